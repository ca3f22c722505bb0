// Attention forward kernels for head dim 128, causal mask, every compiled exp2 split.
#include "attn_launch.h"

namespace attn {
cudaError_t launch_fwd_d128_causal(const LaunchArgs& a) { return launch_variant<128, true>(a); }
}  // namespace attn
