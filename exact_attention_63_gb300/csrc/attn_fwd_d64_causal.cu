// Attention forward kernels for head dim 64, causal mask, every compiled exp2 split.
#include "attn_launch.h"

namespace attn {
cudaError_t launch_fwd_d64_causal(const LaunchArgs& a) { return launch_variant<64, true>(a); }
}  // namespace attn
