"""Plant plausible mistakes in the oracle and check that a pin catches each.

Each mutant is one textual edit of ``oracle/attention.py``, executed as a
fresh module and swapped into the ``oracle`` package for the duration of the
test (CPU only; nothing on the GPU side is involved).
"""

import importlib.util
import os
import types

import pytest

import oracle
import oracle_pins

SRC_PATH = os.path.join(os.path.dirname(oracle.__file__), "attention.py")

MUTANTS = {
    "dropped_scale": ("return scale * (q @ k.T)", "return (q @ k.T)"),
    "flipped_sign": ("return scale * (q @ k.T)", "return -scale * (q @ k.T)"),
    "squared_scale": ("return scale * (q @ k.T)", "return scale * scale * (q @ k.T)"),
    "causal_off_by_one": ("keys[None, :] <= rows[:, None]", "keys[None, :] < rows[:, None]"),
    "causal_transposed": ("keys[None, :] <= rows[:, None]", "keys[None, :] >= rows[:, None]"),
    "causal_ignored": ("    if not causal:\n        return np.ones", "    if True:\n        return np.ones"),
    "pv_uses_keys": ("= P @ v[:kmax]", "= P @ k[:kmax]"),
    "lse_log2": ("M + np.log(np.where(L > 0, L, 1.0))", "M + np.log2(np.where(L > 0, L, 1.0))"),
    "lse_drops_max": ("M + np.log(np.where(L > 0, L, 1.0))", "np.log(np.where(L > 0, L, 1.0))"),
    "denominator_counts_masked": ("    L = E.sum(axis=1)", "    L = np.exp(s - shift[:, None]).sum(axis=1)"),
    "unnormalised_p": ("E / np.where(finite, L, 1.0)[:, None]", "E"),
    "double_shift": ("np.exp(masked - shift[:, None])", "np.exp(masked - 2 * shift[:, None])"),
    "causal_prefix_short": ("int(min(Sk, r.max() + 1 + causal_offset))", "int(min(Sk, r.max() + causal_offset))"),
    "forward_swaps_kv": ("attention_head(q[b, :, h, :], k[b, :, g, :], v[b, :, g, :]",
                         "attention_head(q[b, :, h, :], v[b, :, g, :], k[b, :, g, :]"),
    "gqa_interleaved_heads": ("return h // (H // H_kv)", "return h % H_kv"),
    "gqa_ignores_grouping": ("            g = kv_head(h, H, H_kv)\n            O[b, :, h, :]",
                             "            g = min(h, H_kv - 1)\n            O[b, :, h, :]"),
    "varlen_ignores_grouping": ("            g = kv_head(h, H, H_kv)\n            if k1 <= k0:",
                                "            g = min(h, H_kv - 1)\n            if k1 <= k0:"),
    "fp8_drops_descale_v": ("v = e4m3_to_f64(v8) * float(descale_v)", "v = e4m3_to_f64(v8)"),
    "fp8_descale_k_for_q": ("q = e4m3_to_f64(q8) * float(descale_q)", "q = e4m3_to_f64(q8) * float(descale_k)"),
    "bwd_rows_drop_d": ("dS = P * (dO[rows] @ v[krows].T - D[rows][:, None])", "dS = P * (dO[rows] @ v[krows].T)"),
    "bwd_rows_dv_one_chunk": ("        dV += P.T @ dO[rows]", "        dV = P.T @ dO[rows]"),
    "offset_ignored": ("keys[None, :] <= rows[:, None] + causal_offset", "keys[None, :] <= rows[:, None]"),
    "offset_negated": ("keys[None, :] <= rows[:, None] + causal_offset", "keys[None, :] <= rows[:, None] - causal_offset"),
    "forward_drops_offset": ("                                                         causal_offset=causal_offset)",
                             "                                                         causal_offset=0)"),
    "rows_drop_offset": ("rows=rows, causal_offset=causal_offset)", "rows=rows)"),
    "bwd_dv_untransposed": ("    dV = P.T @ dO", "    dV = P @ dO[:P.shape[1]] if P.shape[0] >= P.shape[1] else P.T @ dO * 0.5"),
    "bwd_ds_drops_d": ("    dS = P * (dP - D[:, None])", "    dS = P * dP"),
    "bwd_group_overwrites": ("            dK[b, :, g] += dk", "            dK[b, :, g] = dk"),
    "bwd_dk_unscaled": ("scale * (dS.T @ q), dV, D", "(dS.T @ q), dV, D"),
    "bwd_dq_uses_v": ("return scale * (dS @ k), scale", "return scale * (dS @ v), scale"),
    "bwd_dq_unscaled": ("return scale * (dS @ k), scale", "return (dS @ k), scale"),
    "bwd_dv_from_dp": ("    dV = P.T @ dO", "    dV = (P * (dO @ v.T)).T @ dO"),
    "varlen_global_offset": ("        off = (k1 - k0) - (q1 - q0) if (causal and bottom_right) else 0",
                             "        off = (cu_k[-1] - cu_q[-1]) if (causal and bottom_right) else 0"),
    "varlen_keys_from_start": ("k[k0:k1, g, :], v[k0:k1, g, :], scale", "k[0:k1 - k0, g, :], v[0:k1 - k0, g, :], scale"),
    "varlen_lse_row_major": ("O[q0:q1, h, :], LSE[h, q0:q1] = attention_head", "O[q0:q1, h, :], LSE[h, 0:q1 - q0] = attention_head"),
    "forward_lse_transposed_heads": ("LSE[b, h, :] = attention_head", "LSE[b, (h + 1) % H, :] = attention_head"),
    "combine_plain_mean": ("O = (w[..., None] * Os).sum(axis=0)", "O = Os.mean(axis=0)"),
    "combine_lse_max_only": ("LSE = np.where(finite, shift + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)",
                             "LSE = np.where(finite, shift, -np.inf)"),
}


def _load_mutant(old, new):
    with open(SRC_PATH) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    mod = types.ModuleType("oracle_attention_mutant")
    exec(compile(src.replace(old, new), SRC_PATH + ":mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    mod = _load_mutant(*MUTANTS[name])
    for fn in ("attention_forward", "attention_head", "attention_rows", "attention_varlen", "attention_backward",
               "attention_backward_head", "head_probabilities", "head_scores", "kv_head", "visible_mask",
               "combine_partials", "attention_forward_fp8", "e4m3_to_f64", "attention_backward_rows"):
        monkeypatch.setattr(oracle, fn, getattr(mod, fn))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_source_passes_all_pins(monkeypatch):
    mod = _load_mutant("ROW_CHUNK = 1024", "ROW_CHUNK = 1024")
    for fn in ("attention_forward", "attention_head", "head_probabilities", "head_scores",
               "visible_mask", "combine_partials"):
        monkeypatch.setattr(oracle, fn, getattr(mod, fn))
    for pin in oracle_pins.ALL_PINS:
        pin()
