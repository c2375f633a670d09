"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Each mutant is the oracle's C source with one textual change, compiled into a
temporary directory on the CPU.  A mutant that every pin passes would mean the
pins cannot see that kind of mistake.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "silu_sign": ("z / (1.0 + exp(-z))", "z / (1.0 + exp(z))"),
    "bias_dropped": ("if (bias) acc += (double)bias[e];", ""),
    "tie_to_higher_id": ("logits[e] > logits[best]", "logits[e] >= logits[best]"),
    "no_renormalisation": ("w[s] = exp(logits[idx[s]] - lmax) / den;", "w[s] = exp(logits[idx[s]] - lmax);"),
    "softmax_over_all": ("for (int s = 0; s < k; ++s) den += exp(logits[idx[s]] - lmax);",
                         "for (int e2 = 0; e2 < E; ++e2) den += exp(logits[e2] - lmax);"),
    "q_unsigned": ("(int)(int8_t)blk[2 + j]", "(int)blk[2 + j]"),
    "scale_byte_order": ("blk[0] | (blk[1] << 8)", "blk[1] | (blk[0] << 8)"),
    "half_exponent": ("expo - 25", "expo - 24"),
    "gate_up_swapped": ("h[r] = silu(g[r]) * u[r];", "h[r] = silu(u[r]) * g[r];"),
    "residual_dropped": ("residual ? xt[o] + acc[o] : acc[o]", "acc[o]"),
    "bucket_unstable": ("int p = off[e] + cnt[e]++;", "int p = off[e + 1] - 1 - cnt[e]++;"),
    "combine_slot_shift": ("int e = it[s];", "int e = it[(s + 1) % k];"),
    "block_stride": ("#define ORACLE_Q8_BLOCK_BYTES 34", "#define ORACLE_Q8_BLOCK_BYTES 36"),
    "q4_nibble_swap": ("int lo = q4b[2 + j] & 0x0F, hi = q4b[2 + j] >> 4;",
                       "int hi = q4b[2 + j] & 0x0F, lo = q4b[2 + j] >> 4;"),
    "q4_offset": ("(double)(hi - 8) * d4", "(double)(hi - 7) * d4"),
    "q4_interleaved": ("w[b * ORACLE_Q8_BLOCK_ELEMS + j] = (double)(lo - 8) * d4;\n"
                       "            w[b * ORACLE_Q8_BLOCK_ELEMS + 16 + j]",
                       "w[b * ORACLE_Q8_BLOCK_ELEMS + 2 * j] = (double)(lo - 8) * d4;\n"
                       "            w[b * ORACLE_Q8_BLOCK_ELEMS + 2 * j + 1]"),
    "q4_block_stride": ("#define ORACLE_Q4_BLOCK_BYTES 18", "#define ORACLE_Q4_BLOCK_BYTES 17"),
    "bf16_round_half_up": ("bits = (bits + 0x7fffu + lsb) & 0xffff0000u;", "bits = (bits + 0x8000u) & 0xffff0000u;"),
    "bf16_not_applied": ("expert_input_bf16 ? to_bf16_via_f32(xt[j]) : xt[j]", "xt[j]"),
    "forced_selection_ignored": ("forced_idx ? forced_idx + (size_t)t * k : NULL", "NULL"),
    "router_index": ("const float* wr = Wr + (size_t)e * dm;", "const float* wr = Wr + (size_t)(E - 1 - e) * dm;"),
    "route_idx_stride": ("NULL, idx + (size_t)t * k, w + (size_t)t * k, lg)",
                         "NULL, idx + (size_t)t, w + (size_t)t * k, lg)"),
    "route_weight_stride": ("NULL, idx + (size_t)t * k, w + (size_t)t * k, lg)",
                            "NULL, idx + (size_t)t * k, w + (size_t)t, lg)"),
    "route_logits_stride": ("            memcpy(logits + (size_t)t * E, lg, sizeof(double) * (size_t)E);\n        free(lg);",
                            "            memcpy(logits + (size_t)t * k, lg, sizeof(double) * (size_t)E);\n        free(lg);"),
    "route_token_offset": ("route_token(x + (size_t)t * dm, dm,", "route_token(x + (size_t)t * E, dm,"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/absent"
    mpath = os.path.join(tmp_path, "mutant.c")
    with open(mpath, "w") as fh:
        fh.write(src.replace(old, new))
    lib = os.path.join(tmp_path, f"liboracle_{name}.so")
    oracle.build(mpath, lib, openmp=False)
    orc = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
