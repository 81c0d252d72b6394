"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle.c, applies one plausible mistake (a dropped term, a
wrong sign, a transposed operand, a wrong index, a broken tie rule ...),
compiles the copy on the CPU and runs the pins against it.  At least one pin
must fail for every mistake; that is what makes the pins worth trusting.
Every edit keeps all memory accesses in bounds.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import pins

MUTANTS = {
    "swiglu_drops_up": ("a[j] = silu(h[j]) * h[I + j];", "a[j] = silu(h[j]);"),
    "swiglu_gate_up_swapped": ("a[j] = silu(h[j]) * h[I + j];", "a[j] = silu(h[I + j]) * h[j];"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "gateup_lora_unscaled": ("h[j] += scaling * s;", "h[j] += s;"),
    "down_lora_dropped": ("d[o] += scaling * s;", "d[o] += 0.0 * s;"),
    "A13_transposed": ("s += xm[i] * bf16_bits_to_double(A[(size_t)q * H + i]);",
                       "s += xm[i] * bf16_bits_to_double(A[(size_t)i * r + q]);"),
    "B2_transposed": ("s += t2[q] * bf16_bits_to_double(B[(size_t)o * r + q]);",
                      "s += t2[q] * bf16_bits_to_double(B[(size_t)q * H + o]);"),
    "B13_wrong_expert": ("const uint16_t* B = B13 + ((size_t)l * E_tot + e) * 2 * I * r;",
                         "const uint16_t* B = B13 + ((size_t)l * E_tot + 0) * 2 * I * r;"),
    "out_scale_dropped": ("y[(size_t)m * H + o] = (double)out_scale * acc[o];",
                          "y[(size_t)m * H + o] = acc[o];"),
    "combine_weight_dropped": ("acc[o] += w * d[o];", "acc[o] += d[o];"),
    "ties_to_higher_id": ("return id_a < id_b;", "return id_a > id_b;"),
    "shared_weight_rsf": ("w[top_k + j] = 1.0 / (double)routed_scaling_factor;",
                          "w[top_k + j] = (double)routed_scaling_factor;"),
    "shared_id_offset": ("ids[top_k + j] = E + j;", "ids[top_k + j] = E - 1 + j;"),
    "softmax_never_renormalises": ("if (renormalize) {\n                for (int k = 0; k < top_k; ++k) denom",
                                   "if (0) {\n                for (int k = 0; k < top_k; ++k) denom"),
    "sigmoid_weight_includes_bias": ("w[k] = 1.0 / (1.0 + exp(-(double)l[ids[k]]));",
                                     "w[k] = (double)key[ids[k]];"),
    "sigmoid_key_ignores_bias": ("key[e] = sg + (bias ? bias[e] : 0.0f);", "key[e] = sg;"),
    "align_descending_slots": ("for (long f = 0; f < slots; ++f)\n            if (topk_ids[f] == e)",
                               "for (long f = slots - 1; f >= 0; --f)\n            if (topk_ids[f] == e)"),
    "align_no_padding": ("while ((pos - start) % block_m != 0) sorted_ids[pos++] = sentinel;", ""),
    "align_tail_not_filled": ("for (long b = pos / block_m; b < max_padded / block_m; ++b) expert_ids[b] = -1;", ""),
    # MXFP8
    "mx_shared_exponent_off_by_one": ("se = (e - 1) - 8;", "se = (e - 1) - 7;"),
    "mx_rounds_toward_zero": ("const double q = rint(a / step) * step;", "const double q = floor(a / step) * step;"),
    "mx_no_saturation": ("if (!(a < 448.0)) return sign | 0x7E;", "if (!(a < 480.0)) return sign | 0x7E;"),
    "mx_negative_zero_unsigned": ("if (q == 0.0) return sign;", "if (q == 0.0) return 0;"),
    "mx_subnormals_flushed": ("if (q < ldexp(1.0, -6)) return sign | (uint8_t)(q / ldexp(1.0, -9));",
                              "if (q < ldexp(1.0, -6)) return sign;"),
    "mx_decode_bias_8": ("v = ldexp(1.0 + m / 8.0, E - 7);", "v = ldexp(1.0 + m / 8.0, E - 8);"),
    "mx_swiglu_output_not_quantized": ("mx_round_trip(act, I, actq);",
                                       "for (int j = 0; j < I; ++j) actq[j] = act[j];"),
    "mx_x_not_quantized": ("mx_round_trip(xm, H, xq);", "for (int i = 0; i < H; ++i) xq[i] = xm[i];"),
    "mx_adapter_reads_quantized_x": ("expert_mx(xq, xm,", "expert_mx(xq, xq,"),
    "mx_shrink_not_rounded": ("ts[q] = bf16_round(scaling * acc_q);", "ts[q] = scaling * acc_q;"),
    "mx_scale_of_next_block": ("sv[S2[(size_t)o * (I / 32) + j / 32]]", "sv[S2[(size_t)o * (I / 32) + (j / 32 + 1) % (I / 32)]]"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle._SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, source, name):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique/found"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(source.replace(old, new))
    so = str(tmp_path / "liboracle_mutant.so")
    oracle.build(str(src), so)
    lib = oracle.load(so)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as exc:  # noqa: PERF203
            caught.append(pin.__name__)
            break
    assert caught, f"no pin caught the planted mistake {name}"
