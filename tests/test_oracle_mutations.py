"""Plant plausible mistakes in copies of the oracle source; the pins must catch each one.

This shows the pins are strong enough: a dropped term, a wrong sign, a wrong
index or a swapped operand anywhere in the oracle makes at least one pin fail.
The planted copies are compiled into a temporary directory on the CPU; the
oracle itself is untouched.
"""
import pytest

import oracle.oracle as orc
from _pins import ALL_PINS

SRC = orc._SRC

MUTATIONS = {
    "recurrence_uses_raw_x": ("h[n] = a * h[n] + delta * Bt[n] * u;", "h[n] = a * h[n] + delta * Bt[n] * xt;"),
    "decay_sign": ("double a = exp(delta * (double)A_d[n]);", "double a = exp(-delta * (double)A_d[n]);"),
    "decay_drops_delta": ("double a = exp(delta * (double)A_d[n]);", "double a = exp((double)A_d[n]);"),
    "input_drops_delta": ("h[n] = a * h[n] + delta * Bt[n] * u;", "h[n] = a * h[n] + Bt[n] * u;"),
    "readout_before_update": ("        y += Ct[n] * h[n];\n", "        y += 0.0;\n"),
    "C_and_B_swapped": ("Ct[n] = widen(Cm, in_dtype, ib + n);", "Ct[n] = widen(Bm, in_dtype, ib + n);"),
    "skip_uses_raw_x": ("y += D_d * u;", "y += D_d * xt;"),
    "skip_dropped": ("y += D_d * u;", "y += 0.0 * u;"),
    "gate_without_silu": ("return y * silu(zt);", "return y * zt;"),
    "conv_current_tap_dropped": ("xc += (double)conv_w_d[W - 1] * xt;", "xc += 0.0 * xt;"),
    "conv_taps_reversed": ("xc += (double)conv_w_d[k] * hist[k];", "xc += (double)conv_w_d[W - 2 - k] * hist[k];"),
    "conv_bias_dropped": ("double xc = conv_b_d;", "double xc = 0.0;"),
    "conv_history_stores_u": ("if (W > 1) hist[W - 2] = xt;", "if (W > 1) hist[W - 2] = u;"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "softplus_branch_sign": ("v + log1p(exp(-v))", "v + log1p(exp(v))"),
    "softplus_drops_bias": ("softplus(dtt + dt_bias_d)", "softplus(dtt)"),
    "state_in_ignored": ("h[n] = ssm_state_in ? ssm_state_in[((int64_t)b * Dn + d) * N + n] : 0.0;",
                         "h[n] = 0.0;"),
    "conv_state_in_ignored": ("hist[k] = conv_state_in ? conv_state_in[((int64_t)b * (W - 1) + k) * Dn + d] : 0.0;",
                              "hist[k] = 0.0;"),
    "decode_conv_state_not_written": (
        "for (int k = 0; k < W - 1; ++k) conv_state[((int64_t)b * (W - 1) + k) * Dn + d] = hist[k];",
        "(void)0;"),
    "chunk_carry_drops_decay": ("carry = Aagg * carry + Bagg;", "carry = carry + Bagg;"),
    "q8_scale_128": ("inv = 127.0f / amax;", "inv = 128.0f / amax;"),
    "q8_ties_away": ("float r = rintf(t);", "float r = roundf(t);"),
    # (widening the clamp is unobservable: |x * inv| <= 127 (1 + 2^-23)^2 < 127.5)
    "q8_clamp_126": ("if (r > 127.0f) r = 127.0f;", "if (r > 126.0f) r = 126.0f;"),
    "q8_per_partial_amax": ("for (int p = 0; p < P; ++p)\n            for (int64_t i = j0; i < j1; ++i) {",
                            "for (int p = 0; p < 1; ++p)\n            for (int64_t i = j0; i < j1; ++i) {"),
    "q8_output_scale": ("float o = (float)s * scale;", "float o = (float)s * inv;"),
    "q8s_absmax_signed": ("const float v = fabsf(widen_f32(x, in_dtype, i));\n            if (v > m) m = v;",
                          "const float v = widen_f32(x, in_dtype, i);\n            if (v > m) m = v;"),
    "q8s_inv_128": ("            inv = 127.0f / a;\n", "            inv = 128.0f / a;\n"),
    "q8s_truncates": ("float r = rintf(widen_f32(x, in_dtype, i) * inv);",
                      "float r = truncf(widen_f32(x, in_dtype, i) * inv);"),
    "q8s_clamp_126": ("r = r > 127.0f ? 127.0f : (r < -127.0f ? -127.0f : r);",
                      "r = r > 126.0f ? 126.0f : (r < -126.0f ? -126.0f : r);"),
    "q8s_sum_skips_last_rank": ("for (int p = 0; p < P; ++p) s += codes[p][i];",
                                "for (int p = 0; p + 1 < P; ++p) s += codes[p][i];"),
    "q8s_scale_of_next_block": ("const float o = (float)s * scales[i / block];",
                                "const float o = (float)s * scales[(i + 1) / block];"),
    "out_proj_W_transposed": ("const double wv = widen(W, in_dtype, n * K + k);",
                              "const double wv = widen(W, in_dtype, k * N + n);"),
    "out_proj_drops_last_k": ("for (int64_t k = 0; k < K; ++k) {\n                const double yv",
                              "for (int64_t k = 0; k < K - 1; ++k) {\n                const double yv"),
    "out_proj_absdot_signed": ("a += fabs(yv) * fabs(wv);", "a += yv * wv;"),
    "out_proj_amax_signed": ("if (fabs(out[i]) > mx) mx = fabs(out[i]);", "if (out[i] > mx) mx = out[i];"),
    "ssd_group_interleaved": ("const int g = h / hpg;", "const int g = h % G;"),
    "ssd_decay_of_group": ("const double a = exp(delta * (double)A[h]);", "const double a = exp(delta * (double)A[g]);"),
    "ssd_input_drops_delta": ("+ delta * xh[p] * Bg[n];", "+ xh[p] * Bg[n];"),
    "ssd_readout_uses_B": ("y += Cg[n] * S[(int64_t)p * N + n];", "y += Bg[n] * S[(int64_t)p * N + n];"),
    "ssd_C_reads_B_channels": ("ch[P + N + n] = (int64_t)H * P + (int64_t)G * N + (int64_t)g * N + n;",
                               "ch[P + N + n] = (int64_t)H * P + (int64_t)g * N + n;"),
    "ssd_skip_dropped": ("y += (double)Dskip[h] * xh[p];", "y += 0.0 * xh[p];"),
    "ssd_dt_of_head_zero": ("widen(dt, in_dtype, row * H + h)", "widen(dt, in_dtype, row * H)"),
    "ssd_gate_offset": ("row * H * P + (int64_t)h * P + p);\n                out", "row * H * P + p);\n                out"),
    "ssd_state_in_ignored": ("S[e] = ssm_state_in ? ssm_state_in[((int64_t)b * H + h) * P * N + e] : 0.0;",
                             "S[e] = 0.0;"),
    "ssd_conv_state_in_ignored": ("hist[c * (W - 1) + k] = conv_state_in ? conv_state_in[((int64_t)b * (W - 1) + k) * Cx + ch[c]] : 0.0;",
                                  "hist[c * (W - 1) + k] = 0.0;"),
    "ssd_conv_history_stores_u": ("if (W > 1) hist[c * (W - 1) + W - 2] = xt;", "if (W > 1) hist[c * (W - 1) + W - 2] = u[c];"),
    "ssd_state_transposed": ("S[(int64_t)p * N + n] = a * S[(int64_t)p * N + n] + delta",
                             "S[(int64_t)p * N + n] = a * S[(int64_t)n * P + p] + delta"),
}


def _caught(lib):
    failures = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            failures.append(f"{pin.__name__}: {str(e)[:80]}")
    return failures


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    text = SRC.read_text()
    assert text.count(old) == 1, f"mutation site for {name} not unique/not found"
    src = tmp_path / "ssm_oracle_mutant.c"
    src.write_text(text.replace(old, new))
    out = orc.build(src, tmp_path / "libmutant.so", force=True)
    failures = _caught(orc.load(out))
    assert failures, f"planted mistake {name!r} passed every pin"
