"""Mutation check of the oracle's pins (run by hand, not collected by pytest):

    python tests/oracle_mutants.py [name ...]

Each mutant plants one plausible mistake (a wrong bias, tie rule, constant,
index, direction, sign, bound or bit order) in a copy of
oracle/nvfp4_oracle.c, in a temporary directory, and runs the CPU pin tests
(tests/test_oracle_*.py) against that copy. A pin set that catches every
mutant leaves no such mistake unnoticed. The one mutant expected to survive
changes the fixed fp32 order of the in-block sums, a reading the pages leave
open (the GPU parity tests hold the kernels to it). Exit status 1 when any
other mutant survives. Nothing here touches the repository's own files or a
GPU."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, replacement[, which occurrence])
MUTANTS = [
    ("e2m1_bias", "return (1.0 + f / 2.0) * ldexp(1.0, e - 1);", "return (1.0 + f / 2.0) * ldexp(1.0, e - 2);"),
    ("e2m1_sub", "if (e == 0) return f * 0.5;", "if (e == 0) return f * 1.0;"),
    ("e4m3_bias", "return (1.0 + f / 8.0) * ldexp(1.0, e - 7);", "return (1.0 + f / 8.0) * ldexp(1.0, e - 8);"),
    ("e4m3_sub", "if (e == 0) return f / 8.0 * ldexp(1.0, -6);", "if (e == 0) return f / 8.0 * ldexp(1.0, -7);"),
    ("ue5m3_bias", "ldexp(1.0, e - 15)", "ldexp(1.0, e - 16)"),
    ("ue5m3_sub", "ldexp(1.0, -14)", "ldexp(1.0, -15)"),
    ("rne_ties_up", "return (lo % 2 == 0) ? lo : hi;", "return hi;"),
    ("rne_ties_down", "return (lo % 2 == 0) ? lo : hi;", "return lo;"),
    ("rne_sat", "if (!(a < val(n - 1))) return n - 1;", "if (!(a < val(n - 1))) return n - 2;"),
    ("bf16_trunc", "return (uint16_t)((u + 0x7FFFu + lsb) >> 16);", "return (uint16_t)(u >> 16);"),
    ("bf16_ties_away", "return (uint16_t)((u + 0x7FFFu + lsb) >> 16);", "return (uint16_t)((u + 0x8000u) >> 16);"),
    ("philox_m0", "0xD2511F53u", "0xD2511F55u"),
    ("philox_m1", "0xCD9E8D57u", "0xCD9E8D55u"),
    ("philox_rounds", "round < 10", "round < 9"),
    ("philox_key0", "k0 += 0x9E3779B9u;", "k0 += 0x9E3779B7u;"),
    ("philox_key1", "k1 += 0xBB67AE85u;", "k1 += 0xBB67AE87u;"),
    ("philox_prod", "uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;", "uint32_t n0 = (uint32_t)(p0 >> 32) ^ c1 ^ k0;"),
    ("philox_out", "out[0] = c0; out[1] = c1;", "out[0] = c1; out[1] = c0;"),
    ("sr_group", "uint64_t j = idx >> 3;", "uint64_t j = idx >> 2;"),
    ("sr_half", "return (idx & 1) ? (word >> 16) : (word & 0xFFFFu);", "return (idx & 1) ? (word & 0xFFFFu) : (word >> 16);"),
    ("sr_word", "uint32_t word = w[(idx & 7) >> 1];", "uint32_t word = w[idx & 3];"),
    ("sr_ctr", "{(uint32_t)j, (uint32_t)(j >> 32), dir, 0u}", "{(uint32_t)j, (uint32_t)(j >> 32), 0u, dir}"),
    ("sr_key", "uint32_t key[2] = {seed, step};", "uint32_t key[2] = {step, seed};"),
    ("e2m1_sr_cmp", "return (uint8_t)(s | (u < p ? lo + 1 : lo));", "return (uint8_t)(s | (u <= p ? lo + 1 : lo));", 0),
    ("e2m1_sr_u", "/ 65536.0", "/ 65535.0", 0),
    ("e2m1_sr_sat", "if (!(a < 6.0)) return (uint8_t)(s | 7);", "if (!(a < 6.0)) return (uint8_t)(s | 6);"),
    ("e2m1_sr_v", "double u = (double)(v16 & 0xFFFFu) / 65536.0;", "double u = 1.0 - (double)(v16 & 0xFFFFu) / 65536.0;", 0),
    ("g_den", "float den = 6.0f * M;", "float den = 4.0f * M;"),
    ("M_fos", "float M = scale_max > 0.0f ? scale_max : (fos ? 256.0f : 448.0f);", "float M = scale_max > 0.0f ? scale_max : 448.0f;", 0),
    ("cand_k", "float den = k * g;", "float den = 6.0f * g;"),
    ("cand_div", "float y = x[i] * inv;", "float y = x[i] / c->d;"),
    ("err_sign", "e[i] = fmaf(-c->qv[i], c->d, x[i]);", "e[i] = fmaf(c->qv[i], c->d, x[i]);"),
    ("fos_strict", "if (sse[1] < sse[0])", "if (sse[1] <= sse[0])"),
    ("fos_rule", "return rule == 1 ? c->sae : (rule == 2 ? c->emax : c->sse);", "return rule == 2 ? c->sae : (rule == 1 ? c->emax : c->sse);"),
    ("block_amax_abs", "float a = fabsf(x[i]);\n    if (a > amax) amax = a;", "float a = x[i];\n    if (a > amax) amax = a;"),
    ("sr_elem_idx", "v16[i] = orc_sr_bits(seed, step, dir, idx0 + (uint64_t)i);", "v16[i] = orc_sr_bits(seed, step, dir, idx0 + (uint64_t)(15 - i));"),
    ("choice_bit", "choice[s * W + b / 32] |= 1u << (b % 32);", "choice[s * W + b / 32] |= 1u << (31 - b % 32);"),
    ("pack_nibble", "codes[(e0 + i) / 2] = (uint8_t)((q[i] & 15) | ((q[i + 1] & 15) << 4));", "codes[(e0 + i) / 2] = (uint8_t)((q[i + 1] & 15) | ((q[i] & 15) << 4));"),
    ("col_dir", "encode_rows(xt, S, C, R, g, fmt, rounding, fos, rule, seed, step, 1,", "encode_rows(xt, S, C, R, g, fmt, rounding, fos, rule, seed, step, 0,"),
    ("col_transpose", "xt[s * R * C + c * R + r] = xf[s * R * C + r * C + c];", "xt[s * R * C + c * R + r] = xf[s * R * C + r * C + (C - 1 - c)];", 0),
    ("amax_inf", "if (a >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;", "if (a > 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;"),
    ("fq_post", "xq[e] = orc_f32_to_bf16(so * q);", "xq[e] = orc_f32_to_bf16(sp * q);"),
    ("ste_in", "int in = (r >= -6.0f) && (r <= 6.0f);", "int in = (r > -6.0f) && (r < 6.0f);"),
    ("ste_tied", "t[i] = in ? (q[i] - r) : q[i];", "t[i] = in ? (q[i] - r) : 0.0f;"),
    ("ste_pre_sign", "gs_pre[b] = -a * block_sum(g, rin);", "gs_pre[b] = a * block_sum(g, rin);"),
    ("ste_gx_gate", "gx[e] = orc_f32_to_bf16(in ? g[i] * a : 0.0f);", "gx[e] = orc_f32_to_bf16(g[i] * a);"),
    ("ste_post", "gs_post[b] = block_sum(g, q);", "gs_post[b] = block_sum(g, rin);"),
    ("e4m3_sr_sat", "if (!(a < 448.0)) return (uint8_t)(s | 0x7E);", "if (!(a < 448.0)) return (uint8_t)(s | 0x7D);"),
    ("e4m3_sr_cmp", "return (uint8_t)(s | (u < p ? lo + 1 : lo));", "return (uint8_t)(s | (u <= p ? lo + 1 : lo));", 1),
    ("mx_exp_round", "(2.0f * m > 1.75f ? 1 : 0)", "(2.0f * m >= 1.75f ? 1 : 0)"),
    ("mx_exp_off", "int e = (e2 - 1) - 8 +", "int e = (e2 - 1) - 9 +"),
    ("mx_exp_clamp", "if (e < -127) e = -127;", "if (e < -126) e = -126;"),
    ("mx_exp_zero", "if (!(amax > 0.0f)) return -127;", "if (!(amax > 0.0f)) return 0;"),
    ("rq_mx_dir", "orc_mx_encode(xt + e0, R, rounding, seed, step, 2,", "orc_mx_encode(xt + e0, R, rounding, seed, step, 1,"),
    ("rq_nv_dir", "encode_rows(xt, S, C, R, g, dst_fmt, rounding, dst_fos, dst_rule, seed, step, 2,", "encode_rows(xt, S, C, R, g, dst_fmt, rounding, dst_fos, dst_rule, seed, step, 1,"),
    ("dq_nibble", "uint8_t c = (e & 1) ? (codes[e / 2] >> 4) : (codes[e / 2] & 15);", "uint8_t c = (e & 1) ? (codes[e / 2] & 15) : (codes[e / 2] >> 4);"),
    ("dq_scale_idx", "float d = orc_scale_value(fmt, scales[e / 16]) * g;", "float d = orc_scale_value(fmt, scales[e / 32]) * g;"),
    ("rq_M", "float M = dst_scale_max > 0.0f ? dst_scale_max : (dst_fos ? 256.0f : 448.0f);", "float M = dst_scale_max > 0.0f ? dst_scale_max : 448.0f;"),
    ("fp8_unit_M", "global_decode_scale(gamax, 448.0f, &u->g);", "global_decode_scale(gamax, 256.0f, &u->g);"),
    ("mse_ties", "if (c == 1 || sse < best_sse)", "if (c == 1 || sse <= best_sse)"),
    ("mse_range", "for (int c = 1; c <= 126; ++c)", "for (int c = 1; c <= 125; ++c)"),
    ("mse_err", "e[i] = fmaf(-q, s, x[i]);", "e[i] = fmaf(q, s, x[i]);"),
    ("export_scale", "scales[b] = so >= 0.0f ? q8_code(so, &u) : 0;", "scales[b] = so >= 0.0f ? q8_code(s_pre[b], &u) : 0;"),
    ("export_inv", "float inv = 1.0f / sp[b];", "float inv = 1.0f / s_pre[b];"),
    ("q8_rg", "static uint8_t q8_code(float s, const fp8_unit* u) { return orc_scale_encode(0, s * u->rg); }", "static uint8_t q8_code(float s, const fp8_unit* u) { return orc_scale_encode(0, s / u->g * 0.5f); }"),
    ("fp8_status", "!(sp_q[b] >= FLT_MIN)", "!(sp_q[b] >= 0.0f)"),
    ("tile_amax", "for (int cc = 0; cc < 16; ++cc) {", "for (int cc = 0; cc < 8; ++cc) {"),
    ("tile_dir", "v16[i] = orc_sr_bits(seed, step, 0, (uint64_t)(e0 + i));", "v16[i] = orc_sr_bits(seed, step, 1, (uint64_t)(e0 + i));"),
    ("tile_k", "encode_candidate(xb, amax, g, 6.0f, fmt, rounding, v16, &cd);", "encode_candidate(xb, amax, g, 4.0f, fmt, rounding, v16, &cd);"),
    ("tile_col_scale", "if (c_scales && r % 16 == 0) c_scales[t / 16] = r_scales[e / 16];", "if (c_scales && r % 16 == 0) c_scales[t / 16] = r_scales[(e + C) / 16 % (R * C / 16)];"),
    ("mx_rows_dir", "orc_mx_encode(xf + e0, C, rounding, seed, step, 0,", "orc_mx_encode(xf + e0, C, rounding, seed, step, 2,"),
    ("mx_cols_dir", "orc_mx_encode(xt + e0, R, rounding, seed, step, 1, (uint64_t)e0, c_codes", "orc_mx_encode(xt + e0, R, rounding, seed, step, 0, (uint64_t)e0, c_codes"),
    ("mx_blk_amax", "if (fabsf(vb[i]) > amax) amax = fabsf(vb[i]);", "if (vb[i] > amax) amax = vb[i];"),
    ("block_sum_order", "acc[p] = fmaf(a[i], b[i], acc[p]);", "acc[0] = fmaf(a[i], b[i], acc[0]);"),
    ("ue5m3_range", "nearest_index((double)t, ue5m3_mag, 256)", "nearest_index((double)t, ue5m3_mag, 255)"),
    ("e4m3_scale_range", "nearest_index((double)t, e4m3_mag, 127)", "nearest_index((double)t, e4m3_mag, 126)"),
    ("rden_clamp", "if (rden > FLT_MAX) rden = FLT_MAX;", ""),
    ("gamax_zero", "if (gamax == 0.0f) { *g = 1.0f; return 0; }", "if (gamax == 0.0f) { *g = 0.5f; return 0; }"),
    ("bad_amax", "if (!(gamax >= 0.0f) || isinf(gamax))", "if (isnan(gamax))"),
    ("scale_ok_pre", "if (!(s_pre >= FLT_MIN) || !(s_pre <= FLT_MAX)) return 0;", "if (!(s_pre > 0.0f)) return 0;"),
    ("quant_nonfinite", "if ((x[i] & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;\n    xf[i] = orc_bf16_to_f32(x[i]);", "xf[i] = orc_bf16_to_f32(x[i]);", 0),
    ("dq_bf16", "dq[i] = orc_f32_to_bf16(dqf[i]);", "dq[i] = (uint16_t)(f2u(dqf[i]) >> 16);"),
    ("mae_abs", "acc[p] = acc[p] + fabsf(e[8 * h + p + 2 * j]);", "acc[p] = acc[p] + e[8 * h + p + 2 * j];"),
    ("maxerr_first", "if (fabsf(e[i]) > m) m = fabsf(e[i]);", "if (fabsf(e[i]) > m) m = e[i];"),
    ("amax_slice", "uint16_t a = x[s * n + i] & 0x7FFFu;", "uint16_t a = x[i] & 0x7FFFu;"),
    ("amax_sign", "uint16_t a = x[s * n + i] & 0x7FFFu;", "uint16_t a = x[s * n + i] & 0xFFFFu;"),
    ("tied_scale", "float sp = s_pre[b], so = s_post ? s_post[b] : s_pre[b];", "float sp = s_pre[b], so = s_post ? s_post[b] : 1.0f;"),
    ("rq_choice", "out_scales, out_choice, NULL);", "out_scales, NULL, NULL);"),
    ("export_nibble", "codes[e / 2] = (uint8_t)((q0 & 15) | ((q1 & 15) << 4));", "codes[e / 2] = (uint8_t)((q1 & 15) | ((q0 & 15) << 4));"),
    ("tile_M", "float M = scale_max > 0.0f ? scale_max : 448.0f;", "float M = scale_max > 0.0f ? scale_max : 256.0f;"),
    ("tile_dq", "r_dq[e0 + i] = orc_f32_to_bf16(cd.qv[i] * cd.d);", "r_dq[e0 + i] = orc_f32_to_bf16(cd.qv[i]);"),
    ("mx_scale_idx", "r_scales + e0 / 32);", "r_scales + e0 / 16);"),
    ("dq_M_fos", "float M = scale_max > 0.0f ? scale_max : (fos ? 256.0f : 448.0f);", "float M = scale_max > 0.0f ? scale_max : 448.0f;", 1),
    ("fq_nonfinite", "      if ((x[e] & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;\n      float r = orc_bf16_to_f32(x[e]) * inv;", "      float r = orc_bf16_to_f32(x[e]) * inv;"),
    ("sg_nonfinite_g", "if ((x[e] & 0x7FFFu) >= 0x7F80u || (gq[e] & 0x7FFFu) >= 0x7F80u)", "if ((x[e] & 0x7FFFu) >= 0x7F80u)"),
    ("dq_nonfinite", "if (!isfinite(out[e])) st |= ORC_ST_NONFINITE_INPUT;", ""),
    ("mse_nonfinite", "      if ((h & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;\n      xb[i] = orc_bf16_to_f32(h);", "      xb[i] = orc_bf16_to_f32(h);"),
    ("export_nonfinite", "if ((x[e] & 0x7FFFu) >= 0x7F80u || (x[e + 1] & 0x7FFFu) >= 0x7F80u)", "if ((x[e] & 0x7FFFu) >= 0x7F80u)"),
    ("tile_nonfinite", "            if ((h & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;\n            float a = fabsf", "            float a = fabsf"),
    ("mx_nonfinite", "if ((x[i] & 0x7FFFu) >= 0x7F80u) st |= ORC_ST_NONFINITE_INPUT;\n    xf[i] = orc_bf16_to_f32(x[i]);\n  }\n  if (blocks & 1)\n    for", "xf[i] = orc_bf16_to_f32(x[i]);\n  }\n  if (blocks & 1)\n    for"),
    ("rq_src_fmt", "int st = orc_dequant(src_fmt, src_scale_max, src_fos,", "int st = orc_dequant(0, src_scale_max, src_fos,"),
    ("rq_src_M", "int st = orc_dequant(src_fmt, src_scale_max, src_fos,", "int st = orc_dequant(src_fmt, 0.0f, src_fos,"),
    ("quant_scale_max", "float M = scale_max > 0.0f ? scale_max : (fos ? 256.0f : 448.0f);", "float M = fos ? 256.0f : 448.0f;", 0),
    ("fp8_post_sign", "!(so >= 0.0f && so <= FLT_MAX)", "!(so <= FLT_MAX)"),
    ("tile_col_nibble", "if (t & 1) c_codes[t / 2] = (uint8_t)((c_codes[t / 2] & 0x0F) | (q << 4));", "if (!(t & 1)) c_codes[t / 2] = (uint8_t)((c_codes[t / 2] & 0x0F) | (q << 4));"),
    ("rq_transpose", "for (int64_t c = 0; c < C; ++c) xt[s * R * C + c * R + r] = xh[s * R * C + r * C + c];", "for (int64_t c = 0; c < C; ++c) xt[s * R * C + c * R + r] = xh[s * R * C + r * C + (C - 1 - c)];"),
    ("mx_scale_sign", "float y = ldexpf(vb[i], -e);", "float y = ldexpf(vb[i], e);"),
    ("tile_sr_idx", "if (rounding) v16[i] = orc_sr_bits(seed, step, 0, (uint64_t)(e0 + i));", "if (rounding) v16[i] = orc_sr_bits(seed, step, 0, (uint64_t)(e0 + 15 - i));"),
    ("tile_amax_row", "for (int rr = 0; rr < 16; ++rr)\n          for (int cc = 0; cc < 16; ++cc)", "for (int rr = 0; rr < 1; ++rr)\n          for (int cc = 0; cc < 16; ++cc)"),
]

EXPECTED_SURVIVORS = {"block_sum_order"}


def _prepare(base, name, old, new, occ):
    d = os.path.join(base, name)
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(d, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(d, "tests"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copytree(os.path.join(ROOT, "nvfp4_block_scaled_02_gb300"),
                    os.path.join(d, "nvfp4_block_scaled_02_gb300"),
                    ignore=shutil.ignore_patterns("_build", "*.so", "__pycache__", "csrc"))
    p = os.path.join(d, "oracle", "nvfp4_oracle.c")
    with open(p) as f:
        s = f.read()
    assert s.count(old) > occ, (name, "text not found")
    i = -1
    for _ in range(occ + 1):
        i = s.index(old, i + 1)
    with open(p, "w") as f:
        f.write(s[:i] + new + s[i + len(old):])
    return d


def _run(base, m):
    name, old, new = m[:3]
    d = _prepare(base, name, old, new, m[3] if len(m) > 3 else 0)
    tests = sorted("tests/" + t for t in os.listdir(os.path.join(d, "tests"))
                   if t.startswith("test_oracle_") and t.endswith(".py"))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *tests], cwd=d, capture_output=True, text=True, timeout=1800)
    first = next((l for l in r.stdout.splitlines() if l.startswith("FAILED")), "")
    return name, r.returncode != 0, first


def main(names):
    ms = [m for m in MUTANTS if not names or m[0] in names]
    base = tempfile.mkdtemp(prefix="oracle_mutants_")
    bad = []
    try:
        with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
            for name, caught, first in ex.map(lambda m: _run(base, m), ms):
                print(f"{'caught  ' if caught else 'SURVIVED'} {name:18s} {first[:100]}", flush=True)
                if not caught and name not in EXPECTED_SURVIVORS:
                    bad.append(name)
    finally:
        shutil.rmtree(base, ignore_errors=True)
    print(f"{len(ms) - len(bad)} of {len(ms)} as expected; unexpected survivors: {bad or 'none'}")
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
