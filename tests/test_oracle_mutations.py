"""Plant a mistake in a copy of the oracle and check that the pins catch it.

Each mutant is the oracle's own C source with one plausible slip (a dropped
term, a wrong sign, a transposed operand or index, a wrong divisor, a wrong
offset), compiled on the CPU into a temporary library; the pin suites then
run against it in a child process and must fail.  The real oracle is never
modified.
"""
import concurrent.futures
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")

MUTANTS = {
    "drop_weight_decay": ("float wd = *w * s->decay;", "float wd = *w;"),
    "update_sign": ("*w = wd - upd;", "*w = wd + upd;"),
    "first_moment_reads_v": ("float a = s->beta1 * *m;", "float a = s->beta1 * *v;"),
    "second_moment_not_squared": ("float e = d * g;", "float e = d;"),
    "drop_bias_correction_2": ("float q = root / s->bc2_sqrt;", "float q = root;"),
    "drop_bias_correction_1": ("out->step_size = (float)(lr / bc1);",
                               "out->step_size = (float)lr;"),
    "eps_inside_sqrt": ("float den = q + s->eps;",
                        "float den = sqrtf(v1 + s->eps) / s->bc2_sqrt;"),
    "grad_index_transposed": ("local = local + oracle_bf16_to_float(G[(int64_t)r * M + j][i]);",
                              "local = local + oracle_bf16_to_float(G[(int64_t)j * R + r][i]);"),
    "divide_by_R_only": ("return acc / denom_rm;", "return acc / (float)R;"),
    "drop_last_rank": ("acc = (r == 0) ? local : acc + local;",
                       "acc = (r == 0) ? local : (r == R - 1 ? acc : acc + local);"),
    "bf16_truncates": ("u += 0x7FFFu + kept_lsb;", "u += 0u * kept_lsb;"),
    "bf16_ties_away": ("u += 0x7FFFu + kept_lsb;", "u += 0x8000u + 0u * kept_lsb;"),
    "shard_offset_off_by_one": ("int64_t lo = (int64_t)r * S;\n        int64_t len = n - lo < S ? n - lo : S;\n        if (len <= 0) continue;",
                                "int64_t lo = (int64_t)r * S + (r > 0);\n        int64_t len = n - lo < S ? n - lo : S;\n        if (len <= 0) continue;"),
    "all_gather_own_replica_only": ("memcpy(P[q] + lo, pshard", "memcpy(P[r] + lo + 0 * q, pshard"),
    "ring_allgather_wrong_chunk": ("int32_t c = ((k + 1 - s) % p + p) % p;\n            int64_t lo = CH_LO(c), hi = CH_HI(c);\n            memcpy(msg",
                                   "int32_t c = ((k - s) % p + p) % p;\n            int64_t lo = CH_LO(c), hi = CH_HI(c);\n            memcpy(msg"),
    "zero2_formula_swapped": ("out[2] = N * bp + N * (bg + bo) / P;",
                              "out[2] = N * (bp + bg) + N * bo / P;"),
    "shard_len_no_roundup": ("return (per + align - 1) / align * align;", "return per + 0 * align;"),
    "sumsq_left_to_right": ("return (double)sumsq_tree(g, n, 0, len);",
                            "float acc = 0.0f; for (int64_t i = 0; i < n; ++i) acc += g[i] * g[i]; return (double)acc + 0.0 * len;"),
    "sumsq_double_accumulation": ("return (double)sumsq_tree(g, n, 0, len);",
                                  "double acc = 0.0; for (int64_t i = 0; i < n; ++i) acc += (double)g[i] * (double)g[i]; return acc + 0.0 * len;"),
    "sumsq_leaf_not_squared": ("float x = g[lo];\n        return x * x;",
                               "float x = g[lo];\n        return fabsf(x);"),
    "clip_coef_without_epsilon": ("double coef = (double)max_norm / (norm + 1e-6);",
                                  "double coef = (double)max_norm / norm;"),
    "clip_condition_inverted": ("if (coef < 1.0) {", "if (coef > 1.0) {"),
    "clip_divides": ("float gi = clip ? g[i] * coef : g[i];", "float gi = clip ? g[i] / coef : g[i];"),
    "skip_ignores_flag": ("if (!isfinite(sumsq) && skip_nonfinite) skipped = 1;",
                          "if (!isfinite(sumsq) || skip_nonfinite < 0) skipped = 1;"),
    "zero3_owner_off_by_one": ("int32_t owner = (int32_t)(i / S);", "int32_t owner = (int32_t)((i + 1) / S);"),
    "zero3_counts_every_microbatch": ("if (recv && k % M == 0 && k / M != r) recv[r] += len;",
                                      "if (recv && k / M != r) recv[r] += len;"),
    "zero3_shard_cast_truncates": ("Pshard[lo + k] = oracle_bf16_rne(W[lo + k]);",
                                   "Pshard[lo + k] = (uint16_t)(((union { float f; uint32_t u; }){W[lo + k]}).u >> 16);"),
    "fp16_truncates": ("uint32_t r = a + 0xFFFu + ((a >> 13) & 1u);", "uint32_t r = a + 0u * ((a >> 13) & 1u);"),
    "fp16_subnormal_no_round": ("if (rem > half || (rem == half && (q & 1u))) ++q;", "if (rem > half + rem) ++q;"),
    "int8_scale_128": ("float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    "int8_truncates": ("float q = rintf(xb[k] / s);", "float q = truncf(xb[k] / s);"),
    "sign_uses_max": ("float s = abs_tree(xb, cnt, 0, ORACLE_COMP_BLOCK) / (float)cnt;",
                      "float s = abs_tree(xb, cnt, 0, ORACLE_COMP_BLOCK) / (float)ORACLE_COMP_BLOCK;"),
    "ef_sign_flipped": ("if (E) E[r][i] = x[i] - d[i];", "if (E) E[r][i] = d[i] - x[i];"),
    "ef_not_added": ("x[i] = E ? loc + E[r][i] : loc;", "x[i] = E ? loc + 0.0f * E[r][i] : loc;"),
    "zero3_unit_source_offset": ("ptr[k] = Gu[k] + (a - lo);", "ptr[k] = Gu[k] + (a - lo) * 0;"),
    "zero3_unit_owned_range_clipped_low": ("int64_t a = lo > own_lo ? lo : own_lo;",
                                           "int64_t a = own_lo;"),
    "zero3_unit_counts_own_rank": ("if (recv && k % M == 0 && k / M != r) recv[r] += b - a;",
                                   "if (recv && k % M == 0) recv[r] += b - a;"),
    "zero3_unit_divides_by_R": ("float denom_rm = (float)((double)R * (double)M);",
                                "float denom_rm = (float)((double)R * (double)1);"),
    "zero3_update_casts_before_update": ("oracle_adamw_elem(&s, gshard[i], &W[i], &m[i], &v[i]);\n        Pshard[i] = oracle_bf16_rne(W[i]);",
                                         "Pshard[i] = oracle_bf16_rne(W[i]);\n        oracle_adamw_elem(&s, gshard[i], &W[i], &m[i], &v[i]);"),
    "onebit_warmup_off_by_one": ("if (step <= freeze_step)", "if (step < freeze_step)"),
    "onebit_local_mean_not_divided": ("float gl = loc / denom_m;", "float gl = loc + 0.0f * denom_m;"),
    "onebit_momentum_from_grad_only": ("float ml = s.beta1 * m[i] + s.one_minus_beta1 * gl;",
                                       "float ml = 0.0f * m[i] + s.one_minus_beta1 * gl;"),
    "onebit_worker_ef_sign": ("E[r][i] = xr[i] - dr[i];", "E[r][i] = dr[i] - xr[i];"),
    "onebit_no_server_ef": ("y[i] = dsum[i] / denom_r + Es[i];", "y[i] = dsum[i] / denom_r + 0.0f * Es[i];"),
    "onebit_server_ef_sign": ("Es[i] = y[i] - ds[i];", "Es[i] = ds[i] - y[i];"),
    "onebit_global_server_blocks": ("oracle_compress(ORACLE_COMP_SIGN, y + lo, len, ds + lo);",
                                    "if (r == 0) oracle_compress(ORACLE_COMP_SIGN, y, n + 0 * len, ds);"),
    "onebit_update_skips_server_codec": ("float mi = ds[i];", "float mi = dsum[i] / denom_r;"),
    "onebit_bias_correction_at_t": ("float q = root / sf.bc2_sqrt;", "float q = root / s.bc2_sqrt;"),
}

# Further slips, one per site: the moment coefficients, the bias-correction
# and decay scalars, the decay order, the collectives' first and own terms,
# the codecs' thresholds and sign rules, and the 1-bit update's state.
MUTANTS.update({
    "first_moment_uses_beta2": ("float a = s->beta1 * *m;", "float a = s->beta2 * *m;"),
    "second_moment_uses_one_minus_beta1": ("float d = s->one_minus_beta2 * g;",
                                           "float d = s->one_minus_beta1 * g;"),
    "update_uses_old_first_moment": ("float ratio = m1 / den;", "float ratio = *m / den;"),
    "decay_after_update": ("*w = wd - upd;", "*w = (*w - upd) * s->decay + 0.0f * wd;"),
    "decay_without_lr": ("out->decay = (float)(1.0 - lr * wd);",
                         "out->decay = (float)(1.0 - wd + 0.0 * lr);"),
    "bias_correction_2_uses_beta1": ("double bc2 = 1.0 - pow(b2, t);",
                                     "double bc2 = 1.0 - pow(b1, t);"),
    "rs_sum_skips_first_rank": ("float acc = in[0][lo + k];", "float acc = 0.0f * in[0][lo + k];"),
    "ring_reduce_overwrites": ("cards[dst][e] = cards[dst][e] + msg[(int64_t)k * csz + (e - lo)];",
                               "cards[dst][e] = msg[(int64_t)k * csz + (e - lo)];"),
    "zero3_bytes_params_unsharded": ("out[3] = N * (bp + bg + bo) / P;",
                                     "out[3] = N * bp + N * (bg + bo) / P;"),
    "clip_uses_sumsq_as_norm": ("double norm = sqrt(sumsq);", "double norm = sumsq;"),
    "zero3_gather_counts_own_elements": ("if (owner != card) ++from_others;",
                                         "if (owner != card || 1) ++from_others;"),
    "fp16_overflow_at_max_finite": ("if (a >= 0x477FF000u)", "if (a > 0x477FE000u)"),
    "int8_amax_signed": ("float a = fabsf(xb[k]);", "float a = xb[k];"),
    "sign_of_zero_negative": ("db[k] = xb[k] < 0.0f ? -s : s;", "db[k] = xb[k] <= 0.0f ? -s : s;"),
    "compressed_divides_by_R": ("float g = acc[i] / s.denom_rm;", "float g = acc[i] / (float)R;"),
    "onebit_server_average_not_divided": ("y[i] = dsum[i] / denom_r + Es[i];",
                                          "y[i] = dsum[i] + Es[i] + 0.0f * denom_r;"),
    "onebit_step_size_at_freeze": ("float upd = s.step_size * ratio;",
                                   "float upd = sf.step_size * ratio;"),
    "onebit_no_decay": ("float wd = W[i] * s.decay;", "float wd = W[i];"),
    "onebit_momentum_not_stored": ("m[i] = mi;", "(void)mi;"),
    "zero_rs_reads_unshifted_chunk": (
        "gshard[k] = oracle_avg_grad((const uint16_t* const*)recv_ptr, R, M, k,",
        "gshard[k] = oracle_avg_grad((const uint16_t* const*)G + 0 * (recv_ptr != 0), R, M, k,"),
    "zero3_update_cast_truncates": ("Pshard[i] = oracle_bf16_rne(W[i]);",
                                    "Pshard[i] = (uint16_t)(f2u(W[i]) >> 16);"),
    "zero3_gather_local_index": ("out[i - lo] = Pshard[i];", "out[i - lo] = Pshard[i - lo];"),
    "zero3_unit_counts_whole_unit": (
        "if (recv && k % M == 0 && k / M != r) recv[r] += b - a;",
        "if (recv && k % M == 0 && k / M != r) recv[r] += hi - lo + 0 * (b - a);"),
    "zero3_unit_writes_local_index": (
        "gshard[i] = oracle_avg_grad((const uint16_t* const*)ptr, R, M, i - a, denom_rm);",
        "gshard[i - a] = oracle_avg_grad((const uint16_t* const*)ptr, R, M, i - a, denom_rm);"),
    "mt_ranges_overlap": ("jb->hi = n * (k + 1) / nthreads;",
                          "jb->hi = n * (k + 1) / nthreads + (k + 1 < nthreads);"),
    "denom_R_plus_M": ("out->denom_rm = (float)((double)R * (double)M);",
                       "out->denom_rm = (float)((double)R + (double)M);"),
    "bf16_nan_keeps_payload": ("return (uint16_t)0x7FC0u;", "return (uint16_t)((u >> 16) | 0x40u);"),
    "eps_before_bias_correction": ("float den = q + s->eps;",
                                   "float den = (root + s->eps) / s->bc2_sqrt + 0.0f * q;"),
    "dp_cast_before_update": (
        "float g = oracle_avg_grad(G, R, M, i, s.denom_rm);\n"
        "        oracle_adamw_elem(&s, g, &W[i], &m[i], &v[i]);\n"
        "        uint16_t p = oracle_bf16_rne(W[i]);",
        "float g = oracle_avg_grad(G, R, M, i, s.denom_rm);\n"
        "        uint16_t p = oracle_bf16_rne(W[i]);\n"
        "        oracle_adamw_elem(&s, g, &W[i], &m[i], &v[i]);"),
    "onebit_momentum_coefficients_swapped": (
        "float ml = s.beta1 * m[i] + s.one_minus_beta1 * gl;",
        "float ml = s.beta1 * gl + s.one_minus_beta1 * m[i];"),
    "compressed_ef_of_next_rank": ("x[i] = E ? loc + E[r][i] : loc;",
                                   "x[i] = E ? loc + E[(r + 1) % R][i] : loc;"),
    "clip_norm_of_unaveraged_sum": (
        "for (int64_t i = 0; i < n; ++i) g[i] = oracle_avg_grad(G, R, M, i, s.denom_rm);",
        "for (int64_t i = 0; i < n; ++i) g[i] = oracle_avg_grad(G, R, M, i, 1.0f + 0.0f * s.denom_rm);"),
})


PIN_SUITES = ["tests/test_oracle_pins.py", "tests/test_oracle_collectives.py",
              "tests/test_oracle_clip.py", "tests/test_oracle_zero3.py",
              "tests/test_oracle_compress.py", "tests/test_oracle_onebit.py"]


def _run_mutant(name, workdir):
    """Compile the mutant into its own library and run the pin suites on it in
    a child process; returns (returncode, tail of the child's output)."""
    old, new = MUTANTS[name]
    src = open(SRC).read()
    if src.count(old) != 1:
        return None, f"mutation site for {name} not unique/present"
    mut_src = os.path.join(workdir, "zero_oracle.c")
    with open(mut_src, "w") as f:
        f.write(src.replace(old, new))
    hdr_dir = os.path.join(ROOT, "oracle")
    lib = os.path.join(workdir, "liboracle_mut.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-I", hdr_dir, "-o", lib, mut_src, "-lm", "-lpthread"],
                   check=True)
    env = dict(os.environ, ZERO_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PIN_SUITES], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    return r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """Every mutant's pin run, the children side by side (one per core): each
    is an independent process over its own library, so the outcome of one
    does not depend on the others."""
    workers = max(1, min(len(MUTANTS), os.cpu_count() or 1))
    dirs = {n: str(tmp_path_factory.mktemp(n)) for n in MUTANTS}
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        futs = {n: ex.submit(_run_mutant, n, dirs[n]) for n in MUTANTS}
        return {n: f.result() for n, f in futs.items()}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_results):
    rc, out = mutant_results[name]
    assert rc is not None, out
    assert rc != 0, f"mutant {name} survived the pins:\n{out}"
