"""The oracle's pins catch plausible mistakes.

Each case below plants one mistake in a copy of oracle/santa_oracle.c or of
oracle/analysis.py on the CPU: a wrong operand, index, sign, constant or
rounding rule, or a dropped term.  It then builds or loads the copy and runs
the pins of tests/test_oracle_pins.py against it (the C copy through
SANTA_ORACLE_LIB, the Python copy in place of oracle.analysis).  Every
mutant must make at least one pin fail.  The mistakes are planted in the oracle only; the CUDA library is
not involved.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "santa_oracle.c")

# (name, original text, replacement, which occurrence of the original (0-based), total occurrences)
MUTANTS = [
    # Philox4x32-10 (Salmon et al., SC'11) and the uniform map
    ("philox_operand", "(uint64_t)0xD2511F53u * (uint64_t)c[0]", "(uint64_t)0xD2511F53u * (uint64_t)c[1]", 0, 1),
    ("philox_weyl", "k1 += 0xBB67AE85u;", "k1 += 0xBB67AE86u;", 0, 1),
    ("philox_rounds", "round < 10; ++round", "round < 9; ++round", 0, 1),
    ("uniform_bits", "(words[r % 4u] >> 8)", "(words[r % 4u] >> 9)", 0, 1),
    ("counter_b_h_swapped", "{r / 4u, h, b, step}", "{r / 4u, b, h, step}", 0, 1),
    # thresholds (Sec. 2.1)
    ("systematic_denominator", "t[j] = ((double)j + u) / (double)S;", "t[j] = ((double)j + u) / (double)(S + 1);", 0, 1),
    ("stratified_one_uniform", "santa_oracle_uniform(seed, b, h, step, (uint32_t)j)) / (double)S;",
     "santa_oracle_uniform(seed, b, h, step, 0u)) / (double)S;", 0, 1),
    ("iid_unsorted", "qsort(t, (size_t)S, sizeof(double), cmp_double);", "(void)cmp_double;", 0, 1),
    # scores and softmax (Eq. 1)
    ("scale_dropped_sqrt", "1.0 / sqrt((double)d)", "1.0 / (double)d", 0, 1),
    ("softmax_sign", "p[n] = exp(sc[n] - m)", "p[n] = exp(m - sc[n])", 0, 1),
    ("gqa_head_map", "const int32_t kvh = h / (P->n_q_heads / Hkv);", "const int32_t kvh = h % Hkv;", 0, 5),
    ("query_row", "((int64_t)b * P->n_q_heads + h) * d + k", "((int64_t)h * P->batch + b) * d + k", 0, 1),
    # inverse CDF and gather (App. A.4, Eq. 4)
    ("boundary_left_open", "if (F[mid] <= tj) lo = mid + 1;", "if (F[mid] < tj) lo = mid + 1;", 0, 1),
    ("clamp_to_last_key", "n = last_pos;", "n = nk - 1;", 0, 1),
    ("gather_normaliser", "est[k] *= 1.0 / (double)S;", "est[k] *= 1.0 / (double)(S + 1);", 0, 2),
    ("gather_ignores_offsets", "for (int32_t k = 0; k < d; ++k) est[k] += (double)counts[n]",
     "for (int32_t k = 0; k < d; ++k) est[k] += (double)(counts[n] > 0)", 0, 1),
    ("sample_row_offset", "const int64_t base = ((row0 + n) * Hkv + kvh) * (int64_t)d;\n      for (int32_t k = 0; k < d; ++k) est",
     "const int64_t base = ((n) * Hkv + kvh) * (int64_t)d;\n      for (int32_t k = 0; k < d; ++k) est", 0, 1),
    ("dense_reads_K", "out[k] += p[n] * load_elem(P->dtype, P->V, base + k);",
     "out[k] += p[n] * load_elem(P->dtype, P->K, base + k);", 0, 1),
    ("decode_padding", "if (Jrow) Jrow[j] = -1;", "if (Jrow) Jrow[j] = 0;", 0, 1),
    # tile samplers (App. O, Alg. 3-5; App. P, Alg. 6-8)
    ("prop_smallest_remainder", "frac[t] > frac[best]", "frac[t] < frac[best]", 0, 1),
    ("prop_ties_to_higher_tile", "frac[t] > frac[best]", "frac[t] >= frac[best]", 0, 1),
    ("prop_no_cap", "frac[best] = -1.0;", "frac[best] -= 0.5;", 0, 1),
    ("tile_counts_ceil", "c[n] = (int32_t)(floor(hi) - floor(lo));", "c[n] = (int32_t)(ceil(hi) - ceil(lo));", 0, 1),
    ("tile_mass_drops_l", "W[t] = exp(m[t] - mstar) * l[t];", "W[t] = exp(m[t] - mstar);", 0, 1),
    ("flash_weight_uses_S", "(W[t] / Z) / (double)bud[t]", "(W[t] / Z) / (double)S", 0, 1),
    ("flash_tile_budget_floor", "floor((double)S / (double)T + 0.5)", "floor((double)S / (double)T)", 0, 1),
    ("tile_delta_from_budget", "inv_delta = bud[t] > 0 ? (double)bud[t] / l[t]", "inv_delta = bud[t] > 0 ? (double)S / l[t]", 0, 1),
    # storage widening and rounding
    ("bf16_shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15", 0, 1),
    ("fp16_exponent_bias", "expo - 25", "expo - 24", 0, 1),
    ("fp16_subnormal_scale", "ldexp((double)mant, -24)", "ldexp((double)mant, -23)", 0, 1),
    ("fp16_round_half_up", "if (r > half || (r == half && (q & 1u))) ++q;", "if (r >= half) ++q;", 0, 1),
    ("bf16_round_half_up", "u += 0x7fffu + ((u >> 16) & 1u);", "u += 0x8000u;", 0, 1),
    # Bernoulli qK^T with the mean group query (App. C, Eq. 10-13)
    ("bernoulli_drops_norm", "const float mh = (norm * (float)c) / (float)nsamp;",
     "const float mh = ((float)c) / (float)nsamp;", 0, 1),
    ("bernoulli_stream", "(uint32_t)(H + kvh)", "(uint32_t)(kvh)", 0, 1),
    ("bernoulli_norm_is_sum", "if (m[i] > norm) norm = m[i];", "norm += m[i];", 0, 1),
    ("bernoulli_plain_threshold", "(a24 < (double)pr * 16777216.0)", "(a24 <= (double)pr * 16777216.0 + 1.0)", 0, 1),
    ("bernoulli_abs_dropped", "acc += fabsf(q[g * d + i]);", "acc += q[g * d + i];", 0, 1),
    ("bernoulli_stratified_strict", "(double)n * 16777216.0 + a24 < (double)nsamp",
     "(double)n * 16777216.0 + a24 <= (double)nsamp", 0, 1),
    ("bernoulli_stratum_index", "(double)n * 16777216.0 + a24", "(double)(n + 1) * 16777216.0 + a24", 0, 1),
    # more of the score, sampling and decode plumbing
    ("tile_stats_sum", "for (int64_t n = lo; n < hi; ++n) sum += exp(s[n] - mx);",
     "for (int64_t n = lo; n < hi; ++n) sum += exp(s[n]);", 0, 1),
    ("softmax_Z_drops_first_key", "p[n] = exp(sc[n] - m); Z += p[n];", "p[n] = exp(sc[n] - m); Z += n ? p[n] : 0.0;",
     0, 1),
    ("decode_ignores_S_per_seq", "const int32_t Sb = S_per_seq ? S_per_seq[b] : S;", "const int32_t Sb = S;", 1, 2),
    ("scores_row_offset", "const int64_t base = ((row0 + n) * Hkv + kvh) * (int64_t)d;\n    for (int32_t k = 0; k < d; ++k) dot",
     "const int64_t base = ((n) * Hkv + kvh) * (int64_t)d;\n    for (int32_t k = 0; k < d; ++k) dot", 0, 1),
    ("gather_row_offset", "((row0 + J[j]) * Hkv + kvh)", "((J[j]) * Hkv + kvh)", 0, 1),
    ("dense_row_offset", "const int64_t base = ((row0 + n) * Hkv + kvh) * (int64_t)d;\n    for (int32_t k = 0; k < d; ++k) out",
     "const int64_t base = ((n) * Hkv + kvh) * (int64_t)d;\n    for (int32_t k = 0; k < d; ++k) out", 0, 1),
    ("prop_budget_rounds", "St[t] = (int32_t)floor(q);", "St[t] = (int32_t)floor(q + 0.5);", 0, 1),
    ("sample_delta_one_side", "dist = a < c ? a : c;", "dist = a;", 0, 1),
    ("tile_delta_one_side", "dx[n] = d1 < d2 ? d1 : d2;", "dx[n] = d1;", 0, 1),
    ("tile_delta_scale", "dx[n] *= W[t] / (Z * (double)bud[t]);", "dx[n] *= W[t] / Z;", 0, 1),
    ("tile_a0_stream", "santa_oracle_uniform(seed, (uint32_t)b, (uint32_t)h, step, (uint32_t)t)",
     "santa_oracle_uniform(seed, (uint32_t)b, (uint32_t)h, step, (uint32_t)(t + 1))", 0, 1),
]


# the closed forms of oracle/analysis.py, same format
PY_MUTANTS = [
    ("iid_trace_drops_mean", "- mu @ mu)", ")", 0, 1),
    ("iid_trace_not_over_S", "    return tr / S", "    return tr", 0, 1),
    ("iid_coordinate_drops_mean", "(V * V) - mu * mu) / S", "(V * V)) / S", 0, 1),
    ("stratum_upper_edge", "((m + 1) / S)", "((m + 2) / S)", 0, 1),
    ("stratified_trace_over_S", "return float(tr_m.sum()) / (S * S)", "return float(tr_m.sum()) / S", 0, 1),
    ("stratified_coordinate_over_S", "return var_m.sum(axis=0) / (S * S)", "return var_m.sum(axis=0) / S", 0, 1),
    ("breakpoints_sign", "u = (S * F)[:, None] - np.arange(S)[None, :]", "u = (S * F)[:, None] + np.arange(S)[None, :]",
     0, 1),
    ("offset_piece_length", "* (b - a)", "* (b + a)", 0, 1),
    ("replicate_divisor", "/ (R - 1)", "/ R", 0, 1),
    ("count_bounds_swapped", "return np.floor(Sp), np.ceil(Sp)", "return np.ceil(Sp), np.floor(Sp)", 0, 1),
    ("unique_keys_exponent", "-np.expm1(S * np.log1p(-p))", "-np.expm1((S - 1) * np.log1p(-p))", 0, 1),
    ("causal_mask_off_by_one", "np.triu_indices(n, 1)", "np.triu_indices(n, 2)", 0, 1),
    ("coverage_complement", "np.mean(-np.expm1(log_none))", "np.mean(np.exp(log_none))", 0, 1),
    ("coverage_axis", "np.log1p(-P).sum(axis=0)", "np.log1p(-P).sum(axis=1)", 0, 1),
]
PY_SRC = os.path.join(ROOT, "oracle", "analysis.py")

# loads a mutated analysis.py in place of oracle.analysis, then runs the pins
PY_DRIVER = """
import importlib.util, sys
sys.path.insert(0, sys.argv[1])
import oracle
spec = importlib.util.spec_from_file_location("oracle.analysis", sys.argv[2])
mod = importlib.util.module_from_spec(spec)
spec.loader.exec_module(mod)
sys.modules["oracle.analysis"] = mod
oracle.analysis = mod
import pytest
sys.exit(pytest.main([sys.argv[3], "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"]))
"""


def mutate(src: str, orig: str, repl: str, occ: int, total: int) -> str:
    assert src.count(orig) == total, f"{orig!r} occurs {src.count(orig)} times, expected {total}"
    pos = -1
    for _ in range(occ + 1):
        pos = src.index(orig, pos + 1)
    return src[:pos] + repl + src[pos + len(orig):]


def run_pins(lib_path: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, SANTA_ORACLE_LIB=lib_path, OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_oracle_pins.py"), "-x", "-q",
                           "-p", "no:cacheprovider", "-m", "not gpu"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def build_mutant(tmp, name, orig=None, repl=None, occ=0, total=1):
    src = open(SRC).read()
    if orig is not None:
        src = mutate(src, orig, repl, occ, total)
    c_path = os.path.join(tmp, f"{name}.c")
    so_path = os.path.join(tmp, f"lib{name}.so")
    with open(c_path, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-w",
                    "-I", os.path.join(ROOT, "oracle"), "-o", so_path, c_path, "-lm"], check=True)
    return so_path


def test_unmutated_copy_passes(tmp_path):
    """Control: the same build recipe without a mutation passes every pin."""
    so = build_mutant(str(tmp_path), "control")
    r = run_pins(so)
    assert r.returncode == 0, r.stdout[-2000:]


def test_every_mutant_fails_a_pin(tmp_path):
    def one(m):
        name = m[0]
        so = build_mutant(str(tmp_path), *m)
        r = run_pins(so)
        return name, r.returncode, r.stdout.strip().splitlines()[-1:] if r.stdout else []

    with ThreadPoolExecutor(max_workers=max(1, min(6, (os.cpu_count() or 2) // 2))) as ex:
        results = list(ex.map(one, MUTANTS))
    survivors = [(n, tail) for n, rc, tail in results if rc == 0]
    assert not survivors, f"mutants no pin catches: {survivors}"


def test_every_closed_form_mutant_fails_a_pin(tmp_path):
    import oracle
    oracle.build()

    def one(m):
        name, orig, repl, occ, total = m
        path = os.path.join(str(tmp_path), f"analysis_{name}.py")
        with open(path, "w") as f:
            f.write(mutate(open(PY_SRC).read(), orig, repl, occ, total))
        r = subprocess.run([sys.executable, "-c", PY_DRIVER, ROOT, path, os.path.join(HERE, "test_oracle_pins.py")],
                           cwd=ROOT, env=dict(os.environ, OMP_NUM_THREADS="2"), capture_output=True, text=True,
                           timeout=600)
        return name, r.returncode, r.stdout.strip().splitlines()[-1:] if r.stdout else []

    with ThreadPoolExecutor(max_workers=max(1, min(6, (os.cpu_count() or 2) // 2))) as ex:
        results = list(ex.map(one, PY_MUTANTS))
    assert all(rc in (0, 1) for _, rc, _ in results), results   # 1: a pin failed; anything else is a harness error
    survivors = [(n, tail) for n, rc, tail in results if rc == 0]
    assert not survivors, f"closed-form mutants no pin catches: {survivors}"
