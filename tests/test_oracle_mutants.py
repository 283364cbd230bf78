"""Planted mistakes: the oracle's pins must reject a wrong oracle.

Each mutant below is one plausible slip in oracle/vdit_oracle.c: a dropped
term, a wrong sign, an off-by-one, a transposed index, a wrong stride. The test
compiles a copy of the C source with that one change (gcc, on the CPU, the
flags of oracle.build()), points the oracle package at it through
VDIT_ORACLE_LIB and runs the pin files that cover the changed function. Every
mutant must make at least one pin fail; the unmutated source, built and loaded
the same way, must pass all of them. No GPU is involved and nothing here
touches the CUDA library.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "vdit_oracle.c")

SCHED = "test_oracle_schedule.py"
ATTN = "test_oracle_attention.py"
FRAME = "test_oracle_frame_bound.py"
PRO = "test_oracle_prologue.py"

# name, text in the source (must occur once), replacement, pin files that must catch it
MUTANTS = [
    # token mask and block schedule ("Deleting the Mask", Fig. 3)
    ("window_off_by_one", "if (d <= (int64_t)W)", "if (d < (int64_t)W)", [SCHED, ATTN]),
    ("reference_on_query_frame", "if (ref >= 0 && fj == (int64_t)ref)",
     "if (ref >= 0 && fi == (int64_t)ref)", [SCHED, ATTN]),
    ("reference_dropped", "if (ref >= 0 && fj == (int64_t)ref)", "if (0)", [SCHED, ATTN]),
    ("csr_column_shifted", "col_idx[nnz] = (int32_t)kb;", "col_idx[nnz] = (int32_t)(kb + (qb & 1));",
     [SCHED]),
    ("run_end_short", "runs[4 * f + 1] = (int32_t)hi[0];", "runs[4 * f + 1] = (int32_t)hi[0] - 1;",
     [SCHED]),
    ("second_run_dropped", "runs[4 * f + 3] = nr > 1 ? (int32_t)hi[1] : 0;",
     "runs[4 * f + 3] = nr > 1 ? (int32_t)lo[1] : 0;", [SCHED]),
    ("pairs_count_blocks", "pairs += cnt;", "pairs += cnt > 0;", [SCHED]),
    # block census (partial blocks under tiles that straddle frames)
    ("census_ragged_tile_full_area", "int64_t area = (i1 - i0) * (j1 - j0);",
     "int64_t area = (int64_t)bs * bs;", [SCHED]),
    ("census_partial_as_full", "if (live == area)", "if (live * 2 >= area)", [SCHED]),
    # exact bf16 reading
    ("bf16_read_rounded", "uint32_t u = ((uint32_t)((const uint16_t *)p)[idx]) << 16;",
     "uint32_t u = (((uint32_t)((const uint16_t *)p)[idx]) << 16) | 0x8000u;", [ATTN]),
    # key statistics and eligibility ("Unchaining the Softmax")
    ("mean_over_n_minus_1", "cc[d] /= (double)N;", "cc[d] /= (double)(N - 1);", [ATTN]),
    ("radius_uncentred", "double x = elem(k, kb + j * ks[2] + d, dtype) - cc[d];",
     "double x = elem(k, kb + j * ks[2] + d, dtype);", [ATTN]),
    ("gap_without_factor_2", "G[bh] = 2.0 * scale * qmax[bh] * R[bh];",
     "G[bh] = scale * qmax[bh] * R[bh];", [ATTN]),
    ("qmax_not_square_rooted", "qmax[bh] = sqrt(q2);", "qmax[bh] = q2;", [ATTN]),
    ("eligibility_strict", "elig[bh] = ((float)G[bh] <= (float)tau) ? 1 : 0;",
     "elig[bh] = ((float)G[bh] < (float)tau * 0.5f) ? 1 : 0;", [ATTN]),
    # row bound
    ("bound_minus_norm_term", "m[r] = scale * (dot + sqrt(nn) * R[bh]);",
     "m[r] = scale * (dot - sqrt(nn) * R[bh]);", [ATTN]),
    ("bound_without_mean_term", "m[r] = scale * (dot + sqrt(nn) * R[bh]);",
     "m[r] = scale * (sqrt(nn) * R[bh]);", [ATTN]),
    # masked attention (plain definition)
    ("scale_dropped", "s[j] = scale * acc;", "s[j] = acc;", [ATTN]),
    ("lse_without_max", "lse[r] = m + log(l);", "lse[r] = log(l);", [ATTN]),
    ("value_of_query_row", "out[d] += p * elem(v, vb + j * vs[2] + d, dtype);",
     "out[d] += p * elem(v, vb + i * vs[2] + d, dtype);", [ATTN]),
    ("not_normalised", "out[d] /= l;", "out[d] /= 1.0;", [ATTN]),
    ("key_rows_with_query_stride", "acc += qrow[d] * elem(k, kb + j * ks[2] + d, dtype);",
     "acc += qrow[d] * elem(k, kb + j * qs[2] + d, dtype);", [ATTN]),
    ("exp_shift_half_max", "double p = exp(s[j] - m);", "double p = exp(s[j] - 0.5 * m);",
     [ATTN]),
    # per-query-frame statistics and bound
    ("frame_radius_ignores_mask", "if (vo_mask(T, W, ref, f * T, j) && kn[j] > r)",
     "if (kn[j] > r)", [FRAME]),
    ("frame_qmax_spills_into_next_frame", "for (int64_t i = f * T; i < (f + 1) * T; ++i) {",
     "for (int64_t i = f * T; i < (f + 2) * T && i < N; ++i) {", [FRAME]),
    ("frame_bound_without_mean_term", "m[r] = scale * (dot + sqrt(nn) * Rf[bh * F + i / T]);",
     "m[r] = scale * (sqrt(nn) * Rf[bh * F + i / T]);", [FRAME]),
    ("frame_bound_uses_frame_0", "m[r] = scale * (dot + sqrt(nn) * Rf[bh * F + i / T]);",
     "m[r] = scale * (dot + sqrt(nn) * Rf[bh * F]);", [FRAME]),
    # fused pre-attention chain ("Layout Is the ABI", Fig. 5)
    ("rmsnorm_without_gain", "y[c] = elem(x, xo + c, dtype) * inv * gamma[c];",
     "y[c] = elem(x, xo + c, dtype) * inv;", [PRO]),
    ("rmsnorm_without_mean", "const double inv = 1.0 / sqrt(ss / (double)C + eps);",
     "const double inv = 1.0 / sqrt(ss + eps);", [PRO]),
    ("weights_transposed", "acc += y[c] * elem(w, o * C + c, dtype);",
     "acc += y[c] * elem(w, c * (3 * HD) + o, dtype);", [PRO]),
    ("rotation_sign", "zh[i] = u * cos(a) - wv * sin(a);", "zh[i] = u * cos(a) + wv * sin(a);",
     [PRO]),
    ("rotation_adjacent_pairs", "const double u = zh[i], wv = zh[i + D / 2];",
     "const double u = zh[i], wv = zh[(i + 1) % D];", [PRO]),
    ("rotation_frequency", "const double t = pow(base, -2.0 * i / (double)D);",
     "const double t = pow(base, -1.0 * i / (double)D);", [PRO]),
    ("values_rotated_too", "for (int part = 0; part < 2; ++part) {", "for (int part = 0; part < 3; ++part) {",
     [PRO]),
]


def _pin_run(lib, files):
    """Run the given pin files against the oracle library `lib`; pytest's exit code."""
    env = dict(os.environ, VDIT_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu"]
    cmd += [os.path.join(HERE, f) for f in files]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Build the unmutated source and every mutant, then run each against its pin
    files, several at a time. Returns {name: (exit code, output tail)}."""
    src = open(SRC).read()
    out_dir = tmp_path_factory.mktemp("oracle_mutants")
    jobs = [("control", src, [SCHED, ATTN, FRAME, PRO])]
    for name, old, new, files in MUTANTS:
        assert src.count(old) == 1, f"{name}: the mutated text must occur exactly once"
        jobs.append((name, src.replace(old, new), files))

    def run(job):
        name, text, files = job
        c = os.path.join(out_dir, f"{name}.c")
        with open(c, "w") as f:
            f.write(text)
        so = os.path.join(out_dir, f"lib{name}.so")
        oracle.compile_source(c, so)
        return name, _pin_run(so, files)

    with ThreadPoolExecutor(max_workers=max(2, min(8, (os.cpu_count() or 2) // 2))) as ex:
        return dict(ex.map(run, jobs))


def test_control_build_passes_every_pin(outcomes):
    """The mechanism itself (copy, compile, load through VDIT_ORACLE_LIB) leaves
    the pins green, so a failing mutant is failing on its planted mistake."""
    rc, tail = outcomes["control"]
    assert rc == 0, tail


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_reject_mutant(outcomes, name):
    rc, tail = outcomes[name]
    # exit code 1: some test failed (not a collection error or a crash)
    assert rc == 1, f"mutant {name} survived the pins (pytest exit {rc}):\n{tail}"
