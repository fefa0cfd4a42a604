"""The oracle's pins catch plausible mistakes: mutation tests on the CPU.

Each case plants one plausible mistake in a copy of oracle/vc_oracle.c (a
dropped term, a flipped sign, a wrong index or constant, a changed rounding
rule), builds the copy with the oracle's own flags, and runs the named pin
files against it in a subprocess (the oracle loads the copy through its
library override).  The pins must fail on assertions.  The unmutated copy,
built the same way, passes the same files.  Nothing here touches the CUDA
library; the mistakes live only in temporary copies.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

import oracle
from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "vc_oracle.c")

# (id, what goes wrong, text in vc_oracle.c, replacement, pin files that must fail)
MUTANTS = [
    # ExpCast-FP8 (paper summary, 方法步骤详情 step 4)
    ("beta_dropped", "ExpCast constant 120 instead of 120 + beta",
     "#define VCO_BETA_PLUS_120 119.65f", "#define VCO_BETA_PLUS_120 120.0f", ["test_oracle_expcast.py"]),
    ("round_floor", "ExpCast rounds down instead of to nearest",
     "float r = nearbyintf(t);                  /* RNE */", "float r = floorf(t);", ["test_oracle_expcast.py"]),
    ("no_upper_clip", "ExpCast byte not clipped at 120",
     "    if (r > 120.0f) return 120;\n", "", ["test_oracle_expcast.py"]),
    # E4M3 codec (前置知识, E4M3 浮点格式)
    ("subnormal_scale", "subnormal step 2^-10 instead of 2^-9",
     "if (e == 0) v = (double)m * ldexp(1.0, -9);", "if (e == 0) v = (double)m * ldexp(1.0, -10);",
     ["test_oracle_codecs.py"]),
    ("exponent_bias", "exponent bias 8 instead of 7",
     "else        v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else        v = ldexp(1.0 + (double)m / 8.0, e - 8);",
     ["test_oracle_codecs.py"]),
    ("saturate_to_nan", "values beyond 448 become NaN instead of 448",
     "if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;", ["test_oracle_codecs.py"]),
    ("ties_away", "encoder ties away from zero instead of to even",
     "double mq = nearbyint(q);                 /* in [8, 16]", "double mq = floor(q + 0.5);                 /* in [8, 16]",
     ["test_oracle_codecs.py"]),
    ("bf16_truncates", "bf16 conversion truncates",
     "    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;\n", "", ["test_oracle_codecs.py"]),
    # grouping (方法步骤详情 step 1)
    ("mean_off_by_one", "centroid divides by count + 1",
     "C[(int64_t)i * d + c] = (float)(sum[(int64_t)i * d + c] / (double)cnt[i]);",
     "C[(int64_t)i * d + c] = (float)(sum[(int64_t)i * d + c] / (double)(cnt[i] + 1));", ["test_oracle_kmeans.py"]),
    ("assign_farthest", "assignment keeps the farthest centroid",
     "if (dist < best) { best = dist; arg = i; }", "if (!(dist < best) || best == INFINITY) { best = dist; arg = i; }",
     ["test_oracle_kmeans.py"]),
    ("cold_start_first_k", "cold start takes the first k tokens",
     "int src = (int)(((int64_t)i * N) / k);", "int src = i;", ["test_oracle_kmeans.py"]),
    ("argsort_unstable", "equal labels in reverse token order",
     "for (int n = 0; n < N; ++n)\n                if (z[n] == lab) p[pos++] = n;",
     "for (int n = N - 1; n >= 0; --n)\n                if (z[n] == lab) p[pos++] = n;", ["test_oracle_kmeans.py"]),
    # block fill (独立分析的弱点, weakness one)
    ("fill_farthest", "block-fill chain moves to the farthest centroid",
     "if (best < 0 || sum < bestd) { best = c; bestd = sum; }",
     "if (best < 0 || sum > bestd) { best = c; bestd = sum; }", ["test_oracle_block_fill.py"]),
    ("fill_drops_blocks", "whole blocks left out of the permutation",
     "int f = n[c] - n[c] % VCO_BLOCK, seen = 0;\n            for (int t = 0; t < N && seen < f; ++t)",
     "int f = 0, seen = 0;\n            for (int t = 0; t < N && seen < f; ++t)", ["test_oracle_block_fill.py"]),
    # rotary + Hadamard ahead of the quantizer
    ("rotary_sign", "rotation with the wrong sign",
     "y[2 * i] = a - b;", "y[2 * i] = a + b;", ["test_oracle_preproc.py"]),
    ("rotary_k_position", "K rows rotated at their permuted slot, not their token's position",
     "rope ? rope + (int64_t)src * d : NULL,", "rope ? rope + (int64_t)(t0 + r) * d : NULL,",
     ["test_oracle_preproc.py"]),
    ("hadamard_no_inverse", "Q scale without the 1/d of the Hadamard pair",
     "float q_mul = hadamard ? 1.0f / (float)d : 1.0f;", "float q_mul = 1.0f;", ["test_oracle_preproc.py"]),
    ("butterfly_sign", "Hadamard butterfly difference reversed",
     "y[i + st] = a - b;", "y[i + st] = b - a;", ["test_oracle_preproc.py"]),
    # block quantization and V-Smooth (方法步骤详情 step 2)
    ("qk_scale_240", "Q/K block scale amax/240",
     "float s = amax / 448.0f;\n        float inv", "float s = amax / 240.0f;\n        float inv",
     ["test_oracle_quant.py"]),
    ("mean_unrounded", "residual against the unrounded mean",
     "m = vco_bf16_to_f32(mb);", "m = sum / (float)cnt;", ["test_oracle_quant.py"]),
    ("channel_scale_first_block", "V channel scale from the first block only",
     "for (int t = 0; t < N; ++t) {\n                float a = fabsf(R[(int64_t)t * d + c]);",
     "for (int t = 0; t < N && t < 128; ++t) {\n                float a = fabsf(R[(int64_t)t * d + c]);",
     ["test_oracle_quant.py"]),
    # attention, online softmax, mean restore (方法步骤详情 steps 3-4)
    ("mean_restore_dropped", "r_ij mu_j term left out",
     "for (int c = 0; c < d; ++c) A[c] += r * (double)vco_bf16_to_f32(mj[c]);",
     "for (int c = 0; c < d; ++c) A[c] += 0.0 * (double)vco_bf16_to_f32(mj[c]);", ["test_oracle_attention.py"]),
    ("rescale_sign", "rescale exp2(m' - m) instead of exp2(m - m')",
     "exp2((double)m - (double)mnew);", "exp2((double)mnew - (double)m);", ["test_oracle_attention.py"]),
    ("l_not_rescaled", "normaliser not rescaled",
     "l = alpha * l + r;", "l = l + r;", ["test_oracle_attention.py"]),
    ("exact_offset", "exp-then-cast without the 2^8 factor",
     "float off = 8.0f - mnew;", "float off = 0.0f - mnew;", ["test_oracle_attention.py"]),
    ("score_term_dropped", "first channel left out of the score",
     "for (int c = 0; c < d; ++c) s += qd[c] * dec[kr[c]];", "for (int c = 1; c < d; ++c) s += qd[c] * dec[kr[c]];",
     ["test_oracle_attention.py"]),
    ("query_scale_block0", "every query row takes block 0's scale",
     "            float sqi = sq[(int64_t)bh * nblk + i / VCO_BLOCK];\n            double* A",
     "            float sqi = sq[(int64_t)bh * nblk];\n            double* A", ["test_oracle_attention.py"]),
    ("ref_unscaled", "fidelity reference without the softmax scale",
     "s[n] = acc * scale;", "s[n] = acc;", ["test_oracle_attention.py"]),
    ("C_sign", "ExpCast offset adds the running max instead of subtracting it",
     "return fmaf(-8.0f, m_new, VCO_BETA_PLUS_120);", "return fmaf(8.0f, m_new, VCO_BETA_PLUS_120);",
     ["test_oracle_expcast.py"]),
    ("tail_mean_over_128", "the ragged block's mean divides by 128",
     "uint16_t mb = vco_bf16_rne(sum / (float)cnt);", "uint16_t mb = vco_bf16_rne(sum / 128.0f);",
     ["test_oracle_quant.py"]),
    ("rotary_half_pairs", "rotary pairs (i, i + d/2) instead of (2i, 2i + 1)",
     "float x0 = y[2 * i], x1 = y[2 * i + 1];", "float x0 = y[i], x1 = y[i + d / 2];",
     ["test_oracle_preproc.py"]),
    ("empty_cluster_zeroed", "an empty cluster's centroid reset to zero",
     "if (cnt[i] == 0) continue;", "if (cnt[i] == 0) { for (int c = 0; c < d; ++c) C[(int64_t)i * d + c] = 0.0f; continue; }",
     ["test_oracle_kmeans.py"]),
    ("labels_descending", "pi sorts the labels in descending order",
     "for (int lab = 0; lab < k; ++lab)", "for (int lab = k - 1; lab >= 0; --lab)", ["test_oracle_kmeans.py"]),
    ("chain_starts_high", "leftover chain starts at the highest label",
     "for (int c = 0; c < k; ++c)\n            if (n[c] % VCO_BLOCK) { last = c; break; }",
     "for (int c = k - 1; c >= 0; --c)\n            if (n[c] % VCO_BLOCK) { last = c; break; }",
     ["test_oracle_block_fill.py"]),
    # 4-bit V residual (方法步骤详情 step 2, 4-bit path; the MX reading)
    ("e2m1_ties_away", "E2M1 ties go to the odd code",
     "if (dd < bd || (dd == bd && (c & 1) == 0))", "if (dd < bd || (dd == bd && (c & 1) == 1))",
     ["test_oracle_v4.py"]),
    ("e2m1_no_saturation", "E2M1 without the explicit saturation at 6",
     "    if (a >= 6.0) return (uint8_t)(sign | 7);", "", ["test_oracle_v4.py"]),
    ("mx_exponent_off", "MX group exponent one too high (maximum lands in [2, 4))",
     "            e = ex - 1 - 2;", "            e = ex - 1 - 1;", ["test_oracle_v4.py"]),
    ("v4_scale_448", "4-bit channel scale amax/448 instead of amax/6",
     "    *sv_c = amax / 6.0f;", "    *sv_c = amax / 448.0f;", ["test_oracle_v4.py"]),
    # range-adaptive ExpCast (独立分析的弱点, weakness two: beta by score range)
    ("piece_from_floor", "piece read off floor(t0) instead of rint(t0)",
     "long k = (long)nearbyintf(t0);            /* RNE */", "long k = (long)floorf(t0);",
     ["test_oracle_expcast_pieces.py"]),
    ("piece_table_reversed", "beta table in reverse piece order",
     "{-0.195f, -0.635f, -0.685f, -0.535f}", "{-0.535f, -0.685f, -0.635f, -0.195f}",
     ["test_oracle_expcast_pieces.py"]),
    ("piece_width_four", "pieces four codes wide instead of two",
     "VCO_BETA_PIECE[(k >> 1) & 3]", "VCO_BETA_PIECE[(k >> 2) & 3]", ["test_oracle_expcast_pieces.py"]),
    # hybrid bytes (独立分析的弱点, weakness two)
    ("hybrid_inverted", "hybrid vote inverted",
     "if (diff >= -margin) flags", "if (diff < -margin) flags", ["test_oracle_hybrid.py"]),
    ("hybrid_group_64", "hybrid vote over 64-row groups",
     "int i = rows[ri], g = i / 32;", "int i = rows[ri], g = i / 64;", ["test_oracle_hybrid.py"]),
]

ALL_PINS = sorted({f for m in MUTANTS for f in m[4]})


def _pytest(lib, pins):
    env = dict(os.environ, OMP_NUM_THREADS="2", PYTHONDONTWRITEBYTECODE="1")
    env[oracle.LIB_OVERRIDE_ENV] = lib
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider"] + \
        [os.path.join(ROOT, "tests", f) for f in pins]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-1500:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Build every mutant (and the unmutated copy) and run its pins, in parallel."""
    with open(SRC) as f:
        text = f.read()
    work = tmp_path_factory.mktemp("mutants")
    jobs = {"unmutated": (text, ALL_PINS)}
    for mid, _, old, new, pins in MUTANTS:
        assert text.count(old) == 1, "mutation site of %s must occur exactly once" % mid
        jobs[mid] = (text.replace(old, new), pins)

    def run(item):
        mid, (src, pins) = item
        c = os.path.join(str(work), mid + ".c")
        with open(c, "w") as f:
            f.write(src)
        lib = obuild.compile_c(c, os.path.join(str(work), "lib_" + mid + ".so"))
        return mid, _pytest(lib, pins)

    workers = max(2, min(8, (os.cpu_count() or 4) // 2))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        return dict(ex.map(run, jobs.items()))


def test_unmutated_copy_passes_every_pin(outcomes):
    rc, out = outcomes["unmutated"]
    assert rc == 0, out


@pytest.mark.parametrize("mid,what", [(m[0], m[1]) for m in MUTANTS], ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(outcomes, mid, what):
    rc, out = outcomes[mid]
    # exit code 1: tests ran and at least one failed (not a crash, not a collection error)
    assert rc == 1, "%s (%s) was not caught:\n%s" % (mid, what, out)
