"""Mutation check of the CPU oracle's pins (a script, not collected by pytest).

Each mutant is one small, plausible mistake in a function under ``oracle/``
(a dropped term, a wrong sign, index, bound, operand or order).  For each, the
repository is copied to a scratch directory, the mistake is planted there,
and the oracle pin tests run on the CPU; a mutant must make at least one of
them fail.  Mutants marked equivalent cannot change any result (the reason is
given beside each) and must pass.

    python tests/oracle_mutants.py [--dst DIR] [--only I ...]

The source tree itself is never modified; the copy lives in DIR/oracle_mutants_copy
(DIR defaults to a new temporary directory) and is removed at the end.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_TESTS = ["tests/test_oracle_pins.py", "tests/test_topk_pins.py", "tests/test_sparse_pins.py"]

# (file, text, replacement, what the mistake is, reason when it is equivalent)
MUTANTS = [
    ('oracle/msa_oracle.c',
     'ldexp((double)m, -24)',
     'ldexp((double)m, -25)',
     'half subnormal exp', None),
    ('oracle/msa_oracle.c',
     'ldexp((double)(m + 1024), e - 25)',
     'ldexp((double)(m + 1024), e - 24)',
     'half normal exp', None),
    ('oracle/msa_oracle.c',
     'v = m ? NAN : INFINITY;\n    else\n        v = ldexp((double)(m + 1024)',
     'v = INFINITY;\n    else\n        v = ldexp((double)(m + 1024)',
     'half nan', None),
    ('oracle/msa_oracle.c',
     '(uint32_t)h << 16',
     '((uint32_t)h << 16) | 1u',
     'bf16 low bit', None),
    ('oracle/msa_oracle.c',
     'if (e == 15 && m == 7)',
     'if (e == 15 && m >= 6)',
     'e4m3 nan', None),
    ('oracle/msa_oracle.c',
     'ldexp((double)m, -9)',
     'ldexp((double)m, -10)',
     'e4m3 subnormal', None),
    ('oracle/msa_oracle.c',
     'ldexp((double)(m + 8), e - 10)',
     'ldexp((double)(m + 8), e - 9)',
     'e4m3 normal', None),
    ('oracle/msa_oracle.c',
     'ldexp((double)m, -16)',
     'ldexp((double)m, -15)',
     'e5m2 subnormal', None),
    ('oracle/msa_oracle.c',
     'ldexp((double)(m + 4), e - 17)',
     'ldexp((double)(m + 4), e - 16)',
     'e5m2 normal', None),
    ('oracle/msa_oracle.c',
     'ldexp((double)m, -1)           /*',
     'ldexp((double)m, 0)           /*',
     'e2m1 subnormal', None),
    ('oracle/msa_oracle.c',
     'ldexp((double)(m + 2), e - 2)',
     'ldexp((double)(m + 2), e - 1)',
     'e2m1 normal', None),
    ('oracle/msa_oracle.c',
     'ldexp(1.0, (int)b - 127)',
     'ldexp(1.0, (int)b - 126)',
     'e8m0 bias', None),
    ('oracle/msa_oracle.c',
     'const int G = fmt ? 16 : 32;',
     'const int G = fmt ? 32 : 16;',
     'fp4 group size', None),
    ('oracle/msa_oracle.c',
     '(d & 1) ? (byte >> 4) : (byte & 15)',
     '(d & 1) ? (byte & 15) : (byte >> 4)',
     'fp4 nibble order', "query and key bytes are read with the same order and a byte's two codes share a scale group, so every dot product is unchanged"),
    ('oracle/msa_oracle.c',
     'return v * (fmt ? e4m3_to_double(sb) : e8m0_to_double(sb));',
     'return v * (fmt ? e8m0_to_double(sb) : e8m0_to_double(sb));',
     'nvfp4 scale type', None),
    ('oracle/msa_oracle.c',
     'a->cu_q[b] <= t && t < a->cu_q[b + 1]',
     'a->cu_q[b] <= t && t <= a->cu_q[b + 1]',
     'request_of bound', None),
    ('oracle/msa_oracle.c',
     'int64_t row = (int64_t)a->cu_k[b] + j;',
     'int64_t row = (int64_t)a->cu_k[b] + j + (j > 0);',
     'TND row', None),
    ('oracle/msa_oracle.c',
     '*scale_idx = row * a->H_kv + hk;',
     '*scale_idx = row * a->H_kv;',
     'TND scale idx', None),
    ('oracle/msa_oracle.c',
     'return page * a->page_stride + (off * a->H_kv + hk) * ru;',
     'return page * a->page_stride + ((int64_t)hk * a->P + off) * ru;',
     'BBND offset', None),
    ('oracle/msa_oracle.c',
     '*scale_idx = (page * a->H_kv + hk) * (int64_t)a->P + off;',
     '*scale_idx = (page * a->P + off) * (int64_t)a->H_kv + hk;',
     'paged scale idx', None),
    ('oracle/msa_oracle.c',
     'a->sparse_mode == 3 ? L - Lq + i : INT64_MAX',
     'a->sparse_mode == 3 ? L - Lq + i - 1 : INT64_MAX',
     'qpos off by one', None),
    ('oracle/msa_oracle.c',
     'if (j >= L || j > qpos)',
     'if (j > L || j > qpos)',
     'kv_len mask', None),
    ('oracle/msa_oracle.c',
     'if (j >= L || j > qpos)',
     'if (j >= L || j >= qpos)',
     'causal mask', None),
    ('oracle/msa_oracle.c',
     'if (!any || s > best)',
     'if (!any || s < best)',
     'max -> min', None),
    ('oracle/msa_oracle.c',
     '            if (a->k_dtype == 2)\n                s *= (double)a->scale[sidx];                 /* DEQUANT (column scale) */\n            if (!any || s > best)                            /* MAX */\n                best = s;\n',
     '            if (!any || s > best)                            /* MAX */\n                best = s;\n            if (a->k_dtype == 2 && j == beta * a->P + a->P - 1)\n                best *= (double)a->scale[sidx];\n',
     'int8 scale after the max', None),
    ('oracle/msa_oracle.c',
     'dst[beta] = 1e29f;',
     'dst[beta] = dst[beta] == 1e30f ? 1e30f : 1e29f;',
     'init overrides local', None),
    ('oracle/msa_oracle.c',
     'int64_t lo = sl + 1 - a->local_blocks;',
     'int64_t lo = sl - a->local_blocks;',
     'local window lo', None),
    ('oracle/msa_oracle.c',
     'for (int64_t beta = lo; beta <= sl && beta < a->MB; ++beta)',
     'for (int64_t beta = lo; beta < sl && beta < a->MB; ++beta)',
     'local window hi', None),
    ('oracle/msa_oracle.c',
     'if (L > 0 && (a->init_blocks > 0 || a->local_blocks > 0))',
     'if ((a->init_blocks > 0 || a->local_blocks > 0))',
     'local mask on empty kv', None),
    ('oracle/msa_oracle.c',
     'const int hk = h / g;',
     'const int hk = h % a->H_kv;',
     'gqa head map', None),
    ('oracle/msa_oracle.c',
     '(t * a->H_q + h) * ng, d, a->fp4_format) *',
     '(t * a->H_q + h) * ng + (d >= 64), d, a->fp4_format) *',
     'fp4 q scale row', None),
    ('oracle/msa_oracle.c',
     'dst[beta] = any ? (float)best : a->fill_value;',
     'dst[beta] = any ? (float)(best + 1e-30) : a->fill_value;',
     'score nudged before rounding', None),
    ('oracle/msa_oracle.c',
     'for (int64_t beta = 0; beta < a->MB; ++beta) {\n        double best',
     'for (int64_t beta = 0; beta < a->MB - (a->MB > 3); ++beta) {\n        double best',
     'last column skipped', None),
    ('oracle/msa_oracle.c',
     'for (int64_t beta = 0; beta < a->init_blocks && beta < a->MB; ++beta)',
     'for (int64_t beta = 0; beta <= a->init_blocks && beta < a->MB; ++beta)',
     'init range', None),
    ('oracle/topk.py',
     'order = np.lexsort((idx, -s.astype(np.float64)))',
     'order = np.lexsort((-idx, -s.astype(np.float64)))',
     'tie order', None),
    ('oracle/topk.py',
     'chosen = np.sort(idx[order[:k]])',
     'chosen = idx[order[:k]]',
     'not sorted by index', None),
    ('oracle/topk.py',
     'valid = s > np.float32(-np.inf)',
     'valid = s >= np.float32(-np.inf)',
     '-inf selectable', None),
    ('oracle/topk.py',
     'gs = np.fmax.reduce(sc.reshape(R, g, T, MBp), axis=1)',
     'gs = sc.reshape(R, g, T, MBp)[:, 0]',
     'group score first head', None),
    ('oracle/topk.py',
     'gs = np.fmax.reduce(sc.reshape(R, g, T, MBp), axis=1)',
     'gs = np.fmax.reduce(sc.reshape(g, R, T, MBp), axis=0)',
     'group head interleave', None),
    ('oracle/topk.py',
     'if 0 <= qpos < L and qpos // P < MB:',
     'if 0 <= qpos <= L and qpos // P < MB:',
     'local block bound', 'q_pos = kv_len - Lq + i is at most kv_len - 1, so q_pos <= kv_len never admits more'),
    ('oracle/topk.py',
     'qpos = L - Lq + i',
     'qpos = L - Lq + i - 1',
     'local qpos', None),
    ('oracle/topk.py',
     'rest[loc] = np.float32(-np.inf)',
     'pass',
     'local duplicate', None),
    ('oracle/topk.py',
     'row_topk(rest, MB, k - 1)',
     'row_topk(rest, MB, k)',
     'local slot extra', None),
    ('oracle/sparse_attention.py',
     'if j < L and (case.sparse_mode != 3 or j <= qpos):',
     'if j < L and (case.sparse_mode != 3 or j < qpos):',
     'sparse causal', None),
    ('oracle/sparse_attention.py',
     'if beta < 0 or beta >= MB or beta >= nb:',
     'if beta < 0 or beta >= MB:',
     'sparse blocks past the last', 'a block at or past ceil(kv_len / P) holds no position below kv_len, so it adds no key'),
    ('oracle/sparse_attention.py',
     's = scale * (kk @ q[t, h])',
     's = (kk @ q[t, h])',
     'sm scale', None),
    ('oracle/sparse_attention.py',
     'LSE[t, h] = m + math.log(w.sum())',
     'LSE[t, h] = math.log(w.sum())',
     'lse max', None),
    ('oracle/sparse_attention.py',
     '        r = h // g\n        Lq',
     '        r = h % case.H_kv\n        Lq',
     'sparse head map', None),
    ('oracle/sparse_attention.py',
     'vv = _key_rows(case, value, b, js, r)',
     'vv = _key_rows(case, case.key, b, js, r)',
     'V is K', None),
    ('oracle/sparse_attention.py',
     'O[t, h] = (w[:, None] * vv).sum(axis=0) / w.sum()',
     'O[t, h] = (w[:, None] * vv).sum(axis=0) / (w.sum() + 1e-3)',
     'normaliser', None),
    ('oracle/sparse_attention.py',
     'scale = 1.0 / math.sqrt(D) if sm_scale is None',
     'scale = 1.0 / D if sm_scale is None',
     'default scale', None),
    ('oracle/sparse_attention.py',
     'base = int(case.cu_seqlens_k[b])',
     'base = int(case.cu_seqlens_k[b]) + 1',
     'sparse TND base', None),
    ('oracle/sparse_attention.py',
     'L = int(case.cu_seqlens_k[b + 1] - case.cu_seqlens_k[b])',
     'L = int(case.cu_seqlens_k[b + 1] - case.cu_seqlens_k[b]) - 1',
     'sparse TND length', None),
    ('oracle/sparse_attention.py',
     'qpos = L - Lq + (t - cu[b])',
     'qpos = L - Lq + (t - cu[b]) - 1',
     'sparse qpos', None),
    ('oracle/sparse_attention.py',
     'for j in range(beta * P, beta * P + P):',
     'for j in range(beta * P, beta * P + P - 1):',
     'sparse block width', None),
    ('oracle/sparse_attention.py',
     'return _f64(cache[pages, off, r])',
     'return _f64(cache[pages, off, 0])',
     'sparse bbnd head', None),
    ('oracle/topk.py',
     's = np.asarray(row, dtype=np.float32)[:MB]',
     's = np.asarray(row, dtype=np.float32)',
     'padding selectable', None),
    ('oracle/topk.py',
     'h, t = divmod(int(r), T)',
     't, h = divmod(int(r), H)',
     'block_topk row order', None),
    ('oracle/topk.py',
     'r, t = divmod(int(flat), T)',
     't, r = divmod(int(flat), R)',
     'group_topk row order', None),
    ('oracle/sparse_attention.py',
     't, h = divmod(int(flat), H_q)',
     'h, t = divmod(int(flat), T)',
     'sparse row order', None),
    ('oracle/msa_oracle.c',
     'int h = (int)(rows[r] / a->T);\n        int64_t t = rows[r] % a->T;',
     'int h = (int)(rows[r] % a->H_q);\n        int64_t t = rows[r] / a->H_q;',
     'oracle row order', None),
    ('oracle/topk.py',
     'out[: chosen.shape[0]] = chosen',
     'out[k - chosen.shape[0]:] = chosen',
     'tail at front', None),
    ('oracle/msa_oracle.c',
     'const int64_t qrow = (t * a->H_q + h) * row_units(a);',
     'const int64_t qrow = (t * a->H_q + (h ^ 1)) * row_units(a);',
     'query head', None),
    ('oracle/msa_oracle.c',
     'return page * a->page_stride + ((int64_t)hk * a->P + off) * ru;  /* BNBD */',
     'return page * a->page_stride + (off * a->H_kv + hk) * ru;  /* BNBD */',
     'BNBD offset', None),
    ('oracle/msa_oracle.c',
     'return a->k_dtype == 5 ? a->D / 2 : a->D;',
     'return a->D;',
     'fp4 row units', None),
]


def run_one(dst: str, mutant) -> bool:
    """Plant one mutant in a fresh copy; True when the pin tests fail."""
    path, old, new, _, _ = mutant
    if os.path.exists(dst):
        shutil.rmtree(dst)
    shutil.copytree(ROOT, dst, ignore=shutil.ignore_patterns(
        ".git", "_work", "gpurun_out", "__pycache__", ".pytest_cache", "*.so", "_build"))
    target = os.path.join(dst, path)
    with open(target) as fh:
        src = fh.read()
    if src.count(old) != 1:
        raise SystemExit(f"mutant text not found exactly once in {path}: {old[:60]!r}")
    with open(target, "w") as fh:
        fh.write(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu",
                        "-p", "no:cacheprovider", *PIN_TESTS],
                       cwd=dst, capture_output=True, text=True)
    return r.returncode != 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--dst", default=None,
                    help="directory under which the mutated copy is made (default: a new "
                         "temporary directory); only its subdirectory oracle_mutants_copy "
                         "is written and removed")
    ap.add_argument("--only", type=int, nargs="*", default=None, help="mutant numbers to run")
    args = ap.parse_args()
    parent = args.dst or tempfile.mkdtemp(prefix="oracle_mutants_")
    os.makedirs(parent, exist_ok=True)
    scratch = os.path.join(parent, "oracle_mutants_copy")
    bad = 0
    for i, m in enumerate(MUTANTS):
        if args.only is not None and i not in args.only:
            continue
        killed = run_one(scratch, m)
        expect_killed = m[4] is None
        ok = killed == expect_killed
        bad += not ok
        state = "killed" if killed else "survived"
        note = "" if expect_killed else " (equivalent)"
        print(f"{i:3d} {m[0]:28s} {m[3]:34s} {state}{note}{'' if ok else '  <-- UNEXPECTED'}",
              flush=True)
    shutil.rmtree(scratch, ignore_errors=True)
    if args.dst is None:
        shutil.rmtree(parent, ignore_errors=True)
    print("all as expected" if not bad else f"{bad} unexpected")
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
