"""Row-parallel driver of the CPU oracle for the GPU parity tests (test infrastructure only).

Checks many query rows of the indexer at once: for each row the oracle quantises the query (Hadamard + FP8),
scores the row's candidate pools on the GPU's own FP8 keys, selects and builds the index row, and the result
is compared with what the GPU produced for that row.  Rows are independent, so chunks of rows run in
separate processes of a ``spawn`` pool (never forked: the parent holds a CUDA context).  This module imports
only numpy and the oracle, so that the workers start without torch.  The oracle itself is unchanged: this
file only calls it row by row.
"""
from __future__ import annotations

import os

import numpy as np

from oracle import kpool_oracle as O

# Tolerance of the index rows: bit-exact, except pools whose oracle score lies within this relative distance
# of the row's topk-th score (boundary pools, counted and reported).
BOUNDARY_RTOL = 1e-3

_SHARED = {}


def compare_rows(gpu_rows, layout, rows, oracle_scores, topk, W):
    """Compares GPU index rows with the oracle's selection rule.  Returns a dict of counts; 'hard' counts rows
    that differ other than at boundary pools (pools whose oracle score is within BOUNDARY_RTOL of the row's
    topk-th score)."""
    stats = {"rows": 0, "exact": 0, "boundary_rows": 0, "boundary_pools": 0, "hard": 0, "hard_rows": []}
    for n, i in enumerate(rows):
        i = int(i)
        d, r, n_i, tail = O.query_geometry(layout, i)
        S = oracle_scores[n]
        sel = O.select_pools(S, topk)
        want = O.index_row(layout, i, sel, W)
        got = gpu_rows[n]
        stats["rows"] += 1
        if np.array_equal(got, want):
            stats["exact"] += 1
            continue
        # structural validity of the GPU row
        valid = got[got >= 0]
        nv = 4 * min(topk, n_i) + tail
        s_d = int(layout["cu_seqlens"][d])
        ok = (len(valid) == nv and np.all(got[nv:] == -1) and np.all(np.diff(valid) > 0)
              and valid.min() >= s_d and valid.max() <= i)
        if ok and tail:
            ok = valid[-tail:].tolist() == list(range(i - tail + 1, i + 1))
        gsel = np.zeros(0, np.int64)
        if ok:
            blocks = (valid[:nv - tail] - s_d).reshape(-1, 4)
            ok = bool(np.all(blocks == blocks[:, :1] + np.arange(4)) and np.all(blocks[:, 0] % 4 == 0))
            gsel = blocks[:, 0] // 4
        if not ok:
            stats["hard"] += 1
            stats["hard_rows"].append(i)
            continue
        Sd = np.asarray(S, np.float64)
        kth = np.sort(Sd)[::-1][min(topk, n_i) - 1]
        diff = set(gsel.tolist()) ^ set(sel.tolist())
        near = all(abs(Sd[p] - kth) <= BOUNDARY_RTOL * abs(kth) for p in diff)
        if near:
            stats["boundary_rows"] += 1
            stats["boundary_pools"] += len(diff) // 2
        else:
            stats["hard"] += 1
            stats["hard_rows"].append(i)
    return stats


def merge_stats(parts):
    out = {"rows": 0, "exact": 0, "boundary_rows": 0, "boundary_pools": 0, "hard": 0, "hard_rows": []}
    for s in parts:
        for k in ("rows", "exact", "boundary_rows", "boundary_pools", "hard"):
            out[k] += s[k]
        out["hard_rows"] += s["hard_rows"]
    return out


def _init(shared):
    _SHARED.clear()
    _SHARED.update(shared)


def _bf16_bits_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


U32 = 2.0 ** -24          # unit roundoff of fp32


def gamma(n: int) -> float:
    """Bound on the relative error of an n-term fp32 sum (n u / (1 - n u))."""
    return n * U32 / (1.0 - n * U32)


def score_error_bound(qd_abs, kd_abs, ws_abs, sk, o_abs):
    """Per-pool bound on |GPU score - oracle score| for one query row.  The E4M3 products are exact in fp32;
    the GPU sums the d_i products of a head in fp32 (error <= gamma(d_i) * sum |q k|), takes ReLU (exact), sums
    the H_i weighted heads in fp32 (error <= gamma(H_i + 2) * sum |ws| ReLU, and ReLU(x) <= sum |q k|), scales by
    s_k (one rounding); the oracle's fp64 result is rounded to fp32 once.  So
    |d| <= s_k * (gamma(d_i) + gamma(H_i + 2)) * sum_h |ws_h| A_hp + 2^-23 |S_p|, A_hp = sum_d |q_hd| |k_pd|."""
    A = qd_abs @ kd_abs.T                                        # [H_i, n]
    hi, di = qd_abs.shape
    return sk * (gamma(di) + gamma(hi + 2)) * (ws_abs @ A) + 2.0 ** -23 * o_abs


def check_chunk(task):
    """One chunk of rows: (rows, q_idx bf16 bits [n,H_i,d_i], GPU q8 [n,H_i,d_i], GPU ws [n,H_i], GPU scores
    (one array or None per row), GPU index rows [n,W]).  Returns the q8/ws mismatch counts, the worst score
    error relative to the row's largest oracle score, the worst ratio of a score's error to its own bound
    (:func:`score_error_bound`), and the row comparison counts."""
    rows, qbits, q8_g, ws_g, sc_g, idx_g = task
    sh = _SHARED
    q8_o, sq_o = O.quantize_queries(_bf16_bits_to_f32(qbits))
    q8_bad = int(np.count_nonzero(np.any(q8_o != q8_g, axis=(1, 2))))
    ws_o = (sh["w"][rows] * sq_o).astype(np.float32)
    ws_bad = int(np.count_nonzero(np.any(ws_o.view(np.uint32) != ws_g.view(np.uint32), axis=1)))
    S_o = O.scores_fp8(q8_o, sq_o, sh["k8"], sh["s_k"], sh["w"], sh["layout"], rows)
    if "kd_abs" not in sh:
        sh["kd_abs"] = np.abs(O.e4m3_decode(sh["k8"]))
    worst = 0.0
    worst_bound = 0.0
    for n, g in enumerate(sc_g):
        if g is None:
            continue
        o = S_o[n].astype(np.float64)
        scale = max(np.abs(o).max(), 1e-30)
        err = np.abs(np.asarray(g, np.float64) - o)
        worst = max(worst, float(err.max() / scale))
        d, _, n_i, _ = O.query_geometry(sh["layout"], int(rows[n]))
        p0 = int(sh["layout"]["cu_pools"][d])
        bound = score_error_bound(np.abs(O.e4m3_decode(q8_o[n])), sh["kd_abs"][p0:p0 + n_i],
                                  np.abs(ws_o[n].astype(np.float64)),
                                  np.asarray(sh["s_k"][p0:p0 + n_i], np.float64), np.abs(o))
        worst_bound = max(worst_bound, float((err / np.maximum(bound, 1e-300)).max()))
    stats = compare_rows(idx_g, sh["layout"], rows, S_o, sh["topk"], sh["W"])
    return {"q8_bad": q8_bad, "ws_bad": ws_bad, "worst": worst, "worst_bound": worst_bound, "stats": stats}


def check_rows(rows, qbits, q8_g, ws_g, scores_g, idx_g, shared, workers=None, chunk=256):
    """All rows, in chunks over a spawn pool of ``workers`` processes (default: the host's cores; 1 runs
    in this process).  Returns the merged result of :func:`check_chunk`."""
    rows = np.asarray(rows, np.int64)
    tasks = [(rows[a:a + chunk], qbits[a:a + chunk], q8_g[a:a + chunk], ws_g[a:a + chunk], scores_g[a:a + chunk],
              idx_g[a:a + chunk]) for a in range(0, len(rows), chunk)]
    workers = workers or os.cpu_count() or 1
    if workers <= 1 or len(tasks) <= 1:
        _init(shared)
        parts = [check_chunk(t) for t in tasks]
    else:
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        # one BLAS thread per worker process (set before the children import numpy)
        saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            with ProcessPoolExecutor(max_workers=min(workers, len(tasks)), mp_context=mp.get_context("spawn"),
                                     initializer=_init, initargs=(shared,)) as ex:
                parts = list(ex.map(check_chunk, tasks))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
    return {"q8_bad": sum(p["q8_bad"] for p in parts), "ws_bad": sum(p["ws_bad"] for p in parts),
            "worst": max((p["worst"] for p in parts), default=0.0),
            "worst_bound": max((p["worst_bound"] for p in parts), default=0.0),
            "stats": merge_stats([p["stats"] for p in parts])}
