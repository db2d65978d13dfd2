"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare its outputs with the CPU oracle.  Test infrastructure only."""
from __future__ import annotations

import numpy as np
import torch

from oracle import kpool_oracle as O
from pooled_key_dsa_gb300 import kpooldsa as K
from pooled_key_dsa_gb300 import workloads
from tests import oracle_rows as OR

# Tolerances (floating point): pooled keys within 1e-5 of the magnitude of the
# keys they mix; attention output 2e-2 max / 5e-3 mean absolute; LSE 1e-3
# absolute; index rows bit-exact except pools whose oracle score lies within
# 1e-3 relative of the row's topk-th score.
KPOOL_RTOL = 1e-5
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 5e-3
LSE_ABS = 1e-3
BOUNDARY_RTOL = OR.BOUNDARY_RTOL


def params_of(wl: workloads.Workload) -> K.Params:
    return K.make_params(topk=wl.topk, n_idx_heads=wl.n_idx_heads, d_idx=wl.d_idx, n_heads=wl.n_heads,
                         d_lat=wl.d_lat, scale=wl.scale)


def to_dev(inp: workloads.Inputs, dev="cuda"):
    d = {
        "cu_seqlens": torch.from_numpy(inp.cu_seqlens).to(dev),
        "q_idx": inp.q_idx.to(dev),
        "k": inp.k.to(dev),
        "gate": torch.from_numpy(inp.gate).to(dev),
        "ape": torch.from_numpy(inp.ape).to(dev),
        "w": torch.from_numpy(inp.w).to(dev),
        "kv_lat": inp.kv_lat.to(dev),
    }
    if inp.q_lat is not None:
        d["q_lat"] = inp.q_lat.to(dev)
    return d


def run_indexer(wl, dev_inp, topk=None, W=None):
    """kpool_build + dsa_index on the device; returns host copies of the
    layout, pooled keys, workspace intermediates and index rows."""
    p = params_of(wl)
    topk = wl.topk if topk is None else topk
    W = K.row_width(topk) if W is None else W
    kp, lay = K.kpool_build(dev_inp["k"], dev_inp["gate"], dev_inp["ape"], dev_inp["cu_seqlens"], p)
    nbytes = K.workspace_bytes(p, wl.T, lay.n_docs)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    idx = K.dsa_index(dev_inp["q_idx"], dev_inp["w"], kp, lay, topk, p, workspace=ws, W=W)
    st = K.check_status(lay.status)
    off = K.workspace_offsets(p, wl.T, lay.n_docs)
    T, Hi, di, P = wl.T, wl.n_idx_heads, wl.d_idx, wl.T // 4
    wsc = ws.cpu().numpy()
    res = {
        "status": st,
        "cu_pools": lay.cu_pools.cpu().numpy(),
        "pool_tok_start": lay.pool_tok_start.cpu().numpy()[:P],
        "tok_doc": lay.tok_doc.cpu().numpy()[:T],
        "kpool": kp.cpu().numpy()[:P],
        "q8": wsc[off.q8:off.q8 + T * Hi * di].reshape(T, Hi, di),
        "ws": wsc[off.ws:off.ws + T * Hi * 4].view(np.float32).reshape(T, Hi),
        "k8": wsc[off.k8:off.k8 + P * di].reshape(P, di),
        "s_k": wsc[off.s_k:off.s_k + P * 4].view(np.float32),
        "pair_base": wsc[off.pair_base:off.pair_base + (lay.n_docs + 1) * 8].view(np.int64),
        "scores_raw": wsc[off.scores:off.total].view(np.float32),
        "indices": idx.cpu().numpy(),
        "indices_dev": idx,
        "layout": lay,
        "W": W,
        "topk": topk,
    }
    return res


def gpu_row_scores(res, layout, i):
    """The GPU's scores of query row i (compact triangle), or None if the row
    keeps every candidate and is not scored."""
    d, r, n_i, _ = O.query_geometry(layout, i)
    if n_i <= res["topk"]:
        return None
    a, b = divmod(r, 4)
    start = int(res["pair_base"][d]) + 2 * a * (a - 1) + a * (b + 1)
    return res["scores_raw"][start:start + n_i]


compare_rows = OR.compare_rows

# One summary line per parity check of the index rows (rows, bit-exact, boundary rows and pools, hard), printed
# again at the end of the pytest run so that the counts reach the run's record even under -q.
PARITY_LOG = []


def record(line: str) -> None:
    PARITY_LOG.append(line)
    print(line)


def check_index_rows(wl, res, inp, lay_o, rows, workers=None):
    """Oracle check of the given query rows of the GPU indexer, in parallel over rows: the query FP8 codes and
    head weights bit-exact, the scores within 1e-5 of each row's largest, the index rows by the selection rule
    (bit-exact up to counted boundary pools).  Returns the merged counts."""
    rows = np.asarray(rows, np.int64)
    qbits = inp.q_idx.view(torch.int16).numpy().view(np.uint16)
    scores = [gpu_row_scores(res, lay_o, int(i)) for i in rows]
    shared = {"k8": res["k8"], "s_k": res["s_k"], "w": inp.w, "layout": lay_o, "topk": res["topk"], "W": res["W"]}
    return OR.check_rows(rows, qbits[rows], res["q8"][rows], res["ws"][rows], scores, res["indices"][rows], shared,
                         workers=workers)


def attention_check(out_gpu, lse_gpu, out_ref, lse_ref):
    """Max/mean absolute output error and max LSE error (finite LSEs)."""
    o = out_gpu.astype(np.float64)
    e = np.abs(o - out_ref.astype(np.float64))
    fin = np.isfinite(lse_ref)
    lse_err = float(np.abs(lse_gpu[fin].astype(np.float64) - lse_ref[fin]).max()) if fin.any() else 0.0
    assert np.array_equal(np.isfinite(lse_gpu), fin)
    return float(e.max()), float(e.mean()), lse_err


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def sample_rows(wl, n_uniform=256, seed=0):
    """Fixed, seeded sample of query rows: document starts and ends, the
    2048-position cutover region of every document, the last rows, and
    uniform rows."""
    rng = np.random.default_rng(seed)
    cu = wl.cu_seqlens
    rows = set()
    for d in range(len(cu) - 1):
        s, e = int(cu[d]), int(cu[d + 1])
        for r in list(range(0, 6)) + list(range(2044, 2057)) + [e - s - 2, e - s - 1]:
            if 0 <= r < e - s:
                rows.add(s + r)
    rows.update(range(max(0, wl.T - 4), wl.T))
    rows.update(rng.integers(0, wl.T, n_uniform).tolist())
    return np.array(sorted(rows), dtype=np.int64)
