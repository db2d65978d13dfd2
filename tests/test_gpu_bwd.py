"""Sparse latent attention backward on the GPU, through the C ABI, against the oracle.

Tolerances, derived from the arithmetic: P and dZ' enter the MMAs as bf16
(relative rounding up to 2^-9 each), sums are fp32, dq is returned in bf16
(2^-9 relative) and delta is formed from the forward's bf16 output.  Summed
over many slots these errors average out, so over a whole tensor the relative
RMS error stays below 4e-3 and no element is off by more than 2e-2 of the
tensor's largest magnitude.  (For context, the pages report cuDNN's sparse MLA
at 1.7e-3 relative RMSE for dQ and 3.7e-3 for dKV against a reference.)
"""
import numpy as np
import pytest
import torch

from oracle import kpool_oracle as O
from pooled_key_dsa_gb300 import build as B
from pooled_key_dsa_gb300 import kpooldsa as K
from pooled_key_dsa_gb300 import workloads
from tests import kpool_parity as KP

pytestmark = pytest.mark.gpu

REL_RMSE = 4e-3
MAX_REL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    K.lib()


def _close(gpu, ref, what):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    scale = np.sqrt((r ** 2).mean())
    rel_rmse = np.sqrt(((g - r) ** 2).mean()) / scale
    max_rel = np.abs(g - r).max() / np.abs(r).max()
    assert rel_rmse <= REL_RMSE and max_rel <= MAX_REL, (what, rel_rmse, max_rel)
    return rel_rmse


def _random_rows(T, W, rng, empty=()):
    idx = np.full((T, W), -1, np.int32)
    for i in range(T):
        if i in empty:
            continue
        n = int(rng.integers(1, W + 1))
        idx[i, :n] = np.sort(rng.choice(T, n, replace=False))
    return idx


def _fwd_bwd(q, kv, idx, scale, dout, status=None):
    out, lse = K.sparse_mla_fwd(q, kv, idx, scale, status=status)
    dq, dkv = K.sparse_mla_bwd(q, kv, idx, scale, out, lse, dout, status=status)
    return out, lse, dq, dkv


def test_backward_parity_several_blocks_and_ragged_rows():
    # 1200 queries (several per CTA), rows of 1..256 slots (up to 4 blocks, ragged), some empty rows
    wl = workloads.custom("bwd_rand", 31, (1200,), n_heads=64)
    q, kv = workloads.layer_attention_inputs(wl, 0)
    dout = workloads.dout_input(wl)
    rng = np.random.default_rng(5)
    idx = _random_rows(wl.T, 256, rng, empty={0, 7, 8, 160, 312})
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, dq, dkv = _fwd_bwd(q.cuda(), kv.cuda(), torch.from_numpy(idx).cuda(), wl.scale, dout.cuda(), st)
    assert K.check_status(st) == 0
    ref = O.sparse_attention_bwd(q.float().numpy(), kv.float().numpy(), idx, wl.scale, dout.float().numpy(),
                                 np.arange(wl.T))
    dq_g = dq.float().cpu().numpy()
    assert np.all(dq_g[[0, 7, 8, 160, 312]] == 0)
    _close(dq_g, ref["dq"], "dq")
    _close(dkv.cpu().numpy(), ref["dkv"], "dkv")


@pytest.mark.parametrize("H", [1, 4, 20])
def test_backward_small_head_counts(H):
    wl = workloads.custom("bwd_heads", 9, (300,), n_heads=H)
    q, kv = workloads.layer_attention_inputs(wl, 0)
    dout = workloads.dout_input(wl)
    idx = np.full((wl.T, 128), -1, np.int32)
    for i in range(wl.T):                       # causal rows, the last 128 positions
        lo = max(0, i - 127)
        idx[i, :i - lo + 1] = np.arange(lo, i + 1)
    out, lse, dq, dkv = _fwd_bwd(q.cuda(), kv.cuda(), torch.from_numpy(idx).cuda(), wl.scale, dout.cuda())
    ref = O.sparse_attention_bwd(q.float().numpy(), kv.float().numpy(), idx, wl.scale, dout.float().numpy(),
                                 np.arange(wl.T))
    _close(dq.float().cpu().numpy(), ref["dq"], "dq")
    _close(dkv.cpu().numpy(), ref["dkv"], "dkv")


def test_backward_tiny_workload_on_its_index_rows():
    wl = workloads.workload(0)
    inp = workloads.all_inputs(wl)
    d = KP.to_dev(inp)
    p = KP.params_of(wl)
    kp, lay = K.kpool_build(d["k"], d["gate"], d["ape"], d["cu_seqlens"], p)
    idx = K.dsa_index(d["q_idx"], d["w"], kp, lay, wl.topk, p, W=wl.W)
    dout = workloads.dout_input(wl)
    out, lse, dq, dkv = _fwd_bwd(d["q_lat"], d["kv_lat"], idx, wl.scale, dout.cuda(), lay.status)
    assert K.check_status(lay.status) == 0
    ref = O.sparse_attention_bwd(inp.q_lat.float().numpy(), inp.kv_lat.float().numpy(), idx.cpu().numpy(),
                                 wl.scale, dout.float().numpy(), np.arange(wl.T))
    _close(dq.float().cpu().numpy(), ref["dq"], "dq")
    _close(dkv.cpu().numpy(), ref["dkv"], "dkv")


def _identity_gap(q, kv, dq, dkv, dout, out):
    """<dkv, kv> - <dq, q> - <dout, out> (zero by the logit-scaling identity), in float64, relative to the sum of
    the absolute products (a bound on how far elementwise rounding can move the three sums)."""
    a, b, c = dkv.double() * kv.double(), dq.double() * q.double(), dout.double() * out.double()
    gap = float(a.sum() - b.sum() - c.sum())
    return abs(gap) / float(a.abs().sum() + b.abs().sum() + c.abs().sum())


@pytest.mark.parametrize("cfg", [2, 3])
def test_backward_full_size_sampled(cfg):
    # the forward's own index rows at full size: dq on sampled rows; dkv on the last 48 latent rows
    # (only the queries at or after them can select them, so the oracle takes just those queries);
    # the scaling identity over the whole tensors
    wl = workloads.workload(cfg)
    inp = workloads.all_inputs(wl)
    d = KP.to_dev(inp)
    p = KP.params_of(wl)
    kp, lay = K.kpool_build(d["k"], d["gate"], d["ape"], d["cu_seqlens"], p)
    idx = K.dsa_index(d["q_idx"], d["w"], kp, lay, wl.topk, p, W=wl.W)
    dout = workloads.dout_input(wl).cuda()
    out, lse, dq, dkv = _fwd_bwd(d["q_lat"], d["kv_lat"], idx, wl.scale, dout, lay.status)
    assert K.check_status(lay.status) == 0
    idx_h = idx.cpu().numpy()
    kv_np = inp.kv_lat.float().numpy()
    rows = np.unique(np.concatenate([np.linspace(0, wl.T - 1, 24).astype(np.int64),
                                     [2047, 2048, 2051, wl.T - 1]]))
    dsel = torch.from_numpy(rows).cuda()
    ref = O.sparse_attention_bwd(inp.q_lat[rows].float().numpy(), kv_np, idx_h[rows], wl.scale,
                                 dout[dsel].float().cpu().numpy(), rows)
    _close(dq[dsel].float().cpu().numpy(), ref["dq"], "dq")
    tail = np.arange(wl.T - 48, wl.T)
    ref_t = O.sparse_attention_bwd(inp.q_lat[tail].float().numpy(), kv_np, idx_h[tail], wl.scale,
                                   dout[torch.from_numpy(tail).cuda()].float().cpu().numpy(), tail)
    _close(dkv[wl.T - 48:].cpu().numpy(), ref_t["dkv"][wl.T - 48:], "dkv tail")
    assert _identity_gap(d["q_lat"], d["kv_lat"], dq, dkv, dout, out) < 1e-3


def test_backward_empty_rows_out_of_range_and_repeatability():
    wl = workloads.custom("bwd_edge", 12, (700,), n_heads=64)
    q, kv = workloads.layer_attention_inputs(wl, 0)
    dout = workloads.dout_input(wl)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(3)
    empty = {i for i in range(wl.T) if (i // n_sm) % 3 == 1}        # consecutive empty queries per CTA
    idx = _random_rows(wl.T, 192, rng, empty=empty)
    idx[5, 2] = wl.T + 3                                             # out of range: skipped and flagged
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd, kvd, idd, dd = q.cuda(), kv.cuda(), torch.from_numpy(idx).cuda(), dout.cuda()
    out, lse, dq, dkv = _fwd_bwd(qd, kvd, idd, wl.scale, dd, st)
    assert K.check_status(st) == K.CODES["KPOOL_ERR_INDEX_RANGE"]
    dq2, dkv2 = K.sparse_mla_bwd(qd, kvd, idd, wl.scale, out, lse, dd)
    assert torch.equal(dq, dq2)                                      # dq has a fixed summation order
    # dkv: fp32 atomics whose order varies between runs.  An element sums up to ~1000 contributions, so two
    # runs differ by the rounding of two summation orders (a few 1e-6 absolute at this magnitude), which a
    # fixed 1e-6 floor does not cover near zero; the floor is set by the tensor's own scale instead.
    assert torch.allclose(dkv, dkv2, rtol=1e-5, atol=2e-5 * float(dkv.abs().max()))
    ref_idx = idx.copy()
    ref_idx[(ref_idx < -1) | (ref_idx >= wl.T)] = -1
    ref = O.sparse_attention_bwd(q.float().numpy(), kv.float().numpy(), ref_idx, wl.scale, dout.float().numpy(),
                                 np.arange(wl.T))
    dq_g = dq.float().cpu().numpy()
    assert np.all(dq_g[sorted(empty)] == 0)
    _close(dq_g, ref["dq"], "dq")
    _close(dkv.cpu().numpy(), ref["dkv"], "dkv")
