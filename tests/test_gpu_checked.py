"""The KPOOL_CHECKED build of the library: its internal bounds checks (computed token, pool and
score positions of the pooling, scoring and select kernels; each failure would record
KPOOL_ERR_CHECK) stay quiet on the seeded workloads and edge layouts, and its results equal the
default build's bit for bit."""
import numpy as np
import pytest
import torch

from pooled_key_dsa_gb300 import build as B
from pooled_key_dsa_gb300 import kpooldsa as K
from pooled_key_dsa_gb300 import workloads
from tests import kpool_parity as KP

pytestmark = pytest.mark.gpu


def _forward(wl):
    inp = workloads.all_inputs(wl)
    dev = KP.to_dev(inp)
    p = KP.params_of(wl)
    kp, lay = K.kpool_build(dev["k"], dev["gate"], dev["ape"], dev["cu_seqlens"], p)
    idx = K.dsa_index(dev["q_idx"], dev["w"], kp, lay, wl.topk, p, W=wl.W)
    out, lse = K.sparse_mla_fwd(dev["q_lat"], dev["kv_lat"], idx, wl.scale, status=lay.status)
    st = K.check_status(lay.status)
    return st, kp.cpu(), idx.cpu(), out.cpu(), lse.cpu()


@pytest.mark.parametrize("case", ["tiny", "packed8192", "short_docs", "scored_d128"])
def test_checked_build_is_quiet_and_equal(case):
    B.build()
    B.build(checked=True)
    assert torch.cuda.is_available()
    wl = {"tiny": lambda: workloads.workload(0),
          "packed8192": lambda: workloads.workload(2),
          "short_docs": lambda: workloads.custom("checked_short", 41, (1, 3, 4, 5, 0, 9, 2050, 4099), topk=16,
                                                 n_heads=8),
          "scored_d128": lambda: workloads.custom("checked_d128", 42, (2600, 1497, 7), topk=64)}[case]()
    ref = _forward(wl)
    assert ref[0] == 0
    K.use_checked_library(True)
    try:
        got = _forward(wl)
    finally:
        K.use_checked_library(False)
    assert got[0] == 0, K.ERRORS.get(got[0], got[0])
    for a, b in zip(ref[1:], got[1:]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def _host_forward(wl, n_chunks):
    inp = workloads.all_inputs(wl)
    host = {"k": inp.k, "gate": torch.from_numpy(inp.gate), "ape": torch.from_numpy(inp.ape),
            "cu_seqlens": torch.from_numpy(inp.cu_seqlens), "q_idx": inp.q_idx, "w": torch.from_numpy(inp.w),
            "q_lat": inp.q_lat, "kv_lat": inp.kv_lat}
    host = {k: v.contiguous().pin_memory() for k, v in host.items()}
    H = inp.q_lat.shape[1]
    host["out"] = torch.empty(tuple(inp.q_lat.shape), dtype=torch.bfloat16).pin_memory()
    host["lse"] = torch.empty((wl.T, H), dtype=torch.float32).pin_memory()
    dev = {k: torch.empty(tuple(v.shape), dtype=v.dtype, device="cuda") for k, v in host.items()}
    p = KP.params_of(wl)
    lay = K.PoolLayout(dev["cu_seqlens"], wl.T)
    dev["kpool"] = torch.empty((max(wl.T // 4, 1), wl.d_idx), dtype=torch.float32, device="cuda")
    dev["workspace"] = torch.empty(K.workspace_bytes(p, wl.T, lay.n_docs), dtype=torch.uint8, device="cuda")
    dev["indices"] = torch.empty((wl.T, wl.W), dtype=torch.int32, device="cuda")
    s = K.forward_host(host, dev, lay, p, n_chunks=n_chunks)
    s.synchronize()
    return K.check_status(lay.status, s), dev["indices"].cpu(), host["out"].clone(), host["lse"].clone()


def test_checked_build_on_the_blocked_host_forward():
    # the host forward indexes each query-row block on its own: block edges inside documents, blocks without
    # scored rows, and an item range per block; the checked build's bounds checks must stay quiet there too
    B.build()
    B.build(checked=True)
    wl = workloads.custom("checked_blocks", 43, (3, 5, 700, 9, 2051, 2060, 1), topk=64)
    ref = _host_forward(wl, 37)
    assert ref[0] == 0
    K.use_checked_library(True)
    try:
        got = _host_forward(wl, 37)
    finally:
        K.use_checked_library(False)
    assert got[0] == 0, K.ERRORS.get(got[0], got[0])
    for a, b in zip(ref[1:], got[1:]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
