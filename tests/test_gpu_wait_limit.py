"""The bounded waits of the two tcgen05 kernels of the forward run out, on demand, and leave the context usable.

Every mbarrier wait of the scoring and sparse attention kernels gives up after about two seconds, records
KPOOL_ERR_TIMEOUT, and every warp role then leaves its loop, waits for its copies and MMAs in flight and frees
TMEM.  kpool_debug_inject_stall makes one role of each kernel wait first on a barrier that nothing completes
(a flag that nothing sets), so that path runs here.  The next normal call on the same context must then give
results bit-identical to a clean run: TMEM was freed (a kernel that leaked it could not allocate again) and no
copy was left writing."""
import numpy as np
import pytest
import torch

from pooled_key_dsa_gb300 import build as B
from pooled_key_dsa_gb300 import kpooldsa as K
from pooled_key_dsa_gb300 import workloads
from tests import kpool_parity as KP

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    K.lib()
    yield
    K.debug_inject_stall(0)


def _index(wl, dev, p, layout, kp):
    layout.status.zero_()
    idx = K.dsa_index(dev["q_idx"], dev["w"], kp, layout, wl.topk, p, W=wl.W)
    return idx, K.check_status(layout.status)


def test_stalled_waits_time_out_and_the_next_calls_match_a_clean_run():
    # two documents long enough for scored rows (topk 64 pools), d_i = 128 so the tcgen05 scorer runs,
    # more query rows than SMs so the attention runs its persistent instance
    wl = workloads.custom("stall", 31, (2600, 1497), topk=64)
    inp = workloads.indexer_inputs(wl)
    dev = KP.to_dev(inp)
    p = KP.params_of(wl)
    kp, layout = K.kpool_build(dev["k"], dev["gate"], dev["ape"], dev["cu_seqlens"], p)
    assert K.check_status(layout.status) == 0
    q = workloads.q_lat(wl).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    idx0, st = _index(wl, dev, p, layout, kp)
    assert st == 0
    out0, lse0 = K.sparse_mla_fwd(q, dev["kv_lat"], idx0, wl.scale, status=status)
    assert K.check_status(status) == 0

    # scoring: its TMA producer never loads, so the MMA issuer and the epilogue warps time out too
    K.debug_inject_stall(K.STALL_SCORE)
    try:
        _, st = _index(wl, dev, p, layout, kp)
    finally:
        K.debug_inject_stall(0)
    assert st == K.CODES["KPOOL_ERR_TIMEOUT"], K.ERRORS.get(st, st)
    idx1, st = _index(wl, dev, p, layout, kp)
    assert st == 0
    assert torch.equal(idx1, idx0)

    # sparse attention: its row scanner never publishes a block count, so every role's wait runs out
    K.debug_inject_stall(K.STALL_SPARSE_MLA)
    try:
        status.zero_()
        K.sparse_mla_fwd(q, dev["kv_lat"], idx0, wl.scale, status=status)
        st = K.check_status(status)
    finally:
        K.debug_inject_stall(0)
    assert st == K.CODES["KPOOL_ERR_TIMEOUT"], K.ERRORS.get(st, st)
    status.zero_()
    out1, lse1 = K.sparse_mla_fwd(q, dev["kv_lat"], idx0, wl.scale, status=status)
    assert K.check_status(status) == 0
    assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))
    assert np.array_equal(lse1.cpu().numpy().view(np.uint32), lse0.cpu().numpy().view(np.uint32))
