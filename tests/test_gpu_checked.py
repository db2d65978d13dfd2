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
