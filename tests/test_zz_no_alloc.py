"""dsa_index_noalloc: the indexer for callers that cannot allocate device
memory (custom-op hosts that own all device memory, fixed memory pools,
loops that must not call cudaMalloc).  Its scratch is a static device array
inside the library, so this test checks, through the C ABI, that two calls in
a row give the same index rows as dsa_index with a caller-allocated
workspace, and that sizes past the array's limit are refused.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from pooled_key_dsa_gb300 import build as B
from pooled_key_dsa_gb300 import kpooldsa as K
from pooled_key_dsa_gb300 import workloads

pytestmark = pytest.mark.gpu


def _inputs(wl):
    inp = workloads.indexer_inputs(wl)
    p = K.make_params(topk=wl.topk, n_idx_heads=wl.n_idx_heads, d_idx=wl.d_idx, n_heads=wl.n_heads,
                      d_lat=wl.d_lat, scale=wl.scale)
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    kp, lay = K.kpool_build(inp.k.cuda(), torch.from_numpy(inp.gate).cuda(), torch.from_numpy(inp.ape).cuda(), cu, p)
    return p, lay, kp, inp.q_idx.cuda(), torch.from_numpy(inp.w).cuda()


def test_no_alloc_entry_matches_dsa_index_on_two_calls():
    B.build()
    assert torch.cuda.is_available()
    K.lib()
    # two different workloads in a row: the second call must not see the first's leftovers
    for wl in (workloads.custom("noalloc_a", 21, (2600, 1000, 496)),
               workloads.custom("noalloc_b", 22, (4093,), n_idx_heads=16, topk=300)):
        p, lay, kp, q_idx, w = _inputs(wl)
        ref = K.dsa_index(q_idx, w, kp, lay, wl.topk, p)
        got = K.dsa_index_noalloc(q_idx, w, kp, lay, wl.topk, p)
        torch.cuda.synchronize()
        assert K.check_status(lay.status) == 0
        np.testing.assert_array_equal(got.cpu().numpy(), ref.cpu().numpy())
        assert int((got >= 0).sum(dim=1).max()) == 4 * wl.topk + 3


def test_no_alloc_entry_refuses_sizes_past_its_limit():
    B.build()
    wl = workloads.custom("noalloc_big", 23, (4097,))
    p, lay, kp, q_idx, w = _inputs(wl)
    idx = torch.empty((wl.T, wl.W), dtype=torch.int32, device="cuda")
    rc = K.lib().dsa_index_noalloc(ctypes.c_void_p(q_idx.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                   ctypes.c_void_p(kp.data_ptr()), ctypes.byref(lay.c), wl.topk, ctypes.byref(p),
                                   ctypes.c_void_p(idx.data_ptr()), wl.W, None)
    assert rc == K.CODES["KPOOL_ERR_SHAPE"]
