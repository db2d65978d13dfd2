"""IndexShare: a shared DSA layer reuses the index rows of the full layer that
ran the indexer and calls only the sparse attention (NeMo AutoModel "GLM-5 /
GLM-5.1 / GLM-5.2 / GLM-5.3 (MoE + DSA)", Key Features: shared DSA layers reuse
the previous full layer's top-k selection).  Its outputs are checked against the oracle's attention on the
same rows, and the shared rows are the indexer layer's, bit for bit."""
import numpy as np
import pytest
import torch

from oracle import kpool_oracle as O
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


@pytest.mark.parametrize("cfg", [0, 2])
def test_shared_layer_attention_on_the_indexer_layers_rows(cfg):
    wl = workloads.workload(cfg)
    inp = workloads.indexer_inputs(wl)
    d = KP.to_dev(inp)
    p = KP.params_of(wl)
    kp, lay = K.kpool_build(d["k"], d["gate"], d["ape"], d["cu_seqlens"], p)
    idx = K.dsa_index(d["q_idx"], d["w"], kp, lay, wl.topk, p, W=wl.W)
    assert K.check_status(lay.status) == 0
    rows_before = idx.clone()

    q1, kv1 = workloads.layer_attention_inputs(wl, 1)
    q0, kv0 = workloads.layer_attention_inputs(wl, 0)
    assert torch.equal(kv0, inp.kv_lat) and not torch.equal(kv1, kv0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = K.sparse_mla_fwd(q1.cuda(), kv1.cuda(), idx, wl.scale, status=status)
    assert K.check_status(status) == 0
    assert torch.equal(idx, rows_before)          # the shared rows are only read

    rows = KP.sample_rows(wl, n_uniform=64, seed=11)
    q_rows = q1[rows].float().numpy()
    o_ref, l_ref = O.sparse_attention(q_rows, kv1.float().numpy(), idx.cpu().numpy()[rows], wl.scale, rows)
    mx, mean, lse_err = KP.attention_check(out[rows].float().cpu().numpy(), lse[rows].cpu().numpy(), o_ref, l_ref)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and lse_err <= KP.LSE_ABS, (mx, mean, lse_err)
