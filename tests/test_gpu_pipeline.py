"""Row-block attention and the pipelined host-buffer forward, through the C ABI.

Rows of the attention are independent, so a split into row blocks must give
exactly the unsplit results; the pipelined host forward must give exactly the
device path's index rows and outputs, and those agree with the oracle on
sampled rows."""
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


def _device_path(wl, d):
    p = KP.params_of(wl)
    kp, lay = K.kpool_build(d["k"], d["gate"], d["ape"], d["cu_seqlens"], p)
    idx = K.dsa_index(d["q_idx"], d["w"], kp, lay, wl.topk, p, W=wl.W)
    out, lse = K.sparse_mla_fwd(d["q_lat"], d["kv_lat"], idx, wl.scale, status=lay.status)
    assert K.check_status(lay.status) == 0
    return idx, out, lse


def test_row_blocks_give_the_unsplit_attention():
    wl = workloads.workload(2)                      # 6 packed documents, T = 8192
    inp = workloads.all_inputs(wl)
    d = KP.to_dev(inp)
    idx, out, lse = _device_path(wl, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_b = torch.full_like(out, float("nan"))
    lse_b = torch.full_like(lse, float("nan"))
    for r0, r1 in ((0, 1), (1, 2999), (2999, 3000), (3000, wl.T)):   # uneven blocks, single rows
        K.sparse_mla_fwd_rows(d["q_lat"][r0:r1], d["kv_lat"], idx[r0:r1], wl.scale, out=out_b[r0:r1],
                              lse=lse_b[r0:r1], status=status)
    assert K.check_status(status) == 0
    assert torch.equal(out_b, out)
    assert torch.equal(lse_b, lse)


# Block counts and workloads: config 0 (d_i = 64) runs the whole indexer before the blocks; the others index
# block by block, with block edges inside documents, blocks of a few query groups (64 blocks), one block, and
# a packed set of tiny documents (no scored rows) beside documents past the scoring cutover (topk 64 pools).
MIXED = ("mixed_docs", 37, (3, 5, 700, 9, 2051, 2060, 1), 64)


@pytest.mark.parametrize("cfg,n_chunks", [(0, 3), (2, 5), (2, 64), (1, 1), (1, 16), (MIXED, 7), (MIXED, 37)])
def test_host_pipeline_matches_the_device_path_and_the_oracle(cfg, n_chunks):
    if isinstance(cfg, tuple):
        name, seed, lens, topk = cfg
        wl = workloads.custom(name, seed, lens, topk=topk)
    else:
        wl = workloads.workload(cfg)
    inp = workloads.all_inputs(wl)
    d = KP.to_dev(inp)
    idx, out, lse = _device_path(wl, d)

    host = {"k": inp.k, "gate": torch.from_numpy(inp.gate), "ape": torch.from_numpy(inp.ape),
            "cu_seqlens": torch.from_numpy(inp.cu_seqlens), "q_idx": inp.q_idx, "w": torch.from_numpy(inp.w),
            "q_lat": inp.q_lat, "kv_lat": inp.kv_lat}
    host = {k: v.contiguous().pin_memory() for k, v in host.items()}
    host["out"] = torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory()
    host["lse"] = torch.empty(tuple(lse.shape), dtype=lse.dtype).pin_memory()
    dev = {k: torch.empty(tuple(v.shape), dtype=v.dtype, device="cuda") for k, v in host.items()}
    p = KP.params_of(wl)
    lay = K.PoolLayout(dev["cu_seqlens"], wl.T)
    dev["kpool"] = torch.empty((max(wl.T // 4, 1), wl.d_idx), dtype=torch.float32, device="cuda")
    dev["workspace"] = torch.empty(K.workspace_bytes(p, wl.T, lay.n_docs), dtype=torch.uint8, device="cuda")
    dev["indices"] = torch.empty((wl.T, wl.W), dtype=torch.int32, device="cuda")
    s_compute = K.forward_host(host, dev, lay, p, n_chunks=n_chunks)
    s_compute.synchronize()
    assert K.check_status(lay.status, s_compute) == 0
    assert torch.equal(dev["indices"], idx)
    assert torch.equal(host["out"], out.cpu())
    assert torch.equal(host["lse"], lse.cpu())

    # sampled rows against the oracle (index rows are the device path's, which the parity tests pin)
    rows = np.unique(np.linspace(0, wl.T - 1, 24).astype(np.int64))
    q_rows = inp.q_lat[rows].float().numpy()
    o_ref, l_ref = O.sparse_attention(q_rows, inp.kv_lat.float().numpy(), idx.cpu().numpy()[rows], wl.scale, rows)
    mx, mean, lse_err = KP.attention_check(host["out"][rows].float().numpy(), host["lse"][rows].numpy(), o_ref, l_ref)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and lse_err <= KP.LSE_ABS, (mx, mean, lse_err)
