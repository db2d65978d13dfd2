"""Absorbed-MLA projections on the GPU, through the C ABI, against the oracle.

Tolerance, derived from the arithmetic: the kernels sum exact bf16 products
in fp32 (at most 512 terms, so the sum is off by at most 512 * 2^-24 of the
sum of |products|) and round the result to bf16 (half an ulp: at most 2^-8
of |value|).  Each element must satisfy
    |gpu - oracle| <= 2^-8 * |oracle| + 2^-14 * sum_k |a_k b_k|.
"""
import numpy as np
import pytest
import torch

from oracle import absorb_oracle as A
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


def _check(gpu, ref, absref):
    g = gpu.float().cpu().numpy().astype(np.float64)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * absref
    bad = np.abs(g - ref) > bound
    assert not bad.any(), (int(bad.sum()), float(np.abs(g - ref).max()))


def _absorb_ref(q_nope, w, dn, dv):
    qn = q_nope.float().numpy()
    wn = w.float().numpy()
    return A.absorb_q(qn, wn, dn, dv), A.absorb_q(np.abs(qn), np.abs(wn), dn, dv)


def _vproj_ref(o_lat, w, dn, dv):
    on = o_lat.float().numpy()
    wn = w.float().numpy()
    return A.v_proj(on, wn, dn, dv), A.v_proj(np.abs(on), np.abs(wn), dn, dv)


# T spans several 128-token tiles with a ragged tail, a single partial tile, one token
@pytest.mark.parametrize("T,H,dn,dv", [(300, 64, 128, 128), (1000, 5, 64, 64), (77, 3, 128, 64), (1, 2, 64, 128),
                                       (640, 17, 128, 128)])
def test_absorb_and_v_proj_parity(T, H, dn, dv):
    wl = workloads.custom("proj", 21, (T,), n_heads=H)
    q_nope, w = workloads.proj_inputs(wl, dn, dv)
    o_lat = workloads.o_lat_input(wl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_lat = K.mla_absorb_q(q_nope.cuda(), w.cuda(), dn, dv, status=st)
    o_v = K.mla_v_proj(o_lat.cuda(), w.cuda(), dn, dv, status=st)
    assert K.check_status(st) == 0
    _check(q_lat, *_absorb_ref(q_nope, w, dn, dv))
    _check(o_v, *_vproj_ref(o_lat, w, dn, dv))


def test_output_rows_past_the_tensor_are_untouched():
    # the last tile is partial: nothing past T rows may be written
    T, H, dn, dv = 200, 4, 128, 128
    wl = workloads.custom("proj_tail", 22, (T,), n_heads=H)
    q_nope, w = workloads.proj_inputs(wl, dn, dv)
    buf = torch.full((T + 60, H, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    K.mla_absorb_q(q_nope.cuda(), w.cuda(), dn, dv, out=buf[:T])
    torch.cuda.synchronize()
    assert torch.all(buf[T:] == 7.0)
    vbuf = torch.full((T + 60, H, dv), 7.0, dtype=torch.bfloat16, device="cuda")
    K.mla_v_proj(workloads.o_lat_input(wl).cuda(), w.cuda(), dn, dv, out=vbuf[:T])
    torch.cuda.synchronize()
    assert torch.all(vbuf[T:] == 7.0)


def test_full_size_sampled_rows():
    # the benchmark's shape: 32768 tokens, 64 heads, d_nope = d_v = 128; sampled token rows vs the oracle
    wl = workloads.workload(3)
    dn = dv = 128
    q_nope, w = workloads.proj_inputs(wl, dn, dv)
    rows = np.unique(np.concatenate([[0, 127, 128, wl.T - 1], np.linspace(0, wl.T - 1, 40).astype(np.int64)]))
    q_lat = K.mla_absorb_q(q_nope.cuda(), w.cuda(), dn, dv)
    _check(q_lat[torch.from_numpy(rows).cuda()], *_absorb_ref(q_nope[rows], w, dn, dv))
    del q_lat
    o_lat = workloads.o_lat_input(wl)
    o_v = K.mla_v_proj(o_lat.cuda(), w.cuda(), dn, dv)
    _check(o_v[torch.from_numpy(rows).cuda()], *_vproj_ref(o_lat[rows], w, dn, dv))


def test_absorbed_layer_chain_against_the_oracle():
    # q_nope -> absorb -> sparse latent attention on the layer's index rows -> V projection
    wl = workloads.workload(2)
    dn = dv = 128
    inp = workloads.indexer_inputs(wl)
    q_nope, w = workloads.proj_inputs(wl, dn, dv)
    d = KP.to_dev(inp)
    p = KP.params_of(wl)
    kp, lay = K.kpool_build(d["k"], d["gate"], d["ape"], d["cu_seqlens"], p)
    idx = K.dsa_index(d["q_idx"], d["w"], kp, lay, wl.topk, p, W=wl.W)
    q_lat = K.mla_absorb_q(q_nope.cuda(), w.cuda(), dn, dv, status=lay.status)
    out, lse = K.sparse_mla_fwd(q_lat, d["kv_lat"], idx, wl.scale, status=lay.status)
    o_v = K.mla_v_proj(out, w.cuda(), dn, dv, status=lay.status)
    assert K.check_status(lay.status) == 0

    rows = np.unique(np.linspace(0, wl.T - 1, 24).astype(np.int64))
    ql_ref = A.absorb_q(q_nope[rows].float().numpy(), w.float().numpy(), dn, dv)
    # attention in the oracle runs on the GPU's own q_lat and index rows (each step is pinned on its own)
    o_ref, l_ref = O.sparse_attention(q_lat[torch.from_numpy(rows).cuda()].float().cpu().numpy(),
                                      inp.kv_lat.float().numpy(), idx.cpu().numpy()[rows], wl.scale, rows)
    _check(q_lat[torch.from_numpy(rows).cuda()], ql_ref, A.absorb_q(np.abs(q_nope[rows].float().numpy()),
                                                                    np.abs(w.float().numpy()), dn, dv))
    mx, mean, lse_err = KP.attention_check(out[torch.from_numpy(rows).cuda()].float().cpu().numpy(),
                                           lse[torch.from_numpy(rows).cuda()].cpu().numpy(), o_ref, l_ref)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and lse_err <= KP.LSE_ABS
    # the V projection of the GPU's own attention output
    o_sel = out[torch.from_numpy(rows).cuda()].cpu()
    _check(o_v[torch.from_numpy(rows).cuda()], *_vproj_ref(o_sel, w, dn, dv))
