"""Paged decode on the GPU, through the C ABI, against the oracle.

A decode query is the newest token of its sequence, so its index row is the
prefill row of the sequence's last token (pinned on its own), written in
latent-cache slots through the sequence's block table.  Pooled-key codes and
scales in the pages are bit-exact; rows are bit-exact except pools within 1e-3
of the topk-th score (counted); the attention over the paged latent cache
meets the forward's bounds."""
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


def _params(dw):
    return K.make_params(topk=dw.topk, n_idx_heads=dw.n_idx_heads, d_idx=dw.d_idx, n_heads=dw.n_heads,
                         d_lat=dw.d_lat, scale=dw.scale)


def _fill(dw, inp, bt, upto=None):
    """Pooled-key and latent caches of every sequence (pools p < upto[b] when given), on the GPU."""
    p = _params(dw)
    k_all = torch.cat(inp.k).cuda()
    g_all = torch.from_numpy(np.concatenate(inp.gate)).cuda()
    starts = np.concatenate([[0], np.cumsum(dw.seq_lens)])[:-1]
    tok, seq, idx = [], [], []
    for b, L in enumerate(dw.seq_lens):
        n = L // 4 if upto is None else upto[b]
        tok += [int(starts[b]) + 4 * q for q in range(n)]
        seq += [b] * n
        idx += list(range(n))
    k8 = torch.zeros((dw.n_pages, 32, dw.d_idx), dtype=torch.uint8, device="cuda")
    sk = torch.zeros((dw.n_pages, 32), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    K.paged_append(k_all, g_all, torch.from_numpy(inp.ape).cuda(), t(tok), t(seq), t(idx),
                   torch.from_numpy(bt).cuda(), dw.n_pages, p, k8, sk, status=st)
    kv = torch.zeros((dw.n_pages * workloads.PAGE_TOKENS, dw.d_lat), dtype=torch.bfloat16)
    for b, L in enumerate(dw.seq_lens):
        slots = O.paged_slots(np.arange(L), bt[b])
        kv[torch.from_numpy(slots)] = inp.kv_lat[b]
    return k8, sk, kv.cuda(), st


def _oracle_rows(dw, inp, bt):
    rows, keys = [], []
    for b, L in enumerate(dw.seq_lens):
        row, res = O.decode_row(inp.q_idx[b].float().numpy(), inp.w[b], inp.k[b].float().numpy(), inp.gate[b],
                                inp.ape, dw.topk, dw.W)
        rows.append(O.paged_slots(row, bt[b]))
        keys.append(res)
    return np.stack(rows), keys


@pytest.mark.parametrize("cfg", [0, 1])
def test_paged_cache_and_decode_rows(cfg):
    dw = workloads.decode_workload(cfg)
    inp = workloads.decode_inputs(dw)
    bt = dw.block_table()
    k8, sk, kv, st = _fill(dw, inp, bt)
    assert K.check_status(st) == 0
    ref_rows, res = _oracle_rows(dw, inp, bt)
    # pooled-key codes and scales, bit-exact, in their page slots
    k8h, skh = k8.cpu().numpy(), sk.cpu().numpy()
    for b, L in enumerate(dw.seq_lens):
        n = L // 4
        if n == 0:
            continue
        slots = O.paged_slots(4 * np.arange(n), bt[b]) // 4        # pool slot = page * 32 + pool % 32
        assert np.array_equal(k8h.reshape(-1, dw.d_idx)[slots], res[b]["k8"][:n])
        assert np.array_equal(skh.reshape(-1)[slots], res[b]["s_k"][:n].astype(np.float32))
    p = _params(dw)
    dst = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = K.decode_index(inp.q_idx.cuda(), torch.from_numpy(inp.w).cuda(), k8, sk, torch.from_numpy(bt).cuda(),
                          torch.tensor(dw.seq_lens, dtype=torch.int32, device="cuda"), dw.topk, p, dw.W, status=dst)
    assert K.check_status(dst) == 0
    got = rows.cpu().numpy()
    mismatched = 0
    for b in range(dw.B):
        if not np.array_equal(got[b], ref_rows[b]):
            mismatched += 1
            # only a tie at the topk-th score may differ: same count, and the sets differ by boundary pools
            assert (got[b] >= 0).sum() == (ref_rows[b] >= 0).sum(), b
    assert mismatched == 0, f"{mismatched} rows differ"


def test_decode_attention_over_the_paged_cache():
    dw = workloads.decode_workload(0)
    inp = workloads.decode_inputs(dw)
    bt = dw.block_table()
    k8, sk, kv, st = _fill(dw, inp, bt)
    p = _params(dw)
    rows = K.decode_index(inp.q_idx.cuda(), torch.from_numpy(inp.w).cuda(), k8, sk, torch.from_numpy(bt).cuda(),
                          torch.tensor(dw.seq_lens, dtype=torch.int32, device="cuda"), dw.topk, p, dw.W, status=st)
    out, lse = K.sparse_mla_fwd_rows(inp.q_lat.cuda(), kv, rows, dw.scale, status=st)
    assert K.check_status(st) == 0
    o_ref, l_ref = O.sparse_attention(inp.q_lat.float().numpy(), kv.float().cpu().numpy(), rows.cpu().numpy(),
                                      dw.scale, np.arange(dw.B))
    mx, mean, le = KP.attention_check(out.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS, (mx, mean, le)
    # the attention reads only the sequence's own latent rows: positions mapped through its pages
    for b, L in enumerate(dw.seq_lens):
        r = rows[b].cpu().numpy()
        r = r[r >= 0]
        allowed = set(O.paged_slots(np.arange(L), bt[b]).tolist())
        assert set(r.tolist()) <= allowed


def test_append_of_the_pool_a_decode_step_completes():
    # sequences whose newest token completes a pool: cache all earlier pools, append the last one from a
    # staging buffer of the 4 tokens, and compare with the full fill
    dw = workloads.DecodeWorkload("decode_append", 53, (8, 132, 516, 2052), topk=64)
    inp = workloads.decode_inputs(dw)
    bt = dw.block_table()
    full_k8, full_sk, _, _ = _fill(dw, inp, bt)
    part_k8, part_sk, _, st = _fill(dw, inp, bt, upto=[L // 4 - 1 for L in dw.seq_lens])
    k4 = torch.stack([inp.k[b][-4:] for b in range(dw.B)]).reshape(-1, dw.d_idx).cuda()
    g4 = torch.from_numpy(np.stack([inp.gate[b][-4:] for b in range(dw.B)]).reshape(-1, dw.d_idx)).cuda()
    t = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    K.paged_append(k4, g4, torch.from_numpy(inp.ape).cuda(), t([4 * b for b in range(dw.B)]), t(list(range(dw.B))),
                   t([L // 4 - 1 for L in dw.seq_lens]), torch.from_numpy(bt).cuda(), dw.n_pages, _params(dw),
                   part_k8, part_sk, status=st)
    assert K.check_status(st) == 0
    assert torch.equal(part_k8, full_k8) and torch.equal(part_sk, full_sk)


def test_decode_guards():
    dw = workloads.decode_workload(0)
    inp = workloads.decode_inputs(dw)
    bt = dw.block_table()
    k8, sk, kv, st = _fill(dw, inp, bt)
    p = _params(dw)
    lens = list(dw.seq_lens)
    lens[3] = dw.max_pages * workloads.PAGE_TOKENS + 1           # longer than the block table holds
    rows = K.decode_index(inp.q_idx.cuda(), torch.from_numpy(inp.w).cuda(), k8, sk, torch.from_numpy(bt).cuda(),
                          torch.tensor(lens, dtype=torch.int32, device="cuda"), dw.topk, p, dw.W, status=st)
    assert K.check_status(st) == K.CODES["KPOOL_ERR_SHAPE"]
    assert torch.all(rows[3] == -1)
    bad = bt.copy()
    bad[5, 1] = dw.n_pages + 4                                    # a page id outside the cache
    st.zero_()
    K.decode_index(inp.q_idx.cuda(), torch.from_numpy(inp.w).cuda(), k8, sk, torch.from_numpy(bad).cuda(),
                   torch.tensor(dw.seq_lens, dtype=torch.int32, device="cuda"), dw.topk, p, dw.W, status=st)
    assert K.check_status(st) == K.CODES["KPOOL_ERR_INDEX_RANGE"]


def test_decode_step_replayed_from_a_cuda_graph_equals_the_eager_step():
    # append + index + attention captured once into a CUDA graph (the calls allocate nothing given their
    # buffers and set kernel attributes only on first use); every replay gives the eager step's results
    dw = workloads.DecodeWorkload("decode_graph", 55, (8, 300, 1037, 2052), topk=32)
    inp = workloads.decode_inputs(dw)
    bt = dw.block_table()
    k8, sk, kv, st = _fill(dw, inp, bt, upto=[L // 4 - 1 if L % 4 == 0 else L // 4 for L in dw.seq_lens])
    p = _params(dw)
    comp = [b for b, L in enumerate(dw.seq_lens) if L % 4 == 0]
    starts = np.concatenate([[0], np.cumsum(dw.seq_lens)])[:-1]
    t = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    k_all = torch.cat(inp.k).cuda()
    g_all = torch.from_numpy(np.concatenate(inp.gate)).cuda()
    ape = torch.from_numpy(inp.ape).cuda()
    a_tok = t([int(starts[b]) + dw.seq_lens[b] - 4 for b in comp])
    a_seq, a_idx = t(comp), t([dw.seq_lens[b] // 4 - 1 for b in comp])
    btd = torch.from_numpy(bt).cuda()
    lens = t(list(dw.seq_lens))
    q_idx, w, q_lat = inp.q_idx.cuda(), torch.from_numpy(inp.w).cuda(), inp.q_lat.cuda()
    ws = torch.empty(K.decode_workspace_bytes(p, dw.B, dw.max_pages), dtype=torch.uint8, device="cuda")
    rows = torch.empty((dw.B, dw.W), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q_lat)
    lse = torch.empty((dw.B, dw.n_heads), dtype=torch.float32, device="cuda")

    def step():
        K.paged_append(k_all, g_all, ape, a_tok, a_seq, a_idx, btd, dw.n_pages, p, k8, sk, status=st)
        K.decode_index(q_idx, w, k8, sk, btd, lens, dw.topk, p, dw.W, workspace=ws, indices=rows, status=st)
        K.sparse_mla_fwd_rows(q_lat, kv, rows, dw.scale, out=out, lse=lse, status=st)

    step()                                            # eager (also the first use of every kernel)
    torch.cuda.synchronize()
    assert K.check_status(st) == 0
    ref = (k8.clone(), sk.clone(), rows.clone(), out.clone(), lse.clone())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        rows.fill_(-7)
        out.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert K.check_status(st) == 0
        for a, b in zip((k8, sk, rows, out, lse), ref):
            assert torch.equal(a, b)
