"""GPU-vs-oracle parity of every step of the KPool-DSA forward, through the C
ABI, on the seeded workloads and edge cases."""
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


def _check_layout(res, lay_o, wl):
    assert res["status"] == 0
    np.testing.assert_array_equal(res["cu_pools"], lay_o["cu_pools"])
    np.testing.assert_array_equal(res["pool_tok_start"][:lay_o["n_pools"]], lay_o["pool_tok_start"])
    np.testing.assert_array_equal(res["tok_doc"], lay_o["tok_doc"])


def _check_kpool(res, inp, lay_o):
    kp_o = O.pool_keys(inp.k.float().numpy(), inp.gate, inp.ape, lay_o)
    P = lay_o["n_pools"]
    kp_g = res["kpool"][:P]
    kf = np.abs(inp.k.float().numpy())
    mag = np.stack([kf[lay_o["pool_tok_start"] + j] for j in range(4)]).max(axis=0) if P else np.zeros((0, 1))
    err = np.abs(kp_g.astype(np.float64) - kp_o.astype(np.float64))
    assert np.all(err <= KP.KPOOL_RTOL * mag + 1e-30), float((err / np.maximum(mag, 1e-30)).max())
    assert np.all(res["kpool"][P:] == 0)
    return kp_o


def _full_parity(idx, rows=None, attn_rows=None):
    return _parity_of(workloads.workload(idx), rows, attn_rows)


def _parity_of(wl, rows=None, attn_rows=None, attention=True):
    inp = workloads.indexer_inputs(wl)
    dev = KP.to_dev(inp)
    res = KP.run_indexer(wl, dev)
    lay_o = O.pool_layout(wl.cu_seqlens)
    _check_layout(res, lay_o, wl)
    kp_o = _check_kpool(res, inp, lay_o)

    # FP8 keys: the oracle's quantiser on the GPU's pooled keys is bit-exact,
    # and so is the oracle's own end-to-end chain
    k8_o, sk_o = O.quantize_keys(res["kpool"])
    np.testing.assert_array_equal(res["k8"], k8_o)
    np.testing.assert_array_equal(res["s_k"].view(np.uint32), sk_o.view(np.uint32))
    k8_e2e, _ = O.quantize_keys(kp_o)
    assert np.array_equal(res["k8"][:lay_o["n_pools"]], k8_e2e)

    rows = np.arange(wl.T) if rows is None else np.asarray(rows, np.int64)
    chk = KP.check_index_rows(wl, res, inp, lay_o, rows)
    st = chk["stats"]
    KP.record(f"[{wl.name}] index rows: {st['rows']} checked ({'all' if len(rows) == wl.T else 'sample'} of "
              f"{wl.T}), {st['exact']} bit-exact, {st['boundary_rows']} boundary rows ({st['boundary_pools']} "
              f"pools), hard {st['hard']}; q8 rows off {chk['q8_bad']}, ws rows off {chk['ws_bad']}; "
              f"score rel err {chk['worst']:.2e}, worst error / its per-pool bound {chk['worst_bound']:.2e}")
    assert chk["q8_bad"] == 0 and chk["ws_bad"] == 0
    assert chk["worst"] <= 1e-5, chk["worst"]
    assert chk["worst_bound"] <= 1.0, chk["worst_bound"]
    assert st["hard"] == 0, st["hard_rows"][:10]
    if not attention:
        return wl, res

    # attention, evaluated by the oracle on the GPU's own index rows
    attn_rows = rows if attn_rows is None else np.asarray(attn_rows, np.int64)
    ql = workloads.q_lat(wl)
    out, lse = K.sparse_mla_fwd(ql.cuda(), dev["kv_lat"], res["indices_dev"], wl.scale)
    torch.cuda.synchronize()
    out_g = out[torch.from_numpy(attn_rows).cuda()].float().cpu().numpy()
    lse_g = lse[torch.from_numpy(attn_rows).cuda()].cpu().numpy()
    out_o, lse_o = O.sparse_attention(ql[torch.from_numpy(attn_rows)].float().numpy(), inp.kv_lat.float().numpy(),
                                      res["indices"][attn_rows], wl.scale, attn_rows)
    mx, mean, le = KP.attention_check(out_g, lse_g, out_o, lse_o)
    KP.record(f"[{wl.name}] attention ({len(attn_rows)} rows): max abs {mx:.3e}, mean abs {mean:.3e}, lse {le:.3e}")
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS
    return wl, res


@pytest.mark.parametrize("hi", [4, 8, 16, 64])
def test_tensor_core_scoring_head_counts(hi):
    """The tcgen05 scoring kernel at every indexer head count it takes (d_i = 128): 256 / H_i queries per
    work item, 1 to 8 queries per 32-column chunk; two documents, both long enough to have scored rows."""
    wl = workloads.custom(f"heads{hi}", 20 + hi, (1637, 1130), n_idx_heads=hi, d_idx=128, topk=64, n_heads=4)
    _parity_of(wl, attention=False)


def test_parity_tiny_workload():
    _full_parity(0)


def test_parity_single_doc_4096_cutover():
    """Every index row; attention on the seeded sample."""
    wl = workloads.workload(1)
    _full_parity(1, rows=None, attn_rows=KP.sample_rows(wl, n_uniform=400, seed=1))


def test_parity_packed_8192_six_docs():
    """Every index row; attention on the seeded sample."""
    wl = workloads.workload(2)
    _full_parity(2, rows=None, attn_rows=KP.sample_rows(wl, n_uniform=400, seed=2))


def test_parity_headline_32768():
    """Every index row; attention on the seeded sample."""
    wl = workloads.workload(3)
    _full_parity(3, rows=None, attn_rows=KP.sample_rows(wl, n_uniform=256, seed=3))


@pytest.mark.slow
def test_parity_long_131072():
    """Several thousand index rows (the seeded sample, the last 64 rows of every document and 4096 uniform
    rows); attention on the seeded sample."""
    wl = workloads.workload(4)
    sample = KP.sample_rows(wl, n_uniform=192, seed=4)
    extra = [np.arange(max(s, e - 64), e) for s, e in zip(wl.cu_seqlens[:-1], wl.cu_seqlens[1:])]
    uni = np.random.default_rng(44).integers(0, wl.T, 4096)
    rows = np.unique(np.concatenate([sample, uni, *extra]))
    _full_parity(4, rows=rows, attn_rows=sample)


# ----------------------------------------------------------------- stage isolation

def _scores_buffer(wl, lay_o, topk, S_rows, rows):
    """Oracle scores placed in the workspace's compact triangle layout."""
    cu = wl.cu_seqlens
    pair_base = np.zeros(len(cu), np.int64)
    for d in range(len(cu) - 1):
        L = int(cu[d + 1] - cu[d])
        a, b = divmod(L, 4)
        pair_base[d + 1] = pair_base[d] + 2 * a * (a - 1) + a * (b + 1)
    buf = np.zeros(max(int(pair_base[-1]), 1), np.float32)
    for n, i in enumerate(rows):
        d, r, n_i, _ = O.query_geometry(lay_o, int(i))
        a, b = divmod(r, 4)
        s = int(pair_base[d]) + 2 * a * (a - 1) + a * (b + 1)
        buf[s:s + n_i] = S_rows[n]
    return buf, pair_base


def _stage_select(wl, S_rows, topk):
    lay_o = O.pool_layout(wl.cu_seqlens)
    rows = np.arange(wl.T)
    buf, pb = _scores_buffer(wl, lay_o, topk, S_rows, rows)
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    p = KP.params_of(wl)
    k = torch.zeros((wl.T, wl.d_idx), dtype=torch.bfloat16, device="cuda")
    gate = torch.zeros((wl.T, wl.d_idx), dtype=torch.float32, device="cuda")
    ape = torch.zeros((4, wl.d_idx), dtype=torch.float32, device="cuda")
    _, lay = K.kpool_build(k, gate, ape, cu, p)
    W = K.row_width(topk)
    idx = K.stage_select(torch.from_numpy(buf).cuda(), torch.from_numpy(pb).cuda(), lay, topk, W=W)
    got = idx.cpu().numpy()
    want = np.stack([O.index_row(lay_o, i, O.select_pools(S_rows[i], topk), W) for i in range(wl.T)])
    return got, want


def test_stage_select_bit_exact_on_oracle_scores():
    wl = workloads.workload(1)
    inp = workloads.indexer_inputs(wl)
    r = O.indexer(inp.q_idx.float().numpy(), inp.k.float().numpy(), inp.gate, inp.ape, inp.w, wl.cu_seqlens,
                  wl.topk, wl.W, with_scores=True)
    got, want = _stage_select(wl, r["scores"], wl.topk)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("kind", ["few_values", "zeros_signed", "all_equal", "negative", "nan_and_inf"])
def test_stage_select_ties(kind):
    wl = workloads.custom("ties", 7, (1500, 1037, 3), topk=64)
    lay_o = O.pool_layout(wl.cu_seqlens)
    rng = np.random.default_rng({"few_values": 1, "zeros_signed": 2, "all_equal": 3, "negative": 4,
                                 "nan_and_inf": 5}[kind])
    S = []
    for i in range(wl.T):
        n = O.query_geometry(lay_o, i)[2]
        if kind == "few_values":
            s = rng.integers(-2, 3, n).astype(np.float32) * np.float32(0.25)
        elif kind == "zeros_signed":
            s = np.where(rng.random(n) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
            s[rng.random(n) < 0.05] = 1.0
        elif kind == "all_equal":
            s = np.full(n, 3.5, np.float32)
        elif kind == "nan_and_inf":                  # NaN ranks lowest: long rows keep some NaN pools
            s = rng.standard_normal(n).astype(np.float32)
            s[rng.random(n) < 0.85] = np.nan
            s[rng.random(n) < 0.02] = np.inf
            s[rng.random(n) < 0.05] = -np.inf          # below every number but above NaN
        else:
            s = -np.abs(rng.standard_normal(n)).astype(np.float32)
        S.append(s)
    got, want = _stage_select(wl, S, wl.topk)
    np.testing.assert_array_equal(got, want)


def _long_row_select(lens, kind, min_n, seed):
    """Stage select over one compact score triangle of documents `lens` (standard normal scores), the
    rows of more than min_n pools overwritten with the pattern `kind`; compares those rows and 200
    others with the oracle."""
    wl = workloads.custom("long_rows", seed, lens, topk=512)
    lay_o = O.pool_layout(wl.cu_seqlens)
    cu = wl.cu_seqlens
    pair_base = np.zeros(len(cu), np.int64)
    for d in range(len(cu) - 1):
        a, b = divmod(int(cu[d + 1] - cu[d]), 4)
        pair_base[d + 1] = pair_base[d] + 2 * a * (a - 1) + a * (b + 1)
    rng = np.random.default_rng(seed)
    buf = rng.standard_normal(int(pair_base[-1]), dtype=np.float32)

    def start(i):
        d, r, n_i, _ = O.query_geometry(lay_o, i)
        a, b = divmod(r, 4)
        return int(pair_base[d]) + 2 * a * (a - 1) + a * (b + 1), n_i

    long_rows = [i for i in range(wl.T) if O.query_geometry(lay_o, i)[2] > min_n]
    assert len(long_rows) > 200
    for i in long_rows:
        s0, n = start(i)
        if kind == "ties_across_chunks":             # 100 pools above the tie, 700 tied, 300 of them in chunk 0
            x = -np.abs(rng.standard_normal(n)).astype(np.float32)
            pick = rng.permutation(8192)[:300]
            x[pick] = 1.0
            late = 8192 + rng.permutation(n - 8192)[:500]
            x[late[:400]] = 1.0
            x[late[400:]] = 2.0
        elif kind == "increasing":                   # every kept pool in the last chunk
            x = np.arange(n, dtype=np.float32) * np.float32(0.001)
        elif kind == "all_equal":
            x = np.full(n, -3.5, np.float32)
        else:
            continue
        buf[s0:s0 + n] = x
    check = long_rows + sorted(rng.choice(np.setdiff1d(np.arange(wl.T), long_rows), 200, replace=False).tolist())
    cu_d = torch.from_numpy(cu).cuda()
    p = KP.params_of(wl)
    k = torch.zeros((wl.T, wl.d_idx), dtype=torch.bfloat16, device="cuda")
    gate = torch.zeros((wl.T, wl.d_idx), dtype=torch.float32, device="cuda")
    ape = torch.zeros((4, wl.d_idx), dtype=torch.float32, device="cuda")
    _, lay = K.kpool_build(k, gate, ape, cu_d, p)
    W = K.row_width(wl.topk)
    got = K.stage_select(torch.from_numpy(buf).cuda(), torch.from_numpy(pair_base).cuda(), lay, wl.topk,
                         W=W).cpu().numpy()
    for i in check:
        s0, n = start(i)
        want = O.index_row(lay_o, i, O.select_pools(buf[s0:s0 + n], wl.topk), W)
        np.testing.assert_array_equal(got[i], want, err_msg=f"row {i} (n = {n})")


@pytest.mark.parametrize("kind", ["normal", "ties_across_chunks", "increasing", "all_equal"])
def test_stage_select_rows_longer_than_8192_pools(kind):
    """Rows of 8193 to 16392 candidate pools (documents of 32769 to 65571 tokens) are copied whole into
    shared memory and ranked in chunks of 8192 pools.  The patterns put the kept pools in the first
    chunk only, in the second only, or split the tie at the threshold across both."""
    _long_row_select((4 * (8192 + 700) + 2, 1001), kind, 8192, 81)


@pytest.mark.slow
@pytest.mark.parametrize("kind", ["normal", "ties_across_chunks"])
def test_stage_select_rows_longer_than_16392_pools(kind):
    """Rows of more than 16392 candidate pools (documents of more than 65571 tokens) are read from
    global memory on every pass, with the keys of the chosen level-1 bin in a shared candidate list."""
    _long_row_select((4 * (16392 + 60) + 3,), kind, 16392, 82)


# ----------------------------------------------------------------- edge cases

@pytest.mark.parametrize("lens", [(1,), (3,), (4,), (5, 0, 7), (2, 1, 3, 2), (130, 0, 0, 257), (4096 + 3,)])
def test_edge_layouts_and_rows(lens):
    wl = workloads.custom("edge", 11, lens, n_idx_heads=4, d_idx=64, topk=8, n_heads=4)
    inp = workloads.indexer_inputs(wl)
    dev = KP.to_dev(inp)
    res = KP.run_indexer(wl, dev)
    lay_o = O.pool_layout(wl.cu_seqlens)
    _check_layout(res, lay_o, wl)
    _check_kpool(res, inp, lay_o)
    rows = np.arange(wl.T)
    r = O.indexer(inp.q_idx.float().numpy(), inp.k.float().numpy(), inp.gate, inp.ape, inp.w, wl.cu_seqlens,
                  wl.topk, wl.W, with_scores=True)
    stats = KP.compare_rows(res["indices"], lay_o, rows, r["scores"], wl.topk, res["W"])
    assert stats["hard"] == 0


def test_invalid_cu_seqlens_sets_status_and_empty_rows():
    wl = workloads.custom("bad", 3, (40, 24), n_idx_heads=4, d_idx=64, topk=8, n_heads=4)
    inp = workloads.indexer_inputs(wl)
    dev = KP.to_dev(inp)
    dev["cu_seqlens"] = torch.tensor([0, 50, 40], dtype=torch.int32, device="cuda")   # decreasing, wrong end
    res = KP.run_indexer(wl, dev)
    assert res["status"] == K.CODES["KPOOL_ERR_LAYOUT"]
    assert res["cu_pools"][-1] == -1
    assert np.all(res["indices"] == -1)
    assert np.all(res["kpool"] == 0)


def test_sparse_mla_index_range_and_empty_rows():
    wl = workloads.custom("mla_edge", 5, (300,), n_heads=64)
    inp = workloads.indexer_inputs(wl)
    ql = workloads.q_lat(wl)
    T, W = wl.T, 256
    rng = np.random.default_rng(0)
    idx = np.full((T, W), -1, np.int32)
    for i in range(T):
        n = min(i + 1, int(rng.integers(0, 200)))
        idx[i, :n] = np.sort(rng.choice(T, n, replace=False))
    idx[5, 3] = T + 7            # out of range: skipped and flagged
    idx[6, 0] = -5
    idx[7, :] = -1               # empty row
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = K.sparse_mla_fwd(ql.cuda(), inp.kv_lat.cuda(), torch.from_numpy(idx).cuda(), wl.scale, status=st)
    assert K.check_status(st) == K.CODES["KPOOL_ERR_INDEX_RANGE"]
    ref_idx = idx.copy()
    ref_idx[(ref_idx < -1) | (ref_idx >= T)] = -1
    rows = np.arange(T)
    out_o, lse_o = O.sparse_attention(ql.float().numpy(), inp.kv_lat.float().numpy(), ref_idx, wl.scale, rows)
    out_g, lse_g = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(out_g[7] == 0) and np.all(np.isneginf(lse_g[7]))
    mx, mean, le = KP.attention_check(out_g, lse_g, out_o, lse_o)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS


def test_sparse_mla_holes_and_late_rescales():
    """Rows mixing fully valid 64-slot blocks (the softmax's fast path) with blocks that have invalid
    slots in the middle of the row (the masked path), and rows where a slot of a late full block
    beats the running max by far, so that O^T is rescaled after several blocks have been added."""
    wl = workloads.custom("mla_holes", 9, (700,), n_heads=64)
    inp = workloads.indexer_inputs(wl)
    ql = workloads.q_lat(wl)
    kv = inp.kv_lat.float().clone()
    T, W = wl.T, 640
    rng = np.random.default_rng(3)
    idx = np.full((T, W), -1, np.int32)
    for i in range(T):
        n = min(i + 1, W)
        row = np.sort(rng.choice(i + 1, n, replace=False)).astype(np.int32)
        if i % 3 == 1:                           # holes: about a fifth of the entries invalid
            row[rng.random(n) < 0.2] = -1
        idx[i, :n] = row
    # late large logits: for every fourth long row, one slot of its sixth block gets the direction
    # of one head's query, so that this head's logit there (~12) beats its running max by far while
    # the key's entries stay of the usual size
    big = []
    for i in range(400, T, 4):
        j = 5 * 64 + 7
        if idx[i, j] >= 0 and int(idx[i, j]) not in big:
            r = int(idx[i, j])
            qh = ql[i, i % 64].float()
            kv[r] = qh / qh.norm() * 12.0 / wl.scale / qh.norm()
            big.append(r)
    kv_b = kv.to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = K.sparse_mla_fwd(ql.cuda(), kv_b.cuda(), torch.from_numpy(idx).cuda(), wl.scale, status=st)
    assert K.check_status(st) == 0
    rows = np.arange(T)
    out_o, lse_o = O.sparse_attention(ql.float().numpy(), kv_b.float().numpy(), idx, wl.scale, rows)
    mx, mean, le = KP.attention_check(out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS, (mx, mean, le)
    assert len(big) > 10


def test_sparse_mla_rescales_from_several_warps_and_last_blocks():
    """Running-max moves that O^T already depends on, raised in one block by heads of different softmax
    warps at once, again for a head in a later block, and in a row's last block (whose rescale must be
    done before the last PV, while the softmax warps wait for the epilogue)."""
    wl = workloads.custom("mla_rescales", 12, (700,), n_heads=64)
    inp = workloads.indexer_inputs(wl)
    ql = workloads.q_lat(wl)
    kv = inp.kv_lat.float().clone()
    T, W = wl.T, 640
    rng = np.random.default_rng(5)
    idx = np.full((T, W), -1, np.int32)
    for i in range(T):
        n = min(i + 1, W)
        idx[i, :n] = np.sort(rng.choice(i + 1, n, replace=False)).astype(np.int32)
    used = set()

    def aim(i, h, j, logit):
        r = int(idx[i, j])
        if r < 0 or r in used:
            return False
        qh = ql[i, h].float()
        kv[r] = qh / qh.norm() * logit / wl.scale / qh.norm()
        used.add(r)
        return True

    hits = 0
    for i in range(200, T, 3):
        n = min(i + 1, W)
        nb = (n + 63) // 64
        b1 = 1 + i % max(1, nb - 2)
        for k, h in enumerate((i % 64, (i + 21) % 64, (i + 42) % 64)):      # three warps, one block
            hits += aim(i, h, b1 * 64 + 3 + 5 * k, 12.0 + 3.0 * k)
        if b1 + 1 < nb - 1:                                                   # the same head again later
            hits += aim(i, i % 64, (b1 + 1) * 64 + 9, 26.0)
        hits += aim(i, (i + 7) % 64, n - 1, 20.0)                             # the row's last slot
    kv_b = kv.to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = K.sparse_mla_fwd(ql.cuda(), kv_b.cuda(), torch.from_numpy(idx).cuda(), wl.scale, status=st)
    assert K.check_status(st) == 0
    rows = np.arange(T)
    out_o, lse_o = O.sparse_attention(ql.float().numpy(), kv_b.float().numpy(), idx, wl.scale, rows)
    mx, mean, le = KP.attention_check(out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS, (mx, mean, le)
    assert hits > 200


@pytest.mark.parametrize("H, W", [(48, 130), (16, 256), (64, 2176)])
def test_one_query_per_cta_launches(H, W):
    """Launches with at most one query per CTA (as a decode step makes) take the kernel's one-query instance,
    whose row scanner reads the row with 16-byte loads when W is a multiple of 4 and 4-byte loads otherwise."""
    T, n_rows = 3000, 40
    rng = np.random.default_rng(H + W)
    q = torch.from_numpy(rng.standard_normal((n_rows, H, 512), dtype=np.float32)).to(torch.bfloat16)
    kv = torch.from_numpy(rng.standard_normal((T, 512), dtype=np.float32)).to(torch.bfloat16)
    idx = np.full((n_rows, W), -1, np.int32)
    for i in range(n_rows):
        n = int(rng.integers(0, W + 1))
        idx[i, :n] = rng.choice(T, n, replace=False)
    idx[3, :] = -1                               # an empty row
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = K.sparse_mla_fwd_rows(q.cuda(), kv.cuda(), torch.from_numpy(idx).cuda(), 1.0 / np.sqrt(512),
                                     status=st)
    assert K.check_status(st) == 0
    out_o, lse_o = O.sparse_attention(q.float().numpy(), kv.float().numpy(), idx, 1.0 / np.sqrt(512),
                                      np.arange(n_rows))
    mx, mean, le = KP.attention_check(out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS, (mx, mean, le)


@pytest.mark.parametrize("hi, di", [(32, 128), (4, 64)])
def test_indexer_queries_only_8_byte_aligned(hi, di):
    """q_idx is documented as 8-byte aligned: a view starting 8 bytes into an allocation (so not 16-byte
    aligned) gives the same codes, head weights and index rows as an aligned copy."""
    wl = workloads.custom("qalign", 17, (700, 333), n_idx_heads=hi, d_idx=di, topk=32, n_heads=4)
    inp = workloads.indexer_inputs(wl)
    dev = KP.to_dev(inp)
    ref = KP.run_indexer(wl, dev)
    n = dev["q_idx"].numel()
    buf = torch.empty(n + 4, dtype=torch.bfloat16, device="cuda")
    buf[4:] = dev["q_idx"].reshape(-1)
    shifted = buf[4:].view(dev["q_idx"].shape)
    assert shifted.data_ptr() % 16 == 8
    dev2 = dict(dev, q_idx=shifted)
    got = KP.run_indexer(wl, dev2)
    assert got["status"] == 0
    np.testing.assert_array_equal(got["q8"], ref["q8"])
    np.testing.assert_array_equal(got["ws"].view(np.uint32), ref["ws"].view(np.uint32))
    np.testing.assert_array_equal(got["indices"], ref["indices"])


def test_small_head_counts_attention():
    for H in (1, 4, 20, 48):
        wl = workloads.custom("heads", 9, (97,), n_heads=H)
        inp = workloads.indexer_inputs(wl)
        ql = workloads.q_lat(wl)
        T = wl.T
        idx = np.full((T, 128), -1, np.int32)
        for i in range(T):
            idx[i, :i + 1] = np.arange(i + 1)
        out, lse = K.sparse_mla_fwd(ql.cuda(), inp.kv_lat.cuda(), torch.from_numpy(idx).cuda(), wl.scale)
        out_o, lse_o = O.sparse_attention(ql.float().numpy(), inp.kv_lat.float().numpy(), idx, wl.scale,
                                          np.arange(T))
        mx, mean, le = KP.attention_check(out.float().cpu().numpy(), lse.cpu().numpy(), out_o, lse_o)
        assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS, (H, mx, mean, le)


def test_dense_equivalence_below_cutover_on_gpu():
    """topk >= every document's pool count: GPU rows are the causal prefix of
    the document and GPU attention equals dense causal attention."""
    wl = workloads.custom("dense", 13, (700, 321), n_idx_heads=8, d_idx=128, topk=256, n_heads=16)
    inp = workloads.indexer_inputs(wl)
    dev = KP.to_dev(inp)
    res = KP.run_indexer(wl, dev)
    cu = wl.cu_seqlens
    for i in range(wl.T):
        d = 0 if i < cu[1] else 1
        row = res["indices"][i]
        assert row[row >= 0].tolist() == list(range(int(cu[d]), i + 1))
    ql = workloads.q_lat(wl)
    out, lse = K.sparse_mla_fwd(ql.cuda(), dev["kv_lat"], res["indices_dev"], wl.scale)
    q = ql.float().double()
    kv = inp.kv_lat.float().double()
    ref = torch.zeros_like(q)
    for d in range(2):
        s, e = int(cu[d]), int(cu[d + 1])
        qq = q[s:e].permute(1, 0, 2)
        kk = kv[s:e][None].expand(wl.n_heads, -1, -1)
        ref[s:e] = torch.nn.functional.scaled_dot_product_attention(qq, kk, kk, is_causal=True,
                                                                    scale=wl.scale).permute(1, 0, 2)
    err = (out.float().cpu().double() - ref).abs()
    assert err.max() <= KP.OUT_MAX_ABS and err.mean() <= KP.OUT_MEAN_ABS


def test_determinism_and_document_isolation():
    wl = workloads.workload(2)
    inp = workloads.indexer_inputs(wl)
    dev = KP.to_dev(inp)
    a = KP.run_indexer(wl, dev)
    b = KP.run_indexer(wl, dev)
    np.testing.assert_array_equal(a["indices"], b["indices"])
    # perturb the last document: every other document's rows are unchanged
    s = int(wl.cu_seqlens[-2])
    dev2 = dict(dev)
    dev2["q_idx"] = dev["q_idx"].clone()
    dev2["q_idx"][s:] = -dev2["q_idx"][s:]
    dev2["k"] = dev["k"].clone()
    dev2["k"][s:] *= 2
    c = KP.run_indexer(wl, dev2)
    np.testing.assert_array_equal(a["indices"][:s], c["indices"][:s])
    ql = workloads.q_lat(wl).cuda()
    o1, l1 = K.sparse_mla_fwd(ql, dev["kv_lat"], a["indices_dev"], wl.scale)
    kv2 = dev["kv_lat"].clone()
    kv2[s:] = 1.0
    o2, l2 = K.sparse_mla_fwd(ql, kv2, c["indices_dev"], wl.scale)
    assert torch.equal(o1[:s], o2[:s]) and torch.equal(l1[:s], l2[:s])


def test_sparse_mla_runs_of_empty_rows():
    # Each CTA walks rows i, i + n_sm, ...; whole bands of empty rows give every CTA
    # consecutive empty queries, between and after non-empty ones.
    wl = workloads.custom("mla_empty_runs", 11, (1900,), n_heads=64)
    inp = workloads.indexer_inputs(wl)
    ql = workloads.q_lat(wl)
    T, W = wl.T, 256
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(1)
    idx = np.full((T, W), -1, np.int32)
    for i in range(T):
        band = (i // n_sm) % 4
        if band in (1, 2):
            continue                              # two consecutive empty queries per CTA
        n = int(rng.integers(1, W + 1))
        idx[i, :n] = np.sort(rng.choice(T, n, replace=False))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = K.sparse_mla_fwd(ql.cuda(), inp.kv_lat.cuda(), torch.from_numpy(idx).cuda(), wl.scale, status=st)
    assert K.check_status(st) == 0
    rows = np.arange(T)
    out_o, lse_o = O.sparse_attention(ql.float().numpy(), inp.kv_lat.float().numpy(), idx, wl.scale, rows)
    out_g, lse_g = out.float().cpu().numpy(), lse.cpu().numpy()
    empty = np.all(idx < 0, axis=1)
    assert np.all(out_g[empty] == 0) and np.all(np.isneginf(lse_g[empty]))
    mx, mean, le = KP.attention_check(out_g[~empty], lse_g[~empty], out_o[~empty], lse_o[~empty])
    assert mx <= KP.OUT_MAX_ABS and mean <= KP.OUT_MEAN_ABS and le <= KP.LSE_ABS
