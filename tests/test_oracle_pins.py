"""Pins of the CPU oracle against facts fixed outside it: values worked out by
hand from the pages' rule, closed forms, library routines and brute force.
No GPU needed."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import torch

from oracle import kpool_oracle as O
from pooled_key_dsa_gb300 import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- layout

def test_layout_hand_example():
    g = _gold("tiny_rows.json")
    cu = np.concatenate([[0], np.cumsum(g["doc_lens"])])
    lay = O.pool_layout(cu)
    assert lay["cu_pools"].tolist() == g["layout"]["cu_pools"]
    assert lay["pool_tok_start"].tolist() == g["layout"]["pool_tok_start"]
    assert lay["tok_doc"].tolist() == g["layout"]["tok_doc"]


def test_layout_tiny_workload_pools():
    wl = workloads.workload(0)
    lay = O.pool_layout(wl.cu_seqlens)
    # 301 = 4*75 + 1 and 211 = 4*52 + 3: pools end mid-document
    assert lay["cu_pools"].tolist() == [0, 75, 127]
    assert lay["pool_tok_start"][75] == 301
    assert lay["pool_tok_start"][74] == 296


def test_layout_short_and_empty_docs():
    lay = O.pool_layout([0, 3, 3, 4, 9, 17])     # lengths 3, 0, 1, 5, 8
    assert lay["cu_pools"].tolist() == [0, 0, 0, 0, 1, 3]
    assert lay["pool_tok_start"].tolist() == [4, 9, 13]


# ----------------------------------------------------------------- pooling

def _pool_case(seed, T=16, d=8):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, d)).astype(np.float32)
    gate = rng.standard_normal((T, d)).astype(np.float32)
    ape = (0.1 * rng.standard_normal((4, d))).astype(np.float32)
    return k, gate, ape


def test_pool_constant_gate_is_ape_softmax_mean():
    k, _, ape = _pool_case(1)
    gate = np.full_like(k, 0.7)
    lay = O.pool_layout([0, 16])
    kp = O.pool_keys(k, gate, ape, lay)
    wts = scipy.special.softmax(ape.astype(np.float64), axis=0)       # library softmax
    for p in range(4):
        ref = (wts * k[4 * p:4 * p + 4].astype(np.float64)).sum(axis=0)
        np.testing.assert_allclose(kp[p], ref, rtol=1e-6, atol=1e-7)


def test_pool_constant_gate_and_ape_is_mean():
    k, _, _ = _pool_case(2)
    lay = O.pool_layout([0, 16])
    kp = O.pool_keys(k, np.full_like(k, -3.0), np.full((4, 8), 0.25, np.float32), lay)
    ref = k.astype(np.float64).reshape(4, 4, 8).mean(axis=1)
    np.testing.assert_allclose(kp, ref, rtol=1e-6, atol=1e-7)


def test_pool_dominant_gate_selects_token():
    k, gate, ape = _pool_case(3)
    lay = O.pool_layout([0, 16])
    gate = gate.copy()
    for p in range(4):
        gate[4 * p + (p % 4), :] = 200.0        # token j=p%4 dominates its pool
    kp = O.pool_keys(k, gate, ape, lay)
    for p in range(4):
        np.testing.assert_allclose(kp[p], k[4 * p + p % 4], rtol=0, atol=1e-30)


def test_pool_per_document_restart():
    # two documents: pools start at each document's first token
    k, gate, ape = _pool_case(4, T=13)
    lay = O.pool_layout([0, 5, 13])      # doc lens 5 and 8: pools at 0, 5, 9
    assert lay["pool_tok_start"].tolist() == [0, 5, 9]
    kp = O.pool_keys(k, gate, ape, lay)
    # each pool only depends on its own 4 tokens
    k2 = k.copy()
    k2[4] = 1e3         # token 4 is the partial tail of doc 0: in no pool
    np.testing.assert_array_equal(O.pool_keys(k2, gate, ape, lay), kp)


# ----------------------------------------------------------------- Hadamard

@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_hadamard_matches_sylvester_matrix(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((5, d)).astype(np.float32)
    Hm = scipy.linalg.hadamard(d).astype(np.float64) / math.sqrt(d)   # textbook Sylvester order
    np.testing.assert_allclose(O.hadamard_f32(x), x.astype(np.float64) @ Hm.T, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("d", [64, 128])
def test_hadamard_orthonormal_and_e0(d):
    I = np.eye(d, dtype=np.float32)
    Hm = O.hadamard_f32(I).astype(np.float64)          # rows: H e_j
    np.testing.assert_allclose(Hm @ Hm.T, np.eye(d), atol=1e-6)
    np.testing.assert_allclose(Hm[0], np.full(d, 1 / math.sqrt(d)), rtol=1e-7)
    x = np.random.default_rng(0).standard_normal((100, d)).astype(np.float32)
    n0 = np.linalg.norm(x.astype(np.float64), axis=1)
    n1 = np.linalg.norm(O.hadamard_f32(x).astype(np.float64), axis=1)
    np.testing.assert_allclose(n1, n0, rtol=1e-6)


def test_hadamard_is_fp32_butterfly_bitwise():
    """The fp32 stages are applied one at a time: a d=4 case worked out by
    hand, each intermediate exactly representable."""
    x = np.array([[1.0, 2.0, 4.0, 8.0]], np.float32)
    # h=1 pairs (0,1),(2,3): (3, -1, 12, -4)
    # h=2 pairs (0,2),(1,3): (3+12, -1-4, 3-12, -1+4) = (15, -5, -9, 3); times 1/2
    np.testing.assert_array_equal(O.hadamard_f32(x), np.array([[7.5, -2.5, -4.5, 1.5]], np.float32))


# ----------------------------------------------------------------- FP8

def test_e4m3_known_codes():
    dec = O.e4m3_decode_table()
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert dec[0x38] == 1.0 and dec[0x08] == 2.0 ** -6 and dec[0x01] == 2.0 ** -9
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert dec[0x00] == 0.0 and np.signbit(dec[0x80])


def test_e4m3_round_trip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    np.testing.assert_array_equal(O.e4m3_encode(vals), codes)


def test_e4m3_ties_to_even_at_every_midpoint():
    pos = np.array([c for c in range(0x7F)], np.int64)          # 0 .. 0x7E, ascending values
    vals = O.e4m3_decode(pos)
    for a, b in zip(pos[:-1], pos[1:]):
        mid = (O.e4m3_decode([a])[0] + O.e4m3_decode([b])[0]) / 2.0
        assert np.float32(mid) == mid                     # midpoints are fp32-exact
        want = a if a % 2 == 0 else b                     # even mantissa wins
        assert O.e4m3_encode(np.float32(mid))[()] == want, (a, b, mid)
        assert O.e4m3_encode(-np.float32(mid))[()] == (want | 0x80)
        lo = np.nextafter(np.float32(mid), np.float32(-1))
        hi = np.nextafter(np.float32(mid), np.float32(1e9))
        assert O.e4m3_encode(lo)[()] == a and O.e4m3_encode(hi)[()] == b
    assert vals[-1] == 448.0


def test_e4m3_agrees_with_torch_cast():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(40),
        rng.uniform(-448, 448, 200000).astype(np.float32),
        (rng.standard_normal(50000) * 1e-2).astype(np.float32),     # subnormal range
    ])
    ours = O.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()   # library cast
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_saturates():
    assert O.e4m3_encode(np.float32(500.0))[()] == 0x7E
    assert O.e4m3_encode(np.float32(-1e30))[()] == 0xFE
    assert O.e4m3_encode(np.float32(464.0))[()] == 0x7E


def test_quantize_scale_and_amax_code():
    x = np.random.default_rng(6).standard_normal((50, 128)).astype(np.float32)
    codes, s = O.quantize_fp8(x)
    amax = np.abs(x).max(axis=1)
    np.testing.assert_array_equal(s, (amax / np.float32(448)).astype(np.float32))
    j = np.abs(x).argmax(axis=1)
    assert set(codes[np.arange(50), j] & 0x7F) == {0x7E}        # the amax element is +-448
    dq = O.e4m3_decode(codes) * s[:, None]
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 above the subnormal range
    big = np.abs(x) > amax[:, None] * 2.0 ** -6 * 1.01
    assert np.all(np.abs(dq - x)[big] <= np.abs(x)[big] * 2.0 ** -4 + 1e-12)
    z_codes, z_s = O.quantize_fp8(np.zeros((2, 64), np.float32))
    assert not z_codes.any() and not z_s.any()


# ----------------------------------------------------------------- scores

def test_score_worked_example():
    g = _gold("score_worked_example.json")
    assert np.array_equal(O.e4m3_decode(g["q8_codes"]), np.array(g["q8_values"]))
    assert np.array_equal(O.e4m3_decode(g["k8_codes"]), np.array(g["k8_values"]))
    lay = O.pool_layout(np.concatenate([[0], np.cumsum(g["doc_lens"])]))
    i = g["query"]
    w = np.zeros((12, 1), np.float32)
    w[i] = g["w"]
    S = O.scores_fp8(np.array([g["q8_codes"]], np.uint8), np.array([g["s_q"]], np.float32),
                     np.array(g["k8_codes"], np.uint8), np.array(g["s_k"], np.float32), w, lay, [i])
    np.testing.assert_array_equal(S[0], np.array(g["scores"], np.float32))
    assert O.select_pools(S[0], 2).tolist() == g["top2_pools"]


def test_score_dots_exact_against_fractions():
    """The float64 dot of E4M3 codes equals the exact rational sum."""
    rng = np.random.default_rng(7)
    q8 = rng.integers(0, 256, (3, 128)).astype(np.uint8)
    k8 = rng.integers(0, 256, (5, 128)).astype(np.uint8)
    q8[(q8 & 0x7F) == 0x7F] = 0
    k8[(k8 & 0x7F) == 0x7F] = 0
    fl = O.e4m3_decode(q8) @ O.e4m3_decode(k8).T
    dec = [Fraction(float(v)) if not np.isnan(v) else None for v in O.e4m3_decode_table()]
    for a in range(3):
        for b in range(5):
            ex = sum(dec[x] * dec[y] for x, y in zip(q8[a], k8[b]))
            assert Fraction(float(fl[a, b])) == ex


def test_zero_weights_pick_lowest_pools():
    S = np.zeros(40, np.float32)
    assert O.select_pools(S, 8).tolist() == list(range(8))
    S = np.array([-0.0, 0.0] * 20, np.float32)
    assert O.select_pools(S, 8).tolist() == list(range(8))


def test_select_nan_ranks_below_every_number():
    """NaN is below -inf (reading R6: NaN ranks lowest); among NaNs the lower pool index wins."""
    S = np.array([np.nan, -np.inf, np.nan, -3e38, np.inf, np.nan, 0.0], np.float32)
    assert O.select_pools(S, 4).tolist() == [1, 3, 4, 6]
    assert O.select_pools(S, 5).tolist() == [0, 1, 3, 4, 6]
    assert O.select_pools(S, 6).tolist() == [0, 1, 2, 3, 4, 6]


def test_select_positive_scaling_invariant():
    rng = np.random.default_rng(8)
    S = rng.standard_normal(300).astype(np.float32)
    assert np.array_equal(O.select_pools(S, 50), O.select_pools(S * np.float32(4.0), 50))


# ----------------------------------------------------------------- select / rows

def test_select_matches_full_sort_with_ties():
    rng = np.random.default_rng(9)
    for trial in range(200):
        n = int(rng.integers(1, 60))
        S = rng.integers(-3, 4, n).astype(np.float32) * np.float32(0.5)   # many ties
        if trial % 3 == 0:
            S[S == 0] = -0.0
        k = int(rng.integers(1, 70))
        ranked = sorted(range(n), key=lambda p: (-float(S[p]), p))       # library sort
        assert O.select_pools(S, k).tolist() == sorted(ranked[:min(k, n)])


def test_tiny_rows_golden():
    g = _gold("tiny_rows.json")
    lay = O.pool_layout(np.concatenate([[0], np.cumsum(g["doc_lens"])]))
    for c in g["cases"]:
        i = c["i"]
        sel = O.select_pools(np.array(c["scores"], np.float32), g["topk"])
        row = O.index_row(lay, i, sel, g["W"])
        n = len(c["row"])
        assert row[:n].tolist() == c["row"], c["why"]
        assert np.all(row[n:] == -1)


def test_row_width():
    const = _gold("structural_constants.json")
    W = O.row_width(const["topk_pools"]["value"])
    assert W % const["row_multiple"]["value"] == 0
    assert W >= const["max_raw_slots"]["value"] and W - 128 < const["max_raw_slots"]["value"]
    assert W == 2176
    assert O.row_width(8) == 128


def _valid_closed_form(r, topk):
    return 4 * min(topk, (r + 1) // 4) + (r + 1) % 4


def test_valid_counts_closed_form_and_max():
    const = _gold("structural_constants.json")
    topk = const["topk_pools"]["value"]
    assert 4 * topk == const["index_topk_positions"]["value"]
    lay = O.pool_layout([0, 2200])
    rng = np.random.default_rng(10)
    mx = 0
    for i in list(range(0, 12)) + list(range(2040, 2060)) + [2199]:
        d, r, n_i, tail = O.query_geometry(lay, i)
        S = rng.standard_normal(n_i).astype(np.float32)
        row = O.index_row(lay, i, O.select_pools(S, topk), O.row_width(topk))
        nv = int((row >= 0).sum())
        assert nv == _valid_closed_form(r, topk)
        mx = max(mx, nv)
    assert mx == const["max_raw_slots"]["value"]


def test_dense_below_cutover():
    """With topk >= n_i every candidate is kept, so the row is the whole causal
    prefix of the document: s_d .. i."""
    lay = O.pool_layout([0, 301, 512])
    rng = np.random.default_rng(11)
    for i in [0, 3, 4, 150, 300, 301, 302, 305, 511]:
        d, r, n_i, _ = O.query_geometry(lay, i)
        S = rng.standard_normal(n_i).astype(np.float32)
        row = O.index_row(lay, i, O.select_pools(S, 1000), 512)
        s_d = int(lay["cu_seqlens"][d])
        assert row[row >= 0].tolist() == list(range(s_d, i + 1))


def _closed_form_totals(doc_lens, topk):
    P = sum(L // 4 for L in doc_lens)
    pairs = sum((r + 1) // 4 for L in doc_lens for r in range(L))
    valid = sum(_valid_closed_form(r, topk) for L in doc_lens for r in range(L))
    return P, pairs, valid


@pytest.mark.parametrize("idx,want", [(0, (127, 16762, 16065)),
                                      (1, (1024, 2096128, 6295552)),
                                      (3, (8192, 134209536, 65058816))])
def test_workload_totals(idx, want):
    wl = workloads.workload(idx)
    assert _closed_form_totals(wl.doc_lens, wl.topk) == want


# ----------------------------------------------------------------- attention

def _dense_causal_sdpa(q, kv, cu, scale):
    """Dense causal attention per document with torch's CPU SDPA (library)."""
    T, H, D = q.shape
    out = np.zeros((T, H, D), np.float64)
    for d in range(len(cu) - 1):
        s, e = int(cu[d]), int(cu[d + 1])
        qq = torch.from_numpy(q[s:e].astype(np.float64)).permute(1, 0, 2)          # [H, L, D]
        kk = torch.from_numpy(kv[s:e].astype(np.float64))[None].expand(H, -1, -1)
        o = torch.nn.functional.scaled_dot_product_attention(qq, kk, kk, is_causal=True, scale=scale)
        out[s:e] = o.permute(1, 0, 2).numpy()
    return out


def test_attention_dense_equivalence_small():
    rng = np.random.default_rng(12)
    cu = np.array([0, 37, 60])
    T, H, D = 60, 3, 32
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    kv = rng.standard_normal((T, D)).astype(np.float32)
    lay = O.pool_layout(cu)
    W = 128
    idx = np.stack([O.index_row(lay, i, O.select_pools(np.zeros(O.query_geometry(lay, i)[2], np.float32), 100), W)
                    for i in range(T)])
    out, lse = O.sparse_attention(q, kv, idx, 1 / math.sqrt(D), list(range(T)))
    ref = _dense_causal_sdpa(q, kv, cu, 1 / math.sqrt(D))
    np.testing.assert_allclose(out, ref, rtol=1e-5, atol=1e-5)


def test_attention_constant_values_and_lse_closed_form():
    rng = np.random.default_rng(13)
    T, H, D = 20, 2, 16
    kv = np.tile(rng.standard_normal((1, D)).astype(np.float32), (T, 1))
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    idx = np.full((T, 128), -1, np.int32)
    for i in range(T):
        idx[i, :i + 1] = np.arange(i + 1)
    out, _ = O.sparse_attention(q, kv, idx, 0.3, list(range(T)))
    np.testing.assert_allclose(out, np.broadcast_to(kv[0], out.shape), rtol=1e-6)   # convex combination
    # q = 0: all logits 0, softmax uniform: lse = ln(n), out = mean of the rows
    kv2 = rng.standard_normal((T, D)).astype(np.float32)
    out2, lse2 = O.sparse_attention(np.zeros_like(q), kv2, idx, 0.3, list(range(T)))
    for i in range(T):
        np.testing.assert_allclose(lse2[i], math.log(i + 1), rtol=1e-6)
        np.testing.assert_allclose(out2[i, 0], kv2[:i + 1].mean(axis=0), rtol=1e-5, atol=1e-6)


def test_attention_lse_matches_library_logsumexp():
    rng = np.random.default_rng(14)
    T, H, D = 9, 2, 8
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    kv = rng.standard_normal((T, D)).astype(np.float32)
    idx = np.full((1, 128), -1, np.int32)
    idx[0, :5] = [0, 2, 3, 7, 8]
    _, lse = O.sparse_attention(q[[8]], kv, idx, 0.5, [8])
    for h in range(H):
        z = [0.5 * float(np.dot(q[8, h].astype(np.float64), kv[j].astype(np.float64))) for j in [0, 2, 3, 7, 8]]
        assert abs(lse[0, h] - scipy.special.logsumexp(z)) < 1e-6


def test_attention_empty_row():
    out, lse = O.sparse_attention(np.ones((1, 2, 4), np.float32), np.ones((3, 4), np.float32),
                                  np.full((1, 128), -1, np.int32), 1.0, [0])
    assert not out.any() and np.all(np.isneginf(lse))


# ----------------------------------------------------------------- paged decode

def test_paged_slots_hand_example():
    bt = [7, 2, 5]                       # pages of positions 0-127, 128-255, 256-383
    row = [0, 1, 127, 128, 255, 256, 300, -1]
    assert O.paged_slots(row, bt).tolist() == [896, 897, 1023, 256, 383, 640, 684, -1]


def test_decode_row_is_the_prefill_row_of_the_last_token():
    wl = workloads.workload(1)                 # one document: the decode query is its last token
    inp = workloads.indexer_inputs(wl)
    L = 700
    k = inp.k[:L].float().numpy()
    row, _ = O.decode_row(inp.q_idx[L - 1].float().numpy(), inp.w[L - 1], k, inp.gate[:L], inp.ape, 64,
                          O.row_width(64))
    full = O.indexer(inp.q_idx[:L].float().numpy(), k, inp.gate[:L], inp.ape, inp.w[:L], np.array([0, L]), 64,
                     O.row_width(64), rows=np.array([L - 1]))
    assert np.array_equal(row, full["indices"][0])
