"""Pins of the absorbed-MLA projection oracle against facts fixed outside it.

The absorbed form must give the same attention as multi-latent attention run
the unabsorbed way: kv_b_proj applied to every latent row as a plain linear
layer (torch on CPU), the result split per head into key and value, softmax
attention over the keys, values summed.  One-hot weights check which rows of
kv_b_proj each projection reads.  No GPU needed."""
import numpy as np
import torch

from oracle import absorb_oracle as A
from oracle import kpool_oracle as O


def _unabsorbed_mla(q_nope, latent, w_kv_b, rows_idx, scale, d_nope, d_v):
    """Textbook multi-latent attention with the latent expanded first."""
    H = q_nope.shape[1]
    kv = torch.nn.functional.linear(torch.from_numpy(latent), torch.from_numpy(w_kv_b))   # [n, H*(dn+dv)]
    kv = kv.view(latent.shape[0], H, d_nope + d_v)
    k_nope, v = kv[..., :d_nope], kv[..., d_nope:]
    outs = []
    for t, idx in enumerate(rows_idx):
        sel = torch.from_numpy(idx[idx >= 0])
        q = torch.from_numpy(q_nope[t])                                     # [H, dn]
        logits = scale * torch.einsum("hn,jhn->hj", q, k_nope[sel])
        p = torch.softmax(logits, dim=-1)
        outs.append(torch.einsum("hj,jhv->hv", p, v[sel]))
    return torch.stack(outs).numpy()


def test_absorbed_attention_equals_unabsorbed_mla():
    rng = np.random.default_rng(7)
    T, H, dn, dv, D = 11, 3, 8, 5, 512
    q_nope = rng.standard_normal((T, H, dn))
    latent = rng.standard_normal((T, D))
    w = rng.standard_normal((H * (dn + dv), D)) / np.sqrt(D)
    idx = np.full((T, 16), -1, np.int64)
    for t in range(T):                       # causal rows with a gap, so the sets differ
        sel = [j for j in range(t + 1) if j != t - 2]
        idx[t, :len(sel)] = sel
    scale = 0.37
    ref = _unabsorbed_mla(q_nope, latent, w, idx, scale, dn, dv)

    q_lat = A.absorb_q(q_nope, w, dn, dv)
    out_lat, _ = O.sparse_attention(q_lat, latent, idx, scale, np.arange(T))
    # the attention oracle returns fp32; redo its float64 sums here for a tight check
    out64 = np.zeros((T, H, D))
    for t in range(T):
        sel = idx[t][idx[t] >= 0]
        z = scale * q_lat[t] @ latent[sel].T
        p = np.exp(z - z.max(axis=1, keepdims=True))
        out64[t] = (p / p.sum(axis=1, keepdims=True)) @ latent[sel]
    np.testing.assert_allclose(out_lat, out64, rtol=1e-5, atol=1e-6)
    o_v = A.v_proj(out64, w, dn, dv)
    np.testing.assert_allclose(o_v, ref, rtol=1e-10, atol=1e-12)


def test_absorbed_logits_equal_key_dot_products():
    rng = np.random.default_rng(3)
    T, H, dn, dv, D = 4, 2, 16, 16, 512
    q_nope = rng.standard_normal((T, H, dn))
    latent = rng.standard_normal((6, D))
    w = rng.standard_normal((H * (dn + dv), D))
    kv = torch.nn.functional.linear(torch.from_numpy(latent), torch.from_numpy(w)).view(6, H, dn + dv).numpy()
    q_lat = A.absorb_q(q_nope, w, dn, dv)
    for h in range(H):
        np.testing.assert_allclose(q_lat[:, h] @ latent.T, q_nope[:, h] @ kv[:, h, :dn].T, rtol=1e-10, atol=1e-9)


def test_one_hot_weights_pick_the_head_slices():
    T, H, dn, dv, D = 3, 4, 6, 3, 512
    rng = np.random.default_rng(5)
    q_nope = rng.standard_normal((T, H, dn))
    o_lat = rng.standard_normal((T, H, D))
    h, n, v, c = 2, 4, 1, 300
    w = np.zeros((H * (dn + dv), D))
    w[h * (dn + dv) + n, c] = 1.0            # key row n of head h reads latent column c
    w[h * (dn + dv) + dn + v, c + 1] = 1.0   # value row v of head h reads latent column c+1
    q_lat = A.absorb_q(q_nope, w, dn, dv)
    expect = np.zeros((T, H, D))
    expect[:, h, c] = q_nope[:, h, n]
    assert np.array_equal(q_lat, expect)
    o_v = A.v_proj(o_lat, w, dn, dv)
    expect_v = np.zeros((T, H, dv))
    expect_v[:, h, v] = o_lat[:, h, c + 1]
    assert np.array_equal(o_v, expect_v)


def test_split_rejects_mismatched_weight():
    w = np.zeros((10, 512))
    try:
        A.split_kv_b(w, 2, 3, 3)
    except ValueError:
        return
    raise AssertionError("a weight with the wrong row count must be rejected")
