"""Pins of the oracle's sparse attention backward against facts fixed outside it:
torch autograd through a separately written attention, a closed form for a
single slot, and an identity that follows from how the logits scale.
No GPU needed."""
import numpy as np
import torch

from oracle import kpool_oracle as O


def _rows(T, W, rng, dup_free=True):
    idx = np.full((T, W), -1, np.int64)
    for i in range(T):
        n = int(rng.integers(1, min(i + 1, W) + 1))
        idx[i, :n] = np.sort(rng.choice(i + 1, n, replace=False))
    return idx


def _autograd(q, kv, idx, scale, dout):
    """Gradients of sum(dout * out) by torch autograd, attention written with gather + softmax."""
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kvt = torch.tensor(kv, dtype=torch.float64, requires_grad=True)
    outs = []
    for i in range(q.shape[0]):
        sel = torch.from_numpy(idx[i][idx[i] >= 0])
        k = kvt.index_select(0, sel)                              # [n, D]
        a = torch.softmax(scale * qt[i] @ k.T, dim=-1)            # [H, n]
        outs.append(a @ k)
    out = torch.stack(outs)
    (out * torch.from_numpy(dout)).sum().backward()
    return qt.grad.numpy(), kvt.grad.numpy(), out.detach().numpy()


def test_backward_matches_torch_autograd():
    rng = np.random.default_rng(11)
    T, H, D, W = 23, 3, 512, 12
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((T, D))
    dout = rng.standard_normal((T, H, D))
    idx = _rows(T, W, rng)
    scale = 1.0 / np.sqrt(D)
    g = O.sparse_attention_bwd(q, kv, idx, scale, dout, np.arange(T))
    dq, dkv, out = _autograd(q, kv, idx, scale, dout)
    np.testing.assert_allclose(g["out"], out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dq"], dq, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dkv"], dkv, rtol=1e-9, atol=1e-11)


def test_single_slot_closed_form():
    # one valid slot: p = 1, so the logit gradient vanishes (dq = 0) and the
    # latent row receives dout summed over heads
    rng = np.random.default_rng(2)
    T, H, D = 6, 4, 512
    q = rng.standard_normal((1, H, D))
    kv = rng.standard_normal((T, D))
    dout = rng.standard_normal((1, H, D))
    idx = np.array([[3, -1, -1, -1]])
    g = O.sparse_attention_bwd(q, kv, idx, 0.3, dout, np.array([5]), T=T)
    assert np.abs(g["dq"]).max() < 1e-12
    expect = np.zeros((T, D))
    expect[3] = dout[0].sum(axis=0)
    np.testing.assert_allclose(g["dkv"], expect, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["out"][0], np.broadcast_to(kv[3], (H, D)), rtol=1e-12)
    assert np.allclose(g["lse"][0], 0.3 * q[0] @ kv[3])


def test_scaling_identity():
    # Scaling every latent row by (1 + e) scales out by (1 + e) and every logit by (1 + e), as scaling q by
    # (1 + e) would; so <dkv, kv> - <dq, q> = <dout, out>.
    rng = np.random.default_rng(4)
    T, H, D, W = 40, 5, 512, 16
    q = rng.standard_normal((T, H, D))
    kv = rng.standard_normal((T, D))
    dout = rng.standard_normal((T, H, D))
    idx = _rows(T, W, rng)
    g = O.sparse_attention_bwd(q, kv, idx, 0.05, dout, np.arange(T))
    lhs = (g["dkv"] * kv).sum() - (g["dq"] * q).sum()
    rhs = (dout * g["out"]).sum()
    assert abs(lhs - rhs) <= 1e-9 * (abs(rhs) + 1.0)


def test_forward_part_agrees_with_the_forward_oracle():
    rng = np.random.default_rng(8)
    T, H, D, W = 17, 2, 512, 10
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    kv = rng.standard_normal((T, D)).astype(np.float32)
    idx = _rows(T, W, rng)
    idx[4] = -1                                   # an empty row: zero gradients, lse = -inf
    g = O.sparse_attention_bwd(q, kv, idx, 0.1, np.ones((T, H, D)), np.arange(T))
    out, lse = O.sparse_attention(q, kv, idx, 0.1, np.arange(T))
    np.testing.assert_allclose(g["out"], out, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(g["lse"], lse, rtol=1e-6, atol=1e-6)
    assert np.all(g["dq"][4] == 0) and np.all(np.isneginf(g["lse"][4]))
