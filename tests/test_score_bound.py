"""The per-pool error bound that the GPU parity tests put on FP8 indexer scores (tests/oracle_rows.py) holds for
fp32 evaluations of the score in several summation orders, and is tight enough that a dropped head term or a
missing pool scale falls outside it."""
import numpy as np
import pytest

from oracle import kpool_oracle as O
from tests import oracle_rows as OR


def _codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7F) == 0x7F, np.uint8(0x3F), c)     # no NaN codes


def _fp32_scores(q8, ws, k8, sk, order):
    """The score as a GPU would evaluate it: exact E4M3 products summed in fp32 (in the given order), ReLU,
    fp32 sum of the weighted heads over four partial sums, fp32 product with the pool scale."""
    qd = O.e4m3_decode(q8).astype(np.float32)
    kd = O.e4m3_decode(k8).astype(np.float32)
    hi, di = qd.shape
    out = np.empty(kd.shape[0], np.float32)
    for p in range(kd.shape[0]):
        res = [np.float32(0)] * 4
        for h in range(hi):
            acc = np.float32(0)
            for d in order:
                acc = np.float32(acc + qd[h, d] * kd[p, d])      # the product is exact in fp32
            res[h % 4] = np.float32(res[h % 4] + np.float32(ws[h] * max(acc, np.float32(0))))
        out[p] = np.float32(np.float32(np.float32(res[0] + res[1]) + np.float32(res[2] + res[3])) * sk[p])
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bound_holds_for_fp32_evaluations_and_catches_mistakes(seed):
    rng = np.random.default_rng(seed)
    hi, di, n = 8, 32, 24
    q8 = _codes(rng, (1, hi, di))
    k8 = _codes(rng, (n, di))
    w = rng.standard_normal((1, hi)).astype(np.float32)
    s_q = np.abs(rng.standard_normal((1, hi))).astype(np.float32) + np.float32(0.01)
    s_k = np.abs(rng.standard_normal(n)).astype(np.float32) + np.float32(0.01)
    ws = (w[0] * s_q[0]).astype(np.float32)
    layout = O.pool_layout(np.array([0, 4 * n + 3], np.int32))
    row = np.array([4 * n + 2])                                   # sees all n pools
    w_tok = np.zeros((4 * n + 3, hi), np.float32)               # w is indexed by token
    w_tok[row[0]] = w[0]
    S = O.scores_fp8(q8, s_q, k8, s_k, w_tok, layout, row)[0].astype(np.float64)
    bound = OR.score_error_bound(np.abs(O.e4m3_decode(q8[0])), np.abs(O.e4m3_decode(k8)), np.abs(ws.astype(np.float64)),
                                 s_k.astype(np.float64), np.abs(S))
    for order in (range(di), range(di - 1, -1, -1), rng.permutation(di)):
        g = _fp32_scores(q8[0], ws, k8, s_k, list(order)).astype(np.float64)
        assert np.all(np.abs(g - S) <= bound)
    # a dropped head term, or the pool scale left out, is far outside the bound
    g = _fp32_scores(q8[0], ws, k8, s_k, list(range(di))).astype(np.float64)
    qd = O.e4m3_decode(q8[0])
    kd = O.e4m3_decode(k8)
    dropped = g - ws[0] * np.maximum(qd[0] @ kd.T, 0.0) * s_k
    moved = np.abs(dropped - S) > bound
    assert moved[np.abs(ws[0] * np.maximum(qd[0] @ kd.T, 0.0) * s_k) > 1e-3 * np.abs(S).max()].all()
    unscaled = g / s_k
    assert np.any(np.abs(unscaled - S) > bound)


def test_gamma_matches_its_definition():
    u = 2.0 ** -24
    for n in (1, 32, 128, 34):
        assert OR.gamma(n) == pytest.approx(n * u / (1 - n * u), rel=1e-15)
