"""CPU oracle for the absorbed-MLA projections either side of the sparse
attention.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it; the library never does.  It shares no code with the CUDA path.

Sources (pages, by title and section):
  [PR3699]  NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog:
            the K projection is absorbed into the query, attention runs over
            the shared 512-wide latent K/V, and the model-owned V projection is
            applied afterwards.
  [LORA]    miles "GLM-5.3-Flash" recipe, section 6 "LoRA RL": the DSA attention
            absorbs the kv_b_proj weight into the query and the output without
            calling that module.

Readings where the pages are silent:
  * kv_b_proj is a bias-free linear map from the 512-wide latent to
    n_heads * (d_nope + d_v) features, stored [out, in] = [H*(d_nope+d_v), 512];
    per head the first d_nope output rows are the key (no-position) part and
    the next d_v rows the value part (the multi-latent attention layout the
    GLM DSA layers inherit);
  * d_nope and d_v are parameters; the pages give neither.

Every step is float64.
"""
from __future__ import annotations

import numpy as np


def split_kv_b(w_kv_b, n_heads: int, d_nope: int, d_v: int) -> tuple[np.ndarray, np.ndarray]:
    """kv_b_proj weight [H*(d_nope+d_v), D] -> (W_UK [H, d_nope, D], W_UV [H, d_v, D])
    [LORA]: head h owns rows h*(d_nope+d_v) .. (h+1)*(d_nope+d_v)-1, key rows first."""
    w = np.asarray(w_kv_b, dtype=np.float64)
    D = w.shape[1]
    if w.shape[0] != n_heads * (d_nope + d_v):
        raise ValueError("kv_b_proj rows must be n_heads * (d_nope + d_v)")
    per_head = w.reshape(n_heads, d_nope + d_v, D)
    return per_head[:, :d_nope, :], per_head[:, d_nope:, :]


def absorb_q(q_nope, w_kv_b, d_nope: int, d_v: int) -> np.ndarray:
    """Query absorption [PR3699]: the no-position key of latent row c is
    k[h] = W_UK[h] c, so q_nope[h] . k[h] = (W_UK[h]^T q_nope[h]) . c and the
    latent query is q_lat[t,h,:] = sum_n q_nope[t,h,n] W_UK[h][n,:].
    q_nope [T, H, d_nope] -> q_lat [T, H, D] (float64)."""
    q = np.asarray(q_nope, dtype=np.float64)
    H = q.shape[1]
    w_uk, _ = split_kv_b(w_kv_b, H, d_nope, d_v)
    out = np.empty((q.shape[0], H, w_uk.shape[2]), dtype=np.float64)
    for h in range(H):
        out[:, h, :] = q[:, h, :] @ w_uk[h]
    return out


def v_proj(o_lat, w_kv_b, d_nope: int, d_v: int) -> np.ndarray:
    """V projection of the latent attention output [PR3699]: the value of latent
    row c is v[h] = W_UV[h] c, and softmax weights sum linearly, so the head
    output is o_v[t,h,:] = W_UV[h] o_lat[t,h,:].
    o_lat [T, H, D] -> o_v [T, H, d_v] (float64)."""
    o = np.asarray(o_lat, dtype=np.float64)
    H = o.shape[1]
    _, w_uv = split_kv_b(w_kv_b, H, d_nope, d_v)
    out = np.empty((o.shape[0], H, d_v), dtype=np.float64)
    for h in range(H):
        out[:, h, :] = o[:, h, :] @ w_uv[h].T
    return out
