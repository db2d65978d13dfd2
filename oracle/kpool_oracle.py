"""CPU oracle for the KPool-DSA forward.  TEST INFRASTRUCTURE ONLY.

Plain, slow NumPy restatement of what the pooled-key DeepSeek Sparse Attention
layer of GLM-5.3-Flash computes.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the library never does.  It shares
no code with the CUDA path.

Sources (pages, by title and section):
  [PR4036]  prime-rl PR "GLM-5.3-Flash text model", Summary, the bullet on
            "The DSA indexer with k-pool compression": per-document pools of 4
            starting at each document's first token; per-channel
            softmax(gate + ape)-weighted mean; Hadamard rotation of queries and
            pooled keys (fp32 butterfly) before FP8 scoring; a query scores the
            complete pools that end at or before it, keeps the top 512, and also
            attends to its own incomplete pool; index rows padded to a multiple
            of 128; the pool layout is built once per forward.
  [PR3699]  NeMo AutoModel PR "add GLM-5.3-Flash training support", Changelog
            (K projection absorbed into the query; attention over the shared
            512-wide latent K/V) and section "cuDNN sparse MLA parity and
            performance" (64 query heads, index_topk=2048, index_kpool=4,
            2051 raw sparse slots).
  [MILES]   miles "GLM-5.3-Flash" recipe, section 1 "Model Introduction"
            (NoPE MLA, kpool-compressed lightning indexer, 64 attention heads).

Readings where the pages are silent (each one a parameter or a stated choice):
  * indexer score = s_k[p] * sum_h (w[i,h] * s_q[i,h]) * ReLU(q8[i,h] . k8[p]),
    no other scalar; top-k ties go to the lower pool index; -0 counts as +0;
  * FP8 format is OCP E4M3 ("fn": max 448, no infinities), one exact fp32
    absmax scale per vector, round-to-nearest-even with saturation;
  * Hadamard: Sylvester (natural) order, radix-2 stages with strides
    1, 2, 4, ..., d/2, then one multiply by fp32(1/sqrt(d));
  * when (r+1) % 4 == 0 the query's own pool is complete and only competes in
    the top-k, so the own tail holds (r+1) % 4 <= 3 tokens (2048 + 3 = 2051);
  * index rows list the valid positions in ascending order, then -1;
  * attention scale is a parameter (1/sqrt(512)); LSE is the natural log;
  * the backward (section 9) is the exact gradient of that attention, with
    the latent row as both key and value (its gradient sums both roles).

Every floating-point step is float64 unless a step says fp32, in which case it
is np.float32 arithmetic in the same order as written here.
"""
from __future__ import annotations

import math

import numpy as np

KPOOL = 4


# ----------------------------------------------------------------- 1. layout

def pool_layout(cu_seqlens, kpool: int = KPOOL) -> dict:
    """PoolLayout [PR4036]: pools restart at every document's first token; a
    document of length L holds floor(L/kpool) complete pools; a trailing group
    of L % kpool tokens gets no pooled key."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = cu[1:] - cu[:-1]
    if np.any(lens < 0):
        raise ValueError("cu_seqlens must be non-decreasing")
    n_pools = lens // kpool
    cu_pools = np.concatenate([[0], np.cumsum(n_pools)]).astype(np.int64)
    pool_tok_start = np.empty(int(cu_pools[-1]), dtype=np.int64)
    tok_doc = np.empty(int(cu[-1]), dtype=np.int64)
    for d in range(len(lens)):
        for m in range(int(n_pools[d])):
            pool_tok_start[cu_pools[d] + m] = cu[d] + kpool * m
        tok_doc[cu[d]:cu[d + 1]] = d
    return {"cu_seqlens": cu, "cu_pools": cu_pools, "pool_tok_start": pool_tok_start,
            "tok_doc": tok_doc, "n_pools": int(cu_pools[-1]), "kpool": kpool}


# ----------------------------------------------------------------- 2. pooling

def pool_keys(k, gate, ape, layout) -> np.ndarray:
    """Pooled indexer keys [PR4036]: for pool p with tokens t_0..t_{kpool-1},
    kp[p, c] = sum_j a_{j,c} k[t_j, c] with a_{.,c} = softmax_j(gate[t_j,c] +
    ape[j,c]), the softmax taken over the pool's tokens, per channel.
    Float64 throughout; stored as fp32."""
    k = np.asarray(k, dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    ape = np.asarray(ape, dtype=np.float64)
    kp = layout["kpool"]
    P = layout["n_pools"]
    out = np.zeros((P, k.shape[1]), dtype=np.float32)
    for p in range(P):
        t0 = int(layout["pool_tok_start"][p])
        logits = gate[t0:t0 + kp] + ape[:kp]                 # [kpool, d]
        m = logits.max(axis=0)
        e = np.exp(logits - m)
        a = e / e.sum(axis=0)
        out[p] = (a * k[t0:t0 + kp]).sum(axis=0)
    return out


# ----------------------------------------------------------------- 3. Hadamard

def hadamard_f32(x) -> np.ndarray:
    """Orthonormal Walsh-Hadamard transform of the last axis in fp32
    [PR4036: "Hadamard-rotated (same fp32 butterfly order)"]: stages with
    stride h = 1, 2, 4, ..., d/2; in each block of 2h, for j < h,
    (x[j], x[j+h]) <- (x[j] + x[j+h], x[j] - x[j+h]); then every element is
    multiplied once by fp32(1/sqrt(d))."""
    x = np.array(x, dtype=np.float32, copy=True)
    d = x.shape[-1]
    if d & (d - 1):
        raise ValueError("Hadamard width must be a power of two")
    lead = x.shape[:-1]
    h = 1
    while h < d:
        y = x.reshape(lead + (d // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        x = y.reshape(lead + (d,))
        h *= 2
    c = np.float32(1.0 / math.sqrt(d))
    return x * c


# ----------------------------------------------------------------- 4. FP8 E4M3

E4M3_MAX = 448.0


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 OCP E4M3 ("fn") codes: 1 sign bit, 4 exponent
    bits (bias 7), 3 mantissa bits; exponent 0 is subnormal (step 2^-9);
    0x7F / 0xFF are NaN; no infinities."""
    t = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            t[c] = np.nan
        elif e == 0:
            t[c] = s * m * 2.0 ** -9
        else:
            t[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


_DEC = e4m3_decode_table()


def e4m3_decode(codes) -> np.ndarray:
    return _DEC[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Round fp32 values to OCP E4M3: nearest, ties to even, magnitudes above
    448 saturate to 448; the sign bit follows the input (so -0 -> 0x80)."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    sign = np.signbit(v).astype(np.uint8) << 7
    a = np.minimum(np.abs(v), E4M3_MAX)
    _, ex = np.frexp(a)                         # a = f * 2**ex, f in [0.5, 1)
    e = np.maximum(ex.astype(np.int64) - 1, -6)  # unbiased exponent, subnormals at -6
    q = np.rint(np.ldexp(a, (3 - e)))           # mantissa units at that exponent, RNE
    carry = q >= 16                              # rounded up into the next binade
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q).astype(np.int64)
    normal = q >= 8
    exp_field = np.where(normal, e + 7, 0)
    man_field = np.where(normal, q - 8, q)
    return (sign | (exp_field << 3).astype(np.uint8) | man_field.astype(np.uint8)).astype(np.uint8)


def quantize_fp8(xr) -> tuple[np.ndarray, np.ndarray]:
    """Per-vector FP8 cast of Hadamard-rotated fp32 vectors (last axis):
    amax = max|x|; s = amax/448 and inv = 448/amax (fp32 divisions); codes =
    E4M3(x * inv) (fp32 multiply).  An all-zero vector gives codes 0, s = 0."""
    xr = np.asarray(xr, dtype=np.float32)
    amax = np.abs(xr).max(axis=-1)
    safe = np.where(amax > 0, amax, np.float32(1.0)).astype(np.float32)
    inv = (np.float32(E4M3_MAX) / safe).astype(np.float32)
    s = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(0.0))
    codes = e4m3_encode(xr * inv[..., None])
    codes = np.where((amax > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes, s.astype(np.float32)


def quantize_queries(q_idx):
    """q_idx fp32 [T, H_i, d_i] -> (q8 [T,H_i,d_i] uint8, s_q [T,H_i] fp32)."""
    return quantize_fp8(hadamard_f32(q_idx))


def quantize_keys(kpool):
    """pooled keys fp32 [P, d_i] -> (k8 [P,d_i] uint8, s_k [P] fp32)."""
    return quantize_fp8(hadamard_f32(kpool))


# ----------------------------------------------------------------- 5. scores

def query_geometry(layout, i: int) -> tuple[int, int, int, int]:
    """(doc d, in-document position r, number of scorable pools n_i, tail
    length) for query token i.  The candidates are the complete pools of i's
    own document that end at or before i [PR4036]: pool m ends at 4m+3 <= r."""
    d = int(layout["tok_doc"][i])
    r = i - int(layout["cu_seqlens"][d])
    kp = layout["kpool"]
    n_i = (r + 1) // kp
    tail = (r + 1) % kp
    return d, r, n_i, tail


def scores_fp8(q8, s_q, k8, s_k, w, layout, rows) -> list[np.ndarray]:
    """Indexer scores for the given query rows (one fp32 array per row, over
    the row's candidate pools in pool order).  ``q8``/``s_q`` are indexed by
    position in ``rows``; ``w`` by token:
        S[i,p] = s_k[p] * sum_h (w[i,h]*s_q[i,h]) * max(q8[i,h].k8[p], 0).
    The E4M3 dot products are exact in float64 (products of two E4M3 values
    are multiples of 2^-18 below 2^18, and 128 of them sum below 2^43), so
    the BLAS call here is exact whatever its summation order."""
    kdec = e4m3_decode(k8)
    out = []
    for n, i in enumerate(rows):
        d, r, n_i, _ = query_geometry(layout, int(i))
        p0 = int(layout["cu_pools"][d])
        qd = e4m3_decode(q8[n])                                  # [H_i, d_i]
        dots = qd @ kdec[p0:p0 + n_i].T                          # [H_i, n_i], exact
        ws = np.asarray(w[i], np.float64) * np.asarray(s_q[n], np.float64)
        S = (ws[:, None] * np.maximum(dots, 0.0)).sum(axis=0) * np.asarray(s_k[p0:p0 + n_i], np.float64)
        out.append(S.astype(np.float32))
    return out


def scores_exact(q_idx, w, kpool, layout, rows) -> list[np.ndarray]:
    """Exact scorer (no rotation, no FP8): S = sum_h w_h * ReLU(q_h . kp), in
    float64.  Used only to report exact-vs-FP8 set agreement."""
    out = []
    for i in rows:
        d, r, n_i, _ = query_geometry(layout, int(i))
        p0 = int(layout["cu_pools"][d])
        dots = np.asarray(q_idx[i], np.float64) @ np.asarray(kpool[p0:p0 + n_i], np.float64).T
        S = (np.asarray(w[i], np.float64)[:, None] * np.maximum(dots, 0.0)).sum(axis=0)
        out.append(S.astype(np.float32))
    return out


# ----------------------------------------------------------------- 6-7. select and rows

def select_pools(S_row: np.ndarray, topk: int) -> np.ndarray:
    """Indices (relative to the document's first pool) of the top
    min(topk, n) pools by score descending, ties to the lower pool index;
    -0 is +0 and NaN ranks lowest, below -inf.  Returned in ascending pool
    order."""
    S = np.asarray(S_row, dtype=np.float64) + 0.0
    nan = np.isnan(S)
    S = np.where(nan, -np.inf, S)
    n = len(S)
    order = np.lexsort((np.arange(n), -S, nan))  # primary: numbers first, then -S ascending, then pool
    return np.sort(order[:min(topk, n)])


def index_row(layout, i: int, sel_rel: np.ndarray, W: int) -> np.ndarray:
    """Index row of query i [PR4036, PR3699]: positions of the selected pools
    plus the own incomplete pool's tokens up to i, ascending, padded with -1
    to width W."""
    d, r, n_i, tail = query_geometry(layout, i)
    p0 = int(layout["cu_pools"][d])
    kp = layout["kpool"]
    pos = [int(layout["pool_tok_start"][p0 + int(m)]) + j for m in sel_rel for j in range(kp)]
    pos += list(range(i - tail + 1, i + 1))
    pos = sorted(pos)
    if len(pos) > W:
        raise ValueError("index row wider than W")
    row = np.full(W, -1, dtype=np.int32)
    row[:len(pos)] = pos
    return row


def row_width(topk: int, kpool: int = KPOOL) -> int:
    """Smallest multiple of 128 that holds kpool*topk + kpool-1 positions."""
    raw = kpool * topk + kpool - 1
    return 128 * ((raw + 127) // 128)


# ----------------------------------------------------------------- 8. attention

def sparse_attention(q_lat, kv_lat, indices, scale, rows) -> tuple[np.ndarray, np.ndarray]:
    """Absorbed NoPE sparse latent attention [PR3699, MILES]: for query i and
    head h over the valid slots j of its index row,
    z_j = scale * q_lat[i,h] . kv_lat[idx_j]; out[i,h] = sum_j softmax(z)_j kv_lat[idx_j];
    lse[i,h] = ln sum_j exp(z_j).  Float64.  A row with no valid slot gives
    out = 0 and lse = -inf.  Returns (out [len(rows),H,D] fp32, lse [len(rows),H] fp32).
    ``q_lat`` is indexed by position in ``rows`` (it may hold only those rows)."""
    H, D = q_lat.shape[1], q_lat.shape[2]
    outs = np.zeros((len(rows), H, D), dtype=np.float32)
    lses = np.full((len(rows), H), -np.inf, dtype=np.float32)
    for n, i in enumerate(rows):
        idx = np.asarray(indices[n])
        valid = idx[idx >= 0]
        if len(valid) == 0:
            continue
        kv = np.asarray(kv_lat[valid], dtype=np.float64)             # [n, D]
        q = np.asarray(q_lat[n], dtype=np.float64)                    # [H, D]
        z = float(scale) * (q @ kv.T)                                 # [H, n]
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        s = e.sum(axis=1, keepdims=True)
        outs[n] = ((e / s) @ kv).astype(np.float32)
        lses[n] = (m[:, 0] + np.log(s[:, 0])).astype(np.float32)
    return outs, lses


# ----------------------------------------------------------------- whole indexer

def indexer(q_idx, k, gate, ape, w, cu_seqlens, topk, W, rows=None, kpool=KPOOL, with_scores=False):
    """Steps 1-7 for the given query rows (all rows when None).  Inputs are the
    exact fp32 values (bf16 tensors widened).  Returns a dict with the layout,
    pooled keys, FP8 codes/scales, index rows [len(rows), W] and, optionally,
    the per-row candidate scores."""
    q_idx = np.asarray(q_idx, np.float32)
    layout = pool_layout(cu_seqlens, kpool)
    kp = pool_keys(k, gate, ape, layout)
    k8, s_k = quantize_keys(kp)
    T = int(layout["cu_seqlens"][-1])
    rows = np.arange(T) if rows is None else np.asarray(rows)
    q8, s_q = quantize_queries(q_idx[rows])          # indexed by position in rows
    S = scores_fp8(q8, s_q, k8, s_k, w, layout, rows)
    idx = np.stack([index_row(layout, int(i), select_pools(S[n], topk), W)
                    for n, i in enumerate(rows)]) if len(rows) else np.zeros((0, W), np.int32)
    res = {"layout": layout, "kpool": kp, "k8": k8, "s_k": s_k, "q8": q8, "s_q": s_q,
           "rows": rows, "indices": idx}
    if with_scores:
        res["scores"] = S
    return res


# ----------------------------------------------------------------- 9. attention backward

def sparse_attention_bwd(q_lat, kv_lat, indices, scale, dout, rows, T=None) -> dict:
    """Gradients of the absorbed sparse latent attention [PR3699] for the given
    query rows, given dL/dout.  The latent row kv[j] is both key and value, so
    it collects a value term and a key term.  Float64, per query i and head h,
    over the valid slots j of the row:
        p_j   = softmax(scale * q[i,h] . kv[j])
        dp_j  = dout[i,h] . kv[j]
        delta = sum_j p_j dp_j             (= dout[i,h] . out[i,h])
        dz_j  = p_j (dp_j - delta)
        dq[i,h] = scale * sum_j dz_j kv[j]
        dkv[j] += p_j dout[i,h] + scale * dz_j q[i,h]
    ``q_lat``/``dout`` are indexed by position in ``rows``; dkv [T, D] holds the
    contributions of these rows only.  Returns dq [len(rows),H,D], dkv [T,D],
    and the recomputed out [len(rows),H,D] and lse [len(rows),H] (float64)."""
    q_lat = np.asarray(q_lat, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    kv_all = np.asarray(kv_lat, dtype=np.float64)
    T = kv_all.shape[0] if T is None else T
    n, H, D = q_lat.shape
    dq = np.zeros((n, H, D))
    dkv = np.zeros((T, D))
    out = np.zeros((n, H, D))
    lse = np.full((n, H), -np.inf)
    for m in range(n):
        idx = np.asarray(indices[m])
        valid = idx[idx >= 0]
        if len(valid) == 0:
            continue
        kv = kv_all[valid]                                  # [n_v, D]
        z = float(scale) * (q_lat[m] @ kv.T)                # [H, n_v]
        zmax = z.max(axis=1, keepdims=True)
        e = np.exp(z - zmax)
        s = e.sum(axis=1, keepdims=True)
        p = e / s
        out[m] = p @ kv
        lse[m] = zmax[:, 0] + np.log(s[:, 0])
        dp = dout[m] @ kv.T                                 # [H, n_v]
        delta = (dout[m] * out[m]).sum(axis=1, keepdims=True)
        dz = p * (dp - delta)
        dq[m] = float(scale) * (dz @ kv)
        np.add.at(dkv, valid, p.T @ dout[m] + float(scale) * (dz.T @ q_lat[m]))
    return {"dq": dq, "dkv": dkv, "out": out, "lse": lse}


# ----------------------------------------------------------------- 10. paged decode

PAGE_TOKENS = 128


def paged_slots(row, block_table_row) -> np.ndarray:
    """A decode index row in latent-cache slots [PR4036, "Patches and workarounds": 128-token pages of 32
    pools]: the in-sequence position pos lives in slot block_table_row[pos // 128] * 128 + pos % 128;
    -1 stays -1."""
    row = np.asarray(row, dtype=np.int64)
    bt = np.asarray(block_table_row, dtype=np.int64)
    out = np.full(row.shape, -1, dtype=np.int64)
    ok = row >= 0
    out[ok] = bt[row[ok] // PAGE_TOKENS] * PAGE_TOKENS + row[ok] % PAGE_TOKENS
    return out


def decode_row(q_idx, w, k, gate, ape, topk, W):
    """Index row of a decode query: the newest token (position L-1) of a sequence of L tokens whose indexer
    keys and gates are k, gate [L, d_i], with query q_idx [H_i, d_i] and head weights w [H_i].  The same
    rules as the prefill row of query L-1 of a one-document row (steps 1-7); returns in-sequence positions."""
    L = np.asarray(k).shape[0]
    q_all = np.zeros((L,) + np.asarray(q_idx).shape, dtype=np.float32)
    q_all[L - 1] = np.asarray(q_idx, dtype=np.float32)
    w_all = np.zeros((L, np.asarray(w).shape[0]), dtype=np.float32)
    w_all[L - 1] = np.asarray(w, dtype=np.float32)
    res = indexer(q_all, k, gate, ape, w_all, np.array([0, L]), topk, W, rows=np.array([L - 1]))
    return res["indices"][0], res
