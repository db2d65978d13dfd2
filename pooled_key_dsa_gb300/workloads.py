"""Seeded synthetic workloads for the KPool-DSA forward.

This module only draws inputs.  It holds none of the method's arithmetic and is
shared by the tests, the benchmark and the CPU oracle's drivers, so that every
side sees the same bytes.

Five workloads, shaped after the packed-THD rows that the GLM-5.3-Flash pages
train and serve on (NeMo AutoModel PR "add GLM-5.3-Flash training support",
section "cuDNN sparse MLA parity and performance": 64 query heads, a 512-wide
latent K/V, index_topk=2048 = 512 pools of index_kpool=4):

  0  tiny      T=512    docs [301, 211]                 H_i=4,  d_i=64,  topk=8,   H=4
  1  cutover   T=4096   one doc                         H_i=32, d_i=128, topk=512, H=64
  2  packed    T=8192   6 docs ~U[257,3000], no length a multiple of 4
  3  headline  T=32768  one doc
  4  long      T=131072 docs log-uniform in [1024,65536], last one truncated

Value recipe: every tensor comes from its own stream
``numpy.random.default_rng([seed, tensor_id(, chunk)])`` so that any slice can be
regenerated on its own.  Values are fp32 N(0,1); q_idx, k, q_lat and kv_lat are
then rounded to bf16 (round-to-nearest-even, done by torch's dtype cast);
``ape`` is N(0, 0.1**2) (0.1 read as the standard deviation) and
``w`` is N(0,1)/sqrt(H_i).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

# tensor ids of the per-tensor random streams
_DOCS, _QIDX, _K, _GATE, _APE, _W, _QLAT, _KVLAT = range(8)
_CHUNK = 1024          # tokens per independently seeded chunk of the big tensors


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    doc_lens: tuple
    n_idx_heads: int = 32     # H_i
    d_idx: int = 128          # d_i
    topk: int = 512           # pools kept per query
    n_heads: int = 64         # H
    d_lat: int = 512          # D
    kpool: int = 4

    @property
    def T(self) -> int:
        return int(sum(self.doc_lens))

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.doc_lens)]).astype(np.int32)

    @property
    def W(self) -> int:
        """Index-row width: room for 4*topk pooled positions plus a 3-token own
        tail, rounded up to a multiple of 128."""
        raw = self.kpool * self.topk + self.kpool - 1
        return 128 * ((raw + 127) // 128)

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d_lat)))


def _doc_lens_packed8192(seed: int) -> tuple:
    rng = np.random.default_rng([seed, _DOCS])
    while True:
        first = rng.integers(257, 3001, size=5)
        last = 8192 - int(first.sum())
        lens = [int(x) for x in first] + [last]
        if 257 <= last <= 3000 and all(x % 4 != 0 for x in lens):
            return tuple(lens)


def _doc_lens_loguniform(seed: int, total: int = 131072) -> tuple:
    rng = np.random.default_rng([seed, _DOCS])
    lens = []
    while sum(lens) < total:
        u = rng.uniform(math.log(1024), math.log(65536))
        lens.append(int(round(math.exp(u))))
    lens[-1] -= sum(lens) - total
    return tuple(lens)


def workload(idx: int) -> Workload:
    if idx == 0:
        return Workload("tiny_T512_2docs", 0, (301, 211), n_idx_heads=4, d_idx=64,
                        topk=8, n_heads=4)
    if idx == 1:
        return Workload("single_doc_T4096", 1, (4096,))
    if idx == 2:
        return Workload("packed_T8192_6docs", 2, _doc_lens_packed8192(2))
    if idx == 3:
        return Workload("single_doc_T32768", 3, (32768,))
    if idx == 4:
        return Workload("packed_T131072_loguniform", 4, _doc_lens_loguniform(4))
    raise ValueError(f"no workload {idx}")


def custom(name: str, seed: int, doc_lens, **kw) -> Workload:
    """A workload with explicit document lengths (edge-case tests)."""
    return Workload(name, seed, tuple(int(x) for x in doc_lens), **kw)


# --------------------------------------------------------------------------- draws

def _normal(seed: int, tid: int, shape, std: float = 1.0, chunk: int | None = None) -> np.ndarray:
    key = [seed, tid] if chunk is None else [seed, tid, chunk]
    x = np.random.default_rng(key).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def _chunked_bf16(seed: int, tid: int, T: int, row_shape: tuple, rows=None) -> torch.Tensor:
    """bf16 tensor [T, *row_shape] drawn in independently seeded token chunks.
    With ``rows`` given, only those token rows are drawn (same values)."""
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        out = torch.empty((len(rows),) + tuple(row_shape), dtype=torch.bfloat16)
        for c in np.unique(rows // _CHUNK):
            n = min(_CHUNK, T - c * _CHUNK)
            block = _bf16(_normal(seed, tid, (n,) + tuple(row_shape), chunk=int(c)))
            sel = np.nonzero(rows // _CHUNK == c)[0]
            out[torch.from_numpy(sel)] = block[torch.from_numpy(rows[sel] - c * _CHUNK)]
        return out
    out = torch.empty((T,) + tuple(row_shape), dtype=torch.bfloat16)
    n_chunks = (T + _CHUNK - 1) // _CHUNK

    def fill(c):
        n = min(_CHUNK, T - c * _CHUNK)
        out[c * _CHUNK:c * _CHUNK + n] = _bf16(_normal(seed, tid, (n,) + tuple(row_shape), chunk=c))

    with ThreadPoolExecutor(max_workers=8) as ex:
        list(ex.map(fill, range(n_chunks)))
    return out


@dataclass
class Inputs:
    """Host-side inputs of one workload.  bf16 tensors are torch CPU tensors
    (their exact fp32 values are ``.float()``); fp32 tensors are numpy."""
    wl: Workload
    cu_seqlens: np.ndarray
    q_idx: torch.Tensor       # bf16 [T, H_i, d_i]
    k: torch.Tensor           # bf16 [T, d_i]
    gate: np.ndarray          # fp32 [T, d_i]
    ape: np.ndarray           # fp32 [kpool, d_i]
    w: np.ndarray             # fp32 [T, H_i]
    kv_lat: torch.Tensor      # bf16 [T, D]
    q_lat: torch.Tensor | None = field(default=None)   # bf16 [T, H, D] (drawn on demand)


def indexer_inputs(wl: Workload) -> Inputs:
    """Everything except q_lat (which is large; see :func:`q_lat`)."""
    T, Hi, di = wl.T, wl.n_idx_heads, wl.d_idx
    q_idx = _chunked_bf16(wl.seed, _QIDX, T, (Hi, di))
    k = _bf16(_normal(wl.seed, _K, (T, di)))
    gate = _normal(wl.seed, _GATE, (T, di))
    ape = _normal(wl.seed, _APE, (wl.kpool, di), std=0.1)
    w = _normal(wl.seed, _W, (T, Hi)) / np.float32(math.sqrt(Hi))
    w = w.astype(np.float32)
    kv_lat = _chunked_bf16(wl.seed, _KVLAT, T, (wl.d_lat,))
    return Inputs(wl, wl.cu_seqlens, q_idx, k, gate, ape, w, kv_lat)


def q_lat(wl: Workload, rows=None) -> torch.Tensor:
    """bf16 q_lat [T, H, D], or only the given token rows of it."""
    return _chunked_bf16(wl.seed, _QLAT, wl.T, (wl.n_heads, wl.d_lat), rows=rows)


# tensor ids of a further layer's attention inputs: _QLAT + _LAYER_STRIDE * layer, ...
_LAYER_STRIDE = 16


def layer_attention_inputs(wl: Workload, layer: int, rows=None) -> tuple:
    """(q_lat [T, H, D] or the given rows of it, kv_lat [T, D]) of DSA layer ``layer`` of a stack whose
    layers share this workload's index rows (IndexShare: the indexer runs in layer 0 only).  Layer 0 gives
    the workload's own attention inputs; each further layer has its own seeded streams."""
    off = _LAYER_STRIDE * int(layer)
    q = _chunked_bf16(wl.seed, _QLAT + off, wl.T, (wl.n_heads, wl.d_lat), rows=rows)
    kv = _chunked_bf16(wl.seed, _KVLAT + off, wl.T, (wl.d_lat,))
    return q, kv


# tensor ids of the absorbed-MLA projection inputs and of the attention's output gradient
_QNOPE, _WKVB, _OLAT, _DOUT = 8, 9, 10, 11


def proj_inputs(wl: Workload, d_nope: int = 128, d_v: int = 128, rows=None) -> tuple:
    """(q_nope bf16 [T, H, d_nope] or the given token rows of it, w_kv_b bf16 [H*(d_nope+d_v), D]).
    q_nope is N(0,1); the kv_b_proj weight is N(0,1)/sqrt(D), so that a projected latent row has about
    unit variance."""
    H, D = wl.n_heads, wl.d_lat
    q_nope = _chunked_bf16(wl.seed, _QNOPE, wl.T, (H, d_nope), rows=rows)
    w = _bf16(_normal(wl.seed, _WKVB, (H * (d_nope + d_v), D)) / np.float32(math.sqrt(D)))
    return q_nope, w


def o_lat_input(wl: Workload, rows=None) -> torch.Tensor:
    """A stand-in latent attention output, bf16 [T, H, D] N(0,1), for the V projection on its own."""
    return _chunked_bf16(wl.seed, _OLAT, wl.T, (wl.n_heads, wl.d_lat), rows=rows)


def dout_input(wl: Workload, rows=None) -> torch.Tensor:
    """A seeded gradient of the loss w.r.t. the attention output, bf16 [T, H, D] N(0,1)."""
    return _chunked_bf16(wl.seed, _DOUT, wl.T, (wl.n_heads, wl.d_lat), rows=rows)


def all_inputs(wl: Workload) -> Inputs:
    inp = indexer_inputs(wl)
    inp.q_lat = q_lat(wl)
    return inp


# --------------------------------------------------------------------------- paged decode

_DEC_LENS, _DEC_PAGES, _DEC_K, _DEC_GATE, _DEC_APE, _DEC_KV, _DEC_QIDX, _DEC_W, _DEC_QLAT = range(32, 41)
PAGE_TOKENS = 128          # 32 pools of 4 per page (vLLM's index_kpool x 32 block)


@dataclass(frozen=True)
class DecodeWorkload:
    """One decode step over B sequences: sequence b holds seq_lens[b] tokens, the last of which is the
    step's query.  Each sequence is one document; its latent rows and pooled keys live in 128-token pages
    assigned by a seeded permutation (so the block table is not the identity)."""
    name: str
    seed: int
    seq_lens: tuple
    n_idx_heads: int = 32
    d_idx: int = 128
    topk: int = 512
    n_heads: int = 64
    d_lat: int = 512
    kpool: int = 4
    spare_pages: int = 3

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def W(self) -> int:
        raw = self.kpool * self.topk + self.kpool - 1
        return 128 * ((raw + 127) // 128)

    @property
    def pages_per_seq(self) -> list:
        return [(L + PAGE_TOKENS - 1) // PAGE_TOKENS for L in self.seq_lens]

    @property
    def max_pages(self) -> int:
        return max(max(self.pages_per_seq), 1)

    @property
    def n_pages(self) -> int:
        return sum(self.pages_per_seq) + self.spare_pages

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.d_lat)))

    def block_table(self) -> np.ndarray:
        """int32 [B, max_pages]: a seeded permutation of the pages, -1 past each sequence's last page."""
        perm = np.random.default_rng([self.seed, _DEC_PAGES]).permutation(self.n_pages).astype(np.int32)
        bt = np.full((self.B, self.max_pages), -1, np.int32)
        at = 0
        for b, npg in enumerate(self.pages_per_seq):
            bt[b, :npg] = perm[at:at + npg]
            at += npg
        return bt


def decode_workload(idx: int) -> DecodeWorkload:
    if idx == 0:      # tiny: every branch of a row (all pools kept, radix select, tails 0..3, several pages)
        return DecodeWorkload("decode_tiny", 50, (5, 9, 130, 517, 1029, 1100, 2052, 2175), topk=64)
    if idx == 1:      # rows of > 8192 pools take the chunked select
        return DecodeWorkload("decode_long_rows", 51, (33000, 40003, 4099))
    if idx == 2:      # benchmark: 128 sequences, lengths log-uniform in [4096, 32768]
        rng = np.random.default_rng([52, _DEC_LENS])
        lens = np.exp(rng.uniform(math.log(4096), math.log(32768), size=128)).astype(np.int64)
        return DecodeWorkload("decode_B128_loguniform_4K_32K", 52, tuple(int(x) for x in lens))
    raise ValueError(f"no decode workload {idx}")


@dataclass
class DecodeInputs:
    dw: DecodeWorkload
    k: list            # per sequence, bf16 [L_b, d_i]
    gate: list         # per sequence, fp32 [L_b, d_i]
    kv_lat: list       # per sequence, bf16 [L_b, D]
    ape: np.ndarray    # fp32 [kpool, d_i]
    q_idx: torch.Tensor  # bf16 [B, H_i, d_i], the newest token of each sequence
    w: np.ndarray      # fp32 [B, H_i]
    q_lat: torch.Tensor  # bf16 [B, H, D]


def decode_inputs(dw: DecodeWorkload) -> DecodeInputs:
    """Host inputs of a decode workload (small and medium sizes; the benchmark draws its caches on the GPU)."""
    ks, gs, kvs = [], [], []
    for b, L in enumerate(dw.seq_lens):
        ks.append(_bf16(_normal(dw.seed, _DEC_K, (L, dw.d_idx), chunk=b)))
        gs.append(_normal(dw.seed, _DEC_GATE, (L, dw.d_idx), chunk=b))
        kvs.append(_bf16(_normal(dw.seed, _DEC_KV, (L, dw.d_lat), chunk=b)))
    ape = _normal(dw.seed, _DEC_APE, (dw.kpool, dw.d_idx), std=0.1)
    q_idx = _bf16(_normal(dw.seed, _DEC_QIDX, (dw.B, dw.n_idx_heads, dw.d_idx)))
    w = (_normal(dw.seed, _DEC_W, (dw.B, dw.n_idx_heads)) / np.float32(math.sqrt(dw.n_idx_heads))).astype(np.float32)
    q_lat = _bf16(_normal(dw.seed, _DEC_QLAT, (dw.B, dw.n_heads, dw.d_lat)))
    return DecodeInputs(dw, ks, gs, kvs, ape, q_idx, w, q_lat)
