"""ctypes binding of ``libkpooldsa.so`` (C ABI in ``include/kpooldsa.h``).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  If the
library has not been built, importing this module works but every call raises
``KpoolUnavailable`` -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libkpooldsa.so")

KPOOL_OK = 0
ERRORS = {1: "KPOOL_ERR_INVALID_ARG", 2: "KPOOL_ERR_SHAPE", 3: "KPOOL_ERR_ALIGN", 4: "KPOOL_ERR_LAYOUT",
          5: "KPOOL_ERR_INDEX_RANGE", 6: "KPOOL_ERR_TIMEOUT", 7: "KPOOL_ERR_CUDA", 8: "KPOOL_ERR_WORKSPACE",
          9: "KPOOL_ERR_CHECK"}
CODES = {v: k for k, v in ERRORS.items()}

EXPORTED = ("kpool_workspace_bytes", "kpool_workspace_offsets", "kpool_build", "dsa_index", "sparse_mla_fwd",
            "kpool_stage_select", "kpool_set_stage_events", "kpool_check_status", "kpool_strerror", "kpool_version",
            "dsa_index_noalloc", "sparse_mla_fwd_rows", "kpool_forward_host", "mla_absorb_q", "mla_v_proj",
            "sparse_mla_bwd", "kpool_measure_l2_reduce", "kpool_paged_append", "dsa_decode_workspace_bytes",
            "dsa_decode_index", "kpool_cast_e4m3", "kpool_debug_inject_stall")
STALL_SCORE, STALL_SPARSE_MLA = 1, 2


class KpoolUnavailable(ImportError):
    pass


class KpoolError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({strerror(code)})")


class Params(ctypes.Structure):
    _fields_ = [("kpool", ctypes.c_int32), ("topk", ctypes.c_int32), ("n_idx_heads", ctypes.c_int32),
                ("d_idx", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("d_lat", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class LayoutC(ctypes.Structure):
    _fields_ = [("n_docs", ctypes.c_int32), ("T", ctypes.c_int32), ("max_pools", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("cu_pools", ctypes.c_void_p),
                ("pool_tok_start", ctypes.c_void_p), ("tok_doc", ctypes.c_void_p), ("status", ctypes.c_void_p)]


class HostIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("k", "gate", "ape", "cu_seqlens", "q_idx", "w", "q_lat", "kv_lat",
                                                "out", "lse")]


class DevIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("k", "gate", "ape", "cu_seqlens", "q_idx", "w", "q_lat", "kv_lat",
                                                "out", "lse", "kpool")] + \
               [("layout", ctypes.POINTER(LayoutC)), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("indices", ctypes.c_void_p), ("W", ctypes.c_int32)]


MAX_CHUNKS = 64


class WsOffsets(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("q8", "ws", "k8", "s_k", "pair_base", "sched", "scores", "total")]


_lib = None
_LIB_DEFAULT = _LIB_PATH
_LIB_CHECKED = os.path.join(os.path.dirname(_LIB_PATH), "libkpooldsa_checked.so")


def use_checked_library(on: bool) -> None:
    """Switch the binding to the KPOOL_CHECKED build of the library (internal bounds checks that
    record KPOOL_ERR_CHECK in the status word) or back to the default build; later calls load it."""
    global _LIB_PATH, _lib
    _LIB_PATH = _LIB_CHECKED if on else _LIB_DEFAULT
    _lib = None


def lib():
    """The loaded library (raises KpoolUnavailable when it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise KpoolUnavailable(f"{_LIB_PATH} is not built; run pooled_key_dsa_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.kpool_workspace_bytes.argtypes = [ctypes.POINTER(Params), i32, i32]
        L.kpool_workspace_bytes.restype = sz
        L.kpool_workspace_offsets.argtypes = [ctypes.POINTER(Params), i32, i32, ctypes.POINTER(WsOffsets)]
        L.kpool_build.argtypes = [vp, vp, vp, vp, i32, i32, ctypes.POINTER(Params), vp, ctypes.POINTER(LayoutC), vp]
        L.dsa_index.argtypes = [vp, vp, vp, ctypes.POINTER(LayoutC), i32, ctypes.POINTER(Params), vp, sz, vp, i32,
                                vp]
        L.sparse_mla_fwd.argtypes = [vp, vp, vp, i32, i32, i32, ctypes.c_float, vp, vp, vp, vp]
        L.sparse_mla_fwd_rows.argtypes = [vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, vp, vp, vp, vp]
        L.kpool_forward_host.argtypes = [ctypes.POINTER(HostIO), ctypes.POINTER(DevIO), i32, i32,
                                         ctypes.POINTER(Params), i32, vp, vp, vp]
        L.sparse_mla_bwd.argtypes = [vp, vp, vp, i32, i32, i32, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp]
        L.kpool_measure_l2_reduce.argtypes = [vp, i32, vp, i32, vp]
        L.kpool_cast_e4m3.argtypes = [vp, ctypes.c_int64, vp, vp]
        L.kpool_debug_inject_stall.argtypes = [i32]
        L.kpool_paged_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, ctypes.POINTER(Params), vp, vp,
                                         vp, vp]
        L.dsa_decode_workspace_bytes.argtypes = [ctypes.POINTER(Params), i32, i32]
        L.dsa_decode_workspace_bytes.restype = sz
        L.dsa_decode_index.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, ctypes.POINTER(Params), vp, sz, vp,
                                       i32, vp, vp]
        L.mla_absorb_q.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
        L.mla_v_proj.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
        L.kpool_stage_select.argtypes = [vp, vp, ctypes.POINTER(LayoutC), i32, vp, i32, vp]
        L.dsa_index_noalloc.argtypes = [vp, vp, vp, ctypes.POINTER(LayoutC), i32, ctypes.POINTER(Params), vp, i32,
                                        vp]
        L.kpool_check_status.argtypes = [vp, vp]
        L.kpool_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        L.kpool_strerror.argtypes = [ctypes.c_int]
        L.kpool_strerror.restype = ctypes.c_char_p
        L.kpool_version.restype = ctypes.c_char_p
        for name in ("kpool_workspace_offsets", "kpool_build", "dsa_index", "sparse_mla_fwd", "kpool_stage_select",
                     "kpool_set_stage_events", "kpool_check_status", "dsa_index_noalloc", "sparse_mla_fwd_rows",
                     "kpool_forward_host"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().kpool_strerror(int(code)).decode()
    except KpoolUnavailable:
        return "library not built"


def _check(rc: int, what: str):
    if rc != KPOOL_OK:
        raise KpoolError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _want(t, dtype, shape, name):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_params(topk=512, n_idx_heads=32, d_idx=128, n_heads=64, d_lat=512, scale=None, kpool=4) -> Params:
    if scale is None:
        scale = 1.0 / math.sqrt(d_lat)
    return Params(kpool, topk, n_idx_heads, d_idx, n_heads, d_lat, scale)


def row_width(topk: int, kpool: int = 4) -> int:
    raw = kpool * topk + kpool - 1
    return 128 * ((raw + 127) // 128)


class PoolLayout:
    """Device buffers of a PoolLayout plus the C struct that points at them."""

    def __init__(self, cu_seqlens: torch.Tensor, T: int, status: torch.Tensor | None = None):
        _want(cu_seqlens, torch.int32, None, "cu_seqlens")
        dev = cu_seqlens.device
        self.n_docs = cu_seqlens.numel() - 1
        self.T = int(T)
        self.max_pools = self.T // 4
        self.cu_seqlens = cu_seqlens
        self.cu_pools = torch.zeros(self.n_docs + 1, dtype=torch.int32, device=dev)
        self.pool_tok_start = torch.zeros(max(self.max_pools, 1), dtype=torch.int32, device=dev)
        self.tok_doc = torch.zeros(max(self.T, 1), dtype=torch.int32, device=dev)
        self.status = status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
        self.c = LayoutC(self.n_docs, self.T, self.max_pools, cu_seqlens.data_ptr(), self.cu_pools.data_ptr(),
                         self.pool_tok_start.data_ptr(), self.tok_doc.data_ptr(), self.status.data_ptr())


def workspace_bytes(p: Params, T: int, n_docs: int) -> int:
    return int(lib().kpool_workspace_bytes(ctypes.byref(p), T, n_docs))


def workspace_offsets(p: Params, T: int, n_docs: int) -> WsOffsets:
    o = WsOffsets()
    _check(lib().kpool_workspace_offsets(ctypes.byref(p), T, n_docs, ctypes.byref(o)), "kpool_workspace_offsets")
    return o


def kpool_build(k, gate, ape, cu_seqlens, p: Params, kpool_out=None, layout: PoolLayout | None = None,
                stream=None):
    """Pooled keys fp32 [T//4, d_idx] and the PoolLayout (both on k's device)."""
    T, d = k.shape
    _want(k, torch.bfloat16, (T, p.d_idx), "k")
    _want(gate, torch.float32, (T, p.d_idx), "gate")
    _want(ape, torch.float32, (p.kpool, p.d_idx), "ape")
    if layout is None:
        layout = PoolLayout(cu_seqlens, T)
    if kpool_out is None:
        kpool_out = torch.empty((max(layout.max_pools, 1), p.d_idx), dtype=torch.float32, device=k.device)
    _check(lib().kpool_build(_ptr(k), _ptr(gate), _ptr(ape), _ptr(cu_seqlens), layout.n_docs, T, ctypes.byref(p),
                             _ptr(kpool_out), ctypes.byref(layout.c), _stream(stream)), "kpool_build")
    return kpool_out, layout


def dsa_index(q_idx, w, kpool, layout: PoolLayout, topk: int, p: Params, workspace=None, indices=None, W=None,
              stream=None):
    """int32 index rows [T, W] (W defaults to the multiple of 128 above 4*topk+3)."""
    T = layout.T
    _want(q_idx, torch.bfloat16, (T, p.n_idx_heads, p.d_idx), "q_idx")
    _want(w, torch.float32, (T, p.n_idx_heads), "w")
    _want(kpool, torch.float32, None, "kpool")
    W = row_width(topk) if W is None else int(W)
    nbytes = workspace_bytes(p, T, layout.n_docs)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q_idx.device)
    if indices is None:
        indices = torch.empty((T, W), dtype=torch.int32, device=q_idx.device)
    _check(lib().dsa_index(_ptr(q_idx), _ptr(w), _ptr(kpool), ctypes.byref(layout.c), topk, ctypes.byref(p),
                           _ptr(workspace), workspace.numel(), _ptr(indices), W, _stream(stream)), "dsa_index")
    return indices


def dsa_index_noalloc(q_idx, w, kpool, layout: PoolLayout, topk: int, p: Params, indices=None, W=None,
                      stream=None):
    """dsa_index without a workspace, for callers that cannot allocate device
    memory: the library keeps the scratch in one static device array (T up to
    4096, at most 256 documents).  Only ``indices`` is allocated here, and
    only when the caller passes none."""
    T = layout.T
    _want(q_idx, torch.bfloat16, (T, p.n_idx_heads, p.d_idx), "q_idx")
    _want(w, torch.float32, (T, p.n_idx_heads), "w")
    _want(kpool, torch.float32, None, "kpool")
    W = row_width(topk) if W is None else int(W)
    if indices is None:
        indices = torch.empty((T, W), dtype=torch.int32, device=q_idx.device)
    _check(lib().dsa_index_noalloc(_ptr(q_idx), _ptr(w), _ptr(kpool), ctypes.byref(layout.c), topk,
                                   ctypes.byref(p), _ptr(indices), W, _stream(stream)), "dsa_index_noalloc")
    return indices


def sparse_mla_fwd(q_lat, kv_lat, indices, scale: float, out=None, lse=None, status=None, stream=None):
    """(out bf16 [T, H, 512], lse fp32 [T, H])."""
    T, H, D = q_lat.shape
    _want(q_lat, torch.bfloat16, (T, H, D), "q_lat")
    _want(kv_lat, torch.bfloat16, (T, D), "kv_lat")
    _want(indices, torch.int32, None, "indices")
    if indices.dim() != 2 or indices.shape[0] != T:
        raise ValueError("indices must be [T, W]")
    if out is None:
        out = torch.empty_like(q_lat)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q_lat.device)
    _check(lib().sparse_mla_fwd(_ptr(q_lat), _ptr(kv_lat), _ptr(indices), indices.shape[1], T, H, float(scale),
                                _ptr(out), _ptr(lse), _ptr(status), _stream(stream)), "sparse_mla_fwd")
    return out, lse


def sparse_mla_fwd_rows(q_lat, kv_lat, indices, scale: float, out=None, lse=None, status=None, stream=None):
    """sparse_mla_fwd over a block of query rows: q_lat [n, H, 512] and indices [n, W] are the block's rows,
    kv_lat [T, 512] the whole latent (index entries lie in [-1, T))."""
    n, H, D = q_lat.shape
    T = kv_lat.shape[0]
    _want(q_lat, torch.bfloat16, (n, H, D), "q_lat")
    _want(kv_lat, torch.bfloat16, (T, D), "kv_lat")
    _want(indices, torch.int32, None, "indices")
    if indices.dim() != 2 or indices.shape[0] != n:
        raise ValueError("indices must be [n_rows, W]")
    if out is None:
        out = torch.empty_like(q_lat)
    if lse is None:
        lse = torch.empty((n, H), dtype=torch.float32, device=q_lat.device)
    _check(lib().sparse_mla_fwd_rows(_ptr(q_lat), _ptr(kv_lat), _ptr(indices), indices.shape[1], n, T, H,
                                     float(scale), _ptr(out), _ptr(lse), _ptr(status), _stream(stream)),
           "sparse_mla_fwd_rows")
    return out, lse


def sparse_mla_bwd(q_lat, kv_lat, indices, scale: float, out, lse, dout, dq=None, dkv=None, delta=None,
                   status=None, stream=None):
    """Gradients of sparse_mla_fwd: returns (dq bf16 [T, H, 512], dkv fp32 [T, 512]).  out and lse are the
    forward's results; dout is dL/dout.  dkv is accumulated with fp32 atomics (its last bits depend on the
    order in which they land)."""
    T, H, D = q_lat.shape
    _want(q_lat, torch.bfloat16, (T, H, D), "q_lat")
    _want(kv_lat, torch.bfloat16, (T, D), "kv_lat")
    _want(indices, torch.int32, None, "indices")
    if indices.dim() != 2 or indices.shape[0] != T:
        raise ValueError("indices must be [T, W]")
    _want(out, torch.bfloat16, (T, H, D), "out")
    _want(lse, torch.float32, (T, H), "lse")
    _want(dout, torch.bfloat16, (T, H, D), "dout")
    if dq is None:
        dq = torch.empty_like(q_lat)
    if dkv is None:
        dkv = torch.empty((T, D), dtype=torch.float32, device=q_lat.device)
    if delta is None:
        delta = torch.empty((T, H), dtype=torch.float32, device=q_lat.device)
    _want(dq, torch.bfloat16, (T, H, D), "dq")
    _want(dkv, torch.float32, (T, D), "dkv")
    _want(delta, torch.float32, (T, H), "delta")
    _check(lib().sparse_mla_bwd(_ptr(q_lat), _ptr(kv_lat), _ptr(indices), indices.shape[1], T, H, float(scale),
                                _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dkv), _ptr(delta), _ptr(status),
                                _stream(stream)), "sparse_mla_bwd")
    return dq, dkv


def measure_l2_reduce(buf, row_ids, stream=None):
    """Adds 1.0 to every element of the rows buf[row_ids] (fp32 [rows, 512]) with the dkv scatter's fp32
    reductions; a timing aid for the reduction rate that bounds sparse_mla_bwd."""
    _want(buf, torch.float32, None, "buf")
    _want(row_ids, torch.int32, None, "row_ids")
    if buf.dim() != 2 or buf.shape[1] != 512:
        raise ValueError("buf must be [rows, 512]")
    _check(lib().kpool_measure_l2_reduce(_ptr(buf), buf.shape[0], _ptr(row_ids), row_ids.numel(), _stream(stream)),
           "kpool_measure_l2_reduce")


def debug_inject_stall(mask: int) -> None:
    """Test hook of the bounded waits: STALL_SCORE / STALL_SPARSE_MLA make the later launches of the tcgen05
    scoring / sparse attention kernels wait first on a barrier that nothing completes, so that they end with
    KPOOL_ERR_TIMEOUT after the wait limit; 0 restores normal operation."""
    _check(lib().kpool_debug_inject_stall(int(mask)), "kpool_debug_inject_stall")


def cast_e4m3(x, out=None, stream=None):
    """uint8 E4M3 codes of the fp32 tensor x (round to nearest even, saturating at 448): the conversion that
    every FP8 quantiser of the library applies, exposed for value-by-value tests."""
    _want(x, torch.float32, None, "x")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib().kpool_cast_e4m3(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "kpool_cast_e4m3")
    return out


# ----------------------------------------------------------------- paged decode

PAGE_TOKENS = 128          # tokens per page (32 pools of 4)


def decode_workspace_bytes(p: Params, B: int, max_pages: int) -> int:
    return int(lib().dsa_decode_workspace_bytes(ctypes.byref(p), B, max_pages))


def paged_append(k, gate, ape, pool_tok, pool_seq, pool_idx, block_table, n_pages: int, p: Params, k8_cache, sk_cache,
                 status=None, stream=None):
    """Pooled keys of the 4-token rows pool_tok[v].. of k/gate into slot pool_idx[v] of sequence pool_seq[v]'s
    pages (block_table [B, max_pages]) of the caches k8_cache uint8 [n_pages, 32, d_i], sk_cache fp32 [n_pages, 32]."""
    n = pool_tok.numel()
    for name, t in (("pool_tok", pool_tok), ("pool_seq", pool_seq), ("pool_idx", pool_idx)):
        _want(t, torch.int32, (n,), name)
    _want(block_table, torch.int32, None, "block_table")
    _want(k8_cache, torch.uint8, (n_pages, 32, p.d_idx), "k8_cache")
    _want(sk_cache, torch.float32, (n_pages, 32), "sk_cache")
    _check(lib().kpool_paged_append(_ptr(k), _ptr(gate), _ptr(ape), _ptr(pool_tok), _ptr(pool_seq), _ptr(pool_idx), n,
                                    _ptr(block_table), block_table.shape[1], n_pages, ctypes.byref(p), _ptr(k8_cache),
                                    _ptr(sk_cache), _ptr(status), _stream(stream)), "kpool_paged_append")


def decode_index(q_idx, w, k8_cache, sk_cache, block_table, seq_lens, topk: int, p: Params, W: int,
                 workspace=None, indices=None, status=None, stream=None):
    """Index rows of one decode step: latent-cache slots [B, W] for each sequence's newest token."""
    B = q_idx.shape[0]
    n_pages = k8_cache.shape[0]
    _want(q_idx, torch.bfloat16, (B, p.n_idx_heads, p.d_idx), "q_idx")
    _want(w, torch.float32, (B, p.n_idx_heads), "w")
    _want(block_table, torch.int32, None, "block_table")
    _want(seq_lens, torch.int32, (B,), "seq_lens")
    max_pages = block_table.shape[1]
    need = decode_workspace_bytes(p, B, max_pages)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q_idx.device)
    if indices is None:
        indices = torch.empty((B, W), dtype=torch.int32, device=q_idx.device)
    _check(lib().dsa_decode_index(_ptr(q_idx), _ptr(w), _ptr(k8_cache), _ptr(sk_cache), n_pages, _ptr(block_table),
                                  max_pages, _ptr(seq_lens), B, topk, ctypes.byref(p), _ptr(workspace),
                                  workspace.numel(), _ptr(indices), W, _ptr(status), _stream(stream)),
           "dsa_decode_index")
    return indices


def _proj_weight(w_kv_b, H: int, d_nope: int, d_v: int, D: int):
    _want(w_kv_b, torch.bfloat16, (H * (d_nope + d_v), D), "w_kv_b")


def mla_absorb_q(q_nope, w_kv_b, d_nope: int, d_v: int, out=None, status=None, stream=None):
    """Query absorption: q_lat[t,h,:] = q_nope[t,h,:] . W_UK[h] with W_UK[h] the d_nope key rows of head h in the
    kv_b_proj weight w_kv_b [H*(d_nope+d_v), 512].  q_nope [T, H, d_nope] bf16 -> q_lat [T, H, 512] bf16."""
    T, H, dn = q_nope.shape
    if dn != d_nope:
        raise ValueError("q_nope's last dimension must be d_nope")
    _want(q_nope, torch.bfloat16, (T, H, dn), "q_nope")
    _proj_weight(w_kv_b, H, d_nope, d_v, 512)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_nope.device)
    _want(out, torch.bfloat16, (T, H, 512), "q_lat")
    _check(lib().mla_absorb_q(_ptr(q_nope), _ptr(w_kv_b), T, H, d_nope, d_v, _ptr(out), _ptr(status),
                              _stream(stream)), "mla_absorb_q")
    return out


def mla_v_proj(o_lat, w_kv_b, d_nope: int, d_v: int, out=None, status=None, stream=None):
    """V projection: o_v[t,h,:] = W_UV[h] . o_lat[t,h,:] with W_UV[h] the d_v value rows of head h in the
    kv_b_proj weight.  o_lat [T, H, 512] bf16 -> o_v [T, H, d_v] bf16."""
    T, H, D = o_lat.shape
    _want(o_lat, torch.bfloat16, (T, H, 512), "o_lat")
    _proj_weight(w_kv_b, H, d_nope, d_v, D)
    if out is None:
        out = torch.empty((T, H, d_v), dtype=torch.bfloat16, device=o_lat.device)
    _want(out, torch.bfloat16, (T, H, d_v), "o_v")
    _check(lib().mla_v_proj(_ptr(o_lat), _ptr(w_kv_b), T, H, d_nope, d_v, _ptr(out), _ptr(status),
                            _stream(stream)), "mla_v_proj")
    return out


_HOST_KEYS = ("k", "gate", "ape", "cu_seqlens", "q_idx", "w", "q_lat", "kv_lat", "out", "lse")


def forward_host(host: dict, dev: dict, layout: PoolLayout, p: Params, n_chunks: int = 16, streams=None):
    """Whole forward from (page-locked) host tensors with overlapped copies.

    host: CPU tensors k, gate, ape, cu_seqlens, q_idx, w, q_lat, kv_lat (read) and out, lse (written).
    dev:  CUDA tensors of the same names plus kpool, workspace (uint8) and indices; ``layout`` must be built on
          dev["cu_seqlens"].  streams: (s_in, s_compute, s_out) torch streams (three new ones by default).
    Returns s_compute; the forward (including the copies back) is complete when it is."""
    for name in _HOST_KEYS:
        t = host[name]
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or not t.is_contiguous():
            raise TypeError(f"host[{name!r}] must be a contiguous CPU tensor")
        d = dev[name]
        _want(d, t.dtype, tuple(t.shape), f"dev[{name!r}]")
    for name in ("kpool", "workspace", "indices"):
        if not isinstance(dev[name], torch.Tensor) or dev[name].device.type != "cuda":
            raise TypeError(f"dev[{name!r}] must be a CUDA tensor")
    if dev["cu_seqlens"].data_ptr() != layout.c.cu_seqlens:
        raise ValueError("layout must be built on dev['cu_seqlens']")
    if streams is None:
        streams = tuple(torch.cuda.Stream(device=dev["q_lat"].device) for _ in range(3))
    h = HostIO(*[host[n].data_ptr() for n in _HOST_KEYS])
    d = DevIO(*[dev[n].data_ptr() for n in _HOST_KEYS], dev["kpool"].data_ptr(), ctypes.pointer(layout.c),
              dev["workspace"].data_ptr(), dev["workspace"].numel() * dev["workspace"].element_size(),
              dev["indices"].data_ptr(), dev["indices"].shape[1])
    _check(lib().kpool_forward_host(ctypes.byref(h), ctypes.byref(d), layout.n_docs, layout.T, ctypes.byref(p),
                                    int(n_chunks), _stream(streams[0]), _stream(streams[1]), _stream(streams[2])),
           "kpool_forward_host")
    return streams[1]


def stage_select(scores, pair_base, layout: PoolLayout, topk: int, W=None, indices=None, stream=None):
    W = row_width(topk) if W is None else int(W)
    if indices is None:
        indices = torch.empty((layout.T, W), dtype=torch.int32, device=scores.device)
    _check(lib().kpool_stage_select(_ptr(scores), _ptr(pair_base), ctypes.byref(layout.c), topk, _ptr(indices), W,
                                    _stream(stream)), "kpool_stage_select")
    return indices


def check_status(status, stream=None) -> int:
    """Synchronises the stream and returns the device status word."""
    return int(lib().kpool_check_status(_ptr(status), _stream(stream)))


def set_stage_events(events) -> None:
    """Register 4 torch.cuda.Event(enable_timing=True) objects (or None) for
    the dsa_index stage timing hook."""
    if not events:
        _check(lib().kpool_set_stage_events(None, 0), "kpool_set_stage_events")
        return
    for e in events:            # torch creates the CUDA event on first use
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().kpool_set_stage_events(arr, len(events)), "kpool_set_stage_events")


def version() -> str:
    return lib().kpool_version().decode()
