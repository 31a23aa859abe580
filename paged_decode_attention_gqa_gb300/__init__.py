"""Paged decode attention for GB300: Python binding of libzl_decode_attn.so.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library (declared in include/zl_decode_attn.h). There is no CPU
or PyTorch fallback; if the library is missing or fails to load, every call
raises.

    import paged_decode_attention_gqa_gb300 as zl
    out = zl.decode_attn(q, k_pool, v_pool, block_table, seq_lens,
                         page_size=16, scale=128 ** -0.5)

Tensors are torch CUDA tensors (PyTorch provides device memory and streams).
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from ._build import LIB_PATH, build  # noqa: F401  (build() is the public build step)

__all__ = [
    "ZlError", "Params", "AppendParams", "lib", "decode_attn", "decode_attn_mla", "kv_append",
    "workspace_size", "workspace_size_mla", "call", "call_noalloc", "build", "LIB_PATH",
    "DEVERR_BAD_PAGE", "DEVERR_BAD_SEQ_LEN", "DEVERR_TIMEOUT", "HEADER", "declared_symbols",
]

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "zl_decode_attn.h")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = range(5)
SINGLE_LAUNCH = 1  # ZL_DECODE_SINGLE_LAUNCH
TEST_STALL = 0x80000000  # ZL_DECODE_TEST_STALL (failure-detection test hook)
DEVERR_BAD_PAGE, DEVERR_BAD_SEQ_LEN, DEVERR_TIMEOUT, DEVERR_BAD_PREFIX = 1, 2, 4, 8
NOALLOC_WORKSPACE_BYTES = 8 << 20  # ZL_NOALLOC_WORKSPACE_BYTES


class ZlError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (zl_status {status})")
        self.status = status


class Params(ctypes.Structure):
    """Mirror of zl_decode_attn_params."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("q", ctypes.c_void_p),
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("page_stride", ctypes.c_int64),
        ("token_stride", ctypes.c_int64),
        ("head_stride", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
        ("block_table_stride", ctypes.c_int64),
        ("seq_lens", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("D_qk", ctypes.c_int32),
        ("D_v", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("err_flags", ctypes.c_void_p),
        ("num_ctas", ctypes.c_int32),
        ("attn_begin", ctypes.c_void_p),
        ("attn_end", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
        ("shared_prefix_pages", ctypes.c_int32),
        ("k_new", ctypes.c_void_p),
        ("v_new", ctypes.c_void_p),
    ]


class AppendParams(ctypes.Structure):
    """Mirror of zl_kv_append_params."""
    _fields_ = [
        ("struct_size", ctypes.c_size_t),
        ("k_new", ctypes.c_void_p),
        ("v_new", ctypes.c_void_p),
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("page_stride", ctypes.c_int64),
        ("token_stride", ctypes.c_int64),
        ("head_stride", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
        ("block_table_stride", ctypes.c_int64),
        ("seq_lens", ctypes.c_void_p),
        ("B", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("D_k", ctypes.c_int32),
        ("D_v", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("err_flags", ctypes.c_void_p),
    ]


_lib = None
_lib_lock = threading.Lock()


def lib():
    """The loaded library (built first if missing or stale). Raises on failure."""
    global _lib
    with _lib_lock:
        if _lib is None:
            try:
                path = build()
                handle = ctypes.CDLL(path)
            except Exception as e:  # no fallback: the CUDA path is the product
                raise RuntimeError(f"libzl_decode_attn could not be built or loaded: {e}") from e
            P = ctypes.POINTER(Params)
            for name in ("zl_decode_attn", "zl_decode_attn_mla", "zl_decode_attn_noalloc"):
                fn = getattr(handle, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [P, ctypes.c_void_p]
            for name in ("zl_decode_attn_workspace_size", "zl_decode_attn_mla_workspace_size"):
                fn = getattr(handle, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
            handle.zl_decode_attn_launches.restype = ctypes.c_int
            handle.zl_decode_attn_launches.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
            handle.zl_kv_append.restype = ctypes.c_int
            handle.zl_kv_append.argtypes = [ctypes.POINTER(AppendParams), ctypes.c_void_p]
            handle.zl_status_string.restype = ctypes.c_char_p
            handle.zl_status_string.argtypes = [ctypes.c_int]
            _lib = handle
        return _lib


def declared_symbols(header: str = HEADER):
    """Function names the public header declares."""
    text = open(header).read()
    return sorted(set(re.findall(r"^\s*(?:zl_status|const char\*)\s+(zl_\w+)\s*\(", text, re.M)))


def _check(status: int, what: str):
    if status != OK:
        raise ZlError(status, f"{what}: {lib().zl_status_string(status).decode()}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _pool_strides(pool: torch.Tensor, layout: str):
    """(page, token, head) element strides of a 4-D pool in NHD or HND layout."""
    if pool.dim() != 4:
        raise ValueError("pools are 4-D: [pages, slot, head, dim] (NHD) or [pages, head, slot, dim]")
    s = pool.stride()
    if layout == "NHD":
        return s[0], s[1], s[2]
    if layout == "HND":
        return s[0], s[2], s[1]
    raise ValueError(f"unknown layout {layout!r}")


def make_params(q, k_pool, v_pool, block_table, seq_lens, out, *, page_size, scale, Hkv,
                D_v, lse=None, workspace=None, err_flags=None, num_ctas=0, max_seq_len=0,
                layout="NHD", events=None, single_launch=False,
                shared_prefix_pages=0, k_new=None, v_new=None) -> Params:
    """k_new / v_new: the fused KV append (the new tokens' K and V rows, bf16
    [B, q_len, Hkv, D]; MLA: the latent rows in k_new, v_new None); the call
    then stores them in their page slots before attending."""
    B, q_len, Hq, D_qk = q.shape
    ps, ts, hs = _pool_strides(k_pool, layout)
    if v_pool is not None and _pool_strides(v_pool, layout) != (ps, ts, hs):
        raise ValueError("K and V pools must share strides")
    if k_pool.stride(3) != 1 or not q.is_contiguous() or not out.is_contiguous():
        raise ValueError("q, out and the pool rows must be contiguous")
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    p = Params()
    p.struct_size = ctypes.sizeof(Params)
    p.q, p.k_pool, p.v_pool = _ptr(q), _ptr(k_pool), _ptr(v_pool)
    p.page_stride, p.token_stride, p.head_stride = ps, ts, hs
    p.block_table = _ptr(block_table)
    p.block_table_stride = block_table.stride(0)
    p.seq_lens = _ptr(seq_lens)
    p.out, p.lse = _ptr(out), _ptr(lse)
    p.B, p.q_len, p.Hq, p.Hkv, p.D_qk, p.D_v = B, q_len, Hq, Hkv, D_qk, D_v
    p.page_size = page_size
    p.num_pages = k_pool.shape[0]
    p.max_seq_len = int(max_seq_len)
    p.scale = float(scale)
    if workspace is not None:
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    p.err_flags = _ptr(err_flags)
    p.num_ctas = int(num_ctas)
    p.flags = SINGLE_LAUNCH if single_launch else 0
    p.shared_prefix_pages = int(shared_prefix_pages)
    for t in (k_new, v_new):
        if t is not None and not t.is_contiguous():
            raise ValueError("k_new and v_new must be contiguous")
    p.k_new, p.v_new = _ptr(k_new), _ptr(v_new)
    if events is not None:
        p.attn_begin, p.attn_end = events[0].cuda_event, events[1].cuda_event
    # The struct holds raw device pointers: keep the tensors alive with it.
    p.tensors = (q, k_pool, v_pool, block_table, seq_lens, out, lse, workspace, err_flags, events,
                 k_new, v_new)
    return p


def workspace_size(params: Params) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().zl_decode_attn_workspace_size(ctypes.byref(params), ctypes.byref(n)),
           "zl_decode_attn_workspace_size")
    return n.value


def workspace_size_mla(params: Params) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().zl_decode_attn_mla_workspace_size(ctypes.byref(params), ctypes.byref(n)),
           "zl_decode_attn_mla_workspace_size")
    return n.value


_ws_cache: dict = {}


def _workspace(device, nbytes, kind, counters=0):
    """A cached device byte buffer of at least nbytes per (device, kind).

    ``counters``: the call needs that many leading bytes at zero (the arrival
    counters of a single-launch GQA call). They are zeroed again whenever the
    previous user of the buffer may have written there: a call of another
    shape (its partials may sit where this call counts) or a fresh buffer.
    Calls of one shape leave the counters at zero themselves."""
    key = (device.type, device.index, kind)
    buf, last = _ws_cache.get(key, (None, None))
    if buf is None or buf.numel() < nbytes:
        buf, last = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device), None
    if counters and last != (nbytes, counters):
        buf[:counters].zero_()
    _ws_cache[key] = (buf, (nbytes, counters) if counters else None)
    return buf


def launches(params: Params) -> int:
    """Kernel launches one zl_decode_attn call with these params enqueues."""
    n = ctypes.c_int32(0)
    _check(lib().zl_decode_attn_launches(ctypes.byref(params), ctypes.byref(n)),
           "zl_decode_attn_launches")
    return int(n.value)


def call_noalloc(params: Params, stream=None):
    """zl_decode_attn_noalloc: the library's own static scratch, no workspace
    argument and no allocation (see the header for its limits)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    _check(lib().zl_decode_attn_noalloc(ctypes.byref(params), ctypes.c_void_p(stream.cuda_stream)),
           "zl_decode_attn_noalloc")


def call(params: Params, *, mla: bool, stream=None):
    """Invoke the entry point on ``stream`` (default: torch's current stream)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    fn = lib().zl_decode_attn_mla if mla else lib().zl_decode_attn
    _check(fn(ctypes.byref(params), ctypes.c_void_p(stream.cuda_stream)),
           "zl_decode_attn_mla" if mla else "zl_decode_attn")


def _run(q, k_pool, v_pool, block_table, seq_lens, *, mla, page_size, scale, Hkv, D_v, out, lse,
         workspace, err_flags, num_ctas, max_seq_len, layout, stream, events, single_launch=False,
         shared_prefix_pages=0, k_new=None, v_new=None):
    if out is None:
        out = torch.empty(q.shape[:3] + (D_v,), dtype=torch.bfloat16, device=q.device)
    p = make_params(q, k_pool, v_pool, block_table, seq_lens, out, page_size=page_size,
                    scale=scale, Hkv=Hkv, D_v=D_v, lse=lse, err_flags=err_flags,
                    num_ctas=num_ctas, max_seq_len=max_seq_len, layout=layout, events=events,
                    single_launch=single_launch, shared_prefix_pages=shared_prefix_pages,
                    k_new=k_new, v_new=v_new)
    need = workspace_size_mla(p) if mla else workspace_size(p)
    if workspace is None:
        counters = 8 * q.shape[0] * Hkv if single_launch else 0
        workspace = _workspace(q.device, need,
                               "mla" if mla else ("gqa1" if single_launch else "gqa"), counters)
    p.workspace = workspace.data_ptr()
    p.workspace_bytes = workspace.numel() * workspace.element_size()
    call(p, mla=mla, stream=stream)
    return out


def decode_attn(q, k_pool, v_pool, block_table, seq_lens, *, page_size, scale, out=None, lse=None,
                workspace=None, err_flags=None, num_ctas=0, max_seq_len=0, layout="NHD",
                stream=None, events=None, single_launch=False, shared_prefix_pages=0,
                k_new=None, v_new=None):
    """GQA/MHA/MQA paged decode attention (zl_decode_attn).

    q [B, q_len, Hq, 128] bf16; k_pool, v_pool [pages, page_size, Hkv, 128]
    (layout "NHD") or [pages, Hkv, page_size, 128] ("HND") bf16; block_table
    int32 [B, max_pages]; seq_lens int32 [B]. Returns out [B, q_len, Hq, 128]
    bf16. single_launch: merge split-KV partials inside the attention kernel
    (ZL_DECODE_SINGLE_LAUNCH; a caller's workspace must then hold zeroed
    arrival counters, see the header; the default cached one is kept so).
    shared_prefix_pages: the first pages of every block-table row are the same
    shared prefix (read once per group of sequences; see the header).
    k_new, v_new: the q_len new tokens' K and V rows [B, q_len, Hkv, 128] bf16;
    the call stores them in their page slots (as kv_append does) and then
    attends, in the same launch.
    """
    Hkv = k_pool.shape[2] if layout == "NHD" else k_pool.shape[1]
    return _run(q, k_pool, v_pool, block_table, seq_lens, mla=False, page_size=page_size,
                scale=scale, Hkv=Hkv, D_v=q.shape[3], out=out, lse=lse, workspace=workspace,
                err_flags=err_flags, num_ctas=num_ctas, max_seq_len=max_seq_len, layout=layout,
                stream=stream, events=events, single_launch=single_launch,
                shared_prefix_pages=shared_prefix_pages, k_new=k_new, v_new=v_new)


def decode_attn_mla(q, kv_pool, block_table, seq_lens, *, page_size, scale, D_v=512, out=None,
                    lse=None, workspace=None, err_flags=None, num_ctas=0, max_seq_len=0,
                    stream=None, events=None, kv_new=None):
    """Absorbed MLA paged decode (zl_decode_attn_mla).

    q [B, q_len, Hq, 576] bf16; kv_pool [pages, page_size, 1, 576] bf16 (V =
    first D_v columns). Returns out [B, q_len, Hq, D_v] bf16. kv_new: the new
    tokens' latent rows [B, q_len, 1, 576] bf16, stored in their page slots by
    the same launch before it attends.
    """
    return _run(q, kv_pool, None, block_table, seq_lens, mla=True, page_size=page_size,
                scale=scale, Hkv=1, D_v=D_v, out=out, lse=lse, workspace=workspace,
                err_flags=err_flags, num_ctas=num_ctas, max_seq_len=max_seq_len, layout="NHD",
                stream=stream, events=events, k_new=kv_new)


def make_append_params(k_new, v_new, k_pool, v_pool, block_table, seq_lens, *, page_size,
                       layout="NHD", err_flags=None) -> AppendParams:
    B, q_len, Hkv, D_k = k_new.shape
    ps, ts, hs = _pool_strides(k_pool, layout)
    if (v_pool is None) != (v_new is None):
        raise ValueError("v_new and v_pool are given together (both None for a latent-only pool)")
    if v_pool is not None and _pool_strides(v_pool, layout) != (ps, ts, hs):
        raise ValueError("K and V pools must share strides")
    if not k_new.is_contiguous() or (v_new is not None and not v_new.is_contiguous()):
        raise ValueError("k_new and v_new must be contiguous")
    if k_pool.stride(3) != 1 or block_table.stride(1) != 1:
        raise ValueError("pool rows and block_table rows must be contiguous")
    p = AppendParams()
    p.struct_size = ctypes.sizeof(AppendParams)
    p.k_new, p.v_new, p.k_pool, p.v_pool = _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool)
    p.page_stride, p.token_stride, p.head_stride = ps, ts, hs
    p.block_table = _ptr(block_table)
    p.block_table_stride = block_table.stride(0)
    p.seq_lens = _ptr(seq_lens)
    p.B, p.q_len, p.Hkv, p.D_k = B, q_len, Hkv, D_k
    p.D_v = 0 if v_new is None else v_new.shape[3]
    p.page_size = page_size
    p.num_pages = k_pool.shape[0]
    p.err_flags = _ptr(err_flags)
    p.tensors = (k_new, v_new, k_pool, v_pool, block_table, seq_lens, err_flags)
    return p


def kv_append(k_new, v_new, k_pool, v_pool, block_table, seq_lens, *, page_size, layout="NHD",
              err_flags=None, stream=None):
    """Paged KV append (zl_kv_append): new token i of sequence b goes to logical
    position seq_lens[b] - q_len + i of its cache, in place.

    k_new [B, q_len, Hkv, D_k] bf16, v_new [B, q_len, Hkv, D_v] bf16 or None
    (latent-only pool, v_pool None); pools, block_table and seq_lens as for
    decode_attn (seq_lens count the new tokens).
    """
    p = make_append_params(k_new, v_new, k_pool, v_pool, block_table, seq_lens,
                           page_size=page_size, layout=layout, err_flags=err_flags)
    if stream is None:
        stream = torch.cuda.current_stream()
    _check(lib().zl_kv_append(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream)),
           "zl_kv_append")
