"""Oracle for paged decode attention: a plain fp64 CPU implementation.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import this package. The CUDA library does not
import, link or call it, and this package imports nothing from the CUDA
library.

The arithmetic lives in ``zl_oracle.c`` (C, binary64, OpenMP over query rows);
this module compiles it with gcc and marshals numpy arrays through ctypes.

Sources for what is computed: "ZhiLight：知乎开源的高性能 LLM 推理加速引擎",
section "4. Tensor Core 上的 Flash Attention" (decode-phase fused batch
attention) and section "技术架构：五层模块化设计" (flash_decoding / flash_mla);
"ZhiLight: Zhihu's CUDA Inference Engine for Llama and DeepSeek on PCIe GPUs",
section "Dual streams, host all-reduce and the memory model" (fused batch
attention for decoding, prefix cache, DeepseekV2 MLA). The formula itself is
the standard scaled-dot-product attention; zl_oracle.c writes it out.

Pins (tests/test_oracle_pins.py): torch's fp64 scaled_dot_product_attention on
gathered dense K/V, scipy's softmax and logsumexp on closed-form one-hot
cases, single-token / constant-V / zero-query closed forms, token permutation,
page remapping, split-and-merge, GQA head mapping, MLA column sharing; the KV
append against a numpy fancy-index gather of the written slots.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "zl_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "libzl_oracle.so")

BAD_PAGE = 1
BAD_LEN = 2

_lock = threading.Lock()
_default = None


def compile_oracle(src: str = SOURCE, out: str = LIB_PATH, extra_flags=()) -> str:
    """Compile ``src`` into a shared library at ``out`` with gcc (portable flags)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        c_int = ctypes.c_int
        lib.zl_oracle_decode_attn.restype = c_int
        lib.zl_oracle_decode_attn.argtypes = [
            u16p, u16p, u16p, i64, i64, i64, i32p, i64, i32p,
            c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
            ctypes.c_double, f64p, f64p, c_int]
        lib.zl_oracle_attend_range.restype = c_int
        lib.zl_oracle_attend_range.argtypes = [
            u16p, u16p, u16p, i64, i64, i64, i32p, c_int, c_int, c_int, c_int, c_int,
            ctypes.c_double, i64, i64, f64p, f64p, f64p]
        lib.zl_oracle_lse_merge.restype = None
        lib.zl_oracle_lse_merge.argtypes = [f64p, f64p, c_int, c_int, f64p, f64p]
        lib.zl_oracle_kv_append.restype = c_int
        lib.zl_oracle_kv_append.argtypes = [
            u16p, u16p, u16p, u16p, i64, i64, i64, i32p, i64, i32p,
            c_int, c_int, c_int, c_int, c_int, c_int, c_int]
        lib.zl_oracle_max_threads.restype = c_int
        lib.zl_oracle_max_threads.argtypes = []
        self._lib = lib

    def max_threads(self) -> int:
        return int(self._lib.zl_oracle_max_threads())

    def decode_attn(self, q, k_pool, v_pool, strides, block_table, seq_lens, *, Hkv, page_size,
                    num_pages, scale, D_v=None, num_threads=0):
        """Batched paged decode attention in fp64.

        q           uint16 (bf16 bits) [B, q_len, Hq, D_qk]
        k_pool      uint16 buffer; row (page, slot, head) starts at
                    page*strides[0] + slot*strides[1] + head*strides[2]
        v_pool      like k_pool, or None for MLA (V = first D_v columns of K)
        block_table int32 [B, max_pages]
        seq_lens    int32 [B]
        Returns (out fp64 [B, q_len, Hq, D_v], lse fp64 [B, q_len, Hq], status bits).
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        B, q_len, Hq, D_qk = q.shape
        D_v = D_qk if D_v is None else D_v
        k_pool = np.ascontiguousarray(k_pool).view(np.uint16)
        v_arr = None if v_pool is None else np.ascontiguousarray(v_pool).view(np.uint16)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        assert bt.ndim == 2 and bt.shape[0] == B and sl.shape == (B,)
        out = np.zeros((B, q_len, Hq, D_v), dtype=np.float64)
        lse = np.zeros((B, q_len, Hq), dtype=np.float64)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        st = self._lib.zl_oracle_decode_attn(
            _ptr(q, ctypes.c_uint16), _ptr(k_pool, ctypes.c_uint16),
            _ptr(v_arr, ctypes.c_uint16) if v_arr is not None else ctypes.cast(None, u16p),
            int(strides[0]), int(strides[1]), int(strides[2]),
            _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32),
            B, q_len, Hq, int(Hkv), D_qk, int(D_v), int(page_size), int(num_pages),
            float(scale), _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
            int(num_threads))
        return out, lse, int(st)

    def attend_range(self, q_row, k_pool, v_pool, strides, bt_row, *, kh, page_size, num_pages,
                     scale, t_begin, t_end, D_v=None, want_weights=False):
        """One query row over tokens [t_begin, t_end) of one sequence.

        Returns (out fp64 [D_v], lse, weights or None, status).
        """
        q_row = np.ascontiguousarray(q_row, dtype=np.uint16).reshape(-1)
        D_qk = q_row.shape[0]
        D_v = D_qk if D_v is None else D_v
        k_pool = np.ascontiguousarray(k_pool).view(np.uint16)
        v_arr = None if v_pool is None else np.ascontiguousarray(v_pool).view(np.uint16)
        bt_row = np.ascontiguousarray(bt_row, dtype=np.int32)
        out = np.zeros(D_v, dtype=np.float64)
        lse = np.zeros(1, dtype=np.float64)
        n = max(int(t_end) - int(t_begin), 0)
        w = np.zeros(max(n, 1), dtype=np.float64) if want_weights else None
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        st = self._lib.zl_oracle_attend_range(
            _ptr(q_row, ctypes.c_uint16), _ptr(k_pool, ctypes.c_uint16),
            _ptr(v_arr, ctypes.c_uint16) if v_arr is not None else ctypes.cast(None, u16p),
            int(strides[0]), int(strides[1]), int(strides[2]), _ptr(bt_row, ctypes.c_int32),
            int(kh), D_qk, int(D_v), int(page_size), int(num_pages), float(scale),
            int(t_begin), int(t_end), _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
            _ptr(w, ctypes.c_double) if w is not None else ctypes.cast(None, f64p))
        return out, float(lse[0]), (w[:n] if w is not None else None), int(st)

    def kv_append(self, k_new, v_new, k_pool, v_pool, strides, block_table, seq_lens, *,
                  page_size, num_pages):
        """Write the new tokens into copies of the pools; returns (k_pool', v_pool', status).

        k_new  uint16 [B, q_len, Hkv, D_k]; v_new uint16 [B, q_len, Hkv, D_v] or None (MLA)
        k_pool, v_pool  uint16 pools (any shape; strides in elements as for decode_attn);
                        v_pool None for MLA. The inputs are not modified.
        """
        k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
        B, q_len, Hkv, D_k = k_new.shape
        v_new = None if v_new is None else np.ascontiguousarray(v_new, dtype=np.uint16)
        D_v = D_k if v_new is None else v_new.shape[3]
        k_out = np.array(np.asarray(k_pool).view(np.uint16), copy=True, order="C")
        v_out = None if v_pool is None else np.array(np.asarray(v_pool).view(np.uint16),
                                                     copy=True, order="C")
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        assert bt.ndim == 2 and bt.shape[0] == B and sl.shape == (B,)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        none = ctypes.cast(None, u16p)
        st = self._lib.zl_oracle_kv_append(
            _ptr(k_new, ctypes.c_uint16), _ptr(v_new, ctypes.c_uint16) if v_new is not None else none,
            _ptr(k_out, ctypes.c_uint16), _ptr(v_out, ctypes.c_uint16) if v_out is not None else none,
            int(strides[0]), int(strides[1]), int(strides[2]), _ptr(bt, ctypes.c_int32),
            bt.shape[1], _ptr(sl, ctypes.c_int32), B, q_len, Hkv, D_k, int(D_v), int(page_size),
            int(num_pages))
        return k_out, v_out, int(st)

    def lse_merge(self, parts, lses):
        """Merge S normalised partials ``parts`` [S, D] with their ``lses`` [S]."""
        parts = np.ascontiguousarray(parts, dtype=np.float64)
        lses = np.ascontiguousarray(lses, dtype=np.float64)
        S, D = parts.shape
        out = np.zeros(D, dtype=np.float64)
        lse = np.zeros(1, dtype=np.float64)
        self._lib.zl_oracle_lse_merge(_ptr(parts, ctypes.c_double), _ptr(lses, ctypes.c_double),
                                      S, D, _ptr(out, ctypes.c_double),
                                      _ptr(lse, ctypes.c_double))
        return out, float(lse[0])


def build() -> str:
    """Compile the oracle library in-tree (under oracle/_build/)."""
    with _lock:
        return compile_oracle()


def load(lib_path: str | None = None) -> Oracle:
    """Return the oracle, compiling it first if it is missing or stale."""
    global _default
    if lib_path is not None:
        return Oracle(lib_path)
    with _lock:
        if _default is None:
            stale = (not os.path.exists(LIB_PATH)
                     or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE))
            if stale:
                compile_oracle()
            _default = Oracle(LIB_PATH)
        return _default
