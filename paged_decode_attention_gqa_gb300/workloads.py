"""Seeded synthetic inputs for paged decode attention.

This module only makes inputs: sequence lengths, page placement, block tables,
bf16 values and NaN poison. It holds none of the attention arithmetic, so both
the CUDA path and the CPU oracle can consume what it makes without sharing any
computation.

Recipe (the same for every workload):
  * Structure (lengths, page placement, channel choice) comes from numpy PCG64
    seeded with ``SeedSequence(seed, spawn_key=(0,))``, drawn in the order
    lengths -> page placement -> extra choices.
  * Values are N(0, 1) float32 drawn in chunks of ``_CHUNK`` values; chunk c of
    tensor k (1 = Q, 2 = K pool, 3 = V pool) uses PCG64 seeded with
    ``SeedSequence(seed, spawn_key=(k, c))``, so the bits do not depend on the
    thread count. Pools are drawn in the canonical [page, slot, head, dim]
    order; the HND layout is a permutation of the same values.
  * float32 -> bf16 is round-to-nearest-even (torch ``.to(torch.bfloat16)``).
  * Pool pages no block table references, and the slots past the last token of
    each sequence's last page, hold NaN (bf16 0x7FC0), so any read of them
    shows up in the output.
  * Block-table entries past a sequence's last page are -1.

Workloads are named after what they model; ``WORKLOADS`` lists them.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_CHUNK = 1 << 22
BF16_NAN = 0x7FC0


@dataclass
class Workload:
    name: str
    seed: int
    B: int
    q_len: int
    Hq: int
    Hkv: int
    D_qk: int
    D_v: int
    page_size: int
    num_pages: int
    scale: float
    layout: str                  # "NHD": [page, slot, head, dim]; "HND": [page, head, slot, dim]
    seq_lens: np.ndarray         # int32 [B]
    block_table: np.ndarray      # int32 [B, max_pages]
    q: torch.Tensor              # bf16 [B, q_len, Hq, D_qk]
    k_pool: torch.Tensor         # bf16, layout above
    v_pool: torch.Tensor | None  # bf16, same layout; None for MLA (V = first D_v cols of K)
    notes: dict = field(default_factory=dict)
    mla: bool = False            # V is the first D_v columns of the K (latent) row

    @property
    def strides(self):
        """(page, token, head) strides of the pools, in elements."""
        P, H, D = self.page_size, self.Hkv, self.D_qk
        if self.layout == "NHD":
            return (P * H * D, H * D, D)
        return (H * P * D, D, P * D)

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    def to(self, device) -> "Workload":
        """A copy whose tensors live on ``device`` (structure stays in numpy)."""
        w = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        w.q = self.q.to(device)
        w.k_pool = self.k_pool.to(device)
        w.v_pool = None if self.v_pool is None else self.v_pool.to(device)
        return w

    @staticmethod
    def bits(t: torch.Tensor) -> np.ndarray:
        """bf16 tensor -> numpy uint16 bits (host copy)."""
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal_bf16(seed: int, key: int, shape, scale_channels=None, factor=8.0) -> torch.Tensor:
    """N(0,1) float32 values in ``shape`` (chunked, per-chunk seeds) rounded to bf16.

    ``scale_channels``: indices along the last axis multiplied by ``factor``
    in float32 before rounding.
    """
    n = int(np.prod(shape))
    flat = torch.empty(n, dtype=torch.bfloat16)
    last = shape[-1]
    nchunks = (n + _CHUNK - 1) // _CHUNK
    if scale_channels is not None:
        assert _CHUNK % last == 0
        scale_channels = np.asarray(scale_channels)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(key, c))))
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        if scale_channels is not None:
            x = x.reshape(-1, last)
            x[:, scale_channels] *= np.float32(factor)
            x = x.reshape(-1)
        flat[lo:hi] = torch.from_numpy(x).to(torch.bfloat16)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(nchunks)))
    return flat.view(*shape)


def new_token_rows(seed: int, B: int, q_len: int, Hkv: int, D_k: int, D_v: int | None = None):
    """The new tokens' K and V rows for a KV append, bf16 N(0,1):
    k_new [B, q_len, Hkv, D_k] and v_new [B, q_len, Hkv, D_v] (None when D_v is None)."""
    k_new = _normal_bf16(seed, 11, (B, q_len, Hkv, D_k))
    v_new = None if D_v is None else _normal_bf16(seed, 12, (B, q_len, Hkv, D_v))
    return k_new, v_new


def _poison_pool(pool_nhd: torch.Tensor, used_pages: np.ndarray, tails) -> None:
    """NaN into unreferenced pages and tail slots (pool in [page, slot, head, dim])."""
    nan = torch.tensor(BF16_NAN, dtype=torch.int16).view(torch.bfloat16)
    unused = np.setdiff1d(np.arange(pool_nhd.shape[0]), used_pages)
    if unused.size:
        pool_nhd[torch.from_numpy(unused)] = nan
    for page, first_dead_slot in tails:
        pool_nhd[page, first_dead_slot:] = nan


def build_workload(name, seed, *, B, Hq, Hkv, D_qk, page_size, seq_lens, block_table, num_pages,
                   scale, D_v=None, q_len=1, mla=False, layout="NHD", k_scale_channels=None,
                   poison=True, notes=None, values=True) -> Workload:
    """Draw the values for a workload whose structure is already fixed.

    ``values=False`` returns the structure only (tensors left as None).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    block_table = np.asarray(block_table, dtype=np.int32)
    D_v = D_qk if D_v is None else D_v
    P = page_size
    if not values:
        return Workload(name=name, seed=seed, B=B, q_len=q_len, Hq=Hq, Hkv=Hkv, D_qk=D_qk,
                        D_v=D_v, page_size=P, num_pages=num_pages, scale=float(scale),
                        layout=layout, seq_lens=seq_lens, block_table=block_table, q=None,
                        k_pool=None, v_pool=None, notes=dict(notes or {}), mla=mla)
    q = _normal_bf16(seed, 1, (B, q_len, Hq, D_qk))
    k = _normal_bf16(seed, 2, (num_pages, P, Hkv, D_qk), k_scale_channels)
    v = None if mla else _normal_bf16(seed, 3, (num_pages, P, Hkv, D_qk))
    if poison:
        used, tails = [], []
        for b in range(B):
            L = int(seq_lens[b])
            npg = (L + P - 1) // P
            used.extend(block_table[b, :npg].tolist())
            if L % P:
                tails.append((int(block_table[b, npg - 1]), L % P))
        used = np.unique(np.asarray(used, dtype=np.int64))
        _poison_pool(k, used, tails)
        if v is not None:
            _poison_pool(v, used, tails)
    if layout == "HND":
        k = k.permute(0, 2, 1, 3).contiguous()
        v = None if v is None else v.permute(0, 2, 1, 3).contiguous()
    else:
        assert layout == "NHD"
    return Workload(name=name, seed=seed, B=B, q_len=q_len, Hq=Hq, Hkv=Hkv, D_qk=D_qk, D_v=D_v,
                    page_size=P, num_pages=num_pages, scale=float(scale), layout=layout,
                    seq_lens=seq_lens, block_table=block_table, q=q, k_pool=k, v_pool=v,
                    notes=dict(notes or {}), mla=mla)


def _structure_rng(seed):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(0,))))


def place_pages(rng, seq_lens, page_size, num_pages, shared_prefix_pages=0):
    """Block tables over a randomly permuted pool.

    Pages are taken in order from one seeded permutation of the pool: first the
    shared prefix pages (the same ids in every table), then each sequence's
    private pages, sequence by sequence.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = seq_lens.shape[0]
    npg = (seq_lens + page_size - 1) // page_size
    max_pages = int(npg.max()) if B else 0
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
    prefix = perm[:shared_prefix_pages]
    pos = shared_prefix_pages
    for b in range(B):
        table[b, :shared_prefix_pages] = prefix
        own = int(npg[b]) - shared_prefix_pages
        table[b, shared_prefix_pages:npg[b]] = perm[pos:pos + own]
        pos += own
    assert pos <= num_pages
    return table


def _pool_for(pages_needed, factor=1.25):
    return int(math.ceil(pages_needed * factor))


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def tiny_gqa(seed=1001, layout="NHD", poison=True, values=True) -> Workload:
    """4 seqs, 8 query / 2 KV heads, D 128, lengths {17,64,100,256}, page 16,
    64-page pool, pages taken from a seeded permutation, the rest NaN."""
    rng = _structure_rng(seed)
    lens = np.array([17, 64, 100, 256], dtype=np.int32)
    table = place_pages(rng, lens, 16, 64)
    return build_workload("tiny_gqa", seed, B=4, Hq=8, Hkv=2, D_qk=128, page_size=16,
                          seq_lens=lens, block_table=table, num_pages=64,
                          scale=1.0 / math.sqrt(128), layout=layout, poison=poison, values=values)


def llama3_8b_decode(seed=1002, layout="NHD", poison=True, B=64, values=True,
                     q_len=1) -> Workload:
    """Llama-3-8B attention shape: 64 seqs, 32 query / 8 KV heads, D 128,
    lengths U[512, 4096], page 16, pool 1.25x, 4 of 128 K channels scaled x8.
    q_len > 1: that many new query tokens per sequence (speculative decode)."""
    rng = _structure_rng(seed)
    lens = rng.integers(512, 4096, size=B, endpoint=True).astype(np.int32)
    pages = int(((lens + 15) // 16).sum())
    num_pages = _pool_for(pages)
    table = place_pages(rng, lens, 16, num_pages)
    channels = np.sort(rng.choice(128, 4, replace=False))
    return build_workload("llama3_8b_decode", seed, B=B, Hq=32, Hkv=8, D_qk=128, page_size=16,
                          seq_lens=lens, block_table=table, num_pages=num_pages,
                          scale=1.0 / math.sqrt(128), layout=layout, k_scale_channels=channels,
                          poison=poison, notes={"k_scaled_channels": channels.tolist()},
                          values=values, q_len=q_len)


def mqa32_decode(seed=1006, layout="NHD", poison=True, B=64, values=True,
                 q_len=1) -> Workload:
    """Many-head multi-query attention: the Llama-3-8B lengths (64 seqs,
    U[512, 4096], page 16, pool 1.25x) with 32 query heads on one KV head, D
    128 -- more than 16 heads per KV head, so two row groups of 16."""
    rng = _structure_rng(seed)
    lens = rng.integers(512, 4096, size=B, endpoint=True).astype(np.int32)
    pages = int(((lens + 15) // 16).sum())
    num_pages = _pool_for(pages)
    table = place_pages(rng, lens, 16, num_pages)
    return build_workload("mqa32_decode", seed, B=B, Hq=32, Hkv=1, D_qk=128, page_size=16,
                          seq_lens=lens, block_table=table, num_pages=num_pages,
                          scale=1.0 / math.sqrt(128), layout=layout, poison=poison,
                          values=values, q_len=q_len)


def llama70b_prefix_decode(seed=1003, layout="NHD", poison=True, sigma=1.0, values=True,
                           B=128) -> Workload:
    """70B attention shape with prefix sharing: 128 seqs, 64 query / 8 KV heads,
    D 128, page 16; a 2048-token prefix on the same physical pages in every
    table plus a private lognormal suffix (median 300, sigma 1, cap 6144). (A
    smaller B takes the first B suffixes of the same draw; for profiling.)"""
    rng = _structure_rng(seed)
    prefix = 2048
    z = rng.standard_normal(128)[:B]
    suffix = np.clip(np.rint(np.exp(math.log(300.0) + sigma * z)), 1, 6144).astype(np.int64)
    lens = (prefix + suffix).astype(np.int32)
    pfx_pages = prefix // 16
    unique = pfx_pages + int(((suffix + 15) // 16).sum())
    num_pages = _pool_for(unique)
    table = place_pages(rng, lens, 16, num_pages, shared_prefix_pages=pfx_pages)
    return build_workload("llama70b_prefix_decode", seed, B=B, Hq=64, Hkv=8, D_qk=128,
                          page_size=16, seq_lens=lens, block_table=table, num_pages=num_pages,
                          scale=1.0 / math.sqrt(128), layout=layout, poison=poison,
                          notes={"shared_prefix_tokens": prefix, "unique_pages": unique},
                          values=values)


def long_context_decode(seed=1004, layout="NHD", poison=True, values=True, B=8) -> Workload:
    """Long contexts: 8 seqs, 32 query / 8 KV heads, D 128, lengths
    U[32768, 131072], page 64, random placement, pool 1.25x. (A smaller B takes
    the first B lengths of the same draw; used for profiling captures.)"""
    rng = _structure_rng(seed)
    lens = rng.integers(32768, 131072, size=8, endpoint=True).astype(np.int32)[:B]
    pages = int(((lens + 63) // 64).sum())
    num_pages = _pool_for(pages)
    table = place_pages(rng, lens, 64, num_pages)
    return build_workload("long_context_decode", seed, B=B, Hq=32, Hkv=8, D_qk=128,
                          page_size=64, seq_lens=lens, block_table=table, num_pages=num_pages,
                          scale=1.0 / math.sqrt(128), layout=layout, poison=poison, values=values)


def mla_decode(seed=1005, poison=True, B=64, values=True, q_len=1) -> Workload:
    """Absorbed MLA (DeepSeek-V3 shape): 64 seqs, 128 query heads over one
    latent KV row of 512 + 64 rope (QK over 576, V = the 512 latent), lengths
    U[1024, 8192], page 64, random pages, scale 1/sqrt(192). q_len > 1: that
    many new query tokens per sequence (multi-token prediction)."""
    rng = _structure_rng(seed)
    lens = rng.integers(1024, 8192, size=B, endpoint=True).astype(np.int32)
    pages = int(((lens + 63) // 64).sum())
    num_pages = _pool_for(pages)
    table = place_pages(rng, lens, 64, num_pages)
    return build_workload("mla_decode", seed, B=B, Hq=128, Hkv=1, D_qk=576, D_v=512,
                          page_size=64, seq_lens=lens, block_table=table, num_pages=num_pages,
                          scale=1.0 / math.sqrt(192), mla=True, poison=poison, values=values,
                          q_len=q_len)


WORKLOADS = {
    "tiny_gqa": tiny_gqa,
    "llama3_8b_decode": llama3_8b_decode,
    "llama70b_prefix_decode": llama70b_prefix_decode,
    "long_context_decode": long_context_decode,
    "mla_decode": mla_decode,
    "mqa32_decode": mqa32_decode,
}


def random_case(seed, *, B, Hq, Hkv, D=128, page_size=16, lens=None, max_len=300, layout="NHD",
                pool_factor=1.5, poison=True, q_len=1, mla=False, D_v=None, scale=None,
                shared_prefix_pages=0, values=True) -> Workload:
    """A small randomized case for parity sweeps (explicit or random lengths)."""
    rng = _structure_rng(seed)
    if lens is None:
        lens = rng.integers(1, max_len, size=B, endpoint=True)
    lens = np.asarray(lens, dtype=np.int32)
    assert lens.shape == (B,)
    own = np.maximum((lens.astype(np.int64) + page_size - 1) // page_size - shared_prefix_pages, 0)
    pages = int(own.sum()) + shared_prefix_pages
    num_pages = max(1, _pool_for(pages, pool_factor))
    table = place_pages(rng, lens, page_size, num_pages, shared_prefix_pages)
    if scale is None:
        scale = 1.0 / math.sqrt(D if not mla else 192)
    return build_workload(f"random_{seed}", seed, B=B, Hq=Hq, Hkv=Hkv, D_qk=D, page_size=page_size,
                          seq_lens=lens, block_table=table, num_pages=num_pages, scale=scale,
                          D_v=D_v, q_len=q_len, mla=mla, layout=layout, poison=poison, values=values)
