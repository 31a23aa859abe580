"""Shared helpers for the GPU parity tests: run a workload through the C-ABI and
through the oracle on the same bits, and compare element by element.

Tolerance (per element, bf16 output vs the fp64 oracle):
    |gpu - oracle| <= ATOL + RTOL * |oracle|,  ATOL = RTOL = 1e-2.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300.workloads import Workload

ATOL = 1e-2
RTOL = 1e-2


class GpuRun:
    def __init__(self, out, lse, err):
        self.out, self.lse, self.err = out, lse, err

    def out64(self):
        return self.out.float().cpu().numpy().astype(np.float64)

    def lse64(self):
        return self.lse.cpu().numpy().astype(np.float64)


def device_inputs(wl: Workload):
    dev = torch.device("cuda")
    return dict(q=wl.q.to(dev), k=wl.k_pool.to(dev),
                v=None if wl.v_pool is None else wl.v_pool.to(dev),
                bt=torch.from_numpy(wl.block_table).to(dev),
                sl=torch.from_numpy(wl.seq_lens).to(dev))


def run_gpu(wl: Workload, inputs=None, *, num_ctas=0, max_seq_len=None, block_table=None,
            seq_lens=None, shared_prefix_pages=0, single_launch=False) -> GpuRun:
    d = inputs or device_inputs(wl)
    bt = d["bt"] if block_table is None else block_table
    sl = d["sl"] if seq_lens is None else seq_lens
    lse = torch.full((wl.B, wl.q_len, wl.Hq), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    msl = wl.max_seq_len if max_seq_len is None else max_seq_len
    if wl.mla:
        out = zl.decode_attn_mla(d["q"], d["k"], bt, sl, page_size=wl.page_size, scale=wl.scale,
                                 D_v=wl.D_v, lse=lse, err_flags=err, num_ctas=num_ctas,
                                 max_seq_len=msl)
    else:
        out = zl.decode_attn(d["q"], d["k"], d["v"], bt, sl, page_size=wl.page_size,
                             scale=wl.scale, lse=lse, err_flags=err, num_ctas=num_ctas,
                             max_seq_len=msl, layout=wl.layout,
                             shared_prefix_pages=shared_prefix_pages,
                             single_launch=single_launch)
    torch.cuda.synchronize()
    return GpuRun(out, lse, err)


def run_oracle(wl: Workload, block_table=None, seq_lens=None):
    orc = oracle.load()
    return orc.decode_attn(Workload.bits(wl.q), Workload.bits(wl.k_pool),
                           None if wl.v_pool is None else Workload.bits(wl.v_pool), wl.strides,
                           wl.block_table if block_table is None else block_table,
                           wl.seq_lens if seq_lens is None else seq_lens, Hkv=wl.Hkv,
                           page_size=wl.page_size, num_pages=wl.num_pages, scale=wl.scale,
                           D_v=wl.D_v)


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_inf = np.isinf(ref) & (got == ref)
    with np.errstate(invalid="ignore"):  # inf - inf where both are -inf (masked below)
        diff = np.where(both_inf, 0.0, np.abs(got - ref))
    bound = ATOL + RTOL * np.abs(np.where(both_inf, 0.0, ref))
    bad = ~(diff <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first at "
            f"{tuple(i)}: gpu {got[tuple(i)]!r} oracle {ref[tuple(i)]!r}; "
            f"max abs err {np.nanmax(diff):.3e}")


def max_errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    return float(d.max()), float((d / np.maximum(np.abs(ref), 1e-6)).max())
