"""Absorbed MLA paged decode on the GPU against the oracle (element by element)."""
import numpy as np
import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _mla_case(seed, lens, page_size=64, pool_factor=1.5):
    return wl.random_case(seed, B=len(lens), Hq=128, Hkv=1, D=576, D_v=512, mla=True,
                          page_size=page_size, lens=lens, pool_factor=pool_factor)


def _parity(w, **kw):
    g = run_gpu(w, **kw)
    ref, ref_lse, st = run_oracle(w)
    assert st == 0
    assert int(g.err.item()) == 0
    assert_close(g.out64(), ref, f"{w.name} out")
    assert_close(g.lse64(), ref_lse, f"{w.name} lse")
    return g


def test_mla_one_tile():
    _parity(_mla_case(600, [64]), num_ctas=2)


def test_mla_small():
    _parity(_mla_case(601, [1, 31, 32, 33, 63, 64, 65, 127, 128, 200, 513]))


@pytest.mark.parametrize("num_ctas", [2, 6, 30, 152, 1000])
def test_mla_any_split(num_ctas):
    _parity(_mla_case(602, [700, 1500, 33, 2048]), num_ctas=num_ctas)


@pytest.mark.parametrize("P", [64, 128, 256])
def test_mla_page_sizes(P):
    _parity(_mla_case(603 + P, [P - 1, P, P + 1, 3 * P + 5], page_size=P))


def test_mla_page_remap_is_bit_identical():
    w = _mla_case(610, [300, 900, 64], pool_factor=2.0)
    d = device_inputs(w)
    g1 = run_gpu(w, d)
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(9))
    k2 = torch.empty_like(d["k"])
    k2[perm.cuda()] = d["k"]
    bt = w.block_table.copy()
    bt[bt >= 0] = perm.numpy()[bt[bt >= 0]]
    g2 = run_gpu(w, dict(d, k=k2, bt=torch.from_numpy(bt).cuda()))
    assert torch.equal(g1.out.view(torch.int16), g2.out.view(torch.int16))


def test_mla_empty_and_bad_page():
    w = _mla_case(611, [200, 0, 400, 130])
    d = device_inputs(w)
    bt = w.block_table.copy()
    bt[2, 3] = -1
    g = run_gpu(w, d, block_table=torch.from_numpy(bt).cuda())
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    assert (g.out[1] == 0).all() and (g.out[2] == 0).all()
    ref, _, _ = run_oracle(w, block_table=bt)
    assert_close(g.out64(), ref, "mla empty/bad")


def test_mla_full_workload():
    _parity(wl.mla_decode())
