"""17 to 32 query heads per kv head with one query token (MQA-like shapes; the
heads of a kv head go in two row groups of at most 16 that share every CTA)
against the oracle, element by element: lengths at tile edges, splits of
every size, page sizes and layouts, bad pages, empty sequences, page
remapping, the full 32-head MQA workload."""
import numpy as np
import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

EDGES = [1, 15, 16, 17, 127, 128, 129, 255, 256, 300, 1000]


def _parity(w, **kw):
    g = run_gpu(w, **kw)
    ref, ref_lse, st = run_oracle(w)
    assert st == 0
    assert int(g.err.item()) == 0
    assert_close(g.out64(), ref, f"{w.name} out")
    assert_close(g.lse64(), ref_lse, f"{w.name} lse")
    assert not torch.isnan(g.out.float()).any()
    return g


@pytest.mark.parametrize("Hq,Hkv", [(32, 1), (17, 1), (24, 1), (64, 2), (128, 4), (96, 4)])
def test_heads_per_kv_head(Hq, Hkv):
    w = wl.random_case(1200 + Hq + Hkv, B=len(EDGES), Hq=Hq, Hkv=Hkv, lens=EDGES)
    _parity(w)


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 152, 777, 5000])
def test_any_split(num_ctas):
    w = wl.random_case(1210, B=5, Hq=32, Hkv=1, max_len=1500)
    _parity(w, num_ctas=num_ctas)


def test_split_vs_unsplit_close():
    w = wl.random_case(1211, B=3, Hq=32, Hkv=2, lens=[3000, 129, 2048])
    a = run_gpu(w, num_ctas=1).out64()
    b = run_gpu(w, num_ctas=300).out64()
    assert np.abs(a - b).max() <= 2e-2


@pytest.mark.parametrize("P", [16, 32, 64, 128])
def test_page_sizes_and_layouts(P):
    for layout in ("NHD", "HND"):
        w = wl.random_case(1220 + P, B=4, Hq=32, Hkv=2, page_size=P, max_len=5 * P + 3,
                           layout=layout)
        _parity(w)


def test_short_contexts_one_cta_per_unit():
    """max_seq_len shows every unit short: one CTA per unit, no merge launch;
    without it the kernel decides the same on the device."""
    lens = [0, 1, 16, 17, 64, 128]
    w = wl.random_case(1230, B=len(lens), Hq=32, Hkv=1, lens=lens)
    g = _parity(w)
    assert torch.all(g.out[0] == 0) and torch.all(torch.isneginf(g.lse[0].cpu()))
    _parity(w, max_seq_len=0)


def test_page_remap_and_repeat_are_bit_identical():
    w = wl.random_case(1240, B=4, Hq=32, Hkv=1, max_len=900, pool_factor=2.0)
    d = device_inputs(w)
    g1 = run_gpu(w, d)
    g2 = run_gpu(w, d)
    assert torch.equal(g1.out.view(torch.int16), g2.out.view(torch.int16))
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(3))
    k2, v2 = torch.empty_like(d["k"]), torch.empty_like(d["v"])
    k2[perm.cuda()] = d["k"]
    v2[perm.cuda()] = d["v"]
    bt = w.block_table.copy()
    bt[bt >= 0] = perm.numpy()[bt[bt >= 0]]
    g3 = run_gpu(w, dict(d, k=k2, v=v2, bt=torch.from_numpy(bt).cuda()))
    assert torch.equal(g1.out.view(torch.int16), g3.out.view(torch.int16))


@pytest.mark.parametrize("num_ctas", [0, 40])
def test_bad_page_zeroes_its_sequence(num_ctas):
    w = wl.random_case(1250, B=4, Hq=32, Hkv=1, lens=[300, 500, 129, 40])
    d = device_inputs(w)
    bt = d["bt"].clone()
    bt[1, 9] = -2                 # inside a chunk of sequence 1
    bt[2, 8] = w.num_pages + 3    # the last (one-token) tile of sequence 2
    g = run_gpu(w, d, block_table=bt, num_ctas=num_ctas)
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    ref, ref_lse, st = run_oracle(w, block_table=bt.cpu().numpy())
    assert st & 1
    assert_close(g.out64(), ref, "out")
    assert_close(g.lse64(), ref_lse, "lse")
    for b in (1, 2):
        assert torch.all(g.out[b] == 0)
    assert torch.all(g.out[0].abs().sum(-1) > 0)


def test_mqa32_full_workload():
    _parity(wl.mqa32_decode())


def test_launch_count():
    w = wl.random_case(1260, B=2, Hq=32, Hkv=1, lens=[2000, 3000])
    d = device_inputs(w)
    out = torch.empty(w.B, 1, w.Hq, 128, dtype=torch.bfloat16, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=w.page_size,
                       scale=w.scale, Hkv=w.Hkv, D_v=128)
    assert zl.launches(p) == 2  # one attention launch for both row groups, and its merge
