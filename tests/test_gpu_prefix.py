"""Shared-prefix decode (shared_prefix_pages > 0): the prefix pages are read
once per group of sequences and each row's prefix result is folded into its
own suffix. Element by element against the oracle, which knows nothing of
the sharing (it reads every sequence's pages through its own table)."""
import numpy as np
import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _parity(w, npref, **kw):
    g = run_gpu(w, shared_prefix_pages=npref, **kw)
    ref, ref_lse, st = run_oracle(w)
    assert st == 0
    assert int(g.err.item()) == 0
    assert_close(g.out64(), ref, f"{w.name} out")
    assert_close(g.lse64(), ref_lse, f"{w.name} lse")
    assert not torch.isnan(g.out.float()).any()
    return g


def _case(seed, *, B, Hq, Hkv, npref, P=16, q_len=1, extra=None, layout="NHD"):
    rng = np.random.default_rng(seed)
    base = npref * P + q_len - 1
    lens = base + (rng.integers(0, 400, size=B) if extra is None else np.asarray(extra))
    return wl.random_case(seed, B=B, Hq=Hq, Hkv=Hkv, page_size=P, lens=lens, q_len=q_len,
                          shared_prefix_pages=npref, layout=layout)


def test_llama70b_shared_prefix_full():
    w = wl.llama70b_prefix_decode()
    npref = w.notes["shared_prefix_tokens"] // w.page_size
    _parity(w, npref)


@pytest.mark.parametrize("Hq,Hkv,q_len", [(64, 8, 1), (32, 8, 1), (16, 8, 1), (8, 8, 1),
                                          (32, 8, 2), (16, 8, 4), (16, 1, 1), (12, 3, 1)])
def test_groups_and_query_tokens(Hq, Hkv, q_len):
    """g * q_len rows per sequence, 16 / (g * q_len) sequences per group (the
    last group partly empty for B = 7)."""
    w = _case(1200 + Hq + Hkv + q_len, B=7, Hq=Hq, Hkv=Hkv, npref=6, q_len=q_len)
    _parity(w, 6)


@pytest.mark.parametrize("npref,B", [(20, 5), (64, 40), (129, 3)])
def test_long_prefixes(npref, B):
    """Long prefixes (20, 64 and 129 pages of 16 tokens) cut between several
    CTAs, with 2 sequences per prefix group at g = 8 and a partly empty last
    group for odd B."""
    w = _case(1260 + npref + B, B=B, Hq=64, Hkv=8, npref=npref)
    _parity(w, npref)


def test_suffix_edges():
    """Sequences that end exactly at the prefix, one token past it, at tile and
    page edges, and long ones."""
    extra = [0, 1, 15, 16, 17, 31, 32, 33, 700]
    w = _case(1210, B=len(extra), Hq=32, Hkv=8, npref=5, extra=extra)
    _parity(w, 5)


@pytest.mark.parametrize("B", [300, 400])
def test_many_sequences_around_the_small_table(B):
    """Prefix groups plus sequences make the table's units: 150 + 300 fit the
    small shared-memory table, 200 + 400 take the full one."""
    rng = np.random.default_rng(B)
    w = _case(1300 + B, B=B, Hq=64, Hkv=8, npref=4, extra=rng.integers(0, 40, size=B))
    _parity(w, 4)


@pytest.mark.parametrize("num_ctas", [1, 3, 40, 151, 900])
def test_any_grid(num_ctas):
    w = _case(1220, B=9, Hq=32, Hkv=8, npref=8)
    _parity(w, 8, num_ctas=num_ctas)


@pytest.mark.parametrize("P", [32, 64])
def test_page_sizes_and_hnd(P):
    for layout in ("NHD", "HND"):
        w = _case(1230 + P, B=6, Hq=16, Hkv=4, npref=3, P=P, layout=layout)
        _parity(w, 3)


def test_matches_plain_path_and_repeats():
    """Same inputs through the plain path: close (the pieces differ, so not the
    same bits); the shared-prefix path repeats bit for bit."""
    w = _case(1240, B=10, Hq=64, Hkv=8, npref=10)
    d = device_inputs(w)
    a = run_gpu(w, d, shared_prefix_pages=10)
    b = run_gpu(w, d, shared_prefix_pages=10)
    c = run_gpu(w, d)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert_close(a.out64(), c.out64(), "shared prefix vs plain")


def test_page_remap_is_bit_identical():
    w = _case(1250, B=6, Hq=32, Hkv=8, npref=4)
    d = device_inputs(w)
    g1 = run_gpu(w, d, shared_prefix_pages=4)
    # move every used page to another slot of a larger pool (prefix stays shared)
    n = w.num_pages
    perm = np.random.default_rng(7).permutation(2 * n)[:n]
    k2 = torch.full((2 * n,) + tuple(w.k_pool.shape[1:]), float("nan"), dtype=torch.bfloat16)
    v2 = k2.clone()
    k2[torch.from_numpy(perm)] = w.k_pool
    v2[torch.from_numpy(perm)] = w.v_pool
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    d2 = dict(d, k=k2.cuda(), v=v2.cuda(), bt=torch.from_numpy(bt2).cuda())
    w2 = wl.Workload(**{f: getattr(w, f) for f in w.__dataclass_fields__})
    w2.num_pages = 2 * n
    g2 = run_gpu(w2, d2, shared_prefix_pages=4)
    assert torch.equal(g1.out.view(torch.int16), g2.out.view(torch.int16))


def test_violations_are_flagged():
    """A sequence whose first pages differ from the others', or one shorter
    than the prefix, sets ZL_DEVERR_BAD_PREFIX."""
    w = _case(1260, B=5, Hq=32, Hkv=8, npref=4)
    d = device_inputs(w)
    bt = w.block_table.copy()
    bt[3, 1] = bt[3, 1] + 1 if bt[3, 1] + 1 < w.num_pages else bt[3, 1] - 1
    g = run_gpu(w, d, block_table=torch.from_numpy(bt).cuda(), shared_prefix_pages=4)
    assert int(g.err.item()) & zl.DEVERR_BAD_PREFIX
    sl = w.seq_lens.copy()
    sl[2] = 4 * 16 - 5
    g = run_gpu(w, d, seq_lens=torch.from_numpy(sl).cuda(), shared_prefix_pages=4)
    assert int(g.err.item()) & zl.DEVERR_BAD_PREFIX


def test_bad_prefix_page_zeroes_everything():
    w = _case(1270, B=4, Hq=32, Hkv=8, npref=3)
    d = device_inputs(w)
    bt = w.block_table.copy()
    bt[:, 1] = w.num_pages + 9
    g = run_gpu(w, d, block_table=torch.from_numpy(bt).cuda(), shared_prefix_pages=3)
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    assert torch.all(g.out.float() == 0)
