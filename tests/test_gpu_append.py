"""Paged KV append (zl_kv_append) on the GPU against the oracle: the pools
after the append must be bit-identical to the oracle's, everywhere."""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _append_both(w, k_new, v_new, *, block_table=None, seq_lens=None):
    """Run the append on device copies of w's pools and in the oracle; return
    (gpu K, gpu V, gpu flags, oracle K, oracle V, oracle status)."""
    bt = w.block_table if block_table is None else block_table
    sl = w.seq_lens if seq_lens is None else seq_lens
    kp = w.k_pool.cuda()
    vp = None if w.v_pool is None else w.v_pool.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    zl.kv_append(k_new.cuda(), None if v_new is None else v_new.cuda(), kp, vp,
                 torch.from_numpy(bt).cuda(), torch.from_numpy(sl).cuda(),
                 page_size=w.page_size, layout=w.layout, err_flags=err)
    torch.cuda.synchronize()
    ko, vo, st = oracle.load().kv_append(
        _u16(k_new), None if v_new is None else _u16(v_new), _u16(w.k_pool),
        None if w.v_pool is None else _u16(w.v_pool), w.strides, bt, sl,
        page_size=w.page_size, num_pages=w.num_pages)
    return kp, vp, int(err.item()), ko, vo, st


def _assert_pools_equal(kp, vp, ko, vo):
    assert np.array_equal(_u16(kp), ko.reshape(kp.shape)), "K pool differs"
    if vp is None:
        assert vo is None
    else:
        assert np.array_equal(_u16(vp), vo.reshape(vp.shape)), "V pool differs"


@pytest.mark.parametrize("q_len", [1, 2, 4])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_append_bit_exact(q_len, layout):
    w = wl.random_case(900 + q_len, B=7, Hq=32, Hkv=8, max_len=200, q_len=q_len, layout=layout)
    k_new, v_new = wl.new_token_rows(900 + q_len, w.B, q_len, 8, 128, 128)
    kp, vp, err, ko, vo, st = _append_both(w, k_new, v_new)
    assert err == 0 and st == 0
    _assert_pools_equal(kp, vp, ko, vo)
    assert not np.array_equal(ko, _u16(w.k_pool))    # something was written


@pytest.mark.parametrize("Hkv,P", [(1, 16), (2, 32), (4, 64), (8, 128)])
def test_append_heads_and_pages(Hkv, P):
    w = wl.random_case(910 + Hkv, B=5, Hq=2 * Hkv, Hkv=Hkv, page_size=P, max_len=3 * P, q_len=3)
    k_new, v_new = wl.new_token_rows(910 + Hkv, w.B, 3, Hkv, 128, 128)
    kp, vp, err, ko, vo, st = _append_both(w, k_new, v_new)
    assert err == 0 and st == 0
    _assert_pools_equal(kp, vp, ko, vo)


def test_append_latent_pool():
    """Latent-only (MLA) pool: one 576-wide row per token, no V pool."""
    w = wl.random_case(920, B=6, Hq=128, Hkv=1, D=576, page_size=64, max_len=300, mla=True,
                       D_v=512, q_len=2)
    k_new, _ = wl.new_token_rows(920, w.B, 2, 1, 576)
    kp, vp, err, ko, vo, st = _append_both(w, k_new, None)
    assert err == 0 and st == 0 and vp is None
    _assert_pools_equal(kp, vp, ko, vo)


def test_append_errors():
    """A sequence shorter than q_len writes nothing; a bad page id skips its
    token; both are flagged; everything else is appended."""
    w = wl.random_case(930, B=5, Hq=16, Hkv=4, lens=[40, 2, 50, 33, 64], q_len=3)
    k_new, v_new = wl.new_token_rows(930, w.B, 3, 4, 128, 128)
    bt = w.block_table.copy()
    bt[2, (50 - 1) // 16] = w.num_pages + 3
    kp, vp, err, ko, vo, st = _append_both(w, k_new, v_new, block_table=bt)
    assert st == 3 and err == 3
    _assert_pools_equal(kp, vp, ko, vo)


def test_append_then_attend():
    """The new tokens' slots start as NaN; after the append, decode attention on
    the same stream matches the oracle's attention over the oracle's appended pools."""
    q_len = 2
    w = wl.random_case(940, B=6, Hq=32, Hkv=8, max_len=300, q_len=q_len)
    k_new, v_new = wl.new_token_rows(940, w.B, q_len, 8, 128, 128)
    for b, L in enumerate(w.seq_lens):                 # wipe the new tokens' slots
        for t in range(L - q_len, L):
            page, slot = w.block_table[b, t // 16], t % 16
            w.k_pool[page, slot] = float("nan")
            w.v_pool[page, slot] = float("nan")
    kp, vp, err, ko, vo, st = _append_both(w, k_new, v_new)
    assert err == 0 and st == 0
    _assert_pools_equal(kp, vp, ko, vo)
    d = dict(q=w.q.cuda(), k=kp, v=vp, bt=torch.from_numpy(w.block_table).cuda(),
             sl=torch.from_numpy(w.seq_lens).cuda())
    g = run_gpu(w, d)
    w.k_pool = torch.from_numpy(ko.view(np.int16)).view(torch.bfloat16).reshape(w.k_pool.shape)
    w.v_pool = torch.from_numpy(vo.view(np.int16)).view(torch.bfloat16).reshape(w.v_pool.shape)
    ref, ref_lse, st = run_oracle(w)
    assert st == 0 and int(g.err.item()) == 0
    assert_close(g.out64(), ref, "out")
    assert_close(g.lse64(), ref_lse, "lse")


def test_append_full_size_llama3_8b():
    """Llama-3-8B shape at batch 64: the whole ~0.7 GB of pools bit-identical."""
    w = wl.llama3_8b_decode()
    k_new, v_new = wl.new_token_rows(950, w.B, 1, 8, 128, 128)
    kp, vp, err, ko, vo, st = _append_both(w, k_new, v_new)
    assert err == 0 and st == 0
    _assert_pools_equal(kp, vp, ko, vo)
