"""Fused KV append (k_new / v_new in the decode call): the attention launch
stores the new tokens' rows in their page slots and attends over them. After
the call the pools must be bit-identical to the oracle's append, the output
bit-identical to a separate zl_kv_append followed by the same decode call,
and within tolerance of the oracle's attention over the appended cache. The
new tokens' slots start as NaN, so reading them before they are stored would
show."""
import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, run_oracle

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _wipe_new_slots(w):
    """NaN in every slot the call's new tokens go to (valid sequences only)."""
    cap = w.block_table.shape[1] * w.page_size
    for b, L in enumerate(w.seq_lens):
        if not (w.q_len <= L <= cap):
            continue
        for t in range(L - w.q_len, L):
            page, slot = w.block_table[b, t // w.page_size], t % w.page_size
            if not 0 <= page < w.num_pages:
                continue
            if w.layout == "NHD":
                w.k_pool[page, slot] = float("nan")
                if w.v_pool is not None:
                    w.v_pool[page, slot] = float("nan")
            else:
                w.k_pool[page, :, slot] = float("nan")
                w.v_pool[page, :, slot] = float("nan")


def _decode(w, kp, vp, bt, sl, k_new=None, v_new=None, **kw):
    lse = torch.full((w.B, w.q_len, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = w.q.cuda()
    if w.mla:
        out = zl.decode_attn_mla(q, kp, bt, sl, page_size=w.page_size, scale=w.scale, D_v=w.D_v,
                                 lse=lse, err_flags=err, max_seq_len=w.max_seq_len,
                                 kv_new=k_new, **kw)
    else:
        out = zl.decode_attn(q, kp, vp, bt, sl, page_size=w.page_size, scale=w.scale, lse=lse,
                             err_flags=err, max_seq_len=w.max_seq_len, layout=w.layout,
                             k_new=k_new, v_new=v_new, **kw)
    torch.cuda.synchronize()
    return out, lse, int(err.item())


def _check(w, seed, *, block_table=None, expect_err=0, oracle_parity=True, **kw):
    Hkv = w.Hkv
    if w.mla:
        k_new, v_new = wl.new_token_rows(seed, w.B, w.q_len, 1, w.D_qk)
    else:
        k_new, v_new = wl.new_token_rows(seed, w.B, w.q_len, Hkv, 128, 128)
    _wipe_new_slots(w)
    bt_np = w.block_table if block_table is None else block_table
    bt = torch.from_numpy(bt_np).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    kn = k_new.cuda()
    vn = None if v_new is None else v_new.cuda()
    # fused: one call
    kp, vp = w.k_pool.cuda(), None if w.v_pool is None else w.v_pool.cuda()
    out, lse, err = _decode(w, kp, vp, bt, sl, kn, vn, **kw)
    assert err == expect_err
    # separate: zl_kv_append, then the same decode call
    kp2, vp2 = w.k_pool.cuda(), None if w.v_pool is None else w.v_pool.cuda()
    zl.kv_append(kn, vn, kp2, vp2, bt, sl, page_size=w.page_size, layout=w.layout)
    out2, lse2, err2 = _decode(w, kp2, vp2, bt, sl, **kw)
    assert err2 == expect_err
    assert torch.equal(kp.view(torch.int16), kp2.view(torch.int16)), "K pools differ"
    if vp is not None:
        assert torch.equal(vp.view(torch.int16), vp2.view(torch.int16)), "V pools differ"
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "out differs"
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32)), "lse differs"
    # the oracle's append, bit for bit, and its attention over the result
    ko, vo, st = oracle.load().kv_append(
        _u16(k_new), None if v_new is None else _u16(v_new), _u16(w.k_pool),
        None if w.v_pool is None else _u16(w.v_pool), w.strides, bt_np, w.seq_lens,
        page_size=w.page_size, num_pages=w.num_pages)
    assert np.array_equal(_u16(kp), ko.reshape(kp.shape)), "K pool differs from the oracle's"
    if vp is not None:
        assert np.array_equal(_u16(vp), vo.reshape(vp.shape)), "V pool differs from the oracle's"
    if oracle_parity:
        w.k_pool = torch.from_numpy(ko.view(np.int16)).view(torch.bfloat16).reshape(w.k_pool.shape)
        if vp is not None:
            w.v_pool = torch.from_numpy(vo.view(np.int16)).view(torch.bfloat16).reshape(
                w.v_pool.shape)
        ref, ref_lse, st = run_oracle(w, block_table=bt_np)
        assert st == expect_err
        assert_close(out.float().cpu().numpy().astype(np.float64), ref, "out")
        assert_close(lse.cpu().numpy().astype(np.float64), ref_lse, "lse")
    return out


@pytest.mark.parametrize("q_len", [1, 2, 4, 8])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_fused_append_gqa(q_len, layout):
    """4 query heads per kv head: 1-4 tokens in one row group, 8 in two groups
    that share every CTA."""
    w = wl.random_case(1500 + q_len, B=7, Hq=32, Hkv=8, max_len=300, q_len=q_len, layout=layout)
    _check(w, 1500 + q_len)


@pytest.mark.parametrize("Hq,Hkv,q_len", [(32, 1, 1), (32, 1, 2), (64, 2, 1), (16, 16, 3),
                                          (12, 3, 5)])
def test_fused_append_head_groups(Hq, Hkv, q_len):
    """Many heads per kv head (two groups per CTA, or four groups on separate
    CTAs that each store the same rows), MHA, odd head and token counts."""
    w = wl.random_case(1510 + Hq + q_len, B=5, Hq=Hq, Hkv=Hkv, max_len=400, q_len=q_len)
    _check(w, 1510 + Hq + q_len)


@pytest.mark.parametrize("num_ctas", [1, 7, 152, 1000])
def test_fused_append_any_grid(num_ctas):
    w = wl.random_case(1520, B=6, Hq=32, Hkv=8, max_len=700, q_len=2)
    _check(w, 1520, num_ctas=num_ctas)


@pytest.mark.parametrize("P", [16, 32, 64, 128])
def test_fused_append_page_edges(P):
    """New tokens at every page and tile edge: the first slot of a page, the
    last, and tokens spanning two pages."""
    lens = sorted({2, 3, 16, 17, P, P + 1, P + 2, 2 * P + 1})
    w = wl.random_case(1530 + P, B=len(lens), Hq=16, Hkv=4, page_size=P, lens=lens, q_len=2)
    _check(w, 1530 + P)


def test_fused_append_single_launch():
    """One launch per row group (8 tokens at g = 4), each storing the rows it reads."""
    w = wl.random_case(1540, B=5, Hq=32, Hkv=8, max_len=500, q_len=8)
    _check(w, 1540, single_launch=True)


def test_fused_append_shared_prefix():
    rng = np.random.default_rng(1550)
    npref, P = 4, 16
    lens = npref * P + 2 + rng.integers(0, 200, size=9)  # the new tokens lie past the prefix
    w = wl.random_case(1550, B=9, Hq=32, Hkv=8, page_size=P, lens=lens, q_len=2,
                       shared_prefix_pages=npref)
    _check(w, 1550, shared_prefix_pages=npref)


def test_fused_append_errors():
    """A sequence shorter than q_len stores nothing (bad length); a new token on
    a bad page is skipped (bad page); the rest is stored and attended."""
    w = wl.random_case(1560, B=5, Hq=16, Hkv=4, lens=[40, 2, 50, 33, 64], q_len=3)
    bt = w.block_table.copy()
    bt[2, (50 - 1) // 16] = w.num_pages + 3
    _check(w, 1560, block_table=bt, expect_err=zl.DEVERR_BAD_PAGE, oracle_parity=False)


@pytest.mark.parametrize("q_len", [1, 2])
@pytest.mark.parametrize("num_ctas", [0, 2, 40])
def test_fused_append_mla(q_len, num_ctas):
    w = wl.random_case(1570 + q_len, B=6, Hq=128, Hkv=1, D=576, page_size=64, max_len=500,
                       mla=True, D_v=512, q_len=q_len)
    _check(w, 1570 + q_len, num_ctas=num_ctas)


def test_fused_append_full_size_llama3_8b():
    w = wl.llama3_8b_decode()
    _check(w, 1580)
