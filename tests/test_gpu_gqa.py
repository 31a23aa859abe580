"""GQA paged decode attention on the GPU against the oracle (element by element)."""
import numpy as np
import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _parity(w, **kw):
    g = run_gpu(w, **kw)
    ref, ref_lse, st = run_oracle(w)
    assert st == 0
    assert int(g.err.item()) == 0
    assert_close(g.out64(), ref, f"{w.name} out")
    assert_close(g.lse64(), ref_lse, f"{w.name} lse")
    assert not torch.isnan(g.out.float()).any()
    return g


def test_tiny_gqa():
    _parity(wl.tiny_gqa())


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (16, 4), (32, 8), (64, 8), (16, 1), (12, 3),
                                    (64, 4), (6, 2), (10, 5)])
def test_group_sizes(Hq, Hkv):
    """g = 1..16 and every heads-per-CTA choice (8, 4, 2, 1)."""
    w = wl.random_case(100 + Hq * 7 + Hkv, B=5, Hq=Hq, Hkv=Hkv, max_len=200)
    _parity(w)


@pytest.mark.parametrize("P", [16, 32, 64, 128])
def test_page_sizes_and_edges(P):
    """Lengths at every tile/page edge: 1, 15, 16, 17, P-1, P, P+1, 2P+3."""
    lens = sorted({1, 15, 16, 17, P - 1, P, P + 1, 2 * P + 3})
    w = wl.random_case(200 + P, B=len(lens), Hq=16, Hkv=4, page_size=P, lens=lens)
    _parity(w)


def test_hnd_layout_is_bit_identical_to_nhd():
    a = wl.random_case(301, B=6, Hq=32, Hkv=8, max_len=300)
    b = wl.random_case(301, B=6, Hq=32, Hkv=8, max_len=300, layout="HND")
    ga, gb = _parity(a), _parity(b)
    assert torch.equal(ga.out.view(torch.int16), gb.out.view(torch.int16))


@pytest.mark.parametrize("B,Hq,Hkv", [(511, 8, 2), (512, 8, 2), (600, 32, 1)])
@pytest.mark.parametrize("hint", [True, False])
def test_batches_around_the_small_table(B, Hq, Hkv, hint):
    """Up to 511 sequences keep their tile offsets in the small shared-memory
    table (more CTAs fit on an SM), more in the full one: both sides of the
    edge (512 and 513 entries), and the two-row-group instance (32 heads on
    one kv head) on the full one; with and without max_seq_len."""
    w = wl.random_case(500 + B + Hq, B=B, Hq=Hq, Hkv=Hkv, max_len=48)
    _parity(w, **({} if hint else {"max_seq_len": 0}))


@pytest.mark.parametrize("num_ctas", [1, 2, 7, 64, 151, 1000, 5000])
def test_any_split_matches(num_ctas):
    """Every grid size (one CTA = unsplit, many CTAs = many split pieces)."""
    w = wl.random_case(400, B=7, Hq=32, Hkv=8, max_len=700)
    _parity(w, num_ctas=num_ctas)


@pytest.mark.parametrize("trend", ["rising", "falling", "spike"])
@pytest.mark.parametrize("num_ctas", [0, 1, 37])
def test_softmax_base_moves_often(trend, num_ctas):
    """Scores that climb by much more than 2^8 from tile to tile (the kernel's
    softmax base moves on nearly every tile), that fall after a large first
    tile (P far below 1 against a stale base), or that jump at one token late
    in the context; whole and split, against the oracle."""
    w = wl.random_case(1600 + num_ctas + len(trend), B=4, Hq=32, Hkv=8,
                       lens=[700, 333, 1000, 17])
    k = w.k_pool.float()
    for b, L in enumerate(w.seq_lens):
        for t in range(int(L)):
            page, slot = w.block_table[b, t // w.page_size], t % w.page_size
            if trend == "rising":
                f = 1.0 + 40.0 * t / L
            elif trend == "falling":
                f = 41.0 - 40.0 * t / L
            else:
                f = 30.0 if t == int(L) * 3 // 4 else 1.0
            k[page, slot] *= f
    w.k_pool = k.to(torch.bfloat16)
    _parity(w, num_ctas=num_ctas)


def test_split_vs_unsplit_close():
    w = wl.random_case(401, B=4, Hq=32, Hkv=8, lens=[1000, 2000, 17, 513])
    d = device_inputs(w)
    one = run_gpu(w, d, num_ctas=1).out64()
    many = run_gpu(w, d, num_ctas=300).out64()
    assert_close(many, one, "split vs unsplit")


def test_page_remap_is_bit_identical():
    w = wl.random_case(500, B=6, Hq=32, Hkv=8, max_len=400, pool_factor=2.0)
    d = device_inputs(w)
    g1 = run_gpu(w, d)
    # move every page to another physical slot, same logical content
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(5))
    k2 = torch.empty_like(d["k"])
    v2 = torch.empty_like(d["v"])
    k2[perm.cuda()] = d["k"]
    v2[perm.cuda()] = d["v"]
    bt = w.block_table.copy()
    bt[bt >= 0] = perm.numpy()[bt[bt >= 0]]
    d2 = dict(d, k=k2, v=v2, bt=torch.from_numpy(bt).cuda())
    g2 = run_gpu(w, d2)
    assert torch.equal(g1.out.view(torch.int16), g2.out.view(torch.int16))
    assert torch.equal(g1.lse, g2.lse)


def test_repeat_calls_are_bit_identical():
    w = wl.random_case(501, B=8, Hq=32, Hkv=8, max_len=900)
    d = device_inputs(w)
    a, b = run_gpu(w, d), run_gpu(w, d)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_single_token_returns_v0_exactly():
    w = wl.random_case(502, B=3, Hq=16, Hkv=4, lens=[1, 1, 1])
    g = run_gpu(w)
    v = w.v_pool
    for b in range(3):
        page = w.block_table[b, 0]
        for h in range(16):
            assert torch.equal(g.out[b, 0, h].cpu().view(torch.int16),
                               v[page, 0, h // 4].view(torch.int16))


def test_empty_sequence_gives_zeros_and_neg_inf():
    w = wl.random_case(503, B=4, Hq=16, Hkv=4, lens=[30, 0, 77, 0])
    g = run_gpu(w)
    ref, ref_lse, _ = run_oracle(w)
    assert int(g.err.item()) == 0
    assert (g.out[1] == 0).all() and (g.out[3] == 0).all()
    assert torch.isinf(g.lse[1]).all() and (g.lse[1] < 0).all()
    assert_close(g.out64(), ref, "empty")


def test_bad_page_sets_flag_and_zeros_that_sequence():
    w = wl.random_case(504, B=4, Hq=32, Hkv=8, lens=[100, 300, 50, 400])
    d = device_inputs(w)
    bt = w.block_table.copy()
    bt[1, 3] = w.num_pages + 7
    g = run_gpu(w, d, block_table=torch.from_numpy(bt).cuda())
    ref, _, st = run_oracle(w, block_table=bt)
    assert st & zl.DEVERR_BAD_PAGE
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    assert (g.out[1] == 0).all()
    assert_close(g.out64(), ref, "bad page")


def test_bad_page_in_split_sequence():
    w = wl.random_case(505, B=2, Hq=32, Hkv=8, lens=[2000, 1500])
    d = device_inputs(w)
    bt = w.block_table.copy()
    bt[0, 100] = -3
    g = run_gpu(w, d, num_ctas=40, block_table=torch.from_numpy(bt).cuda())
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    assert (g.out[0] == 0).all()
    ref, _, _ = run_oracle(w, block_table=bt)
    assert_close(g.out64(), ref, "bad page split")


def test_oversize_seq_len_sets_flag():
    w = wl.random_case(506, B=3, Hq=16, Hkv=4, lens=[40, 60, 20])
    d = device_inputs(w)
    sl = w.seq_lens.copy()
    sl[2] = w.block_table.shape[1] * w.page_size + 1
    g = run_gpu(w, d, seq_lens=torch.from_numpy(sl).cuda())
    assert int(g.err.item()) & zl.DEVERR_BAD_SEQ_LEN
    assert (g.out[2] == 0).all()
    ref, _, st = run_oracle(w, seq_lens=sl)
    assert st & 2
    assert_close(g.out64(), ref, "oversize len")


def test_workspace_too_small_is_rejected():
    w = wl.random_case(507, B=2, Hq=16, Hkv=4, lens=[40, 60])
    d = device_inputs(w)
    out = torch.empty(2, 1, 16, 128, dtype=torch.bfloat16, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=16,
                       scale=w.scale, Hkv=4, D_v=128)
    need = zl.workspace_size(p)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    with pytest.raises(zl.ZlError) as e:
        zl.call(p, mla=False)
    assert e.value.status == zl.ERR_WORKSPACE


def test_runs_on_a_side_stream():
    w = wl.random_case(508, B=5, Hq=32, Hkv=8, max_len=500)
    d = device_inputs(w)
    ref = run_gpu(w, d).out
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = zl.decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], page_size=16,
                             scale=w.scale)
    s.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_llama3_8b_full():
    _parity(wl.llama3_8b_decode())


def test_llama70b_prefix_full():
    _parity(wl.llama70b_prefix_decode())


def test_long_context_full():
    _parity(wl.long_context_decode())


def test_mqa32_full():
    """32 query heads on one kv head (two row groups of 16 heads, both in every
    CTA), the Llama-3-8B lengths, the whole output against the oracle."""
    _parity(wl.mqa32_decode())


def test_cuda_graph_capture_of_the_default_path():
    """The default call (attention kernel + merge kernel as a programmatic
    dependent launch) captures into a CUDA graph; replays give the eager bits."""
    w = wl.random_case(509, B=8, Hq=32, Hkv=8, max_len=2500)
    d = device_inputs(w)
    out = torch.empty(w.B, 1, w.Hq, 128, dtype=torch.bfloat16, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=16,
                       scale=w.scale, Hkv=8, D_v=128)
    ws = torch.zeros(zl.workspace_size(p), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    zl.call(p, mla=False)
    torch.cuda.synchronize()
    eager = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        zl.call(p, mla=False, stream=s)
    for _ in range(4):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    ref, _, _ = run_oracle(w)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "graph replay")


def _launches(w, **kw):
    d = device_inputs(w)
    out = torch.empty((w.B, w.q_len, w.Hq, 128), dtype=torch.bfloat16, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=w.page_size,
                       scale=w.scale, Hkv=w.Hkv, D_v=128, max_seq_len=w.max_seq_len, **kw)
    return zl.launches(p)


def test_short_contexts_take_one_cta_per_unit():
    """max_seq_len shows every (sequence, head group) is short (here 7 tiles x
    64 KB of K and V): one CTA each, one launch, nothing to merge."""
    w = wl.random_case(410, B=6, Hq=32, Hkv=8, max_len=100)
    assert _launches(w) == 1
    assert _launches(w, num_ctas=152) == 2  # an explicit grid cuts as usual
    _parity(w)


def test_longer_contexts_are_cut_and_merged():
    w = wl.random_case(411, B=6, Hq=32, Hkv=8, lens=[3000, 40, 900, 1, 2500, 128])
    assert _launches(w) == 2
    _parity(w)


def test_short_contexts_with_empty_and_bad_sequences():
    w = wl.random_case(412, B=5, Hq=16, Hkv=4, lens=[0, 70, 1, 33, 64])
    d = device_inputs(w)
    bt = w.block_table.copy()
    bt[3, 1] = -1
    assert _launches(w) == 1
    g = run_gpu(w, d, block_table=torch.from_numpy(bt).cuda())
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    assert (g.out[0] == 0).all() and (g.out[3, :, 4:8] == 0).all()
    ref, _, _ = run_oracle(w, block_table=bt)
    assert_close(g.out64(), ref, "short contexts, empty and bad")
