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


@pytest.mark.parametrize("num_ctas", [0, 12])
def test_mla_bad_page_seen_by_the_newest_token_only(num_ctas):
    """Two query tokens; the bad page holds only the newest token (position
    L - 1 starts its page), so only the second token's rows are zeroed."""
    P = 64
    lens = [P + 1, 3 * P + 1, 150]
    w = wl.random_case(615, B=len(lens), Hq=128, Hkv=1, D=576, D_v=512, mla=True,
                       page_size=P, lens=lens, pool_factor=1.5, q_len=2)
    d = device_inputs(w)
    bt = w.block_table.copy()
    bt[0, 1] = -1
    bt[1, 3] = w.num_pages
    g = run_gpu(w, d, block_table=torch.from_numpy(bt).cuda(), num_ctas=num_ctas)
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    ref, ref_lse, st = run_oracle(w, block_table=bt)
    assert st & 1
    assert_close(g.out64(), ref, "mla newest-page out")
    assert_close(g.lse64(), ref_lse, "mla newest-page lse")
    for b in (0, 1):
        assert (g.out[b, 1] == 0).all() and (g.out[b, 0] != 0).any()


def test_mla_full_workload():
    _parity(wl.mla_decode())


def test_mla_max_units():
    """1024 (sequence, query token) units, the most one call takes: the tile
    prefix and cost arrays in shared memory are full."""
    rng = np.random.default_rng(614)
    _parity(_mla_case(614, rng.integers(1, 100, size=1024, endpoint=True).tolist()))


def test_mla_output_16_byte_aligned():
    """An output that is 16- but not 32-byte aligned takes 16-byte stores."""
    w = _mla_case(612, [300, 64, 1000])
    d = device_inputs(w)
    n = w.B * w.q_len * w.Hq * w.D_v
    buf = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(w.B, w.q_len, w.Hq, w.D_v)
    assert out.data_ptr() % 32 == 16
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    zl.decode_attn_mla(d["q"], d["k"], d["bt"], d["sl"], page_size=w.page_size, scale=w.scale,
                       D_v=w.D_v, out=out, err_flags=err, max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, _, _ = run_oracle(w)
    assert_close(out.float().cpu().numpy(), ref, "mla out at 16-byte alignment")


@pytest.mark.parametrize("q_len", [2, 3])
def test_mla_multi_token(q_len):
    """q_len query tokens per sequence (multi-token prediction): token i sees the
    first L - q_len + 1 + i tokens; contexts shorter than q_len included."""
    lens = [1, 2, 3, 64, 65, 130, 700]
    w = wl.random_case(620 + q_len, B=len(lens), Hq=128, Hkv=1, D=576, D_v=512, mla=True,
                       page_size=64, lens=lens, q_len=q_len)
    _parity(w)


def test_mla_multi_token_split_and_last_row():
    """Split across many clusters; the last query token's rows equal a q_len = 1
    call with that query, bit for bit."""
    w = wl.random_case(630, B=5, Hq=128, Hkv=1, D=576, D_v=512, mla=True, page_size=64,
                       max_len=900, q_len=2)
    g = _parity(w, num_ctas=60)
    w1 = wl.random_case(630, B=5, Hq=128, Hkv=1, D=576, D_v=512, mla=True, page_size=64,
                        max_len=900, q_len=1)
    w1.q = w.q[:, -1:].contiguous()
    g1 = run_gpu(w1, num_ctas=60)
    ref1, _, _ = run_oracle(w1)
    assert_close(g1.out64(), ref1, "q_len 1")
    assert_close(g.out64()[:, -1:], g1.out64(), "last row vs q_len 1")


def test_mla_deepseek_mtp_shape_sampled():
    """The DeepSeek-V3 shape with 2 query tokens (one extra MTP token): sampled
    sequences against the oracle at full context lengths."""
    w = wl.mla_decode(q_len=2)
    g = run_gpu(w)
    rng = np.random.default_rng(11)
    bs = rng.choice(w.B, size=4, replace=False)
    ws = wl.build_workload("sampled", 0, B=len(bs), Hq=128, Hkv=1, D_qk=576, D_v=512,
                           page_size=64, seq_lens=w.seq_lens[bs], block_table=w.block_table[bs],
                           num_pages=w.num_pages, scale=w.scale, q_len=2, mla=True, values=False)
    ws.q, ws.k_pool, ws.v_pool = w.q[bs].contiguous(), w.k_pool, None
    ref, ref_lse, st = run_oracle(ws)
    assert st == 0
    assert_close(g.out64()[bs], ref, "sampled out")
    assert_close(g.lse64()[bs], ref_lse, "sampled lse")


@pytest.mark.parametrize("trend", ["rising", "falling", "spike"])
@pytest.mark.parametrize("num_ctas", [0, 2, 40])
def test_mla_softmax_max_moves_often(trend, num_ctas):
    """The rope columns of the latent rows scaled so that the scores climb far
    past 2^8 from tile to tile (the kernel's running max moves and O in TMEM is
    rescaled), fall after a large first tile, or jump at one late token; whole
    and split. (Only the rope: scaling the latent would scale V as well, and
    the bf16 rounding of P would then exceed the absolute tolerance wherever
    large V rows cancel.)"""
    w = _mla_case(1650 + num_ctas + len(trend), [700, 1500, 65, 1024])
    k = w.k_pool.float()
    for b, L in enumerate(w.seq_lens):
        for t in range(int(L)):
            page, slot = w.block_table[b, t // w.page_size], t % w.page_size
            if trend == "rising":
                f = 1.0 + 40.0 * t / L
            elif trend == "falling":
                f = 41.0 - 40.0 * t / L
            else:
                f = 40.0 if t == int(L) * 3 // 4 else 1.0
            k[page, slot, :, 512:] *= f
    w.k_pool = k.to(torch.bfloat16)
    _parity(w, num_ctas=num_ctas)
