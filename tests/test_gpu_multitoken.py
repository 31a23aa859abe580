"""Multi-token decode queries (q_len > 1: speculative / multi-token-prediction
steps) on the GPU against the oracle, element by element.

Query token i of a sequence with L cached tokens (the q_len new ones included)
sees tokens t < L - q_len + 1 + i; the oracle's causal pin fixes that reading.
"""
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


@pytest.mark.parametrize("Hq,Hkv,q_len", [
    (32, 8, 2), (32, 8, 3), (32, 8, 4),      # Llama-3 group of 4: 8, 12, 16 rows
    (16, 8, 2), (16, 8, 5), (16, 8, 8),      # group of 2
    (8, 8, 7), (8, 8, 16),                   # MHA: one head, up to 16 tokens
    (10, 2, 3),                              # group of 5: 15 rows
    (64, 8, 2),                              # group of 8: 16 rows
])
def test_group_and_q_len(Hq, Hkv, q_len):
    w = wl.random_case(700 + 31 * Hq + 7 * Hkv + q_len, B=5, Hq=Hq, Hkv=Hkv, max_len=260,
                       q_len=q_len)
    _parity(w)


@pytest.mark.parametrize("q_len", [2, 4])
def test_short_contexts(q_len):
    """L = 0, L < q_len (rows that see nothing give zeros and lse = -inf), L = q_len,
    and lengths at the tile edges."""
    lens = [0, 1, q_len - 1, q_len, q_len + 1, 15, 16, 17, 33]
    w = wl.random_case(800 + q_len, B=len(lens), Hq=32, Hkv=8, lens=lens, q_len=q_len)
    g = _parity(w)
    out = g.out.float().cpu()
    for b, L in enumerate(lens):
        for i in range(q_len):
            if L - q_len + 1 + i <= 0:
                assert torch.all(out[b, i] == 0)
                assert torch.all(torch.isneginf(g.lse[b, i].cpu()))


@pytest.mark.parametrize("num_ctas", [1, 3, 64, 151, 1000])
def test_any_split(num_ctas):
    w = wl.random_case(810, B=6, Hq=32, Hkv=8, max_len=600, q_len=3)
    _parity(w, num_ctas=num_ctas)


@pytest.mark.parametrize("P", [16, 64])
def test_page_sizes_and_hnd(P):
    for layout in ("NHD", "HND"):
        w = wl.random_case(820 + P, B=4, Hq=16, Hkv=4, page_size=P, max_len=5 * P, q_len=4,
                           layout=layout)
        _parity(w)


def test_last_row_equals_single_token_call():
    """The last of q_len query tokens sees the whole cache: the same row as a
    q_len = 1 call with that query, bit for bit (rows of the tensor-core tile
    are independent, and the split is the same)."""
    w = wl.random_case(830, B=5, Hq=32, Hkv=8, max_len=400, q_len=4)
    g = run_gpu(w)
    w1 = wl.random_case(830, B=5, Hq=32, Hkv=8, max_len=400, q_len=1)
    w1.q = w.q[:, -1:].contiguous()
    g1 = run_gpu(w1)
    assert torch.equal(g.out[:, -1:].view(torch.int16), g1.out.view(torch.int16))
    assert torch.equal(g.lse[:, -1:], g1.lse)


def test_bad_first_page_zeroes_every_row():
    w = wl.random_case(840, B=3, Hq=32, Hkv=8, lens=[40, 50, 60], q_len=3)
    d = device_inputs(w)
    bt = d["bt"].clone()
    bt[1, 0] = w.num_pages + 5
    g = run_gpu(w, d, block_table=bt)
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    ref, ref_lse, st = run_oracle(w, block_table=bt.cpu().numpy())
    assert st & 1
    assert_close(g.out64(), ref, "out")
    assert_close(g.lse64(), ref_lse, "lse")
    assert torch.all(g.out[1].float() == 0)


@pytest.mark.parametrize("Hq,q_len,num_ctas,single", [
    (32, 3, 0, False),     # one row group of 12 rows, whole units
    (32, 3, 40, False),    # units cut between CTAs: the bad rows cross the merge
    (32, 3, 40, True),     # ... merged inside the attention kernel
    (32, 8, 0, False),     # two row groups of 4 tokens in every CTA
    (32, 8, 40, False),
    (64, 2, 40, False),    # group of 8: 16 rows, the upper half of the tile
])
def test_bad_page_seen_by_the_newest_token_only(Hq, q_len, num_ctas, single):
    """A bad page that holds only the newest token (position L - 1 is the first
    slot of its page): only the last query row sees it, so only that row of the
    sequence is zeroed (lse = -inf); the rows before it keep their values. The
    oracle zeroes exactly the rows whose visible range holds the bad page."""
    P = 16
    lens = [P * 2 + 1, P * 3 + 1, 70, 45]  # sequences 0 and 1 end one token into a page
    w = wl.random_case(845 + Hq + q_len, B=len(lens), Hq=Hq, Hkv=8, lens=lens, q_len=q_len,
                       page_size=P)
    d = device_inputs(w)
    bt = d["bt"].clone()
    bt[0, 2] = -3                  # the page of sequence 0's newest token
    bt[1, 3] = w.num_pages + 1     # the page of sequence 1's newest token
    g = run_gpu(w, d, block_table=bt, num_ctas=num_ctas, single_launch=single)
    assert int(g.err.item()) & zl.DEVERR_BAD_PAGE
    ref, ref_lse, st = run_oracle(w, block_table=bt.cpu().numpy())
    assert st & 1
    assert_close(g.out64(), ref, "out")
    assert_close(g.lse64(), ref_lse, "lse")
    out = g.out.float().cpu()
    for b in (0, 1):
        assert torch.all(out[b, -1] == 0)
        assert torch.all(torch.isneginf(g.lse[b, -1].cpu()))
        assert torch.all(out[b, :-1].abs().sum(-1) > 0)  # the other rows are not zeroed


def test_full_size_llama3_8b_mtp_sampled():
    """Llama-3-8B decode shape at batch 64 with 4 query tokens per sequence,
    sampled rows against the oracle at full context lengths."""
    w = wl.random_case(850, B=64, Hq=32, Hkv=8, max_len=4096, q_len=4, pool_factor=1.1)
    g = run_gpu(w)
    rng = np.random.default_rng(5)
    bs = rng.choice(w.B, size=6, replace=False)
    sub_lens = w.seq_lens[bs]
    ws = wl.build_workload("sampled", 0, B=len(bs), Hq=32, Hkv=8, D_qk=128,
                           page_size=w.page_size, seq_lens=sub_lens,
                           block_table=w.block_table[bs], num_pages=w.num_pages, scale=w.scale,
                           q_len=4, values=False)
    ws.q, ws.k_pool, ws.v_pool = w.q[bs].contiguous(), w.k_pool, w.v_pool
    ref, ref_lse, st = run_oracle(ws)
    assert st == 0
    assert_close(g.out64()[bs], ref, "sampled out")
    assert_close(g.lse64()[bs], ref_lse, "sampled lse")


# More query rows than one tensor-core tile holds (g * q_len > 16): the tokens
# go in groups of 16 / g that run side by side in one launch (one launch per
# group in single-launch mode), each group with its own causal limits. Two
# groups run in every CTA (half the kv heads per CTA); more groups split the
# grid's CTAs between them.
@pytest.mark.parametrize("Hq,Hkv,q_len", [
    (32, 8, 8), (32, 8, 5), (32, 8, 13),     # group of 4: 4 + 4, 4 + 1, 4 + 4 + 4 + 1
    (64, 8, 3),                              # group of 8: 2 + 1
    (128, 8, 2),                             # group of 16: one token per group
    (16, 8, 17),                             # group of 2: 8 + 8 + 1
    (8, 1, 3),                               # one kv head (1 per CTA): 2 + 1
    (16, 4, 5),                              # four kv heads (2 per CTA): 4 + 1
])
def test_token_groups(Hq, Hkv, q_len):
    w = wl.random_case(900 + 31 * Hq + 7 * Hkv + q_len, B=5, Hq=Hq, Hkv=Hkv, max_len=300,
                       q_len=q_len)
    _parity(w)


def test_token_groups_short_contexts():
    """Groups whose rows see nothing (L < q_len), and lengths at the tile edges."""
    q_len = 6
    lens = [0, 1, 3, 5, 6, 7, 15, 16, 17, 21, 22, 40]
    w = wl.random_case(910, B=len(lens), Hq=32, Hkv=8, lens=lens, q_len=q_len)
    g = _parity(w)
    out = g.out.float().cpu()
    for b, L in enumerate(lens):
        for i in range(q_len):
            if L - q_len + 1 + i <= 0:
                assert torch.all(out[b, i] == 0)
                assert torch.all(torch.isneginf(g.lse[b, i].cpu()))


@pytest.mark.parametrize("num_ctas", [1, 7, 151, 1000])
def test_token_groups_any_split(num_ctas):
    w = wl.random_case(920, B=6, Hq=32, Hkv=8, max_len=700, q_len=8)
    _parity(w, num_ctas=num_ctas)


def test_token_groups_single_launch():
    w = wl.random_case(930, B=6, Hq=32, Hkv=8, max_len=700, q_len=7)
    d = device_inputs(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.empty((w.B, w.q_len, w.Hq), dtype=torch.float32, device="cuda")
    out = zl.decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], page_size=w.page_size,
                         scale=w.scale, lse=lse, err_flags=err, max_seq_len=w.max_seq_len,
                         single_launch=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, ref_lse, _ = run_oracle(w)
    assert_close(out.float().cpu().numpy(), ref, "single launch, token groups")
    assert_close(lse.double().cpu().numpy(), ref_lse, "single launch, token groups lse")


def test_token_groups_last_row_matches_single_token_call():
    """The last of 8 query tokens (in the second group) sees the whole cache:
    the same row as a q_len = 1 call with that query. The two-group launch
    cuts the tile line with its own plan (half the kv heads per CTA), so the
    rounding order differs from the one-token call: equal within the
    tolerance, not bit for bit."""
    w = wl.random_case(940, B=5, Hq=32, Hkv=8, max_len=400, q_len=8)
    d = device_inputs(w)
    g = run_gpu(w, d)
    q1 = d["q"][:, -1:].contiguous()
    out1 = zl.decode_attn(q1, d["k"], d["v"], d["bt"], d["sl"], page_size=w.page_size,
                          scale=w.scale, max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert_close(g.out[:, -1].double().cpu().numpy(), out1[:, 0].double().cpu().numpy(),
                 "last of 8 tokens vs a one-token call")


# More than 16 query heads per kv head (many-head MQA, wide GQA): each token's
# g heads go in ceil(g / 16) chunks of at most 16 rows (the last may be
# smaller), one row group per (token, chunk); two groups share every CTA, more
# split the grid.
@pytest.mark.parametrize("Hq,Hkv,q_len", [
    (32, 1, 1),                              # MQA, 32 heads: two chunks of 16
    (48, 1, 1),                              # three chunks of 16
    (17, 1, 1),                              # chunks of 9 and 8
    (71, 1, 1),                              # five chunks: 15, 15, 15, 15, 11
    (64, 2, 1),                              # g = 32 over two kv heads
    (32, 1, 3),                              # 3 tokens x 2 chunks: six groups
    (40, 2, 2),                              # g = 20: chunks of 10, 2 tokens
])
def test_many_heads_per_kv_head(Hq, Hkv, q_len):
    w = wl.random_case(950 + 13 * Hq + 5 * Hkv + q_len, B=5, Hq=Hq, Hkv=Hkv, max_len=300,
                       q_len=q_len)
    _parity(w)


@pytest.mark.parametrize("num_ctas", [1, 3, 152, 777])
def test_many_heads_any_split(num_ctas):
    w = wl.random_case(960, B=4, Hq=32, Hkv=1, max_len=600, q_len=2)
    _parity(w, num_ctas=num_ctas)


def test_many_heads_short_contexts():
    """One CTA per unit (no merge) with head chunks; lengths at tile edges and
    rows that see nothing."""
    lens = [0, 1, 2, 15, 16, 17, 33, 40]
    w = wl.random_case(970, B=len(lens), Hq=48, Hkv=1, lens=lens, q_len=2)
    g = _parity(w)
    out = g.out.float().cpu()
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(g.lse[0].cpu()))
    assert torch.all(out[1, 0] == 0)  # token 0 of a 1-token cache sees nothing


def test_many_heads_single_launch():
    """Single-launch mode: one launch per (token, head chunk) group, each with
    its merge inside the attention kernel."""
    w = wl.random_case(980, B=6, Hq=32, Hkv=1, max_len=700, q_len=2)
    d = device_inputs(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.empty((w.B, w.q_len, w.Hq), dtype=torch.float32, device="cuda")
    out = zl.decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], page_size=w.page_size,
                         scale=w.scale, lse=lse, err_flags=err, max_seq_len=w.max_seq_len,
                         single_launch=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, ref_lse, _ = run_oracle(w)
    assert_close(out.float().cpu().numpy(), ref, "single launch, head chunks")
    assert_close(lse.double().cpu().numpy(), ref_lse, "single launch, head chunks lse")


@pytest.mark.parametrize("Hq,Hkv,q_len,num_ctas", [
    (128, 1, 60, 0),     # 480 row groups: more than the default grid's CTAs
    (32, 1, 2, 3),       # 4 groups over 3 CTAs: one CTA each
    (32, 8, 13, 7),      # 4 token groups over 7 CTAs: one CTA each
    (32, 1, 3, 13),      # 6 groups, 2 CTAs each
    (32, 8, 8, 5),       # two groups in every CTA
])
def test_row_groups_stay_inside_the_workspace(Hq, Hkv, q_len, num_ctas):
    """A workspace of exactly the reported size, followed by a guard region:
    every launch plan of row groups (one CTA per group when there are more
    groups than CTAs) leaves the guard untouched and matches the oracle."""
    w = wl.random_case(990 + Hq + 3 * q_len + num_ctas, B=4, Hq=Hq, Hkv=Hkv, max_len=400,
                       q_len=q_len)
    d = device_inputs(w)
    out = torch.empty((w.B, w.q_len, w.Hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.q_len, w.Hq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(page_size=w.page_size, scale=w.scale, Hkv=w.Hkv, D_v=128, lse=lse,
              err_flags=err, num_ctas=num_ctas)
    n = zl.workspace_size(zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, **kw))
    guard = 1 << 20
    buf = torch.full((n + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, workspace=buf[:n], **kw)
    zl.call(p, mla=False)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert bool(torch.all(buf[n:] == 0xA5)), "a launch wrote past the workspace"
    ref, ref_lse, _ = run_oracle(w)
    assert_close(out.double().cpu().numpy(), ref, "row groups, exact workspace")
    assert_close(lse.double().cpu().numpy(), ref_lse, "row groups, exact workspace lse")


@pytest.mark.parametrize("Hq,Hkv,q_len", [(32, 8, 8), (32, 1, 1)])
def test_two_groups_per_cta_capture_into_a_cuda_graph(Hq, Hkv, q_len):
    """A two-group call (8 tokens at g = 4; 32 heads on one kv head) and its
    merge launch capture into a CUDA graph; replays give the eager bits."""
    w = wl.random_case(1010 + Hq + q_len, B=6, Hq=Hq, Hkv=Hkv, max_len=1500, q_len=q_len)
    d = device_inputs(w)
    out = torch.empty((w.B, w.q_len, w.Hq, 128), dtype=torch.bfloat16, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=w.page_size,
                       scale=w.scale, Hkv=w.Hkv, D_v=128)
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
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    ref, _, _ = run_oracle(w)
    assert_close(out.double().cpu().numpy(), ref, "two groups per CTA, graph replay")
