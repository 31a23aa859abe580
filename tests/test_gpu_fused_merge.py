"""Single-launch split-KV (ZL_DECODE_SINGLE_LAUNCH): the last warp to finish
a piece of a (sequence, kv head) merges the partials, through arrival counters
in the workspace. These tests cover what that adds: the counters returning to
zero, stale counters from another call ignored, CUDA graph capture and replay,
results that do not depend on arrival order, and bit-identity with the
two-launch path (merge kernel as a programmatic dependent launch)."""
import numpy as np
import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs, run_oracle

pytestmark = pytest.mark.gpu


def _setup(w, num_ctas=0, single_launch=True):
    d = device_inputs(w)
    out = torch.empty(w.B, w.q_len, w.Hq, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.B, w.q_len, w.Hq, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=w.page_size,
                       scale=w.scale, Hkv=w.Hkv, D_v=128, lse=lse, err_flags=err,
                       num_ctas=num_ctas, layout=w.layout, single_launch=single_launch)
    ws = torch.zeros(zl.workspace_size(p), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    p.keep_alive = d  # the params hold raw pointers into these tensors
    return p, out, lse, err, ws


def _check(w, out, lse, err):
    torch.cuda.synchronize()
    ref, ref_lse, st = run_oracle(w)
    assert st == 0 and int(err.item()) == 0
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "out")
    assert_close(lse.cpu().numpy().astype(np.float64), ref_lse, "lse")


def test_counters_return_to_zero_and_calls_repeat_bit_identically():
    w = wl.random_case(960, B=6, Hq=32, Hkv=8, max_len=900)
    p, out, lse, err, ws = _setup(w, num_ctas=97)
    n_count = w.B * w.Hkv * 8
    outs = []
    for _ in range(3):
        zl.call(p, mla=False)
        torch.cuda.synchronize()
        assert int(ws[:n_count].count_nonzero().item()) == 0
        outs.append(out.clone())
    _check(w, out, lse, err)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_stale_counters_of_another_call_are_ignored():
    """Counter words tagged with another call (as a call stopped by a device
    error would leave them) do not disturb the next call."""
    w = wl.random_case(961, B=5, Hq=32, Hkv=8, max_len=700, q_len=2)
    p, out, lse, err, ws = _setup(w, num_ctas=64)
    zl.call(p, mla=False)
    torch.cuda.synchronize()
    good = out.clone()
    words = ws[: w.B * w.Hkv * 8].view(torch.int64)
    words.copy_(torch.full_like(words, (0x7FFFFFF0 << 32) | 1))
    out.zero_()
    zl.call(p, mla=False)
    _check(w, out, lse, err)
    assert torch.equal(out.view(torch.int16), good.view(torch.int16))


def test_workspace_reused_across_shapes():
    a = wl.random_case(962, B=4, Hq=32, Hkv=8, max_len=1200)
    b = wl.random_case(963, B=9, Hq=16, Hkv=4, max_len=400, q_len=3)
    pa, oa, la, ea, ws = _setup(a, num_ctas=50)
    pb, ob, lb, eb, _ = _setup(b, num_ctas=77)
    big = torch.zeros(max(ws.numel(), zl.workspace_size(pb)), dtype=torch.uint8, device="cuda")
    for p in (pa, pb):
        p.workspace, p.workspace_bytes = big.data_ptr(), big.numel()
    zl.call(pa, mla=False)
    zl.call(pb, mla=False)
    zl.call(pa, mla=False)
    _check(a, oa, la, ea)
    _check(b, ob, lb, eb)


def test_cuda_graph_capture_and_replay():
    """The call is capturable (no allocation, no sync, one stream); replays of
    the captured graph give the eager result bit for bit."""
    w = wl.random_case(964, B=8, Hq=32, Hkv=8, max_len=1500)
    p, out, lse, err, ws = _setup(w)
    zl.call(p, mla=False)
    torch.cuda.synchronize()
    eager = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        zl.call(p, mla=False, stream=s)
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    _check(w, out, lse, err)


@pytest.mark.parametrize("num_ctas", [2, 3, 152, 600, 3000])
def test_split_results_independent_of_grid_timing(num_ctas):
    """Heavily split units (many pieces per (sequence, kv head)), including
    CTAs with empty ranges, against the oracle."""
    w = wl.random_case(965 + num_ctas, B=3, Hq=32, Hkv=8, lens=[2000, 37, 700])
    p, out, lse, err, ws = _setup(w, num_ctas=num_ctas)
    zl.call(p, mla=False)
    _check(w, out, lse, err)


@pytest.mark.parametrize("case", [
    dict(B=7, Hq=32, Hkv=8, max_len=3000, num_ctas=0),
    dict(B=3, Hq=32, Hkv=8, max_len=9000, num_ctas=0),
    dict(B=5, Hq=16, Hkv=4, max_len=800, num_ctas=333, q_len=3),
    dict(B=4, Hq=64, Hkv=8, max_len=2000, num_ctas=17),
    dict(B=6, Hq=8, Hkv=1, max_len=1500, num_ctas=40, q_len=2),
    dict(B=6, Hq=4, Hkv=4, max_len=1500, num_ctas=40, q_len=16),
])
def test_single_launch_bit_identical_to_two_launches(case):
    case = dict(case)
    num_ctas = case.pop("num_ctas")
    w = wl.random_case(970 + case["B"], **case)
    p1, o1, l1, e1, _ = _setup(w, num_ctas=num_ctas, single_launch=True)
    p2, o2, l2, e2, _ = _setup(w, num_ctas=num_ctas, single_launch=False)
    zl.call(p1, mla=False)
    zl.call(p2, mla=False)
    _check(w, o1, l1, e1)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
