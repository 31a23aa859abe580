"""zl_decode_attn_noalloc: the entry point for callers that cannot allocate
device memory (no workspace argument; the library's own static scratch).

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test. It must pass alone in a fresh
process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs, run_oracle

pytestmark = pytest.mark.gpu


def _params(w, d, out, lse, err=None, single_launch=False, max_seq_len=None):
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=w.page_size,
                       scale=w.scale, Hkv=w.Hkv, D_v=w.D_v, lse=lse, err_flags=err,
                       max_seq_len=w.max_seq_len if max_seq_len is None else max_seq_len,
                       single_launch=single_launch)
    return p


def _noalloc_against_oracle(w, single_launch, max_seq_len=None):
    """One zl_decode_attn_noalloc call through the C ABI, checked against the oracle."""
    d = device_inputs(w)
    out = torch.full((w.B, w.q_len, w.Hq, w.D_v), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((w.B, w.q_len, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = _params(w, d, out, lse, err, single_launch, max_seq_len)
    stream = torch.cuda.current_stream()
    rc = zl.lib().zl_decode_attn_noalloc(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream))
    assert rc == zl.OK, zl.lib().zl_status_string(rc)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, ref_lse, st = run_oracle(w)
    assert st == 0
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"{w.name} noalloc out")
    assert_close(lse.cpu().numpy().astype(np.float64), ref_lse, f"{w.name} noalloc lse")
    return p


def test_noalloc_matches_workspace_entry_point_twice():
    w = wl.llama3_8b_decode(B=16)
    d = device_inputs(w)
    # the existing entry point, with a caller-owned workspace
    ref_out = torch.empty(w.B, 1, w.Hq, w.D_v, dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(w.B, 1, w.Hq, dtype=torch.float32, device="cuda")
    p = _params(w, d, ref_out, ref_lse)
    ws = torch.zeros(zl.workspace_size(p), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    stream = torch.cuda.current_stream()
    assert zl.lib().zl_decode_attn(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream)) == zl.OK
    torch.cuda.synchronize()
    # the allocation-free entry point, called twice in a row through the C ABI
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        q = _params(w, d, out, lse)
        rc = zl.lib().zl_decode_attn_noalloc(ctypes.byref(q), ctypes.c_void_p(stream.cuda_stream))
        assert rc == zl.OK, zl.lib().zl_status_string(rc)
        torch.cuda.synchronize()
        assert_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), "noalloc out")
        assert_close(lse.cpu().numpy(), ref_lse.cpu().numpy(), "noalloc lse")


def test_noalloc_rejects_a_workspace_beyond_its_maximum():
    w = wl.random_case(910, B=2, Hq=64, Hkv=4, lens=[40, 60])
    d = device_inputs(w)
    out = torch.empty(2, 1, 64, 128, dtype=torch.bfloat16, device="cuda")
    p = _params(w, d, out, None)
    p.num_ctas = 20000  # 20000 CTAs x 2 slots x 4 kv heads x 16 rows x 512 B > 8 MiB
    p.max_seq_len = 0
    assert zl.workspace_size(p) > zl.NOALLOC_WORKSPACE_BYTES
    stream = torch.cuda.current_stream()
    rc = zl.lib().zl_decode_attn_noalloc(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream))
    assert rc == zl.ERR_WORKSPACE


def test_noalloc_single_launch_after_calls_of_other_shapes():
    """The one mode whose calls share state through the array: single-launch
    arrival counters. A plain call leaves partials where a larger single-launch
    call counts; the entry point clears its counters first, so each call in
    this sequence matches the oracle (and the last repeats a shape)."""
    small = wl.random_case(920, B=4, Hq=32, Hkv=8, max_len=900)
    large = wl.random_case(921, B=24, Hq=32, Hkv=8, max_len=700)
    mqa = wl.random_case(922, B=5, Hq=32, Hkv=1, max_len=500, q_len=2)
    _noalloc_against_oracle(small, single_launch=False, max_seq_len=0)
    _noalloc_against_oracle(large, single_launch=True, max_seq_len=0)
    _noalloc_against_oracle(small, single_launch=False, max_seq_len=0)
    _noalloc_against_oracle(small, single_launch=True, max_seq_len=0)
    # 32 heads on one kv head, two query tokens: four row groups, one launch
    # each in single-launch mode, sharing the array's slots and counters
    _noalloc_against_oracle(mqa, single_launch=True, max_seq_len=0)
    _noalloc_against_oracle(mqa, single_launch=False, max_seq_len=0)
    _noalloc_against_oracle(large, single_launch=True, max_seq_len=0)


def test_noalloc_takes_a_smaller_grid_when_the_default_one_does_not_fit():
    """The 70B head shape (64 query heads over 8 kv heads) at the default grid
    needs more partial slots than the array holds (152 CTAs x 2 slots x 8 kv
    heads x 8 rows, ~10 MB); the call runs on a grid that fits instead."""
    w = wl.random_case(923, B=12, Hq=64, Hkv=8, max_len=3000)
    d = device_inputs(w)
    out = torch.empty(w.B, 1, w.Hq, 128, dtype=torch.bfloat16, device="cuda")
    p = _params(w, d, out, None, max_seq_len=0)
    assert zl.workspace_size(p) > zl.NOALLOC_WORKSPACE_BYTES
    _noalloc_against_oracle(w, single_launch=False, max_seq_len=0)
    _noalloc_against_oracle(w, single_launch=True, max_seq_len=0)


def test_noalloc_with_fused_append():
    """The fused KV append through the no-workspace entry point: the same pools
    and output, bit for bit, as the workspace entry point with the same rows."""
    w = wl.random_case(925, B=6, Hq=32, Hkv=8, max_len=400, q_len=2)
    k_new, v_new = wl.new_token_rows(925, w.B, 2, 8, 128, 128)
    kn, vn = k_new.cuda(), v_new.cuda()
    outs, pools = [], []
    for noalloc in (False, True):
        d = device_inputs(w)
        out = torch.empty((w.B, w.q_len, w.Hq, w.D_v), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        if noalloc:
            p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out,
                               page_size=w.page_size, scale=w.scale, Hkv=w.Hkv, D_v=w.D_v,
                               err_flags=err, max_seq_len=w.max_seq_len, k_new=kn, v_new=vn)
            zl.call_noalloc(p)
        else:
            zl.decode_attn(d["q"], d["k"], d["v"], d["bt"], d["sl"], page_size=w.page_size,
                           scale=w.scale, out=out, err_flags=err, max_seq_len=w.max_seq_len,
                           k_new=kn, v_new=vn)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append(out)
        pools.append((d["k"], d["v"]))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    for a, b in zip(pools[0], pools[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
