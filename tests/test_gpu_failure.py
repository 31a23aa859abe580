"""Failure detection without a GPU fault: a call whose pipeline wait runs out
reports ZL_DEVERR_TIMEOUT on the host and leaves the context usable.

The stall is made with the ZL_DECODE_TEST_STALL hook: the attention kernel's
producer waits on a word that nothing sets, its bounded wait (~50 ms) runs
out, every CTA stops early. Nothing traps, nothing hangs; the next call on the
same stream, buffers and workspace computes the right result."""
import numpy as np
import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs, run_oracle

pytestmark = pytest.mark.gpu


def _setup(w, single_launch):
    d = device_inputs(w)
    out = torch.empty(w.B, w.q_len, w.Hq, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.B, w.q_len, w.Hq, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=w.page_size,
                       scale=w.scale, Hkv=w.Hkv, D_v=128, lse=lse, err_flags=err,
                       single_launch=single_launch)
    ws = torch.zeros(zl.workspace_size(p), dtype=torch.uint8, device="cuda")
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    return p, out, lse, err, ws


@pytest.mark.parametrize("single_launch", [False, True])
def test_stalled_call_reports_timeout_and_next_call_is_correct(single_launch):
    w = wl.random_case(990, B=6, Hq=32, Hkv=8, max_len=1500)
    p, out, lse, err, ws = _setup(w, single_launch)
    ref, ref_lse, st = run_oracle(w)
    assert st == 0

    p.flags |= zl.TEST_STALL
    zl.call(p, mla=False)            # returns at once: the error is a device flag
    torch.cuda.synchronize()         # the context is fine: no exception here
    assert int(err.item()) & zl.DEVERR_TIMEOUT

    p.flags &= ~zl.TEST_STALL
    err.zero_()
    zl.call(p, mla=False)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "out after a timeout")
    assert_close(lse.cpu().numpy().astype(np.float64), ref_lse, "lse after a timeout")


def test_timeout_is_reported_within_its_bound():
    """The stalled call ends in well under a second (its wait is bounded)."""
    w = wl.random_case(991, B=3, Hq=16, Hkv=4, max_len=300)
    p, out, lse, err, ws = _setup(w, False)
    p.flags |= zl.TEST_STALL
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    zl.call(p, mla=False)
    b.record()
    torch.cuda.synchronize()
    assert int(err.item()) & zl.DEVERR_TIMEOUT
    ms = a.elapsed_time(b)
    assert 40.0 <= ms < 1000.0, ms
