"""zl_decode_attn_noalloc: the entry point for callers that cannot allocate
device memory (no workspace argument; the library's own static scratch).

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test. It must pass alone in a fresh
process and after the rest of the suite.
"""
import ctypes

import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl
from paged_decode_attention_gqa_gb300 import workloads as wl
from parity import assert_close, device_inputs

pytestmark = pytest.mark.gpu


def _params(w, d, out, lse):
    p = zl.make_params(d["q"], d["k"], d["v"], d["bt"], d["sl"], out, page_size=w.page_size,
                       scale=w.scale, Hkv=w.Hkv, D_v=w.D_v, lse=lse, max_seq_len=w.max_seq_len)
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
    assert zl.workspace_size(p) > (8 << 20)
    stream = torch.cuda.current_stream()
    rc = zl.lib().zl_decode_attn_noalloc(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream))
    assert rc == zl.ERR_WORKSPACE
