"""The C-ABI library: it builds, loads, exports what the header declares, and
rejects bad arguments on the host before touching the GPU (CPU only)."""
import ctypes

import pytest
import torch

import paged_decode_attention_gqa_gb300 as zl


def test_builds_and_exports_every_declared_symbol():
    lib = zl.lib()
    names = zl.declared_symbols()
    assert {"zl_decode_attn", "zl_decode_attn_mla", "zl_decode_attn_workspace_size",
            "zl_decode_attn_mla_workspace_size", "zl_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    lib = zl.lib()
    for code in range(5):
        assert lib.zl_status_string(code)
    assert lib.zl_status_string(0) == b"ok"


def _params(**over):
    """A fully valid-looking GQA parameter block with fake aligned pointers."""
    p = zl.Params()
    p.struct_size = ctypes.sizeof(zl.Params)
    fake = 1 << 20
    p.q = p.k_pool = p.v_pool = p.out = fake
    p.block_table = p.seq_lens = fake
    p.page_stride, p.token_stride, p.head_stride = 16 * 8 * 128, 8 * 128, 128
    p.block_table_stride = 8
    p.B, p.q_len, p.Hq, p.Hkv, p.D_qk, p.D_v = 4, 1, 32, 8, 128, 128
    p.page_size, p.num_pages = 16, 64
    p.scale = 128 ** -0.5
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over,code", [
    (dict(struct_size=8), zl.ERR_INVALID_ARG),
    (dict(B=0), zl.ERR_INVALID_ARG),
    (dict(Hkv=0), zl.ERR_INVALID_ARG),
    (dict(Hq=30), zl.ERR_INVALID_ARG),           # Hq % Hkv != 0
    (dict(scale=0.0), zl.ERR_INVALID_ARG),
    (dict(scale=float("nan")), zl.ERR_INVALID_ARG),
    (dict(num_ctas=-1), zl.ERR_INVALID_ARG),
    (dict(q=None), zl.ERR_INVALID_ARG),
    (dict(v_pool=None), zl.ERR_INVALID_ARG),
    (dict(out=None), zl.ERR_INVALID_ARG),
    (dict(q=(1 << 20) + 2), zl.ERR_INVALID_ARG),  # misaligned
    (dict(token_stride=100), zl.ERR_INVALID_ARG),  # not a multiple of 8 elements
    (dict(D_qk=64, D_v=64), zl.ERR_UNSUPPORTED),
    (dict(Hq=8 * 129), zl.ERR_UNSUPPORTED),        # 129 query heads per kv head
    (dict(q_len=129), zl.ERR_UNSUPPORTED),         # more query tokens than one call takes
    (dict(q_len=5, shared_prefix_pages=1), zl.ERR_UNSUPPORTED),  # 4 x 5 rows, shared prefix
    (dict(q_len=0), zl.ERR_INVALID_ARG),
    (dict(flags=2), zl.ERR_INVALID_ARG),           # unknown flag bit
    (dict(flags=zl.TEST_STALL | 4), zl.ERR_INVALID_ARG),
    (dict(page_size=8), zl.ERR_UNSUPPORTED),
    (dict(B=5000), zl.ERR_UNSUPPORTED),
    (dict(k_new=1 << 20), zl.ERR_INVALID_ARG),     # fused append: K rows without V rows
    (dict(v_new=1 << 20), zl.ERR_INVALID_ARG),     # ... V rows without K rows
    (dict(k_new=(1 << 20) + 8, v_new=1 << 20), zl.ERR_INVALID_ARG),  # misaligned new rows
])
def test_host_validation(over, code):
    p = _params(**over)
    assert zl.lib().zl_decode_attn(ctypes.byref(p), None) == code


def test_null_params():
    assert zl.lib().zl_decode_attn(None, None) == zl.ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert zl.lib().zl_decode_attn_workspace_size(None, ctypes.byref(n)) == zl.ERR_INVALID_ARG


def test_no_cpu_fallback():
    """Without a GPU the valid call fails loudly instead of computing on the CPU."""
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = _params()
    assert zl.lib().zl_decode_attn(ctypes.byref(p), None) != zl.OK


def _mla_params(**over):
    p = _params(Hq=128, Hkv=1, D_qk=576, D_v=512, page_size=64, v_pool=None)
    p.page_stride, p.token_stride, p.head_stride = 64 * 576, 576, 576
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over,code", [
    (dict(struct_size=8), zl.ERR_INVALID_ARG),
    (dict(Hkv=2, Hq=128), zl.ERR_INVALID_ARG),
    (dict(v_pool=1 << 20), zl.ERR_INVALID_ARG),   # MLA takes V from the latent row
    (dict(q=None), zl.ERR_INVALID_ARG),
    (dict(D_qk=512, D_v=512), zl.ERR_UNSUPPORTED),
    (dict(Hq=64), zl.ERR_UNSUPPORTED),
    (dict(page_size=16), zl.ERR_UNSUPPORTED),
    (dict(page_size=48), zl.ERR_UNSUPPORTED),
    (dict(page_size=32), zl.ERR_UNSUPPORTED),
    (dict(B=600, q_len=2), zl.ERR_UNSUPPORTED),    # 1200 (sequence, token) pairs
    (dict(B=3000), zl.ERR_UNSUPPORTED),
    (dict(flags=zl.SINGLE_LAUNCH), zl.ERR_UNSUPPORTED),
    (dict(flags=zl.TEST_STALL), zl.ERR_UNSUPPORTED),
    (dict(flags=4), zl.ERR_INVALID_ARG),
    (dict(k_new=1 << 20, v_new=1 << 20), zl.ERR_INVALID_ARG),  # latent rows only: no v_new
    (dict(v_new=1 << 20), zl.ERR_INVALID_ARG),
    (dict(k_new=(1 << 20) + 2), zl.ERR_INVALID_ARG),
])
def test_mla_host_validation(over, code):
    p = _mla_params(**over)
    assert zl.lib().zl_decode_attn_mla(ctypes.byref(p), None) == code


def _append_params(**over):
    """A valid-looking zl_kv_append parameter block with fake aligned pointers."""
    p = zl.AppendParams()
    p.struct_size = ctypes.sizeof(zl.AppendParams)
    fake = 1 << 20
    p.k_new = p.v_new = p.k_pool = p.v_pool = p.block_table = p.seq_lens = fake
    p.page_stride, p.token_stride, p.head_stride = 16 * 8 * 128, 8 * 128, 128
    p.block_table_stride = 8
    p.B, p.q_len, p.Hkv, p.D_k, p.D_v, p.page_size, p.num_pages = 4, 1, 8, 128, 128, 16, 64
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("over", [
    dict(struct_size=8), dict(B=0), dict(q_len=0), dict(Hkv=0), dict(page_size=0),
    dict(num_pages=0), dict(block_table_stride=0), dict(D_k=12), dict(D_k=2048), dict(D_v=4),
    dict(k_new=None), dict(k_pool=None), dict(block_table=None), dict(seq_lens=None),
    dict(v_new=None),                        # V pool without new V rows
    dict(v_pool=None),                       # new V rows without a V pool
    dict(k_new=(1 << 20) + 8),               # misaligned
    dict(seq_lens=(1 << 20) + 2),
    dict(token_stride=100), dict(head_stride=0),
])
def test_append_host_validation(over):
    p = _append_params(**over)
    assert zl.lib().zl_kv_append(ctypes.byref(p), None) == zl.ERR_INVALID_ARG


def test_append_null_params_and_no_cpu_fallback():
    assert zl.lib().zl_kv_append(None, None) == zl.ERR_INVALID_ARG
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for over in (dict(), dict(v_new=None, v_pool=None, D_k=576, D_v=0)):
        p = _append_params(**over)
        assert zl.lib().zl_kv_append(ctypes.byref(p), None) == zl.ERR_CUDA


def test_binding_constants_match_the_header():
    """The Python names mirror the header's #defines."""
    import re
    text = open(zl.HEADER).read()

    def define(name):
        m = re.search(r"#define\s+" + name + r"\s+\(?([0-9a-fx]+)u?(?:\s*<<\s*(\d+))?", text)
        assert m, name
        v = int(m.group(1), 0)
        return v << int(m.group(2)) if m.group(2) else v

    assert define("ZL_DECODE_SINGLE_LAUNCH") == zl.SINGLE_LAUNCH
    assert define("ZL_DECODE_TEST_STALL") == zl.TEST_STALL
    assert define("ZL_DEVERR_BAD_PAGE") == zl.DEVERR_BAD_PAGE
    assert define("ZL_DEVERR_BAD_PREFIX") == zl.DEVERR_BAD_PREFIX
    assert define("ZL_NOALLOC_WORKSPACE_BYTES") == zl.NOALLOC_WORKSPACE_BYTES
