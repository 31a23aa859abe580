"""Input generators: determinism and the structure each workload promises (CPU)."""
import numpy as np
import torch

from paged_decode_attention_gqa_gb300 import workloads as wl


def test_tiny_is_deterministic_and_poisoned():
    a, b = wl.tiny_gqa(), wl.tiny_gqa()
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))
    assert list(a.seq_lens) == [17, 64, 100, 256]
    used = np.unique(np.concatenate([a.block_table[i, :(L + 15) // 16]
                                     for i, L in enumerate(a.seq_lens)]))
    assert used.size == 29 and a.num_pages == 64
    unused = np.setdiff1d(np.arange(64), used)
    assert torch.isnan(a.k_pool[torch.from_numpy(unused)].float()).all()
    assert torch.isnan(a.v_pool[torch.from_numpy(unused)].float()).all()
    # tail of the 17-token sequence: slot 1.. of its second page are NaN
    last = a.block_table[0, 1]
    assert torch.isnan(a.k_pool[last, 1:].float()).all()
    assert not torch.isnan(a.k_pool[last, 0].float()).any()
    assert not torch.isnan(a.q.float()).any()


def test_other_seed_differs():
    a, b = wl.tiny_gqa(seed=1), wl.tiny_gqa(seed=2)
    assert not torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))


def test_hnd_is_a_permutation_of_nhd():
    a = wl.tiny_gqa()
    h = wl.tiny_gqa(layout="HND")
    assert torch.equal(a.k_pool.view(torch.int16),
                       h.k_pool.permute(0, 2, 1, 3).contiguous().view(torch.int16))
    assert h.strides == (2 * 16 * 128, 128, 16 * 128)


def test_structures_of_large_workloads():
    c2 = wl.llama3_8b_decode(values=False)
    assert c2.B == 64 and c2.Hq == 32 and c2.Hkv == 8 and c2.page_size == 16
    assert c2.seq_lens.min() >= 512 and c2.seq_lens.max() <= 4096
    pages = ((c2.seq_lens + 15) // 16).sum()
    assert c2.num_pages == int(np.ceil(1.25 * pages))
    assert len(c2.notes["k_scaled_channels"]) == 4

    c3 = wl.llama70b_prefix_decode(values=False)
    assert c3.B == 128 and c3.Hq == 64 and c3.Hkv == 8
    assert (c3.seq_lens >= 2049).all() and (c3.seq_lens <= 2048 + 6144).all()
    assert (c3.block_table[:, :128] == c3.block_table[0, :128]).all()
    priv = np.concatenate([c3.block_table[i, 128:(L + 15) // 16]
                           for i, L in enumerate(c3.seq_lens)])
    assert np.unique(priv).size == priv.size
    assert not np.isin(priv, c3.block_table[0, :128]).any()

    c4 = wl.long_context_decode(values=False)
    assert c4.page_size == 64 and c4.B == 8
    assert c4.seq_lens.min() >= 32768 and c4.seq_lens.max() <= 131072

    c5 = wl.mla_decode(values=False)
    assert c5.mla and c5.Hkv == 1 and c5.D_qk == 576 and c5.D_v == 512
    assert abs(c5.scale - 192 ** -0.5) < 1e-15

    m = wl.mqa32_decode(values=False)
    assert m.B == 64 and m.Hq == 32 and m.Hkv == 1 and m.page_size == 16 and not m.mla
    assert m.seq_lens.min() >= 512 and m.seq_lens.max() <= 4096
    assert m.num_pages == int(np.ceil(1.25 * ((m.seq_lens + 15) // 16).sum()))


def test_pages_are_distinct_without_prefix():
    c2 = wl.llama3_8b_decode(values=False)
    ids = np.concatenate([c2.block_table[i, :(L + 15) // 16] for i, L in enumerate(c2.seq_lens)])
    assert np.unique(ids).size == ids.size
    assert ids.min() >= 0 and ids.max() < c2.num_pages


def test_random_case_structure():
    w = wl.random_case(7, B=6, Hq=16, Hkv=4, lens=[1, 15, 16, 17, 0, 300])
    assert w.q.shape == (6, 1, 16, 128) and w.k_pool.shape[1:] == (16, 4, 128)
    assert (w.block_table[4] == -1).all()
    h = wl.random_case(7, B=6, Hq=16, Hkv=4, lens=[1, 15, 16, 17, 0, 300], layout="HND")
    assert torch.equal(w.k_pool.view(torch.int16),
                       h.k_pool.permute(0, 2, 1, 3).contiguous().view(torch.int16))
    m = wl.random_case(8, B=2, Hq=16, Hkv=1, D=576, D_v=512, mla=True, page_size=64)
    assert m.mla and m.v_pool is None and m.k_pool.shape[1:] == (64, 1, 576)


def _bench_module():
    import importlib.util
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py")
    spec = importlib.util.spec_from_file_location("zl_bench", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_roofline_bytes_count_shared_pages_once():
    """bench.py's roofline bytes: distinct (page, slot) rows, checked against a
    plain loop; equal to the logical bytes when no page is shared."""
    bench = _bench_module()
    for name in ("tiny_gqa", "llama70b_prefix_decode"):
        w = wl.WORKLOADS[name]()
        seen = set()
        for b in range(w.B):
            L = int(w.seq_lens[b])
            for t in range(L):
                seen.add((int(w.block_table[b, t // w.page_size]), t % w.page_size))
        want = len(seen) * w.Hkv * 2 * w.D_qk * 2
        assert bench.unique_kv_bytes(w) == want
        if name == "tiny_gqa":
            assert want == bench.kv_bytes(w)
        else:
            assert want < bench.kv_bytes(w) / 4  # the 2048-token prefix is shared by 128
