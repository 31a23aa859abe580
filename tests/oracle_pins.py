"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with:
  * torch's fp64 ``scaled_dot_product_attention`` (a library routine) on the
    dense, logical K/V that the paged pool was built from;
  * scipy's ``softmax`` / ``logsumexp`` on one-hot constructions where the
    scores are known exactly;
  * closed forms (single token, constant V, zero query, empty context);
  * invariants (token permutation, page remapping, pool layout, split+merge).

The pages the oracle follows print no worked example, so no pin uses stored
values from them; every expected value here comes from a library routine, a
closed form or an invariant.

The same pins run against mutated copies of the oracle in
``test_oracle_mutants.py``: each plausible mistake must fail at least one.
"""

from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

TOL = 1e-12


# ----------------------------------------------------------------------------
# construction helpers (inputs only; no attention arithmetic)
# ----------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """float -> nearest bf16 value, returned as float64."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


class PagedCase:
    """Logical dense K/V per sequence, scattered into a randomly placed pool."""

    def __init__(self, rng, lens, Hq, Hkv, D, P, *, q_len=1, D_v=None, mla=False, layout="NHD",
                 q=None, k=None, v=None, extra_pages=3, scale=None):
        self.lens = [int(x) for x in lens]
        self.B, self.Hq, self.Hkv, self.D, self.P = len(lens), Hq, Hkv, D, P
        self.q_len, self.mla, self.layout = q_len, mla, layout
        self.D_v = D if D_v is None else D_v
        self.scale = (1.0 / math.sqrt(D)) if scale is None else scale
        self.q = bf16_round(rng.standard_normal((self.B, q_len, Hq, D))) if q is None else q
        self.k = k if k is not None else [bf16_round(rng.standard_normal((L, Hkv, D)))
                                          for L in self.lens]
        if mla:
            self.v = [kb[..., :self.D_v] for kb in self.k]
        else:
            self.v = v if v is not None else [bf16_round(rng.standard_normal((L, Hkv, D)))
                                              for L in self.lens]
        npg = [(L + P - 1) // P for L in self.lens]
        self.num_pages = sum(npg) + extra_pages
        perm = rng.permutation(self.num_pages)
        self.table = np.full((self.B, max(max(npg), 1)), -1, dtype=np.int32)
        pos = 0
        for b in range(self.B):
            self.table[b, :npg[b]] = perm[pos:pos + npg[b]]
            pos += npg[b]
        self.build_pools(rng)

    def build_pools(self, rng=None):
        nan = np.float64("nan")
        kp = np.full((self.num_pages, self.P, self.Hkv, self.D), nan)
        vp = np.full((self.num_pages, self.P, self.Hkv, self.D), nan)
        for b, L in enumerate(self.lens):
            for t in range(L):
                page, slot = self.table[b, t // self.P], t % self.P
                kp[page, slot] = self.k[b][t]
                if not self.mla:
                    vp[page, slot] = self.v[b][t]
        if self.layout == "HND":
            kp = kp.transpose(0, 2, 1, 3).copy()
            vp = vp.transpose(0, 2, 1, 3).copy()
        self.k_pool = bf16_bits(kp)
        self.v_pool = None if self.mla else bf16_bits(vp)

    @property
    def strides(self):
        P, H, D = self.P, self.Hkv, self.D
        return (P * H * D, H * D, D) if self.layout == "NHD" else (H * P * D, D, P * D)

    def run(self, oracle, **kw):
        return oracle.decode_attn(bf16_bits(self.q), self.k_pool, self.v_pool, self.strides,
                                  self.table, np.array(self.lens, dtype=np.int32), Hkv=self.Hkv,
                                  page_size=self.P, num_pages=self.num_pages, scale=self.scale,
                                  D_v=self.D_v, **kw)

    def sdpa(self, b):
        """torch fp64 SDPA on sequence b's dense K/V (GQA via enable_gqa)."""
        L = self.lens[b]
        q = torch.from_numpy(self.q[b]).permute(1, 0, 2)[None]              # [1,Hq,q_len,D]
        k = torch.from_numpy(self.k[b]).permute(1, 0, 2)[None]              # [1,Hkv,L,D]
        v = torch.from_numpy(np.ascontiguousarray(self.v[b])).permute(1, 0, 2)[None]
        mask = None
        if self.q_len > 1:
            i = torch.arange(self.q_len)[:, None]
            t = torch.arange(L)[None, :]
            mask = t <= (L - self.q_len + i)
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=self.scale,
                                           enable_gqa=(self.Hq != self.Hkv))
        return o[0].permute(1, 0, 2).numpy()                                 # [q_len,Hq,D_v]


def _close(a, b, tol=TOL, what=""):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert np.all(np.isfinite(a)) and err <= tol, f"{what}: max|diff| = {err}"


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def pin_sdpa_dense(oracle):
    """Random tiny paged cases == torch fp64 SDPA on the logical dense K/V."""
    rng = np.random.default_rng(11)
    shapes = [  # lens, Hq, Hkv, D, P
        ([1, 7, 40], 4, 4, 8, 4),
        ([33, 16], 8, 2, 8, 16),
        ([17, 5, 29], 8, 1, 128, 16),
        ([40], 4, 2, 128, 8),
        ([3, 31], 16, 4, 16, 4),
        ([9, 23], 32, 1, 8, 4),     # many-head MQA (32 query heads on one kv head)
        ([14], 71, 1, 8, 8),        # 71 heads: no even split into chunks of 16
        ([30, 5], 40, 2, 8, 16),    # 20 query heads per kv head
    ]
    for lens, Hq, Hkv, D, P in shapes:
        case = PagedCase(rng, lens, Hq, Hkv, D, P)
        out, _, st = case.run(oracle)
        assert st == 0
        for b in range(case.B):
            _close(out[b], case.sdpa(b), 1e-12, f"sdpa lens={lens} b={b}")


def pin_gqa_head_mapping(oracle):
    """Query head h reads kv head h // (Hq/Hkv), checked with very different kv heads."""
    rng = np.random.default_rng(12)
    L, Hq, Hkv, D = 20, 8, 4, 8
    k = bf16_round(rng.standard_normal((L, Hkv, D)))
    v = np.zeros((L, Hkv, D))
    for kh in range(Hkv):
        v[:, kh, :] = 10.0 * (kh + 1)      # output of head h is 10*(h//2 + 1)
    case = PagedCase(rng, [L], Hq, Hkv, D, 4, k=[k], v=[v])
    out, _, _ = case.run(oracle)
    for h in range(Hq):
        _close(out[0, 0, h], np.full(D, 10.0 * (h // (Hq // Hkv) + 1)), 1e-12, f"head {h}")
    _close(out[0], case.sdpa(0), 1e-12, "gqa sdpa")


def pin_softmax_onehot(oracle):
    """One-hot construction: scores equal known bf16 values, so the output rows
    are scipy's softmax and lse is scipy's logsumexp."""
    rng = np.random.default_rng(13)
    for L, spread in [(1, 1.0), (2, 1.0), (9, 3.0), (37, 20.0), (100, 0.25)]:
        D = 128
        x = bf16_round(rng.standard_normal(L) * spread)
        q = np.zeros((1, 1, 1, D))
        q[0, 0, 0, 0] = 1.0
        k = np.zeros((L, 1, D))
        k[:, 0, 0] = x
        v = np.zeros((L, 1, D))
        for t in range(L):
            v[t, 0, t % D] = 1.0 if t < D else 0.0
        scale = 0.5
        case = PagedCase(rng, [L], 1, 1, D, 16, q=q, k=[k], v=[v], scale=scale)
        out, lse, st = case.run(oracle)
        w = scipy.special.softmax(scale * x)
        expect = np.zeros(D)
        for t in range(L):
            expect[t % D] += w[t]
        _close(out[0, 0, 0], expect, 1e-13, f"softmax L={L}")
        _close(lse[0, 0, 0], scipy.special.logsumexp(scale * x), 1e-12, f"lse L={L}")
        # the weight vector itself
        o2, l2, wts, st2 = oracle.attend_range(bf16_bits(q[0, 0, 0]), case.k_pool, case.v_pool,
                                               case.strides, case.table[0], kh=0, page_size=16,
                                               num_pages=case.num_pages, scale=scale, t_begin=0,
                                               t_end=L, want_weights=True)
        _close(wts, w, 1e-13, "weights")
        assert abs(wts.sum() - 1.0) <= 1e-12 and np.all(wts >= 0)


def pin_large_scores(oracle):
    """Scores in the thousands: the max-subtracted softmax stays finite and
    agrees with SDPA (which is stable); an unstable exp overflows."""
    rng = np.random.default_rng(14)
    L, D = 24, 128
    q = bf16_round(rng.standard_normal((1, 1, 2, D)) * 24.0)
    k = bf16_round(rng.standard_normal((L, 1, D)) * 24.0)
    case = PagedCase(rng, [L], 2, 1, D, 16, q=q, k=[k])
    out, lse, _ = case.run(oracle)
    _close(out[0], case.sdpa(0), 1e-10, "large scores")
    assert np.all(np.isfinite(lse))


def pin_single_token(oracle):
    """L = 1: the output is exactly V_0 (weight 1), bit for bit."""
    rng = np.random.default_rng(15)
    case = PagedCase(rng, [1, 1], 8, 2, 128, 16)
    out, _, _ = case.run(oracle)
    for b in range(2):
        for h in range(8):
            assert np.array_equal(out[b, 0, h], case.v[b][0, h // 4]), "single token"


def pin_constant_v(oracle):
    """All V rows equal c: the output is c whatever the scores."""
    rng = np.random.default_rng(16)
    lens = [5, 77, 130]
    c = bf16_round(rng.standard_normal((2, 64)))
    v = [np.broadcast_to(c, (L, 2, 64)).copy() for L in lens]
    case = PagedCase(rng, lens, 8, 2, 64, 16, v=v)
    out, _, _ = case.run(oracle)
    for b in range(3):
        for h in range(8):
            _close(out[b, 0, h], c[h // 4], 1e-12, "constant V")


def pin_zero_query(oracle):
    """q = 0: uniform weights, so out = mean of V over the context and lse = ln L."""
    rng = np.random.default_rng(17)
    lens = [1, 16, 45]
    q = np.zeros((3, 1, 4, 32))
    case = PagedCase(rng, lens, 4, 2, 32, 16, q=q)
    out, lse, _ = case.run(oracle)
    for b, L in enumerate(lens):
        for h in range(4):
            _close(out[b, 0, h], case.v[b][:, h // 2].mean(axis=0), 1e-12, "zero query")
            _close(lse[b, 0, h], math.log(L), 1e-12, "zero query lse")


def pin_token_permutation(oracle):
    """Attention has no positional term: permuting the tokens (K and V
    together) leaves the output unchanged."""
    rng = np.random.default_rng(18)
    a = PagedCase(rng, [50, 23], 8, 2, 16, 8)
    out_a, lse_a, _ = a.run(oracle)
    for b in range(2):
        perm = rng.permutation(a.lens[b])
        a.k[b] = a.k[b][perm]
        a.v[b] = a.v[b][perm]
    a.build_pools()
    out_b, lse_b, _ = a.run(oracle)
    _close(out_a, out_b, 1e-12, "permutation")
    _close(lse_a, lse_b, 1e-12, "permutation lse")


def pin_page_remap(oracle):
    """Same logical content on other physical pages: identical bits."""
    rng = np.random.default_rng(19)
    a = PagedCase(rng, [61, 16, 33], 8, 2, 32, 16, extra_pages=5)
    out_a, lse_a, _ = a.run(oracle)
    perm = rng.permutation(a.num_pages).astype(np.int32)
    a.table = np.where(a.table >= 0, perm[np.maximum(a.table, 0)], -1).astype(np.int32)
    a.build_pools()
    out_b, lse_b, _ = a.run(oracle)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b), "page remap"


def pin_layout(oracle):
    """NHD and HND pools with the same logical content give identical bits."""
    rng = np.random.default_rng(20)
    a = PagedCase(rng, [37, 64], 8, 4, 16, 16)
    out_a, lse_a, _ = a.run(oracle)
    a.layout = "HND"
    a.build_pools()
    out_b, lse_b, _ = a.run(oracle)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b), "layout"


def pin_split_merge(oracle):
    """Partials over arbitrary cuts, merged by log-sum-exp, equal the unsplit row."""
    rng = np.random.default_rng(21)
    L, D = 97, 32
    case = PagedCase(rng, [L], 4, 2, D, 16)
    full, lse_full, _ = case.run(oracle)
    for cuts in ([0, 97], [0, 1, 97], [0, 16, 16, 50, 97], [0, 3, 40, 41, 96, 97]):
        for h in range(4):
            parts, lses = [], []
            for t0, t1 in zip(cuts[:-1], cuts[1:]):
                o, l, _, st = oracle.attend_range(
                    bf16_bits(case.q[0, 0, h]), case.k_pool, case.v_pool, case.strides,
                    case.table[0], kh=h // 2, page_size=16, num_pages=case.num_pages,
                    scale=case.scale, t_begin=t0, t_end=t1)
                parts.append(o)
                lses.append(l)
            o, l = oracle.lse_merge(np.stack(parts), np.array(lses))
            _close(o, full[0, 0, h], 1e-12, f"merge {cuts}")
            _close(l, lse_full[0, 0, h], 1e-12, f"merge lse {cuts}")
    # all-empty merge
    o, l = oracle.lse_merge(np.zeros((2, D)), np.array([-np.inf, -np.inf]))
    assert np.all(o == 0) and l == -np.inf


def pin_mla(oracle):
    """MLA (V = first D_v columns of the latent row) equals a separate V pool
    holding that copy, and equals SDPA on the dense latent."""
    rng = np.random.default_rng(22)
    lens = [9, 70]
    a = PagedCase(rng, lens, 16, 1, 576, 64, D_v=512, mla=True, scale=1 / math.sqrt(192))
    out_a, lse_a, _ = a.run(oracle)
    for b in range(2):
        _close(out_a[b], a.sdpa(b), 1e-12, "mla sdpa")
    b_ = PagedCase(rng, lens, 16, 1, 576, 64, D_v=512, scale=1 / math.sqrt(192), q=a.q,
                   k=a.k, v=[np.concatenate([kb[..., :512], np.zeros((kb.shape[0], 1, 64))], -1)
                             for kb in a.k])
    b_.table, b_.num_pages = a.table, a.num_pages
    b_.build_pools()
    out_b, lse_b, _ = b_.run(oracle)
    _close(out_a, out_b, 0.0, "mla vs explicit V")
    _close(lse_a, lse_b, 0.0, "mla lse")


def pin_mla_absorption(oracle):
    """The absorbed reading: (W_UK^T q_nope) . c == q_nope . (W_UK c) in fp64,
    so attention over the latent with the absorbed query equals attention over
    the up-projected keys (here checked through the oracle's scores)."""
    rng = np.random.default_rng(23)
    dl, dn, L = 16, 8, 12
    W = rng.standard_normal((dn, dl))
    q_nope = rng.standard_normal(dn)
    c = bf16_round(rng.standard_normal((L, dl)))
    q_abs = W.T @ q_nope                      # absorbed query over the latent
    s_abs = c @ q_abs
    s_up = (c @ W.T) @ q_nope                 # keys up-projected, then dot
    _close(s_abs, s_up, 1e-12, "absorption identity")
    # the oracle on the latent with the absorbed query (exactly bf16) equals
    # softmax of those scores applied to the latent
    qb = bf16_round(q_abs)
    case = PagedCase(rng, [L], 1, 1, dl, 4, q=qb.reshape(1, 1, 1, dl), k=[c[:, None, :]],
                     v=[c[:, None, :]], scale=1.0)
    out, _, _ = case.run(oracle)
    w = scipy.special.softmax(c @ qb)
    _close(out[0, 0, 0], w @ c, 1e-12, "absorbed attention")


def pin_multi_token_causal(oracle):
    """q_len > 1: query i sees tokens t <= L - q_len + i (bottom-right causal)."""
    rng = np.random.default_rng(24)
    for q_len, Hq, Hkv in ((2, 8, 2), (4, 8, 2), (3, 32, 1)):
        case = PagedCase(rng, [20, 9, 33], Hq, Hkv, 16, 8, q_len=q_len)
        out, _, _ = case.run(oracle)
        for b in range(3):
            _close(out[b], case.sdpa(b), 1e-12, f"causal q_len={q_len} Hq={Hq}")


def pin_degenerate(oracle):
    """Empty context, bad page ids and oversize lengths: zeros, lse -inf, status bits."""
    rng = np.random.default_rng(25)
    case = PagedCase(rng, [16, 7, 30], 4, 2, 16, 16)
    lens = np.array(case.lens, dtype=np.int32)
    q = bf16_bits(case.q)

    def run(table, lens_):
        return oracle.decode_attn(q, case.k_pool, case.v_pool, case.strides, table, lens_,
                                  Hkv=2, page_size=16, num_pages=case.num_pages, scale=case.scale)

    ref, _, st = run(case.table, lens)
    assert st == 0
    l0 = lens.copy()
    l0[1] = 0
    out, lse, st = run(case.table, l0)
    assert st == 0 and np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    assert np.array_equal(out[0], ref[0]) and np.array_equal(out[2], ref[2])
    bad = case.table.copy()
    bad[2, 1] = case.num_pages            # out of range
    out, lse, st = run(bad, lens)
    assert st & 1 and np.all(out[2] == 0) and np.all(lse[2] == -np.inf)
    assert np.array_equal(out[0], ref[0])
    big = lens.copy()
    big[0] = case.table.shape[1] * 16 + 1
    out, lse, st = run(case.table, big)
    assert st & 2 and np.all(out[0] == 0) and np.all(lse[0] == -np.inf)


def _append_inputs(case, q_len):
    """New-token rows of a PagedCase and its pools with those rows overwritten by
    junk (the state before the append). Pure numpy indexing."""
    knew = np.stack([case.k[b][L - q_len:] for b, L in enumerate(case.lens)])
    vnew = None if case.mla else np.stack([np.ascontiguousarray(case.v[b][L - q_len:])
                                           for b, L in enumerate(case.lens)])
    junk = np.uint16(0x7F81)                      # a NaN pattern that no input holds
    kb = case.k_pool.copy()
    vb = None if case.mla else case.v_pool.copy()
    for b, L in enumerate(case.lens):
        for t in range(L - q_len, L):
            page, slot = case.table[b, t // case.P], t % case.P
            for arr in (kb, vb):
                if arr is None:
                    continue
                if case.layout == "NHD":
                    arr[page, slot] = junk
                else:
                    arr[page, :, slot] = junk
    return bf16_bits(knew), None if vnew is None else bf16_bits(vnew), kb, vb


def pin_kv_append(oracle):
    """Appending the last q_len tokens of every sequence to pools that lack them
    gives, bit for bit, the pools built directly from the dense K/V (every other
    element untouched), for both layouts and for the latent-only (MLA) pool."""
    rng = np.random.default_rng(26)
    for q_len, layout, mla in ((1, "NHD", False), (3, "NHD", False), (2, "HND", False),
                               (4, "NHD", True)):
        lens = [20, 9, 33, 5]
        case = PagedCase(rng, lens, 4, 2, 16, 8, q_len=q_len, layout=layout, mla=mla,
                         D_v=8 if mla else None)
        knew, vnew, kb, vb = _append_inputs(case, q_len)
        assert not np.array_equal(kb, case.k_pool)
        ko, vo, st = oracle.kv_append(knew, vnew, kb, vb, case.strides, case.table,
                                      np.array(lens, dtype=np.int32), page_size=case.P,
                                      num_pages=case.num_pages)
        assert st == 0
        assert np.array_equal(ko, case.k_pool), ("K pool", q_len, layout)
        if mla:
            assert vo is None
        else:
            assert np.array_equal(vo, case.v_pool), ("V pool", q_len, layout)


def pin_kv_append_errors(oracle):
    """A sequence shorter than q_len writes nothing (bit 2); a bad page id skips
    only its token (bit 1); the other sequences are appended as usual."""
    rng = np.random.default_rng(27)
    q_len = 3
    case = PagedCase(rng, [12, 19, 30], 2, 2, 8, 4, q_len=q_len)
    knew, vnew, kb, vb = _append_inputs(case, q_len)
    lens = np.array(case.lens, dtype=np.int32)
    short = lens.copy()
    short[0] = 2
    ko, vo, st = oracle.kv_append(knew, vnew, kb, vb, case.strides, case.table, short,
                                  page_size=4, num_pages=case.num_pages)
    assert st == 2
    own0 = case.table[0, :3]
    assert np.array_equal(ko[own0], kb[own0]) and np.array_equal(vo[own0], vb[own0])
    rest = np.setdiff1d(np.arange(case.num_pages), own0)
    assert np.array_equal(ko[rest], case.k_pool[rest])
    table = case.table.copy()
    last = (case.lens[2] - 1) // 4
    good_page = table[2, last]
    table[2, last] = -1                   # the page of sequence 2's newest tokens
    ko, vo, st = oracle.kv_append(knew, vnew, kb, vb, case.strides, table, lens, page_size=4,
                                  num_pages=case.num_pages)
    assert st == 1
    assert np.array_equal(ko[good_page], kb[good_page])
    others = np.setdiff1d(np.arange(case.num_pages), [good_page])
    assert np.array_equal(ko[others], case.k_pool[others])
    assert np.array_equal(vo[others], case.v_pool[others])


ALL_PINS = [
    pin_sdpa_dense, pin_gqa_head_mapping, pin_softmax_onehot, pin_large_scores,
    pin_single_token, pin_constant_v, pin_zero_query, pin_token_permutation, pin_page_remap,
    pin_layout, pin_split_merge, pin_mla, pin_mla_absorption, pin_multi_token_causal,
    pin_degenerate, pin_kv_append, pin_kv_append_errors,
]
