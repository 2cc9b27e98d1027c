"""Pins of the FP64 attention oracle against facts fixed outside it.

Each test ties the oracle to something it does not compute itself: a closed
form, an invariant of the definition, the merge rule printed on the pages, or
an independent library routine (torch float64 on the CPU) on tiny shapes.
A plausible mistake in the oracle (dropped scale, wrong sign, transposed
operand, wrong group map, causal off-by-one, log base) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _torch_attention(q, k, v, causal, scale):
    """Library brute force: float64 torch softmax on the CPU (tiny shapes)."""
    q, k, v = (torch.as_tensor(x, dtype=torch.float64) for x in (q, k, v))
    B, Nq, Hq, d = q.shape
    Hkv = k.shape[2]
    kk = k.repeat_interleave(Hq // Hkv, dim=2)
    vv = v.repeat_interleave(Hq // Hkv, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", q, kk) * scale
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(k.shape[1])[None, :]
        s = s.masked_fill(j > i, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), vv)
    return o.numpy(), lse.numpy()


# ---------------------------------------------------------------- decoders
def test_decoders_match_library_conversion():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for elem, tdt in ((oracle.ELEM_BF16, torch.bfloat16), (oracle.ELEM_F16, torch.float16)):
        mine = oracle.decode(bits, elem)
        ref = torch.from_numpy(bits.view(np.int16)).view(tdt).double().numpy()
        same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
        assert same.all(), f"elem {elem}: {np.count_nonzero(~same)} patterns differ"


# ------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2)])
def test_zero_query_gives_mean_of_allowed_values(causal, Hq, Hkv):
    """Q = 0: every allowed logit is 0, so P is uniform over the allowed keys:
    O_i = mean of allowed V rows and LSE_i = ln |J_i|."""
    B, Nq, Nk, d = 2, 9, 13, 8
    q = np.zeros((B, Nq, Hq, d))
    k = _rand((B, Nk, Hkv, d), 1)
    v = _rand((B, Nk, Hkv, d), 2)
    o, lse = oracle.attention_full(q, k, v, causal=causal, scale=0.37)
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            for i in range(Nq):
                n = min(i + 1, Nk) if causal else Nk
                np.testing.assert_allclose(o[b, i, h], v[b, :n, h // g].mean(axis=0),
                                           rtol=0, atol=1e-13)
                assert abs(lse[b, h, i] - math.log(n)) < 1e-13


def test_one_hot_dominant_logit_selects_that_value_row():
    """A key whose logit exceeds all others by >= 55 takes all the weight:
    O_i = V[j*] to within e^-55 relative, LSE_i = s_{j*} + ln(1 + tiny)."""
    B, Nk, H, d = 1, 50, 1, 16
    scale = 1 / math.sqrt(d)
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, 1, H, d))
    k = 0.01 * rng.standard_normal((B, Nk, H, d))
    v = rng.standard_normal((B, Nk, H, d))
    jstar = 31
    qv = q[0, 0, 0]
    k[0, jstar, 0] = (60.0 / scale) * qv / np.dot(qv, qv)   # logit exactly 60
    o, lse = oracle.attention_full(q, k, v, causal=False, scale=scale)
    np.testing.assert_allclose(o[0, 0, 0], v[0, jstar, 0], rtol=1e-20, atol=1e-20)
    assert abs(lse[0, 0, 0] - 60.0) < 1e-12
    # the dominant key wins only because of its sign: flip it and it is ignored
    k[0, jstar, 0] *= -1
    o2, _ = oracle.attention_full(q, k, v, causal=False, scale=scale)
    assert np.abs(o2[0, 0, 0] - v[0, jstar, 0]).max() > 0.1


def test_causal_first_row_is_first_value_row():
    B, N, H, d = 1, 7, 3, 4
    q, k, v = _rand((B, N, H, d), 7), _rand((B, N, H, d), 8), _rand((B, N, H, d), 9)
    o, lse = oracle.attention_full(q, k, v, causal=True, scale=0.5)
    np.testing.assert_allclose(o[0, 0], v[0, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, :, 0], 0.5 * np.einsum("hd,hd->h", q[0, 0], k[0, 0]),
                               rtol=0, atol=1e-14)


# ------------------------------------------------- merge rule of the pages
@pytest.mark.parametrize("splits", [[1], [17], [5, 40], [3, 11, 29, 60]])
def test_streaming_merge_rule_matches_whole_softmax(splits):
    """Pages' merge rule (m = max(m_a, m_b), z = z_a e^(m_a-m) + z_b e^(m_b-m)):
    attention over disjoint key blocks, merged pairwise, equals attention over
    all keys.  This is the identity the GPU's streaming softmax rests on."""
    B, Nq, Nk, Hq, Hkv, d = 2, 6, 64, 4, 2, 16
    q = _rand((B, Nq, Hq, d), 11)
    k = 2.0 * _rand((B, Nk, Hkv, d), 12)
    v = _rand((B, Nk, Hkv, d), 13)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention_full(q, k, v, causal=False, scale=scale)
    edges = [0] + list(splits) + [Nk]
    o_acc = lse_acc = None
    for a, b in zip(edges[:-1], edges[1:]):
        o_p, lse_p = oracle.attention_full(q, k[:, a:b], v[:, a:b], causal=False, scale=scale)
        lse_p = lse_p.transpose(0, 2, 1)          # -> [B, Nq, Hq] to match o's leading axes
        if o_acc is None:
            o_acc, lse_acc = o_p, lse_p
        else:
            o_acc, lse_acc = oracle.merge_partials(o_acc, lse_acc, o_p, lse_p)
    np.testing.assert_allclose(o_acc, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_acc.transpose(0, 2, 1), lse_ref, rtol=0, atol=1e-12)


# ------------------------------------------------ library brute force
@pytest.mark.parametrize("B,Nq,Nk,Hq,Hkv,d,causal", [
    (1, 5, 5, 1, 1, 4, False),
    (2, 7, 11, 4, 2, 8, False),
    (2, 7, 11, 4, 2, 8, True),      # causal, Nq < Nk: top-left aligned
    (1, 13, 6, 6, 3, 8, True),      # causal, Nq > Nk: rows >= Nk see every key
    (1, 33, 64, 8, 1, 16, True),    # multi-query group
])
def test_matches_library_bruteforce_float64(B, Nq, Nk, Hq, Hkv, d, causal):
    q = _rand((B, Nq, Hq, d), 21)
    k = _rand((B, Nk, Hkv, d), 22)
    v = _rand((B, Nk, Hkv, d), 23)
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attention_full(q, k, v, causal=causal, scale=scale)
    o_t, lse_t = _torch_attention(q, k, v, causal, scale)
    np.testing.assert_allclose(o, o_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t, rtol=0, atol=1e-12)


@pytest.mark.parametrize("elem,tdt", [(oracle.ELEM_BF16, torch.bfloat16),
                                      (oracle.ELEM_F16, torch.float16)])
def test_raw_16bit_inputs_match_library_bruteforce(elem, tdt):
    """The oracle decodes raw 16-bit inputs itself; a library float64 pass on
    the same (library-decoded) values must agree."""
    g = torch.Generator().manual_seed(3)
    B, Nq, Nk, Hq, Hkv, d = 1, 9, 20, 4, 2, 8
    q = torch.randn(B, Nq, Hq, d, generator=g).to(tdt)
    k = torch.randn(B, Nk, Hkv, d, generator=g).to(tdt)
    v = torch.randn(B, Nk, Hkv, d, generator=g).to(tdt)
    bits = [x.view(torch.int16).numpy().view(np.uint16) for x in (q, k, v)]
    o, lse = oracle.attention_full(*bits, causal=True, scale=0.3, elem=elem)
    o_t, lse_t = _torch_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                  True, 0.3)
    np.testing.assert_allclose(o, o_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t, rtol=0, atol=1e-12)


def test_selected_rows_equal_full_rows():
    B, N, Hq, Hkv, d = 2, 21, 4, 1, 8
    q, k, v = _rand((B, N, Hq, d), 31), _rand((B, N, Hkv, d), 32), _rand((B, N, Hkv, d), 33)
    o, lse = oracle.attention_full(q, k, v, causal=True, scale=0.25)
    rows = np.array([[0, 0, 0], [1, 3, 20], [0, 2, 7], [1, 1, 13]])
    qr = q[rows[:, 0], rows[:, 2], rows[:, 1]]
    o_r, lse_r = oracle.attention_rows(qr, k, v, Hq=Hq, causal=True, scale=0.25, rows=rows)
    np.testing.assert_array_equal(o_r, o[rows[:, 0], rows[:, 2], rows[:, 1]])
    np.testing.assert_array_equal(lse_r, lse[rows[:, 0], rows[:, 1], rows[:, 2]])


# ---------------------------------------------------------- invariants
def test_key_permutation_invariance_noncausal():
    B, N, H, d = 1, 40, 2, 8
    q, k, v = _rand((B, 5, H, d), 41), _rand((B, N, H, d), 42), _rand((B, N, H, d), 43)
    perm = np.random.default_rng(44).permutation(N)
    o1, l1 = oracle.attention_full(q, k, v, causal=False, scale=0.4)
    o2, l2 = oracle.attention_full(q, k[:, perm], v[:, perm], causal=False, scale=0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_changes_only_lse(causal):
    """K -> K + u on every key adds scale*q.u to every logit of a row:
    softmax is unchanged, LSE shifts by exactly scale*q.u."""
    B, N, H, d = 1, 30, 2, 8
    scale = 0.3
    q, k, v = _rand((B, N, H, d), 51), _rand((B, N, H, d), 52), _rand((B, N, H, d), 53)
    u = _rand((d,), 54)
    o1, l1 = oracle.attention_full(q, k, v, causal=causal, scale=scale)
    o2, l2 = oracle.attention_full(q, k + u, v, causal=causal, scale=scale)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    shift = scale * np.einsum("bihd,d->bhi", q, u)
    np.testing.assert_allclose(l2 - l1, shift, rtol=0, atol=1e-12)


def test_value_affine_map():
    B, N, H, d = 2, 25, 2, 8
    q, k, v = _rand((B, N, H, d), 61), _rand((B, N, H, d), 62), _rand((B, N, H, d), 63)
    o1, _ = oracle.attention_full(q, k, v, causal=True, scale=0.35)
    o2, _ = oracle.attention_full(q, k, -2.5 * v + 0.75, causal=True, scale=0.35)
    np.testing.assert_allclose(o2, -2.5 * o1 + 0.75, rtol=0, atol=1e-12)


def test_output_is_convex_combination():
    B, N, H, d = 1, 50, 2, 8
    q, k, v = 3 * _rand((B, N, H, d), 71), _rand((B, N, H, d), 72), _rand((B, N, H, d), 73)
    o, _ = oracle.attention_full(q, k, v, causal=True, scale=0.5)
    for i in range(N):
        lo = v[:, : i + 1].min(axis=1)
        hi = v[:, : i + 1].max(axis=1)
        assert np.all(o[:, i] >= lo - 1e-12) and np.all(o[:, i] <= hi + 1e-12)


# ---------------------------------------------------- the pages' numbers
def test_pages_flop_ratio_fixture():
    """The pages print one worked number for this path: GEMM flops per score
    (4 * d) over one softmax exponential per score is 512 at head_dim 128.
    The bench's FLOP count (4 * B * Hq * Nq * Nk * d, halved under the causal
    mask) must reproduce it per score."""
    with open(os.path.join(GOLDEN, "pages_facts.json")) as f:
        facts = json.load(f)
    fx = facts["gemm_to_softmax_flop_ratio"]
    import bench
    d = fx["head_dim"]
    flops = bench.attention_flops(B=1, Hq=1, Nq=1000, Nk=1000, d=d, causal=False)
    assert flops / (1000 * 1000) == fx["value"]
