"""Pins of the FP8 / Hadamard part of the oracle (numpy, CPU only)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
import synth


def test_e4m3_encode_exhaustive_vs_library():
    """Every finite bfloat16 value, clamped to +-448, encodes exactly as the
    library's float32 -> float8_e4m3fn conversion does (RNE, ties to even)."""
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).astype(np.uint32).view(np.float32)
    x = np.clip(f[np.isfinite(f)], -448.0, 448.0).astype(np.float32)
    mine = fp8.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref), np.count_nonzero(mine != ref)


def test_e4m3_encode_saturates_and_rounds_half_even():
    assert fp8.e4m3_encode([448.0])[0] == 0x7E
    assert fp8.e4m3_encode([1e9])[0] == 0x7E            # finite overflow saturates
    assert fp8.e4m3_encode([-1e9])[0] == 0xFE
    assert fp8.e4m3_encode([np.nan])[0] == 0x7F
    assert fp8.e4m3_encode([2.0 ** -10])[0] == 0x00     # half of the smallest subnormal: to even
    assert fp8.e4m3_encode([3 * 2.0 ** -10])[0] == 0x02  # 1.5 quanta -> 2 (even)
    assert fp8.e4m3_encode([1.0625])[0] == 0x38         # 1 + 1/16: tie between 1 and 1.125 -> 1


def test_e4m3_decode_all_codes_vs_library():
    codes = np.arange(256, dtype=np.uint8)
    mine = fp8.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    same = (mine == ref) | (np.isnan(mine) & np.isnan(ref))
    assert same.all()
    assert np.nanmax(mine) == 448.0 and mine[1] == 2.0 ** -9


@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_is_orthogonal_up_to_d(d):
    H = fp8.hadamard_matrix(d)
    assert np.array_equal(H @ H.T, d * np.eye(d, dtype=np.int64))
    assert np.array_equal(H, H.T)


def test_hadamard_d2_closed_form():
    assert np.array_equal(fp8.hadamard_matrix(2), np.array([[1, 1], [1, -1]]))
    assert np.array_equal(fp8.hadamard_matrix(4)[3], np.array([1, -1, -1, 1]))


def test_transform_leaves_attention_unchanged_gqa():
    """(Q M)(K M)^T = Q K^T for orthogonal M shared by a query group and its
    key/value head: oracle attention on transformed Q, K equals the raw one."""
    B, N, Hq, Hkv, d = 1, 40, 4, 2, 16
    rng = np.random.default_rng(0)
    q = rng.standard_normal((B, N, Hq, d))
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    signs = synth.hadamard_signs(Hkv, d, seed=3).numpy()
    qt = fp8.incoherent_transform(q, signs)
    kt = fp8.incoherent_transform(k, signs)
    o1, l1 = oracle.attention_full(q, k, v, causal=True, scale=0.25)
    o2, l2 = oracle.attention_full(qt, kt, v, causal=True, scale=0.25)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)
    # signs that differ between a query head and its key/value head break it
    bad = signs.copy()
    bad[:, 0] *= -1
    qb = fp8.incoherent_transform(q, bad)
    o3, _ = oracle.attention_full(qb, kt, v, causal=True, scale=0.25)
    assert np.abs(o3 - o1).max() > 1e-3


def test_block_quantisation_properties():
    """descale = amax / 448 per (b, h, 128-token block); every code decodes to
    within half an E4M3 spacing of x / descale; the block maximum maps to 448;
    an all-zero block has descale 1 and zero codes; the last block is partial."""
    B, N, H, d = 2, 300, 3, 8
    rng = np.random.default_rng(1)
    x = rng.standard_normal((B, N, H, d)).astype(np.float32)
    x[1, 128:256, 2] = 0.0                      # an all-zero block
    codes, ds = fp8.quantize_blocks(x)
    assert ds.shape == (B, H, 3)
    assert ds[1, 2, 1] == 1.0 and not codes[1, 128:256, 2].any()
    for b in range(B):
        for h in range(H):
            for t in range(3):
                blk = x[b, t * 128:(t + 1) * 128, h]
                amax = np.float32(np.abs(blk).max())
                if amax == 0:
                    continue
                assert ds[b, h, t] == np.float32(amax / np.float32(448.0))
                q = blk.astype(np.float64) / np.float64(ds[b, h, t])
                dec = fp8.e4m3_decode(codes[b, t * 128:(t + 1) * 128, h])
                # spacing of E4M3 at |q|: 2^(floor(log2|q|) - 3), at least 2^-9
                e = np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6)))
                assert np.all(np.abs(dec - q) <= 0.5 * np.exp2(e - 3) * (1 + 1e-6))
                assert np.abs(dec).max() == 448.0
                np.testing.assert_array_equal(codes[b, t * 128:(t + 1) * 128, h].ravel(),
                                              _nearest_code(q))


def _nearest_code(q):
    """Brute force over the E4M3 codebook, independent of fp8.e4m3_encode:
    the finite code whose value (from its bit fields) is nearest to q, ties to
    the code with the even last significand bit, beyond +-448 the largest
    finite magnitude."""
    q = np.asarray(q, dtype=np.float64).ravel()
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.int64)
    e, m = (codes >> 3) & 0xF, codes & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (8 + m) * 2.0 ** (e - 10))
    val = np.where(codes & 0x80, -mag, mag)
    dist = np.abs(q[:, None] - val[None, :])
    best = dist.min(axis=1, keepdims=True)
    tie = dist == best
    # among tied codes take the even significand (one of two neighbours is
    # even); +0 and -0 tie for 0: prefer the sign of q
    score = np.where(tie, 0, 4) + (codes[None, :] & 1) * 2 + (
        (codes[None, :] >> 7) != (np.signbit(q)[:, None]).astype(np.int64))
    return codes[np.argmin(score, axis=1)].astype(np.uint8)


def test_block_quantisation_rounds_exact_quotient_at_midpoints():
    """Values placed exactly on E4M3 rounding midpoints of x / descale round
    to the even neighbour, and values one float32 ulp off a midpoint round
    to the nearer side: the code is decided by the exact quotient x / descale
    ("FlashAttention（V3）深度解析" section 4.3: a scale per block; the
    quantised value is the block's value divided by its scale)."""
    # block amax 448 * 2^-4 = 28: descale = 1/16 exactly, so x / descale = 16 x
    mids = np.array([1.0625, 1.1875, 3.125, 13.5, 200.0, 2.0 ** -10, 3 * 2.0 ** -10], np.float64)
    x = (mids / 16.0).astype(np.float32)
    assert np.array_equal(x.astype(np.float64) * 16.0, mids)      # exactly on midpoints
    up = np.nextafter(x, np.float32(np.inf))
    dn = np.nextafter(x, np.float32(0.0))
    blk = np.zeros((1, 128, 1, 4), np.float32)
    blk[0, 0, 0, 0] = 28.0
    vals = np.concatenate([x, up, dn])
    blk[0, 1:1 + len(vals), 0, 0] = vals
    codes, ds = fp8.quantize_blocks(blk)
    assert ds[0, 0, 0] == np.float32(1.0 / 16.0)
    got = codes[0, 1:1 + len(vals), 0, 0]
    np.testing.assert_array_equal(got, _nearest_code(vals.astype(np.float64) * 16.0))
    dec = fp8.e4m3_decode(got).reshape(3, -1)
    assert np.all(dec[1] > dec[2])          # one ulp above / below a midpoint split
    # ties to even: 1.0625 -> 1.0 (code 0x38), 1.1875 -> 1.25 (0x3A)
    assert got[0] == 0x38 and got[1] == 0x3A


def test_fp8_error_with_hadamard_not_worse_on_outliers():
    """The claim on the pages (incoherent processing lowers FP8 error) holds
    for the oracle's own quantisation on the outlier workload recipe: the
    attention output from dequantised Hadamard-processed Q, K is no further
    from the exact output than plain per-block FP8."""
    B, N, H, d = 1, 512, 2, 128
    q, k, v = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=0,
                                outlier_frac=1e-3)
    q, k, v = (t.double().numpy() for t in (q, k, v))
    scale = 1 / math.sqrt(d)
    o_ref, _ = oracle.attention_full(q, k, v, causal=False, scale=scale)
    signs = synth.hadamard_signs(H, d, seed=0).numpy()
    errs = {}
    for had in (False, True):
        cq, dq, _ = fp8.prepare(q, signs, had)
        ck, dk, _ = fp8.prepare(k, signs, had)
        cv, dv, _ = fp8.prepare(v, signs, False)
        o, _ = oracle.attention_full(fp8.dequantize(cq, dq), fp8.dequantize(ck, dk),
                                     fp8.dequantize(cv, dv), causal=False, scale=scale)
        errs[had] = math.sqrt(np.mean((o - o_ref) ** 2))
    assert errs[True] <= errs[False], errs


# --- rotary embedding (rotate-half reading) -------------------------------

def test_rope_small_closed_form():
    """d = 4, base 10000: frequencies 1 and 10000^(-1/2) = 0.01; channel c
    pairs with c + 2.  Rotating unit vectors by hand at tokens 0, 1, 2."""
    N, d = 3, 4
    x = np.zeros((1, N, 4, d))
    for h in range(4):
        x[0, :, h, h] = 1.0                 # head h holds unit vector e_h
    y = fp8.rope(x, base=10000.0)
    for n in range(N):
        a0, a1 = n * 1.0, n * 0.01
        want = np.array([
            [math.cos(a0), 0.0, math.sin(a0), 0.0],     # e_0 -> cos e_0 + sin e_2
            [0.0, math.cos(a1), 0.0, math.sin(a1)],     # e_1 -> cos e_1 + sin e_3
            [-math.sin(a0), 0.0, math.cos(a0), 0.0],    # e_2 -> -sin e_0 + cos e_2
            [0.0, -math.sin(a1), 0.0, math.cos(a1)],    # e_3 -> -sin e_1 + cos e_3
        ])
        np.testing.assert_allclose(y[0, n], want, atol=1e-15)


def test_rope_is_complex_rotation_and_relative():
    """(x_c + i x_{c+d/2}) is multiplied by exp(i (pos0 + n) theta_c): norms
    are kept, position 0 is the identity, and q.k after rotation depends only
    on the difference of the two positions."""
    rng = np.random.default_rng(3)
    B, N, H, d = 1, 6, 2, 64
    x = rng.standard_normal((B, N, H, d))
    y = fp8.rope(x, base=500.0, pos0=7)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    theta = 500.0 ** (-np.arange(d // 2) / (d // 2))
    rot = np.exp(1j * (7 + np.arange(N))[:, None] * theta[None, :])
    zr = z * rot[None, :, None, :]
    np.testing.assert_allclose(y, np.concatenate([zr.real, zr.imag], -1), atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    np.testing.assert_array_equal(fp8.rope(x, pos0=0)[:, 0], x[:, 0])
    # relative positions: the same q and k vectors at every token
    q = np.broadcast_to(x[:, :1], x.shape)
    k = np.broadcast_to(x[:, 1:2], x.shape)
    s0 = np.einsum("bmhc,bnhc->bhmn", fp8.rope(q), fp8.rope(k))
    s5 = np.einsum("bmhc,bnhc->bhmn", fp8.rope(q, pos0=5), fp8.rope(k, pos0=5))
    np.testing.assert_allclose(s0, s5, atol=1e-12)
    # ... and it does change with the offset between them
    s_shift = np.einsum("bmhc,bnhc->bhmn", fp8.rope(q), fp8.rope(k, pos0=1))
    assert np.abs(s_shift - s0).max() > 1e-3


def test_prepare_rope_then_transform_keeps_rotated_scores():
    """The transform is applied after the rotation, so the float32 values that
    are quantised give the rotated Q K^T (to float32 rounding); in the other
    order they would not."""
    rng = np.random.default_rng(4)
    B, N, H, d = 1, 40, 2, 64
    q, k = rng.standard_normal((B, N, H, d)), rng.standard_normal((B, N, H, d))
    signs = synth.hadamard_signs(H, d, seed=1).numpy()
    _, _, yq = fp8.prepare(q, signs, True, rope_base=10000.0)
    _, _, yk = fp8.prepare(k, signs, True, rope_base=10000.0)
    want = np.einsum("bmhc,bnhc->bhmn", fp8.rope(q), fp8.rope(k))
    got = np.einsum("bmhc,bnhc->bhmn", yq.astype(np.float64), yk.astype(np.float64))
    np.testing.assert_allclose(got, want, atol=1e-4)
    wrong = np.einsum("bmhc,bnhc->bhmn", fp8.rope(fp8.incoherent_transform(q, signs)),
                      fp8.rope(fp8.incoherent_transform(k, signs)))
    assert np.abs(wrong - want).max() > 1e-2


# --- per-tensor quantisation (the baseline FP8 scheme) -----------------------

def test_per_tensor_quantisation_properties():
    B, N, H, d = 2, 300, 3, 64
    x, _, _ = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=9,
                                outlier_frac=1e-3)
    y = x.float().numpy()
    codes, ds, _ = fp8.prepare(y, per_tensor=True)
    amax = np.float32(np.abs(y).max())
    assert ds.shape == (B, H, 3)
    assert np.all(ds == np.float32(amax / np.float32(448.0)))
    dec = fp8.e4m3_decode(codes)
    assert np.abs(dec).max() == 448.0
    # every code is the E4M3 rounding of value / descale
    qv = y.astype(np.float64) / np.float64(ds.flat[0])
    e = np.floor(np.log2(np.maximum(np.abs(qv), 2.0 ** -6)))
    assert np.all(np.abs(dec - qv) <= 0.5 * np.exp2(e - 3) * (1 + 1e-6))
    np.testing.assert_array_equal(codes[:, :, :, :8].ravel(), _nearest_code(qv[:, :, :, :8]))
    # a tensor of one block is quantised as that block
    one = y[:1, :128, :1]
    c1, d1, _ = fp8.prepare(one, per_tensor=True)
    c2, d2, _ = fp8.prepare(one)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(d1, d2)
    # an all-zero tensor: descale 1, zero codes
    cz, dz, _ = fp8.prepare(np.zeros((1, 5, 2, 64)), per_tensor=True)
    assert not cz.any() and np.all(dz == 1.0)


def test_error_study_ordering_on_channel_outliers():
    """On channel-structured outliers (4 channels per key/value head, x5 in
    Q and K for every token) the per-block + Hadamard scheme's error is less
    than half the per-tensor baseline's and below per-block alone."""
    B, N, H, d = 1, 256, 2, 128
    q, k, v = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=0,
                                channel_outliers=4, channel_scale=5.0)
    q, k, v = (t.double().numpy() for t in (q, k, v))
    scale = 1 / math.sqrt(d)
    o_ref, _ = oracle.attention_full(q, k, v, causal=False, scale=scale)
    signs = synth.hadamard_signs(H, d, seed=0).numpy()
    err = {}
    for name, pt, had in (("tensor", True, False), ("block", False, False),
                          ("block+H", False, True)):
        deq = []
        for t, h in ((q, had), (k, had), (v, False)):
            c, ds, _ = fp8.prepare(t, signs, h, per_tensor=pt)
            deq.append(fp8.dequantize(c, ds))
        o, _ = oracle.attention_full(*deq, causal=False, scale=scale)
        err[name] = math.sqrt(np.mean((o - o_ref) ** 2))
    assert err["block+H"] * 2 < err["tensor"], err
    assert err["block+H"] < err["block"], err
