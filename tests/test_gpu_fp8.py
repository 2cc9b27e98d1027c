"""GPU parity of the FP8 path: the prep kernel (per-block E4M3 quantisation,
optional Hadamard transform; the per-tensor baseline; the fused rotary
variant and its tables) and the FP8 fused forward.

* Prep without the transform: codes (E4M3 of the exact quotient x /
  descale, ties to even) and descales must match the oracle bit for bit, in
  both layouts.  bfloat16 inputs put about 0.1 % of quotients exactly on an
  E4M3 rounding midpoint, so this checks the kernel's tie decision too.
* Prep with the transform: the float32 butterfly and the oracle's float64
  product may round the last bit differently, which can move a value across
  an E4M3 rounding boundary.  Codes are checked against the exact value with
  that slack; descales to float32 rounding.
* FP8 forward: the kernel run on the oracle's own codes and descales against
  the oracle on the same dequantised values (identical inputs: the kernel's
  arithmetic); the whole GPU chain (prep + forward) against the same, bit
  for bit where the codes are bit-exact; and against the oracle on the
  original BF16 values (the truth): no error beyond the quantisation
  scheme's own, RMS <= 5e-2 where the scheme can reach it (x10 outliers),
  and with the transform no worse than without it on outlier-injected
  inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import fp8 as ofp8
from parity import errors

pytestmark = pytest.mark.gpu


def _signs(G, d, dev="cuda"):
    return synth.hadamard_signs(G, d, seed=0).to(dev)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [300, 4096])
def test_prep_bit_exact_without_transform(gpu_lib, d, N):
    B, H = 2, 3
    x, _, _ = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=5,
                                outlier_frac=1e-3)
    codes, ds = gpu_lib.attn_prep_fp8(x.cuda())
    codes_t, ds_t = gpu_lib.attn_prep_fp8(x.cuda(), transpose_out=True)
    assert gpu_lib.get_status() == 0
    xf = x.float().numpy()
    oc, ods, _ = ofp8.prepare(xf, None, False)
    np.testing.assert_array_equal(ds.cpu().numpy(), ods)
    np.testing.assert_array_equal(ds_t.cpu().numpy(), ods)
    t = np.arange(N) // 128
    q_exact = xf.astype(np.float64) / ods.astype(np.float64)[:, :, t].transpose(0, 2, 1)[..., None]
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    npad = (N + 15) // 16 * 16
    ct = codes_t.cpu().numpy()
    assert ct.shape == (B, H, d, npad)
    np.testing.assert_array_equal(ct[..., :N], oc.transpose(0, 2, 3, 1))
    assert not ct[..., N:].any()   # padding keys are zero codes
    # the inputs do exercise near-ties: quotients within 2^-21 of an E4M3
    # rounding midpoint, where a float32 reciprocal-and-product alone can
    # round the other way (the descale's own rounding puts bfloat16 values
    # whose x * 448 / amax is a midpoint about 2^-25 off it)
    lo = ofp8.e4m3_encode(q_exact * (1 - 2.0 ** -21))
    hi = ofp8.e4m3_encode(q_exact * (1 + 2.0 ** -21))
    assert np.count_nonzero(lo != hi) > 0


@pytest.mark.parametrize("d", [64, 128, 256])
def test_prep_with_transform_matches_oracle(gpu_lib, d):
    B, N, Hq, Hkv = 1, 520, 4, 2
    x, _, _ = synth.attn_inputs(B, N, N, Hq, Hkv, d, dtype=torch.bfloat16, seed=6,
                                outlier_frac=1e-3)
    signs = _signs(Hkv, d)
    codes, ds = gpu_lib.attn_prep_fp8(x.cuda(), signs=signs, sign_heads=Hkv)
    assert gpu_lib.get_status() == 0
    y64 = ofp8.incoherent_transform(x.double().numpy(), signs.cpu().numpy())
    _, ods, y32 = ofp8.prepare(x.double().numpy(), signs.cpu().numpy(), True)
    g_ds = ds.cpu().numpy()
    np.testing.assert_allclose(g_ds, ods, rtol=4e-6, atol=0)
    t = np.arange(N) // 128
    q_exact = y64 / ods.astype(np.float64)[:, :, t].transpose(0, 2, 1)[..., None]
    tol = 4e-6 * np.abs(q_exact) + 1e-30
    lo, hi = ofp8.e4m3_encode(q_exact - tol), ofp8.e4m3_encode(q_exact + tol)
    g = codes.cpu().numpy()
    ok = (g == lo) | (g == hi)
    assert ok.all(), np.argwhere(~ok)[:5]
    # and almost all codes are the exact nearest-even code
    assert np.mean(g != ofp8.e4m3_encode(q_exact)) < 1e-3


def _fp8_forward(gpu_lib, q, k, v, causal, hadamard, Hkv):
    d = q.shape[-1]
    signs = _signs(Hkv, d) if hadamard else None
    q8, qd = gpu_lib.attn_prep_fp8(q, signs=signs, sign_heads=Hkv if hadamard else None)
    k8, kd = gpu_lib.attn_prep_fp8(k, signs=signs, sign_heads=Hkv if hadamard else None)
    v8, vd = gpu_lib.attn_prep_fp8(v, transpose_out=True)
    o, lse = gpu_lib.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=causal, hadamard=hadamard)
    assert gpu_lib.get_status() == 0
    return o, lse


def _oracle_codes(q, k, v, hadamard, Hkv, per_tensor=False, rope=False):
    """The oracle's FP8 preparation of Q, K, V: [(codes, descale)] x 3 (numpy,
    BSHD) and the dequantised float64 values."""
    d = q.shape[-1]
    sg = synth.hadamard_signs(Hkv, d, seed=0).numpy() if hadamard else None
    codes, deq = [], []
    for t, had, rot in ((q, hadamard, rope), (k, hadamard, rope), (v, False, False)):
        c, ds, _ = ofp8.prepare(t.double().cpu().numpy(), sg, had, per_tensor=per_tensor,
                                rope_base=10000.0 if rot else None)
        codes.append((c, ds))
        deq.append(ofp8.dequantize(c, ds))
    return codes, deq


def _oracle_on(deq, causal, Hq, rows=None):
    """FP64 oracle attention on dequantised values (every row or `rows`)."""
    qd, kd, vd = deq
    scale = 1 / math.sqrt(qd.shape[-1])
    if rows is None:
        return oracle.attention_full(qd, kd, vd, causal=causal, scale=scale)
    return oracle.attention_rows(qd[rows[:, 0], rows[:, 2], rows[:, 1]], kd, vd,
                                 Hq=Hq, causal=causal, scale=scale, rows=rows)


def _oracle_dequant(q, k, v, causal, hadamard, Hkv, rows=None, per_tensor=False, rope=False):
    """Oracle on its own FP8 quantisation of the same inputs (dequantised)."""
    _, deq = _oracle_codes(q, k, v, hadamard, Hkv, per_tensor, rope)
    return _oracle_on(deq, causal, q.shape[2], rows)


def _forward_on_codes(gpu_lib, codes, causal, hadamard):
    """The FP8 forward kernel on given codes and descales (here the oracle's):
    Q, K as BSHD, V moved to the key-contiguous layout the kernel reads."""
    (cq, dq), (ck, dk), (cv, dv) = codes
    B, N, Hkv, d = cv.shape
    npad = (N + 15) // 16 * 16
    vt = np.zeros((B, Hkv, d, npad), dtype=np.uint8)
    vt[..., :N] = cv.transpose(0, 2, 3, 1)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    o, lse = gpu_lib.attn_fwd_fp8(dev(cq), dev(ck), dev(vt), dev(dq), dev(dk), dev(dv),
                                  causal=causal, hadamard=hadamard)
    assert gpu_lib.get_status() == 0
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp8_forward_vs_dequantised_oracle(gpu_lib, causal, hadamard, d):
    """Ragged multi-tile GQA case, x50 outliers, every row.

    * The forward kernel on the oracle's own codes and descales against the
      oracle on the same dequantised values: the remaining error is the E4M3
      rounding of P (relative 2^-4 at most) and the bfloat16 output.
    * The whole GPU chain (prep, then forward): without the transform its
      codes equal the oracle's (test_prep_bit_exact_without_transform), so
      its output must equal the forward on the oracle's codes bit for bit.
      With the transform a code may be one step off where the float32
      butterfly and the oracle's float64 product straddle a rounding
      midpoint (test_prep_with_transform_matches_oracle); on an outlier one
      such step moves a few logits: 99 % of the rows stay within the LSE
      bound."""
    B, N, Hq, Hkv = 1, 700, 4, 2
    q, k, v = synth.attn_inputs(B, N, N, Hq, Hkv, d, dtype=torch.bfloat16, seed=7,
                                outlier_frac=1e-3, device="cuda")
    codes, deq = _oracle_codes(q, k, v, hadamard, Hkv)
    o, lse = _forward_on_codes(gpu_lib, codes, causal, hadamard)
    o_ref, lse_ref = _oracle_on(deq, causal, Hq)
    e = errors(o, lse, o_ref, lse_ref)
    assert e["nonfinite"] == 0, e
    assert e["o_rel_rms"] <= 4e-2, e
    assert e["lse_max_abs"] <= 2e-3, e
    oc, lc = _fp8_forward(gpu_lib, q, k, v, causal, hadamard, Hkv)
    if not hadamard:
        assert torch.equal(oc, o) and torch.equal(lc, lse)
    else:
        ec = errors(oc, lc, o_ref, lse_ref)
        assert ec["nonfinite"] == 0 and ec["o_rel_rms"] <= 4e-2, ec
        dl = np.abs(lc.double().cpu().numpy() - lse_ref)
        assert np.mean(dl <= 2e-3) >= 0.99, np.mean(dl <= 2e-3)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_several_units_per_cta(gpu_lib, causal, d):
    """GQA with several work units per persistent CTA (B=1, Hq=32, Hkv=4,
    N=4096: 512 units of 256 query rows), so that the per-tile barrier phases
    (S released, P buffers full and free) carry over unit boundaries; sampled
    rows of every head against the oracle on the dequantised inputs."""
    B, N, Hq, Hkv = 1, 4096, 32, 4
    q, k, v = synth.attn_inputs(B, N, N, Hq, Hkv, d, dtype=torch.bfloat16, seed=31,
                                outlier_frac=1e-3, outlier_scale=10.0, device="cuda")
    codes, deq = _oracle_codes(q, k, v, False, Hkv)
    o, lse = _forward_on_codes(gpu_lib, codes, causal, False)
    rows = synth.sample_rows(B, Hq, N, per_head=16, seed=3)
    idx = torch.as_tensor(rows, device="cuda")
    og = o[idx[:, 0], idx[:, 2], idx[:, 1]].double().cpu().numpy()
    lg = lse[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    o_ref, lse_ref = _oracle_on(deq, causal, Hq, rows=rows)
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    rel_rms = math.sqrt(np.mean((og - o_ref) ** 2) / np.mean(o_ref ** 2))
    assert rel_rms <= 4e-2, rel_rms
    assert np.max(np.abs(lg - lse_ref)) <= 2e-3, np.max(np.abs(lg - lse_ref))


@pytest.mark.parametrize("outlier_scale", [50.0, 10.0])
def test_fp8_full_workload_accuracy_and_hadamard(gpu_lib, outlier_scale):
    """B=4, H=16, N=4096, d=128, 0.1% of entries multiplied by `outlier_scale`.

    Against the oracle on the original BF16 values (the truth), sampled rows:
    * the GPU adds no error beyond the quantisation scheme itself: its RMS is
      within 10 % of the RMS of the oracle run on its own E4M3 quantisation of
      the same inputs;
    * the Hadamard-processed run is no worse than plain FP8;
    * at x10 outliers the RMS error is <= 5e-2.  At x50 the scheme's own error
      (E4M3 rounding of Q and K when outliers make logits reach the hundreds)
      is above that bound for any implementation of it, so the bound there is
      the scheme's own error."""
    B, N, H, d = 4, 4096, 16, 128
    q, k, v = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=0,
                                outlier_frac=1e-3, outlier_scale=outlier_scale, device="cuda")
    rows = synth.sample_rows(B, H, N, per_head=32, seed=0)
    idx = torch.as_tensor(rows, device="cuda")
    q_rows = synth.raw_bits(q[idx[:, 0], idx[:, 2], idx[:, 1]])
    o_ref, lse_ref = oracle.attention_rows(q_rows, synth.raw_bits(k), synth.raw_bits(v), Hq=H,
                                           causal=False, scale=1 / math.sqrt(d), rows=rows,
                                           elem=oracle.ELEM_BF16)
    rms, rms_scheme = {}, {}
    for had in (False, True):
        o, lse = _fp8_forward(gpu_lib, q, k, v, False, had, H)
        og = o[idx[:, 0], idx[:, 2], idx[:, 1]].double().cpu().numpy()
        lg = lse[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
        assert np.isfinite(og).all() and np.isfinite(lg).all()
        rms[had] = math.sqrt(np.mean((og - o_ref) ** 2))
        o_sch, _ = _oracle_dequant(q, k, v, False, had, H, rows=rows)
        rms_scheme[had] = math.sqrt(np.mean((o_sch - o_ref) ** 2))
        assert rms[had] <= 1.10 * rms_scheme[had] + 1e-3, (had, rms, rms_scheme)
    assert rms[True] <= rms[False], rms
    if outlier_scale <= 10.0:
        assert rms[False] <= 5e-2 and rms[True] <= 5e-2, rms


def test_fp8_full_workload_every_row_vs_dequantised_oracle(gpu_lib):
    """B=4, H=16, N=4096, d=128, x50 outliers, with and without the transform,
    in the bench's launch configuration: all 262,144 rows of the forward
    kernel run on the oracle's own E4M3 codes against the FP64 oracle on the
    same dequantised values (the kernel's arithmetic up to the E4M3 rounding
    of P and the bfloat16 output); without the transform the whole GPU chain
    gives the same output bit for bit."""
    B, N, H, d = 4, 4096, 16, 128
    q, k, v = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=0,
                                outlier_frac=1e-3, device="cuda")
    for had in (False, True):
        codes, deq = _oracle_codes(q, k, v, had, H)
        o, lse = _forward_on_codes(gpu_lib, codes, False, had)
        o_ref, lse_ref = _oracle_on(deq, False, H)
        e = errors(o, lse, o_ref, lse_ref)
        assert e["nonfinite"] == 0, (had, e)
        assert e["o_rel_rms"] <= 4e-2, (had, e)
        assert e["lse_max_abs"] <= 2e-3, (had, e)
        if not had:
            # the GPU chain's codes equal the oracle's: the same output
            oc, lc = _fp8_forward(gpu_lib, q, k, v, False, False, H)
            assert torch.equal(oc, o) and torch.equal(lc, lse)


# --- per-tensor baseline ------------------------------------------------------

@pytest.mark.parametrize("d,N,H", [(64, 1000, 3), (128, 1000, 3), (256, 1000, 3),
                                   (128, 4000, 16)])
def test_prep_per_tensor_bit_exact_without_transform(gpu_lib, d, N, H):
    """Small cases, and one with several times more tiles than CTAs (most
    tiles of both passes claimed from the launch's counter)."""
    B = 2
    x, _, _ = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=21,
                                outlier_frac=1e-3)
    codes, ds = gpu_lib.attn_prep_fp8_per_tensor(x.cuda())
    codes_t, ds_t = gpu_lib.attn_prep_fp8_per_tensor(x.cuda(), transpose_out=True)
    assert gpu_lib.get_status() == 0
    xf = x.float().numpy()
    oc, ods, _ = ofp8.prepare(xf, per_tensor=True)
    np.testing.assert_array_equal(ds.cpu().numpy(), ods)
    np.testing.assert_array_equal(ds_t.cpu().numpy(), ods)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(codes_t.cpu().numpy()[..., :N], oc.transpose(0, 2, 3, 1))
    # a second call on other data leaves nothing behind (descale[0] is reused
    # as the amax accumulator)
    z = torch.zeros_like(x).cuda()
    cz, dz = gpu_lib.attn_prep_fp8_per_tensor(z, descale=ds)
    assert not cz.any() and bool((dz == 1.0).all())


def _codes_near(g, q_exact, rel=4e-6, abs_=4e-5):
    """Every code is the E4M3 code of a value within the tolerance of the
    exact scaled value; almost all are the exact nearest-even code."""
    tol = rel * np.abs(q_exact) + abs_
    lo, hi = ofp8.e4m3_encode(q_exact - tol), ofp8.e4m3_encode(q_exact + tol)
    ok = (g == lo) | (g == hi)
    assert ok.all(), np.argwhere(~ok)[:5]
    assert np.mean(g != ofp8.e4m3_encode(q_exact)) < 1e-3


def test_prep_per_tensor_with_transform(gpu_lib):
    B, N, Hq, Hkv, d = 1, 700, 4, 2, 128
    x, _, _ = synth.attn_inputs(B, N, N, Hq, Hkv, d, dtype=torch.bfloat16, seed=22,
                                outlier_frac=1e-3)
    signs = _signs(Hkv, d)
    codes, ds = gpu_lib.attn_prep_fp8_per_tensor(x.cuda(), signs=signs, sign_heads=Hkv)
    assert gpu_lib.get_status() == 0
    y64 = ofp8.incoherent_transform(x.double().numpy(), signs.cpu().numpy())
    _, ods, _ = ofp8.prepare(x.double().numpy(), signs.cpu().numpy(), True, per_tensor=True)
    g_ds = ds.cpu().numpy()
    np.testing.assert_allclose(g_ds, ods, rtol=4e-6, atol=0)
    assert np.all(g_ds == g_ds.flat[0])
    _codes_near(codes.cpu().numpy(), y64 / float(ods.flat[0]))


# --- rotary embedding fused into the prep -------------------------------------

@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("pos0", [0, 123457])
def test_rope_table_matches_oracle(gpu_lib, d, pos0):
    N = 3000
    cos, sin = gpu_lib.attn_rope_table(N, d, base=10000.0, pos0=pos0)
    assert gpu_lib.get_status() == 0
    oc, osn = ofp8.rope_tables(N, d, 10000.0, pos0)
    # double-precision evaluation rounded once to float32: within half a
    # float32 ulp of 1 (plus the double evaluation's own error)
    np.testing.assert_allclose(cos.cpu().numpy(), oc, rtol=0, atol=7e-8)
    np.testing.assert_allclose(sin.cpu().numpy(), osn, rtol=0, atol=7e-8)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("hadamard", [False, True])
def test_prep_rope_matches_oracle(gpu_lib, d, hadamard):
    """Rotation, transform and block quantisation in one pass, against the
    oracle's float64 rotation (and transform) of the same rows: codes within
    the float32 rounding of the exact scaled value, descales to float32
    rounding; ragged last block."""
    B, N, Hq, Hkv = 2, 650, 4, 2
    x, _, _ = synth.attn_inputs(B, N, N, Hq, Hkv, d, dtype=torch.bfloat16, seed=23,
                                outlier_frac=1e-3)
    cos, sin = gpu_lib.attn_rope_table(N, d)
    signs = _signs(Hkv, d) if hadamard else None
    codes, ds = gpu_lib.attn_prep_fp8_rope(x.cuda(), cos, sin, signs=signs,
                                           sign_heads=Hkv if hadamard else None)
    assert gpu_lib.get_status() == 0
    y64 = ofp8.rope(x.double().numpy(), 10000.0)
    if hadamard:
        y64 = ofp8.incoherent_transform(y64, signs.cpu().numpy())
    _, ods, _ = ofp8.prepare(x.double().numpy(), signs.cpu().numpy() if hadamard else None,
                             hadamard, rope_base=10000.0)
    g_ds = ds.cpu().numpy()
    np.testing.assert_allclose(g_ds, ods, rtol=4e-6, atol=0)
    t = np.arange(N) // 128
    q_exact = y64 / ods.astype(np.float64)[:, :, t].transpose(0, 2, 1)[..., None]
    _codes_near(codes.cpu().numpy(), q_exact)


@pytest.mark.parametrize("variant", ["per_tensor", "per_tensor_hadamard", "rope", "rope_hadamard"])
def test_fp8_forward_variants_vs_dequantised_oracle(gpu_lib, variant):
    """The forward on the oracle's per-tensor and rotated codes, every row,
    against the oracle on the same dequantised values; then the GPU chain."""
    B, N, Hq, Hkv, d = 1, 700, 4, 2, 128
    q, k, v = synth.attn_inputs(B, N, N, Hq, Hkv, d, dtype=torch.bfloat16, seed=24,
                                outlier_frac=1e-3, outlier_scale=10.0, device="cuda")
    had = variant.endswith("hadamard")
    signs = _signs(Hkv, d) if had else None
    sh = Hkv if had else None
    pt, rot = variant.startswith("per_tensor"), variant.startswith("rope")
    codes, deq = _oracle_codes(q, k, v, had, Hkv, per_tensor=pt, rope=rot)
    o, lse = _forward_on_codes(gpu_lib, codes, True, had)
    o_ref, lse_ref = _oracle_on(deq, True, Hq)
    e = errors(o, lse, o_ref, lse_ref)
    assert e["nonfinite"] == 0, e
    assert e["o_rel_rms"] <= 4e-2, e
    assert e["lse_max_abs"] <= 2e-3, e
    # the GPU chain: identical codes (per-tensor without the transform) give
    # the identical output; float32 rotation / transform leave 99 % of rows
    # within the bound (see test_fp8_forward_vs_dequantised_oracle)
    if pt:
        q8, qd = gpu_lib.attn_prep_fp8_per_tensor(q, signs=signs, sign_heads=sh)
        k8, kd = gpu_lib.attn_prep_fp8_per_tensor(k, signs=signs, sign_heads=sh)
        v8, vd = gpu_lib.attn_prep_fp8_per_tensor(v, transpose_out=True)
    else:
        cos, sin = gpu_lib.attn_rope_table(N, d)
        q8, qd = gpu_lib.attn_prep_fp8_rope(q, cos, sin, signs=signs, sign_heads=sh)
        k8, kd = gpu_lib.attn_prep_fp8_rope(k, cos, sin, signs=signs, sign_heads=sh)
        v8, vd = gpu_lib.attn_prep_fp8(v, transpose_out=True)
    oc, lc = gpu_lib.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=True, hadamard=had)
    assert gpu_lib.get_status() == 0
    if variant == "per_tensor":
        assert torch.equal(oc, o) and torch.equal(lc, lse)
    else:
        ec = errors(oc, lc, o_ref, lse_ref)
        assert ec["nonfinite"] == 0 and ec["o_rel_rms"] <= 4e-2, ec
        dl = np.abs(lc.double().cpu().numpy() - lse_ref)
        assert np.mean(dl <= 2e-3) >= 0.99, np.mean(dl <= 2e-3)


def test_prep_rope_hadamard_full_size_sampled(gpu_lib):
    """The rotary + transform prep at the FP8 workload's size (B=4, H=16,
    N=4096, d=128, x50 outliers), in the launch configuration the bench uses:
    every descale, and the codes of sampled rows, against the oracle."""
    B, N, H, d = 4, 4096, 16, 128
    q, _, _ = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=0,
                                outlier_frac=1e-3, device="cuda")
    cos, sin = gpu_lib.attn_rope_table(N, d)
    signs = _signs(H, d)
    codes, ds = gpu_lib.attn_prep_fp8_rope(q, cos, sin, signs=signs, sign_heads=H)
    assert gpu_lib.get_status() == 0
    x = q.double().cpu().numpy()
    _, ods, _ = ofp8.prepare(x, signs.cpu().numpy(), True, rope_base=10000.0)
    g_ds = ds.cpu().numpy()
    np.testing.assert_allclose(g_ds, ods, rtol=4e-6, atol=0)
    rows = synth.sample_rows(B, H, N, per_head=16, seed=3)
    # exact rotated + transformed values of the sampled rows only
    xr = x[rows[:, 0], rows[:, 2], rows[:, 1]]                       # [R, d]
    cos_t, sin_t = ofp8.rope_tables(N, d, 10000.0)
    c, s_ = cos_t[rows[:, 2]], sin_t[rows[:, 2]]
    a, b = xr[:, : d // 2], xr[:, d // 2:]
    rot = np.concatenate([a * c - b * s_, b * c + a * s_], axis=-1)
    sg = signs.cpu().numpy().astype(np.float64)[rows[:, 1]]
    y = (rot * sg) @ ofp8.hadamard_matrix(d).astype(np.float64) / np.sqrt(d)
    q_exact = y / ods.astype(np.float64)[rows[:, 0], rows[:, 1], rows[:, 2] // 128][:, None]
    g = codes.cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    _codes_near(g, q_exact)


# --- Q, K, V prepared in one launch ------------------------------------------

@pytest.mark.parametrize("variant", ["plain", "hadamard", "rope_hadamard"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_prep_qkv_one_launch_equals_separate_calls(gpu_lib, variant, d):
    """attn_prep_fp8_qkv gives the codes and descales of the three separate
    calls bit for bit (GQA, Nq != Nk, ragged last blocks); without the
    transform they are also the oracle's."""
    B, Nq, Nk, Hq, Hkv = 2, 650, 390, 4, 2
    q, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=torch.bfloat16, seed=25,
                                outlier_frac=1e-3, device="cuda")
    signs = _signs(Hkv, d) if variant != "plain" else None
    rope = gpu_lib.attn_rope_table(max(Nq, Nk), d) if variant == "rope_hadamard" else None
    got = gpu_lib.attn_prep_fp8_qkv(q, k, v, signs=signs, rope=rope)
    assert gpu_lib.get_status() == 0
    if rope is None:
        want = (*gpu_lib.attn_prep_fp8(q, signs=signs, sign_heads=Hkv),
                *gpu_lib.attn_prep_fp8(k, signs=signs, sign_heads=Hkv),
                *gpu_lib.attn_prep_fp8(v, transpose_out=True))
    else:
        cq, sq = gpu_lib.attn_rope_table(Nq, d)
        ck, sk = gpu_lib.attn_rope_table(Nk, d)
        want = (*gpu_lib.attn_prep_fp8_rope(q, cq, sq, signs=signs, sign_heads=Hkv),
                *gpu_lib.attn_prep_fp8_rope(k, ck, sk, signs=signs, sign_heads=Hkv),
                *gpu_lib.attn_prep_fp8(v, transpose_out=True))
    for g, w in zip(got, want):
        assert g.shape == w.shape and torch.equal(g, w)
    if variant == "plain":
        for t, (c, ds) in zip((q, k), ((got[0], got[1]), (got[2], got[3]))):
            oc, ods, _ = ofp8.prepare(t.float().cpu().numpy(), None, False)
            np.testing.assert_array_equal(c.cpu().numpy(), oc)
            np.testing.assert_array_equal(ds.cpu().numpy(), ods)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_prep_qkv_claimed_tiles_bit_exact_repeated_and_on_two_streams(gpu_lib, d):
    """A launch with several times more tiles than CTAs (most tiles are
    claimed from the launch's counter while others run): codes and descales
    are the oracle's, bit for bit (ragged last block, transposed V), on
    every one of several calls in a row (each launch leaves its counter at
    zero for the next), and two launches running at once on two streams give
    the codes of sequential calls."""
    B, N, H = 2, 4000, 16
    q, k, v = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=26,
                                outlier_frac=1e-3, device="cuda")
    first = gpu_lib.attn_prep_fp8_qkv(q, k, v)
    assert gpu_lib.get_status() == 0
    for t, c, ds in ((q, first[0], first[1]), (k, first[2], first[3])):
        oc, ods, _ = ofp8.prepare(t.float().cpu().numpy(), None, False)
        np.testing.assert_array_equal(ds.cpu().numpy(), ods)
        np.testing.assert_array_equal(c.cpu().numpy(), oc)
    oc, ods, _ = ofp8.prepare(v.float().cpu().numpy(), None, False)
    np.testing.assert_array_equal(first[5].cpu().numpy(), ods)
    np.testing.assert_array_equal(first[4].cpu().numpy()[..., :N], oc.transpose(0, 2, 3, 1))
    for _ in range(5):
        again = gpu_lib.attn_prep_fp8_qkv(q, k, v)
        for g, w in zip(again, first):
            assert torch.equal(g, w)
    # a second problem, prepared alone, then both at once on two streams
    q2, k2, v2 = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=27,
                                   outlier_frac=1e-3, device="cuda")
    alone = gpu_lib.attn_prep_fp8_qkv(q2, k2, v2)
    out1 = tuple(torch.empty_like(t) for t in first)
    out2 = tuple(torch.empty_like(t) for t in alone)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        gpu_lib.attn_prep_fp8_qkv(q, k, v, out=out1, stream=s1)
        gpu_lib.attn_prep_fp8_qkv(q2, k2, v2, out=out2, stream=s2)
    torch.cuda.synchronize()
    assert gpu_lib.get_status() == 0
    for g, w in zip(out1, first):
        assert torch.equal(g, w)
    for g, w in zip(out2, alone):
        assert torch.equal(g, w)
