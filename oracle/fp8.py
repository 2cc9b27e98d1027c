"""FP8 E4M3 codec, Hadamard matrix and per-block quantisation (numpy oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources and readings
--------------------
* Block quantisation: "FlashAttention（V3）深度解析" (dtcms.com), section 4.3
  "块量化与非一致处理": each block keeps a scale factor so that it can be
  brought back to its floating-point range; dequantisation is fused into the
  attention pipeline.  Reading taken: symmetric per-block scale, no offset
  (FP8 is sign-magnitude), one block = 128 tokens x d of one (batch, head);
  descale = amax / 448 (448 = largest finite E4M3 value) rounded to float32,
  descale = 1 for an all-zero block; code = E4M3(x / descale) rounded to
  nearest-even with saturation to +-448, the quotient of the float32 value
  and the float32 descale taken exactly (no intermediate rounding that could
  move it across an E4M3 rounding boundary).  The last block of a sequence
  may be partial.
* FP8 format: the pages say "FP8" (H100 FP8 tensor cores, 1978 TFLOPS, in
  the Together AI summary card "FlashAttention-3——利用异步与低精度加速注意力机制");
  the code on the dtcms.com page (section 11, FP8Support.fp32_to_fp8_conversion)
  clamps to +-240 and rounds to a 1/16 grid, which is not E4M3; that garbled
  helper is not followed.  The format here is OCP E4M3FN: 1 sign, 4 exponent
  bits (bias 7), 3 mantissa bits, subnormals kept, no infinities, S.1111.111
  is NaN, largest finite value 448.
* Incoherent processing: the summary card, section "低精度优化：非相干处理":
  each attention head is multiplied by a random orthogonal matrix (a Hadamard
  transform with random signs) to spread outliers before FP8 quantisation.
  Reading taken: M_h = diag(sigma_h) H_d / sqrt(d), H_d the Sylvester
  Hadamard matrix H[i, j] = (-1)^popcount(i & j), applied to Q and K only
  (Q M (K M)^T = Q K^T for orthogonal M, so O needs no inverse transform);
  sigma_h in {+1, -1}^d is an input, one row per key/value head, shared by the
  query heads of that group.

* Per-tensor FP8 (the baseline of the error comparison): the summary card,
  same section, says incoherent processing gives 2.6 times lower error than
  "baseline FP8" without naming that baseline.  Reading taken: one scale for
  the whole tensor (all batches, heads and tokens), descale = amax / 448,
  codes = E4M3(x / descale) as for a block.  The descale
  is written for every (b, head, block) so that the same forward consumes
  either scheme.
* Rotary embedding fused with the transform: the summary card, same section,
  says the Hadamard transform can be fused with rotary embedding (a
  bandwidth-bound step) at no extra cost.  The pages define no rotary
  variant.  Reading taken: the rotate-half form, channel c paired with
  c + d/2 for c < d/2, angle (pos0 + n) * base^(-2c/d) for token n, base
  10000 by default; (x_c, x_{c+d/2}) -> (x_c cos - x_{c+d/2} sin,
  x_{c+d/2} cos + x_c sin).  It is applied to Q and K before the Hadamard
  transform (the rotation must act on the model's own Q and K; M is applied
  after it so that Q M (K M)^T is still the rotated Q K^T), never to V.

Precision of the quantisation decision: the values that are quantised are
float32 (the inputs themselves, or the rotated / transformed values formed in
float64 and rounded once to float32); the block amax is exact; the descale
amax / 448 is rounded to float32 once (it is what the forward pass reads); the
code is the E4M3 rounding of the exact quotient value / descale.  The
quotient is formed in float64: a float32 value over a float32 descale lies
on an E4M3 rounding midpoint exactly when its float64 rounding does (a
midpoint times the descale has at most 29 significant bits, so a quotient
that misses a midpoint misses it by far more than a float64 ulp), so the
float64 division decides every code as the exact quotient would.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3FN byte codes to float64 from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    v = np.where(e == 0, sub, normal)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return sign * v


def e4m3_encode(x) -> np.ndarray:
    """Encode real values to E4M3FN codes: round to nearest, ties to even
    significand, saturate finite overflow to +-448, NaN to 0x7F."""
    xv = np.asarray(x, dtype=np.float64)
    a = np.abs(xv)
    sign = np.signbit(xv)
    # binade exponent of |x| (frexp is exact: a = f * 2^ex, f in [0.5, 1)),
    # floored at the smallest normal binade 2^-6 and capped at the top binade 2^8
    _, ex = np.frexp(np.where(np.isfinite(a) & (a > 0), a, 1.0))
    e = np.clip(ex.astype(np.float64) - 1.0, -6.0, 8.0)
    quantum = np.exp2(e - 3.0)            # spacing of representable values in the binade
    k = np.rint(np.where(np.isfinite(a), a, E4M3_MAX) / quantum)  # half-to-even
    v = k * quantum
    # a value that rounds up past its binade lands on the next power of two,
    # which is representable; finite overflow saturates to the largest value
    v = np.minimum(v, E4M3_MAX)
    # v is now exactly representable: build its code
    _, vex = np.frexp(np.where(v > 0, v, 1.0))
    ve = vex.astype(np.float64) - 1.0
    is_sub = v < 2.0 ** -6
    mant_sub = np.rint(v / 2.0 ** -9).astype(np.int64)
    ebits = (ve + 7.0).astype(np.int64)
    mant_norm = np.rint((v / np.exp2(ve) - 1.0) * 8.0).astype(np.int64)
    code = np.where(is_sub, mant_sub, (ebits << 3) | mant_norm)
    code = np.where(sign, code | 0x80, code)
    code = np.where(np.isnan(xv), 0x7F, code)
    return code.astype(np.uint8)


def hadamard_matrix(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix: H[i, j] = (-1)^popcount(i & j)  (integer +-1)."""
    if d < 1 or (d & (d - 1)) != 0:
        raise ValueError("d must be a power of two")
    i = np.arange(d)[:, None]
    j = np.arange(d)[None, :]
    bits = np.bitwise_and(i, j)
    pc = np.zeros_like(bits)
    t = bits.copy()
    while np.any(t):
        pc += t & 1
        t >>= 1
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def incoherent_transform(x, signs, sign_heads: int | None = None) -> np.ndarray:
    """x [B, N, H, d] -> (x * sigma_g(h)) @ H_d / sqrt(d) in float64.

    signs: [G, d] of +-1; head h uses row h // (H // G)."""
    x = np.asarray(x, dtype=np.float64)
    B, N, H, d = x.shape
    s = np.asarray(signs, dtype=np.float64)
    G = s.shape[0] if sign_heads is None else sign_heads
    if H % G != 0:
        raise ValueError("H must be a multiple of the number of sign rows")
    sig = s[np.arange(H) // (H // G)]            # [H, d]
    Hd = hadamard_matrix(d).astype(np.float64)
    return np.einsum("bnhc,cj->bnhj", x * sig[None, None], Hd) / np.sqrt(d)


def quantize_blocks(y32: np.ndarray, block: int = BLOCK):
    """Per-(b, h, 128-token block) symmetric quantisation of float32 values.

    y32 : [B, N, H, d] float32.
    Returns (codes uint8 [B, N, H, d], descale float32 [B, H, ceil(N/block)]).
    """
    y32 = np.asarray(y32, dtype=np.float32)
    B, N, H, d = y32.shape
    nb = (N + block - 1) // block
    codes = np.zeros((B, N, H, d), dtype=np.uint8)
    descale = np.ones((B, H, nb), dtype=np.float32)
    for t in range(nb):
        n0, n1 = t * block, min(N, (t + 1) * block)
        blk = y32[:, n0:n1]                                   # [B, n, H, d]
        amax = np.abs(blk).max(axis=(1, 3)).astype(np.float32)  # [B, H], exact
        ds = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        descale[:, :, t] = ds
        # q = x / descale, decided as the exact quotient (see the module notes)
        q = blk.astype(np.float64) / ds.astype(np.float64)[:, None, :, None]
        codes[:, n0:n1] = e4m3_encode(q)
    return codes, descale


def quantize_tensor(y32: np.ndarray, block: int = BLOCK):
    """One symmetric scale for the whole tensor (the per-tensor FP8 baseline).

    y32 : [B, N, H, d] float32.  Returns (codes uint8 [B, N, H, d], descale
    float32 [B, H, ceil(N/block)]) with every descale equal to amax / 448 (1
    for an all-zero tensor), amax taken over every element."""
    y32 = np.asarray(y32, dtype=np.float32)
    B, N, H, d = y32.shape
    nb = (N + block - 1) // block
    amax = np.float32(np.abs(y32).max()) if y32.size else np.float32(0.0)
    ds = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    codes = e4m3_encode(y32.astype(np.float64) / np.float64(ds))   # exact quotient decides
    return codes, np.full((B, H, nb), ds, dtype=np.float32)


def rope_tables(N: int, d: int, base: float = 10000.0, pos0: int = 0):
    """cos and sin of the rotary angles, float64 [N, d/2]:
    angle[n, c] = (pos0 + n) * base^(-2c/d)."""
    if d % 2:
        raise ValueError("d must be even")
    c = np.arange(d // 2, dtype=np.float64)
    freq = np.power(np.float64(base), -2.0 * c / d)
    ang = (pos0 + np.arange(N, dtype=np.float64))[:, None] * freq[None, :]
    return np.cos(ang), np.sin(ang)


def rope(x, base: float = 10000.0, pos0: int = 0) -> np.ndarray:
    """Rotate-half rotary embedding of x [B, N, H, d] in float64: channel c
    and c + d/2 rotate by angle[n, c] (see rope_tables)."""
    x = np.asarray(x, dtype=np.float64)
    B, N, H, d = x.shape
    cos, sin = rope_tables(N, d, base, pos0)
    cos, sin = cos[None, :, None, :], sin[None, :, None, :]
    a, b = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def prepare(x, signs=None, hadamard: bool = False, per_tensor: bool = False,
            rope_base: float | None = None, rope_pos0: int = 0):
    """The oracle of the FP8 preparation step on one tensor [B, N, H, d].

    x is the exact input (bf16 values as float32/float64).  Steps, in order:
    rotary embedding (when rope_base is given), the Hadamard transform (when
    hadamard), rounding to float32, then per-block (default) or per-tensor
    quantisation.  Returns (codes uint8 [B, N, H, d], descale float32
    [B, H, nblocks], y32) where y32 is the float32 tensor that was quantised."""
    x = np.asarray(x)
    if rope_base is None and not hadamard:
        y32 = np.asarray(x, dtype=np.float32)
    else:
        y = np.asarray(x, dtype=np.float64)
        if rope_base is not None:
            y = rope(y, rope_base, rope_pos0)
        if hadamard:
            y = incoherent_transform(y, signs)
        y32 = y.astype(np.float32)
    codes, ds = quantize_tensor(y32) if per_tensor else quantize_blocks(y32)
    return codes, ds, y32


def dequantize(codes, descale, block: int = BLOCK) -> np.ndarray:
    """codes [B, N, H, d], descale [B, H, nb] -> float64 values."""
    v = e4m3_decode(codes)
    B, N, H, d = v.shape
    t = np.arange(N) // block
    ds = np.asarray(descale, dtype=np.float64)[:, :, t]       # [B, H, N]
    return v * ds.transpose(0, 2, 1)[..., None]
