"""Seeded synthetic inputs for attention workloads.

This module is the only code that both the GPU path's callers (tests, smoke,
bench) and the CPU oracle's callers share.  It draws random numbers and casts
them; it holds none of the attention method's arithmetic.

Recipe (every workload):
* Q, K, V are iid N(0, 1) drawn in float32 from a ``torch.Generator`` seeded
  with ``seed``, in BSHD layout ([B, N, H, d], d innermost), drawn in the
  order Q, K, V, then cast to the working dtype with round-to-nearest-even.
* Outlier injection (the FP8 workload): after each tensor's normal draw, a
  uniform draw from the same generator selects entries with probability
  ``outlier_frac`` (0.1 %), which are multiplied by ``outlier_scale`` (50).
* Channel outliers (a second outlier structure for the FP8 error study):
  from a CPU generator seeded with ``seed + 11``, ``channel_outliers``
  channels are chosen per key/value head (a random permutation's first
  entries); every token's value in them is multiplied by ``channel_scale`` in
  K and in the query heads of that group; V is left as drawn.
* Hadamard signs: +-1 per (key/value head, channel) from a generator seeded
  with ``seed + 7``.
* Sampled query rows: uniform per (b, h) from a generator seeded with
  ``seed + 1``, always including rows {0, 1, 127, 128, N - 1} that exist.
"""
from __future__ import annotations

import numpy as np
import torch


def _draw(shape, gen, device, outlier_frac, outlier_scale):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        t = torch.where(u < outlier_frac, t * outlier_scale, t)
    return t


def _channel_mult(Hkv, d, gen, n_channels, scale):
    mult = torch.ones(Hkv, d, dtype=torch.float32)
    for h in range(Hkv):
        mult[h, torch.randperm(d, generator=gen)[:n_channels]] = scale
    return mult


def attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=torch.bfloat16, seed=0, device="cpu",
                outlier_frac=0.0, outlier_scale=50.0, channel_outliers=0, channel_scale=10.0):
    """Return (q, k, v) in BSHD with the given dtype on ``device``.

    With ``device='cuda'`` the draw uses a CUDA generator (a different but
    equally seeded stream), which keeps multi-GB workloads off the host."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    q = _draw((B, Nq, Hq, d), gen, dev, outlier_frac, outlier_scale)
    k = _draw((B, Nk, Hkv, d), gen, dev, outlier_frac, outlier_scale)
    v = _draw((B, Nk, Hkv, d), gen, dev, outlier_frac, outlier_scale)
    if channel_outliers > 0:
        cgen = torch.Generator().manual_seed(int(seed) + 11)
        mult = _channel_mult(Hkv, d, cgen, channel_outliers, channel_scale).to(dev)
        q = q * mult.repeat_interleave(Hq // Hkv, dim=0)
        k = k * mult
    return q.to(dtype), k.to(dtype), v.to(dtype)


def hadamard_signs(G, d, seed=0) -> torch.Tensor:
    """[G, d] int8 of +-1 (one row per key/value head)."""
    gen = torch.Generator().manual_seed(int(seed) + 7)
    bits = torch.randint(0, 2, (G, d), generator=gen)
    return (1 - 2 * bits).to(torch.int8)


def sample_rows(B, H, N, per_head, seed=0) -> np.ndarray:
    """[R, 3] int64 of (b, h, i): ``per_head`` rows per (b, h) plus fixed edge rows."""
    rng = np.random.default_rng(int(seed) + 1)
    fixed = [i for i in (0, 1, 127, 128, N - 1) if 0 <= i < N]
    out = []
    for b in range(B):
        for h in range(H):
            extra = rng.choice(N, size=min(per_head, N), replace=False)
            idx = np.unique(np.concatenate([np.asarray(fixed, dtype=np.int64), extra]))
            for i in idx:
                out.append((b, h, int(i)))
    return np.asarray(out, dtype=np.int64).reshape(-1, 3)


def raw_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 bit patterns of a 16-bit float tensor (no value conversion)."""
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("16-bit float tensor expected")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
