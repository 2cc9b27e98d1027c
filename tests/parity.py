"""Helpers of the GPU parity tests: run the CUDA path, run the oracle on the
same seeded inputs, and compare with the stated tolerances.

Tolerances (FP16/BF16 forward): O max-abs error <= 1e-2, O RMS error <= 2e-3,
|LSE error| <= 1e-3, all against the FP64 oracle on the exact input values.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth

O_MAX_ABS = 1e-2
O_RMS = 2e-3
LSE_ABS = 1e-3


def oracle_for(q, k, v, causal, scale, rows=None):
    """FP64 oracle on the exact 16-bit values of q, k, v (torch tensors, any
    device).  rows=None: every row, returns (O [B,Nq,Hq,d], LSE [B,Hq,Nq]);
    else rows [R,3] of (b, h, i), returns (O [R,d], LSE [R])."""
    elem = oracle.ELEM_BF16 if q.dtype == torch.bfloat16 else oracle.ELEM_F16
    kb, vb = synth.raw_bits(k), synth.raw_bits(v)
    if rows is None:
        return oracle.attention_full(synth.raw_bits(q), kb, vb, causal=causal, scale=scale,
                                     elem=elem)
    idx = torch.as_tensor(rows, dtype=torch.long, device=q.device)
    q_rows = q[idx[:, 0], idx[:, 2], idx[:, 1]]
    return oracle.attention_rows(synth.raw_bits(q_rows), kb, vb, Hq=q.shape[2], causal=causal,
                                 scale=scale, rows=rows, elem=elem)


def errors(o_gpu, lse_gpu, o_ref, lse_ref):
    o = o_gpu.detach().double().cpu().numpy() if torch.is_tensor(o_gpu) else o_gpu
    l = lse_gpu.detach().double().cpu().numpy() if torch.is_tensor(lse_gpu) else lse_gpu
    d = o - o_ref
    return {
        "o_max_abs": float(np.abs(d).max()) if d.size else 0.0,
        "o_rms": float(math.sqrt(np.mean(d ** 2))) if d.size else 0.0,
        "o_rel_rms": float(np.linalg.norm(d) / max(np.linalg.norm(o_ref), 1e-300)) if d.size else 0.0,
        "lse_max_abs": float(np.abs(l - lse_ref).max()) if l.size else 0.0,
        "nonfinite": int(np.count_nonzero(~np.isfinite(o)) + np.count_nonzero(~np.isfinite(l))),
    }


def assert_within(err, o_max_abs=O_MAX_ABS, o_rms=O_RMS, lse_abs=LSE_ABS):
    assert err["nonfinite"] == 0, err
    assert err["o_max_abs"] <= o_max_abs, err
    assert err["o_rms"] <= o_rms, err
    assert err["lse_max_abs"] <= lse_abs, err


def gather_rows(o, lse, rows):
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    return o[idx[:, 0], idx[:, 2], idx[:, 1]], lse[idx[:, 0], idx[:, 1], idx[:, 2]]
