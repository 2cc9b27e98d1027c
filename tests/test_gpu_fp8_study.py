"""FP8 error study on the GPU: the four quantisation schemes (one scale per
tensor or per 128-token block, with or without the Hadamard transform) on
the FP8 workload shape (B=4, H=16, N=4096, d=128), against the FP64 oracle
on the original BF16 values (sampled rows).

The summary card (FlashAttention-3 summary, low-precision section) reports
2.6 times lower error than baseline FP8 for the transform, on a workload it
does not state.  Two outlier structures stand in for it:
* entry outliers: 0.1 % of the entries of Q, K and V multiplied by 10 or 50;
* channel outliers: 4 channels per key/value head multiplied by 5 in Q and K
  for every token (the structure the transform is meant to spread).

Set ATTN_FP8_STUDY_JSON to a file name to have the table written there."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

SCHEMES = ("tensor", "tensor+H", "block", "block+H")
RECIPES = {
    "entry_x10": dict(outlier_frac=1e-3, outlier_scale=10.0),
    "entry_x50": dict(outlier_frac=1e-3, outlier_scale=50.0),
    "channel4_x5": dict(channel_outliers=4, channel_scale=5.0),
}


def _scheme_forward(gpu_lib, q, k, v, scheme, signs):
    per_tensor = scheme.startswith("tensor")
    had = scheme.endswith("+H")
    prep = gpu_lib.attn_prep_fp8_per_tensor if per_tensor else gpu_lib.attn_prep_fp8
    sg = signs if had else None
    sh = signs.shape[0] if had else None
    q8, qd = prep(q, signs=sg, sign_heads=sh)
    k8, kd = prep(k, signs=sg, sign_heads=sh)
    v8, vd = prep(v, transpose_out=True)
    o, _ = gpu_lib.attn_fwd_fp8(q8, k8, v8, qd, kd, vd, causal=False, hadamard=had)
    assert gpu_lib.get_status() == 0
    return o


def test_fp8_error_study(gpu_lib):
    B, N, H, d = 4, 4096, 16, 128
    table = {}
    for name, recipe in RECIPES.items():
        q, k, v = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=0,
                                    device="cuda", **recipe)
        rows = synth.sample_rows(B, H, N, per_head=32, seed=0)
        idx = torch.as_tensor(rows, device="cuda")
        q_rows = synth.raw_bits(q[idx[:, 0], idx[:, 2], idx[:, 1]])
        o_ref, _ = oracle.attention_rows(q_rows, synth.raw_bits(k), synth.raw_bits(v), Hq=H,
                                         causal=False, scale=1 / math.sqrt(d), rows=rows,
                                         elem=oracle.ELEM_BF16)
        signs = synth.hadamard_signs(H, d, seed=0).cuda()
        errs = {}
        for scheme in SCHEMES:
            o = _scheme_forward(gpu_lib, q, k, v, scheme, signs)
            og = o[idx[:, 0], idx[:, 2], idx[:, 1]].double().cpu().numpy()
            assert np.isfinite(og).all()
            errs[scheme] = math.sqrt(np.mean((og - o_ref) ** 2))
        errs["ratio_tensor_over_blockH"] = errs["tensor"] / errs["block+H"]
        table[name] = errs
    out = os.environ.get("ATTN_FP8_STUDY_JSON")
    if out:
        with open(out, "w") as f:
            json.dump({"workload": "B4_H16_N4096_d128", "rows_per_head": 32,
                       "metric": "RMS(O_fp8 - O_exact)", "table": table}, f, indent=1)
    print(json.dumps(table, indent=1))
    for name, errs in table.items():
        # the transform never hurts, and block + transform beats the baseline
        assert errs["block+H"] <= errs["block"], (name, errs)
        assert errs["block+H"] <= errs["tensor"], (name, errs)
    assert table["channel4_x5"]["ratio_tensor_over_blockH"] >= 2.0, table
