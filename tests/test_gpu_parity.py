"""GPU parity of the FP16/BF16 fused forward against the FP64 oracle.

Element-by-element on every row for shapes the oracle finishes in seconds
(several tiles, ragged tails, causal with Nq != Nk, grouped heads) and for
the B=4, H=16, N=4096 workloads; on sampled rows for the long causal GQA
workloads, in the launch configuration the bench times.
"""
import math

import numpy as np
import pytest
import torch

import synth
from parity import assert_within, errors, gather_rows, oracle_for

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


def _run(gpu_lib, B, Nq, Nk, Hq, Hkv, d, causal, dtype, seed=0, rows=None, device="cpu"):
    q, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=DT[dtype], seed=seed, device=device)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = gpu_lib.attn_fwd(q, k, v, causal=causal, scale=scale)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, causal, scale, rows)
    if rows is not None:
        o, lse = gather_rows(o, lse, rows)
    return errors(o, lse, o_ref, lse_ref)


def test_tiny_fp16_noncausal(gpu_lib):
    """B=1, H=2, Nq=Nk=128, d=64, FP16: the smallest workload, every row."""
    assert_within(_run(gpu_lib, 1, 128, 128, 2, 2, 64, False, "f16"))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_ragged_multi_tile_gqa(gpu_lib, d, causal, dtype):
    """Several 128-row tiles with a ragged tail, two query heads per key head."""
    assert_within(_run(gpu_lib, 2, 777, 777, 4, 2, d, causal, dtype, seed=1))


@pytest.mark.parametrize("Nq,Nk", [(300, 1000), (1000, 300), (129, 127), (1, 1), (1, 700),
                                   (640, 640), (255, 257)])
@pytest.mark.parametrize("causal", [False, True])
def test_unequal_lengths_and_edges(gpu_lib, Nq, Nk, causal):
    assert_within(_run(gpu_lib, 1, Nq, Nk, 8, 1, 128, causal, "bf16", seed=2))


@pytest.mark.parametrize("Nq,Hq,Hkv,d", [(16, 64, 8, 128), (32, 16, 2, 128), (5, 32, 4, 64),
                                          (12, 16, 2, 256), (3, 48, 16, 128)])
def test_few_queries_gqa_packed(gpu_lib, Nq, Hq, Hkv, d):
    """Non-causal, few query rows per head: when a GQA group divides 128 and
    its rows fit the unit's query tiles, the heads of the group share tile
    rows (one K/V stream per group); a group of 3 takes the plain kernel."""
    assert_within(_run(gpu_lib, 2, Nq, 1500, Hq, Hkv, d, False, "bf16", seed=6))


def test_many_heads_small_sequence(gpu_lib):
    """More work units than SMs with tiny sequences (every CTA loops)."""
    assert_within(_run(gpu_lib, 3, 200, 200, 64, 8, 64, True, "bf16", seed=3))


def test_repeated_calls_are_deterministic(gpu_lib):
    q, k, v = synth.attn_inputs(2, 513, 513, 4, 4, 128, dtype=torch.bfloat16, seed=4,
                                device="cuda")
    o1, l1 = gpu_lib.attn_fwd(q, k, v, causal=True)
    o2, l2 = gpu_lib.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_query_is_noop(gpu_lib):
    q = torch.empty(2, 0, 4, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(2, 10, 4, 128, device="cuda").to(torch.bfloat16)
    o, lse = gpu_lib.attn_fwd(q, k, k)
    assert o.shape == (2, 0, 4, 128) and lse.shape == (2, 4, 0)


def test_misaligned_view_is_rejected(gpu_lib):
    base = torch.zeros(1 * 64 * 2 * 128 + 32, dtype=torch.bfloat16, device="cuda")
    q = base[32:].view(1, 64, 2, 128)   # 64-byte offset
    k = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gpu_lib.AttnError) as ei:
        gpu_lib.attn_fwd(q, k, k)
    assert ei.value.code == -3


# ---------------------------------------------------------------- full sizes
@pytest.mark.parametrize("d", [64, 128, 256])
def test_full_bf16_mha_4096_every_row(gpu_lib, d):
    """B=4, H=16, Nq=Nk=4096, BF16, non-causal (the bench workload at d=128,
    in the bench's launch configuration): all 262,144 rows against the FP64
    oracle."""
    assert_within(_run(gpu_lib, 4, 4096, 4096, 16, 16, d, False, "bf16", device="cuda"))


def test_full_causal_gqa_32k_sampled(gpu_lib):
    """B=1, Hq=64, Hkv=8, N=32768, causal BF16 (Llama-3-70B-shaped layer):
    256 sampled query rows per head."""
    rows = synth.sample_rows(1, 64, 32768, per_head=256, seed=0)
    assert_within(_run(gpu_lib, 1, 32768, 32768, 64, 8, 128, True, "bf16", rows=rows,
                       device="cuda"))


def test_full_causal_gqa_128k_sampled(gpu_lib):
    """B=1, Hq=64, Hkv=8, N=131072, causal BF16 (long-context prefill):
    64 sampled query rows per head."""
    rows = synth.sample_rows(1, 64, 131072, per_head=64, seed=0)
    assert_within(_run(gpu_lib, 1, 131072, 131072, 64, 8, 128, True, "bf16", rows=rows,
                       device="cuda"))
