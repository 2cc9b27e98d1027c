"""GPU parity of the split-key-range forward (decode-like shapes) against the
FP64 oracle, and its agreement with the unsplit kernel."""
import ctypes
import math

import pytest
import torch

import synth
from parity import assert_within, errors, oracle_for

pytestmark = pytest.mark.gpu


def _inputs(B, Nq, Nk, Hq, Hkv, d, seed, device="cpu"):
    q, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=torch.bfloat16, seed=seed,
                                device=device)
    return q.cuda(), k.cuda(), v.cuda()


@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (16, 5000), (128, 3000), (200, 2500)])
@pytest.mark.parametrize("splits", [1, 3, 64, None])
def test_splitkv_matches_oracle(gpu_lib, Nq, Nk, splits):
    B, Hq, Hkv, d = 2, 8, 2, 128
    q, k, v = _inputs(B, Nq, Nk, Hq, Hkv, d, seed=11)
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=splits)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, 1 / math.sqrt(d))
    assert_within(errors(o, lse, o_ref, lse_ref))


@pytest.mark.parametrize("d", [64, 256])
def test_splitkv_head_dims(gpu_lib, d):
    q, k, v = _inputs(1, 5, 4000, 4, 4, d, seed=12)
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=7)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, 1 / math.sqrt(d))
    assert_within(errors(o, lse, o_ref, lse_ref))


def test_splitkv_agrees_with_unsplit_kernel(gpu_lib):
    q, k, v = _inputs(1, 64, 8192, 16, 4, 128, seed=13)
    o1, l1 = gpu_lib.attn_fwd(q, k, v, causal=False)
    o2, l2 = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=16)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_splitkv_decode_128k_every_row(gpu_lib):
    """One query per head against 131072 keys (B=1, Hq=64, Hkv=8, d=128):
    the long-context decode shape, default split count, every row."""
    q, k, v = synth.attn_inputs(1, 1, 131072, 64, 8, 128, dtype=torch.bfloat16, seed=14,
                                device="cuda")
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, 1 / math.sqrt(128))
    assert_within(errors(o, lse, o_ref, lse_ref))


def test_splitkv_decode_1m_keys_every_row(gpu_lib):
    """One query per head against 1,048,576 keys (B=1, Hq=8, Hkv=1, d=128): a
    million-token context, default split count, every row against the oracle."""
    q, k, v = synth.attn_inputs(1, 1, 1 << 20, 8, 1, 128, dtype=torch.bfloat16, seed=17,
                                device="cuda")
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, 1 / math.sqrt(128))
    assert_within(errors(o, lse, o_ref, lse_ref))


def test_splitkv_rejects_small_workspace(gpu_lib):
    q, k, v = _inputs(1, 4, 4096, 2, 2, 128, seed=15)
    need = gpu_lib.splitkv_workspace_bytes(1, 2, 4, 128, 8)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(gpu_lib.AttnError) as ei:
        gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=8, workspace=ws)
    assert ei.value.code == -1
    lib = gpu_lib.load()
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 4, device="cuda")
    rc = lib.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), 1, 2, 2, 4, 4096, 128, 0, 0.1, 1, None, 0,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -1   # num_splits < 1


@pytest.mark.parametrize("Hq,Hkv", [(6, 1), (16, 1), (12, 4)])
def test_splitkv_group_packing_and_fallback(gpu_lib, Hq, Hkv):
    """Groups that divide 128 share query tiles (16/1); others (6/1, 12/4 with a
    group of 3) run one head per tile.  Both must match the oracle."""
    q, k, v = _inputs(2, 9, 3000, Hq, Hkv, 128, seed=16)
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=5)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, 1 / math.sqrt(128))
    assert_within(errors(o, lse, o_ref, lse_ref))


@pytest.mark.parametrize("Hq,Hkv,Nq", [(16, 2, 1), (16, 2, 16), (64, 8, 2), (8, 8, 3), (12, 4, 5)])
def test_splitkv_single_split_packed(gpu_lib, Hq, Hkv, Nq):
    """With one split, GQA groups that divide 128 still share query tiles when
    the packed rows fit (the kernel then writes O and LSE itself, without a
    workspace); other shapes take the plain kernel."""
    q, k, v = _inputs(3, Nq, 2000, Hq, Hkv, 128, seed=18)
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=1)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, 1 / math.sqrt(128))
    assert_within(errors(o, lse, o_ref, lse_ref))


def test_splitkv_batched_decode_every_row(gpu_lib):
    """A batch of 32 sequences, one query per head each, 8192 cached keys
    (B=32, Hq=64, Hkv=8, d=128), default split count, every row."""
    q, k, v = synth.attn_inputs(32, 1, 8192, 64, 8, 128, dtype=torch.bfloat16, seed=19,
                                device="cuda")
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, 1 / math.sqrt(128))
    assert_within(errors(o, lse, o_ref, lse_ref))
