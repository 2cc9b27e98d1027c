"""attn_fwd_splitkv_noalloc: the split-key-range forward for callers that
cannot allocate device memory (code running under CUDA graph capture, programs
that hand all device memory to their own pool, allocation-free request paths).

It keeps its partial results in a fixed array inside the library instead of a
caller or library allocation.  These tests call it through the C ABI and check
its output against attn_fwd_splitkv, within the tolerances of the other parity
tests, on two calls in a row with different inputs (so that anything left in
the shared array by the first call would show up in the second), and check
that a problem too large for the array is refused.

This file is named to be collected last.
"""
import ctypes
import math

import pytest
import torch

import synth
from parity import LSE_ABS, O_MAX_ABS, O_RMS

pytestmark = pytest.mark.gpu


def _call(lib, q, k, v, o, lse, splits, d):
    B, Nq, Hq, _ = q.shape
    _, Nk, Hkv, _ = k.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, splits,
                                        1.0 / math.sqrt(d), 1, stream)


def test_noalloc_matches_splitkv_on_two_calls(gpu_lib):
    lib = gpu_lib.load()
    B, Nq, Nk, Hq, Hkv, d, splits = 2, 3, 20000, 16, 4, 128, 12
    for call in range(2):
        q, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=torch.bfloat16, seed=40 + call,
                                    device="cuda")
        o_ref, lse_ref = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=splits)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call(lib, q, k, v, o, lse, splits, d) == 0
        torch.cuda.synchronize()
        if call == 1:
            # the first call may load the library's device image; after that
            # a call takes no device memory at all
            assert torch.cuda.mem_get_info()[0] == free_before
        diff = (o.float() - o_ref.float())
        assert diff.abs().max().item() <= O_MAX_ABS
        assert diff.pow(2).mean().sqrt().item() <= O_RMS
        assert (lse - lse_ref).abs().max().item() <= LSE_ABS
        assert torch.isfinite(o.float()).all()


def test_noalloc_refuses_problems_larger_than_its_array(gpu_lib):
    lib = gpu_lib.load()
    # 256 splits x 64 heads x 128 rows x 129 floats is far over 16 MiB
    B, Nq, Nk, Hq, Hkv, d = 1, 128, 40000, 64, 8, 128
    q = torch.zeros(B, Nq, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, Nk, Hkv, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device="cuda")
    assert _call(lib, q, k, k, o, lse, 256, d) == gpu_lib.ERR_SCRATCH
