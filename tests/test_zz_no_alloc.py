"""attn_fwd_splitkv_noalloc: the split-key-range forward for callers that
cannot allocate device memory (programs whose device memory belongs to their
own pool or arena, and services that forbid allocation on the request path,
where an allocation could block, synchronise the device or fail).

It keeps its partial results and its status word in a fixed array inside the
library instead of a caller workspace or a library allocation.  These tests
call it through the C ABI and compare every output row with the FP64 oracle,
within the tolerances of the other parity tests, on two calls in a row with
different inputs (anything the first call left in the shared array would
show up in the second), for each head dimension, with several splits and
with one; they check that attn_get_status (which reads the array's status
word) reports no problem afterwards, that the second call takes no device
memory, and that a problem too large for the array is refused.

This file is named to be collected last.
"""
import ctypes
import math

import pytest
import torch

import synth
from parity import assert_within, errors, oracle_for

pytestmark = pytest.mark.gpu

DT = {"bf16": (torch.bfloat16, 1), "f16": (torch.float16, 0)}


def _call(lib, q, k, v, o, lse, splits, d, dtype_code):
    B, Nq, Hq, _ = q.shape
    _, Nk, Hkv, _ = k.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, splits,
                                        1.0 / math.sqrt(d), dtype_code, stream)


@pytest.mark.parametrize("d,splits,dtype", [(64, 12, "bf16"), (128, 12, "bf16"),
                                            (256, 12, "f16"), (128, 1, "bf16")])
def test_noalloc_matches_oracle_on_two_calls(gpu_lib, d, splits, dtype):
    lib = gpu_lib.load()
    tdt, code = DT[dtype]
    B, Nq, Nk, Hq, Hkv = 2, 3, 20000, 16, 4
    for call in range(2):
        q, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=tdt, seed=40 + call,
                                    device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call(lib, q, k, v, o, lse, splits, d, code) == 0
        torch.cuda.synchronize()
        if call == 1:
            # the first call may load the library's device image; after that
            # a call takes no device memory at all
            assert torch.cuda.mem_get_info()[0] == free_before
        assert gpu_lib.get_status() == 0
        o_ref, lse_ref = oracle_for(q, k, v, False, 1.0 / math.sqrt(d))
        assert_within(errors(o, lse, o_ref, lse_ref))


def test_noalloc_refuses_problems_larger_than_its_array(gpu_lib):
    lib = gpu_lib.load()
    # 256 splits x 64 heads x 128 rows x 129 floats is far over 16 MiB
    B, Nq, Nk, Hq, Hkv, d = 1, 128, 40000, 64, 8, 128
    q = torch.zeros(B, Nq, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, Nk, Hkv, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device="cuda")
    assert _call(lib, q, k, k, o, lse, 256, d, 1) == gpu_lib.ERR_SCRATCH
