"""Failure path of the kernels' bounded waits, on the GPU without a fault: a
wait that nothing completes runs out, the status word reports it, and the
context stays usable for the next call."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import errors

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_stays_usable(gpu_lib):
    assert gpu_lib.get_status() == gpu_lib.OK
    gpu_lib.selftest_bounded_wait()
    assert gpu_lib.get_status() == gpu_lib.ERR_TIMEOUT
    assert gpu_lib.get_status() == gpu_lib.OK   # read and cleared
    # the next forward runs normally and matches the oracle
    B, N, H, d = 1, 300, 2, 64
    q, k, v = synth.attn_inputs(B, N, N, H, H, d, dtype=torch.bfloat16, seed=5, device="cuda")
    o, lse = gpu_lib.attn_fwd(q, k, v)
    assert gpu_lib.get_status() == gpu_lib.OK
    o_ref, lse_ref = oracle.attention_full(*(synth.raw_bits(t) for t in (q, k, v)),
                                           causal=False, scale=1 / math.sqrt(d),
                                           elem=oracle.ELEM_BF16)
    e = errors(o, lse, o_ref, lse_ref)
    assert e["o_max_abs"] <= 1e-2 and e["lse_max_abs"] <= 1e-3, e
