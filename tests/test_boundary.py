"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any CUDA call."""
import math
import os
import re

import pytest

from tiled_attention_forward_02_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert set(_declared_functions()) == set(attn.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


A = 0x10000000  # a 128-byte aligned fake device address (never dereferenced)


def _fwd(**kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, B=1, Hq=2, Hkv=1, Nq=10, Nk=10, d=128, causal=0,
                scale=0.1, dtype=attn.ATTN_BF16, stream=0)
    args.update(kw)
    return attn.fwd_raw(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                        args["Hq"], args["Hkv"], args["Nq"], args["Nk"], args["d"], args["causal"],
                        args["scale"], args["dtype"], args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=3, Hkv=2), attn.ERR_INVALID_ARG),          # Hq % Hkv != 0
    (dict(Hkv=0), attn.ERR_INVALID_ARG),
    (dict(B=-1), attn.ERR_INVALID_ARG),
    (dict(Nq=-5), attn.ERR_INVALID_ARG),
    (dict(Nk=0), attn.ERR_INVALID_ARG),                 # keys required when Nq > 0
    (dict(causal=2), attn.ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ERR_INVALID_ARG),
    (dict(scale=-1.0), attn.ERR_INVALID_ARG),
    (dict(scale=math.nan), attn.ERR_INVALID_ARG),
    (dict(scale=math.inf), attn.ERR_INVALID_ARG),
    (dict(Nq=1 << 31), attn.ERR_INVALID_ARG),
    (dict(q=0), attn.ERR_INVALID_ARG),
    (dict(lse=0), attn.ERR_INVALID_ARG),
    (dict(d=96), attn.ERR_UNSUPPORTED),
    (dict(d=32), attn.ERR_UNSUPPORTED),
    (dict(dtype=7), attn.ERR_UNSUPPORTED),
    (dict(q=A + 64), attn.ERR_MISALIGNED),              # TMA base must be 128-byte aligned
    (dict(o=A + 16), attn.ERR_MISALIGNED),
    (dict(lse=A + 4), attn.ERR_MISALIGNED),
])
def test_fwd_rejects_bad_arguments_on_host(lib, kw, code):
    assert _fwd(**kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(Nq=0), dict(Nq=0, Nk=0, q=0, k=0, v=0, o=0, lse=0)])
def test_fwd_empty_problem_is_a_noop(lib, kw):
    assert _fwd(**kw) == attn.OK


def test_fp8_and_prep_reject_bad_arguments_on_host(lib):
    L = lib
    # prep: unsupported d, bad transpose flag, sign heads not dividing H, misaligned
    assert L.attn_prep_fp8(A, A, A, 1, 4, 100, 96, None, 0, 0, None) == attn.ERR_UNSUPPORTED
    assert L.attn_prep_fp8(A, A, A, 1, 4, 100, 128, None, 0, 3, None) == attn.ERR_INVALID_ARG
    assert L.attn_prep_fp8(A, A, A, 1, 4, 100, 128, A, 3, 0, None) == attn.ERR_INVALID_ARG
    assert L.attn_prep_fp8(A + 8, A, A, 1, 4, 100, 128, None, 0, 0, None) == attn.ERR_MISALIGNED
    assert L.attn_prep_fp8(A, A, A, 0, 4, 100, 128, None, 0, 0, None) == attn.OK
    # fp8 forward: d = 96 not covered, bad hadamard flag, null descale
    args = [A, A, A, A, A, A, A, A, 1, 2, 2, 10, 10, 128, 0, 0.1, 0, None]
    bad = list(args); bad[13] = 96
    assert L.attn_fwd_fp8(*bad) == attn.ERR_UNSUPPORTED
    bad = list(args); bad[16] = 2
    assert L.attn_fwd_fp8(*bad) == attn.ERR_INVALID_ARG
    bad = list(args); bad[3] = None
    assert L.attn_fwd_fp8(*bad) == attn.ERR_INVALID_ARG
    bad = list(args); bad[4] = A + 4
    assert L.attn_fwd_fp8(*bad) == attn.ERR_MISALIGNED


def test_prep_variants_reject_bad_arguments_on_host(lib):
    L = lib
    # per-tensor: same checks as the per-block prep
    assert L.attn_prep_fp8_per_tensor(A, A, A, 1, 4, 100, 96, None, 0, 0, None) == attn.ERR_UNSUPPORTED
    assert L.attn_prep_fp8_per_tensor(A, A, A, 1, 4, 100, 128, A, 3, 0, None) == attn.ERR_INVALID_ARG
    assert L.attn_prep_fp8_per_tensor(A, A + 8, A, 1, 4, 100, 128, None, 0, 0, None) == attn.ERR_MISALIGNED
    assert L.attn_prep_fp8_per_tensor(A, A, A, 1, 4, 0, 128, None, 0, 0, None) == attn.OK
    # rotary prep: tables required and 16-byte aligned
    assert L.attn_prep_fp8_rope(A, A, A, 1, 4, 100, 128, None, A, None, 0, None) == attn.ERR_INVALID_ARG
    assert L.attn_prep_fp8_rope(A, A, A, 1, 4, 100, 128, A + 4, A, None, 0, None) == attn.ERR_MISALIGNED
    assert L.attn_prep_fp8_rope(A, A, A, 1, 4, 100, 100, A, A, None, 0, None) == attn.ERR_UNSUPPORTED
    assert L.attn_prep_fp8_rope(A, A, A, 0, 4, 100, 128, None, None, None, 0, None) == attn.OK
    # tables: odd or too large d, base <= 1, negative offset, empty
    assert L.attn_rope_table(A, A, 10, 7, 10000.0, 0, None) == attn.ERR_INVALID_ARG
    assert L.attn_rope_table(A, A, 10, 512, 10000.0, 0, None) == attn.ERR_INVALID_ARG
    assert L.attn_rope_table(A, A, 10, 128, 1.0, 0, None) == attn.ERR_INVALID_ARG
    assert L.attn_rope_table(A, A, 10, 128, 10000.0, -1, None) == attn.ERR_INVALID_ARG
    assert L.attn_rope_table(A, A, 0, 128, 10000.0, 0, None) == attn.OK


def test_strerror_covers_every_code(lib):
    for c in (attn.OK, attn.ERR_INVALID_ARG, attn.ERR_UNSUPPORTED, attn.ERR_MISALIGNED,
              attn.ERR_CUDA, attn.ERR_TIMEOUT, attn.ERR_DEVICE):
        assert attn.strerror(c)
    assert "unknown" in attn.strerror(12345)


def test_valid_call_without_device_reports_cuda_error(lib):
    """Valid arguments reach the CUDA runtime; with no GPU visible the call
    must come back with ATTN_ERR_CUDA (no crash, no CPU fallback)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    assert _fwd() == attn.ERR_CUDA
    assert "cuda" in attn.strerror(attn.ERR_CUDA).lower()


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)


def test_splitkv_workspace_size_and_host_checks(lib):
    # splits x B x Hq x Nq rows of d floats (padded to 256 bytes), then one float per row
    assert lib.attn_splitkv_workspace_bytes(1, 2, 4, 128, 8) == 64 * 128 * 4 + 64 * 4
    assert lib.attn_splitkv_workspace_bytes(1, 2, 3, 64, 1) == 1536 + 24
    assert lib.attn_splitkv_workspace_bytes(1, 2, 4, 128, 0) == 0
    args = [A, A, A, A, A, 1, 2, 2, 4, 4096, 128, 4, 0.1, 1, A, 1 << 20, None]
    bad = list(args); bad[11] = 0
    assert lib.attn_fwd_splitkv(*bad) == attn.ERR_INVALID_ARG        # no split
    bad = list(args); bad[10] = 96
    assert lib.attn_fwd_splitkv(*bad) == attn.ERR_UNSUPPORTED
    bad = list(args); bad[14] = None
    assert lib.attn_fwd_splitkv(*bad) == attn.ERR_INVALID_ARG        # workspace missing
    bad = list(args); bad[15] = 1024
    assert lib.attn_fwd_splitkv(*bad) == attn.ERR_INVALID_ARG        # workspace too small
    bad = list(args); bad[14] = A + 64
    assert lib.attn_fwd_splitkv(*bad) == attn.ERR_MISALIGNED
