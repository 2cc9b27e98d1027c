"""Python binding of the C-ABI attention library (``include/attn.h``).

Argument marshalling only: shape/dtype/device checks, output allocation with
torch (device memory is plumbing), and one ctypes call per entry point on the
current torch stream.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback of any kind.  If the shared library is
missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libattn.so")

ATTN_F16, ATTN_BF16 = 0, 1
OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED = -1, -2, -3
ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = -4, -5, -6
ERR_SCRATCH = -7

EXPORTS = ("attn_fwd", "attn_prep_fp8", "attn_fwd_fp8", "attn_get_status", "attn_strerror",
           "attn_launch_count", "attn_fwd_splitkv", "attn_splitkv_workspace_bytes",
           "attn_splitkv_default_splits", "attn_fwd_splitkv_noalloc", "attn_prep_fp8_per_tensor",
           "attn_rope_table", "attn_prep_fp8_rope", "attn_selftest_bounded_wait",
           "attn_prep_fp8_qkv")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: error {code}: {strerror(code)}")


def load():
    """Load ``lib/libattn.so`` (built by ``build.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.attn_fwd.restype = i32
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i64, i32, i32, f32, i32, vp]
    lib.attn_prep_fp8.restype = i32
    lib.attn_prep_fp8.argtypes = [vp, vp, vp, i32, i32, i64, i32, vp, i32, i32, vp]
    lib.attn_fwd_fp8.restype = i32
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i64, i32, i32,
                                 f32, i32, vp]
    lib.attn_get_status.restype = i32
    lib.attn_get_status.argtypes = [vp]
    lib.attn_selftest_bounded_wait.restype = i32
    lib.attn_selftest_bounded_wait.argtypes = [vp]
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_strerror.argtypes = [i32]
    lib.attn_launch_count.restype = i64
    lib.attn_launch_count.argtypes = []
    lib.attn_fwd_splitkv.restype = i32
    lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i64, i32, i32, f32,
                                     i32, vp, ctypes.c_size_t, vp]
    lib.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_splitkv_workspace_bytes.argtypes = [i32, i32, i64, i32, i32]
    lib.attn_fwd_splitkv_noalloc.restype = i32
    lib.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i64, i32, i32,
                                             f32, i32, vp]
    lib.attn_splitkv_default_splits.restype = i32
    lib.attn_splitkv_default_splits.argtypes = [i32, i32, i32, i64, i64, i32]
    lib.attn_prep_fp8_per_tensor.restype = i32
    lib.attn_prep_fp8_per_tensor.argtypes = [vp, vp, vp, i32, i32, i64, i32, vp, i32, i32, vp]
    lib.attn_rope_table.restype = i32
    lib.attn_rope_table.argtypes = [vp, vp, i64, i32, ctypes.c_double, i64, vp]
    lib.attn_prep_fp8_qkv.restype = i32
    lib.attn_prep_fp8_qkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i64,
                                      i32, vp, vp, vp, vp]
    lib.attn_prep_fp8_rope.restype = i32
    lib.attn_prep_fp8_rope.argtypes = [vp, vp, vp, i32, i32, i64, i32, vp, vp, vp, i32, vp]
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().attn_strerror(int(code)).decode()


def launch_count() -> int:
    return int(load().attn_launch_count())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _check(rc: int, where: str):
    if rc != OK:
        raise AttnError(rc, where)


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (BSHD)")


def _check_outputs(q, out, lse):
    """Caller-provided outputs must match what the kernels write."""
    B, Nq, Hq, _ = q.shape
    _need_cuda(out, lse)
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must have the shape and dtype of q")
    if tuple(lse.shape) != (B, Hq, Nq) or lse.dtype != torch.float32:
        raise ValueError("lse must be float32 [B, Hq, Nq]")


def fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, Nq, Nk, d, causal, scale, dtype,
            stream) -> int:
    """Direct C call with raw integers (used by the boundary tests)."""
    return load().attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, Nq, Nk, d, causal,
                           scale, dtype, stream)


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             stream=None):
    """O, LSE = attention(q, k, v).  q: [B, Nq, Hq, d]; k, v: [B, Nk, Hkv, d]
    (fp16 or bf16, contiguous, CUDA).  Returns (O [B, Nq, Hq, d], LSE [B, Hq, Nq] fp32)."""
    _need_cuda(q, k, v)
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be float16 or all bfloat16")
    B, Nq, Hq, d = q.shape
    Bk, Nk, Hkv, dk = k.shape
    if v.shape != k.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch between q, k, v")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _check_outputs(q, out, lse)
    dt = ATTN_BF16 if q.dtype == torch.bfloat16 else ATTN_F16
    rc = load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                         int(bool(causal)), float(scale), dt, _stream(stream))
    _check(rc, "attn_fwd")
    return out, lse


def splitkv_workspace_bytes(B, Hq, Nq, d, num_splits) -> int:
    return int(load().attn_splitkv_workspace_bytes(B, Hq, Nq, d, num_splits))


def splitkv_default_splits(B, Hq, Hkv, Nq, Nk, d) -> int:
    return int(load().attn_splitkv_default_splits(B, Hq, Hkv, Nq, Nk, d))


def attn_fwd_splitkv(q, k, v, num_splits: int | None = None, scale: float | None = None,
                     out=None, lse=None, workspace=None, stream=None):
    """Non-causal attention with the key range split over several CTAs and an
    LSE merge (decode-like shapes).  Same arguments and results as attn_fwd
    with causal=False; `workspace` is a uint8 CUDA tensor of at least
    splitkv_workspace_bytes(...) bytes (allocated here if None)."""
    _need_cuda(q, k, v)
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be float16 or all bfloat16")
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    if num_splits is None:
        num_splits = splitkv_default_splits(B, Hq, Hkv, Nq, Nk, d)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _check_outputs(q, out, lse)
    if workspace is None and num_splits > 1:
        nbytes = splitkv_workspace_bytes(B, Hq, Nq, d, num_splits)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dt = ATTN_BF16 if q.dtype == torch.bfloat16 else ATTN_F16
    rc = load().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Nq,
                                 Nk, d, int(num_splits), float(scale), dt, _ptr(workspace),
                                 ws_bytes, _stream(stream))
    _check(rc, "attn_fwd_splitkv")
    return out, lse


def _prep_buffers(x, signs, sign_heads, transpose_out, out, descale):
    _need_cuda(x)
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    B, N, H, d = x.shape
    nb = (N + 127) // 128
    if transpose_out:
        npad = (N + 15) // 16 * 16
        shape = (B, H, d, npad)
    else:
        shape = (B, N, H, d)
    if out is None:
        out = torch.empty(shape, dtype=torch.uint8, device=x.device)
    if descale is None:
        descale = torch.empty((B, H, nb), dtype=torch.float32, device=x.device)
    if signs is not None:
        _need_cuda(signs)
        if signs.dtype != torch.int8 or signs.shape[1] != d:
            raise ValueError("signs must be int8 [G, d]")
        sign_heads = signs.shape[0] if sign_heads is None else sign_heads
    return out, descale, int(sign_heads or 0)


def attn_prep_fp8(x, signs=None, sign_heads: int | None = None, transpose_out: bool = False,
                  out=None, descale=None, stream=None):
    """Per-128-token-block E4M3 quantisation of x [B, N, H, d] (bf16), with the
    optional Hadamard transform (signs [G, d] int8 +-1 on the device).
    Returns (codes uint8, descale fp32 [B, H, ceil(N/128)]); codes are
    [B, N, H, d], or [B, H, d, Npad] (Npad = N rounded up to 16) when
    ``transpose_out``."""
    out, descale, sh = _prep_buffers(x, signs, sign_heads, transpose_out, out, descale)
    B, N, H, d = x.shape
    rc = load().attn_prep_fp8(_ptr(x), _ptr(out), _ptr(descale), B, H, N, d, _ptr(signs), sh,
                              int(bool(transpose_out)), _stream(stream))
    _check(rc, "attn_prep_fp8")
    return out, descale


def attn_prep_fp8_qkv(q, k, v, signs=None, rope=None, out=None, stream=None):
    """The FP8 preparation of one attention call in one launch: Q and K per
    block (with the transform when ``signs`` [Hkv, d] is given, rotated first
    when ``rope`` = (cos, sin) from attn_rope_table covering max(Nq, Nk)
    positions), V transposed.  Returns (q8, qd, k8, kd, v8t, vd), the same as
    the separate attn_prep_fp8 / attn_prep_fp8_rope calls.  ``out`` may hold
    those six tensors to be written in place."""
    _need_cuda(q, k, v)
    if q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must be bfloat16")
    B, Nq, Hq, d = q.shape
    _, Nk, Hkv, _ = k.shape
    if v.shape != k.shape:
        raise ValueError("k and v must have the same shape")
    if out is None:
        dev = q.device
        npad = (Nk + 15) // 16 * 16
        out = (torch.empty(q.shape, dtype=torch.uint8, device=dev),
               torch.empty((B, Hq, (Nq + 127) // 128), dtype=torch.float32, device=dev),
               torch.empty(k.shape, dtype=torch.uint8, device=dev),
               torch.empty((B, Hkv, (Nk + 127) // 128), dtype=torch.float32, device=dev),
               torch.empty((B, Hkv, d, npad), dtype=torch.uint8, device=dev),
               torch.empty((B, Hkv, (Nk + 127) // 128), dtype=torch.float32, device=dev))
    q8, qd, k8, kd, v8, vd = out
    if signs is not None:
        _need_cuda(signs)
        if signs.dtype != torch.int8 or tuple(signs.shape) != (Hkv, d):
            raise ValueError("signs must be int8 [Hkv, d]")
    cos, sin = (None, None) if rope is None else rope
    rc = load().attn_prep_fp8_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(k8), _ptr(v8),
                                  _ptr(qd), _ptr(kd), _ptr(vd), B, Hq, Hkv, Nq, Nk, d,
                                  _ptr(signs), _ptr(cos), _ptr(sin), _stream(stream))
    _check(rc, "attn_prep_fp8_qkv")
    return q8, qd, k8, kd, v8, vd


def attn_prep_fp8_per_tensor(x, signs=None, sign_heads: int | None = None,
                             transpose_out: bool = False, out=None, descale=None, stream=None):
    """One E4M3 scale for the whole tensor (the baseline FP8 scheme); same
    arguments and outputs as attn_prep_fp8, every descale entry equal."""
    out, descale, sh = _prep_buffers(x, signs, sign_heads, transpose_out, out, descale)
    B, N, H, d = x.shape
    rc = load().attn_prep_fp8_per_tensor(_ptr(x), _ptr(out), _ptr(descale), B, H, N, d,
                                         _ptr(signs), sh, int(bool(transpose_out)),
                                         _stream(stream))
    _check(rc, "attn_prep_fp8_per_tensor")
    return out, descale


def attn_rope_table(N: int, d: int, base: float = 10000.0, pos0: int = 0, device="cuda",
                    stream=None):
    """cos, sin float32 [N, d/2] of the rotate-half rotary angles
    (pos0 + n) * base^(-2c/d), computed on the device."""
    cos = torch.empty((N, d // 2), dtype=torch.float32, device=device)
    sin = torch.empty((N, d // 2), dtype=torch.float32, device=device)
    _need_cuda(cos)
    rc = load().attn_rope_table(_ptr(cos), _ptr(sin), int(N), int(d), float(base), int(pos0),
                                _stream(stream))
    _check(rc, "attn_rope_table")
    return cos, sin


def attn_prep_fp8_rope(x, rope_cos, rope_sin, signs=None, sign_heads: int | None = None,
                       out=None, descale=None, stream=None):
    """Rotary embedding (tables from attn_rope_table, [N, d/2] float32), then
    the optional Hadamard transform, then per-block E4M3 quantisation of a Q
    or K tensor x [B, N, H, d] (bf16).  Returns (codes [B, N, H, d], descale)."""
    out, descale, sh = _prep_buffers(x, signs, sign_heads, False, out, descale)
    B, N, H, d = x.shape
    _need_cuda(rope_cos, rope_sin)
    if (rope_cos.dtype != torch.float32 or rope_sin.dtype != torch.float32
            or tuple(rope_cos.shape) != (N, d // 2) or tuple(rope_sin.shape) != (N, d // 2)
            or not rope_cos.is_contiguous() or not rope_sin.is_contiguous()):
        raise ValueError("rope tables must be contiguous float32 [N, d/2]")
    rc = load().attn_prep_fp8_rope(_ptr(x), _ptr(out), _ptr(descale), B, H, N, d,
                                   _ptr(rope_cos), _ptr(rope_sin), _ptr(signs), sh,
                                   _stream(stream))
    _check(rc, "attn_prep_fp8_rope")
    return out, descale


def attn_fwd_fp8(q8, k8, v8t, q_descale, k_descale, v_descale, *, Hq: int | None = None,
                 causal: bool = False, scale: float | None = None, hadamard: bool = False,
                 out=None, lse=None, stream=None):
    """FP8 forward.  q8 [B, Nq, Hq, d], k8 [B, Nk, Hkv, d] uint8 E4M3 codes,
    v8t [B, Hkv, d, Nkpad]; descales fp32 per 128-token block.
    Returns (O bf16 [B, Nq, Hq, d], LSE fp32 [B, Hq, Nq])."""
    _need_cuda(q8, k8, v8t, q_descale, k_descale, v_descale)
    B, Nq, Hq_, d = q8.shape
    _, Nk, Hkv, _ = k8.shape
    if out is None:
        out = torch.empty((B, Nq, Hq_, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, Hq_, Nq), dtype=torch.float32, device=q8.device)
    _need_cuda(out, lse)
    if tuple(out.shape) != (B, Nq, Hq_, d) or out.dtype != torch.bfloat16:
        raise ValueError("out must be bfloat16 [B, Nq, Hq, d]")
    if tuple(lse.shape) != (B, Hq_, Nq) or lse.dtype != torch.float32:
        raise ValueError("lse must be float32 [B, Hq, Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = load().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(q_descale), _ptr(k_descale),
                             _ptr(v_descale), _ptr(out), _ptr(lse), B, Hq_, Hkv, Nq, Nk, d,
                             int(bool(causal)), float(scale), int(bool(hadamard)), _stream(stream))
    _check(rc, "attn_fwd_fp8")
    return out, lse


def get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word as a code."""
    return int(load().attn_get_status(_stream(stream)))


def selftest_bounded_wait(stream=None):
    """Launch the library's bounded-wait self test (a wait that runs out after
    about 2 s and sets the timeout status); read the result with get_status."""
    _check(int(load().attn_selftest_bounded_wait(_stream(stream))), "attn_selftest_bounded_wait")
