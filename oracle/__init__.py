"""FP64 CPU oracle for the tiled attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / reference leg of ``bench.py`` may import this package.
The product path (the CUDA library and its Python binding) never imports it,
and it imports nothing from the product package.

Contents
--------
``attention_rows``   plain two-pass FP64 attention for selected query rows
                     (C, ``attn_oracle.c``).
``attention_full``   the same for every query row.
``merge_partials``   the pages' streaming-softmax merge rule, used by the
                     pins to tie the oracle to the algorithm the GPU runs.
``fp8``              E4M3 codec, Sylvester Hadamard matrix and per-block FP8
                     quantisation (numpy), see ``oracle/fp8.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import fp8  # noqa: F401  (re-exported sub-module)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_DIR = os.path.join(_HERE, "lib")
_LIB_PATH = os.path.join(_LIB_DIR, "liboracle.so")
_SRC = os.path.join(_HERE, "attn_oracle.c")

ELEM_F16, ELEM_BF16, ELEM_F32, ELEM_F64 = 0, 1, 2, 3

_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``oracle/lib/liboracle.so`` with gcc."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread",
                    "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        ll = ctypes.c_longlong
        vp = ctypes.c_void_p
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [vp, vp, vp, ctypes.c_int, ll, ll, ll, ll, ll,
                                              ctypes.c_int, ctypes.c_double, vp, vp, vp, ll,
                                              vp, vp, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [vp, ctypes.c_int, ll, vp]
        _lib = lib
    return _lib


def _elem_of(a: np.ndarray, elem: int | None) -> int:
    if elem is not None:
        return elem
    if a.dtype == np.float64:
        return ELEM_F64
    if a.dtype == np.float32:
        return ELEM_F32
    raise TypeError("16-bit inputs must be passed as uint16 bit patterns with an explicit elem")


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def decode(raw: np.ndarray, elem: int) -> np.ndarray:
    """Decode raw 16/32/64-bit elements to float64 with the oracle's decoders."""
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.size, dtype=np.float64)
    rc = _load().oracle_decode(raw.ctypes.data, elem, raw.size, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_decode failed ({rc})")
    return out.reshape(raw.shape)


def attention_rows(q_rows, k, v, *, Hq: int, causal: bool, scale: float, rows,
                   elem: int | None = None, nthreads: int | None = None):
    """FP64 attention for selected query rows.

    q_rows : [R, d] (the query vectors of the selected rows)
    k, v   : [B, Nk, Hkv, d]  (BSHD, d innermost)
    rows   : [R, 3] integer array of (b, h, i): batch, query head, query index
    elem   : element code of the raw arrays (uint16 inputs need ELEM_F16/ELEM_BF16)
    Returns (O [R, d] float64, LSE [R] float64, natural log).
    """
    q_rows = np.ascontiguousarray(q_rows)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    el = _elem_of(k, elem)
    if not (q_rows.dtype == k.dtype == v.dtype):
        raise TypeError("q_rows, k, v must share one raw dtype")
    B, Nk, Hkv, d = k.shape
    if v.shape != k.shape or q_rows.shape != (rows.shape[0], d):
        raise ValueError("shape mismatch")
    R = rows.shape[0]
    rb = np.ascontiguousarray(rows[:, 0])
    rh = np.ascontiguousarray(rows[:, 1])
    ri = np.ascontiguousarray(rows[:, 2])
    o = np.zeros((R, d), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    nt = nthreads or default_threads()
    rc = _load().oracle_attention_rows(q_rows.ctypes.data, k.ctypes.data, v.ctypes.data, el, B, Hq,
                                       Hkv, Nk, d, int(bool(causal)), float(scale),
                                       rb.ctypes.data, rh.ctypes.data, ri.ctypes.data, R,
                                       o.ctypes.data, lse.ctypes.data, nt)
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed ({rc})")
    return o, lse


def all_rows(B: int, H: int, N: int) -> np.ndarray:
    """Every (b, h, i) in BSHD order of the query tensor rows."""
    b, i, h = np.meshgrid(np.arange(B), np.arange(N), np.arange(H), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1).astype(np.int64)


def attention_full(q, k, v, *, causal: bool, scale: float, elem: int | None = None,
                   nthreads: int | None = None):
    """FP64 attention for every query row.

    q : [B, Nq, Hq, d];  k, v : [B, Nk, Hkv, d].
    Returns O [B, Nq, Hq, d] float64 and LSE [B, Hq, Nq] float64.
    """
    B, Nq, Hq, d = q.shape
    rows = all_rows(B, Hq, Nq)
    q_rows = np.ascontiguousarray(q).reshape(B * Nq * Hq, d)
    o, lse = attention_rows(q_rows, k, v, Hq=Hq, causal=causal, scale=scale, rows=rows,
                            elem=elem, nthreads=nthreads)
    o = o.reshape(B, Nq, Hq, d)
    lse = lse.reshape(B, Nq, Hq).transpose(0, 2, 1).copy()
    return o, lse


def merge_partials(o_a, lse_a, o_b, lse_b):
    """Combine two partial softmax results over disjoint key sets.

    The pages' merge rule ("FlashAttention（V3）深度解析", section 4.2):
    m = max(m_a, m_b), z = z_a e^(m_a - m) + z_b e^(m_b - m).  A partial result
    (O_x, LSE_x) is the pair m_x = LSE_x, z_x = 1, so the merged output is the
    z-weighted mean of the two normalised outputs and LSE = m + ln z.
    """
    m = np.maximum(lse_a, lse_b)
    wa = np.exp(lse_a - m)
    wb = np.exp(lse_b - m)
    z = wa + wb
    o = (wa[..., None] * o_a + wb[..., None] * o_b) / z[..., None]
    return o, m + np.log(z)
