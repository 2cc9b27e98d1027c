"""The method's degenerate and edge cases through the CUDA path, element by
element against the FP64 oracle and against their closed forms.

* Q = 0: every allowed logit is 0, so O is the mean of the allowed V rows and
  LSE = ln |J| (causal: the prefix mean of V[0..i]), for Nq != Nk in both
  directions.
* Lazy rescale: the kernels move a row's softmax reference, and rescale O and
  l in tensor memory, only when the running maximum grows by more than 2^8
  (16-bit inputs).  Inputs whose logits rise by about 12 log2 units from
  each 128-key tile to the next make that branch run on every tile of every
  row (counted here, from the same values, before the comparison), in the
  two-tile, one-tile (d = 256) and split-key-range instances.  The branch
  applies the merge rule of "FlashAttention（V3）深度解析" section 4.2
  (m = max(m_a, m_b), z = z_a e^(m_a - m) + z_b e^(m_b - m)).
* One dominant key planted in the last key tile of rows that span eight or
  more tiles, with a logit gap of at least 60 over every other key: O equals
  that key's V row and LSE its logit (the reference moves by the gap at the
  last tile).
"""
import math

import numpy as np
import pytest
import torch

import synth
from parity import assert_within, errors, oracle_for

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}
LOG2E = 1.4426950408889634
TAU = 8.0   # the 16-bit kernels' rescale threshold, log2 units


def _allowed(i, Nk, causal):
    return min(i + 1, Nk) if causal else Nk


# ----------------------------------------------------------------- Q = 0
@pytest.mark.parametrize("Nq,Nk", [(300, 1000), (1000, 300)])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_zero_query_gives_mean_of_allowed_values(gpu_lib, Nq, Nk, d, causal, dtype):
    B, Hq, Hkv = 1, 4, 2
    _, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=DT[dtype], seed=8)
    q = torch.zeros(B, Nq, Hq, d, dtype=DT[dtype])
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = gpu_lib.attn_fwd(q, k, v, causal=causal, scale=scale)
    assert gpu_lib.get_status() == 0
    # closed form from the V values alone
    vv = v.double().cpu().numpy()                                   # [B, Nk, Hkv, d]
    csum = np.cumsum(vv, axis=1)
    n = np.array([_allowed(i, Nk, causal) for i in range(Nq)])      # |J| per row
    mean = csum[:, n - 1] / n[None, :, None, None]                   # [B, Nq, Hkv, d]
    o_cf = np.repeat(mean, Hq // Hkv, axis=2)                        # query head h -> h / group
    lse_cf = np.broadcast_to(np.log(n)[None, None, :], (B, Hq, Nq))
    assert_within(errors(o, lse, o_cf, lse_cf))
    o_ref, lse_ref = oracle_for(q, k, v, causal, scale)
    assert_within(errors(o, lse, o_ref, lse_ref))


def test_zero_query_split_key_range(gpu_lib):
    """The same closed form through the split-key-range path (GQA group packed
    into tile rows, several splits merged)."""
    B, Nq, Nk, Hq, Hkv, d = 2, 3, 5000, 16, 4, 128
    _, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=torch.bfloat16, seed=9)
    q = torch.zeros(B, Nq, Hq, d, dtype=torch.bfloat16)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=7)
    assert gpu_lib.get_status() == 0
    mean = v.double().cpu().numpy().mean(axis=1)                    # [B, Hkv, d]
    o_cf = np.repeat(mean, Hq // Hkv, axis=1)[:, None].repeat(Nq, axis=1)
    lse_cf = np.full((B, Hq, Nq), math.log(Nk))
    assert_within(errors(o, lse, o_cf, lse_cf))


# ------------------------------------------------------------ lazy rescale
def _ramp_inputs(B, Nq, Nk, Hq, Hkv, d, dtype, seed, step_log2=12.0):
    """Q = 0.3 g + 1, K = 0.3 h + a_t (a_t constant over key tile t, rising by
    step_log2 / (sqrt(d) log2 e) per tile), V = N(0, 1), g, h, V iid N(0, 1):
    the scaled logit of every row rises by about step_log2 log2 units from
    one key tile to the next, with a spread of about 0.4 log2 units over the
    keys of a tile, so that even a causal diagonal tile with one allowed key
    raises the maximum by more than the threshold."""
    q, k, v = synth.attn_inputs(B, Nq, Nk, Hq, Hkv, d, dtype=torch.float32, seed=seed)
    delta = step_log2 / (math.sqrt(d) * LOG2E)
    ramp = (torch.arange(Nk) // 128).float() * delta                 # a_t per key
    q = 0.3 * q + 1.0
    k = 0.3 * k + ramp[None, :, None, None]
    return q.to(dtype), k.to(dtype), v.to(dtype)


def _count_rescales(q, k, causal, scale, j0_tiles=None):
    """For every (b, h, i): the number of key tiles at which the kernels' rule
    (reference = max of the first tile of the range, moved when a tile's
    maximum exceeds it by more than TAU log2 units) must move the reference,
    counting only moves clear of the threshold by 0.5.  j0_tiles: tiles per
    key range (split instances start a fresh reference per range)."""
    qd = q.double().cpu().numpy()
    kd = k.double().cpu().numpy()
    B, Nq, Hq, d = qd.shape
    Nk, Hkv = kd.shape[1], kd.shape[2]
    G = Hq // Hkv
    nt = (Nk + 127) // 128
    out = np.zeros((B, Hq, Nq), dtype=np.int64)
    for b in range(B):
        for h in range(Hq):
            s = qd[b, :, h] @ kd[b, :, h // G].T * scale * LOG2E    # [Nq, Nk] log2 units
            if causal:
                s = np.where(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None], s, -np.inf)
            tm = np.stack([s[:, t * 128:(t + 1) * 128].max(axis=1) for t in range(nt)], axis=1)
            per = j0_tiles or nt
            for r0 in range(0, nt, per):
                ref = tm[:, r0]
                for t in range(r0 + 1, min(r0 + per, nt)):
                    fin = np.isfinite(tm[:, t])
                    move = fin & (tm[:, t] > ref + TAU + 0.5)
                    near = fin & (np.abs(tm[:, t] - ref - TAU) <= 0.5)
                    out[b, h] += move
                    assert not near.any()     # no decision within 0.5 of the threshold
                    ref = np.where(move, tm[:, t], ref)
    return out


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_lazy_rescale_fires_every_tile(gpu_lib, d, causal, dtype):
    """Rows spanning 9 key tiles (ragged last tile), every later tile moving
    the reference; two query tiles per unit for d <= 128, one for d = 256."""
    B, N, Hq, Hkv = 1, 1100, 4, 2
    q, k, v = _ramp_inputs(B, N, N, Hq, Hkv, d, DT[dtype], seed=11)
    scale = 1.0 / math.sqrt(d)
    moves = _count_rescales(q, k, causal, scale)
    span = np.array([(_allowed(i, N, causal) + 127) // 128 for i in range(N)])
    # every tile after the first moves the reference, in every row
    assert np.array_equal(moves, np.broadcast_to(span - 1, moves.shape)), moves.min()
    assert moves.sum() > 0
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o, lse = gpu_lib.attn_fwd(q, k, v, causal=causal, scale=scale)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, causal, scale)
    assert_within(errors(o, lse, o_ref, lse_ref))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_lazy_rescale_fires_in_split_key_ranges(gpu_lib, d):
    """The split instances: each 8-tile key range starts its own reference and
    moves it at each of its later tiles; the ranges are merged afterwards."""
    B, Nq, Nk, Hq, Hkv = 1, 5, 4096, 8, 2
    q, k, v = _ramp_inputs(B, Nq, Nk, Hq, Hkv, d, torch.bfloat16, seed=12)
    scale = 1.0 / math.sqrt(d)
    moves = _count_rescales(q, k, False, scale, j0_tiles=8)
    assert np.all(moves == 4 * 7), moves.min()        # 4 ranges x 7 moves
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o, lse = gpu_lib.attn_fwd_splitkv(q, k, v, num_splits=4, scale=scale)
    assert gpu_lib.get_status() == 0
    o_ref, lse_ref = oracle_for(q, k, v, False, scale)
    assert_within(errors(o, lse, o_ref, lse_ref))


# ------------------------------------------------------- one dominant key
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_dominant_key_in_last_tile_selects_its_value(gpu_lib, d, causal):
    """Q = g + 1, K = N(0, 1) except key j* (in the last of 9 key tiles) set to
    20 in every channel: for every row that sees j*, the scaled logit of j*
    exceeds every other logit of the row by at least 60, so O = V[j*] and LSE
    = that logit up to e^-60."""
    B, N, Hq, Hkv = 1, 1100, 4, 2
    q, k, v = synth.attn_inputs(B, N, N, Hq, Hkv, d, dtype=torch.float32, seed=13)
    q = q + 1.0
    jstar = 1050
    k[:, jstar] = 20.0
    q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    G = Hq // Hkv
    rows_see = np.arange(N) >= jstar if causal else np.ones(N, bool)
    for h in range(Hq):
        s = qd[0, :, h] @ kd[0, :, h // G].T * scale                 # [N, N]
        if causal:
            s = np.where(np.arange(N)[None, :] <= np.arange(N)[:, None], s, -np.inf)
        others = np.delete(s, jstar, axis=1).max(axis=1)
        gap = s[:, jstar] - others
        assert np.all(gap[rows_see] >= 60.0), gap[rows_see].min()
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o, lse = gpu_lib.attn_fwd(qc, kc, vc, causal=causal, scale=scale)
    assert gpu_lib.get_status() == 0
    og = o.double().cpu().numpy()[0]                                  # [N, Hq, d]
    lg = lse.double().cpu().numpy()[0]                                # [Hq, N]
    for h in range(Hq):
        want_o = vd[0, jstar, h // G]
        want_l = qd[0, :, h] @ kd[0, jstar, h // G] * scale
        assert np.abs(og[rows_see, h] - want_o).max() <= 1e-2
        assert np.abs(lg[h, rows_see] - want_l[rows_see]).max() <= 1e-3
    o_ref, lse_ref = oracle_for(qc, kc, vc, causal, scale)
    assert_within(errors(o, lse, o_ref, lse_ref))
