"""A step-by-step model of the fused attention kernel's online softmax, in
numpy (fp32 where the kernel computes in fp32), checked against the fp64
oracle on the CPU.

The model takes the kernel's order of operations, not the oracle's: key
blocks of 128, each row's block split into two halves of 64 keys; each half
exponentiates against a provisional maximum (the running maximum, raised so
that p <= 2^64, or in the row's first block the half's own maximum); the
row's maximum m_new then follows from both halves and p moves to it where the
two differ (p * exp2(m_use - m_new)); O and l are rescaled lazily, only when a
block's maximum exceeds the running one by more than 8 (log2 units); p is
rounded to bf16 before its product with V, and l sums the unrounded p.

Score patterns that reach every branch (a later block far above the running
maximum, a maximum that climbs block by block, negative and zero alpha, blocks
whose upper half holds no keys) must keep every intermediate finite, every p
at most 2^8 once moved to the row's maximum, and O within the oracle's bound.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from dense_matmul_tensor_gb300 import workloads as wl

D = 128
BLOCK = 128
HALF = 64
RESCALE_LOG2 = 8.0
SPEC_LOG2 = 64.0


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even) -> fp32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32)


def _model(q, k, v, alpha):
    """O [Lq, D] float64 for one batch item (q, k, v: float32 [L, D])."""
    f32 = np.float32
    sc = f32(float(alpha) * 1.4426950408889634)
    Lq, Lk = q.shape[0], k.shape[0]
    m = np.full(Lq, -np.inf, f32)
    l = np.zeros((2, Lq), f32)
    o = np.zeros((Lq, D), f32)
    for j in range(-(-Lk // BLOCK)):
        valid = min(BLOCK, Lk - j * BLOCK)
        s = np.zeros((Lq, BLOCK), f32)  # keys past Lk: zero-filled K rows
        s[:, :valid] = (q.astype(np.float64) @ k[j * BLOCK:j * BLOCK + valid].astype(np.float64).T).astype(f32)
        z = s * sc
        mine, p = [], []
        for h in range(2):
            vh = valid - HALF * h
            zh = z[:, HALF * h:HALF * (h + 1)]
            mine.append(zh[:, :vh].max(axis=1) if vh > 0 else np.full(Lq, -np.inf, f32))
        m_use = [mine[h] if j == 0 else np.maximum(m, mine[h] - f32(SPEC_LOG2)) for h in range(2)]
        for h in range(2):
            with np.errstate(over="ignore", invalid="ignore"):
                ph = np.exp2(z[:, HALF * h:HALF * (h + 1)] - m_use[h][:, None]).astype(f32)
            keys = HALF * h + np.arange(HALF)
            ph[:, keys >= valid] = 0.0
            assert np.isfinite(ph).all()
            assert (ph <= f32(2.0 ** SPEC_LOG2)).all()
            p.append(ph)
        m_blk = np.maximum(mine[0], mine[1])
        grow = (m_blk > m + f32(RESCALE_LOG2)) if j > 0 else np.zeros(Lq, bool)
        m_new = m_blk if j == 0 else np.where(grow, m_blk, m)
        for h in range(2):
            moved = m_use[h] != m_new
            r = np.where(moved, np.exp2((m_use[h] - m_new).astype(f32)), f32(1.0)).astype(f32)
            p[h] = (p[h] * r[:, None]).astype(f32)
            assert (p[h] <= f32(2.0 ** RESCALE_LOG2) * f32(1.0 + 2.0 ** -20)).all()
        if j > 0:
            r = np.where(grow, np.exp2((m - m_new).astype(f32)), f32(1.0)).astype(f32)
            o *= r[:, None]
            l *= r[None, :]
        m = m_new
        for h in range(2):
            l[h] += p[h].sum(axis=1, dtype=f32)
        pb = _bf16_round(np.concatenate(p, axis=1))
        o += (pb[:, :valid].astype(np.float64) @ v[j * BLOCK:j * BLOCK + valid].astype(np.float64)).astype(f32)
        assert np.isfinite(o).all() and np.isfinite(l).all()
    out = o / (l[0] + l[1])[:, None]
    return _bf16_round(out.astype(f32)).astype(np.float64)


def _check(Q, K, V, alpha):
    batch, Lq, _ = Q.shape
    Lk = K.shape[1]
    ref, bnd = oracle.attention(Q, K, V, batch=batch, Lq=Lq, Lk=Lk, D=D, alpha=alpha)
    tol = oracle.attention_tolerance(ref, bnd, Q, K, V, alpha=alpha)
    q, k, v = (oracle.decode(x, "bf16").astype(np.float32) for x in (Q, K, V))
    worst = 0.0
    for b in range(batch):
        got = _model(q[b], k[b], v[b], alpha)
        err = np.abs(got - ref[b])
        assert (err <= tol[b]).all(), float((err / tol[b]).max())
        worst = max(worst, float((err / tol[b]).max()))
    return worst


def _scale_keys(K, lo, hi, log2_factor):
    """K with rows [lo, hi) scaled by 2^log2_factor (exact in bf16)."""
    k = oracle.decode(K, "bf16").astype(np.float32)
    k[:, lo:hi, :] *= np.float32(2.0 ** log2_factor)
    return (k.view(np.uint32) >> 16).astype(np.uint16)


ALPHA = float(np.float32(1.0 / math.sqrt(D)))


@pytest.mark.parametrize("alpha", [ALPHA, 1.0, -0.2, 0.0])
def test_model_matches_oracle_on_random_scores(alpha):
    Q, K, V = wl.attention_qkv(2, 48, D, Lk=1000, seed=81)
    _check(Q, K, V, alpha)


@pytest.mark.parametrize("alpha", [1.0, -1.0])
def test_model_survives_a_block_far_above_the_running_maximum(alpha):
    # block 1 exceeds block 0 by thousands (log2 units): its halves start from
    # m - 64 < mine and O, l from block 0 rescale to (nearly) zero
    Q, K, V = wl.attention_qkv(1, 40, D, Lk=400, seed=82)
    _check(Q, _scale_keys(K, 128, 256, 6), V, alpha)


def test_model_follows_a_maximum_that_climbs_block_by_block():
    # block j scaled by 2^(j/2): the maximum rises every other block, sometimes
    # by more than the lazy-rescale threshold and sometimes by less
    Q, K, V = wl.attention_qkv(1, 40, D, Lk=1024, seed=83)
    for j in range(8):
        K = _scale_keys(K, j * BLOCK, (j + 1) * BLOCK, j // 2)
    _check(Q, K, V, 0.5)


@pytest.mark.parametrize("Lk", [1, 64, 65, 129, 200])
def test_model_on_blocks_whose_upper_half_is_short_or_empty(Lk):
    Q, K, V = wl.attention_qkv(1, 24, D, Lk=Lk, seed=84 + Lk)
    _check(Q, K, V, ALPHA)
