"""Fused attention O = softmax(alpha Q K^T) V on the GPU through the C ABI,
element by element against the fp64 oracle (``oracle.attention``).

The kernel rounds the probabilities to bf16 before their product with V, as
the two-step pair does, accumulates in fp32 and rounds O to bf16 once; the
acceptance bound per element is ``oracle.attention_tolerance``:
(2^-8 + 2^-14 + eta_i) * (sum_c p_ic |V_cd| + |O_id|) + Lk * 2^-126 * max|V|,
with eta_i the stated fp32 score allowance carried through the exponential.
Every operand sits inside a larger buffer whose padding and guards hold NaN,
so a read outside Q, K or V turns O into NaN; O's padding holds a sentinel
that must survive.
"""
from __future__ import annotations

import math
import time

import numpy as np
import pytest
import torch

import oracle
from dense_matmul_tensor_gb300 import bmm as api
from dense_matmul_tensor_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

D = 128
NAN16 = np.int16(0x7FC0)
O_SENTINEL = np.int16(np.array([0xC0DE], np.uint16).view(np.int16)[0])
ALPHA = float(np.float32(1.0 / math.sqrt(D)))


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _place(bits, rows, ld, stride, fill, dev, guard=4096):
    """[batch, rows, D] bit array -> device int16 buffer with row stride ld,
    batch stride `stride`, `guard` fill elements before and after."""
    batch = bits.shape[0]
    span = (batch - 1) * stride + (rows - 1) * ld + D if batch and rows else 0
    host = np.full(guard + span + guard, fill, dtype=np.int16)
    for b in range(batch):
        for i in range(rows):
            o = guard + b * stride + i * ld
            host[o:o + D] = bits[b, i].view(np.int16)
    buf = torch.from_numpy(host).to(dev)
    return buf, guard


def run_attn(Q, K, V, *, alpha, lds=(D, D, D, D), pads=(0, 0, 0, 0), plan_env=None):
    """Run the fused kernel on bit arrays Q [b, Lq, D], K and V [b, Lk, D];
    returns (O float64 [b, Lq, D], status of the device error word)."""
    batch, Lq, _ = Q.shape
    Lk = K.shape[1]
    ldq, ldk, ldv, ldo = lds
    sq, sk, sv, so = (Lq * ldq + pads[0], Lk * ldk + pads[1], Lk * ldv + pads[2],
                      Lq * ldo + pads[3])
    dev = torch.device("cuda:0")
    qb, qo = _place(Q, Lq, ldq, sq, NAN16, dev)
    kb, ko = _place(K, Lk, ldk, sk, NAN16, dev)
    vb, vo = _place(V, Lk, ldv, sv, NAN16, dev)
    zero = np.zeros((batch, Lq, D), np.uint16)
    ob, oo = _place(zero, Lq, ldo, so, O_SENTINEL, dev)
    ob.fill_(int(O_SENTINEL))
    desc = api.make_attn_desc(batch=batch, Lq=Lq, Lk=Lk, alpha=alpha, ldq=ldq, ldk=ldk, ldv=ldv,
                              ldo=ldo, strideQ=sq, strideK=sk, strideV=sv, strideO=so)
    es = 2
    with api.AttnPlan(desc) as plan:
        plan.run(qb.data_ptr() + qo * es, kb.data_ptr() + ko * es, vb.data_ptr() + vo * es,
                 ob.data_ptr() + oo * es, torch.cuda.current_stream())
        torch.cuda.synchronize()
        st, word = plan.device_error()
    assert st == api.BMM_OK, f"device error word {word:#x}"
    host = ob.cpu().numpy()
    # everything outside the rows of O is untouched
    mask = np.ones(host.size, bool)
    for b in range(batch):
        for i in range(Lq):
            o = oo + b * so + i * ldo
            mask[o:o + D] = False
    assert np.all(host[mask] == O_SENTINEL), "write outside O"
    out = np.empty((batch, Lq, D), np.float64)
    vals = torch.from_numpy(host).view(torch.bfloat16).double().numpy()
    for b in range(batch):
        for i in range(Lq):
            o = oo + b * so + i * ldo
            out[b, i] = vals[o:o + D]
    return out


def check(O, Q, K, V, alpha):
    batch, Lq, _ = Q.shape
    ref, bnd = oracle.attention(Q, K, V, batch=batch, Lq=Lq, Lk=K.shape[1], D=D, alpha=alpha)
    assert not np.isnan(O).any(), "NaN in O: a read outside Q, K or V"
    tol = oracle.attention_tolerance(ref, bnd, Q, K, V, alpha=alpha)
    err = np.abs(O - ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} elements out of bound; worst at "
                           f"{np.unravel_index(np.argmax(err - tol), err.shape)}: "
                           f"{O.flat[np.argmax(err - tol)]} vs {ref.flat[np.argmax(err - tol)]}")
    return float((err / tol).max())


SHAPES = [
    (1, 128, 128),     # one tile, one key block
    (2, 200, 77),      # ragged query tile, one partial key block
    (3, 129, 300),     # a 1-row second tile, 2 full + 1 partial key blocks
    (1, 1, 1),         # the degenerate softmax over one key: O = V's row
    (2, 64, 1000),     # eight key blocks, the last 104 wide
    (1, 300, 129),     # a one-key last block
    (1, 130, 64),      # one block of exactly the lower key half (the upper half holds none)
    (2, 100, 65),      # one key in the upper half of the only block
]


@pytest.mark.parametrize("batch,Lq,Lk", SHAPES)
def test_fused_attention_matches_oracle(batch, Lq, Lk):
    _need_gpu()
    Q, K, V = wl.attention_qkv(batch, Lq, D, Lk=Lk, seed=11 + Lq + Lk)
    O = run_attn(Q, K, V, alpha=ALPHA)
    check(O, Q, K, V, ALPHA)


def test_persistent_ctas_carry_ring_phases_across_tiles():
    # 160 x 2 = 320 query tiles on at most 152 CTAs: each CTA runs two or three
    # tiles of three key blocks, so every barrier ring (and both O buffers)
    # wraps across tiles
    _need_gpu()
    Q, K, V = wl.attention_qkv(160, 130, D, Lk=260, seed=21)
    O = run_attn(Q, K, V, alpha=ALPHA)
    check(O, Q, K, V, ALPHA)


def test_padded_rows_and_batch_strides():
    _need_gpu()
    Q, K, V = wl.attention_qkv(3, 150, D, Lk=200, seed=31)
    O = run_attn(Q, K, V, alpha=ALPHA, lds=(136, 144, 192, 160), pads=(8, 64, 8, 24))
    check(O, Q, K, V, ALPHA)


@pytest.mark.parametrize("alpha", [-0.2, 0.0, 1.0])
def test_scale_sign_zero_and_sharp(alpha):
    # alpha < 0 flips which key dominates; alpha = 0 gives the mean of V's rows;
    # alpha = 1 on unit-normal data (scores of order 10) gives a peaked softmax
    _need_gpu()
    Q, K, V = wl.attention_qkv(2, 130, D, Lk=300, seed=41)
    O = run_attn(Q, K, V, alpha=alpha)
    check(O, Q, K, V, alpha)
    if alpha == 0.0:
        mean = oracle.decode(V, "bf16").mean(axis=1)
        assert np.allclose(O, mean[:, None, :], rtol=2.0 ** -7, atol=1e-3)


@pytest.mark.parametrize("alpha", [1.0, -1.0])
def test_a_later_block_far_above_the_running_maximum(alpha):
    # keys 128..255 scaled by 2^6: block 1's scores exceed block 0's maximum
    # by far more than 2^64 in log2 units, so its exponentials must be redone
    # against its own maximum and O, l from block 0 rescale to (nearly) zero;
    # block 2 falls back far below the new maximum
    _need_gpu()
    Q, K, V = wl.attention_qkv(2, 130, D, Lk=400, seed=71)
    k = oracle.decode(K, "bf16").astype(np.float32)
    k[:, 128:256, :] *= 64.0
    K = (k.view(np.uint32) >> 16).astype(np.uint16)  # exact: a power-of-two scale
    O = run_attn(Q, K, V, alpha=alpha)
    check(O, Q, K, V, alpha)


def test_repeat_runs_are_bitwise_identical():
    _need_gpu()
    Q, K, V = wl.attention_qkv(4, 256, D, Lk=384, seed=51)
    a = run_attn(Q, K, V, alpha=ALPHA)
    b = run_attn(Q, K, V, alpha=ALPHA)
    assert np.array_equal(a, b)


def test_full_workload_every_element_and_convexity():
    """batch 128, Lq = Lk = 2048, D = 128 (the attention pair's shape, with the
    pair's inputs): every element of O against the oracle, and for every row
    the property that O is a convex combination of V's rows:
    min_c V_cd <= O_id <= max_c V_cd, within O's final rounding."""
    _need_gpu()
    batch, L = 128, 2048
    Q, K, V = wl.attention_qkv(batch, L, D)
    dev = torch.device("cuda:0")
    q = torch.from_numpy(Q.view(np.int16)).to(dev)
    k = torch.from_numpy(K.view(np.int16)).to(dev)
    v = torch.from_numpy(V.view(np.int16)).to(dev)
    o = torch.full_like(q, int(NAN16))
    desc = api.make_attn_desc(batch=batch, Lq=L, Lk=L, alpha=ALPHA)
    with api.AttnPlan(desc) as plan:
        plan.run(q, k, v, o, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.device_error()[0] == api.BMM_OK
    of = o.view(torch.bfloat16).float()
    assert bool(torch.isfinite(of).all())
    vf = v.view(torch.bfloat16).float()
    lo, hi = vf.amin(dim=1, keepdim=True), vf.amax(dim=1, keepdim=True)
    slack = 2.0 ** -7 * torch.maximum(lo.abs(), hi.abs())
    assert bool(((of >= lo - slack) & (of <= hi + slack)).all())
    O = of.double().cpu().numpy()
    del q, k, v, o, of, vf
    worst = check(O, Q, K, V, ALPHA)
    print(f"attention 128x2048x2048x128: max err/tol over all {O.size} elements = {worst:.4f}")


def test_expired_wait_is_reported_and_the_next_run_is_clean(monkeypatch):
    _need_gpu()
    Q, K, V = wl.attention_qkv(2, 256, D, Lk=512, seed=61)
    monkeypatch.setenv("DMT_BMM_TEST_STALL_MMA", "1")
    monkeypatch.setenv("DMT_BMM_WAIT_TIMEOUT_MS", "50")
    dev = torch.device("cuda:0")
    q, k, v = (torch.from_numpy(x.view(np.int16)).to(dev) for x in (Q, K, V))
    o = torch.zeros_like(q)
    with api.AttnPlan(api.make_attn_desc(batch=2, Lq=256, Lk=512, alpha=ALPHA)) as plan:
        t0 = time.perf_counter()
        plan.run(q, k, v, o, torch.cuda.current_stream())
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        st, word = plan.device_error()
    assert st == api.BMM_ERR_DEVICE_TIMEOUT
    assert word >> 28 == 0xB
    assert elapsed < 5.0
    monkeypatch.delenv("DMT_BMM_TEST_STALL_MMA")
    monkeypatch.delenv("DMT_BMM_WAIT_TIMEOUT_MS")
    O = run_attn(Q, K, V, alpha=ALPHA)
    check(O, Q, K, V, ALPHA)


def test_empty_problems_launch_nothing():
    _need_gpu()
    for batch, Lq in ((0, 128), (2, 0)):
        with api.AttnPlan(api.make_attn_desc(batch=batch, Lq=Lq, Lk=16, alpha=ALPHA)) as plan:
            plan.run(None, None, None, None, torch.cuda.current_stream())
        torch.cuda.synchronize()
