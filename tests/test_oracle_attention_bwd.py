"""Pins of the backward oracle (``oracle.attention_bwd``): torch autograd in
fp64, central finite differences of the forward oracle, the closed form of a
one-token sequence, the invariants sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i,
and the ring: block gradients summed over every ring step of every split
equal the full gradients ("Scaling video training with parallelism",
section 2, Ring Attention)."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import attention_bwd as B
from oracle import plan as P


def _inputs(cu, H, Hkv, D, seed=0, scale_in=1.0):
    rng = np.random.default_rng(seed)
    T = cu[-1]
    q = rng.standard_normal((T, H, D)) * scale_in
    k = rng.standard_normal((T, Hkv, D)) * scale_in
    v = rng.standard_normal((T, Hkv, D))
    do = rng.standard_normal((T, H, D))
    return q, k, v, do


def _torch_grads(q, k, v, do, cu, causal, scale):
    """Autograd of a dense-mask softmax attention written in torch fp64."""
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    T, H, D = q.shape
    Hkv = k.shape[1]
    outs = []
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        rows = []
        for h in range(H):
            g = h * Hkv // H
            S = scale * qt[a:b, h] @ kt[a:b, g].T
            if causal:
                S = S.masked_fill(torch.ones(b - a, b - a, dtype=torch.bool).triu(1), float("-inf"))
            rows.append(torch.softmax(S, dim=-1) @ vt[a:b, g])
        outs.append(torch.stack(rows, dim=1))
    O = torch.cat(outs, dim=0)
    O.backward(torch.tensor(do))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


CASES = [((0, 5, 17, 30), 4, 2, 8, True), ((0, 9, 20), 2, 2, 4, False), ((0, 1, 2, 40), 6, 3, 16, True),
         ((0, 33), 2, 1, 8, True)]


@pytest.mark.parametrize("case", CASES)
def test_matches_torch_autograd(case):
    cu, H, Hkv, D, causal = case
    q, k, v, do = _inputs(cu, H, Hkv, D, seed=len(cu))
    got = B.packed_attention_bwd(q, k, v, do, cu, causal, 0.3)
    ref = _torch_grads(q, k, v, do, cu, causal, 0.3)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)


def test_central_finite_differences():
    cu, H, Hkv, D, causal, scale = (0, 6, 13), 4, 2, 5, True, 0.45
    q, k, v, do = _inputs(cu, H, Hkv, D, seed=3)
    dq, dk, dv = B.packed_attention_bwd(q, k, v, do, cu, causal, scale)

    def f(q_, k_, v_):
        return float(np.sum(A.packed_attention(q_, k_, v_, cu, causal, scale)[0] * do))

    rng = np.random.default_rng(4)
    eps = 1e-5
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(12):
            xs = [q.copy(), k.copy(), v.copy()]
            idx = tuple(int(rng.integers(0, n)) for n in xs[which].shape)
            xs[which][idx] += eps
            fp = f(*xs)
            xs[which][idx] -= 2 * eps
            fm = f(*xs)
            fd = (fp - fm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


def test_one_token_sequence_closed_form():
    # one visible key: P = 1, so dV = dO and dS = dO.v - dO.v = 0 (dQ = dK = 0)
    cu = (0, 1, 2)
    q, k, v, do = _inputs(cu, 2, 2, 4, seed=5)
    dq, dk, dv = B.packed_attention_bwd(q, k, v, do, cu, True, 0.7)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)


@pytest.mark.parametrize("causal", [True, False])
def test_invariants_per_sequence_and_kv_head(causal):
    cu, H, Hkv, D = (0, 7, 30, 64), 6, 2, 8
    q, k, v, do = _inputs(cu, H, Hkv, D, seed=6, scale_in=2.0)
    dq, dk, dv = B.packed_attention_bwd(q, k, v, do, cu, causal, 0.5)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for g in range(Hkv):
            heads = [h for h in range(H) if h * Hkv // H == g]
            # the rows of dS sum to zero, so the keys' gradients cancel
            assert np.abs(dk[a:b, g].sum(axis=0)).max() < 1e-10
            # every row of P sums to one
            np.testing.assert_allclose(dv[a:b, g].sum(axis=0), do[a:b][:, heads].sum(axis=(0, 1)), atol=1e-10)


@pytest.mark.parametrize("mode,cp,causal,grid", [("zigzag", 2, True, None), ("zigzag", 4, True, None),
                                                 ("contiguous", 3, True, None), ("zigzag", 3, False, None),
                                                 ("grid2d", 4, False, (2, 4, 6))])
def test_ring_steps_sum_to_the_full_gradients(mode, cp, causal, grid):
    cu = (0, 48) if grid else (0, 24, 61, 100)
    H, Hkv, D, scale = 4, 2, 8, 0.4
    q, k, v, do = _inputs(cu, H, Hkv, D, seed=7)
    O, L = A.packed_attention(q, k, v, cu, causal, scale)
    full = B.packed_attention_bwd(q, k, v, do, cu, causal, scale)
    plan = P.make_plan(cu, cp, mode, grid)
    kv_rank, _ = P.ring_schedule(plan, causal)
    acc = [np.zeros_like(x) for x in full]
    for r in range(cp):
        qr = P.rank_rows(plan, r)
        for t in range(cp):
            kr = P.rank_rows(plan, kv_rank[r, t])
            gq, gk, gv = B.block_attention_bwd(q, k, v, do, O, L, cu, qr, kr, causal, scale)
            acc[0][qr] += gq
            acc[1][kr] += gk
            acc[2][kr] += gv
    for a_, f_ in zip(acc, full):
        np.testing.assert_allclose(a_, f_, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("threads,batch", [(None, None), (3, 2), (1, 1)])
def test_dq_at_rows_equals_the_full_backward(causal, threads, batch):
    """Row batches of any size, on any number of threads, give the full
    backward's dQ rows (unsorted rows, several sequences, G = 2)."""
    cu, H, Hkv, D = (0, 40, 41, 90), 4, 2, 8
    q, k, v, do = _inputs(cu, H, Hkv, D, seed=8)
    full = B.packed_attention_bwd(q, k, v, do, cu, causal, 0.35)[0]
    rows = np.array([77, 0, 5, 39, 40, 41, 89, 12, 60])
    got = B.dq_at_rows(q, k, v, do, cu, rows, causal, 0.35, threads=threads, batch=batch)
    np.testing.assert_allclose(got, full[rows], rtol=1e-11, atol=1e-13)
