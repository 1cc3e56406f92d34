"""Pins for the fp64 attention oracle: brute force, a library routine, closed
forms and the invariants the split must keep.  CPU only."""

import math

import numpy as np
import pytest
import torch

import inputs
from oracle import attention as A
from oracle import merge as M
from oracle import plan as P


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def brute_force(q, k, v, cu, causal, scale):
    """Dense-mask attention with explicit Python loops and math.exp."""
    T, H, D = q.shape
    Hkv = k.shape[1]
    group = H // Hkv
    seq, pos = [], []
    s = 0
    for t in range(T):
        while t >= cu[s + 1]:
            s += 1
        seq.append(s)
        pos.append(t - cu[s])
    O = np.zeros((T, H, D))
    LSE = np.zeros((H, T))
    for h in range(H):
        g = h // group
        for i in range(T):
            scores = {}
            for j in range(T):
                if seq[j] != seq[i] or (causal and pos[j] > pos[i]):
                    continue
                acc = 0.0
                for d in range(D):
                    acc += q[i, h, d] * k[j, g, d]
                scores[j] = scale * acc
            mx = max(scores.values())
            wts = {j: math.exp(sv - mx) for j, sv in scores.items()}
            Z = sum(wts.values())
            for d in range(D):
                O[i, h, d] = sum(w * v[j, g, d] for j, w in wts.items()) / Z
            LSE[h, i] = mx + math.log(Z)
    return O, LSE


CASES = [
    ((0, 5, 17, 40), 4, 2, 8, True),
    ((0, 5, 17, 40), 4, 2, 8, False),
    ((0, 1, 2, 30, 31), 2, 1, 4, True),
    ((0, 48), 3, 3, 6, True),
]


@pytest.mark.parametrize("cu,H,Hkv,D,causal", CASES)
def test_oracle_matches_brute_force(cu, H, Hkv, D, causal):
    T = cu[-1]
    q, k, v = _rand((T, H, D), 1), _rand((T, Hkv, D), 2), _rand((T, Hkv, D), 3)
    scale = 0.37
    O, L = A.packed_attention(q, k, v, cu, causal, scale, row_block=7)
    Ob, Lb = brute_force(q, k, v, cu, causal, scale)
    assert np.abs(O - Ob).max() < 1e-12
    assert np.abs(L - Lb).max() < 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_oracle_matches_torch_sdpa(causal):
    """Per-sequence attention equals torch's scaled_dot_product_attention (fp64
    CPU) with K/V heads repeated for GQA, and LSE equals torch.logsumexp."""
    cu = (0, 33, 100, 161)
    H, Hkv, D = 8, 2, 16
    T = cu[-1]
    q, k, v = _rand((T, H, D), 4), _rand((T, Hkv, D), 5), _rand((T, Hkv, D), 6)
    scale = 1 / math.sqrt(D)
    O, L = A.packed_attention(q, k, v, cu, causal, scale)
    for a, b in zip(cu[:-1], cu[1:]):
        qt = torch.from_numpy(q[a:b]).permute(1, 0, 2)[None]
        kt = torch.from_numpy(k[a:b]).permute(1, 0, 2).repeat_interleave(H // Hkv, 0)[None]
        vt = torch.from_numpy(v[a:b]).permute(1, 0, 2).repeat_interleave(H // Hkv, 0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)
        assert np.abs(O[a:b] - ref[0].permute(1, 0, 2).numpy()).max() < 1e-12
        s = scale * (qt @ kt.transpose(-1, -2))
        if causal:
            s = s.masked_fill(torch.ones(b - a, b - a, dtype=torch.bool).triu(1), float("-inf"))
        lse = torch.logsumexp(s, dim=-1)[0].numpy()
        assert np.abs(L[:, a:b] - lse).max() < 1e-12


def test_zero_queries_give_log_count_and_prefix_mean():
    cu = (0, 7, 30)
    H, D = 2, 5
    T = cu[-1]
    q = np.zeros((T, H, D))
    k, v = _rand((T, H, D), 7), _rand((T, H, D), 8)
    O, L = A.packed_attention(q, k, v, cu, True, 0.5)
    for a, b in zip(cu[:-1], cu[1:]):
        for i in range(a, b):
            n = i - a + 1
            assert abs(L[0, i] - math.log(n)) < 1e-14
            assert np.abs(O[i] - v[a:i + 1].mean(axis=0)).max() < 1e-14
    Ob, Lb = A.packed_attention(q, k, v, cu, False, 0.5)
    for a, b in zip(cu[:-1], cu[1:]):
        assert np.abs(Lb[:, a:b] - math.log(b - a)).max() < 1e-14
        assert np.abs(Ob[a:b] - v[a:b].mean(axis=0)).max() < 1e-14


def test_first_token_sees_only_itself():
    cu = (0, 9, 20, 21)
    H, Hkv, D = 4, 2, 6
    T = cu[-1]
    q, k, v = _rand((T, H, D), 9), _rand((T, Hkv, D), 10), _rand((T, Hkv, D), 11)
    O, L = A.packed_attention(q, k, v, cu, True, 0.25)
    for a in cu[:-1]:
        for h in range(H):
            g = h // (H // Hkv)
            assert np.array_equal(O[a, h], v[a, g])
            assert abs(L[h, a] - 0.25 * float(q[a, h] @ k[a, g])) < 1e-14


def test_dominant_key_selects_its_value():
    cu = (0, 40)
    H, D = 1, 8
    q, k, v = _rand((40, H, D), 12, 0.01), _rand((40, H, D), 13, 0.01), _rand((40, H, D), 14)
    q[25, 0] = 1.0
    k[3, 0] = 100.0  # score 100*... dominates every other key for row 25
    O, _ = A.packed_attention(q, k, v, cu, False, 1.0)
    assert np.abs(O[25, 0] - v[3, 0]).max() < 1e-12


def test_block_partials_merge_to_full_for_random_partitions():
    cu = (0, 50, 77, 140)
    H, Hkv, D = 4, 2, 8
    T = cu[-1]
    q, k, v = _rand((T, H, D), 15), _rand((T, Hkv, D), 16), _rand((T, Hkv, D), 17)
    O, L = A.packed_attention(q, k, v, cu, True, 0.3)
    rng = np.random.default_rng(18)
    for nparts in (1, 2, 3, 7):
        owner = rng.integers(0, nparts, T)
        parts = [A.block_attention(q, k, v, cu, np.arange(T), np.nonzero(owner == p)[0], True, 0.3)
                 for p in range(nparts)]
        Om, Lm = M.lse_merge([p[0] for p in parts], [p[1] for p in parts])
        assert np.abs(Om - O).max() < 1e-12
        assert np.abs(Lm - L).max() < 1e-12


def _ring_emulation(q, k, v, cu, plan, causal, scale):
    """Every virtual rank runs cp ring steps of block attention over the KV
    shard it holds at that step; partials are merged and scattered back."""
    T, H, D = q.shape
    O = np.full((T, H, D), np.nan)
    L = np.full((H, T), np.nan)
    kv_rank, _ = P.ring_schedule(plan, causal)
    for r in range(plan.cp):
        q_rows = P.rank_rows(plan, r)
        parts = [A.block_attention(q, k, v, cu, q_rows, P.rank_rows(plan, kv_rank[r, t]), causal, scale)
                 for t in range(plan.cp)]
        Om, Lm = M.lse_merge([p[0] for p in parts], [p[1] for p in parts])
        O[q_rows] = Om
        L[:, q_rows] = Lm
    return O, L


@pytest.mark.parametrize("mode,cps", [("zigzag", (1, 2, 4)), ("contiguous", (1, 3, 4))])
def test_cp_split_does_not_change_the_result(mode, cps):
    w = inputs.workload("tiny_packed_fp32")
    q, k, v = (t.numpy().astype(np.float64) for t in inputs.make_qkv(w))
    O, L = A.packed_attention(q, k, v, w.cu_seqlens, True, w.scale)
    for cp in cps:
        plan = P.make_plan(w.cu_seqlens, cp, mode)
        Or, Lr = _ring_emulation(q, k, v, w.cu_seqlens, plan, True, w.scale)
        assert np.abs(Or - O).max() < 1e-12, cp
        assert np.abs(Lr - L).max() < 1e-12, cp


def test_grid2d_split_does_not_change_bidirectional_result():
    F, h, wd = 2, 5, 6
    T = F * h * wd
    H, D = 2, 8
    q, k, v = _rand((T, H, D), 19), _rand((T, H, D), 20), _rand((T, H, D), 21)
    O, L = A.packed_attention(q, k, v, (0, T), False, 0.35)
    for cp in (1, 2, 4):
        plan = P.grid2d((0, T), cp, (F, h, wd))
        Or, Lr = _ring_emulation(q, k, v, (0, T), plan, False, 0.35)
        assert np.abs(Or - O).max() < 1e-12
        assert np.abs(Lr - L).max() < 1e-12


def test_no_attention_crosses_sequence_boundaries():
    cu = (0, 20, 45, 60)
    H, D = 2, 4
    T = cu[-1]
    q, k, v = _rand((T, H, D), 22), _rand((T, H, D), 23), _rand((T, H, D), 24)
    for causal in (True, False):
        O, L = A.packed_attention(q, k, v, cu, causal, 0.5)
        k2, v2 = k.copy(), v.copy()
        k2[:20] += 3.0
        v2[45:] -= 5.0
        O2, L2 = A.packed_attention(q, k2, v2, cu, causal, 0.5)
        assert np.array_equal(O[20:45], O2[20:45])
        assert np.array_equal(L[:, 20:45], L2[:, 20:45])


def test_causal_mask_ignores_future_keys():
    cu = (0, 64)
    H, D = 2, 4
    q, k, v = _rand((64, H, D), 25), _rand((64, H, D), 26), _rand((64, H, D), 27)
    O, L = A.packed_attention(q, k, v, cu, True, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[40:] = 7.0
    v2[40:] = -7.0
    O2, L2 = A.packed_attention(q, k2, v2, cu, True, 0.5)
    assert np.array_equal(O[:40], O2[:40])
    assert np.array_equal(L[:, :40], L2[:, :40])
    assert not np.array_equal(O[40:], O2[40:])


def test_sampled_rows_equal_full_oracle():
    w = inputs.custom((0, 100, 300, 333), H=8, Hkv=2, D=16, dtype="bf16", causal=True)
    q, k, v = inputs.make_qkv(w)
    O, L = A.packed_attention(q, k, v, w.cu_seqlens, True, w.scale)
    rows = np.array([0, 1, 99, 100, 150, 299, 300, 332])
    Os, Ls = A.attention_at_rows(q, k, v, w.cu_seqlens, rows, True, w.scale, threads=2, batch=3)
    assert np.abs(Os - O[rows]).max() < 1e-13
    assert np.abs(Ls - L[:, rows]).max() < 1e-13
    Ob, Lbd = A.packed_attention(q, k, v, w.cu_seqlens, False, w.scale)
    Os, Ls = A.attention_at_rows(q, k, v, w.cu_seqlens, rows, False, w.scale, threads=2, batch=3)
    assert np.abs(Os - Ob[rows]).max() < 1e-13
    assert np.abs(Ls - Lbd[:, rows]).max() < 1e-13
