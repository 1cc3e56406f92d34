"""Pins of the teacher-forcing oracle (clean/noisy pairs, "Scaling video
training with parallelism", section 4, LongLive-2.0 balanced SP)."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import plan as P
from oracle import teacher_forcing as TF


def test_mask_hand_worked():
    # one sample of 8 tokens, N = 2: clean chunks {0,1}, {2,3}; noisy {4,5}, {6,7}
    want = np.array([
        [1, 1, 0, 0, 0, 0, 0, 0],   # clean chunk 0: clean chunk 0
        [1, 1, 0, 0, 0, 0, 0, 0],
        [1, 1, 1, 1, 0, 0, 0, 0],   # clean chunk 1: clean chunks 0, 1
        [1, 1, 1, 1, 0, 0, 0, 0],
        [0, 0, 0, 0, 1, 1, 0, 0],   # noisy chunk 0: itself only
        [0, 0, 0, 0, 1, 1, 0, 0],
        [1, 1, 0, 0, 0, 0, 1, 1],   # noisy chunk 1: clean chunk 0 and itself
        [1, 1, 0, 0, 0, 0, 1, 1],
    ], dtype=bool)
    assert np.array_equal(TF.allowed((0, 8), 2), want)


def test_mask_keeps_samples_apart_and_counts_pairs():
    rng = np.random.default_rng(0)
    for _ in range(10):
        N = int(rng.integers(1, 5))
        lens = 2 * rng.integers(N, 30, size=rng.integers(1, 4))
        cu = np.concatenate([[0], np.cumsum(lens)])
        m = TF.allowed(cu, N)
        seq = np.searchsorted(cu, np.arange(cu[-1]), side="right") - 1
        assert not (m & (seq[:, None] != seq[None, :])).any()
        assert TF.allowed_pairs(cu, N) == int(m.sum())
        assert m.any(axis=1).all()       # every query sees at least its own chunk


def test_masked_attention_matches_torch_sdpa():
    cu, N, H, Hkv, D = (0, 20, 56), 3, 4, 2, 8
    rng = np.random.default_rng(1)
    q, k, v = rng.standard_normal((56, H, D)), rng.standard_normal((56, Hkv, D)), rng.standard_normal((56, Hkv, D))
    mask = TF.allowed(cu, N)
    O, L = TF.masked_attention(q, k, v, mask, 0.3)
    qt = torch.tensor(q).transpose(0, 1)
    kt = torch.tensor(k).repeat_interleave(H // Hkv, dim=1).transpose(0, 1)
    vt = torch.tensor(v).repeat_interleave(H // Hkv, dim=1).transpose(0, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.tensor(mask), scale=0.3)
    np.testing.assert_allclose(O, ref.transpose(0, 1).numpy(), atol=1e-12)
    s = 0.3 * torch.einsum("htd,hsd->hts", qt, kt).masked_fill(~torch.tensor(mask), float("-inf"))
    np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


def test_one_chunk_is_two_bidirectional_halves():
    cu, H, D = (0, 30), 2, 8
    rng = np.random.default_rng(2)
    q, k, v = rng.standard_normal((30, H, D)), rng.standard_normal((30, H, D)), rng.standard_normal((30, H, D))
    O, L = TF.masked_attention(q, k, v, TF.allowed(cu, 1), 0.5)
    O2, L2 = A.packed_attention(q, k, v, (0, 15, 30), False, 0.5)
    np.testing.assert_allclose(O, O2, atol=1e-12)
    np.testing.assert_allclose(L, L2, atol=1e-12)


def test_noisy_chunk_is_attention_over_its_key_set():
    cu, N, H, D = (0, 48), 4, 2, 8
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((48, H, D)), rng.standard_normal((48, H, D)), rng.standard_normal((48, H, D))
    O, L = TF.masked_attention(q, k, v, TF.allowed(cu, N), 0.4)
    for j in range(N):
        noisy = np.arange(24 + 6 * j, 24 + 6 * j + 6)
        keys = np.concatenate([np.arange(0, 6 * j), noisy])
        Ob, Lb = A.block_attention(q, k, v, (0, 48), noisy, keys, False, 0.4)
        np.testing.assert_allclose(O[noisy], Ob, atol=1e-12)
        np.testing.assert_allclose(L[:, noisy], Lb, atol=1e-12)


def test_paired_plan_gives_each_rank_its_time_chunks():
    cu, cp, N = (0, 40, 100), 2, 4
    pl = TF.paired_plan(cu, cp, N)
    seq, stream, chunk = TF.token_roles(cu, N)
    assert np.array_equal(np.sort(pl.index_map), np.arange(100))
    for r in range(cp):
        rows = P.rank_rows(pl, r)
        assert set(chunk[rows] // (N // cp)) == {r}
        # pair by pair: clean chunk then noisy chunk of the same time chunk
        for s in range(2):
            rs = rows[seq[rows] == s]
            keys = list(zip(chunk[rs], stream[rs]))
            assert keys == sorted(keys)
    kv, kind = P.ring_schedule(pl, True)
    assert kv[:, 0].tolist() == [0, 1] and (kv[:, 1:] == -1).all()
    with pytest.raises(ValueError):
        TF.paired_plan((0, 41), 2, 4)     # odd length
    with pytest.raises(ValueError):
        TF.paired_plan((0, 40), 3, 4)     # N not a multiple of cp


def test_sampled_rows_equal_the_dense_mask_attention():
    cu, N, H, Hkv, D = (0, 20, 56), 3, 4, 2, 8
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((56, H, D)), rng.standard_normal((56, Hkv, D)), rng.standard_normal((56, Hkv, D))
    O, L = TF.masked_attention(q, k, v, TF.allowed(cu, N), 0.3)
    rows = np.array([0, 3, 9, 10, 19, 20, 30, 38, 47, 55])
    Or, Lr = TF.attention_at_rows(q, k, v, cu, N, rows, 0.3)
    np.testing.assert_allclose(Or, O[rows], atol=1e-12)
    np.testing.assert_allclose(Lr, L[:, rows], atol=1e-12)
