"""The library's planner (C++) matches the oracle's independent restatement
bit for bit: chunk table, owners, rank offsets, local cu_seqlens, index map
and ring schedule."""

import numpy as np
import pytest

import inputs
from oracle import plan as P


def _compare(cpattn, cu, cp, mode, grid=None):
    ref = P.make_plan(cu, cp, mode, grid)
    got = cpattn.cpattn_plan(cu, cp, mode, grid)
    info = got.info()
    assert info["total_tokens"] == ref.T
    assert info["n_chunks"] == len(ref.chunk_ranks)
    assert (info["split_h"], info["split_w"]) == (ref.split_h, ref.split_w)
    assert np.array_equal(got.chunk_offsets(), ref.chunk_offsets)
    assert np.array_equal(got.chunk_ranks(), ref.chunk_ranks)
    assert np.array_equal(got.rank_offsets(), ref.rank_offsets)
    assert np.array_equal(got.index_map(), ref.index_map)
    for r in range(cp):
        assert np.array_equal(got.local_cu_seqlens(r), ref.local_cu_seqlens[r])
    for causal in ((False,) if P.MODES.get(mode, mode) == P.GRID2D else (False, True)):
        kv, kind = got.ring_schedule(causal)
        rkv, rkind = P.ring_schedule(ref, causal)
        assert np.array_equal(kv, rkv) and np.array_equal(kind, rkind)


@pytest.mark.parametrize("name", ["tiny_packed_fp32", "dynamic_cp_microbatch", "long_video_200k_gqa",
                                  "video_latent_grid2d"])
def test_workload_plans_match_oracle(cpattn, name):
    w = inputs.workload(name)
    _compare(cpattn, w.cu_seqlens, w.cp, w.mode, w.grid)


@pytest.mark.slow
def test_million_token_plan_matches_oracle(cpattn):
    w = inputs.workload("single_seq_1m_gqa")
    _compare(cpattn, w.cu_seqlens, w.cp, w.mode)


@pytest.mark.parametrize("seed", range(6))
def test_random_plans_match_oracle(cpattn, seed):
    rng = np.random.default_rng(seed)
    for cp in (1, 2, 3, 4, 8):
        lens = rng.integers(2 * cp, 300, size=rng.integers(1, 7))
        cu = np.concatenate([[0], np.cumsum(lens)])
        _compare(cpattn, cu, cp, "zigzag")
        _compare(cpattn, cu, cp, "contiguous")
    for cp in (1, 2, 4, 6, 8):
        F, h, w = rng.integers(1, 4), rng.integers(4, 20), rng.integers(4, 20)
        try:
            ref = P.grid2d((0, F * h * w), cp, (F, h, w))
        except P.PlanError:
            with pytest.raises(cpattn.CpattnError):
                cpattn.cpattn_plan([0, F * h * w], cp, "grid2d", (F, h, w))
            continue
        _compare(cpattn, (0, F * h * w), cp, "grid2d", (F, h, w))


def _compare_mesh(cpattn, cu, u, r):
    ref = P.ulysses2d(cu, u, r)
    got = cpattn.cpattn_plan_2d(cu, u, r)
    info = got.info()
    assert (info["mode"], info["cp_size"], info["split_h"], info["split_w"]) == (P.ULYSSES2D, u * r, u, r)
    assert info["n_chunks"] == len(ref.chunk_ranks)
    assert np.array_equal(got.chunk_offsets(), ref.chunk_offsets)
    assert np.array_equal(got.chunk_ranks(), ref.chunk_ranks)
    assert np.array_equal(got.rank_offsets(), ref.rank_offsets)
    assert np.array_equal(got.index_map(), ref.index_map)
    assert np.array_equal(got.a2a_map(), P.a2a_map(ref))
    for g in range(u * r):
        assert np.array_equal(got.local_cu_seqlens(g), ref.local_cu_seqlens[g])
    for causal in (False, True):
        kv, kind = got.ring_schedule(causal)
        rkv, rkind = P.ring_schedule(ref, causal)
        assert np.array_equal(kv, rkv) and np.array_equal(kind, rkind)


@pytest.mark.parametrize("seed", range(4))
def test_ulysses_ring_mesh_plans_match_oracle(cpattn, seed):
    rng = np.random.default_rng(50 + seed)
    for u, r in ((1, 1), (1, 4), (2, 1), (2, 2), (4, 2), (3, 3), (8, 1)):
        lens = rng.integers(2 * r, 400, size=rng.integers(1, 6))
        cu = np.concatenate([[0], np.cumsum(lens)])
        _compare_mesh(cpattn, cu, u, r)


def test_long_video_as_the_4x2_mesh_matches_oracle(cpattn):
    w = inputs.workload("long_video_200k_gqa")
    _compare_mesh(cpattn, w.cu_seqlens, 4, 2)


def test_mesh_plan_errors(cpattn):
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan_2d((0, 3), 1, 2)        # a sequence shorter than 2*ring
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan_2d((0, 8), 5, 2)        # ring shards of 4 tokens for 5 Ulysses ranks
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan((0, 64), 4, "ulysses2d")  # only cpattn_plan_2d builds mesh plans
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan((0, 64), 4, "zigzag").a2a_map()


@pytest.mark.parametrize("seed", range(4))
def test_paired_plans_match_oracle(cpattn, seed):
    from oracle import teacher_forcing as TF
    rng = np.random.default_rng(80 + seed)
    for cp in (1, 2, 4):
        N = cp * int(rng.integers(1, 4))
        lens = 2 * rng.integers(N, 200, size=rng.integers(1, 4))
        cu = np.concatenate([[0], np.cumsum(lens)])
        ref = TF.paired_plan(cu, cp, N)
        got = cpattn.cpattn_plan_paired(cu, cp, N)
        info = got.info()
        assert (info["mode"], info["split_h"], info["split_w"]) == (TF.PAIRED, cp, 1)
        assert np.array_equal(got.chunk_offsets(), ref.chunk_offsets)
        assert np.array_equal(got.chunk_ranks(), ref.chunk_ranks)
        assert np.array_equal(got.rank_offsets(), ref.rank_offsets)
        assert np.array_equal(got.index_map(), ref.index_map)
        assert np.array_equal(got.a2a_map(), P.a2a_map(ref))
        for r in range(cp):
            assert np.array_equal(got.local_cu_seqlens(r), ref.local_cu_seqlens[r])
        kv, kind = got.ring_schedule(True)
        rkv, rkind = P.ring_schedule(ref, True)
        assert np.array_equal(kv, rkv) and np.array_equal(kind, rkind)
        assert got.allowed_pairs() == TF.allowed_pairs(cu, N)
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan_paired((0, 41), 1, 2)       # odd length
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan_paired((0, 40), 3, 4)       # chunks not a multiple of cp


def test_allowed_pairs_of_standard_plans(cpattn):
    cu = (0, 10, 30)
    pl = cpattn.cpattn_plan(cu, 2, "zigzag")
    assert pl.allowed_pairs(True) == 55 + 210 and pl.allowed_pairs(False) == 100 + 400
