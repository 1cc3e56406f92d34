"""Pins for the oracle's context-parallel planner: the pages' worked examples,
closed forms and permutation/balance invariants.  CPU only."""

import json
import os

import numpy as np
import pytest

import inputs
from oracle import plan as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_mmsp_worked_example_contiguous():
    g = _golden("mmsp_worked_example.json")
    cu = np.concatenate([[0], np.cumsum(g["segments"])])
    plan = P.contiguous(cu, g["cp"])
    for r in range(g["cp"]):
        assert plan.rank_offsets[r + 1] - plan.rank_offsets[r] == g["rank_tokens"][r]
        lc = plan.local_cu_seqlens[r]
        pieces = [int(x) for x in np.diff(lc) if x > 0]
        assert pieces == g["rank_segments"][r]


def test_optimal_split_table():
    g = _golden("optimal_split.json")
    for cp, pair in g["closest_square_pairs"].items():
        assert list(P.optimal_split(int(cp))) == pair
    e = g["latent_45x80_cp8"]
    plan = P.grid2d((0, 16 * 45 * 80), 8, (16, 45, 80))
    assert (plan.split_h, plan.split_w) == (e["split_h"], e["split_w"])
    assert P.split_sizes(45, 2) == e["h_pieces"]
    assert P.split_sizes(80, 4) == e["w_pieces"]


def test_grid_orientation_follows_larger_side():
    assert (P.grid2d((0, 80 * 45), 8, (1, 80, 45)).split_h,) == (4,)
    p = P.grid2d((0, 36), 2, (1, 6, 6))
    assert (p.split_h, p.split_w) == (1, 2)
    with pytest.raises(P.PlanError):
        P.split_sizes(9, 4)  # ceil(9/4)=3 gives only three pieces


def test_zigzag_chunk_sizes_uneven():
    sizes = P.zigzag_chunk_sizes(200996, 8)
    assert sizes == [12563] * 4 + [12562] * 12
    assert sum(sizes) == 200996


def _assert_permutation(plan):
    assert np.array_equal(np.sort(plan.index_map), np.arange(plan.T))
    assert plan.rank_offsets[0] == 0 and plan.rank_offsets[-1] == plan.T


def test_zigzag_rank_owns_chunk_pair():
    cu = (0, 64, 264, 520)
    plan = P.zigzag(cu, 2)
    _assert_permutation(plan)
    C = 4
    assert plan.chunk_offsets.tolist() == [0, 16, 32, 48, 64, 114, 164, 214, 264, 328, 392, 456, 520]
    assert plan.chunk_ranks.tolist() == [0, 1, 1, 0] * 3
    for r in range(2):
        rows = P.rank_rows(plan, r).tolist()
        exp = []
        for s in range(3):
            for j in (r, C - 1 - r):
                a = plan.chunk_offsets[s * C + j]
                b = plan.chunk_offsets[s * C + j + 1]
                exp.extend(range(a, b))
        assert rows == exp
    assert plan.local_cu_seqlens.tolist() == [[0, 32, 132, 260], [0, 32, 132, 260]]


@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_zigzag_causal_work_is_balanced(cp):
    """For C | L every rank owns c^2 (C-1) + c(c+1) allowed causal pairs."""
    C, c = 2 * cp, 24
    L = C * c
    cu = (0, L, 2 * L)
    plan = P.zigzag(cu, cp)
    for r in range(cp):
        rows = P.rank_rows(plan, r)
        pos = rows % L
        pairs = int((pos + 1).sum())  # each query sees pos+1 keys
        assert pairs == 2 * (c * c * (C - 1) + c * (c + 1))


def test_zigzag_workload_plans():
    w = inputs.workload("dynamic_cp_microbatch")
    plan = P.zigzag(w.cu_seqlens, w.cp)
    _assert_permutation(plan)
    lens = w.lengths()
    assert lens.sum() == 32768 and lens.min() >= 64 and lens.max() <= 16384
    assert np.all(lens % 8 == 0)
    assert np.all(np.diff(plan.rank_offsets) == 32768 // 4)


def test_zigzag_rejects_short_sequences_and_bad_cu():
    with pytest.raises(P.PlanError):
        P.zigzag((0, 3, 10), 2)
    with pytest.raises(P.PlanError):
        P.zigzag((1, 10), 1)
    with pytest.raises(P.PlanError):
        P.zigzag((0, 10, 10), 1)


def test_grid2d_shards_are_boxes():
    F, h, w = 3, 7, 10
    plan = P.grid2d((0, F * h * w), 4, (F, h, w))
    _assert_permutation(plan)
    assert (plan.split_h, plan.split_w) == (2, 2)
    for r in range(4):
        rows = P.rank_rows(plan, r)
        f, y, x = rows // (h * w), (rows // w) % h, rows % w
        ih, iw = divmod(r, 2)
        assert set(y) == set(range([0, 4][ih], [4, 7][ih]))
        assert set(x) == set(range([0, 5][iw], [5, 10][iw]))
        assert len(rows) == F * len(set(y)) * len(set(x))
        assert np.all(np.diff(f * h * w + y * w + x) > 0)  # (f, y, x) row-major order


def test_ring_schedule_visits_every_shard_once():
    for mode, cp in (("zigzag", 4), ("contiguous", 3)):
        plan = P.make_plan((0, 40, 96), cp, mode)
        kv, kind = P.ring_schedule(plan, True)
        for r in range(cp):
            assert sorted(kv[r].tolist()) == list(range(cp))
            assert kv[r, 0] == r and kind[r, 0] == P.DIAG
            for t in range(cp):
                assert kv[r, t] == (r - t) % cp


def test_zigzag_mask_kinds_agree_with_positions():
    """KV_HEAD: only the lower kv chunk is visible, to all q rows; Q_TAIL: only
    the upper q chunk sees anything, and it sees all kv rows."""
    cp, C = 4, 8
    L = 8 * 13 + 5
    cu = (0, L)
    plan = P.zigzag(cu, cp)
    kv, kind = P.ring_schedule(plan, True)
    off = plan.chunk_offsets
    for r in range(cp):
        for t in range(1, cp):
            k = kv[r, t]
            q_rows = P.rank_rows(plan, r)
            kv_rows = P.rank_rows(plan, k)
            vis = kv_rows[None, :] <= q_rows[:, None]
            nq_low = off[r + 1] - off[r]
            nk_low = off[k + 1] - off[k]
            if kind[r, t] == P.KV_HEAD:
                assert vis[:, :nk_low].all() and not vis[:, nk_low:].any()
            else:
                assert kind[r, t] == P.Q_TAIL
                assert not vis[:nq_low].any() and vis[nq_low:].all()


def test_contiguous_sizes():
    plan = P.contiguous((0, 5, 11), 4)
    assert np.diff(plan.rank_offsets).tolist() == [3, 3, 3, 2]
    with pytest.raises(P.PlanError):
        P.contiguous((0, 2), 3)


# ------------------------------------------------------- Ulysses x ring mesh

def test_mesh_with_one_ulysses_rank_is_the_zigzag_ring():
    for cu, r in (((0, 100, 357), 2), ((0, 64, 264, 520), 4), ((0, 9),  1)):
        z, m = P.zigzag(cu, r), P.ulysses2d(cu, 1, r)
        assert np.array_equal(z.index_map, m.index_map) and np.array_equal(z.rank_offsets, m.rank_offsets)


def test_mesh_with_one_ring_group_is_a_contiguous_split():
    for cu, u in (((0, 100, 357), 4), ((0, 777), 3)):
        c, m = P.contiguous(cu, u), P.ulysses2d(cu, u, 1)
        assert np.array_equal(m.index_map, np.arange(cu[-1])) and np.array_equal(c.rank_offsets, m.rank_offsets)


def test_longvila_4x2_mesh_layout():
    # 8-way SP over two nodes as a 4 x 2 mesh: ranks 0-3 (one node) share ring
    # shard 0, ranks 4-7 ring shard 1; the Ulysses groups split each shard evenly
    cu = (0, 1600)
    m = P.ulysses2d(cu, 4, 2)
    ring = P.zigzag(cu, 2)
    assert np.array_equal(m.rank_offsets, [0, 200, 400, 600, 800, 1000, 1200, 1400, 1600])
    assert np.array_equal(np.sort(m.index_map[:800]), np.sort(P.rank_rows(ring, 0)))
    kv, kind = P.ring_schedule(m, True)
    assert kv[5].tolist() == [5, 1, -1, -1, -1, -1, -1, -1]      # rank (i=1, j=1): its shard, then ring shard 0
    assert kind[5, :2].tolist() == [P.DIAG, P.KV_HEAD]


def test_a2a_map_is_the_head_regroup():
    cu, u = (0, 50, 123), 2
    m = P.ulysses2d(cu, u, 2)
    a2a = P.a2a_map(m)
    T, H, D = 123, 4, 3
    assert np.array_equal(np.sort(a2a), np.arange(u * T))
    x = np.arange(T * H * D).reshape(T, H, D)
    buf = x.reshape(T * u, (H // u) * D)[a2a].reshape(u, T, H // u, D)
    for i in range(u):
        assert np.array_equal(buf[i], x[m.index_map][:, i * (H // u):(i + 1) * (H // u)])


@pytest.mark.parametrize("causal", [True, False])
def test_mesh_ring_reproduces_packed_attention(causal):
    """Every rank (i, j) after the all-to-all: its head group's queries of ring
    shard j over the ring shards in ring order, merged exactly, equal the
    packed attention of those rows and heads."""
    from oracle import attention as A
    from oracle import merge as M
    cu, u, r, H, Hkv, D = (0, 37, 130), 2, 2, 4, 2, 8
    rng = np.random.default_rng(1)
    q, k, v = rng.standard_normal((130, H, D)), rng.standard_normal((130, Hkv, D)), rng.standard_normal((130, Hkv, D))
    O, L = A.packed_attention(q, k, v, cu, causal, 0.4)
    m = P.ulysses2d(cu, u, r)
    kv, _ = P.ring_schedule(m, causal)
    ring_rows = [m.index_map[m.rank_offsets[j * u]:m.rank_offsets[(j + 1) * u]] for j in range(r)]
    for g in range(u * r):
        i, j = g % u, g // u
        hs, ks = slice(i * H // u, (i + 1) * H // u), slice(i * Hkv // u, (i + 1) * Hkv // u)
        parts = []
        for t in range(r):
            kr = kv[g, t] // u
            parts.append(A.block_attention(q[:, hs], k[:, ks], v[:, ks], cu, ring_rows[j], ring_rows[kr], causal, 0.4))
        Og, Lg = M.lse_merge([p_[0] for p_ in parts], [p_[1] for p_ in parts])
        np.testing.assert_allclose(Og, O[ring_rows[j]][:, hs], atol=1e-12)
        np.testing.assert_allclose(Lg, L[hs][:, ring_rows[j]], atol=1e-12)
