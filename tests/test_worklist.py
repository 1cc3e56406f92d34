"""The work lists the planner hands the kernels, replayed on the CPU.

Each list is walked the way the kernel walks it (every tile against every
pair of its runs, the position mask only inside runs flagged for it) and the
(query, key) pairs it visits are counted; the counts must equal the mask's
plain definition, once per pair: same sequence and, when causal, key
position <= query position ("Scaling video training with parallelism",
section 2: blockwise attention over the KV blocks of the ring), or the
teacher-forcing mask for paired plans.  Also checked: every query (forward)
or key (backward) row lies in exactly one tile, tiles hold consecutive
positions of one sequence owned by one rank (whole calls on global rows:
query tiles cut from the sequence's end and owned by the rank of their last
row, KV tiles cut from its start and owned by the rank of their first key),
runs are in ring order (rank (r - t) mod cp at step t forward,
(k + t) mod cp backward), the per-tile piece counts the kernels loop over,
longest-first order, and the rank-local output rows of one ring step."""

import numpy as np
import pytest

from oracle import teacher_forcing as TF

# Kernel tile shapes: (rows per tile, keys or queries per piece, pieces per
# kernel tile).
FWD_TILES = {"bf16": (128, 64, 1), "fp32": (64, 32, 1)}
BWD_TILES = {"bf16": (128, 64, 1), "fp32": (32, 64, 1)}


def seq_pos(cu):
    cu = np.asarray(cu, dtype=np.int64)
    t = np.arange(cu[-1])
    seq = np.searchsorted(cu, t, side="right") - 1
    return seq, t - cu[seq]


def definition(cu, causal):
    """Dense [T, T] mask (query token, key token) from its definition."""
    seq, pos = seq_pos(cu)
    m = seq[:, None] == seq[None, :]
    if causal:
        m &= pos[None, :] <= pos[:, None]
    return m


def rank_maps(plan, gathered):
    """Buffer row -> token and token -> rank for zigzag / contiguous (global
    rows) and grid2d (gathered rank-major rows) plans; local row of a token."""
    idx = plan.index_map()
    ro = plan.rank_offsets()
    T = len(idx)
    rank_of_tok = np.empty(T, dtype=np.int64)
    local = np.empty(T, dtype=np.int64)
    for r in range(len(ro) - 1):
        rank_of_tok[idx[ro[r]:ro[r + 1]]] = r
        local[idx[ro[r]:ro[r + 1]]] = np.arange(ro[r + 1] - ro[r])
    tok_of_row = idx if gathered else np.arange(T)
    return tok_of_row, rank_of_tok, local


def replay(tiles, runs, tok_of_row, seq, pos, causal, tile_rows, piece, backward, rank_of_tok=None, cp=None,
           q_rank=None, step=None, local=None, gathered=False, per_tile=1):
    """Pair counts [query token, key token] of a work list, with the structural
    checks of every tile and run.  The positions a list carries are the
    tokens' positions in their sequence, except on gathered grid2d rows
    (bidirectional only), where they are the gathered rows."""
    T = len(seq)
    row_pos = np.arange(len(tok_of_row)) if gathered else pos[tok_of_row]
    packed = q_rank is None and not gathered and rank_of_tok is not None
    seq_len = np.bincount(seq)
    count = np.zeros((T, T), dtype=np.int32)
    seen = np.zeros(T, dtype=np.int32)
    assert (np.diff(tiles[:, 6]) <= 0).all(), "tiles are not longest-first"
    for row0, pos0, out0, rows, rb, re, pieces, rank in tiles:
        assert 1 <= rows <= tile_rows
        tt = tok_of_row[row0:row0 + rows]
        assert (seq[tt] == seq[tt[0]]).all() and (row_pos[row0:row0 + rows] == pos0 + np.arange(rows)).all()
        seen[tt] += 1
        if packed and not backward:
            # a whole forward call on global rows: query tiles are cut from the
            # sequence, ending at its last row, and owned by the rank of their
            # last row (they may hold the end of one chunk and the start of
            # the next)
            assert rank_of_tok[tt[-1]] == rank
            assert (seq_len[seq[tt[0]]] - (pos0 + rows)) % tile_rows == 0 and (rows == tile_rows or pos0 == 0)
        elif packed:
            # the backward's KV tiles: cut from the sequence's first row on,
            # owned by the rank of their first key
            assert rank_of_tok[tt[0]] == rank
            assert pos0 % tile_rows == 0 and (rows == tile_rows or pos0 + rows == seq_len[seq[tt[0]]])
        elif rank_of_tok is not None:
            assert (rank_of_tok[tt] == rank).all()
            if q_rank is not None:
                assert rank == (q_rank if not backward else (q_rank - step) % cp)
                if not backward:
                    assert (local[tt] == out0 + np.arange(rows)).all(), "partial output rows"
        steps, n_pieces = [], 0
        for krow0, kpos0, klen, masked in runs[rb:re]:
            assert klen >= 1
            ot = tok_of_row[krow0:krow0 + klen]
            assert (seq[ot] == seq[tt[0]]).all() and (row_pos[krow0:krow0 + klen] == kpos0 + np.arange(klen)).all()
            q_t, k_t = (ot, tt) if backward else (tt, ot)
            vis = pos[k_t][None, :] <= pos[q_t][:, None]
            if masked:
                assert causal, "a masked run in a bidirectional list"
            else:
                assert not causal or vis.all(), "an unmasked run holds a pair the mask forbids"
                vis = np.ones_like(vis)
            count[np.ix_(q_t, k_t)] += vis
            n_pieces += -(-klen // piece)
            if rank_of_tok is not None:
                other = rank_of_tok[ot]
                assert (other == other[0]).all(), "a run spans two ranks"
                t = (other[0] - rank) % cp if backward else (rank - other[0]) % cp
                steps.append(int(t))
                if q_rank is not None:
                    assert t == step
        assert steps == sorted(steps), "runs out of ring order"
        assert pieces == -(-n_pieces // per_tile)
    return count, seen


CASES = [
    ((0, 64, 264, 520), 2, "zigzag", None, True),
    ((0, 64, 264, 520), 2, "zigzag", None, False),
    ((0, 300, 557, 1200), 3, "zigzag", None, True),
    ((0, 300, 557, 1200), 4, "zigzag", None, True),
    ((0, 8, 40, 300), 2, "zigzag", None, True),
    ((0, 1000), 4, "zigzag", None, True),
    ((0, 300, 557, 1200), 3, "contiguous", None, True),
    ((0, 300, 557, 1200), 3, "contiguous", None, False),
    ((0, 2 * 9 * 20), 4, "grid2d", (2, 9, 20), False),
    ((0, 3 * 7 * 11), 6, "grid2d", (3, 7, 11), False),
]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("backward", [False, True], ids=["fwd", "bwd"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[2]}-cp{c[1]}-T{c[0][-1]}-{'causal' if c[4] else 'bidir'}")
def test_whole_call_visits_every_allowed_pair_once(cpattn, case, backward, dtype):
    cu, cp, mode, grid, causal = case
    plan = cpattn.cpattn_plan(cu, cp, mode, grid)
    tok_of_row, rank_of_tok, _ = rank_maps(plan, mode == "grid2d")
    seq, pos = seq_pos(cu)
    rows, piece, per = (BWD_TILES if backward else FWD_TILES)[dtype]
    tiles, runs = plan.worklist(backward, dtype, causal)
    count, seen = replay(tiles, runs, tok_of_row, seq, pos, causal, rows, piece, backward, rank_of_tok, cp,
                         gathered=(mode == "grid2d"), per_tile=per)
    assert (seen == 1).all()
    assert np.array_equal(count, definition(cu, causal).astype(np.int32))


@pytest.mark.parametrize("backward", [False, True], ids=["fwd", "bwd"])
@pytest.mark.parametrize("case", [CASES[2], CASES[7], CASES[8]], ids=["zigzag", "contiguous", "grid2d"])
def test_ring_steps_partition_the_pairs(cpattn, case, backward):
    cu, cp, mode, grid, causal = case
    plan = cpattn.cpattn_plan(cu, cp, mode, grid)
    tok_of_row, rank_of_tok, local = rank_maps(plan, mode == "grid2d")
    seq, pos = seq_pos(cu)
    rows, piece, per = (BWD_TILES if backward else FWD_TILES)["bf16"]
    total = np.zeros((len(seq), len(seq)), dtype=np.int32)
    for r in range(cp):
        for t in range(cp):
            tiles, runs = plan.worklist(backward, "bf16", causal, r, t)
            count, seen = replay(tiles, runs, tok_of_row, seq, pos, causal, rows, piece, backward, rank_of_tok, cp,
                                 q_rank=r, step=t, local=local, gathered=(mode == "grid2d"), per_tile=per)
            # forward: every query row of rank r once per step; backward: every key row of rank (r - t) mod cp
            owner = r if not backward else (r - t) % cp
            assert (seen[rank_of_tok == owner] == 1).all() and (seen[rank_of_tok != owner] == 0).all()
            if backward:
                assert (count[rank_of_tok != r, :] == 0).all()
            total += count
    assert np.array_equal(total, definition(cu, causal).astype(np.int32))


@pytest.mark.parametrize("kind", ["mesh", "paired"])
def test_head_sharded_lists_cover_every_group(cpattn, kind):
    if kind == "mesh":
        cu, u = (0, 300, 557, 1200), 2
        plan = cpattn.cpattn_plan_2d(cu, u, 2)
        want = definition(cu, True)
    else:
        cu, u, N = (0, 96, 256), 4, 8
        plan = cpattn.cpattn_plan_paired(cu, u, N)
        want = TF.allowed(cu, N)
    T = cu[-1]
    idx = plan.index_map()
    seq, pos = seq_pos(cu)
    tiles, runs = plan.worklist(False, "bf16", True)
    tok_of_row = idx[np.arange(u * T) % T]
    group = np.arange(u * T) // T
    for row0, _, _, rows, rb, re, _, _ in tiles:
        g = group[row0]
        assert (group[row0:row0 + rows] == g).all()
        for krow0, _, klen, masked in runs[rb:re]:
            assert (group[krow0:krow0 + klen] == g).all(), "a run reads another head group's rows"
            if kind == "paired":
                assert masked == 0
    # paired lists carry no position mask (every run is fully visible under the
    # teacher-forcing mask), so they are replayed as unmasked lists
    count, seen = replay(tiles, runs, tok_of_row, seq, pos, kind == "mesh", 128, 64, False, per_tile=1)
    assert (seen == u).all()
    assert np.array_equal(count, u * want.astype(np.int32))


def test_worklist_rejects_what_the_calls_reject(cpattn):
    g = cpattn.cpattn_plan([0, 2 * 9 * 20], 4, "grid2d", (2, 9, 20))
    with pytest.raises(cpattn.CpattnError):
        g.worklist(False, "bf16", True)            # causal grid2d
    z = cpattn.cpattn_plan([0, 520], 2, "zigzag")
    with pytest.raises(cpattn.CpattnError):
        z.worklist(False, "bf16", True, 2, 0)      # rank out of range
    with pytest.raises(cpattn.CpattnError):
        z.worklist(True, "bf16", True, 0, 2)       # step out of range
    m = cpattn.cpattn_plan_2d([0, 300, 557, 1200], 2, 2)
    with pytest.raises(cpattn.CpattnError):
        m.worklist(True, "bf16", True)             # no backward on mesh plans
    p = cpattn.cpattn_plan_paired([0, 96, 256], 4, 8)
    with pytest.raises(cpattn.CpattnError):
        p.worklist(False, "bf16", False)           # the teacher-forcing mask needs causal


@pytest.mark.parametrize("seed", range(4))
def test_random_layouts(cpattn, seed):
    """Seeded random lengths, CP sizes, grids and meshes: every list visits
    every allowed pair once."""
    rng = np.random.default_rng(1000 + seed)
    for cp in (1, 2, 3, 4, 8):
        lens = rng.integers(2 * cp, 260, size=rng.integers(1, 6))
        cu = tuple(int(x) for x in np.concatenate([[0], np.cumsum(lens)]))
        seq, pos = seq_pos(cu)
        for mode in ("zigzag", "contiguous"):
            plan = cpattn.cpattn_plan(cu, cp, mode)
            tok_of_row, rank_of_tok, _ = rank_maps(plan, False)
            for causal in (True, False):
                for backward in (False, True):
                    dtype = ("bf16", "fp32")[int(rng.integers(0, 2))]
                    rows, piece, per = (BWD_TILES if backward else FWD_TILES)[dtype]
                    tiles, runs = plan.worklist(backward, dtype, causal)
                    count, seen = replay(tiles, runs, tok_of_row, seq, pos, causal, rows, piece, backward,
                                         rank_of_tok, cp, per_tile=per)
                    assert (seen == 1).all()
                    assert np.array_equal(count, definition(cu, causal).astype(np.int32)), (cu, cp, mode, causal)
    for cp in (2, 4, 6, 8):
        F, h, w = (int(x) for x in (rng.integers(1, 3), rng.integers(4, 16), rng.integers(4, 16)))
        try:
            plan = cpattn.cpattn_plan([0, F * h * w], cp, "grid2d", (F, h, w))
        except cpattn.CpattnError:
            continue                                  # a side too short for its pieces
        cu = (0, F * h * w)
        seq, pos = seq_pos(cu)
        tok_of_row, rank_of_tok, _ = rank_maps(plan, True)
        for backward in (False, True):
            rows, piece, per = (BWD_TILES if backward else FWD_TILES)["bf16"]
            tiles, runs = plan.worklist(backward, "bf16", False)
            count, seen = replay(tiles, runs, tok_of_row, seq, pos, False, rows, piece, backward, rank_of_tok, cp,
                                 gathered=True, per_tile=per)
            assert (seen == 1).all() and np.array_equal(count, definition(cu, False).astype(np.int32))
    for u, r in ((2, 2), (4, 1), (1, 4), (2, 3)):
        lens = rng.integers(2 * r, 240, size=rng.integers(1, 5))
        cu = tuple(int(x) for x in np.concatenate([[0], np.cumsum(lens)]))
        plan = cpattn.cpattn_plan_2d(cu, u, r)
        T = cu[-1]
        seq, pos = seq_pos(cu)
        tok_of_row = plan.index_map()[np.arange(u * T) % T]
        tiles, runs = plan.worklist(False, "bf16", True)
        count, seen = replay(tiles, runs, tok_of_row, seq, pos, True, 128, 64, False, per_tile=1)
        assert (seen == u).all() and np.array_equal(count, u * definition(cu, True).astype(np.int32)), (cu, u, r)
