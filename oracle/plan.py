"""Context-parallel split planner, restated independently for plan parity.

Test infrastructure only (see the package docstring).  Integer-only.

Modes:

* ZIGZAG - each packed sequence of length L is cut into C = 2*cp contiguous
  chunks of sizes floor(L/C) + [j < L mod C]; virtual rank r owns chunks r and
  C-1-r of every sequence, in that order.  The pages name ZIGZAG-RINGATTN as
  the load-balanced ring split (LongVILA news article, Fig. 5 and Table 2);
  the pairing of chunk i with chunk 2cp-1-i is the one the workload fixes.
  Every sequence must have at least C tokens.
* GRID2D - one latent of F x h x w tokens, flattened (frame, row, column)
  row-major, is cut into split_h x split_w tiles (LongCat-Video
  context-parallel article, tensor split strategy): (split_h, split_w) is the
  factor pair of cp closest to square (get_optimal_split), the larger factor
  going to the larger spatial side and, on a tie, split_h <= split_w.  Each
  side is cut torch-split style into pieces of ceil(n/parts) with the
  remainder last; rank = ih*split_w + iw owns its tile across all frames.
* CONTIGUOUS - the packed T tokens are cut into cp contiguous ranges, the
  first T mod cp ranges one token longer (the token-level stage of LongVILA's
  two-stage MM-SP sharding, "Scaling video training with parallelism",
  section 3, Fig. 2).

* ULYSSES2D - the 2D-Attention mesh of u x r virtual ranks (LongVILA news
  article, 2D attention parallelism and Fig. 3 left: independent Ulysses
  (all-to-all) and Ring (P2P) groups, e.g. 8-way SP as a 4 x 2 mesh; USP and
  LoongTrain's head-context parallelism, "Scaling video training with
  parallelism", section 2).  Rank g = j*u + i (i the Ulysses index inside a
  ring group, j the ring index).  The ring dimension is the zigzag split over
  r (ring shard j = chunks j and 2r-1-j of every sequence); the u ranks of
  ring group j hold u contiguous pieces of ring shard j's local rows (sizes
  floor(T_j/u) + [i < T_j mod u]).  The all-to-all gives rank (i, j) every
  row of ring shard j for the query and KV heads of head group i (H/u and
  Hkv/u heads; "Ulysses ... when the number of heads supports the split",
  section 2).  Chunks are the maximal runs of consecutive global rows of one
  sequence owned by one rank.

Ring schedule: at step t, rank r computes with the KV shard of rank
(r - t) mod cp ("Scaling video training with parallelism", section 2, Ring
Attention: KV blocks circulate around the ring).  The mask kind records which
part of the pair can interact under a causal mask.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

ZIGZAG, GRID2D, CONTIGUOUS, ULYSSES2D, PAIRED = 0, 1, 2, 3, 4
MODES = {"zigzag": ZIGZAG, "grid2d": GRID2D, "contiguous": CONTIGUOUS, "ulysses2d": ULYSSES2D}

# mask kinds of a (q rank, ring step) pair
SKIP, FULL, DIAG, KV_HEAD, Q_TAIL = 0, 1, 2, 3, 4


class PlanError(ValueError):
    pass


@dataclass
class Plan:
    mode: int
    cp: int
    T: int
    n_seqs: int
    chunk_offsets: np.ndarray      # int64 [n_chunks+1]: global start of each chunk, then T
    chunk_ranks: np.ndarray        # int32 [n_chunks]
    rank_offsets: np.ndarray       # int64 [cp+1]: start of each rank in index_map
    local_cu_seqlens: np.ndarray   # int32 [cp, n_seqs+1]
    index_map: np.ndarray          # int64 [T]: rank-major local row -> global row
    split_h: int = 0
    split_w: int = 0


def optimal_split(cp: int):
    """Factor pair (a, b), a <= b, a*b = cp, with b - a smallest."""
    a = int(np.floor(np.sqrt(cp)))
    while a > 1 and cp % a:
        a -= 1
    return a, cp // a


def split_sizes(n: int, parts: int):
    """torch.split(ceil(n/parts)) piece sizes; error unless exactly ``parts``."""
    size = -(-n // parts)
    sizes = []
    left = n
    while left > 0:
        sizes.append(min(size, left))
        left -= size
    if len(sizes) != parts:
        raise PlanError(f"cannot cut {n} into {parts} pieces of {size}")
    return sizes


def zigzag_chunk_sizes(L: int, cp: int):
    C = 2 * cp
    base, rem = divmod(L, C)
    return [base + (1 if j < rem else 0) for j in range(C)]


def _check_cu(cu):
    cu = [int(c) for c in cu]
    if len(cu) < 2 or cu[0] != 0:
        raise PlanError("cu_seqlens must start at 0 and hold at least one sequence")
    for a, b in zip(cu[:-1], cu[1:]):
        if b <= a:
            raise PlanError("cu_seqlens must be strictly increasing")
    return cu


def _local_cu(index_map, rank_offsets, cu, cp):
    n = len(cu) - 1
    out = np.zeros((cp, n + 1), dtype=np.int32)
    bounds = np.asarray(cu, dtype=np.int64)
    for r in range(cp):
        rows = index_map[rank_offsets[r]:rank_offsets[r + 1]]
        seq = np.searchsorted(bounds, rows, side="right") - 1
        counts = np.bincount(seq, minlength=n)
        out[r, 1:] = np.cumsum(counts)
    return out


def zigzag(cu_seqlens, cp: int) -> Plan:
    cu = _check_cu(cu_seqlens)
    if cp < 1:
        raise PlanError("cp must be >= 1")
    C = 2 * cp
    n = len(cu) - 1
    offs, ranks = [], []
    per_rank = [[] for _ in range(cp)]
    for s in range(n):
        L = cu[s + 1] - cu[s]
        if L < C:
            raise PlanError(f"sequence {s} has {L} < 2*cp tokens")
        sizes = zigzag_chunk_sizes(L, cp)
        starts = [cu[s] + sum(sizes[:j]) for j in range(C)]
        for j in range(C):
            offs.append(starts[j])
            ranks.append(j if j < cp else C - 1 - j)
        for r in range(cp):
            for j in (r, C - 1 - r):
                per_rank[r].extend(range(starts[j], starts[j] + sizes[j]))
    offs.append(cu[-1])
    index_map = np.asarray([g for r in range(cp) for g in per_rank[r]], dtype=np.int64)
    rank_offsets = np.zeros(cp + 1, dtype=np.int64)
    rank_offsets[1:] = np.cumsum([len(p) for p in per_rank])
    return Plan(ZIGZAG, cp, cu[-1], n, np.asarray(offs, dtype=np.int64),
                np.asarray(ranks, dtype=np.int32), rank_offsets,
                _local_cu(index_map, rank_offsets, cu, cp), index_map)


def grid2d(cu_seqlens, cp: int, grid) -> Plan:
    cu = _check_cu(cu_seqlens)
    if cp < 1:
        raise PlanError("cp must be >= 1")
    if len(cu) != 2:
        raise PlanError("grid2d plans one latent (one sequence)")
    F, h, w = (int(x) for x in grid)
    if F < 1 or h < 1 or w < 1 or F * h * w != cu[-1]:
        raise PlanError("grid frames*height*width must equal T")
    a, b = optimal_split(cp)
    split_h, split_w = (b, a) if h > w else (a, b)
    hs = split_sizes(h, split_h)
    ws = split_sizes(w, split_w)
    h0 = np.concatenate([[0], np.cumsum(hs)])
    w0 = np.concatenate([[0], np.cumsum(ws)])
    per_rank = []
    for ih in range(split_h):
        for iw in range(split_w):
            rows = []
            for f in range(F):
                for y in range(h0[ih], h0[ih + 1]):
                    base = f * h * w + y * w
                    rows.extend(range(base + w0[iw], base + w0[iw + 1]))
            per_rank.append(rows)
    offs, ranks = [], []
    for f in range(F):
        for y in range(h):
            ih = int(np.searchsorted(h0, y, side="right") - 1)
            for iw in range(split_w):
                offs.append(f * h * w + y * w + int(w0[iw]))
                ranks.append(ih * split_w + iw)
    offs.append(cu[-1])
    index_map = np.asarray([g for r in range(cp) for g in per_rank[r]], dtype=np.int64)
    rank_offsets = np.zeros(cp + 1, dtype=np.int64)
    rank_offsets[1:] = np.cumsum([len(p) for p in per_rank])
    return Plan(GRID2D, cp, cu[-1], 1, np.asarray(offs, dtype=np.int64),
                np.asarray(ranks, dtype=np.int32), rank_offsets,
                _local_cu(index_map, rank_offsets, cu, cp), index_map, split_h, split_w)


def contiguous(cu_seqlens, cp: int) -> Plan:
    cu = _check_cu(cu_seqlens)
    if cp < 1:
        raise PlanError("cp must be >= 1")
    T = cu[-1]
    if T < cp:
        raise PlanError("fewer tokens than ranks")
    q, rem = divmod(T, cp)
    sizes = [q + (1 if r < rem else 0) for r in range(cp)]
    starts = [sum(sizes[:r]) for r in range(cp)]
    offs = np.asarray(starts + [T], dtype=np.int64)
    index_map = np.arange(T, dtype=np.int64)
    rank_offsets = offs.copy()
    return Plan(CONTIGUOUS, cp, T, len(cu) - 1, offs, np.arange(cp, dtype=np.int32),
                rank_offsets, _local_cu(index_map, rank_offsets, cu, cp), index_map)


def ulysses2d(cu_seqlens, u: int, r: int) -> Plan:
    cu = _check_cu(cu_seqlens)
    if u < 1 or r < 1:
        raise PlanError("ulysses and ring degrees must be >= 1")
    T = cu[-1]
    cp = u * r
    ring = zigzag(cu, r)
    per_rank = [None] * cp
    for j in range(r):
        rows = rank_rows(ring, j)
        if len(rows) < u:
            raise PlanError("a ring shard has fewer tokens than the Ulysses degree")
        q, rem = divmod(len(rows), u)
        start = 0
        for i in range(u):
            size = q + (1 if i < rem else 0)
            per_rank[j * u + i] = rows[start:start + size]
            start += size
    index_map = np.concatenate(per_rank).astype(np.int64)
    rank_offsets = np.zeros(cp + 1, dtype=np.int64)
    rank_offsets[1:] = np.cumsum([len(x) for x in per_rank])
    owner = np.empty(T, dtype=np.int64)
    for g in range(cp):
        owner[per_rank[g]] = g
    seq = np.searchsorted(np.asarray(cu), np.arange(T), side="right") - 1
    starts = [t for t in range(T) if t == 0 or owner[t] != owner[t - 1] or seq[t] != seq[t - 1]]
    offs = np.asarray(starts + [T], dtype=np.int64)
    return Plan(ULYSSES2D, cp, T, len(cu) - 1, offs, owner[starts].astype(np.int32), rank_offsets,
                _local_cu(index_map, rank_offsets, cu, cp), index_map, u, r)


def a2a_map(plan: Plan) -> np.ndarray:
    """The all-to-all as one row gather: viewing a [T, H, D] tensor as
    [T*u, H/u*D] rows (row t*u + i = token t's head group i), row
    i*T + p of the head-sharded buffer is token index_map[p]'s head group i;
    head group i's rows are the ring shards in ring order."""
    u = plan.split_h
    return np.concatenate([plan.index_map * u + i for i in range(u)]).astype(np.int64)


def make_plan(cu_seqlens, cp: int, mode, grid=None) -> Plan:
    mode = MODES.get(mode, mode)
    if mode == ZIGZAG:
        return zigzag(cu_seqlens, cp)
    if mode == GRID2D:
        return grid2d(cu_seqlens, cp, grid)
    if mode == CONTIGUOUS:
        return contiguous(cu_seqlens, cp)
    if mode == ULYSSES2D:
        u, r = int(grid[0]), int(grid[1])
        if u * r != cp:
            raise PlanError("cp must equal ulysses * ring")
        return ulysses2d(cu_seqlens, u, r)
    raise PlanError("unknown mode")


def ring_schedule(plan: Plan, causal: bool):
    """(kv_rank [cp,cp], mask_kind [cp,cp]) for (q rank r, step t).  For a
    ULYSSES2D plan the ring runs over the r ring groups after the all-to-all:
    rank (i, j) at step t < r works with ring shard (j - t) mod r of its head
    group, held by rank ((j - t) mod r)*u + i; steps t >= r are -1 / SKIP."""
    cp = plan.cp
    kv = np.zeros((cp, cp), dtype=np.int32)
    kind = np.zeros((cp, cp), dtype=np.int32)
    if plan.mode in (ULYSSES2D, PAIRED):   # PAIRED: a Ulysses layout with one ring group
        u, r = plan.split_h, plan.split_w
        for g in range(cp):
            i, j = g % u, g // u
            for t in range(cp):
                if t >= r:
                    kv[g, t], kind[g, t] = -1, SKIP
                    continue
                k = (j - t) % r
                kv[g, t] = k * u + i
                kind[g, t] = FULL if not causal else (DIAG if k == j else (KV_HEAD if k < j else Q_TAIL))
        return kv, kind
    for r in range(cp):
        for t in range(cp):
            k = (r - t) % cp
            kv[r, t] = k
            if not causal:
                kind[r, t] = FULL
            elif k == r:
                kind[r, t] = DIAG
            elif plan.mode == ZIGZAG:
                kind[r, t] = KV_HEAD if k < r else Q_TAIL
            elif plan.mode == CONTIGUOUS:
                kind[r, t] = FULL if k < r else SKIP
            else:
                raise PlanError("causal masks are not defined for grid2d plans")
    return kv, kind


def rank_rows(plan: Plan, r: int) -> np.ndarray:
    """Global rows of rank r in its local order."""
    return plan.index_map[plan.rank_offsets[r]:plan.rank_offsets[r + 1]]
