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

Ring schedule: at step t, rank r computes with the KV shard of rank
(r - t) mod cp ("Scaling video training with parallelism", section 2, Ring
Attention: KV blocks circulate around the ring).  The mask kind records which
part of the pair can interact under a causal mask.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

ZIGZAG, GRID2D, CONTIGUOUS = 0, 1, 2
MODES = {"zigzag": ZIGZAG, "grid2d": GRID2D, "contiguous": CONTIGUOUS}

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


def make_plan(cu_seqlens, cp: int, mode, grid=None) -> Plan:
    mode = MODES.get(mode, mode)
    if mode == ZIGZAG:
        return zigzag(cu_seqlens, cp)
    if mode == GRID2D:
        return grid2d(cu_seqlens, cp, grid)
    if mode == CONTIGUOUS:
        return contiguous(cu_seqlens, cp)
    raise PlanError("unknown mode")


def ring_schedule(plan: Plan, causal: bool):
    """(kv_rank [cp,cp], mask_kind [cp,cp]) for (q rank r, step t)."""
    cp = plan.cp
    kv = np.zeros((cp, cp), dtype=np.int32)
    kind = np.zeros((cp, cp), dtype=np.int32)
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
