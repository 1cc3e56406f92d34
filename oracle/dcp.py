"""Dynamic context-parallel (Dynamic-CP) scheduling, restated for parity.

Test infrastructure only (see the package docstring).

"Speeding up Variable-Length Training with Dynamic Context Parallelism and
NVIDIA Megatron Core", data-scheduling section:

* Workload model: a sample's cost grows as O(S^2) (attention) plus O(S)
  (the per-token operators); its activation memory grows as O(S).  Here
  workload(S) = attn_coef * S(S+1)/2 + lin_coef * S (integers; with
  attn_coef = 4*D*H it is the causal attention FLOP count) and memory(S) = S
  tokens.
* Balance (Eq. 1-3): DP ranks finish together when
  W_i (m_i V + p - 1) is the same for every rank i (Eq. 1), so
  W_i = W_1 (m_1 V + p - 1) / (m_i V + p - 1) (Eq. 2), and the quotas must
  cover the batch: sum_i W_i m_i = total workload (Eq. 3).  Here m_i is rank
  i's micro-batch count, V the virtual pipeline stages and p the pipeline
  stage count.
* Two-objective heuristic: a sample whose workload exceeds the micro-batch
  quota gets a larger CP size (power of two up to max_cp); then memory leads:
  the lowest-compute samples are placed first to fill the buckets, and the
  remaining samples, in descending order, go one by one to the bucket that
  the same rule picks.

Readings (the page is prose): every micro-batch has the same quota
Q = ceil(total / n_micro) (Eq. 2-3 with the same micro-batch count on every
DP rank, as the runtime section constrains it); a sample's CP size is the
smallest power of two c <= max_cp with workload <= c*Q and S <= c*cap (else
max_cp); a micro-batch split over c GPUs puts workload/c on each, kept as the
integer load = workload * (max_cp / c); the n_micro lowest-workload samples
open one micro-batch each; every other sample (descending workload, ties by
index) joins the micro-batch with the least load after the placement among
those whose tokens stay within c*cap, else the least-loaded one (ties by
index); a micro-batch's CP size is the largest of its samples'.  The sweep's
knee and its choice near the knee are read in ``sweep``.

Pins (tests/test_oracle_dcp.py): Eq. 1-3 against a hand-solved case and a
linear solve of the equations; CP choice against exhaustive search;
placement invariants, the memory cap, Graham's list-scheduling bound against
a brute-force optimum on tiny batches, and a hand-worked schedule; the knee
on hand-made curves.  The heuristic rule itself is a reading of prose: beyond
those pins its parity is unpinned.
"""

from __future__ import annotations


def workload(S: int, attn_coef: int, lin_coef: int) -> int:
    return attn_coef * (S * (S + 1) // 2) + lin_coef * S


def quotas(m, V: int, p: int, total: float):
    """Per-rank micro-batch workload W_i from Eq. 2 and Eq. 3."""
    # Eq. 1: W_i (m_i V + p - 1) = K for all i;  Eq. 3: sum_i W_i m_i = total
    K = total / sum(mi / (mi * V + p - 1) for mi in m)
    return [K / (mi * V + p - 1) for mi in m]


def choose_cp(w: int, S: int, quota: int, cap: int, max_cp: int) -> int:
    c = 1
    while c <= max_cp:
        if w <= c * quota and S <= c * cap:
            return c
        c *= 2
    return max_cp


def schedule(lengths, n_buckets: int, max_cp: int, cap: int, attn_coef: int, lin_coef: int):
    """Returns (micro-batch of each sample, CP size of each sample, CP size of
    each micro-batch, workload of each micro-batch, tokens of each
    micro-batch).  A micro-batch's per-GPU load is its workload over its CP
    size; it is kept as the integer load = workload * (max_cp / cp)."""
    n = len(lengths)
    S = [int(x) for x in lengths]
    w = [workload(s, attn_coef, lin_coef) for s in S]
    total = sum(w)
    quota = -(-total // n_buckets)
    cp = [choose_cp(w[s], S[s], quota, cap, max_cp) for s in range(n)]
    bucket = [-1] * n
    b_work = [0] * n_buckets
    b_tok = [0] * n_buckets
    b_cp = [1] * n_buckets

    def load_after(b, s):
        c = max(b_cp[b], cp[s])
        return (b_work[b] + w[s]) * (max_cp // c), c

    def place(b, s):
        bucket[s] = b
        b_work[b] += w[s]
        b_tok[b] += S[s]
        b_cp[b] = max(b_cp[b], cp[s])

    # memory first: the lowest-workload samples open the micro-batches
    order_up = sorted(range(n), key=lambda s: (w[s], s))
    for b, s in enumerate(order_up[:n_buckets]):
        place(b, s)
    # the rest in descending workload, each to the least-loaded micro-batch
    # that stays within the per-GPU token cap
    for s in sorted(order_up[n_buckets:], key=lambda s: (-w[s], s)):
        best, best_load, fall, fall_load = -1, 0, -1, 0
        for b in range(n_buckets):
            ld, c = load_after(b, s)
            if fall < 0 or ld < fall_load:
                fall, fall_load = b, ld
            if b_tok[b] + S[s] <= c * cap and (best < 0 or ld < best_load):
                best, best_load = b, ld
        place(best if best >= 0 else fall, s)
    return bucket, cp, b_cp, b_work, b_tok


def loads(b_work, b_cp, max_cp: int):
    return [wk * (max_cp // c) for wk, c in zip(b_work, b_cp)]


def sweep(lengths, dp: int, pp: int, vpp: int, mult: int, max_cp: int, cap: int, attn_coef: int, lin_coef: int):
    """The micro-batch count grid of the solver's runtime section: every DP
    rank takes the same m, swept from pp to mult*pp.  budget(m) is the largest
    per-GPU micro-batch load (workload * max_cp / cp) of the schedule with
    dp*m micro-batches.

    Readings: the knee is the grid point farthest below the chord from the
    first to the last point of the budget curve, both axes scaled to [0, 1]
    (for integer exactness: the m minimising (m - m0)*Y + (budget - b_last)*X
    with X = m_last - m0, Y = b0 - b_last; the first m when X or Y <= 0).  In
    place of the simulator, the chosen m is the one in {knee-1, knee, knee+1}
    with the smallest Eq. 1 step time budget(m) * (m V + p - 1).  Ties go to the
    smaller m.  Returns (ms, budgets, knee m, chosen m)."""
    ms = list(range(pp, mult * pp + 1))
    budgets = []
    for m in ms:
        _, _, b_cp, b_work, _ = schedule(lengths, dp * m, max_cp, cap, attn_coef, lin_coef)
        budgets.append(max(loads(b_work, b_cp, max_cp)))
    k = knee(budgets)
    best = choose_near_knee(ms, budgets, k, vpp, pp)
    return ms, budgets, ms[k], ms[best]


def knee(budgets) -> int:
    """Index of the point farthest below the chord from the first to the last
    point, both axes scaled to [0, 1]; 0 when the curve does not fall."""
    X = len(budgets) - 1
    Y = budgets[0] - budgets[-1]
    if X <= 0 or Y <= 0:
        return 0
    score = [i * Y + (budgets[i] - budgets[-1]) * X for i in range(len(budgets))]
    return min(range(len(budgets)), key=lambda i: (score[i], i))


def choose_near_knee(ms, budgets, k: int, vpp: int, pp: int) -> int:
    """Index in {k-1, k, k+1} with the least Eq. 1 step time."""
    cand = [i for i in (k - 1, k, k + 1) if 0 <= i < len(ms)]
    return min(cand, key=lambda i: (budgets[i] * (ms[i] * vpp + pp - 1), i))
