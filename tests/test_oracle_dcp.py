"""Pins of the Dynamic-CP scheduler oracle ("Speeding up Variable-Length
Training with Dynamic Context Parallelism and NVIDIA Megatron Core",
data-scheduling section, Eq. 1-3, and the runtime section's grid search)."""

import itertools

import numpy as np
import pytest

from oracle import dcp


# ------------------------------------------------------------------ Eq. 1-3

def test_quotas_hand_solved():
    # m = (1, 3), V = 1, p = 2: Eq. 1 gives 2 W1 = 4 W2, Eq. 3 W1 + 3 W2 = 100,
    # so 5 W2 = 100: W2 = 20, W1 = 40.
    assert dcp.quotas([1, 3], 1, 2, 100.0) == pytest.approx([40.0, 20.0], rel=1e-15)


@pytest.mark.parametrize("seed", range(5))
def test_quotas_solve_the_linear_system(seed):
    rng = np.random.default_rng(seed)
    dp = int(rng.integers(2, 9))
    m = rng.integers(1, 17, dp).tolist()
    V, p = int(rng.integers(1, 5)), int(rng.integers(1, 9))
    total = float(rng.uniform(1e6, 1e12))
    # rows: W_1 a_1 - W_i a_i = 0 (Eq. 1 against rank 1), sum_i m_i W_i = total (Eq. 3)
    a = [mi * V + p - 1 for mi in m]
    A = np.zeros((dp, dp))
    b = np.zeros(dp)
    for i in range(1, dp):
        A[i - 1, 0], A[i - 1, i] = a[0], -a[i]
    A[dp - 1, :] = m
    b[dp - 1] = total
    assert dcp.quotas(m, V, p, total) == pytest.approx(np.linalg.solve(A, b).tolist(), rel=1e-10)


def test_quotas_special_cases():
    # the same micro-batch count everywhere: the batch splits evenly
    assert dcp.quotas([4, 4, 4], 2, 4, 1200.0) == pytest.approx([100.0] * 3, rel=1e-15)
    # one stage, no virtual stages: every rank's whole share W_i m_i is total / dp
    w = dcp.quotas([1, 2, 5, 10], 1, 1, 400.0)
    assert [wi * mi for wi, mi in zip(w, [1, 2, 5, 10])] == pytest.approx([100.0] * 4, rel=1e-14)


# ----------------------------------------------------------- workload, CP size

def test_workload_is_the_causal_pair_count_plus_tokens():
    for S in (1, 2, 7, 100):
        pairs = sum(1 for i in range(S) for j in range(S) if j <= i)
        assert dcp.workload(S, 3, 5) == 3 * pairs + 5 * S


def test_choose_cp_is_the_smallest_feasible_power_of_two():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        max_cp = 2 ** int(rng.integers(0, 6))
        w, S = int(rng.integers(0, 10**6)), int(rng.integers(1, 5000))
        quota, cap = int(rng.integers(1, 10**5)), int(rng.integers(1, 2000))
        c = dcp.choose_cp(w, S, quota, cap, max_cp)
        feasible = [t for t in (2 ** e for e in range(11)) if t <= max_cp and w <= t * quota and S <= t * cap]
        assert c == (feasible[0] if feasible else max_cp)


# -------------------------------------------------------------- the schedule

def _check_invariants(lengths, n_micro, max_cp, cap, ac, lc, res):
    bucket, cp, b_cp, b_work, b_tok = res
    w = [dcp.workload(int(S), ac, lc) for S in lengths]
    assert sorted(set(bucket)) <= list(range(n_micro)) and -1 not in bucket
    for b in range(n_micro):
        members = [s for s in range(len(lengths)) if bucket[s] == b]
        assert b_work[b] == sum(w[s] for s in members)
        assert b_tok[b] == sum(int(lengths[s]) for s in members)
        assert b_cp[b] == max([cp[s] for s in members], default=1)
    assert sum(b_work) == sum(w)
    # the n_micro lowest-workload samples open distinct micro-batches
    low = sorted(range(len(lengths)), key=lambda s: (w[s], s))[:n_micro]
    assert len({bucket[s] for s in low}) == len(low)


@pytest.mark.parametrize("seed", range(6))
def test_schedule_invariants(seed):
    rng = np.random.default_rng(200 + seed)
    n = int(rng.integers(1, 150))
    lengths = np.clip(np.exp(rng.normal(np.log(512), 1.2, n)), 64, 16384).astype(int)
    n_micro = int(rng.integers(1, 40))
    max_cp, cap = 2 ** int(rng.integers(0, 4)), int(rng.integers(4096, 65536))
    ac, lc = 4 * 128 * 32, int(rng.integers(0, 10**5))
    res = dcp.schedule(lengths, n_micro, max_cp, cap, ac, lc)
    _check_invariants(lengths, n_micro, max_cp, cap, ac, lc, res)


def test_memory_cap_holds_when_there_is_room():
    rng = np.random.default_rng(7)
    lengths = rng.integers(64, 2048, 300)
    # room for every sample many times over: no micro-batch may exceed cp * cap
    for max_cp in (1, 4):
        _, _, b_cp, _, b_tok = dcp.schedule(lengths, 64, max_cp, 20000, 2, 0)
        assert all(t <= c * 20000 for t, c in zip(b_tok, b_cp))


@pytest.mark.parametrize("seed", range(8))
def test_graham_bound_against_brute_force_optimum(seed):
    """With one GPU per micro-batch and no memory limit the placement is list
    scheduling: each sample joins the least-loaded micro-batch, so the largest
    load is within (2 - 1/n_micro) of the best possible (Graham, 1966)."""
    rng = np.random.default_rng(300 + seed)
    n, nb = int(rng.integers(3, 9)), int(rng.integers(2, 4))
    lengths = rng.integers(1, 60, n)
    w = [dcp.workload(int(S), 2, 1) for S in lengths]
    opt = min(max(sum(w[s] for s in range(n) if a[s] == b) for b in range(nb))
              for a in itertools.product(range(nb), repeat=n))
    _, _, b_cp, b_work, _ = dcp.schedule(lengths, nb, 1, 10**9, 2, 1)
    got = max(dcp.loads(b_work, b_cp, 1))
    assert opt <= got <= (2 - 1 / nb) * opt + 1e-9
    assert got <= sum(w) / nb + max(w)


def test_hand_worked_schedule_memory_decides():
    # S = (6,1,1,1,1,1,1), workload S(S+1) (attn_coef 2), 2 micro-batches,
    # max_cp 2, cap 4 tokens.  Workloads (42,2,2,2,2,2,2), total 54, quota 27.
    # Sample 0: 42 > 27 at cp 1, fits at cp 2 (42 <= 54, 6 <= 8).  Samples 1, 2
    # open micro-batches 0, 1.  Sample 0: loads after 44 and 44, tie -> 0
    # (cp 2, 7 tokens).  Samples 3, 4, 5: micro-batch 1 at loads 8, 12, 16
    # (cp 1, so load = 2 * work) beats 46.  Sample 6: micro-batch 1 would hold
    # 5 > 4 tokens, so it joins micro-batch 0 (load 46, 8 <= 8 tokens).
    bucket, cp, b_cp, b_work, b_tok = dcp.schedule([6, 1, 1, 1, 1, 1, 1], 2, 2, 4, 2, 0)
    assert bucket == [0, 0, 1, 1, 1, 1, 0]
    assert cp == [2, 1, 1, 1, 1, 1, 1]
    assert (b_cp, b_work, b_tok) == ([2, 1], [46, 8], [8, 4])
    assert dcp.loads(b_work, b_cp, 2) == [46, 16]


def test_hand_worked_schedule_over_the_cap_falls_back():
    # S = (4,1,2,3,6), workload S(S+1): (20,2,6,12,42), total 82, 2 micro-batches,
    # quota 41, max_cp 2, cap 5.  Sample 4 needs cp 2.  Samples 1, 2 open the
    # micro-batches; sample 4 -> 0 (load 44 < 48); sample 0 fits neither
    # (11 > 10, 6 > 5 tokens), so it takes the least load after: 1 (52 < 64);
    # sample 3 -> 0 (load 56, 10 <= 10 tokens; micro-batch 1 would hold 9 > 5).
    bucket, cp, b_cp, b_work, b_tok = dcp.schedule([4, 1, 2, 3, 6], 2, 2, 5, 2, 0)
    assert bucket == [1, 0, 1, 0, 0]
    assert cp == [1, 1, 1, 1, 2]
    assert (b_cp, b_work, b_tok) == ([2, 1], [56, 26], [10, 6])


def test_more_micro_batches_than_samples():
    bucket, cp, b_cp, b_work, b_tok = dcp.schedule([5, 3], 4, 4, 100, 1, 0)
    assert sorted(bucket) == [0, 1] and b_work[2:] == [0, 0] and b_cp[2:] == [1, 1]
    assert dcp.schedule([], 3, 2, 10, 1, 0) == ([], [], [1, 1, 1], [0, 0, 0], [0, 0, 0])


# ------------------------------------------------------------------- the knee

def test_knee_on_hand_made_curves():
    # X = 4, Y = 100: scores 400, 180, 240, 320, 400 -> index 1
    assert dcp.knee([100, 20, 10, 5, 0]) == 1
    # a straight line has no knee: every score ties, the first point wins
    assert dcp.knee([40, 30, 20, 10, 0]) == 0
    assert dcp.knee([5, 5, 5]) == 0 and dcp.knee([1, 2, 3]) == 0 and dcp.knee([9]) == 0
    # near the knee the Eq. 1 step time budget * (mV + p - 1) decides:
    # m = 2, 3, 4 with V = 1, p = 2: 100*3, 70*4, 60*5 -> m = 3
    assert dcp.choose_near_knee([2, 3, 4, 5], [100, 70, 60, 59], 1, 1, 2) == 1


def test_sweep_picks_within_the_grid():
    rng = np.random.default_rng(11)
    lengths = np.clip(np.exp(rng.normal(np.log(512), 1.2, 120)), 64, 16384).astype(int)
    ms, budgets, k, best = dcp.sweep(lengths, 2, 2, 2, 4, 8, 16384, 4 * 128 * 32, 0)
    assert ms == list(range(2, 9)) and len(budgets) == len(ms)
    assert k in ms and abs(best - k) <= 1
