"""The library's Dynamic-CP scheduler (host C++ behind the C ABI) against the
oracle: every integer output bit-exact, the Eq. 1-3 quotas to rounding.

Sample lengths follow the long-tailed distributions of the Dynamic-CP
article's Fig. 1-2 (lognormal, median 512, clipped to [64, 16384]) plus a
video-like mix of a few very long samples."""

import numpy as np
import pytest

from oracle import dcp as D

KEYS = ("sample_micro", "sample_cp", "micro_cp", "micro_work", "micro_tokens")


def _lengths(seed, n, kind="lognormal"):
    rng = np.random.default_rng(seed)
    if kind == "lognormal":
        return np.clip(np.exp(rng.normal(np.log(512), 1.2, n)), 64, 16384).astype(np.int64)
    if kind == "video":
        L = rng.integers(300, 4000, n)
        L[rng.choice(n, max(1, n // 20), replace=False)] = rng.integers(100_000, 400_000, max(1, n // 20))
        return L.astype(np.int64)
    return np.full(n, 777, dtype=np.int64)   # all equal: every tie rule in play


CASES = [
    # seed, n, kind, n_micro, max_cp, cap, attn_coef, lin_coef
    (0, 200, "lognormal", 16, 8, 8192, 4 * 128 * 32, 0),
    (1, 300, "lognormal", 64, 4, 16384, 4 * 128 * 32, 24 * 4096 * 128),
    (2, 50, "video", 8, 16, 131072, 4 * 128 * 24, 0),
    (3, 40, "equal", 6, 2, 2000, 1, 1),
    (4, 7, "lognormal", 20, 8, 4096, 4 * 128 * 32, 0),   # more micro-batches than samples
    (5, 500, "lognormal", 3, 1, 10**12, 2, 0),            # one GPU per micro-batch, no memory limit
    (6, 120, "lognormal", 24, 32, 512, 4 * 128 * 32, 0),  # tight cap: large CP sizes, fallbacks
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_schedule_bit_exact(cpattn, case):
    seed, n, kind, nm, max_cp, cap, ac, lc = case
    L = _lengths(seed, n, kind)
    got = cpattn.cpattn_dcp_schedule(L, nm, max_cp, cap, ac, lc)
    ref = D.schedule(L.tolist(), nm, max_cp, cap, ac, lc)
    for key, r in zip(KEYS, ref):
        assert np.array_equal(got[key], np.asarray(r, dtype=got[key].dtype)), key


@pytest.mark.parametrize("case", [(0, 200, "lognormal", 4, 2, 1, 8), (2, 60, "video", 2, 4, 2, 6),
                                  (3, 30, "equal", 3, 1, 1, 5)])
def test_sweep_bit_exact(cpattn, case):
    seed, n, kind, dp, pp, vpp, mult = case
    L = _lengths(seed, n, kind)
    got = cpattn.cpattn_dcp_sweep(L, dp, pp, vpp, mult, 8, 16384, 4 * 128 * 32, 0)
    ms, budgets, knee, best = D.sweep(L.tolist(), dp, pp, vpp, mult, 8, 16384, 4 * 128 * 32, 0)
    assert got["m"].tolist() == ms
    assert got["budgets"].tolist() == budgets
    assert (got["knee_m"], got["best_m"]) == (knee, best)


def test_quotas_match(cpattn):
    rng = np.random.default_rng(9)
    for _ in range(20):
        dp = int(rng.integers(1, 17))
        m = rng.integers(1, 33, dp).tolist()
        V, p, total = int(rng.integers(1, 5)), int(rng.integers(1, 9)), float(rng.uniform(0, 1e15))
        np.testing.assert_allclose(cpattn.cpattn_dcp_quotas(m, V, p, total), D.quotas(m, V, p, total), rtol=1e-13)


def test_empty_batch_and_plans_from_the_schedule(cpattn):
    got = cpattn.cpattn_dcp_schedule(np.zeros(0, np.int64), 3, 2, 10, 1, 0)
    assert got["micro_cp"].tolist() == [1, 1, 1] and got["micro_work"].tolist() == [0, 0, 0]
    # every micro-batch becomes a valid context-parallel plan of its own CP size
    L = _lengths(0, 60)
    sched = cpattn.cpattn_dcp_schedule(L, 8, 8, 4096, 4 * 128 * 32, 0)
    seen = []
    for ids, cu, cp in cpattn.dcp_micro_batches(L, sched):
        seen.extend(ids.tolist())
        if len(ids):
            plan = cpattn.cpattn_plan(cu, cp, "zigzag")
            assert plan.info()["total_tokens"] == int(L[ids].sum()) and plan.info()["cp_size"] == cp
    assert sorted(seen) == list(range(60))


@pytest.mark.parametrize("bad", [
    dict(max_cp=3), dict(max_cp=0), dict(max_cp=2048), dict(cap_tokens=0), dict(attn_coef=-1),
    dict(n_micro=0), dict(lengths=[5, 0, 3]), dict(lengths=[1 << 41]),
    dict(lengths=[1 << 24] * 4, attn_coef=1 << 20),   # total workload * max_cp beyond int64
])
def test_schedule_rejects_bad_arguments(cpattn, bad):
    args = dict(lengths=[10, 20, 30], n_micro=2, max_cp=4, cap_tokens=100, attn_coef=1, lin_coef=0)
    args.update(bad)
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_dcp_schedule(np.asarray(args["lengths"], np.int64), args["n_micro"], args["max_cp"],
                                   args["cap_tokens"], args["attn_coef"], args["lin_coef"])
    assert e.value.status == cpattn.INVALID_ARG


def test_quotas_and_sweep_reject_bad_arguments(cpattn):
    for m, V, p, total in (([0, 1], 1, 1, 1.0), ([1], 0, 1, 1.0), ([1], 1, 0, 1.0), ([1], 1, 1, -1.0),
                           ([1], 1, 1, float("nan"))):
        with pytest.raises(cpattn.CpattnError):
            cpattn.cpattn_dcp_quotas(m, V, p, total)
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_dcp_sweep([10, 20], 1, 0, 1, 2, 4, 100, 1)
