"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch each one.  The real oracle is restored after every case."""

import math

import numpy as np
import pytest
import torch

import oracle.attention as A
import oracle.merge as M
from tests.test_oracle_attention import brute_force


def _case():
    cu = (0, 6, 19)
    rng = np.random.default_rng(0)
    q, k, v = rng.standard_normal((19, 4, 4)), rng.standard_normal((19, 2, 4)), rng.standard_normal((19, 2, 4))
    return cu, q, k, v


def _err_vs_brute(causal=True, scale=0.4):
    cu, q, k, v = _case()
    O, L = A.packed_attention(q, k, v, cu, causal, scale)
    Ob, Lb = brute_force(q, k, v, cu, causal, scale)
    return max(np.abs(O - Ob).max(), np.abs(L - Lb).max())


def test_real_oracle_passes():
    assert _err_vs_brute() < 1e-12


def test_wrong_gqa_grouping_is_caught(monkeypatch):
    monkeypatch.setattr(A, "kv_head", lambda h, H, Hkv: h % Hkv)
    assert _err_vs_brute() > 1e-3


def test_dropped_scale_is_caught(monkeypatch):
    real = A._softmax_rows

    def planted(S, V):
        return real(S / 0.4, V)  # as if the scale had been left out

    monkeypatch.setattr(A, "_softmax_rows", planted)
    assert _err_vs_brute() > 1e-3


def test_off_by_one_causal_mask_is_caught(monkeypatch):
    monkeypatch.setattr(A, "causal_visible", lambda kpos, qpos: kpos < qpos)
    cu, q, k, v = _case()
    O, L = A.packed_attention(q, k, v, cu, True, 0.4)
    # the first token of each sequence now sees nothing: the closed form
    # O = v_first, lse = scale q.k_first no longer holds
    assert not np.array_equal(O[0, 0], v[0, 0])
    assert _err_vs_brute() > 1e-3 or not np.isfinite(_err_vs_brute())


def test_transposed_value_operand_is_caught():
    cu, q, k, v = _case()
    # a mistake that uses K in place of V in the P.V product
    O, _ = A.packed_attention(q, k, k, cu, True, 0.4)
    Ob, _ = brute_force(q, k, v, cu, True, 0.4)
    assert np.abs(O - Ob).max() > 1e-3


def test_unnormalised_merge_is_caught(monkeypatch):
    rng = np.random.default_rng(1)
    o = [rng.standard_normal((3, 1, 2)) for _ in range(2)]
    l = [rng.standard_normal((1, 3)) for _ in range(2)]
    good_O, good_L = M.lse_merge(o, l)
    w = [np.exp(x) for x in l]
    ref = (w[0].T[:, :, None] * o[0] + w[1].T[:, :, None] * o[1]) / (w[0] + w[1]).T[:, :, None]
    assert np.abs(good_O - ref).max() < 1e-13

    def planted(o_parts, lse_parts):
        lse = np.stack(lse_parts)
        Mx = lse.max(axis=0)
        coef = np.exp(lse - Mx)  # forgets to divide by the total weight
        return np.einsum("phr,prhd->rhd", coef, np.stack(o_parts)), Mx

    bad_O, _ = planted(o, l)
    assert np.abs(bad_O - ref).max() > 1e-3


def test_sdpa_pin_detects_missing_causal_mask():
    cu, q, k, v = _case()
    O_bidir, _ = A.packed_attention(q, k, v, cu, False, 0.4)
    a, b = 6, 19
    H, Hkv = 4, 2
    qt = torch.from_numpy(q[a:b]).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k[a:b]).permute(1, 0, 2).repeat_interleave(H // Hkv, 0)[None]
    vt = torch.from_numpy(v[a:b]).permute(1, 0, 2).repeat_interleave(H // Hkv, 0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.4)
    assert np.abs(O_bidir[a:b] - ref[0].permute(1, 0, 2).numpy()).max() > 1e-3
    assert math.isfinite(float(ref.abs().max()))


# ------------------------------------------------- Dynamic-CP scheduler slips

def _run_pin(fn):
    try:
        fn()
    except AssertionError:
        return False
    return True


def test_dcp_quota_sign_slip_is_caught(monkeypatch):
    import oracle.dcp as D
    from tests import test_oracle_dcp as T
    monkeypatch.setattr(D, "quotas", lambda m, V, p, total: [
        (total / sum(mi / (mi * V + p + 1) for mi in m)) / (mi * V + p + 1) for mi in m])  # p+1 for p-1
    assert not _run_pin(T.test_quotas_hand_solved)


def test_dcp_most_loaded_choice_is_caught(monkeypatch):
    import oracle.dcp as D
    from tests import test_oracle_dcp as T

    def planted(lengths, n_buckets, max_cp, cap, ac, lc):
        # one GPU per micro-batch, no memory limit (the Graham pin's setting),
        # but each later sample joins the MOST loaded micro-batch
        w = [D.workload(int(S), ac, lc) for S in lengths]
        order = sorted(range(len(w)), key=lambda s: (w[s], s))
        bucket, b_work = [-1] * len(w), [0] * n_buckets
        for i, s in enumerate(order[:n_buckets]):
            bucket[s] = i
            b_work[i] += w[s]
        for s in sorted(order[n_buckets:], key=lambda s: (-w[s], s)):
            b = max(range(n_buckets), key=lambda b: (b_work[b], -b))
            bucket[s] = b
            b_work[b] += w[s]
        return bucket, [1] * len(w), [1] * n_buckets, b_work, [0] * n_buckets

    monkeypatch.setattr(D, "schedule", planted)
    caught = [not _run_pin(lambda s=s: T.test_graham_bound_against_brute_force_optimum(s)) for s in range(8)]
    assert any(caught)


def test_dcp_dropped_memory_check_is_caught(monkeypatch):
    import oracle.dcp as D
    from tests import test_oracle_dcp as T
    real = D.schedule
    monkeypatch.setattr(D, "schedule", lambda lengths, nb, max_cp, cap, ac, lc:
                        real(lengths, nb, max_cp, 10**18, ac, lc))
    assert not _run_pin(T.test_hand_worked_schedule_memory_decides)


def test_dcp_knee_axis_swap_is_caught(monkeypatch):
    import oracle.dcp as D
    from tests import test_oracle_dcp as T

    def planted(budgets):  # the X and Y scalings swapped
        X, Y = len(budgets) - 1, budgets[0] - budgets[-1]
        if X <= 0 or Y <= 0:
            return 0
        score = [i * X + (budgets[i] - budgets[-1]) * Y for i in range(len(budgets))]
        return min(range(len(budgets)), key=lambda i: (score[i], i))

    monkeypatch.setattr(D, "knee", planted)
    assert not _run_pin(T.test_knee_on_hand_made_curves)


# ------------------------------------------------------------ backward slips

def _bwd_pins_hold():
    from tests import test_oracle_attention_bwd as T
    ok = True
    for case in T.CASES:
        ok &= _run_pin(lambda c=case: T.test_matches_torch_autograd(c))
    ok &= _run_pin(T.test_central_finite_differences)
    return ok


def _planted_block_grads(mistake):
    def grads(Qh, Kg, Vg, dOh, lse, delta, allowed, scale):
        S = scale * (Qh @ Kg.T)
        with np.errstate(invalid="ignore", over="ignore"):
            P = np.where(allowed, np.exp(S - lse[:, None]), 0.0)
        P[~np.isfinite(lse)] = 0.0
        dV = (P @ dOh) if mistake == "untransposed_dv" else P.T @ dOh
        dP = dOh @ Vg.T
        d = dP.sum(axis=1) if mistake == "unweighted_delta" else delta
        dS = P * (dP - d[:, None])
        dQ = scale * (dS @ Kg)
        dK = (dS.T @ Qh) if mistake == "unscaled_dk" else scale * (dS.T @ Qh)
        return dQ, dK, dV
    return grads


def test_real_backward_oracle_passes():
    assert _bwd_pins_hold()


@pytest.mark.parametrize("mistake", ["untransposed_dv", "unweighted_delta", "unscaled_dk"])
def test_backward_slips_are_caught(monkeypatch, mistake):
    import oracle.attention_bwd as Bw
    monkeypatch.setattr(Bw, "_block_grads", _planted_block_grads(mistake))
    assert not _bwd_pins_hold()
