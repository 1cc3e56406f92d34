"""Pins for the oracle's LSE merge, loss normalisation and FLOP count.  CPU only."""

import math

import numpy as np

import inputs
from oracle import attention as A
from oracle import flops as F
from oracle import loss as LN
from oracle import merge as M


def _parts(n, R=5, H=2, D=3, seed=0):
    rng = np.random.default_rng(seed)
    return ([rng.standard_normal((R, H, D)) for _ in range(n)],
            [rng.standard_normal((H, R)) * 3 for _ in range(n)])


def test_merge_of_equal_lse_is_average_plus_ln2():
    o, l = _parts(2)
    l[1] = l[0].copy()
    O, L = M.lse_merge(o, l)
    assert np.abs(L - (l[0] + math.log(2))).max() < 1e-14
    assert np.abs(O - (o[0] + o[1]) / 2).max() < 1e-14


def test_merge_weights_by_exp_lse():
    o, l = _parts(3, seed=1)
    O, L = M.lse_merge(o, l)
    w = [np.exp(x) for x in l]
    Z = sum(w)
    assert np.abs(L - np.log(Z)).max() < 1e-13
    ref = sum(wi.T[:, :, None] * oi for wi, oi in zip(w, o)) / Z.T[:, :, None]
    assert np.abs(O - ref).max() < 1e-13


def test_merge_is_commutative_and_associative():
    o, l = _parts(4, seed=2)
    O, L = M.lse_merge(o, l)
    O2, L2 = M.lse_merge(o[::-1], l[::-1])
    assert np.abs(O - O2).max() < 1e-14 and np.abs(L - L2).max() < 1e-14
    Oab, Lab = M.lse_merge(o[:2], l[:2])
    Ocd, Lcd = M.lse_merge(o[2:], l[2:])
    O3, L3 = M.lse_merge([Oab, Ocd], [Lab, Lcd])
    assert np.abs(O - O3).max() < 1e-14 and np.abs(L - L3).max() < 1e-14


def test_merge_ignores_empty_partials():
    o, l = _parts(2, seed=3)
    l[1][:] = -np.inf
    o[1][:] = 123.0
    O, L = M.lse_merge(o, l)
    assert np.array_equal(L, l[0])
    assert np.abs(O - o[0]).max() < 1e-15
    l[0][:] = -np.inf
    O, L = M.lse_merge(o, l)
    assert np.all(L == -np.inf) and np.all(O == 0)


def test_merge_of_halves_equals_attention_over_union():
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((30, 2, 4)), rng.standard_normal((30, 2, 4)), rng.standard_normal((30, 2, 4))
    cu = (0, 30)
    O, L = A.packed_attention(q, k, v, cu, False, 0.7)
    a = A.block_attention(q, k, v, cu, np.arange(30), np.arange(0, 11), False, 0.7)
    b = A.block_attention(q, k, v, cu, np.arange(30), np.arange(11, 30), False, 0.7)
    Om, Lm = M.lse_merge([a[0], b[0]], [a[1], b[1]])
    assert np.abs(Om - O).max() < 1e-13 and np.abs(Lm - L).max() < 1e-13


def test_loss_norm_closed_form():
    loss = np.array([1.0, 2.0, 4.0, 8.0], dtype=np.float32)
    valid = np.array([1, 0, 1, 1], dtype=np.uint8)
    val, cnt = LN.token_loss_norm(loss, valid)
    assert cnt == 3 and val == (1 + 4 + 8) / 3
    val, cnt = LN.token_loss_norm(loss, np.ones(4, np.uint8))
    assert cnt == 4 and val == 15 / 4
    val, cnt = LN.token_loss_norm(loss, np.zeros(4, np.uint8))
    assert cnt == 0 and val == 0.0


def test_loss_norm_on_microbatch_workload():
    w = inputs.workload("dynamic_cp_microbatch")
    loss, valid = inputs.make_loss_inputs(w)
    val, cnt = LN.token_loss_norm(loss.numpy(), valid.numpy())
    assert cnt == w.T - 3276
    assert abs(val - loss.numpy().astype(np.float64)[valid.numpy() == 1].mean()) < 1e-12


def test_flops_closed_form_and_brute_count():
    cu = (0, 64, 264, 520)
    assert F.fwd_flops(cu, 4, 64, True) == 4 * 64 * 4 * (64 * 65 // 2 + 200 * 201 // 2 + 256 * 257 // 2)
    assert F.fwd_flops(cu, 4, 64, True) == 56397824
    # brute count of allowed pairs from the dense mask definition
    seq, pos = A.seq_ids_and_positions(cu)
    for causal in (True, False):
        allowed = seq[:, None] == seq[None, :]
        if causal:
            allowed &= pos[None, :] <= pos[:, None]
        assert F.fwd_flops(cu, 3, 16, causal) == 4 * 16 * 3 * int(allowed.sum())
    assert F.fwd_flops((0, 200996), 32, 128, True) == 4 * 128 * 32 * 200996 * 200997 // 2
    assert F.fwd_flops((0, 57600), 24, 128, False) == 4 * 128 * 24 * 57600 ** 2
    # max_seqlen-based counting would overestimate a packed batch
    assert F.fwd_flops(cu, 4, 64, True) < 4 * 64 * 4 * 3 * (256 * 257 // 2)
