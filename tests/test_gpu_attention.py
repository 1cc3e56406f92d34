"""GPU parity of the packed forward (cpattn_fwd through the C ABI) against the
fp64 oracle, on small ragged cases and at the workloads' full sizes."""

import math
import os

import numpy as np
import pytest
import torch

import inputs
from oracle import attention as A
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    import context_attention_cpattn_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    m.build()
    m.lib()
    return m


SMALL = [
    # cu_seqlens, H, Hkv, D, causal, mode, cp
    ((0, 300, 557), 2, 2, 128, True, "zigzag", 2),            # ragged chunks, several tiles
    ((0, 300, 557), 2, 2, 128, False, "zigzag", 2),
    ((0, 4, 9, 300, 1111), 8, 2, 128, True, "zigzag", 2),     # GQA, 1-token chunks
    ((0, 1000, 1290), 4, 4, 64, True, "zigzag", 4),           # D = 64
    ((0, 700, 1500, 1501, 2600), 4, 1, 128, True, "contiguous", 3),  # ranks cut sequences
    ((0, 777), 2, 2, 128, True, "zigzag", 1),                 # cp = 1 is plain attention
    ((0, 2048), 2, 2, 128, True, "zigzag", 8),                # tiles exactly 128
]


@pytest.mark.parametrize("case", SMALL, ids=[f"case{i}" for i in range(len(SMALL))])
def test_bf16_small_cases_full_oracle(cp, case):
    cu, H, Hkv, D, causal, mode, cps = case
    w = inputs.custom(cu, H, Hkv, D, dtype="bf16", causal=causal, mode=mode, cp=cps)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(cu, cps, mode)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, cu, causal, w.scale)
    U.check(o, lse, O, L, "bf16", str(case))


def test_bf16_sharp_softmax_unscaled_inputs(cp):
    """N(0,1) inputs without the 1/sqrt(D) scaling: a peaked softmax whose
    output is far from the value mean, so a wrong O cannot hide under the
    absolute bound."""
    cu = (0, 513, 1400, 2048)
    w = inputs.custom(cu, 4, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=4, value_scale=1.0)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(cu, 4, "zigzag")
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, cu, True, w.scale)
    U.check(o, lse, O, L, "bf16", "sharp")


def test_bf16_grid2d_small(cp):
    F, h, wd = 3, 9, 20
    T = F * h * wd
    w = inputs.custom((0, T), 2, 2, 128, dtype="bf16", causal=False, mode="grid2d", cp=8, grid=(F, h, wd))
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan((0, T), 8, "grid2d", (F, h, wd))
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, (0, T), False, w.scale)
    U.check(o, lse, O, L, "bf16", "grid2d")


def test_fp32_tiny_packed_workload_full_oracle(cp):
    w = inputs.workload("tiny_packed_fp32")
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, w.cu_seqlens, True, w.scale)
    U.check(o, lse, O, L, "fp32", "tiny")


def test_fp32_bidirectional_and_gqa(cp):
    cu = (0, 100, 333)
    w = inputs.custom(cu, 4, 2, 128, dtype="fp32", causal=False, mode="zigzag", cp=2)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(cu, 2, "zigzag")
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, cu, False, w.scale)
    U.check(o, lse, O, L, "fp32", "fp32-gqa")


def test_repeated_calls_are_bitwise_stable(cp):
    w = inputs.workload("dynamic_cp_microbatch")
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode)
    o1, l1 = U.run_fwd(cp, plan, w, qd, kd, vd)
    o2, l2 = U.run_fwd(cp, plan, w, qd, kd, vd)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _sampled(cp, name, n_rows):
    w = inputs.workload(name)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    rows = U.boundary_rows(plan, n_rows, w.T, seed=w.seed)
    O, L = A.attention_at_rows(q, k, v, w.cu_seqlens, rows, w.causal, w.scale)
    stats = U.check(o[torch.from_numpy(rows).cuda()], lse[:, torch.from_numpy(rows).cuda()], O, L, "bf16", name)
    # every row written (the outputs started as NaN)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    return stats


def test_dynamic_cp_microbatch_full_size(cp):
    _sampled(cp, "dynamic_cp_microbatch", 2048)


def test_long_video_200k_gqa_full_size(cp):
    _sampled(cp, "long_video_200k_gqa", 512)


def test_video_latent_grid2d_full_size(cp):
    _sampled(cp, "video_latent_grid2d", 512)


def test_single_seq_1m_gqa_full_size(cp):
    _sampled(cp, "single_seq_1m_gqa", int(os.environ.get("CPATTN_1M_ROWS", "1024")))


def test_dynamic_cp_micro_batches_each_at_their_own_cp_size(cp):
    """A global batch packed by the Dynamic-CP scheduler: every micro-batch
    runs the packed forward at the CP size chosen for it and matches the
    oracle on all rows."""
    rng = np.random.default_rng(5)
    lengths = np.clip(np.exp(rng.normal(np.log(256), 1.0, 24)), 16, 2048).astype(np.int64)
    sched = cp.cpattn_dcp_schedule(lengths, 4, 4, 1024, 4 * 128 * 4, 0)
    sizes = set()
    for ids, cu, cps in cp.dcp_micro_batches(lengths, sched):
        if not len(ids):
            continue
        sizes.add(cps)
        w = inputs.custom(tuple(int(x) for x in cu), 4, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=cps)
        (q, k, v), (qd, kd, vd) = U.device_inputs(w)
        plan = cp.cpattn_plan(cu, cps, "zigzag")
        o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
        O, L = A.packed_attention(q, k, v, w.cu_seqlens, True, w.scale)
        U.check(o, lse, O, L, "bf16", f"dcp cp={cps}")
    assert len(sizes) > 1      # the batch really mixes CP sizes
