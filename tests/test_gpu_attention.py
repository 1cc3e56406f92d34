"""GPU parity of the packed forward (cpattn_fwd through the C ABI) against the
fp64 oracle, on small ragged cases and at the workloads' full sizes."""

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
    """The workload at full size through cpattn_fwd; the oracle on every
    chunk-boundary row plus ``n_rows`` seeded rows (all heads), or on every
    row when ``n_rows`` is None."""
    w = inputs.workload(name)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    rows = np.arange(w.T) if n_rows is None else U.boundary_rows(plan, n_rows, w.T, seed=w.seed)
    O, L = A.attention_at_rows(q, k, v, w.cu_seqlens, rows, w.causal, w.scale)
    idx = torch.from_numpy(rows).cuda()
    stats = U.check(o[idx], lse[:, idx], O, L, "bf16", name)
    # every row written (the outputs started as NaN)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    return stats


def test_dynamic_cp_microbatch_full_size_every_row(cp):
    """The 32K micro-batch against the oracle on every row and head."""
    _sampled(cp, "dynamic_cp_microbatch", None)


def test_long_video_200k_gqa_full_size(cp):
    _sampled(cp, "long_video_200k_gqa", 4096)


def test_video_latent_grid2d_full_size(cp):
    _sampled(cp, "video_latent_grid2d", 4096)


def test_single_seq_1m_gqa_full_size(cp):
    """4,096 seeded query rows (plus every chunk-boundary row) on all 32
    heads, the extent the 1M-token workload states."""
    _sampled(cp, "single_seq_1m_gqa", 4096)


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


MESH = [
    # cu_seqlens, H, Hkv, D, causal, ulysses, ring
    ((0, 300, 557), 4, 2, 128, True, 2, 1),
    ((0, 300, 557, 1200), 8, 4, 128, True, 2, 2),
    ((0, 1000, 1290), 4, 4, 64, False, 4, 1),
    ((0, 2048), 8, 8, 128, True, 4, 2),
    ((0, 33, 250, 251 + 260), 8, 2, 128, True, 2, 4),
]


@pytest.mark.parametrize("case", MESH, ids=[f"mesh{i}" for i in range(len(MESH))])
def test_ulysses_ring_mesh_forward(cp, case):
    """2D-Attention mesh: all-to-all head regroup, ring over the ring
    groups, reverse all-to-all; equals packed attention."""
    cu, H, Hkv, D, causal, u, r = case
    w = inputs.custom(cu, H, Hkv, D, dtype="bf16", causal=causal, mode="zigzag", cp=r)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan_2d(cu, u, r)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, cu, causal, w.scale)
    U.check(o, lse, O, L, "bf16", f"mesh {u}x{r}")


def test_ulysses_ring_mesh_fp32(cp):
    cu = (0, 100, 333)
    w = inputs.custom(cu, 4, 2, 64, dtype="fp32", causal=True, mode="zigzag", cp=2)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan_2d(cu, 2, 2)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, cu, True, w.scale)
    U.check(o, lse, O, L, "fp32", "mesh fp32")


def test_long_video_200k_as_the_4x2_mesh_full_size(cp):
    w = inputs.workload("long_video_200k_gqa")
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan_2d(w.cu_seqlens, 4, 2)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    rows = U.boundary_rows(plan, 512, w.T, seed=w.seed)
    O, L = A.attention_at_rows(q, k, v, w.cu_seqlens, rows, True, w.scale)
    idx = torch.from_numpy(rows).cuda()
    U.check(o[idx], lse[:, idx], O, L, "bf16", "long video 4x2 mesh")
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


def test_mesh_needs_heads_divisible_by_the_ulysses_degree(cp):
    plan = cp.cpattn_plan_2d((0, 256), 4, 1)
    qd = torch.zeros(256, 6, 128, dtype=torch.bfloat16, device="cuda")
    kd = torch.zeros(256, 2, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cp.cpattn_workspace_size(plan, 6, 2, 128, torch.bfloat16, True), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(cp.CpattnError) as e:
        cp.cpattn_fwd(plan, qd, kd, kd, torch.empty_like(qd), torch.empty(6, 256, device="cuda"), ws)
    assert e.value.status == cp.UNSUPPORTED


PAIRED = [
    # cu_seqlens, H, Hkv, D, cp, time chunks
    ((0, 40, 100), 4, 2, 128, 2, 4),
    ((0, 512), 8, 8, 128, 4, 8),
    ((0, 300, 700), 8, 4, 64, 2, 2),
    ((0, 2 * 4 * 300), 4, 4, 128, 4, 4),
]


@pytest.mark.parametrize("case", PAIRED, ids=[f"paired{i}" for i in range(len(PAIRED))])
def test_paired_teacher_forcing_forward(cp, case):
    """Clean/noisy pairs behind the Ulysses all-to-all with the
    teacher-forcing mask; equals the dense-mask oracle."""
    from oracle import teacher_forcing as TF
    cu, H, Hkv, D, cps, N = case
    w = inputs.custom(cu, H, Hkv, D, dtype="bf16", causal=True, mode="zigzag", cp=1)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan_paired(cu, cps, N)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = TF.masked_attention(q, k, v, TF.allowed(cu, N), w.scale)
    U.check(o, lse, O, L, "bf16", f"paired cp={cps} N={N}")


def test_paired_teacher_forcing_fp32(cp):
    from oracle import teacher_forcing as TF
    cu = (0, 64, 200)
    w = inputs.custom(cu, 4, 2, 64, dtype="fp32", causal=True, mode="zigzag", cp=1)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan_paired(cu, 2, 4)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = TF.masked_attention(q, k, v, TF.allowed(cu, 4), w.scale)
    U.check(o, lse, O, L, "fp32", "paired fp32")


def test_teacher_forcing_pairs_full_size(cp):
    from oracle import teacher_forcing as TF
    w = inputs.workload("teacher_forcing_pairs")
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan_paired(w.cu_seqlens, w.cp, w.grid[0])
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    rows = U.boundary_rows(plan, 384, w.T, seed=w.seed)
    O, L = TF.attention_at_rows(q, k, v, w.cu_seqlens, w.grid[0], rows, w.scale)
    idx = torch.from_numpy(rows).cuda()
    U.check(o[idx], lse[:, idx], O, L, "bf16", "teacher forcing pairs")
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()


def test_paired_plans_need_the_teacher_forcing_mask(cp):
    plan = cp.cpattn_plan_paired((0, 256), 2, 2)
    qd = torch.zeros(256, 2, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(cp.cpattn_workspace_size(plan, 2, 2, 128, torch.bfloat16, False), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(cp.CpattnError) as e:
        cp.cpattn_fwd(plan, qd, qd, qd, torch.empty_like(qd), torch.empty(2, 256, device="cuda"), ws, causal=False)
    assert e.value.status == cp.UNSUPPORTED
