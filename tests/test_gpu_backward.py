"""GPU parity of the backward (cpattn_bwd and the per-step cpattn_block_bwd
through the C ABI) against the fp64 backward oracle.

Tolerances (derived from the arithmetic, written here): the bf16 kernel
rounds P and dS to bf16 (relative 2^-9 per element) before the tensor-core
products and reads the forward's bf16 O for delta, so each gradient carries
a relative error of a few 1e-3; the bound is a per-head relative RMS of
2e-2 on dQ, dK and dV plus a max-abs error of 5% of the tensor's largest
magnitude.  fp32: 1e-5 of the largest magnitude."""

import numpy as np
import pytest
import torch

import inputs
from oracle import attention_bwd as B
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

BWD_BF16_REL_RMS = 2e-2
BWD_BF16_MAX = 5e-2
BWD_FP32 = 1e-5


@pytest.fixture(scope="module")
def cp():
    import context_attention_cpattn_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    m.build()
    m.lib()
    return m


def check_grads(got, ref, dtype, where):
    stats = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        x = g.detach().to("cpu", torch.float64).numpy()
        assert np.isfinite(x).all(), f"{where}: non-finite {name}"
        err = np.abs(x - r)
        scale = max(np.abs(r).max(initial=0), 1e-30)
        stats[name + "_max_rel"] = float(err.max(initial=0) / scale)
        if dtype == "bf16":
            num = np.sqrt((err ** 2).sum(axis=(0, 2)))
            den = np.sqrt((r ** 2).sum(axis=(0, 2)))
            rel = num / np.maximum(den, 1e-30)
            stats[name + "_rel_rms"] = float(rel.max(initial=0))
            assert stats[name + "_rel_rms"] <= BWD_BF16_REL_RMS, (where, name, stats)
            assert stats[name + "_max_rel"] <= BWD_BF16_MAX, (where, name, stats)
        else:
            assert stats[name + "_max_rel"] <= BWD_FP32, (where, name, stats)
    print(where, stats)
    return stats


def _setup(cp, w):
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    do = inputs.make_dout(w)
    dod = do.cuda()
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    o, lse = U.run_fwd(cp, plan, w, qd, kd, vd)
    return (q, k, v, do), (qd, kd, vd, dod), plan, o, lse


def _run_bwd(cp, plan, w, qd, kd, vd, o, lse, dod):
    T, H, D = qd.shape
    ws = torch.empty(cp.cpattn_bwd_workspace_size(plan, H, kd.shape[1], D, qd.dtype, w.causal), dtype=torch.uint8,
                     device="cuda")
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    cp.cpattn_bwd(plan, qd, kd, vd, o, lse, dod, dq, dk, dv, ws, scale=w.scale, causal=w.causal)
    cp.cpattn_sync_status(ws)
    return dq, dk, dv


SMALL = [
    # cu_seqlens, H, Hkv, D, causal, mode, cp, grid
    ((0, 300, 557), 2, 2, 128, True, "zigzag", 2, None),
    ((0, 300, 557), 2, 2, 128, False, "zigzag", 2, None),
    ((0, 4, 9, 300, 1111), 8, 2, 128, True, "zigzag", 2, None),
    ((0, 700, 1500, 1501, 2600), 4, 1, 128, True, "contiguous", 3, None),
    ((0, 777), 2, 2, 128, True, "zigzag", 1, None),
    ((0, 2048), 2, 2, 128, True, "zigzag", 8, None),
    ((0, 3 * 9 * 20), 2, 2, 128, False, "grid2d", 8, (3, 9, 20)),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"case{i}" for i in range(len(SMALL))])
def test_bf16_backward_small_cases(cp, case):
    cu, H, Hkv, D, causal, mode, cps, grid = case
    w = inputs.custom(cu, H, Hkv, D, dtype="bf16", causal=causal, mode=mode, cp=cps, grid=grid)
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    got = _run_bwd(cp, plan, w, qd, kd, vd, o, lse, dod)
    ref = B.packed_attention_bwd(q, k, v, do, cu, causal, w.scale)
    check_grads(got, ref, "bf16", str(case))


def test_bf16_backward_sharp_softmax(cp):
    cu = (0, 513, 1400, 2048)
    w = inputs.custom(cu, 4, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=4, value_scale=1.0)
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    got = _run_bwd(cp, plan, w, qd, kd, vd, o, lse, dod)
    check_grads(got, B.packed_attention_bwd(q, k, v, do, cu, True, w.scale), "bf16", "sharp")


@pytest.mark.parametrize("case", [((0, 64, 264, 520), 4, 4, 64, True, "zigzag", 2),
                                  ((0, 100, 333), 4, 2, 128, False, "zigzag", 2),
                                  ((0, 90, 200), 2, 1, 64, True, "contiguous", 3)])
def test_fp32_backward(cp, case):
    cu, H, Hkv, D, causal, mode, cps = case
    w = inputs.custom(cu, H, Hkv, D, dtype="fp32", causal=causal, mode=mode, cp=cps)
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    got = _run_bwd(cp, plan, w, qd, kd, vd, o, lse, dod)
    check_grads(got, B.packed_attention_bwd(q, k, v, do, cu, causal, w.scale), "fp32", str(case))


@pytest.mark.parametrize("dtype,mode", [("bf16", "zigzag"), ("fp32", "zigzag"), ("bf16", "grid2d")])
def test_block_backward_ring_steps_add_up(cp, dtype, mode):
    if mode == "grid2d":
        cu, causal, grid = (0, 2 * 9 * 20), False, (2, 9, 20)
    else:
        cu, causal, grid = (0, 300, 557, 1200), True, None
    w = inputs.custom(cu, 8, 2, 128, dtype=dtype, causal=causal, mode=mode, cp=4, grid=grid)
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    T, H, D = qd.shape
    ws = torch.empty(cp.cpattn_bwd_workspace_size(plan, H, 2, D, qd.dtype, causal), dtype=torch.uint8,
                     device="cuda")
    dq = torch.zeros(T, H, D, dtype=torch.float32, device="cuda")
    dk = torch.zeros(T, 2, D, dtype=torch.float32, device="cuda")
    dv = torch.zeros(T, 2, D, dtype=torch.float32, device="cuda")
    for r in range(w.cp):
        for t in range(w.cp):
            cp.cpattn_block_bwd(plan, qd, kd, vd, o, lse, dod, dq, dk, dv, ws, r, t, scale=w.scale, causal=causal)
            cp.cpattn_sync_status(ws)
    ref = B.packed_attention_bwd(q, k, v, do, cu, causal, w.scale)
    check_grads((dq, dk, dv), ref, dtype, f"ring {dtype} {mode}")


def test_backward_rejects_unsupported_shapes(cp):
    plan = cp.cpattn_plan((0, 256), 2, "zigzag")
    with pytest.raises(cp.CpattnError) as e:
        cp.cpattn_bwd_workspace_size(plan, 2, 2, 64, torch.bfloat16, True)
    assert e.value.status == cp.UNSUPPORTED


def test_dynamic_cp_microbatch_backward_full_size(cp):
    """The 32K-token micro-batch (H = 32, D = 128, zigzag cp = 4): dQ at every
    chunk-boundary row plus 512 sampled rows from the oracle row by row; dK and
    dV of every sequence of at most 2048 tokens from the full oracle; and on
    every sequence and KV head the invariants sum_j dV_j = sum_i dO_i
    (relative to sqrt(sum_i |dO_i|^2)) and sum_j dK_j = 0 (relative to
    sqrt(sum_j |dK_j|^2))."""
    w = inputs.workload("dynamic_cp_microbatch")
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    dq, dk, dv = _run_bwd(cp, plan, w, qd, kd, vd, o, lse, dod)
    cu = np.asarray(w.cu_seqlens)
    rows = U.boundary_rows(plan, 512, w.T, seed=w.seed)
    ref_dq = B.dq_at_rows(q, k, v, do, cu, rows, True, w.scale)
    got_dq = dq[torch.from_numpy(rows).cuda()].to("cpu", torch.float64).numpy()
    err = got_dq - ref_dq
    rel = np.sqrt((err ** 2).sum(axis=(0, 2))) / np.sqrt((ref_dq ** 2).sum(axis=(0, 2)))
    assert rel.max() <= BWD_BF16_REL_RMS, rel.max()
    assert np.abs(err).max() <= BWD_BF16_MAX * np.abs(ref_dq).max()
    dk64 = dk.to("cpu", torch.float64).numpy()
    dv64 = dv.to("cpu", torch.float64).numpy()
    do64 = do.to(torch.float64).numpy()
    short = [s for s in range(len(cu) - 1) if cu[s + 1] - cu[s] <= 2048]
    assert len(short) >= 5
    for s in short:
        a, b = int(cu[s]), int(cu[s + 1])
        r_dq, r_dk, r_dv = B.packed_attention_bwd(q[a:b], k[a:b], v[a:b], do[a:b], (0, b - a), True, w.scale)
        check_grads((dq[a:b], dk[a:b], dv[a:b]), (r_dq, r_dk, r_dv), "bf16", f"sequence {s} ({b - a} tokens)")
    worst_v = worst_k = 0.0
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        for g in range(w.Hkv):
            heads = [h for h in range(w.H) if h * w.Hkv // w.H == g]
            lhs = dv64[a:b, g].sum(axis=0)
            rhs = do64[a:b][:, heads].sum(axis=(0, 1))
            worst_v = max(worst_v, np.linalg.norm(lhs - rhs) / np.sqrt((do64[a:b][:, heads] ** 2).sum() + 1e-30))
            worst_k = max(worst_k, np.linalg.norm(dk64[a:b, g].sum(axis=0)) /
                          np.sqrt((dk64[a:b, g] ** 2).sum() + 1e-30))
    print("invariants: sum dV - sum dO", worst_v, "sum dK", worst_k)
    assert worst_v <= 2e-2 and worst_k <= 2e-2


@pytest.mark.parametrize("dtype,mode", [("bf16", "contiguous"), ("fp32", "contiguous")])
def test_block_backward_contiguous_ring(cp, dtype, mode):
    cu = (0, 700, 1500, 1501, 2600) if dtype == "bf16" else (0, 90, 200, 201, 300)
    w = inputs.custom(cu, 8, 2, 128 if dtype == "bf16" else 64, dtype=dtype, causal=True, mode=mode, cp=3)
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    T, H, D = qd.shape
    ws = torch.empty(cp.cpattn_bwd_workspace_size(plan, H, 2, D, qd.dtype, True), dtype=torch.uint8, device="cuda")
    acc = [torch.zeros(T, n, D, dtype=torch.float32, device="cuda") for n in (H, 2, 2)]
    for r in range(w.cp):
        for t in range(w.cp):
            cp.cpattn_block_bwd(plan, qd, kd, vd, o, lse, dod, *acc, ws, r, t, scale=w.scale, causal=True)
            cp.cpattn_sync_status(ws)
    check_grads(acc, B.packed_attention_bwd(q, k, v, do, cu, True, w.scale), dtype, f"ring {dtype} {mode}")


def test_bf16_backward_gqa_group_of_eight(cp):
    cu = (0, 700, 1500)
    w = inputs.custom(cu, 32, 4, 128, dtype="bf16", causal=True, mode="zigzag", cp=2)
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    got = _run_bwd(cp, plan, w, qd, kd, vd, o, lse, dod)
    check_grads(got, B.packed_attention_bwd(q, k, v, do, cu, True, w.scale), "bf16", "gqa 32/4")


def _full_size_single_sequence(cp, name, n_rows):
    """One long sequence at full size: dQ at chunk-boundary and sampled rows
    from the oracle row by row, and sum_j dV_j = sum_i dO_i, sum_j dK_j = 0 on
    every KV head.  The dV bound is relative to sqrt(sum_i |dO_i|^2): with
    near-uniform attention every P of a row sits near 1/row, so its bf16
    rounding carries a per-row bias of up to 2^-9 that the sum over rows
    weights by dO_i; the dK bound is relative to sqrt(sum_j |dK_j|^2)."""
    w = inputs.workload(name)
    (q, k, v, do), (qd, kd, vd, dod), plan, o, lse = _setup(cp, w)
    dq, dk, dv = _run_bwd(cp, plan, w, qd, kd, vd, o, lse, dod)
    rows = inputs.sample_rows(w.T, n_rows, w.seed, must_include=plan.chunk_offsets()[1:-1][:64].tolist())
    ref = B.dq_at_rows(q, k, v, do, w.cu_seqlens, rows, w.causal, w.scale)
    got = dq[torch.from_numpy(rows).cuda()].to("cpu", torch.float64).numpy()
    err = got - ref
    rel = np.sqrt((err ** 2).sum(axis=(0, 2))) / np.sqrt((ref ** 2).sum(axis=(0, 2)))
    assert rel.max() <= BWD_BF16_REL_RMS, rel.max()
    assert np.abs(err).max() <= BWD_BF16_MAX * np.abs(ref).max()
    G = w.H // w.Hkv
    sum_dv = dv.to(torch.float64).sum(dim=0)                    # [Hkv, D]
    do_g = dod.to(torch.float64).view(w.T, w.Hkv, G, w.D)
    sum_do = do_g.sum(dim=(0, 2))
    norm_v = do_g.pow(2).sum(dim=(0, 2, 3)).sqrt()
    worst_v = ((sum_dv - sum_do).norm(dim=1) / norm_v).max().item()
    sum_dk = dk.to(torch.float64).sum(dim=0)
    norm_k = dk.to(torch.float64).pow(2).sum(dim=(0, 2)).sqrt()
    worst_k = (sum_dk.norm(dim=1) / norm_k).max().item()
    print(name, "dQ rel rms", rel.max(), "invariants", worst_v, worst_k)
    assert worst_v <= 2e-2 and worst_k <= 2e-2
    assert torch.isfinite(dk).all() and torch.isfinite(dv).all() and torch.isfinite(dq).all()


def test_long_video_200k_backward_full_size(cp):
    _full_size_single_sequence(cp, "long_video_200k_gqa", 1024)


def test_video_latent_grid2d_backward_full_size(cp):
    _full_size_single_sequence(cp, "video_latent_grid2d", 2048)


def test_single_seq_1m_backward_full_size(cp):
    _full_size_single_sequence(cp, "single_seq_1m_gqa", 256)
