"""GPU parity of the materialised ring (cpattn_block_fwd per step, then
cpattn_merge), the per-token loss normalisation and the row permutations."""

import numpy as np
import pytest
import torch

import inputs
from oracle import attention as A
from oracle import loss as LN
from oracle import merge as M
from oracle import plan as P
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


def _ring(cp, w, qd, kd, vd):
    """Every rank: cp block steps then the merge, scattered to global rows."""
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    T, H, D = qd.shape
    ws = torch.empty(cp.cpattn_workspace_size(plan, H, kd.shape[1], D, qd.dtype, w.causal), dtype=torch.uint8,
                     device="cuda")
    ro = plan.rank_offsets()
    idx = torch.from_numpy(plan.index_map()).cuda()
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    parts_all = []
    for r in range(w.cp):
        Tr = int(ro[r + 1] - ro[r])
        po = [torch.full((Tr, H, D), float("nan"), dtype=torch.float32, device="cuda") for _ in range(w.cp)]
        pl = [torch.full((H, Tr), float("nan"), dtype=torch.float32, device="cuda") for _ in range(w.cp)]
        for t in range(w.cp):
            cp.cpattn_block_fwd(plan, qd, kd, vd, po[t], pl[t], ws, r, t, scale=w.scale, causal=w.causal)
            cp.cpattn_sync_status(ws)
        cp.cpattn_merge(po, pl, o, lse, out_rows=idx[int(ro[r]):int(ro[r + 1])])
        parts_all.append((po, pl))
    torch.cuda.synchronize()
    return plan, o, lse, parts_all


@pytest.mark.parametrize("name_or_case", ["tiny_packed_fp32", "bf16_gqa", "bf16_grid2d", "bf16_contiguous"])
def test_materialised_ring_matches_oracle(cp, name_or_case):
    if name_or_case == "tiny_packed_fp32":
        w = inputs.workload(name_or_case)
    elif name_or_case == "bf16_gqa":
        w = inputs.custom((0, 300, 557, 1200), 8, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=4)
    elif name_or_case == "bf16_contiguous":
        w = inputs.custom((0, 300, 557, 1200), 4, 4, 64, dtype="bf16", causal=True, mode="contiguous", cp=3)
    else:
        w = inputs.custom((0, 2 * 9 * 20), 2, 2, 128, dtype="bf16", causal=False, mode="grid2d", cp=4,
                          grid=(2, 9, 20))
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan, o, lse, parts = _ring(cp, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, w.cu_seqlens, w.causal, w.scale)
    U.check(o, lse, O, L, w.dtype, name_or_case)
    # each block partial against the oracle's block attention
    ref_plan = P.make_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    kv_rank, _ = P.ring_schedule(ref_plan, w.causal)
    for r in (0, w.cp - 1):
        q_rows = P.rank_rows(ref_plan, r)
        for t in range(w.cp):
            Ob, Lb = A.block_attention(q, k, v, w.cu_seqlens, q_rows, P.rank_rows(ref_plan, kv_rank[r, t]),
                                       w.causal, w.scale)
            po, pl = parts[r][0][t], parts[r][1][t]
            U.check(po, pl, Ob, Lb, w.dtype if w.dtype == "fp32" else "bf16", f"{name_or_case} r{r} t{t}")


def test_merge_kernel_against_oracle(cp):
    rng = np.random.default_rng(3)
    rows, H, D, n = 777, 3, 128, 5
    o_parts = [rng.standard_normal((rows, H, D)).astype(np.float32) for _ in range(n)]
    lse_parts = [(rng.standard_normal((H, rows)) * 4).astype(np.float32) for _ in range(n)]
    lse_parts[2][:, :100] = -np.inf          # partials with no visible key
    for p in range(n):
        lse_parts[p][:, 5] = -np.inf         # a row with nothing at all
    O, L = M.lse_merge(o_parts, lse_parts)
    od = [torch.from_numpy(x).cuda() for x in o_parts]
    ld = [torch.from_numpy(x).cuda() for x in lse_parts]
    out = torch.empty((rows, H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((H, rows), dtype=torch.float32, device="cuda")
    cp.cpattn_merge(od, ld, out, lse)
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    assert np.abs(got - O).max() < 1e-5
    gl = lse.cpu().double().numpy()
    assert np.array_equal(np.isfinite(gl), np.isfinite(L))
    fin = np.isfinite(L)
    assert np.abs(gl[fin] - L[fin]).max() < 1e-5 * max(1.0, np.abs(L[fin]).max())
    assert np.all(got[5] == 0)


def test_loss_norm_matches_oracle(cp):
    w = inputs.workload("dynamic_cp_microbatch")
    loss, valid = inputs.make_loss_inputs(w)
    ref, count = LN.token_loss_norm(loss.numpy(), valid.numpy())
    out = torch.empty(1, dtype=torch.float64, device="cuda")
    cnt = torch.empty(1, dtype=torch.int64, device="cuda")
    f32 = torch.empty(1, dtype=torch.float32, device="cuda")
    cp.cpattn_token_loss_norm(loss.cuda(), valid.cuda(), out, cnt, f32)
    torch.cuda.synchronize()
    assert int(cnt.item()) == count == w.T - 3276
    assert abs(out.item() - ref) <= 1e-12 * abs(ref)
    assert abs(f32.item() - ref) <= 1e-6 * abs(ref)
    # ragged length, unaligned tail and the empty-valid case
    for T in (1, 17, 1000003):
        l = torch.rand(T) * 5
        vmask = (torch.rand(T) > 0.3).to(torch.uint8)
        ref, count = LN.token_loss_norm(l.numpy(), vmask.numpy())
        cp.cpattn_token_loss_norm(l.cuda(), vmask.cuda(), out, cnt)
        torch.cuda.synchronize()
        assert int(cnt.item()) == count
        assert abs(out.item() - ref) <= 1e-12 * max(abs(ref), 1e-300)
    cp.cpattn_token_loss_norm(l.cuda(), torch.zeros(T, dtype=torch.uint8, device="cuda"), out, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 0 and out.item() == 0.0


def test_loss_norm_is_deterministic(cp):
    l = (torch.rand(1 << 20) * 3).cuda()
    vmask = (torch.rand(1 << 20) > 0.1).to(torch.uint8).cuda()
    outs = []
    for _ in range(3):
        out = torch.empty(1, dtype=torch.float64, device="cuda")
        cnt = torch.empty(1, dtype=torch.int64, device="cuda")
        cp.cpattn_token_loss_norm(l, vmask, out, cnt)
        outs.append(out.item())
    assert outs[0] == outs[1] == outs[2]


def test_gather_scatter_round_trip(cp):
    F, h, wd = 4, 45, 80
    T = F * h * wd
    plan = cp.cpattn_plan((0, T), 8, "grid2d", (F, h, wd))
    idx_np = plan.index_map()
    ref = P.grid2d((0, T), 8, (F, h, wd))
    assert np.array_equal(idx_np, ref.index_map)
    x = torch.randn(T, 24, 128, dtype=torch.bfloat16, device="cuda")
    idx = torch.from_numpy(idx_np).cuda()
    shards = torch.empty_like(x)
    cp.cpattn_gather_rows(x, shards, idx)
    back = torch.empty_like(x)
    cp.cpattn_scatter_rows(shards, back, idx)
    torch.cuda.synchronize()
    assert torch.equal(shards, x[idx])
    assert torch.equal(back, x)
    # out-of-range indices are skipped
    bad = idx.clone()
    bad[7] = T + 5
    dst = torch.zeros_like(x)
    cp.cpattn_gather_rows(x, dst, bad)
    torch.cuda.synchronize()
    assert torch.equal(dst[7], torch.zeros_like(dst[7]))
    assert torch.equal(dst[8], x[idx[8]])


def test_device_fault_word_reports_nothing_on_clean_runs(cp):
    w = inputs.custom((0, 256), 2, 2, 128, dtype="bf16")
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan((0, 256), 2, "zigzag")
    ws = torch.empty(cp.cpattn_workspace_size(plan, 2, 2, 128, torch.bfloat16, True), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(qd)
    lse = torch.empty(2, 256, dtype=torch.float32, device="cuda")
    cp.cpattn_fwd(plan, qd, kd, vd, o, lse, ws)
    cp.cpattn_sync_status(ws)
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_copy_kernel_between_pinned_host_and_device(cp):
    """cpattn_copy moves bytes exactly: pinned host -> device, device -> pinned
    host, device -> device, with a few and with many blocks."""
    g = torch.Generator().manual_seed(3)
    h = torch.randint(0, 2 ** 31 - 1, (3 << 20,), generator=g, dtype=torch.int32).pin_memory()
    d = torch.empty(h.shape, dtype=torch.int32, device="cuda")
    for blocks in (3, 0):
        d.fill_(-1)
        cp.cpattn_copy(d, h, n_blocks=blocks)
        torch.cuda.synchronize()
        assert torch.equal(d.cpu(), h)
        back = torch.full(h.shape, -1, dtype=torch.int32).pin_memory()
        cp.cpattn_copy(back, d, n_blocks=blocks)
        torch.cuda.synchronize()
        assert torch.equal(back, h)
    d2 = torch.empty_like(d)
    cp.cpattn_copy(d2, d)
    torch.cuda.synchronize()
    assert torch.equal(d2, d)
    with pytest.raises(cp.CpattnError):
        cp.cpattn_copy(d[1:3], d[5:7])          # 8 bytes: not a multiple of 16
    with pytest.raises(cp.CpattnError):
        cp.cpattn_copy(d, torch.empty(h.shape, dtype=torch.int32))   # pageable host memory
