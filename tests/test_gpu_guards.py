"""Guard regions around every buffer the library writes.

compute-sanitizer is not available, so each output and each workspace sits
between two guard regions holding a known pattern; after the call the guards
must be untouched.  The shapes are ragged (tiles end mid-tile, chunks of
uneven size, a grid whose sides do not divide evenly) and cover the whole
forward (bf16 zigzag with GQA, fp32, grid2d, a 2 x 2 Ulysses-ring mesh), one
materialised ring step and the LSE merge, the backward (bf16 and fp32) and
the loss normalisation."""

import numpy as np
import pytest
import torch

import inputs

pytestmark = pytest.mark.gpu

GUARD = 8192  # elements on each side; keeps every view 16-byte aligned


@pytest.fixture(scope="module")
def cp():
    import context_attention_cpattn_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    m.build()
    m.lib()
    return m


class Guarded:
    """A tensor of `shape` inside a larger buffer whose head and tail hold
    `fill`; `.t` is the tensor handed to the library."""

    def __init__(self, shape, dtype, fill, device="cuda"):
        self.n = int(np.prod(shape))
        self.fill = fill
        self.buf = torch.full((self.n + 2 * GUARD,), fill, dtype=dtype, device=device)
        self.t = self.buf[GUARD:GUARD + self.n].view(*shape)

    def intact(self) -> bool:
        ref = torch.full((GUARD,), self.fill, dtype=self.buf.dtype, device=self.buf.device)
        return bool(torch.equal(self.buf[:GUARD], ref) and torch.equal(self.buf[GUARD + self.n:], ref))


def _ws(nbytes):
    return Guarded((max(int(nbytes), 1),), torch.uint8, 0xA5)


def _fwd(cp, plan, w, qd, kd, vd):
    T, H, D = qd.shape
    o = Guarded((T, H, D), qd.dtype, -7.25)
    lse = Guarded((H, T), torch.float32, -7.25)
    ws = _ws(cp.cpattn_workspace_size(plan, H, kd.shape[1], D, qd.dtype, w.causal))
    cp.cpattn_fwd(plan, qd, kd, vd, o.t, lse.t, ws.t, scale=w.scale, causal=w.causal)
    cp.cpattn_sync_status(ws.t)
    torch.cuda.synchronize()
    return o, lse, ws


def _device(w):
    q, k, v = inputs.make_qkv(w)
    return q.cuda(), k.cuda(), v.cuda()


@pytest.mark.parametrize("case", ["bf16_zigzag_gqa", "fp32_tiny", "bf16_grid2d", "bf16_mesh_2x2"])
def test_forward_writes_stay_inside_outputs_and_workspace(cp, case):
    if case == "bf16_zigzag_gqa":
        w = inputs.custom((0, 200, 333, 520), 4, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=2)
        plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    elif case == "fp32_tiny":
        w = inputs.workload("tiny_packed_fp32")
        plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    elif case == "bf16_grid2d":
        w = inputs.custom((0, 2 * 9 * 20), 2, 2, 128, dtype="bf16", causal=False, mode="grid2d", cp=4,
                          grid=(2, 9, 20))
        plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    else:
        w = inputs.custom((0, 300, 557, 1200), 8, 4, 128, dtype="bf16", causal=True)
        plan = cp.cpattn_plan_2d(w.cu_seqlens, 2, 2)
    qd, kd, vd = _device(w)
    o, lse, ws = _fwd(cp, plan, w, qd, kd, vd)
    assert o.intact() and lse.intact() and ws.intact(), case
    assert torch.isfinite(o.t).all() and torch.isfinite(lse.t).all(), case


def test_ring_step_and_merge_writes_stay_inside(cp):
    w = inputs.custom((0, 200, 333, 520), 4, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=2)
    qd, kd, vd = _device(w)
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    T, H, D = qd.shape
    ro = plan.rank_offsets()
    idx = torch.from_numpy(plan.index_map()).cuda()
    ws = _ws(cp.cpattn_workspace_size(plan, H, kd.shape[1], D, qd.dtype, w.causal))
    o = Guarded((T, H, D), qd.dtype, -7.25)
    lse = Guarded((H, T), torch.float32, -7.25)
    guards = [ws, o, lse]
    for r in range(w.cp):
        Tr = int(ro[r + 1] - ro[r])
        po = [Guarded((Tr, H, D), torch.float32, -7.25) for _ in range(w.cp)]
        pl = [Guarded((H, Tr), torch.float32, -7.25) for _ in range(w.cp)]
        guards += po + pl
        for t in range(w.cp):
            cp.cpattn_block_fwd(plan, qd, kd, vd, po[t].t, pl[t].t, ws.t, r, t, scale=w.scale, causal=w.causal)
            cp.cpattn_sync_status(ws.t)
        cp.cpattn_merge([x.t for x in po], [x.t for x in pl], o.t, lse.t, out_rows=idx[int(ro[r]):int(ro[r + 1])])
    torch.cuda.synchronize()
    assert all(g.intact() for g in guards)
    assert torch.isfinite(o.t).all() and torch.isfinite(lse.t).all()


@pytest.mark.parametrize("case", ["bf16", "fp32"])
def test_backward_writes_stay_inside_outputs_and_workspace(cp, case):
    if case == "bf16":
        w = inputs.custom((0, 200, 333, 520), 4, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=2)
    else:
        w = inputs.workload("tiny_packed_fp32")
    qd, kd, vd = _device(w)
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    o, lse, _ = _fwd(cp, plan, w, qd, kd, vd)
    dod = inputs.make_dout(w).cuda()
    T, H, D = qd.shape
    Hkv = kd.shape[1]
    dq = Guarded((T, H, D), qd.dtype, -7.25)
    dk = Guarded((T, Hkv, D), kd.dtype, -7.25)
    dv = Guarded((T, Hkv, D), vd.dtype, -7.25)
    ws = _ws(cp.cpattn_bwd_workspace_size(plan, H, Hkv, D, qd.dtype, w.causal))
    cp.cpattn_bwd(plan, qd, kd, vd, o.t, lse.t, dod, dq.t, dk.t, dv.t, ws.t, scale=w.scale, causal=w.causal)
    cp.cpattn_sync_status(ws.t)
    torch.cuda.synchronize()
    assert dq.intact() and dk.intact() and dv.intact() and ws.intact(), case
    assert torch.isfinite(dq.t).all() and torch.isfinite(dk.t).all() and torch.isfinite(dv.t).all(), case


def test_loss_norm_writes_stay_inside(cp):
    T = 4099
    gen = torch.Generator().manual_seed(5)
    loss = (torch.rand(T, generator=gen) * 12).cuda()
    valid = (torch.rand(T, generator=gen) > 0.1).to(torch.uint8).cuda()
    out = Guarded((1,), torch.float64, -7.25)
    cnt = Guarded((1,), torch.int64, -7)
    f32 = Guarded((1,), torch.float32, -7.25)
    cp.cpattn_token_loss_norm(loss, valid, out.t, cnt.t, f32.t)
    torch.cuda.synchronize()
    assert out.intact() and cnt.intact() and f32.intact()
    assert int(cnt.t.item()) == int(valid.sum().item())
