"""The device fault path, exercised without a GPU fault.

Every wait inside the kernels is bounded.  Here a test-only setting shortens
the bound to 2 ms and makes block 0 of the bf16 forward skip loading its first
V tile, so its MMA thread waits on a barrier that nothing completes.  The
wait runs out, the kernel records the fault in the workspace, lets its copies
in flight land, frees its tensor memory and returns; cpattn_sync_status must
report CPATTN_DEVICE_FAULT for block 0, and a following clean call on the
same context must match the oracle."""

import time

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


def test_an_expired_wait_is_reported_and_the_context_stays_usable(cp):
    cu = (0, 300, 557, 1200)
    w = inputs.custom(cu, 4, 2, 128, dtype="bf16", causal=True, mode="zigzag", cp=2)
    (q, k, v), (qd, kd, vd) = U.device_inputs(w)
    plan = cp.cpattn_plan(cu, 2, "zigzag")
    T, H, D = qd.shape
    ws = torch.empty(cp.cpattn_workspace_size(plan, H, 2, D, qd.dtype, True), dtype=torch.uint8, device="cuda")
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    cp.cpattn_debug_wait_fault(2000, True)
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        cp.cpattn_fwd(plan, qd, kd, vd, o, lse, ws, scale=w.scale, causal=True)
        with pytest.raises(cp.CpattnError) as e:
            cp.cpattn_sync_status(ws)
        elapsed = time.perf_counter() - t0
    finally:
        cp.cpattn_debug_wait_fault(0, False)
    assert e.value.status == cp.DEVICE_FAULT
    # a wait-timeout fault (code 1) in block 0; which of its waits ran out first (the
    # MMA thread's wait for V_0, or the warps waiting behind it) depends on timing
    assert "kernel fault 1 in block 0 at" in str(e.value), str(e.value)
    assert elapsed < 2.0                                       # the kernel returned after the short limit
    assert torch.isnan(o).any()                                # block 0 stopped early: rows left unwritten
    # the same context, a clean call
    o2, lse2 = U.run_fwd(cp, plan, w, qd, kd, vd)
    O, L = A.packed_attention(q, k, v, cu, True, w.scale)
    U.check(o2, lse2, O, L, "bf16", "after the fault")
