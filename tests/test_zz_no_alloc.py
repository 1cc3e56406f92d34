"""cpattn_fwd_static, the forward for callers that cannot allocate device
memory (a plugin interface that passes only input and output buffers, or a
process whose device memory another allocator owns), gives the results of the
workspace forward cpattn_fwd on two calls in a row, bit for bit, and both
match the oracle.  After each call the static array's fault word is read back
through cpattn_static_sync_status.

This file is collected last on purpose: a run that stops at the first failure
has run every other test before it.  It also passes alone in a fresh process.
"""

import ctypes

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


def _static_forward(cp, plan, w, qd, kd, vd):
    """Through the C ABI directly: no workspace argument at all."""
    T, H, D = qd.shape
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    L = cp.lib()
    dt = cp.DTYPE_BF16 if qd.dtype == torch.bfloat16 else cp.DTYPE_FP32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    s = L.cpattn_fwd_static(plan.handle, ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()),
                            ctypes.c_void_p(vd.data_ptr()), dt, H, kd.shape[1], D, w.scale, int(w.causal),
                            ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)
    assert s == cp.OK, L.cpattn_last_error_string()
    s = L.cpattn_static_sync_status(stream)     # synchronises; the fault word must be clear
    assert s == cp.OK, L.cpattn_last_error_string()
    return o, lse


def test_static_scratch_forward_matches_workspace_forward(cp):
    cases = [inputs.workload("dynamic_cp_microbatch"), inputs.workload("tiny_packed_fp32"),
             inputs.custom((0, 300, 557), 8, 2, 128, dtype="bf16", causal=True, mode="contiguous", cp=3)]
    for w in cases:
        (q, k, v), (qd, kd, vd) = U.device_inputs(w)
        plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode)
        o_ws, l_ws = U.run_fwd(cp, plan, w, qd, kd, vd)
        first = _static_forward(cp, plan, w, qd, kd, vd)
        second = _static_forward(cp, plan, w, qd, kd, vd)   # the scratch still holds the first call's list
        for name, (o, lse) in (("first", first), ("second", second)):
            # the same kernel on the same work list: identical bits
            assert torch.equal(o, o_ws) and torch.equal(lse, l_ws), f"{w.name} {name} call"
        # and the oracle, on every row (the micro-batch) or all of it
        rows = np.arange(w.T)
        O, L = A.attention_at_rows(q, k, v, w.cu_seqlens, rows, w.causal, w.scale)
        U.check(second[0], second[1], O, L, w.dtype, f"{w.name} static vs oracle")


def _buffers(T, H, Hkv, D):
    """Device buffers that fit a call on T tokens, so that a call which
    wrongly went ahead would still stay inside its buffers."""
    q = torch.zeros(T, H, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(T, Hkv, D, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    o = torch.empty_like(q)
    lse = torch.empty(H, T, dtype=torch.float32, device="cuda")
    return [ctypes.c_void_p(t.data_ptr()) for t in (q, k, v)], ctypes.c_void_p(o.data_ptr()), \
        ctypes.c_void_p(lse.data_ptr()), (q, k, v, o, lse)


def test_static_scratch_rejects_what_it_cannot_hold(cp):
    L = cp.lib()
    plans = [cp.cpattn_plan([0, 2 * 9 * 20], 4, "grid2d", (2, 9, 20)),
             cp.cpattn_plan_2d([0, 256], 2, 2),
             cp.cpattn_plan_paired([0, 64], 2, 4)]
    (q, k, v), o, lse, keep = _buffers(2 * 9 * 20, 4, 4, 128)
    for plan in plans:
        s = L.cpattn_fwd_static(plan.handle, q, k, v, cp.DTYPE_BF16, 4, 4, 128, 0.1, 1, o, lse, None)
        assert s == cp.UNSUPPORTED, plan.mode
    # many short sequences with a large cp: every tile reads 2cp one-token
    # chunks, and the work list outgrows the 8 MiB array (checked here on the
    # host before the call)
    n, ln = 10000, 64
    big = cp.cpattn_plan(np.arange(0, ln * (n + 1), ln), 32, "zigzag")
    tiles, runs = big.worklist(False, "bf16", True)
    r256 = lambda x: -(-x // 256) * 256
    assert 256 + r256(len(tiles) * 32) + r256(len(runs) * 16) > 8 << 20
    (q, k, v), o, lse, keep = _buffers(n * ln, 2, 2, 128)
    s = L.cpattn_fwd_static(big.handle, q, k, v, cp.DTYPE_BF16, 2, 2, 128, 0.1, 1, o, lse, None)
    torch.cuda.synchronize()
    assert s == cp.WORKSPACE
    assert b"static scratch holds" in L.cpattn_last_error_string()
