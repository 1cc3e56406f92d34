"""The C-ABI library loads on a host without a GPU, exports every function
the header declares, and rejects bad arguments before touching the device."""

import ctypes

import numpy as np
import pytest
import torch

# Tests that pass made-up addresses (never dereferenced: every call fails an
# argument check first) run only where no GPU can be reached, so that a check
# that went missing could never launch a kernel on them.
host_only = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="made-up device addresses: run only without a reachable GPU")


def test_every_declared_symbol_is_exported(cpattn):
    names = cpattn.header_functions()
    assert len(names) >= 20
    L = cpattn.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(cpattn._SIGNATURES), "binding and header disagree"


def test_version(cpattn):
    assert "sm_103a" in cpattn.version()


def test_fwd_flops_matches_closed_form(cpattn):
    assert cpattn.cpattn_fwd_flops([0, 64, 264, 520], 4, 64, True) == 56397824
    assert cpattn.cpattn_fwd_flops([0, 1 << 20], 32, 128, True) == 4 * 128 * 32 * (1 << 20) * ((1 << 20) + 1) // 2
    assert cpattn.cpattn_fwd_flops([0, 57600], 24, 128, False) == 4 * 128 * 24 * 57600 ** 2


@pytest.mark.parametrize("cu,cp,mode", [
    ([0, 3, 10], 2, "zigzag"),       # a sequence shorter than 2*cp
    ([1, 10], 1, "zigzag"),          # cu[0] != 0
    ([0, 10, 10], 1, "contiguous"),  # empty sequence
    ([0, 2], 3, "contiguous"),       # fewer tokens than ranks
    ([0, 10], 0, "zigzag"),          # cp < 1
])
def test_plan_rejects_bad_inputs(cpattn, cu, cp, mode):
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_plan(cu, cp, mode)
    assert e.value.status == cpattn.INVALID_ARG


def test_grid_plan_rejects_bad_grids(cpattn):
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan([0, 100], 4, "grid2d", (1, 9, 11))   # 9*11 != 100
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan([0, 9 * 4], 16, "grid2d", (1, 9, 4))  # 16 = 4 x 4 but 9 rows cannot give 4 pieces of 3
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_plan([0, 50, 100], 2, "grid2d", (1, 10, 10))  # two sequences


@host_only
def test_host_side_argument_errors(cpattn):
    L = cpattn.lib()
    plan = cpattn.cpattn_plan([0, 256], 2, "zigzag")
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    ws = ctypes.c_void_p(1 << 20)
    # unsupported head dim
    s = L.cpattn_fwd(plan.handle, fake, fake, fake, cpattn.DTYPE_BF16, 4, 4, 96, 0.1, 1, fake, fake, ws, 1 << 30, None)
    assert s == cpattn.UNSUPPORTED
    # H not a multiple of Hkv
    s = L.cpattn_fwd(plan.handle, fake, fake, fake, cpattn.DTYPE_BF16, 6, 4, 128, 0.1, 1, fake, fake, ws, 1 << 30, None)
    assert s == cpattn.INVALID_ARG
    # NULL q
    s = L.cpattn_fwd(plan.handle, None, fake, fake, cpattn.DTYPE_BF16, 4, 4, 128, 0.1, 1, fake, fake, ws, 1 << 30, None)
    assert s == cpattn.INVALID_ARG
    # misaligned workspace
    s = L.cpattn_fwd(plan.handle, fake, fake, fake, cpattn.DTYPE_BF16, 4, 4, 128, 0.1, 1, fake, fake,
                     ctypes.c_void_p((1 << 20) + 16), 1 << 30, None)
    assert s == cpattn.WORKSPACE
    # workspace too small
    s = L.cpattn_fwd(plan.handle, fake, fake, fake, cpattn.DTYPE_BF16, 4, 4, 128, 0.1, 1, fake, fake, ws, 16, None)
    assert s == cpattn.WORKSPACE
    assert b"workspace too small" in L.cpattn_last_error_string()
    # block step out of range
    s = L.cpattn_block_fwd(plan.handle, fake, fake, fake, cpattn.DTYPE_BF16, 4, 4, 128, 0.1, 1, 0, 2, fake, fake,
                           ws, 1 << 30, None)
    assert s == cpattn.INVALID_ARG
    # merge with too many partials
    arr = (ctypes.c_void_p * 65)()
    s = L.cpattn_merge(65, arr, arr, 10, 4, 128, None, 10, fake, cpattn.DTYPE_BF16, fake, None)
    assert s == cpattn.INVALID_ARG
    # causal grid2d is not defined
    gplan = cpattn.cpattn_plan([0, 16 * 45 * 80], 8, "grid2d", (16, 45, 80))
    out = ctypes.c_size_t()
    s = L.cpattn_workspace_size(gplan.handle, 24, 24, 128, cpattn.DTYPE_BF16, 1, ctypes.byref(out))
    assert s == cpattn.UNSUPPORTED


def test_workspace_size_grows_with_grid_shards(cpattn):
    z = cpattn.cpattn_plan([0, 4096], 4, "zigzag")
    g = cpattn.cpattn_plan([0, 16 * 45 * 80], 8, "grid2d", (16, 45, 80))
    wz = cpattn.cpattn_workspace_size(z, 32, 8, 128, "bf16", True)
    wg = cpattn.cpattn_workspace_size(g, 24, 24, 128, "bf16", False)
    assert 256 < wz < (1 << 22)
    T = 16 * 45 * 80
    assert wg >= T * 8 + 3 * T * 24 * 128 * 2


@host_only
def test_backward_and_mesh_argument_errors(cpattn):
    """Every rejection below happens in the host-side checks, before any
    device call (the pointers are never dereferenced)."""
    L = cpattn.lib()
    fake = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 20)
    plan = cpattn.cpattn_plan([0, 256], 2, "zigzag")
    bf, f32 = cpattn.DTYPE_BF16, cpattn.DTYPE_FP32

    def bwd(p=plan, dtype=bf, H=4, Hkv=4, D=128, scale=0.1, causal=1, o=fake, dq=fake, ws_ptr=ws, ws_bytes=1 << 30):
        return L.cpattn_bwd(p.handle, fake, fake, fake, o, fake, fake, dtype, H, Hkv, D, scale, causal, dq, fake,
                            fake, ws_ptr, ws_bytes, None)

    assert bwd(D=64) == cpattn.UNSUPPORTED                      # bf16 backward needs D = 128
    assert bwd(dtype=f32, D=96) == cpattn.UNSUPPORTED           # head dim
    assert bwd(H=6) == cpattn.INVALID_ARG                       # H not a multiple of Hkv
    assert bwd(o=None) == cpattn.INVALID_ARG                    # NULL O
    assert bwd(dq=ctypes.c_void_p((1 << 20) + 8)) == cpattn.INVALID_ARG  # misaligned dQ
    assert bwd(scale=0.0) == cpattn.INVALID_ARG
    assert bwd(scale=float("inf")) == cpattn.INVALID_ARG
    assert bwd(ws_ptr=ctypes.c_void_p((1 << 20) + 64)) == cpattn.WORKSPACE
    assert bwd(ws_bytes=64) == cpattn.WORKSPACE
    assert b"workspace too small" in L.cpattn_last_error_string()
    # per-step backward: rank and step ranges
    s = L.cpattn_block_bwd(plan.handle, fake, fake, fake, fake, fake, fake, bf, 4, 4, 128, 0.1, 1, 2, 0, fake, fake,
                           fake, ws, 1 << 30, None)
    assert s == cpattn.INVALID_ARG
    s = L.cpattn_block_bwd(plan.handle, fake, fake, fake, fake, fake, fake, bf, 4, 4, 128, 0.1, 1, 0, -1, fake, fake,
                           fake, ws, 1 << 30, None)
    assert s == cpattn.INVALID_ARG
    out = ctypes.c_size_t()
    # causal grid2d has no backward either
    gplan = cpattn.cpattn_plan([0, 2 * 9 * 20], 4, "grid2d", (2, 9, 20))
    assert L.cpattn_bwd_workspace_size(gplan.handle, 2, 2, 128, bf, 1, ctypes.byref(out)) == cpattn.UNSUPPORTED
    assert L.cpattn_bwd_workspace_size(gplan.handle, 2, 2, 128, bf, 0, ctypes.byref(out)) == cpattn.OK
    # mesh and paired plans: whole forward only; heads must split over the Ulysses degree
    mesh = cpattn.cpattn_plan_2d([0, 300, 557, 1200], 2, 2)
    assert L.cpattn_bwd_workspace_size(mesh.handle, 8, 4, 128, bf, 1, ctypes.byref(out)) == cpattn.UNSUPPORTED
    assert bwd(p=mesh, H=8, Hkv=4) == cpattn.UNSUPPORTED
    s = L.cpattn_fwd(mesh.handle, fake, fake, fake, bf, 6, 3, 128, 0.1, 1, fake, fake, ws, 1 << 30, None)
    assert s == cpattn.UNSUPPORTED                              # 3 KV heads over u = 2
    s = L.cpattn_block_fwd(mesh.handle, fake, fake, fake, bf, 8, 4, 128, 0.1, 1, 0, 0, fake, fake, ws, 1 << 30, None)
    assert s == cpattn.UNSUPPORTED
    paired = cpattn.cpattn_plan_paired([0, 64], 2, 4)
    s = L.cpattn_fwd(paired.handle, fake, fake, fake, bf, 4, 4, 128, 0.1, 0, fake, fake, ws, 1 << 30, None)
    assert s == cpattn.UNSUPPORTED                              # the teacher-forcing mask needs causal = 1


@pytest.mark.parametrize("args", [
    ([0, 100], 0, 2),        # ulysses < 1
    ([0, 100], 2, 0),        # ring < 1
    ([0, 3], 1, 2),          # a sequence shorter than 2 * ring
])
def test_mesh_plan_rejects_bad_inputs(cpattn, args):
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_plan_2d(*args)
    assert e.value.status == cpattn.INVALID_ARG


@pytest.mark.parametrize("args", [
    ([0, 41], 2, 4),         # odd sample length: no clean/noisy halves
    ([0, 40], 3, 4),         # chunks not a multiple of cp
    ([0, 6], 2, 4),          # fewer tokens per stream than chunks
])
def test_paired_plan_rejects_bad_inputs(cpattn, args):
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_plan_paired(*args)
    assert e.value.status == cpattn.INVALID_ARG


def test_every_plan_entry_point_rejects_a_null_plan(cpattn):
    """NULL plan, NULL pointers and zero sizes: each call returns
    CPATTN_INVALID_ARG without touching memory (destroy of NULL is a no-op)."""
    L = cpattn.lib()
    names = [n for n in cpattn._SIGNATURES if n.startswith("cpattn_plan_get") or n in (
        "cpattn_workspace_size", "cpattn_fwd", "cpattn_block_fwd", "cpattn_bwd_workspace_size", "cpattn_bwd",
        "cpattn_block_bwd", "cpattn_fwd_static", "cpattn_plan_allowed_pairs")]
    assert len(names) >= 17
    for n in names:
        sig = cpattn._SIGNATURES[n]
        args = [None] + [None if t is ctypes.c_void_p else 0 for t in sig[1:]]
        assert getattr(L, n)(*args) == cpattn.INVALID_ARG, n
    assert L.cpattn_plan_destroy(None) == cpattn.OK


@host_only
def test_merge_permute_and_loss_argument_errors(cpattn):
    L = cpattn.lib()
    fake = ctypes.c_void_p(1 << 20)
    arr = (ctypes.c_void_p * 2)(1 << 20, 1 << 21)
    bf = cpattn.DTYPE_BF16
    assert L.cpattn_merge(0, arr, arr, 10, 4, 128, None, 10, fake, bf, fake, None) == cpattn.INVALID_ARG
    assert L.cpattn_merge(2, None, None, 10, 4, 128, None, 10, fake, bf, fake, None) == cpattn.INVALID_ARG
    assert L.cpattn_merge(2, arr, arr, 10, 4, 96, None, 10, fake, bf, fake, None) == cpattn.UNSUPPORTED
    assert L.cpattn_merge(2, arr, arr, -1, 4, 128, None, 10, fake, bf, fake, None) == cpattn.INVALID_ARG
    assert L.cpattn_merge(2, arr, arr, 10, 4, 128, None, 5, fake, bf, fake, None) == cpattn.INVALID_ARG
    assert L.cpattn_merge(2, arr, arr, 10, 4, 128, None, 10, None, bf, fake, None) == cpattn.INVALID_ARG
    assert L.cpattn_gather_rows(fake, 10, fake, fake, 10, 24, None) == cpattn.INVALID_ARG      # row bytes % 16
    assert L.cpattn_gather_rows(ctypes.c_void_p((1 << 20) + 4), 10, fake, fake, 10, 32, None) == cpattn.INVALID_ARG
    assert L.cpattn_gather_rows(fake, 10, fake, None, 10, 32, None) == cpattn.INVALID_ARG
    assert L.cpattn_scatter_rows(fake, fake, 10, fake, -3, 32, None) == cpattn.INVALID_ARG
    assert L.cpattn_token_loss_norm(None, fake, 10, fake, fake, None, None) == cpattn.INVALID_ARG
    assert L.cpattn_token_loss_norm(fake, fake, -1, fake, fake, None, None) == cpattn.INVALID_ARG


def test_fault_path_test_settings_reject_bad_arguments(cpattn):
    """The fault-path test settings (host only, nothing launched)."""
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_debug_wait_fault(0, True)          # a withheld load needs a short limit
    assert e.value.status == cpattn.INVALID_ARG
    with pytest.raises(cpattn.CpattnError):
        cpattn.cpattn_debug_wait_fault(20_000_000, False)  # above 10 s
    cpattn.cpattn_debug_wait_fault(1000, True)
    cpattn.cpattn_debug_wait_fault(0, False)             # back to the defaults
