"""The C-ABI library loads on a host without a GPU, exports every function
the header declares, and rejects bad arguments before touching the device."""

import ctypes

import numpy as np
import pytest


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
