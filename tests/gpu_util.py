"""Helpers for the GPU parity tests: run the library on a workload and compare
with the fp64 oracle under the stated tolerances."""

from __future__ import annotations

import math

import numpy as np
import torch

import inputs

# Tolerances.  bf16 outputs: max-abs 2e-2 on O and 1e-3 relative on LSE, the
# workload statement's bounds; because O is small for near-uniform attention,
# a per-head relative RMS bound of 1e-2 is checked as well.  fp32: 1e-5.
# The LSE bound carries an absolute floor of 1e-6: for a row that sees one key,
# lse is that key's score, which can be ~0, and its fp32 rounding is ~1e-7.
BF16_O_ABS = 2e-2
BF16_LSE_REL = 1e-3
BF16_O_REL_RMS = 1e-2
FP32_TOL = 1e-5
LSE_ABS_FLOOR = 1e-6


def device_inputs(w: inputs.Workload):
    q, k, v = inputs.make_qkv(w)
    return (q, k, v), (q.cuda(), k.cuda(), v.cuda())


def run_fwd(cp, plan, w, qd, kd, vd, causal=None):
    causal = w.causal if causal is None else causal
    T, H, D = qd.shape
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(cp.cpattn_workspace_size(plan, H, kd.shape[1], D, qd.dtype, causal), dtype=torch.uint8,
                     device="cuda")
    cp.cpattn_fwd(plan, qd, kd, vd, o, lse, ws, scale=w.scale, causal=causal)
    cp.cpattn_sync_status(ws)
    return o, lse


def check(o_gpu, lse_gpu, o_ref, lse_ref, dtype, where=""):
    """Element-wise comparison; returns a dict of the observed errors."""
    o = o_gpu.detach().to("cpu", torch.float64).numpy()
    l = lse_gpu.detach().to("cpu", torch.float64).numpy()
    assert np.isfinite(o).all(), f"{where}: non-finite O"
    err_o = np.abs(o - o_ref)
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), finite), f"{where}: -inf pattern of LSE differs"
    err_l = np.abs(l[finite] - lse_ref[finite])
    rel_l = err_l / np.maximum(np.abs(lse_ref[finite]), LSE_ABS_FLOOR / BF16_LSE_REL if dtype == "bf16" else 1.0)
    stats = {"o_max_abs": float(err_o.max(initial=0)), "lse_max_rel": float(rel_l.max(initial=0))}
    if dtype == "bf16":
        num = np.sqrt((err_o ** 2).sum(axis=(0, 2)))
        den = np.sqrt((o_ref ** 2).sum(axis=(0, 2)))
        rel_rms = num / np.maximum(den, 1e-30)
        stats["o_rel_rms_max"] = float(rel_rms.max(initial=0))
        assert stats["o_max_abs"] <= BF16_O_ABS, (where, stats)
        assert stats["lse_max_rel"] <= BF16_LSE_REL, (where, stats)
        assert stats["o_rel_rms_max"] <= BF16_O_REL_RMS, (where, stats)
    else:
        lse_err = err_l / np.maximum(np.abs(lse_ref[finite]), 1.0)
        stats["lse_max"] = float(lse_err.max(initial=0))
        assert stats["o_max_abs"] <= FP32_TOL, (where, stats)
        assert stats["lse_max"] <= FP32_TOL, (where, stats)
    return stats


def boundary_rows(plan, n_extra: int, T: int, seed: int) -> np.ndarray:
    """Rows at every chunk boundary (first/last row of each chunk) plus a
    seeded uniform sample."""
    offs = plan.chunk_offsets()
    edges = np.unique(np.concatenate([offs[:-1], offs[1:] - 1, [0, T - 1]]))
    if len(edges) > 2000:
        edges = edges[np.linspace(0, len(edges) - 1, 2000).astype(int)]
    return inputs.sample_rows(T, n_extra, seed, must_include=edges.tolist())
