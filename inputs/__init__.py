"""Seeded synthetic workloads for packed variable-length context-parallel attention.

This module holds workload shapes, the sequence-length draw and seeded value
generation only.  It contains none of the attention, planning, merge or loss
arithmetic: both the fp64 oracle tests and the CUDA path take their inputs from
here, and nothing else is shared between them.

Workloads (named by what they are, after the pages' workloads):

* ``tiny_packed_fp32`` - three packed sequences {64, 200, 256}, H=4, D=64,
  fp32 N(0,1), causal, zigzag cp=2.
* ``dynamic_cp_microbatch`` - a Dynamic-CP style packed micro-batch: lengths
  drawn from a long-tailed lognormal (median 512, clipped to [64, 16384]) until
  T=32768, H=32, D=128, bf16 N(0,1)/sqrt(D), causal, zigzag cp=4, with 10% of
  tokens flagged invalid for the per-token loss normalisation
  ("Speeding up Variable-Length Training with Dynamic Context Parallelism and
  NVIDIA Megatron Core", Fig. 1 and the THD packing section).
* ``long_video_200k_gqa`` - 1024 frames x 196 visual tokens + 300 text tokens
  as one causal sequence (T=200,996), H=32, Hkv=8, D=128, zigzag cp=8
  (LongVILA news article, stage-5 long-video training).
* ``video_latent_grid2d`` - a 16 x 45 x 80 video latent (T=57,600), H=24,
  D=128, bidirectional, cp=8 split as an h x w tile grid (LongCat-Video
  context-parallel article, tensor split strategy).
* ``single_seq_1m_gqa`` - one causal sequence of 2**20 tokens, H=32, Hkv=8,
  D=128, zigzag cp=16.

Values are N(0,1) draws from numpy's PCG64, keyed by (seed, tensor, block),
scaled by 1/sqrt(D) for the bf16 workloads and rounded to the tensor dtype
(round-to-nearest-even for bf16).  Generation is block-parallel so that the
largest workload (6.4e9 values) is produced in seconds on a many-core host; the
values depend only on the seed, never on the thread count.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np
import torch

DEFAULT_SEED = 20261202

# Values are generated in blocks of this many elements; each block has its own
# PCG64 stream keyed by (seed, tensor id, block index).
_BLOCK = 1 << 22

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "loss": 4, "lengths": 5, "valid": 6, "dout": 7}


@dataclass(frozen=True)
class Workload:
    name: str
    cu_seqlens: Tuple[int, ...]
    H: int
    Hkv: int
    D: int
    dtype: str               # "fp32" or "bf16"
    causal: bool
    mode: str                # "zigzag", "grid2d" or "contiguous"
    cp: int
    grid: Optional[Tuple[int, int, int]] = None   # (frames, height, width) for grid2d
    value_scale: float = 1.0
    invalid_fraction: float = 0.0
    seed: int = DEFAULT_SEED
    notes: str = field(default="", compare=False)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def n_seqs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(D)."""
        return 1.0 / math.sqrt(self.D)

    def lengths(self) -> np.ndarray:
        cu = np.asarray(self.cu_seqlens, dtype=np.int64)
        return cu[1:] - cu[:-1]


def _rng(seed: int, tensor: str, block: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=seed, spawn_key=(_TENSOR_IDS[tensor], block))
    return np.random.Generator(np.random.PCG64(ss))


def lognormal_lengths(total: int, median: float, sigma: float, lo: int, hi: int,
                      multiple: int, seed: int) -> np.ndarray:
    """Draw sequence lengths from a clipped lognormal until they sum to ``total``.

    Each length is round(exp(ln(median) + sigma*z)), clipped to [lo, hi] and
    rounded down to a multiple of ``multiple`` (so zigzag chunks divide it).
    The last sequence takes the remainder; a remainder shorter than ``lo`` is
    appended to the previous sequence.
    """
    assert total % multiple == 0
    rng = _rng(seed, "lengths")
    out = []
    acc = 0
    while True:
        z = rng.standard_normal()
        L = int(round(math.exp(math.log(median) + sigma * z)))
        L = min(max(L, lo), hi)
        L = (L // multiple) * multiple
        if acc + L >= total:
            rem = total - acc
            if rem < lo and out:
                out[-1] += rem
            else:
                out.append(rem)
            break
        out.append(L)
        acc += L
    return np.asarray(out, dtype=np.int64)


def _cu(lengths) -> Tuple[int, ...]:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return tuple(cu)


def workload(name: str, seed: int = DEFAULT_SEED) -> Workload:
    """Return the named workload with its sequence layout fixed by ``seed``."""
    if name == "tiny_packed_fp32":
        return Workload(name, (0, 64, 264, 520), H=4, Hkv=4, D=64, dtype="fp32",
                        causal=True, mode="zigzag", cp=2, value_scale=1.0, seed=seed)
    if name == "dynamic_cp_microbatch":
        cp = 4
        lens = lognormal_lengths(32768, 512.0, 1.0, 64, 16384, 2 * cp, seed)
        return Workload(name, _cu(lens), H=32, Hkv=32, D=128, dtype="bf16",
                        causal=True, mode="zigzag", cp=cp,
                        value_scale=1.0 / math.sqrt(128), invalid_fraction=0.1, seed=seed)
    if name == "long_video_200k_gqa":
        return Workload(name, (0, 1024 * 196 + 300), H=32, Hkv=8, D=128, dtype="bf16",
                        causal=True, mode="zigzag", cp=8,
                        value_scale=1.0 / math.sqrt(128), seed=seed)
    if name == "video_latent_grid2d":
        F, h, w = 16, 45, 80
        return Workload(name, (0, F * h * w), H=24, Hkv=24, D=128, dtype="bf16",
                        causal=False, mode="grid2d", cp=8, grid=(F, h, w),
                        value_scale=1.0 / math.sqrt(128), seed=seed)
    if name == "single_seq_1m_gqa":
        return Workload(name, (0, 1 << 20), H=32, Hkv=8, D=128, dtype="bf16",
                        causal=True, mode="zigzag", cp=16,
                        value_scale=1.0 / math.sqrt(128), seed=seed)
    if name == "teacher_forcing_pairs":
        # [clean ; noisy] x 8 time chunks of 3 latent frames x (30 x 52) patches; grid = (time chunks,)
        return Workload(name, (0, 2 * 8 * 3 * 30 * 52), H=24, Hkv=24, D=128, dtype="bf16",
                        causal=True, mode="paired", cp=8, grid=(8,),
                        value_scale=1.0 / math.sqrt(128), seed=seed)
    raise KeyError(name)


WORKLOADS = ("tiny_packed_fp32", "dynamic_cp_microbatch", "long_video_200k_gqa",
             "video_latent_grid2d", "single_seq_1m_gqa")


def custom(cu_seqlens, H, Hkv, D, dtype="bf16", causal=True, mode="zigzag", cp=2,
           grid=None, value_scale=None, seed=DEFAULT_SEED, name="custom") -> Workload:
    """A workload of arbitrary shape (for tests), values N(0,1)*value_scale."""
    if value_scale is None:
        value_scale = 1.0 if dtype == "fp32" else 1.0 / math.sqrt(D)
    return Workload(name, tuple(int(c) for c in cu_seqlens), H=H, Hkv=Hkv, D=D,
                    dtype=dtype, causal=causal, mode=mode, cp=cp, grid=grid,
                    value_scale=value_scale, seed=seed)


def _fill_normal(out: np.ndarray, seed: int, tensor: str, scale: float, threads: int):
    n = out.size
    nblocks = (n + _BLOCK - 1) // _BLOCK

    def work(b):
        lo = b * _BLOCK
        hi = min(n, lo + _BLOCK)
        seg = out[lo:hi]
        _rng(seed, tensor, b).standard_normal(out=seg, dtype=np.float32)
        if scale != 1.0:
            seg *= np.float32(scale)

    if nblocks == 1 or threads <= 1:
        for b in range(nblocks):
            work(b)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(nblocks)))


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def normal_tensor(shape, dtype: torch.dtype, seed: int, tensor: str, scale: float,
                  pin: bool = False, threads: Optional[int] = None) -> torch.Tensor:
    """N(0,1)*scale values of ``shape`` rounded to ``dtype``, on the host."""
    threads = threads or _threads()
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=dtype, pin_memory=pin)
    chunk = _BLOCK * 16
    tmp = np.empty(min(n, chunk), dtype=np.float32) if dtype != torch.float32 else None
    if dtype == torch.float32:
        _fill_normal(out.numpy(), seed, tensor, scale, threads)
        return out.view(*shape)
    # Generate fp32 in pieces aligned to the block size, then round to dtype.
    nb_total = (n + _BLOCK - 1) // _BLOCK
    b0 = 0
    while b0 < nb_total:
        b1 = min(nb_total, b0 + chunk // _BLOCK)
        lo, hi = b0 * _BLOCK, min(n, b1 * _BLOCK)
        piece = tmp[: hi - lo]

        def work(b, lo=lo, piece=piece):
            s = b * _BLOCK - lo
            e = min(piece.size, s + _BLOCK)
            seg = piece[s:e]
            _rng(seed, tensor, b).standard_normal(out=seg, dtype=np.float32)
            if scale != 1.0:
                seg *= np.float32(scale)

        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(b0, b1)))
        out[lo:hi].copy_(torch.from_numpy(piece))
        b0 = b1
    return out.view(*shape)


def make_qkv(w: Workload, pin: bool = False):
    """Host Q [T,H,D], K [T,Hkv,D], V [T,Hkv,D] in the workload dtype."""
    dt = w.torch_dtype
    q = normal_tensor((w.T, w.H, w.D), dt, w.seed, "q", w.value_scale, pin)
    k = normal_tensor((w.T, w.Hkv, w.D), dt, w.seed, "k", w.value_scale, pin)
    v = normal_tensor((w.T, w.Hkv, w.D), dt, w.seed, "v", w.value_scale, pin)
    return q, k, v


def make_dout(w: Workload, pin: bool = False):
    """Host upstream gradient dO [T,H,D] for the backward: N(0,1) in the
    workload dtype."""
    return normal_tensor((w.T, w.H, w.D), w.torch_dtype, w.seed, "dout", 1.0, pin)


def make_loss_inputs(w: Workload):
    """Per-token fp32 losses in [0, 12) and a uint8 valid mask with exactly
    floor(invalid_fraction*T) zeros chosen by a seeded permutation."""
    T = w.T
    loss = _rng(w.seed, "loss").random(T, dtype=np.float32) * np.float32(12.0)
    valid = np.ones(T, dtype=np.uint8)
    n_invalid = int(math.floor(w.invalid_fraction * T))
    if n_invalid:
        idx = _rng(w.seed, "valid").permutation(T)[:n_invalid]
        valid[idx] = 0
    return torch.from_numpy(loss), torch.from_numpy(valid)


def sample_rows(T: int, n: int, seed: int, must_include=()) -> np.ndarray:
    """``n`` distinct token indices drawn uniformly from [0, T) (sorted), plus
    any ``must_include`` indices (e.g. chunk boundaries)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(entropy=seed, spawn_key=(99,))))
    n = min(n, T)
    rows = rng.choice(T, size=n, replace=False)
    rows = np.union1d(rows, np.asarray([r for r in must_include if 0 <= r < T], dtype=np.int64))
    return np.sort(rows.astype(np.int64))
