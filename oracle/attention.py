"""fp64 softmax attention over packed (THD) sequences - the oracle's definition.

Test infrastructure only (see the package docstring).

For a packed batch with ``cu_seqlens`` (sequence s owns tokens
[cu[s], cu[s+1])), each query token i of sequence s and query head h attends
to the keys j of the same sequence that the mask allows:

    allowed(i, j) = seq(i) == seq(j) and (not causal or pos(j) <= pos(i))

with pos measured from the start of the sequence (THD packing keeps samples
independent: Dynamic-CP article, dynamic rescheduling and packing, Fig. 1).
Query head h reads KV head g(h) = floor(h * Hkv / H) (contiguous groups).

    s_ij   = scale * sum_d Q[i,h,d] K[j,g(h),d]
    lse_i  = m_i + ln sum_j exp(s_ij - m_i),    m_i = max_j s_ij
    O[i,h] = sum_j exp(s_ij - lse_i) V[j,g(h)]

A row with no allowed key has O = 0 and lse = -inf.  All arithmetic is fp64 on
the exact values the GPU receives.  Rows are independent, so evaluating a group
of rows with one matrix product is the same definition row by row; a matrix
product and ``np.exp`` are the only library steps.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def kv_head(h: int, H: int, Hkv: int) -> int:
    """KV head read by query head ``h``: contiguous groups of H/Hkv heads."""
    return (h * Hkv) // H


def causal_visible(kpos, qpos):
    """Causal rule inside one sequence: key position <= query position."""
    return kpos <= qpos


def to_f64(x) -> np.ndarray:
    """Exact fp64 copy of a torch tensor (fp32 or bf16) or numpy array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _softmax_rows(S: np.ndarray, V: np.ndarray):
    """Softmax-weighted sum for each row of S (masked entries are -inf).

    S is a temporary of the caller and is overwritten: S - m and its
    exponential are formed in place (the same operations as out of place, with
    fewer full-size temporaries)."""
    m = S.max(axis=1)
    ok = np.isfinite(m)
    m_safe = np.where(ok, m, 0.0)
    S -= m_safe[:, None]
    P = np.exp(S, out=S)
    l = P.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        O = (P @ V) / l[:, None]
        lse = m_safe + np.log(l)
    O[~ok] = 0.0
    lse[~ok] = -np.inf
    return O, lse


def packed_attention(q, k, v, cu_seqlens, causal: bool, scale: float, row_block: int = 256):
    """Attention of every token; returns (O [T,H,D] fp64, LSE [H,T] fp64)."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    T, H, D = q.shape
    Hkv = k.shape[1]
    cu = [int(c) for c in cu_seqlens]
    O = np.zeros((T, H, D))
    LSE = np.full((H, T), -np.inf)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(H):
            g = kv_head(h, H, Hkv)
            for i0 in range(a, b, row_block):
                i1 = min(b, i0 + row_block)
                kend = i1 if causal else b
                S = scale * (q[i0:i1, h, :] @ k[a:kend, g, :].T)
                if causal:
                    qpos = np.arange(i0, i1)[:, None] - a
                    kpos = np.arange(a, kend)[None, :] - a
                    S = np.where(causal_visible(kpos, qpos), S, -np.inf)
                O[i0:i1, h, :], LSE[h, i0:i1] = _softmax_rows(S, v[a:kend, g, :])
    return O, LSE


def seq_ids_and_positions(cu_seqlens):
    """Sequence id and in-sequence position of every token."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T = int(cu[-1])
    seq = np.zeros(T, dtype=np.int64)
    pos = np.zeros(T, dtype=np.int64)
    for s in range(len(cu) - 1):
        seq[cu[s]:cu[s + 1]] = s
        pos[cu[s]:cu[s + 1]] = np.arange(cu[s + 1] - cu[s])
    return seq, pos


def block_attention(q, k, v, cu_seqlens, q_rows, kv_rows, causal: bool, scale: float):
    """Attention of the query rows ``q_rows`` over the key rows ``kv_rows`` only.

    This is one block of blockwise (ring) attention: it returns the partial
    output normalised over the allowed keys inside ``kv_rows`` and its
    log-sum-exp, (O [len(q_rows),H,D], LSE [H,len(q_rows)]).  Rows with no
    allowed key in the block get O = 0 and lse = -inf.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    T, H, D = q.shape
    Hkv = k.shape[1]
    seq, pos = seq_ids_and_positions(cu_seqlens)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    kv_rows = np.asarray(kv_rows, dtype=np.int64)
    allowed = seq[q_rows][:, None] == seq[kv_rows][None, :]
    if causal:
        allowed &= causal_visible(pos[kv_rows][None, :], pos[q_rows][:, None])
    O = np.zeros((len(q_rows), H, D))
    LSE = np.full((H, len(q_rows)), -np.inf)
    if len(q_rows) == 0 or len(kv_rows) == 0:
        return O, LSE
    for h in range(H):
        g = kv_head(h, H, Hkv)
        S = scale * (q[q_rows, h, :] @ k[kv_rows, g, :].T)
        S = np.where(allowed, S, -np.inf)
        O[:, h, :], LSE[h, :] = _softmax_rows(S, v[kv_rows, g, :])
    return O, LSE


def attention_at_rows(q, k, v, cu_seqlens, rows, causal: bool, scale: float,
                      threads: int | None = None, batch: int | None = None):
    """Attention of the sampled query rows ``rows`` (all heads) over their full
    sequences; returns (O [R,H,D] fp64, LSE [H,R] fp64).

    Used at sizes where the whole output is too large for the CPU: each
    sampled row is still computed from its full definition.  ``q`` may be the
    full [T,H,D] tensor; ``k``/``v`` are full [T,Hkv,D] tensors (torch or
    numpy, any float dtype).  For each KV head and each sequence holding a
    sampled row, the keys up to the last sampled row are converted to fp64
    once; independent row batches run on one thread pool (numpy releases the
    GIL).  The causal rule is applied by setting the scores of the keys after
    each query's position to -inf.
    """
    rows = np.asarray(rows, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    H = q.shape[1]
    Hkv = k.shape[1]
    D = q.shape[2]
    R = len(rows)
    G = H // Hkv
    seq = np.searchsorted(cu, rows, side="right") - 1
    qr = to_f64(q[rows]) if not isinstance(q, np.ndarray) else q[rows].astype(np.float64)
    O = np.zeros((R, H, D))
    LSE = np.full((H, R), -np.inf)
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    batch = batch or max(16, 128 // G)    # about 128 (row, head) pairs per matrix product
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for g in range(Hkv):
            heads = [h for h in range(H) if kv_head(h, H, Hkv) == g]
            assert len(heads) == G
            for s in np.unique(seq):
                idx_s = np.nonzero(seq == s)[0]
                a, b = int(cu[s]), int(cu[s + 1])
                kend_s = int(rows[idx_s].max()) + 1 if causal else b
                k_s = to_f64(k[a:kend_s, g, :])   # keys of this sequence up to the last sampled row
                v_s = to_f64(v[a:kend_s, g, :])

                def work(idx, a=a, b=b, k_s=k_s, v_s=v_s):
                    rr = rows[idx]
                    kend = int(rr.max()) + 1 if causal else b
                    Qb = qr[idx][:, heads, :].reshape(len(idx) * G, D)
                    S = Qb @ k_s[: kend - a].T
                    S *= scale
                    if causal:
                        for r, qpos in enumerate(np.repeat(rr - a, G)):
                            S[r, qpos + 1:] = -np.inf     # keys after the query's position
                    Ob, Lb = _softmax_rows(S, v_s[: kend - a])
                    return idx, Ob.reshape(len(idx), G, D), Lb.reshape(len(idx), G)

                # longest batches first, so the pool's threads finish together
                batches = [idx_s[i:i + batch] for i in range(0, len(idx_s), batch)][::-1]
                for idx, Ob, Lb in ex.map(work, batches):
                    for gi, h in enumerate(heads):
                        O[idx, h, :] = Ob[:, gi, :]
                        LSE[h, idx] = Lb[:, gi]
    return O, LSE
