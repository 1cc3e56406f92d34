"""fp64 gradients of packed softmax attention - the backward's definition.

Test infrastructure only (see the package docstring).

The pages train with this attention ("Scaling video training with
parallelism", opening section and section 2, Ring Attention: blockwise
attention with the KV blocks passed around a ring, forward and backward;
Dynamic-CP article: post-training and pre-training), so the backward pass is
the plain derivative of the forward of ``oracle.attention``.  With
s_ij = scale q_i.k_j on allowed pairs, P_ij = exp(s_ij - lse_i) and
O_i = sum_j P_ij v_j, for an upstream gradient dO the chain rule gives

    dV_j   = sum_i P_ij dO_i
    dP_ij  = dO_i . v_j
    delta_i = sum_j P_ij dP_ij            (= dO_i . O_i)
    dS_ij  = P_ij (dP_ij - delta_i)
    dQ_i   = scale sum_j dS_ij k_j
    dK_j   = scale sum_i dS_ij q_i

where dK and dV of a KV head sum over the query heads that read it.  A row
with no allowed key contributes nothing.  A ring step's backward block uses
the final (merged) O and LSE of its query rows: P over the block's keys is
exp(s - lse) with the full-row lse, so the block gradients of all ring steps
add up to the full gradients.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .attention import causal_visible, kv_head, packed_attention, seq_ids_and_positions, to_f64


def _block_grads(Qh, Kg, Vg, dOh, lse, delta, allowed, scale):
    """Gradients of one (query rows, key rows) block for one query head."""
    S = scale * (Qh @ Kg.T)
    with np.errstate(invalid="ignore", over="ignore"):
        P = np.where(allowed, np.exp(S - lse[:, None]), 0.0)
    P[~np.isfinite(lse)] = 0.0
    dV = P.T @ dOh
    dP = dOh @ Vg.T
    dS = P * (dP - delta[:, None])
    dQ = scale * (dS @ Kg)
    dK = scale * (dS.T @ Qh)
    return dQ, dK, dV


def packed_attention_bwd(q, k, v, dout, cu_seqlens, causal: bool, scale: float):
    """(dQ [T,H,D], dK [T,Hkv,D], dV [T,Hkv,D]) in fp64 from the definition:
    the forward (O, LSE) is recomputed here by ``oracle.attention``."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    T, H, D = q.shape
    Hkv = k.shape[1]
    O, LSE = packed_attention(q, k, v, cu_seqlens, causal, scale)
    delta = np.einsum("thd,thd->ht", do, O)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    cu = [int(c) for c in cu_seqlens]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        pos = np.arange(b - a)
        allowed = causal_visible(pos[None, :], pos[:, None]) if causal else np.ones((b - a, b - a), bool)
        for h in range(H):
            g = kv_head(h, H, Hkv)
            gq, gk, gv = _block_grads(q[a:b, h], k[a:b, g], v[a:b, g], do[a:b, h], LSE[h, a:b], delta[h, a:b],
                                      allowed, scale)
            dQ[a:b, h] += gq
            dK[a:b, g] += gk
            dV[a:b, g] += gv
    return dQ, dK, dV


def block_attention_bwd(q, k, v, dout, O, LSE, cu_seqlens, q_rows, kv_rows, causal: bool, scale: float):
    """One ring step's backward block: the gradients that the query rows
    ``q_rows`` send through the key rows ``kv_rows``, using the final O [T,H,D]
    and LSE [H,T] of the whole forward.  Returns (dQ [len(q_rows),H,D],
    dK [len(kv_rows),Hkv,D], dV [len(kv_rows),Hkv,D])."""
    q, k, v, do, O, LSE = to_f64(q), to_f64(k), to_f64(v), to_f64(dout), to_f64(O), to_f64(LSE)
    T, H, D = q.shape
    Hkv = k.shape[1]
    seq, pos = seq_ids_and_positions(cu_seqlens)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    kv_rows = np.asarray(kv_rows, dtype=np.int64)
    dQ = np.zeros((len(q_rows), H, D))
    dK = np.zeros((len(kv_rows), Hkv, D))
    dV = np.zeros((len(kv_rows), Hkv, D))
    if len(q_rows) == 0 or len(kv_rows) == 0:
        return dQ, dK, dV
    allowed = seq[q_rows][:, None] == seq[kv_rows][None, :]
    if causal:
        allowed &= causal_visible(pos[kv_rows][None, :], pos[q_rows][:, None])
    delta = np.einsum("thd,thd->ht", do[q_rows], O[q_rows])
    for h in range(H):
        g = kv_head(h, H, Hkv)
        gq, gk, gv = _block_grads(q[q_rows, h], k[kv_rows, g], v[kv_rows, g], do[q_rows, h], LSE[h, q_rows],
                                  delta[h], allowed, scale)
        dQ[:, h] += gq
        dK[:, g] += gk
        dV[:, g] += gv
    return dQ, dK, dV


def dq_at_rows(q, k, v, dout, cu_seqlens, rows, causal: bool, scale: float,
               threads: int | None = None, batch: int | None = None):
    """dQ [R,H,D] of the sampled query rows ``rows`` (all heads), each from
    its full definition: the row's own forward (P, O, delta) over its
    sequence's allowed keys, then dP, dS and dQ as in the module docstring.
    For sizes where the whole backward is too large for the CPU.

    For each KV head and each sequence holding a sampled row, the keys and
    values up to the last sampled row are converted to fp64 once.  The rows
    are cut into batches (the query heads that read the KV head stacked in
    one matrix product; at most ``batch`` rows, fewer where the score matrix
    would pass 2**24 entries or where fewer batches than threads would be
    left) that run on one thread pool, largest first (numpy releases the
    GIL).  The causal rule sets the scores of the keys after each query's
    position to -inf; P and dS are formed in place in the score and dP
    temporaries."""
    rows = np.asarray(rows, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G = H // Hkv
    seq = np.searchsorted(cu, rows, side="right") - 1
    qr, dor = to_f64(q[rows]), to_f64(dout[rows])
    dQ = np.zeros((len(rows), H, D))
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    batch = batch or max(16, 128 // G)    # about 128 (row, head) pairs per matrix product

    def work(idx, heads, a, n, Kg, Vg):
        rr = rows[idx]
        Qb = qr[idx][:, heads, :].reshape(len(idx) * G, D)
        dOb = dor[idx][:, heads, :].reshape(len(idx) * G, D)
        S = Qb @ Kg[:n].T
        S *= scale
        if causal:
            for r, qpos in enumerate(np.repeat(rr - a, G)):
                S[r, qpos + 1:] = -np.inf     # keys after the query's position
        S -= S.max(axis=1, keepdims=True)
        P = np.exp(S, out=S)
        P /= P.sum(axis=1, keepdims=True)
        O = P @ Vg[:n]
        delta = np.sum(dOb * O, axis=1)
        dS = dOb @ Vg[:n].T                   # dP
        dS -= delta[:, None]
        dS *= P
        return idx, heads, (scale * (dS @ Kg[:n])).reshape(len(idx), G, D)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for g in range(Hkv):
            heads = [h for h in range(H) if kv_head(h, H, Hkv) == g]
            assert len(heads) == G
            tasks = []
            for s in np.unique(seq):
                idx_s = np.nonzero(seq == s)[0]
                a, b = int(cu[s]), int(cu[s + 1])
                kend_s = int(rows[idx_s].max()) + 1 if causal else b
                Kg, Vg = to_f64(k[a:kend_s, g]), to_f64(v[a:kend_s, g])
                bs = max(1, min(batch, (1 << 24) // (G * (kend_s - a)), -(-len(idx_s) // threads)))
                for i in range(0, len(idx_s), bs):
                    idx = idx_s[i:i + bs]
                    n = (int(rows[idx].max()) + 1 if causal else b) - a
                    tasks.append((len(idx) * n, idx, a, n, Kg, Vg))
            tasks.sort(key=lambda t: -t[0])
            for f in [ex.submit(work, idx, heads, a, n, Kg, Vg) for _, idx, a, n, Kg, Vg in tasks]:
                idx, hs, dQb = f.result()
                dQ[np.ix_(idx, hs)] = dQb
    return dQ
