"""Teacher-forcing attention on clean/noisy pairs, restated for parity.

Test infrastructure only (see the package docstring).

"Scaling video training with parallelism", section 4 (LongLive-2.0):
autoregressive teacher forcing lays out each sample as two streams over the
same time chunks, [clean history latents ; noisy target latents]; balanced
SP gives every rank the clean/noisy pair of the same time chunk, and the
teacher-forcing mask is built in the token order after the Ulysses
all-to-all.

Readings (the page is cut off before it defines the mask):

* A sample of L tokens (L even) is clean tokens [0, L/2) and noisy tokens
  [L/2, L); each stream is cut into N time chunks of floor((L/2)/N) +
  [j < (L/2) mod N] tokens (every chunk non-empty).
* The mask is the plain teacher-forcing block mask: a clean token of chunk
  j sees the clean tokens of chunks <= j; a noisy token of chunk j sees the
  clean tokens of chunks < j and the noisy tokens of chunk j.  Samples are
  independent (packed THD).
* With cp ranks and N = m*cp chunks, rank k holds chunks [k*m, (k+1)*m),
  each as its clean chunk then its noisy chunk (pair by pair); the Ulysses
  all-to-all then gives every rank all tokens in that rank order for its
  head group (mode ULYSSES2D with u = cp, r = 1 in the plan's terms).

Parity of the mask itself is "partly unpinned": it is a reading, pinned by
a dense-mask library routine, its one-chunk special case and a second
formulation, not by the page.
"""

from __future__ import annotations

import numpy as np

from .attention import _softmax_rows, kv_head, to_f64
from .plan import Plan, _check_cu, _local_cu

PAIRED = 4


def chunk_sizes(half: int, N: int):
    return [half // N + (1 if j < half % N else 0) for j in range(N)]


def token_roles(cu_seqlens, N: int):
    """Per token: sample id, stream (0 clean, 1 noisy) and time chunk."""
    cu = _check_cu(cu_seqlens)
    T = cu[-1]
    seq = np.zeros(T, dtype=np.int64)
    stream = np.zeros(T, dtype=np.int64)
    chunk = np.zeros(T, dtype=np.int64)
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        if L % 2 or L // 2 < N:
            raise ValueError(f"sample {s}: length {L} must be even with at least N tokens per stream")
        sizes = chunk_sizes(L // 2, N)
        pos = cu[s]
        for st in (0, 1):
            for j in range(N):
                seq[pos:pos + sizes[j]] = s
                stream[pos:pos + sizes[j]] = st
                chunk[pos:pos + sizes[j]] = j
                pos += sizes[j]
    return seq, stream, chunk


def allowed(cu_seqlens, N: int) -> np.ndarray:
    """Dense [T, T] teacher-forcing mask (query row, key column)."""
    seq, stream, chunk = token_roles(cu_seqlens, N)
    same = seq[:, None] == seq[None, :]
    qs, ks = stream[:, None], stream[None, :]
    qc, kc = chunk[:, None], chunk[None, :]
    clean_q = (qs == 0) & (ks == 0) & (kc <= qc)
    noisy_q = (qs == 1) & (((ks == 0) & (kc < qc)) | ((ks == 1) & (kc == qc)))
    return same & (clean_q | noisy_q)


def masked_attention(q, k, v, mask, scale: float):
    """(O [T,H,D], LSE [H,T]) of softmax attention under a dense mask."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    T, H, D = q.shape
    Hkv = k.shape[1]
    O = np.zeros((T, H, D))
    LSE = np.full((H, T), -np.inf)
    for h in range(H):
        g = kv_head(h, H, Hkv)
        S = np.where(mask, scale * (q[:, h] @ k[:, g].T), -np.inf)
        O[:, h], LSE[h] = _softmax_rows(S, v[:, g])
    return O, LSE


def paired_plan(cu_seqlens, cp: int, N: int) -> Plan:
    """Rank k holds time chunks [k*m, (k+1)*m) of every sample (m = N/cp),
    each as clean chunk then noisy chunk."""
    cu = _check_cu(cu_seqlens)
    if cp < 1 or N < 1 or N % cp:
        raise ValueError("N must be a positive multiple of cp")
    m = N // cp
    seq, stream, chunk = token_roles(cu, N)
    T = cu[-1]
    per_rank = [[] for _ in range(cp)]
    for s in range(len(cu) - 1):
        rows = np.arange(cu[s], cu[s + 1])
        for j in range(N):
            for st in (0, 1):
                sel = rows[(stream[rows] == st) & (chunk[rows] == j)]
                per_rank[j // m].extend(sel.tolist())
    index_map = np.asarray([t for r in range(cp) for t in per_rank[r]], dtype=np.int64)
    rank_offsets = np.zeros(cp + 1, dtype=np.int64)
    rank_offsets[1:] = np.cumsum([len(x) for x in per_rank])
    owner = chunk // m
    starts = [t for t in range(T) if t == 0 or seq[t] != seq[t - 1] or stream[t] != stream[t - 1]
              or chunk[t] != chunk[t - 1]]
    offs = np.asarray(starts + [T], dtype=np.int64)
    return Plan(PAIRED, cp, T, len(cu) - 1, offs, owner[starts].astype(np.int32), rank_offsets,
                _local_cu(index_map, rank_offsets, cu, cp), index_map, cp, 1)


def allowed_pairs(cu_seqlens, N: int) -> int:
    """Number of allowed (query, key) pairs, counted from the chunk sizes."""
    cu = _check_cu(cu_seqlens)
    total = 0
    for s in range(len(cu) - 1):
        sizes = chunk_sizes((cu[s + 1] - cu[s]) // 2, N)
        prefix = np.concatenate([[0], np.cumsum(sizes)])
        for j in range(N):
            total += sizes[j] * prefix[j + 1]              # clean chunk j: clean chunks <= j
            total += sizes[j] * (prefix[j] + sizes[j])     # noisy chunk j: clean < j and itself
    return int(total)


def attention_at_rows(q, k, v, cu_seqlens, N: int, rows, scale: float):
    """(O [R,H,D], LSE [H,R]) of the sampled query rows under the
    teacher-forcing mask, each row over its own key set (no T x T mask).
    Rows of the same (sample, stream, chunk) share their key set, so they are
    evaluated together."""
    seq, stream, chunk = token_roles(cu_seqlens, N)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    H, D = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    O = np.zeros((len(rows), H, D))
    LSE = np.full((H, len(rows)), -np.inf)
    groups = {}
    for n, t in enumerate(rows):
        groups.setdefault((int(seq[t]), int(stream[t]), int(chunk[t])), []).append(n)
    for (s_, st, j), idx in groups.items():
        idx = np.asarray(idx)
        ks = np.arange(int(cu[s_]), int(cu[s_ + 1]))
        if st == 0:
            keys = ks[(stream[ks] == 0) & (chunk[ks] <= j)]
        else:
            keys = ks[((stream[ks] == 0) & (chunk[ks] < j)) | ((stream[ks] == 1) & (chunk[ks] == j))]
        Qr = to_f64(q[rows[idx]])
        for g in range(Hkv):
            Kg, Vg = to_f64(k[keys, g]), to_f64(v[keys, g])
            for h in [h for h in range(H) if kv_head(h, H, Hkv) == g]:
                O[idx, h], LSE[h, idx] = _softmax_rows(scale * (Qr[:, h] @ Kg.T), Vg)
    return O, LSE
