"""THD-aware forward FLOP count (exact integers).

Test infrastructure only (see the package docstring).

FLOPs are counted from the real sequence lengths, never from max_seqlen, which
overestimates packed variable-length batches (Dynamic-CP article, section
"Loss computation and FLOPS statistics").  Each allowed (query, key, query
head) triple costs 2*D FLOPs in Q.K^T and 2*D in P.V; a sequence of length L
has L(L+1)/2 allowed pairs under a causal mask and L^2 without.
"""

from __future__ import annotations


def allowed_pairs(L: int, causal: bool) -> int:
    return L * (L + 1) // 2 if causal else L * L


def fwd_flops(cu_seqlens, H: int, D: int, causal: bool) -> int:
    cu = [int(c) for c in cu_seqlens]
    pairs = sum(allowed_pairs(b - a, causal) for a, b in zip(cu[:-1], cu[1:]))
    return 4 * D * H * pairs
