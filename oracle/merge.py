"""Exact log-sum-exp merge of attention partials (fp64).

Test infrastructure only (see the package docstring).

Ring attention computes a query block's attention one KV block at a time
("Scaling video training with parallelism", section 2, Ring Attention); the
pages do not spell out how the per-block results are combined.  The plain
reading is the identity that recombines softmax partials exactly: a partial
p holds O_p = sum_{j in p} e^{s_j} v_j / sum_{j in p} e^{s_j} and
lse_p = ln sum_{j in p} e^{s_j}, so over all partials

    M   = max_p lse_p
    lse = M + ln sum_p exp(lse_p - M)
    O   = sum_p exp(lse_p - lse) * O_p

A partial with lse_p = -inf (no allowed key) contributes nothing; if every
partial is -inf the merged row is O = 0, lse = -inf.
"""

from __future__ import annotations

import numpy as np


def lse_merge(o_parts, lse_parts):
    """Merge partials.  o_parts: list of [R,H,D]; lse_parts: list of [H,R].
    Returns (O [R,H,D] fp64, LSE [H,R] fp64)."""
    o = np.stack([np.asarray(x, dtype=np.float64) for x in o_parts])      # [P,R,H,D]
    lse = np.stack([np.asarray(x, dtype=np.float64) for x in lse_parts])  # [P,H,R]
    M = lse.max(axis=0)                                                   # [H,R]
    ok = np.isfinite(M)
    M_safe = np.where(ok, M, 0.0)
    w = np.exp(lse - M_safe[None])                                        # [P,H,R]
    Z = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        out_lse = np.where(ok, M_safe + np.log(Z), -np.inf)
    coef = np.where(ok[None], np.exp(lse - np.where(ok, out_lse, 0.0)[None]), 0.0)  # [P,H,R]
    out_o = np.einsum("phr,prhd->rhd", coef, o)
    return out_o, out_lse
