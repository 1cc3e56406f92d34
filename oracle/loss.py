"""Per-token loss normalisation over valid tokens (fp64).

Test infrastructure only (see the package docstring).

With variable-length THD packing each micro-batch holds a different number of
real tokens, so the loss is the sum over valid tokens divided by the number of
valid tokens, which keeps padding from biasing it (Dynamic-CP article, section
"Loss computation and FLOPS statistics").  With no valid token the result is 0
(and the count 0).
"""

from __future__ import annotations

import numpy as np


def token_loss_norm(loss, valid):
    """Returns (mean loss over valid tokens as fp64, valid count as int)."""
    loss = np.asarray(loss, dtype=np.float64)
    valid = np.asarray(valid) != 0
    count = int(valid.sum())
    total = float(loss[valid].sum()) if count else 0.0
    return (total / count if count else 0.0), count
