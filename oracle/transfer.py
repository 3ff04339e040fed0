"""Packed transfer form of one sequence -- the plain definition.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The news summary ("system gains") reports that in the prefill/decode-
separated setting the head-aware layout cuts KV transfer bytes by up to 6.3x:
only what each head keeps travels.  This module states what travels, from
the page model (oracle/pagemodel.py) and the dense K/V:

  * rows(unit) = the positions the unit stores after n tokens, in position
    order (every slot of pagemodel.stored_positions that is not empty);
  * payload = for every (layer, KV head) unit in order, K[rows] then V[rows];
  * transfer bytes = 2 * d * bytes_per_element * sum of |rows| over units,
    against 2 * d * bytes_per_element * n * layers * KV heads for dense KV.
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np

from . import pagemodel


def unit_rows(kind: int, sink: int, window: int, idx, n: int, page: int) -> List[int]:
    """Positions a unit keeps after n tokens, ascending."""
    tab = pagemodel.stored_positions(kind, sink, window, idx, n, page)
    return sorted(p for pg in tab for p in pg if p >= 0)


def payload(policies: Sequence[Sequence[tuple]], n_layer: Sequence[int],
            k_dense: Sequence[np.ndarray], v_dense: Sequence[np.ndarray], page: int) -> np.ndarray:
    """The packed payload as a flat array of the K/V element type.

    policies[l][h] = (kind, sink, window, idx); k_dense[l], v_dense[l] are
    [n_l, Hkv, d] arrays of one layer."""
    parts = []
    for l, row in enumerate(policies):
        for h, (kind, sink, window, idx) in enumerate(row):
            r = unit_rows(kind, sink, window, idx, n_layer[l], page)
            parts.append(np.asarray(k_dense[l])[r, h].reshape(-1))
            parts.append(np.asarray(v_dense[l])[r, h].reshape(-1))
    return np.concatenate(parts) if parts else np.zeros(0)


def transfer_ratio(policies, n_layer, page: int) -> float:
    """Dense KV bytes over packed KV bytes (payload only)."""
    kept = sum(len(unit_rows(k, s, w, i, n_layer[l], page))
               for l, row in enumerate(policies) for (k, s, w, i) in row)
    dense = sum(n_layer[l] * len(row) for l, row in enumerate(policies))
    return dense / kept
