"""The step's cache state after the append, as the oracle computes it.

A workload holds the pools before the step (``cache_len = L - 1`` tokens per
sequence) and the step's new token in ``k_new``/``v_new``. Every reference
value a test compares against is computed by the oracle from the pools after
the append, and those pools come from ``oracle.append`` too: the input
generator only draws values and never places the new token itself
("PagedAttention: The Cache Was Storing Nothing" §1-§2.2: the cache grows by
one token per step, written into the tail block the table names).
"""

from __future__ import annotations

import oracle


def pools_after_append(wl):
    """Copies of the workload's pools with the step's token appended by the oracle."""
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, kp, vp, wl.block_tables, wl.cache_lens)
    return kp, vp


def append_in_place(wl) -> None:
    """Append the step's token into the workload's own host pools with the oracle."""
    oracle.append(wl.k_new, wl.v_new, wl.k_pool, wl.v_pool, wl.block_tables, wl.cache_lens)
