"""Expert-parallel dispatch / combine plan (host logic).

The pages' Ascend deployment ("MoE and output stages" of the pypto DSpark page) shards the 256 routed
experts over the cards of an EP group and moves token rows with a dispatch and a combine collective.  On
one GB300 all experts are resident and the layer runs data-parallel replicas; this module is the plan for
an EP-sharded layout, exercised with CPU ranks:

* rank r owns the experts [r E/ep, (r + 1) E/ep) and runs the shared expert on its own tokens;
* dispatch: every (token, slot) pair of a rank's tokens goes to the owner of its expert, in the order
  (destination rank, expert, token, slot), with the expert id alongside;
* the receiver groups what it got by (expert, source rank, arrival order) -- expert-major, deterministic
  -- runs its grouped FFN on that order and returns every row to its source in the order it arrived;
* combine: the source puts each returned row back at its (token, slot) and sums the slots in the fixed
  order 0..k-1, then the shared row, exactly as the single-GPU combine does.

Only index bookkeeping lives here: no arithmetic of the layer.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def owner(expert: np.ndarray, n_experts: int, ep: int) -> np.ndarray:
    """Rank that owns each expert id (contiguous blocks of n_experts / ep)."""
    if n_experts % ep:
        raise ValueError("n_experts must be a multiple of the EP size")
    return np.asarray(expert) // (n_experts // ep)


@dataclass
class SendPlan:
    order: np.ndarray        # int64 [T k]: flat (token * k + slot) indices in send order
    expert: np.ndarray       # int32 [T k]: the expert of each sent row, same order
    counts: np.ndarray       # int64 [ep]: rows to each destination rank


def plan_dispatch(ids: np.ndarray, n_experts: int, ep: int) -> SendPlan:
    """Send order of one rank's routed rows: by destination rank, then expert, then token, then slot."""
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    flat_e = ids.reshape(-1)
    flat = np.arange(T * k, dtype=np.int64)
    dest = owner(flat_e, n_experts, ep)
    order = np.lexsort((flat % k, flat // k, flat_e, dest))  # last key sorts first
    counts = np.bincount(dest, minlength=ep).astype(np.int64)
    return SendPlan(order, flat_e[order].astype(np.int32), counts)


@dataclass
class RecvPlan:
    order: np.ndarray        # int64 [n]: received-row indices in expert-major compute order
    offsets: np.ndarray      # int64 [E / ep + 1]: row offsets of the local experts in that order
    local_expert: np.ndarray  # int32 [n]: local expert index of each row in compute order


def plan_receive(expert: np.ndarray, src_counts: np.ndarray, n_experts: int, ep: int, rank: int) -> RecvPlan:
    """Compute order on the receiving rank: rows grouped by local expert; within an expert by source
    rank, then arrival order (received rows arrive concatenated by source rank)."""
    expert = np.asarray(expert, dtype=np.int64)
    per = n_experts // ep
    local = expert - rank * per
    if expert.size and (local.min() < 0 or local.max() >= per):
        raise ValueError("a received row names an expert this rank does not own")
    src = np.repeat(np.arange(len(src_counts)), src_counts)
    arrival = np.arange(expert.size)
    order = np.lexsort((arrival, src, local))
    offsets = np.concatenate([[0], np.cumsum(np.bincount(local, minlength=per))]).astype(np.int64)
    return RecvPlan(order, offsets, local[order].astype(np.int32))


def combine_rows(returned: np.ndarray, plan: SendPlan, T: int, k: int, shared: np.ndarray | None) -> np.ndarray:
    """Token outputs from the rows returned in send order: slots 0..k-1 in order, then the shared row."""
    rows = np.empty((T * k,) + returned.shape[1:], dtype=returned.dtype)
    rows[plan.order] = returned
    rows = rows.reshape((T, k) + returned.shape[1:])
    out = rows[:, 0].copy()
    for j in range(1, k):
        out = out + rows[:, j]
    if shared is not None:
        out = out + shared
    return out
