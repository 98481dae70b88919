"""Oracle of the MoE expert dispatch and combine around the grouped GEMM
(TEST INFRASTRUCTURE ONLY: the same import rules as the rest of ``oracle``).

Routing-replay page, "R3: Rollout Routing Replay": the rollout records each
token's top-k expert choices per MoE layer as integer indices, and the experts
are then fed from those recorded indices instead of a fresh router pass.  What
this module computes from a [T, k] index array:

* the dispatch plan: for each expert e, the rows of its segment in the grouped
  layout, filled with the (token, slot) pairs routed to e in increasing
  flattened pair order (token-major, then slot).  Readings: the pages fix no
  order inside a segment, and the stable one (increasing token) is the
  plainest; an index outside [0, E) drops its pair (a padded or unrouted
  slot), which then has no row.
* dispatch with quantisation: row r of the grouped activation is the token row
  it came from, quantised in 1x128 groups exactly as a dense activation row
  (the quantiser is per row, so gathering first and quantising afterwards is
  the definition);
* combine: out[t] = sum over the token's slots j of gate[t, j] * y[row(t, j)],
  in fp64 (the pages leave the precision open), over the slots that have a row.
  Reading: the combine weights are an input (the router's top-k weights, as the
  MoE layer of the pages' Qwen3-30B-A3B model forms them); replaying indices
  fixes which experts run, not how their outputs are weighted.

Plain Python loops where the step is a loop over pairs; fp64 numpy otherwise.
"""
from __future__ import annotations

import numpy as np


def dispatch_plan(topk: np.ndarray, experts: int):
    """Returns (offsets int32 [E+1], row_of_pair int32 [T*k], token_of_row
    int32 [T*k]).  Rows past offsets[E] (there are as many as dropped pairs)
    have token -1; dropped pairs have row -1."""
    idx = np.asarray(topk, dtype=np.int64)
    tokens, k = idx.shape
    pairs = tokens * k
    flat = idx.reshape(-1)
    counts = [0] * experts
    for e in flat:
        if 0 <= e < experts:
            counts[int(e)] += 1
    offsets = np.zeros(experts + 1, dtype=np.int32)
    for e in range(experts):
        offsets[e + 1] = offsets[e] + counts[e]
    row_of_pair = np.full(pairs, -1, dtype=np.int32)
    token_of_row = np.full(pairs, -1, dtype=np.int32)
    fill = [int(offsets[e]) for e in range(experts)]  # next free row of each segment
    for p in range(pairs):  # increasing pair order: stable within each segment
        e = int(flat[p])
        if 0 <= e < experts:
            row_of_pair[p] = fill[e]
            token_of_row[fill[e]] = p // k
            fill[e] += 1
    return offsets, row_of_pair, token_of_row


def gather_rows(x_bf16_bits: np.ndarray, token_of_row: np.ndarray) -> np.ndarray:
    """The grouped activation before quantisation: row r is x[token_of_row[r]]
    (bf16 bit patterns); rows without a token are returned as zeros and flagged
    by the caller."""
    x = np.asarray(x_bf16_bits, dtype=np.uint16)
    tor = np.asarray(token_of_row, dtype=np.int64)
    out = np.zeros((tor.size, x.shape[1]), dtype=np.uint16)
    live = tor >= 0
    out[live] = x[tor[live]]
    return out


def dispatch_quant(x_bf16_bits: np.ndarray, token_of_row: np.ndarray, fmt: int, quant_act_group):
    """Gather, then the 1x128 activation quantiser (passed in: the oracle's
    own `quant_act_group`).  Returns (codes [R, K], scales [K/128, R], live
    rows mask)."""
    g = gather_rows(x_bf16_bits, token_of_row)
    q, s = quant_act_group(g, fmt)
    return q, s, np.asarray(token_of_row) >= 0


def combine(y: np.ndarray, row_of_pair: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """fp64 [T, N]: the weighted sum of each token's expert output rows.
    y holds the expert outputs as values (fp64 or anything numpy converts)."""
    y = np.asarray(y, dtype=np.float64)
    rop = np.asarray(row_of_pair, dtype=np.int64)
    w = np.asarray(gate, dtype=np.float64)
    tokens, k = w.shape
    rop = rop.reshape(tokens, k)
    out = np.zeros((tokens, y.shape[1]), dtype=np.float64)
    for j in range(k):
        has = rop[:, j] >= 0
        out[has] += w[has, j:j + 1] * y[rop[has, j]]
    return out
