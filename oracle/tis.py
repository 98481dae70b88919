"""Oracle of the token-level truncated importance sampling (TIS) weight and the
train-inference mismatch KL estimate (TEST INFRASTRUCTURE ONLY: the same
import rules as the rest of ``oracle``).

FP8-RL page, "Method steps", step 4 (and the importance-sampling background
paragraph): for each token sampled by the FP8 rollout policy, the training
policy's log-probability lp_train and the rollout's lp_rollout give the weight
w = pi_theta / pi_fp8 = exp(lp_train - lp_rollout), truncated at C = 2.
Reading: the pages write the truncation both as clip(w, C) and as a clip to
[-C, C]; w is positive, so both mean min(w, C).

Precision-alignment page, "how the gap is measured": the mismatch is the mean,
over all generated tokens, of (rollout log-probability - training
log-probability), an estimate of KL(pi_fp8 || pi_theta) per token.

Reading for both: a token mask selects the generated (response) tokens; a
masked-out token gets weight 0 and is left out of the mean; no generated token
gives a mean of 0.  Everything in fp64 (the pages leave the precision open).
"""
from __future__ import annotations

import math

import numpy as np

TIS_CLIP = 2.0


def tis_weights(lp_train: np.ndarray, lp_rollout: np.ndarray, mask: np.ndarray | None = None,
                clip: float = TIS_CLIP) -> np.ndarray:
    """fp64 [n]: min(exp(lp_train - lp_rollout), clip) on masked-in tokens, 0 elsewhere."""
    lt = np.asarray(lp_train, dtype=np.float64)
    lr = np.asarray(lp_rollout, dtype=np.float64)
    d = lt - lr
    with np.errstate(over="ignore"):
        w = np.minimum(np.exp(d), clip)
    if mask is not None:
        w = np.where(np.asarray(mask) != 0, w, 0.0)
    return w


def mismatch_kl(lp_train: np.ndarray, lp_rollout: np.ndarray, mask: np.ndarray | None = None):
    """(mean, sum, count): the per-token mean of lp_rollout - lp_train over
    the masked-in tokens; the sum is exact (math.fsum of the exact fp64
    differences of the fp32 inputs)."""
    lt = np.asarray(lp_train, dtype=np.float64)
    lr = np.asarray(lp_rollout, dtype=np.float64)
    sel = np.ones(lt.shape, dtype=bool) if mask is None else np.asarray(mask) != 0
    terms = (lr - lt)[sel]
    total = math.fsum(terms.tolist())
    count = int(sel.sum())
    return (total / count if count else 0.0), total, count
