"""CPU oracle of the draft LM head.

TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle/``).

[EAGLE blog] (CSDN, section 1.2): the draft model is one decoder layer on top
of the target's features, and it reuses the target's LM head to turn its
output features into a distribution over the vocabulary.  The logits of a
feature row x are W x, W the LM head [V, H]; a library matrix product in
float64 is the whole computation.
"""
import numpy as np


def lm_head_logits(features: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """features [M, H], weight [V, H] (any float dtype) -> fp64 logits [M, V]."""
    return features.astype(np.float64) @ weight.astype(np.float64).T


def lm_head_error_bound(features: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """|sum_h x_h w_h| rounding bound of an fp32-accumulated product:
    H * 2^-24 * sum_h |x_h w_h| (the standard bound for recursive summation,
    generous for the pairwise / tensor-core orders)."""
    H = features.shape[1]
    mag = np.abs(features.astype(np.float64)) @ np.abs(weight.astype(np.float64)).T
    return H * 2.0 ** -24 * mag
