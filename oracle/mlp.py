"""BlockPilot block-size predictor (fp64).

BlockPilot page section 3: after prefill, the full-vocabulary next-token
distribution at the last position is the request's state; a two-layer MLP
scores the candidate block sizes and the best one is used for the whole
request.  Section 2: the candidates are B-3 .. B+3 around the training block
size B.  Section 4: hidden width 2048.  Section 7: the raw probabilities
(not re-normalised, not a softmax of probabilities) are the input.

Definition:  x = softmax(last_logits) per request;  h = ReLU(x W1 + b1);
z = h W2 + b2;  choice = argmax z (lowest index on ties);
block = B - (n_out - 1) // 2 + choice.
"""
from __future__ import annotations

import numpy as np

from .attention import as_f64


def blockpilot(last_logits, W1, b1, W2, b2, block=16):
    x = as_f64(last_logits)
    x = np.exp(x - x.max(axis=1, keepdims=True))
    x /= x.sum(axis=1, keepdims=True)
    h = np.maximum(x @ as_f64(W1) + np.asarray(b1, np.float64), 0.0)
    z = h @ as_f64(W2) + np.asarray(b2, np.float64)
    choice = np.array([int(np.nonzero(row == row.max())[0][0]) for row in z], np.int32)
    n_out = z.shape[1]
    return z, choice, (block - (n_out - 1) // 2 + choice).astype(np.int32)
