"""AdamW on the LoRA factors, in float64.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may use this module.

The pages train the adapters with a plain learning rate ("Fine tune an 8B model on a 4GB
laptop GPU (Soup setup)", section "Step 1, the config": lr 2e-5) and name no optimizer.
Reading: AdamW, the decoupled-weight-decay Adam of Loshchilov and Hutter, step t >= 1:

    m = b1 m + (1 - b1) g
    v = b2 v + (1 - b2) g^2
    p = p - lr ( (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps) + wd p )
"""
from __future__ import annotations

import numpy as np


def adamw_step(p, g, m, v, t, lr, b1=0.9, b2=0.999, eps=1e-8, wd=0.0):
    """Returns the updated (p, m, v) as float64 arrays."""
    p = np.asarray(p, np.float64)
    g = np.asarray(g, np.float64)
    m = b1 * np.asarray(m, np.float64) + (1.0 - b1) * g
    v = b2 * np.asarray(v, np.float64) + (1.0 - b2) * g * g
    mhat = m / (1.0 - b1 ** t)
    vhat = v / (1.0 - b2 ** t)
    p = p - lr * (mhat / (np.sqrt(vhat) + eps) + wd * p)
    return p, m, v
