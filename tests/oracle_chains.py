"""Oracle runs over several error-feedback steps of one tensor, for the
full-size parity tests.  Kept free of torch and CUDA so that a pool of
processes (started with "spawn") can run many tensors at once on the host
cores while the GPU side waits."""
import numpy as np

import oracle


def hybrid_chain(grads, k, bits, group, rounding, seed):
    """EF + Top-K + QSGD of one tensor over len(grads) steps (step s uses
    Philox step s), starting from a zero residual.  Returns per step
    (idx, codes, scales, err')."""
    e = np.zeros(grads[0].size, np.float32)
    out = []
    for step, g in enumerate(grads):
        idx, codes, scales, e = oracle.ef_topk_quant(g, e, k, bits, group, rounding, seed, step)
        out.append((idx, codes, scales, e.copy()))
    return out


def tern_chain(grads, seed):
    """EF + TernGrad (one scale per tensor, stochastic) over len(grads)
    steps from a zero residual.  Returns per step (codes, scales, err')."""
    e = np.zeros(grads[0].size, np.float32)
    out = []
    for step, g in enumerate(grads):
        codes, scales, e = oracle.ef_quant(g, e, 2, 0, "tern", "stochastic", seed, step)
        out.append((codes, scales, e.copy()))
    return out
