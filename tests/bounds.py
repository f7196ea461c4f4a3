"""Error bounds derived from the arithmetic, shared by the GPU tests."""
import numpy as np

import oracle


def delta_error_bound(f, scale, causal):
    """Elementwise bounds on the dQ, dK error caused by delta_lp (FP64, oracle values).

    The kernel forms delta = rowsum(dO o O) from its stored BF16 O ("Why
    Low-Precision Transformer Training Fails", Figure 3: delta_lp).  That O
    differs from the exact one by at most 2^-9 (P|V|) from the BF16 P in the
    P V product plus 2^-9 |O| <= 2^-9 (P|V|) from the final rounding, so
    |delta_lp - delta| <= 2^-8 sum_k |dO_ik| (P|V|)_ik =: e_i, and the
    resulting dS error is at most P_ij e_i, giving
    |dQ err| <= scale (P e) |K| and |dK err| <= scale (P e)^T |Q|.
    f: single-head dict of q, k, v, do ([N, d] arrays).
    """
    p, _, _ = oracle.probabilities(f["q"], f["k"], scale, causal)
    pv = p @ np.abs(f["v"].astype(np.float64))
    e = 2.0 ** -8 * (np.abs(f["do"].astype(np.float64)) * pv).sum(axis=1)
    pe = p * e[:, None]
    return (scale * pe @ np.abs(f["k"].astype(np.float64)),
            scale * pe.T @ np.abs(f["q"].astype(np.float64)))
