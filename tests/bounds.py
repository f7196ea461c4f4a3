"""Error estimates derived from the arithmetic, shared by the GPU tests."""
import numpy as np

import oracle

# Unit roundoff of BF16 (8 significand bits, round to nearest even): a rounded
# value differs from x by at most U_BF16 * |x|.
U_BF16 = 2.0 ** -8


def delta_error_rms(f, scale, causal):
    """RMS size of the dQ, dK error that delta_lp carries (FP64, oracle values).

    The kernels form delta = rowsum(dO o O) from the stored BF16 O ("Why
    Low-Precision Transformer Training Fails", Figure 3: delta_lp).  That O is
    bf16(sum_j bf16(P~_ij) V_j / l_i) with l_i the FP32 row sum of the
    unrounded P~, so, to first order,
        O_lp - O = sum_j eps_ij P_ij V_j + eta_i o O_i,
    eps_ij the relative rounding error of P~_ij to BF16 and eta_ik that of
    the final rounding, each at most U_BF16 in size.  The row's largest P~
    is exactly 1 (exp2 of 0, or of a rounding residue below BF16 resolution),
    so eps is 0 at the row's arg max.  Hence
        e_i := delta_lp_i - delta_i = sum_j eps_ij P_ij dP_ij + sum_k eta_ik O_ik dO_ik
    with dP = dO V^T.  Treating the roundings as independent, zero-mean and
    of variance at most U_BF16^2 / 3 (uniform on [-U|x|, U|x|]):
        E[e_i^2] <= s_i^2 = U^2/3 (sum_{j != argmax} P_ij^2 dP_ij^2 + sum_k O_ik^2 dO_ik^2).
    e_i enters dS_ij = P_ij (dP_ij - delta_i) as -P_ij e_i, so
        dQ_i error = -scale e_i (P K)_i,   dK_j error = -scale sum_i P_ij e_i Q_i,
    and, the e_i being independent across rows,
        E|dQ err|^2 = scale^2 sum_i s_i^2 |(P K)_i|^2,
        E|dK err|^2 = scale^2 sum_ij P_ij^2 s_i^2 |Q_i|^2.
    Returns (sqrt E|dQ err|^2, sqrt E|dK err|^2): upper estimates of the
    Frobenius norm of the delta-induced error (not worst-case bounds).
    f: single-head dict of q, k, v, do ([N, d] arrays).
    """
    q, k, v, do = (np.asarray(f[n], dtype=np.float64) for n in ("q", "k", "v", "do"))
    p, _, _ = oracle.probabilities(q, k, scale, causal)
    o = p @ v
    dp = do @ v.T
    p_off = p.copy()
    p_off[np.arange(p.shape[0]), p.argmax(axis=1)] = 0.0
    s2 = (U_BF16 ** 2 / 3.0) * ((p_off * dp) ** 2).sum(axis=1) \
        + (U_BF16 ** 2 / 3.0) * ((o * do) ** 2).sum(axis=1)
    pk = p @ k
    rms_dq = scale * np.sqrt((s2 * (pk * pk).sum(axis=1)).sum())
    rms_dk = scale * np.sqrt(((p * p) * (s2 * (q * q).sum(axis=1))[:, None]).sum())
    return float(rms_dq), float(rms_dk)


def delta_error_worst(f, scale, causal):
    """Elementwise worst-case bounds on the dQ, dK error caused by delta_lp.

    For tiny problems (a handful of keys), where an RMS estimate says little.
    With the notation of delta_error_rms, |sum_j eps_ij P_ij V_j| <=
    U (P|V|) and the final rounding adds at most U (1 + U) (P|V|), so
    |O_lp - O| <= 2.01 U (P|V|) elementwise, |delta_lp - delta|_i <=
    2.01 U sum_k |dO_ik| (P|V|)_ik =: e_i, and the dS error P_ij e_i gives
    |dQ err| <= scale (P e) |K| and |dK err| <= scale (P e)^T |Q|.
    Returns the two elementwise bound arrays.
    """
    q, k, v, do = (np.asarray(f[n], dtype=np.float64) for n in ("q", "k", "v", "do"))
    p, _, _ = oracle.probabilities(q, k, scale, causal)
    e = 2.01 * U_BF16 * (np.abs(do) * (p @ np.abs(v))).sum(axis=1)
    pe = p * e[:, None]
    return scale * pe @ np.abs(k), scale * pe.T @ np.abs(q)
