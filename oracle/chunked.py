"""Independent fp64 chunked form of the gated-delta recurrence (oracle self-check).

Test infrastructure only. It exists to show that the chunk-parallel
formulation the prefill kernel implements is the same function as the
sequential scan of the "Delta-rule recurrence" section of "fm_kernel_ssm.h"
(the scan kept there as the permanent reference for the chunked path). The
chunking itself (64-token chunks joined by ceil(T/64) sequential state links)
follows the "Mamba-2 SSD chunked prefill scan" note of "ssm_mamba.rs"; the
algebra below is derived from the recurrence alone, since the pages print no
chunked algorithm for this layer.

Derivation (plain orientation S[i][j], per head; within one chunk let
Gam_t = g_1 + ... + g_t and S_0 the state entering the chunk):
  unrolling S_t = e^{g_t} S_{t-1} + k_t u_t^T gives
      S_t = e^{Gam_t} S_0 + sum_{s<=t} e^{Gam_t - Gam_s} k_s u_s^T;
  substituting into u_t = beta_t (v_t - e^{g_t} S_{t-1}^T k_t) gives
      (I + A) U = diag(beta) V - diag(beta e^{Gam}) K S_0,
      A[t,s] = beta_t e^{Gam_t - Gam_s} (k_t . k_s) for s < t, else 0;
  the readout o_t = scale S_t^T q_t gives
      O = scale (diag(e^{Gam}) Q S_0 + (Mask o Q K^T) U),
      Mask[t,s] = e^{Gam_t - Gam_s} for s <= t, else 0;
  and the chunk's end state is
      S_C = e^{Gam_C} S_0 + K^T diag(e^{Gam_C - Gam}) U.
Library primitives used as steps: matrix products and scipy's unit lower
triangular solve.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def chunked_scan(q, k, v, g, beta, S0, chunk, scale):
    """q, k, v [T][d]; g, beta [T]; S0 [d][d] plain orientation.

    Returns (S_T, y [T][d]) in float64.
    """
    q, k, v, g, beta = (np.asarray(a, np.float64) for a in (q, k, v, g, beta))
    S = np.array(S0, np.float64, copy=True)
    T, d = q.shape
    y = np.empty((T, d))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        n = c1 - c0
        Q, K, V = q[c0:c1], k[c0:c1], v[c0:c1]
        G, Bt = g[c0:c1], beta[c0:c1]
        Gam = np.cumsum(G)
        diff = Gam[:, None] - Gam[None, :]
        lower = np.tril(np.ones((n, n), bool), -1)
        lower_eq = np.tril(np.ones((n, n), bool), 0)
        decay_strict = np.exp(np.where(lower, diff, -np.inf))
        decay_incl = np.exp(np.where(lower_eq, diff, -np.inf))
        A = Bt[:, None] * decay_strict * (K @ K.T)
        rhs = Bt[:, None] * V - (Bt * np.exp(Gam))[:, None] * (K @ S)
        U = solve_triangular(np.eye(n) + A, rhs, lower=True, unit_diagonal=True)
        y[c0:c1] = scale * (np.exp(Gam)[:, None] * (Q @ S) + (decay_incl * (Q @ K.T)) @ U)
        S = np.exp(Gam[-1]) * S + K.T @ (np.exp(Gam[-1] - Gam)[:, None] * U)
    return S, y
