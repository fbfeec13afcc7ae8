"""Quadratic ("attention") form of the SSD scan, numpy float64, tiny inputs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The state-space duality of the Mamba-2 SSD layer ("Compiler-First State Space
Duality and Portable O(1) Autoregressive Caching for Inference", abstract:
diagonal per-head dynamics, einsum-dominated compute, a static causal mask --
Table 7) says the whole recurrence over a sequence equals one masked matrix
product per head:

    y = (Lmask o (C B^T)) (dt o x) + exp(cum a) o (C h0^T) + D x
    Lmask[i, j] = exp(sum_{k=j+1..i} a_k) for j <= i, 0 otherwise
    a_k = dt_k * A_h

and the final state is

    h_L = exp(sum_k a_k) h0 + sum_j exp(sum_{k=j+1..L-1} a_k) dt_j x_j B_j^T.

Each segment sum is an explicit sum over its own index range (not a
difference of prefix sums), so this form shares no arithmetic with the
token-by-token oracle: it is the independent cross-check of it. O(L^2) memory;
meant for L up to a few hundred.
"""
from __future__ import annotations

import numpy as np


def _segsum(a: np.ndarray) -> np.ndarray:
    """S[i, j] = sum_{k=j+1..i} a[k] for j <= i (empty sum = 0), -inf above the diagonal."""
    L = a.shape[0]
    S = np.full((L, L), -np.inf)
    for i in range(L):
        for j in range(i + 1):
            S[i, j] = float(np.sum(a[j + 1:i + 1]))
    return S


def ssd_quadratic(x, dt, A, B, C, D=None, init_state=None):
    """Quadratic form. Shapes as in ``oracle.ssd_seq``. Returns (y, final_state)."""
    x = np.asarray(x, dtype=np.float64)
    dt = np.asarray(dt, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    Bm = np.asarray(B, dtype=np.float64)
    Cm = np.asarray(C, dtype=np.float64)
    Bsz, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    y = np.zeros((Bsz, L, H, P))
    hT = np.zeros((Bsz, H, P, N))
    for b in range(Bsz):
        for h in range(H):
            g = h // (H // G)
            a = dt[b, :, h] * A[h]                      # [L]
            Lmask = np.exp(_segsum(a))                  # [L, L], zero above the diagonal
            CB = Cm[b, :, g, :] @ Bm[b, :, g, :].T      # [L, L]
            M = Lmask * CB * dt[b, None, :, h]          # column j scaled by dt_j
            yy = M @ x[b, :, h, :]                      # [L, P]
            # decay from the start of the sequence to each token, and to the end
            to_i = np.array([float(np.sum(a[:i + 1])) for i in range(L)])
            if init_state is not None:
                h0 = np.asarray(init_state, dtype=np.float64)[b, h]       # [P, N]
                yy = yy + np.exp(to_i)[:, None] * (Cm[b, :, g, :] @ h0.T)
                hT[b, h] = np.exp(float(np.sum(a))) * h0
            if D is not None:
                yy = yy + float(D[h]) * x[b, :, h, :]
            y[b, :, h, :] = yy
            # final state: contributions of every token, decayed to the end
            w = np.array([np.exp(float(np.sum(a[j + 1:]))) * dt[b, j, h] for j in range(L)])
            hT[b, h] += (x[b, :, h, :] * w[:, None]).T @ Bm[b, :, g, :]
    return y, hT
