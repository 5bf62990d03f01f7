"""CPU fp64 model of the chunkwise-parallel KDA form (test helper).

This is NOT the oracle.  It restates the chunked algebra that the CUDA prefill
kernels implement, so that the algebra itself can be checked against the
token-by-token oracle in fp64 (and so that kernel intermediates can be
inspected stage by stage).  It imports nothing from the CUDA path or from
``oracle/``.

Chunking follows the lineage essay "GPT-2부터 Kimi K3까지", section "병렬화
트릭": split the sequence into chunks of C tokens, use masked attention inside
a chunk and the carried state plus one matmul between chunks, and resolve all
deltas of a chunk at once through a Householder (UT) reparameterisation.  The
algebra for the per-channel gate, derived from the token recurrence:

  gamma_r = sum_{i<=r} g_i             (per channel, inside the chunk)
  A[r,i]  = beta_r sum_c k_rc k_ic exp(gamma_rc - gamma_ic),   i < r
  P[r,i]  =        sum_c q_rc k_ic exp(gamma_rc - gamma_ic),   i <= r
  (I + A) U = Diag(beta) (V - (K * exp(gamma)) S)
  O       = (Q * exp(gamma)) S + P U
  S_next  = Diag(exp(gamma_C)) S + (K * exp(gamma_C - gamma))^T U
"""
from __future__ import annotations

import numpy as np


def chunk_step(q, k, v, g, beta, S):
    """One chunk (L tokens, L >= 1) for one head.  Returns (O, S_next, parts)."""
    L = q.shape[0]
    gam = np.cumsum(g, axis=0)                       # [L, dk]
    Gam = np.exp(gam)
    diff = gam[:, None, :] - gam[None, :, :]         # [r, i, c] = gamma_rc - gamma_ic
    lower = np.tril(np.ones((L, L), dtype=bool))
    E = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)), 0.0)
    A = beta[:, None] * np.einsum("rc,ic,ric->ri", k, k, E)
    A = np.tril(A, -1)
    P = np.einsum("rc,ic,ric->ri", q, k, E)          # inclusive lower
    Tm = np.linalg.inv(np.eye(L) + A)
    W = Tm @ (beta[:, None] * (k * Gam))
    Ut = Tm @ (beta[:, None] * v)
    U = Ut - W @ S
    O = (q * Gam) @ S + P @ U
    Kbar = k * np.exp(gam[-1][None, :] - gam)
    S_next = Gam[-1][:, None] * S + Kbar.T @ U
    parts = dict(gamma=gam, A=A, P=P, T=Tm, W=W, Ut=Ut, U=U, Kbar=Kbar)
    return O, S_next, parts


def prefill(q, k, v, g, beta, S0, cu_seqlens, chunk):
    """Chunked prefill over a packed batch (all fp64 numpy arrays).

    Shapes as in the oracle: q, k, g [T, H, dk]; v [T, H, dv]; beta [T, H];
    S0 [N, H, dk, dv] or None.  Chunks never cross a sequence boundary; the
    last chunk of a sequence may be partial.
    """
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    o = np.zeros((T, H, dv))
    S_T = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], dtype=np.float64)
            for c0 in range(cu[n], cu[n + 1], chunk):
                c1 = min(c0 + chunk, cu[n + 1])
                O, S, _ = chunk_step(q[c0:c1, h], k[c0:c1, h], v[c0:c1, h],
                                     g[c0:c1, h], beta[c0:c1, h], S)
                o[c0:c1, h] = O
            S_T[n, h] = S
    return o, S_T
