"""Chunkwise (WY) form of the gated delta rule forward, fp64 numpy.

TEST INFRASTRUCTURE (see the package docstring).  Used on tiny inputs only:
it cross-checks the token recurrence and exposes the per-chunk intermediates
that the three GPU stages produce.

Per segment and value head, tokens are cut into chunks of C (64 by default,
the chunk size FlashQLA's varlen path uses: "Findings from integrating
FlashQLA's Blackwell GDN kernels into a JAX trainer", section 1,
``prepare_chunk_indices(cu, 64)``; "FlashQLA GDN backend produces different
tokens ...", Setup, ``chunk_size=64``).  For a chunk with rows i, j (local
token index), entering state S (dk x dv):

  stage 1 (prep)
    G_i   = sum_{t <= i} g_t                          (chunk-local, inclusive)
    A_ij  = beta_i exp(G_i - G_j) (k_i . k_j)  for j < i, else 0
    Tm    = (I + A)^-1                                (forward substitution)
    W     = Tm diag(beta exp(G)) K
    U     = Tm diag(beta) V
  stage 2 (state scan)
    h     = S                                         (state entering the chunk)
    V'    = U - W S
    S    <- exp(G_last) S + (diag(exp(G_last - G)) K)^T V'
  stage 3 (output)
    O     = scale [ diag(exp(G)) Q h + (M o (Q K^T)) V' ],  M_ij = exp(G_i - G_j), j <= i

The algebra follows from unrolling the recurrence inside a chunk: the delta
form S_t = a_t S_{t-1} + k_t w_t^T with w_t = beta_t (v_t - a_t S_{t-1}^T k_t)
gives (I + A) Wmat = diag(beta) V - diag(beta exp(G)) K S, i.e. Wmat = V'.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _segment_bounds(cu, T):
    """cu_seqlens made non-decreasing by a running maximum, clamped to [0, T]."""
    out = []
    prev = 0
    for i, c in enumerate(cu):
        c = min(max(int(c), 0), T)
        if i > 0 and c < prev:
            c = prev
        out.append(c)
        prev = c
    return [(out[i], out[i + 1]) for i in range(len(out) - 1)]


def forward_substitution_inverse(A):
    """(I + A)^-1 for strictly lower-triangular A, row by row."""
    n = A.shape[0]
    Tm = np.zeros_like(A)
    for i in range(n):
        Tm[i] = -A[i, :i] @ Tm[:i] if i else 0.0
        Tm[i, i] = 1.0
    return Tm


def chunked_wy(q, k, v, g, beta, scale, h0, cu_seqlens, C=64, want_ht=True,
               intermediates=False, o_init=np.nan):
    """Chunkwise fp64 forward.  Same argument layouts as ``oracle.recurrent``.

    Returns (o, ht) or, with ``intermediates=True``, (o, ht, inter) where
    ``inter`` maps (segment, head, chunk_start) to a dict of the chunk's
    G, A, Tm, W, U, h, v_new.
    """
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    T, Hk, dk = q.shape
    H, dv = v.shape[1], v.shape[2]
    group = H // Hk
    n_seq = len(cu) - 1
    o = np.full((T, H, dv), o_init, dtype=np.float64)
    ht = np.zeros((n_seq, H, dk, dv)) if want_ht else None
    inter = {}
    for n, (s, e) in enumerate(_segment_bounds(cu, T)):
        for h in range(H):
            hk = h // group
            S = h0[n, h].copy() if h0 is not None else np.zeros((dk, dv))
            for cs in range(s, e, C):
                ce = min(cs + C, e)
                Qc, Kc, Vc = q[cs:ce, hk], k[cs:ce, hk], v[cs:ce, h]
                gc, bc = g[cs:ce, h], beta[cs:ce, h]
                # stage 1
                G = np.cumsum(gc)
                D = np.exp(G[:, None] - G[None, :])
                A = np.tril(bc[:, None] * D * (Kc @ Kc.T), -1)
                Tm = forward_substitution_inverse(A)
                W = Tm @ ((bc * np.exp(G))[:, None] * Kc)
                U = Tm @ (bc[:, None] * Vc)
                # stage 2
                h_in = S.copy()
                Vn = U - W @ S
                S = np.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * Kc).T @ Vn
                # stage 3
                M = np.tril(D)
                o[cs:ce, h] = scale * ((np.exp(G)[:, None] * Qc) @ h_in + (M * (Qc @ Kc.T)) @ Vn)
                if intermediates:
                    inter[(n, h, cs)] = dict(G=G, A=A, Tm=Tm, W=W, U=U, h=h_in, v_new=Vn)
            if want_ht:
                ht[n, h] = S
    if intermediates:
        return o, ht, inter
    return o, ht
