"""Independent fp64 formulations that pin the oracle (test infrastructure only).

Each function restates the method in a different form from the token loop in
``gdn_oracle.cpp`` and uses different library routines for its steps, so a
mistake in one (a dropped term, a wrong sign or index, a transposed operand)
shows up as a disagreement with the other:

  * ``gdn_transition``  the gated delta rule as a product of transition
                        matrices A_t = alpha_t (I - beta_t k_t k_t^T); the
                        state after t tokens is a sum over s of
                        (A_t ... A_{s+1}) beta_s k_s v_s^T plus the decayed
                        initial state. Quadratic in T: tiny inputs only.
  * ``conv_direct``     the causal depthwise conv as a direct sum per output,
                        SiLU via scipy's logistic function.
  * ``gdn_chunked``     the chunk (WY / UT-transform) form of the same rule:
                        within a chunk of L tokens the per-token delta vectors
                        solve a unit lower-triangular system, then the output
                        and the carried state are dense products. This is the
                        plainest reading of "a chunked prefill form for long
                        prompts" (r9700-stack v0.2.3 notes, section 1, which
                        name vLLM's chunked GDN core without writing it out).
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit


def _split_heads(qkv, Hk, Hv, Dk, Dv):
    T = qkv.shape[0]
    q = qkv[:, : Hk * Dk].reshape(T, Hk, Dk)
    k = qkv[:, Hk * Dk: 2 * Hk * Dk].reshape(T, Hk, Dk)
    v = qkv[:, 2 * Hk * Dk:].reshape(T, Hv, Dv)
    return q, k, v


def _gates(a, b, A_log, dt_bias, gate_mode):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if gate_mode == 1:
        return a, b
    # softplus through logaddexp(0, x) = log(e^0 + e^x)
    g = -np.exp(np.asarray(A_log, np.float64))[None, :] * np.logaddexp(0.0, a + dt_bias[None, :])
    beta = expit(b)
    return g, beta


def _unit(x, eps):
    n = np.sqrt(np.einsum("...i,...i->...", x, x) + eps)
    return x / n[..., None]


def gdn_transition(qkv, a, b, A_log, dt_bias, Hk, Hv, Dk, Dv, S0=None,
                   scale=None, eps=1e-6, gate_mode=0):
    """One sequence. Returns (o [T][Hv][Dv], S_T [Hv][Dk][Dv])."""
    qkv = np.asarray(qkv, np.float64)
    T = qkv.shape[0]
    scale = Dk ** -0.5 if scale is None else scale
    q, k, v = _split_heads(qkv, Hk, Hv, Dk, Dv)
    g, beta = _gates(a, b, np.asarray(A_log), np.asarray(dt_bias, np.float64), gate_mode)
    group = Hv // Hk
    o = np.zeros((T, Hv, Dv))
    S_T = np.zeros((Hv, Dk, Dv))
    eye = np.eye(Dk)
    for h in range(Hv):
        kh = h // group
        kk = _unit(k[:, kh], eps)
        qq = _unit(q[:, kh], eps)
        S0h = np.zeros((Dk, Dv)) if S0 is None else np.asarray(S0[h], np.float64)
        A = [np.exp(g[t, h]) * (eye - beta[t, h] * np.outer(kk[t], kk[t])) for t in range(T)]

        def prod(t_hi, t_lo):  # A_{t_hi} ... A_{t_lo+1}; identity when empty
            P = eye.copy()
            for s in range(t_lo + 1, t_hi + 1):
                P = A[s] @ P
            return P

        for t in range(T):
            St = prod(t, -1) @ S0h
            for s in range(t + 1):
                St = St + prod(t, s) @ (beta[s, h] * np.outer(kk[s], v[s, h]))
            o[t, h] = scale * (St.T @ qq[t])
            if t == T - 1:
                S_T[h] = St
        if T == 0:
            S_T[h] = S0h
    return o, S_T


def conv_direct(x, hist, w, bias=None):
    """One sequence. x [T][C], hist [W-1][C], w [C][W] -> (y [T][C], hist_out)."""
    x = np.asarray(x, np.float64)
    hist = np.asarray(hist, np.float64)
    w = np.asarray(w, np.float64)
    W = w.shape[1]
    full = np.concatenate([hist, x], axis=0)
    T = x.shape[0]
    y = np.zeros_like(x)
    for t in range(T):
        window = full[t: t + W]                  # [W][C], oldest first
        z = np.sum(window.T * w, axis=1)
        if bias is not None:
            z = z + bias
        y[t] = z * expit(z)
    return y, full[T: T + W - 1].copy()


def gdn_chunked(qkv, a, b, A_log, dt_bias, Hk, Hv, Dk, Dv, S0=None, chunk=64,
                scale=None, eps=1e-6, gate_mode=0):
    """One sequence, chunk form. Returns (o [T][Hv][Dv], S_T [Hv][Dk][Dv]).

    Within a chunk with state S at its start, gamma_t = sum_{s<=t} g_s and
        A   = strictly-lower( beta_t e^{gamma_t-gamma_s} k_t.k_s )
        Tm  = (I + A)^{-1}
        U   = Tm diag(beta) V,    Wm = Tm diag(beta e^gamma) K
        Vn  = U - Wm S                       (the per-token delta vectors)
        O   = scale ( diag(e^gamma) Q S + (Q K^T o Gamma o causal) Vn )
        S  <- e^{gamma_L} S + (diag(e^{gamma_L - gamma}) K)^T Vn
    """
    qkv = np.asarray(qkv, np.float64)
    T = qkv.shape[0]
    scale = Dk ** -0.5 if scale is None else scale
    q, k, v = _split_heads(qkv, Hk, Hv, Dk, Dv)
    g, beta = _gates(a, b, np.asarray(A_log), np.asarray(dt_bias, np.float64), gate_mode)
    group = Hv // Hk
    o = np.zeros((T, Hv, Dv))
    S_T = np.zeros((Hv, Dk, Dv))
    for h in range(Hv):
        kh = h // group
        K = _unit(k[:, kh], eps)
        Q = _unit(q[:, kh], eps)
        V = v[:, h]
        S = np.zeros((Dk, Dv)) if S0 is None else np.asarray(S0[h], np.float64).copy()
        for c0 in range(0, T, chunk):
            sl = slice(c0, min(T, c0 + chunk))
            Kc, Qc, Vc = K[sl], Q[sl], V[sl]
            L = Kc.shape[0]
            gam = np.cumsum(g[sl, h])
            bet = beta[sl, h]
            Gam = np.exp(gam[:, None] - gam[None, :])
            low = np.tril(np.ones((L, L)), -1)
            A = low * (bet[:, None] * Gam * (Kc @ Kc.T))
            Tm = np.linalg.inv(np.eye(L) + A)
            U = Tm @ (bet[:, None] * Vc)
            Wm = Tm @ ((bet * np.exp(gam))[:, None] * Kc)
            Vn = U - Wm @ S
            causal = np.tril(np.ones((L, L)))
            P = (Qc @ Kc.T) * Gam * causal
            o[sl, h] = scale * (np.exp(gam)[:, None] * (Qc @ S) + P @ Vn)
            S = np.exp(gam[-1]) * S + (np.exp(gam[-1] - gam)[:, None] * Kc).T @ Vn
        S_T[h] = S
    return o, S_T
