"""O2: the chunked (WY / UT) form of the delta rule, numpy fp64.

TEST INFRASTRUCTURE ONLY, for tiny brute-force checks: it must equal the
sequential recurrence O1 (fw_oracle.c) to rounding for every chunk length,
which pins the algorithm the tensor-core kernel implements independently of
the GPU.

The pages give the recurrence (Fast Weights Transformer guide,
xdnf.cn/news/308600, section "FastWeightsAttention: the new update rule") and
say that the chunked library computes in parallel inside a chunk while passing
the memory between chunks (lucidrains fast-weight-attention write-up,
section 4.2 "long sequences, chunked in parallel").  They give no chunk
algorithm; this one follows from the recurrence alone:

  W_t = W_{t-1} + u_t phi(k_t)^T,   u_t = beta_t (v_t - W_{t-1} phi(k_t)).
  Inside a chunk that starts from state S, W_{t-1} = S + sum_{s<t} u_s phi(k_s)^T,
  so  u_t + beta_t sum_{s<t} (phi(k_t).phi(k_s)) u_s = beta_t (v_t - S phi(k_t)),
  i.e. (I + A) U = diag(beta) (V - K S^T) with A = strict_lower(diag(beta) K K^T).
  The read uses the updated weights, so
  y_t = S phi(q_t) + sum_{s<=t} (phi(q_t).phi(k_s)) u_s,
  i.e. Y = Q S^T + tril_inclusive(Q K^T) U,  and the next state is S + U^T K.

K, Q are the chunk's phi(k), phi(q) rows (C x d_dot), V is C x d_v, S is
d_v x d_dot.  The unit-lower system is solved by plain forward substitution.
"""
import numpy as np

from . import dpfp


def _forward_substitution_unit_lower(M, R):
    """Solve (I + M) U = R for strictly-lower M (C x C), R (C x n)."""
    C = M.shape[0]
    U = np.zeros_like(R)
    for t in range(C):
        U[t] = R[t] - M[t, :t] @ U[:t]
    return U


def delta_forward_chunked(q, k, v, beta, W0=None, nu: int = 1, eps: float = 1e-6, chunk: int = 64):
    """Same contract as oracle.delta_forward, computed chunk by chunk."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    B, H, L, d_key = q.shape
    d_v = v.shape[-1]
    d_dot = 2 * d_key * nu
    phq = dpfp(q, nu, eps)
    phk = dpfp(k, nu, eps)
    y = np.zeros((B, H, L, d_v))
    W_final = np.zeros((B, H, d_v, d_dot))
    for b in range(B):
        for h in range(H):
            S = np.zeros((d_v, d_dot)) if W0 is None else np.array(W0[b, h], dtype=np.float64)
            for c0 in range(0, L, chunk):
                c1 = min(L, c0 + chunk)
                K = phk[b, h, c0:c1]
                Q = phq[b, h, c0:c1]
                V = v[b, h, c0:c1]
                bt = beta[b, h, c0:c1]
                A = np.tril(bt[:, None] * (K @ K.T), k=-1)
                U = _forward_substitution_unit_lower(A, bt[:, None] * (V - K @ S.T))
                y[b, h, c0:c1] = Q @ S.T + np.tril(Q @ K.T) @ U
                S = S + U.T @ K
            W_final[b, h] = S
    return y, W_final


def _dpfp_backward(x_raw, gphi, nu: int, eps: float):
    """dL/dk of the DPFP map for rows of raw keys x_raw [..., d_key], given
    dL/dphi [..., 2 d_key nu]: the quotient rule of the normalisation, both
    factors of every rolled product, the two ReLU halves of [k, -k]."""
    k = np.asarray(x_raw, dtype=np.float64)
    d_key = k.shape[-1]
    n = 2 * d_key
    x = np.concatenate([np.maximum(k, 0.0), np.maximum(-k, 0.0)], axis=-1)
    prods = [x * np.roll(x, i, axis=-1) for i in range(1, nu + 1)]   # block i: x_j x_{(j - i) mod n}
    p = np.concatenate(prods, axis=-1)
    s = p.sum(axis=-1, keepdims=True) + eps
    gp = gphi / s - (gphi * p).sum(axis=-1, keepdims=True) / (s * s)
    gx = np.zeros_like(x)
    for i in range(1, nu + 1):
        g = gp[..., (i - 1) * n:i * n]
        gx += g * np.roll(x, i, axis=-1)                  # d/dx_j of x_j x_{j - i}
        gx += np.roll(g * x, -i, axis=-1)                 # d/dx_{j - i}: the product at j lands on j - i
    return gx[..., :d_key] * (k > 0) - gx[..., d_key:] * (k < 0)


def delta_backward_chunked(q, k, v, beta, gy, W0=None, gW=None, nu: int = 1, eps: float = 1e-6,
                           chunk: int = 64):
    """Same contract as oracle.delta_backward, computed chunk by chunk: the
    transpose of the chunk algebra above.  With X = V - K S^T, M = (I + A)^-1,
    T = M diag(beta), U = T X, P = tril_inclusive(Q K^T), Y = Q S^T + P U and
    S' = S + U^T K, given dY and dS' (the gradient of the next chunk's start
    state):
      dU = P^T dY + K dS'^T,  dX = T^T dU,  dT = dU X^T,  dP = tril_inclusive(dY U^T),
      dS = dS' + dY^T Q - dX^T K                      (to the previous chunk),
      dV = dX,  dQ = dY S + dP K,
      dA = -M^T (dT diag(beta)) M^T (kept strictly lower),  B = diag(beta) dA,
      dK = U dS' - dX S + dP^T Q + (B + B^T) K,
      dbeta = sum over rows of M * dT + row sums of dA * (K K^T),
    then the DPFP backward of the key and query rows.  Returns (gq, gk, gv,
    gbeta, gW0)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    gy = np.asarray(gy, dtype=np.float64)
    B, H, L, d_key = q.shape
    d_v = v.shape[-1]
    d_dot = 2 * d_key * nu
    phq = dpfp(q, nu, eps)
    phk = dpfp(k, nu, eps)
    gphq = np.zeros_like(phq)
    gphk = np.zeros_like(phk)
    gv = np.zeros_like(v)
    gbeta = np.zeros_like(beta)
    gW0 = np.zeros((B, H, d_v, d_dot))
    for b in range(B):
        for h in range(H):
            S = np.zeros((d_v, d_dot)) if W0 is None else np.array(W0[b, h], dtype=np.float64)
            saved = []
            for c0 in range(0, L, chunk):
                c1 = min(L, c0 + chunk)
                K, Q, V, bt = phk[b, h, c0:c1], phq[b, h, c0:c1], v[b, h, c0:c1], beta[b, h, c0:c1]
                C = c1 - c0
                KK = K @ K.T
                A = np.tril(bt[:, None] * KK, k=-1)
                M = np.linalg.inv(np.eye(C) + A)
                T = M * bt[None, :]
                X = V - K @ S.T
                U = T @ X
                P = np.tril(Q @ K.T)
                saved.append((c0, c1, K, Q, bt, KK, M, T, X, U, P, S))
                S = S + U.T @ K
            dS = np.zeros((d_v, d_dot)) if gW is None else np.array(gW[b, h], dtype=np.float64)
            for c0, c1, K, Q, bt, KK, M, T, X, U, P, S in reversed(saved):
                dY = gy[b, h, c0:c1]
                dU = P.T @ dY + K @ dS.T
                dX = T.T @ dU
                dT = dU @ X.T
                dP = np.tril(dY @ U.T)
                dA = np.tril(-(M.T @ (dT * bt[None, :]) @ M.T), k=-1)
                Bm = bt[:, None] * dA
                gphq[b, h, c0:c1] = dY @ S + dP @ K
                gphk[b, h, c0:c1] = U @ dS - dX @ S + dP.T @ Q + (Bm + Bm.T) @ K
                gv[b, h, c0:c1] = dX
                gbeta[b, h, c0:c1] = np.sum(M * dT, axis=0) + np.sum(dA * KK, axis=1)
                dS = dS + dY.T @ Q - dX.T @ K
            gW0[b, h] = dS
    return (_dpfp_backward(q, gphq, nu, eps), _dpfp_backward(k, gphk, nu, eps), gv, gbeta, gW0)
