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
