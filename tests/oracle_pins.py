"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, written so that each takes an oracle object (oracle.OracleLib) and raises
AssertionError on a mismatch.  tests/test_oracle_pins.py runs them against the
oracle as built; tests/test_oracle_mutants.py runs them against copies of the
oracle with a planted mistake and expects at least one to fail.

None of these re-types the oracle's own loop: they compare it with
hand-worked fractions (tests/golden/), with an FFT identity for the DPFP block
sums, with closed forms and invariants of the recurrence, and with the
independent chunked forms of the forward and the backward (oracle/chunked.py).
"""
import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _frac(s):
    return float(Fraction(s))


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- DPFP pins
def pin_dpfp_hand(o):
    """Hand-worked DPFP values (exact with eps = 0; scaled by s/(s+eps) otherwise)."""
    for case in _load("dpfp_hand.json")["cases"]:
        k = np.array(case["k"], dtype=np.float64)
        want = np.array([_frac(x) for x in case["phi"]])
        got = o.dpfp(k, case["nu"], 0.0)
        assert got.shape == want.shape, (got.shape, want.shape)
        assert np.allclose(got, want, rtol=0, atol=1e-15), (case["k"], got, want)
        s = _frac(case["s"])
        got_eps = o.dpfp(k, case["nu"], 1e-6)
        assert np.allclose(got_eps, want * s / (s + 1e-6), rtol=1e-14, atol=1e-16)


def _autocorr_fft(x):
    """Circular autocorrelation r[i] = sum_j x[j] x[(j - i) mod n] via the FFT."""
    X = np.fft.fft(x)
    return np.real(np.fft.ifft(X * np.conj(X)))


def pin_dpfp_block_sums_fft(o):
    """Block i of the unnormalised phi sums to the circular autocorrelation of
    x = ReLU([k,-k]) at lag i; after normalisation the total is s/(s+eps)."""
    rng = _rng(1)
    for d_key, nu in [(2, 1), (3, 2), (8, 1), (8, 5), (16, 3), (16, 31), (64, 3)]:
        k = rng.standard_normal((5, d_key))
        for eps in (0.0, 1e-6, 0.5):
            phi = o.dpfp(k, nu, eps)
            n = 2 * d_key
            assert phi.shape == (5, n * nu)
            for r in range(5):
                x = np.concatenate([np.maximum(k[r], 0), np.maximum(-k[r], 0)])
                ac = _autocorr_fft(x)
                blocks = np.array([ac[i] for i in range(1, nu + 1)])
                s = blocks.sum()
                got_blocks = phi[r].reshape(nu, n).sum(axis=1)
                assert np.allclose(got_blocks, blocks / (s + eps), rtol=1e-10, atol=1e-13), \
                    (d_key, nu, eps, got_blocks, blocks / (s + eps))


def pin_dpfp_invariants(o):
    """phi >= 0; scale invariance phi(c k) = phi(k) for c > 0 (eps = 0); the
    sign flip k -> -k swaps the halves of x, which rolls every block of phi by
    d_key; block i = d_key (reachable when nu >= d_key) is identically zero;
    zero input gives zero output without NaN."""
    rng = _rng(2)
    for d_key, nu in [(2, 3), (4, 4), (8, 2), (16, 1), (5, 9)]:
        n = 2 * d_key
        k = rng.standard_normal((7, d_key))
        phi = o.dpfp(k, nu, 0.0)
        assert np.all(phi >= 0)
        assert np.allclose(o.dpfp(3.7 * k, nu, 0.0), phi, rtol=1e-12, atol=1e-15)
        flipped = o.dpfp(-k, nu, 0.0).reshape(7, nu, n)
        rolled = np.roll(phi.reshape(7, nu, n), -d_key, axis=2)
        assert np.allclose(flipped, rolled, rtol=1e-12, atol=1e-15)
        if nu >= d_key:
            assert np.all(phi.reshape(7, nu, n)[:, d_key - 1, :] == 0.0)
    z = o.dpfp(np.zeros((3, 8)), 2, 1e-6)
    assert np.all(z == 0.0) and not np.any(np.isnan(z))


def pin_dpfp_sparsity_and_gram(o):
    """Each phi entry is a product of two ReLU outputs, so for nu = 1 and a
    random k roughly a quarter of the 2*d_key entries are non-zero (adjacent
    pairs of x of the same sign); and ||phi||^2 <= (sum phi)^2 = 1 for eps = 0.
    The sparsity statistic is loose: it catches a dropped ReLU, not rounding."""
    rng = _rng(3)
    k = rng.standard_normal((4000, 64))
    phi = o.dpfp(k, 1, 0.0)
    nnz = np.count_nonzero(phi) / phi.size
    assert 0.20 < nnz < 0.30, nnz
    assert np.all(np.sum(phi * phi, axis=1) <= 1.0 + 1e-12)


# ------------------------------------------------------- recurrence pins
def pin_recurrence_hand(o):
    """Hand-worked two-step and exact-overwrite examples."""
    for case in _load("recurrence_hand.json")["cases"]:
        k = np.array(case["k"], dtype=np.float64)[None, None]
        q = np.array(case["q"], dtype=np.float64)[None, None]
        v = np.array(case["v"], dtype=np.float64)[None, None]
        beta = np.array([_frac(b) for b in case["beta"]])[None, None]
        y_want = np.array([[_frac(x) for x in row] for row in case["y"]])
        W_want = np.array([[_frac(x) for x in row] for row in case["W_final"]])
        y, W = o.delta_forward(q, k, v, beta, None, case["nu"], 0.0)
        assert np.allclose(y[0, 0], y_want, rtol=0, atol=1e-14), (case["name"], y[0, 0], y_want)
        assert np.allclose(W[0, 0], W_want, rtol=0, atol=1e-14), (case["name"], W[0, 0], W_want)
        y6, W6 = o.delta_forward(q, k, v, beta, None, case["nu"], 1e-6)
        assert np.allclose(y6[0, 0], y_want, rtol=1e-5, atol=1e-6)
        assert np.allclose(W6[0, 0], W_want, rtol=1e-5, atol=1e-6)


def _rand_inputs(rng, B, H, L, d_key, nu, d_v, with_w0=True):
    q = rng.standard_normal((B, H, L, d_key))
    k = rng.standard_normal((B, H, L, d_key))
    v = rng.standard_normal((B, H, L, d_v))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, L))))
    W0 = 0.1 * rng.standard_normal((B, H, d_v, 2 * d_key * nu)) if with_w0 else None
    return q, k, v, beta, W0


def pin_beta_zero(o):
    """beta = 0 never writes: W_final = W0 and y_t = W0 phi(q_t)."""
    rng = _rng(4)
    q, k, v, beta, W0 = _rand_inputs(rng, 2, 2, 9, 4, 2, 3)
    y, W = o.delta_forward(q, k, v, np.zeros_like(beta), W0, 2, 1e-6)
    assert np.array_equal(W, W0)
    pq = o.dpfp(q, 2, 1e-6)
    assert np.allclose(y, np.einsum("bhvd,bhtd->bhtv", W0, pq), rtol=1e-12, atol=1e-14)


def pin_one_step_closed_form(o):
    """From W0 = 0 one step gives W1 = beta v phi(k)^T and
    y1 = beta v (phi(k) . phi(q))."""
    rng = _rng(5)
    q, k, v, beta, _ = _rand_inputs(rng, 3, 2, 1, 8, 3, 5, with_w0=False)
    y, W = o.delta_forward(q, k, v, beta, None, 3, 1e-6)
    pk = o.dpfp(k, 3, 1e-6)[:, :, 0]
    pq = o.dpfp(q, 3, 1e-6)[:, :, 0]
    bv = beta[:, :, 0, None] * v[:, :, 0]
    assert np.allclose(W, bv[..., None] * pk[:, :, None, :], rtol=1e-12, atol=1e-15)
    dot = np.sum(pk * pq, axis=-1)
    assert np.allclose(y[:, :, 0], bv * dot[..., None], rtol=1e-12, atol=1e-15)


def pin_linearity(o):
    """For fixed k, q, beta the outputs are jointly linear in (V, W0)."""
    rng = _rng(6)
    q, k, v1, beta, W01 = _rand_inputs(rng, 1, 2, 11, 4, 1, 3)
    _, _, v2, _, W02 = _rand_inputs(rng, 1, 2, 11, 4, 1, 3)
    a, b = 0.7, -1.3
    y1, Wf1 = o.delta_forward(q, k, v1, beta, W01, 1, 1e-6)
    y2, Wf2 = o.delta_forward(q, k, v2, beta, W02, 1, 1e-6)
    y3, Wf3 = o.delta_forward(q, k, a * v1 + b * v2, beta, a * W01 + b * W02, 1, 1e-6)
    assert np.allclose(y3, a * y1 + b * y2, rtol=1e-10, atol=1e-12)
    assert np.allclose(Wf3, a * Wf1 + b * Wf2, rtol=1e-10, atol=1e-12)


def pin_value_channel_permutation(o):
    """Rows of W evolve independently: permuting the d_v channels of V and W0
    permutes y and W_final the same way."""
    rng = _rng(7)
    q, k, v, beta, W0 = _rand_inputs(rng, 2, 1, 10, 3, 2, 6)
    perm = rng.permutation(6)
    y, W = o.delta_forward(q, k, v, beta, W0, 2, 1e-6)
    yp, Wp = o.delta_forward(q, k, v[..., perm], beta, W0[:, :, perm], 2, 1e-6)
    assert np.allclose(yp, y[..., perm], rtol=1e-13, atol=1e-15)
    assert np.allclose(Wp, W[:, :, perm], rtol=1e-13, atol=1e-15)


def pin_contraction_bound(o):
    """Each step maps W to W (I - beta phi phi^T) + beta v phi^T and
    ||I - beta phi phi^T||_2 <= 1 (0 <= beta <= 1, ||phi||_2 <= 1), so
    ||W_t||_F <= ||W_{t-1}||_F + beta_t ||v_t|| ||phi(k_t)||."""
    rng = _rng(8)
    q, k, v, beta, W0 = _rand_inputs(rng, 1, 1, 40, 4, 1, 3)
    bound = np.linalg.norm(W0[0, 0])
    pk = o.dpfp(k, 1, 1e-6)[0, 0]
    for t in range(40):
        bound += beta[0, 0, t] * np.linalg.norm(v[0, 0, t]) * np.linalg.norm(pk[t])
    _, W = o.delta_forward(q, k, v, beta, W0, 1, 1e-6)
    assert np.linalg.norm(W[0, 0]) <= bound * (1 + 1e-12)


def pin_one_hot_recall(o):
    """d_key = 64: a key whose only non-zero entries are two adjacent positive
    values has a one-hot phi (nu = 1).  Keys on disjoint positions are
    orthogonal, so with beta = 1 every stored value is recalled exactly and a
    second write to the same key replaces the first."""
    d_key, d_v = 64, 5
    rng = _rng(9)
    pos = [3, 10, 20, 40, 3]
    L = len(pos)
    k = np.zeros((1, 1, L, d_key))
    for t, a in enumerate(pos):
        k[0, 0, t, a] = 1.0 + rng.random()
        k[0, 0, t, a + 1] = 1.0 + rng.random()
    q = k.copy()
    v = rng.standard_normal((1, 1, L, d_v))
    beta = np.ones((1, 1, L))
    y, W = o.delta_forward(q, k, v, beta, None, 1, 0.0)
    assert np.allclose(y[0, 0], v[0, 0], rtol=0, atol=1e-14)
    # query all keys against the final state: the repeated key holds its last value
    qs = k[:, :, :4].copy()
    pq = o.dpfp(qs, 1, 0.0)[0, 0]
    recalled = pq @ W[0, 0].T
    want = v[0, 0, [4, 1, 2, 3]]
    assert np.allclose(recalled, want, rtol=0, atol=1e-14)


def pin_chunked_equals_sequential(o, chunked):
    """O1 (one token at a time) equals O2 (chunked WY form) to rounding for
    every chunk length and every L in 1..9, with and without W0."""
    rng = _rng(10)
    for L in range(1, 10):
        for d_key, nu, d_v in [(2, 1, 1), (3, 2, 2), (4, 3, 5)]:
            for with_w0 in (False, True):
                q, k, v, beta, W0 = _rand_inputs(rng, 2, 1, L, d_key, nu, d_v, with_w0)
                y1, W1 = o.delta_forward(q, k, v, beta, W0, nu, 1e-6)
                for C in sorted({1, 2, 3, L}):
                    y2, W2 = chunked(q, k, v, beta, W0, nu, 1e-6, C)
                    sy = max(1.0, np.abs(y1).max())
                    sw = max(1.0, np.abs(W1).max())
                    assert np.abs(y2 - y1).max() <= 1e-12 * sy, (L, C, np.abs(y2 - y1).max())
                    assert np.abs(W2 - W1).max() <= 1e-12 * sw, (L, C)


def pin_chunked_backward_equals_sequential(o, chunked_backward):
    """The sequential backward (one token at a time, walked in reverse) equals
    the chunked backward (the transpose of the WY chunk algebra) to rounding,
    for every chunk length, with and without W0 and an incoming dW."""
    rng = _rng(13)
    for L in (1, 2, 5, 9):
        for d_key, nu, d_v in [(2, 1, 1), (3, 2, 2), (4, 3, 5)]:
            for with_w0 in (False, True):
                q, k, v, beta, W0 = _rand_inputs(rng, 2, 1, L, d_key, nu, d_v, with_w0)
                gy = rng.normal(size=v.shape)
                gW = rng.normal(size=(2, 1, d_v, 2 * d_key * nu)) if with_w0 else None
                want = o.delta_backward(q, k, v, beta, gy, W0, gW, nu, 1e-6)
                for C in sorted({1, 2, 3, L}):
                    got = chunked_backward(q, k, v, beta, gy, W0, gW, nu, 1e-6, C)
                    for name, a, b in zip(("gq", "gk", "gv", "gbeta", "gW0"), got, want):
                        scale = max(1.0, np.abs(b).max())
                        assert np.abs(a - b).max() <= 1e-11 * scale, (L, C, name, np.abs(a - b).max())


def pin_decode_stepped_equals_forward(o):
    """The token-wise variant stepped over L tokens equals the forward over
    the same tokens, in y and in the final state."""
    rng = _rng(11)
    q, k, v, beta, W0 = _rand_inputs(rng, 2, 3, 7, 4, 2, 3)
    y, W = o.delta_forward(q, k, v, beta, W0, 2, 1e-6)
    Ws = W0.copy()
    for t in range(7):
        yt, Ws = o.delta_decode_step(q[:, :, t], k[:, :, t], v[:, :, t], beta[:, :, t], Ws, 2, 1e-6)
        assert np.allclose(yt, y[:, :, t], rtol=1e-13, atol=1e-15)
    assert np.allclose(Ws, W, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------- the projections
def pin_projection_selection(o):
    """With W_all made of unit columns that pick features of x (and W_beta
    picking a feature equal to log 3, or a zero column), the projections are
    those features, split into heads, and beta is sigmoid(log 3) = 3/4 or
    sigmoid(0) = 1/2 exactly."""
    import oracle
    B, L, H, d_key, d_v = 2, 3, 2, 2, 3
    N = H * (2 * d_key + d_v + 1)
    d_model = 2 * H * d_key + H * d_v + 1
    rng = _rng(40)
    x = rng.standard_normal((B, L, d_model))
    x[..., -1] = np.log(3.0)
    W = np.zeros((d_model, N))
    for c in range(2 * H * d_key + H * d_v):
        W[c, c] = 1.0                                  # q, k, v take features 0 .. 2 H d_key + H d_v - 1
    W[-1, N - H] = 1.0                                 # head 0's beta from log 3; head 1's from a zero column
    q, k, v, beta = oracle.project(x, W, H, d_key, d_v)
    for h in range(H):
        assert np.array_equal(q[:, h], x[..., h * d_key:(h + 1) * d_key])
        assert np.array_equal(k[:, h], x[..., H * d_key + h * d_key:H * d_key + (h + 1) * d_key])
        assert np.array_equal(v[:, h], x[..., 2 * H * d_key + h * d_v:2 * H * d_key + (h + 1) * d_v])
    assert np.allclose(beta[:, 0], 0.75, rtol=0, atol=1e-15) and np.all(beta[:, 1] == 0.5)


# ---------------------------------------------------------------- backward
def _fd_loss(o, q, k, v, beta, W0, gy, gW, nu):
    y, Wf = o.delta_forward(q, k, v, beta, W0, nu, 1e-6)
    return float((gy * y).sum() + (gW * Wf).sum())


def pin_backward_finite_differences(o):
    """Every gradient of the backward (q, k, v, beta, W0) equals the central
    finite difference of L = sum(gy * y) + sum(gW * W_final) through the
    forward, entry by entry; inputs are kept away from the ReLU kink."""
    rng = _rng(30)
    B, H, L, d_key, nu, d_v = 1, 2, 5, 3, 2, 2
    d_dot = 2 * d_key * nu

    def away(a):
        return np.sign(a) * (np.abs(a) + 0.2)
    q, k = away(rng.standard_normal((B, H, L, d_key))), away(rng.standard_normal((B, H, L, d_key)))
    v = rng.standard_normal((B, H, L, d_v))
    beta = rng.uniform(0.1, 0.9, (B, H, L))
    W0 = rng.standard_normal((B, H, d_v, d_dot))
    gy = rng.standard_normal((B, H, L, d_v))
    gW = rng.standard_normal((B, H, d_v, d_dot))
    grads = o.delta_backward(q, k, v, beta, gy, W0, gW, nu, 1e-6)
    args = [q, k, v, beta, W0]
    h = 1e-6
    for which, g in enumerate(grads):
        x = args[which]
        for idx in np.ndindex(x.shape):
            xp, xm = [a.copy() for a in args], [a.copy() for a in args]
            xp[which][idx] += h
            xm[which][idx] -= h
            fd = (_fd_loss(o, *xp, gy, gW, nu) - _fd_loss(o, *xm, gy, gW, nu)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, g[idx])


def pin_backward_special_cases(o):
    """beta = 0: the state never changes, so gv = 0, gk = 0, gW0 = the summed
    read-out gradients plus gW, and gq is the plain read-out gradient; the
    backward is linear in (gy, gW)."""
    rng = _rng(31)
    B, H, L, d_key, nu, d_v = 2, 1, 6, 4, 1, 3
    d_dot = 2 * d_key * nu
    q, k = rng.standard_normal((B, H, L, d_key)), rng.standard_normal((B, H, L, d_key))
    v = rng.standard_normal((B, H, L, d_v))
    W0 = rng.standard_normal((B, H, d_v, d_dot))
    gy = rng.standard_normal((B, H, L, d_v))
    gW = rng.standard_normal((B, H, d_v, d_dot))
    gq, gk, gv, gb, gW0 = o.delta_backward(q, k, v, np.zeros((B, H, L)), gy, W0, gW, nu, 1e-6)
    pq = o.dpfp(q, nu, 1e-6)
    assert np.allclose(gv, 0.0) and np.allclose(gk, 0.0)
    assert np.allclose(gW0, gW + np.einsum("bhtv,bhtd->bhvd", gy, pq), rtol=1e-12, atol=1e-12)
    beta = rng.uniform(0, 1, (B, H, L))
    g1 = o.delta_backward(q, k, v, beta, gy, W0, gW, nu, 1e-6)
    g2 = o.delta_backward(q, k, v, beta, 2 * gy, W0, 2 * gW, nu, 1e-6)
    for x1, x2 in zip(g1, g2):
        assert np.allclose(x2, 2 * x1, rtol=1e-12, atol=1e-13)


# ------------------------------------------------- sum rule (linear attention)
def _attention_form(o, q, k, v, W0, z0, nu, normalize):
    """The kernel-attention form the sum rule is the recurrence of (the
    guide's linear self-attention section): with weights
    w_ij = phi(k_j) . phi(q_i) for j <= i,
    num_i = W0 phi(q_i) + sum_j v_j w_ij,  den_i = z0 . phi(q_i) + sum_j w_ij.
    Built from the DPFP map and plain matrix products, all L^2 weights at once."""
    pq, pk = o.dpfp(q, nu, 1e-6), o.dpfp(k, nu, 1e-6)       # [B,H,L,d_dot]
    L = q.shape[2]
    w = np.einsum("bhid,bhjd->bhij", pq, pk) * np.tril(np.ones((L, L)))
    num = np.einsum("bhij,bhjv->bhiv", w, v) + np.einsum("bhvd,bhid->bhiv", W0, pq)
    den = w.sum(-1) + np.einsum("bhd,bhid->bhi", z0, pq)
    y = num / den[..., None] if normalize else num
    W = W0 + np.einsum("bhjv,bhjd->bhvd", v, pk)
    z = z0 + pk.sum(2)
    return y, W, z


def pin_linear_attention_form(o):
    """The sum-rule recurrence equals its kernel-attention form (the ratio of
    weighted sums over all earlier tokens), normalised or not, with an
    initial state carried in."""
    rng = _rng(20)
    for normalize in (True, False):
        B, H, L, d_key, nu, d_v = 2, 3, 9, 4, 2, 3
        q, k, v = (rng.standard_normal((B, H, L, n)) for n in (d_key, d_key, d_v))
        d_dot = 2 * d_key * nu
        W0 = rng.standard_normal((B, H, d_v, d_dot))
        z0 = np.abs(rng.standard_normal((B, H, d_dot))) + 0.1    # a running sum of phi >= 0
        y1, W1, z1 = o.linear_forward(q, k, v, W0, z0, nu, normalize, 1e-6)
        y2, W2, z2 = _attention_form(o, q, k, v, W0, z0, nu, normalize)
        assert np.allclose(y1, y2, rtol=1e-11, atol=1e-13), (normalize, np.abs(y1 - y2).max())
        assert np.allclose(W1, W2, rtol=1e-12, atol=1e-13)
        assert np.allclose(z1, z2, rtol=1e-12, atol=1e-13)


def pin_linear_first_token_and_convexity(o):
    """Normalised, from a zero state: the first output is v_1 itself (the
    single weight cancels), and every output is a convex combination of the
    values so far, so it stays inside their range channel by channel."""
    rng = _rng(21)
    B, H, L, d_key, nu, d_v = 2, 2, 12, 5, 2, 4
    k = rng.standard_normal((B, H, L, d_key))
    q = k + 0.3 * rng.standard_normal((B, H, L, d_key))
    q[:, :, 0] = k[:, :, 0]                                       # phi(q_1) . phi(k_1) > 0
    v = rng.standard_normal((B, H, L, d_v))
    y, _, _ = o.linear_forward(q, k, v, None, None, nu, True, 1e-6)
    assert np.allclose(y[:, :, 0], v[:, :, 0], rtol=1e-12, atol=1e-14)
    for t in range(L):
        lo, hi = v[:, :, : t + 1].min(2), v[:, :, : t + 1].max(2)
        assert np.all(y[:, :, t] >= lo - 1e-12) and np.all(y[:, :, t] <= hi + 1e-12), t


def pin_linear_zero_denominator(o):
    """A query with phi(q) = 0 (q = 0) has a zero denominator: its output is
    0 (the reading taken where the pages give no guard), never NaN; the
    unnormalised output is 0 as well, and the state is unaffected by q."""
    rng = _rng(22)
    q = rng.standard_normal((1, 1, 4, 3))
    k = rng.standard_normal((1, 1, 4, 3))
    v = rng.standard_normal((1, 1, 4, 2))
    q[:, :, 2] = 0.0
    for normalize in (True, False):
        y, W, z = o.linear_forward(q, k, v, None, None, 1, normalize, 1e-6)
        assert np.all(np.isfinite(y)) and np.all(y[:, :, 2] == 0.0)
        _, W2, z2 = o.linear_forward(rng.standard_normal(q.shape), k, v, None, None, 1, normalize, 1e-6)
        assert np.array_equal(W, W2) and np.array_equal(z, z2)


ALL_PINS = [
    pin_dpfp_hand, pin_dpfp_block_sums_fft, pin_dpfp_invariants, pin_dpfp_sparsity_and_gram,
    pin_recurrence_hand, pin_beta_zero, pin_one_step_closed_form, pin_linearity,
    pin_value_channel_permutation, pin_contraction_bound, pin_one_hot_recall,
    pin_decode_stepped_equals_forward, pin_linear_attention_form, pin_linear_first_token_and_convexity,
    pin_linear_zero_denominator, pin_backward_finite_differences, pin_backward_special_cases,
    pin_projection_selection,
]


# ---------------------------------------------------- token-wise layer stack
# These take the OracleLib `o` (its sequence-level forward O1 is the
# independent reference for the stack's per-token state updates) and the
# stack module `st` (oracle/stack.py or a mutated copy).
def _torch_layer_norm(x, gamma=None, beta=None, eps=1e-5):
    import torch
    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    g = None if gamma is None else torch.from_numpy(np.asarray(gamma, dtype=np.float64))
    b = None if beta is None else torch.from_numpy(np.asarray(beta, dtype=np.float64))
    return torch.nn.functional.layer_norm(t, (t.shape[-1],), g, b, eps).numpy()


def _stack_layer(rng, H, d_key, d_v, d_model, d_ff, B, nu, zero=()):
    N = H * (2 * d_key + d_v + 1)
    ly = dict(W_in=rng.normal(0, 1 / np.sqrt(d_model), (d_model, N + 8)),
              W_o=rng.normal(0, 1 / np.sqrt(H * d_v), (H * d_v, d_model)), b_o=rng.normal(0, 0.1, d_model),
              ln_gamma=1 + rng.normal(0, 0.1, d_model), ln_beta=rng.normal(0, 0.1, d_model),
              W_1=rng.normal(0, 1 / np.sqrt(d_model), (d_model, d_ff)), b_1=rng.normal(0, 0.1, d_ff),
              W_2=rng.normal(0, 1 / np.sqrt(d_ff), (d_ff, d_model)), b_2=rng.normal(0, 0.1, d_model),
              W=rng.normal(0, 0.1, (B, H, d_v, 2 * d_key * nu)))
    for name in zero:
        ly[name] = np.zeros_like(ly[name])
    return ly


def pin_stack_layer_norm(o, st):
    """The norm equals PyTorch's LayerNorm (biased variance, eps inside the
    square root, then gamma and beta); without gamma / beta each row has mean
    0 and variance var / (var + eps); a constant row maps to beta."""
    rng = _rng(40)
    x = rng.normal(0.3, 2.0, (7, 48))
    g, b = rng.normal(1, 0.2, 48), rng.normal(0, 0.2, 48)
    assert np.allclose(st.layer_norm(x, g, b, 1e-5), _torch_layer_norm(x, g, b, 1e-5), rtol=0, atol=1e-12)
    z = st.layer_norm(x, None, None, 1e-5)
    var = x.var(axis=-1)
    assert np.allclose(z.mean(axis=-1), 0, atol=1e-12)
    assert np.allclose(z.var(axis=-1), var / (var + 1e-5), rtol=1e-12, atol=0)
    c = st.layer_norm(np.full((2, 48), 3.5), g, b, 1e-5)
    assert np.allclose(c, np.broadcast_to(b, c.shape), rtol=0, atol=1e-12)


def pin_stack_zero_weights(o, st):
    """With every weight matrix zero, q = k = 0 so phi = 0: no layer changes
    its fast weights or the residual stream beyond its biases (none here), and
    the output is the final norm of the input."""
    rng = _rng(41)
    H, d_key, d_v, d_model, d_ff, B, nu = 2, 4, 3, 6, 5, 3, 2
    layers = []
    for _ in range(2):
        ly = _stack_layer(rng, H, d_key, d_v, d_model, d_ff, B, nu, zero=("W_in", "W_o", "W_1", "W_2"))
        ly.update(b_o=None, b_1=None, b_2=None)
        layers.append(ly)
    x = rng.normal(0, 1, (B, d_model))
    g, b = rng.normal(1, 0.2, d_model), rng.normal(0, 0.2, d_model)
    out, res, states = st.stack_step(x, layers, H, d_key, d_v, nu, g, b)
    assert np.allclose(res, x, rtol=0, atol=0)
    assert np.allclose(out, _torch_layer_norm(x, g, b), rtol=0, atol=1e-12)
    for ly, W in zip(layers, states):
        assert np.array_equal(W, ly["W"])


def _project_sequence(o, xs, W_in, H, d_key, d_v):
    """q, k, v, beta [B, H, T, *] of the token sequence xs [T, B, d_model]."""
    from oracle import project
    return project(np.transpose(xs, (1, 0, 2)), W_in, H, d_key, d_v)


def pin_stack_state_follows_forward(o, st):
    """One layer whose output map and second feed-forward map are zero leaves
    the residual stream as it is, so stepping it token by token over a
    sequence must leave its fast weights where the sequence-level recurrence
    O1 (one C loop over the tokens) leaves them, and each output is the final
    norm of that token's input."""
    rng = _rng(42)
    H, d_key, d_v, d_model, d_ff, B, nu, T = 2, 4, 3, 8, 6, 3, 2, 5
    ly = _stack_layer(rng, H, d_key, d_v, d_model, d_ff, B, nu, zero=("W_o", "W_2"))
    ly.update(b_o=None, b_2=None)
    xs = rng.normal(0, 1, (T, B, d_model))
    W = ly["W"]
    for t in range(T):
        out, res, (W,) = st.stack_step(xs[t], [dict(ly, W=W)], H, d_key, d_v, nu)
        assert np.allclose(res, xs[t], rtol=0, atol=0)
        assert np.allclose(out, _torch_layer_norm(xs[t]), rtol=0, atol=1e-12)
    q, k, v, beta = _project_sequence(o, xs, ly["W_in"], H, d_key, d_v)
    _, W_ref = o.delta_forward(q, k, v, beta, ly["W"], nu)
    assert np.allclose(W, W_ref, rtol=1e-12, atol=1e-12)


def pin_stack_attention_output(o, st):
    """With d_model = H d_v, the identity as output map and the feed-forward
    block reduced to its last bias c2, a layer's residual output is
    x_t + y_t + b_o + c2, with y_t the heads' outputs of O1 over the sequence
    laid side by side (head h in columns h d_v .. (h + 1) d_v - 1)."""
    rng = _rng(43)
    H, d_key, d_v, d_ff, B, nu, T = 3, 4, 2, 5, 2, 1, 4
    d_model = H * d_v
    ly = _stack_layer(rng, H, d_key, d_v, d_model, d_ff, B, nu, zero=("W_1", "W_2"))
    ly.update(W_o=np.eye(d_model), b_1=None)
    xs = rng.normal(0, 1, (T, B, d_model))
    q, k, v, beta = _project_sequence(o, xs, ly["W_in"], H, d_key, d_v)
    y_ref, _ = o.delta_forward(q, k, v, beta, ly["W"], nu)
    W = ly["W"]
    for t in range(T):
        _, res, (W,) = st.stack_step(xs[t], [dict(ly, W=W)], H, d_key, d_v, nu)
        want = xs[t] + y_ref[:, :, t, :].reshape(B, d_model) + ly["b_o"] + ly["b_2"]
        assert np.allclose(res, want, rtol=1e-12, atol=1e-12)


def pin_stack_feed_forward(o, st):
    """With the projections zero (y = 0), identity linear maps in the
    feed-forward block and a first bias far above |LN(x)|, ReLU passes
    everything: x1 = x + b_o + LN(x + b_o) + b_1 + b_2; with the first bias
    far below, ReLU blocks everything: x1 = x + b_o + b_2."""
    rng = _rng(44)
    H, d_key, d_v, B, nu = 2, 4, 4, 3, 1
    d_model = d_ff = 8
    x = rng.normal(0, 1, (B, d_model))
    for sign in (1.0, -1.0):
        ly = _stack_layer(rng, H, d_key, d_v, d_model, d_ff, B, nu, zero=("W_in",))
        ly.update(W_1=np.eye(d_model), W_2=np.eye(d_model), b_1=np.full(d_ff, sign * 1e3))
        _, res, _ = st.stack_step(x, [ly], H, d_key, d_v, nu)
        a = x + ly["b_o"]
        if sign > 0:
            want = a + _torch_layer_norm(a, ly["ln_gamma"], ly["ln_beta"]) + ly["b_1"] + ly["b_2"]
        else:
            want = a + ly["b_2"]
        assert np.allclose(res, want, rtol=1e-12, atol=1e-9)


def pin_stack_composition(o, st):
    """Layers apply in order, each to the previous one's residual output and
    each with its own fast weights: a two-layer step equals the first layer's
    step followed by the second's."""
    rng = _rng(45)
    H, d_key, d_v, d_model, d_ff, B, nu = 2, 4, 4, 8, 6, 3, 2
    l1 = _stack_layer(rng, H, d_key, d_v, d_model, d_ff, B, nu)
    l2 = _stack_layer(rng, H, d_key, d_v, d_model, d_ff, B, nu)
    x = rng.normal(0, 1, (B, d_model))
    _, r12, (W1, W2) = st.stack_step(x, [l1, l2], H, d_key, d_v, nu)
    _, r1, (V1,) = st.stack_step(x, [l1], H, d_key, d_v, nu)
    _, r2, (V2,) = st.stack_step(r1, [l2], H, d_key, d_v, nu)
    assert np.allclose(r12, r2, rtol=1e-12, atol=1e-12)
    assert np.array_equal(W1, V1) and np.array_equal(W2, V2)
    assert not np.allclose(W1, l1["W"]) and not np.allclose(W2, l2["W"])


STACK_PINS = (pin_stack_layer_norm, pin_stack_zero_weights, pin_stack_state_follows_forward,
              pin_stack_attention_output, pin_stack_feed_forward, pin_stack_composition)
