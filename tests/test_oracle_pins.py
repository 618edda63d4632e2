"""Pins of the f64 oracle against facts fixed outside the oracle itself.

Which pin covers which oracle routine:
  scan_kda        hand-derived three-token recurrence (golden fixture), the same case embedded
                  at D=128 inside a two-head varlen batch, beta=0 closed form, orthonormal-key
                  recall, dense-matrix product form, chunked UT/WY form, default scale.
  scan_gdn        equals scan_kda with the gate broadcast; dense product form; recall.
  conv_silu       one-hot tap weights reproduce shifted samples; ring contents after T < K-1,
                  T = K-1 and T > K-1 rows; NULL weights pass rows through.
  l2norm          output norm closed form; direction kept; eps inside the sqrt.
  gate_kda        f + dt_bias = 0 gives lb/2; monotone limits; per-channel bias indexing.
  gate_gdn        alpha + dt_bias = 0 gives -exp(A_log) ln 2; large-argument limit.
  sigmoid         closed values.
  gated_rmsnorm   w = 1, z -> +inf reduces to a plain RMSNorm closed form; gate factor.
  gated_rmsnorm_silu   the SiLU-gated mode at hand values (sigmoid(ln 3) = 3/4) and z -> +inf.
  forward         split-at-every-point state carry (bit-equal); T-token call equals T chained
                  one-token calls (bit-equal).
  forward (Hk)    grouped queries equal the plain mixer on q/k heads replicated in the tiled
                  order h % Hk (outputs, state, ring).
  scan_kda_rect   (value width Dv != key width) equals the square routine on each value-column
  (forward Dv)    block, bit for bit; the dense product form with a Dk x Dv state; the whole
                  mixer with Dv = 2D equals two mixers on the halves of each value head, and its
                  y is the gated RMSNorm over the full width.
  matvec_rows     one-hot weight rows select inputs exactly; small-integer case equals exact
  (proj6)         integer dot products; a band matrix's closed form; the six outputs' order.
Every check is a plain function so test_oracle_mutations.py can run it against mutated oracle
builds and show that each planted mistake is caught.
"""

import json
import os

import numpy as np
import pytest

from oracle import oracle as orc
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _math_to_M(S):
    return np.ascontiguousarray(S.T)


# ------------------------------------------------------------------------------------------
# scan
# ------------------------------------------------------------------------------------------

def check_three_token_golden():
    fx = json.load(open(os.path.join(GOLDEN, "three_token_recurrence.json")))
    D = fx["D"]
    tk = fx["tokens"]
    q = np.array([t["q"] for t in tk], float).reshape(3, 1, D)
    k = np.array([t["k"] for t in tk], float).reshape(3, 1, D)
    v = np.array([t["v"] for t in tk], float).reshape(3, 1, D)
    g = np.log(np.array([t["decay"] for t in tk], float)).reshape(3, 1, D)
    beta = np.array([t["beta"] for t in tk], float).reshape(3, 1)
    o, st = orc.scan_kda(q, k, v, g, beta, np.zeros((1, 1, D, D)), scale=fx["scale"])
    np.testing.assert_allclose(o.reshape(3, D), fx["expected_o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(st[0, 0], fx["expected_state_M_col_i"], rtol=0, atol=1e-14)


def check_three_token_embedded():
    """The golden case inside D=128, head 1 of 2, second sequence of a varlen pair; every other
    channel and the first sequence carry unrelated data that must not leak in."""
    fx = json.load(open(os.path.join(GOLDEN, "three_token_recurrence.json")))
    D, H = 128, 2
    ki, vj = (5, 77), (3, 100)  # key-dim channels and value-dim channels used by the case
    rng = _rng(1)
    T0 = 4  # first sequence: random data
    rows = T0 + 3
    q = np.zeros((rows, H, D)); k = np.zeros((rows, H, D)); v = np.zeros((rows, H, D))
    g = np.zeros((rows, H, D)); beta = np.zeros((rows, H))
    q[:T0] = rng.standard_normal((T0, H, D)); k[:T0] = _unit_rows(rng, (T0, H, D))
    v[:T0] = rng.standard_normal((T0, H, D)); g[:T0] = -rng.uniform(0, 1, (T0, H, D))
    beta[:T0] = rng.uniform(0, 1, (T0, H))
    # head 0 of the second sequence: random too
    q[T0:, 0] = rng.standard_normal((3, D)); k[T0:, 0] = _unit_rows(rng, (3, D))
    v[T0:, 0] = rng.standard_normal((3, D)); g[T0:, 0] = -rng.uniform(0, 1, (3, D))
    beta[T0:, 0] = 0.3
    for t, tok in enumerate(fx["tokens"]):
        r = T0 + t
        for a in range(2):
            q[r, 1, ki[a]] = tok["q"][a]
            k[r, 1, ki[a]] = tok["k"][a]
            v[r, 1, vj[a]] = tok["v"][a]
            g[r, 1, ki[a]] = np.log(tok["decay"][a])
        beta[r, 1] = tok["beta"]
    S0 = np.zeros((2, H, D, D))
    S0[0] = rng.standard_normal((H, D, D)) * 0.1
    S0[1, 0] = rng.standard_normal((D, D)) * 0.1
    o, st = orc.scan_kda(q, k, v, g, beta, S0, cu_seqlens=[0, T0, rows], scale=1.0)
    exp_o = np.array(fx["expected_o"])
    got = o[T0:, 1]
    want = np.zeros((3, D))
    want[:, vj[0]] = exp_o[:, 0]
    want[:, vj[1]] = exp_o[:, 1]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)
    M = st[1, 1]
    Sexp = np.array(fx["expected_S_math_rows_key_dim"])
    want_M = np.zeros((D, D))
    for a in range(2):
        for b in range(2):
            want_M[vj[b], ki[a]] = Sexp[a, b]
    np.testing.assert_allclose(M, want_M, rtol=0, atol=1e-14)
    # the other units match the dense product form on their own data
    for n, (r0, r1), h in ((0, (0, T0), 0), (0, (0, T0), 1), (1, (T0, rows), 0)):
        ob, Sb = brute.dense_product_scan(q[r0:r1, h], k[r0:r1, h], v[r0:r1, h], g[r0:r1, h],
                                          beta[r0:r1, h], S0[n, h].T, 1.0)
        np.testing.assert_allclose(o[r0:r1, h], ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(st[n, h], Sb.T, rtol=0, atol=1e-12)


def check_beta_zero_closed_form():
    """beta = 0: S_T = Diag(exp(sum g)) S0 and o_t = scale (Diag(exp(G_t)) S0)^T q_t."""
    rng = _rng(2)
    T, D = 6, 8
    q = rng.standard_normal((T, 1, D)); k = _unit_rows(rng, (T, 1, D))
    v = rng.standard_normal((T, 1, D)); g = -rng.uniform(0, 2, (T, 1, D))
    S0 = rng.standard_normal((D, D))
    o, st = orc.scan_kda(q, k, v, g, np.zeros((T, 1)), _math_to_M(S0)[None, None], scale=0.5)
    G = np.cumsum(g[:, 0], axis=0)
    for t in range(T):
        want = 0.5 * (np.exp(G[t])[:, None] * S0).T @ q[t, 0]
        np.testing.assert_allclose(o[t, 0], want, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(st[0, 0], (np.exp(G[-1])[:, None] * S0).T, rtol=1e-13,
                               atol=1e-13)


def check_orthonormal_recall(scan=None):
    """g = 0, beta = 1, keys = an orthonormal basis, S0 = 0: after token t, S^T k_s = v_s for
    every s <= t, so the readout with q_t = k_t is scale * v_t, and S_T^T k_j = v_j for all j."""
    scan = scan or orc.scan_kda
    rng = _rng(3)
    D = 8
    Qm, _ = np.linalg.qr(rng.standard_normal((D, D)))
    keys = Qm.T  # rows orthonormal
    v = rng.standard_normal((D, 1, D))
    k = keys.reshape(D, 1, D)
    g = np.zeros((D, 1, D)) if scan is orc.scan_kda else np.zeros((D, 1))
    o, st = scan(k, k, v, g, np.ones((D, 1)), np.zeros((1, 1, D, D)), scale=0.25)
    np.testing.assert_allclose(o[:, 0], 0.25 * v[:, 0], rtol=0, atol=1e-12)
    S = st[0, 0].T
    np.testing.assert_allclose(keys @ S, v[:, 0], rtol=0, atol=1e-12)


def check_dense_product_form():
    rng = _rng(4)
    for D, T in ((2, 5), (4, 9), (8, 12)):
        q = rng.standard_normal((T, 1, D)); k = _unit_rows(rng, (T, 1, D))
        v = rng.standard_normal((T, 1, D)); g = -5 * rng.uniform(0, 1, (T, 1, D))
        beta = rng.uniform(0, 1, (T, 1)); S0 = rng.standard_normal((D, D))
        o, st = orc.scan_kda(q, k, v, g, beta, _math_to_M(S0)[None, None], scale=0.7)
        ob, Sb = brute.dense_product_scan(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0,
                                          0.7)
        np.testing.assert_allclose(o[:, 0], ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(st[0, 0], Sb.T, rtol=1e-12, atol=1e-12)


def check_chunked_form_every_chunk_size():
    rng = _rng(5)
    for D, T in ((2, 7), (4, 10), (8, 12)):
        q = rng.standard_normal((T, 1, D)); k = _unit_rows(rng, (T, 1, D))
        v = rng.standard_normal((T, 1, D)); g = -5 * rng.uniform(0, 1, (T, 1, D))
        beta = rng.uniform(0, 1, (T, 1)); S0 = rng.standard_normal((D, D))
        o, st = orc.scan_kda(q, k, v, g, beta, _math_to_M(S0)[None, None], scale=0.3)
        for chunk in range(1, T + 1):
            oc, Sc = brute.chunked_scan(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0, 0.3,
                                        chunk)
            scale_o = max(1.0, np.abs(o).max())
            np.testing.assert_allclose(o[:, 0] / scale_o, oc / scale_o, rtol=0, atol=1e-11)
            np.testing.assert_allclose(st[0, 0], Sc.T, rtol=1e-10, atol=1e-11)


def check_default_scale():
    """scale defaults to head_dim^-1/2 and multiplies the readout only."""
    rng = _rng(6)
    T, D = 4, 16
    args = (rng.standard_normal((T, 1, D)), _unit_rows(rng, (T, 1, D)),
            rng.standard_normal((T, 1, D)), -rng.uniform(0, 1, (T, 1, D)),
            rng.uniform(0, 1, (T, 1)), rng.standard_normal((1, 1, D, D)))
    o1, s1 = orc.scan_kda(*args, scale=1.0)
    od, sd = orc.scan_kda(*args)
    np.testing.assert_allclose(od, o1 / 4.0, rtol=1e-14, atol=0)
    np.testing.assert_array_equal(sd, s1)


def check_gdn_equals_broadcast_kda():
    rng = _rng(7)
    T, H, D = 9, 3, 8
    q = rng.standard_normal((T, H, D)); k = _unit_rows(rng, (T, H, D))
    v = rng.standard_normal((T, H, D)); gs = -rng.uniform(0, 3, (T, H))
    beta = rng.uniform(0, 1, (T, H)); S0 = rng.standard_normal((1, H, D, D))
    og, sg = orc.scan_gdn(q, k, v, gs, beta, S0)
    ok, sk = orc.scan_kda(q, k, v, np.repeat(gs[:, :, None], D, axis=2), beta, S0)
    np.testing.assert_allclose(og, ok, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sg, sk, rtol=1e-12, atol=1e-12)
    # and the scalar routine against the dense product form directly
    for h in range(H):
        ob, Sb = brute.dense_product_scan(q[:, h], k[:, h], v[:, h],
                                          np.repeat(gs[:, h, None], D, axis=1), beta[:, h],
                                          S0[0, h].T, D ** -0.5)
        np.testing.assert_allclose(og[:, h], ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sg[0, h], Sb.T, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------
# prologue / epilogue steps
# ------------------------------------------------------------------------------------------

def _silu(x):
    return x / (1.0 + np.exp(-x))


def check_conv_one_hot_shift():
    """w[c] = e_{K-1-s} makes y_t = silu(sample s steps back); the ring is the last K-1 raw
    samples of [ring_in, rows], oldest first, for T below, at and above K-1."""
    rng = _rng(8)
    K, Cch = 4, 3 * 5
    for T in (1, 2, 3, 7):
        x = rng.standard_normal((T, Cch))
        ring = rng.standard_normal((Cch, K - 1))
        w = np.zeros((Cch, K))
        shifts = np.arange(Cch) % K
        w[np.arange(Cch), K - 1 - shifts] = 1.0
        y, ro = orc.conv_silu(x, w, ring)
        for c in range(Cch):
            hist = np.concatenate([ring[c], x[:, c]])  # xt
            for t in range(T):
                np.testing.assert_allclose(y[t, c], _silu(hist[K - 1 + t - shifts[c]]),
                                           rtol=1e-15, atol=0)
            np.testing.assert_array_equal(ro[c], hist[T:T + K - 1])
        # NULL weights: rows pass through unchanged
        y0, r0 = orc.conv_silu(x, None, None)
        np.testing.assert_array_equal(y0, x)
        assert r0 is None


def check_conv_taps_general():
    """Random weights: y_t = silu(sum_j w_j xt[t+j]) written as a correlation over the padded
    history, compared at 1e-15."""
    rng = _rng(9)
    K, Cch, T = 4, 6, 9
    x = rng.standard_normal((T, Cch)); ring = rng.standard_normal((Cch, K - 1))
    w = rng.standard_normal((Cch, K))
    y, _ = orc.conv_silu(x, w, ring)
    for c in range(Cch):
        hist = np.concatenate([ring[c], x[:, c]])
        want = _silu(np.correlate(hist, w[c], mode="valid"))
        np.testing.assert_allclose(y[:, c], want, rtol=1e-14, atol=1e-15)


def check_l2norm():
    rng = _rng(10)
    D = 16
    x = rng.standard_normal((5, D)) * np.array([1e-4, 1e-2, 1, 10, 1e3])[:, None]
    eps = 1e-6
    y = orc.l2norm(x, D, eps)
    ss = (x * x).sum(1)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.sqrt(ss / (ss + eps)), rtol=1e-13)
    cos = (x * y).sum(1) / (np.linalg.norm(x, axis=1) * np.linalg.norm(y, axis=1))
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)
    z = orc.l2norm(np.zeros((1, D)), D, eps)
    np.testing.assert_array_equal(z, 0.0)


def check_gates():
    H, D = 2, 4
    C = H * D
    dt = np.linspace(-1, 1, C)
    a_log = np.log(np.array([2.0, 8.0]))
    f = -np.tile(dt, (3, 1))  # f + dt_bias = 0 everywhere
    np.testing.assert_array_equal(orc.gate_kda(f, dt, a_log, -5.0), -2.5)
    f2 = np.tile(dt * 0, (1, 1)) + 1e3
    np.testing.assert_allclose(orc.gate_kda(f2, dt, a_log, -5.0), -5.0, rtol=1e-15)
    f3 = np.zeros((1, C)) - 1e3
    assert np.all(orc.gate_kda(f3, dt, a_log, -5.0) > -1e-100)
    # per-channel bias and per-head rate: one channel differs
    f4 = np.zeros((1, C)); dt4 = np.zeros(C); dt4[5] = 0.3
    g4 = orc.gate_kda(f4, dt4, a_log, -5.0)
    want = -5.0 / (1.0 + np.exp(-(8.0 * 0.3)))
    np.testing.assert_allclose(g4[0, 5], want, rtol=1e-15)
    assert np.all(np.delete(g4[0], 5) == -2.5)
    # GDN: alpha + dt_bias = 0 -> softplus(0) = ln 2
    alpha = -np.array([[0.5, -0.25]])
    gg = orc.gate_gdn(alpha, np.array([0.5, -0.25]), a_log)
    np.testing.assert_allclose(gg[0], -np.exp(a_log) * np.log(2.0), rtol=1e-15)
    gbig = orc.gate_gdn(np.array([[40.0, -40.0]]), np.zeros(2), np.zeros(2))
    np.testing.assert_allclose(gbig[0], [-40.0, -np.exp(-40.0)], rtol=1e-14)
    np.testing.assert_array_equal(orc.sigmoid(np.array([0.0])), [0.5])


def check_gated_rmsnorm():
    rng = _rng(11)
    D = 32
    o = rng.standard_normal((4, D))
    eps = 1e-6
    y = orc.gated_rmsnorm(o, np.ones(D), np.full((4, D), 1e3), eps)
    want = o / np.sqrt((o ** 2).mean(1, keepdims=True) + eps)
    np.testing.assert_allclose(y, want, rtol=1e-14)
    w = rng.uniform(0.5, 1.5, D); z = rng.standard_normal((4, D))
    y2 = orc.gated_rmsnorm(o, w, z, eps)
    np.testing.assert_allclose(y2, want * w / (1 + np.exp(-z)), rtol=1e-13)


def check_gated_rmsnorm_silu():
    """The SiLU-gated mode (GDN's gated_rmsnorm): hand values, D = 2, o = (3, 4), w = 1, eps = 0,
    so o / rms = (3, 4) / sqrt(12.5); silu(0) = 0 and silu(ln 3) = (3/4) ln 3 exactly
    (sigmoid(ln 3) = 3/4).  And z -> +inf: silu(z) = z, a plain RMSNorm times z."""
    o = np.array([[3.0, 4.0], [3.0, 4.0]])
    z = np.array([[0.0, np.log(3.0)], [np.log(3.0), 0.0]])
    y = orc.gated_rmsnorm(o, np.ones(2), z, 0.0, gate="silu")
    r = np.sqrt(12.5)
    np.testing.assert_allclose(y, [[0.0, 4.0 / r * 0.75 * np.log(3.0)],
                                   [3.0 / r * 0.75 * np.log(3.0), 0.0]], rtol=1e-15, atol=0)
    rng = _rng(12)
    D = 32
    o = rng.standard_normal((4, D))
    y = orc.gated_rmsnorm(o, np.ones(D), np.full((4, D), 1e3), 1e-6, gate="silu")
    want = o / np.sqrt((o ** 2).mean(1, keepdims=True) + 1e-6) * 1e3
    np.testing.assert_allclose(y, want, rtol=1e-14)


# ------------------------------------------------------------------------------------------
# whole-mixer state carry
# ------------------------------------------------------------------------------------------

def _tiny_layer(rng, T, H=2, D=8, K=4, gate_mode=0):
    C = H * D
    d = dict(q_raw=rng.standard_normal((T, C)), k_raw=rng.standard_normal((T, C)),
             v_raw=rng.standard_normal((T, C)), conv_w=0.5 * rng.standard_normal((3 * C, K)),
             ring_in=rng.standard_normal((1, 3 * C, K - 1)),
             f_raw=rng.standard_normal((T, C) if gate_mode == 0 else (T, H)),
             dt_bias=0.5 * rng.standard_normal(C if gate_mode == 0 else H),
             a_log=np.log(rng.uniform(1, 16, H)), beta_raw=rng.standard_normal((T, H)),
             state_in=0.02 * rng.standard_normal((1, H, D, D)),
             norm_w=1 + 0.1 * rng.standard_normal(D), gate_raw=rng.standard_normal((T, C)))
    return d


def _slice_rows(d, r0, r1):
    out = dict(d)
    for key in ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw"):
        out[key] = d[key][r0:r1]
    return out


def check_split_state_carry():
    rng = _rng(12)
    T, H, D = 9, 2, 8
    for gate_mode in (0, 1):
        d = _tiny_layer(rng, T, H, D, gate_mode=gate_mode)
        full = orc.forward(H=H, D=D, gate_mode=gate_mode, **d)
        for p in range(0, T + 1):
            a = orc.forward(H=H, D=D, gate_mode=gate_mode, **_slice_rows(d, 0, p))
            rest = _slice_rows(d, p, T)
            rest["state_in"] = a["state_out"]
            rest["ring_in"] = a["ring_out"]
            b = orc.forward(H=H, D=D, gate_mode=gate_mode, **rest)
            np.testing.assert_array_equal(np.concatenate([a["y"], b["y"]]), full["y"])
            np.testing.assert_array_equal(b["state_out"], full["state_out"])
            np.testing.assert_array_equal(b["ring_out"], full["ring_out"])


def check_chained_single_tokens_equal_multi_token():
    rng = _rng(13)
    T, H, D = 4, 2, 8
    d = _tiny_layer(rng, T, H, D)
    full = orc.forward(H=H, D=D, **d)
    st, ring = d["state_in"], d["ring_in"]
    ys = []
    for t in range(T):
        step = _slice_rows(d, t, t + 1)
        step["state_in"], step["ring_in"] = st, ring
        r = orc.forward(H=H, D=D, **step)
        st, ring = r["state_out"], r["ring_out"]
        ys.append(r["y"])
    np.testing.assert_array_equal(np.concatenate(ys), full["y"])
    np.testing.assert_array_equal(st, full["state_out"])
    np.testing.assert_array_equal(ring, full["ring_out"])


def check_varlen_equals_separate_calls():
    rng = _rng(14)
    H, D = 2, 8
    Ls = [3, 0, 5, 1]
    parts = [_tiny_layer(rng, L, H, D) for L in Ls]
    cat = {k: np.concatenate([p[k] for p in parts]) for k in
           ("q_raw", "k_raw", "v_raw", "f_raw", "beta_raw", "gate_raw", "ring_in", "state_in")}
    shared = dict(conv_w=parts[0]["conv_w"], dt_bias=parts[0]["dt_bias"],
                  a_log=parts[0]["a_log"], norm_w=parts[0]["norm_w"])
    cu = np.concatenate([[0], np.cumsum(Ls)])
    packed = orc.forward(H=H, D=D, cu_seqlens=cu, **cat, **shared)
    for n, p in enumerate(parts):
        p = dict(p, **shared)
        one = orc.forward(H=H, D=D, **p)
        np.testing.assert_array_equal(packed["y"][cu[n]:cu[n + 1]], one["y"])
        np.testing.assert_array_equal(packed["state_out"][n], one["state_out"][0])
        np.testing.assert_array_equal(packed["ring_out"][n], one["ring_out"][0])
    # an empty sequence keeps its state and ring
    np.testing.assert_array_equal(packed["state_out"][1], cat["state_in"][1])
    np.testing.assert_array_equal(packed["ring_out"][1], cat["ring_in"][1])


# ------------------------------------------------------------------------------------------
# stage 1: the projections that read x
# ------------------------------------------------------------------------------------------

def check_matvec_one_hot_rows():
    """Weight rows that are one-hot pick one input entry each: out[s][r] = x[s][p(r)] exactly."""
    rng = _rng(40)
    rows, in_f, t = 7, 19, 3
    p = rng.permutation(in_f)[:rows]
    w = np.zeros((rows, in_f))
    w[np.arange(rows), p] = 1.0
    x = rng.standard_normal((t, in_f))
    np.testing.assert_array_equal(orc.matvec_rows(w, x), x[:, p])


def check_matvec_exact_integers():
    """Small integer weights and inputs: every partial sum is an exact integer in f64, so the
    result equals the exact integer dot products computed here with Python ints, row by row and
    token by token (a non-square shape, so a transposed operand or a swapped stride cannot
    pass)."""
    rng = _rng(41)
    rows, in_f, t = 5, 11, 4
    w = rng.integers(-9, 10, size=(rows, in_f))
    x = rng.integers(-9, 10, size=(t, in_f))
    want = np.array([[sum(int(w[r, k]) * int(x[s, k]) for k in range(in_f)) for r in range(rows)]
                     for s in range(t)], dtype=float)
    np.testing.assert_array_equal(orc.matvec_rows(w.astype(float), x.astype(float)), want)


def check_matvec_band():
    """w[r][r] = r + 1 and w[r][r+1] = 2 (a band): out[s][r] = (r+1) x[s][r] + 2 x[s][r+1]."""
    rng = _rng(42)
    rows, in_f, t = 6, 9, 2
    w = np.zeros((rows, in_f))
    for r in range(rows):
        w[r, r] = r + 1.0
        w[r, r + 1] = 2.0
    x = rng.standard_normal((t, in_f))
    want = np.stack([(np.arange(rows) + 1.0) * x[s, :rows] + 2.0 * x[s, 1:rows + 1]
                     for s in range(t)])
    np.testing.assert_allclose(orc.matvec_rows(w, x), want, rtol=0, atol=1e-14)


def check_proj6_order_and_shapes():
    """The six projections come back in the pages' order [q, k, v, forget-down, gate-down,
    beta] with shapes [t, rows of each weight]; each weight tagged by a distinct constant row
    sum shows which output it produced."""
    t, in_f = 2, 8
    dims = (6, 6, 6, 3, 3, 2)
    ws = [np.full((d, in_f), float(i + 1)) for i, d in enumerate(dims)]
    x = np.ones((t, in_f))
    outs = orc.proj6(x, *ws)
    assert [o.shape for o in outs] == [(t, d) for d in dims]
    for i, o in enumerate(outs):
        np.testing.assert_array_equal(o, np.full_like(o, (i + 1) * in_f))


def check_gqa_equals_replicated_heads():
    """Grouped queries (value head h reads query/key head h % Hk) equal the plain mixer run on
    q/k raw channels, conv weights and ring rows replicated to H heads in that tiled order: the
    outputs, the state and the v part of the ring agree, and each replicated q/k ring row equals
    its source head's."""
    rng = _rng(43)
    D, H, Hk, K, T = 4, 6, 2, 3, 7
    C, Cq = H * D, Hk * D
    tiled = np.arange(H) % Hk
    chan = np.concatenate([np.arange(h * D, (h + 1) * D) for h in tiled])   # q/k channel per slot
    q = rng.standard_normal((T, Cq))
    k = rng.standard_normal((T, Cq))
    v = rng.standard_normal((T, C))
    wq, wk, wv = (rng.standard_normal((Cq, K)), rng.standard_normal((Cq, K)),
                  rng.standard_normal((C, K)))
    rq, rk, rv = (rng.standard_normal((Cq, K - 1)), rng.standard_normal((Cq, K - 1)),
                  rng.standard_normal((C, K - 1)))
    shared = dict(f_raw=rng.standard_normal((T, C)), dt_bias=rng.standard_normal(C),
                  a_log=np.log(rng.uniform(1, 16, H)), beta_raw=rng.standard_normal((T, H)),
                  state_in=0.1 * rng.standard_normal((1, H, D, D)), norm_w=1 + rng.standard_normal(D),
                  gate_raw=rng.standard_normal((T, C)), D=D, H=H)
    gqa = orc.forward(q_raw=q, k_raw=k, v_raw=v, conv_w=np.concatenate([wq, wk, wv]),
                      ring_in=np.concatenate([rq, rk, rv])[None], Hk=Hk, **shared)
    full = orc.forward(q_raw=q[:, chan], k_raw=k[:, chan], v_raw=v,
                       conv_w=np.concatenate([wq[chan], wk[chan], wv]),
                       ring_in=np.concatenate([rq[chan], rk[chan], rv])[None], **shared)
    for key in ("y", "o", "state_out"):
        np.testing.assert_array_equal(gqa[key], full[key])
    np.testing.assert_array_equal(gqa["ring_out"][0, 2 * Cq:], full["ring_out"][0, 2 * C:])
    np.testing.assert_array_equal(gqa["ring_out"][0, :Cq][chan], full["ring_out"][0, :C])
    np.testing.assert_array_equal(gqa["ring_out"][0, Cq:2 * Cq][chan], full["ring_out"][0, C:2 * C])
    assert gqa["q_hat"].shape == (T, Cq)


def check_rect_scan_is_column_blocks():
    """A value width Dv = 3 Dk: every value column of S evolves on its own, so the rectangular
    routine equals the square routine run on each Dk-wide block of value columns, bit for bit
    (state blocks and outputs), and with Dv = Dk it is the square routine itself."""
    rng = _rng(44)
    T, H, Dk, m = 6, 2, 4, 3
    Dv = m * Dk
    q, k = _unit_rows(rng, (T, H, Dk)), _unit_rows(rng, (T, H, Dk))
    v = rng.standard_normal((T, H, Dv))
    g = -rng.random((T, H, Dk))
    b = rng.random((T, H))
    s0 = rng.standard_normal((1, H, Dv, Dk))
    o, st = orc.scan_kda_rect(q, k, v, g, b, s0)
    assert o.shape == (T, H, Dv) and st.shape == (1, H, Dv, Dk)
    for j in range(m):
        sl = slice(j * Dk, (j + 1) * Dk)
        oj, sj = orc.scan_kda(q, k, v[:, :, sl], g, b, s0[:, :, sl], scale=Dk ** -0.5)
        np.testing.assert_array_equal(o[:, :, sl], oj)
        np.testing.assert_array_equal(st[:, :, sl], sj)


def check_rect_scan_dense_product():
    """The rectangular routine against the dense product form written out here:
    S <- (I - b k k^T) Diag(a) S + b k v^T with S of shape Dk x Dv, readout scale S^T q."""
    rng = _rng(45)
    T, Dk, Dv = 5, 3, 7
    q, k = _unit_rows(rng, (T, 1, Dk)), _unit_rows(rng, (T, 1, Dk))
    v = rng.standard_normal((T, 1, Dv))
    g = -rng.random((T, 1, Dk))
    b = rng.random((T, 1))
    S = rng.standard_normal((Dk, Dv))
    o, st = orc.scan_kda_rect(q, k, v, g, b, np.ascontiguousarray(S.T)[None, None], scale=1.0)
    for t in range(T):
        kt, bt = k[t, 0], b[t, 0]
        S = (np.eye(Dk) - bt * np.outer(kt, kt)) @ np.diag(np.exp(g[t, 0])) @ S + bt * np.outer(kt, v[t, 0])
        np.testing.assert_allclose(o[t, 0], S.T @ q[t, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(st[0, 0], S.T, rtol=0, atol=1e-12)


def check_forward_value_width():
    """The whole mixer with Dv = 2 D: its readout and state equal two mixers run on the halves of
    every value head (v raw channels, conv weight and ring rows, state), and y is the gated RMSNorm
    of that readout over each full 2 D-wide head."""
    rng = _rng(46)
    D, H, K, T = 4, 2, 3, 6
    Dv = 2 * D
    C, Cv = H * D, H * Dv
    q, k = rng.standard_normal((T, C)), rng.standard_normal((T, C))
    v = rng.standard_normal((T, Cv))
    wq, wk, wv = (rng.standard_normal((C, K)), rng.standard_normal((C, K)),
                  rng.standard_normal((Cv, K)))
    rq, rk, rv = (rng.standard_normal((C, K - 1)), rng.standard_normal((C, K - 1)),
                  rng.standard_normal((Cv, K - 1)))
    s0 = 0.1 * rng.standard_normal((1, H, Dv, D))
    shared = dict(f_raw=rng.standard_normal((T, C)), dt_bias=rng.standard_normal(C),
                  a_log=np.log(rng.uniform(1, 16, H)), beta_raw=rng.standard_normal((T, H)), D=D,
                  H=H)
    w_norm, z = 1 + rng.standard_normal(Dv), rng.standard_normal((T, Cv))
    full = orc.forward(q_raw=q, k_raw=k, v_raw=v, conv_w=np.concatenate([wq, wk, wv]),
                       ring_in=np.concatenate([rq, rk, rv])[None], state_in=s0, Dv=Dv,
                       norm_w=w_norm, gate_raw=z, **shared)
    for half in range(2):
        ch = np.concatenate([np.arange(h * Dv + half * D, h * Dv + (half + 1) * D)
                             for h in range(H)])
        part = orc.forward(q_raw=q, k_raw=k, v_raw=v[:, ch],
                           conv_w=np.concatenate([wq, wk, wv[ch]]),
                           ring_in=np.concatenate([rq, rk, rv[ch]])[None],
                           state_in=np.ascontiguousarray(s0[:, :, half * D:(half + 1) * D]),
                           scale=D ** -0.5, **shared)
        np.testing.assert_array_equal(full["o"][:, ch], part["o"])
        np.testing.assert_array_equal(full["state_out"][:, :, half * D:(half + 1) * D],
                                      part["state_out"])
        np.testing.assert_array_equal(full["ring_out"][0, 2 * C:][ch], part["ring_out"][0, 2 * C:])
    np.testing.assert_array_equal(full["y"], orc.gated_rmsnorm(full["o"], w_norm, z))


ALL_CHECKS = [
    check_three_token_golden, check_three_token_embedded, check_beta_zero_closed_form,
    check_orthonormal_recall, check_dense_product_form, check_chunked_form_every_chunk_size,
    check_default_scale, check_gdn_equals_broadcast_kda, check_conv_one_hot_shift,
    check_conv_taps_general, check_l2norm, check_gates, check_gated_rmsnorm,
    check_gated_rmsnorm_silu,
    check_split_state_carry, check_chained_single_tokens_equal_multi_token,
    check_varlen_equals_separate_calls, check_matvec_one_hot_rows, check_matvec_exact_integers,
    check_matvec_band, check_proj6_order_and_shapes, check_gqa_equals_replicated_heads,
    check_rect_scan_is_column_blocks, check_rect_scan_dense_product, check_forward_value_width,
]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__[len("check_"):])
def test_pin(check):
    check()


def test_gdn_orthonormal_recall():
    check_orthonormal_recall(orc.scan_gdn)
