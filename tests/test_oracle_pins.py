"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's loop: each expected value comes from a different statement
of the same quantity -- the worked demo's causal convolution in exact rational arithmetic, the
LTI convolution kernel, the semiseparable (materialised-matrix) form with products of
exponentials written as one exponential of a sum, tree-shaped compositions of the scan operator,
and library routines for softplus and the logistic function. ``test_mutants_are_caught`` builds
deliberately broken copies of the oracle and checks that every one of them fails some pin.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def _demo_inputs():
    vals = {}
    with open(os.path.join(HERE, "golden", "lti_demo.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            vals[k] = v
    return (Fraction(vals["A"][0]), Fraction(vals["B"][0]), Fraction(vals["C"][0]),
            [Fraction(s) for s in vals["x"]])


def _one_channel(u, delta, A, B, C, Dskip=None, z=None, bias=None, softplus=False, lib=None):
    """Run the oracle on a single (batch=1, dim=1) channel given plain float sequences."""
    L = len(u)
    N = len(A)
    y, h = oracle.fwd(_f32(u).reshape(1, L, 1), _f32(delta).reshape(1, L, 1),
                      _f32(A).reshape(1, N), _f32(B).reshape(1, L, N), _f32(C).reshape(1, L, N),
                      None if Dskip is None else _f32([Dskip]),
                      None if z is None else _f32(z).reshape(1, L, 1),
                      None if bias is None else _f32([bias]), softplus=softplus, lib=lib)
    return y[0, :, 0], h[0, 0]


# ---------------------------------------------------------------------------------------------
# 1. The worked LTI demo ("架构变体：Mamba/SSM", "Python 演示"): scan == causal convolution.
# ---------------------------------------------------------------------------------------------
def pin_worked_example(lib=None):
    A, B, C, x = _demo_inputs()
    L = len(x)
    # Exact causal convolution with K[k] = C*B*A^k, in rationals (the page's closed form).
    y_exact = [sum(C * B * A ** k * x[t - k] for k in range(t + 1)) for t in range(L)]
    # Hand-checkable values of that convolution (the page does not print them).
    assert y_exact[:3] == [Fraction(1, 10), Fraction(-3, 20), Fraction(1, 40)]
    # Map onto the selective scan: dt = 1 (softplus off), exp(dt*A_cont) = 0.9, B_t = 0.2,
    # C_t = 1, no skip, no gate. A_cont = ln 0.9 and the inputs are rounded to fp32, so compare
    # (i) to the closed form evaluated on the fp32-rounded parameters to 1e-13, and (ii) to the
    # page's exact values within the parameter rounding (A^k drifts by <= k * 2^-24 relative).
    a_cont = float(np.float32(math.log(0.9)))
    xf = [float(np.float32(float(v))) for v in x]
    bf = float(np.float32(0.2))
    y, h = _one_channel(xf, [1.0] * L, [a_cont], [[bf]] * L, [[1.0]] * L, lib=lib)
    a = math.exp(a_cont)
    y_cf = [math.fsum(bf * a ** k * xf[t - k] for k in range(t + 1)) for t in range(L)]
    np.testing.assert_allclose(y, y_cf, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(y, [float(v) for v in y_exact], rtol=2e-6, atol=1e-7)
    assert abs(h[0] - y_cf[-1]) < 1e-14  # C = 1: the final state is the last output


def pin_selective_demo(lib=None):
    """The demo's selective variant: B_t = 0.2 * sigmoid(x_t), fed to the scan as B."""
    A, B, C, x = _demo_inputs()
    xf = [float(np.float32(float(v))) for v in x]
    Bt = [float(np.float32(0.2 * expit(v))) for v in xf]
    a_cont = float(np.float32(math.log(0.9)))
    a = math.exp(a_cont)
    L = len(xf)
    y, _ = _one_channel(xf, [1.0] * L, [a_cont], [[b] for b in Bt], [[1.0]] * L, lib=lib)
    # Unrolled sum y_t = sum_{s<=t} a^(t-s) B_s x_s.
    y_cf = [math.fsum(a ** (t - s) * Bt[s] * xf[s] for s in range(t + 1)) for t in range(L)]
    np.testing.assert_allclose(y, y_cf, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# 2. LTI special case, general N: constant dt, B, C  =>  y = K_d * u (causal convolution).
#    ("架构变体：Mamba/SSM", "并行卷积": with fixed parameters the recurrence unrolls into a
#    convolution whose weights depend only on the lag.)
# ---------------------------------------------------------------------------------------------
def pin_lti_convolution(lib=None):
    rng = np.random.default_rng(11)
    batch, L, dim, N = 2, 40, 3, 5
    u = _f32(rng.standard_normal((batch, L, dim)))
    z = _f32(rng.standard_normal((batch, L, dim)))
    A = _f32(-np.exp(rng.uniform(0, math.log(16), (dim, N))))
    Bv = _f32(rng.standard_normal((batch, N)))
    Cv = _f32(rng.standard_normal((batch, N)))
    Dskip = _f32(rng.standard_normal(dim))
    bias = _f32(rng.uniform(-3, 0.5, dim))
    delta = _f32(np.broadcast_to(rng.standard_normal((1, 1, dim)), (batch, L, dim)))
    Bm = _f32(np.broadcast_to(Bv[:, None, :], (batch, L, N)))
    Cm = _f32(np.broadcast_to(Cv[:, None, :], (batch, L, N)))
    y, h = oracle.fwd(u, delta, A, Bm, Cm, Dskip, z, bias, softplus=True, lib=lib)
    dt = np.logaddexp(0.0, delta[0, 0].astype(np.float64) + bias.astype(np.float64))  # (dim,)
    k = np.arange(L)
    for b in range(batch):
        for d in range(dim):
            K = np.zeros(L)
            for n in range(N):
                K += (float(Cv[b, n]) * dt[d] * float(Bv[b, n])
                      * np.exp(dt[d] * float(A[d, n])) ** k)
            uu = u[b, :, d].astype(np.float64)
            conv = np.convolve(K, uu)[:L] + float(Dskip[d]) * uu
            zz = z[b, :, d].astype(np.float64)
            ref = conv * zz * expit(zz)
            np.testing.assert_allclose(y[b, :, d], ref, rtol=1e-11, atol=1e-13)
            # Final state: h[n] = sum_s exp(dt A)^(L-1-s) dt B[n] u_s
            for n in range(N):
                hn = math.fsum(np.exp(dt[d] * float(A[d, n])) ** (L - 1 - s) * dt[d]
                               * float(Bv[b, n]) * float(uu[s]) for s in range(L))
                assert abs(h[b, d, n] - hn) <= 1e-12 * (1 + abs(hn))


# ---------------------------------------------------------------------------------------------
# 3. General time-varying case: the materialised (semiseparable-matrix) form
#    y[t] = sum_{s<=t} sum_n C_t[n] exp(A[n] * sum_{s<tau<=t} dt_tau) dt_s B_s[n] u_s + D u_t.
#    Products of per-step exponentials are taken as one exponential of the summed steps.
# ---------------------------------------------------------------------------------------------
def _matrix_form(u, delta, A, Bm, Cm, Dskip, z, bias, softplus):
    batch, L, dim = u.shape
    N = Bm.shape[2]
    y = np.zeros((batch, L, dim))
    h = np.zeros((batch, dim, N))
    for b in range(batch):
        for d in range(dim):
            x = delta[b, :, d].astype(np.float64) + (0.0 if bias is None else float(bias[d]))
            dt = np.logaddexp(0.0, x) if softplus else x
            cum = np.concatenate([[0.0], np.cumsum(dt)])  # cum[t+1] = dt_0 + ... + dt_t
            uu = u[b, :, d].astype(np.float64)
            for t in range(L):
                acc = []
                for s in range(t + 1):
                    seg = cum[t + 1] - cum[s + 1]  # sum of dt over s < tau <= t
                    for n in range(N):
                        acc.append(float(Cm[b, t, n]) * math.exp(float(A[d, n]) * seg) * dt[s]
                                   * float(Bm[b, s, n]) * uu[s])
                yt = math.fsum(acc) + (0.0 if Dskip is None else float(Dskip[d]) * uu[t])
                if z is not None:
                    zz = float(z[b, t, d])
                    yt *= zz * expit(zz)
                y[b, t, d] = yt
            for n in range(N):
                h[b, d, n] = math.fsum(
                    math.exp(float(A[d, n]) * (cum[L] - cum[s + 1])) * dt[s] * float(Bm[b, s, n])
                    * uu[s] for s in range(L))
    return y, h


def pin_matrix_form(lib=None):
    rng = np.random.default_rng(5)
    batch, L, dim, N = 2, 9, 3, 4
    u = _f32(rng.standard_normal((batch, L, dim)))
    delta = _f32(rng.standard_normal((batch, L, dim)))
    z = _f32(rng.standard_normal((batch, L, dim)))
    A = _f32(-np.exp(rng.uniform(-1, 2, (dim, N))))
    Bm = _f32(rng.standard_normal((batch, L, N)))
    Cm = _f32(rng.standard_normal((batch, L, N)))
    Dskip = _f32(rng.standard_normal(dim))
    bias = _f32(rng.uniform(-2, 1, dim))
    for sp, zz, DD, bb in [(True, z, Dskip, bias), (False, None, None, None)]:
        d_in = delta if sp else _f32(np.abs(delta) * 0.3)
        y, h = oracle.fwd(u, d_in, A, Bm, Cm, DD, zz, bb, softplus=sp, lib=lib)
        yr, hr = _matrix_form(u, d_in, A, Bm, Cm, DD, zz, bb, sp)
        np.testing.assert_allclose(y, yr, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(h, hr, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# 4. Associativity of the scan operator ("架构变体：Mamba/SSM", "硬件感知算法": the update rule is
#    associative, so the scan can be evaluated as a tree). Every bracketing of
#    (a2,b2) o (a1,b1) = (a2*a1, a2*b1 + b2) over L <= 7 steps must give the sequential state.
# ---------------------------------------------------------------------------------------------
def _compose(p, q):  # p earlier, q later
    return (q[0] * p[0], q[0] * p[1] + q[1])


def _all_brackets(items):
    if len(items) == 1:
        yield items[0]
        return
    for i in range(1, len(items)):
        for left in _all_brackets(items[:i]):
            for right in _all_brackets(items[i:]):
                yield _compose(left, right)


def pin_associativity(lib=None):
    rng = np.random.default_rng(3)
    for L in range(1, 8):
        N = 2
        u = _f32(rng.standard_normal(L))
        delta = _f32(rng.standard_normal(L))
        A = _f32(-np.exp(rng.uniform(-1, 1.5, N)))
        Bm = _f32(rng.standard_normal((L, N)))
        Cm = _f32(rng.standard_normal((L, N)))
        bias = -1.0
        _, h = _one_channel(u, delta, A, Bm, Cm, bias=bias, softplus=True, lib=lib)
        dt = np.logaddexp(0.0, delta.astype(np.float64) + float(np.float32(bias)))
        for n in range(N):
            pairs = [(math.exp(dt[t] * float(A[n])), dt[t] * float(Bm[t, n]) * float(u[t]))
                     for t in range(L)]
            count = 0
            for agg in _all_brackets(pairs):
                count += 1
                assert abs(agg[1] - h[n]) <= 1e-13 * (1 + abs(h[n]))
            assert count == math.comb(2 * (L - 1), L - 1) // L  # Catalan number C_{L-1}


# ---------------------------------------------------------------------------------------------
# 5. Delta -> 0 leaves the state unchanged (softplus off, dt = 0 on a window).
# ---------------------------------------------------------------------------------------------
def pin_delta_zero(lib=None):
    rng = np.random.default_rng(8)
    L, N = 30, 6
    u = _f32(rng.standard_normal(L))
    delta = _f32(np.abs(rng.standard_normal(L)) * 0.2)
    delta[10:20] = 0.0
    A = _f32(-np.arange(1, N + 1))
    Bm = _f32(rng.standard_normal((L, N)))
    Cm = _f32(rng.standard_normal((L, N)))
    Cm[10:20] = Cm[10]  # constant readout over the window
    Dskip = 0.7
    y, _ = _one_channel(u, delta, A, Bm, Cm, Dskip=Dskip, softplus=False, lib=lib)
    core = y - float(np.float32(Dskip)) * u.astype(np.float64)
    # The state entering the window is the state at t = 9; with dt = 0 it never changes.
    assert np.ptp(core[10:20]) < 1e-14 * (1 + np.abs(core[10:20]).max())
    assert abs(core[10] - core[9]) > 1e-6 or np.allclose(Cm[9], Cm[10])
    # dt = 0 everywhere: the state stays zero and y is the gated skip term.
    z = _f32(rng.standard_normal(L))
    y0, h0 = _one_channel(u, np.zeros(L), A, Bm, Cm, Dskip=Dskip, z=z, softplus=False, lib=lib)
    assert np.all(h0 == 0.0)
    ref = float(np.float32(Dskip)) * u.astype(np.float64) * z * expit(z.astype(np.float64))
    np.testing.assert_allclose(y0, ref, rtol=1e-15, atol=0)


# ---------------------------------------------------------------------------------------------
# 6. Skip and gate special cases: C = 0 => y = Dskip*u*SiLU(z); B = 0 => h_last = 0.
# ---------------------------------------------------------------------------------------------
def pin_skip_gate(lib=None):
    rng = np.random.default_rng(9)
    batch, L, dim, N = 2, 12, 4, 3
    u = _f32(rng.standard_normal((batch, L, dim)))
    delta = _f32(rng.standard_normal((batch, L, dim)))
    z = _f32(rng.standard_normal((batch, L, dim)) * 3)
    A = _f32(-np.arange(1, N + 1) * np.ones((dim, 1)))
    Bm = _f32(rng.standard_normal((batch, L, N)))
    Dskip = _f32(rng.standard_normal(dim))
    y, h = oracle.fwd(u, delta, A, Bm, np.zeros_like(Bm), Dskip, z, None, softplus=True, lib=lib)
    zz = z.astype(np.float64)
    ref = Dskip.astype(np.float64) * u * zz * expit(zz)
    np.testing.assert_allclose(y, ref, rtol=1e-15, atol=1e-300)
    assert np.abs(h).max() > 0.01  # the state itself is not zero, only unread
    y2, h2 = oracle.fwd(u, delta, A, np.zeros_like(Bm), Bm, None, None, None, lib=lib)
    assert np.all(h2 == 0.0) and np.all(y2 == 0.0)


# ---------------------------------------------------------------------------------------------
# 7. Softplus against numpy's logaddexp(0, x); bias is added before softplus.
#    (A = 0, B = C = u = 1, one step: y = h = dt.)
# ---------------------------------------------------------------------------------------------
def pin_softplus(lib=None):
    xs = _f32(np.concatenate([np.linspace(-12, 30, 85), [-40.0, 50.0, 0.0, 1e-3, -1e-3]]))
    dim = xs.size
    ones = np.ones((1, 1, dim), np.float32)
    for bias in (None, _f32(np.linspace(-2.0, 1.0, dim))):
        y, _ = oracle.fwd(ones, xs.reshape(1, 1, dim), np.zeros((dim, 1), np.float32),
                          np.ones((1, 1, 1), np.float32), np.ones((1, 1, 1), np.float32),
                          None, None, bias, softplus=True, lib=lib)
        x = xs.astype(np.float64) + (0.0 if bias is None else bias.astype(np.float64))
        np.testing.assert_allclose(y[0, 0], np.logaddexp(0.0, x), rtol=1e-15, atol=0)
        y_off, _ = oracle.fwd(ones, xs.reshape(1, 1, dim), np.zeros((dim, 1), np.float32),
                              np.ones((1, 1, 1), np.float32), np.ones((1, 1, 1), np.float32),
                              None, None, bias, softplus=False, lib=lib)
        np.testing.assert_array_equal(y_off[0, 0], x)


# ---------------------------------------------------------------------------------------------
# 8. bf16 io: the oracle reads bf16 bit patterns as exactly the fp32 values they encode.
# ---------------------------------------------------------------------------------------------
def _bf16_bits(x):
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def _bf16_to_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def pin_bf16_widening(lib=None):
    rng = np.random.default_rng(21)
    batch, L, dim, N = 2, 15, 5, 4
    arrs = [rng.standard_normal(s) for s in
            [(batch, L, dim)] * 3 + [(batch, L, N)] * 2]
    bits = [_bf16_bits(a) for a in arrs]
    vals = [_bf16_to_f32(b) for b in bits]
    A = _f32(-np.arange(1, N + 1) * np.ones((dim, 1)))
    Dskip = _f32(rng.standard_normal(dim))
    bias = _f32(rng.uniform(-3, -1, dim))
    ub, db, zb, Bb, Cb = bits
    uf, df, zf, Bf, Cf = vals
    y1, h1 = oracle.fwd(ub, db, A, Bb, Cb, Dskip, zb, bias, io="bf16", lib=lib)
    y2, h2 = oracle.fwd(uf, df, A, Bf, Cf, Dskip, zf, bias, io="f32", lib=lib)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(h1, h2)
    # and the widening itself: bf16 0x3FC0 = 1.5, 0xC040 = -3.0
    assert _bf16_to_f32(np.array([0x3FC0, 0xC040], np.uint16)).tolist() == [1.5, -3.0]


# ---------------------------------------------------------------------------------------------
# 9. Initial state h0 (recurrent mode: the state is all that carries from one step to the next,
#    "Mamba：选择性状态空间模型入门教程", "Mamba 的关键创新：选择性机制").
# ---------------------------------------------------------------------------------------------
def _h0_inputs(rng, batch, L, dim, N):
    u, z = (_f32(rng.standard_normal((batch, L, dim))) for _ in range(2))
    delta = _f32(rng.standard_normal((batch, L, dim)))
    Bm, Cm = (_f32(rng.standard_normal((batch, L, N))) for _ in range(2))
    A = _f32(-np.exp(rng.uniform(0, math.log(8), (dim, N))))
    Dskip = _f32(rng.standard_normal(dim))
    bias = _f32(rng.uniform(-3, -1, dim))
    h0 = _f32(rng.standard_normal((batch, dim, N)))
    return u, delta, A, Bm, Cm, Dskip, z, bias, h0


def pin_h0_free_decay(lib=None):
    """u = 0: no input enters, so h_t = exp(A sum_{s<=t} dt_s) h0 (one exponential of the summed
    steps) and y_t = (C_t . h_t) SiLU(z_t)."""
    rng = np.random.default_rng(21)
    batch, L, dim, N = 2, 24, 3, 6
    u, delta, A, Bm, Cm, Dskip, z, bias, h0 = _h0_inputs(rng, batch, L, dim, N)
    u0 = np.zeros_like(u)
    y, h = oracle.fwd(u0, delta, A, Bm, Cm, Dskip, z, bias, softplus=True, lib=lib, h0=h0)
    dt = np.logaddexp(0.0, delta.astype(np.float64) + bias.astype(np.float64))  # (batch, L, dim)
    cum = np.cumsum(dt, axis=1)
    for b in range(batch):
        for d in range(dim):
            ht = np.exp(cum[b, :, d, None] * A[d].astype(np.float64)[None, :]) \
                * h0[b, d].astype(np.float64)[None, :]                     # (L, N)
            zz = z[b, :, d].astype(np.float64)
            ref = np.einsum("tn,tn->t", Cm[b].astype(np.float64), ht) * zz * expit(zz)
            np.testing.assert_allclose(y[b, :, d], ref, rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(h[b, d], ht[-1], rtol=1e-12, atol=1e-15)
    # First-order factor: h_t = prod_{s<=t} (1 + dt_s A) h0, with steps small enough to decay.
    bs = _f32(bias - 3.0)
    y, h = oracle.fwd(u0, delta, A, Bm, Cm, Dskip, z, bs, softplus=True, lib=lib, h0=h0,
                      euler=True)
    dt = np.logaddexp(0.0, delta.astype(np.float64) + bs.astype(np.float64))
    for b in range(batch):
        for d in range(dim):
            fac = 1.0 + dt[b, :, d, None] * A[d].astype(np.float64)[None, :]   # (L, N)
            ht = np.cumprod(fac, axis=0) * h0[b, d].astype(np.float64)[None, :]
            zz = z[b, :, d].astype(np.float64)
            ref = np.einsum("tn,tn->t", Cm[b].astype(np.float64), ht) * zz * expit(zz)
            np.testing.assert_allclose(y[b, :, d], ref, rtol=1e-11, atol=1e-13)


def pin_h0_superposition(lib=None):
    """The scan is linear in (h0, inputs) for fixed steps: y(h0, u) = y(0, u) + y(h0, u = 0)."""
    rng = np.random.default_rng(22)
    batch, L, dim, N = 2, 30, 4, 5
    u, delta, A, Bm, Cm, Dskip, z, bias, h0 = _h0_inputs(rng, batch, L, dim, N)
    y1, h1 = oracle.fwd(u, delta, A, Bm, Cm, Dskip, z, bias, lib=lib, h0=h0)
    y2, h2 = oracle.fwd(u, delta, A, Bm, Cm, Dskip, z, bias, lib=lib)
    y3, h3 = oracle.fwd(np.zeros_like(u), delta, A, Bm, Cm, Dskip, z, bias, lib=lib, h0=h0)
    scale = np.abs(y2).max() + np.abs(y3).max()
    np.testing.assert_allclose(y1, y2 + y3, rtol=0, atol=1e-13 * scale)
    np.testing.assert_allclose(h1, h2 + h3, rtol=0, atol=1e-13 * (np.abs(h2).max() + np.abs(h3).max()))


def pin_h0_split_sequence(lib=None):
    """Running steps [0, L1) and then [L1, L) from the carried state equals one run over [0, L)
    (the carried state rounded to fp32 on the way, as the library's h_last / h0 are)."""
    rng = np.random.default_rng(23)
    batch, L, dim, N, L1 = 2, 40, 3, 7, 17
    u, delta, A, Bm, Cm, Dskip, z, bias, _ = _h0_inputs(rng, batch, L, dim, N)
    for euler in (False, True):
        # Euler is stable only for dt |A| < 2: give it smaller steps.
        bs = _f32(bias - 3.0) if euler else bias
        y, h = oracle.fwd(u, delta, A, Bm, Cm, Dskip, z, bs, lib=lib, euler=euler)
        ya, ha = oracle.fwd(u[:, :L1].copy(), delta[:, :L1].copy(), A, Bm[:, :L1].copy(),
                            Cm[:, :L1].copy(), Dskip, z[:, :L1].copy(), bs, lib=lib, euler=euler)
        yb, hb = oracle.fwd(u[:, L1:].copy(), delta[:, L1:].copy(), A, Bm[:, L1:].copy(),
                            Cm[:, L1:].copy(), Dskip, z[:, L1:].copy(), bs, lib=lib,
                            h0=ha.astype(np.float32), euler=euler)
        np.testing.assert_array_equal(ya, y[:, :L1])
        scale = np.abs(y).max()
        np.testing.assert_allclose(yb, y[:, L1:], rtol=0, atol=1e-6 * scale)
        np.testing.assert_allclose(hb, h, rtol=0, atol=1e-6 * np.abs(h).max())


# ---------------------------------------------------------------------------------------------
# 10. First-order (Euler) decay factor 1 + dt A: with constant dt, B, C the recurrence unrolls
#     into a causal convolution with K[k] = sum_n C dt B (1 + dt A)^k ("架构变体：Mamba/SSM",
#     "并行卷积"; the factor is the first-order expansion of exp(dt A), "从RNN到Mamba" 3.2).
# ---------------------------------------------------------------------------------------------
def pin_euler_lti(lib=None):
    rng = np.random.default_rng(12)
    batch, L, dim, N = 2, 36, 3, 4
    u = _f32(rng.standard_normal((batch, L, dim)))
    A = _f32(-np.exp(rng.uniform(0, math.log(8), (dim, N))))
    Bv = _f32(rng.standard_normal((batch, N)))
    Cv = _f32(rng.standard_normal((batch, N)))
    Dskip = _f32(rng.standard_normal(dim))
    delta = _f32(np.broadcast_to(rng.uniform(0.01, 0.1, (1, 1, dim)), (batch, L, dim)))
    Bm = _f32(np.broadcast_to(Bv[:, None, :], (batch, L, N)))
    Cm = _f32(np.broadcast_to(Cv[:, None, :], (batch, L, N)))
    y, h = oracle.fwd(u, delta, A, Bm, Cm, Dskip, None, None, softplus=False, lib=lib, euler=True)
    dt = delta[0, 0].astype(np.float64)
    k = np.arange(L)
    for b in range(batch):
        for d in range(dim):
            K = np.zeros(L)
            for n in range(N):
                K += float(Cv[b, n]) * dt[d] * float(Bv[b, n]) * (1.0 + dt[d] * float(A[d, n])) ** k
            uu = u[b, :, d].astype(np.float64)
            ref = np.convolve(K, uu)[:L] + float(Dskip[d]) * uu
            np.testing.assert_allclose(y[b, :, d], ref, rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# 11. Causal depthwise Conv1d + SiLU ahead of the scan ("Mamba: Linear-Time Sequence Modeling
#     with Selective State Spaces" notes, "架构：极简设计": Linear -> Conv1d -> SiLU).
# ---------------------------------------------------------------------------------------------
def pin_conv1d_numpy(lib=None):
    """Against numpy.convolve with the taps reversed (w[W-1] weighs the current step) and
    scipy's logistic function; widths 1 .. 5."""
    rng = np.random.default_rng(31)
    batch, L, dim = 2, 23, 3
    x = _f32(rng.standard_normal((batch, L, dim)))
    for width in range(1, 6):
        w = _f32(rng.standard_normal((dim, width)))
        bias = _f32(rng.standard_normal(dim))
        y = oracle.conv1d(x, w, bias, lib=lib)
        y_lin = oracle.conv1d(x, w, None, silu=False, lib=lib)
        for b in range(batch):
            for d in range(dim):
                lin = np.convolve(x[b, :, d].astype(np.float64),
                                  w[d, ::-1].astype(np.float64))[:L]
                np.testing.assert_allclose(y_lin[b, :, d], lin, rtol=1e-13, atol=1e-13)
                a = lin + float(bias[d])
                np.testing.assert_allclose(y[b, :, d], a * expit(a), rtol=1e-12, atol=1e-13)


def pin_conv1d_stream(lib=None):
    """With the previous W - 1 inputs given, the output is the tail of one convolution over the
    concatenated sequence (a streamed sequence matches an unsplit one)."""
    rng = np.random.default_rng(32)
    batch, L, dim, width = 2, 19, 4, 4
    x = _f32(rng.standard_normal((batch, L + width - 1, dim)))
    w = _f32(rng.standard_normal((dim, width)))
    bias = _f32(rng.standard_normal(dim))
    full = oracle.conv1d(x, w, bias, lib=lib)
    tail = oracle.conv1d(x[:, width - 1:].copy(), w, bias, x_prev=x[:, :width - 1].copy(),
                         lib=lib)
    np.testing.assert_array_equal(tail, full[:, width - 1:])


# ---------------------------------------------------------------------------------------------
# 12. Backward pass: the gradient of sum(dy * y) + sum(dh_last * h_last). Pinned against torch
#     autograd of an independent float64 statement of the forward (vectorised over batch,
#     channels and states) and against central differences of that forward.
# ---------------------------------------------------------------------------------------------
def _torch_forward(t, softplus, euler):
    import torch
    u, delta, A, Bm, Cm = t["u"], t["delta"], t["A"], t["B"], t["C"]
    Dv, z, bias, h0 = t.get("D"), t.get("z"), t.get("bias"), t.get("h0")
    batch, L, dim = u.shape
    N = A.shape[1]
    h = h0 if h0 is not None else torch.zeros(batch, dim, N, dtype=torch.float64)
    ys = []
    for s in range(L):
        x = delta[:, s] + (bias if bias is not None else 0.0)
        dt = torch.nn.functional.softplus(x) if softplus else x
        a = 1.0 + dt[..., None] * A if euler else torch.exp(dt[..., None] * A)
        h = a * h + (dt * u[:, s])[..., None] * Bm[:, s, None, :]
        y = (h * Cm[:, s, None, :]).sum(-1) + (Dv * u[:, s] if Dv is not None else 0.0)
        if z is not None:
            y = y * z[:, s] * torch.sigmoid(z[:, s])
        ys.append(y)
    return torch.stack(ys, 1), h


def _bwd_case(seed, softplus, euler, with_opt):
    rng = np.random.default_rng(seed)
    batch, L, dim, N = 2, 13, 3, 4
    c = {"u": _f32(rng.standard_normal((batch, L, dim))),
         "delta": _f32(rng.standard_normal((batch, L, dim)) * (0.02 if euler else 1.0)),
         "A": _f32(-np.exp(rng.uniform(0, math.log(8), (dim, N)))),
         "B": _f32(rng.standard_normal((batch, L, N))),
         "C": _f32(rng.standard_normal((batch, L, N)))}
    if with_opt:
        c.update({"D": _f32(rng.standard_normal(dim)), "z": _f32(rng.standard_normal((batch, L, dim))),
                  "bias": _f32(rng.uniform(-3, -1, dim)),
                  "h0": _f32(rng.standard_normal((batch, dim, N)))})
    if euler:
        c["delta"] = _f32(np.abs(c["delta"]))
    dy = _f32(rng.standard_normal((batch, L, dim)))
    dh = _f32(rng.standard_normal((batch, dim, N)))
    return c, dy, dh


_BWD_KEYS = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "bias": "ddelta_bias", "h0": "dh0"}


def _oracle_grads(c, dy, dh, softplus, euler, lib):
    return oracle.bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], c.get("D"), c.get("z"),
                      c.get("bias"), dy, dh, softplus=softplus, h0=c.get("h0"), euler=euler,
                      lib=lib)


def pin_bwd_autograd(lib=None):
    import torch
    for seed, softplus, euler, with_opt in [(41, True, False, True), (42, False, True, False),
                                            (43, True, True, True), (44, False, False, False)]:
        c, dy, dh = _bwd_case(seed, softplus, euler, with_opt)
        tt = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in c.items()}
        y, h = _torch_forward(tt, softplus, euler)
        # the torch statement computes the same forward as the oracle
        yo, ho = oracle.fwd(c["u"], c["delta"], c["A"], c["B"], c["C"], c.get("D"), c.get("z"),
                            c.get("bias"), softplus=softplus, h0=c.get("h0"), euler=euler,
                            lib=lib)
        np.testing.assert_allclose(y.detach().numpy(), yo, rtol=1e-12, atol=1e-12)
        loss = (y * torch.tensor(dy, dtype=torch.float64)).sum() + \
            (h * torch.tensor(dh, dtype=torch.float64)).sum()
        loss.backward()
        g = _oracle_grads(c, dy, dh, softplus, euler, lib)
        for k, v in tt.items():
            ref = v.grad.numpy()
            got = g[_BWD_KEYS[k]]
            np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10 * (1 + np.abs(ref).max()),
                                       err_msg=f"{k} softplus={softplus} euler={euler}")


def pin_bwd_finite_difference(lib=None):
    """Central differences (step 1e-6) of the float64 forward's loss at sampled elements."""
    import torch
    softplus, euler = True, False
    c, dy, dh = _bwd_case(45, softplus, euler, True)
    g = _oracle_grads(c, dy, dh, softplus, euler, lib)
    dyt, dht = torch.tensor(dy, dtype=torch.float64), torch.tensor(dh, dtype=torch.float64)

    def loss_of(cc):
        tt = {k: torch.tensor(v, dtype=torch.float64) for k, v in cc.items()}
        y, h = _torch_forward(tt, softplus, euler)
        return float((y * dyt).sum() + (h * dht).sum())

    rng = np.random.default_rng(46)
    for k, v in c.items():
        for _ in range(3):
            idx = tuple(int(rng.integers(0, s)) for s in v.shape)
            plus = {kk: vv.astype(np.float64) for kk, vv in c.items()}
            minus = {kk: vv.astype(np.float64) for kk, vv in c.items()}
            eps = 1e-6
            plus[k][idx] += eps
            minus[k][idx] -= eps
            fd = (loss_of(plus) - loss_of(minus)) / (2 * eps)
            got = g[_BWD_KEYS[k]][idx]
            assert abs(got - fd) <= 1e-6 * (1 + abs(fd)), (k, idx, got, fd)


# ---------------------------------------------------------------------------------------------
# Magnitudes: the scale of every output's (and gradient's) terms, which the parity metric uses
# for outputs that cancel. Pinned by what they must be: with no negative term they equal the
# value itself, and they never fall below its absolute value.
# ---------------------------------------------------------------------------------------------
def pin_magnitude_forward(lib=None):
    rng = np.random.default_rng(51)
    batch, L, dim, N = 2, 40, 5, 16
    pos = lambda *s: _f32(np.abs(rng.standard_normal(s)))  # noqa: E731
    A = _f32(-np.arange(1, N + 1) * np.ones((dim, 1)) * 0.3)
    args = (pos(batch, L, dim), _f32(rng.standard_normal((batch, L, dim))), A, pos(batch, L, N),
            pos(batch, L, N), pos(dim), pos(batch, L, dim), _f32(rng.uniform(-3, -1, dim)))
    # every term non-negative (exp factors, softplus steps, and positive u, B, C, D, z, SiLU(z))
    y, h, m = oracle.fwd(*args, want_mag=True, lib=lib)
    np.testing.assert_array_equal(m, y)
    # random signs: the magnitude bounds the value
    args = (_f32(rng.standard_normal((batch, L, dim))), _f32(rng.standard_normal((batch, L, dim))),
            A, _f32(rng.standard_normal((batch, L, N))), _f32(rng.standard_normal((batch, L, N))),
            _f32(rng.standard_normal(dim)), _f32(rng.standard_normal((batch, L, dim))),
            _f32(rng.uniform(-3, -1, dim)))
    y, h, m = oracle.fwd(*args, want_mag=True, lib=lib)
    assert np.all(m >= np.abs(y)) and np.all(m > 0)


def pin_magnitude_backward(lib=None):
    for softplus, euler in [(True, False), (False, True)]:
        c, dy, dh = _bwd_case(52, softplus, euler, True)
        g = oracle.bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], c.get("D"), c.get("z"),
                       c.get("bias"), dy, dh, softplus=softplus, h0=c.get("h0"), euler=euler,
                       lib=lib)
        m = oracle.bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], c.get("D"), c.get("z"),
                       c.get("bias"), dy, dh, softplus=softplus, h0=c.get("h0"), euler=euler,
                       lib=lib, mag=True)
        for k in g:
            assert np.all(m[k] >= np.abs(g[k]) * (1 - 1e-12)), (k, softplus, euler)
        # no negative term anywhere: non-negative inputs and a non-negative A (a growing state,
        # fine for 13 steps), positive steps; then every magnitude equals its gradient
        pc = {k: _f32(np.abs(v)) for k, v in c.items()}
        pdy, pdh = _f32(np.abs(dy)), _f32(np.abs(dh))
        gp = oracle.bwd(pc["u"], pc["delta"], pc["A"], pc["B"], pc["C"], pc["D"], pc["z"], None,
                        pdy, pdh, softplus=softplus, h0=pc["h0"], euler=euler, lib=lib)
        mp = oracle.bwd(pc["u"], pc["delta"], pc["A"], pc["B"], pc["C"], pc["D"], pc["z"], None,
                        pdy, pdh, softplus=softplus, h0=pc["h0"], euler=euler, lib=lib, mag=True)
        for k in gp:
            np.testing.assert_allclose(mp[k], gp[k], rtol=1e-12, atol=0, err_msg=k)


PINS = [pin_worked_example, pin_selective_demo, pin_lti_convolution, pin_matrix_form,
        pin_associativity, pin_delta_zero, pin_skip_gate, pin_softplus, pin_bf16_widening,
        pin_h0_free_decay, pin_h0_superposition, pin_h0_split_sequence, pin_euler_lti,
        pin_conv1d_numpy, pin_conv1d_stream, pin_bwd_autograd, pin_bwd_finite_difference,
        pin_magnitude_forward, pin_magnitude_backward]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(None)


def test_channel_entry_matches_whole_tensor_entry():
    """The per-channel entry used for sampled checks agrees exactly with the whole-tensor one."""
    rng = np.random.default_rng(4)
    batch, L, dim, N = 2, 33, 6, 16
    u, delta, z = (_f32(rng.standard_normal((batch, L, dim))) for _ in range(3))
    Bm, Cm = (_f32(rng.standard_normal((batch, L, N))) for _ in range(2))
    A = _f32(-np.arange(1, N + 1) * np.ones((dim, 1)))
    Dskip = _f32(rng.standard_normal(dim))
    bias = _f32(rng.uniform(-4, -1, dim))
    y, h = oracle.fwd(u, delta, A, Bm, Cm, Dskip, z, bias)
    for b, d in [(0, 0), (1, 5), (1, 2)]:
        yc, hc = oracle.fwd_channel(u[b, :, d].copy(), delta[b, :, d].copy(), A[d], Bm[b], Cm[b],
                                    float(Dskip[d]), z[b, :, d].copy(), float(bias[d]))
        np.testing.assert_array_equal(yc, y[b, :, d])
        np.testing.assert_array_equal(hc, h[b, d])


MUTANTS = {
    1: "readout before the state update",
    2: "sign of the exponent flipped",
    3: "skip term dropped",
    4: "B read at the wrong step",
    5: "dt missing from the input term",
    6: "sigmoid gate instead of SiLU",
    7: "softplus dropped",
    8: "bias added after softplus",
    9: "Euler step instead of zero-order hold",
    10: "B and C swapped",
    11: "B/C rows taken from another batch",
    12: "initial state ignored",
    13: "initial state not decayed at the first step",
    14: "Euler factor with the page's sign (1 - dt A)",
    15: "convolution reads future steps",
    16: "convolution taps in reverse order",
    17: "SiLU after the convolution dropped",
    18: "convolution bias dropped",
    19: "backward: the decay's dependence on dt dropped",
    20: "backward: adjoint carried with the earlier step's factor",
    21: "backward: dC from the previous state",
    22: "backward: softplus derivative dropped",
    23: "backward: gate derivative taken as the sigmoid alone",
    24: "magnitude: the skip term left out",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda k: MUTANTS[k].replace(" ", "_"))
def test_mutants_are_caught(mutant, tmp_path):
    """A plausible mistake planted in a copy of the oracle must fail at least one pin."""
    path = oracle.build(mutant=mutant, out=str(tmp_path / f"m{mutant}.so"))
    lib = oracle.load(path)
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant '{MUTANTS[mutant]}' passed every pin"
