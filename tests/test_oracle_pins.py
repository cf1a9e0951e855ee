"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Each pin is an independent computation (a closed form, a brute-force
expansion, a dense quadratic form, a hand-worked example or an invariant),
chosen so that a dropped term, a wrong sign or index or a transposed operand
in the oracle fails at least one of them.  CPU only.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from selective_state_space_146_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _ev(s):
    return float(eval(str(s), {"__builtins__": {}}, {"log": math.log, "exp": math.exp}))


def _rand_case(rng, Bsz, Dch, N, L, gate=True, skip=True, bias=True):
    u = rng.standard_normal((Bsz, Dch, L))
    delta = 0.3 * rng.standard_normal((Bsz, Dch, L))
    A = -rng.uniform(0.2, 3.0, (Dch, N))  # not a ladder: catches n-index mix-ups
    Bm = rng.standard_normal((Bsz, N, L))
    Cm = rng.standard_normal((Bsz, N, L))
    D = rng.standard_normal(Dch) if skip else None
    z = rng.standard_normal((Bsz, Dch, L)) if gate else None
    db = rng.uniform(-2.0, 0.5, Dch) if bias else None
    return u, delta, A, Bm, Cm, D, z, db


def _softplus(x):
    return math.log1p(math.exp(x)) if x <= 0 else x + math.log1p(math.exp(-x))


# --------------------------------------------------------------------------
# Hand-worked examples (golden fixture).


def test_golden_selective_hand_worked():
    g = json.load(open(GOLDEN))
    for case in g["selective"]:
        N, L = case["N"], case["L"]
        A = np.array([[_ev(v) for v in row] for row in case["A"]])
        u = np.array(case["u"], float).reshape(1, 1, L)
        dl = np.array(case["delta"], float).reshape(1, 1, L)
        Bm = np.array(case["B"], float).reshape(1, N, L)
        Cm = np.array(case["C"], float).reshape(1, N, L)
        D = None if case["D"] is None else np.array([case["D"]], float)
        z = None if case["z"] is None else np.array([_ev(v) for v in case["z"]]).reshape(1, 1, L)
        db = None if case["delta_bias"] is None else np.array([_ev(case["delta_bias"])])
        y, last = oracle.selective_scan(u, dl, A, Bm, Cm, D, z, db, softplus=case["softplus"])
        want_y = np.array([_ev(v) for v in case["y"]])
        want_s = np.array([_ev(v) for v in case["last_state"]])
        np.testing.assert_allclose(y.ravel(), want_y, rtol=1e-13, atol=1e-13, err_msg=case["name"])
        np.testing.assert_allclose(last.ravel(), want_s, rtol=1e-13, atol=1e-13, err_msg=case["name"])


def test_golden_ssd_hand_worked():
    g = json.load(open(GOLDEN))
    for case in g["ssd"]:
        L, H, P, G, N = (case[k] for k in "LHPGN")
        x = np.array(case["x"], float).reshape(1, L, H, P)
        dt = np.array(case["dt"], float).reshape(1, L, H)
        A = np.array([_ev(v) for v in case["A_head"]])
        Bm = np.array(case["B"], float).reshape(1, L, G, N)
        Cm = np.array(case["C"], float).reshape(1, L, G, N)
        D = np.array(case["D"], float)
        y, last = oracle.ssd(x, dt, A, Bm, Cm, D)
        want_y = np.vectorize(_ev)(np.array(case["y"], dtype=object)).astype(float)
        want_s = np.vectorize(_ev)(np.array(case["last_state"], dtype=object)).astype(float)
        np.testing.assert_allclose(y.reshape(L, H, P), want_y, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(last.reshape(H, P, N), want_s, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# P1: with input-independent delta, B and C the system is time invariant and
# the scan is a causal convolution with kernel K_k = sum_n C_n Abar_n^k Bbar_n
# (study notes §3.2; paper talk §2.2).


@pytest.mark.parametrize("softplus", [False, True])
def test_lti_equals_causal_convolution(softplus):
    rng = np.random.default_rng(1)
    Dch, N, L = 3, 5, 300
    A = -rng.uniform(0.05, 2.0, (Dch, N))
    dconst = rng.uniform(0.05, 0.6, Dch)
    Bn = rng.standard_normal(N)
    Cn = rng.standard_normal(N)
    Dv = rng.standard_normal(Dch)
    u = rng.standard_normal((1, Dch, L))
    delta = np.broadcast_to(dconst[None, :, None], (1, Dch, L)).copy()
    Bm = np.broadcast_to(Bn[None, :, None], (1, N, L)).copy()
    Cm = np.broadcast_to(Cn[None, :, None], (1, N, L)).copy()
    y, _ = oracle.selective_scan(u, delta, A, Bm, Cm, Dv, None, None, softplus=softplus)
    for d in range(Dch):
        dl = _softplus(dconst[d]) if softplus else dconst[d]
        abar = np.exp(dl * A[d])
        k = np.arange(L)
        K = ((abar[None, :] ** k[:, None]) * (dl * Bn)[None, :] * Cn[None, :]).sum(1)
        conv = np.array([np.dot(K[: t + 1], u[0, d, t::-1]) for t in range(L)])
        want = conv + Dv[d] * u[0, d]
        np.testing.assert_allclose(y[0, d], want, rtol=1e-11, atol=1e-12 * np.abs(want).max())


# --------------------------------------------------------------------------
# P2: delta -> 0 leaves the state at zero and y = D u (times the gate).


def test_delta_zero_limit():
    rng = np.random.default_rng(2)
    u, _, A, Bm, Cm, D, z, _ = _rand_case(rng, 2, 4, 6, 50)
    zero = np.zeros_like(u)
    y, last = oracle.selective_scan(u, zero, A, Bm, Cm, D, z, None, softplus=False)
    gate = z / (1.0 + np.exp(-z))
    np.testing.assert_array_equal(last, 0.0)
    np.testing.assert_allclose(y, D[None, :, None] * u * gate, rtol=0, atol=1e-15)
    # softplus(-40) ~ 4e-18: the same limit up to that size.
    y2, last2 = oracle.selective_scan(u, zero, A, Bm, Cm, D, z, np.full(4, -40.0), softplus=True)
    np.testing.assert_allclose(y2, D[None, :, None] * u * gate, rtol=0, atol=1e-12)
    assert np.abs(last2).max() < 1e-12


# --------------------------------------------------------------------------
# P3: brute-force unrolling h_t = sum_{s<=t} (prod_{r=s+1..t} Abar_r) Bbar_s u_s
# with plain Python floats and explicit products.


def _brute_selective(u, delta, A, Bm, Cm, D, z, db, softplus):
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    if Bm.ndim == 4:  # one B, C per group of Dch / G consecutive channels
        G = Bm.shape[1]
        grp = [d // (Dch // G) for d in range(Dch)]
        return _brute_grouped(u, delta, A, Bm, Cm, D, z, db, softplus, grp)
    y = np.zeros((Bsz, Dch, L))
    last = np.zeros((Bsz, Dch, N))
    for b, d in itertools.product(range(Bsz), range(Dch)):
        dl = []
        for t in range(L):
            v = float(delta[b, d, t]) + (float(db[d]) if db is not None else 0.0)
            dl.append(_softplus(v) if softplus else v)

        def h_at(t, n):  # state after step t, as an explicit sum of products
            acc = 0.0
            for s in range(t + 1):
                prod = 1.0
                for r in range(s + 1, t + 1):
                    prod *= math.exp(dl[r] * A[d, n])
                acc += prod * dl[s] * Bm[b, n, s] * u[b, d, s]
            return acc

        for t in range(L):
            out = sum(Cm[b, n, t] * h_at(t, n) for n in range(N))
            if D is not None:
                out += D[d] * u[b, d, t]
            if z is not None:
                out *= z[b, d, t] / (1.0 + math.exp(-z[b, d, t]))
            y[b, d, t] = out
        last[b, d] = [h_at(L - 1, n) for n in range(N)]
    return y, last


def _brute_grouped(u, delta, A, Bm, Cm, D, z, db, softplus, grp):
    """Channel d of a grouped call, unrolled with its group's B, C written out
    as a per-channel 3-D copy, one channel at a time."""
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    y = np.zeros((Bsz, Dch, L))
    last = np.zeros((Bsz, Dch, N))
    for d in range(Dch):
        Bd = np.stack([Bm[b, grp[d]] for b in range(Bsz)])  # (Bsz, N, L)
        Cd = np.stack([Cm[b, grp[d]] for b in range(Bsz)])
        yd, ld = _brute_selective(u[:, d:d + 1], delta[:, d:d + 1], A[d:d + 1], Bd, Cd,
                                  None if D is None else D[d:d + 1],
                                  None if z is None else z[:, d:d + 1],
                                  None if db is None else db[d:d + 1], softplus)
        y[:, d] = yd[:, 0]
        last[:, d] = ld[:, 0]
    return y, last


@pytest.mark.parametrize("L", [1, 2, 5, 8])
@pytest.mark.parametrize("flags", [(True, True, True, True), (False, False, False, False),
                                   (True, False, True, False)])
def test_brute_force_unrolling(L, flags):
    gate, skip, bias, softplus = flags
    rng = np.random.default_rng(10 + L)
    u, delta, A, Bm, Cm, D, z, db = _rand_case(rng, 2, 3, 4, L, gate, skip, bias)
    y, last = oracle.selective_scan(u, delta, A, Bm, Cm, D, z, db, softplus=softplus)
    yb, lb = _brute_selective(u, delta, A, Bm, Cm, D, z, db, softplus)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(last, lb, rtol=1e-12, atol=1e-13)




@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("L", [1, 3, 6])
def test_grouped_brute_force_unrolling(G, L):
    """B, C per channel group (G = Dch: one per channel) against the explicit
    sums of products, channel by channel with the group's B, C."""
    rng = np.random.default_rng(100 + 10 * G + L)
    Bsz, Dch, N = 2, 4, 3
    u, delta, A, _, _, D, z, db = _rand_case(rng, Bsz, Dch, N, L)
    Bm = rng.standard_normal((Bsz, G, N, L))
    Cm = rng.standard_normal((Bsz, G, N, L))
    y, last = oracle.selective_scan(u, delta, A, Bm, Cm, D, z, db)
    yb, lb = _brute_selective(u, delta, A, Bm, Cm, D, z, db, True)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(last, lb, rtol=1e-12, atol=1e-13)


def test_grouped_with_copies_of_one_B_equals_shared():
    """Every group holding the same B, C gives the shared-B, C scan."""
    rng = np.random.default_rng(7)
    Bsz, Dch, N, L, G = 2, 6, 5, 40, 3
    u, delta, A, Bm, Cm, D, z, db = _rand_case(rng, Bsz, Dch, N, L)
    Bg = np.repeat(Bm[:, None], G, axis=1)
    Cg = np.repeat(Cm[:, None], G, axis=1)
    y1, s1 = oracle.selective_scan(u, delta, A, Bm, Cm, D, z, db)
    y2, s2 = oracle.selective_scan(u, delta, A, Bg, Cg, D, z, db)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(s1, s2)
# --------------------------------------------------------------------------
# P4: the final state is the carry: running [0, L1) and then [L1, L) from
# that state reproduces y and the final state exactly (paper talk §5.3, §5.4:
# chunks with the state passed across the boundary).


def test_split_invariance_selective():
    rng = np.random.default_rng(4)
    u, delta, A, Bm, Cm, D, z, db = _rand_case(rng, 2, 5, 7, 91)
    y, last = oracle.selective_scan(u, delta, A, Bm, Cm, D, z, db)
    for L1 in (1, 40, 90):
        sl1, sl2 = slice(0, L1), slice(L1, None)
        y1, s1 = oracle.selective_scan(u[..., sl1], delta[..., sl1], A, Bm[..., sl1], Cm[..., sl1],
                                       D, z[..., sl1], db)
        y2, s2 = oracle.selective_scan(u[..., sl2], delta[..., sl2], A, Bm[..., sl2], Cm[..., sl2],
                                       D, z[..., sl2], db, h0=s1)
        np.testing.assert_array_equal(np.concatenate([y1, y2], -1), y)
        np.testing.assert_array_equal(s2, last)


def test_split_invariance_ssd():
    rng = np.random.default_rng(5)
    Bsz, L, H, P, G, N = 2, 37, 4, 3, 2, 5
    x = rng.standard_normal((Bsz, L, H, P))
    dt = rng.uniform(0.01, 0.5, (Bsz, L, H))
    A = -rng.uniform(0.5, 4, H)
    Bm = rng.standard_normal((Bsz, L, G, N))
    Cm = rng.standard_normal((Bsz, L, G, N))
    D = rng.standard_normal(H)
    y, last = oracle.ssd(x, dt, A, Bm, Cm, D)
    y1, s1 = oracle.ssd(x[:, :20], dt[:, :20], A, Bm[:, :20], Cm[:, :20], D)
    y2, s2 = oracle.ssd(x[:, 20:], dt[:, 20:], A, Bm[:, 20:], Cm[:, 20:], D, h0=s1)
    np.testing.assert_array_equal(np.concatenate([y1, y2], 1), y)
    np.testing.assert_array_equal(s2, last)


# --------------------------------------------------------------------------
# P5: linearity in u of the pre-gate output; zero cases.


def test_linearity_and_zero_cases():
    rng = np.random.default_rng(6)
    u1, delta, A, Bm, Cm, D, _, db = _rand_case(rng, 1, 4, 6, 64, gate=False)
    u2 = rng.standard_normal(u1.shape)
    a, b = 0.7, -1.9
    y1, s1 = oracle.selective_scan(u1, delta, A, Bm, Cm, D, None, db)
    y2, s2 = oracle.selective_scan(u2, delta, A, Bm, Cm, D, None, db)
    y3, s3 = oracle.selective_scan(a * u1 + b * u2, delta, A, Bm, Cm, D, None, db)
    np.testing.assert_allclose(y3, a * y1 + b * y2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(s3, a * s1 + b * s2, rtol=1e-11, atol=1e-12)
    y0, _ = oracle.selective_scan(u1, delta, A, Bm, np.zeros_like(Cm), np.zeros(4), None, db)
    np.testing.assert_array_equal(y0, 0.0)
    yz, sz = oracle.selective_scan(np.zeros_like(u1), delta, A, Bm, Cm, D, None, db)
    np.testing.assert_array_equal(yz, 0.0)
    np.testing.assert_array_equal(sz, 0.0)
    # the skip term is exactly D * u when C = 0
    yd, _ = oracle.selective_scan(u1, delta, A, Bm, np.zeros_like(Cm), D, None, db)
    np.testing.assert_allclose(yd, D[None, :, None] * u1, rtol=0, atol=0)


# --------------------------------------------------------------------------
# P6: SSD is the selective scan with one scalar A per head, delta = dt, and
# channels d = (h, p) reading their group's B and C.


def test_ssd_is_selective_scan_with_scalar_A():
    rng = np.random.default_rng(7)
    Bsz, L, H, P, G, N = 2, 29, 4, 3, 2, 6
    x = rng.standard_normal((Bsz, L, H, P))
    dt = rng.uniform(0.01, 0.6, (Bsz, L, H))
    A = -rng.uniform(0.5, 5, H)
    Bm = rng.standard_normal((Bsz, L, G, N))
    Cm = rng.standard_normal((Bsz, L, G, N))
    D = rng.standard_normal(H)
    y, last = oracle.ssd(x, dt, A, Bm, Cm, D)
    hpg = H // G
    for g in range(G):
        heads = list(range(g * hpg, (g + 1) * hpg))
        # channels (h, p) of this group, h-major
        u = x[:, :, heads, :].transpose(0, 2, 3, 1).reshape(Bsz, hpg * P, L)
        dl = np.repeat(dt[:, :, heads].transpose(0, 2, 1), P, axis=1)
        Asel = np.repeat(A[heads], P)[:, None] * np.ones((1, N))
        Bs = Bm[:, :, g, :].transpose(0, 2, 1)
        Cs = Cm[:, :, g, :].transpose(0, 2, 1)
        Ds = np.repeat(D[heads], P)
        ys, ss = oracle.selective_scan(u, dl, Asel, Bs, Cs, Ds, None, None, softplus=False)
        np.testing.assert_allclose(ys.reshape(Bsz, hpg, P, L).transpose(0, 3, 1, 2),
                                   y[:, :, heads, :], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(ss.reshape(Bsz, hpg, P, N), last[:, heads], rtol=1e-12,
                                   atol=1e-12)


# --------------------------------------------------------------------------
# P7: the SSD "attention" (dual, quadratic) form equals the recurrence
# (study notes §5.1: the SSM / attention duality):
#   y_t = sum_{s<=t} (C_t . B_s) exp(sum_{r=s+1..t} dt_r A) dt_s x_s + D x_t


def test_ssd_quadratic_dual_form():
    rng = np.random.default_rng(8)
    Bsz, L, H, P, G, N = 2, 200, 4, 5, 2, 8
    x = rng.standard_normal((Bsz, L, H, P))
    dt = rng.uniform(0.001, 0.2, (Bsz, L, H))
    A = -rng.uniform(1, 8, H)
    Bm = rng.standard_normal((Bsz, L, G, N))
    Cm = rng.standard_normal((Bsz, L, G, N))
    D = rng.standard_normal(H)
    y, last = oracle.ssd(x, dt, A, Bm, Cm, D)
    hpg = H // G
    for b in range(Bsz):
        for h in range(H):
            g = h // hpg
            cs = np.concatenate([[0.0], np.cumsum(dt[b, :, h] * A[h])])  # cs[t+1] = sum_{r<=t}
            seg = cs[1:, None] - cs[None, 1:]  # sum_{r=s+1..t} for t >= s
            mask = np.tril(np.ones((L, L), bool))
            Lmat = np.where(mask, np.exp(np.where(mask, seg, 0.0)), 0.0) * dt[b, None, :, h]
            CB = Cm[b, :, g, :] @ Bm[b, :, g, :].T
            want = (Lmat * CB) @ x[b, :, h, :] + D[h] * x[b, :, h, :]
            np.testing.assert_allclose(y[b, :, h, :], want, rtol=1e-10, atol=1e-11)
            # final state: sum_s exp(sum_{r=s+1..L-1} dt_r A) dt_s x_s B_s^T
            w = np.exp(cs[-1] - cs[1:]) * dt[b, :, h]
            S = (x[b, :, h, :] * w[:, None]).T @ Bm[b, :, g, :]
            np.testing.assert_allclose(last[b, h], S, rtol=1e-10, atol=1e-11)


# --------------------------------------------------------------------------
# The causal depthwise conv1d + SiLU in front of the scan (study notes §4.3,
# paper talk §3.1).


def _conv_silu_by_numpy(x, w, bias):
    """The same map through numpy's convolution (a different algorithm):
    left-pad by W-1 zeros, correlate with the taps, add the bias, SiLU."""
    Bsz, D, L = x.shape
    W = w.shape[1]
    out = np.empty_like(x)
    for b in range(Bsz):
        for d in range(D):
            pad = np.concatenate([np.zeros(W - 1), x[b, d]])
            pre = np.convolve(pad, w[d][::-1], mode="valid") + (bias[d] if bias is not None else 0)
            out[b, d] = pre / (1 + np.exp(-pre))
    return out


def test_conv_identity_and_delay_kernels():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((2, 5, 40))
    ident = np.zeros((5, 4))
    ident[:, 3] = 1.0
    u = oracle.causal_conv1d_silu(x, ident)
    np.testing.assert_allclose(u, x / (1 + np.exp(-x)), rtol=1e-15, atol=1e-15)
    delay = np.zeros((5, 4))
    delay[:, 0] = 1.0
    u = oracle.causal_conv1d_silu(x, delay)
    np.testing.assert_array_equal(u[..., :3], 0.0)
    np.testing.assert_allclose(u[..., 3:], x[..., :-3] / (1 + np.exp(-x[..., :-3])), rtol=1e-15)
    bias = rng.standard_normal(5)
    u = oracle.causal_conv1d_silu(x, np.zeros((5, 4)), bias)
    np.testing.assert_allclose(u, np.broadcast_to((bias / (1 + np.exp(-bias)))[None, :, None],
                                                  u.shape), rtol=1e-15)


@pytest.mark.parametrize("W", [1, 2, 4])
def test_conv_matches_numpy_convolution(W):
    rng = np.random.default_rng(40 + W)
    x = rng.standard_normal((2, 6, 33))
    w = rng.standard_normal((6, W))
    bias = rng.standard_normal(6)
    np.testing.assert_allclose(oracle.causal_conv1d_silu(x, w, bias), _conv_silu_by_numpy(x, w, bias),
                               rtol=1e-12, atol=1e-13)


def test_conv_then_scan_composes():
    rng = np.random.default_rng(45)
    x = rng.standard_normal((1, 4, 30))
    w = rng.standard_normal((4, 4))
    cb = rng.standard_normal(4)
    _, delta, A, Bm, Cm, D, z, db = _rand_case(rng, 1, 4, 5, 30)
    y, s = oracle.conv_selective_scan(x, w, cb, delta, A, Bm, Cm, D, z, db)
    u = _conv_silu_by_numpy(x, w, cb)
    y2, s2 = oracle.selective_scan(u, delta, A, Bm, Cm, D, z, db)
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s, s2, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Planted mistakes: a copy of the oracle with one plausible bug (made in a
# temporary copy of the C source, compiled on the CPU) must fail at least one
# of the pins above.


_MUTANTS = {
    "no_decay": ("hp[n] = abar * hp[n] + bbar * ur[t];", "hp[n] = hp[n] + bbar * ur[t];"),
    "input_sign": ("hp[n] = abar * hp[n] + bbar * ur[t];", "hp[n] = abar * hp[n] - bbar * ur[t];"),
    "readout_before_update": (
        "hp[n] = abar * hp[n] + bbar * ur[t];\n                out += Cg[n * L + t] * hp[n];",
        "out += Cg[n * L + t] * hp[n];\n                hp[n] = abar * hp[n] + bbar * ur[t];"),
    "group_index": ("int64_t g = d / (D / G);", "int64_t g = d % G;"),
    "A_transposed": ("exp(dlt * A[d * N + n])", "exp(dlt * A[n * D + d])"),
    "gate_sign": ("out * zr[t] / (1.0 + exp(-zr[t]))", "out * zr[t] / (1.0 + exp(zr[t]))"),
    "softplus_dropped": ("if (softplus) dlt = softplus_d(dlt);", ""),
    "skip_dropped": ("if (Dv) out += Dv[d] * ur[t];", ""),
    "ssd_B_C_swapped": ("out += cr[n] * S[p * N + n];", "out += br[n] * S[p * N + n];"),
    "ssd_no_dt_on_input": ("a * S[p * N + n] + dtv * xr[p] * br[n]", "a * S[p * N + n] + xr[p] * br[n]"),
    "ssd_group_index": ("int64_t g = hh / heads_per_group;", "int64_t g = hh % G;"),
    "conv_taps_reversed": ("int64_t s = t - (W - 1) + k;", "int64_t s = t - k;"),
    "conv_bias_dropped": ("double pre = bias ? bias[d] : 0.0;", "double pre = 0.0;"),
    "conv_no_silu": ("ur[t] = pre / (1.0 + exp(-pre));", "ur[t] = pre;"),
    "bwd_no_adjoint_carry": ("g[n] *= abar; /* carry to step t-1 */", ""),
    "bwd_dz_missing_term": ("(sg + zr[t] * sg * (1.0 - sg))", "(sg)"),
    "bwd_dA_wrong_state": ("dA[d * N + n] += g[n] * hs[t * N + n] * abar * dl;",
                           "dA[d * N + n] += g[n] * hs[(t + 1) * N + n] * abar * dl;"),
    "bwd_softplus_chain_dropped": ("double dx = softplus ? ddl / (1.0 + exp(-x)) : ddl;",
                                   "double dx = ddl;"),
}


def _pins_pass(lib):
    """Run the pins against a given oracle library; True if all hold."""
    try:
        rng = np.random.default_rng(11)
        u, delta, A, Bm, Cm, D, z, db = _rand_case(rng, 1, 3, 4, 6)
        y, last = lib.selective_scan(u, delta, A, Bm, Cm, D, z, db, softplus=True)
        yb, lb = _brute_selective(u, delta, A, Bm, Cm, D, z, db, True)
        if not (np.allclose(y, yb, rtol=1e-12, atol=1e-13) and np.allclose(last, lb, rtol=1e-12,
                                                                            atol=1e-13)):
            return False
        Bg = rng.standard_normal((1, 3, 4, 6))
        Cg = rng.standard_normal((1, 3, 4, 6))
        u6 = np.concatenate([u, u], axis=1)
        d6 = np.concatenate([delta, delta], axis=1)
        A6, D6, db6 = np.concatenate([A, A]), np.concatenate([D, D]), np.concatenate([db, db])
        z6 = np.concatenate([z, z], axis=1)
        yg, lg = lib.selective_scan(u6, d6, A6, Bg, Cg, D6, z6, db6, softplus=True)
        ygb, lgb = _brute_selective(u6, d6, A6, Bg, Cg, D6, z6, db6, True)
        if not (np.allclose(yg, ygb, rtol=1e-12, atol=1e-13) and
                np.allclose(lg, lgb, rtol=1e-12, atol=1e-13)):
            return False
        Bsz, L, H, P, G, N = 1, 24, 4, 3, 2, 5
        x = rng.standard_normal((Bsz, L, H, P))
        dt = rng.uniform(0.01, 0.3, (Bsz, L, H))
        Ah = -rng.uniform(1, 4, H)
        Bs = rng.standard_normal((Bsz, L, G, N))
        Cs = rng.standard_normal((Bsz, L, G, N))
        Dh = rng.standard_normal(H)
        ys, _ = lib.ssd(x, dt, Ah, Bs, Cs, Dh)
        for h in range(H):
            g = h // (H // G)
            cs = np.concatenate([[0.0], np.cumsum(dt[0, :, h] * Ah[h])])
            seg = cs[1:, None] - cs[None, 1:]
            mask = np.tril(np.ones((L, L), bool))
            Lm = np.where(mask, np.exp(np.where(mask, seg, 0.0)), 0.0) * dt[0, None, :, h]
            want = (Lm * (Cs[0, :, g] @ Bs[0, :, g].T)) @ x[0, :, h] + Dh[h] * x[0, :, h]
            if not np.allclose(ys[0, :, h], want, rtol=1e-10, atol=1e-11):
                return False
        xc = rng.standard_normal((2, 3, 17))
        wc = rng.standard_normal((3, 4))
        bc = rng.standard_normal(3)
        uc = lib.causal_conv1d_silu(xc, wc, bc)
        if not np.allclose(uc, _conv_silu_by_numpy(xc, wc, bc), rtol=1e-12, atol=1e-13):
            return False
        return _bwd_matches_finite_differences(lib, seed=17)
    except ValueError:
        return False


def _bwd_matches_finite_differences(lib, seed, Bsz=2, Dch=3, N=4, L=7):
    """Directional derivatives of sum(dout * out) by central differences of
    the forward oracle, against the backward oracle, for every input."""
    try:
        rng = np.random.default_rng(seed)
        u, delta, A, Bm, Cm, D, z, db = _rand_case(rng, Bsz, Dch, N, L)
        dout = rng.standard_normal(u.shape)
        grads = lib.selective_scan_bwd(u, delta, A, Bm, Cm, D, z, db, dout, softplus=True)
        args = dict(u=u, delta=delta, A=A, B=Bm, C=Cm, D=D, z=z, delta_bias=db)
        names = dict(u="du", delta="ddelta", A="dA", B="dB", C="dC", D="dD", z="dz",
                     delta_bias="ddelta_bias")
        eps = 1e-6
        for k, gname in names.items():
            v = rng.standard_normal(args[k].shape)
            plus = dict(args); plus[k] = args[k] + eps * v
            minus = dict(args); minus[k] = args[k] - eps * v
            yp, _ = lib.selective_scan(**plus, softplus=True)
            ym, _ = lib.selective_scan(**minus, softplus=True)
            fd = float(np.sum(dout * (yp - ym)) / (2 * eps))
            an = float(np.sum(grads[gname] * v))
            if not abs(fd - an) <= 1e-6 * max(1.0, abs(fd)):
                return False
        return True
    except ValueError:
        return False


def test_pins_pass_on_the_oracle():
    assert _pins_pass(oracle)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_backward_matches_finite_differences(seed):
    assert _bwd_matches_finite_differences(oracle, seed)


def test_backward_without_optional_inputs():
    """No gate, no skip, no bias, softplus off: the remaining gradients still
    match finite differences."""
    rng = np.random.default_rng(5)
    u, delta, A, Bm, Cm, _, _, _ = _rand_case(rng, 1, 2, 3, 6, gate=False, skip=False, bias=False)
    dout = rng.standard_normal(u.shape)
    g = oracle.selective_scan_bwd(u, delta, A, Bm, Cm, None, None, None, dout, softplus=False)
    assert g["dz"] is None and g["dD"] is None and g["ddelta_bias"] is None
    eps = 1e-6
    for k, arr, gn in (("u", u, "du"), ("delta", delta, "ddelta"), ("A", A, "dA"),
                       ("B", Bm, "dB"), ("C", Cm, "dC")):
        v = rng.standard_normal(arr.shape)
        args = dict(u=u, delta=delta, A=A, B=Bm, C=Cm)
        ap = dict(args); ap[k] = arr + eps * v
        am = dict(args); am[k] = arr - eps * v
        yp, _ = oracle.selective_scan(**ap, softplus=False)
        ym, _ = oracle.selective_scan(**am, softplus=False)
        fd = np.sum(dout * (yp - ym)) / (2 * eps)
        assert abs(fd - np.sum(g[gn] * v)) <= 1e-6 * max(1.0, abs(fd)), k


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_planted_mistake_fails_a_pin(name, tmp_path):
    old, new = _MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.compile_source(str(mutant), str(tmp_path / "libmut.so")))
    assert not _pins_pass(lib), f"planted mistake {name} was not caught"


# --------------------------------------------------------------------------
# The input recipe: checks on the generator (not the method).


def test_input_recipe_properties():
    x = inputs.selective_inputs(1, 64, 16, 256, "f32", seed=0)
    assert x["u"].dtype.is_floating_point and tuple(x["u"].shape) == (1, 64, 256)
    sp = np.log1p(np.exp(x["delta_bias"].double().numpy()))
    assert sp.min() >= 1e-3 * 0.999 and sp.max() <= 1e-1 * 1.001
    np.testing.assert_array_equal(x["A"].numpy()[5], -np.arange(1, 17, dtype=np.float32))
    x2 = inputs.selective_inputs(1, 64, 16, 256, "f32", seed=0)
    assert all((x[k] is None and x2[k] is None) or bool((x[k] == x2[k]).all()) for k in x)
    s = inputs.ssd_inputs(1, 64, 4, 8, 16, 1, "bf16", seed=0)
    assert float(s["dt"].float().min()) > 0
    assert float(s["A_head"].max()) <= -1.0 + 1e-6 and float(s["A_head"].min()) >= -16.0 - 1e-4
