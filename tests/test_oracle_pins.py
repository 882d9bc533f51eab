"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against a formulation that does not share its code or its
shape of computation: the convolution view of an LTI system, the continuous-time solution
that exact ZOH samples, the materialised lower-triangular (semiseparable) matrix, a
library filter or cumulative sum, limits of delta, and the chunked SSD decomposition.
A dropped term, a wrong sign or index, or a swapped operand in the oracle fails at least
one of them.
"""
import json
import os

import numpy as np
import pytest
from scipy.signal import lfilter

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softplus_lib(v):
    # log(1 + e^v) through numpy's logaddexp, not the oracle's formula
    return np.logaddexp(0.0, v)


def _rng(seed):
    return np.random.default_rng(seed)


def _problem(rng, b, L, d, n, gate=True, dskip=True, bias_lo=-5.0, bias_hi=-1.0):
    return dict(
        x=rng.standard_normal((b, L, d)),
        delta=rng.standard_normal((b, L, d)),
        A=-rng.uniform(0.5, 8.0, size=(d, n)),
        B=rng.standard_normal((b, L, n)),
        C=rng.standard_normal((b, L, n)),
        D=rng.standard_normal(d) if dskip else None,
        z=rng.standard_normal((b, L, d)) if gate else None,
        delta_bias=rng.uniform(bias_lo, bias_hi, size=d),
    )


# ---------------------------------------------------------------- LTI: recurrence == convolution

def _lti_inputs(n, L, delta, Bval, C, x):
    A = -np.arange(1, n + 1, dtype=np.float64)[None, :]
    return dict(x=x[None, :, None], delta=np.full((1, L, 1), delta), A=A,
                B=np.full((1, L, n), Bval), C=np.tile(C[None, None, :], (1, L, 1)))


def _conv_output(n, L, delta, Bval, C, x, zoh):
    a = -np.arange(1, n + 1, dtype=np.float64)
    abar = np.exp(delta * a)
    bbar = (abar - 1.0) / a * Bval if zoh else delta * Bval * np.ones(n)
    powers = abar[None, :] ** np.arange(L)[:, None]          # (L, n): A_bar^k
    K = powers @ (C * bbar)                                  # K_k = C . A_bar^k . B_bar
    return np.convolve(K, x)[:L], K


@pytest.mark.parametrize("zoh", [True, False])
def test_lti_recurrence_equals_convolution_page_example(zoh):
    """The pages' worked example: n=16, L=256, delta=0.01, A=-(1..16), B=0.5; recurrent and
    convolution modes agree to 1e-14 (exact ZOH on the page; the delta*B form must agree too)."""
    g = json.load(open(os.path.join(GOLDEN, "lti_recurrent_vs_conv.json")))
    n, L, delta, Bval = g["n"], g["seq_len"], g["delta"], g["B"]
    rng = _rng(42)
    C = rng.standard_normal(n) * 0.1
    t = np.linspace(0, 1, L)
    x = np.sin(2 * np.pi * 3 * t) + 0.5 * np.sin(2 * np.pi * 15 * t) + 0.2 * rng.standard_normal(L)
    inp = _lti_inputs(n, L, delta, Bval, C, x)
    y, _ = oracle.ssm_scan_ref(**inp, delta_softplus=False, zoh=zoh)
    y_conv, K = _conv_output(n, L, delta, Bval, C, x, zoh)
    assert np.max(np.abs(y[0, :, 0] - y_conv)) <= g["max_abs_diff"]
    # the kernel's lag-0 tap is C.B_bar: the output includes the current input
    assert abs(y[0, 0, 0] - K[0] * x[0]) <= 1e-15


def test_lti_random_long_convolution():
    rng = _rng(7)
    n, L = 8, 1000
    C = rng.standard_normal(n)
    x = rng.standard_normal(L)
    for delta in (1e-3, 0.05, 0.7):
        inp = _lti_inputs(n, L, delta, 1.3, C, x)
        y, _ = oracle.ssm_scan_ref(**inp, delta_softplus=False)
        y_conv, _ = _conv_output(n, L, delta, 1.3, C, x, zoh=False)
        assert np.max(np.abs(y[0, :, 0] - y_conv)) <= 1e-12 * max(1.0, np.max(np.abs(y_conv)))


def test_zoh_samples_the_continuous_solution():
    """Exact ZOH is exact for piecewise-constant input: with constant x and h(0)=0 the
    continuous system h' = a h + b x has h(t) = (b x / -a)(1 - e^{a t}); step k of the
    recurrence (which includes input k) is h((k+1) delta)."""
    n, L, delta = 6, 300, 0.037
    a = -np.array([0.3, 1.0, 2.5, 4.0, 7.0, 11.0])
    bvec = np.array([0.5, -1.0, 2.0, 0.25, 1.5, -0.75])
    xval = 1.7
    for k_n in range(n):
        inp = dict(x=np.full((1, L, 1), xval), delta=np.full((1, L, 1), delta), A=a[None, :],
                   B=np.tile(bvec[None, None, :], (1, L, 1)),
                   C=np.tile(np.eye(n)[k_n][None, None, :], (1, L, 1)))
        y, h_last = oracle.ssm_scan_ref(**inp, delta_softplus=False, zoh=True)
        tgrid = (np.arange(L) + 1) * delta
        h_exact = bvec[k_n] * xval / (-a[k_n]) * (1.0 - np.exp(a[k_n] * tgrid))
        np.testing.assert_allclose(y[0, :, 0], h_exact, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(h_last[0, 0, :], bvec * xval / (-a) * (1 - np.exp(a * L * delta)),
                                   rtol=1e-12)


def test_n1_lti_matches_library_filter():
    """N=1, constant delta: a first-order IIR filter h_t = a h_{t-1} + b x_t (scipy lfilter)."""
    rng = _rng(3)
    L = 777
    x = rng.standard_normal(L)
    a_cont, delta, bval, cval = -2.3, 0.11, 0.8, -1.7
    inp = dict(x=x[None, :, None], delta=np.full((1, L, 1), delta), A=np.array([[a_cont]]),
               B=np.full((1, L, 1), bval), C=np.full((1, L, 1), cval))
    y, h_last = oracle.ssm_scan_ref(**inp, delta_softplus=False)
    h = lfilter([delta * bval], [1.0, -np.exp(delta * a_cont)], x)
    np.testing.assert_allclose(y[0, :, 0], cval * h, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h_last[0, 0, 0], h[-1], rtol=1e-12)


# ---------------------------------------------------------------- semiseparable brute force

def _brute_force_mamba1(p, zoh=False):
    """y = M x per channel with M[t, s] = sum_n C[t,n] exp(A[n] * sum_{k=s+1..t} dt_k) Bbar_s[n]."""
    x, A, B, C = p["x"], p["A"], p["B"], p["C"]
    b, L, d = x.shape
    dt = _softplus_lib(p["delta"] + p["delta_bias"][None, None, :])
    y = np.zeros_like(x)
    h_last = np.zeros((b, d, A.shape[1]))
    for bi in range(b):
        for di in range(d):
            cs = np.concatenate([[0.0], np.cumsum(dt[bi, :, di])])      # cs[t+1] = sum_{k<=t}
            a = A[di]
            # decay[t, s, n] = exp(a_n * (cs[t+1] - cs[s+1]))
            seg = cs[1:, None] - cs[None, 1:]
            tri = np.tril(np.ones((L, L), dtype=bool))
            decay = np.exp(np.where(tri, seg, 0.0)[:, :, None] * a[None, None, :])
            if zoh:
                bbar = np.expm1(dt[bi, :, di][:, None] * a[None, :]) / a[None, :] * B[bi]
            else:
                bbar = dt[bi, :, di][:, None] * B[bi]
            M = np.einsum("tn,tsn,sn->ts", C[bi], decay, bbar) * tri
            yy = M @ x[bi, :, di]
            if p.get("D") is not None:
                yy = yy + p["D"][di] * x[bi, :, di]
            if p.get("z") is not None:
                zz = p["z"][bi, :, di]
                yy = yy * zz / (1.0 + np.exp(-zz))
            y[bi, :, di] = yy
            h_last[bi, di] = np.einsum("sn,sn,s->n", decay[-1], bbar, x[bi, :, di])
    return y, h_last


@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("gate,dskip", [(True, True), (False, False), (True, False)])
def test_mamba1_matches_semiseparable_matrix(gate, dskip, zoh):
    rng = _rng(11)
    p = _problem(rng, 2, 37, 3, 5, gate=gate, dskip=dskip)
    y, h_last = oracle.ssm_scan_ref(**p, zoh=zoh)
    y_bf, h_bf = _brute_force_mamba1(p, zoh=zoh)
    np.testing.assert_allclose(y, y_bf, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h_last, h_bf, rtol=1e-11, atol=1e-12)


def test_first_tokens_follow_the_pages_expansion():
    g = json.load(open(os.path.join(GOLDEN, "first_tokens.json")))
    rng = _rng(5)
    n, L = 4, 3
    a = -np.array([1.0, 2.0, 3.0, 4.0])
    delta = 0.3
    Bv, Cv = rng.standard_normal(n), rng.standard_normal(n)
    u = rng.standard_normal(L)
    inp = dict(x=u[None, :, None], delta=np.full((1, L, 1), delta), A=a[None, :],
               B=np.tile(Bv[None, None, :], (1, L, 1)), C=np.tile(Cv[None, None, :], (1, L, 1)))
    y, _ = oracle.ssm_scan_ref(**inp, delta_softplus=False)
    abar, bbar = np.exp(delta * a), delta * Bv
    for k, terms in g["terms"].items():
        expect = sum(np.dot(Cv, abar ** pw * bbar) * u[j] for pw, j in terms)
        assert abs(y[0, int(k), 0] - expect) <= 1e-14


# ---------------------------------------------------------------- special cases and limits

def test_a_zero_is_a_cumulative_sum():
    rng = _rng(21)
    p = _problem(rng, 2, 50, 3, 4, gate=False, dskip=False)
    p["A"] = np.zeros_like(p["A"])
    y, h_last = oracle.ssm_scan_ref(**p)
    dt = _softplus_lib(p["delta"] + p["delta_bias"])
    for bi in range(2):
        for di in range(3):
            hh = np.cumsum(dt[bi, :, di, None] * p["B"][bi] * p["x"][bi, :, di, None], axis=0)
            np.testing.assert_allclose(y[bi, :, di], np.sum(p["C"][bi] * hh, axis=1), rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(h_last[bi, di], hh[-1], rtol=1e-12, atol=1e-12)


def test_b_zero_leaves_only_the_skip_and_gate():
    rng = _rng(22)
    p = _problem(rng, 1, 40, 5, 3)
    p["B"] = np.zeros_like(p["B"])
    y, h_last = oracle.ssm_scan_ref(**p)
    z = p["z"]
    np.testing.assert_allclose(y, p["D"][None, None, :] * p["x"] * z / (1 + np.exp(-z)), rtol=1e-13, atol=1e-14)
    assert np.all(h_last == 0.0)


def test_small_delta_limit_keeps_the_state_and_drops_the_input():
    """delta -> 0: A_bar -> 1 and B_bar -> 0, so y -> D x, and to first order the SSM part is
    C_t . sum_{s<=t} dt_s B_s x_s (selection: 'small delta ignores the input')."""
    rng = _rng(23)
    p = _problem(rng, 1, 60, 2, 4, gate=False, dskip=False)
    p["delta_bias"] = np.full(2, -30.0)
    y, _ = oracle.ssm_scan_ref(**p)
    dt = _softplus_lib(p["delta"] + p["delta_bias"])
    assert np.max(dt) < 1e-11
    first = np.einsum("tn,tdn->td", p["C"][0], np.cumsum(dt[0, :, :, None] * p["B"][0][:, None, :] * p["x"][0, :, :, None], axis=0))
    np.testing.assert_allclose(y[0], first, rtol=1e-8, atol=0)
    q = dict(p, D=np.array([0.7, -1.2]))
    yq, _ = oracle.ssm_scan_ref(**q)
    np.testing.assert_allclose(yq[0], q["D"][None, :] * p["x"][0], rtol=0, atol=1e-10)


def test_large_delta_limit_forgets_the_past():
    """delta -> inf with A < 0: A_bar -> 0, so y_t -> dt_t (C_t . B_t) x_t + D x_t."""
    rng = _rng(24)
    p = _problem(rng, 1, 30, 3, 4, gate=False, dskip=True)
    p["delta_bias"] = np.full(3, 60.0)
    y, _ = oracle.ssm_scan_ref(**p)
    dt = _softplus_lib(p["delta"] + p["delta_bias"])
    expect = dt[0] * np.sum(p["C"][0] * p["B"][0], axis=1)[:, None] * p["x"][0] + p["D"][None, :] * p["x"][0]
    np.testing.assert_allclose(y[0], expect, rtol=1e-12)


def test_softplus_matches_library_and_is_stable():
    v = np.array([-800.0, -40.0, -1e-3, 0.0, 1e-3, 5.0, 40.0, 800.0])
    np.testing.assert_allclose(oracle.softplus(v), np.logaddexp(0.0, v), rtol=1e-15, atol=0)
    # the C recurrence applies the same softplus: one step, one state, C=B=x=1, A=0
    for vv in v:
        inp = dict(x=np.ones((1, 1, 1)), delta=np.full((1, 1, 1), vv), A=np.zeros((1, 1)),
                   B=np.ones((1, 1, 1)), C=np.ones((1, 1, 1)))
        y, _ = oracle.ssm_scan_ref(**inp)
        assert y[0, 0, 0] == pytest.approx(np.logaddexp(0.0, vv), rel=1e-15, abs=0)


# ---------------------------------------------------------------- invariances

def test_split_and_resume_through_h0():
    rng = _rng(31)
    p = _problem(rng, 2, 90, 3, 6)
    y, h_last = oracle.ssm_scan_ref(**p)
    L1 = 41
    first = {k: (v[:, :L1] if k in ("x", "delta", "B", "C", "z") else v) for k, v in p.items()}
    second = {k: (v[:, L1:] if k in ("x", "delta", "B", "C", "z") else v) for k, v in p.items()}
    y1, h1 = oracle.ssm_scan_ref(**first)
    y2, h2 = oracle.ssm_scan_ref(**second, h0=h1)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h2, h_last, rtol=1e-13, atol=1e-14)


def test_reverse_is_the_scan_of_the_flipped_sequence():
    rng = _rng(32)
    p = _problem(rng, 2, 45, 3, 4)
    y_rev, h_rev = oracle.ssm_scan_ref(**p, reverse=True)
    flipped = {k: (np.ascontiguousarray(v[:, ::-1]) if k in ("x", "delta", "B", "C", "z") else v) for k, v in p.items()}
    y_f, h_f = oracle.ssm_scan_ref(**flipped)
    np.testing.assert_allclose(y_rev, y_f[:, ::-1], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(h_rev, h_f, rtol=1e-14, atol=1e-15)


def test_channels_are_independent_and_b_c_shared():
    """Running channels one at a time gives the same result (no cross-channel leakage)."""
    rng = _rng(33)
    p = _problem(rng, 2, 30, 4, 3)
    y, h = oracle.ssm_scan_ref(**p)
    for di in range(4):
        q = dict(p)
        for k in ("x", "delta", "z"):
            q[k] = p[k][:, :, di:di + 1]
        q["A"], q["D"], q["delta_bias"] = p["A"][di:di + 1], p["D"][di:di + 1], p["delta_bias"][di:di + 1]
        yd, hd = oracle.ssm_scan_ref(**q)
        np.testing.assert_array_equal(yd[:, :, 0], y[:, :, di])
        np.testing.assert_array_equal(hd[:, 0], h[:, di])


# ---------------------------------------------------------------- SSD (Mamba-2)

def _ssd_problem(rng, b, L, H, P, N, gate=False, dskip=False):
    return dict(
        x=rng.standard_normal((b, L, H, P)),
        delta=rng.standard_normal((b, L, H)),
        A=-rng.uniform(1.0, 16.0, size=H),
        B=rng.standard_normal((b, L, 1, N)),
        C=rng.standard_normal((b, L, 1, N)),
        D=rng.standard_normal(H) if dskip else None,
        z=rng.standard_normal((b, L, H, P)) if gate else None,
        delta_bias=rng.uniform(-6.0, -2.0, size=H),
    )


def _brute_force_ssd(p):
    x, A, B, C = p["x"], p["A"], p["B"][:, :, 0], p["C"][:, :, 0]
    b, L, H, P = x.shape
    dt = _softplus_lib(p["delta"] + p["delta_bias"][None, None, :])
    y = np.zeros_like(x)
    tri = np.tril(np.ones((L, L), dtype=bool))
    for bi in range(b):
        G = C[bi] @ B[bi].T                                       # (t, s): C_t . B_s
        for h in range(H):
            cs = np.cumsum(dt[bi, :, h])
            seg = np.where(tri, cs[:, None] - cs[None, :], 0.0)
            M = G * np.exp(A[h] * seg) * dt[bi, :, h][None, :] * tri
            yy = M @ x[bi, :, h, :]
            if p.get("D") is not None:
                yy = yy + p["D"][h] * x[bi, :, h, :]
            if p.get("z") is not None:
                zz = p["z"][bi, :, h, :]
                yy = yy * zz / (1 + np.exp(-zz))
            y[bi, :, h, :] = yy
    return y


@pytest.mark.parametrize("gate,dskip", [(False, False), (True, True)])
def test_ssd_matches_semiseparable_matrix(gate, dskip):
    rng = _rng(41)
    p = _ssd_problem(rng, 2, 33, 3, 4, 5, gate, dskip)
    y, _ = oracle.ssd_scan_ref(**p)
    np.testing.assert_allclose(y, _brute_force_ssd(p), rtol=1e-11, atol=1e-12)


def test_ssd_equals_mamba1_with_a_tied_per_head():
    """A head of P channels with one scalar A and one delta per head is P Mamba-1 channels
    whose A rows are all A_h and whose deltas are equal."""
    rng = _rng(42)
    b, L, H, P, N = 2, 40, 3, 4, 6
    p = _ssd_problem(rng, b, L, H, P, N, gate=True, dskip=True)
    y, h_last = oracle.ssd_scan_ref(**p)
    m1 = dict(
        x=p["x"].reshape(b, L, H * P),
        delta=np.repeat(p["delta"], P, axis=2),
        A=np.repeat(p["A"], P)[:, None] * np.ones((1, N)),
        B=p["B"][:, :, 0], C=p["C"][:, :, 0],
        D=np.repeat(p["D"], P), z=p["z"].reshape(b, L, H * P),
        delta_bias=np.repeat(p["delta_bias"], P),
    )
    y1, h1 = oracle.ssm_scan_ref(**m1)
    np.testing.assert_allclose(y.reshape(b, L, H * P), y1, rtol=1e-12, atol=1e-13)
    # SSD state (b, H, N, P) vs Mamba-1 state (b, H*P, N)
    np.testing.assert_allclose(h_last.transpose(0, 1, 3, 2).reshape(b, H * P, N), h1, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 100])
def test_ssd_chunked_equals_recurrence(chunk):
    rng = _rng(43)
    p = _ssd_problem(rng, 1, 100, 2, 8, 16, gate=True, dskip=True)
    h0 = rng.standard_normal((1, 2, 16, 8))
    y, h_last = oracle.ssd_scan_ref(**p, h0=h0)
    yc, hc = oracle.ssd_chunked_ref(**p, chunk=chunk, h0=h0)
    np.testing.assert_allclose(yc, y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, h_last, rtol=1e-11, atol=1e-12)


def test_ssd_groups_map_heads_to_their_group():
    rng = _rng(44)
    b, L, H, P, N, G = 1, 20, 4, 3, 5, 2
    p = _ssd_problem(rng, b, L, H, P, N)
    p["B"] = rng.standard_normal((b, L, G, N))
    p["C"] = rng.standard_normal((b, L, G, N))
    y, h = oracle.ssd_scan_ref(**p)
    for g in range(G):
        q = dict(p)
        hs = slice(g * (H // G), (g + 1) * (H // G))
        q["x"], q["delta"], q["A"], q["delta_bias"] = p["x"][:, :, hs], p["delta"][:, :, hs], p["A"][hs], p["delta_bias"][hs]
        q["B"], q["C"] = p["B"][:, :, g:g + 1], p["C"][:, :, g:g + 1]
        yg, hg = oracle.ssd_scan_ref(**q)
        np.testing.assert_array_equal(yg, y[:, :, hs])
        np.testing.assert_array_equal(hg, h[:, hs])


# ---------------------------------------------------------------- planted mistakes are caught

def test_a_planted_index_slip_is_caught(monkeypatch):
    """Sanity of the pins themselves: an oracle that reads B one step late fails the
    semiseparable brute force."""
    rng = _rng(51)
    p = _problem(rng, 1, 20, 2, 3)
    bad = dict(p)
    bad["B"] = np.concatenate([p["B"][:, :1], p["B"][:, :-1]], axis=1)
    y_bad, _ = oracle.ssm_scan_ref(**bad)
    y_bf, _ = _brute_force_mamba1(p)
    assert np.max(np.abs(y_bad - y_bf)) > 1e-3


# ---------------------------------------------------------------- causal conv1d + SiLU prologue

def _conv_problem(rng, b, L, d, K, with_prev=False):
    x = rng.standard_normal((b, L, d))
    w = rng.standard_normal((d, K))
    bias = rng.standard_normal(d)
    prev = rng.standard_normal((b, K - 1, d)) if with_prev else None
    return x, w, bias, prev


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv1d_matches_the_pages_layer(K):
    """The pages' layer is a depthwise convolution with kernel d_conv, padding d_conv - 1 and
    the output cut to the first L steps, then SiLU: run exactly that through torch's conv1d
    (float64, CPU) and its SiLU."""
    import torch
    rng = _rng(70 + K)
    b, L, d = 2, 37, 5
    x, w, bias, _ = _conv_problem(rng, b, L, d, K)
    xt = torch.from_numpy(x).transpose(1, 2)                            # (b, d, L)
    ref = torch.nn.functional.conv1d(xt, torch.from_numpy(w)[:, None, :], torch.from_numpy(bias),
                                     padding=K - 1, groups=d)[:, :, :L]
    ref = torch.nn.functional.silu(ref).transpose(1, 2).numpy()
    np.testing.assert_allclose(oracle.causal_conv1d_ref(x, w, bias), ref, rtol=1e-13, atol=1e-13)


def test_conv1d_matches_numpy_convolve_per_channel():
    """Without SiLU each channel is numpy's full convolution with the reversed taps, cut to
    the first L outputs (causal: output t sees inputs t-K+1 .. t)."""
    rng = _rng(75)
    b, L, d, K = 2, 50, 3, 4
    x, w, bias, _ = _conv_problem(rng, b, L, d, K)
    y = oracle.causal_conv1d_ref(x, w, bias, apply_silu=False)
    for bi in range(b):
        for di in range(d):
            ref = np.convolve(x[bi, :, di], w[di, ::-1])[:L] + bias[di]
            np.testing.assert_allclose(y[bi, :, di], ref, rtol=1e-13, atol=1e-13)


def test_conv1d_identity_and_delay_taps():
    """Taps (0, 0, 0, 1) pass x through unchanged; taps (1, 0, 0, 0) delay it by three steps
    with zeros in front (the causal zero padding)."""
    rng = _rng(76)
    x = rng.standard_normal((1, 20, 2))
    ident = np.tile(np.array([0.0, 0.0, 0.0, 1.0]), (2, 1))
    np.testing.assert_array_equal(oracle.causal_conv1d_ref(x, ident, apply_silu=False), x)
    delay = np.tile(np.array([1.0, 0.0, 0.0, 0.0]), (2, 1))
    y = oracle.causal_conv1d_ref(x, delay, apply_silu=False)
    np.testing.assert_array_equal(y[:, :3], 0.0)
    np.testing.assert_array_equal(y[:, 3:], x[:, :-3])


def test_conv1d_previous_inputs_resume_a_split_sequence():
    """Convolving the second half with the last K-1 inputs of the first half as x_prev gives
    the second half of the convolution of the whole sequence."""
    rng = _rng(77)
    b, L, d, K = 2, 40, 3, 4
    x, w, bias, _ = _conv_problem(rng, b, L, d, K)
    whole = oracle.causal_conv1d_ref(x, w, bias)
    first = oracle.causal_conv1d_ref(x[:, :17], w, bias)
    second = oracle.causal_conv1d_ref(x[:, 17:], w, bias, x_prev=x[:, 17 - (K - 1):17])
    np.testing.assert_allclose(np.concatenate([first, second], axis=1), whole, rtol=0, atol=1e-14)


def test_silu_matches_the_logistic_function():
    """silu(v) = v * sigmoid(v) against scipy's logistic function, including large |v|."""
    from scipy.special import expit
    v = np.array([-800.0, -40.0, -3.5, -1e-8, 0.0, 1e-8, 0.7, 12.0, 800.0])
    np.testing.assert_allclose(oracle.silu(v), v * expit(v), rtol=1e-15, atol=0)


def test_a_planted_conv_tap_reversal_is_caught():
    """A convolution with its taps in the wrong order (x_t times weight[:, 0]) fails the
    numpy-convolve pin."""
    rng = _rng(78)
    x, w, bias, _ = _conv_problem(rng, 1, 30, 2, 4)
    bad = oracle.causal_conv1d_ref(x, w[:, ::-1], bias, apply_silu=False)
    ref = np.convolve(x[0, :, 0], w[0, ::-1])[:30] + bias[0]
    assert np.max(np.abs(bad[0, :, 0] - ref)) > 1e-3
