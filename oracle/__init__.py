"""Test infrastructure: the fp64 CPU oracle for the selective scan and the SSD scan.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use
this package. It shares no code with the CUDA library: the recurrences live in
``ssm_oracle.c`` (plain C, double precision, sequential in time) and the chunked SSD
form below is plain numpy. Inputs may be numpy arrays or torch tensors in any dtype; they
are widened to float64 exactly as stored (a bf16 input is read as its bf16 value).

Functions
---------
ssm_scan_ref     Mamba selective scan: softplus(delta + bias), A_bar = exp(delta*A),
                 B_bar x = delta*B*x (or exact ZOH), h_t = A_bar h_{t-1} + B_bar x_t,
                 y_t = C_t.h_t + D x_t, times silu(z_t).
                 Pages: "Mamba/SSM complete guide" section 5 listing ``selective_scan``;
                 "論文解説: Mamba" (0h-n0) "選択機構" and "Hardware-Aware Parallel Scan";
                 "State Space Model / Mamba" (disassemble-channel) "Zero-Order Hold".
ssd_scan_ref     Mamba-2 recurrence with a scalar A per head, sequential.
                 Pages: "Mamba-2 / SSD" (abeam) "基本アイデア"; "Mamba/SSM complete
                 guide" section 6 "SSD演算の概念".
causal_conv1d_ref  Causal depthwise conv1d over time (kernel K, left zero padding or the
                 K-1 previous inputs), then SiLU: the prologue of the Mamba block's x branch.
                 Pages: "Mamba/SSM complete guide" section 5 `MambaBlock` (nn.Conv1d with
                 groups = d_inner, kernel d_conv, padding d_conv - 1, output cut to the first
                 L steps, then F.silu); "論文解説: Mamba" "Mambaブロックの全体構成"
                 (convolution with d_conv = 4, then SiLU).
ssd_chunked_ref  The same SSD output through the chunked block decomposition (diagonal
                 blocks by matrix products, chunk-to-chunk hand-off through the state).
                 Pages: "Mamba-2 / SSD" (abeam) "基本アイデア" (diagonal blocks as ordinary
                 block products, off-diagonal blocks as a low-rank state hand-off);
                 "Mamba/SSM complete guide" section 6 (intra-chunk matrix products,
                 inter-chunk state recurrence).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into oracle/liboracle.so with gcc (-O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fno-fast-math", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.oracle_ssm_scan_f64.argtypes = [i64, i64, i64, i64] + [dp] * 8 + [ci, dp, ci, ci, dp, dp, ci]
            lib.oracle_ssm_scan_f64.restype = ci
            lib.oracle_ssd_scan_f64.argtypes = [i64] * 6 + [dp] * 8 + [ci, dp, dp, dp, ci]
            lib.oracle_ssd_scan_f64.restype = ci
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle uses by default (OpenMP's count for this process)."""
    return int(_load().oracle_max_threads())


def f64(a):
    """Widen an array or tensor to a C-contiguous float64 numpy array (None passes through)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen in torch (numpy has no bf16), then hand over
        a = a.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def ssm_scan_ref(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 h0=None, zoh=False, reverse=False, nthreads=None):
    """fp64 selective scan. Shapes: x, delta, z (b, L, d); A (d, n); B, C (b, L, n);
    D, delta_bias (d); h0 (b, d, n). Returns (y (b, L, d), h_last (b, d, n)) as float64."""
    x, delta, A, B, C = f64(x), f64(delta), f64(A), f64(B), f64(C)
    D, z, delta_bias, h0 = f64(D), f64(z), f64(delta_bias), f64(h0)
    b, L, d = x.shape
    n = A.shape[1]
    assert delta.shape == (b, L, d) and A.shape == (d, n)
    assert B.shape == (b, L, n) and C.shape == (b, L, n)
    assert z is None or z.shape == (b, L, d)
    assert D is None or D.shape == (d,)
    assert delta_bias is None or delta_bias.shape == (d,)
    assert h0 is None or h0.shape == (b, d, n)
    y = np.zeros((b, L, d))
    h_last = np.zeros((b, d, n))
    rc = _load().oracle_ssm_scan_f64(b, L, d, n, _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                     _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
                                     _ptr(h0), int(bool(zoh)), int(bool(reverse)),
                                     _ptr(y), _ptr(h_last), int(nthreads or max_threads()))
    if rc != 0:
        raise ValueError(f"oracle_ssm_scan_f64 failed ({rc})")
    return y, h_last


def ssd_scan_ref(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 h0=None, nthreads=None):
    """fp64 SSD recurrence. Shapes: x, z (b, L, H, P); delta (b, L, H); A, D, delta_bias (H);
    B, C (b, L, G, N) or (b, L, N) for one group; h0 (b, H, N, P).
    Returns (y (b, L, H, P), h_last (b, H, N, P)) as float64."""
    x, delta, A, B, C = f64(x), f64(delta), f64(A), f64(B), f64(C)
    D, z, delta_bias, h0 = f64(D), f64(z), f64(delta_bias), f64(h0)
    if B.ndim == 3:
        B, C = B[:, :, None, :].copy(), C[:, :, None, :].copy()
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert delta.shape == (b, L, H) and A.shape == (H,)
    assert B.shape == (b, L, G, N) and C.shape == (b, L, G, N)
    y = np.zeros((b, L, H, P))
    h_last = np.zeros((b, H, N, P))
    rc = _load().oracle_ssd_scan_f64(b, L, H, P, N, G, _ptr(x), _ptr(delta), _ptr(A), _ptr(B),
                                     _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                                     int(bool(delta_softplus)), _ptr(h0), _ptr(y), _ptr(h_last),
                                     int(nthreads or max_threads()))
    if rc != 0:
        raise ValueError(f"oracle_ssd_scan_f64 failed ({rc})")
    return y, h_last


def softplus(v):
    """log(1 + e^v) in float64, as max(v, 0) + log1p(e^-|v|)."""
    v = np.asarray(v, dtype=np.float64)
    return np.maximum(v, 0.0) + np.log1p(np.exp(-np.abs(v)))


def silu(v):
    """v * sigmoid(v) = v / (1 + e^-v) in float64 (written to avoid overflow of e^-v)."""
    v = np.asarray(v, dtype=np.float64)
    e = np.exp(-np.abs(v))
    return np.where(v >= 0, v / (1.0 + e), v * e / (1.0 + e))


def causal_conv1d_ref(x, weight, bias=None, apply_silu=True, x_prev=None):
    """fp64 causal depthwise convolution along t, then SiLU.

    x (b, L, d); weight (d, K); bias (d) or None; x_prev (b, K-1, d): the K-1 inputs that
    precede x[:, 0] (zeros when None, which is the zero padding of d_conv - 1 steps on the
    left). With xp = x_prev followed by x along t,
        y[b, t, d] = bias[d] + sum_{k=0}^{K-1} weight[d, k] * xp[b, t + k, d],
    so weight[:, K-1] multiplies x_t and weight[:, 0] multiplies x_{t-K+1} (a convolution
    layer's cross-correlation, kept to the first L outputs). Then y = silu(y) if apply_silu.
    Returns y (b, L, d) as float64."""
    x, weight, bias, x_prev = f64(x), f64(weight), f64(bias), f64(x_prev)
    b, L, d = x.shape
    K = weight.shape[1]
    assert weight.shape == (d, K) and K >= 1
    assert bias is None or bias.shape == (d,)
    if x_prev is None:
        x_prev = np.zeros((b, K - 1, d))
    assert x_prev.shape == (b, K - 1, d)
    xp = np.concatenate([x_prev, x], axis=1)          # (b, K - 1 + L, d)
    y = np.zeros((b, L, d)) if bias is None else np.broadcast_to(bias, (b, L, d)).copy()
    for k in range(K):
        y += weight[:, k] * xp[:, k:k + L, :]
    return silu(y) if apply_silu else y


def ssd_chunked_ref(x, delta, A, B, C, chunk, D=None, z=None, delta_bias=None,
                    delta_softplus=True, h0=None):
    """fp64 SSD output through the chunked block decomposition, in the order:
    1. dt = softplus(delta + bias); a_t = dt * A_h; cum = inclusive cumulative sum of a
       inside each chunk.
    2. G = C_c B_c^T over the state dimension (one per chunk and group).
    3. M[i, j] = G[i, j] * exp(cum_i - cum_j) * dt_j for j <= i, 0 above the diagonal.
    4. Y_diag = M X_c.
    5. Y_off[i] = exp(cum_i) * C_i S_prev (the state handed over from earlier chunks).
    6. S = exp(cum_last) S_prev + sum_j exp(cum_last - cum_j) dt_j B_j^T x_j.
    7. y = Y_diag + Y_off (+ D x) (* silu z).
    Shapes as in ssd_scan_ref. The last chunk may be shorter than ``chunk``."""
    x, delta, A, B, C = f64(x), f64(delta), f64(A), f64(B), f64(C)
    D, z, delta_bias, h0 = f64(D), f64(z), f64(delta_bias), f64(h0)
    if B.ndim == 3:
        B, C = B[:, :, None, :], C[:, :, None, :]
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    dt = delta + (delta_bias[None, None, :] if delta_bias is not None else 0.0)
    if delta_softplus:
        dt = softplus(dt)
    y = np.zeros((b, L, H, P))
    h_last = np.zeros((b, H, N, P))
    for bi in range(b):
        for h in range(H):
            g = h // hpg
            S = h0[bi, h].copy() if h0 is not None else np.zeros((N, P))
            for c0 in range(0, L, chunk):
                c1 = min(c0 + chunk, L)
                Xc, Bc, Cc = x[bi, c0:c1, h, :], B[bi, c0:c1, g, :], C[bi, c0:c1, g, :]
                dtc = dt[bi, c0:c1, h]
                cum = np.cumsum(dtc * A[h])
                Gm = Cc @ Bc.T
                seg = cum[:, None] - cum[None, :]
                causal = np.tril(np.ones((c1 - c0, c1 - c0), dtype=bool))
                M = np.where(causal, Gm * np.exp(np.where(causal, seg, 0.0)) * dtc[None, :], 0.0)
                Ydiag = M @ Xc
                Yoff = np.exp(cum)[:, None] * (Cc @ S)
                w = np.exp(cum[-1] - cum) * dtc
                S = np.exp(cum[-1]) * S + (Bc * w[:, None]).T @ Xc
                y[bi, c0:c1, h, :] = Ydiag + Yoff
            h_last[bi, h] = S
    if D is not None:
        y = y + D[None, None, :, None] * x
    if z is not None:
        y = y * (z / (1.0 + np.exp(-z)))
    return y, h_last
