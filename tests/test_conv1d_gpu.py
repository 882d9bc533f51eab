"""GPU parity of the causal conv1d + SiLU prologue: the standalone kernel and the scan with the
prologue fused (TMA path, chunked TMA path and generic path), against the fp64 oracle."""
import pytest
import torch

import oracle
from selective_state_space_127_b300 import binding, causal_conv1d_fwd, check_status, new_workspace, ssm_scan_fwd
from selective_state_space_127_b300.synth import make_scan_inputs
from conftest import rel_l2

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
TOL_H = {"f32": 1e-5, "bf16": 1e-4}
_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _conv_inputs(b, L, D, K, dt, seed, with_prev):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(b, L, D, generator=g).to(_DT[dt])
    w = torch.randn(D, K, generator=g) / K ** 0.5
    bias = 0.1 * torch.randn(D, generator=g)
    prev = torch.randn(b, K - 1, D, generator=g).to(_DT[dt]) if with_prev else None
    return x, w, bias, prev


CONV_CASES = [
    # b, L, D, K, dtype, silu, x_prev
    (1, 1, 8, 4, "bf16", True, False),
    (2, 3, 16, 4, "bf16", True, True),       # shorter than the window
    (2, 77, 40, 4, "bf16", True, True),      # ragged runs
    (3, 300, 1536, 4, "bf16", True, False),
    (1, 129, 24, 3, "f32", True, True),
    (2, 64, 64, 2, "f32", False, False),
    (1, 50, 12, 1, "f32", True, False),
    (2, 1000, 256, 4, "f32", False, True),
]


@pytest.mark.parametrize("b,L,D,K,dt,silu,with_prev", CONV_CASES)
def test_conv1d_matches_oracle(cuda_dev, b, L, D, K, dt, silu, with_prev):
    x, w, bias, prev = _conv_inputs(b, L, D, K, dt, 500 + L + D + K, with_prev)
    y = causal_conv1d_fwd(x.to(cuda_dev), w.to(cuda_dev), bias.to(cuda_dev), silu=silu,
                          x_prev=prev.to(cuda_dev) if prev is not None else None)
    torch.cuda.synchronize()
    ref = oracle.causal_conv1d_ref(x, w, bias, apply_silu=silu, x_prev=prev)
    assert rel_l2(y.float().cpu().numpy(), ref) <= TOL[dt]


def test_conv1d_split_sequence_resumes_through_x_prev(cuda_dev):
    x, w, bias, _ = _conv_inputs(2, 200, 32, 4, "f32", 77, False)
    xd, wd, bd = x.to(cuda_dev), w.to(cuda_dev), bias.to(cuda_dev)
    whole = causal_conv1d_fwd(xd, wd, bd)
    first = causal_conv1d_fwd(xd[:, :90].contiguous(), wd, bd)
    second = causal_conv1d_fwd(xd[:, 90:].contiguous(), wd, bd, x_prev=xd[:, 87:90].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([first, second], dim=1), whole)


def _fused_case(b, L, D, N, dt, K, seed, with_prev, gate=True, dskip=True):
    inp = make_scan_inputs(b, L, D, N, dt, seed=seed, d_skip="normal" if dskip else "none", gate=gate)
    _, w, cb, prev = _conv_inputs(b, L, D, K, dt, seed + 1, with_prev)
    return inp, w, cb, prev


def _fused_ref(inp, w, cb, prev, h0=None):
    u = oracle.causal_conv1d_ref(inp["x"], w, cb, x_prev=prev)
    return oracle.ssm_scan_ref(**dict(inp, x=u), h0=h0)


def _to(dev, inp):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def _misaligned_copy(t):
    big = torch.empty(t.shape[:-1] + (t.shape[-1] + 1,), dtype=t.dtype, device=t.device)
    v = big[..., 1:]
    v.copy_(t)
    return v


FUSED_CASES = [
    # b, L, D, N, dtype, K, x_prev, chunk_len
    (2, 77, 40, 16, "bf16", 4, True, 0),
    (1, 300, 48, 16, "bf16", 4, False, 0),
    (3, 129, 24, 32, "bf16", 2, True, 0),
    (1, 70, 32, 64, "f32", 4, True, 0),
    (2, 64, 16, 16, "f32", 3, False, 0),
    (1, 2100, 32, 16, "bf16", 4, True, 512),   # chunked: the halo of a chunk is the previous chunk's tail
    (2, 1000, 16, 16, "f32", 4, False, 256),
]


@pytest.mark.parametrize("b,L,D,N,dt,K,with_prev,chunk", FUSED_CASES)
def test_fused_prologue_matches_oracle_on_both_paths(cuda_dev, b, L, D, N, dt, K, with_prev, chunk):
    inp, w, cb, prev = _fused_case(b, L, D, N, dt, K, 6000 + L + D + N + K, with_prev)
    g = _to(cuda_dev, inp)
    cw = dict(conv_weight=w.to(cuda_dev), conv_bias=cb.to(cuda_dev),
              conv_x_prev=prev.to(cuda_dev) if prev is not None else None)
    ws = new_workspace(binding.scan_workspace_size(**g, chunk_len=chunk, **cw), cuda_dev)
    y_fast, h_fast = ssm_scan_fwd(**g, chunk_len=chunk, workspace=ws, **cw)
    y_gen, h_gen = ssm_scan_fwd(**dict(g, x=_misaligned_copy(g["x"])), **cw)
    torch.cuda.synchronize()
    y_ref, h_ref = _fused_ref(inp, w, cb, prev)
    assert rel_l2(y_fast.float().cpu().numpy(), y_ref) <= TOL[dt]
    assert rel_l2(h_fast.cpu().numpy(), h_ref) <= TOL_H[dt]
    assert rel_l2(y_gen.float().cpu().numpy(), y_ref) <= TOL[dt]
    assert rel_l2(h_gen.cpu().numpy(), h_ref) <= TOL_H[dt]
    assert check_status(ws) == binding.SSM_OK


def test_fused_prologue_split_and_resume(cuda_dev):
    """Two calls (the second with h0 = the first's h_last and conv_x_prev = the first's last
    three raw inputs) give the output of one call."""
    inp, w, cb, _ = _fused_case(2, 640, 32, 16, "bf16", 4, 6100, False)
    g = _to(cuda_dev, inp)
    cw = dict(conv_weight=w.to(cuda_dev), conv_bias=cb.to(cuda_dev))
    y_all, h_all = ssm_scan_fwd(**g, **cw)
    cut = 257
    first = {k: (v[:, :cut] if k in ("x", "delta", "z", "B", "C") else v) for k, v in g.items()}
    second = {k: (v[:, cut:] if k in ("x", "delta", "z", "B", "C") else v) for k, v in g.items()}
    y1, h1 = ssm_scan_fwd(**first, **cw)
    y2, h2 = ssm_scan_fwd(**second, h0=h1, conv_x_prev=g["x"][:, cut - 3:cut].contiguous(), **cw)
    torch.cuda.synchronize()
    y_split = torch.cat([y1, y2], dim=1).float().cpu().numpy()
    assert rel_l2(y_split, y_all.float().cpu().numpy()) <= 1e-2
    assert rel_l2(h2.cpu().numpy(), h_all.cpu().numpy()) <= 1e-5


def test_fused_prologue_decode_step_advances_conv_window(cuda_dev):
    """Single-token steps (the generic kernel) with h0 == h_last in place and the last three
    raw inputs as conv_x_prev reproduce the full-sequence output."""
    inp, w, cb, _ = _fused_case(2, 12, 16, 16, "f32", 4, 6200, False)
    g = _to(cuda_dev, inp)
    cw = dict(conv_weight=w.to(cuda_dev), conv_bias=cb.to(cuda_dev))
    y_all, h_all = ssm_scan_fwd(**g, **cw)
    h = torch.zeros(2, 16, 16, device=cuda_dev)
    xp = torch.zeros(2, 3, 16, device=cuda_dev)
    ys = []
    for t in range(12):
        step = {k: (v[:, t:t + 1] if k in ("x", "delta", "z", "B", "C") else v) for k, v in g.items()}
        y, _ = ssm_scan_fwd(**step, h0=h, h_last=h, conv_x_prev=xp, **cw)
        ys.append(y)
        xp = torch.cat([xp[:, 1:], g["x"][:, t:t + 1]], dim=1).contiguous()
    torch.cuda.synchronize()
    assert rel_l2(torch.cat(ys, dim=1).cpu().numpy(), y_all.cpu().numpy()) <= 1e-6
    assert rel_l2(h.cpu().numpy(), h_all.cpu().numpy()) <= 1e-6


def test_fused_prologue_at_workload_size_sampled(cuda_dev):
    """b8 D1536 L2048 N16 bf16 with the prologue (the launch configuration the benchmark
    times): eight channels checked against the oracle over the whole sequence."""
    inp, w, cb, _ = _fused_case(8, 2048, 1536, 16, "bf16", 4, 6300, False)
    g = _to(cuda_dev, inp)
    y, h = ssm_scan_fwd(**g, conv_weight=w.to(cuda_dev), conv_bias=cb.to(cuda_dev))
    torch.cuda.synchronize()
    idx = torch.arange(0, 1536, 192)
    sub = {k: (v.index_select(2, idx) if k in ("x", "delta", "z") else v) for k, v in inp.items()}
    for k in ("D", "delta_bias"):
        sub[k] = inp[k].index_select(0, idx)
    sub["A"] = inp["A"].index_select(0, idx)
    y_ref, h_ref = _fused_ref(sub, w.index_select(0, idx), cb.index_select(0, idx), None)
    assert rel_l2(y.index_select(2, idx.to(cuda_dev)).float().cpu().numpy(), y_ref) <= TOL["bf16"]
    assert rel_l2(h.index_select(1, idx.to(cuda_dev)).cpu().numpy(), h_ref) <= TOL_H["bf16"]


def test_fused_prologue_with_exact_zoh_and_h0(cuda_dev):
    """The conv prologue together with the exact-ZOH discretisation and an initial state (the
    generic kernel takes this combination) against the oracle."""
    inp, w, cb, prev = _fused_case(2, 150, 24, 16, "f32", 4, 6400, True)
    h0 = torch.randn(2, 24, 16, generator=torch.Generator().manual_seed(64))
    g = _to(cuda_dev, inp)
    y, h = ssm_scan_fwd(**g, h0=h0.to(cuda_dev), zoh=True, conv_weight=w.to(cuda_dev), conv_bias=cb.to(cuda_dev),
                        conv_x_prev=prev.to(cuda_dev))
    torch.cuda.synchronize()
    u = oracle.causal_conv1d_ref(inp["x"], w, cb, x_prev=prev)
    y_ref, h_ref = oracle.ssm_scan_ref(**dict(inp, x=u), h0=h0, zoh=True)
    assert rel_l2(y.cpu().numpy(), y_ref) <= TOL["f32"]
    assert rel_l2(h.cpu().numpy(), h_ref) <= TOL_H["f32"]
