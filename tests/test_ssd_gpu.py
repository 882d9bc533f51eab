"""GPU parity of the SSD chunked scan (through the C ABI) against the fp64 oracle.

Shapes with bf16 I/O, P = 64, N = 128 and a chunk that is a multiple of 128 take the
tensor-core kernel; the others take the CUDA-core recurrence kernel.

Tolerances: rel-L2 <= 1e-5 for fp32 I/O and <= 2e-2 for bf16 I/O on y. The final state is
fp32; on the tensor-core path the MMA operands w*x (the decayed inputs of the state update)
and the carried state (operand of C S) are rounded to bf16, a relative error of at most 2^-9
per element that averages to about 1e-3 over the 128-term products, so h_last is held to
5e-3 for bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_127_b300 import ssd_chunk_scan_fwd
from selective_state_space_127_b300.synth import SSD_WORKLOAD, make_ssd_inputs, ssd_workload_inputs
from conftest import rel_l2

pytestmark = pytest.mark.gpu

TOL_Y = {"f32": 1e-5, "bf16": 2e-2}
TOL_H = {"f32": 1e-5, "bf16": 5e-3}


def _to(dev, inp):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def _misaligned_copy(t):
    """Same values in a view whose base is off the 16-byte grid (the tensor-core kernel
    refuses it, so the CUDA-core kernel runs)."""
    big = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    v = big[1:].view(t.shape)
    v.copy_(t)
    return v


CASES = [
    # b, L, H, P, N, G, Q, dtype, gate, dskip
    (1, 1, 1, 1, 1, 1, 1, "f32", False, False),
    (2, 37, 3, 8, 16, 1, 16, "f32", True, True),
    (1, 300, 4, 64, 128, 1, 256, "bf16", False, False),
    (2, 100, 4, 32, 64, 2, 64, "bf16", True, True),
    (1, 513, 2, 64, 128, 1, 256, "bf16", False, False),
    (1, 64, 2, 16, 32, 1, 32, "f32", False, True),
]


@pytest.mark.parametrize("b,L,H,P,N,G,Q,dt,gate,dskip", CASES)
def test_random_shapes_match_oracle(cuda_dev, b, L, H, P, N, G, Q, dt, gate, dskip):
    inp = make_ssd_inputs(b, L, H, P, N, dt, seed=500 + L + H + P + N, d_skip="normal" if dskip else "none",
                          gate=gate, ngroups=G)
    y, h = ssd_chunk_scan_fwd(**_to(cuda_dev, inp), chunk_size=Q)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssd_scan_ref(**inp)
    assert rel_l2(y.float().cpu().numpy(), y_ref) <= TOL_Y[dt]
    assert rel_l2(h.cpu().numpy(), h_ref) <= TOL_H[dt]


def test_h0_and_chunk_size_invariance(cuda_dev):
    inp = make_ssd_inputs(1, 200, 2, 64, 128, "bf16", seed=77)
    h0 = torch.randn(1, 2, 128, 64, generator=torch.Generator().manual_seed(1))
    g = _to(cuda_dev, inp)
    outs = []
    for Q in (32, 64, 128, 256):
        y, h = ssd_chunk_scan_fwd(**g, chunk_size=Q, h0=h0.to(cuda_dev))
        outs.append((y.float().cpu().numpy(), h.cpu().numpy()))
    y_ref, h_ref = oracle.ssd_scan_ref(**inp, h0=h0)
    for y, h in outs:
        assert rel_l2(y, y_ref) <= TOL_Y["bf16"]
        assert rel_l2(h, h_ref) <= TOL_H["bf16"]
        assert rel_l2(y, outs[0][0]) <= 1e-2


def test_full_size_workload_whole_tensors(cuda_dev):
    """Every element of y and h_last of the full-size SSD workload against the oracle, a slice
    of heads at a time: rel-L2 over the whole tensors and an element-wise bound, so an error
    confined to one head, one batch row or one block fails.

    The bound is the usual one for sums of rounded products: the tensor-core path rounds the
    MMA operands (the masked decayed C B^T block, w*x, the carried state) to bf16, a relative
    error of at most 2^-9 per term, so |y - y_ref| <= 2^-6 y_abs + 2^-8 |y_ref| (terms plus the
    final rounding of y to bf16) and |h - h_ref| <= 2^-6 h_abs, where y_abs and h_abs are the
    oracle run on |x|, |B|, |C|: the sums of the terms' magnitudes."""
    w = SSD_WORKLOAD
    inp = ssd_workload_inputs(device=cuda_dev)
    y, h = ssd_chunk_scan_fwd(**inp, chunk_size=w.chunk)
    torch.cuda.synchronize()
    ny = dy = nh = dh = 0.0
    excess_y = excess_h = -np.inf
    for h0 in range(0, w.nheads, 16):
        h1 = min(w.nheads, h0 + 16)
        sub = dict(inp)
        sub["x"] = inp["x"][:, :, h0:h1]
        sub["delta"] = inp["delta"][:, :, h0:h1]
        sub["A"] = inp["A"][h0:h1]
        sub["delta_bias"] = inp["delta_bias"][h0:h1]
        host = {k: (v.cpu() if v is not None else None) for k, v in sub.items()}
        y_ref, h_ref = oracle.ssd_scan_ref(**host)
        y_abs, h_abs = oracle.ssd_scan_ref(**dict(host, x=host["x"].abs(), B=host["B"].abs(), C=host["C"].abs()))
        y_s = y[:, :, h0:h1].float().cpu().numpy().astype(np.float64)
        h_s = h[:, h0:h1].cpu().numpy().astype(np.float64)
        excess_y = max(excess_y, float((np.abs(y_s - y_ref) - (2.0 ** -6 * y_abs + 2.0 ** -8 * np.abs(y_ref))).max()))
        excess_h = max(excess_h, float((np.abs(h_s - h_ref) - 2.0 ** -6 * h_abs).max()))
        ny += float(((y_s - y_ref) ** 2).sum())
        dy += float((y_ref ** 2).sum())
        nh += float(((h_s - h_ref) ** 2).sum())
        dh += float((h_ref ** 2).sum())
    ey, eh = np.sqrt(ny / dy), np.sqrt(nh / dh)
    print(f"SSD workload: rel-L2 y {ey:.3e} h_last {eh:.3e}; element excess y {excess_y:.2e} h {excess_h:.2e}")
    assert ey <= TOL_Y["bf16"]
    assert eh <= TOL_H["bf16"]
    assert excess_y <= 0.0 and excess_h <= 0.0


TC_CASES = [
    # b, L, H, P, N, G, Q, gate, dskip, h0
    (1, 128, 2, 64, 128, 1, 128, False, False, False),
    (2, 333, 4, 64, 128, 2, 128, True, True, True),     # ragged last block, 2 groups, D, z, h0
    (1, 77, 3, 64, 128, 1, 256, False, True, False),    # shorter than one block
    (2, 1000, 2, 64, 128, 1, 256, False, False, True),
]


@pytest.mark.parametrize("b,L,H,P,N,G,Q,gate,dskip,with_h0", TC_CASES)
def test_tensor_core_path_matches_oracle_and_cuda_core_path(cuda_dev, b, L, H, P, N, G, Q, gate, dskip, with_h0):
    inp = make_ssd_inputs(b, L, H, P, N, "bf16", seed=900 + L + H + G, d_skip="normal" if dskip else "none",
                          gate=gate, ngroups=G)
    h0 = torch.randn(b, H, N, P, generator=torch.Generator().manual_seed(L)) if with_h0 else None
    g = _to(cuda_dev, inp)
    h0_d = h0.to(cuda_dev) if h0 is not None else None
    y_tc, h_tc = ssd_chunk_scan_fwd(**g, chunk_size=Q, h0=h0_d)
    y_cc, h_cc = ssd_chunk_scan_fwd(**dict(g, x=_misaligned_copy(g["x"])), chunk_size=64, h0=h0_d)  # CUDA cores
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssd_scan_ref(**inp, h0=h0)
    assert rel_l2(y_tc.float().cpu().numpy(), y_ref) <= TOL_Y["bf16"]
    assert rel_l2(h_tc.cpu().numpy(), h_ref) <= TOL_H["bf16"]
    assert rel_l2(y_cc.float().cpu().numpy(), y_ref) <= TOL_Y["bf16"]
    assert rel_l2(h_cc.cpu().numpy(), h_ref) <= 1e-4
    assert rel_l2(y_tc.float().cpu().numpy(), y_cc.float().cpu().numpy()) <= TOL_Y["bf16"]


def test_tensor_core_path_empty_sequence_copies_h0(cuda_dev):
    inp = make_ssd_inputs(1, 0, 2, 64, 128, "bf16", seed=5)
    g = _to(cuda_dev, inp)
    h0 = torch.randn(1, 2, 128, 64, device=cuda_dev)
    y, h = ssd_chunk_scan_fwd(**g, chunk_size=256, h0=h0)
    torch.cuda.synchronize()
    assert y.shape == (1, 0, 2, 64) and torch.equal(h, h0)
