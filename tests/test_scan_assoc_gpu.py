"""GPU parity of the in-tile associative scan (algorithm="assoc") against the fp64 oracle and
against the default serial walk, through the C ABI.

The two algorithms compute the same recurrence in a different order of fp32 operations, so they
agree to rounding, not bit for bit; both are held to the oracle with the tolerances of the
serial path's tests (rel-L2 <= 1e-5 for fp32 I/O, <= 2e-2 for y and 1e-4 for h_last with bf16
I/O).
"""
import pytest
import torch

import oracle
from selective_state_space_127_b300 import binding, check_status, new_workspace, ssm_scan_fwd
from selective_state_space_127_b300.synth import make_scan_inputs
from conftest import rel_l2

pytestmark = pytest.mark.gpu

TOL_Y = {"f32": 1e-5, "bf16": 2e-2}
TOL_H = {"f32": 1e-5, "bf16": 1e-4}

# b, L, D, N, dtype, gate, d_skip, softplus, chunk_len, with h0
CASES = [
    (2, 300, 40, 16, "f32", True, "normal", True, 0, False),     # ragged L and channel tile
    (1, 1000, 32, 32, "bf16", True, "ones", True, 96, True),     # N = 32, chunks + carry, h0
    (3, 257, 64, 16, "bf16", False, "none", False, 0, False),    # no gate, no skip, raw dt
    (1, 2048, 16, 16, "f32", True, "normal", True, 256, True),   # chunks in fp32
    (2, 3, 16, 16, "bf16", True, "normal", True, 0, True),       # shorter than one tile
]


def _to(dev, inp):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


@pytest.mark.parametrize("b,L,D,N,dt,gate,dskip,sp,q,with_h0", CASES)
def test_assoc_scan_matches_oracle_and_serial_walk(cuda_dev, b, L, D, N, dt, gate, dskip, sp, q, with_h0):
    inp = make_scan_inputs(b, L, D, N, dt, seed=9100 + L + D + N, d_skip=dskip, gate=gate)
    if not sp:   # raw dt is used as given: positive steps (delta + bias would be negative here)
        inp = dict(inp, delta=(inp["delta"].float().abs() * 0.05).to(inp["delta"].dtype), delta_bias=None)
    h0 = torch.randn(b, D, N, generator=torch.Generator().manual_seed(L + 7)) if with_h0 else None
    g = _to(cuda_dev, inp)
    h0_d = h0.to(cuda_dev) if h0 is not None else None
    kw = dict(delta_softplus=sp, h0=h0_d, chunk_len=q)
    ws = new_workspace(binding.scan_workspace_size(**g, algorithm="assoc", **kw), cuda_dev)
    y_a, h_a = ssm_scan_fwd(**g, workspace=ws, algorithm="assoc", **kw)
    y_s, h_s = ssm_scan_fwd(**g, **kw)
    torch.cuda.synchronize()
    assert check_status(ws) == binding.SSM_OK
    y_ref, h_ref = oracle.ssm_scan_ref(**inp, h0=h0, delta_softplus=sp)
    assert rel_l2(y_a.float().cpu().numpy(), y_ref) <= TOL_Y[dt]
    assert rel_l2(h_a.cpu().numpy(), h_ref) <= TOL_H[dt]
    # against the serial walk: the same inputs, the same rounding of y to the I/O dtype
    assert rel_l2(h_a.cpu().numpy(), h_s.cpu().numpy()) <= 1e-5
    assert rel_l2(y_a.float().cpu().numpy(), y_s.float().cpu().numpy()) <= (1e-5 if dt == "f32" else 4e-3)


def test_assoc_scan_refuses_what_it_does_not_take(cuda_dev):
    inp = _to(cuda_dev, make_scan_inputs(1, 64, 16, 16, "bf16", seed=9200))
    for kw in (dict(reverse=True), dict(zoh=True)):
        with pytest.raises(binding.SSMError) as e:
            ssm_scan_fwd(**inp, algorithm="assoc", **kw)
        assert e.value.status == binding.SSM_ERR_UNSUPPORTED
    # a strided (non-TMA) layout
    x = inp["x"]
    wide = torch.zeros(x.shape[0], x.shape[1], x.shape[2] + 3, dtype=x.dtype, device=cuda_dev)
    wide[..., :x.shape[2]] = x
    with pytest.raises(binding.SSMError) as e:
        ssm_scan_fwd(**dict(inp, x=wide[..., :x.shape[2]]), algorithm="assoc")
    assert e.value.status == binding.SSM_ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        ssm_scan_fwd(**inp, algorithm="blelloch")
