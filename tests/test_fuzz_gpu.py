"""Seeded random configurations of the selective scan (shapes, dtypes, both algorithms, strided
inputs and every optional feature together) against the fp64 oracle, so that combinations the
targeted tests do not name are exercised on whichever kernel the library picks for them."""
import random

import pytest
import torch

import oracle
from selective_state_space_127_b300 import binding, check_status, new_workspace, ssm_scan_fwd
from selective_state_space_127_b300.synth import make_scan_inputs
from conftest import rel_l2

pytestmark = pytest.mark.gpu

TOL_Y = {"f32": 1e-5, "bf16": 2e-2}
TOL_H = {"f32": 1e-5, "bf16": 1e-4}


def _config(i):
    r = random.Random(9000 + i)
    cfg = dict(
        b=r.choice([1, 2, 3]),
        L=r.choice([1, 2, 5, 17, 33, 64, 100, 257, 700]),
        D=r.choice([8, 16, 24, 40, 72]),
        N=r.choice([4, 8, 16, 32, 64]),
        dt=r.choice(["f32", "bf16"]),
        gate=r.random() < 0.5,
        dskip=r.random() < 0.5,
        softplus=r.random() < 0.8,
        h0=r.random() < 0.5,
        chunk=r.choice([0, 0, 0, 64, 96]),
    )
    variant = r.choice(["plain", "plain", "zoh", "reverse", "conv"])
    cfg["zoh"] = variant == "zoh"
    cfg["reverse"] = variant == "reverse"
    cfg["conv"] = r.choice([2, 3, 4]) if variant == "conv" else 0
    # drawn last, so the earlier fields of configuration i stay what they were
    cfg["algorithm"] = "assoc" if variant == "plain" and cfg["N"] in (16, 32) and r.random() < 0.3 else "serial"
    cfg["strided_x"] = cfg["algorithm"] == "serial" and r.random() < 0.2   # the generic kernel
    return cfg


@pytest.mark.parametrize("i", range(120))
def test_random_configuration_matches_oracle(cuda_dev, i):
    c = _config(i)
    inp = make_scan_inputs(c["b"], c["L"], c["D"], c["N"], c["dt"], seed=9100 + i,
                           d_skip="normal" if c["dskip"] else "none", gate=c["gate"])
    if not c["softplus"]:
        inp["delta"] = (inp["delta"].float().abs() * 0.05).to(inp["delta"].dtype)
        inp["delta_bias"] = torch.full_like(inp["delta_bias"], 1e-3)
    g = torch.Generator().manual_seed(9200 + i)
    h0 = torch.randn(c["b"], c["D"], c["N"], generator=g) if c["h0"] else None
    kw = dict(delta_softplus=c["softplus"], zoh=c["zoh"], reverse=c["reverse"], chunk_len=c["chunk"],
              algorithm=c["algorithm"])
    conv = {}
    x_ref = inp["x"]
    if c["conv"]:
        w = torch.randn(c["D"], c["conv"], generator=g) / c["conv"] ** 0.5
        cb = 0.1 * torch.randn(c["D"], generator=g)
        conv = dict(conv_weight=w.to(cuda_dev), conv_bias=cb.to(cuda_dev))
        x_ref = oracle.causal_conv1d_ref(inp["x"], w, cb)
    dev_inp = {k: (v.to(cuda_dev) if v is not None else None) for k, v in inp.items()}
    if c["strided_x"]:   # x as a view with a row stride of D + 3 elements
        x = dev_inp["x"]
        wide = torch.zeros(x.shape[0], x.shape[1], x.shape[2] + 3, dtype=x.dtype, device=cuda_dev)
        wide[..., :x.shape[2]] = x
        dev_inp["x"] = wide[..., :x.shape[2]]
    h0_d = h0.to(cuda_dev) if h0 is not None else None
    ws = new_workspace(binding.scan_workspace_size(**dev_inp, h0=h0_d, **kw, **conv), cuda_dev)
    y, h = ssm_scan_fwd(**dev_inp, h0=h0_d, workspace=ws, **kw, **conv)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssm_scan_ref(**dict(inp, x=x_ref), h0=h0, delta_softplus=c["softplus"], zoh=c["zoh"],
                                       reverse=c["reverse"])
    assert rel_l2(y.float().cpu().numpy(), y_ref) <= TOL_Y[c["dt"]], c
    assert rel_l2(h.cpu().numpy(), h_ref) <= TOL_H[c["dt"]], c
    assert check_status(ws) == binding.SSM_OK


def _ssd_config(i):
    r = random.Random(9500 + i)
    P, N = r.choice([(64, 128), (64, 128), (32, 64), (16, 32), (8, 16), (64, 64)])
    H = r.choice([1, 2, 4, 6])
    G = r.choice([g for g in (1, 2, 3) if H % g == 0])
    return dict(b=r.choice([1, 2]), L=r.choice([1, 7, 64, 128, 130, 300, 513]), H=H, P=P, N=N, G=G,
                Q=r.choice([16, 64, 128, 256]), dt=r.choice(["bf16", "bf16", "f32"]), gate=r.random() < 0.4,
                dskip=r.random() < 0.5, h0=r.random() < 0.5)


@pytest.mark.parametrize("i", range(24))
def test_random_ssd_configuration_matches_oracle(cuda_dev, i):
    from selective_state_space_127_b300 import ssd_chunk_scan_fwd
    from selective_state_space_127_b300.synth import make_ssd_inputs
    c = _ssd_config(i)
    inp = make_ssd_inputs(c["b"], c["L"], c["H"], c["P"], c["N"], c["dt"], seed=9600 + i,
                          d_skip="normal" if c["dskip"] else "none", gate=c["gate"], ngroups=c["G"])
    h0 = torch.randn(c["b"], c["H"], c["N"], c["P"], generator=torch.Generator().manual_seed(9700 + i)) if c["h0"] else None
    dev_inp = {k: (v.to(cuda_dev) if v is not None else None) for k, v in inp.items()}
    ws = new_workspace(binding.WORKSPACE_HEADER_BYTES, cuda_dev)
    y, h = ssd_chunk_scan_fwd(**dev_inp, chunk_size=c["Q"], h0=h0.to(cuda_dev) if h0 is not None else None,
                              workspace=ws)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssd_scan_ref(**inp, h0=h0)
    # the tensor-core kernel (bf16, P = 64, N = 128) carries bf16 operands: h within 5e-3
    tol_h = 5e-3 if c["dt"] == "bf16" else 1e-5
    assert rel_l2(y.float().cpu().numpy(), y_ref) <= TOL_Y[c["dt"]], c
    assert rel_l2(h.cpu().numpy(), h_ref) <= tol_h, c
    assert check_status(ws) == binding.SSM_OK
