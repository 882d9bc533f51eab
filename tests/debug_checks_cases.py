"""Calls that reach every kernel of the library, for the debug-build check in
test_debug_checks_gpu.py: the TMA scan (split sequence with the state in place, reverse, the
conv1d prologue, exact ZOH), the generic and short-sequence scan kernels, the standalone conv1d,
and the SSD scan on the tensor-core and CUDA-core kernels.

run(dev) makes each call with a workspace of its own and returns the outputs and the status
word of each workspace. Run as a script (python tests/debug_checks_cases.py OUT) it saves them
to OUT with torch.save; the library loaded is the one SSMSCAN_LIBRARY names."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from selective_state_space_127_b300 import binding  # noqa: E402
from selective_state_space_127_b300.synth import make_scan_inputs, make_ssd_inputs  # noqa: E402


def _to(dev, inp):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def _misaligned(t):
    big = torch.empty(t.shape[:-1] + (t.shape[-1] + 1,), dtype=t.dtype, device=t.device)
    v = big[..., 1:]
    v.copy_(t)
    return v


def run(dev):
    out = {}

    def ws():
        return binding.new_workspace(64 << 20, dev)

    def scan(name, inp, **kw):
        w = ws()
        y, h = binding.ssm_scan_fwd(**inp, workspace=w, **kw)
        out[name + ".y"], out[name + ".h"] = y, h
        out[name + ".status"] = binding.check_status(w)

    g = torch.Generator().manual_seed(1)
    inp = _to(dev, make_scan_inputs(2, 700, 40, 16, "bf16", seed=71, d_skip="normal"))
    state = torch.randn(2, 40, 16, generator=g).to(dev)
    scan("split_in_place", inp, h0=state, h_last=state, chunk_len=64)
    h0a = torch.randn(2, 40, 32, generator=torch.Generator().manual_seed(2)).to(dev)
    scan("assoc_split", _to(dev, make_scan_inputs(2, 700, 40, 32, "bf16", seed=78)), h0=h0a, chunk_len=96,
         algorithm="assoc")
    scan("reverse_f32", _to(dev, make_scan_inputs(1, 300, 48, 32, "f32", seed=72)), reverse=True)
    cw, cb = (torch.randn(32, 4, generator=g) / 2).to(dev), (0.1 * torch.randn(32, generator=g)).to(dev)
    inp = _to(dev, make_scan_inputs(2, 200, 32, 16, "bf16", seed=73))
    prev = torch.randn(2, 3, 32, generator=g).to(torch.bfloat16).to(dev)
    scan("conv_prologue", inp, conv_weight=cw, conv_bias=cb, conv_x_prev=prev, chunk_len=96)
    scan("zoh_n64", _to(dev, make_scan_inputs(1, 130, 24, 64, "bf16", seed=74)), zoh=True)
    inp = _to(dev, make_scan_inputs(2, 90, 20, 17, "f32", seed=75))
    scan("generic", dict(inp, x=_misaligned(inp["x"])))
    inp = _to(dev, make_scan_inputs(3, 1, 48, 16, "bf16", seed=76, d_skip="normal"))
    state = torch.randn(3, 48, 16, generator=g).to(dev)
    scan("decode", inp, h0=state, h_last=state)

    x = torch.randn(2, 100, 64, generator=g).to(torch.bfloat16).to(dev)
    xp = torch.randn(2, 3, 64, generator=g).to(torch.bfloat16).to(dev)
    w64, b64 = (torch.randn(64, 4, generator=g) / 2).to(dev), (0.1 * torch.randn(64, generator=g)).to(dev)
    w = ws()
    out["conv1d.y"] = binding.causal_conv1d_fwd(x, w64, b64, x_prev=xp, workspace=w)
    out["conv1d.status"] = binding.check_status(w)

    for name, args in (("ssd_tc", (1, 300, 2, 64, 128, "bf16")), ("ssd_ref", (2, 70, 4, 32, 64, "f32"))):
        sinp = _to(dev, make_ssd_inputs(*args, seed=77, d_skip="normal", gate=name == "ssd_ref",
                                        ngroups=2 if name == "ssd_ref" else 1))
        h0 = torch.randn(args[0], args[2], args[4], args[3], generator=g).to(dev)
        w = ws()
        y, h = binding.ssd_chunk_scan_fwd(**sinp, chunk_size=128, h0=h0, workspace=w)
        out[name + ".y"], out[name + ".h"] = y, h
        out[name + ".status"] = binding.check_status(w)
    torch.cuda.synchronize()
    return out


if __name__ == "__main__":
    res = run(torch.device("cuda:0"))
    torch.save({k: (v.cpu() if torch.is_tensor(v) else v) for k, v in res.items()}, sys.argv[1])
    print("library:", binding.LIB_PATH)
