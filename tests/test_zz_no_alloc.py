"""The allocation-free scan entry point, ssm_scan_fwd_noalloc, called through the C ABI.

It serves callers that cannot allocate device memory or pass a workspace: its chunk-carry
scratch lives in a fixed buffer inside the library. Here it must reproduce the workspace
entry point's results on a long sequence that is split into chunks (so the scratch is used),
on two calls in a row (the buffer keeps the previous call's contents), and it must refuse a
call whose scratch need exceeds the buffer before launching anything.

This file sorts last so that a stop-at-first-failure run has run every other test first.
"""
import pytest
import torch

from selective_state_space_127_b300 import binding, ssm_scan_fwd
from selective_state_space_127_b300.synth import make_scan_inputs
from conftest import rel_l2

pytestmark = pytest.mark.gpu

TOL_Y_BF16 = 2e-2      # the bf16 I/O tolerance of the scan tests
TOL_H = 1e-4           # fp32 final state with bf16 inputs


def _to(dev, inp):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_dev):
    inp = _to(cuda_dev, make_scan_inputs(2, 3000, 48, 16, "bf16", seed=777, d_skip="normal"))
    q = 256
    need = binding.scan_workspace_size(**inp, chunk_len=q)
    assert 0 < need <= binding.NOALLOC_SCRATCH_BYTES
    y_ws, h_ws = ssm_scan_fwd(**inp, chunk_len=q)
    torch.cuda.synchronize()
    y_out = torch.empty_like(y_ws)
    h_out = torch.empty_like(h_ws)
    for call in range(2):
        y_out.fill_(float("nan"))
        h_out.fill_(float("nan"))
        binding.ssm_scan_fwd_noalloc(**inp, chunk_len=q, out=y_out, h_last=h_out)
        torch.cuda.synchronize()
        assert binding.device_status() == binding.SSM_OK
        assert rel_l2(y_out.float().cpu().numpy(), y_ws.float().cpu().numpy()) <= TOL_Y_BF16, call
        assert rel_l2(h_out.cpu().numpy(), h_ws.cpu().numpy()) <= TOL_H, call


def test_noalloc_refuses_a_scratch_need_beyond_its_buffer(cuda_dev):
    inp = _to(cuda_dev, make_scan_inputs(1, 4096, 1024, 64, "bf16", seed=778))
    q = 16   # 256 chunks: (256 - 1) * 1024 * 65 * 4 bytes of scratch, far above 16 MiB
    assert binding.scan_workspace_size(**inp, chunk_len=q) > binding.NOALLOC_SCRATCH_BYTES
    before = binding.kernel_launch_count()
    with pytest.raises(binding.SSMError) as e:
        binding.ssm_scan_fwd_noalloc(**inp, chunk_len=q)
    assert e.value.status == binding.SSM_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
    assert binding.kernel_launch_count() == before
