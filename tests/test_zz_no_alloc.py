"""The allocation-free scan entry point, ssm_scan_fwd_noalloc, called through the C ABI.

Some callers cannot hand the library a workspace: a host application whose device memory is
planned once at start-up, or a plugin inside a runtime that owns every device allocation.
For them the chunk-carry scratch lives in a fixed buffer inside the library. Here that entry
point must reproduce the workspace entry point's results bit for bit on a long sequence that
is split into chunks (so the scratch is used), on two calls in a row with different inputs
and initial states (the buffer keeps the previous call's contents, so a read of stale scratch
would show), and it must refuse a call whose scratch need exceeds the buffer before
launching anything.

This file sorts last so that a stop-at-first-failure run has run every other test first.
"""
import pytest
import torch

from selective_state_space_127_b300 import binding, ssm_scan_fwd
from selective_state_space_127_b300.synth import make_scan_inputs

pytestmark = pytest.mark.gpu


def _to(dev, inp):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_dev):
    q = 256
    calls = [(make_scan_inputs(2, 3000, 48, 16, "bf16", seed=777, d_skip="normal"), None),
             (make_scan_inputs(2, 3000, 48, 16, "bf16", seed=779, d_skip="normal"),
              torch.randn(2, 48, 16, generator=torch.Generator().manual_seed(780)))]
    for call, (inp, h0) in enumerate(calls):
        g = _to(cuda_dev, inp)
        h0_d = h0.to(cuda_dev) if h0 is not None else None
        need = binding.scan_workspace_size(**g, h0=h0_d, chunk_len=q)
        assert binding.WORKSPACE_HEADER_BYTES < need <= binding.noalloc_scratch_bytes()
        y_ws, h_ws = ssm_scan_fwd(**g, h0=h0_d, chunk_len=q)
        y_out = torch.full_like(y_ws, float("nan"))
        h_out = torch.full_like(h_ws, float("nan"))
        binding.ssm_scan_fwd_noalloc(**g, h0=h0_d, chunk_len=q, out=y_out, h_last=h_out)
        torch.cuda.synchronize()
        assert binding.check_status(None) == binding.SSM_OK, call
        # the same kernels on the same inputs: identical results
        assert torch.equal(y_out, y_ws), call
        assert torch.equal(h_out, h_ws), call


def test_noalloc_refuses_a_scratch_need_beyond_its_buffer(cuda_dev):
    inp = _to(cuda_dev, make_scan_inputs(1, 4096, 1024, 64, "bf16", seed=778))
    q = 16   # 256 chunks: 256 * 1024 * 64 * 4 bytes of carries alone, far above 16 MiB
    assert binding.scan_workspace_size(**inp, chunk_len=q) > binding.noalloc_scratch_bytes()
    before = binding.kernel_launch_count()
    with pytest.raises(binding.SSMError) as e:
        binding.ssm_scan_fwd_noalloc(**inp, chunk_len=q)
    assert e.value.status == binding.SSM_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
    assert binding.kernel_launch_count() == before
