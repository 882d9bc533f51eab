"""GPU tests of the TMA selective-scan path: parity with the oracle on layouts it takes,
agreement with the generic path, and the bounded-wait timeout (host-injected, no fault)."""
import pytest
import torch

import oracle
from selective_state_space_127_b300 import binding, check_status, new_workspace, ssm_scan_fwd
from selective_state_space_127_b300.synth import make_scan_inputs
from conftest import rel_l2

pytestmark = pytest.mark.gpu

TOL_Y = {"f32": 1e-5, "bf16": 2e-2}
TOL_H = {"f32": 1e-5, "bf16": 1e-4}


def _to(dev, inp):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def _misaligned_copy(t):
    """Same values in a view whose base is off the 16-byte grid (the TMA path refuses it)."""
    big = torch.empty(t.shape[:-1] + (t.shape[-1] + 1,), dtype=t.dtype, device=t.device)
    v = big[..., 1:]
    v.copy_(t)
    return v


FAST_CASES = [
    # b, L, D, N, dtype, gate, dskip, softplus
    (1, 1, 16, 16, "bf16", True, True, True),
    (2, 77, 40, 16, "bf16", True, True, True),
    (3, 300, 48, 64, "f32", True, False, True),
    (1, 70, 32, 64, "bf16", True, True, True),
    (1, 129, 24, 32, "bf16", False, True, True),
    (2, 64, 64, 16, "f32", False, False, True),
    (1, 1000, 16, 16, "bf16", True, True, True),
    (2, 45, 32, 32, "f32", True, True, False),
]


@pytest.mark.parametrize("b,L,D,N,dt,gate,dskip,sp", FAST_CASES)
def test_tma_path_matches_oracle_and_generic_path(cuda_dev, b, L, D, N, dt, gate, dskip, sp):
    inp = make_scan_inputs(b, L, D, N, dt, seed=3000 + L + D + N, d_skip="normal" if dskip else "none", gate=gate)
    if not sp:
        inp["delta"] = (inp["delta"].float().abs() * 0.05).to(inp["delta"].dtype)
        inp["delta_bias"] = torch.full_like(inp["delta_bias"], 1e-3)
    g = _to(cuda_dev, inp)
    ws = new_workspace(binding.scan_workspace_size(**g, delta_softplus=sp), cuda_dev)
    y_fast, h_fast = ssm_scan_fwd(**g, delta_softplus=sp, workspace=ws)
    slow = dict(g, x=_misaligned_copy(g["x"]))
    y_gen, h_gen = ssm_scan_fwd(**slow, delta_softplus=sp)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssm_scan_ref(**inp, delta_softplus=sp)
    yf, yg = y_fast.float().cpu().numpy(), y_gen.float().cpu().numpy()
    assert rel_l2(yf, y_ref) <= TOL_Y[dt]
    assert rel_l2(h_fast.cpu().numpy(), h_ref) <= TOL_H[dt]
    assert rel_l2(yg, y_ref) <= TOL_Y[dt]
    # same fp32 recurrence, different softplus evaluation and summation order
    assert rel_l2(h_fast.cpu().numpy(), h_gen.cpu().numpy()) <= 2e-6
    assert check_status(ws) == binding.SSM_OK


def test_bf16_outputs_are_the_rounded_oracle(cuda_dev):
    """With fp32 state the only visible error on bf16 y should be the final rounding: nearly
    every element equals the oracle's value rounded to bf16, and the rest differ by one bf16
    step (or by fp32-level noise where y is near zero)."""
    inp = make_scan_inputs(4, 512, 256, 16, "bf16", seed=99)
    y, _ = ssm_scan_fwd(**_to(cuda_dev, inp))
    y_ref, _ = oracle.ssm_scan_ref(**inp)
    y_ref_b = torch.from_numpy(y_ref).to(torch.bfloat16)
    same = (y.cpu() == y_ref_b).float().mean().item()
    scale = float(torch.from_numpy(y_ref).pow(2).mean().sqrt())
    near = (y.cpu().float() - y_ref_b.float()).abs() <= y_ref_b.float().abs() * 2 ** -7 + 1e-5 * scale
    assert same >= 0.97, same
    assert near.all()


def test_injected_missing_copy_times_out_and_context_survives(cuda_dev):
    """The test hook withholds the first TMA copy: the bounded wait gives up after about a
    second, the status word of that call's workspace reads SSM_ERR_TIMEOUT, and the next call
    works normally."""
    inp = _to(cuda_dev, make_scan_inputs(1, 16, 32, 16, "bf16", seed=5))
    ws = new_workspace(binding.scan_workspace_size(**inp), cuda_dev)
    assert check_status(ws) == binding.SSM_OK
    ssm_scan_fwd(**inp, debug_flags=binding.SSM_DEBUG_SKIP_FIRST_LOAD, workspace=ws)
    assert check_status(ws, clear=True) == binding.SSM_ERR_TIMEOUT
    assert check_status(ws) == binding.SSM_OK
    y, h = ssm_scan_fwd(**inp, workspace=ws)
    assert check_status(ws) == binding.SSM_OK
    y_ref, h_ref = oracle.ssm_scan_ref(**{k: (v.cpu() if v is not None else None) for k, v in inp.items()})
    assert rel_l2(y.float().cpu().numpy(), y_ref) <= TOL_Y["bf16"]


def test_timeout_is_reported_only_to_the_workspace_that_had_it(cuda_dev):
    """Two calls on two streams with two workspaces: the one whose first copy is withheld
    reads SSM_ERR_TIMEOUT from its own workspace; the other call's workspace reads SSM_OK."""
    inp = _to(cuda_dev, make_scan_inputs(1, 16, 32, 16, "bf16", seed=15))
    need = binding.scan_workspace_size(**inp)
    ws_a, ws_b = new_workspace(need, cuda_dev), new_workspace(need, cuda_dev)
    s_a, s_b = torch.cuda.Stream(device=cuda_dev), torch.cuda.Stream(device=cuda_dev)
    torch.cuda.synchronize()
    ssm_scan_fwd(**inp, debug_flags=binding.SSM_DEBUG_SKIP_FIRST_LOAD, workspace=ws_a, stream=s_a)
    y, h = ssm_scan_fwd(**inp, workspace=ws_b, stream=s_b)
    assert check_status(ws_b, stream=s_b) == binding.SSM_OK
    assert check_status(ws_a, stream=s_a) == binding.SSM_ERR_TIMEOUT
    y_ref, h_ref = oracle.ssm_scan_ref(**{k: (v.cpu() if v is not None else None) for k, v in inp.items()})
    assert rel_l2(y.float().cpu().numpy(), y_ref) <= TOL_Y["bf16"]


def test_in_place_state_with_a_split_sequence(cuda_dev):
    """h_last may be the h0 buffer when the sequence is split into chunks: the output pass of
    the first chunk reads a copy of h0 that the carry kernel made, not the buffer the last
    chunk overwrites."""
    inp = make_scan_inputs(2, 1000, 48, 16, "bf16", seed=4321, d_skip="normal")
    h0 = torch.randn(2, 48, 16, generator=torch.Generator().manual_seed(4322))
    g = _to(cuda_dev, inp)
    y_ref_gpu, h_ref_gpu = ssm_scan_fwd(**g, h0=h0.to(cuda_dev), chunk_len=64)
    state = h0.to(cuda_dev)
    y, h = ssm_scan_fwd(**g, h0=state, h_last=state, chunk_len=64)
    torch.cuda.synchronize()
    assert h.data_ptr() == state.data_ptr()
    assert torch.equal(y, y_ref_gpu)
    assert torch.equal(state, h_ref_gpu)
    y_ref, h_ref = oracle.ssm_scan_ref(**inp, h0=h0)
    assert rel_l2(y.float().cpu().numpy(), y_ref) <= TOL_Y["bf16"]
    assert rel_l2(state.cpu().numpy(), h_ref) <= TOL_H["bf16"]


def test_phase_events_time_each_kernel_of_a_split_call(cuda_dev):
    """The phase events bracket the three kernels of a split sequence (local pass, carry,
    output pass) and the single kernel of an unsplit one; unused trailing events are recorded
    at the end of the call."""
    inp = _to(cuda_dev, make_scan_inputs(1, 8192, 32, 16, "bf16", seed=4323))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ssm_scan_fwd(**inp, chunk_len=1024, phase_events=ev)
    torch.cuda.synchronize()
    parts = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    assert all(p > 0 for p in parts), parts
    ssm_scan_fwd(**inp, chunk_len=8192, phase_events=ev)
    torch.cuda.synchronize()
    assert ev[0].elapsed_time(ev[1]) > 0
    assert ev[1].elapsed_time(ev[3]) < 0.01


def test_workspace_size_is_header_plus_carries(cuda_dev):
    inp = _to(cuda_dev, make_scan_inputs(2, 64, 16, 16, "bf16", seed=4324))
    hdr = binding.WORKSPACE_HEADER_BYTES
    assert binding.scan_workspace_size(**inp) == hdr
    # two chunks of 32 steps: two carry slots of b * D * N floats, one Σdt slot of b * D
    assert binding.scan_workspace_size(**inp, chunk_len=32) == hdr + (2 * 2 * 16 * 16 + 2 * 16) * 4


def test_debug_hook_is_refused_where_it_could_leave_copies_in_flight(cuda_dev):
    inp = _to(cuda_dev, make_scan_inputs(1, 100, 32, 16, "bf16", seed=6))
    with pytest.raises(binding.SSMError) as e:
        ssm_scan_fwd(**inp, debug_flags=binding.SSM_DEBUG_SKIP_FIRST_LOAD)
    assert e.value.status == binding.SSM_ERR_INVALID_ARG


CHUNK_CASES = [
    # b, L, D, N, dtype, chunk_len, with h0
    (1, 1000, 32, 16, "bf16", 64, True),      # 16 chunks, ragged last chunk
    (2, 777, 48, 16, "f32", 100, False),      # chunk rounded up to 112 steps
    (1, 300, 16, 32, "f32", 48, True),
    (1, 257, 40, 64, "bf16", 128, True),      # ragged channel tile too
]


@pytest.mark.parametrize("b,L,D,N,dt,q,with_h0", CHUNK_CASES)
def test_chunked_sequence_matches_oracle_and_single_chunk(cuda_dev, b, L, D, N, dt, q, with_h0):
    """The sequence split into chunks (local pass, carry, output pass) gives the oracle's
    result and agrees with the one-chunk run up to fp32 rounding."""
    inp = make_scan_inputs(b, L, D, N, dt, seed=4000 + L + D + N + q, d_skip="normal")
    h0 = torch.randn(b, D, N, generator=torch.Generator().manual_seed(L)) if with_h0 else None
    g = _to(cuda_dev, inp)
    h0_d = h0.to(cuda_dev) if h0 is not None else None
    ws = new_workspace(binding.scan_workspace_size(**g, chunk_len=q), cuda_dev)
    y_c, h_c = ssm_scan_fwd(**g, h0=h0_d, chunk_len=q, workspace=ws)
    y_1, h_1 = ssm_scan_fwd(**g, h0=h0_d, chunk_len=L)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssm_scan_ref(**inp, h0=h0)
    assert rel_l2(y_c.float().cpu().numpy(), y_ref) <= TOL_Y[dt]
    assert rel_l2(h_c.cpu().numpy(), h_ref) <= TOL_H[dt]
    assert rel_l2(h_c.cpu().numpy(), h_1.cpu().numpy()) <= 2e-6
    assert rel_l2(y_c.float().cpu().numpy(), y_1.float().cpu().numpy()) <= (2e-6 if dt == "f32" else 4e-3)
    assert check_status(ws) == binding.SSM_OK


def test_automatic_split_for_few_channels(cuda_dev):
    """One channel tile and a long sequence: the library splits the sequence by itself and
    asks for workspace; the result matches the oracle."""
    inp = make_scan_inputs(1, 4096, 16, 16, "bf16", seed=4242)
    g = _to(cuda_dev, inp)
    lib = binding.load_library()
    y, h = ssm_scan_fwd(**g)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssm_scan_ref(**inp)
    assert rel_l2(y.float().cpu().numpy(), y_ref) <= TOL_Y["bf16"]
    assert rel_l2(h.cpu().numpy(), h_ref) <= TOL_H["bf16"]
    assert binding.scan_workspace_size(**g) > binding.WORKSPACE_HEADER_BYTES


VARIANT_CASES = [
    # b, L, D, N, dtype, zoh, reverse, chunk_len, with h0
    (2, 77, 40, 16, "bf16", True, False, 0, True),
    (1, 300, 48, 64, "f32", True, False, 0, False),
    (2, 129, 24, 32, "f32", True, False, 0, True),
    (1, 1000, 32, 16, "f32", True, False, 96, True),    # ZOH through the chunked path
    (2, 77, 40, 16, "bf16", False, True, 0, True),
    (1, 300, 48, 64, "f32", False, True, 0, False),
    (3, 129, 24, 32, "f32", False, True, 0, True),
    (1, 4096, 16, 16, "bf16", False, True, 0, False),   # would be split forward; reverse is one chunk
]


@pytest.mark.parametrize("b,L,D,N,dt,zoh,rev,q,with_h0", VARIANT_CASES)
def test_zoh_and_reverse_on_the_tma_path(cuda_dev, b, L, D, N, dt, zoh, rev, q, with_h0):
    """Exact-ZOH and reverse-direction kernels of the TMA path against the oracle and the
    generic kernel (forced by a misaligned copy of x)."""
    A = None
    if zoh:
        # A with zeros (the dt B limit), tiny and large magnitudes: both branches of the
        # ZOH coefficient (series for |dt A| < 1/8, (A_bar - 1) / A above)
        row = -torch.logspace(-4, 1.5, N, dtype=torch.float64)
        row[::5] = 0.0
        A = row.to(torch.float32).repeat(D, 1)
    inp = make_scan_inputs(b, L, D, N, dt, seed=7000 + L + D + N + 2 * zoh + rev, d_skip="normal", A=A)
    h0 = torch.randn(b, D, N, generator=torch.Generator().manual_seed(L + 1)) if with_h0 else None
    g = _to(cuda_dev, inp)
    h0_d = h0.to(cuda_dev) if h0 is not None else None
    ws = new_workspace(binding.scan_workspace_size(**g, zoh=zoh, reverse=rev, chunk_len=q), cuda_dev)
    y_f, h_f = ssm_scan_fwd(**g, h0=h0_d, zoh=zoh, reverse=rev, chunk_len=q, workspace=ws)
    y_g, h_g = ssm_scan_fwd(**dict(g, x=_misaligned_copy(g["x"])), h0=h0_d, zoh=zoh, reverse=rev)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssm_scan_ref(**inp, h0=h0, zoh=zoh, reverse=rev)
    assert rel_l2(y_f.float().cpu().numpy(), y_ref) <= TOL_Y[dt]
    assert rel_l2(h_f.cpu().numpy(), h_ref) <= TOL_H[dt]
    assert rel_l2(y_g.float().cpu().numpy(), y_ref) <= TOL_Y[dt]
    assert rel_l2(h_f.cpu().numpy(), h_g.cpu().numpy()) <= 1e-5
    if rev:
        assert binding.scan_workspace_size(**g, reverse=True) == binding.WORKSPACE_HEADER_BYTES
    assert check_status(ws) == binding.SSM_OK


def test_tiny_chunk_len_on_a_long_sequence_is_capped_at_the_grid_limit(cuda_dev):
    """chunk_len = 32 on 2.2 M steps would need more than 65535 chunks (the grid's z extent):
    the library lengthens the chunks and the result still matches the oracle."""
    L = 2_200_000
    inp = make_scan_inputs(1, L, 16, 16, "bf16", seed=4343, d_skip="normal")
    g = _to(cuda_dev, inp)
    need = binding.scan_workspace_size(**g, chunk_len=32)
    assert binding.WORKSPACE_HEADER_BYTES < need <= binding.WORKSPACE_HEADER_BYTES + 65535 * 16 * 17 * 4
    ws = new_workspace(need, cuda_dev)
    y, h = ssm_scan_fwd(**g, chunk_len=32, workspace=ws)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssm_scan_ref(**inp)
    assert rel_l2(y[:, -20000:].float().cpu().numpy(), y_ref[:, -20000:]) <= TOL_Y["bf16"]
    assert rel_l2(h.cpu().numpy(), h_ref) <= TOL_H["bf16"]
    assert check_status(ws) == binding.SSM_OK
