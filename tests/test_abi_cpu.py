"""Host-side checks of the C ABI (no GPU needed, no kernel launched)."""
import ctypes
import os
import re
import subprocess

import pytest

from selective_state_space_127_b300 import binding
from selective_state_space_127_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssmscan.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SSMSCAN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.check_output(["nm", "-D", "--defined-only", binding.LIB_PATH]).decode()
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [f for f in _declared_functions() if f not in exported]
    assert not missing, missing
    for f in _declared_functions():
        assert hasattr(lib, f)


def test_library_needs_no_cuda_shared_runtime():
    out = subprocess.check_output(["ldd", binding.LIB_PATH]).decode()
    assert "libcudart" not in out and "libtorch" not in out


def test_abi_version_and_status_strings(lib):
    assert lib.ssm_abi_version() == binding.ABI_VERSION
    for code in range(7):
        assert lib.ssm_status_string(code).decode() == binding._status_name(code)


def _c_offsets(struct, fields):
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"ssmscan.h\"\nint main(void){\n"
    for f in fields:
        src += f'printf("%zu\\n", offsetof({struct}, {f}));\n'
    src += f'printf("%zu\\n", sizeof({struct}));\nreturn 0;}}\n'
    return src


@pytest.mark.parametrize("struct,cls", [("ssm_scan_params", binding.ScanParams),
                                        ("ssd_scan_params", binding.SSDParams),
                                        ("ssm_conv1d_params", binding.Conv1dParams)])
def test_ctypes_struct_layout_matches_header(tmp_path, struct, cls):
    fields = [f for f, _ in cls._fields_]
    c = tmp_path / "probe.c"
    c.write_text(_c_offsets(struct, fields))
    exe = tmp_path / "probe"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)])
    vals = [int(v) for v in subprocess.check_output([str(exe)]).decode().split()]
    assert vals[:-1] == [getattr(cls, f).offset for f in fields]
    assert vals[-1] == ctypes.sizeof(cls)


def _valid_scan_params():
    p = binding.ScanParams()
    p.batch, p.seqlen, p.dim, p.dstate = 2, 8, 4, 16
    p.io_dtype = binding.SSM_DTYPE_BF16
    p.delta_softplus = 1
    # aligned, never-dereferenced, non-overlapping addresses: validation only
    for i, name in enumerate(("x", "delta", "B", "C", "A", "y")):
        setattr(p, name, (i + 1) << 20)
    p.x_stride[:] = (32, 4, 1)
    p.delta_stride[:] = (32, 4, 1)
    p.y_stride[:] = (32, 4, 1)
    p.B_stride[:] = (128, 16, 1)
    p.C_stride[:] = (128, 16, 1)
    return p


def test_workspace_query_accepts_valid_params(lib):
    p = _valid_scan_params()
    assert lib.ssm_scan_workspace_size(ctypes.byref(p)) != ctypes.c_size_t(-1).value


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, binding.SSM_ERR_INVALID_ARG),
    ("dim", -1, binding.SSM_ERR_INVALID_ARG),
    ("seqlen", -5, binding.SSM_ERR_INVALID_ARG),
    ("dstate", 0, binding.SSM_ERR_INVALID_ARG),
    ("dstate", 257, binding.SSM_ERR_UNSUPPORTED),
    ("io_dtype", 7, binding.SSM_ERR_INVALID_ARG),
    ("discretization", 3, binding.SSM_ERR_INVALID_ARG),
    ("reverse", 2, binding.SSM_ERR_INVALID_ARG),
    ("A", 0, binding.SSM_ERR_INVALID_ARG),
    ("x", 0, binding.SSM_ERR_INVALID_ARG),
    ("y", (1 << 20) + 1, binding.SSM_ERR_INVALID_ARG),
    ("chunk_len", -1, binding.SSM_ERR_INVALID_ARG),
])
def test_invalid_scan_args_are_rejected_before_launch(lib, field, value, status):
    p = _valid_scan_params()
    setattr(p, field, value)
    assert lib.ssm_scan_workspace_size(ctypes.byref(p)) == ctypes.c_size_t(-1).value
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == status
    assert lib.ssm_last_error().decode() != ""


def _header_define(name):
    m = re.search(r"#define\s+" + name + r"\s+(.+)", open(HEADER).read())
    return eval(m.group(1).replace("u", ""))


def test_header_constants_match_the_library_and_binding(lib):
    assert lib.ssm_noalloc_scratch_bytes() == _header_define("SSM_NOALLOC_SCRATCH_BYTES")
    assert binding.noalloc_scratch_bytes() == _header_define("SSM_NOALLOC_SCRATCH_BYTES")
    assert binding.WORKSPACE_HEADER_BYTES == _header_define("SSM_WORKSPACE_HEADER_BYTES")
    assert binding.ABI_VERSION == _header_define("SSMSCAN_ABI_VERSION")


@pytest.mark.parametrize("name", ["x", "delta", "B", "C", "A"])
def test_output_overlapping_an_input_is_rejected(lib, name):
    p = _valid_scan_params()
    p.y = getattr(p, name) + 32           # y's range starts inside the input's range
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    assert "overlap" in lib.ssm_last_error().decode()
    p = _valid_scan_params()
    p.h_last = getattr(p, name)           # the final state over an input
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG


def test_h_last_may_be_h0_but_not_partly_overlap_it(lib):
    p = _valid_scan_params()
    p.h0 = p.h_last = 7 << 20
    assert lib.ssm_scan_workspace_size(ctypes.byref(p)) != ctypes.c_size_t(-1).value
    p.h_last = (7 << 20) + 64
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG


def test_phase_event_fields_are_checked(lib):
    p = _valid_scan_params()
    p.n_phase_events = 2                  # no array
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    p = _valid_scan_params()
    p.reserved2 = 1
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG


def test_algorithm_field_is_checked(lib):
    """algorithm: 0 (serial walk) or 1 (in-tile associative scan); anything else is an argument
    error, and the associative scan refuses what it does not take before any launch."""
    p = _valid_scan_params()
    p.algorithm = 2
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    assert lib.ssm_scan_workspace_size(ctypes.byref(p)) == ctypes.c_size_t(-1).value
    for field, value in (("reverse", 1), ("discretization", binding.SSM_DISC_ZOH), ("dstate", 64)):
        p = _valid_scan_params()
        p.algorithm = binding.SSM_SCAN_ALGO_ASSOC
        setattr(p, field, value)
        assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_UNSUPPORTED, field


def test_workspace_sizes_include_the_status_header(lib):
    p = _valid_scan_params()              # bf16, dense, 16-byte aligned: the TMA path
    p.seqlen = 64
    p.x_stride[:] = p.delta_stride[:] = p.y_stride[:] = (64 * 16, 16, 1)
    p.dim = 16
    p.B_stride[:] = p.C_stride[:] = (64 * 16, 16, 1)
    # the TMA path needs the driver's tensor-map encoder; without a driver (a CPU-only host)
    # the library picks the generic kernel, which needs no workspace
    n1 = lib.ssm_scan_workspace_size(ctypes.byref(p))
    p.chunk_len = 32                      # two chunks: carries after the header
    n2 = lib.ssm_scan_workspace_size(ctypes.byref(p))
    if n1 != 0:
        assert n1 == binding.WORKSPACE_HEADER_BYTES
        assert n2 == binding.WORKSPACE_HEADER_BYTES + (2 * 2 * 16 * 16 + 1 * 2 * 16) * 4
    else:
        assert n2 == 0
    p.seqlen = 1                          # the short-sequence kernel has no device-side waits
    assert lib.ssm_scan_workspace_size(ctypes.byref(p)) == 0
    c = _valid_conv_params()
    assert lib.ssm_causal_conv1d_workspace_size(ctypes.byref(c)) == binding.WORKSPACE_HEADER_BYTES
    assert lib.ssm_causal_conv1d_fwd(ctypes.byref(c), None) == binding.SSM_ERR_WORKSPACE


def test_overlapping_output_strides_are_rejected(lib):
    p = _valid_scan_params()
    p.y_stride[:] = (32, 1, 1)   # t and d step onto the same elements
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    p = _valid_scan_params()
    p.x_stride[:] = (32, -4, 1)
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG


def test_invalid_ssd_args_are_rejected_before_launch(lib):
    p = binding.SSDParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk_size = 1, 16, 6, 8, 16, 4, 8
    fake = 1 << 20
    for name in ("x", "delta", "A", "B", "C", "y"):
        setattr(p, name, fake)
    p.io_dtype, p.delta_softplus = binding.SSM_DTYPE_BF16, 1
    assert lib.ssd_chunk_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG   # 4 does not divide 6
    p.ngroups = 2
    p.chunk_size = 0
    assert lib.ssd_chunk_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    p.chunk_size = 8
    assert lib.ssd_chunk_scan_workspace_size(ctypes.byref(p)) != ctypes.c_size_t(-1).value


def test_null_params_are_rejected(lib):
    assert lib.ssm_scan_fwd(None, None) == binding.SSM_ERR_INVALID_ARG
    assert lib.ssd_chunk_scan_fwd(None, None) == binding.SSM_ERR_INVALID_ARG


def test_conv_prologue_args_are_checked_before_launch(lib):
    fake = 1 << 20
    p = _valid_scan_params()
    p.conv_weight, p.conv_width = fake, 5            # more than 4 taps
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    p.conv_width = 0
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    p.conv_width, p.reverse = 4, 1                    # the prologue is causal: forward only
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_UNSUPPORTED
    p.reverse, p.conv_x_prev = 0, fake + 1            # x_prev not aligned to bf16
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    p.conv_x_prev, p.reserved2 = 0, 1
    assert lib.ssm_scan_fwd(ctypes.byref(p), None) == binding.SSM_ERR_INVALID_ARG
    p.reserved2 = 0
    assert lib.ssm_scan_workspace_size(ctypes.byref(p)) != ctypes.c_size_t(-1).value


def _valid_conv_params():
    p = binding.Conv1dParams()
    p.batch, p.seqlen, p.dim, p.width = 2, 64, 16, 4
    p.io_dtype, p.silu = binding.SSM_DTYPE_BF16, 1
    p.x, p.weight, p.y = 1 << 20, 1 << 21, 1 << 22
    return p


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, binding.SSM_ERR_INVALID_ARG),
    ("seqlen", -1, binding.SSM_ERR_INVALID_ARG),
    ("width", 0, binding.SSM_ERR_INVALID_ARG),
    ("width", 5, binding.SSM_ERR_INVALID_ARG),
    ("io_dtype", 3, binding.SSM_ERR_INVALID_ARG),
    ("silu", 2, binding.SSM_ERR_INVALID_ARG),
    ("reserved", 1, binding.SSM_ERR_INVALID_ARG),
    ("weight", 0, binding.SSM_ERR_INVALID_ARG),
    ("x", (1 << 20) + 8, binding.SSM_ERR_INVALID_ARG),     # not 16-byte aligned
    ("dim", 12, binding.SSM_ERR_UNSUPPORTED),              # 24 bytes of bf16 per row
    ("y", (1 << 20) + 1024, binding.SSM_ERR_INVALID_ARG),  # overlaps x
])
def test_invalid_conv1d_args_are_rejected_before_launch(lib, field, value, status):
    p = _valid_conv_params()
    setattr(p, field, value)
    assert lib.ssm_causal_conv1d_fwd(ctypes.byref(p), None) == status
    assert lib.ssm_last_error().decode() != ""
    assert lib.ssm_causal_conv1d_fwd(None, None) == binding.SSM_ERR_INVALID_ARG


def test_debug_build_exports_the_same_symbols():
    from selective_state_space_127_b300.build import DEBUG_LIB_PATH, build as build_lib
    build_lib(debug_checks=True)
    out = subprocess.check_output(["nm", "-D", "--defined-only", DEBUG_LIB_PATH]).decode()
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    assert set(_declared_functions()) <= exported
    lib = ctypes.CDLL(DEBUG_LIB_PATH)
    lib.ssm_status_string.restype = ctypes.c_char_p
    assert lib.ssm_status_string(binding.SSM_ERR_BOUNDS).decode() == "SSM_ERR_BOUNDS"
