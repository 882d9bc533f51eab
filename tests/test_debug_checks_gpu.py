"""The index-checking debug build of the library (libssmscan_debug.so, -DSSM_DEBUG_CHECKS):
on calls that reach every kernel, its kernels find no index outside its array (every status
word reads SSM_OK) and its results equal the normal build's bit for bit (the checks only add
comparisons). The debug build runs in a process of its own (SSMSCAN_LIBRARY selects it)."""
import os
import subprocess
import sys

import pytest
import torch

from selective_state_space_127_b300 import binding
from selective_state_space_127_b300.build import DEBUG_LIB_PATH, build

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
import debug_checks_cases  # noqa: E402

pytestmark = pytest.mark.gpu


def test_debug_build_finds_no_bad_index_and_matches_the_normal_build(cuda_dev, tmp_path):
    build(debug_checks=True)
    dump = tmp_path / "debug.pt"
    env = dict(os.environ, SSMSCAN_LIBRARY=os.path.basename(DEBUG_LIB_PATH))
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_checks_cases.py"), str(dump)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "libssmscan_debug.so" in r.stdout
    dbg = torch.load(dump)
    ref = debug_checks_cases.run(cuda_dev)
    assert set(dbg) == set(ref)
    for k, v in dbg.items():
        if k.endswith(".status"):
            assert v == binding.SSM_OK, (k, v)
            assert ref[k] == binding.SSM_OK, k
        else:
            assert torch.equal(v, ref[k].cpu()), k
