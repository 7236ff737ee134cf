"""The checked build (-DLP_CHECKED) on a GB300.

Every kernel of the checked library tests the indexes and TMA coordinates it
computes against the extents derived from the call's arguments, and records a
failed test in a check word instead of faulting.  Over small parity cases of
every entry point (logits path with ragged and unaligned rows, temperature and
shards; fused path with fewer than 16 rows, ragged V, shards, lse and the
no-alloc call; the backward with fp32 and bf16 grad_W and saved statistics)
the check word must stay 0 and every output must have the bits of the normal
build.
"""

import os
import subprocess
import sys

import pytest
import torch

from invariant_token_logprobs_gb300 import _build_lib, lp, synth
from _checked_cases import run_cases

pytestmark = pytest.mark.gpu


def test_checked_build_clean_and_bitwise_equal(tmp_path):
    lp.load()
    checked = _build_lib.build(checked=True)
    ref = run_cases(lp, synth)
    path = str(tmp_path / "checked.pt")
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_checked_child.py")
    env = dict(os.environ, LP_LIBRARY=checked)
    res = subprocess.run([sys.executable, child, path], capture_output=True, text=True, env=env,
                         timeout=600)
    assert res.returncode == 0, res.stdout + res.stderr
    got = torch.load(path)
    assert got["backend"] == "lp.sm103a.bitwise.v1+checked"
    assert got["status"] == 0
    assert got["word"] == 0, f"check word {got['word']:#x}"
    assert set(got["out"]) == set(ref)
    for k in ref:
        assert torch.equal(got["out"][k], ref[k]), k


def test_normal_build_check_word_is_zero():
    import ctypes
    lib = lp.load()
    word = ctypes.c_uint32(1)
    assert lib.lp_get_check_word(ctypes.byref(word)) == 0 and word.value == 0
    assert lp.lp_backend_id() == "lp.sm103a.bitwise.v1"
