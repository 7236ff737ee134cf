"""Child process of tests/test_gpu_checked.py: runs the shared parity cases
with the library named by LP_LIBRARY (the checked build) and saves the outputs,
the backend id and the check word."""

import ctypes
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from invariant_token_logprobs_gb300 import lp, synth  # noqa: E402
from _checked_cases import run_cases  # noqa: E402


def main(path):
    lib = lp.load(build_if_needed=False)
    out = run_cases(lp, synth)
    word = ctypes.c_uint32(0xFFFFFFFF)
    st = lib.lp_get_check_word(ctypes.byref(word))
    torch.save({"out": out, "backend": lp.lp_backend_id(), "status": st, "word": word.value}, path)


if __name__ == "__main__":
    main(sys.argv[1])
