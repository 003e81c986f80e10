"""The bounds-checked debug build, the stand-in for a memory checker (compute-sanitizer is
not available on this machine): the library compiled with -DGQA_BOUNDS_CHECK checks every
global store of every kernel against the extent of its buffer, skips a store that would
leave it and sets GQA_DEV_BOUNDS in the device status.  A probe shows the guard firing on a
store past a declared extent (the buffer itself is larger: nothing leaves the allocation),
then representative parity suites run against the checked library in a child process: any
store out of its buffer would set the status bit their checks read, or leave an output
element unwritten (NaN-filled outputs, guarded margins)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# every kernel and store path: split decode (cluster and ticket combines, fused append, pages,
# f8 and int8 codes), tensor-core prefill (masks with the block map), RoPE/append, the
# CUDA-core kernel, the past copy
SUITES = ["tests/test_gpu_decode.py", "tests/test_gpu_prefill.py", "tests/test_gpu_rope_append.py",
          "tests/test_gpu_paged.py", "tests/test_gpu_mask_skip.py::test_dead_tiles_are_never_read",
          "tests/test_gpu_q8.py::test_split_decode_q8", "tests/test_gpu_q8.py::test_cuda_core_q8"]


@pytest.fixture(scope="module")
def checked_lib():
    from sliding_window_gb300 import build
    return build.build(checked=True)


def test_guard_skips_and_reports_a_store_past_its_extent(checked_lib):
    import ctypes
    lib = ctypes.CDLL(checked_lib)
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.gqa_test_bounds_check(ctypes.c_void_p(buf.data_ptr()), ctypes.c_void_p(st.data_ptr()), None) == 0
    torch.cuda.synchronize()
    b = buf.cpu()
    assert int(b[8]) == 5 and int(b[40]) == 0  # the in-extent store landed, the other did not
    assert int(st.item()) == 16  # GQA_DEV_BOUNDS


def test_parity_suites_pass_on_the_checked_build(checked_lib):
    env = dict(os.environ, GQA_CHECKED_BUILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] + SUITES,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
