"""The FA_DEBUG build (libfa_debug.so): every computed TMA coordinate, output
row and TMEM base column is checked before use, and a failed check sets a
device status bit (5 for the forward kernel, 12 for the backward kernels)
instead of trapping.

The test runs the parity suites of the forward (bf16, 8-bit, CTA pair), the
backward and the split-KV path in a child process whose FA_LIBRARY points at
the debug library.  Those suites check after every test that the device
status word is clear, so every shape they cover must pass all address checks
as well as match the oracle.  The full-size workloads are left out to bound
the time."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_fa_gpu.py", "tests/test_bwd_gpu.py", "tests/test_fp8_gpu.py", "tests/test_decode_gpu.py",
          "tests/test_fwd_pair_gpu.py"]


@pytest.mark.gpu
def test_parity_suites_pass_every_debug_check():
    from exact_attention_42_gb300.build import build
    path = build(debug=True)
    env = dict(os.environ, FA_LIBRARY=path)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
           "-k", "not full_size and not headline", *SUITES]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((res.stdout + res.stderr).splitlines()[-30:])
    assert res.returncode == 0, "parity suites on the debug build failed:\n" + tail
    assert " passed" in res.stdout, tail


@pytest.mark.gpu
def test_debug_library_is_the_one_loaded():
    # The child must really run the debug build: FA_LIBRARY selects it.
    from exact_attention_42_gb300.build import build
    path = build(debug=True)
    code = "import exact_attention_42_gb300 as fa; fa.lib(); print(fa.lib_path())"
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=dict(os.environ, FA_LIBRARY=path),
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().endswith("libfa_debug.so")
