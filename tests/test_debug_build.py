"""The FA_DEBUG build compiles here (nvcc cross-compiles sm_103a without a
GPU) and exports the same C ABI as the release library."""
import subprocess

from exact_attention_42_gb300.build import LIB_PATH, build


def _exports(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.split() and line.split()[-1].startswith("fa_")}


def test_debug_library_builds_with_the_release_abi():
    release = build()
    debug = build(debug=True)
    assert debug != release and debug.endswith("libfa_debug.so")
    assert _exports(debug) == _exports(release) and "fa_fwd" in _exports(debug)
