"""The C ABI from plain C: tests/c_abi/host_calls.c includes include/dllm.h,
compiles as pedantic C99 with warnings as errors, links libdllm.so and runs
the host entry points against hand-computed values (no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_calls_from_plain_c(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler on this machine")
    import denoise_step_token_gb300 as dllm
    dllm.load()   # the library is built and loadable
    lib_dir = os.path.dirname(os.path.abspath(dllm.__file__))
    exe = str(tmp_path / "host_calls")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "host_calls.c"), "-L", lib_dir, "-ldllm",
           "-Wl,-rpath," + lib_dir, "-lm", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "ok" in run.stdout
