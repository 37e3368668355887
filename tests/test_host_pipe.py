"""The ordering logic of the host-buffer forward pass, checked on the CPU.

``host_pipe_check.cpp`` runs the pipeline of ``csrc/host_pipe.h`` against a
fake set of stream operations that models CUDA's stream and event ordering,
with a failure injected at every call in turn: on success every chunk's
kernel follows its copy-in and every copy-out its kernel, and the caller's
stream resumes after the last copy-out; on a failure part-way the error is
reported and the caller's stream still waits for everything queued.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_pipeline_ordering_and_failure_fence(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = tmp_path / "host_pipe_check"
    src = os.path.join(ROOT, "tests", "host_pipe_check.cpp")
    inc = os.path.join(ROOT, "online_softmax_fa_gb300", "csrc")
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-I", inc, src, "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
