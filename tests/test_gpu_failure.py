"""The bounded waits that keep every kernel from hanging, exercised on the GPU
without a fault: a CTA waits on an mbarrier that nothing arrives on (the wait
every decode kernel uses, from pa_device.cuh), the wait gives up after its time
limit and reports it, and the context stays usable for a decode afterwards."""
import ctypes
import os
import shutil
import subprocess

import pytest
import torch

from paritylib import compare, make_inputs, oracle_decode, run_decode, shape

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _build_probe(tmp):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    lib = os.path.join(tmp, "libwaitprobe.so")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "paged_kv_cache_251_gb300", "csrc"),
           os.path.join(HERE, "gpu_wait_probe.cu"), "-o", lib]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return ctypes.CDLL(lib)


def test_a_wait_that_nothing_completes_gives_up_and_the_context_stays_usable(tmp_path):
    probe = _build_probe(str(tmp_path))
    status = ctypes.c_uint(0)
    elapsed = ctypes.c_ulonglong(0)
    assert probe.wait_probe_run(ctypes.byref(status), ctypes.byref(elapsed)) == 0
    assert status.value == 2, "the wait reported a phase that never completed"
    assert 1.9e9 <= elapsed.value <= 10e9, f"gave up after {elapsed.value / 1e9:.2f} s, the limit is 2 s"
    # the same process decodes correctly afterwards
    inp = make_inputs(shape("after", 4, 8, 2, 128, 16, torch.bfloat16, seed=3), [300, 17, 600, 1])
    got, err = run_decode(inp)
    assert err == 0
    compare(got, oracle_decode(inp), torch.bfloat16)
