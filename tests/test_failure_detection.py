"""Failure detection without a GPU fault: a bounded wait on an mbarrier that
nothing signals gives up after its limit and reports MLA_ERR_TIMEOUT; the
context stays usable. Host-side failures (bad plans, bad indices) are covered
in the parity tests."""
import ctypes
import os
import shutil
import subprocess

import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.gpu
def test_bounded_wait_times_out_and_reports(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = tmp_path / "libwait.so"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-I", os.path.join(ROOT, "mla_decode_attention_09_gb300", "csrc"),
                    os.path.join(HERE, "gpu_selftest", "bounded_wait.cu"), "-o", str(so)], check=True)
    lib = ctypes.CDLL(str(so))
    lib.run_wait_on_silent_barrier.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    limit_ns = 5_000_000  # 5 ms
    assert lib.run_wait_on_silent_barrier(limit_ns, status.data_ptr(), waited.data_ptr()) == 0
    assert int(status.item()) == -5
    assert limit_ns <= int(waited.item()) < 1_000_000_000
    # the context is still usable
    x = torch.arange(10, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 45.0
