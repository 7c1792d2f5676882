"""GPU test of mla_decode_noalloc, the entry point for callers that may not
allocate device memory: for example a plug-in whose host framework's caching
allocator already holds the GPU's memory, or a serving loop that cannot afford
cudaMalloc's implicit synchronisation. Instead of a plan's workspace it keeps
its work list and partial results in a fixed array inside the library.

Its output must match the regular mla_decode (with a planned workspace) and
the float64 oracle within the parity tolerances, on two calls in a row that
reuse the same fixed array.
This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

TOL = {mi.MODE_BF16: (2e-2, 1e-2), mi.MODE_FP8: (6e-2, 3e-2)}
MLA_ERR_NOALLOC_LIMIT = -11


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_09_gb300 import build
    build.build()
    import mla_decode_attention_09_gb300 as m
    return m


def _close(a: torch.Tensor, b: torch.Tensor, mode: int):
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(x))
    max_abs = float(np.abs(x - y).max()) if x.size else 0.0
    denom = float(np.linalg.norm(y))
    rel = float(np.linalg.norm(x - y) / denom) if denom > 0 else 0.0
    atol, rtol = TOL[mode]
    assert max_abs <= atol and rel <= rtol, (max_abs, rel)


def _noalloc(lib, d: mi.Inputs, ip_host: torch.Tensor, ks, out, status):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mla_decode_noalloc(d.q.data_ptr(), d.kv.data_ptr(), ks.data_ptr(), ip_host.data_ptr(),
                                  d.kv_indptr.data_ptr(), d.kv_indices.data_ptr(), d.batch, d.kv.shape[0],
                                  out.data_ptr(), ctypes.c_float(d.sm_scale), d.mode, status.data_ptr(), stream)


@pytest.mark.parametrize("mode,lengths", [
    (mi.MODE_BF16, [700, 333, 64, 1000, 0, 17]),
    (mi.MODE_FP8, [1024] * 64),
])
def test_noalloc_matches_planned_decode_twice(mla, mode, lengths):
    inp = mi.make_inputs(lengths, mode, seed=77 + mode, permute=True, extra_slots=5)
    d = inp.to("cuda")
    ks = d.kv_scale_tensor("cuda")
    ip_host = inp.kv_indptr.to(torch.int32).contiguous()

    plan = mla.plan(ip_host, 0, num_kv_slots=inp.kv.shape[0])
    ref = mla.decode(d.q, d.kv, ks, d.kv_indptr, d.kv_indices, sm_scale=inp.sm_scale, dtype_mode=mode, plan=plan)
    assert plan.check_error() == 0

    expect, _ = oracle.decode(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.sm_scale, mode, inp.kv_scale)

    lib = mla.load_library()
    status = torch.full((1,), 123, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the second call reuses whatever the first left in the fixed array
        out = torch.full((inp.batch, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, d, ip_host, ks, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(out, ref, mode)
        _close(out, torch.from_numpy(expect), mode)


def test_noalloc_rejects_oversized_requests(mla):
    lib = mla.load_library()
    inp = mi.make_inputs([1] * 1025, mi.MODE_BF16, seed=3)
    d = inp.to("cuda")
    ks = d.kv_scale_tensor("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((inp.batch, 16, 512), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, d, inp.kv_indptr.contiguous(), ks, out, status) == MLA_ERR_NOALLOC_LIMIT
    assert "mla_decode_noalloc" in lib.mla_strerror(MLA_ERR_NOALLOC_LIMIT).decode()
