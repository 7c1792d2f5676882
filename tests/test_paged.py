"""GPU parity of the paged layout (mla_decode_paged) against the float64 oracle.

The KV buffer is viewed as [num_pages, page_size, 576]; kv_indptr counts pages,
kv_indices holds page ids and kv_last_page_len the tokens of each last page
(kernelbot amd-mixed-mla submission 641982 "v86", _run_a8w8). Tolerances as in
test_parity: bf16 2e-2 / 1e-2, fp8 6e-2 / 3e-2 (max-abs / relative L2).
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle
from test_parity import FP8_KERNEL_IDS, FP8_KERNELS, MODE_IDS, MODES, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_09_gb300 import build
    build.build()
    import mla_decode_attention_09_gb300 as m
    return m


def oracle_paged(inp: mi.Inputs, seq_ids=None):
    out, _ = oracle.decode_paged(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.kv_last_page_len, inp.page_size,
                                 inp.sm_scale, inp.mode, inp.kv_scale, seq_ids=seq_ids)
    return out


def run_paged(mla, inp: mi.Inputs, num_sms=0, **opts):
    d = inp.to("cuda")
    plan = mla.plan_paged(inp.kv_indptr, inp.kv_last_page_len, inp.page_size, num_sms,
                          num_kv_slots=max(inp.kv.shape[0], 1), **opts)
    out = torch.full((inp.batch, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.decode_paged(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, d.kv_last_page_len,
                     inp.page_size, out, sm_scale=inp.sm_scale, dtype_mode=inp.mode, plan=plan)
    return out, plan


LENGTHS = [1, 15, 17, 63, 64, 65, 1000, 0, 129, 2, 300]


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("ps", [2, 3, 8, 16, 24, 32, 64, 128, 256])
@pytest.mark.parametrize("order", ["contiguous", "shuffled"])
def test_paged_lengths(mla, mode, k8, ps, order):
    inp = mi.make_paged_inputs(LENGTHS, ps, mode, seed=200 + ps + mode, permute=order == "shuffled", extra_pages=5)
    out, plan = run_paged(mla, inp, num_sms=7, min_rows_per_split=16, granularity=16, **k8)
    assert plan.check_error() == 0
    assert plan.info()["num_split_seqs"] > 0
    compare(out, oracle_paged(inp), mode, f"paged ps={ps} {order}")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_paged_whole_sequences_default_plan(mla, mode, k8):
    inp = mi.make_paged_inputs([3000, 1, 257, 4096], 8, mode, seed=31, permute=True)
    out, plan = run_paged(mla, inp, **k8)
    assert plan.check_error() == 0
    compare(out, oracle_paged(inp), mode, "paged default plan")


@pytest.mark.parametrize("k8", FP8_KERNELS, ids=FP8_KERNEL_IDS)
@pytest.mark.parametrize("ps", [8, 16, 32, 64])
@pytest.mark.parametrize("checked", [True, False])
def test_paged_unused_rows_of_last_pages_are_ignored(mla, k8, ps, checked):
    # Pages of 16..64 rows arrive as whole pages, so the rows of a last page past
    # kv_last_page_len are read too. Poison them with e4m3 NaN codes (0x7f): the
    # output must not see them. Tails of 1, ps - 1 and a few rows; the default plan
    # (tiles start on page boundaries), with and without the pool size.
    inp = mi.make_paged_inputs([3 * ps + 5, 1, 5 * ps - 1, 130, 2 * ps], ps, mi.MODE_FP8, seed=40 + ps,
                               permute=True, extra_pages=3)
    for b in range(inp.batch):
        lo, hi = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
        if hi > lo:
            page, used = int(inp.kv_indices[hi - 1]), int(inp.kv_last_page_len[b])
            inp.kv[page * ps + used:(page + 1) * ps] = 0x7F
    d = inp.to("cuda")
    plan = mla.plan_paged(inp.kv_indptr, inp.kv_last_page_len, ps,
                          num_kv_slots=inp.kv.shape[0] if checked else 0, **k8)
    out = torch.full((inp.batch, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.decode_paged(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, d.kv_last_page_len, ps,
                     out, sm_scale=inp.sm_scale, dtype_mode=inp.mode, plan=plan)
    assert plan.check_error() == 0
    compare(out, oracle_paged(inp), mi.MODE_FP8, f"poisoned last pages ps={ps}")


@pytest.mark.parametrize("k8", FP8_KERNELS, ids=FP8_KERNEL_IDS)
def test_paged_last_page_mismatch_is_reported(mla, k8):
    inp = mi.make_paged_inputs([40, 33], 8, mi.MODE_FP8, seed=3)
    d = inp.to("cuda")
    plan = mla.plan_paged(inp.kv_indptr, inp.kv_last_page_len, 8, **k8)
    lp = d.kv_last_page_len.clone()
    lp[1] = 2  # device disagrees with the plan for sequence 1
    out = torch.zeros((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    mla.decode_paged(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, lp, 8, out,
                     sm_scale=inp.sm_scale, dtype_mode=inp.mode, plan=plan)
    assert plan.check_error() == -3
    # the agreeing sequence is still decoded
    compare(out[:1], oracle_paged(inp, seq_ids=[0]), mi.MODE_FP8, "paged mismatch, other sequence")


@pytest.mark.parametrize("k8", FP8_KERNELS, ids=FP8_KERNEL_IDS)
def test_paged_out_of_range_page_is_reported(mla, k8):
    inp = mi.make_paged_inputs([40, 33], 8, mi.MODE_FP8, seed=4)
    inp.kv_indices[2] = inp.kv.shape[0] // 8  # one past the last page
    d = inp.to("cuda")
    plan = mla.plan_paged(inp.kv_indptr, inp.kv_last_page_len, 8, num_kv_slots=inp.kv.shape[0], **k8)
    out = torch.zeros((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    mla.decode_paged(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, d.kv_last_page_len, 8, out,
                     sm_scale=inp.sm_scale, dtype_mode=inp.mode, plan=plan)
    assert plan.check_error() == -8


def test_paged_and_row_plans_are_not_interchangeable(mla):
    inp = mi.make_paged_inputs([40, 33], 8, mi.MODE_BF16, seed=5)
    d = inp.to("cuda")
    out = torch.zeros((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    paged = mla.plan_paged(inp.kv_indptr, inp.kv_last_page_len, 8)
    rows = mla.plan(inp.kv_indptr)
    with pytest.raises(mla.MLAError) as e:
        mla.decode(d.q, d.kv, None, d.kv_indptr, d.kv_indices, out, plan=paged)
    assert e.value.status == -1
    with pytest.raises(mla.MLAError) as e:
        mla.decode_paged(d.q, d.kv, None, d.kv_indptr, d.kv_indices, d.kv_last_page_len, 8, out, plan=rows)
    assert e.value.status == -1
    with pytest.raises(mla.MLAError) as e:  # page size differs from the plan's
        mla.decode_paged(d.q, d.kv, None, d.kv_indptr, d.kv_indices, d.kv_last_page_len, 4, out, plan=paged)
    assert e.value.status == -1


# The pages' paged configuration for long sequences: fp8, page_size 8, pages in order
# (kv_indices = arange, every last page full), B = 64, kv_len = 8192; and shuffled pages.
@pytest.mark.parametrize("order", ["contiguous", "shuffled"])
def test_paged_full_size(mla, order):
    lengths = [8192] * 64
    inp = mi.make_paged_inputs(lengths, 8, mi.MODE_FP8, seed=77, permute=order == "shuffled")
    out, plan = run_paged(mla, inp)
    assert plan.check_error() == 0
    # every sequence, element by element
    compare(out, oracle_paged(inp), mi.MODE_FP8, f"paged full size {order}")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("ps", [16, 64])
def test_half_shuffled_pages(mla, mode, k8, ps):
    """Page order kept for half of the pages and shuffled for the rest: tiles inside runs of pages
    in order load as one box, the others as page boxes (or row copies where a page is out of step)."""
    lengths = [1500, 700, 2000, 130]
    inp = mi.make_paged_inputs(lengths, ps, mode, seed=77, extra_pages=3)
    ix = inp.kv_indices.clone()
    g = torch.Generator().manual_seed(5)
    n = ix.numel()
    pick = torch.nonzero(torch.rand(n, generator=g) < 0.5).flatten()
    ix[pick] = ix[pick][torch.randperm(pick.numel(), generator=g)]
    inp.kv_indices = ix
    out, _ = run_paged(mla, inp, **k8)
    compare(out, oracle_paged(inp), mode, f"half-shuffled pages of {ps}")
