"""GPU parity: the CUDA library (through the C ABI) against the float64 oracle,
element by element, on the same seeded inputs.

Tolerances (max-abs error, relative L2 error of the whole output):
bf16 2e-2 / 1e-2, fp8 6e-2 / 3e-2. a16w8 (bf16 Q x e4m3 KV) is held to the bf16
bound: its query is exact (two e4m3 terms of a scaled copy on the tensor-memory
kernel, f16 on the warp-level one), and its weights keep about 8 (e4m3 hi + lo)
or 11 (f16) significant bits.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

TOL = {mi.MODE_BF16: (2e-2, 1e-2), mi.MODE_FP8: (6e-2, 3e-2), mi.MODE_A16W8: (2e-2, 1e-2)}


@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_09_gb300 import build
    build.build()
    import mla_decode_attention_09_gb300 as m
    return m


# fp8 stage-1 kernels: the tcgen05 / TMA kernel (default) in both of its MMA
# issue instances, and the warp-level mma.sync kernel
KERNELS = {"tcgen05": {"fp8_issuers": 2}, "tcgen05-1issuer": {"fp8_issuers": 1}, "mma": {"fp8_kernel": 1}}
FP8_KERNELS = list(KERNELS.values())
FP8_KERNEL_IDS = list(KERNELS)


def run(mla, inp: mi.Inputs, num_sms=0, **opts):
    d = inp.to("cuda")
    plan = mla.plan(inp.kv_indptr, num_sms, num_kv_slots=max(inp.kv.shape[0], 1), **opts)
    out = torch.full((inp.batch, 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.decode(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, out, sm_scale=inp.sm_scale,
               dtype_mode=inp.mode, plan=plan)
    assert plan.check_error() == 0
    return out, plan


def compare(got: torch.Tensor, ref: np.ndarray, mode: int, what: str = ""):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel_l2 = float(np.linalg.norm(g - ref) / denom) if denom > 0 else float(np.linalg.norm(g - ref))
    atol, rtol = TOL[mode]
    assert max_abs <= atol and rel_l2 <= rtol, f"{what}: max_abs={max_abs:.3e} rel_l2={rel_l2:.3e}"
    return max_abs, rel_l2


def oracle_out(inp: mi.Inputs, seq_ids=None):
    out, _ = oracle.decode(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.sm_scale, inp.mode, inp.kv_scale,
                           seq_ids=seq_ids)
    return out


ODD = [1, 15, 17, 63, 64, 65, 1000, 0, 129, 2]


# a16w8 runs on the tensor-memory kernel by default (the bf16 query as two e4m3 terms) and on the
# warp-level kernel with fp8_kernel = 1
MODES = ([(mi.MODE_BF16, {})] + [(mi.MODE_FP8, k) for k in FP8_KERNELS]
         + [(mi.MODE_A16W8, {}), (mi.MODE_A16W8, {"fp8_kernel": 1})])
MODE_IDS = ["bf16"] + [f"fp8-{k}" for k in FP8_KERNEL_IDS] + ["a16w8-tcgen05", "a16w8-mma"]


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("split", ["whole", "split"])
def test_odd_lengths(mla, mode, k8, split):
    inp = mi.make_inputs(ODD, mode, seed=100 + mode, permute=True, extra_slots=37)
    opts = {} if split == "whole" else {"min_rows_per_split": 16, "granularity": 16}
    out, plan = run(mla, inp, num_sms=152 if split == "whole" else 5, **k8, **opts)
    info = plan.info()
    if split == "split":
        assert info["num_split_seqs"] > 0
    compare(out, oracle_out(inp), mode, f"odd lengths {split}")


def mixed_tile_inputs(mode: int) -> mi.Inputs:
    """Rows in order, except that every third 128-row chunk of a sequence has its rows shuffled among
    themselves, and the chunk after it has one row moved to a spare slot: box-loaded tiles and
    row-copied tiles alternate within each sequence."""
    lengths = [1500, 700, 2000, 130, 5]
    inp = mi.make_inputs(lengths, mode, seed=321, extra_slots=5)
    ix = inp.kv_indices.clone()
    g = torch.Generator().manual_seed(9)
    ip = inp.kv_indptr.tolist()
    for b in range(len(lengths)):
        for k, t0 in enumerate(range(ip[b], ip[b + 1], 128)):
            t1 = min(t0 + 128, ip[b + 1])
            if k % 3 == 1:
                ix[t0:t1] = ix[t0:t1][torch.randperm(t1 - t0, generator=g)]
            elif k % 3 == 2 and t1 - t0 > 1:
                ix[t0 + (t1 - t0) // 2] = inp.kv.shape[0] - 1 - (k % 5)
    inp.kv_indices = ix
    return inp


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("split", ["whole", "split"])
def test_mixed_box_and_row_copied_tiles(mla, mode, k8, split):
    inp = mixed_tile_inputs(mode)
    opts = {} if split == "whole" else {"min_rows_per_split": 64}
    out, plan = run(mla, inp, num_sms=152 if split == "whole" else 7, **k8, **opts)
    if split == "split":
        assert plan.info()["num_split_seqs"] > 0
    compare(out, oracle_out(inp), mode, f"mixed tiles {split}")


@pytest.mark.parametrize("k8", [{}, {"fp8_kernel": 1}], ids=["a16w8-tcgen05", "a16w8-mma"])
@pytest.mark.parametrize("q_std", [1.0, 2.0])
def test_a16w8_keeps_the_bf16_query(mla, k8, q_std):
    # The same inputs decoded as fp8 (query cast to e4m3) differ from the a16w8 definition by more
    # than the bf16 tolerance, so a kernel that rounded the query to one e4m3 term would fail here.
    inp = mi.make_inputs([300, 1000, 37, 2048], mi.MODE_A16W8, seed=700, permute=True, extra_slots=9, q_std=q_std)
    ref = oracle_out(inp)
    as_fp8, _ = oracle.decode(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.sm_scale, mi.MODE_FP8, inp.kv_scale)
    gap = np.linalg.norm(as_fp8 - ref) / np.linalg.norm(ref)
    assert gap > 2 * TOL[mi.MODE_A16W8][1], f"test inputs do not separate the modes (rel-L2 {gap:.2e})"
    out, plan = run(mla, inp, num_sms=20, **k8)
    assert plan.check_error() == 0
    compare(out, ref, mi.MODE_A16W8, f"a16w8 q_std={q_std}")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_one_long_sequence_many_splits(mla, mode, k8):
    inp = mi.make_inputs([5003], mode, seed=7)
    out, plan = run(mla, inp, num_sms=152, min_rows_per_split=16, granularity=16, **k8)
    assert plan.info()["num_partial_slots"] > 100
    compare(out, oracle_out(inp), mode, "one long sequence")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_many_short_sequences(mla, mode, k8):
    # 3000 sequences of 0..200 rows at random slots: many items per CTA, with empty and
    # one-row sequences among them; every sequence is compared
    rng = np.random.default_rng(77 + mode)
    lengths = [int(x) for x in rng.integers(0, 201, 3000)]
    lengths[5] = 0
    lengths[6] = 1
    inp = mi.make_inputs(lengths, mode, seed=400 + mode, permute=True)
    out, plan = run(mla, inp, **k8)
    assert plan.check_error() == 0
    compare(out, oracle_out(inp), mode, "many short sequences")


@pytest.mark.parametrize("mode,k8", [(mi.MODE_BF16, {}), (mi.MODE_FP8, {})], ids=["bf16", "fp8-tcgen05"])
def test_one_very_long_sequence(mla, mode, k8):
    # 300,000 rows in one sequence, split over every CTA by the default plan
    inp = mi.make_inputs([300_000], mode, seed=500 + mode)
    out, plan = run(mla, inp, **k8)
    assert plan.info()["num_ctas"] >= 100
    compare(out, oracle_out(inp), mode, "one very long sequence")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_degenerate_inputs(mla, mode, k8):
    # sequence 0: zero query (every score equal: the mean of the value rows); sequence 1: all its
    # KV rows identical (that row); sequences 2-3: one row each (the row itself); split plans
    inp = mi.make_inputs([700, 300, 1, 1], mode, seed=600 + mode)
    inp.q[0] = 0
    rows = inp.kv_indices[int(inp.kv_indptr[1]):int(inp.kv_indptr[2])].long()
    inp.kv[rows] = inp.kv[rows[0]].clone()
    out, plan = run(mla, inp, num_sms=7, min_rows_per_split=16, granularity=16, **k8)
    assert plan.check_error() == 0
    ref = oracle_out(inp)
    compare(out, ref, mode, "degenerate inputs")
    # the closed forms hold for the oracle's values too (exact up to its float64 rounding)
    kv = inp.kv.float() if mode == mi.MODE_BF16 else None
    if kv is not None:
        r0 = inp.kv_indices[:700].long()
        assert np.allclose(ref[0], kv[r0, :512].double().mean(0).numpy()[None, :], atol=1e-9)
        assert np.allclose(ref[1], kv[rows[0], :512].double().numpy()[None, :], atol=1e-9)


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_peaked_scores(mla, mode, k8):
    # larger query norm -> sharply peaked softmax; exercises the running-max rescale
    inp = mi.make_inputs([300, 1, 77, 2000], mode, seed=9, q_std=6.0)
    out, _ = run(mla, inp, num_sms=4, min_rows_per_split=16, **k8)
    compare(out, oracle_out(inp), mode, "peaked")


@pytest.mark.parametrize("k8", FP8_KERNELS, ids=FP8_KERNEL_IDS)
@pytest.mark.parametrize("q_std", [2.0, 3.0])
@pytest.mark.parametrize("split", ["whole", "split"])
def test_fp8_sharp_softmax(mla, k8, q_std, split):
    # queries of std 2 and 3 give scores of std ~2 and ~3: a few rows carry most of the
    # weight, so every weight's rounding shows in the output (one e4m3 term per weight
    # left the fp8 bound here; the hi + lo pair and f16 P stay inside it)
    inp = mi.make_inputs(ODD + [3000, 333], mi.MODE_FP8, seed=700 + int(q_std), permute=True, extra_slots=21,
                         q_std=q_std)
    opts = {} if split == "whole" else {"min_rows_per_split": 16, "granularity": 16}
    out, _ = run(mla, inp, num_sms=152 if split == "whole" else 9, **k8, **opts)
    compare(out, oracle_out(inp), mi.MODE_FP8, f"fp8 q_std={q_std} {split}")


@pytest.mark.parametrize("k8", FP8_KERNELS, ids=FP8_KERNEL_IDS)
def test_fp8_query_cast_saturates(mla, k8):
    # entries beyond +-448 exercise the saturating direct cast of the query
    inp = mi.make_inputs([40, 9], mi.MODE_FP8, seed=13)
    inp.q[0, 3, :50] = 1000.0
    inp.q[1, 5, 100:140] = -600.0
    out, _ = run(mla, inp, **k8)
    ref = oracle_out(inp)
    compare(out, ref, mi.MODE_FP8, "fp8 saturation")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_stage1_plus_reduce_equals_decode_and_is_deterministic(mla, mode, k8):
    inp = mi.make_inputs([700, 333, 64], mode, seed=21)
    a, plan = run(mla, inp, num_sms=6, min_rows_per_split=16, **k8)
    b, _ = run(mla, inp, num_sms=6, min_rows_per_split=16, **k8)
    assert torch.equal(a, b)
    d = inp.to("cuda")
    c = torch.empty_like(a)
    mla.decode_stage1(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, c, plan=plan,
                      sm_scale=inp.sm_scale, dtype_mode=mode)
    mla.decode_reduce(c, plan=plan)
    assert plan.check_error() == 0
    assert torch.equal(a, c)


def test_empty_batch_and_empty_sequences(mla):
    inp = mi.make_inputs([0, 0, 0], mi.MODE_BF16, seed=1, extra_slots=4)
    out, _ = run(mla, inp)
    assert torch.count_nonzero(out) == 0
    inp0 = mi.make_inputs([], mi.MODE_FP8, seed=1, extra_slots=4)
    out0, _ = run(mla, inp0)
    assert out0.shape == (0, 16, 512)


def test_plan_mismatch_is_reported(mla):
    inp = mi.make_inputs([100, 50], mi.MODE_BF16, seed=3)
    d = inp.to("cuda")
    plan = mla.plan(torch.tensor([0, 60, 150], dtype=torch.int32), 0, num_kv_slots=inp.kv.shape[0])
    out = torch.zeros((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    mla.decode(d.q, d.kv, None, d.kv_indptr, d.kv_indices, out, dtype_mode=0, plan=plan)
    assert plan.check_error() == -3   # MLA_ERR_PLAN_MISMATCH
    assert plan.check_error() == 0    # cleared after reading


@pytest.mark.parametrize("mode,k8", [(mi.MODE_FP8, k) for k in FP8_KERNELS] + [(mi.MODE_A16W8, {})],
                         ids=[f"fp8-{k}" for k in FP8_KERNEL_IDS] + ["a16w8-tcgen05"])
def test_out_of_range_index_is_reported(mla, mode, k8):
    inp = mi.make_inputs([30, 20], mode, seed=4)
    inp.kv_indices[7] = inp.kv.shape[0] + 5
    d = inp.to("cuda")
    plan = mla.plan(inp.kv_indptr, 0, num_kv_slots=inp.kv.shape[0], **k8)
    out = torch.zeros((2, 16, 512), dtype=torch.bfloat16, device="cuda")
    mla.decode(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, out, plan=plan, dtype_mode=mode)
    assert plan.check_error() == -8   # MLA_ERR_INDEX; the bad row was read as zeros
    assert torch.isfinite(out.float()).all()


def test_host_argument_errors(mla):
    inp = mi.make_inputs([10], mi.MODE_BF16, seed=2).to("cuda")
    plan = mla.plan(inp.kv_indptr.cpu(), 0)
    out = torch.empty((1, 16, 512), dtype=torch.bfloat16, device="cuda")
    lib = mla.load_library()
    s = torch.cuda.current_stream().cuda_stream
    args = [inp.q.data_ptr(), inp.kv.data_ptr(), None, inp.kv_indptr.data_ptr(), inp.kv_indices.data_ptr(),
            out.data_ptr(), 0.04, 0, plan.handle, s]
    bad = list(args); bad[7] = 5
    assert lib.mla_decode(*bad) == -2            # dtype
    bad = list(args); bad[0] = inp.q.data_ptr() + 2
    assert lib.mla_decode(*bad) == -6            # alignment
    bad = list(args); bad[7] = 1
    assert lib.mla_decode(*bad) == -1            # fp8 without kv_scale
    bad = list(args); bad[7] = 2
    assert lib.mla_decode(*bad) == -1            # a16w8 without kv_scale
    assert lib.mla_decode(*args) == 0
    assert plan.check_error() == 0


# ---------------------------------------------------------------- full-size workloads

# the default plan (no options) is the launch configuration the benchmark times
FULL = ([(n, "default") for n in mi.WORKLOADS] + [(n, k) for n, w in mi.WORKLOADS.items() if w.mode == mi.MODE_FP8
                                                  for k in ("tcgen05-1issuer", "mma")]
        + [(n, k) for n in mi.EXTRA_WORKLOADS for k in ("default", "mma")])

_FULL_REF = {}


def full_reference(name: str, inp: mi.Inputs) -> np.ndarray:
    """The oracle over every sequence of a full-size workload (computed once per workload)."""
    if name not in _FULL_REF:
        _FULL_REF.clear()  # one workload's reference held at a time
        _FULL_REF[name] = oracle_out(inp)
    return _FULL_REF[name]


@pytest.mark.parametrize("name,kernel", FULL, ids=[f"{n}-{k}" for n, k in FULL])
def test_full_size_workload(mla, name, kernel):
    # every sequence, element by element, against the oracle
    inp = mi.make_workload(name)
    out, plan = run(mla, inp, **KERNELS.get(kernel, {}))
    compare(out, full_reference(name, inp), inp.mode, name)


@pytest.mark.parametrize("k8", FP8_KERNELS, ids=FP8_KERNEL_IDS)
@pytest.mark.parametrize("q_std", [2.0, 3.0])
def test_full_size_fp8_sharp_softmax(mla, k8, q_std):
    # the fp8 B = 64, kv_len = 8192 shape with queries of std 2 and 3, every sequence compared
    w = mi.get_workload("fp8_b64_l8192")
    inp = mi.make_inputs(mi.workload_lengths(w), w.mode, w.seed + 40 + int(q_std), q_std=q_std)
    out, _ = run(mla, inp, **k8)
    compare(out, full_reference(f"fp8_b64_l8192-q{q_std}", inp), mi.MODE_FP8, f"full size q_std={q_std}")
