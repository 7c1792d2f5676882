"""GPU parity of multi-token decode (mla_decode_multi) against the float64 oracle.

Sequence b has q_b query tokens (rows qo_indptr[b] .. of q and out), the last
q_b tokens of the sequence; causally, query token j sees the first
L_b - q_b + j + 1 KV tokens (kernelbot amd-mixed-mla submission 690201 "V6c",
_build_cache: qo_indptr = arange(B+1) * q_seq_len). Tolerances as test_parity.
"""
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


def oracle_multi(inp, q, qo, causal):
    out, _ = oracle.decode_multi(q, inp.kv, qo, inp.kv_indptr, inp.kv_indices, inp.sm_scale, inp.mode, inp.kv_scale,
                                 causal=causal, kv_last_page_len=inp.kv_last_page_len, page_size=inp.page_size)
    return out


def run_multi(mla, inp, q, qo, causal, num_sms=0, **opts):
    d = inp.to("cuda")
    plan = mla.plan_multi(qo, inp.kv_indptr, num_sms, causal=causal, page_size=inp.page_size,
                          kv_last_page_len_host=inp.kv_last_page_len, num_kv_slots=max(inp.kv.shape[0], 1), **opts)
    out = torch.full((int(qo[-1]), 16, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.decode_multi(q.cuda(), d.kv, d.kv_scale_tensor("cuda"), qo.cuda(), d.kv_indptr, d.kv_indices, out, plan=plan,
                     kv_last_page_len=d.kv_last_page_len, sm_scale=inp.sm_scale, dtype_mode=inp.mode)
    return out, plan


LENGTHS = [300, 10, 0, 1, 1000, 77, 2, 129]
Q_LENS = [2, 3, 1, 4, 3, 1, 5, 2]


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("layout", ["rows", "pages8"])
@pytest.mark.parametrize("split", ["whole", "split"])
def test_multi_tokens(mla, mode, k8, causal, layout, split):
    inp = (mi.make_paged_inputs(LENGTHS, 8, mode, seed=300 + mode, permute=True, extra_pages=3) if layout == "pages8"
           else mi.make_inputs(LENGTHS, mode, seed=300 + mode, permute=True, extra_slots=11))
    q, qo = mi.make_query_tokens(Q_LENS, seed=310 + mode, q_std=2.0)
    opts = {} if split == "whole" else {"min_rows_per_split": 16, "granularity": 16}
    out, plan = run_multi(mla, inp, q, qo, causal, num_sms=152 if split == "whole" else 6, **k8, **opts)
    assert plan.check_error() == 0
    if split == "split":
        assert plan.info()["num_split_seqs"] > 0
    compare(out, oracle_multi(inp, q, qo, causal), mode, f"multi {layout} {split} causal={causal}")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("qn", [2, 4])
@pytest.mark.parametrize("split", ["whole", "split"])
@pytest.mark.parametrize("layout", ["rows", "pages64"])
def test_multi_tokens_equal_counts(mla, mode, k8, qn, split, layout):
    # every sequence has qn query tokens: token-parallel plans (one CTA per row range and query
    # token), whole and split into many ranges, over rows or shuffled pages of 64 (page boxes)
    lengths = [1, 130, 640, 1000, 3 * 128 + 5, 7 * 128, 2000]
    inp = (mi.make_paged_inputs(lengths, 64, mode, seed=320 + mode + qn, permute=True, extra_pages=3)
           if layout == "pages64" else mi.make_inputs(lengths, mode, seed=320 + mode + qn, permute=True, extra_slots=7))
    # queries of std 2: a sharper softmax than N(0, 1), where each weight's rounding in P.V shows
    q, qo = mi.make_query_tokens([qn] * len(lengths), seed=330 + qn, q_std=2.0)
    opts = {} if split == "whole" else {"min_rows_per_split": 16, "granularity": 16}
    out, plan = run_multi(mla, inp, q, qo, True, num_sms=152 if split == "whole" else 12, **k8, **opts)
    assert plan.check_error() == 0
    ref = oracle_multi(inp, q, qo, True)
    compare(out, ref, mode, f"equal query counts q={qn} {split}")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_multi_tokens_equal_counts_with_empty_sequences(mla, mode, k8):
    # equal query counts where there are KV rows (a token-parallel plan), and empty sequences
    # holding other numbers of query tokens, whose outputs are zeros
    lengths, q_lens = [0, 300, 0, 200, 5], [3, 2, 5, 2, 2]
    inp = mi.make_inputs(lengths, mode, seed=340 + mode, permute=True, extra_slots=3)
    q, qo = mi.make_query_tokens(q_lens, seed=341, q_std=1.0)
    out, plan = run_multi(mla, inp, q, qo, True, num_sms=9, **k8)
    assert plan.check_error() == 0
    compare(out, oracle_multi(inp, q, qo, True), mode, "equal counts with empty sequences")


def test_multi_query_mismatch_is_reported(mla):
    inp = mi.make_inputs([64, 40], mi.MODE_BF16, seed=8)
    q, qo = mi.make_query_tokens([2, 2], seed=9)
    d = inp.to("cuda")
    plan = mla.plan_multi(qo, inp.kv_indptr)
    bad = torch.tensor([0, 1, 4], dtype=torch.int32, device="cuda")  # device disagrees for sequence 1
    out = torch.zeros((4, 16, 512), dtype=torch.bfloat16, device="cuda")
    mla.decode_multi(q.cuda(), d.kv, None, bad, d.kv_indptr, d.kv_indices, out, plan=plan, dtype_mode=0)
    assert plan.check_error() == -3
    with pytest.raises(mla.MLAError) as e:  # a multi-token plan serves decode_multi only
        mla.decode(d.q, d.kv, None, d.kv_indptr, d.kv_indices, torch.zeros((2, 16, 512), dtype=torch.bfloat16,
                                                                         device="cuda"), plan=plan)
    assert e.value.status == -1


# Speculative-decode shape: fp8, B = 64, kv_len = 8192, two query tokens per sequence. On the
# tensor-core kernel the default plan takes the tokens in pairs; token_pairs = -1 keeps one CTA
# per token.
@pytest.mark.parametrize("k8", FP8_KERNELS + [{"token_pairs": -1}], ids=FP8_KERNEL_IDS + ["tcgen05-per-token"])
def test_multi_full_size(mla, k8):
    inp = mi.make_workload("fp8_b64_l8192")
    q, qo = mi.make_query_tokens([2] * 64, seed=91)
    out, plan = run_multi(mla, inp, q, qo, True, **k8)
    assert plan.check_error() == 0
    # every query row, element by element
    compare(out, oracle_multi(inp, q, qo, True), mi.MODE_FP8, "multi full size")


# ---------------------------------------------------------------- token pairs (fp8, tensor cores)
# Multi-token plans with equal even query counts also hold a token-pair list (option token_pairs,
# on by default): fp8 on the tensor-core kernel takes tokens 2v and 2v+1 of a sequence in one pass
# over their rows (mla_decode_attention_09_gb300/csrc/stage1_umma_pairs.cu).
PAIRS = {"token_pairs": 1}


def pair_items(mla, qo, inp, num_sms, causal, **opts):
    """The host planner's items for the same request (no GPU): checks what a case exercises."""
    return mla.plan_compute_host_multi(qo, inp.kv_indptr, num_sms, causal=causal, page_size=inp.page_size,
                                       kv_last_page_len_host=inp.kv_last_page_len, token_pairs=1, **opts)["items"]


@pytest.mark.parametrize("qn", [2, 4])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("split", ["whole", "split"])
@pytest.mark.parametrize("layout", ["rows", "pages64", "pages8", "pages3"])
def test_token_pairs(mla, qn, causal, split, layout):
    lengths = [1, 2, 3, 130, 640, 1000, 3 * 128 + 5, 7 * 128, 2000, 65]
    mode = mi.MODE_FP8
    seed = 400 + qn + (10 if causal else 0)
    if layout == "rows":
        inp = mi.make_inputs(lengths, mode, seed=seed, permute=True, extra_slots=7)
    else:
        inp = mi.make_paged_inputs(lengths, int(layout[5:]), mode, seed=seed, permute=True, extra_pages=3)
    q, qo = mi.make_query_tokens([qn] * len(lengths), seed=seed + 1, q_std=2.0)
    opts = {} if split == "whole" else {"min_rows_per_split": 16, "granularity": 16}
    num_sms = 152 if split == "whole" else 12
    items = pair_items(mla, qo, inp, num_sms, causal, **opts)
    assert (items[:, 7] >= 0).all()  # a pair plan
    out, plan = run_multi(mla, inp, q, qo, causal, num_sms=num_sms, **PAIRS, **opts)
    assert plan.check_error() == 0
    if split == "split":
        assert plan.info()["num_split_seqs"] > 0
    compare(out, oracle_multi(inp, q, qo, causal), mode, f"token pairs q={qn} {layout} {split} causal={causal}")


@pytest.mark.parametrize("q_std", [1.0, 3.0])
def test_token_pairs_sharp_softmax(mla, q_std):
    lengths = [2000, 1000, 4096, 130, 7]
    inp = mi.make_inputs(lengths, mi.MODE_FP8, seed=430, permute=True, extra_slots=5)
    q, qo = mi.make_query_tokens([2] * len(lengths), seed=431, q_std=q_std)
    out, plan = run_multi(mla, inp, q, qo, True, num_sms=20, **PAIRS)
    assert plan.check_error() == 0
    compare(out, oracle_multi(inp, q, qo, True), mi.MODE_FP8, f"token pairs q_std={q_std}")


def test_token_pairs_edge_items(mla):
    """Pieces where the first token of a pair sees none of the rows (its causal prefix ends at the
    piece's start), whole items where it sees nothing at all, and sequences without rows that hold
    an odd number of query tokens (single-token items writing zeros)."""
    lengths, q_lens = [65, 129, 1, 2, 0, 0], [2, 2, 2, 2, 3, 0]
    inp = mi.make_inputs(lengths, mi.MODE_FP8, seed=440, permute=True, extra_slots=3)
    q, qo = mi.make_query_tokens(q_lens, seed=441, q_std=2.0)
    opts = {"min_rows_per_split": 16, "granularity": 16, "item_cost_rows": -1}
    items = pair_items(mla, qo, inp, 20, True, **opts)
    pair = items[:, 7]
    assert ((pair >= 0) & (pair == items[:, 1]) & (items[:, 2] > items[:, 1]) & (items[:, 3] >= 0)).sum() >= 2
    assert ((pair >= 0) & (pair == items[:, 1]) & (items[:, 2] > items[:, 1]) & (items[:, 3] < 0)).sum() >= 1
    assert (pair < 0).sum() == 3
    out, plan = run_multi(mla, inp, q, qo, True, num_sms=20, **PAIRS, **opts)
    assert plan.check_error() == 0
    compare(out, oracle_multi(inp, q, qo, True), mi.MODE_FP8, "token pairs edge items")


@pytest.mark.parametrize("mode,k8", MODES, ids=MODE_IDS)
def test_token_pair_plans_serve_every_mode(mla, mode, k8):
    # a plan with a token-pair list (the default for equal even counts): fp8 on the tensor-core
    # kernel takes the pairs, every other mode and kernel the ordinary list
    inp = mi.make_inputs([300, 40, 1000, 2], mode, seed=450 + mode, permute=True, extra_slots=5)
    q, qo = mi.make_query_tokens([2, 2, 2, 2], seed=451, q_std=2.0)
    out, plan = run_multi(mla, inp, q, qo, True, num_sms=12, min_rows_per_split=16, granularity=16, **k8)
    assert plan.token_pairs and plan.check_error() == 0
    compare(out, oracle_multi(inp, q, qo, True), mode, f"token-pair plan, mode {mode}")


@pytest.mark.parametrize("qn", [2, 4])
@pytest.mark.parametrize("split", ["whole", "split"])
@pytest.mark.parametrize("layout", ["rows", "pages64"])
def test_multi_tokens_equal_counts_per_token_ctas(mla, qn, split, layout):
    # fp8 on the tensor-core kernel with the token-pair list turned off: one CTA per token
    lengths = [1, 130, 640, 1000, 3 * 128 + 5, 7 * 128, 2000]
    mode = mi.MODE_FP8
    inp = (mi.make_paged_inputs(lengths, 64, mode, seed=460 + qn, permute=True, extra_pages=3)
           if layout == "pages64" else mi.make_inputs(lengths, mode, seed=460 + qn, permute=True, extra_slots=7))
    q, qo = mi.make_query_tokens([qn] * len(lengths), seed=470 + qn, q_std=2.0)
    opts = {} if split == "whole" else {"min_rows_per_split": 16, "granularity": 16}
    out, plan = run_multi(mla, inp, q, qo, True, num_sms=152 if split == "whole" else 12, token_pairs=-1, **opts)
    assert not plan.token_pairs and plan.check_error() == 0
    compare(out, oracle_multi(inp, q, qo, True), mode, f"per-token CTAs q={qn} {split}")


@pytest.mark.parametrize("qn", [2, 4])
def test_token_pairs_full_size(mla, qn):
    inp = mi.make_workload("fp8_b64_l8192")
    q, qo = mi.make_query_tokens([qn] * 64, seed=92 + qn)
    out, plan = run_multi(mla, inp, q, qo, True, **PAIRS)
    assert plan.check_error() == 0
    compare(out, oracle_multi(inp, q, qo, True), mi.MODE_FP8, f"token pairs full size q={qn}")


def test_token_pairs_out_of_range_index_is_reported(mla):
    inp = mi.make_inputs([300, 200], mi.MODE_FP8, seed=4)
    inp.kv_indices[7] = inp.kv.shape[0] + 5
    q, qo = mi.make_query_tokens([2, 2], seed=5)
    out, plan = run_multi(mla, inp, q, qo, True)
    assert plan.token_pairs
    assert plan.check_error() == -8   # MLA_ERR_INDEX; the bad row was read as zeros
    assert torch.isfinite(out.float()).all()


def test_token_pairs_query_mismatch_is_reported(mla):
    # the device qo_indptr disagrees with the plan: the pair kernel checks both rows of a pair and
    # skips the items instead of reading another sequence's query
    inp = mi.make_inputs([64, 40], mi.MODE_FP8, seed=8)
    q, qo = mi.make_query_tokens([2, 2], seed=9)
    d = inp.to("cuda")
    plan = mla.plan_multi(qo, inp.kv_indptr, num_kv_slots=inp.kv.shape[0])
    assert plan.token_pairs
    bad = torch.tensor([0, 1, 4], dtype=torch.int32, device="cuda")
    out = torch.zeros((4, 16, 512), dtype=torch.bfloat16, device="cuda")
    mla.decode_multi(q.cuda(), d.kv, d.kv_scale_tensor("cuda"), bad, d.kv_indptr, d.kv_indices, out, plan=plan,
                     dtype_mode=mi.MODE_FP8)
    assert plan.check_error() == -3   # MLA_ERR_PLAN_MISMATCH
    assert not out.float().abs().any()  # nothing was written
