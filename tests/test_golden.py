"""Golden fixtures (tests/golden/): values the pages print, and worked cases whose exact
output follows from the definition.

problem_constants.txt holds the constants printed by kernelbot amd-mixed-mla 689529
"MLA decode V3" (module constants, docstring) and 690201 "V6c" (docstring). They are
checked against the C header, the input module and the oracle's e4m3 cast.

closed_forms.txt holds one-sequence cases with constant rows and a constant query, whose
output O is worked out by hand in the file. The oracle must reproduce O in float64 on the
CPU; every stage-1 kernel must produce its bf16 rounding exactly, both on the sequence as
written and with its rows repeated until the plan splits it (repeating every row k times
multiplies the softmax's numerator and denominator by k, so O is unchanged). The same
values hold in every KV layout (rows spread over pages in any order, the unused rows of
the last page poisoned), and for every query token of a sequence when each token sees
all of its rows (several tokens, not causal), so those paths are checked against them too.
"""
import os
import re

import numpy as np
import pytest
import torch

import mla_inputs as mi

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")
HEADER = os.path.join(os.path.dirname(HERE), "include", "mla_decode.h")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln for ln in (x.strip() for x in f) if ln and not ln.startswith("#")]


def constants():
    out = {}
    for ln in _lines("problem_constants.txt"):
        name, value = ln.split()[:2]
        out[name] = float(value)
    return out


def cases():
    out = []
    for ln in _lines("closed_forms.txt"):
        name, a, rows, expect, expect_bf16 = ln.split()[:5]
        out.append((name, float(a), [float(x) for x in rows.split(",")], float(expect), float(expect_bf16)))
    return out


CASES = cases()
CASE_IDS = [c[0] for c in CASES]


def make_case(a: float, rows, mode: int, repeat: int = 1) -> mi.Inputs:
    """One sequence: row r holds rows[r % len(rows)] in all 576 dims, the query holds a everywhere."""
    vals = torch.tensor(list(rows) * repeat, dtype=torch.float32)
    kv = vals[:, None].expand(-1, mi.QK_DIM).contiguous()
    q = torch.full((1, mi.HEADS, mi.QK_DIM), a, dtype=torch.float32).to(torch.bfloat16)
    n = kv.shape[0]
    ip = torch.tensor([0, n], dtype=torch.int32)
    ix = torch.arange(n, dtype=torch.int32)
    if mode == mi.MODE_BF16:
        kvq = kv.to(torch.bfloat16)
        assert torch.equal(kvq.float(), kv)
        return mi.Inputs(mode, q, kvq, 1.0, ip, ix, sm_scale=mi.SM_SCALE)
    codes = kv.to(torch.float8_e4m3fn)
    assert torch.equal(codes.float(), kv)  # the fixtures' values are exact in e4m3
    return mi.Inputs(mode, q, codes.view(torch.uint8).contiguous(), 1.0, ip, ix, sm_scale=mi.SM_SCALE)


POISON = 448.0  # the unused rows of a last page: exact in bf16 and e4m3, and far from every case's rows


def make_paged_case(a: float, rows, mode: int, repeat: int, page_size: int, seed: int = 7) -> mi.Inputs:
    """make_case's rows laid out in pages of page_size, in a shuffled page order, with the
    unused rows of the last page holding POISON."""
    base = make_case(a, rows, mode, repeat)
    n = base.kv.shape[0]
    pages = -(-n // page_size)
    perm = torch.randperm(pages, generator=torch.Generator().manual_seed(seed))
    fill = torch.full((1, mi.QK_DIM), POISON)
    fill = fill.to(torch.bfloat16) if mode == mi.MODE_BF16 else fill.to(torch.float8_e4m3fn).view(torch.uint8)
    buf = fill.expand(pages * page_size, -1).clone()
    for p_log in range(pages):
        lo, hi = p_log * page_size, min((p_log + 1) * page_size, n)
        dst = int(perm[p_log]) * page_size
        buf[dst:dst + hi - lo] = base.kv[lo:hi]
    ip = torch.tensor([0, pages], dtype=torch.int32)
    last = torch.tensor([n - (pages - 1) * page_size], dtype=torch.int32)
    return mi.Inputs(mode, base.q, buf.contiguous(), 1.0, ip, perm.to(torch.int32), sm_scale=mi.SM_SCALE,
                     page_size=page_size, kv_last_page_len=last)


# ---------------------------------------------------------------- printed constants

def _header_defines():
    with open(HEADER) as f:
        text = f.read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(MLA_\w+)\s+(\d+)\b", text)}


def test_header_constants_are_the_pages():
    c, d = constants(), _header_defines()
    assert d["MLA_NUM_HEADS"] == c["num_heads"]
    assert d["MLA_NUM_KV_HEADS"] == c["num_kv_heads"]
    assert d["MLA_QK_HEAD_DIM"] == c["qk_head_dim"]
    assert d["MLA_V_HEAD_DIM"] == c["v_head_dim"]
    assert d["MLA_PAGE_SIZE"] == c["page_size"]


def test_input_constants_are_the_pages():
    c = constants()
    assert (mi.HEADS, mi.QK_DIM, mi.V_DIM) == (c["num_heads"], c["qk_head_dim"], c["v_head_dim"])
    assert c["sm_scale"] == 1.0 / 24.0 == 1.0 / np.sqrt(c["qk_head_dim"])
    # the library receives sm_scale as fp32
    assert mi.SM_SCALE == float(np.float32(c["sm_scale"]))
    assert mi.FP8_MAX == c["e4m3_max"]


def test_oracle_e4m3_range_is_the_pages(oracle_lib):
    """The direct fp8 cast of the query (scale 1) saturates at the printed e4m3 range."""
    import oracle
    c = constants()
    table = oracle.e4m3_decode_table(oracle_lib)
    finite = table[np.isfinite(table)]
    assert finite.max() == c["e4m3_max"] and finite.min() == -c["e4m3_max"]
    q = torch.tensor([1000.0, -1000.0, 448.0, 500.0, -464.0, 1.0], dtype=torch.bfloat16)
    got = table[oracle.q_to_e4m3(q, oracle_lib)]
    assert got.tolist() == [448.0, -448.0, 448.0, 448.0, -448.0, c["q_scale"]]


# ---------------------------------------------------------------- closed forms, oracle

def test_fixture_bf16_column_is_the_rounding_of_the_exact_value():
    for name, _, _, expect, expect_bf16 in CASES:
        assert float(torch.tensor(expect, dtype=torch.float64).to(torch.bfloat16)) == expect_bf16, name


@pytest.mark.parametrize("mode", [mi.MODE_BF16, mi.MODE_FP8, mi.MODE_A16W8], ids=["bf16", "fp8", "a16w8"])
@pytest.mark.parametrize("case", CASES, ids=CASE_IDS)
def test_closed_forms_oracle(oracle_lib, case, mode):
    import oracle
    name, a, rows, expect, _ = case
    inp = make_case(a, rows, mode)
    out, _ = oracle.decode(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.sm_scale, mode, inp.kv_scale,
                           lib=oracle_lib)
    np.testing.assert_allclose(out, np.full_like(out, expect), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms, every stage-1 kernel

@pytest.fixture(scope="module")
def mla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_09_gb300 import build
    build.build()
    import mla_decode_attention_09_gb300 as m
    return m


KERNELS = [
    ("bf16", mi.MODE_BF16, {}),
    ("fp8-tcgen05", mi.MODE_FP8, {"fp8_issuers": 2}),
    ("fp8-tcgen05-1issuer", mi.MODE_FP8, {"fp8_issuers": 1}),
    ("fp8-mma", mi.MODE_FP8, {"fp8_kernel": 1}),
    ("a16w8-tcgen05", mi.MODE_A16W8, {}),
    ("a16w8-mma", mi.MODE_A16W8, {"fp8_kernel": 1}),
]


@pytest.mark.gpu
@pytest.mark.parametrize("repeat", [1, 2000], ids=["as-written", "split"])
@pytest.mark.parametrize("kernel", KERNELS, ids=[k[0] for k in KERNELS])
@pytest.mark.parametrize("case", CASES, ids=CASE_IDS)
def test_closed_forms_gpu(mla, case, kernel, repeat):
    name, a, rows, _, expect_bf16 = case
    _, mode, opts = kernel
    inp = make_case(a, rows, mode, repeat)
    d = inp.to("cuda")
    plan = mla.plan(inp.kv_indptr, 0, num_kv_slots=inp.kv.shape[0], **opts)
    if repeat > 1:
        assert plan.info()["num_split_seqs"] == 1  # the sequence goes through the reduce
    out = torch.empty((1, mi.HEADS, mi.V_DIM), dtype=torch.bfloat16, device="cuda")
    mla.decode(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, out, plan=plan,
               sm_scale=d.sm_scale, dtype_mode=mode)
    assert plan.check_error() == 0
    got = out.float().cpu()
    assert torch.equal(got, torch.full_like(got, expect_bf16)), (name, got.min().item(), got.max().item())


@pytest.mark.gpu
@pytest.mark.parametrize("page_size", [3, 8, 16, 64], ids=lambda p: f"pages{p}")
@pytest.mark.parametrize("kernel", KERNELS, ids=[k[0] for k in KERNELS])
@pytest.mark.parametrize("case", CASES, ids=CASE_IDS)
def test_closed_forms_gpu_paged(mla, case, kernel, page_size):
    """Pages in shuffled order, the last page's unused rows poisoned; split over CTAs."""
    name, a, rows, _, expect_bf16 = case
    _, mode, opts = kernel
    inp = make_paged_case(a, rows, mode, 500, page_size)
    d = inp.to("cuda")
    plan = mla.plan_paged(inp.kv_indptr, inp.kv_last_page_len, page_size, num_kv_slots=inp.kv.shape[0], **opts)
    out = torch.empty((1, mi.HEADS, mi.V_DIM), dtype=torch.bfloat16, device="cuda")
    mla.decode_paged(d.q, d.kv, d.kv_scale_tensor("cuda"), d.kv_indptr, d.kv_indices, d.kv_last_page_len, page_size,
                     out, plan=plan, sm_scale=d.sm_scale, dtype_mode=mode)
    assert plan.check_error() == 0
    got = out.float().cpu()
    assert torch.equal(got, torch.full_like(got, expect_bf16)), (name, got.min().item(), got.max().item())


@pytest.mark.gpu
@pytest.mark.parametrize("q_len", [2, 3, 4])
@pytest.mark.parametrize("kernel", KERNELS, ids=[k[0] for k in KERNELS])
@pytest.mark.parametrize("case", CASES, ids=CASE_IDS)
def test_closed_forms_gpu_multi(mla, case, kernel, q_len):
    """q_len tokens that each see every row (not causal): every token's output is O. With an
    even q_len, fp8 on the tensor cores takes the tokens in pairs."""
    name, a, rows, _, expect_bf16 = case
    _, mode, opts = kernel
    inp = make_case(a, rows, mode, 500)
    q = inp.q.expand(q_len, -1, -1).contiguous()
    qo = torch.tensor([0, q_len], dtype=torch.int32)
    d = inp.to("cuda")
    plan = mla.plan_multi(qo, inp.kv_indptr, causal=False, num_kv_slots=inp.kv.shape[0], **opts)
    if mode == mi.MODE_FP8 and "fp8_kernel" not in opts:
        assert plan.token_pairs == (q_len % 2 == 0)
    out = torch.empty((q_len, mi.HEADS, mi.V_DIM), dtype=torch.bfloat16, device="cuda")
    mla.decode_multi(q.cuda(), d.kv, d.kv_scale_tensor("cuda"), qo.cuda(), d.kv_indptr, d.kv_indices, out, plan=plan,
                     sm_scale=d.sm_scale, dtype_mode=mode)
    assert plan.check_error() == 0
    got = out.float().cpu()
    assert torch.equal(got, torch.full_like(got, expect_bf16)), (name, got.min().item(), got.max().item())
