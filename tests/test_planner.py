"""CPU tests of the host split-KV planner (through the C ABI's host-only entry)."""
import numpy as np
import pytest

import mla_decode_attention_09_gb300 as mla


def _check_plan(lengths, num_sms, **opts):
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    r = mla.plan_compute_host(ip, num_sms, **opts)
    items, wip, red = r["items"], r["work_indptr"], r["reduce"]
    G = opts.get("granularity", 128)
    min_split = opts.get("min_rows_per_split", 128)
    cpsm = opts.get("ctas_per_sm", 1)
    total = int(ip[-1])
    # CTA ranges: CSR over the item list, at most num_sms * ctas_per_sm CTAs
    assert wip[0] == 0 and wip[-1] == len(items) and np.all(np.diff(wip) >= 0)
    assert 1 <= r["num_ctas"] <= num_sms * cpsm or (len(lengths) == 0 and r["num_ctas"] <= 1)
    # every row of every sequence covered exactly once, in order
    by_seq = {}
    for b, t0, t1, slot, L in items:
        assert 0 <= b < len(lengths) and L == lengths[b]
        by_seq.setdefault(int(b), []).append((int(t0), int(t1), int(slot)))
    assert sorted(by_seq) == list(range(len(lengths)))
    next_slot = 0
    red_map = {int(b): (int(s0), int(n)) for b, s0, n in red}
    for b, parts in by_seq.items():
        L = lengths[b]
        pos = 0
        for t0, t1, _ in parts:
            assert t0 == pos and t1 >= t0
            if t1 != L:
                assert t1 % G == 0, "cuts fall on the granularity"
            pos = t1
        assert pos == L
        if len(parts) == 1:
            assert parts[0][2] == -1 and b not in red_map
        else:
            s0, n = red_map[b]
            assert n == len(parts) and [p[2] for p in parts] == list(range(s0, s0 + n))
            assert s0 == next_slot
            next_slot += n
            assert all(t1 > t0 for t0, t1, _ in parts), "no empty partial"
    assert next_slot == r["num_slots"]
    # load balance in granules (G rows; a sequence's last granule may be shorter): every CTA
    # holds floor or ceil of (granules / CTAs), and no CTA more than the target
    if total:
        max_ctas = num_sms * cpsm
        U = sum(-(-L // G) for L in lengths)
        target = max(-(-U // max_ctas), -(-min_split // G))
        gran = [sum(-(-int(items[i, 2] - items[i, 1]) // G) for i in range(wip[c], wip[c + 1]))
                for c in range(r["num_ctas"])]
        assert sum(gran) == U
        assert max(gran) <= target
        assert max(gran) - min(gran) <= 1
        rows = [sum(int(items[i, 2] - items[i, 1]) for i in range(wip[c], wip[c + 1])) for c in range(r["num_ctas"])]
        assert sum(rows) == total
    return r


@pytest.mark.parametrize("lengths,num_sms", [
    ([1024] * 4, 152), ([8192] * 4, 152), ([1024] * 64, 152), ([8192] * 64, 152),
    ([1], 152), ([0], 152), ([0, 5, 0], 4), ([17, 15, 1000, 63, 64, 65], 3), ([1000], 1),
    ([4096] * 3, 2), (list(range(0, 300, 7)), 5),
])
def test_plan_invariants(lengths, num_sms):
    _check_plan(lengths, num_sms)


def test_plan_invariants_random():
    rng = np.random.default_rng(0)
    for _ in range(300):
        B = int(rng.integers(1, 40))
        lengths = [int(x) for x in rng.integers(0, 3000, B)]
        if rng.random() < 0.2:
            lengths[int(rng.integers(0, B))] = 0
        opts = {}
        if rng.random() < 0.5:
            opts["min_rows_per_split"] = int(rng.choice([16, 64, 256, 1024]))
        if rng.random() < 0.3:
            opts["granularity"] = int(rng.choice([1, 8, 16, 64, 128]))
        _check_plan(lengths, int(rng.integers(1, 160)), **opts)


def test_plan_headline_shapes():
    # B=64 x 8192 over 152 SMs: every SM busy, each sequence split in 2-4 chunks
    r = _check_plan([8192] * 64, 152)
    assert r["num_ctas"] == 152
    assert 64 * 2 <= r["num_slots"] <= 64 * 4
    # B=4 x 1024 bf16: small problem, one 128-row tile per CTA (the minimum chunk)
    r = _check_plan([1024] * 4, 152)
    assert r["num_ctas"] == 32
    # every CTA gets 26 or 27 of the 4096 tiles of B=64 x 8192
    r = mla.plan_compute_host(np.arange(65, dtype=np.int32) * 8192, 152)
    tiles = [sum(-(-int(t1 - t0) // 128) for _, t0, t1, _, _ in r["items"][r["work_indptr"][c]:r["work_indptr"][c + 1]])
             for c in range(152)]
    assert set(tiles) <= {26, 27}


def test_plan_rejects_bad_indptr():
    with pytest.raises(mla.MLAError) as e:
        mla.plan_compute_host(np.array([0, 5, 3], dtype=np.int32), 4)
    assert e.value.status == -10
    with pytest.raises(mla.MLAError) as e:
        mla.plan_compute_host(np.array([1, 5], dtype=np.int32), 4)
    assert e.value.status == -10
    with pytest.raises(mla.MLAError) as e:
        mla.plan_compute_host(np.array([0, 5], dtype=np.int32), 0)
    assert e.value.status == -1


# ---------------------------------------------------------------- paged layout

def _paged_layout(lengths, ps):
    pages = [(L + ps - 1) // ps for L in lengths]
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(pages)
    last = np.array([L - (p - 1) * ps if p else 1 for L, p in zip(lengths, pages)], dtype=np.int32)
    return ip, last


@pytest.mark.parametrize("ps", [1, 2, 3, 8, 64, 300])
def test_paged_plan_equals_row_plan_on_token_counts(ps):
    """A paged plan is the row plan of the sequences' token counts: (pages - 1) * page_size + last."""
    lengths = [0, 1, 17, 1000, 5, 8192, 129, 300, 301]
    ip, last = _paged_layout(lengths, ps)
    opts = dict(min_rows_per_split=16, granularity=16)
    got = mla.plan_compute_host_paged(ip, last, ps, 11, **opts)
    tok = np.zeros(len(lengths) + 1, dtype=np.int32)
    tok[1:] = np.cumsum(lengths)
    ref = mla.plan_compute_host(tok, 11, **opts)
    for k in ("items", "work_indptr", "reduce"):
        assert np.array_equal(got[k], ref[k]), k
    assert got["num_slots"] == ref["num_slots"]
    assert [int(L) for L in got["items"][:, 4]] == [lengths[b] for b in got["items"][:, 0]]


def test_paged_plan_rejects_bad_layouts():
    ip = np.array([0, 2, 3], dtype=np.int32)
    for bad in ([0, 1], [1, 9], [-1, 1]):
        with pytest.raises(mla.MLAError) as e:
            mla.plan_compute_host_paged(ip, np.array(bad, dtype=np.int32), 8, 4)
        assert e.value.status == -10
    # no pages: the last page length is not looked at
    r = mla.plan_compute_host_paged(np.array([0, 0, 1], dtype=np.int32), np.array([0, 3], dtype=np.int32), 8, 4)
    assert [int(x) for x in r["items"][:, 4]] == [0, 3]
    with pytest.raises(mla.MLAError) as e:
        mla.plan_compute_host_paged(ip, np.array([1, 1], dtype=np.int32), 0, 4)
    assert e.value.status == -1
    with pytest.raises(mla.MLAError) as e:
        mla.plan_compute_host_paged(ip, None, 8, 4)
    assert e.value.status == -1
    # a sequence of more than 2^31 - 1 tokens does not fit the 32-bit token offsets
    with pytest.raises(mla.MLAError) as e:
        mla.plan_compute_host_paged(np.array([0, 1 << 24], dtype=np.int32), np.array([256], dtype=np.int32), 256, 4)
    assert e.value.status == -10


# ---------------------------------------------------------------- several query tokens per sequence

def _visible(L, q, j, causal):
    return min(max(L - q + j + 1, 0), L) if causal else L


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("num_sms,opts", [(7, dict(min_rows_per_split=16, granularity=16)), (152, {})])
def test_multi_plan_covers_every_query_token(causal, num_sms, opts):
    lengths = [300, 10, 0, 1, 4096, 77, 2]
    q_lens = [2, 3, 1, 4, 3, 0, 5]
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    qo = np.zeros(len(q_lens) + 1, dtype=np.int32)
    qo[1:] = np.cumsum(q_lens)
    r = mla.plan_compute_host_multi(qo, ip, num_sms, causal=causal, **opts)
    items, wip, red = r["items"], r["work_indptr"], r["reduce"]
    assert wip[0] == 0 and wip[-1] == len(items)
    by_row = {}
    for b, t0, t1, slot, L, q_row, q_tok in items:
        assert L == lengths[b] and q_row == qo[b] + q_tok and 0 <= q_tok < q_lens[b]
        by_row.setdefault(int(q_row), []).append((int(t0), int(t1), int(slot)))
    assert sorted(by_row) == list(range(int(qo[-1])))  # every query row is produced
    red_map = {int(rw): (int(s0), int(n)) for rw, s0, n in red}
    for b in range(len(lengths)):
        for j in range(q_lens[b]):
            parts = by_row[int(qo[b]) + j]
            n = _visible(lengths[b], q_lens[b], j, causal)
            pos = 0
            for t0, t1, _ in parts:  # contiguous cover of the visible tokens, in order
                assert t0 == pos
                pos = t1
            assert pos == n
            if len(parts) == 1:
                assert parts[0][2] == -1 and int(qo[b]) + j not in red_map
            else:
                s0, cnt = red_map[int(qo[b]) + j]
                assert [p[2] for p in parts] == list(range(s0, s0 + cnt))
    # the query tokens of a sequence's row range sit back to back in one CTA
    for c in range(r["num_ctas"]):
        seq_order = [int(items[i, 0]) for i in range(wip[c], wip[c + 1]) if items[i, 2] > items[i, 1]]
        assert all(seq_order[k] <= seq_order[k + 1] for k in range(len(seq_order) - 1))


def test_multi_plan_with_one_query_token_is_the_row_plan():
    lengths = [700, 5, 0, 4096, 129]
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    qo = np.arange(len(lengths) + 1, dtype=np.int32)
    for causal in (True, False):
        m = mla.plan_compute_host_multi(qo, ip, 9, causal=causal, min_rows_per_split=16, granularity=16)
        r = mla.plan_compute_host(ip, 9, min_rows_per_split=16, granularity=16)
        assert np.array_equal(m["items"][:, :5], r["items"])
        assert np.array_equal(m["work_indptr"], r["work_indptr"]) and np.array_equal(m["reduce"], r["reduce"])


def test_multi_plan_balances_weighted_granules():
    """Every KV granule weighs the number of query tokens of its sequence."""
    lengths, q_lens = [8192] * 8 + [1024] * 8, [4] * 8 + [1] * 8
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    qo = np.zeros(len(q_lens) + 1, dtype=np.int32)
    qo[1:] = np.cumsum(q_lens)
    r = mla.plan_compute_host_multi(qo, ip, 20, causal=False)
    items, wip = r["items"], r["work_indptr"]
    w = [sum(-(-int(items[i, 2] - items[i, 1]) // 128) for i in range(wip[c], wip[c + 1]))
         for c in range(r["num_ctas"])]
    assert sum(w) == sum(-(-L // 128) * q for L, q in zip(lengths, q_lens))
    assert max(w) - min(w) <= 4  # one granule of the heaviest sequence


def test_multi_plan_rejects_bad_query_offsets():
    ip = np.array([0, 10, 20], dtype=np.int32)
    for bad in ([1, 2, 3], [0, 3, 2]):
        with pytest.raises(mla.MLAError) as e:
            mla.plan_compute_host_multi(np.array(bad, dtype=np.int32), ip, 4)
        assert e.value.status == -10
