"""CPU tests of the host split-KV planner (through the C ABI's host-only entry)."""
import numpy as np
import pytest

import mla_decode_attention_09_gb300 as mla


def _even_split_costs(gl, n_ctas, item_units, unit):
    """Costs of the ranges that cut the granules of all sequences, laid end to end, evenly:
    range k holds granules [U k / n, U (k + 1) / n); a sequence it touches adds one item."""
    U = sum(gl)
    starts = np.cumsum([0] + gl)
    costs = []
    for k in range(n_ctas):
        a, b = U * k // n_ctas, U * (k + 1) // n_ctas
        if b <= a:
            continue
        touched = sum(1 for i, g in enumerate(gl) if g and starts[i] < b and starts[i] + g > a)
        costs.append((b - a) * unit + touched * item_units)
    return costs


def _check_plan(lengths, num_sms, **opts):
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    r = mla.plan_compute_host(ip, num_sms, **opts)
    items, wip, red = r["items"], r["work_indptr"], r["reduce"]
    G = opts.get("granularity", 64)
    min_split = opts.get("min_rows_per_split", 64)
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
    # Load balance. A CTA's cost is its granules (G rows; a sequence's last granule may be
    # shorter) plus a fixed cost per item it starts (item_cost_rows, default 256 rows). The
    # planner minimises the largest cost: it is never above that of cutting the granules
    # evenly, which is checked when the minimum split is one granule. Without item costs
    # that means at most ceil(granules / CTAs) granules per CTA.
    if total:
        max_ctas = num_sms * cpsm
        ic = opts.get("item_cost_rows", 0)
        ic = 256 if ic == 0 else max(ic, 0)
        unit = 16
        item_units = ic * unit // G
        min_gran = -(-min_split // G)
        gl = [-(-L // G) for L in lengths]
        U = sum(gl)
        gran = [sum(-(-int(items[i, 2] - items[i, 1]) // G) for i in range(wip[c], wip[c + 1]))
                for c in range(r["num_ctas"])]
        nit = [sum(1 for i in range(wip[c], wip[c + 1]) if items[i, 2] > items[i, 1]) for c in range(r["num_ctas"])]
        cost = [g * unit + n * item_units for g, n in zip(gran, nit)]
        assert sum(gran) == U
        rows = [sum(int(items[i, 2] - items[i, 1]) for i in range(wip[c], wip[c + 1])) for c in range(r["num_ctas"])]
        assert sum(rows) == total
        if min_gran == 1:
            assert max(cost) <= max(_even_split_costs(gl, max_ctas, item_units, unit))
            if ic == 0:
                assert max(gran) <= -(-U // max_ctas)
        else:
            # every piece of a split sequence holds min_rows_per_split rows at least, unless it
            # is the sequence's last piece and the whole remainder
            for b in range(len(lengths)):
                parts = [(int(t0), int(t1)) for bb, t0, t1, _, _ in items if bb == b]
                if len(parts) > 1:
                    assert all(t1 - t0 >= min(min_gran * G, lengths[b]) for t0, t1 in parts[:-1])
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
    # B=64 x 8192 over 152 SMs: (nearly) every SM busy, each sequence split in 2-4 chunks
    r = _check_plan([8192] * 64, 152)
    assert 150 <= r["num_ctas"] <= 152
    assert 64 * 2 <= r["num_slots"] <= 64 * 4
    # B=4 x 1024 bf16: small problem, one 64-row granule per CTA (the default minimum chunk)
    r = _check_plan([1024] * 4, 152)
    assert r["num_ctas"] == 64
    # with 128-row granules (the tensor-memory kernel's tile), one tile per CTA
    r = _check_plan([1024] * 4, 152, granularity=128, min_rows_per_split=128)
    assert r["num_ctas"] == 32
    # B=64 x 8192, 4096 tiles. Without item costs every CTA gets 27 tiles at most. With the
    # default cost of two tiles per item, CTAs that hold two sequence pieces get fewer tiles
    # than those holding one, and the largest cost (tiles + 2 x items) drops from 31 to 30.
    def tiles_items(r):
        t, n = [], []
        for c in range(r["num_ctas"]):
            its = r["items"][r["work_indptr"][c]:r["work_indptr"][c + 1]]
            t.append(sum(-(-int(t1 - t0) // 128) for _, t0, t1, _, _ in its))
            n.append(len(its))
        return np.array(t), np.array(n)
    ip = np.arange(65, dtype=np.int32) * 8192
    g128 = dict(granularity=128, min_rows_per_split=128)
    t, n = tiles_items(mla.plan_compute_host(ip, 152, item_cost_rows=-1, **g128))
    assert t.sum() == 4096 and t.max() == 27 and (t + 2 * n).max() == 31
    t, n = tiles_items(mla.plan_compute_host(ip, 152, **g128))
    assert t.sum() == 4096 and (t + 2 * n).max() == 30 and len(t) >= 150
    assert t[n == 2].max() < t[n == 1].max()


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
    for b, t0, t1, slot, L, q_row, q_tok, _pair in items:
        assert L == lengths[b] and q_row == qo[b] + q_tok and 0 <= q_tok < q_lens[b]
        by_row.setdefault(int(q_row), []).append((int(t0), int(t1), int(slot)))
    assert sorted(by_row) == list(range(int(qo[-1])))  # every query row is produced
    red_map = {int(rw): (int(s0), int(n)) for rw, s0, n, _stride in red}
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
        assert np.array_equal(m["work_indptr"], r["work_indptr"]) and np.array_equal(m["reduce"][:, :3], r["reduce"])
        assert not m["items"][:, 7].any() and not m["reduce"][:, 3].any()


def test_multi_plan_balances_weighted_granules():
    """Every KV granule weighs the number of query tokens of its sequence."""
    lengths, q_lens = [8192] * 8 + [1024] * 8, [4] * 8 + [1] * 8
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    qo = np.zeros(len(q_lens) + 1, dtype=np.int32)
    qo[1:] = np.cumsum(q_lens)
    r = mla.plan_compute_host_multi(qo, ip, 20, causal=False, item_cost_rows=-1, granularity=128,
                                    min_rows_per_split=128)
    items, wip = r["items"], r["work_indptr"]
    w = [sum(-(-int(items[i, 2] - items[i, 1]) // 128) for i in range(wip[c], wip[c + 1]))
         for c in range(r["num_ctas"])]
    U = sum(-(-L // 128) * q for L, q in zip(lengths, q_lens))
    assert sum(w) == U
    assert max(w) <= -(-U // 20) + 3  # the even share, plus less than one granule of the heaviest sequence


def test_multi_plan_rejects_bad_query_offsets():
    ip = np.array([0, 10, 20], dtype=np.int32)
    for bad in ([1, 2, 3], [0, 3, 2]):
        with pytest.raises(mla.MLAError) as e:
            mla.plan_compute_host_multi(np.array(bad, dtype=np.int32), ip, 4)
        assert e.value.status == -10


def test_multi_plan_token_parallel():
    """Equal query counts: the row ranges are planned for one token, and CTAs r*Q .. r*Q+Q-1
    hold the Q tokens of range r, each over the same rows (clipped to its causal prefix)."""
    B, L, Q = 16, 3000, 3
    ip = np.arange(B + 1, dtype=np.int32) * L
    qo = np.arange(B + 1, dtype=np.int32) * Q
    r = mla.plan_compute_host_multi(qo, ip, 40, causal=True)
    items, wip = r["items"], r["work_indptr"]
    assert r["num_ctas"] % Q == 0 and r["num_ctas"] <= 40
    for rg in range(r["num_ctas"] // Q):
        per_tok = [[tuple(int(v) for v in x[:3]) for x in items[wip[rg * Q + j]:wip[rg * Q + j + 1]]] for j in range(Q)]
        for j in range(Q):
            assert all(int(x[6]) == j for x in items[wip[rg * Q + j]:wip[rg * Q + j + 1]])
            # same sequences and starts; ends differ only where the causal prefix clips them
            assert [(b, t0) for b, t0, _ in per_tok[j]] == [(b, t0) for b, t0, _ in per_tok[0]]
            for (b, t0, t1), (_, _, t1_0) in zip(per_tok[j], per_tok[0]):
                assert t1 - t1_0 in (0, j) and t1 <= L - Q + j + 1
    # every query row covered once, in order (the reduce map is checked by the general test)
    by_row = {}
    for x in items:
        by_row.setdefault(int(x[5]), []).append((int(x[1]), int(x[2])))
    for row, parts in by_row.items():
        b, j = divmod(row, Q)
        pos = 0
        for t0, t1 in parts:
            assert t0 == pos
            pos = t1
        assert pos == L - Q + j + 1
    # off: each range's tokens back to back in one CTA
    r2 = mla.plan_compute_host_multi(qo, ip, 40, causal=True, token_parallel=-1)
    toks = {int(x[6]) for x in r2["items"][r2["work_indptr"][0]:r2["work_indptr"][1]]}
    assert toks == set(range(Q))


def test_multi_plan_token_parallel_random():
    """Token-parallel plans with empty sequences holding other query counts, and equal counts
    elsewhere: a valid CSR within the grid, every query row produced, causal prefixes covered."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        B = int(rng.integers(1, 30))
        Q = int(rng.choice([2, 3, 4, 8]))
        lengths = [int(x) for x in rng.integers(0, 2000, B)]
        q_lens = []
        for L in lengths:
            if L == 0 and rng.random() < 0.5:
                q_lens.append(int(rng.integers(0, 12)))  # an empty sequence may hold any number of tokens
            else:
                q_lens.append(Q)
        if rng.random() < 0.2:
            lengths[int(rng.integers(0, B))] = 0
        ip = np.zeros(B + 1, dtype=np.int32)
        ip[1:] = np.cumsum(lengths)
        qo = np.zeros(B + 1, dtype=np.int32)
        qo[1:] = np.cumsum(q_lens)
        num_sms = int(rng.integers(1, 160))
        opts = {"min_rows_per_split": 16, "granularity": 16} if rng.random() < 0.5 else {}
        r = mla.plan_compute_host_multi(qo, ip, num_sms, causal=True, **opts)
        items, wip = r["items"], r["work_indptr"]
        assert 1 <= r["num_ctas"] <= max(num_sms, 1) and wip[0] == 0 and wip[-1] == len(items)
        assert np.all(np.diff(wip) >= 0)
        by_row = {}
        for b, t0, t1, slot, L, q_row, q_tok, _pair in items:
            assert L == lengths[b] and q_row == qo[b] + q_tok
            by_row.setdefault(int(q_row), []).append((int(t0), int(t1)))
        assert sorted(by_row) == list(range(int(qo[-1])))
        for b in range(B):
            for j in range(q_lens[b]):
                parts = [p for p in by_row[int(qo[b]) + j] if p[1] > p[0]]
                n = min(max(lengths[b] - q_lens[b] + j + 1, 0), lengths[b])
                pos = 0
                for t0, t1 in parts:
                    assert t0 == pos
                    pos = t1
                assert pos == n


def _pair_rows(items):
    """Expand a token-pair plan's items into per-query-row parts (first token, end token, slot)."""
    by_row = {}
    for b, t0, t1, slot, L, q_row, q_tok, pair in (tuple(int(v) for v in x) for x in items):
        if pair >= 0:  # rows q_row (token q_tok, over [t0, pair)) and q_row + 1 (over [t0, t1))
            assert t0 <= pair <= t1 or t1 == t0 == 0
            by_row.setdefault(q_row, []).append((t0, min(pair, t1), slot))
            by_row.setdefault(q_row + 1, []).append((t0, t1, slot + 1 if slot >= 0 else -1))
        else:
            by_row.setdefault(q_row, []).append((t0, t1, slot))
    return by_row


def _check_pair_plan(lengths, q_lens, num_sms, causal, **opts):
    ip = np.zeros(len(lengths) + 1, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    qo = np.zeros(len(q_lens) + 1, dtype=np.int32)
    qo[1:] = np.cumsum(q_lens)
    r = mla.plan_compute_host_multi(qo, ip, num_sms, causal=causal, token_pairs=1, **opts)
    items, wip, red = r["items"], r["work_indptr"], r["reduce"]
    counts = {q for L, q in zip(lengths, q_lens) if L > 0 and q > 0}
    if len(counts) != 1 or min(counts) % 2:  # not a pair plan: the ordinary one
        plain = mla.plan_compute_host_multi(qo, ip, num_sms, causal=causal, **opts)
        assert all(np.array_equal(r[k], plain[k]) for k in ("items", "work_indptr", "reduce"))
        return r
    assert wip[0] == 0 and wip[-1] == len(items) and np.all(np.diff(wip) >= 0)
    assert 1 <= r["num_ctas"] <= num_sms * opts.get("ctas_per_sm", 1)
    for x in items:
        b, q_row, q_tok, pair = int(x[0]), int(x[5]), int(x[6]), int(x[7])
        assert q_row == qo[b] + q_tok and int(x[4]) == lengths[b]
        if pair >= 0:  # a pair starts at an even token of a sequence with rows
            assert q_tok % 2 == 0 and q_tok + 1 < q_lens[b] and lengths[b] > 0
        else:
            assert lengths[b] == 0 and int(x[2]) == int(x[1]) == 0
    by_row = _pair_rows(items)
    assert sorted(by_row) == list(range(int(qo[-1])))  # every query row is produced
    red_map = {int(rw): (int(s0), int(n), int(st)) for rw, s0, n, st in red}
    used = []
    for b in range(len(lengths)):
        for j in range(q_lens[b]):
            row = int(qo[b]) + j
            parts = by_row[row]
            n = _visible(lengths[b], q_lens[b], j, causal)
            pos = 0
            for t0, t1, _ in parts:  # the non-empty parts cover the visible tokens in order
                if t1 > t0:
                    assert t0 == pos
                    pos = t1
            assert pos == n
            if len(parts) == 1:
                assert parts[0][2] == -1 and row not in red_map
            else:
                s0, cnt, st = red_map[row]
                assert cnt == len(parts) and st == 2
                assert [p[2] for p in parts] == list(range(s0, s0 + 2 * cnt, 2))
                used += [p[2] for p in parts]
    assert sorted(used) == list(range(r["num_slots"]))  # every slot written once
    return r


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Q", [2, 4, 6])
def test_pair_plan_covers_every_query_token(causal, Q):
    """Token pairs: an item covers tokens 2v (over [t_begin, pair field)) and 2v+1 (over [t_begin,
    end)); each row's slots lie two apart; ranges are token-parallel over the Q/2 pairs."""
    B, L = 16, 3000
    r = _check_pair_plan([L] * B, [Q] * B, 40, causal)
    items, wip = r["items"], r["work_indptr"]
    U = Q // 2
    assert r["num_ctas"] % U == 0
    assert (items[:, 7] >= 0).all()
    for rg in range(r["num_ctas"] // U):
        for v in range(U):
            assert all(int(x[6]) == 2 * v for x in items[wip[rg * U + v]:wip[rg * U + v + 1]])


def test_pair_plan_edge_lengths():
    """Sequences shorter than their query count (tokens that see nothing), one-row sequences,
    sequences without rows holding any number of tokens, and ranges that hold only the last row."""
    for causal in (True, False):
        _check_pair_plan([1, 2, 3, 0, 129, 0, 64, 65], [2, 2, 2, 3, 2, 0, 2, 2], 5, causal,
                         min_rows_per_split=16, granularity=16)
        _check_pair_plan([4096, 4, 0, 8193], [4, 4, 5, 4], 3, causal, min_rows_per_split=16, granularity=16)
        _check_pair_plan([65, 65], [2, 2], 8, causal, min_rows_per_split=16, granularity=16, item_cost_rows=-1)


def test_pair_plan_needs_equal_even_counts():
    lengths = [500, 600, 700]
    ip = np.zeros(4, dtype=np.int32)
    ip[1:] = np.cumsum(lengths)
    for q_lens in ([3, 3, 3], [2, 4, 2], [1, 1, 1]):
        qo = np.zeros(4, dtype=np.int32)
        qo[1:] = np.cumsum(q_lens)
        on = mla.plan_compute_host_multi(qo, ip, 20, causal=True, token_pairs=1)
        off = mla.plan_compute_host_multi(qo, ip, 20, causal=True)
        assert not on["items"][:, 7].any() and not on["reduce"][:, 3].any()
        for k in ("items", "work_indptr", "reduce"):
            assert np.array_equal(on[k], off[k])


def test_pair_plan_random():
    rng = np.random.default_rng(11)
    for _ in range(300):
        B = int(rng.integers(1, 24))
        Q = int(rng.choice([2, 4, 6, 8]))
        lengths = [int(x) for x in rng.integers(0, 3000, B)]
        for k in range(B):
            if rng.random() < 0.15:
                lengths[k] = int(rng.integers(0, 4))
        q_lens = [Q if L > 0 else int(rng.integers(0, 9)) for L in lengths]
        opts = {"min_rows_per_split": 16, "granularity": 16} if rng.random() < 0.5 else {}
        if rng.random() < 0.3:
            opts["token_parallel"] = -1
        _check_pair_plan(lengths, q_lens, int(rng.integers(1, 160)), bool(rng.random() < 0.8), **opts)
