"""Pins for the float64 oracle: each checks it against something other than
itself — the OCP e4m3 / bf16 definitions and torch's own float8 / bfloat16
conversions (library routines), closed forms of softmax attention, torch's
float64 scaled_dot_product_attention on tiny inputs (a library routine for the
same definition), and invariances of the method. Every pin takes the oracle
library handle so the planted-mistake test can run them on mutated copies.
"""
from __future__ import annotations

import math
import warnings

import numpy as np
import torch

import mla_inputs as mi
import oracle

H, D, DV = oracle.HEADS, oracle.QK_DIM, oracle.V_DIM


def _torch_kv_values(inp: mi.Inputs) -> torch.Tensor:
    """KV values as float64 through torch's own decoders (bf16, or e4m3fn x kv_scale)."""
    if inp.mode == mi.MODE_BF16:
        return inp.kv.to(torch.float64)
    return inp.kv.view(torch.float8_e4m3fn).to(torch.float64) * inp.kv_scale


def _torch_q_values(inp: mi.Inputs) -> torch.Tensor:
    if inp.mode == mi.MODE_FP8:  # direct cast with scale 1 (|q| << 464, where torch's cast agrees with RNE)
        return inp.q.to(torch.float8_e4m3fn).to(torch.float64)
    return inp.q.to(torch.float64)


def sdpa_reference(inp: mi.Inputs):
    """torch float64 SDPA on the same values; returns (out [B,16,512], lse [B,16])."""
    kvv = _torch_kv_values(inp)
    qv = _torch_q_values(inp)
    ip = inp.kv_indptr.tolist()
    outs, lses = [], []
    for b in range(inp.batch):
        rows = inp.kv_indices[ip[b]:ip[b + 1]].long()
        k = kvv[rows]                                  # [L,576]
        qb = qv[b]                                     # [16,576]
        o = torch.nn.functional.scaled_dot_product_attention(
            qb[None, :, None, :], k[None, None].expand(1, H, -1, -1),
            k[None, None, :, :DV].expand(1, H, -1, -1), scale=inp.sm_scale)[0, :, 0, :]
        s = (qb @ k.T) * inp.sm_scale
        outs.append(o)
        lses.append(torch.logsumexp(s, dim=1))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


# ---------------------------------------------------------------- codecs

def pin_bf16_decode(lib):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([lib.oracle_bf16_decode(int(b)) for b in bits[::97]])
    r = ref[::97]
    assert np.array_equal(np.isnan(got), np.isnan(r))
    assert np.array_equal(got[~np.isnan(r)], r[~np.isnan(r)])


def pin_e4m3_decode_table(lib):
    got = oracle.e4m3_decode_table(lib)
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    # landmarks of the OCP definition
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x38] == 1.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def _all_bf16():
    bits = np.arange(65536, dtype=np.uint16)
    vals = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return bits, vals


def pin_e4m3_encode_vs_torch(lib):
    """Every bf16 value: RNE codes equal torch's cast where torch does not overflow (|x| < 464)."""
    bits, vals = _all_bf16()
    got = oracle.q_to_e4m3(bits, lib)
    f = vals.to(torch.float64).numpy()
    ok = np.isfinite(f) & (np.abs(f) < 464.0)
    ref = vals[torch.from_numpy(ok)].to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[ok], ref)


def pin_e4m3_encode_saturates(lib):
    """Magnitudes past the largest finite value saturate to +-448 (satfinite); NaN stays NaN."""
    bits, vals = _all_bf16()
    got = oracle.q_to_e4m3(bits, lib)
    f = vals.to(torch.float64).numpy()
    big = ~np.isnan(f) & (np.abs(f) >= 464.0)
    assert np.all(got[big & (f > 0)] == 0x7E) and np.all(got[big & (f < 0)] == 0xFE)
    nan = np.isnan(f)
    assert np.all((got[nan] & 0x7F) == 0x7F)
    # exact ties round to the even code: 1 + 1/16 lies halfway between 1 and 1.125 -> 1.0 (0x38)
    assert lib.oracle_e4m3_encode(1.0 + 1.0 / 16) == 0x38
    assert lib.oracle_e4m3_encode(1.125 + 1.0 / 16) == 0x3A          # between 0x39 and 0x3A -> even 0x3A
    assert lib.oracle_e4m3_encode(2.0 ** -10) == 0x00                 # half of the smallest subnormal -> 0
    assert lib.oracle_e4m3_encode(3 * 2.0 ** -10) == 0x02             # 1.5 subnormal steps -> even code 2


# ---------------------------------------------------------------- attention

def _inputs(lengths, mode, seed=11, **kw):
    return mi.make_inputs(lengths, mode, seed, **kw)


def _dec(inp, lib, **kw):
    return oracle.decode(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.sm_scale, inp.mode, inp.kv_scale,
                         lib=lib, **kw)


def pin_single_row(lib):
    """L = 1: softmax weight 1, so O equals the value part of that row, and LSE equals its score."""
    for mode in (0, 1, 2):
        inp = _inputs([1, 1, 1], mode, permute=True, extra_slots=5)
        out, lse = _dec(inp, lib)
        kvv = _torch_kv_values(inp).numpy()
        qv = _torch_q_values(inp).numpy()
        for b in range(3):
            row = int(inp.kv_indices[b])
            assert np.array_equal(out[b], np.broadcast_to(kvv[row, :DV], (H, DV)))
            np.testing.assert_allclose(lse[b], (qv[b] @ kvv[row]) * inp.sm_scale, rtol=1e-12, atol=1e-12)


def pin_identical_rows(lib):
    """All rows equal: uniform weights over equal vectors give that vector."""
    for mode in (0, 1):
        inp = _inputs([7, 33], mode)
        inp.kv[:] = inp.kv[3]
        out, lse = _dec(inp, lib)
        v = _torch_kv_values(inp).numpy()[3, :DV]
        np.testing.assert_allclose(out, np.broadcast_to(v, out.shape), rtol=1e-13, atol=1e-13)


def pin_uniform_scores(lib):
    """q = 0 (and sm_scale = 0): all scores equal, O is the plain mean of the value rows, LSE = log L."""
    inp = _inputs([5, 64, 1], 0)
    inp.q.zero_()
    out, lse = _dec(inp, lib)
    kvv = _torch_kv_values(inp).numpy()
    ip = inp.kv_indptr.tolist()
    for b in range(3):
        mean = kvv[ip[b]:ip[b + 1], :DV].mean(axis=0)
        np.testing.assert_allclose(out[b], np.broadcast_to(mean, (H, DV)), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], math.log(ip[b + 1] - ip[b]), rtol=1e-13)
    inp2 = _inputs([9], 1)
    out2, _ = oracle.decode(inp2.q, inp2.kv, inp2.kv_indptr, inp2.kv_indices, 0.0, 1, inp2.kv_scale, lib=lib)
    mean2 = _torch_kv_values(inp2).numpy()[:9, :DV].mean(axis=0)
    np.testing.assert_allclose(out2[0], np.broadcast_to(mean2, (H, DV)), rtol=1e-12, atol=1e-13)


def pin_two_rows(lib):
    """L = 2: O = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1 (closed form of a two-way softmax)."""
    inp = _inputs([2], 0, seed=5)
    out, _ = _dec(inp, lib)
    kvv = _torch_kv_values(inp).numpy()
    qv = _torch_q_values(inp).numpy()[0]
    s = (qv @ kvv[:2].T) * inp.sm_scale
    w0 = 1.0 / (1.0 + np.exp(s[:, 1] - s[:, 0]))
    ref = w0[:, None] * kvv[0, :DV] + (1 - w0)[:, None] * kvv[1, :DV]
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-13)


def pin_convex_hull(lib):
    """Every output element lies within the range of its column over the sequence's value rows."""
    inp = _inputs([40, 3], 1, q_std=4.0)
    out, _ = _dec(inp, lib)
    kvv = _torch_kv_values(inp).numpy()
    ip = inp.kv_indptr.tolist()
    for b in range(2):
        v = kvv[ip[b]:ip[b + 1], :DV]
        assert np.all(out[b] >= v.min(axis=0) - 1e-12) and np.all(out[b] <= v.max(axis=0) + 1e-12)


def pin_permutation(lib):
    """Moving a sequence's rows to other slots (and its indices with them) leaves O unchanged."""
    for mode in (0, 1):
        inp = _inputs([13, 29], mode, seed=3)
        out, lse = _dec(inp, lib)
        perm = torch.randperm(inp.kv.shape[0], generator=torch.Generator().manual_seed(9))
        inv = torch.argsort(perm)
        moved = mi.Inputs(inp.mode, inp.q, inp.kv[perm].contiguous(), inp.kv_scale, inp.kv_indptr,
                          inv[inp.kv_indices.long()].to(torch.int32), inp.sm_scale)
        out2, lse2 = _dec(moved, lib)
        np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-13)


def pin_library_sdpa(lib):
    """Tiny inputs against torch's float64 scaled_dot_product_attention + logsumexp, all modes."""
    for mode in (0, 1, 2):
        inp = _inputs([1, 6, 17, 40], mode, seed=21 + mode, permute=True, extra_slots=11, q_std=2.0)
        out, lse = _dec(inp, lib)
        ref, ref_lse = sdpa_reference(inp)
        np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-11, atol=1e-12)


def pin_split_combine(lib):
    """Softmax over a union of disjoint row sets = LSE-weighted merge of the per-set results."""
    for mode in (0, 1):
        inp = _inputs([50], mode, seed=8, q_std=3.0)
        full, full_lse = _dec(inp, lib)
        cuts = [0, 16, 17, 48, 50]
        parts = [oracle.decode_range(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.sm_scale, 0, a, b,
                                     mode, inp.kv_scale, lib=lib) for a, b in zip(cuts[:-1], cuts[1:])]
        po = np.stack([p[0] for p in parts])
        pl = np.stack([p[1] for p in parts])
        # an empty part must not change the result
        po = np.concatenate([po, np.zeros((1, H, DV))])
        pl = np.concatenate([pl, np.full((1, H), -np.inf)])
        out, lse = oracle.combine(po, pl, lib)
        np.testing.assert_allclose(out, full[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, full_lse[0], rtol=1e-13)


def pin_empty_and_errors(lib):
    inp = _inputs([0, 4, 0], 0)
    out, lse = _dec(inp, lib)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    bad = mi.Inputs(inp.mode, inp.q, inp.kv, 1.0, inp.kv_indptr, inp.kv_indices.clone(), inp.sm_scale)
    bad.kv_indices[1] = 10_000
    try:
        _dec(bad, lib)
    except ValueError:
        return
    raise AssertionError("out-of-range row index was not reported")


# ---------------------------------------------------------------- paged layout

def _paged(lengths, ps, mode, seed, **kw):
    return mi.make_paged_inputs(lengths, ps, mode, seed, **kw)


def _dec_paged(inp, lib, **kw):
    return oracle.decode_paged(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.kv_last_page_len, inp.page_size,
                               inp.sm_scale, inp.mode, inp.kv_scale, lib=lib, **kw)


def sdpa_reference_paged(inp: mi.Inputs, lengths):
    """torch float64 SDPA over each sequence's tokens, gathered by viewing the buffer as
    [num_pages, page_size, 576] (the pages' own view), indexing it with the page ids and
    keeping the first L_b rows (``lengths`` are the generator's token counts)."""
    kvv = _torch_kv_values(inp)
    pages = kvv.view(-1, inp.page_size, D)
    qv = _torch_q_values(inp)
    ip = inp.kv_indptr.tolist()
    outs, lses = [], []
    for b, L in enumerate(lengths):
        if L == 0:
            outs.append(torch.zeros(H, DV, dtype=torch.float64))
            lses.append(torch.full((H,), -math.inf, dtype=torch.float64))
            continue
        ids = inp.kv_indices[ip[b]:ip[b + 1]].long()
        k = pages[ids].reshape(-1, D)[:L]
        qb = qv[b]
        o = torch.nn.functional.scaled_dot_product_attention(
            qb[None, :, None, :], k[None, None].expand(1, H, -1, -1),
            k[None, None, :, :DV].expand(1, H, -1, -1), scale=inp.sm_scale)[0, :, 0, :]
        outs.append(o)
        lses.append(torch.logsumexp((qb @ k.T) * inp.sm_scale, dim=1))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


def pin_paged_library_sdpa(lib):
    """Paged buffers (ragged last pages, shuffled page order, unused pages) against torch
    SDPA over the tokens gathered through the [pages, page_size, 576] view, all modes."""
    cases = [([1, 9, 16, 0, 37], 8), ([3, 4, 1, 12], 2), ([33, 64, 5], 16), ([7, 2], 3)]
    for k, (lengths, ps) in enumerate(cases):
        for mode in (0, 1, 2):
            inp = _paged(lengths, ps, mode, seed=40 + 3 * k + mode, permute=True, extra_pages=3, q_std=2.0)
            out, lse = _dec_paged(inp, lib)
            ref, ref_lse = sdpa_reference_paged(inp, lengths)
            np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse, ref_lse, rtol=1e-11, atol=1e-12)


def pin_paged_unit_pages(lib):
    """page_size 1 with full last pages is the row-addressed decode."""
    inp = _inputs([1, 6, 17], 1, seed=12, permute=True, extra_slots=4)
    out, lse = _dec(inp, lib)
    ones = torch.ones(inp.batch, dtype=torch.int32)
    out2, lse2 = oracle.decode_paged(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, ones, 1, inp.sm_scale, 1,
                                     inp.kv_scale, lib=lib)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_paged_permutation(lib):
    """Moving whole pages to other page slots (and their ids with them) leaves O unchanged."""
    for mode in (0, 1):
        inp = _paged([13, 29, 8], 4, mode, seed=5, extra_pages=2)
        out, lse = _dec_paged(inp, lib)
        n_pages = inp.kv.shape[0] // 4
        perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(4))
        inv = torch.argsort(perm)
        kv_moved = inp.kv.view(n_pages, 4, D)[perm].reshape(-1, D).contiguous()
        moved = mi.Inputs(inp.mode, inp.q, kv_moved, inp.kv_scale, inp.kv_indptr,
                          inv[inp.kv_indices.long()].to(torch.int32), inp.sm_scale, 4, inp.kv_last_page_len)
        out2, lse2 = _dec_paged(moved, lib)
        np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-13)


def pin_paged_unused_rows_ignored(lib):
    """Rows past a sequence's last used token (the rest of its last page, and unused pages)
    do not enter the result: overwriting them with extreme values changes nothing."""
    for mode in (0, 1):
        lengths, ps = [5, 16, 11], 8
        inp = _paged(lengths, ps, mode, seed=6, extra_pages=2)
        out, lse = _dec_paged(inp, lib)
        used = torch.zeros(inp.kv.shape[0], dtype=torch.bool)
        ip = inp.kv_indptr.tolist()
        for b, L in enumerate(lengths):
            for t in range(L):
                used[int(inp.kv_indices[ip[b] + t // ps]) * ps + t % ps] = True
        assert int(used.sum()) == sum(lengths)
        big = inp.kv.clone()
        big[~used] = (torch.tensor(3.0e4, dtype=torch.bfloat16) if mode == 0
                      else torch.tensor(0x7E, dtype=torch.uint8))
        out2, lse2 = _dec_paged(mi.Inputs(inp.mode, inp.q, big, inp.kv_scale, inp.kv_indptr, inp.kv_indices,
                                          inp.sm_scale, ps, inp.kv_last_page_len), lib)
        assert np.array_equal(out2, out) and np.array_equal(lse2, lse)


def pin_paged_errors(lib):
    """A last page length outside [1, page_size], or a page id past the buffer, is reported."""
    inp = _paged([5, 9], 4, 0, seed=7)
    for bad_last in (0, 5):
        lp = inp.kv_last_page_len.clone()
        lp[1] = bad_last
        try:
            oracle.decode_paged(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, lp, 4, inp.sm_scale, 0, lib=lib)
        except ValueError:
            continue
        raise AssertionError(f"last page length {bad_last} was not reported")
    ix = inp.kv_indices.clone()
    ix[-1] = inp.kv.shape[0] // 4
    try:
        oracle.decode_paged(inp.q, inp.kv, inp.kv_indptr, ix, inp.kv_last_page_len, 4, inp.sm_scale, 0, lib=lib)
    except ValueError:
        return
    raise AssertionError("page id past the buffer was not reported")


# ---------------------------------------------------------------- multi-token decode

def _gather_kv(inp: mi.Inputs, b: int, L: int) -> torch.Tensor:
    """Sequence b's first L KV tokens as float64 [L, 576]: row indices, or the page view."""
    kvv = _torch_kv_values(inp)
    ip = inp.kv_indptr.tolist()
    if inp.page_size == 1:
        return kvv[inp.kv_indices[ip[b]:ip[b + 1]].long()][:L]
    return kvv.view(-1, inp.page_size, D)[inp.kv_indices[ip[b]:ip[b + 1]].long()].reshape(-1, D)[:L]


def sdpa_reference_multi(inp: mi.Inputs, q, qo, lengths, causal: bool):
    """torch float64 SDPA per sequence: its query rows against its KV tokens, masked with torch's
    lower-right causal bias when ``causal`` (the query tokens are the sequence's last ones)."""
    from torch.nn.attention.bias import causal_lower_right
    if inp.mode == mi.MODE_FP8:
        qv = q.to(torch.float8_e4m3fn).to(torch.float64)
    else:
        qv = q.to(torch.float64)
    qo = qo.tolist()
    outs, lses = [], []
    for b, L in enumerate(lengths):
        qb = qv[qo[b]:qo[b + 1]]                      # [n, 576]
        n = qb.shape[0]
        if n == 0:
            continue
        k = _gather_kv(inp, b, L)
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            mask = (causal_lower_right(n, L)._materialize(torch.device("cpu")) if causal
                    else torch.ones(n, L, dtype=torch.bool))
        for h in range(H):
            sh = torch.einsum("nd,td->nt", qb[:, h], k) * inp.sm_scale
            sh = sh.masked_fill(~mask, -math.inf)
            lse = torch.logsumexp(sh, dim=1)
            with warnings.catch_warnings():  # rows with no visible key give NaN there; zeroed below
                warnings.simplefilter("ignore")
                o = torch.nn.functional.scaled_dot_product_attention(
                    qb[None, None, :, h], k[None, None], k[None, None, :, :DV], attn_mask=mask[None, None],
                    scale=inp.sm_scale)[0, 0]
            o = torch.where(torch.isinf(lse)[:, None], torch.zeros_like(o), o)
            outs.append((qo[b], h, o))
            lses.append((qo[b], h, lse))
    total = qo[-1]
    out = torch.zeros(total, H, DV, dtype=torch.float64)
    lse_all = torch.zeros(total, H, dtype=torch.float64)
    for r0, h, o in outs:
        out[r0:r0 + o.shape[0], h] = o
    for r0, h, l in lses:
        lse_all[r0:r0 + l.shape[0], h] = l
    return out.numpy(), lse_all.numpy()


def _dec_multi(inp, q, qo, causal, lib):
    return oracle.decode_multi(q, inp.kv, qo, inp.kv_indptr, inp.kv_indices, inp.sm_scale, inp.mode, inp.kv_scale,
                               causal=causal, kv_last_page_len=inp.kv_last_page_len, page_size=inp.page_size, lib=lib)


def pin_multi_single_token(lib):
    """One query token per sequence, causal or not, is the single-token decode."""
    inp = _inputs([1, 9, 40], 1, seed=14, permute=True, extra_slots=3)
    out, lse = _dec(inp, lib)
    qo = torch.arange(inp.batch + 1, dtype=torch.int32)
    for causal in (False, True):
        out2, lse2 = _dec_multi(inp, inp.q, qo, causal, lib)
        assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_multi_library_sdpa(lib):
    """Several query tokens per sequence against torch float64 SDPA with and without the lower-right
    causal mask: row addressing and paged, all modes."""
    lengths, q_lens = [5, 40, 17, 64, 3], [1, 3, 4, 2, 3]
    for mode in (0, 1, 2):
        for paged in (False, True):
            inp = (_paged(lengths, 8, mode, seed=60 + mode, permute=True, extra_pages=2) if paged
                   else _inputs(lengths, mode, seed=60 + mode, permute=True, extra_slots=7))
            q, qo = mi.make_query_tokens(q_lens, seed=70 + mode, q_std=2.0)
            for causal in (False, True):
                out, lse = _dec_multi(inp, q, qo, causal, lib)
                ref, ref_lse = sdpa_reference_multi(inp, q, qo, lengths, causal)
                np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
                np.testing.assert_allclose(lse, ref_lse, rtol=1e-11, atol=1e-12)


def pin_multi_more_queries_than_tokens(lib):
    """Causal, with more query tokens than KV tokens: the first q_b - L_b query tokens see nothing
    (zeros, LSE -inf); the others see their prefix."""
    lengths, q_lens = [2, 6], [5, 6]
    inp = _inputs(lengths, 0, seed=17)
    q, qo = mi.make_query_tokens(q_lens, seed=18)
    out, lse = _dec_multi(inp, q, qo, True, lib)
    assert np.all(out[:3] == 0) and np.all(np.isneginf(lse[:3]))
    ref, ref_lse = sdpa_reference_multi(inp, q, qo, lengths, True)
    np.testing.assert_allclose(out[3:], ref[3:], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[3:], ref_lse[3:], rtol=1e-11, atol=1e-12)


ALL_PINS = [
    pin_bf16_decode, pin_e4m3_decode_table, pin_e4m3_encode_vs_torch, pin_e4m3_encode_saturates,
    pin_single_row, pin_identical_rows, pin_uniform_scores, pin_two_rows, pin_convex_hull,
    pin_permutation, pin_library_sdpa, pin_split_combine, pin_empty_and_errors,
    pin_paged_library_sdpa, pin_paged_unit_pages, pin_paged_permutation, pin_paged_unused_rows_ignored,
    pin_paged_errors, pin_multi_single_token, pin_multi_library_sdpa, pin_multi_more_queries_than_tokens,
]
