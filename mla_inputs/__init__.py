"""Seeded synthetic inputs for MLA decode (shared by the tests, the oracle
checks, the smoke check and the benchmark).

This module only draws and lays out data; it holds none of the attention
arithmetic. The leaderboard harness that fed the pages' kernels is not
available, so its inputs are stood in for by draws of the same shapes and
distributions: Q and KV ~ N(0,1) rounded to bf16 (the pages argue from Q
being randn with std ~1 — kernelbot amd-mixed-mla submission 689529
"MLA decode V3", docstring); fp8 KV is the bf16 KV quantised per tensor to
OCP e4m3fn with kv_scale = amax|KV| / 448 (the pages receive kv_data["fp8"]
as (buffer, scale) but do not show how it was made). The benchmark workloads
use page_size = 1, so kv_indptr / kv_indices address single rows; paged inputs
(make_paged_inputs) view the buffer as [num_pages, page_size, 576] with
kv_indptr counting pages, kv_indices holding page ids and kv_last_page_len the
tokens used in each sequence's last page (submission 641982 "v86", _run_a8w8).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HEADS = 16
QK_DIM = 576
V_DIM = 512
FP8_MAX = 448.0

# float32 value of 1/sqrt(576) = 1/24, the softmax scale the pages fix
SM_SCALE = float(np.float32(1.0 / math.sqrt(QK_DIM)))

MODE_BF16 = 0   # bf16 Q x bf16 KV
MODE_FP8 = 1    # Q cast to e4m3 in the kernel (scale 1) x e4m3 KV with per-tensor scale
MODE_A16W8 = 2  # bf16 Q x e4m3 KV


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: int
    batch: int
    kv_len: int | tuple[int, int]   # fixed length, or inclusive (lo, hi) for a seeded uniform draw
    permute: bool                    # kv_indices a seeded random permutation of the slots
    seed: int

    def describe(self) -> str:
        kind = {MODE_BF16: "bf16", MODE_FP8: "fp8", MODE_A16W8: "a16w8"}[self.mode]
        lens = (f"kv_len~U[{self.kv_len[0]},{self.kv_len[1]}]" if isinstance(self.kv_len, tuple)
                else f"kv_len={self.kv_len}")
        return f"{kind} B={self.batch} {lens}{' randperm slots' if self.permute else ''}"


# The five benchmark workloads (16 q heads / 1 latent KV head, 576 / 512, page_size 1).
WORKLOADS = {
    "bf16_b4_l1024": Workload("bf16_b4_l1024", MODE_BF16, 4, 1024, False, 1),
    "fp8_b4_l8192": Workload("fp8_b4_l8192", MODE_FP8, 4, 8192, False, 2),
    "fp8_b64_l1024": Workload("fp8_b64_l1024", MODE_FP8, 64, 1024, False, 3),
    "fp8_b64_l8192": Workload("fp8_b64_l8192", MODE_FP8, 64, 8192, False, 4),
    "bf16_b128_ragged": Workload("bf16_b128_ragged", MODE_BF16, 128, (512, 8192), True, 5),
}

# Further shapes for the modes beyond the benchmark workloads: the fp8 headline shape with a bf16 query.
EXTRA_WORKLOADS = {
    "a16w8_b64_l8192": Workload("a16w8_b64_l8192", MODE_A16W8, 64, 8192, False, 6),
}


@dataclasses.dataclass
class Inputs:
    mode: int
    q: torch.Tensor            # bf16 [B,16,576]
    kv: torch.Tensor           # bf16 [slots,576] (mode 0) or uint8 e4m3 codes [slots,576]
    kv_scale: float            # per-tensor fp32 dequantisation scale (1.0 in mode 0)
    kv_indptr: torch.Tensor    # int32 [B+1] (pages when page_size > 1)
    kv_indices: torch.Tensor   # int32 [R] (page ids when page_size > 1)
    sm_scale: float = SM_SCALE
    page_size: int = 1
    kv_last_page_len: torch.Tensor | None = None   # int32 [B] when page_size > 1

    @property
    def batch(self) -> int:
        return self.kv_indptr.numel() - 1

    @property
    def rows(self) -> int:
        """KV rows (tokens) the decode reads."""
        return int(self.lengths().sum())

    @property
    def kv_row_bytes(self) -> int:
        return QK_DIM * (2 if self.mode == MODE_BF16 else 1)

    def kv_scale_tensor(self, device) -> torch.Tensor:
        return torch.tensor([self.kv_scale], dtype=torch.float32, device=device)

    def to(self, device) -> "Inputs":
        lp = None if self.kv_last_page_len is None else self.kv_last_page_len.to(device)
        return Inputs(self.mode, self.q.to(device), self.kv.to(device), self.kv_scale,
                      self.kv_indptr.to(device), self.kv_indices.to(device), self.sm_scale, self.page_size, lp)

    def lengths(self) -> np.ndarray:
        """Tokens per sequence."""
        ip = self.kv_indptr.cpu().numpy().astype(np.int64)
        pages = ip[1:] - ip[:-1]
        if self.page_size == 1 and self.kv_last_page_len is None:
            return pages
        last = (np.full(pages.shape, self.page_size, np.int64) if self.kv_last_page_len is None
                else self.kv_last_page_len.cpu().numpy().astype(np.int64))
        return np.where(pages > 0, (pages - 1) * self.page_size + last, 0)


def quantize_kv_e4m3(kv_bf16: torch.Tensor) -> tuple[torch.Tensor, float]:
    """Per-tensor e4m3fn quantisation of the bf16 KV (input preparation, not the method)."""
    amax = kv_bf16.abs().max().float()
    scale = (amax / FP8_MAX).clamp_min(torch.finfo(torch.float32).tiny)
    codes = (kv_bf16.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, float(scale)


def make_inputs(lengths, mode: int, seed: int, permute: bool = False, extra_slots: int = 0,
                q_std: float = 1.0, device: str = "cpu") -> Inputs:
    """Seeded inputs for arbitrary per-sequence KV lengths.

    The KV pool holds sum(lengths) + extra_slots rows; sequences take their rows
    in order (kv_indices = arange) unless ``permute`` shuffles the slot order.
    """
    lengths = [int(x) for x in lengths]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    batch = len(lengths)
    total = sum(lengths)
    slots = total + int(extra_slots)
    q = (torch.randn((batch, HEADS, QK_DIM), generator=g, device=device) * q_std).to(torch.bfloat16)
    kv = torch.randn((max(slots, 1), QK_DIM), generator=g, device=device).to(torch.bfloat16)[:slots]
    ip = torch.zeros(batch + 1, dtype=torch.int64)
    if batch:
        ip[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    kv_indptr = ip.to(torch.int32).to(device)
    if permute:
        kv_indices = torch.randperm(slots, generator=g, device=device)[:total].to(torch.int32)
    else:
        kv_indices = torch.arange(total, dtype=torch.int32, device=device)
    if mode == MODE_BF16:
        return Inputs(mode, q, kv.contiguous(), 1.0, kv_indptr, kv_indices)
    codes, scale = quantize_kv_e4m3(kv)
    return Inputs(mode, q, codes.contiguous(), scale, kv_indptr, kv_indices)


def make_paged_inputs(lengths, page_size: int, mode: int, seed: int, permute: bool = False, extra_pages: int = 0,
                      q_std: float = 1.0, device: str = "cpu") -> Inputs:
    """Seeded inputs in the paged layout: sequence b takes ceil(L_b / page_size)
    pages, the last one holding L_b - (pages - 1) * page_size tokens (its other
    rows are unused and hold random data). Pages are taken in order unless
    ``permute`` shuffles the page order; ``extra_pages`` adds unused pages."""
    lengths = [int(x) for x in lengths]
    ps = int(page_size)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    batch = len(lengths)
    pages = [(L + ps - 1) // ps for L in lengths]
    last = [L - (p - 1) * ps if p > 0 else 1 for L, p in zip(lengths, pages)]
    total_pages = sum(pages)
    pool_pages = total_pages + int(extra_pages)
    rows = pool_pages * ps
    q = (torch.randn((batch, HEADS, QK_DIM), generator=g, device=device) * q_std).to(torch.bfloat16)
    kv = torch.randn((max(rows, 1), QK_DIM), generator=g, device=device).to(torch.bfloat16)[:rows]
    ip = torch.zeros(batch + 1, dtype=torch.int64)
    if batch:
        ip[1:] = torch.cumsum(torch.tensor(pages, dtype=torch.int64), 0)
    kv_indptr = ip.to(torch.int32).to(device)
    if permute:
        kv_indices = torch.randperm(pool_pages, generator=g, device=device)[:total_pages].to(torch.int32)
    else:
        kv_indices = torch.arange(total_pages, dtype=torch.int32, device=device)
    lp = torch.tensor(last, dtype=torch.int32, device=device)
    if mode == MODE_BF16:
        return Inputs(mode, q, kv.contiguous(), 1.0, kv_indptr, kv_indices, SM_SCALE, ps, lp)
    codes, scale = quantize_kv_e4m3(kv)
    return Inputs(mode, q, codes.contiguous(), scale, kv_indptr, kv_indices, SM_SCALE, ps, lp)


def make_query_tokens(q_lens, seed: int, q_std: float = 1.0, device: str = "cpu"):
    """Multi-token queries: q_lens[b] seeded N(0, q_std) query tokens per sequence, as a bf16
    [sum(q_lens), 16, 576] array with row offsets qo_indptr int32 [B+1]
    (the pages' qo_indptr = arange(B + 1) * q_seq_len, generalised to per-sequence counts)."""
    q_lens = [int(x) for x in q_lens]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = (torch.randn((sum(q_lens), HEADS, QK_DIM), generator=g, device=device) * q_std).to(torch.bfloat16)
    qo = torch.zeros(len(q_lens) + 1, dtype=torch.int64)
    if q_lens:
        qo[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0)
    return q, qo.to(torch.int32).to(device)


def workload_lengths(w: Workload) -> list[int]:
    if isinstance(w.kv_len, tuple):
        g = torch.Generator()
        g.manual_seed(1000 + w.seed)
        lo, hi = w.kv_len
        return [int(x) for x in torch.randint(lo, hi + 1, (w.batch,), generator=g)]
    return [w.kv_len] * w.batch


def get_workload(name: str) -> Workload:
    return WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]


def make_workload(name_or_w, device: str = "cpu", seed_offset: int = 0) -> Inputs:
    w = get_workload(name_or_w) if isinstance(name_or_w, str) else name_or_w
    return make_inputs(workload_lengths(w), w.mode, w.seed + seed_offset, permute=w.permute, device=device)


def workload_bytes(w: Workload) -> dict:
    """Algorithmic bytes one decode call must move: KV rows read, Q (bf16) read, O (bf16) written."""
    rows = sum(workload_lengths(w))
    row_bytes = QK_DIM * (2 if w.mode == MODE_BF16 else 1)
    q_bytes = w.batch * HEADS * QK_DIM * 2
    o_bytes = w.batch * HEADS * V_DIM * 2
    return {"rows": rows, "kv": rows * row_bytes, "q": q_bytes, "o": o_bytes,
            "index": rows * 4, "total": rows * row_bytes + q_bytes + o_bytes}
