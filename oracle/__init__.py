"""Float64 CPU oracle for MLA decode (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package; the product library never does. It wraps the
plain C implementation in ``mla_oracle.c`` (compiled here with gcc, OpenMP
over independent (sequence, head) pairs) with numpy marshalling.

What the oracle computes, and the readings it takes where the pages are
silent, are stated at the top of ``mla_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HEADS = 16
QK_DIM = 576
V_DIM = 512

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library; returns its path."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def load(path: str | None = None):
    """Load (building first if needed) the oracle library and declare its C signatures."""
    global _lib
    if path is None:
        with _lock:
            if _lib is None:
                if _stale():
                    build()
                _lib = _declare(ctypes.CDLL(_LIB_PATH))
            return _lib
    return _declare(ctypes.CDLL(path))


def _declare(lib):
    P = ctypes.c_void_p
    i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_decode.restype = f64
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = f64
    lib.oracle_e4m3_encode.argtypes = [f64]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_decode.argtypes = [i32, P, P, i64, i32, f32, P, P, f64, P, i32, P, P]
    lib.oracle_decode.restype = i32
    lib.oracle_decode_paged.argtypes = [i32, P, P, i64, i32, f32, P, P, P, i32, f64, P, i32, P, P]
    lib.oracle_decode_paged.restype = i32
    lib.oracle_decode_multi.argtypes = [i32, P, P, i64, i32, f32, P, P, P, P, i32, i32, f64, P, P]
    lib.oracle_decode_multi.restype = i32
    lib.oracle_decode_range.argtypes = [i32, P, P, i64, i32, f32, P, P, f64, i32, i64, i64, P, P]
    lib.oracle_decode_range.restype = i32
    lib.oracle_combine.argtypes = [i32, P, P, P, P]
    lib.oracle_combine.restype = i32
    lib.oracle_q_to_e4m3.argtypes = [P, i64, P]
    lib.oracle_q_to_e4m3.restype = None
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = i32
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """bf16 data as raw uint16 bits (accepts a uint16 array or a torch bf16 tensor)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        a = a.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


def _kv_bytes(kv, mode: int) -> np.ndarray:
    if mode == 0:
        return _u16(kv)
    if hasattr(kv, "dtype") and "float8" in str(kv.dtype):
        kv = kv.contiguous().view(__import__("torch").uint8).numpy()
    elif hasattr(kv, "numpy"):
        kv = kv.contiguous().numpy()
    return np.ascontiguousarray(kv, dtype=np.uint8)


def _i32(a) -> np.ndarray:
    if hasattr(a, "numpy"):
        a = a.contiguous().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def decode(q, kv, kv_indptr, kv_indices, sm_scale: float, mode: int = 0, kv_scale: float = 1.0,
           seq_ids=None, lib=None):
    """Oracle MLA decode. Returns (out [n,16,512] float64, lse [n,16] float64).

    q: bf16 [B,16,576] (uint16 bits or torch bf16); kv: [slots,576] bf16 (mode 0)
    or e4m3 bytes (modes 1, 2); kv_indptr int32 [B+1]; kv_indices int32 [R].
    ``sm_scale`` should be the float32 value the device receives.
    """
    lib = lib or load()
    qb = _u16(q).reshape(-1)
    kvb = _kv_bytes(kv, mode)
    ip = _i32(kv_indptr)
    ix = _i32(kv_indices)
    batch = ip.shape[0] - 1
    num_slots = kvb.size // QK_DIM
    sids = None if seq_ids is None else _i32(seq_ids)
    n = batch if sids is None else sids.shape[0]
    out = np.zeros((n, HEADS, V_DIM), dtype=np.float64)
    lse = np.zeros((n, HEADS), dtype=np.float64)
    rc = lib.oracle_decode(batch, _ptr(qb), _ptr(kvb), num_slots, mode, float(kv_scale), _ptr(ip),
                           _ptr(ix if ix.size else np.zeros(1, np.int32)), float(sm_scale),
                           None if sids is None else _ptr(sids), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode failed with code {rc}")
    return out, lse


def decode_paged(q, kv, kv_indptr, kv_indices, kv_last_page_len, page_size: int, sm_scale: float, mode: int = 0,
                 kv_scale: float = 1.0, seq_ids=None, lib=None):
    """Oracle MLA decode over a paged KV buffer. Returns (out [n,16,512], lse [n,16]) float64.

    kv: [num_pages * page_size, 576] (the buffer viewed as pages of page_size rows);
    kv_indptr int32 [B+1] in pages; kv_indices int32 page ids; kv_last_page_len
    int32 [B] (None: every last page full).
    """
    lib = lib or load()
    qb = _u16(q).reshape(-1)
    kvb = _kv_bytes(kv, mode)
    ip = _i32(kv_indptr)
    ix = _i32(kv_indices)
    lp = None if kv_last_page_len is None else _i32(kv_last_page_len)
    batch = ip.shape[0] - 1
    sids = None if seq_ids is None else _i32(seq_ids)
    n = batch if sids is None else sids.shape[0]
    out = np.zeros((n, HEADS, V_DIM), dtype=np.float64)
    lse = np.zeros((n, HEADS), dtype=np.float64)
    rc = lib.oracle_decode_paged(batch, _ptr(qb), _ptr(kvb), kvb.size // QK_DIM, mode, float(kv_scale), _ptr(ip),
                                 _ptr(ix if ix.size else np.zeros(1, np.int32)),
                                 None if lp is None else _ptr(lp if lp.size else np.zeros(1, np.int32)),
                                 int(page_size), float(sm_scale), None if sids is None else _ptr(sids), n,
                                 _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode_paged failed with code {rc}")
    return out, lse


def decode_multi(q, kv, qo_indptr, kv_indptr, kv_indices, sm_scale: float, mode: int = 0, kv_scale: float = 1.0,
                 causal: bool = True, kv_last_page_len=None, page_size: int = 1, lib=None):
    """Oracle multi-token decode: q [qo_indptr[B],16,576] -> (out [qo_indptr[B],16,512], lse [..,16]) float64.

    Sequence b's query tokens are rows qo_indptr[b] .. qo_indptr[b+1]-1; with ``causal`` token j sees
    the first L_b - q_b + j + 1 KV tokens. KV addressing as decode_paged (page_size 1 = rows).
    """
    lib = lib or load()
    qb = _u16(q).reshape(-1)
    kvb = _kv_bytes(kv, mode)
    qo = _i32(qo_indptr)
    ip = _i32(kv_indptr)
    ix = _i32(kv_indices)
    lp = None if kv_last_page_len is None else _i32(kv_last_page_len)
    batch = ip.shape[0] - 1
    n = int(qo[-1]) if batch > 0 else 0
    out = np.zeros((n, HEADS, V_DIM), dtype=np.float64)
    lse = np.zeros((n, HEADS), dtype=np.float64)
    rc = lib.oracle_decode_multi(batch, _ptr(qb if qb.size else np.zeros(1, np.uint16)), _ptr(kvb), kvb.size // QK_DIM,
                                 mode, float(kv_scale), _ptr(qo), _ptr(ip),
                                 _ptr(ix if ix.size else np.zeros(1, np.int32)),
                                 None if lp is None else _ptr(lp if lp.size else np.zeros(1, np.int32)),
                                 int(page_size), int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode_multi failed with code {rc}")
    return out, lse


def decode_range(q, kv, kv_indptr, kv_indices, sm_scale: float, b: int, t_begin: int, t_end: int,
                 mode: int = 0, kv_scale: float = 1.0, lib=None):
    """Attention of sequence b over its rows [t_begin, t_end): (out [16,512], lse [16])."""
    lib = lib or load()
    qb = _u16(q).reshape(-1)
    kvb = _kv_bytes(kv, mode)
    ip = _i32(kv_indptr)
    ix = _i32(kv_indices)
    out = np.zeros((HEADS, V_DIM), dtype=np.float64)
    lse = np.zeros((HEADS,), dtype=np.float64)
    rc = lib.oracle_decode_range(ip.shape[0] - 1, _ptr(qb), _ptr(kvb), kvb.size // QK_DIM, mode, float(kv_scale),
                                 _ptr(ip), _ptr(ix if ix.size else np.zeros(1, np.int32)), float(sm_scale),
                                 b, t_begin, t_end, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode_range failed with code {rc}")
    return out, lse


def combine(part_out: np.ndarray, part_lse: np.ndarray, lib=None):
    """Merge per-split (O, LSE) of one sequence: ([S,16,512], [S,16]) -> ([16,512], [16])."""
    lib = lib or load()
    po = np.ascontiguousarray(part_out, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    out = np.zeros((HEADS, V_DIM), dtype=np.float64)
    lse = np.zeros((HEADS,), dtype=np.float64)
    lib.oracle_combine(po.shape[0], _ptr(po), _ptr(pl), _ptr(out), _ptr(lse))
    return out, lse


def q_to_e4m3(q, lib=None) -> np.ndarray:
    """The mode-1 direct cast, element-wise: bf16 -> e4m3 codes (uint8), same shape."""
    lib = lib or load()
    qb = _u16(q)
    out = np.zeros(qb.shape, dtype=np.uint8)
    lib.oracle_q_to_e4m3(_ptr(qb), qb.size, _ptr(out))
    return out


def e4m3_decode_table(lib=None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def threads(lib=None) -> int:
    return (lib or load()).oracle_threads()
