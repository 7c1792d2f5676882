"""GB300 (sm_103a) MLA decode: Python binding of libmla_decode.so.

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels (stage 1 + split reduce) behind the C ABI declared in
``include/mla_decode.h``. PyTorch supplies device memory and streams. There is
no fallback: if the compiled library is missing or cannot be loaded, every
call raises.

    import mla_decode_attention_09_gb300 as mla
    plan = mla.plan(kv_indptr_host)                     # host split-KV planner (cached)
    out = mla.decode(q, kv, kv_scale, kv_indptr, kv_indices, plan=plan)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

HEADS = 16
QK_DIM = 576
V_DIM = 512
SM_SCALE = 1.0 / math.sqrt(QK_DIM)
MODE_BF16 = 0
MODE_FP8 = 1
MODE_A16W8 = 2  # bf16 q x e4m3 kv (pass dtype_mode explicitly: kv bytes alone do not tell it from MODE_FP8)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_decode.so")

MLA_OK = 0
STATUS = {
    0: "MLA_OK", -1: "MLA_ERR_ARG", -2: "MLA_ERR_DTYPE", -3: "MLA_ERR_PLAN_MISMATCH", -4: "MLA_ERR_CUDA",
    -5: "MLA_ERR_TIMEOUT", -6: "MLA_ERR_ALIGN", -7: "MLA_ERR_NOMEM", -8: "MLA_ERR_INDEX", -9: "MLA_ERR_DEVICE",
    -10: "MLA_ERR_INDPTR", -11: "MLA_ERR_NOALLOC_LIMIT",
}

# Every symbol include/mla_decode.h declares.
EXPORTS = (
    "mla_decode_plan", "mla_decode_plan_ex", "mla_plan_release", "mla_plan_get_info", "mla_plan_destroy",
    "mla_plan_workspace_bytes", "mla_decode",
    "mla_decode_stage1", "mla_decode_reduce", "mla_plan_check_error", "mla_strerror", "mla_version",
    "mla_plan_compute_host", "mla_decode_noalloc", "mla_decode_plan_paged", "mla_decode_paged",
    "mla_plan_compute_host_paged", "mla_decode_plan_multi", "mla_decode_multi", "mla_plan_compute_host_multi",
)


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_strerror(status)})")


class PlanOptions(ctypes.Structure):
    _fields_ = [("num_kv_slots", ctypes.c_int64), ("min_rows_per_split", ctypes.c_int),
                ("granularity", ctypes.c_int), ("ctas_per_sm", ctypes.c_int), ("fp8_kernel", ctypes.c_int),
                ("fp8_issuers", ctypes.c_int), ("item_cost_rows", ctypes.c_int),
                ("token_parallel", ctypes.c_int), ("token_pairs", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("num_ctas", ctypes.c_int), ("num_work_items", ctypes.c_int),
                ("num_partial_slots", ctypes.c_int), ("num_split_seqs", ctypes.c_int), ("device", ctypes.c_int),
                ("total_rows", ctypes.c_int64), ("max_rows_per_cta", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("token_pairs", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load libmla_decode.so (raises OSError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError(f"{p} not found: build it with `python -m mla_decode_attention_09_gb300.build`")
        lib = ctypes.CDLL(p)
        V, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.mla_decode_plan.argtypes = [I, V, I, ctypes.POINTER(V)]
        lib.mla_decode_plan_ex.argtypes = [I, V, I, ctypes.POINTER(PlanOptions), ctypes.POINTER(V)]
        lib.mla_plan_release.argtypes = [V]
        lib.mla_plan_get_info.argtypes = [V, ctypes.POINTER(PlanInfo)]
        lib.mla_plan_destroy.argtypes = [V]
        lib.mla_plan_workspace_bytes.argtypes = [V]
        lib.mla_plan_workspace_bytes.restype = ctypes.c_size_t
        dec = [V, V, V, V, V, V, F, I, V, V]
        lib.mla_decode.argtypes = dec
        lib.mla_decode_stage1.argtypes = dec
        lib.mla_decode_reduce.argtypes = [V, V, V]
        lib.mla_plan_check_error.argtypes = [V, V]
        lib.mla_strerror.argtypes = [I]
        lib.mla_strerror.restype = ctypes.c_char_p
        lib.mla_version.argtypes = []
        lib.mla_plan_compute_host.argtypes = [I, V, I, ctypes.POINTER(PlanOptions), V, V, I, V, I, V, I]
        lib.mla_decode_noalloc.argtypes = [V, V, V, V, V, V, I, I64, V, F, I, V, V]
        lib.mla_decode_plan_paged.argtypes = [I, V, V, I, I, ctypes.POINTER(PlanOptions), ctypes.POINTER(V)]
        lib.mla_decode_paged.argtypes = [V, V, V, V, V, V, I, V, F, I, V, V]
        lib.mla_plan_compute_host_paged.argtypes = [I, V, V, I, I, ctypes.POINTER(PlanOptions), V, V, I, V, I, V,
                                                    I]
        lib.mla_decode_plan_multi.argtypes = [I, V, V, V, I, I, I, ctypes.POINTER(PlanOptions), ctypes.POINTER(V)]
        lib.mla_decode_multi.argtypes = [V, V, V, V, V, V, V, I, V, F, I, V, V]
        lib.mla_plan_compute_host_multi.argtypes = [I, V, V, V, I, I, I, ctypes.POINTER(PlanOptions), V, V, I, V, I,
                                                    V, I]
        for name in EXPORTS:
            if name not in ("mla_strerror", "mla_plan_workspace_bytes"):
                getattr(lib, name).restype = I
        if path is None:
            _lib = lib
        return lib


def _strerror(status: int) -> str:
    try:
        return load_library().mla_strerror(status).decode()
    except OSError:
        return "library not loaded"


def _check(status: int, what: str):
    if status != MLA_OK:
        raise MLAError(status, what)


def _opts(num_kv_slots=0, min_rows_per_split=0, granularity=0, ctas_per_sm=0, fp8_kernel=0,
          fp8_issuers=0, item_cost_rows=0, token_parallel=0, token_pairs=0) -> PlanOptions:
    return PlanOptions(int(num_kv_slots), int(min_rows_per_split), int(granularity), int(ctas_per_sm),
                       int(fp8_kernel), int(fp8_issuers), int(item_cost_rows), int(token_parallel),
                       int(token_pairs))


def _host_indptr(kv_indptr) -> torch.Tensor:
    t = kv_indptr if isinstance(kv_indptr, torch.Tensor) else torch.as_tensor(kv_indptr)
    return t.detach().to("cpu", torch.int32).contiguous()


class Plan:
    """A split-KV plan (work list, reduce map and partial workspace) owned by the library.

    With ``page_size`` given the plan is for the paged layout (kv_indptr counts
    pages, ``kv_last_page_len_host`` the tokens of each last page) and serves
    decode_paged only.
    """

    def __init__(self, kv_indptr_host, num_sms: int = 0, *, page_size: int | None = None,
                 kv_last_page_len_host=None, qo_indptr_host=None, causal: bool = True, **options):
        lib = load_library()
        ip = _host_indptr(kv_indptr_host)
        self.batch = ip.numel() - 1
        self._lib = lib
        self._handle = ctypes.c_void_p()
        o = _opts(**options)
        self.multi = qo_indptr_host is not None
        self.paged = page_size is not None and not self.multi
        self.page_size = int(page_size) if page_size is not None else 1
        self.causal = bool(causal)
        if self.multi:
            qo = _host_indptr(qo_indptr_host)
            lp = None if kv_last_page_len_host is None else _host_indptr(kv_last_page_len_host)
            _check(lib.mla_decode_plan_multi(self.batch, qo.data_ptr(), ip.data_ptr(),
                                             None if lp is None else lp.data_ptr(), self.page_size,
                                             int(self.causal), int(num_sms), ctypes.byref(o),
                                             ctypes.byref(self._handle)), "mla_decode_plan_multi")
            self.qo_indptr_host = qo
            self.num_q_rows = int(qo[-1]) if self.batch > 0 else 0
        elif self.paged:
            lp = None if kv_last_page_len_host is None else _host_indptr(kv_last_page_len_host)
            _check(lib.mla_decode_plan_paged(self.batch, ip.data_ptr(), None if lp is None else lp.data_ptr(),
                                             self.page_size, int(num_sms), ctypes.byref(o),
                                             ctypes.byref(self._handle)), "mla_decode_plan_paged")
            self.kv_last_page_len_host = lp
        else:
            _check(lib.mla_decode_plan_ex(self.batch, ip.data_ptr(), int(num_sms), ctypes.byref(o),
                                          ctypes.byref(self._handle)), "mla_decode_plan")
        self.kv_indptr_host = ip

    @property
    def handle(self):
        return self._handle

    @property
    def token_pairs(self) -> bool:
        """The plan also holds a token-pair work list (used by fp8 decodes on the tensor-core kernel)."""
        return bool(self.info()["token_pairs"])

    def info(self) -> dict:
        inf = PlanInfo()
        _check(self._lib.mla_plan_get_info(self._handle, ctypes.byref(inf)), "mla_plan_get_info")
        return inf.as_dict()

    def check_error(self, stream=None) -> int:
        """Synchronise the stream and return (and clear) the kernels' error status."""
        return self._lib.mla_plan_check_error(self._handle, _stream_ptr(stream))

    def release(self):
        if self._handle:
            self._lib.mla_plan_release(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.release()
        except Exception:
            pass


def plan(kv_indptr_host, num_sms: int = 0, **options) -> Plan:
    """Build (or fetch from the library's cache) the plan for this batch layout."""
    return Plan(kv_indptr_host, num_sms, **options)


def plan_paged(kv_indptr_host, kv_last_page_len_host, page_size: int, num_sms: int = 0, **options) -> Plan:
    """Plan for the paged layout: kv_indptr in pages of ``page_size`` tokens,
    ``kv_last_page_len_host`` [B] the tokens used in each sequence's last page."""
    return Plan(kv_indptr_host, num_sms, page_size=page_size, kv_last_page_len_host=kv_last_page_len_host,
                **options)


def plan_multi(qo_indptr_host, kv_indptr_host, num_sms: int = 0, *, causal: bool = True, page_size: int = 1,
               kv_last_page_len_host=None, **options) -> Plan:
    """Plan for several query tokens per sequence (rows qo_indptr[b] .. of q and out)."""
    return Plan(kv_indptr_host, num_sms, page_size=page_size, kv_last_page_len_host=kv_last_page_len_host,
                qo_indptr_host=qo_indptr_host, causal=causal, **options)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _mode_of(kv: torch.Tensor) -> int:
    if kv.dtype == torch.bfloat16:
        return MODE_BF16
    if kv.dtype in (torch.uint8, torch.float8_e4m3fn):
        return MODE_FP8
    raise ValueError(f"kv dtype {kv.dtype} not supported (bf16, or e4m3 bytes as uint8 / float8_e4m3fn)")


def _validate(q, kv, kv_scale, kv_indptr, kv_indices, out, mode, p: Plan):
    if q.dtype != torch.bfloat16 or q.dim() != 3 or tuple(q.shape[1:]) != (HEADS, QK_DIM):
        raise ValueError(f"q must be bf16 [B,{HEADS},{QK_DIM}], got {q.dtype} {tuple(q.shape)}")
    if kv.dim() != 2 or kv.shape[1] != QK_DIM:
        raise ValueError(f"kv must be [slots,{QK_DIM}], got {tuple(kv.shape)}")
    if q.shape[0] != p.batch or kv_indptr.numel() != p.batch + 1:
        raise ValueError("batch of q / kv_indptr does not match the plan")
    if out.dtype != torch.bfloat16 or tuple(out.shape) != (p.batch, HEADS, V_DIM):
        raise ValueError(f"out must be bf16 [B,{HEADS},{V_DIM}]")
    for name, t in (("q", q), ("kv", kv), ("kv_indptr", kv_indptr), ("kv_indices", kv_indices), ("out", out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if kv_indptr.dtype != torch.int32 or kv_indices.dtype != torch.int32:
        raise ValueError("kv_indptr and kv_indices must be int32")
    if mode != MODE_BF16 and (kv_scale is None or kv_scale.dtype != torch.float32 or not kv_scale.is_cuda):
        raise ValueError("fp8 KV needs kv_scale as a float32 CUDA tensor of one element")


def _call(fn, q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale, mode, p, stream):
    ks = kv_scale.data_ptr() if kv_scale is not None else None
    return fn(q.data_ptr(), kv.data_ptr(), ks, kv_indptr.data_ptr(), kv_indices.data_ptr(), out.data_ptr(),
              float(sm_scale), int(mode), p.handle, _stream_ptr(stream))


def decode(q, kv, kv_scale, kv_indptr, kv_indices, out=None, *, sm_scale: float = SM_SCALE, dtype_mode=None,
           plan: Plan | None = None, stream=None, validate: bool = True) -> torch.Tensor:
    """One MLA decode call (stage 1 + reduce) on the current CUDA stream.

    q bf16 [B,16,576]; kv bf16 [slots,576] or e4m3 bytes [slots,576] (uint8 or
    float8_e4m3fn view) with kv_scale a float32 [1] CUDA tensor; kv_indptr int32
    [B+1] and kv_indices int32 [R] on the device. Without ``plan`` one is built
    from a host copy of kv_indptr (a device-to-host read).
    """
    mode = _mode_of(kv) if dtype_mode is None else int(dtype_mode)
    p = plan if plan is not None else Plan(kv_indptr, num_kv_slots=kv.shape[0])
    if out is None:
        out = torch.empty((p.batch, HEADS, V_DIM), dtype=torch.bfloat16, device=q.device)
    if validate:
        _validate(q, kv, kv_scale, kv_indptr, kv_indices, out, mode, p)
    _check(_call(load_library().mla_decode, q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale, mode, p,
                 stream), "mla_decode")
    return out


def decode_paged(q, kv, kv_scale, kv_indptr, kv_indices, kv_last_page_len, page_size: int, out=None, *,
                 sm_scale: float = SM_SCALE, dtype_mode=None, plan: Plan | None = None, stream=None,
                 validate: bool = True) -> torch.Tensor:
    """MLA decode over the paged layout: kv [num_pages * page_size, 576], kv_indptr
    int32 [B+1] page offsets, kv_indices int32 page ids and kv_last_page_len int32
    [B] on the device. Without ``plan`` one is built from host copies."""
    mode = _mode_of(kv) if dtype_mode is None else int(dtype_mode)
    p = plan if plan is not None else plan_paged(kv_indptr, kv_last_page_len, page_size, num_kv_slots=kv.shape[0])
    if out is None:
        out = torch.empty((p.batch, HEADS, V_DIM), dtype=torch.bfloat16, device=q.device)
    if validate:
        _validate(q, kv, kv_scale, kv_indptr, kv_indices, out, mode, p)
        if page_size > 1 and (kv_last_page_len is None or kv_last_page_len.dtype != torch.int32
                              or not kv_last_page_len.is_cuda or kv_last_page_len.numel() != p.batch):
            raise ValueError("kv_last_page_len must be an int32 CUDA tensor [B]")
    ks = kv_scale.data_ptr() if kv_scale is not None else None
    lp = kv_last_page_len.data_ptr() if kv_last_page_len is not None else None
    _check(load_library().mla_decode_paged(q.data_ptr(), kv.data_ptr(), ks, kv_indptr.data_ptr(),
                                           kv_indices.data_ptr(), lp, int(page_size), out.data_ptr(),
                                           float(sm_scale), int(mode), p.handle, _stream_ptr(stream)),
           "mla_decode_paged")
    return out


def decode_multi(q, kv, kv_scale, qo_indptr, kv_indptr, kv_indices, out=None, *, plan: Plan,
                 kv_last_page_len=None, sm_scale: float = SM_SCALE, dtype_mode=None, stream=None,
                 validate: bool = True) -> torch.Tensor:
    """Decode of several query tokens per sequence: q bf16 [qo_indptr[B],16,576] -> out bf16
    [qo_indptr[B],16,512], with a plan from plan_multi (its page size and causal flag apply)."""
    mode = _mode_of(kv) if dtype_mode is None else int(dtype_mode)
    if out is None:
        out = torch.empty((plan.num_q_rows, HEADS, V_DIM), dtype=torch.bfloat16, device=q.device)
    if validate:
        if not plan.multi:
            raise ValueError("decode_multi needs a plan from plan_multi")
        if q.dtype != torch.bfloat16 or tuple(q.shape) != (plan.num_q_rows, HEADS, QK_DIM):
            raise ValueError(f"q must be bf16 [{plan.num_q_rows},{HEADS},{QK_DIM}]")
        if out.dtype != torch.bfloat16 or tuple(out.shape) != (plan.num_q_rows, HEADS, V_DIM):
            raise ValueError(f"out must be bf16 [{plan.num_q_rows},{HEADS},{V_DIM}]")
        for name, t in (("q", q), ("kv", kv), ("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr),
                        ("kv_indices", kv_indices), ("out", out)):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if qo_indptr.dtype != torch.int32 or qo_indptr.numel() != plan.batch + 1:
            raise ValueError("qo_indptr must be int32 [B+1]")
        if mode != MODE_BF16 and (kv_scale is None or kv_scale.dtype != torch.float32 or not kv_scale.is_cuda):
            raise ValueError("fp8 KV needs kv_scale as a float32 CUDA tensor of one element")
    ks = kv_scale.data_ptr() if kv_scale is not None else None
    lp = kv_last_page_len.data_ptr() if kv_last_page_len is not None else None
    _check(load_library().mla_decode_multi(q.data_ptr(), kv.data_ptr(), ks, qo_indptr.data_ptr(), kv_indptr.data_ptr(),
                                           kv_indices.data_ptr(), lp, int(plan.page_size), out.data_ptr(),
                                           float(sm_scale), int(mode), plan.handle, _stream_ptr(stream)),
           "mla_decode_multi")
    return out


def decode_stage1(q, kv, kv_scale, kv_indptr, kv_indices, out, *, plan: Plan, sm_scale: float = SM_SCALE,
                  dtype_mode=None, stream=None) -> torch.Tensor:
    """Only the persistent stage-1 kernel (final rows of unsplit sequences + partials)."""
    mode = _mode_of(kv) if dtype_mode is None else int(dtype_mode)
    _validate(q, kv, kv_scale, kv_indptr, kv_indices, out, mode, plan)
    _check(_call(load_library().mla_decode_stage1, q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale, mode,
                 plan, stream), "mla_decode_stage1")
    return out


def decode_reduce(out, *, plan: Plan, stream=None) -> torch.Tensor:
    """Only the split reduce: merges the plan's partials into out."""
    _check(load_library().mla_decode_reduce(out.data_ptr(), plan.handle, _stream_ptr(stream)), "mla_decode_reduce")
    return out


def plan_compute_host(kv_indptr_host, num_sms: int, **options) -> dict:
    """The planner alone on the host (no GPU needed): items, work_indptr and reduce map as numpy arrays."""
    import numpy as np

    lib = load_library()
    ip = _host_indptr(kv_indptr_host)
    batch = ip.numel() - 1
    o = _opts(**options)
    counts = np.zeros(4, dtype=np.int32)
    _check(lib.mla_plan_compute_host(batch, ip.data_ptr(), int(num_sms), ctypes.byref(o),
                                     counts.ctypes.data, None, 0, None, 0, None, 0), "mla_plan_compute_host")
    n_items, n_ctas, n_slots, n_reduce = (int(x) for x in counts)
    items = np.zeros((max(n_items, 1), 5), dtype=np.int32)
    wip = np.zeros(n_ctas + 1, dtype=np.int32)
    red = np.zeros((max(n_reduce, 1), 3), dtype=np.int32)
    _check(lib.mla_plan_compute_host(batch, ip.data_ptr(), int(num_sms), ctypes.byref(o), counts.ctypes.data,
                                     items.ctypes.data, items.shape[0], wip.ctypes.data, wip.shape[0],
                                     red.ctypes.data, red.shape[0]), "mla_plan_compute_host")
    return {"items": items[:n_items], "work_indptr": wip, "reduce": red[:n_reduce], "num_ctas": n_ctas,
            "num_slots": n_slots}


def plan_compute_host_paged(kv_indptr_host, kv_last_page_len_host, page_size: int, num_sms: int,
                            **options) -> dict:
    """plan_compute_host for the paged layout (item offsets are tokens)."""
    import numpy as np

    lib = load_library()
    ip = _host_indptr(kv_indptr_host)
    lp = None if kv_last_page_len_host is None else _host_indptr(kv_last_page_len_host)
    lpp = None if lp is None else lp.data_ptr()
    batch = ip.numel() - 1
    o = _opts(**options)
    counts = np.zeros(4, dtype=np.int32)
    _check(lib.mla_plan_compute_host_paged(batch, ip.data_ptr(), lpp, int(page_size), int(num_sms), ctypes.byref(o),
                                           counts.ctypes.data, None, 0, None, 0, None, 0),
           "mla_plan_compute_host_paged")
    n_items, n_ctas, n_slots, n_reduce = (int(x) for x in counts)
    items = np.zeros((max(n_items, 1), 5), dtype=np.int32)
    wip = np.zeros(n_ctas + 1, dtype=np.int32)
    red = np.zeros((max(n_reduce, 1), 3), dtype=np.int32)
    _check(lib.mla_plan_compute_host_paged(batch, ip.data_ptr(), lpp, int(page_size), int(num_sms), ctypes.byref(o),
                                           counts.ctypes.data, items.ctypes.data, items.shape[0], wip.ctypes.data,
                                           wip.shape[0], red.ctypes.data, red.shape[0]),
           "mla_plan_compute_host_paged")
    return {"items": items[:n_items], "work_indptr": wip, "reduce": red[:n_reduce], "num_ctas": n_ctas,
            "num_slots": n_slots}


def plan_compute_host_multi(qo_indptr_host, kv_indptr_host, num_sms: int, *, causal: bool = True,
                            page_size: int = 1, kv_last_page_len_host=None, **options) -> dict:
    """plan_compute_host for multi-token plans; items have 8 fields (..., query row, query token, pair
    field) and reduce entries 4 (..., slot stride)."""
    import numpy as np

    lib = load_library()
    qo = _host_indptr(qo_indptr_host)
    ip = _host_indptr(kv_indptr_host)
    lp = None if kv_last_page_len_host is None else _host_indptr(kv_last_page_len_host)
    lpp = None if lp is None else lp.data_ptr()
    batch = ip.numel() - 1
    o = _opts(**options)
    counts = np.zeros(4, dtype=np.int32)
    args = (batch, qo.data_ptr(), ip.data_ptr(), lpp, int(page_size), int(bool(causal)), int(num_sms), ctypes.byref(o))
    _check(lib.mla_plan_compute_host_multi(*args, counts.ctypes.data, None, 0, None, 0, None, 0),
           "mla_plan_compute_host_multi")
    n_items, n_ctas, n_slots, n_reduce = (int(x) for x in counts)
    items = np.zeros((max(n_items, 1), 8), dtype=np.int32)
    wip = np.zeros(n_ctas + 1, dtype=np.int32)
    red = np.zeros((max(n_reduce, 1), 4), dtype=np.int32)
    _check(lib.mla_plan_compute_host_multi(*args, counts.ctypes.data, items.ctypes.data, items.shape[0],
                                           wip.ctypes.data, wip.shape[0], red.ctypes.data, red.shape[0]),
           "mla_plan_compute_host_multi")
    return {"items": items[:n_items], "work_indptr": wip, "reduce": red[:n_reduce], "num_ctas": n_ctas,
            "num_slots": n_slots}


def version() -> int:
    return load_library().mla_version()
