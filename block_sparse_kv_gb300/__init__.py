"""Python binding of libbskv: CSR-indexed sparse and paged attention on one GB300.

A thin ctypes layer over the C ABI declared in include/bskv.h. Functions carry the
C names; they marshal torch tensors into pointers, strides and the current CUDA
stream, allocate outputs and workspaces with torch when the caller does not pass
them, and raise on any non-OK status. Every step of the computation runs in the
library's CUDA kernels; there is no CPU fallback. Importing works without a GPU
(plans are host code), but the library must have been built (``build()``).
"""

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "BskvError", "Plan", "load_library", "build",
    "bskv_version", "bskv_last_error_message",
    "bskv_plan_decode", "bskv_plan_bsr", "bskv_plan_mla_sparse",
    "bskv_run_decode", "bskv_run_decode_partial", "bskv_decode_merge", "bskv_run_decode_noalloc",
    "bskv_run_bsr", "bskv_run_mla_sparse",
    "bskv_rope_quantize_fp8", "bskv_merge_states",
    "bskv_get_device_status", "bskv_set_debug_force_timeout",
]

FP16, BF16, FP32, E4M3, INT32, INT64 = range(6)
STATUS = {0: "OK", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_WORKSPACE_TOO_SMALL",
          4: "ERR_CUDA", 5: "ERR_TIMEOUT", 6: "ERR_DEVICE_INDEX"}

_DT = {torch.float16: FP16, torch.bfloat16: BF16, torch.float32: FP32, torch.int32: INT32,
       torch.int64: INT64}
if hasattr(torch, "float8_e4m3fn"):
    _DT[torch.float8_e4m3fn] = E4M3


class BskvError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__("%s -> %s: %s" % (fn, STATUS.get(code, code), msg))
        self.code = code
        self.status = STATUS.get(code, str(code))


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_I64P = ctypes.POINTER(ctypes.c_int64)
_I32P = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "bskv_version": ([], _I32),
    "bskv_last_error_message": ([], ctypes.c_char_p),
    "bskv_plan_decode": ([_I32P, _I32P, _I32P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                          _I32, ctypes.POINTER(_P)], _I32),
    "bskv_plan_bsr": ([_I32P, _I32P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                       ctypes.POINTER(_P)], _I32),
    "bskv_plan_prefill_paged": ([_I32P, _I32P, _I32P, _I32P, _I32, _I32, _I32, _I32, _I32,
                                 _I32, _I32, _I32, _I32, ctypes.POINTER(_P)], _I32),
    "bskv_run_prefill_paged": ([_P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _F, _P], _I32),
    "bskv_plan_bsr_variable": ([_P, _I32P, _I32P, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                _I32, ctypes.POINTER(_P)], _I32),
    "bskv_run_bsr_variable": ([_P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _F, _P],
                              _I32),
    "bskv_plan_bsr_masked": ([_I32P, _I32P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                              ctypes.POINTER(_P)], _I32),
    "bskv_run_bsr_masked": ([_P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _SZ, _P, _I64P, _P, _F,
                             _P], _I32),
    "bskv_plan_mla_sparse": ([_I32P, _I32, _I32, _I32, _I32, _I32, ctypes.POINTER(_P)], _I32),
    "bskv_plan_mla_paged": ([_I32P, _I32P, _I32P, _I32, _I32, _I32, _I32, _I32,
                             ctypes.POINTER(_P)], _I32),
    "bskv_plan_destroy": ([_P], _I32),
    "bskv_plan_metadata": ([_P, ctypes.POINTER(_I32P), _I64P], _I32),
    "bskv_plan_workspace_sizes": ([_P, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)], _I32),
    "bskv_plan_upload": ([_P, _P, _SZ, _P], _I32),
    "bskv_run_decode": ([_P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _F, _P, _SZ, _P], _I32),
    "bskv_run_decode_partial": ([_P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _F, _P, _SZ, _P], _I32),
    "bskv_decode_merge": ([_P, _P, _I64P, _P, _P, _SZ, _P], _I32),
    "bskv_run_decode_noalloc": ([_P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _F, _P], _I32),
    "bskv_run_bsr": ([_P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _I64P, _P, _F, _P, _SZ, _P], _I32),
    "bskv_run_mla_sparse": ([_P, _P, _P, _I64, _P, _F, _F, _P, _P, _P, _SZ, _P], _I32),
    "bskv_run_mla_paged": ([_P, _P, _P, _F, _F, _P, _P, _P, _SZ, _P], _I32),
    "bskv_rope_quantize_fp8": ([_P, _I64P, _P, _I64P, _P, _I64, _I32, _P, _I64P, _P, _I64P,
                                _P, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _I64,
                                _I32, _P, _I32, _I64, _I32, _F, _F, _P], _I32),
    "bskv_rope_quantize_fp8_append_paged": ([_P, _I64P, _P, _I64P, _P, _I64, _I32, _P, _I64P,
                                             _P, _I64P, _P, _I64, _P, _I64, _P, _I64, _P, _P,
                                             _P, _P, _I32, _I32, _I64, _P,
                                             _I32, _P, _I32, _I64, _I32, _F, _F, _P], _I32),
    "bskv_merge_states": ([_P, _P, _I64, _I32, _I32, _I32, _P, _I32, _P, _P], _I32),
    "bskv_get_device_status": ([_I32P, _I32], _I32),
    "bskv_set_debug_force_timeout": ([_I32], _I32),
}


def build(force=False):
    """Compile libbskv.so for sm_103a in-tree (nvcc) and load it."""
    global _lib
    _build.build(force=force)
    _lib = None
    return load_library()


def load_library():
    """Load libbskv.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libbskv.so is missing (%s): build it with "
                           "block_sparse_kv_gb300.build() first" % _build.LIB)
    lib = ctypes.CDLL(_build.LIB)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(fn, code):
    if code != 0:
        msg = load_library().bskv_last_error_message().decode(errors="replace")
        raise BskvError(fn, code, msg)


def _i32_array(x):
    t = torch.as_tensor(x, dtype=torch.int32).contiguous().cpu()
    return t, t.data_ptr()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _strides(*vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def _stream(t=None):
    dev = t.device if t is not None and t.is_cuda else None
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _num_sms(device=None):
    if torch.cuda.is_available():
        d = torch.cuda.current_device() if device is None else torch.device(device).index or 0
        return torch.cuda.get_device_properties(d).multi_processor_count
    raise RuntimeError("num_sms must be given when no GPU is visible")


def bskv_version():
    return load_library().bskv_version()


def bskv_last_error_message():
    return load_library().bskv_last_error_message().decode(errors="replace")


class Plan:
    """Host plan handle plus (after upload) its device int workspace."""

    def __init__(self, handle, kind, **info):
        self._h = ctypes.c_void_p(handle)
        self.kind = kind
        self.info = info
        self.int_ws = None
        self.float_ws = None

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.bskv_plan_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    @property
    def handle(self):
        return self._h

    def metadata(self):
        """The plan's int32 metadata words as a Python list."""
        lib = load_library()
        p = _I32P()
        n = ctypes.c_int64()
        _check("bskv_plan_metadata", lib.bskv_plan_metadata(self._h, ctypes.byref(p), ctypes.byref(n)))
        return [p[i] for i in range(n.value)]

    def workspace_sizes(self):
        lib = load_library()
        a, b = ctypes.c_size_t(), ctypes.c_size_t()
        _check("bskv_plan_workspace_sizes",
               lib.bskv_plan_workspace_sizes(self._h, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def upload(self, device="cuda", int_ws=None, float_ws=None):
        """Copy the metadata to the device (allocating the workspaces unless given)."""
        lib = load_library()
        ib, fb = self.workspace_sizes()
        if int_ws is None:
            int_ws = torch.empty(max(ib, 16), dtype=torch.uint8, device=device)
        if float_ws is None and fb > 0:
            float_ws = torch.empty(fb, dtype=torch.uint8, device=device)
        _check("bskv_plan_upload", lib.bskv_plan_upload(self._h, int_ws.data_ptr(),
                                                        int_ws.numel(), _stream(int_ws)))
        self.int_ws = int_ws
        self.float_ws = float_ws
        return self


def bskv_plan_decode(kv_indptr, kv_indices, kv_last_page_len, num_pages, page_size,
                     num_qo_heads, num_kv_heads, head_dim, dtype=torch.bfloat16, num_sms=None,
                     max_workers=0):
    lib = load_library()
    ip, ipp = _i32_array(kv_indptr)
    ix, ixp = _i32_array(kv_indices)
    lp, lpp = _i32_array(kv_last_page_len)
    batch = ip.numel() - 1
    h = ctypes.c_void_p()
    ns = _num_sms() if num_sms is None else num_sms
    _check("bskv_plan_decode", lib.bskv_plan_decode(
        ctypes.cast(ipp, _I32P), ctypes.cast(ixp, _I32P), ctypes.cast(lpp, _I32P), batch,
        int(num_pages), int(page_size), int(num_qo_heads), int(num_kv_heads), int(head_dim),
        _DT[dtype], int(ns), int(max_workers), ctypes.byref(h)))
    return Plan(h.value, "decode", batch=batch, num_qo_heads=num_qo_heads,
                num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype, page_size=page_size)


def bskv_run_decode(plan, q, kv_cache, out=None, lse=None, return_lse=False, sm_scale=None,
                    _entry="bskv_run_decode"):
    """Decode one query token per request; kv_cache [pages, 2, Hkv, page_size, D] (any
    strides with a contiguous last dim)."""
    lib = load_library()
    if plan.int_ws is None:
        plan.upload(q.device)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if sm_scale is None:
        sm_scale = 0.0  # the library applies 1/sqrt(head_dim)
    fw = plan.float_ws
    ks = kv_cache.stride()
    _check(_entry, getattr(lib, _entry)(
        plan.handle, q.data_ptr(), _strides(q.stride(0), q.stride(1)), kv_cache.data_ptr(),
        _strides(ks[0], ks[1], ks[2], ks[3]), out.data_ptr(), _strides(out.stride(0), out.stride(1)),
        _ptr(lse), float(sm_scale), _ptr(fw), 0 if fw is None else fw.numel(), _stream(q)))
    return (out, lse) if return_lse else out


def bskv_run_decode_partial(plan, q, kv_cache, out=None, lse=None, return_lse=False,
                            sm_scale=None):
    """Attention kernel of the decode only (see bskv_decode_merge)."""
    return bskv_run_decode(plan, q, kv_cache, out, lse, return_lse, sm_scale,
                           _entry="bskv_run_decode_partial")


def bskv_decode_merge(plan, out, lse=None):
    """Merge the split-KV partial states a bskv_run_decode_partial left in the plan's
    float workspace into out (and lse)."""
    lib = load_library()
    fw = plan.float_ws
    _check("bskv_decode_merge", lib.bskv_decode_merge(
        plan.handle, out.data_ptr(), _strides(out.stride(0), out.stride(1)), _ptr(lse), _ptr(fw),
        0 if fw is None else fw.numel(), _stream(out)))
    return out


def bskv_run_decode_noalloc(plan, q, kv_cache, out, lse=None, sm_scale=None):
    """Decode without any device allocation by the library or by this call: for callers
    that cannot allocate (see bskv.h). The caller passes the output (and optional lse);
    the plan is not uploaded, its metadata goes into a library-owned static array."""
    lib = load_library()
    B, Hq, D = q.shape
    if plan.kind != "decode" or (B, Hq, D) != (plan.info["batch"], plan.info["num_qo_heads"],
                                                plan.info["head_dim"]):
        raise ValueError("q %s does not match the decode plan" % (tuple(q.shape),))
    if tuple(out.shape) != (B, Hq, D) or out.dtype != plan.info["dtype"] or out.device != q.device:
        raise ValueError("out must be a %s tensor of shape %s on %s"
                         % (plan.info["dtype"], (B, Hq, D), q.device))
    if lse is not None and (tuple(lse.shape) != (B, Hq) or lse.dtype != torch.float32
                            or lse.device != q.device or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 tensor of shape %s on %s"
                         % ((B, Hq), q.device))
    if kv_cache.device != q.device:
        raise ValueError("kv_cache must be on %s" % q.device)
    if sm_scale is None:
        sm_scale = 0.0  # the library applies 1/sqrt(head_dim)
    ks = kv_cache.stride()
    _check("bskv_run_decode_noalloc", lib.bskv_run_decode_noalloc(
        plan.handle, q.data_ptr(), _strides(q.stride(0), q.stride(1)), kv_cache.data_ptr(),
        _strides(ks[0], ks[1], ks[2], ks[3]), out.data_ptr(), _strides(out.stride(0), out.stride(1)),
        _ptr(lse), float(sm_scale), _stream(q)))
    return out


def bskv_plan_bsr(indptr, indices, M, N, R, C, num_qo_heads, num_kv_heads, head_dim,
                  causal=False, dtype=torch.float16, num_sms=None):
    lib = load_library()
    ip, ipp = _i32_array(indptr)
    ix, ixp = _i32_array(indices)
    h = ctypes.c_void_p()
    ns = _num_sms() if num_sms is None else num_sms
    _check("bskv_plan_bsr", lib.bskv_plan_bsr(
        ctypes.cast(ipp, _I32P), ctypes.cast(ixp, _I32P), int(M), int(N), int(R), int(C),
        int(num_qo_heads), int(num_kv_heads), int(head_dim), int(bool(causal)), _DT[dtype],
        int(ns), ctypes.byref(h)))
    return Plan(h.value, "bsr", M=M, N=N, R=R, C=C, num_qo_heads=num_qo_heads,
                num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype)


def bskv_run_bsr(plan, q, k, v, out=None, lse=None, return_lse=False, sm_scale=None):
    lib = load_library()
    if plan.int_ws is None:
        plan.upload(q.device)
    M, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((M, Hq), dtype=torch.float32, device=q.device)
    if sm_scale is None:
        sm_scale = 0.0  # the library applies 1/sqrt(head_dim)
    fw = plan.float_ws
    _check("bskv_run_bsr", lib.bskv_run_bsr(
        plan.handle, q.data_ptr(), _strides(q.stride(0), q.stride(1)), k.data_ptr(),
        _strides(k.stride(0), k.stride(1)), v.data_ptr(), _strides(v.stride(0), v.stride(1)),
        out.data_ptr(), _strides(out.stride(0), out.stride(1)), _ptr(lse), float(sm_scale),
        _ptr(fw), 0 if fw is None else fw.numel(), _stream(q)))
    return (out, lse) if return_lse else out


def bskv_plan_bsr_masked(indptr, indices, M, N, R, C, num_qo_heads, num_kv_heads, head_dim,
                         dtype=torch.float16, num_sms=None):
    """BSR plan whose runs take a per-block token mask (packed bits, bskv_run_bsr_masked)."""
    lib = load_library()
    ip, ipp = _i32_array(indptr)
    ix, ixp = _i32_array(indices)
    h = ctypes.c_void_p()
    ns = _num_sms() if num_sms is None else num_sms
    _check("bskv_plan_bsr_masked", lib.bskv_plan_bsr_masked(
        ctypes.cast(ipp, _I32P), ctypes.cast(ixp, _I32P), int(M), int(N), int(R), int(C),
        int(num_qo_heads), int(num_kv_heads), int(head_dim), _DT[dtype], int(ns),
        ctypes.byref(h)))
    return Plan(h.value, "bsr_masked", M=M, N=N, R=R, C=C, num_qo_heads=num_qo_heads,
                num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype)


def bskv_run_bsr_masked(plan, q, k, v, packed_mask, out=None, lse=None, return_lse=False,
                        sm_scale=None):
    """packed_mask: uint8 device tensor, the (nnz, R, C) mask packed little-endian per byte."""
    lib = load_library()
    if plan.int_ws is None:
        plan.upload(q.device)
    M, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((M, Hq), dtype=torch.float32, device=q.device)
    if sm_scale is None:
        sm_scale = 0.0  # the library applies 1/sqrt(head_dim)
    _check("bskv_run_bsr_masked", lib.bskv_run_bsr_masked(
        plan.handle, q.data_ptr(), _strides(q.stride(0), q.stride(1)), k.data_ptr(),
        _strides(k.stride(0), k.stride(1)), v.data_ptr(), _strides(v.stride(0), v.stride(1)),
        packed_mask.data_ptr(), packed_mask.numel(), out.data_ptr(),
        _strides(out.stride(0), out.stride(1)), _ptr(lse), float(sm_scale), _stream(q)))
    return (out, lse) if return_lse else out


def bskv_plan_bsr_variable(block_mask_map, block_row_sz, block_col_sz, num_qo_heads,
                           num_kv_heads, head_dim, causal=False, dtype=torch.float16,
                           num_sms=None):
    """Variable-block plan: block_mask_map [Hkv, MB, NB] bool, block_row_sz [Hkv, MB],
    block_col_sz [Hkv, NB] int (host copies are made)."""
    lib = load_library()
    bm = torch.as_tensor(block_mask_map).to(torch.uint8).contiguous().cpu()
    rs, rsp = _i32_array(block_row_sz)
    cs, csp = _i32_array(block_col_sz)
    Hkv, MB, NB = bm.shape
    h = ctypes.c_void_p()
    ns = _num_sms() if num_sms is None else num_sms
    _check("bskv_plan_bsr_variable", lib.bskv_plan_bsr_variable(
        ctypes.c_void_p(bm.data_ptr()), ctypes.cast(rsp, _I32P), ctypes.cast(csp, _I32P), int(MB),
        int(NB), int(num_qo_heads), int(num_kv_heads), int(head_dim), int(bool(causal)),
        _DT[dtype], int(ns), ctypes.byref(h)))
    return Plan(h.value, "bsr_variable", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, dtype=dtype, qo_len=int(rs.view(Hkv, MB)[0].sum()))


def bskv_run_bsr_variable(plan, q, k, v, out=None, lse=None, return_lse=False, sm_scale=None):
    """q [Hq, qo_len, D], k/v [Hkv, kv_len, D] -> out [Hq, qo_len, D] (and lse [Hq, qo_len])."""
    lib = load_library()
    if plan.int_ws is None:
        plan.upload(q.device)
    Hq, L, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((Hq, L), dtype=torch.float32, device=q.device)
    if sm_scale is None:
        sm_scale = 0.0  # the library applies 1/sqrt(head_dim)
    _check("bskv_run_bsr_variable", lib.bskv_run_bsr_variable(
        plan.handle, q.data_ptr(), _strides(q.stride(1), q.stride(0)), k.data_ptr(),
        _strides(k.stride(1), k.stride(0)), v.data_ptr(), _strides(v.stride(1), v.stride(0)),
        out.data_ptr(), _strides(out.stride(1), out.stride(0)), _ptr(lse), float(sm_scale),
        _stream(q)))
    return (out, lse) if return_lse else out


def bskv_plan_prefill_paged(qo_indptr, kv_indptr, kv_indices, kv_last_page_len, num_pages,
                            page_size, num_qo_heads, num_kv_heads, head_dim, causal=True,
                            dtype=torch.bfloat16, num_sms=None):
    """Paged prefill plan from HOST ragged query and page-table arrays."""
    lib = load_library()
    qi, qip = _i32_array(qo_indptr)
    ip, ipp = _i32_array(kv_indptr)
    ix, ixp = _i32_array(kv_indices)
    lp, lpp = _i32_array(kv_last_page_len)
    batch = qi.numel() - 1
    h = ctypes.c_void_p()
    ns = _num_sms() if num_sms is None else num_sms
    _check("bskv_plan_prefill_paged", lib.bskv_plan_prefill_paged(
        ctypes.cast(qip, _I32P), ctypes.cast(ipp, _I32P), ctypes.cast(ixp, _I32P),
        ctypes.cast(lpp, _I32P), int(batch), int(num_pages), int(page_size), int(num_qo_heads),
        int(num_kv_heads), int(head_dim), int(bool(causal)), _DT[dtype], int(ns),
        ctypes.byref(h)))
    return Plan(h.value, "prefill_paged", batch=batch, num_qo_heads=num_qo_heads,
                num_kv_heads=num_kv_heads, head_dim=head_dim, dtype=dtype)


def bskv_run_prefill_paged(plan, q, kv_cache, out=None, lse=None, return_lse=False,
                           sm_scale=None):
    """q [total_qo, Hq, D]; kv_cache [pages, 2, Hkv, page_size, D] (any strides)."""
    lib = load_library()
    if plan.int_ws is None:
        plan.upload(q.device)
    T, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
    if sm_scale is None:
        sm_scale = 0.0  # the library applies 1/sqrt(head_dim)
    _check("bskv_run_prefill_paged", lib.bskv_run_prefill_paged(
        plan.handle, q.data_ptr(), _strides(q.stride(0), q.stride(1)), kv_cache.data_ptr(),
        _strides(*kv_cache.stride()[:4]), out.data_ptr(), _strides(out.stride(0), out.stride(1)),
        _ptr(lse), float(sm_scale), _stream(q)))
    return (out, lse) if return_lse else out


def bskv_plan_mla_sparse(seq_lens, batch, q_len, num_heads, top_k, num_sms=None):
    lib = load_library()
    sl, slp = _i32_array(seq_lens)
    h = ctypes.c_void_p()
    ns = _num_sms() if num_sms is None else num_sms
    _check("bskv_plan_mla_sparse", lib.bskv_plan_mla_sparse(
        ctypes.cast(slp, _I32P), int(batch), int(q_len), int(num_heads), int(top_k), int(ns),
        ctypes.byref(h)))
    return Plan(h.value, "mla", batch=batch, q_len=q_len, num_heads=num_heads, top_k=top_k)


def bskv_run_mla_sparse(plan, query, kv_rows, indices, bmm1_scale, bmm2_scale=1.0, out=None,
                        lse=None, return_lse=False):
    """query [B, T, H, 576] uint8/e4m3; kv_rows [rows, 576] (or [pages, page_size, 576])."""
    lib = load_library()
    if plan.int_ws is None:
        plan.upload(query.device)
    B, T, H, _ = query.shape
    rows = kv_rows.numel() // 576
    if out is None:
        out = torch.empty((B, T, H, 512), dtype=torch.bfloat16, device=query.device)
    if lse is None and return_lse:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=query.device)
    fw = plan.float_ws
    _check("bskv_run_mla_sparse", lib.bskv_run_mla_sparse(
        plan.handle, query.data_ptr(), kv_rows.data_ptr(), rows, indices.data_ptr(),
        float(bmm1_scale), float(bmm2_scale), out.data_ptr(), _ptr(lse), _ptr(fw),
        0 if fw is None else fw.numel(), _stream(query)))
    return (out, lse) if return_lse else out


def bskv_plan_mla_paged(kv_indptr, kv_indices, kv_last_page_len, batch, num_pages, page_size,
                        num_heads, num_sms=None):
    """Dense paged MLA decode plan from a HOST CSR page table (one query token per request)."""
    lib = load_library()
    ip, ipp = _i32_array(kv_indptr)
    ix, ixp = _i32_array(kv_indices)
    lp, lpp = _i32_array(kv_last_page_len)
    h = ctypes.c_void_p()
    ns = _num_sms() if num_sms is None else num_sms
    _check("bskv_plan_mla_paged", lib.bskv_plan_mla_paged(
        ctypes.cast(ipp, _I32P), ctypes.cast(ixp, _I32P), ctypes.cast(lpp, _I32P), int(batch),
        int(num_pages), int(page_size), int(num_heads), int(ns), ctypes.byref(h)))
    return Plan(h.value, "mla_paged", batch=batch, num_heads=num_heads, num_pages=num_pages,
                page_size=page_size)


def bskv_run_mla_paged(plan, query, kv_pages, bmm1_scale, bmm2_scale=1.0, out=None, lse=None,
                       return_lse=False):
    """query [B, H, 576] uint8/e4m3; kv_pages [num_pages, page_size, 576] uint8/e4m3."""
    lib = load_library()
    if plan.int_ws is None:
        plan.upload(query.device)
    B, H, _ = query.shape
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=query.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=query.device)
    fw = plan.float_ws
    _check("bskv_run_mla_paged", lib.bskv_run_mla_paged(
        plan.handle, query.data_ptr(), kv_pages.data_ptr(), float(bmm1_scale), float(bmm2_scale),
        out.data_ptr(), _ptr(lse), _ptr(fw), 0 if fw is None else fw.numel(), _stream(query)))
    return (out, lse) if return_lse else out


def bskv_rope_quantize_fp8(q_rope, k_rope, q_nope, k_nope, cos_sin_cache, pos_ids=None,
                           is_neox=True, quant_scale_q=1.0, quant_scale_kv=1.0,
                           q_rope_out=None, k_rope_out=None, q_nope_out=None, k_nope_out=None,
                           pos_ids_k=None):
    """RoPE + FP8 quantisation. pos_ids covers the query rows (and the key rows when
    pos_ids_k is None, the pages' single-nnz form). Outputs are uint8 E4M3 codes."""
    lib = load_library()
    dev = (q_rope if q_rope is not None else k_rope).device
    u8 = torch.uint8
    pos_q = pos_ids
    pos_k = pos_ids if pos_ids_k is None else pos_ids_k
    args = []
    if q_rope is not None:
        nq, H, _ = q_rope.shape
        if q_rope_out is None:
            q_rope_out = torch.empty((nq, H, 64), dtype=u8, device=dev)
        if q_nope_out is None:
            q_nope_out = torch.empty((nq, H, 512), dtype=u8, device=dev)
        args += [q_rope.data_ptr(), _strides(q_rope.stride(0), q_rope.stride(1)), q_nope.data_ptr(),
                 _strides(q_nope.stride(0), q_nope.stride(1)), pos_q.data_ptr(), nq, H,
                 q_rope_out.data_ptr(), _strides(q_rope_out.stride(0), q_rope_out.stride(1)),
                 q_nope_out.data_ptr(), _strides(q_nope_out.stride(0), q_nope_out.stride(1))]
    else:
        args += [None, None, None, None, None, 0, 0, None, None, None, None]
    if k_rope is not None:
        nk = k_rope.shape[0]
        if k_rope_out is None:
            k_rope_out = torch.empty((nk, 64), dtype=u8, device=dev)
        if k_nope_out is None:
            k_nope_out = torch.empty((nk, 512), dtype=u8, device=dev)
        args += [k_rope.data_ptr(), k_rope.stride(0), k_nope.data_ptr(), k_nope.stride(0),
                 pos_k.data_ptr(), nk, k_rope_out.data_ptr(), k_rope_out.stride(0),
                 k_nope_out.data_ptr(), k_nope_out.stride(0)]
    else:
        args += [None, 0, None, 0, None, 0, None, 0, None, 0]
    pos_any = pos_q if pos_q is not None else pos_k
    args += [_DT[pos_any.dtype], cos_sin_cache.data_ptr(), _DT[cos_sin_cache.dtype],
             cos_sin_cache.shape[0], int(bool(is_neox)), float(quant_scale_q),
             float(quant_scale_kv), _stream(cos_sin_cache)]
    _check("bskv_rope_quantize_fp8", lib.bskv_rope_quantize_fp8(*args))
    return q_rope_out, k_rope_out, q_nope_out, k_nope_out


def bskv_rope_quantize_fp8_append_paged(k_rope, k_nope, pos_k, cos_sin_cache, batch_indices,
                                        positions, kv_indptr, kv_indices, kv_pages,
                                        q_rope=None, q_nope=None, pos_q=None, is_neox=True,
                                        quant_scale_q=1.0, quant_scale_kv=1.0, q_rope_out=None,
                                        q_nope_out=None):
    """RoPE + FP8 with the key rows written into kv_pages [num_pages, page_size, 576] (uint8)
    through the device page table (int32 batch_indices, positions, kv_indptr, kv_indices).
    The optional query group is handled as by bskv_rope_quantize_fp8. Returns the query
    outputs (or None)."""
    lib = load_library()
    dev = k_rope.device
    u8 = torch.uint8
    args = []
    if q_rope is not None:
        nq, H, _ = q_rope.shape
        if q_rope_out is None:
            q_rope_out = torch.empty((nq, H, 64), dtype=u8, device=dev)
        if q_nope_out is None:
            q_nope_out = torch.empty((nq, H, 512), dtype=u8, device=dev)
        args += [q_rope.data_ptr(), _strides(q_rope.stride(0), q_rope.stride(1)), q_nope.data_ptr(),
                 _strides(q_nope.stride(0), q_nope.stride(1)), pos_q.data_ptr(), nq, H,
                 q_rope_out.data_ptr(), _strides(q_rope_out.stride(0), q_rope_out.stride(1)),
                 q_nope_out.data_ptr(), _strides(q_nope_out.stride(0), q_nope_out.stride(1))]
    else:
        args += [None, None, None, None, None, 0, 0, None, None, None, None]
    num_pages, page_size, _ = kv_pages.shape
    batch = kv_indptr.numel() - 1
    args += [k_rope.data_ptr(), k_rope.stride(0), k_nope.data_ptr(), k_nope.stride(0),
             pos_k.data_ptr(), k_rope.shape[0], batch_indices.data_ptr(), positions.data_ptr(),
             kv_indptr.data_ptr(), kv_indices.data_ptr(), int(batch), int(page_size),
             int(num_pages), kv_pages.data_ptr(),
             _DT[pos_k.dtype], cos_sin_cache.data_ptr(), _DT[cos_sin_cache.dtype],
             cos_sin_cache.shape[0], int(bool(is_neox)), float(quant_scale_q),
             float(quant_scale_kv), _stream(cos_sin_cache)]
    _check("bskv_rope_quantize_fp8_append_paged", lib.bskv_rope_quantize_fp8_append_paged(*args))
    return q_rope_out, q_nope_out


def bskv_merge_states(v, s, out_dtype=torch.float32, v_out=None, s_out=None):
    """v [seq, S, H, D] float32, s [seq, S, H] float32 -> (v_out [seq, H, D], s_out [seq, H])."""
    lib = load_library()
    seq, S, H, D = v.shape
    v = v.contiguous()
    s = s.contiguous()
    if v_out is None:
        v_out = torch.empty((seq, H, D), dtype=out_dtype, device=v.device)
    if s_out is None:
        s_out = torch.empty((seq, H), dtype=torch.float32, device=v.device)
    _check("bskv_merge_states", lib.bskv_merge_states(
        v.data_ptr(), s.data_ptr(), seq, S, H, D, v_out.data_ptr(), _DT[v_out.dtype],
        s_out.data_ptr(), _stream(v)))
    return v_out, s_out


def bskv_get_device_status(reset=True):
    lib = load_library()
    st = ctypes.c_int32()
    _check("bskv_get_device_status", lib.bskv_get_device_status(ctypes.byref(st), int(bool(reset))))
    return st.value


def bskv_set_debug_force_timeout(on):
    _check("bskv_set_debug_force_timeout", load_library().bskv_set_debug_force_timeout(int(bool(on))))
