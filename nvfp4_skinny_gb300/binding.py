"""Thin ctypes binding over the C ABI in include/nvfp4_skinny.h, include/nvfp4_prefill.h and
include/nvfp4_pack.h.

Argument marshalling only: every step of the projection runs in the CUDA library
(nvfp4_skinny_gb300/_build/libnvfp4skinny.so).  If that library is missing the
functions raise; there is no fallback path.  Torch tensors are accepted for
device buffers (their data pointers are passed through); streams default to
torch's current CUDA stream.
"""
import ctypes
import os

import numpy as np

from . import build as _build

NVFP4_OK = 0
NVFP4_ERR_ARG = 1
NVFP4_ERR_SHAPE = 2
NVFP4_ERR_ALIGN = 3
NVFP4_ERR_M_RANGE = 4
NVFP4_ERR_CUDA = 5
NVFP4_ERR_NOMEM = 6
NVFP4_ERR_TIMEOUT = 7
NVFP4_ERR_SCRATCH_LIMIT = 8
NVFP4_NOALLOC_MAX_K = 32768
NVFP4_NOALLOC_MAX_N = 4194304
NVFP4_OUT_BF16 = 0
NVFP4_OUT_F32 = 1
NVFP4_MAX_M = 32
NVFP4_ABI_VERSION = 4
NVFP4_KERNEL_TCGEN05 = 0
NVFP4_KERNEL_MMA_SYNC = 1
NVFP4_KERNEL_CLUSTER = 2
NVFP4_PLAN_DEFAULT = 0
NVFP4_PLAN_KERNEL_TCGEN05 = 1
NVFP4_PLAN_KERNEL_MMA_SYNC = 2
NVFP4_PLAN_WEIGHTS_AFTER_WAIT = 4
NVFP4_PLAN_KERNEL_CLUSTER = 8
NVFP4_PLAN_DUAL = 16

NVFP4_PACK_OK = 0
NVFP4_PACK_ERR_ARG = -1
NVFP4_PACK_ERR_VALUE = -2

# every symbol the headers declare, per library
CUDA_SYMBOLS = ("nvfp4_status_string", "nvfp4_abi_version", "nvfp4_plan_create", "nvfp4_plan_create_ex",
                "nvfp4_plan_create_flags", "nvfp4_plan_destroy", "nvfp4_skinny_linear", "nvfp4_plan_check", "nvfp4_plan_get_info",
                "nvfp4_skinny_linear_noalloc", "nvfp4_noalloc_check", "nvfp4_skinny_linear_strided", "nvfp4_skinny_linear_silu_mul",
                "nvfp4_quantize_bf16", "nvfp4_skinny_linear_grouped", "nvfp4_skinny_linear_dual",
                "nvfp4_skinny_linear_deinterleaved", "nvfp4_skinny_linear_grouped_tables")
PREFILL_SYMBOLS = ("nvfp4_prefill_geometry", "nvfp4_prefill_plan_create", "nvfp4_prefill_plan_destroy",
                   "nvfp4_prefill_linear", "nvfp4_prefill_linear_ex", "nvfp4_prefill_plan_check",
                   "nvfp4_prefill_plan_get_info")
PACK_SYMBOLS = ("nvfp4_pack_codes", "nvfp4_unpack_codes", "nvfp4_e4m3_encode", "nvfp4_quantize_bf16_host")
NVFP4_PREFILL_MAX_ROWS = 65536


class GroupItem(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("M", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("w_codes", ctypes.c_void_p), ("w_block_scales", ctypes.c_void_p), ("w_global_scale", ctypes.c_float),
                ("reserved2", ctypes.c_float), ("y", ctypes.c_void_p)]


class Nvfp4Error(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, status, where=""):
        self.status = int(status)
        super().__init__("%s: %s" % (where, _status_string(self.status)) if where else _status_string(self.status))


class PlanInfo(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("out_dtype", ctypes.c_int32),
                ("rows_per_block", ctypes.c_int32), ("k_step", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("grid", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("device", ctypes.c_int32), ("row_blocks", ctypes.c_int64), ("k_steps", ctypes.c_int64),
                ("units", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64), ("smem_bytes", ctypes.c_int64),
                ("launches_per_call", ctypes.c_int32), ("kernel", ctypes.c_int32), ("warps_rows", ctypes.c_int32),
                ("warps_k", ctypes.c_int32), ("flags", ctypes.c_uint32), ("cluster_size", ctypes.c_int32)]


class ExpertTables(ctypes.Structure):
    """nvfp4_expert_tables: six DEVICE arrays of `count` entries each."""
    _fields_ = [("w_codes", ctypes.c_void_p), ("w_block_scales", ctypes.c_void_p), ("w_global_scales", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("M", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class PrefillInfo(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("M", ctypes.c_int32), ("bm", ctypes.c_int32),
                ("m_tiles", ctypes.c_int32), ("n_tiles", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("threads", ctypes.c_int32), ("launches_per_call", ctypes.c_int32),
                ("sm_count", ctypes.c_int32), ("max_M", ctypes.c_int32), ("load_stages", ctypes.c_int32),
                ("k_step", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int64)]


_cuda = None
_pack = None


def _lib_path(path):
    if not os.path.exists(path):
        raise ImportError("%s is not built: run nvfp4_skinny_gb300.build.build() (or __graft_entry__.build())"
                          % path)
    return path


def cuda_lib():
    """The CUDA library, loaded once.  Raises ImportError if it has not been built."""
    global _cuda
    if _cuda is None:
        lib = ctypes.CDLL(_lib_path(_build.CUDA_LIB))
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.nvfp4_status_string.restype = ctypes.c_char_p
        lib.nvfp4_status_string.argtypes = [i32]
        lib.nvfp4_abi_version.restype = i32
        lib.nvfp4_abi_version.argtypes = []
        lib.nvfp4_plan_create.restype = i32
        lib.nvfp4_plan_create.argtypes = [i64, i64, ctypes.POINTER(p)]
        lib.nvfp4_plan_create_ex.restype = i32
        lib.nvfp4_plan_create_ex.argtypes = [i64, i64, i32, ctypes.POINTER(p)]
        lib.nvfp4_plan_create_flags.restype = i32
        lib.nvfp4_plan_create_flags.argtypes = [i64, i64, i32, ctypes.c_uint32, ctypes.POINTER(p)]
        lib.nvfp4_plan_destroy.restype = None
        lib.nvfp4_plan_destroy.argtypes = [p]
        lib.nvfp4_skinny_linear.restype = i32
        lib.nvfp4_skinny_linear.argtypes = [p, p, i32, p, p, ctypes.c_float, p, p]
        lib.nvfp4_plan_check.restype = i32
        lib.nvfp4_plan_check.argtypes = [p, p]
        lib.nvfp4_plan_get_info.restype = i32
        lib.nvfp4_plan_get_info.argtypes = [p, ctypes.POINTER(PlanInfo)]
        lib.nvfp4_skinny_linear_strided.restype = i32
        lib.nvfp4_skinny_linear_strided.argtypes = [p, p, i64, i32, p, p, ctypes.c_float, p, i64, p]
        lib.nvfp4_skinny_linear_silu_mul.restype = i32
        lib.nvfp4_skinny_linear_silu_mul.argtypes = [p, p, i64, i32, p, p, ctypes.c_float, p, i64, p]
        lib.nvfp4_skinny_linear_grouped.restype = i32
        lib.nvfp4_skinny_linear_grouped.argtypes = [p, ctypes.POINTER(GroupItem), i32, p]
        lib.nvfp4_skinny_linear_dual.restype = i32
        lib.nvfp4_skinny_linear_dual.argtypes = [p, p, i32, p, p, ctypes.c_float, p, p, p, ctypes.c_float, p, p]
        lib.nvfp4_skinny_linear_deinterleaved.restype = i32
        lib.nvfp4_skinny_linear_deinterleaved.argtypes = [p, p, i32, p, p, ctypes.c_float, p, i32,
                                                          ctypes.POINTER(ctypes.c_int32), p]
        lib.nvfp4_skinny_linear_grouped_tables.restype = i32
        lib.nvfp4_skinny_linear_grouped_tables.argtypes = [p, ctypes.POINTER(ExpertTables), i32, i32, p]
        lib.nvfp4_quantize_bf16.restype = i32
        lib.nvfp4_quantize_bf16.argtypes = [p, i64, i64, i64, ctypes.c_float, p, p, p]
        lib.nvfp4_skinny_linear_noalloc.restype = i32
        lib.nvfp4_skinny_linear_noalloc.argtypes = [i64, i64, i32, p, i32, p, p, ctypes.c_float, p, p]
        lib.nvfp4_noalloc_check.restype = i32
        lib.nvfp4_noalloc_check.argtypes = [p]
        lib.nvfp4_prefill_geometry.restype = i32
        lib.nvfp4_prefill_geometry.argtypes = [i64, i64, i32, i32, ctypes.POINTER(PrefillInfo)]
        lib.nvfp4_prefill_plan_create.restype = i32
        lib.nvfp4_prefill_plan_create.argtypes = [i64, i64, i32, ctypes.POINTER(p)]
        lib.nvfp4_prefill_plan_destroy.restype = None
        lib.nvfp4_prefill_plan_destroy.argtypes = [p]
        lib.nvfp4_prefill_linear.restype = i32
        lib.nvfp4_prefill_linear.argtypes = [p, p, i32, p, p, ctypes.c_float, p, p]
        lib.nvfp4_prefill_linear_ex.restype = i32
        lib.nvfp4_prefill_linear_ex.argtypes = [p, p, i32, p, p, ctypes.c_float, p, i32, i32, i32, p]
        lib.nvfp4_prefill_plan_check.restype = i32
        lib.nvfp4_prefill_plan_check.argtypes = [p, p]
        lib.nvfp4_prefill_plan_get_info.restype = i32
        lib.nvfp4_prefill_plan_get_info.argtypes = [p, i32, ctypes.POINTER(PrefillInfo)]
        _cuda = lib
    return _cuda


def pack_lib():
    """The host packer library, loaded once.  Raises ImportError if it has not been built."""
    global _pack
    if _pack is None:
        lib = ctypes.CDLL(_lib_path(_build.PACK_LIB))
        p, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.nvfp4_pack_codes.restype = ctypes.c_int
        lib.nvfp4_pack_codes.argtypes = [p, i64, i64, p]
        lib.nvfp4_unpack_codes.restype = ctypes.c_int
        lib.nvfp4_unpack_codes.argtypes = [p, i64, i64, p]
        lib.nvfp4_e4m3_encode.restype = ctypes.c_int
        lib.nvfp4_e4m3_encode.argtypes = [p, i64, p, ctypes.POINTER(i64)]
        lib.nvfp4_quantize_bf16_host.restype = ctypes.c_int
        lib.nvfp4_quantize_bf16_host.argtypes = [p, i64, i64, i64, ctypes.c_float, p, p]
        _pack = lib
    return _pack


def _status_string(status):
    try:
        return cuda_lib().nvfp4_status_string(int(status)).decode()
    except ImportError:
        return "status %d" % int(status)


def _ptr(t):
    """Device (or host) address of a torch tensor, a numpy array or an int; None -> NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    raise TypeError("cannot take the address of %r" % type(t))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != NVFP4_OK:
        raise Nvfp4Error(status, where)


class Plan:
    """Owns an nvfp4_plan_t; destroyed with the object (or by destroy())."""

    def __init__(self, handle, N, K, out_dtype):
        self.handle = handle
        self.N, self.K, self.out_dtype = int(N), int(K), int(out_dtype)

    def destroy(self):
        if self.handle is not None:
            cuda_lib().nvfp4_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    @property
    def as_parameter(self):
        if self.handle is None:
            raise ValueError("plan was destroyed")
        return self.handle


def nvfp4_status_string(status):
    return _status_string(status)


def nvfp4_abi_version():
    return int(cuda_lib().nvfp4_abi_version())


def nvfp4_plan_create(N, K):
    """Plan for an [N, K] NVFP4 weight, bfloat16 output."""
    return nvfp4_plan_create_ex(N, K, NVFP4_OUT_BF16)


def nvfp4_plan_create_ex(N, K, out_dtype=NVFP4_OUT_BF16):
    h = ctypes.c_void_p()
    _check(cuda_lib().nvfp4_plan_create_ex(int(N), int(K), int(out_dtype), ctypes.byref(h)), "nvfp4_plan_create_ex")
    return Plan(h.value, N, K, out_dtype)


def nvfp4_plan_create_flags(N, K, out_dtype=NVFP4_OUT_BF16, flags=NVFP4_PLAN_DEFAULT):
    """Plan with NVFP4_PLAN_* flags (kernel choice, weights read only after the dependency wait)."""
    h = ctypes.c_void_p()
    _check(cuda_lib().nvfp4_plan_create_flags(int(N), int(K), int(out_dtype), int(flags), ctypes.byref(h)),
           "nvfp4_plan_create_flags")
    return Plan(h.value, N, K, out_dtype)


def nvfp4_plan_destroy(plan):
    plan.destroy()


def nvfp4_skinny_linear(plan, x, M, w_codes, w_block_scales, w_global_scale, y, stream=None, check=True):
    """Enqueue y = x . dequant(W)^T.  Returns the status (raises on error when check=True)."""
    st = cuda_lib().nvfp4_skinny_linear(plan.as_parameter if isinstance(plan, Plan) else plan, _ptr(x), int(M),
                                        _ptr(w_codes), _ptr(w_block_scales), float(w_global_scale), _ptr(y),
                                        _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear")
    return st


def nvfp4_skinny_linear_strided(plan, x, lda, M, w_codes, w_block_scales, w_global_scale, y, ldc, stream=None,
                                check=True):
    """As nvfp4_skinny_linear with row strides lda (x) and ldc (y) in elements, so x and y may
    be column slices of wider row-major buffers."""
    st = cuda_lib().nvfp4_skinny_linear_strided(plan.as_parameter if isinstance(plan, Plan) else plan, _ptr(x),
                                                int(lda), int(M), _ptr(w_codes), _ptr(w_block_scales),
                                                float(w_global_scale), _ptr(y), int(ldc), _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear_strided")
    return st


def nvfp4_skinny_linear_silu_mul(plan, gate_up, ld_gate_up, M, w_codes, w_block_scales, w_global_scale, y, ldc,
                                 stream=None, check=True):
    """Down projection of a gated MLP: the input is bf16(silu(gate) * up) of a [gate | up] row."""
    st = cuda_lib().nvfp4_skinny_linear_silu_mul(plan.as_parameter if isinstance(plan, Plan) else plan,
                                                 _ptr(gate_up), int(ld_gate_up), int(M), _ptr(w_codes),
                                                 _ptr(w_block_scales), float(w_global_scale), _ptr(y), int(ldc),
                                                 _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear_silu_mul")
    return st


def nvfp4_skinny_linear_grouped(plan, items, stream=None, check=True):
    """Grouped expert projections: items is a sequence of (x, M, w_codes, w_block_scales,
    w_global_scale, y), all for the plan's (N, K)."""
    arr = (GroupItem * len(items))()
    for i, (x, M, codes, scales, gs, y) in enumerate(items):
        arr[i] = GroupItem(_ptr(x), int(M), 0, _ptr(codes), _ptr(scales), float(gs), 0.0, _ptr(y))
    st = cuda_lib().nvfp4_skinny_linear_grouped(plan.as_parameter if isinstance(plan, Plan) else plan, arr,
                                                len(items), _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear_grouped")
    return st


def nvfp4_skinny_linear_dual(plan, x, M, w0, w1, y0, y1, stream=None, check=True):
    """Two projections of one input in one launch on a NVFP4_PLAN_DUAL plan: w0 and w1 are
    (codes, block_scales, global_scale) triples, y0 and y1 their [M, N] outputs."""
    (c0, s0, g0), (c1, s1, g1) = w0, w1
    st = cuda_lib().nvfp4_skinny_linear_dual(plan.as_parameter if isinstance(plan, Plan) else plan, _ptr(x), int(M),
                                             _ptr(c0), _ptr(s0), float(g0), _ptr(y0), _ptr(c1), _ptr(s1), float(g1),
                                             _ptr(y1), _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear_dual")
    return st


def nvfp4_skinny_linear_deinterleaved(plan, x, M, w_codes, w_block_scales, w_global_scale, y, part_rows, stream=None,
                                      check=True):
    """The projection of a weight whose rows interleave len(part_rows) parts per group, stored
    part-major (Q | gate, or Q | K | V | Z)."""
    rows = (ctypes.c_int32 * len(part_rows))(*[int(r) for r in part_rows])
    st = cuda_lib().nvfp4_skinny_linear_deinterleaved(plan.as_parameter if isinstance(plan, Plan) else plan, _ptr(x),
                                                      int(M), _ptr(w_codes), _ptr(w_block_scales),
                                                      float(w_global_scale), _ptr(y), len(part_rows), rows,
                                                      _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear_deinterleaved")
    return st


def nvfp4_skinny_linear_grouped_tables(plan, tables, count, max_M, stream=None, check=True):
    """Grouped experts in one launch; `tables` maps the six field names of nvfp4_expert_tables to
    device tensors (int64 pointer arrays, float32 scales, int32 row counts)."""
    t = ExpertTables(*[_ptr(tables[f]) for f, _ in ExpertTables._fields_])
    st = cuda_lib().nvfp4_skinny_linear_grouped_tables(plan.as_parameter if isinstance(plan, Plan) else plan,
                                                       ctypes.byref(t), int(count), int(max_M), _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear_grouped_tables")
    return st


def nvfp4_quantize_bf16(w, rows, K, ldw, w_global_scale, w_codes, w_block_scales, stream=None, check=True):
    """Quantize a bfloat16 [rows, K] weight (row stride ldw) to NVFP4 codes and block scales."""
    st = cuda_lib().nvfp4_quantize_bf16(_ptr(w), int(rows), int(K), int(ldw), float(w_global_scale), _ptr(w_codes),
                                        _ptr(w_block_scales), _stream(stream))
    if check:
        _check(st, "nvfp4_quantize_bf16")
    return st


def nvfp4_skinny_linear_noalloc(N, K, out_dtype, x, M, w_codes, w_block_scales, w_global_scale, y, stream=None,
                                check=True):
    """Allocation-free call for callers that cannot allocate device memory: same result as
    nvfp4_skinny_linear, scratch in the library's fixed device array (see the header for its
    size, limits and the rule that calls must not overlap on the GPU)."""
    st = cuda_lib().nvfp4_skinny_linear_noalloc(int(N), int(K), int(out_dtype), _ptr(x), int(M), _ptr(w_codes),
                                                _ptr(w_block_scales), float(w_global_scale), _ptr(y),
                                                _stream(stream))
    if check:
        _check(st, "nvfp4_skinny_linear_noalloc")
    return st


def nvfp4_noalloc_check(stream=None):
    """Synchronise the stream; return and clear the allocation-free scratch's error status."""
    return int(cuda_lib().nvfp4_noalloc_check(_stream(stream)))


def nvfp4_plan_check(plan, stream=None):
    """Synchronise the stream and return the plan's device error status (and clear it)."""
    return int(cuda_lib().nvfp4_plan_check(plan.as_parameter, _stream(stream)))


def nvfp4_plan_get_info(plan):
    info = PlanInfo()
    _check(cuda_lib().nvfp4_plan_get_info(plan.as_parameter, ctypes.byref(info)), "nvfp4_plan_get_info")
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_}


# --------------------------------------------------------------------------- prefill

class PrefillPlan:
    """Owns an nvfp4_prefill_plan_t; destroyed with the object (or by destroy())."""

    def __init__(self, handle, N, K, max_M):
        self.handle = handle
        self.N, self.K, self.max_M = int(N), int(K), int(max_M)

    def destroy(self):
        if self.handle is not None:
            cuda_lib().nvfp4_prefill_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    @property
    def as_parameter(self):
        if self.handle is None:
            raise ValueError("plan was destroyed")
        return self.handle


def _info_dict(info):
    return {f: getattr(info, f) for f, _ in PrefillInfo._fields_}


def nvfp4_prefill_geometry(N, K, M, sm_count):
    """The launch geometry of a prefill call (host-only: no GPU needed)."""
    info = PrefillInfo()
    _check(cuda_lib().nvfp4_prefill_geometry(int(N), int(K), int(M), int(sm_count), ctypes.byref(info)),
           "nvfp4_prefill_geometry")
    return _info_dict(info)


def nvfp4_prefill_plan_create(N, K, max_M):
    """Plan for an [N, K] NVFP4 weight and calls of up to max_M activation rows."""
    h = ctypes.c_void_p()
    _check(cuda_lib().nvfp4_prefill_plan_create(int(N), int(K), int(max_M), ctypes.byref(h)),
           "nvfp4_prefill_plan_create")
    return PrefillPlan(h.value, N, K, max_M)


def nvfp4_prefill_plan_destroy(plan):
    plan.destroy()


def nvfp4_prefill_linear(plan, x, M, w_codes, w_block_scales, w_global_scale, y, stream=None, check=True):
    """Enqueue the prefill projection y = x . dequant(W)^T (M up to the plan's max_M)."""
    st = cuda_lib().nvfp4_prefill_linear(plan.as_parameter if isinstance(plan, PrefillPlan) else plan, _ptr(x),
                                         int(M), _ptr(w_codes), _ptr(w_block_scales), float(w_global_scale), _ptr(y),
                                         _stream(stream))
    if check:
        _check(st, "nvfp4_prefill_linear")
    return st


def nvfp4_prefill_linear_ex(plan, x, M, w_codes, w_block_scales, w_global_scale, y, bm=0, splits=0, k_step=0,
                            stream=None, check=True):
    """nvfp4_prefill_linear with an explicit tile height bm, k-split and k per pipeline step
    (0 = automatic)."""
    st = cuda_lib().nvfp4_prefill_linear_ex(plan.as_parameter if isinstance(plan, PrefillPlan) else plan, _ptr(x),
                                            int(M), _ptr(w_codes), _ptr(w_block_scales), float(w_global_scale),
                                            _ptr(y), int(bm), int(splits), int(k_step), _stream(stream))
    if check:
        _check(st, "nvfp4_prefill_linear_ex")
    return st


def nvfp4_prefill_plan_check(plan, stream=None):
    """Synchronise the stream and return the plan's device error status (and clear it)."""
    return int(cuda_lib().nvfp4_prefill_plan_check(plan.as_parameter, _stream(stream)))


def nvfp4_prefill_plan_get_info(plan, M):
    info = PrefillInfo()
    _check(cuda_lib().nvfp4_prefill_plan_get_info(plan.as_parameter, int(M), ctypes.byref(info)),
           "nvfp4_prefill_plan_get_info")
    return _info_dict(info)


# --------------------------------------------------------------------------- packer

def nvfp4_pack_codes(codes):
    """uint8 [N, K] codes (0..15) -> uint8 [N, K/2] packed (low nibble = even k)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = codes.shape
    out = np.empty((N, K // 2), np.uint8)
    st = pack_lib().nvfp4_pack_codes(codes.ctypes.data, N, K, out.ctypes.data)
    if st != NVFP4_PACK_OK:
        raise ValueError("nvfp4_pack_codes failed with %d" % st)
    return out


def nvfp4_unpack_codes(packed, K):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    out = np.empty((N, K), np.uint8)
    st = pack_lib().nvfp4_unpack_codes(packed.ctypes.data, N, int(K), out.ctypes.data)
    if st != NVFP4_PACK_OK:
        raise ValueError("nvfp4_unpack_codes failed with %d" % st)
    return out


def nvfp4_e4m3_encode(scales):
    """float32 array -> uint8 E4M3 bytes (RNE, saturating at 448).  Raises on NaN / negative."""
    s = np.ascontiguousarray(scales, dtype=np.float32)
    out = np.empty(s.shape, np.uint8)
    bad = ctypes.c_int64(-1)
    st = pack_lib().nvfp4_e4m3_encode(s.ctypes.data, s.size, out.ctypes.data, ctypes.byref(bad))
    if st != NVFP4_PACK_OK:
        raise ValueError("nvfp4_e4m3_encode refused element %d (status %d)" % (bad.value, st))
    return out


def nvfp4_quantize_bf16_host(w_bits, K=None, w_global_scale=1.0):
    """uint16 [rows, ldw] bfloat16 bits (the first K columns are the weight) -> (codes uint8
    [rows, K/2], scales uint8 [rows, K/16]) on the host.  A refused call raises ValueError with
    the library's status in its `status` attribute."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    rows, ldw = w.shape
    K = ldw if K is None else int(K)
    codes = np.zeros((rows, max(K, 0) // 2), np.uint8)
    scales = np.zeros((rows, max(K, 0) // 16), np.uint8)
    st = pack_lib().nvfp4_quantize_bf16_host(w.ctypes.data, rows, K, ldw, float(w_global_scale), codes.ctypes.data,
                                              scales.ctypes.data)
    if st != NVFP4_PACK_OK:
        err = ValueError("nvfp4_quantize_bf16_host refused the call (status %d)" % st)
        err.status = st
        raise err
    return codes, scales
