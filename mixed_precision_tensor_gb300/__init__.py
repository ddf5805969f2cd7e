"""Python binding of libtcg, the GB300 (sm_103a) mixed-precision tensor-core GEMM.

D = alpha * op(A) * op(B) + beta * C with FP16/BF16 (or TF32-rounded FP32)
inputs, exact products, FP32 accumulation and an FP32 or round-to-nearest-even
FP16/BF16 output.  The C ABI is declared in ``include/tcg.h``; this module only
marshals arguments into it (ctypes).  PyTorch is used for device memory and
streams.  Every step of the GEMM runs in the library's CUDA kernels: if the
in-tree ``_lib/libtcg.so`` is missing, calls raise -- there is no fallback.

Names mirror the C ABI: ``tcg_create``, ``tcg_destroy``, ``tcg_set_stream``,
``tcg_set_workspace``, ``tcg_gemm_workspace_size``, ``tcg_gemm_ex``,
``tcg_gemm_strided_batched``, ``tcg_get_device_error``, ``tcg_status_string``,
``tcg_set_debug``, ``tcg_launch_count``.  ``Handle`` and ``gemm_rowmajor`` are
conveniences on top of them.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libtcg.so")

# enums (include/tcg.h)
TCG_STATUS_SUCCESS = 0
TCG_STATUS_NOT_INITIALIZED = 1
TCG_STATUS_INVALID_VALUE = 2
TCG_STATUS_NOT_SUPPORTED = 3
TCG_STATUS_ARCH_MISMATCH = 4
TCG_STATUS_EXECUTION_FAILED = 5
TCG_STATUS_TIMEOUT = 6
TCG_STATUS_ALLOC_FAILED = 7
TCG_OP_N, TCG_OP_T = 0, 1
TCG_R_16F, TCG_R_16BF, TCG_R_32F, TCG_R_8F_E4M3, TCG_R_8F_E5M2 = 0, 1, 2, 3, 4
TCG_COMPUTE_32F, TCG_COMPUTE_32F_FAST_TF32, TCG_COMPUTE_32F_3XTF32 = 0, 1, 2

EXPORTS = ("tcg_create", "tcg_destroy", "tcg_set_stream", "tcg_set_workspace",
           "tcg_gemm_workspace_size", "tcg_gemm_ex", "tcg_gemm_strided_batched",
           "tcg_get_device_error", "tcg_last_device_error_bits", "tcg_status_string",
           "tcg_set_debug", "tcg_launch_count", "tcg_set_kernel_options",
           "tcg_gemm_tf32_noalloc", "tcg_noalloc_device_error", "tcg_set_clock_probe",
           "tcg_read_clock_probe", "tcg_set_split_k", "tcg_split_k_plan",
           "tcg_gemm_split_k", "tcg_gemm_ex_host", "tcg_gemm_strided_batched_host",
           "tcg_tail_split_plan", "tcg_gemm_tile_plan", "tcg_set_tile_n",
           "tcg_set_tf32_rounding")

_lock = threading.Lock()
_lib = None


class TcgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {tcg_status_string(status)}" if what else
                         tcg_status_string(status))


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the in-tree libtcg.so (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libtcg.so not found at {p}; build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        i64, vp, ci, f32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        st = ctypes.c_int
        lib.tcg_create.restype = st
        lib.tcg_create.argtypes = [ctypes.POINTER(vp)]
        lib.tcg_destroy.restype = st
        lib.tcg_destroy.argtypes = [vp]
        lib.tcg_set_stream.restype = st
        lib.tcg_set_stream.argtypes = [vp, vp]
        lib.tcg_set_workspace.restype = st
        lib.tcg_set_workspace.argtypes = [vp, vp, ctypes.c_size_t]
        lib.tcg_gemm_workspace_size.restype = st
        lib.tcg_gemm_workspace_size.argtypes = [ci, ci, i64, i64, i64, ci, ci, i64,
                                                ctypes.POINTER(ctypes.c_size_t)]
        lib.tcg_gemm_ex.restype = st
        lib.tcg_gemm_ex.argtypes = [vp, ci, ci, i64, i64, i64, f32, vp, ci, i64, vp, ci, i64,
                                    f32, vp, ci, i64, ci]
        lib.tcg_gemm_strided_batched.restype = st
        lib.tcg_gemm_strided_batched.argtypes = [vp, ci, ci, i64, i64, i64, f32, vp, ci, i64,
                                                 i64, vp, ci, i64, i64, f32, vp, ci, i64, i64,
                                                 i64, ci]
        lib.tcg_tail_split_plan.restype = st
        lib.tcg_tail_split_plan.argtypes = [i64, ci, ci, ctypes.c_double, ctypes.c_double,
                                            ctypes.POINTER(i64), ctypes.POINTER(ci),
                                            ctypes.POINTER(ci)]
        lib.tcg_gemm_tile_plan.restype = st
        lib.tcg_gemm_tile_plan.argtypes = [vp, i64, i64, i64, ci, ci, ci, i64, i64,
                                           ctypes.POINTER(ci), ctypes.POINTER(ci), vp, vp]
        lib.tcg_gemm_ex_host.restype = st
        lib.tcg_gemm_ex_host.argtypes = lib.tcg_gemm_ex.argtypes
        lib.tcg_gemm_strided_batched_host.restype = st
        lib.tcg_gemm_strided_batched_host.argtypes = lib.tcg_gemm_strided_batched.argtypes
        lib.tcg_get_device_error.restype = st
        lib.tcg_get_device_error.argtypes = [vp]
        lib.tcg_last_device_error_bits.restype = ctypes.c_uint32
        lib.tcg_last_device_error_bits.argtypes = [vp]
        lib.tcg_status_string.restype = ctypes.c_char_p
        lib.tcg_status_string.argtypes = [ci]
        lib.tcg_set_debug.restype = st
        lib.tcg_set_debug.argtypes = [vp, ctypes.c_uint64, ci]
        lib.tcg_launch_count.restype = ctypes.c_uint64
        lib.tcg_launch_count.argtypes = [vp]
        lib.tcg_set_kernel_options.restype = st
        lib.tcg_set_kernel_options.argtypes = [vp, ci, ci]
        lib.tcg_set_split_k.restype = st
        lib.tcg_set_split_k.argtypes = [vp, ci]
        lib.tcg_set_tile_n.restype = st
        lib.tcg_set_tile_n.argtypes = [vp, ci]
        lib.tcg_set_tf32_rounding.restype = st
        lib.tcg_set_tf32_rounding.argtypes = [vp, ci]
        lib.tcg_split_k_plan.restype = st
        lib.tcg_split_k_plan.argtypes = [i64, ci, ci, ci, ctypes.POINTER(ci), ctypes.POINTER(ci)]
        lib.tcg_gemm_split_k.restype = st
        lib.tcg_gemm_split_k.argtypes = [vp, i64, i64, i64, ci, ci, i64, ctypes.POINTER(ci),
                                         ctypes.POINTER(i64)]
        lib.tcg_set_clock_probe.restype = st
        lib.tcg_set_clock_probe.argtypes = [vp, ci]
        lib.tcg_read_clock_probe.restype = st
        lib.tcg_read_clock_probe.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64),
                                             ctypes.POINTER(ctypes.c_uint64)]
        lib.tcg_noalloc_device_error.restype = st
        lib.tcg_noalloc_device_error.argtypes = [vp]
        lib.tcg_gemm_tf32_noalloc.restype = st
        lib.tcg_gemm_tf32_noalloc.argtypes = [vp, ci, ci, i64, i64, i64, f32, vp, i64, vp, i64,
                                              f32, vp, i64]
        _lib = lib
        return lib


def _ptr(x) -> int | None:
    """Device pointer of a torch tensor, or an int/None passed through."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


# ---------------------------------------------------------------- raw C ABI
def tcg_create() -> int:
    h = ctypes.c_void_p()
    s = load_library().tcg_create(ctypes.byref(h))
    if s != TCG_STATUS_SUCCESS:
        raise TcgError(s, "tcg_create")
    return h.value


def tcg_destroy(h: int) -> int:
    return load_library().tcg_destroy(h)


def tcg_set_stream(h: int, stream: int | None) -> int:
    return load_library().tcg_set_stream(h, stream)


def tcg_set_workspace(h: int, ptr, nbytes: int) -> int:
    return load_library().tcg_set_workspace(h, _ptr(ptr), nbytes)


def tcg_gemm_workspace_size(transa, transb, m, n, k, Atype, compute, batch_count=1) -> int:
    out = ctypes.c_size_t(0)
    s = load_library().tcg_gemm_workspace_size(transa, transb, m, n, k, Atype, compute,
                                               batch_count, ctypes.byref(out))
    if s != TCG_STATUS_SUCCESS:
        raise TcgError(s, "tcg_gemm_workspace_size")
    return out.value


def tcg_gemm_ex(h, transa, transb, m, n, k, alpha, A, Atype, lda, B, Btype, ldb, beta, C,
                Ctype, ldc, compute) -> int:
    """Status of the C call; A, B, C are torch tensors or raw device pointers."""
    return load_library().tcg_gemm_ex(h, transa, transb, m, n, k, float(alpha), _ptr(A), Atype,
                                      lda, _ptr(B), Btype, ldb, float(beta), _ptr(C), Ctype,
                                      ldc, compute)


def tcg_gemm_strided_batched(h, transa, transb, m, n, k, alpha, A, Atype, lda, strideA, B,
                             Btype, ldb, strideB, beta, C, Ctype, ldc, strideC, batch_count,
                             compute) -> int:
    return load_library().tcg_gemm_strided_batched(
        h, transa, transb, m, n, k, float(alpha), _ptr(A), Atype, lda, strideA, _ptr(B), Btype,
        ldb, strideB, float(beta), _ptr(C), Ctype, ldc, strideC, batch_count, compute)


def tcg_gemm_ex_host(h, transa, transb, m, n, k, alpha, A, Atype, lda, B, Btype, ldb, beta, C,
                     Ctype, ldc, compute) -> int:
    """tcg_gemm_ex with A, B, C in host memory (CPU torch tensors or host addresses);
    returns when C holds D."""
    return load_library().tcg_gemm_ex_host(h, transa, transb, m, n, k, float(alpha), _ptr(A),
                                           Atype, lda, _ptr(B), Btype, ldb, float(beta), _ptr(C),
                                           Ctype, ldc, compute)


def tcg_gemm_strided_batched_host(h, transa, transb, m, n, k, alpha, A, Atype, lda, strideA, B,
                                  Btype, ldb, strideB, beta, C, Ctype, ldc, strideC,
                                  batch_count, compute) -> int:
    return load_library().tcg_gemm_strided_batched_host(
        h, transa, transb, m, n, k, float(alpha), _ptr(A), Atype, lda, strideA, _ptr(B), Btype,
        ldb, strideB, float(beta), _ptr(C), Ctype, ldc, strideC, batch_count, compute)


def tcg_get_device_error(h: int) -> int:
    return load_library().tcg_get_device_error(h)


def tcg_last_device_error_bits(h: int) -> int:
    return load_library().tcg_last_device_error_bits(h)


def tcg_status_string(s: int) -> str:
    return load_library().tcg_status_string(s).decode()


def tcg_set_debug(h: int, wait_limit_ns: int = 0, fault_inject: int = 0) -> int:
    return load_library().tcg_set_debug(h, wait_limit_ns, fault_inject)


def tcg_launch_count(h: int) -> int:
    return load_library().tcg_launch_count(h)


def tcg_set_kernel_options(h: int, cta_group: int = 0, group_m: int = 0) -> int:
    return load_library().tcg_set_kernel_options(h, cta_group, group_m)


def tcg_set_split_k(h: int, splits: int = 0) -> int:
    return load_library().tcg_set_split_k(h, splits)


def tcg_set_tile_n(h: int, tile_n: int = 0) -> int:
    return load_library().tcg_set_tile_n(h, tile_n)


def tcg_set_tf32_rounding(h: int, mode: int = 0) -> int:
    return load_library().tcg_set_tf32_rounding(h, mode)


def tcg_split_k_plan(tiles: int, num_k_blocks: int, clusters: int, forced: int = 0):
    """(status, splits, kb_per_split) of the split-K rule (pure host arithmetic)."""
    s, kb = ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().tcg_split_k_plan(tiles, num_k_blocks, clusters, forced, ctypes.byref(s),
                                         ctypes.byref(kb))
    return st, s.value, kb.value


def tcg_tail_split_plan(tiles: int, num_k_blocks: int, clusters: int, tile_us: float,
                        tile_bytes: float):
    """(status, full_tiles, splits, kb_per_split) of the tail-split rule (host arithmetic)."""
    f, s, kb = ctypes.c_int64(0), ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().tcg_tail_split_plan(tiles, num_k_blocks, clusters, tile_us, tile_bytes,
                                            ctypes.byref(f), ctypes.byref(s), ctypes.byref(kb))
    return st, f.value, s.value, kb.value


def tcg_gemm_tile_plan(h: int, m: int, n: int, k: int, Atype: int, compute: int, Ctype: int,
                       batch: int = 1):
    """(status, tile_m, tile_n, splits, k_per_split): per-tile K ranges of the next call of
    this shape; splits/k_per_split are numpy arrays of shape (batch, tiles_m, tiles_n)."""
    import numpy as np
    lib = load_library()
    tm, tn = ctypes.c_int(0), ctypes.c_int(0)
    # first call for the tile sizes (the arrays' length is only known after it)
    st = lib.tcg_gemm_tile_plan(h, m, n, k, Atype, compute, Ctype, batch, 1 << 62,
                                ctypes.byref(tm), ctypes.byref(tn), None, None)
    if st != 0 and st != 2:
        return st, 0, 0, None, None
    mt = -(-m // tm.value) if tm.value else 0
    nt = -(-n // tn.value) if tn.value else 0
    splits = np.zeros((batch, mt, nt), dtype=np.int32)
    kps = np.zeros((batch, mt, nt), dtype=np.int64)
    st = lib.tcg_gemm_tile_plan(h, m, n, k, Atype, compute, Ctype, batch, splits.size,
                                ctypes.byref(tm), ctypes.byref(tn), splits.ctypes.data,
                                kps.ctypes.data)
    return st, tm.value, tn.value, splits, kps


def tcg_gemm_split_k(h: int, m: int, n: int, k: int, Atype: int, compute: int, batch: int = 1):
    """(status, splits, k_per_split) the next call of this shape on h will use."""
    s, kps = ctypes.c_int(0), ctypes.c_int64(0)
    st = load_library().tcg_gemm_split_k(h, m, n, k, Atype, compute, batch, ctypes.byref(s),
                                         ctypes.byref(kps))
    return st, s.value, kps.value


def tcg_gemm_tf32_noalloc(stream, transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C,
                          ldc) -> int:
    """TF32 GEMM with its scratch in a fixed device array (no allocation); ``stream``
    is a raw cudaStream_t (int) or None.  See include/tcg.h."""
    return load_library().tcg_gemm_tf32_noalloc(stream, transa, transb, m, n, k, float(alpha),
                                                _ptr(A), lda, _ptr(B), ldb, float(beta),
                                                _ptr(C), ldc)


def tcg_set_clock_probe(h, on) -> int:
    """Start (on=1, counters zeroed) or stop adding GEMM kernels' SM cycles and
    nanoseconds to the handle's clock probe.  See include/tcg.h."""
    return load_library().tcg_set_clock_probe(h, int(on))


def tcg_read_clock_probe(h):
    """(status, sm_cycles, ns) summed over the probed GEMM launches (syncs h's stream)."""
    c, n = ctypes.c_uint64(0), ctypes.c_uint64(0)
    st = load_library().tcg_read_clock_probe(h, ctypes.byref(c), ctypes.byref(n))
    return st, c.value, n.value


def tcg_noalloc_device_error(stream) -> int:
    """Synchronise ``stream`` (raw cudaStream_t or None), then return and clear the
    status word of the allocation-free calls.  See include/tcg.h."""
    return load_library().tcg_noalloc_device_error(stream)


# ------------------------------------------------------------ conveniences
_TORCH_TYPE = {}


def dtype_code(t) -> int:
    import torch
    if not _TORCH_TYPE:
        _TORCH_TYPE.update({torch.float16: TCG_R_16F, torch.bfloat16: TCG_R_16BF,
                            torch.float32: TCG_R_32F, torch.float8_e4m3fn: TCG_R_8F_E4M3,
                            torch.float8_e5m2: TCG_R_8F_E5M2})
    return _TORCH_TYPE[t]


class Handle:
    """Owns a tcgHandle_t bound to a torch CUDA stream."""

    def __init__(self, stream=None):
        self.h = tcg_create()
        self.set_stream(stream)

    def set_stream(self, stream=None):
        import torch
        if stream is None and torch.cuda.is_available():
            stream = torch.cuda.current_stream()
        self.stream = stream
        check(tcg_set_stream(self.h, stream.cuda_stream if stream is not None else None),
              "tcg_set_stream")

    def close(self):
        if self.h:
            tcg_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def check(status: int, what: str = "") -> None:
    if status != TCG_STATUS_SUCCESS:
        raise TcgError(status, what)


def _check_rowmajor(A, B, C, host: bool) -> None:
    """Shapes, types, layout and placement that gemm_rowmajor's pointer-level call relies
    on; the library sees only pointers and leading dimensions, so a mismatch here would
    otherwise read the wrong elements rather than fail."""
    if A.dim() not in (2, 3) or B.dim() != A.dim() or C.dim() != A.dim():
        raise ValueError("gemm_rowmajor: A, B, C must all be 2-D or all 3-D (batched)")
    if A.shape[:-2] != B.shape[:-2] or A.shape[:-2] != C.shape[:-2]:
        raise ValueError("gemm_rowmajor: batch sizes of A, B, C differ")
    m, k = A.shape[-2:]
    if B.shape[-2] != k or C.shape[-2:] != (m, B.shape[-1]):
        raise ValueError(f"gemm_rowmajor: shapes {tuple(A.shape)} @ {tuple(B.shape)} -> "
                         f"{tuple(C.shape)} do not agree")
    if A.dtype != B.dtype:
        raise ValueError("gemm_rowmajor: A and B must have the same dtype")
    if not (A.is_contiguous() and B.is_contiguous() and C.is_contiguous()):
        raise ValueError("gemm_rowmajor: A, B, C must be contiguous row-major tensors")
    on_gpu = [t.is_cuda for t in (A, B, C)]
    if host and any(on_gpu):
        raise ValueError("gemm_rowmajor(host=True) takes CPU tensors")
    if not host and not all(on_gpu):
        raise ValueError("gemm_rowmajor takes CUDA tensors (host=True for CPU tensors)")
    if not host and len({t.device for t in (A, B, C)}) != 1:
        raise ValueError("gemm_rowmajor: A, B, C must be on one device")


def gemm_rowmajor(handle: Handle, A, B, C, alpha=1.0, beta=0.0, tf32=False,
                  split3=False, host=False) -> None:
    """Row-major D = alpha*A@B + beta*C in place in C (torch CUDA tensors; CPU tensors,
    preferably pinned, with ``host=True``, through the host-buffer entry points).

    A: (m, k) or (batch, m, k); B: (k, n) or (batch, k, n); C: (m, n) or
    (batch, m, n), all contiguous row-major.  Issued as the column-major call
    gemm(N, N, n, m, k, alpha, B, n, A, k, beta, C, n) (C^T = B^T A^T).
    """
    _check_rowmajor(A, B, C, host)
    batched = A.dim() == 3
    m, k = A.shape[-2:]
    n = B.shape[-1]
    at, ct = dtype_code(A.dtype), dtype_code(C.dtype)
    # FP32 inputs always go through TF32 (one product) or its three-product split
    if split3:
        comp = TCG_COMPUTE_32F_3XTF32
    elif tf32 or at == TCG_R_32F:
        comp = TCG_COMPUTE_32F_FAST_TF32
    else:
        comp = TCG_COMPUTE_32F
    one = tcg_gemm_ex_host if host else tcg_gemm_ex
    many = tcg_gemm_strided_batched_host if host else tcg_gemm_strided_batched
    if not batched:
        s = one(handle.h, TCG_OP_N, TCG_OP_N, n, m, k, alpha, B, at, n, A, at, k, beta, C, ct, n,
                comp)
    else:
        batch = A.shape[0]
        s = many(handle.h, TCG_OP_N, TCG_OP_N, n, m, k, alpha, B, at, n, k * n, A, at, k, m * k,
                 beta, C, ct, n, m * n, batch, comp)
    check(s, "gemm_rowmajor")
