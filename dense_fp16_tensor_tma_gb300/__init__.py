"""Fused fp16 tensor-core GEMM for GB300:  C = epilogue(A @ B + bias).

A thin ctypes binding over the C ABI in include/gemm_f16.h.  It only
marshals arguments (device pointers, sizes, the current CUDA stream); every
step of the computation runs in the library's CUDA kernels.  PyTorch serves
for device memory and streams.  There is no fallback: if the compiled
library is missing, importing this package fails.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgemm_f16.so")

GEMM_EPI_NONE, GEMM_EPI_BIAS, GEMM_EPI_BIAS_RELU, GEMM_EPI_BIAS_GELU_ERF = 0, 1, 2, 3
GEMM_EPI_BIAS_SIGMOID, GEMM_EPI_BIAS_GELU_TANH = 4, 5
EPILOGUES = {"none": GEMM_EPI_NONE, "bias": GEMM_EPI_BIAS, "bias_relu": GEMM_EPI_BIAS_RELU,
             "bias_gelu_erf": GEMM_EPI_BIAS_GELU_ERF, "bias_sigmoid": GEMM_EPI_BIAS_SIGMOID,
             "bias_gelu_tanh": GEMM_EPI_BIAS_GELU_TANH}
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED_DEVICE, GEMM_ERR_MISALIGNED = 0, 1, 2, 3
GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT, GEMM_ERR_NO_MEMORY, GEMM_ERR_SCRATCH_LIMIT = 4, 5, 6, 7

GEMM_F16_TRANS_A, GEMM_F16_TRANS_B, GEMM_F16_PLAN_NOALLOC = 1, 2, 4

EXPORTS = ("gemm_f16", "gemm_f16_ex", "gemm_f16_status_string", "gemm_f16_last_cuda_error",
           "gemm_f16_debug_status", "gemm_f16_release_workspace", "gemm_f16_plan", "gemm_f16_plan_ex",
           "gemm_f16_selftest_timeout", "gemm_f16_noalloc", "gemm_f16_force_config", "gemm_f16_set_pdl",
           "gemm_f16_grouped", "attn_f16_fwd", "attn_f16_debug_status", "attn_f16_last_cuda_error",
           "gemm_f16_debug_inject", "attn_f16_debug_inject", "gemm_f16_force_ksplit", "attn_f16_plan")
GEMM_F16_FAULT_NONE, GEMM_F16_FAULT_SKIP_LOADS, GEMM_F16_FAULT_ENCODE = 0, 1, 2
CONFIGS = {"auto": 0, "pair256x256": 1, "128x256": 2, "128x128": 3, "128x64": 4, "swap": 5, "pair_whole": 6}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
                      "or `python dense_fp16_tensor_tma_gb300/build.py`")

lib = ctypes.CDLL(LIB_PATH)
_vp, _i64, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int


class GemmProblem(ctypes.Structure):
    """gemm_f16_problem_t of include/gemm_f16.h."""
    _fields_ = [("A", _vp), ("lda", _i64), ("B", _vp), ("ldb", _i64), ("bias", _vp), ("C", _vp), ("ldc", _i64),
                ("M", _i64), ("N", _i64), ("K", _i64)]


lib.gemm_f16.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]
lib.gemm_f16.restype = _int
lib.gemm_f16_ex.argtypes = [_vp, _i64, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int, _vp]
lib.gemm_f16_ex.restype = _int
lib.gemm_f16_status_string.argtypes = [_int]
lib.gemm_f16_status_string.restype = ctypes.c_char_p
lib.gemm_f16_last_cuda_error.restype = _int
lib.gemm_f16_debug_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32)]
lib.gemm_f16_debug_status.restype = _int
lib.gemm_f16_release_workspace.restype = _int
lib.gemm_f16_plan.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, ctypes.POINTER(ctypes.c_int64)]
lib.gemm_f16_plan.restype = _int
lib.gemm_f16_plan_ex.argtypes = [_vp, _i64, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int, _int,
                                 ctypes.POINTER(ctypes.c_int64)]
lib.gemm_f16_plan_ex.restype = _int
lib.gemm_f16_selftest_timeout.argtypes = [_vp, ctypes.c_uint32]
lib.gemm_f16_selftest_timeout.restype = _int
lib.gemm_f16_noalloc.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]
lib.gemm_f16_noalloc.restype = _int
lib.gemm_f16_force_config.argtypes = [_int]
lib.gemm_f16_force_config.restype = _int
lib.gemm_f16_grouped.argtypes = [ctypes.POINTER(GemmProblem), _int, _int, _int, _vp]
lib.gemm_f16_grouped.restype = _int
lib.attn_f16_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, ctypes.c_float, _vp]
lib.attn_f16_fwd.restype = _int
lib.attn_f16_debug_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32)]
lib.attn_f16_debug_status.restype = _int
lib.attn_f16_last_cuda_error.restype = _int
lib.attn_f16_plan.argtypes = [_i64, _i64, _i64, _i64, _int, _int, ctypes.POINTER(ctypes.c_int64)]
lib.attn_f16_plan.restype = _int
lib.gemm_f16_set_pdl.argtypes = [_int]
lib.gemm_f16_set_pdl.restype = _int
lib.gemm_f16_force_ksplit.argtypes = [_int]
lib.gemm_f16_force_ksplit.restype = _int
lib.gemm_f16_debug_inject.argtypes = [_int, ctypes.c_uint32]
lib.gemm_f16_debug_inject.restype = _int
lib.attn_f16_debug_inject.argtypes = [_int, ctypes.c_uint32]
lib.attn_f16_debug_inject.restype = _int


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str = "gemm_f16"):
        self.status = status
        msg = gemm_f16_status_string(status)
        if status == GEMM_ERR_CUDA:
            err = lib.attn_f16_last_cuda_error() if where.startswith("attn") else lib.gemm_f16_last_cuda_error()
            msg += f" (cudaError {err})"
        super().__init__(f"{where}: {msg}")


def gemm_f16_status_string(status: int) -> str:
    return lib.gemm_f16_status_string(int(status)).decode()


def _epi(epilogue) -> int:
    return EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)


def _stream_handle(stream, device_index=None):
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:   # the current stream's handle without building a Stream object
            return raw(torch.cuda.current_device() if device_index is None else device_index)
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def gemm_f16_ptr(a_ptr: int, b_ptr: int, bias_ptr: int, c_ptr: int, M: int, N: int, K: int,
                 epilogue=GEMM_EPI_NONE, stream: int = 0) -> int:
    """Raw C-ABI call: device addresses as integers; returns the status code."""
    return lib.gemm_f16(a_ptr or None, b_ptr or None, bias_ptr or None, c_ptr or None,
                        int(M), int(N), int(K), _epi(epilogue), stream or None)


def gemm_f16_ex_ptr(a_ptr: int, lda: int, b_ptr: int, ldb: int, bias_ptr: int, c_ptr: int, ldc: int,
                    M: int, N: int, K: int, epilogue=GEMM_EPI_NONE, flags: int = 0, stream: int = 0) -> int:
    """Raw call of gemm_f16_ex (pitches in elements, GEMM_F16_TRANS_* flags); returns the status code."""
    return lib.gemm_f16_ex(a_ptr or None, int(lda), b_ptr or None, int(ldb), bias_ptr or None, c_ptr or None,
                           int(ldc), int(M), int(N), int(K), _epi(epilogue), int(flags), stream or None)


def _operand_layout(t, name):
    """(stored transposed, row pitch) of a 2-D view whose rows are contiguous
    (strides (ld, 1)) or whose columns are (strides (1, ld): the transpose of a
    row-major matrix, e.g. W.t() of a Linear weight W).  Size-1 dimensions,
    and empty tensors, take any stride."""
    rows, cols = t.shape
    s0, s1 = t.stride()
    if rows == 0 or cols == 0:
        return False, max(cols, 1)   # nothing is read or written: any strides
    if cols <= 1 or s1 == 1:
        if rows <= 1:
            return False, max(cols, 1)
        if s0 >= max(cols, 1):
            return False, s0
    if rows <= 1 or s0 == 1:
        if cols <= 1:
            return True, max(rows, 1)
        if s1 >= max(rows, 1):
            return True, s1
    raise ValueError(f"{name} (shape {tuple(t.shape)}, strides {t.stride()}) needs contiguous rows or "
                     "contiguous columns with non-overlapping lines")


def gemm_f16(A, B, bias, C, epilogue="none", stream=None):
    """C = epilogue(A @ B + bias) into the preallocated fp16 CUDA tensor C.

    A [M,K], B [K,N], C [M,N] and bias [N] (or None for "none") are
    torch.float16 CUDA tensors on the current device.  A and B may be row
    views with any pitch or transposed views (A = X.t(), B = W.t() for a
    weight W [N,K]); they are passed to gemm_f16_ex as pitches and layout
    flags, never copied here.  C needs contiguous rows (any pitch), bias is
    contiguous.  Enqueued on `stream` (default: torch's current stream);
    raises GemmError on a nonzero status.
    """
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    for name, t in (("A", A), ("B", B), ("C", C)) + ((("bias", bias),) if bias is not None else ()):
        if t.dtype != torch.float16 or not t.is_cuda:
            raise ValueError(f"{name} must be a float16 CUDA tensor")
    if bias is not None and (tuple(bias.shape) != (N,) or not bias.is_contiguous()):
        raise ValueError(f"bias must be a contiguous tensor of shape ({N},)")
    ta, lda = _operand_layout(A, "A")
    tb, ldb = _operand_layout(B, "B")
    tc, ldc = _operand_layout(C, "C")
    if tc and M > 1 and N > 1:
        raise ValueError("C needs contiguous rows")
    if tc:
        ldc = N
    flags = (GEMM_F16_TRANS_A if ta else 0) | (GEMM_F16_TRANS_B if tb else 0)
    st = lib.gemm_f16_ex(A.data_ptr() or None, lda, B.data_ptr() or None, ldb,
                         bias.data_ptr() if bias is not None else None, C.data_ptr() or None, ldc,
                         M, N, K, _epi(epilogue), flags, _stream_handle(stream, C.get_device()))
    if st != GEMM_OK:
        raise GemmError(st)
    return C


def gemm_f16_grouped_ptr(problems, epilogue=GEMM_EPI_NONE, flags: int = 0, stream: int = 0) -> int:
    """Raw call of gemm_f16_grouped: `problems` is a sequence of tuples
    (A, lda, B, ldb, bias, C, ldc, M, N, K) of integers (device addresses,
    pitches and sizes).  Returns the status code."""
    arr = (GemmProblem * max(1, len(problems)))()
    for i, q in enumerate(problems):
        arr[i] = GemmProblem(*[(int(x) or None) if k in (0, 2, 4, 5) else int(x) for k, x in enumerate(q)])
    return lib.gemm_f16_grouped(arr, len(problems), _epi(epilogue), int(flags), stream or None)


def gemm_f16_grouped(problems, epilogue="none", stream=None):
    """C_g = epilogue(A_g @ B_g + bias_g) for every (A_g, B_g, bias_g, C_g) in
    `problems`, in one grouped launch per operand layout present (the layouts
    are read from each view as in gemm_f16; bias_g may be None for "none").
    Raises GemmError on a nonzero status."""
    import torch
    by_flags = {}
    dev = None
    for idx, (A, B, bias, C) in enumerate(problems):
        M, K = A.shape
        K2, N = B.shape
        if K2 != K or tuple(C.shape) != (M, N):
            raise ValueError(f"problem {idx}: shape mismatch A {tuple(A.shape)}, B {tuple(B.shape)}, "
                             f"C {tuple(C.shape)}")
        for name, t in (("A", A), ("B", B), ("C", C)) + ((("bias", bias),) if bias is not None else ()):
            if t.dtype != torch.float16 or not t.is_cuda:
                raise ValueError(f"problem {idx}: {name} must be a float16 CUDA tensor")
        if bias is not None and (tuple(bias.shape) != (N,) or not bias.is_contiguous()):
            raise ValueError(f"problem {idx}: bias must be a contiguous tensor of shape ({N},)")
        ta, lda = _operand_layout(A, "A")
        tb, ldb = _operand_layout(B, "B")
        tc, ldc = _operand_layout(C, "C")
        if tc and M > 1 and N > 1:
            raise ValueError(f"problem {idx}: C needs contiguous rows")
        if tc:
            ldc = N
        flags = (GEMM_F16_TRANS_A if ta else 0) | (GEMM_F16_TRANS_B if tb else 0)
        by_flags.setdefault(flags, []).append((A.data_ptr(), lda, B.data_ptr(), ldb,
                                               bias.data_ptr() if bias is not None else 0, C.data_ptr(), ldc,
                                               M, N, K))
        dev = C.get_device()
    handle = _stream_handle(stream, dev)
    for flags, probs in by_flags.items():
        st = gemm_f16_grouped_ptr(probs, epilogue, flags, handle)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_f16_grouped")
    return [C for _, _, _, C in problems]


def gemm_f16_plan(M, N, K, epilogue="none", num_sms=152, a_addr=256, b_addr=256, c_addr=256,
                  bias_addr=256, lda=None, ldb=None, ldc=None, trans_a=False, trans_b=False, noalloc=False):
    """Host-only: the plan gemm_f16 / gemm_f16_ex would pick (dict), without
    touching a device; with noalloc=True the plan of gemm_f16_noalloc.
    Pitches default to the dense ones of the layout."""
    out = (ctypes.c_int64 * 11)()
    lda = lda if lda is not None else (M if trans_a else K)
    ldb = ldb if ldb is not None else (K if trans_b else N)
    ldc = ldc if ldc is not None else N
    flags = ((GEMM_F16_TRANS_A if trans_a else 0) | (GEMM_F16_TRANS_B if trans_b else 0) |
             (GEMM_F16_PLAN_NOALLOC if noalloc else 0))
    st = lib.gemm_f16_plan_ex(a_addr or None, int(lda), b_addr or None, int(ldb), bias_addr or None,
                              c_addr or None, int(ldc), int(M), int(N), int(K), _epi(epilogue), flags,
                              int(num_sms), out)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16_plan")
    keys = ("path", "tile_m", "tile_n", "stages", "ctas", "pack_a", "pack_b", "vec_store", "splits", "scratch",
            "whole_tiles")
    return dict(zip(keys, list(out)))


def gemm_f16_debug_status(stream=None):
    """Synchronise the stream; (status, raw device status word)."""
    word = ctypes.c_uint32(0)
    st = lib.gemm_f16_debug_status(_stream_handle(stream), ctypes.byref(word))
    return st, word.value


def gemm_f16_release_workspace() -> int:
    return lib.gemm_f16_release_workspace()


def gemm_f16_force_config(config) -> int:
    """Pin the kernel configuration ("auto", "pair256x256", "128x256", "128x128",
    "128x64", "swap" or its number) for later calls; returns the previous setting."""
    c = CONFIGS[config] if isinstance(config, str) else int(config)
    prev = lib.gemm_f16_force_config(c)
    if prev < 0:
        raise ValueError(f"unknown configuration {config!r}")
    return prev


def gemm_f16_force_ksplit(splits: int) -> int:
    """Pin the cluster split of K for 128-row tiles (0 automatic, 1 never, 2 or 4
    CTAs per tile) for later calls; returns the previous setting."""
    prev = lib.gemm_f16_force_ksplit(int(splits))
    if prev < 0:
        raise ValueError(f"unknown split {splits!r}")
    return prev


def gemm_f16_set_pdl(enable: bool) -> bool:
    """Programmatic dependent launch of the library's kernels on/off
    (process-wide); returns the previous setting."""
    return bool(lib.gemm_f16_set_pdl(1 if enable else 0))


def gemm_f16_debug_inject(fault: int, wait_us: int = 0) -> int:
    """Test hook: arm one fault (GEMM_F16_FAULT_*) for the next GEMM call that
    reaches it; returns the status code."""
    return lib.gemm_f16_debug_inject(int(fault), int(wait_us))


def attn_f16_debug_inject(fault: int, wait_us: int = 0) -> int:
    """Test hook: arm one fault (GEMM_F16_FAULT_*) for the next attention call."""
    return lib.attn_f16_debug_inject(int(fault), int(wait_us))


def gemm_f16_selftest_timeout(timeout_us: int = 1000, stream=None) -> int:
    return lib.gemm_f16_selftest_timeout(_stream_handle(stream), int(timeout_us))


def gemm_f16_noalloc_ptr(a_ptr: int, b_ptr: int, bias_ptr: int, c_ptr: int, M: int, N: int, K: int,
                         epilogue=GEMM_EPI_NONE, stream: int = 0) -> int:
    """Raw call of gemm_f16_noalloc, the variant that never allocates device memory.

    For callers that cannot allocate (a host framework owns the device memory,
    a serving loop must not synchronise the device through cudaMalloc, or
    allocation after start-up is forbidden).  Any operand repack goes to a
    fixed 32 MiB buffer inside the library; larger repacks return
    GEMM_ERR_SCRATCH_LIMIT.  Calls overlapping on the GPU share that buffer and
    race.  Returns the status code.
    """
    return lib.gemm_f16_noalloc(a_ptr or None, b_ptr or None, bias_ptr or None, c_ptr or None,
                                int(M), int(N), int(K), _epi(epilogue), stream or None)


# ---------------------------------------------------------------- attention forward

def attn_f16_fwd_ptr(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, B: int, H: int, S: int, D: int,
                     causal: bool = False, scale: float = 0.0, stream: int = 0) -> int:
    """Raw call of attn_f16_fwd (device addresses as integers); returns the status code."""
    return lib.attn_f16_fwd(q_ptr or None, k_ptr or None, v_ptr or None, o_ptr or None, int(B), int(H), int(S),
                            int(D), 1 if causal else 0, float(scale), stream or None)


def attn_f16_fwd(Q, K, V, O, causal=False, scale=None, stream=None):
    """O = softmax(scale * Q @ K^T) @ V per (batch, head), into the preallocated
    O.  Q, K, V, O: contiguous torch.float16 CUDA tensors of shape (B, H, S, D),
    D 64 or 128.  scale defaults to 1/sqrt(D).  Raises GemmError on a nonzero
    status."""
    import torch
    shape = tuple(Q.shape)
    if len(shape) != 4 or tuple(K.shape) != shape or tuple(V.shape) != shape or tuple(O.shape) != shape:
        raise ValueError(f"Q, K, V, O must share one (B, H, S, D) shape: {shape}, {tuple(K.shape)}, "
                         f"{tuple(V.shape)}, {tuple(O.shape)}")
    for name, t in (("Q", Q), ("K", K), ("V", V), ("O", O)):
        if t.dtype != torch.float16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float16 CUDA tensor")
    B, H, S, D = shape
    st = lib.attn_f16_fwd(Q.data_ptr() or None, K.data_ptr() or None, V.data_ptr() or None, O.data_ptr() or None,
                          B, H, S, D, 1 if causal else 0, 0.0 if scale is None else float(scale),
                          _stream_handle(stream, O.get_device()))
    if st != GEMM_OK:
        raise GemmError(st, "attn_f16_fwd")
    return O


ATTN_KERNELS = {0: None, 1: "attn_f16_fwd4_kernel", 2: "attn_f16_fwd2_kernel", 3: "attn_f16_fwd3_kernel"}


def attn_f16_plan(B, H, S, D, causal=False, num_sms=152):
    """Host-only: the kernel and work split attn_f16_fwd would use (dict),
    without touching a device."""
    out = (ctypes.c_int64 * 5)()
    st = lib.attn_f16_plan(int(B), int(H), int(S), int(D), 1 if causal else 0, int(num_sms), out)
    if st != GEMM_OK:
        raise GemmError(st, "attn_f16_plan")
    d = dict(zip(("kernel", "units", "pair_units", "causal_pairs", "ctas"), list(out)))
    d["kernel_name"] = ATTN_KERNELS[d["kernel"]]
    return d


def attn_f16_debug_status(stream=None):
    """Synchronise the stream; (status, raw status word) of the attention kernels."""
    word = ctypes.c_uint32(0)
    st = lib.attn_f16_debug_status(_stream_handle(stream), ctypes.byref(word))
    return st, word.value


def attention_flops(B, H, S, D, causal):
    """The pages' FLOP model of attention forward: 4 B H S^2 D, halved when causal."""
    return 4.0 * B * H * S * S * D * (0.5 if causal else 1.0)
