"""ctypes binding to ``libdgt_gemm.so``: argument marshalling only.

The functions ``gemm_tf32``, ``gemm_f16`` and ``gemm_bf16`` have the names
and arguments of the C interface (``include/dgt_gemm.h``) and take raw device
pointers. ``matmul`` takes torch CUDA tensors and derives sizes, leading
dimensions and the current stream from them; ``matmul_from_host`` is the
end-to-end call (``gemm_*_host``) for operands held in (pinned) host memory. Every step of the
product runs in the library's CUDA kernels; there is no other code path, and
a missing or unloadable library raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdgt_gemm.so")

GEMM_B_ROW_MAJOR = 0
GEMM_B_K_MAJOR = 1

GEMM_OK = 0
GEMM_ERR_INVALID_VALUE = 1
GEMM_ERR_MISALIGNED = 2
GEMM_ERR_UNSUPPORTED_DEVICE = 3
GEMM_ERR_LAUNCH = 4
GEMM_ERR_NOT_DEVICE_MEMORY = 5
GEMM_ERR_DRIVER = 6
GEMM_ERR_DEVICE_TIMEOUT = 7
GEMM_ERR_SCRATCH_LIMIT = 8

GEMM_ACT_NONE = 0
GEMM_ACT_RELU = 1
GEMM_ACT_GELU = 2
GEMM_ACT_GELU_TANH = 3
ACTIVATIONS = {None: GEMM_ACT_NONE, "none": GEMM_ACT_NONE, "relu": GEMM_ACT_RELU, "gelu": GEMM_ACT_GELU,
               "gelu_tanh": GEMM_ACT_GELU_TANH}


class Epilogue(ctypes.Structure):
    """gemm_epilogue_t: C = act(alpha * A.B + beta * C + bias[col])."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("activation", ctypes.c_int)]

# Every symbol the C header declares.
EXPORTS = ("gemm_tf32", "gemm_f16", "gemm_bf16", "gemm_tf32_ex", "gemm_f16_ex", "gemm_bf16_ex", "gemm_e4m3", "gemm_e5m2",
           "gemm_status_string", "gemm_get_device_status", "gemm_reset_device_status", "gemm_set_debug",
           "gemm_launch_count", "gemm_set_tuning", "gemm_last_plan", "gemm_free_workspaces",
           "gemm_bf16_static_scratch", "gemm_tf32_strided_batched", "gemm_f16_strided_batched",
           "gemm_bf16_strided_batched", "gemm_e4m3_strided_batched", "gemm_e5m2_strided_batched",
           "gemm_plan_query", "gemm_tf32_host", "gemm_f16_host", "gemm_bf16_host")

_lib = None


class GemmError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} (code {code})")
        self.code = code


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with dense_gemm_tensor_gb300.build.build()")
    lib = ctypes.CDLL(path)
    i64, vp, u32, u64 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64
    for name in ("gemm_tf32", "gemm_f16", "gemm_bf16", "gemm_bf16_static_scratch", "gemm_tf32_host", "gemm_f16_host",
                 "gemm_bf16_host"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int, vp]
        fn.restype = ctypes.c_int
    for name in ("gemm_tf32_ex", "gemm_f16_ex", "gemm_bf16_ex", "gemm_e4m3", "gemm_e5m2"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, ctypes.c_int, ctypes.POINTER(Epilogue), vp]
        fn.restype = ctypes.c_int
    for name in ("gemm_tf32_strided_batched", "gemm_f16_strided_batched", "gemm_bf16_strided_batched",
                 "gemm_e4m3_strided_batched", "gemm_e5m2_strided_batched"):
        fn = getattr(lib, name)
        fn.argtypes = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64, ctypes.c_int,
                       ctypes.POINTER(Epilogue), vp]
        fn.restype = ctypes.c_int
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_get_device_status.argtypes = [vp, ctypes.POINTER(u32)]
    lib.gemm_get_device_status.restype = ctypes.c_int
    lib.gemm_reset_device_status.argtypes = []
    lib.gemm_reset_device_status.restype = ctypes.c_int
    lib.gemm_set_debug.argtypes = [u32, u64]
    lib.gemm_set_debug.restype = ctypes.c_int
    lib.gemm_launch_count.argtypes = []
    lib.gemm_launch_count.restype = u64
    lib.gemm_set_tuning.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gemm_set_tuning.restype = ctypes.c_int
    lib.gemm_last_plan.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    lib.gemm_last_plan.restype = ctypes.c_int
    lib.gemm_free_workspaces.argtypes = []
    lib.gemm_free_workspaces.restype = ctypes.c_int
    ci = ctypes.c_int
    lib.gemm_plan_query.argtypes = [ci, i64, i64, i64, ci, i64, ci, ci, ci, ci, ctypes.POINTER(ctypes.c_int32)]
    lib.gemm_plan_query.restype = ci
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().gemm_status_string(int(code)).decode()


def _call(name, M, N, K, A, lda, B, ldb, C, ldc, layout, stream):
    return getattr(load(), name)(M, N, K, A, lda, B, ldb, C, ldc, layout, stream)


def gemm_tf32(M, N, K, A, lda, B, ldb, C, ldc, layout=GEMM_B_ROW_MAJOR, stream=None) -> int:
    """C = A . B, fp32 operands read as TF32; raw device pointers (ints)."""
    return _call("gemm_tf32", M, N, K, A, lda, B, ldb, C, ldc, layout, stream)


def gemm_f16(M, N, K, A, lda, B, ldb, C, ldc, layout=GEMM_B_ROW_MAJOR, stream=None) -> int:
    """C = A . B with IEEE half operands and output; raw device pointers."""
    return _call("gemm_f16", M, N, K, A, lda, B, ldb, C, ldc, layout, stream)


def gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, layout=GEMM_B_ROW_MAJOR, stream=None) -> int:
    """C = A . B with bfloat16 operands and output; raw device pointers."""
    return _call("gemm_bf16", M, N, K, A, lda, B, ldb, C, ldc, layout, stream)


def gemm_bf16_static_scratch(M, N, K, A, lda, B, ldb, C, ldc, layout=GEMM_B_ROW_MAJOR, stream=None) -> int:
    """gemm_bf16 without any allocation (scratch from the library's fixed
    16 MiB device array); raw device pointers. See the C header for limits."""
    return _call("gemm_bf16_static_scratch", M, N, K, A, lda, B, ldb, C, ldc, layout, stream)


def gemm_ex(dtype_name, M, N, K, A, lda, B, ldb, C, ldc, layout=GEMM_B_ROW_MAJOR, epilogue=None,
            stream=None) -> int:
    """gemm_{tf32,f16,bf16}_ex or gemm_{e4m3,e5m2} with raw device pointers;
    `epilogue` an Epilogue or None."""
    fn = getattr(load(), f"gemm_{dtype_name}" + ("" if dtype_name in ("e4m3", "e5m2") else "_ex"))
    return fn(M, N, K, A, lda, B, ldb, C, ldc, layout, ctypes.byref(epilogue) if epilogue is not None else None,
              stream)


_BY_DTYPE = {torch.float32: "gemm_tf32", torch.float16: "gemm_f16", torch.bfloat16: "gemm_bf16"}
_FP8 = {torch.float8_e4m3fn: "gemm_e4m3", torch.float8_e5m2: "gemm_e5m2"}
_FN = {}  # dtype -> bound C function, filled on first use
_FN_EX = {}


def _raw_stream(stream, device_index: int) -> int:
    """The cudaStream_t of `stream`, or of the device's current stream."""
    if stream is not None:
        return stream.cuda_stream
    try:  # the current stream's handle without building a Stream object
        return torch._C._cuda_getCurrentRawStream(device_index)
    except AttributeError:
        return torch.cuda.current_stream(device_index).cuda_stream


def _rows(t: torch.Tensor, what: str) -> int:
    """Leading dimension of a 2-D tensor with unit column stride."""
    if t.dim() != 2:
        raise ValueError(f"{what} must be 2-D")
    rows, cols = t.shape
    s0, s1 = t.stride()
    if cols > 1 and s1 != 1:
        raise ValueError(f"{what} must have unit stride along its rows")
    return (s0 if s0 > cols else cols) if rows > 1 else cols


def matmul(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None, *, layout: int = GEMM_B_ROW_MAJOR,
           stream: torch.cuda.Stream | None = None, alpha: float = 1.0, beta: float = 0.0,
           bias: torch.Tensor | None = None, activation: str | None = None) -> torch.Tensor:
    """C = A . B on the current CUDA device, or with a fused epilogue
    C = act(alpha * A . B + beta * C + bias) when any of alpha, beta, bias,
    activation ("relu", "gelu", "gelu_tanh") differs from the identity.

    ``A``: M x K. ``B``: K x N for ``layout=GEMM_B_ROW_MAJOR``, or N x K (B
    transposed) for ``layout=GEMM_B_K_MAJOR``. Rows may be padded (stride(0) >
    row length) but elements along a row must be contiguous. The dtype selects
    the entry point: float32 -> gemm_tf32, float16 -> gemm_f16, bfloat16 ->
    gemm_bf16 (the *_ex variants with an epilogue); float8_e4m3fn ->
    gemm_e4m3 and float8_e5m2 -> gemm_e5m2, whose C is bfloat16. ``out`` (M x
    N, the output dtype) may have padded rows too; with beta != 0 it supplies
    the C that is scaled and added. ``bias``: N elements of the output dtype,
    contiguous.
    """
    dt = A.dtype
    if dt in _FP8:
        return _matmul_fp8(A, B, out, layout, stream, alpha, beta, bias, activation)
    fn = _FN.get(dt)
    if fn is None:
        if dt not in _BY_DTYPE:
            raise TypeError("A and B must both be float32, float16 or bfloat16")
        fn = _FN[dt] = getattr(load(), _BY_DTYPE[dt])
    if B.dtype != dt:
        raise TypeError("A and B must have the same dtype")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, K = A.shape
    if layout == GEMM_B_ROW_MAJOR:
        if B.shape[0] != K:
            raise ValueError("B must be K x N")
        N = B.shape[1]
    else:
        if B.shape[1] != K:
            raise ValueError("B must be N x K for the K-major layout")
        N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=A.device)
    elif out.dtype != dt or tuple(out.shape) != (M, N):
        raise ValueError("out must be M x N with the operands' dtype")
    s = _raw_stream(stream, torch.cuda.current_device())
    if alpha == 1.0 and beta == 0.0 and bias is None and activation is None:
        code = fn(M, N, K, A.data_ptr() or None, _rows(A, "A"), B.data_ptr() or None, _rows(B, "B"),
                  out.data_ptr() or None, _rows(out, "out"), layout, s)
        if code != GEMM_OK:
            raise GemmError(code, _BY_DTYPE[dt])
        return out
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(k for k in ACTIVATIONS if k)}")
    if bias is not None:
        if bias.dtype != dt or bias.dim() != 1 or bias.numel() != N or not bias.is_cuda or \
                (N > 1 and bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous CUDA vector of N elements of the operands' dtype")
    fx = _FN_EX.get(dt)
    if fx is None:
        fx = _FN_EX[dt] = getattr(load(), _BY_DTYPE[dt] + "_ex")
    epi = Epilogue(float(alpha), float(beta), bias.data_ptr() if bias is not None else None,
                   ACTIVATIONS[activation])
    code = fx(M, N, K, A.data_ptr() or None, _rows(A, "A"), B.data_ptr() or None, _rows(B, "B"),
              out.data_ptr() or None, _rows(out, "out"), layout, ctypes.byref(epi), s)
    if code != GEMM_OK:
        raise GemmError(code, _BY_DTYPE[dt] + "_ex")
    return out


def _matmul_fp8(A, B, out, layout, stream, alpha, beta, bias, activation):
    dt = A.dtype
    if B.dtype != dt:
        raise TypeError("A and B must have the same FP8 dtype")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, K = A.shape
    if layout == GEMM_B_ROW_MAJOR:
        if B.shape[0] != K:
            raise ValueError("B must be K x N")
        N = B.shape[1]
    else:
        if B.shape[1] != K:
            raise ValueError("B must be N x K for the K-major layout")
        N = B.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    elif out.dtype != torch.bfloat16 or tuple(out.shape) != (M, N):
        raise ValueError("out must be M x N bfloat16")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(k for k in ACTIVATIONS if k)}")
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.dim() != 1 or bias.numel() != N or
                             not bias.is_cuda or (N > 1 and bias.stride(0) != 1)):
        raise ValueError("bias must be a contiguous CUDA bfloat16 vector of N elements")
    epi = Epilogue(float(alpha), float(beta), bias.data_ptr() if bias is not None else None, ACTIVATIONS[activation])
    s = _raw_stream(stream, torch.cuda.current_device())
    fn = getattr(load(), _FP8[dt])
    code = fn(M, N, K, A.data_ptr() or None, _rows(A, "A"), B.data_ptr() or None, _rows(B, "B"),
              out.data_ptr() or None, _rows(out, "out"), layout, ctypes.byref(epi), s)
    if code != GEMM_OK:
        raise GemmError(code, _FP8[dt])
    return out


def bmm(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None, *, layout: int = GEMM_B_ROW_MAJOR,
        stream: torch.cuda.Stream | None = None, alpha: float = 1.0, beta: float = 0.0,
        bias: torch.Tensor | None = None, activation: str | None = None) -> torch.Tensor:
    """Strided batch C[z] = A[z] . B[z] (gemm_*_strided_batched), optionally
    with the fused epilogue. A: batch x M x K; B: batch x K x N (layout 0) or
    batch x N x K (layout 1); a batch stride of 0 (``expand``) repeats one
    matrix. Rows must be contiguous; the other strides come from the tensors.
    FP8 operands (float8_e4m3fn, float8_e5m2) need a K-major B and give a
    bfloat16 C."""
    dt = A.dtype
    if (dt not in _BY_DTYPE and dt not in _FP8) or B.dtype != dt:
        raise TypeError("A and B must both be float32, float16, bfloat16, float8_e4m3fn or float8_e5m2")
    out_dt = torch.bfloat16 if dt in _FP8 else dt
    if A.dim() != 3 or B.dim() != 3 or A.shape[0] != B.shape[0]:
        raise ValueError("A and B must be 3-D with the same batch size")
    batch, M, K = A.shape
    N = B.shape[2] if layout == GEMM_B_ROW_MAJOR else B.shape[1]
    if (B.shape[1] if layout == GEMM_B_ROW_MAJOR else B.shape[2]) != K:
        raise ValueError("B's K dimension does not match A")
    if out is None:
        out = torch.empty((batch, M, N), dtype=out_dt, device=A.device)
    elif out.dtype != out_dt or tuple(out.shape) != (batch, M, N):
        raise ValueError("out must be batch x M x N of the output dtype")
    for t, what in ((A, "A"), (B, "B"), (out, "out")):
        if t.shape[2] > 1 and t.stride(2) != 1:
            raise ValueError(f"{what} must have unit stride along its rows")
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(k for k in ACTIVATIONS if k)}")
    if bias is not None and (bias.dtype != out_dt or bias.dim() != 1 or bias.numel() != N or not bias.is_cuda or
                             (N > 1 and bias.stride(0) != 1)):
        raise ValueError("bias must be a contiguous CUDA vector of N elements of the output dtype")
    epi = Epilogue(float(alpha), float(beta), bias.data_ptr() if bias is not None else None, ACTIVATIONS[activation])
    s = _raw_stream(stream, torch.cuda.current_device())
    ld = lambda t: t.stride(1) if t.shape[1] > 1 else t.shape[2]  # noqa: E731
    bs = lambda t: t.stride(0) if t.shape[0] > 1 else 0  # noqa: E731
    name = (_FP8[dt] if dt in _FP8 else _BY_DTYPE[dt]) + "_strided_batched"
    code = getattr(load(), name)(batch, M, N, K, A.data_ptr() or None, ld(A), bs(A), B.data_ptr() or None, ld(B),
                                 bs(B), out.data_ptr() or None, ld(out), bs(out) if batch > 1 else 0, layout,
                                 ctypes.byref(epi), s)
    if code != GEMM_OK:
        raise GemmError(code, name)
    return out


_HOST_FN = {torch.float32: "gemm_tf32_host", torch.float16: "gemm_f16_host", torch.bfloat16: "gemm_bf16_host"}


def gemm_host(dtype_name, M, N, K, A, lda, B, ldb, C, ldc, layout=GEMM_B_ROW_MAJOR, stream=None) -> int:
    """gemm_{tf32,f16,bf16}_host with raw host pointers (ints) and a raw stream handle."""
    return getattr(load(), f"gemm_{dtype_name}_host")(M, N, K, A, lda, B, ldb, C, ldc, layout, stream)


def matmul_from_host(A_host: torch.Tensor, B_host: torch.Tensor, *, layout: int = GEMM_B_ROW_MAJOR,
                     device: torch.device | str = "cuda", stream: torch.cuda.Stream | None = None,
                     buffers: dict | None = None, wait: bool = True):
    """End-to-end product of host operands through the C call
    gemm_{tf32,f16,bf16}_host: the library copies B and A (in row blocks) to
    its device staging, runs each block's product as it lands, and copies
    each block of C back while the next one computes.

    ``A_host`` / ``B_host``: 2-D CPU tensors (page-locked for the copies to
    overlap), rows contiguous. The result goes to a page-locked host tensor
    cached in ``buffers`` (optional, reused across calls of the same shape).
    With ``wait`` (the default) the call synchronises and returns C; with
    ``wait=False`` it returns ``(C, event)`` at once, C being valid once
    ``event`` has completed. A call that reuses ``buffers`` first waits for
    the previous call on them (it overwrites their C). ``A_host`` and
    ``B_host`` must stay unchanged until the call's event has completed.
    """
    dt = A_host.dtype
    if dt not in _HOST_FN or B_host.dtype != dt:
        raise TypeError("A and B must both be float32, float16 or bfloat16")
    if A_host.is_cuda or B_host.is_cuda:
        raise ValueError("A and B must be host tensors")
    buffers = {} if buffers is None else buffers
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    s = stream if stream is not None else torch.cuda.current_stream(idx)
    if buffers.get("done") is not None:
        buffers["done"].synchronize()
    M, K = A_host.shape
    N = B_host.shape[1] if layout == GEMM_B_ROW_MAJOR else B_host.shape[0]
    if (B_host.shape[0] if layout == GEMM_B_ROW_MAJOR else B_host.shape[1]) != K:
        raise ValueError("B's K dimension does not match A")
    key = (M, N, dt)
    if buffers.get("key") != key:
        buffers.update(key=key, c_host=torch.empty((M, N), dtype=dt, pin_memory=True))
    c = buffers["c_host"]
    with torch.cuda.device(idx):
        code = getattr(load(), _HOST_FN[dt])(M, N, K, A_host.data_ptr() or None, _rows(A_host, "A"),
                                             B_host.data_ptr() or None, _rows(B_host, "B"), c.data_ptr() or None,
                                             N, layout, s.cuda_stream)
    if code != GEMM_OK:
        raise GemmError(code, _HOST_FN[dt])
    done = torch.cuda.Event()
    done.record(s)
    buffers["done"] = done
    if wait:
        done.synchronize()
        return c
    return c, done


def device_status(stream: torch.cuda.Stream | None = None) -> int:
    """Synchronise and read the device status word (0 = no kernel gave up)."""
    out = ctypes.c_uint32(0)
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    code = load().gemm_get_device_status(s, ctypes.byref(out))
    if code not in (GEMM_OK, GEMM_ERR_DEVICE_TIMEOUT):
        raise GemmError(code, "gemm_get_device_status")
    return int(out.value)


def reset_device_status() -> None:
    code = load().gemm_reset_device_status()
    if code != GEMM_OK:
        raise GemmError(code, "gemm_reset_device_status")


def set_debug(flags: int = 0, wait_limit_ns: int = 0) -> None:
    load().gemm_set_debug(flags, wait_limit_ns)


def set_tuning(variant: int = 0, tile_n: int = 0, raster: int = 0, tail_split: int = 0) -> None:
    """Force the kernel variant (1 single CTA, 2 CTA pair, 3 two pairs sharing
    A, 4 CTA pair on the transposed product for row-major B), tile width, band
    height and tail split (1 never, 2 when possible) for later calls (0 = automatic)."""
    code = load().gemm_set_tuning(int(variant), int(tile_n), int(raster), int(tail_split))
    if code != GEMM_OK:
        raise GemmError(code, "gemm_set_tuning")


PLAN_FIELDS = ("kernel", "tile_n", "raster", "grid", "tail_segs", "concurrent_tiles", "tail_start", "work_items")


_KIND_CODE = {"f16": 0, "bf16": 1, "tf32": 2, "e4m3": 3, "e5m2": 4}


def plan_query(dtype: str, M: int, N: int, K: int, *, layout: int = GEMM_B_ROW_MAJOR, batch: int = 1,
               fused: bool = False, sms: int = 152, pair_clusters: int = 76, quad_clusters: int = 36) -> dict:
    """The plan the library's cost model picks for a product, without a device
    (gemm_plan_query; defaults: a GB300's SM and cluster counts)."""
    buf = (ctypes.c_int32 * 6)()
    code = load().gemm_plan_query(_KIND_CODE[dtype], M, N, K, layout, batch, int(fused), sms, pair_clusters,
                                  quad_clusters, buf)
    if code != GEMM_OK:
        raise GemmError(code, "gemm_plan_query")
    return dict(zip(PLAN_FIELDS[:6], list(buf)))


def last_plan() -> dict:
    """Launch plan of this thread's last product-kernel call (see gemm_last_plan)."""
    buf = (ctypes.c_int32 * 8)()
    load().gemm_last_plan(buf)
    return dict(zip(PLAN_FIELDS, list(buf)))


def free_workspaces() -> None:
    """Release the scratch buffers the library holds (waits for the device)."""
    code = load().gemm_free_workspaces()
    if code != GEMM_OK:
        raise GemmError(code, "gemm_free_workspaces")


def launch_count() -> int:
    return int(load().gemm_launch_count())
