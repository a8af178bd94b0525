"""ctypes binding of libtgemm.so (declared in ``include/tgemm.h``).

Argument marshalling only: every step of the product runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. If the
compiled library is missing, every call raises :class:`TgemmError`; there is
no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

TGEMM_OK = 0
TGEMM_ERR_INVALID_ARG = 1
TGEMM_ERR_ALIGNMENT = 2
TGEMM_ERR_CUDA = 3
TGEMM_ERR_DEVICE_TIMEOUT = 4
TGEMM_ERR_UNSUPPORTED = 5

TGEMM_TF32 = 1
TGEMM_BF16 = 2

_HERE = os.path.dirname(os.path.abspath(__file__))

# Every symbol the header declares, with (restype, argtypes).
_VP = ctypes.c_void_p
_SIGNATURES = {
    "gemm_f32": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                _VP, ctypes.c_long, _VP, ctypes.c_long,
                                _VP, ctypes.c_long, _VP]),
    "gemm_tc": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               _VP, ctypes.c_long, _VP, ctypes.c_long,
                               _VP, ctypes.c_long, ctypes.c_int, _VP]),
    "gemm_ex": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               _VP, ctypes.c_long, _VP, ctypes.c_long,
                               _VP, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                               ctypes.c_float, ctypes.c_float, _VP, _VP]),
    "gemm_host": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 _VP, ctypes.c_long, _VP, ctypes.c_long,
                                 _VP, ctypes.c_long, ctypes.c_int, _VP]),
    "gemm_device_status": (ctypes.c_int, [_VP]),
    "gemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gemm_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_longlong]),
    "gemm_set_debug_stall": (ctypes.c_int, [ctypes.c_int]),
    "gemm_set_f32_kernel": (ctypes.c_int, [ctypes.c_int]),
    "gemm_set_tc_kernel": (ctypes.c_int, [ctypes.c_int]),
    "gemm_set_tc_streamk": (ctypes.c_int, [ctypes.c_int]),
    "gemm_set_tc_a_loader": (ctypes.c_int, [ctypes.c_int]),
    "gemm_f32_kernel_count": (ctypes.c_int, []),
    "gemm_f32_kernel_name": (ctypes.c_char_p, [ctypes.c_int]),
    "gemm_last_kernel": (ctypes.c_char_p, []),
    "gemm_tc_tf32_noalloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            _VP, ctypes.c_long, _VP, ctypes.c_long,
                                            _VP, ctypes.c_long, _VP]),
    "gemm_scratch_bytes": (ctypes.c_longlong, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               _VP, ctypes.c_long, _VP, ctypes.c_long,
                                               _VP, ctypes.c_long, ctypes.c_int, ctypes.c_int]),
    "gemm_plan_name": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      _VP, ctypes.c_long, _VP, ctypes.c_long,
                                      _VP, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_char_p, ctypes.c_int]),
    "gemm_tc_peak": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_long,
                                    ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                    _VP]),
}


class TgemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what
                         else f"{status_string(status)} ({status})")


def library_path() -> str:
    return os.environ.get("TGEMM_LIBRARY", os.path.join(_HERE, "_build", "libtgemm.so"))


_lib = None


def load() -> ctypes.CDLL:
    """Load libtgemm.so (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libtgemm.so not found at {path}; build it with "
                "`python -m tiled_matrix_multiplication_sm_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    try:
        return load().gemm_status_string(int(status)).decode()
    except RuntimeError:
        return {0: "ok", 1: "invalid argument", 2: "misaligned operand",
                3: "CUDA error", 4: "device wait timed out",
                5: "unsupported device"}.get(status, "unknown tgemm status")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream: Optional[torch.cuda.Stream], device_index: Optional[int] = None) -> int:
    """The CUDA stream handle to launch on: ``stream``, else the current
    stream of device ``device_index`` (default: the current device)."""
    if stream is not None:
        return int(stream.cuda_stream)
    if device_index is None:
        device_index = torch.cuda.current_device()
    if _raw_stream is not None:
        return int(_raw_stream(device_index))
    return int(torch.cuda.current_stream(device_index).cuda_stream)


def _on_device(device: torch.device, call):
    """Run ``call(device_index)`` with ``device`` current; switches devices
    only when another one is current (a switch costs microseconds)."""
    current = torch.cuda.current_device()
    index = device.index if device.index is not None else current
    if index == current:
        return call(index)
    with torch.cuda.device(index):
        return call(index)


def gemm_f32_raw(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, stream_handle=0) -> int:
    """Direct call of the C entry point; returns its status code."""
    return int(load().gemm_f32(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, stream_handle))


def gemm_tc_raw(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, in_type, stream_handle=0) -> int:
    return int(load().gemm_tc(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, in_type,
                              stream_handle))


def gemm_tc_tf32_noalloc_raw(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, stream_handle=0) -> int:
    """The allocation-free TF32 entry point; returns its status code."""
    return int(load().gemm_tc_tf32_noalloc(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc,
                                           stream_handle))


def _check_matrix(x: torch.Tensor, name: str, dtype: torch.dtype) -> int:
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.ndim != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(x.shape)}")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    rows_stride, col_stride = x.stride()
    cols = x.shape[1]
    if cols > 1 and col_stride != 1:
        raise ValueError(f"{name} must have unit column stride (row-major)")
    # A one-row view keeps its row stride too, so a padded leading dimension
    # is passed through unchanged (it decides which loaders may be used).
    return max(rows_stride, cols, 1)


def _out(out, M, N, device):
    if out is None:
        return torch.empty((M, N), dtype=torch.float32, device=device)
    if tuple(out.shape) != (M, N):
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {(M, N)}")
    return out


def gemm_f32(A: torch.Tensor, B: torch.Tensor, out: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = A @ B on the FP32 CUDA-core path (asynchronous on ``stream``)."""
    lda = _check_matrix(A, "A", torch.float32)
    ldb = _check_matrix(B, "B", torch.float32)
    M, K = A.shape
    if B.shape[0] != K:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} x {tuple(B.shape)}")
    N = B.shape[1]
    C = _out(out, M, N, A.device)
    ldc = _check_matrix(C, "out", torch.float32)
    st = _on_device(A.device, lambda dev: gemm_f32_raw(
        M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
        _stream_handle(stream, dev)))
    if st != TGEMM_OK:
        raise TgemmError(st, "gemm_f32")
    return C


TGEMM_TF32X3 = 3
_TC_TYPES = {"tf32": (TGEMM_TF32, torch.float32), "bf16": (TGEMM_BF16, torch.bfloat16),
             "tf32x3": (TGEMM_TF32X3, torch.float32)}


def gemm_tc(A: torch.Tensor, B: torch.Tensor, in_type: str = "bf16",
            out: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = A @ B on the tcgen05 tensor-core path; ``in_type`` is "tf32", "bf16"
    or "tf32x3" (split TF32, FP32-level accuracy)."""
    code, dtype = _TC_TYPES[in_type]
    lda = _check_matrix(A, "A", dtype)
    ldb = _check_matrix(B, "B", dtype)
    M, K = A.shape
    if B.shape[0] != K:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} x {tuple(B.shape)}")
    N = B.shape[1]
    C = _out(out, M, N, A.device)
    ldc = _check_matrix(C, "out", torch.float32)
    st = _on_device(A.device, lambda dev: gemm_tc_raw(
        M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc, code,
        _stream_handle(stream, dev)))
    if st != TGEMM_OK:
        raise TgemmError(st, "gemm_tc")
    return C


def device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise ``stream`` and return (and clear) the kernels' wait status."""
    return int(load().gemm_device_status(_stream_handle(stream)))


def set_wait_limit_ns(ns: int) -> int:
    return int(load().gemm_set_wait_limit_ns(int(ns)))


def tc_peak(kind: str = "bf16", pair: bool = True, iters: int = 200000,
            stream: Optional[torch.cuda.Stream] = None):
    """Dense MMA rate of the tensor cores (gemm_tc_peak): returns
    (FLOP per SM clock cycle, TFLOP/s over the launch at the running clock)."""
    in_type = {"bf16": TGEMM_BF16, "tf32": TGEMM_TF32}[kind]
    per_clk = ctypes.c_double(0.0)
    tflops = ctypes.c_double(0.0)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = int(load().gemm_tc_peak(in_type, 1 if pair else 0, int(iters), ctypes.byref(per_clk),
                                 ctypes.byref(tflops), int(s.cuda_stream)))
    if st != TGEMM_OK:
        raise TgemmError(st, "gemm_tc_peak")
    return per_clk.value, tflops.value


def set_debug_stall(enable: bool) -> int:
    return int(load().gemm_set_debug_stall(1 if enable else 0))


def set_f32_kernel(kernel_id: int) -> int:
    return int(load().gemm_set_f32_kernel(int(kernel_id)))


def set_tc_kernel(mode: int) -> int:
    """-1: by shape; 0: one-SM tcgen05 kernel (128 x 256 tiles); 1: 2-SM
    (CTA pair) kernel, 256 x 256 tiles; 2: 2-SM kernel, 256 x 512 tiles."""
    return int(load().gemm_set_tc_kernel(int(mode)))


def set_tc_streamk(slots: int) -> int:
    """Stream-K tail of the tensor-core kernels: -1 automatic, 0 never, S > 0
    shared by S SMs or SM pairs where the tail allows it."""
    return int(load().gemm_set_tc_streamk(int(slots)))


def set_tc_a_loader(mode: int) -> int:
    """A with rows 4- but not 16-byte aligned on the tensor paths: -1 / 0
    repacked first, 1 read in place by the GEMM kernel's loader warps."""
    return int(load().gemm_set_tc_a_loader(int(mode)))


def f32_kernel_names():
    lib = load()
    return [lib.gemm_f32_kernel_name(i).decode() for i in range(lib.gemm_f32_kernel_count())]


def last_kernel() -> str:
    return load().gemm_last_kernel().decode()


TGEMM_PATH = {"f32": 0, "tf32": 1, "bf16": 2, "tf32x3": 3}
TGEMM_TRANS_A = 1
TGEMM_TRANS_B = 2
_PATH_DTYPE = {"f32": torch.float32, "tf32": torch.float32, "bf16": torch.bfloat16,
               "tf32x3": torch.float32}


def gemm_ex(A: torch.Tensor, B: torch.Tensor, path: str = "f32", trans_a: bool = False,
            trans_b: bool = False, alpha: float = 1.0, beta: float = 0.0,
            bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """C = alpha * op(A) @ op(B) + beta * C + bias through gemm_ex.

    ``A``/``B`` are the stored matrices: A is K x M when ``trans_a`` (else
    M x K), B is N x K when ``trans_b`` (else K x N). ``bias`` is a CUDA
    float32 vector of N entries; ``out`` is read when ``beta != 0``.
    """
    dtype = _PATH_DTYPE[path]
    lda = _check_matrix(A, "A", dtype)
    ldb = _check_matrix(B, "B", dtype)
    M, K = (A.shape[1], A.shape[0]) if trans_a else (A.shape[0], A.shape[1])
    K2, N = (B.shape[1], B.shape[0]) if trans_b else (B.shape[0], B.shape[1])
    if K != K2:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} / {tuple(B.shape)}")
    if beta != 0.0 and out is None:
        raise ValueError("beta != 0 needs out (the C that is read)")
    C = _out(out, M, N, A.device)
    ldc = _check_matrix(C, "out", torch.float32)
    bias_ptr = None
    if bias is not None:
        if bias.device.type != "cuda" or bias.dtype != torch.float32 or bias.numel() != N:
            raise ValueError("bias must be a CUDA float32 tensor of N entries")
        if not bias.is_contiguous():
            bias = bias.contiguous()
            if stream is not None:
                bias.record_stream(stream)     # the copy lives until `stream` has read it
        bias_ptr = bias.data_ptr()
    flags = (TGEMM_TRANS_A if trans_a else 0) | (TGEMM_TRANS_B if trans_b else 0)
    st = _on_device(A.device, lambda dev: int(load().gemm_ex(
        M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc, TGEMM_PATH[path],
        flags, float(alpha), float(beta), bias_ptr, _stream_handle(stream, dev))))
    if st != TGEMM_OK:
        raise TgemmError(st, "gemm_ex")
    return C


def plan_name_raw(M: int, N: int, K: int, a_ptr: int, lda: int, b_ptr: int, ldb: int,
                  c_ptr: int, ldc: int, path: str = "f32", trans_a: bool = False,
                  trans_b: bool = False, num_sms: int = 152) -> str:
    """The kernels ``gemm_ex`` would launch for this problem on a device with
    ``num_sms`` SMs (gemm_plan_name: no GPU needed; only the pointers'
    alignment matters), in gemm_last_kernel's form."""
    buf = ctypes.create_string_buffer(256)
    flags = (TGEMM_TRANS_A if trans_a else 0) | (TGEMM_TRANS_B if trans_b else 0)
    st = int(load().gemm_plan_name(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, TGEMM_PATH[path],
                                   flags, num_sms, buf, len(buf)))
    if st != TGEMM_OK:
        raise TgemmError(st, "gemm_plan_name")
    return buf.value.decode()


def scratch_bytes(A: torch.Tensor, B: torch.Tensor, path: str = "f32", trans_a: bool = False,
                  trans_b: bool = False, out: Optional[torch.Tensor] = None) -> int:
    """Bytes of device scratch the library's pool would give the product
    ``gemm_ex(A, B, path, trans_a, trans_b, out=out)`` (0: it allocates
    nothing). Without ``out``, C is taken to be a packed, 16-byte-aligned
    M x N float32 matrix."""
    dtype = _PATH_DTYPE[path]
    lda = _check_matrix(A, "A", dtype)
    ldb = _check_matrix(B, "B", dtype)
    M, K = (A.shape[1], A.shape[0]) if trans_a else (A.shape[0], A.shape[1])
    N = B.shape[0] if trans_b else B.shape[1]
    if out is None:
        c_ptr, ldc = 256, max(N, 1)
    else:
        c_ptr, ldc = out.data_ptr(), _check_matrix(out, "out", torch.float32)
    flags = (TGEMM_TRANS_A if trans_a else 0) | (TGEMM_TRANS_B if trans_b else 0)
    n = _on_device(A.device, lambda dev: int(load().gemm_scratch_bytes(
        M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, c_ptr, ldc, TGEMM_PATH[path], flags)))
    if n < 0:
        raise TgemmError(-n, "gemm_scratch_bytes")
    return n


def _check_host_matrix(x: torch.Tensor, name: str, dtype: torch.dtype) -> int:
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor")
    if x.device.type != "cpu":
        raise ValueError(f"{name} must be a host tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if x.shape[1] > 1 and x.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride (row-major)")
    return max(int(x.stride(0)), int(x.shape[1]), 1)


def gemm_host(A: torch.Tensor, B: torch.Tensor, path: str = "f32",
              out: Optional[torch.Tensor] = None,
              stream: Optional[torch.cuda.Stream] = None,
              synchronize: bool = True) -> torch.Tensor:
    """C = A @ B for HOST operands through gemm_host (copies overlapped with
    the product). Returns once C is complete on the host; with
    ``synchronize=False`` it returns once the work is enqueued on ``stream``,
    and C (and the reuse of A, B) waits for that stream to be synchronised --
    two such calls on two streams overlap."""
    dtype = _PATH_DTYPE[path]
    lda = _check_host_matrix(A, "A", dtype)
    ldb = _check_host_matrix(B, "B", dtype)
    M, K = A.shape
    if B.shape[0] != K:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} x {tuple(B.shape)}")
    N = B.shape[1]
    C = out if out is not None else torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    if tuple(C.shape) != (M, N) or C.dtype != torch.float32:
        raise ValueError("out must be a float32 M x N host tensor")
    ldc = _check_host_matrix(C, "out", torch.float32)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = int(load().gemm_host(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
                              TGEMM_PATH[path], int(s.cuda_stream)))
    if st != TGEMM_OK:
        raise TgemmError(st, "gemm_host")
    if synchronize:
        s.synchronize()
    return C


def matmul(A: torch.Tensor, B: torch.Tensor, path: str = "f32",
           out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """End-to-end product through the library for host or device operands.

    ``path`` is "f32" (CUDA cores), "tf32", "bf16" or "tf32x3" (tensor cores;
    "tf32x3" at FP32-level accuracy). Host
    operands go through gemm_host (copies to the device overlapped with the
    product, result copied back, into ``out`` if given -- ideally pinned)
    and the call returns once C is on the host; device operands give a
    device result (in ``out`` if given).
    """
    if path not in _PATH_DTYPE:
        raise ValueError(f"unknown path {path!r}")
    if A.device.type == "cpu":
        return gemm_host(A, B, path, out=out)
    if path == "f32":
        return gemm_f32(A, B, out=out)
    return gemm_tc(A, B, path, out=out)
