"""ctypes binding over the C ABI of ``libgemm_f16.so`` (``include/gemm_f16.h``).

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes a ``cudaStream_t``, and status codes become
exceptions.  Every element of C is computed by the library's sm_103a kernel;
there is no fallback of any kind.  If the library has not been built, every
call raises :class:`LibraryNotBuilt`.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

from . import build as _build

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_ALIGNMENT = -2
GEMM_ERR_UNSUPPORTED_DEVICE = -3
GEMM_ERR_LAUNCH = -4
GEMM_ERR_TIMEOUT = -5
GEMM_ERR_CUDA = -6

# Config argument: id in the low byte, flag bits above (include/gemm_f16.h).
GEMM_F16_CONFIG_ID_MASK = 0xFF
GEMM_F16_NO_SPLIT = 0x100
GEMM_F16_NO_KSPLIT = 0x200
GEMM_F16_KSPLIT_AUTO = 0x400
GEMM_F16_KSPLIT_TAIL = 0x800
GEMM_F16_KSPLIT_SHIFT = 12
GEMM_F16_KSPLIT_MASK = 0x1F000


def ksplit(n: int) -> int:
    """Config flag: cut K into at most n slices (2 <= n <= 16), see gemm_f16.h."""
    return int(n) << GEMM_F16_KSPLIT_SHIFT

HEADER = os.path.join(_build.INCLUDE, "gemm_f16.h")


class LibraryNotBuilt(RuntimeError):
    pass


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status in (GEMM_ERR_INVALID_ARG, GEMM_ERR_ALIGNMENT):
            try:
                detail = lib().gemm_f16_last_error_detail().decode()
            except LibraryNotBuilt:
                pass
        self.detail = detail
        super().__init__(f"{what}: status {status} ({strerror(status)})" + (f": {detail}" if detail else ""))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises LibraryNotBuilt if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise LibraryNotBuilt(f"{_build.LIB} is missing; build it with __graft_entry__.build() "
                              "or python -m dense_fp16_gemm_05_gb300.build")
    L = ctypes.CDLL(_build.LIB)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.gemm_f16.argtypes = [vp, vp, vp, i64, i64, i64, ci, vp]
    L.gemm_f16.restype = ci
    L.gemm_f16_ex.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, vp]
    L.gemm_f16_ex.restype = ci
    L.gemm_f16_ex_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, vp]
    L.gemm_f16_ex_noalloc.restype = ci
    L.gemm_f16_from_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, ci, vp]
    L.gemm_f16_from_host.restype = ci
    L.gemm_f16_check.argtypes = [vp]
    L.gemm_f16_check.restype = ci
    L.gemm_f16_last_timeout_record.argtypes = []
    L.gemm_f16_last_timeout_record.restype = ctypes.c_uint64
    L.gemm_f16_last_error_detail.argtypes = []
    L.gemm_f16_last_error_detail.restype = ctypes.c_char_p
    L.gemm_f16_strerror.argtypes = [ci]
    L.gemm_f16_strerror.restype = ctypes.c_char_p
    L.gemm_f16_version.argtypes = []
    L.gemm_f16_version.restype = ci
    L.gemm_f16_num_configs.argtypes = []
    L.gemm_f16_num_configs.restype = ci
    L.gemm_f16_config_name.argtypes = [ci]
    L.gemm_f16_config_name.restype = ctypes.c_char_p
    L.gemm_f16_auto_config.argtypes = [i64, i64, i64]
    L.gemm_f16_auto_config.restype = ci
    L.gemm_f16_tx.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, ci, ci, vp]
    L.gemm_f16_tx.restype = ci
    L.gemm_f16_relu_backward.argtypes = [vp, vp, vp, i64, vp]
    L.gemm_f16_relu_backward.restype = ci
    L.gemm_f16_config_layouts.argtypes = [ci]
    L.gemm_f16_config_layouts.restype = ci
    L.gemm_f16_selftest_timeout.argtypes = [vp, vp, vp, i64, i64, i64, ci, ctypes.c_uint64, vp]
    L.gemm_f16_selftest_timeout.restype = ci
    L.attention_fwd_f16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float, ci, vp]
    L.attention_fwd_f16.restype = ci
    L.attention_fwd_f16_queue.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float, ci, vp, vp]
    L.attention_fwd_f16_queue.restype = ci
    L.gemm_fp8_block_scaled.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp]
    L.gemm_fp8_block_scaled.restype = ci
    L.gemm_mxfp8_block_scaled.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, ci, vp]
    L.gemm_mxfp8_block_scaled.restype = ci
    pi = ctypes.POINTER(ctypes.c_int)
    L.gemm_fp8_launch_info.argtypes = [i64, i64, i64, pi, pi]
    L.gemm_fp8_launch_info.restype = ci
    L.gemm_f16_launch_info.argtypes = [i64, i64, i64, ci, pi, pi, pi]
    L.gemm_f16_launch_info.restype = ci
    L.gemm_f16_config_cluster_k.argtypes = [ci]
    L.gemm_f16_config_cluster_k.restype = ci
    L.gemm_f16_tma_box_image.argtypes = [vp, i64, i64, i64, i64, i64, vp, vp]
    L.gemm_f16_tma_box_image.restype = ci
    _lib = L
    return L


def header_functions() -> list[str]:
    """Names of the functions declared in include/gemm_f16.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_f16\w*)\s*\(", text)))


def strerror(status: int) -> str:
    try:
        return lib().gemm_f16_strerror(int(status)).decode()
    except LibraryNotBuilt:
        return "library not built"


def version() -> int:
    return int(lib().gemm_f16_version())


def num_configs() -> int:
    return int(lib().gemm_f16_num_configs())


def config_name(config: int) -> str | None:
    r = lib().gemm_f16_config_name(int(config))
    return None if r is None else r.decode()


def config_label(config: int) -> str | None:
    """config_name plus "+nosplit" / "+ksplitN" / "+ksplitauto" / "+noksplit" for the flag bits."""
    name = config_name(config)
    if name is None:
        return None
    c = int(config)
    n = (c & GEMM_F16_KSPLIT_MASK) >> GEMM_F16_KSPLIT_SHIFT
    return (name + ("+nosplit" if c & GEMM_F16_NO_SPLIT else "") + (f"+ksplit{n}" if n else "")
            + ("+ksplitauto" if c & GEMM_F16_KSPLIT_AUTO else "") + ("+ksplittail" if c & GEMM_F16_KSPLIT_TAIL else "")
            + ("+noksplit" if c & GEMM_F16_NO_KSPLIT else ""))


# Raw handle of torch's current stream on a device, without building a
# torch.cuda.Stream object (a few microseconds per call on small problems).
_current_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


class _NoSwitch:
    __slots__ = ()

    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


_NO_SWITCH = _NoSwitch()


def _device_index(device) -> int:
    if isinstance(device, int):
        return device
    idx = (device if isinstance(device, torch.device) else torch.device(device)).index
    return idx if idx is not None else torch.cuda.current_device()


def _device_scope(device):
    """Makes ``device`` (a torch.device, index or name) current for the call;
    no switch when it already is."""
    if _device_index(device) == torch.cuda.current_device():
        return _NO_SWITCH
    return torch.cuda.device(device)


def _stream_handle(stream, device) -> int:
    if stream is None:
        if _current_raw_stream is not None:
            return int(_current_raw_stream(_device_index(device)))
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return int(stream.cuda_stream)
    return int(stream)


def _check_operand(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float16 or t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D float16 tensor, got {t.dtype} {tuple(t.shape)}")


def gemm_f16(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, relu: bool = True,
             stream=None, config: int = 0) -> torch.Tensor:
    """C = ReLU(A @ B) (relu=True) or A @ B, fp16 in and out, fp32 accumulation.

    A (M,K), B (K,N), C (M,N): contiguous float16 CUDA tensors on one device.
    C is allocated (torch.empty) when not given.  The call is asynchronous on
    ``stream`` (default: torch's current stream); errors in the arguments raise
    :class:`GemmError` immediately.
    """
    _check_operand(A, "A")
    _check_operand(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner sizes differ: A {tuple(A.shape)}, B {tuple(B.shape)}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_operand(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    L = _lib if _lib is not None else lib()
    with _device_scope(A.device):
        st = L.gemm_f16_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, int(bool(relu)), int(config),
                           _stream_handle(stream, A.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16")
    return C


def gemm_f16_noalloc(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, relu: bool = True, stream=None,
                     config: int = 0) -> torch.Tensor:
    """gemm_f16 through gemm_f16_ex_noalloc: K-slice partials in the library's
    fixed 16 MiB scratch instead of an allocation (see gemm_f16.h for the size
    limit and the rule that overlapping calls on one device race).  C must be
    given: nothing is allocated."""
    _check_operand(A, "A")
    _check_operand(B, "B")
    _check_operand(C, "C")
    M, K = A.shape
    K2, N = B.shape
    if K != K2 or tuple(C.shape) != (M, N):
        raise ValueError(f"shapes A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)} do not match")
    L = lib()
    with _device_scope(A.device):
        st = L.gemm_f16_ex_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, int(bool(relu)), int(config),
                                   _stream_handle(stream, A.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16_ex_noalloc")
    return C


def gemm_f16_t(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, transa: bool = False,
               transb: bool = False, relu: bool = True, stream=None, config: int = 0) -> torch.Tensor:
    """C = ReLU(op(A) @ op(B)) (relu=True) or op(A) @ op(B), fp16, fp32 accumulation.

    op(A) = A if not transa (A is (M,K)), else A.T (A stored (K,M));
    op(B) = B if not transb (B is (K,N)), else B.T (B stored (N,K)).
    All tensors contiguous float16 CUDA tensors; C (M,N) is allocated if not given.
    """
    _check_operand(A, "A")
    _check_operand(B, "B")
    M, K = (A.shape[1], A.shape[0]) if transa else (A.shape[0], A.shape[1])
    K2, N = (B.shape[1], B.shape[0]) if transb else (B.shape[0], B.shape[1])
    if K != K2:
        raise ValueError(f"inner sizes differ: op(A) {M}x{K}, op(B) {K2}x{N}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_operand(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    with _device_scope(A.device):
        st = lib().gemm_f16_tx(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, int(bool(transa)),
                               int(bool(transb)), int(bool(relu)), int(config), _stream_handle(stream, A.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16_tx")
    return C


def relu_backward(dC: torch.Tensor, C: torch.Tensor, dZ: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dZ = dC where C > 0 else +0 (gradient through the fused ReLU), on the GPU."""
    for t, n in ((dC, "dC"), (C, "C")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float16 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float16 tensor")
    if dC.shape != C.shape:
        raise ValueError(f"dC {tuple(dC.shape)} and C {tuple(C.shape)} differ")
    if dZ is None:
        dZ = torch.empty_like(dC)
    with _device_scope(dC.device):
        st = lib().gemm_f16_relu_backward(dC.data_ptr(), C.data_ptr(), dZ.data_ptr(), dC.numel(),
                                          _stream_handle(stream, dC.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16_relu_backward")
    return dZ


def tma_box_image(X: torch.Tensor, box_rows: int, x: int, y: int, stream=None) -> torch.Tensor:
    """Raw shared-memory image (uint8, box_rows * 128 bytes) of one box of
    box_rows x 64 elements of the 2-D fp16 tensor X at column x, row y, loaded
    by TMA with the GEMM's operand encoding (gemm_f16_tma_box_image)."""
    _check_operand(X, "X")
    rows, cols = X.shape
    out = torch.empty(int(box_rows) * 128, dtype=torch.uint8, device=X.device)
    L = lib()
    with _device_scope(X.device):
        st = L.gemm_f16_tma_box_image(X.data_ptr(), rows, cols, int(box_rows), int(x), int(y), out.data_ptr(),
                                      _stream_handle(stream, X.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16_tma_box_image")
    return out


def config_cluster_k(config: int) -> bool:
    """True if the configuration splits K across a cluster (no workspace)."""
    r = lib().gemm_f16_config_cluster_k(int(config))
    if r < 0:
        raise GemmError(r, "gemm_f16_config_cluster_k")
    return r == 1


def workspace_split_configs() -> list[int]:
    """Fixed configuration ids whose K split uses a workspace."""
    return [c for c in range(1, num_configs() + 1) if not config_cluster_k(c)]


def config_layouts(config: int) -> int:
    return int(lib().gemm_f16_config_layouts(int(config)))


def gemm_f16_raw(A_ptr: int, B_ptr: int, C_ptr: int, M: int, N: int, K: int, relu: int, stream: int = 0,
                 config: int = 0) -> int:
    """The C call with raw pointers; returns the status code (no exception)."""
    return int(lib().gemm_f16_ex(A_ptr, B_ptr, C_ptr, M, N, K, relu, config, stream))


def gemm_f16_from_host(A_host: torch.Tensor, B_host: torch.Tensor, C_host: torch.Tensor,
                       A_dev: torch.Tensor, B_dev: torch.Tensor, C_dev: torch.Tensor,
                       relu: bool = True, stream=None) -> None:
    """End-to-end call: host A, B -> device, GEMM, device C -> host, ordered on ``stream``.

    A and C move in row panels so that copies and GEMMs overlap (see
    gemm_f16.h); the host tensors should be pinned (``pin_memory()``) for
    asynchronous copies.  Returns after enqueueing; synchronising the stream
    is enough before reading C_host.
    """
    for t, n in ((A_host, "A_host"), (B_host, "B_host"), (C_host, "C_host"),
                 (A_dev, "A_dev"), (B_dev, "B_dev"), (C_dev, "C_dev")):
        _check_operand(t, n)
    M, K = A_host.shape
    N = B_host.shape[1]
    L = lib()
    with _device_scope(A_dev.device):
        st = L.gemm_f16_from_host(A_host.data_ptr(), B_host.data_ptr(), C_host.data_ptr(), A_dev.data_ptr(),
                                  B_dev.data_ptr(), C_dev.data_ptr(), M, N, K, int(bool(relu)),
                                  _stream_handle(stream, A_dev.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16_from_host")


def check(stream=None, device=None) -> int:
    """Synchronises the stream and returns the device status (GEMM_OK or an error code)."""
    dev = device if device is not None else torch.cuda.current_device()
    with _device_scope(dev):
        return int(lib().gemm_f16_check(_stream_handle(stream, dev)))


def auto_config(M: int, N: int, K: int) -> int:
    return int(lib().gemm_f16_auto_config(M, N, K))


def launch_info(M: int, N: int, K: int, config: int = 0) -> dict:
    """Grid CTAs, cluster size and tile count that a call would launch with."""
    g, c, t = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = lib().gemm_f16_launch_info(M, N, K, int(config), ctypes.byref(g), ctypes.byref(c), ctypes.byref(t))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_f16_launch_info")
    return {"grid_ctas": g.value, "cluster_size": c.value, "tiles": t.value}


def selftest_timeout(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, config: int = 0,
                     timeout_cycles: int = 1 << 24, stream=None) -> int:
    """Launches the kernel with its producer switched off so that a bounded wait
    runs out (test hook); returns the launch status.  Read the outcome with check()."""
    M, K = A.shape
    N = B.shape[1]
    with _device_scope(A.device):
        return int(lib().gemm_f16_selftest_timeout(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, int(config),
                                                   int(timeout_cycles), _stream_handle(stream, A.device)))


def last_timeout_record() -> int:
    return int(lib().gemm_f16_last_timeout_record())


FP8_BLOCK = 128


def _check_fp8(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D uint8 / float8_e4m3fn tensor, got {t.dtype} {tuple(t.shape)}")


def _check_scales(t: torch.Tensor, name: str, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous float32 tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)}")


def gemm_fp8_block_scaled(A: torch.Tensor, SA: torch.Tensor, W: torch.Tensor, SW: torch.Tensor,
                          C: torch.Tensor | None = None, relu: bool = False, stream=None) -> torch.Tensor:
    """C = R(sum_b SA[:,b] SW[n/128,b] (A_b @ W_b^T)): the FP8 block-scaled linear layer.

    A (M,K) and W (N,K): E4M3 codes (uint8 or float8_e4m3fn) on one CUDA
    device; SA (M, ceil(K/128)) and SW (ceil(N/128), ceil(K/128)) float32;
    C (M,N) float16, allocated when not given.  Asynchronous on ``stream``.
    """
    _check_fp8(A, "A")
    _check_fp8(W, "W")
    M, K = A.shape
    N, K2 = W.shape
    if K != K2:
        raise ValueError(f"inner sizes differ: A {tuple(A.shape)}, W {tuple(W.shape)}")
    KB, NB = -(-K // FP8_BLOCK), -(-N // FP8_BLOCK)
    _check_scales(SA, "SA", (M, KB))
    _check_scales(SW, "SW", (NB, KB))
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_operand(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    L = lib()
    with _device_scope(A.device):
        st = L.gemm_fp8_block_scaled(A.data_ptr(), SA.data_ptr(), W.data_ptr(), SW.data_ptr(), C.data_ptr(),
                                     M, N, K, int(bool(relu)), _stream_handle(stream, A.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_fp8_block_scaled")
    return C


def gemm_mxfp8_block_scaled(A: torch.Tensor, SA: torch.Tensor, W: torch.Tensor, SW: torch.Tensor,
                            C: torch.Tensor | None = None, relu: bool = True, stream=None) -> torch.Tensor:
    """FP8 block-scaled GEMM with power-of-two scales: SA (M, ceil(K/128)) and
    SW (ceil(N/128), ceil(K/128)) uint8 E8M0 exponents; otherwise as
    gemm_fp8_block_scaled (see gemm_f16.h)."""
    _check_fp8(A, "A")
    _check_fp8(W, "W")
    M, K = A.shape
    N, K2 = W.shape
    if K != K2:
        raise ValueError(f"A {tuple(A.shape)} and W {tuple(W.shape)} disagree on K")
    KB, NB = -(-K // 128), -(-N // 128)
    for t, name, shape in ((SA, "SA", (M, KB)), (SW, "SW", (NB, KB))):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous uint8 tensor of shape {shape}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_operand(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    L = lib()
    with _device_scope(A.device):
        st = L.gemm_mxfp8_block_scaled(A.data_ptr(), SA.data_ptr(), W.data_ptr(), SW.data_ptr(), C.data_ptr(),
                                       M, N, K, int(bool(relu)), _stream_handle(stream, A.device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_mxfp8_block_scaled")
    return C


def fp8_launch_info(M: int, N: int, K: int) -> dict:
    g, t = ctypes.c_int(0), ctypes.c_int(0)
    st = lib().gemm_fp8_launch_info(M, N, K, ctypes.byref(g), ctypes.byref(t))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_fp8_launch_info")
    return {"grid_ctas": g.value, "tiles": t.value}


def _launch_stream(stream, device) -> torch.cuda.Stream:
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def attention_fwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor | None = None,
                  sm_scale: float | None = None, causal: bool = False, stream=None,
                  queue: torch.Tensor | bool | None = None) -> torch.Tensor:
    """O = softmax(sm_scale Q K^T [causal]) V per (batch, head).

    Q, K, V (and O): contiguous float16 CUDA tensors of one shape
    (batch, heads, seq, dim), dim 64 or 128; sm_scale defaults to
    1/sqrt(dim).  O is allocated when not given.  Asynchronous on ``stream``.

    ``queue`` (causal only): the work queue of attention_fwd_f16_queue, a
    2-element int32 CUDA tensor that is zero when the launch starts and that
    the kernel leaves zero; one queue serves launches that run one after
    another, launches that may overlap need one each.  None: a fresh zeroed
    queue is made on the launch stream for this call.  False: no queue (the
    fixed shares of attention_fwd_f16).  Results are the same bits either way.
    """
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous 4-D float16 tensor")
    if Q.shape != K.shape or Q.shape != V.shape:
        raise ValueError(f"Q, K, V shapes differ: {tuple(Q.shape)} {tuple(K.shape)} {tuple(V.shape)}")
    B, H, S, D = Q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if O is None:
        O = torch.empty_like(Q)
    if O.dtype != torch.float16 or O.shape != Q.shape or not O.is_contiguous():
        raise ValueError("O must be a contiguous float16 tensor shaped like Q")
    q_ptr = None
    if causal and queue is not False and Q.numel() > 0:
        if queue is None or queue is True:
            with torch.cuda.stream(_launch_stream(stream, Q.device)):
                queue = torch.zeros(2, dtype=torch.int32, device=Q.device)
        if (not isinstance(queue, torch.Tensor) or queue.dtype != torch.int32 or queue.numel() < 2
                or not queue.is_contiguous() or queue.device != Q.device):
            raise ValueError("queue must be a contiguous int32 tensor of >= 2 elements on Q's device")
        q_ptr = queue.data_ptr()
    L = lib()
    with _device_scope(Q.device):
        st = L.attention_fwd_f16_queue(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), B, H, S, D,
                                       float(sm_scale), int(bool(causal)), q_ptr, _stream_handle(stream, Q.device))
    if st != GEMM_OK:
        raise GemmError(st, "attention_fwd_f16_queue")
    return O
