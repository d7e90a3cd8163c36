"""Python binding of libq4_0.so (argument marshalling only).

Every function checks the tensors it is given (dtype, device, shape,
contiguity), passes raw device pointers and the current CUDA stream to the
C ABI declared in include/q4_0.h, and raises Q4Error on a non-zero status.
All arithmetic happens in the library's CUDA kernels; there is no fallback:
if the library is not built, the first call raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libq4_0.so")

# Status codes (include/q4_0.h).
OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_DEVICE_TIMEOUT = -4
ERR_WORKSPACE = -5

# Output element types of q4_0_matmul_ex (include/q4_0.h).
Y_F32 = 0
Y_BF16 = 1

# Every entry point the header declares, with its ctypes signature.
_P, _I64, _SZ, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
SIGNATURES = {
    "q4_0_version": ([], _INT),
    "q4_0_status_string": ([_INT], ctypes.c_char_p),
    "q4_0_weight_bytes": ([_I64, _I64], _SZ),
    "q4_0_quantize": ([_P, _P, _I64, _I64, _P], _INT),
    "q4_0_matmul": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "q4_0_matmul_workspace_bytes": ([_I64, _I64, _I64], _SZ),
    "q4_0_matmul_ws": ([_P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _INT),
    "q4_0_matmul_ex": ([_P, _P, _P, _INT, _I64, _I64, _I64, _P, _SZ, _P], _INT),
    "q4_0_matmul_host_workspace_bytes": ([_I64, _I64, _I64, _INT], _SZ),
    "q4_0_matmul_host": ([_P, _P, _P, _INT, _I64, _I64, _I64, _P, _SZ, _P], _INT),
    "q4_0_matmul_grouped": ([_INT, _P, _P, _P, _INT, _I64, _P, _P, _P], _INT),
    "q4_0_matmul_grouped_launches": ([_INT, _I64, _P, _P], _INT),
    "q4_0_gemv": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "q4_0_gemv_workspace_bytes": ([_I64, _I64], _SZ),
    "q4_0_gemv_ws": ([_P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _INT),
    "q4_0_gemm_workspace_bytes": ([_I64, _I64, _I64], _SZ),
    "q4_0_gemm": ([_P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], _INT),
    "q4_0_gemm_noalloc": ([_P, _P, _P, _I64, _I64, _I64, _P], _INT),
    "q4_0_gemm_plan": ([_I64, _I64, _I64, _P, _P, _P], _INT),
    "q4_0_selftest_wait_timeout": ([_I64, _P], _INT),
    "q4_0_device_error": ([ctypes.POINTER(_INT)], _INT),
}

_lib = None


class Q4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def lib():
    """Load libq4_0.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with q4_weight_only_gb300.build.build() "
                "(nvcc, sm_103a). There is no fallback implementation.")
        l = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = res
        _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().q4_0_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != OK:
        raise Q4Error(status, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def version() -> int:
    return int(lib().q4_0_version())


def weight_bytes(N: int, K: int) -> int:
    return int(lib().q4_0_weight_bytes(N, K))


def quantize(w: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """fp32 [N, K] -> Q4_0 bytes uint8 [N, K/32*18] (device)."""
    _need(w, "w", torch.float32, 2)
    N, K = w.shape
    nbytes = weight_bytes(N, K)
    if nbytes == 0:
        raise ValueError("K must be a positive multiple of 32")
    if out is None:
        out = torch.empty((N, nbytes // N), dtype=torch.uint8, device=w.device)
    _need(out, "out", torch.uint8, 2)
    if out.numel() != nbytes:
        raise ValueError("out has the wrong size")
    _check(lib().q4_0_quantize(w.data_ptr(), out.data_ptr(), N, K, _stream(stream)), "q4_0_quantize")
    return out


def _q4_bytes(N: int, K: int) -> int:
    # q4_0_weight_bytes without a library call (it runs on every matmul call)
    return N * (K // 32) * 18 if N > 0 and K > 0 and K % 32 == 0 else 0


_ws_cache = {}


def _ws_bytes(fn: str, *args) -> int:
    # a workspace size depends on the arguments and on the current device
    # (the GEMM's K split follows its SM count): one library query per
    # distinct (device, call shape)
    key = (fn, torch.cuda.current_device()) + args
    v = _ws_cache.get(key)
    if v is None:
        v = _ws_cache[key] = int(getattr(lib(), fn)(*args))
    return v


def _mm_args(x, wq, N, K, out, out_dtype=torch.float32):
    _need(x, "x", torch.bfloat16, 2)
    _need(wq, "wq", torch.uint8, 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] must equal K")
    if wq.numel() != _q4_bytes(N, K):
        raise ValueError("wq does not hold an N x K Q4_0 matrix")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    _need(out, "out", out_dtype, 2)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    return M, out


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() < nbytes:
        raise ValueError("workspace too small")
    return workspace, workspace.numel()


def matmul(x: torch.Tensor, wq: torch.Tensor, N: int, K: int, out: torch.Tensor = None,
           workspace: torch.Tensor = None, stream=None, out_dtype=torch.float32) -> torch.Tensor:
    """y = x W^T: x bf16 [M, K], wq Q4_0 [N, K] -> [M, N] fp32 (the dispatcher),
    or bf16 with out_dtype=torch.bfloat16 (q4_0_matmul_ex)."""
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
    M, out = _mm_args(x, wq, N, K, out, out_dtype)
    if out_dtype == torch.bfloat16:
        ws, wsb = _workspace(_ws_bytes("q4_0_matmul_workspace_bytes", M, N, K), x.device, workspace)
        _check(lib().q4_0_matmul_ex(x.data_ptr(), wq.data_ptr(), out.data_ptr(), Y_BF16, M, N, K,
                                    ws.data_ptr() if ws is not None else None, wsb, _stream(stream)),
               "q4_0_matmul_ex")
        return out
    ws, wsb = _workspace(_ws_bytes("q4_0_matmul_workspace_bytes", M, N, K), x.device, workspace)
    _check(lib().q4_0_matmul_ws(x.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K,
                                ws.data_ptr() if ws is not None else None, wsb, _stream(stream)),
           "q4_0_matmul")
    return out


def matmul_host(x: torch.Tensor, wq: torch.Tensor, N: int, K: int, out: torch.Tensor = None,
                workspace: torch.Tensor = None, stream=None, out_dtype=torch.float32) -> torch.Tensor:
    """y = x W^T with x and y in host memory, through q4_0_matmul_host: x bf16
    [M, K] on the host (page-locked for asynchronous copies), wq Q4_0 on the
    device, y [M, N] of out_dtype on the host (allocated page-locked when not
    given).  One call copies x in, runs the dispatcher and copies y back on
    the stream; synchronise the stream before reading y.  workspace: a device
    uint8 tensor of at least host_workspace_bytes(M, N, K, out_dtype)."""
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or x.is_cuda or x.dim() != 2 \
            or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D bf16 host tensor")
    _need(wq, "wq", torch.uint8, 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] must equal K")
    if wq.numel() != _q4_bytes(N, K):
        raise ValueError("wq does not hold an N x K Q4_0 matrix")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, pin_memory=True)
    if not isinstance(out, torch.Tensor) or out.dtype != out_dtype or out.is_cuda \
            or tuple(out.shape) != (M, N) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] host tensor of out_dtype")
    yt = Y_BF16 if out_dtype == torch.bfloat16 else Y_F32
    ws, wsb = _workspace(_ws_bytes("q4_0_matmul_host_workspace_bytes", M, N, K, yt), wq.device, workspace)
    _check(lib().q4_0_matmul_host(x.data_ptr(), wq.data_ptr(), out.data_ptr(), yt, M, N, K,
                                  ws.data_ptr() if ws is not None else None, wsb, _stream(stream)),
           "q4_0_matmul_host")
    return out


def matmul_grouped(xs, wqs, Ns, Ks, outs=None, stream=None, out_dtype=torch.float32):
    """y_g = x_g W_g^T for independent problems sharing M, through
    q4_0_matmul_grouped (one persistent decode launch per group where the
    problems allow it).  Returns the list of outputs."""
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")
    G = len(xs)
    if not (len(wqs) == len(Ns) == len(Ks) == G):
        raise ValueError("xs, wqs, Ns and Ks must have the same length")
    outs = list(outs) if outs is not None else [None] * G
    if len(outs) != G:
        raise ValueError("outs must have one tensor per problem")
    M, ys = None, []
    for x, wq, N, K, out in zip(xs, wqs, Ns, Ks, outs):
        m, out = _mm_args(x, wq, N, K, out, out_dtype)
        if M is None:
            M = m
        elif m != M:
            raise ValueError("every x must have the same number of rows")
        ys.append(out)
    if G == 0:
        return ys
    ptrs = lambda ts: ctypes.cast((ctypes.c_void_p * G)(*[t.data_ptr() for t in ts]), ctypes.c_void_p)
    sizes = lambda vs: ctypes.cast((ctypes.c_int64 * G)(*[int(v) for v in vs]), ctypes.c_void_p)
    xa, wa, ya, na, ka = ptrs(xs), ptrs(wqs), ptrs(ys), sizes(Ns), sizes(Ks)
    yt = Y_BF16 if out_dtype == torch.bfloat16 else Y_F32
    _check(lib().q4_0_matmul_grouped(G, xa, wa, ya, yt, M, na, ka, _stream(stream)), "q4_0_matmul_grouped")
    return ys


def grouped_launches(M: int, Ns, Ks) -> int:
    """Kernel launches of a matmul_grouped call with these sizes when the
    grouped decode takes every problem, else -1 (q4_0_matmul_grouped_launches)."""
    G = len(Ns)
    if G == 0 or len(Ks) != G:
        return -1
    na = ctypes.cast((ctypes.c_int64 * G)(*[int(v) for v in Ns]), ctypes.c_void_p)
    ka = ctypes.cast((ctypes.c_int64 * G)(*[int(v) for v in Ks]), ctypes.c_void_p)
    return int(lib().q4_0_matmul_grouped_launches(G, M, na, ka))


def host_workspace_bytes(M: int, N: int, K: int, out_dtype=torch.float32) -> int:
    """Device scratch for matmul_host (q4_0_matmul_host_workspace_bytes)."""
    return int(lib().q4_0_matmul_host_workspace_bytes(M, N, K, Y_BF16 if out_dtype == torch.bfloat16 else Y_F32))


def matmul_alloc(x: torch.Tensor, wq: torch.Tensor, N: int, K: int, out: torch.Tensor = None,
                 stream=None) -> torch.Tensor:
    """Same as matmul, through q4_0_matmul (the library takes its own scratch)."""
    M, out = _mm_args(x, wq, N, K, out)
    _check(lib().q4_0_matmul(x.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K, _stream(stream)),
           "q4_0_matmul")
    return out


def gemv(x: torch.Tensor, wq: torch.Tensor, N: int, K: int, out: torch.Tensor = None,
         workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """The decode kernels alone (M <= 64), through q4_0_gemv_ws."""
    M, out = _mm_args(x, wq, N, K, out)
    ws, wsb = _workspace(int(lib().q4_0_gemv_workspace_bytes(M, K)), x.device, workspace)
    _check(lib().q4_0_gemv_ws(x.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K,
                              ws.data_ptr() if ws is not None else None, wsb, _stream(stream)),
           "q4_0_gemv")
    return out


def gemv_alloc(x: torch.Tensor, wq: torch.Tensor, N: int, K: int, out: torch.Tensor = None,
               stream=None) -> torch.Tensor:
    """Same as gemv, through q4_0_gemv (the library takes its own scratch)."""
    M, out = _mm_args(x, wq, N, K, out)
    _check(lib().q4_0_gemv(x.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K, _stream(stream)),
           "q4_0_gemv")
    return out


def gemm(x: torch.Tensor, wq: torch.Tensor, N: int, K: int, out: torch.Tensor = None,
         workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """The tcgen05 kernel alone (any M)."""
    M, out = _mm_args(x, wq, N, K, out)
    ws, wsb = _workspace(int(lib().q4_0_gemm_workspace_bytes(M, N, K)), x.device, workspace)
    _check(lib().q4_0_gemm(x.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K,
                           ws.data_ptr(), wsb, _stream(stream)), "q4_0_gemm")
    return out



def gemm_plan(M: int, N: int, K: int) -> dict:
    """The launch q4_0_gemm makes for (M, N, K) on the current device:
    {"tile_rows", "splits", "persistent"} (include/q4_0.h, q4_0_gemm_plan)."""
    tr, sp, pe = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().q4_0_gemm_plan(M, N, K, ctypes.byref(tr), ctypes.byref(sp), ctypes.byref(pe)), "q4_0_gemm_plan")
    return {"tile_rows": tr.value, "splits": sp.value, "persistent": bool(pe.value)}

def gemm_noalloc(x: torch.Tensor, wq: torch.Tensor, N: int, K: int, out: torch.Tensor = None,
                 stream=None) -> torch.Tensor:
    """The tcgen05 kernel with the library's fixed scratch array instead of a
    workspace: nothing is allocated on the device by the call (out may be
    given too).  Calls that overlap on the GPU share the array; see
    q4_0_gemm_noalloc in include/q4_0.h."""
    M, out = _mm_args(x, wq, N, K, out)
    _check(lib().q4_0_gemm_noalloc(x.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K,
                                   _stream(stream)), "q4_0_gemm_noalloc")
    return out


def selftest_wait_timeout(limit_us: int = 20000, stream=None) -> int:
    """Run the bounded-wait failure self-check and return the device error
    status it leaves (ERR_DEVICE_TIMEOUT when the path works)."""
    _check(lib().q4_0_selftest_wait_timeout(int(limit_us), _stream(stream)), "q4_0_selftest_wait_timeout")
    return device_error()


def device_error() -> int:
    """Read and clear the device error word (synchronises the device)."""
    code = ctypes.c_int(0)
    _check(lib().q4_0_device_error(ctypes.byref(code)), "q4_0_device_error")
    return code.value
