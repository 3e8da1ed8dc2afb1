"""ctypes binding of the C ABI in include/w4a16.h (argument marshalling only).

Every step of the layer runs in the library's CUDA kernels; this module only turns torch
tensors into device pointers and the current CUDA stream into a stream handle, allocates
outputs when the caller does not pass them, and raises on a non-zero status.  There is no CPU
fallback: if the shared library is missing or fails to load, every call raises.
"""
import contextlib
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_libw4a16.so")
BOUNDS_LIB_PATH = os.path.join(_HERE, "_libw4a16_bounds.so")  # the bounds-checked debug build

OK = 0
ERR_INVALID = -1
ERR_UNSUPPORTED = -2
ERR_MISALIGNED = -3
ERR_WORKSPACE = -4
ERR_CUDA = -5
ERR_DEVICE = -6

OPT_SPLITK_REDUCTION = 1
SPLITK_AUTO = 0
SPLITK_GLOBAL = 1

# name -> (argtypes, restype) of every extern "C" entry point of include/w4a16.h
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "w4a16_packed_bytes": ([_I, _I, _I], _SZ),
    "w4a16_workspace_bytes": ([_I, _I, _I, _I], _SZ),
    "w4a16_repack": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "w4a16_repack_chunk": ([_P, _I64, _P, _I64, _P, _I64, _I, _I, _I, _I, _I, _P, _P], _I),
    "w4a16_gemm": ([_P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "w4a16_dequant": ([_P, _I, _I, _I, _P, _P], _I),
    "w4a16_status_string": ([_I], ctypes.c_char_p),
    "w4a16_last_device_error": ([_P], _I),
    "w4a16_layout_version": ([], _I),
    "w4a16_gemm_noalloc": ([_P, _P, _I, _I, _I, _I, _P, _P], _I),
    "w4a16_set_option": ([_I, _I], _I),
    "w4a16_embed": ([_P, _I, _P, _I, _I, _I, _P, _P], _I),
    "w4a16_awq_to_standard": ([_P, _P, _I, _I, _I, _P, _P, _P], _I),
    "w4a16_selftest_wait_timeout": ([_I64, _P, _P], _I),
    "w4a16_repack_bf16": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "w4a16_repack_chunk_bf16": ([_P, _I64, _P, _I64, _P, _I64, _I, _I, _I, _I, _I, _P, _P], _I),
    "w4a16_gemm_bf16": ([_P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "w4a16_dequant_bf16": ([_P, _I, _I, _I, _P, _P], _I),
    "w4a16_embed_bf16": ([_P, _I, _P, _I, _I, _I, _P, _P], _I),
    "w4a16_bounds_checked": ([], _I),
    "w4a16_selftest_bounds": ([_P, _P], _I),
}

# element type of a layer -> suffix of its entry points
_SUFFIX = {torch.float16: "", torch.bfloat16: "_bf16"}

_libs = {}              # path -> loaded library
_active = [LIB_PATH]    # the library calls go to: the last entry


class W4A16Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %d (%s)" % (fn, status, status_string(status)))


def _load(path):
    L = _libs.get(path)
    if L is None:
        if not os.path.exists(path):
            raise RuntimeError("CUDA library %s is missing: run __graft_entry__.build() first" % path)
        L = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _libs[path] = L
    return L


def lib():
    """The loaded CUDA library (the normal build, or the bounds-checked one inside
    bounds_checked_library()); raises if it has not been built."""
    return _load(_active[-1])


@contextlib.contextmanager
def bounds_checked_library():
    """Within the block, every call of this module goes to the bounds-checked debug build, whose
    kernels check each global access against its buffer's extent (a miss is skipped and makes
    last_device_error() raise).  Its device error word and first-use state are its own."""
    L = _load(BOUNDS_LIB_PATH)
    _active.append(BOUNDS_LIB_PATH)
    try:
        yield L
    finally:
        _active.pop()


def status_string(status):
    return lib().w4a16_status_string(int(status)).decode()


def _check(fn, status):
    if status != OK:
        raise W4A16Error(fn, status)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype, name):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def set_option(option, value):
    """Process-wide option (OPT_SPLITK_REDUCTION: SPLITK_AUTO or SPLITK_GLOBAL)."""
    _check("w4a16_set_option", lib().w4a16_set_option(int(option), int(value)))


def layout_version():
    return lib().w4a16_layout_version()


def packed_bytes(K, N, g):
    return lib().w4a16_packed_bytes(K, N, g)


def workspace_bytes(M, N, K, g):
    return lib().w4a16_workspace_bytes(M, N, K, g)


_HALVES = (torch.float16, torch.bfloat16)


def repack(qweight, qzeros, scales, K, N, g, packed=None, stream=None):
    """AWQ qweight int32 [K, N/8], qzeros int32 [K/g, N/8], scales fp16 or bf16 [K/g, N] ->
    packed uint8 (the scales' type is the layer's element type, recorded in the buffer)."""
    _dev(qweight, torch.int32, "qweight")
    _dev(qzeros, torch.int32, "qzeros")
    _dev(scales, _HALVES, "scales")
    nbytes = packed_bytes(K, N, g)
    if nbytes == 0:
        _check("w4a16_packed_bytes", ERR_UNSUPPORTED)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=qweight.device)
    fn = "w4a16_repack" + _SUFFIX[scales.dtype]
    _check(fn, getattr(lib(), fn)(_ptr(qweight), _ptr(qzeros), _ptr(scales), K, N, g, _ptr(packed),
                                  _stream(stream)))
    return packed


def repack_chunk(qweight_c, qzeros_c, scales_c, K, N, g, n0, n1, packed, stream=None):
    """Repack columns [n0, n1) given the column slices (2-D tensors, unit inner stride)."""
    for t, name in ((qweight_c, "qweight"), (qzeros_c, "qzeros"), (scales_c, "scales")):
        if not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("%s slice must be a 2-D CUDA tensor with unit column stride" % name)
    if scales_c.dtype not in _HALVES:
        raise ValueError("scales must be float16 or bfloat16")
    fn = "w4a16_repack_chunk" + _SUFFIX[scales_c.dtype]
    _check(fn, getattr(lib(), fn)(
        _ptr(qweight_c), qweight_c.stride(0), _ptr(qzeros_c), qzeros_c.stride(0),
        _ptr(scales_c), scales_c.stride(0), K, N, g, n0, n1, _ptr(packed), _stream(stream)))
    return packed


_workspaces = {}
_workspaces_lock = threading.Lock()


def default_workspace(nbytes, device, stream=None):
    """A zero-filled workspace of at least `nbytes` bytes, cached per device and stream.  Every
    completed call leaves it zero-filled, so calls on one stream reuse it; calls on different
    streams get different workspaces, so they may overlap.  (Calls that share a stream run one
    after the other: a call touches the workspace only after the previous kernel in the stream
    has finished.)"""
    index = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    if stream is None:
        stream = torch.cuda.current_stream(index)
    key = (index, stream.cuda_stream)
    with _workspaces_lock:
        ws = _workspaces.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
            _workspaces[key] = ws
    return ws


def gemm(x, packed, M, N, K, g, y=None, workspace=None, stream=None):
    """y [M, N] = x [M, K] . W(packed), in the layer's element type (x fp16 or bf16)."""
    _dev(x, _HALVES, "x")
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    _dev(y, x.dtype, "y")
    need = workspace_bytes(M, N, K, g)
    if need and workspace is None:
        workspace = default_workspace(need, x.device, stream)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    fn = "w4a16_gemm" + _SUFFIX[x.dtype]
    _check(fn, getattr(lib(), fn)(_ptr(x), _ptr(packed), M, N, K, g, _ptr(y), ws_ptr, ws_len, _stream(stream)))
    return y


def gemm_noalloc(x, packed, M, N, K, g, y, stream=None):
    """y = x . W without any workspace: for callers that cannot allocate device memory (the
    library's built-in scratch array serves instead; overlapping calls race on it)."""
    _dev(x, torch.float16, "x")
    _dev(y, torch.float16, "y")
    _check("w4a16_gemm_noalloc", lib().w4a16_gemm_noalloc(_ptr(x), _ptr(packed), M, N, K, g, _ptr(y),
                                                          _stream(stream)))
    return y


def dequant(packed, K, N, g, out=None, stream=None, dtype=torch.float16):
    """W [K, N] from the packed buffer (bit-exact), in the layer's element type (out's dtype
    when out is given, else `dtype`)."""
    if out is None:
        out = torch.empty((K, N), dtype=dtype, device=packed.device)
    _dev(out, _HALVES, "out")
    fn = "w4a16_dequant" + _SUFFIX[out.dtype]
    _check(fn, getattr(lib(), fn)(_ptr(packed), K, N, g, _ptr(out), _stream(stream)))
    return out


def embed(ids, packed, K, N, g, out=None, stream=None, dtype=torch.float16):
    """Rows of the quantized tied embedding: [T, K], row t = column ids[t] of W, in the layer's
    element type (out's dtype when out is given, else `dtype`)."""
    _dev(ids, torch.int32, "ids")
    T = ids.numel()
    if out is None:
        out = torch.empty((T, K), dtype=dtype, device=ids.device)
    _dev(out, _HALVES, "out")
    fn = "w4a16_embed" + _SUFFIX[out.dtype]
    _check(fn, getattr(lib(), fn)(_ptr(ids), T, _ptr(packed), K, N, g, _ptr(out), _stream(stream)))
    return out


def awq_to_standard(qweight, qzeros, K, N, g, stream=None):
    """AWQ int32 tensors -> (qweight_std int32 [K/8, N], qzeros_std int32 [K/g, N/8])."""
    _dev(qweight, torch.int32, "qweight")
    _dev(qzeros, torch.int32, "qzeros")
    qs = torch.empty((K // 8, N), dtype=torch.int32, device=qweight.device)
    zs = torch.empty_like(qzeros)
    _check("w4a16_awq_to_standard", lib().w4a16_awq_to_standard(_ptr(qweight), _ptr(qzeros), K, N, g, _ptr(qs),
                                                                 _ptr(zs), _stream(stream)))
    return qs, zs


def selftest_wait_timeout(limit_ns=1_000_000, stream=None):
    """Forced timeout of the library's bounded waits (see include/w4a16.h): returns the bitmask of
    waits that gave up (3 when both did); the device error word then reports W4A16_ERR_DEVICE."""
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check("w4a16_selftest_wait_timeout", lib().w4a16_selftest_wait_timeout(int(limit_ns), _ptr(status),
                                                                           _stream(stream)))
    return int(status.item())


def selftest_bounds(stream=None):
    """The bounds check on five fixed cases (see include/w4a16.h): returns the bitmask of cases
    judged outside their buffer (0x1C in the bounds-checked build, 0 in the normal one)."""
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check("w4a16_selftest_bounds", lib().w4a16_selftest_bounds(_ptr(status), _stream(stream)))
    return int(status.item())


def bounds_checked():
    """True when calls go to the bounds-checked debug build."""
    return bool(lib().w4a16_bounds_checked())


def last_device_error(stream=None):
    """Synchronize the stream and return (and clear) the device-side error status."""
    return lib().w4a16_last_device_error(_stream(stream))
