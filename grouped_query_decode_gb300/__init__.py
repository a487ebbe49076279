"""GB300 (sm_103a) grouped-query decode attention.

A thin ctypes binding over the C ABI of libgqa_decode.so (include/gqa_decode.h):
the functions here only check and marshal arguments -- every step of the
computation runs in the library's CUDA kernels. There is no CPU fallback: if
the library cannot be built or loaded, every call raises.

    out, lse = torch.empty(...), torch.empty(...)
    gqa_decode(q, k_cache, v_cache, seq_lens, scale, out, lse)

q [B, sq, H, D], k_cache / v_cache [B, G, Tmax, D] and out are bfloat16 CUDA
tensors; seq_lens [B] is int32 on the same device; lse [B, sq, H] float32 or
None. Calls are enqueued on the current torch CUDA stream (or `stream`).
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

GQA_OK = 0
GQA_ERR_INVALID_ARG = -1
GQA_ERR_HEAD_RATIO = -2
GQA_ERR_UNSUPPORTED = -3
GQA_ERR_MISALIGNED = -4
GQA_ERR_WORKSPACE = -5
GQA_ERR_CUDA = -6
GQA_ERR_DEVICE_TIMEOUT = -7

LIB_PATH = _build.LIB_PATH
_lib = None
_lock = threading.Lock()


class GQADecodeError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = strerror(status) if _lib is not None else str(status)
        if status == GQA_ERR_CUDA and _lib is not None:
            msg += f" (cudaError {gqa_decode_last_cuda_error()})"
        super().__init__(f"{what}: {msg}" if what else msg)


class PlanT(ctypes.Structure):
    _fields_ = [("ctas", ctypes.c_int), ("tile_tokens", ctypes.c_int),
                ("row_tiles", ctypes.c_int), ("stages", ctypes.c_int),
                ("threads", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("max_tiles", ctypes.c_longlong)]


def load():
    """Builds (if the sources are newer) and loads libgqa_decode.so."""
    global _lib
    if _lib is not None:           # every call after the first: no lock
        return _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path)
            vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            shape = [i32] * 6
            lib.gqa_decode.argtypes = [vp, vp, vp, vp, f32, vp, vp, *shape, vp]
            lib.gqa_decode.restype = i32
            lib.gqa_decode_ex.argtypes = [vp, vp, vp, vp, f32, vp, vp, *shape, vp, sz, vp]
            lib.gqa_decode_ex.restype = i32
            lib.gqa_decode_append.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp, *shape, vp]
            lib.gqa_decode_append.restype = i32
            lib.gqa_decode_paged.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, *([i32] * 8), vp]
            lib.gqa_decode_paged.restype = i32
            lib.gqa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp, *shape, vp]
            lib.gqa_decode_fp8.restype = i32
            lib.gqa_prefill.argtypes = [vp, vp, vp, vp, f32, vp, vp, *shape, vp]
            lib.gqa_prefill.restype = i32
            lib.gqa_decode_noalloc.argtypes = [vp, vp, vp, vp, f32, vp, vp, *shape, vp]
            lib.gqa_decode_noalloc.restype = i32
            lib.gqa_decode_workspace_bytes.argtypes = shape
            lib.gqa_decode_workspace_bytes.restype = sz
            lib.gqa_decode_plan.argtypes = [*shape, i32, ctypes.POINTER(PlanT)]
            lib.gqa_decode_plan.restype = i32
            lib.gqa_decode_check_error.argtypes = [vp]
            lib.gqa_decode_check_error.restype = i32
            lib.gqa_decode_release_workspace.argtypes = [vp]
            lib.gqa_decode_release_workspace.restype = i32
            lib.gqa_decode_last_cuda_error.argtypes = []
            lib.gqa_decode_last_cuda_error.restype = i32
            lib.gqa_decode_strerror.argtypes = [i32]
            lib.gqa_decode_strerror.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def strerror(status: int) -> str:
    return load().gqa_decode_strerror(int(status)).decode()


def gqa_decode_strerror(status: int) -> str:
    return strerror(status)


def gqa_decode_last_cuda_error() -> int:
    return int(load().gqa_decode_last_cuda_error())


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif hasattr(stream, "device_index") and stream.device_index != device:
        raise ValueError(f"stream is on cuda:{stream.device_index}, the tensors on cuda:{device}")
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _call(device, fn, *args):
    """Calls the library with `device` current (it launches on the current
    device); switches only when another device is current."""
    import torch
    if torch.cuda.current_device() == device:
        return fn(*args)
    with torch.cuda.device(device):
        return fn(*args)


def _check(dev, name, t, dt):
    """dtype, device (the CUDA device `dev`) and contiguity of one tensor; the
    device index doubles as the CUDA check (-1 for host tensors)."""
    if t.dtype != dt:
        raise TypeError(f"{name} must be {dt}, got {t.dtype}")
    d = t.get_device()
    if d < 0:
        raise TypeError(f"{name} must be a CUDA tensor")
    if d != dev:
        raise ValueError(f"{name} is on cuda:{d}, q on cuda:{dev}: all tensors must be on one device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_lse(dev, lse, B, sq, H):
    """lse is optional; when given it is float32 [B, sq, H] on q's device."""
    import torch
    if lse is None:
        return
    _check(dev, "lse", lse, torch.float32)
    if tuple(lse.shape) != (B, sq, H):
        raise ValueError("lse must be [B, sq, H]")


def _shapes(q, k_cache, v_cache, seq_lens, out, lse):
    """Checks the tensors of the contiguous-cache entry points (dtype, one
    CUDA device, contiguity, shapes); returns B, sq, H, G, D, Tmax and the
    device index."""
    import torch
    bf = torch.bfloat16
    dev = q.get_device()
    _check(dev, "q", q, bf)
    _check(dev, "k_cache", k_cache, bf)
    _check(dev, "v_cache", v_cache, bf)
    _check(dev, "seq_lens", seq_lens, torch.int32)
    _check(dev, "out", out, bf)
    if q.dim() != 4 or k_cache.dim() != 4:
        raise ValueError("q is [B, sq, H, D] and k_cache [B, G, Tmax, D]")
    B, sq, H, D = q.shape
    Bk, G, Tmax, Dk = k_cache.shape
    if (Bk, Dk) != (B, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache must be [B, G, Tmax, D] with q's B and D")
    if tuple(seq_lens.shape) != (B,) or tuple(out.shape) != (B, sq, H, D):
        raise ValueError("seq_lens must be [B] and out [B, sq, H, D]")
    _check_lse(dev, lse, B, sq, H)
    return B, sq, H, G, D, Tmax, dev


def gqa_decode(q, k_cache, v_cache, seq_lens, scale, out, lse=None, stream=None):
    """One decode step (library-owned workspace). See include/gqa_decode.h."""
    B, sq, H, G, D, Tmax, dev = _shapes(q, k_cache, v_cache, seq_lens, out, lse)
    rc = _call(dev, load().gqa_decode, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
               seq_lens.data_ptr(), float(scale), out.data_ptr(),
               None if lse is None else lse.data_ptr(), B, sq, H, G, D, Tmax,
               _stream_handle(stream, dev))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode")


def gqa_prefill(q, k_cache, v_cache, seq_lens, scale, out, lse=None, stream=None):
    """Prefill or chunked prefill: the same attention as gqa_decode for any
    number of new tokens sq (no limit on (H/G)*sq), on the tcgen05 kernel.
    The sq new tokens' K/V must already be in the cache; seq_lens counts them."""
    B, sq, H, G, D, Tmax, dev = _shapes(q, k_cache, v_cache, seq_lens, out, lse)
    rc = _call(dev, load().gqa_prefill, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
               seq_lens.data_ptr(), float(scale), out.data_ptr(),
               None if lse is None else lse.data_ptr(), B, sq, H, G, D, Tmax,
               _stream_handle(stream, dev))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_prefill")


def gqa_decode_append(q, k_new, v_new, k_cache, v_cache, seq_lens, scale, out, lse=None,
                      stream=None):
    """One decode step that first appends the sq new tokens' K/V ([B, sq, G, D]
    bf16) to the caches at positions seq_lens[b] - sq + s, in the same launch."""
    B, sq, H, G, D, Tmax, dev = _shapes(q, k_cache, v_cache, seq_lens, out, lse)
    import torch
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _check(dev, name, t, torch.bfloat16)
        if tuple(t.shape) != (B, sq, G, D):
            raise ValueError(f"{name} must be [B, sq, G, D]")
    rc = _call(dev, load().gqa_decode_append, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
               k_cache.data_ptr(), v_cache.data_ptr(), seq_lens.data_ptr(),
               float(scale), out.data_ptr(),
               None if lse is None else lse.data_ptr(), B, sq, H, G, D, Tmax,
               _stream_handle(stream, dev))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode_append")


def gqa_decode_paged(q, k_pages, v_pages, block_table, seq_lens, scale, out, lse=None,
                     stream=None):
    """One decode step over a paged cache: k_pages/v_pages [num_pages, G,
    page_size, D] bf16, block_table [B, max_pages_per_seq] int32."""
    import torch
    dev = q.get_device()
    for name, t, dt in (("q", q, torch.bfloat16), ("k_pages", k_pages, torch.bfloat16),
                        ("v_pages", v_pages, torch.bfloat16), ("block_table", block_table, torch.int32),
                        ("seq_lens", seq_lens, torch.int32), ("out", out, torch.bfloat16)):
        _check(dev, name, t, dt)
    B, sq, H, D = q.shape
    num_pages, G, page_size, Dk = k_pages.shape
    if Dk != D or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("k_pages / v_pages must be [num_pages, G, page_size, D]")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages_per_seq]")
    if tuple(seq_lens.shape) != (B,) or tuple(out.shape) != (B, sq, H, D):
        raise ValueError("seq_lens must be [B] and out [B, sq, H, D]")
    _check_lse(dev, lse, B, sq, H)
    rc = _call(dev, load().gqa_decode_paged, q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
               block_table.data_ptr(), seq_lens.data_ptr(), float(scale),
               out.data_ptr(), None if lse is None else lse.data_ptr(),
               B, sq, H, G, D, page_size, num_pages, block_table.shape[1],
               _stream_handle(stream, dev))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode_paged")


def gqa_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, seq_lens, scale, out, lse=None,
                   stream=None):
    """One decode step over an fp8 cache: k_codes/v_codes [B, G, Tmax, 128]
    uint8 e4m3 codes, k_scale/v_scale [B, G, ceil(Tmax/64)] float32 (one scale
    per 64-token block)."""
    import torch
    dev = q.get_device()
    for name, t, dt in (("q", q, torch.bfloat16), ("k_codes", k_codes, torch.uint8),
                        ("v_codes", v_codes, torch.uint8), ("k_scale", k_scale, torch.float32),
                        ("v_scale", v_scale, torch.float32), ("seq_lens", seq_lens, torch.int32),
                        ("out", out, torch.bfloat16)):
        _check(dev, name, t, dt)
    B, sq, H, D = q.shape
    Bk, G, Tmax, Dk = k_codes.shape
    if (Bk, Dk) != (B, D) or tuple(v_codes.shape) != tuple(k_codes.shape):
        raise ValueError("k_codes / v_codes must be [B, G, Tmax, D]")
    nt = (Tmax + 63) // 64
    if tuple(k_scale.shape) != (B, G, nt) or tuple(v_scale.shape) != (B, G, nt):
        raise ValueError("k_scale / v_scale must be [B, G, ceil(Tmax/64)]")
    if tuple(seq_lens.shape) != (B,) or tuple(out.shape) != (B, sq, H, D):
        raise ValueError("seq_lens must be [B] and out [B, sq, H, D]")
    _check_lse(dev, lse, B, sq, H)
    rc = _call(dev, load().gqa_decode_fp8, q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(),
               k_scale.data_ptr(), v_scale.data_ptr(), seq_lens.data_ptr(),
               float(scale), out.data_ptr(), None if lse is None else lse.data_ptr(),
               B, sq, H, G, D, Tmax, _stream_handle(stream, dev))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode_fp8")


def gqa_decode_ex(q, k_cache, v_cache, seq_lens, scale, out, lse, workspace, stream=None):
    """One decode step with a caller-owned workspace (a CUDA uint8 tensor of at
    least gqa_decode_workspace_bytes(...) bytes)."""
    B, sq, H, G, D, Tmax, dev = _shapes(q, k_cache, v_cache, seq_lens, out, lse)
    import torch
    _check(dev, "workspace", workspace, torch.uint8)
    rc = _call(dev, load().gqa_decode_ex, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
               seq_lens.data_ptr(), float(scale), out.data_ptr(),
               None if lse is None else lse.data_ptr(), B, sq, H, G, D, Tmax,
               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
               _stream_handle(stream, dev))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode_ex")


# Size of the fixed per-device scratch array gqa_decode_noalloc draws from.
GQA_NOALLOC_SCRATCH_BYTES = 8 << 20


def gqa_decode_noalloc(q, k_cache, v_cache, seq_lens, scale, out, lse=None, stream=None):
    """One decode step that allocates no device memory: the scratch comes from
    a fixed 8 MiB array the library keeps on each GPU. For callers that may not
    allocate once running (a pre-reserved memory pool, a framework plugin with
    no allocator, a loop that cannot take cudaMalloc's synchronisation). Calls
    on one device share that array, so calls that overlap on the GPU race."""
    B, sq, H, G, D, Tmax, dev = _shapes(q, k_cache, v_cache, seq_lens, out, lse)
    rc = _call(dev, load().gqa_decode_noalloc, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
               seq_lens.data_ptr(), float(scale), out.data_ptr(),
               None if lse is None else lse.data_ptr(), B, sq, H, G, D, Tmax,
               _stream_handle(stream, dev))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode_noalloc")


def gqa_decode_release_workspace(stream=None, device=None) -> None:
    """Frees the library-owned workspace of (device, stream) after the work
    queued on the stream; the next call on that stream allocates again."""
    import torch
    if device is None:
        device = stream.device_index if hasattr(stream, "device_index") else torch.cuda.current_device()
    rc = _call(device, load().gqa_decode_release_workspace, _stream_handle(stream, device))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode_release_workspace")


def gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax) -> int:
    return int(load().gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax))


def gqa_decode_plan(B, sq, H, G, D, Tmax, num_sms) -> dict:
    plan = PlanT()
    rc = load().gqa_decode_plan(B, sq, H, G, D, Tmax, num_sms, ctypes.byref(plan))
    if rc != GQA_OK:
        raise GQADecodeError(rc, "gqa_decode_plan")
    return {f: getattr(plan, f) for f, _ in PlanT._fields_}


def gqa_decode_check_error(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the device status."""
    import torch
    if device is None:
        device = stream.device_index if hasattr(stream, "device_index") else torch.cuda.current_device()
    dev = device if isinstance(device, int) else torch.device(device).index
    return int(_call(dev, load().gqa_decode_check_error, _stream_handle(stream, dev)))
