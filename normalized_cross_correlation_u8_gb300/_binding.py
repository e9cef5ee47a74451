"""ctypes binding of libcorr.so (include/corr.h, include/corr_peaks.h).

Argument marshalling only: tensors are checked for dtype, shape and device,
their device pointers and the current torch stream are handed to the C ABI,
and every step of the computation runs in the library's CUDA kernels.  There
is no CPU fallback: if the library cannot be loaded, or no GPU is present,
these functions raise.

Host (CPU) tensors are accepted for convenience: they are copied to the
device (asynchronously when pinned), processed there, and the results copied
back, all on the current stream.
"""
import ctypes
import os
import threading

import torch

from . import build as _build

CORR_OK = 0
CORR_EINVAL = -1
CORR_EUNSUPPORTED = -2
CORR_ECUDA = -3
CORR_ETIMEOUT = -4
NCC_MAX_TEMPLATE_PIXELS = 66051
NCC_METHOD_DP4A = 0
NCC_METHOD_BOX = 1
_NCC_METHODS = {"dp4a": NCC_METHOD_DP4A, "box": NCC_METHOD_BOX}

EXPORTS = ["corr_ncc_u8", "corr_ncc_u8_pitched", "corr_ncc_set_method", "corr_ncc_get_method", "corr_xcorr_f32", "corr_xcorr_f32_noalloc", "corr_xcorr_f32_kernel", "corr_device_status", "corr_scratch_reserved", "corr_set_stream",
           "corr_get_stream", "corr_strerror", "corr_last_cuda_error",
           "corr_version", "corr_peak_dp4a", "corr_peak_ffma"]

_lib = None
_lock = threading.Lock()


class CorrError(RuntimeError):
    def __init__(self, code, message, cuda_error=0):
        super().__init__(f"{message} (code {code}"
                         + (f", cudaError {cuda_error})" if cuda_error else ")"))
        self.code = code
        self.cuda_error = cuda_error


def library_path():
    return _build.LIB


def load(build_if_missing=True):
    """Load libcorr.so (building it first when it is missing or stale and
    nvcc is available).  Raises if it cannot be loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing:
            try:
                path = _build.build()
            except RuntimeError:
                if not os.path.exists(path):
                    raise
        if not os.path.exists(path):
            raise ImportError(f"libcorr.so not built ({path}); run "
                              "python -m normalized_cross_correlation_u8_gb300.build")
        lib = ctypes.CDLL(path)
        c_int, vp, c_dbl_p = ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_double)
        lib.corr_ncc_u8.argtypes = [vp, c_int, c_int, vp, c_int, c_int, vp, vp]
        lib.corr_ncc_u8_pitched.argtypes = [vp, c_int, c_int, ctypes.c_size_t, vp, c_int,
                                            c_int, vp, vp]
        lib.corr_ncc_set_method.argtypes = [c_int]
        lib.corr_ncc_get_method.argtypes = []
        lib.corr_xcorr_f32.argtypes = [vp, c_int, vp, c_int, c_int, c_int, vp]
        lib.corr_xcorr_f32_noalloc.argtypes = [vp, c_int, vp, c_int, c_int, c_int, vp]
        lib.corr_scratch_reserved.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
        lib.corr_device_status.argtypes = []
        lib.corr_xcorr_f32_kernel.argtypes = [c_int, c_int, c_int, c_int,
                                              ctypes.POINTER(c_int)]
        lib.corr_set_stream.argtypes = [vp]
        lib.corr_get_stream.argtypes = []
        lib.corr_get_stream.restype = vp
        lib.corr_strerror.argtypes = [c_int]
        lib.corr_strerror.restype = ctypes.c_char_p
        lib.corr_last_cuda_error.argtypes = []
        lib.corr_version.argtypes = []
        lib.corr_peak_dp4a.argtypes = [c_int, c_dbl_p, c_dbl_p]
        lib.corr_peak_ffma.argtypes = [c_dbl_p, c_dbl_p]
        for f in (lib.corr_ncc_u8, lib.corr_ncc_u8_pitched, lib.corr_ncc_set_method,
                  lib.corr_ncc_get_method,
                  lib.corr_xcorr_f32, lib.corr_xcorr_f32_noalloc, lib.corr_scratch_reserved, lib.corr_device_status, lib.corr_xcorr_f32_kernel,
                  lib.corr_set_stream,
                  lib.corr_last_cuda_error, lib.corr_version,
                  lib.corr_peak_dp4a, lib.corr_peak_ffma):
            f.restype = c_int
        _lib = lib
        return lib


def _check(rc):
    if rc != CORR_OK:
        lib = load()
        cuda = lib.corr_last_cuda_error() if rc == CORR_ECUDA else 0
        raise CorrError(rc, lib.corr_strerror(rc).decode(), cuda)


def _bind_stream(device):
    lib = load()
    lib.corr_set_stream(torch.cuda.current_stream(device).cuda_stream)
    return lib


class _Nothing:
    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


_NOTHING = _Nothing()


def _on_device(dev):
    """torch.cuda.device(dev) unless dev is already current (the common
    case, where switching costs two runtime calls for nothing)."""
    if dev.index is None or dev.index == torch.cuda.current_device():
        return _NOTHING
    return torch.cuda.device(dev)


def _require_cuda():
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: the correlation kernels only run on the GPU")


def _u32_empty(shape, device):
    """uint32 output storage (int32 storage where torch lacks uint32)."""
    dt = getattr(torch, "uint32", None)
    try:
        return torch.empty(shape, dtype=dt, device=device)
    except (TypeError, RuntimeError):
        return torch.empty(shape, dtype=torch.int32, device=device)


def ncc_set_method(method):
    """Select how this thread's ncc_u8 calls form SumI / SumISq on the fast
    kernel: "dp4a" (three dp4a per 4 pixels) or "box" (box filters of the
    staged tile, then one dp4a per 4 pixels for SumIT; the default).
    Results are bit-identical."""
    if method not in _NCC_METHODS:
        raise ValueError(f"method must be one of {sorted(_NCC_METHODS)}")
    _check(load().corr_ncc_set_method(_NCC_METHODS[method]))


def ncc_get_method():
    """This thread's ncc_u8 method name ("dp4a" or "box")."""
    code = load().corr_ncc_get_method()
    return {v: k for k, v in _NCC_METHODS.items()}[code]


def ncc_u8_into(image, tmpl, sums_out, coef_out, method=None):
    """Device call: image [h,w] uint8 (rows may be strided, e.g. a crop of a
    larger image: passed as the row pitch), tmpl [ht,wt] uint8, sums_out
    [3,oh,ow] 32-bit (or None), coef_out [oh,ow] float32 (or None), all on
    the same CUDA device, outputs contiguous.  Runs on the current stream.
    `method` ("dp4a" / "box") overrides this thread's method for the call."""
    if image.dtype != torch.uint8 or tmpl.dtype != torch.uint8:
        raise TypeError("image and template must be uint8")
    if image.dim() != 2 or tmpl.dim() != 2:
        raise ValueError("image and template must be 2-D")
    dev = image.device
    if not image.is_cuda or tmpl.device != dev:
        raise ValueError("image and template must be on the same CUDA device")
    h, w = image.shape
    ht, wt = tmpl.shape
    oh, ow = h - ht + 1, w - wt + 1
    for t, shape in ((sums_out, (3, oh, ow)), (coef_out, (oh, ow))):
        if t is not None:
            if t.device != dev or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError(f"output must be a contiguous {shape} tensor on {dev}")
            if t.element_size() != 4:
                raise TypeError("outputs are 32-bit")
    if coef_out is not None and coef_out.dtype != torch.float32:
        raise TypeError("coef_out must be float32")
    if image.stride(1) != 1 or image.stride(0) < w:
        image = image.contiguous()
    pitch = image.stride(0)
    tmpl = tmpl.contiguous()
    if method is not None and method not in _NCC_METHODS:
        raise ValueError(f"method must be one of {sorted(_NCC_METHODS)}")
    args = (image.data_ptr(), w, h, pitch, tmpl.data_ptr(), wt, ht,
            sums_out.data_ptr() if sums_out is not None else None,
            coef_out.data_ptr() if coef_out is not None else None)
    with _on_device(dev):
        lib = _bind_stream(dev)
        if method is None:
            _check(lib.corr_ncc_u8_pitched(*args))
        else:
            prev = lib.corr_ncc_get_method()
            _check(lib.corr_ncc_set_method(_NCC_METHODS[method]))
            try:
                _check(lib.corr_ncc_u8_pitched(*args))
            finally:
                lib.corr_ncc_set_method(prev)
    return sums_out, coef_out


def ncc_u8(image, tmpl, sums=True, coef=True, device=None, method=None):
    """Normalized cross-correlation of a uint8 image with a uint8 template.

    Returns (sums [3, oh, ow] uint32 planes SumI/SumISq/SumIT or None,
    coef [oh, ow] float32 or None).  CUDA inputs stay on their device; CPU
    inputs are copied to `device` (default: the current CUDA device), computed
    there and the results copied back to the host."""
    _require_cuda()
    host = not image.is_cuda
    if host:
        dev = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        image = image.to(dev, non_blocking=True)
        tmpl = tmpl.to(dev, non_blocking=True)
    dev = image.device
    h, w = image.shape
    ht, wt = tmpl.shape
    oh, ow = h - ht + 1, w - wt + 1
    if oh <= 0 or ow <= 0:
        raise CorrError(CORR_EINVAL, "template larger than image")
    s = _u32_empty((3, oh, ow), dev) if sums else None
    c = torch.empty((oh, ow), dtype=torch.float32, device=dev) if coef else None
    ncc_u8_into(image, tmpl, s, c, method=method)
    if host:
        s = s.cpu() if s is not None else None
        c = c.cpu() if c is not None else None
    return s, c


def xcorr_f32_into(left, right, out):
    """Device call: left [nl,H,W], right [nr,H,W] float32, out
    [nl,nr,2H-1,2W-1] float32, same CUDA device, contiguous."""
    for t in (left, right, out):
        if t.dtype != torch.float32:
            raise TypeError("xcorr operates on float32")
    if left.dim() != 3 or right.dim() != 3 or left.shape[1:] != right.shape[1:]:
        raise ValueError("left [nl,H,W] and right [nr,H,W] must share H, W")
    dev = left.device
    if not left.is_cuda or right.device != dev or out.device != dev:
        raise ValueError("all tensors must be on the same CUDA device")
    nl, H, W = left.shape
    nr = right.shape[0]
    if tuple(out.shape) != (nl, nr, 2 * H - 1, 2 * W - 1) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [nl, nr, 2H-1, 2W-1] tensor")
    left, right = left.contiguous(), right.contiguous()
    with _on_device(dev):
        lib = _bind_stream(dev)
        _check(lib.corr_xcorr_f32(left.data_ptr(), nl, right.data_ptr(), nr, H, W,
                                  out.data_ptr()))
    return out


def xcorr_f32_noalloc_into(left, right, out):
    """As xcorr_f32_into, through corr_xcorr_f32_noalloc: the library allocates
    no device memory (its scratch is a fixed 16 MiB array shared by all calls,
    so calls that overlap on the GPU must be ordered by the caller).  Raises
    CorrError (unsupported size) for shapes that need more scratch."""
    for t in (left, right, out):
        if t.dtype != torch.float32:
            raise TypeError("xcorr operates on float32")
    if left.dim() != 3 or right.dim() != 3 or left.shape[1:] != right.shape[1:]:
        raise ValueError("left [nl,H,W] and right [nr,H,W] must share H, W")
    dev = left.device
    if not left.is_cuda or right.device != dev or out.device != dev:
        raise ValueError("all tensors must be on the same CUDA device")
    nl, H, W = left.shape
    nr = right.shape[0]
    if tuple(out.shape) != (nl, nr, 2 * H - 1, 2 * W - 1) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [nl, nr, 2H-1, 2W-1] tensor")
    left, right = left.contiguous(), right.contiguous()
    with _on_device(dev):
        lib = _bind_stream(dev)
        _check(lib.corr_xcorr_f32_noalloc(left.data_ptr(), nl, right.data_ptr(), nr, H, W,
                                          out.data_ptr()))
    return out


def xcorr_f32(left, right, device=None):
    """Full 2D cross-correlation of every (left, right) pair.

    left [nl, H, W] (or [H, W]), right [nr, H, W] (or [H, W]) float32.
    Returns [nl, nr, 2H-1, 2W-1] float32; element [li, ri, dy+H-1, dx+W-1] is
    sum_{y,x} left[li, y, x] * right[ri, y-dy, x-dx]."""
    _require_cuda()
    if left.dim() == 2:
        left = left.unsqueeze(0)
    if right.dim() == 2:
        right = right.unsqueeze(0)
    host = not left.is_cuda
    if host:
        dev = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        left = left.to(dev, non_blocking=True)
        right = right.to(dev, non_blocking=True)
    nl, H, W = left.shape
    nr = right.shape[0]
    out = torch.empty((nl, nr, 2 * H - 1, 2 * W - 1), dtype=torch.float32,
                      device=left.device)
    xcorr_f32_into(left, right, out)
    return out.cpu() if host else out


XCORR_KERNELS = {0: "rows", 1: "rows_win", 2: "bcast", 3: "tiny", 4: "tensor", 5: "warp",
                 6: "tensor_large"}


def xcorr_f32_kernel(nl, nr, H, W):
    """Name of the kernel corr_xcorr_f32 runs for nl x nr pairs of H x W
    matrices ("rows", "rows_win", "bcast", "tiny", "tensor" or "warp")."""
    kind = ctypes.c_int()
    _check(load().corr_xcorr_f32_kernel(nl, nr, H, W, ctypes.byref(kind)))
    return XCORR_KERNELS[kind.value]


def device_status():
    """Synchronise the current stream and raise CorrError (CORR_ETIMEOUT)
    if a library kernel gave up a bounded wait since the last check."""
    _require_cuda()
    lib = _bind_stream(torch.device("cuda", torch.cuda.current_device()))
    _check(lib.corr_device_status())


def scratch_reserved(device=None):
    """Bytes of device memory the library's scratch pool holds on the
    device right now (0 once the calls that used scratch have been
    synchronised)."""
    _require_cuda()
    dev = torch.device(device) if device is not None else torch.device(
        "cuda", torch.cuda.current_device())
    n = ctypes.c_size_t()
    with torch.cuda.device(dev):
        _check(load().corr_scratch_reserved(ctypes.byref(n)))
    return n.value


def peak_dp4a(shf_per_8=0, device=None):
    """Measured unsigned dp4a/s on the device (saturating probe kernel)."""
    _require_cuda()
    dev = torch.device(device) if device is not None else torch.device(
        "cuda", torch.cuda.current_device())
    rate, secs = ctypes.c_double(), ctypes.c_double()
    with torch.cuda.device(dev):
        lib = _bind_stream(dev)
        _check(lib.corr_peak_dp4a(int(shf_per_8), ctypes.byref(rate), ctypes.byref(secs)))
    return rate.value, secs.value


def peak_ffma(device=None):
    """Measured FP32 FMA/s on the device (saturating probe kernel)."""
    _require_cuda()
    dev = torch.device(device) if device is not None else torch.device(
        "cuda", torch.cuda.current_device())
    rate, secs = ctypes.c_double(), ctypes.c_double()
    with torch.cuda.device(dev):
        lib = _bind_stream(dev)
        _check(lib.corr_peak_ffma(ctypes.byref(rate), ctypes.byref(secs)))
    return rate.value, secs.value
