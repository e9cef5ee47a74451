"""GB300 (sm_103a) sliding-window 2D correlation.

Two operations, both computed by hand-written CUDA kernels in libcorr.so and
reached through its C ABI (include/corr.h):

* ncc_u8    -- 8-bit normalized cross-correlation (template matching): exact
               SumI / SumISq / SumIT per valid offset plus the coefficient
               (The CUDA Handbook ch. 15, section 15.5).
* xcorr_f32 -- float32 full 2D cross-correlation of every left/right pair
               over all overlaps ("Efficient GPU-accelerated Parallel
               Cross-correlation" artifact README).

The library is loaded (and built if needed) on first use, not at import.
"""
from ._binding import (CorrError, device_status, load, ncc_get_method, ncc_set_method,  # noqa: F401
                       ncc_u8, ncc_u8_into, peak_dp4a, peak_ffma, scratch_reserved, xcorr_f32,
                       xcorr_f32_into, xcorr_f32_kernel, xcorr_f32_noalloc_into)

__all__ = ["CorrError", "device_status", "load", "ncc_u8", "ncc_u8_into", "ncc_set_method", "ncc_get_method", "xcorr_f32",
           "xcorr_f32_into", "xcorr_f32_kernel", "xcorr_f32_noalloc_into", "scratch_reserved", "peak_dp4a",
           "peak_ffma"]
