"""CPU oracle for the correlation path.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package.  The product library (normalized_cross_correlation_
u8_gb300) never imports it and shares no code with it.
"""
from .oracle import (ncc_u8, ncc_u8_at, template_sums, xcorr_f32,  # noqa: F401
                     xcorr_f32_at, load)
