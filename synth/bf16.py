"""bfloat16 storage helpers (storage format only, no head arithmetic).

bfloat16 values are held as ``uint16`` bit patterns so that numpy, torch and the C
library all see the same bytes.
"""
import numpy as np


def f32_to_bf16(x):
    """Round float32 to bfloat16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b):
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
