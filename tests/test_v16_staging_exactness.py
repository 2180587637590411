"""The fp16 copy of V that a bf16 prefill can stage, restated and checked on
the CPU.  A (sequence, kv head) whose largest bf16 exponent field is E has
its V written as fp16(v * 2^-k) with k = clamp(E - 142, -100, 113), and the
attention result is multiplied back by 2^k.  Claims checked over every finite
bf16 value and every E:
  * nothing overflows: every |v| below 2^(E - 126) lands under 65504;
  * when the largest |v| is at least 2^-85 (E >= 42; below that the clamp at
    -100 binds), every value within 2^30 of it comes back exactly: bf16's
    8-bit significand fits fp16's 11, and the scaled value stays at or above
    fp16's subnormal spacing times 2^7.
"""
import numpy as np


def _shift(E):
    return min(113, max(-100, E - 142))


def test_staged_copy_is_exact_near_the_maximum_and_never_overflows():
    pats = np.arange(1 << 15, dtype=np.uint32)                 # non-negative bf16 patterns
    v = (pats << 16).view(np.float32)
    field = (pats >> 7) & 0xFF
    finite = field < 255
    for E in range(1, 255):
        k = _shift(E)
        sel = finite & (field <= E)                            # values a group with max field E holds
        x = v[sel]
        scaled = (x * np.float32(2.0 ** -k)).astype(np.float16)
        assert np.isfinite(scaled).all(), E
        if E >= 42:
            back = scaled.astype(np.float32) * np.float32(2.0 ** k)
            near = x >= np.float32(2.0 ** (E - 127 - 30))       # within 2^30 of the smallest max
            assert np.array_equal(back[near], x[near]), E
