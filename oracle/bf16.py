"""Round-to-nearest-even from fp64 to bfloat16, written out from the format.

Test infrastructure only (see the package docstring).

bfloat16 keeps the fp32 exponent range (8 exponent bits, bias 127) and 8
significant bits (7 stored).  A finite non-zero x = f * 2**e with 0.5 <= f < 1
(``numpy.frexp``) has its leading bit at weight 2**(e-1), so its 8th
significant bit has weight 2**(e-8).  Below the smallest normal 2**-126 the
spacing stays at 2**-133 (subnormals).  Rounding is to the nearest multiple of
that spacing, ties to even (``numpy.rint`` rounds half to even), and magnitudes
that round past the largest finite value (2 - 2**-7) * 2**127 become inf.
"""

import numpy as np

_MAX_BF16 = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(x):
    """Return fp64 values on the bfloat16 grid: RNE of ``x`` (any shape)."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    _, e = np.frexp(xf)
    quantum_exp = np.maximum(e, -125) - 8
    scaled = np.ldexp(xf, -quantum_exp)           # exact: power-of-two scaling
    r = np.ldexp(np.rint(scaled), quantum_exp)    # ties to even
    r = np.where(np.abs(r) > _MAX_BF16, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def bf16_bits(x):
    """The 16-bit bfloat16 encoding of values already on the bf16 grid."""
    x = np.asarray(x, dtype=np.float64)
    f32 = x.astype(np.float32)  # exact for values on the bf16 grid
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def from_bits(bits):
    """fp64 values of 16-bit bfloat16 encodings."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
