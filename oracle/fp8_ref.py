"""Oracle for the FP8 linear layer (test infrastructure only).

Source: the modded-nanogpt project page ("NanoGPT (124M) in 90 seconds",
"How it works", the precision bullet) runs the MLP, the QKV projections and
the head in FP8. The page gives no recipe, so this follows the plainest one:
per-tensor scaling of each operand to the e4m3 format (OCP 8-bit floating
point: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals, no
infinities, one NaN pattern per sign, largest finite value 448), round to
nearest with ties to even and saturation to +-448, products accumulated in
wide precision, the two scales applied to the result.

Quantization decides integer codes, so it takes its decisions in float32,
as the kernel does: scale = 448 / amax and x * scale are float32 roundings.
Everything else runs in float64.
"""
import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """float64 values of e4m3 codes (uint8): (-1)^s 2^(e-7) (1 + m/8) for e >= 1,
    (-1)^s 2^-6 (m/8) for e = 0; e = 15, m = 7 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


# the 127 non-negative finite codes in increasing order of value (0x00 .. 0x7E)
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x):
    """e4m3 codes of x: the nearest finite value, ties to the even code (the one
    whose last mantissa bit is 0), |x| > 448 saturated to 448, NaN to 0x7F; the
    sign is that of x (a negative x that rounds to zero gives -0, 0x80).
    The choice is made on the value exactly as given (float32 inputs are exact
    in float64)."""
    v = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    dlo, dhi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)  # the sign is kept, zero too
    return np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)


def quantize_e4m3(x):
    """Per-tensor scaling: amax = max |x|; scale = 448 / amax (1 when amax is 0),
    codes = e4m3(x * scale), both products rounded to float32. Returns the codes
    and scale_inv = amax / 448 (float32), the factor that maps codes back."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    scale = np.float32(E4M3_MAX) / amax if amax > 0 else np.float32(1)
    scale_inv = amax / np.float32(E4M3_MAX) if amax > 0 else np.float32(1)
    return e4m3_encode((x32 * scale).astype(np.float32)), np.float32(scale_inv)


def matmul_fp8(a_codes, a_scale_inv, b_codes, b_scale_inv, bias=None):
    """D = (decode(A) decode(B)^T) a_scale_inv b_scale_inv (+ bias), float64;
    A [M, K], B [N, K] (the [out, in] weight layout)."""
    d = e4m3_decode(a_codes) @ e4m3_decode(b_codes).T
    d = d * float(a_scale_inv) * float(b_scale_inv)
    if bias is not None:
        d = d + np.asarray(bias, dtype=np.float64)
    return d
