"""Oracle for the FP8 linear layer (test infrastructure only).

Source: the modded-nanogpt project page ("NanoGPT (124M) in 90 seconds",
"How it works", the precision bullet) runs the MLP, the QKV projections and
the head in FP8. The page gives no recipe, so this follows the plainest one:
per-tensor scaling of each operand to an 8-bit floating-point format, round
to nearest with ties to even and saturation to the largest finite value,
products accumulated in wide precision, the two scales applied to the result.

The two formats are those of the OCP 8-bit floating point specification:
  e4m3  1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals, no
        infinities, one NaN pattern per sign (S.1111.111), largest finite 448;
        the format for weights and activations;
  e5m2  1 sign, 5 exponent bits (bias 15), 2 mantissa bits, subnormals,
        infinities (S.11111.00) and NaNs (S.11111.xx, xx != 0) as in IEEE 754,
        largest finite 57344; the wider range suits gradients.

Quantization decides integer codes, so it takes its decisions in float32,
as the kernel does: scale = max / amax and x * scale are float32 roundings.
Everything else runs in float64.
"""
import numpy as np

# exponent bits, mantissa bits, exponent bias, largest finite value
FORMATS = {
    "e4m3": (4, 3, 7, 448.0),
    "e5m2": (5, 2, 15, 57344.0),
}
E4M3_MAX = FORMATS["e4m3"][3]
E5M2_MAX = FORMATS["e5m2"][3]


def fp8_decode(codes, fmt):
    """float64 values of 8-bit codes (uint8) in format fmt:
    (-1)^s 2^(e-bias) (1 + m/2^mb) for a normal exponent field e >= 1,
    (-1)^s 2^(1-bias) (m/2^mb) for e = 0; the all-ones exponent field holds
    NaN (e4m3: only with m all ones; e5m2: m != 0) and, in e5m2, infinity
    (m = 0)."""
    eb, mb, bias, _ = FORMATS[fmt]
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> mb) & ((1 << eb) - 1)
    m = c & ((1 << mb) - 1)
    frac = m / float(1 << mb)
    mag = np.where(e == 0, np.ldexp(frac, 1 - bias), np.ldexp(1.0 + frac, e - bias))
    top = (1 << eb) - 1
    if fmt == "e4m3":
        mag = np.where((e == top) & (m == (1 << mb) - 1), np.nan, mag)
    else:
        mag = np.where(e == top, np.where(m == 0, np.inf, np.nan), mag)
    return s * mag


def _finite_positive_codes(fmt):
    """The non-negative finite codes of fmt in increasing order of value
    (codes 0x00 up to the largest finite one increase with the value)."""
    codes = np.arange(0x80, dtype=np.uint8)
    v = fp8_decode(codes, fmt)
    keep = np.isfinite(v)
    return codes[keep], v[keep]


_TABLES = {f: _finite_positive_codes(f) for f in FORMATS}


def fp8_encode(x, fmt):
    """Codes of x in format fmt: the nearest finite value, ties to the even
    code (the one whose last mantissa bit is 0), |x| above the largest finite
    value (infinity included) saturated to it, NaN to 0x7F; the sign is that
    of x (a negative x that rounds to zero gives -0, 0x80). The choice is made
    on the value exactly as given (float32 inputs are exact in float64)."""
    codes, values = _TABLES[fmt]
    v = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(v), FORMATS[fmt][3])
    hi = np.clip(np.searchsorted(values, a, side="left"), 0, len(values) - 1)
    lo = np.clip(hi - 1, 0, len(values) - 1)
    dlo, dhi = a - values[lo], values[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0))
    code = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    code = np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)  # the sign is kept, zero too
    return np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)


def e4m3_decode(codes):
    return fp8_decode(codes, "e4m3")


def e4m3_encode(x):
    return fp8_encode(x, "e4m3")


def e5m2_decode(codes):
    return fp8_decode(codes, "e5m2")


def e5m2_encode(x):
    return fp8_encode(x, "e5m2")


def quantize(x, fmt):
    """Per-tensor scaling: amax = max |x|; scale = max_fmt / amax (1 when amax
    is 0), codes = encode(x * scale), both products rounded to float32.
    Returns the codes and scale_inv = amax / max_fmt (float32), the factor
    that maps codes back."""
    fmax = np.float32(FORMATS[fmt][3])
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    scale = fmax / amax if amax > 0 else np.float32(1)
    scale_inv = amax / fmax if amax > 0 else np.float32(1)
    return fp8_encode((x32 * scale).astype(np.float32), fmt), np.float32(scale_inv)


def quantize_e4m3(x):
    return quantize(x, "e4m3")


def quantize_e5m2(x):
    return quantize(x, "e5m2")


def matmul_fp8(a_codes, a_scale_inv, b_codes, b_scale_inv, bias=None, a_fmt="e4m3", b_fmt="e4m3"):
    """D = (decode(A) decode(B)^T) a_scale_inv b_scale_inv (+ bias), float64;
    A [M, K], B [N, K] (the [out, in] weight layout), each in its own format."""
    d = fp8_decode(a_codes, a_fmt) @ fp8_decode(b_codes, b_fmt).T
    d = d * float(a_scale_inv) * float(b_scale_inv)
    if bias is not None:
        d = d + np.asarray(bias, dtype=np.float64)
    return d
