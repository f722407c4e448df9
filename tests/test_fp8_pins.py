"""Pins for the FP8 oracle (e4m3 format, per-tensor quantization, FP8 product),
against the format's published constants, a library conversion and closed
forms; no GPU."""
import numpy as np
import pytest

from oracle import fp8_ref as F


def test_e4m3_format_constants():
    # OCP 8-bit floating point, E4M3: largest finite 448 = 1.75 * 2^8, smallest
    # normal 2^-6, smallest subnormal 2^-9, one NaN pattern per sign, no infinity
    v = F.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x07] == 7 * 2.0 ** -9 and v[0x01] == 2.0 ** -9
    assert v[0x38] == 1.0 and v[0x40] == 2.0 and v[0x30] == 0.5
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and int(np.isnan(v).sum()) == 2
    assert v[0x00] == 0.0 and v[0x80] == 0.0 and np.signbit(v[0x80])
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes 0x00..0x7E increase with value


def test_e4m3_round_trip_every_code():
    codes = np.arange(256, dtype=np.uint8)
    v = F.e4m3_decode(codes)
    fin = ~np.isnan(v)
    assert np.array_equal(F.e4m3_encode(v[fin]), codes[fin])


def test_e4m3_encode_matches_library_conversion():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.uniform(-448, 448, 50000), rng.normal(0, 1e-2, 50000),
                        rng.normal(0, 1e-3, 20000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), ref)


def test_e4m3_ties_saturation_nan():
    enc = lambda a: int(F.e4m3_encode(np.float32(a)))
    assert enc(1.0625) == 0x38 and enc(1.1875) == 0x3A  # midpoints go to the even code
    assert enc(0.5 * 2.0 ** -9) == 0x00 and enc(1.5 * 2.0 ** -9) == 0x02  # subnormal ties
    assert enc(448.0) == 0x7E and enc(449.0) == 0x7E and enc(1e30) == 0x7E and enc(-1e30) == 0xFE
    assert enc(np.nan) == 0x7F
    assert enc(-1e-30) == 0x80  # the sign survives a rounding to zero


def test_quantize_per_tensor_scaling():
    rng = np.random.default_rng(3)
    x = (rng.normal(0, 0.02, (64, 96)) * np.where(rng.random((64, 96)) < 0.01, 50.0, 1.0)).astype(np.float32)
    codes, scale_inv = F.quantize_e4m3(x)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert codes[i] in (0x7E, 0xFE)  # the largest magnitude maps to +-448
    assert scale_inv == np.float32(np.max(np.abs(x))) / np.float32(448.0)
    back = F.e4m3_decode(codes) * float(scale_inv)
    normal = np.abs(x) * (448.0 / np.max(np.abs(x))) >= 2.0 ** -6
    # within half a unit in the last place: 2^-4 relative for normals
    assert np.all(np.abs(back - x)[normal] <= 2.0 ** -4 * np.abs(x)[normal] * (1 + 1e-6))
    zeros, s0 = F.quantize_e4m3(np.zeros(8, np.float32))
    assert np.all(zeros == 0) and s0 == 1.0


def test_matmul_fp8_closed_form():
    # A = [[1, 2], [0.5, -1]], B = [[0.25, 4], [1, 1]] as e4m3 codes, scales 2 and 1/4
    a = F.e4m3_encode(np.array([[1.0, 2.0], [0.5, -1.0]]))
    b = F.e4m3_encode(np.array([[0.25, 4.0], [1.0, 1.0]]))
    d = F.matmul_fp8(a, 2.0, b, 0.25, bias=np.array([1.0, -1.0]))
    # (A B^T) = [[8.25, 3], [-3.875, -0.5]]; times 0.5; plus the bias
    assert np.array_equal(d, np.array([[5.125, 0.5], [-0.9375, -1.25]]))


# ---------------------------------------------------------------- e5m2

def test_e5m2_is_the_top_byte_of_binary16():
    # e5m2 has binary16's sign and exponent fields and the top two bits of its
    # mantissa, so code c is the half-precision number with bit pattern c << 8
    codes = np.arange(256, dtype=np.uint16)
    half = (codes << 8).astype(np.uint16).view(np.float16).astype(np.float64)
    v = F.e5m2_decode(codes.astype(np.uint8))
    assert np.array_equal(np.isnan(v), np.isnan(half))
    fin = ~np.isnan(half)
    assert np.array_equal(v[fin], half[fin])


def test_e5m2_format_constants():
    # OCP 8-bit floating point, E5M2: largest finite 57344 = 1.75 * 2^15,
    # smallest normal 2^-14, smallest subnormal 2^-16, infinities and three
    # NaN patterns per sign
    v = F.e5m2_decode(np.arange(256, dtype=np.uint8))
    assert v[0x7B] == 57344.0 and v[0xFB] == -57344.0
    assert v[0x7C] == np.inf and v[0xFC] == -np.inf
    assert v[0x04] == 2.0 ** -14 and v[0x03] == 3 * 2.0 ** -16 and v[0x01] == 2.0 ** -16
    assert v[0x3C] == 1.0 and v[0x40] == 2.0 and v[0x38] == 0.5
    assert int(np.isnan(v).sum()) == 6 and np.all(np.isnan(v[[0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]]))
    assert np.all(np.diff(v[:0x7C]) > 0)


def test_e5m2_round_trip_every_code():
    codes = np.arange(256, dtype=np.uint8)
    v = F.e5m2_decode(codes)
    fin = np.isfinite(v)
    assert np.array_equal(F.e5m2_encode(v[fin]), codes[fin])


def test_e5m2_encode_matches_library_conversion():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e5m2"):
        pytest.skip("no float8_e5m2 in this torch")
    rng = np.random.default_rng(11)
    # inside the finite range (the library conversion does not saturate beyond it)
    x = np.concatenate([rng.uniform(-57000, 57000, 50000), rng.normal(0, 1.0, 50000),
                        rng.normal(0, 1e-4, 20000), rng.normal(0, 1e-6, 20000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(F.e5m2_encode(x), ref)


def test_e5m2_ties_saturation_nan():
    enc = lambda a: int(F.e5m2_encode(np.float32(a)))
    assert enc(1.125) == 0x3C and enc(1.375) == 0x3E  # midpoints go to the even code
    assert enc(0.5 * 2.0 ** -16) == 0x00 and enc(1.5 * 2.0 ** -16) == 0x02  # subnormal ties
    assert enc(57344.0) == 0x7B and enc(61439.0) == 0x7B and enc(1e30) == 0x7B
    assert enc(np.inf) == 0x7B and enc(-np.inf) == 0xFB  # saturation, not infinity
    assert enc(np.nan) == 0x7F and enc(-1e-30) == 0x80


def test_quantize_e5m2_per_tensor_scaling():
    rng = np.random.default_rng(5)
    x = (rng.normal(0, 1e-3, (48, 80)) * np.where(rng.random((48, 80)) < 0.02, 1e3, 1.0)).astype(np.float32)
    codes, scale_inv = F.quantize_e5m2(x)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert codes[i] in (0x7B, 0xFB)  # the largest magnitude maps to +-57344
    assert scale_inv == np.float32(np.max(np.abs(x))) / np.float32(57344.0)
    back = F.e5m2_decode(codes) * float(scale_inv)
    normal = np.abs(x) * (57344.0 / np.max(np.abs(x))) >= 2.0 ** -14
    # within half a unit in the last place: 2^-3 relative for normals
    assert np.all(np.abs(back - x)[normal] <= 2.0 ** -3 * np.abs(x)[normal] * (1 + 1e-6))


def test_matmul_fp8_mixed_formats_closed_form():
    # A = [[1, -3], [0.25, 6]] in e5m2 with scale 4; B = [[0.5, 2], [1.75, -1]] in e4m3 with scale 1/8
    a = F.e5m2_encode(np.array([[1.0, -3.0], [0.25, 6.0]]))
    b = F.e4m3_encode(np.array([[0.5, 2.0], [1.75, -1.0]]))
    d = F.matmul_fp8(a, 4.0, b, 0.125, a_fmt="e5m2", b_fmt="e4m3")
    # (A B^T) = [[-5.5, 4.75], [12.125, -5.5625]]; times 0.5
    assert np.array_equal(d, np.array([[-2.75, 2.375], [6.0625, -2.78125]]))
    # the same codes read in the other format give other values: the format is not ignored
    assert not np.array_equal(F.matmul_fp8(a, 4.0, b, 0.125, a_fmt="e4m3", b_fmt="e4m3"), d)


# ---- the FP8 linear layer of the oracle's step ----

def _grid_values(rng, shape, table, top):
    """Values drawn from a format's finite values, with the largest finite
    value present (so amax = fmax, the scale is 1 and quantization is exact)."""
    v = rng.choice(table, size=shape) * rng.choice([-1.0, 1.0], size=shape)
    v.reshape(-1)[0] = top
    return v


def test_fp8_linear_exact_on_representable_operands():
    """Operands that are already format values with amax = fmax quantize
    exactly (scale 1), so the FP8 linear layer equals the float64 one; with
    amax = 2 fmax the scale is 1/2, also exact."""
    from oracle import gpt2_ref as R
    rng = np.random.default_rng(11)
    e4 = F.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    e5 = F.e5m2_decode(np.arange(0x7C, dtype=np.uint8))
    x = _grid_values(rng, (6, 5, 16), e4, 448.0)
    w = _grid_values(rng, (12, 16), e4, 448.0)
    b = rng.normal(size=12)
    assert np.array_equal(R.linear_forward_fp8(x, w, b), R.linear_forward(x, w, b))
    assert np.array_equal(R.linear_forward_fp8(2 * x, w), R.linear_forward(2 * x, w))
    dy = _grid_values(rng, (30, 12), e5, 57344.0)
    dx, dw, db = R.linear_backward_fp8(dy, x.reshape(30, 16), w)
    rx, rw, rb = R.linear_backward(dy, x.reshape(30, 16), w)
    assert np.array_equal(dx, rx) and np.array_equal(dw, rw) and np.array_equal(db, rb)


def test_fp8_linear_quantizes_each_operand_per_tensor():
    """A plain operand: the layer equals the product of each operand's
    quantized values (codes times amax / fmax), dy in e5m2, x and w in e4m3;
    the error against the exact product stays within the bound the
    rounding of each operand allows."""
    from oracle import gpt2_ref as R
    rng = np.random.default_rng(12)
    x, w, dy = rng.normal(size=(64, 32)), rng.normal(size=(24, 32)), rng.normal(size=(64, 24))
    qx, sx = F.quantize_e4m3(x)
    qw, sw = F.quantize_e4m3(w)
    ref = (F.e4m3_decode(qx) * float(sx)) @ (F.e4m3_decode(qw) * float(sw)).T
    assert np.allclose(R.linear_forward_fp8(x, w), ref, rtol=0, atol=1e-12)
    # per element |q(a) - a| <= 2^-4 |a| + 2^-10 amax / 448 (half the spacing
    # of normal e4m3 values, and of the subnormals), summed over the products
    ex = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * np.abs(x).max() / 448
    ew = 2.0 ** -4 * np.abs(w) + 2.0 ** -10 * np.abs(w).max() / 448
    bound = ex @ np.abs(w).T + np.abs(x) @ ew.T + ex @ ew.T
    assert np.all(np.abs(R.linear_forward_fp8(x, w) - x @ w.T) <= bound * (1 + 1e-9))
    dx, dw, db = R.linear_backward_fp8(dy, x, w)
    qd, sd = F.quantize_e5m2(dy)
    d = F.e5m2_decode(qd) * float(sd)
    assert np.allclose(dx, d @ (F.e4m3_decode(qw) * float(sw)), rtol=0, atol=1e-12)
    assert np.allclose(dw, d.T @ (F.e4m3_decode(qx) * float(sx)), rtol=0, atol=1e-12)
    assert np.array_equal(db, dy.sum(0))


def test_fp8_step_runs_the_selected_linears_in_fp8():
    """The FP8 step changes the loss and the gradients by quantization-sized
    amounts (not zero, not more than a few percent) and leaves the linears
    that are not selected alone (with fp8=() the step is the bf16 one)."""
    from oracle import gpt2_ref as R
    cfg = R.Config(2, 32, 2, 64, 64, 16)
    params = R.init_params(cfg, 5)
    rng = np.random.default_rng(3)
    tok = rng.integers(0, 64, size=(2, 16))
    tgt = rng.integers(0, 64, size=(2, 16))
    l0, c0 = R.forward(cfg, params, tok, tgt)
    g0 = R.backward(cfg, c0)
    l1, c1 = R.forward(cfg, params, tok, tgt, fp8=())
    assert l1 == l0
    for sel in (("qkv",), ("mlp",), ("head",), ("qkv", "mlp", "head")):
        l2, c2 = R.forward(cfg, params, tok, tgt, fp8=sel)
        g2 = R.backward(cfg, c2)
        assert l2 != l0 and abs(l2 - l0) < 0.05 * l0, (sel, l0, l2)
        for name in ("h0.qkv.w", "h1.fc.w", "wte"):
            err = np.linalg.norm(g2[name] - g0[name]) / np.linalg.norm(g0[name])
            assert err < 0.2, (sel, name, err)
        changed = {n for n in g0 if not np.array_equal(g0[n], g2[n])}
        assert changed, sel
