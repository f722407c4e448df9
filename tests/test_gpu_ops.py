"""Per-kernel parity: each CUDA kernel (through the C ABI) against the oracle.

Inputs are seeded and, in bf16 mode, exactly representable in bf16, so both
sides start from the same values; the oracle computes in float64.
Tolerances: bf16 outputs carry one round-to-nearest-even (relative 2^-9),
checked at 2^-8 relative plus a small floor near zero; fp32 outputs at
1e-5 relative (fp32 accumulation against float64).
"""
import math

import numpy as np
import pytest

from oracle import gpt2_ref as R
from step_gpt_train_gb300 import data
from tests._gpu_util import (BF16_REL, assert_close, dev, dev_f32, host, inputs, rel_l2, torch_dtype)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    from step_gpt_train_gb300 import gpt2 as g
    g.load_library(build=True)
    torch.cuda.set_device(0)
    return torch


def _gemm_ref(A, a_mn, B, b_mn, M, N, K, bias):
    a = A.reshape(K, M).T if a_mn else A.reshape(M, K)
    b = B.reshape(K, N).T if b_mn else B.reshape(N, K)
    d = a.astype(np.float64) @ b.astype(np.float64).T
    if bias is not None:
        d = d + bias
    return d


def tc_accum_atol(K, ref):
    """Error bound of a tensor-core fp32 accumulation over K: the accumulator is
    rounded once per 16-deep MMA step, at most one unit in the last place of the
    running sum each time; the running sum is bounded by 4 max|result| for
    these random inputs."""
    return (K / 16) * 2.0 ** -23 * 4 * float(np.abs(ref).max())


GEMM_CASES = [
    # M, N, K, a_mn, b_mn, d_fp32, bias
    (300, 392, 200, 0, 0, 0, True),    # linear forward, ragged M, N (two 256 tiles), K
    (300, 120, 200, 0, 0, 0, True),    # 128-wide tiles
    (300, 200, 392, 0, 1, 0, False),   # input gradient dX = dY W
    (392, 200, 304, 1, 1, 1, False),   # weight gradient dW = dY^T X, fp32 out
    (128, 256, 4096, 1, 1, 1, False),  # weight gradient with split-K
    (136, 264, 72, 1, 0, 0, False),    # A M-major, B K-major
    (520, 1032, 1000, 0, 0, 1, True),  # fp32 out with bias through the stream-K reduce
    (300, 768, 256, 0, 0, 0, True),    # 192-wide tiles
    (300, 776, 320, 0, 1, 0, False),   # 192-wide tiles, ragged last column tile
    (392, 776, 2000, 1, 1, 1, False),  # stream-K weight gradient, ragged M and N
]


@pytest.mark.parametrize("mode", [1, 0])
@pytest.mark.parametrize("case", GEMM_CASES)
def test_matmul(torch_cuda, mode, case):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_matmul
    M, N, K, a_mn, b_mn, d_fp32, use_bias = case
    A = inputs(1, (M * K,), 1.0, mode)
    B = inputs(2, (N * K,), 1.0, mode)
    bias = inputs(3, (N,), 1.0, mode) if use_bias else None
    dA, dB = dev(A, mode), dev(B, mode)
    dbias = dev(bias, mode) if use_bias else None
    out_dtype = torch.float32 if (d_fp32 or mode == 0) else torch.bfloat16
    D = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    gpt2_op_matmul(D, dA, a_mn, dB, b_mn, M, N, K, bias=dbias)
    torch.cuda.synchronize()
    ref = _gemm_ref(A, a_mn, B, b_mn, M, N, K, bias)
    got = host(D)
    assert np.all(np.isfinite(got))
    if out_dtype == torch.bfloat16:
        assert_close(got, ref, BF16_REL, atol_frac=1e-3, what="bf16 matmul")
    elif mode == 1:
        assert_close(got, ref, 1e-5, atol=tc_accum_atol(K, ref), what="fp32 tensor-core matmul")
    else:
        assert_close(got, ref, 1e-5, atol_frac=1e-5, what="fp32 matmul")


# The CTA-pair kernel's range: at least 512 rows and 1024 columns (256-wide
# pair tiles), or 384 to 960 columns in 192-wide tiles with K from 2048 to
# 16384 (MN-major B there in 64-byte swizzle atoms).
PAIR_CASES = [
    # M, N, K, a_mn, b_mn, d_fp32, bias
    (1000, 1032, 1000, 0, 0, 0, True),   # ragged in every dimension (a half-empty last pair tile)
    (520, 2304, 768, 0, 1, 0, False),    # B MN-major
    (768, 1024, 512, 1, 0, 0, False),    # A MN-major
    (1024, 1280, 256, 1, 1, 1, False),   # both MN-major, fp32 out
    (1000, 768, 2104, 0, 0, 0, True),    # 192-wide tiles, ragged M and K
    (520, 768, 3072, 1, 0, 0, False),    # 192-wide tiles, A MN-major
    (1024, 576, 2048, 0, 0, 1, False),   # 192-wide tiles, fp32 out
    (1000, 768, 2104, 0, 1, 0, False),   # 192-wide tiles, B MN-major (64-byte swizzle), ragged M and K
    (520, 576, 2048, 1, 1, 1, False),    # 192-wide tiles, both MN-major, fp32 out
]


@pytest.mark.parametrize("case", PAIR_CASES)
def test_matmul_pair_kernel(torch_cuda, case):
    """Plain products in the range of the CTA-pair kernel (tcgen05 .cta_group::2,
    one M = 256 product for two SMs; the default there) against the oracle, and
    against the one-CTA kernel on the same inputs (gpt2_debug_matmul_pair(0))."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_matmul, load_library
    lib = load_library()
    M, N, K, a_mn, b_mn, d_fp32, use_bias = case
    A = inputs(111, (M * K,), 1.0, 1)
    B = inputs(112, (N * K,), 1.0, 1)
    bias = inputs(113, (N,), 1.0, 1) if use_bias else None
    dA, dB = dev(A, 1), dev(B, 1)
    dbias = dev(bias, 1) if use_bias else None
    out_dtype = torch.float32 if d_fp32 else torch.bfloat16
    got = {}
    try:
        for pair in (1, 0):
            assert lib.gpt2_debug_matmul_pair(pair) >= 0
            D = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
            gpt2_op_matmul(D, dA, a_mn, dB, b_mn, M, N, K, bias=dbias)
            torch.cuda.synchronize()
            got[pair] = host(D)
    finally:
        lib.gpt2_debug_matmul_pair(1)
    ref = _gemm_ref(A, a_mn, B, b_mn, M, N, K, bias)
    for pair in (1, 0):
        assert np.all(np.isfinite(got[pair]))
        if d_fp32:
            assert_close(got[pair], ref, 1e-5, atol=tc_accum_atol(K, ref), what=f"fp32 matmul, pair={pair}")
        else:
            assert_close(got[pair], ref, BF16_REL, atol_frac=1e-3, what=f"bf16 matmul, pair={pair}")
    # the same products in both kernels: fp32 out to the accumulation bound, bf16
    # out to one rounding (an ulp is up to 2^-7 of the value)
    if d_fp32:
        assert_close(got[1], got[0], 1e-5, atol=tc_accum_atol(K, ref), what="pair vs one-CTA kernel")
    else:
        assert_close(got[1], got[0], 2.0 ** -7, atol=1e-30, what="pair vs one-CTA kernel")


def test_matmul_gelu_pair_kernel(torch_cuda):
    """The GELU and GELU-gradient epilogues (with the bias-gradient column sums)
    in the CTA-pair kernel (gpt2_debug_matmul_pair(2): off by default) against
    the one-CTA kernel's: the stored values to one bf16 rounding, the column
    sums to fp32 summation error."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import (gpt2_op_matmul_gelu, gpt2_op_matmul_gelu_backward_bias, load_library)
    lib = load_library()
    M, N, K, K2 = 1000, 3072, 768, 512
    A = dev(inputs(120, (M, K), 1.0, 1))
    W = dev(inputs(121, (N, K), K ** -0.5, 1))
    b = dev(inputs(122, (N,), 0.5, 1))
    dY = dev(inputs(123, (M, K2), 1.0, 1))
    W2 = dev(inputs(124, (K2, N), K2 ** -0.5, 1))
    res = {}
    try:
        for pair in (2, 0):
            assert lib.gpt2_debug_matmul_pair(pair) >= 0
            dgelu = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            out = torch.full_like(dgelu, float("nan"))
            gpt2_op_matmul_gelu(dgelu, out, A, W, b)
            du = torch.full_like(dgelu, float("nan"))
            dbias = torch.full((N,), float("nan"), device="cuda")
            gpt2_op_matmul_gelu_backward_bias(du, dbias, dY, W2, dgelu)
            torch.cuda.synchronize()
            res[pair] = [host(t) for t in (dgelu, out, du, dbias)]
    finally:
        lib.gpt2_debug_matmul_pair(1)
    for name, x2, x0 in zip(("gelu'", "gelu", "du"), res[2][:3], res[0][:3]):
        assert np.all(np.isfinite(x2)), name
        assert_close(x2, x0, 2.0 ** -7, atol=1e-30, what=f"{name}: pair vs one-CTA kernel")
    scale = float(np.abs(res[0][2].astype(np.float64)).sum(0).max())
    assert_close(res[2][3], res[0][3], 0, atol=1e-5 * scale, what="dbias: pair vs one-CTA kernel")


def test_matmul_full_size_sampled(torch_cuda):
    """Bench-size GEMMs (GPT-2 124M at B*T = 32768); outputs sampled and computed one by one."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_matmul
    rng = np.random.default_rng(5)
    # LM head forward: [32768, 768] x [50304, 768]^T -> bf16 [32768, 50304]
    M, N, K = 32768, 50304, 768
    A = dev(inputs(101, (M, K), 1.0))
    B = dev(inputs(102, (N, K), 0.02))
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    gpt2_op_matmul(D, A, 0, B, 0, M, N, K)
    torch.cuda.synchronize()
    ms, ns = rng.integers(0, M, 3000), rng.integers(0, N, 3000)
    ns[:200] = N - 1 - rng.integers(0, 128, 200)  # the ragged last column tile
    a, b = host(A[ms]), host(B[ns])
    ref = np.einsum("ik,ik->i", a, b)
    got = host(D[ms, ns])
    assert_close(got, ref, BF16_REL, atol_frac=1e-3, what="LM head sampled")
    # MLP projection weight gradient: dW = dY^T X, K = 32768, fp32 out (split-K)
    M, N, K = 768, 3072, 32768
    dY = dev(inputs(103, (K, M), 1.0))
    X = dev(inputs(104, (K, N), 1.0))
    W = torch.empty(M, N, dtype=torch.float32, device="cuda")
    gpt2_op_matmul(W, dY, 1, X, 1, M, N, K)
    torch.cuda.synchronize()
    ms, ns = rng.integers(0, M, 400), rng.integers(0, N, 400)
    ref = np.einsum("ki,ki->i", host(dY[:, ms]), host(X[:, ns]))
    assert_close(host(W[ms, ns]), ref, 1e-5, atol=tc_accum_atol(K, ref), what="dW sampled")


@pytest.mark.parametrize("mode", [1, 0])
@pytest.mark.parametrize("C", [64, 768, 1024, 1600, 2048])  # above 1024 (bf16): the wide-row kernels
def test_layernorm(torch_cuda, mode, C):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_layernorm_backward, gpt2_op_layernorm_forward
    N = 333
    x = inputs(10, (N, C), 2.0, mode) + (inputs(11, (N, 1), 1.0, mode) if mode == 0 else 0)
    x = data.round_to_bf16(x) if mode == 1 else x
    g = inputs(12, (C,), 1.0, mode)
    b = inputs(13, (C,), 1.0, mode)
    dy = inputs(14, (N, C), 1.0, mode)
    dx_, dg_, db_ = dev(x, mode), dev(g, mode), dev(b, mode)
    y = torch.empty_like(dx_)
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    gpt2_op_layernorm_forward(y, mean, rstd, dx_, dg_, db_)
    dx = torch.empty_like(dx_)
    dgam = torch.full((C,), float("nan"), device="cuda")
    dbet = torch.full((C,), float("nan"), device="cuda")
    gpt2_op_layernorm_backward(dx, dgam, dbet, dev(dy, mode), dx_, dg_, mean, rstd)
    torch.cuda.synchronize()
    ry, rmean, rrstd = R.layernorm_forward(x.astype(np.float64), g.astype(np.float64), b.astype(np.float64))
    rdx, rdg, rdb = R.layernorm_backward(dy.astype(np.float64), x.astype(np.float64), g.astype(np.float64),
                                         rmean, rrstd)
    tol = BF16_REL if mode == 1 else 1e-5
    assert_close(host(mean), rmean, 1e-6, atol=1e-6, what="mean")
    assert_close(host(rstd), rrstd, 1e-5, what="rstd")
    assert_close(host(y), ry, tol, atol_frac=1e-3 if mode == 1 else 1e-6, what="y")
    assert_close(host(dx), rdx, 2 * tol, atol_frac=2e-3 if mode == 1 else 1e-6, what="dx")
    assert_close(host(dgam), rdg, 1e-4, atol_frac=1e-5, what="dgamma")
    assert_close(host(dbet), rdb, 1e-4, atol_frac=1e-5, what="dbeta")


@pytest.mark.parametrize("mode", [1, 0])
@pytest.mark.parametrize("C", [64, 768, 1600])  # 1600 (bf16): the wide-row kernels
@pytest.mark.parametrize("accumulate", [0, 1])
def test_residual_layernorm(torch_cuda, mode, C, accumulate):
    """Residual join + LayerNorm forward, and LayerNorm backward into the residual
    gradient with the column sums of the result (the projection bias gradient)."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import (gpt2_op_layernorm_backward_residual,
                                           gpt2_op_residual_layernorm_forward)
    N = 4133  # several grid strides of the backward and a ragged tail
    x = inputs(30, (N, C), 2.0, mode)
    r = inputs(31, (N, C), 1.0, mode)
    g = inputs(32, (C,), 1.0, mode)
    b = inputs(33, (C,), 1.0, mode)
    dy = inputs(34, (N, C), 1.0, mode)
    dres0 = inputs(35, (N, C), 1.0, mode)
    g_, b_ = dev(g, mode), dev(b, mode)
    xsum = torch.empty(N, C, dtype=torch_dtype(mode), device="cuda")
    y = torch.empty_like(xsum)
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    gpt2_op_residual_layernorm_forward(y, mean, rstd, xsum, dev(x, mode), dev(r, mode), g_, b_)
    dres = dev(dres0, mode)
    dgam = torch.full((C,), float("nan"), device="cuda")
    dbet = torch.full((C,), float("nan"), device="cuda")
    dbias = torch.full((C,), float("nan"), device="cuda")
    gpt2_op_layernorm_backward_residual(dres, accumulate, dgam, dbet, dbias, dev(dy, mode), xsum, g_, mean, rstd)
    torch.cuda.synchronize()
    # the sum of two bf16 (or fp32) values, rounded once to the storage type
    s64 = x.astype(np.float64) + r.astype(np.float64)
    s_ref = data.round_to_bf16(s64.astype(np.float32)) if mode == 1 else s64.astype(np.float32)
    assert np.array_equal(host(xsum), s_ref.astype(np.float64)), "residual sum"
    sx = s_ref.astype(np.float64)
    ry, rmean, rrstd = R.layernorm_forward(sx, g.astype(np.float64), b.astype(np.float64))
    rdx, rdg, rdb = R.layernorm_backward(dy.astype(np.float64), sx, g.astype(np.float64), rmean, rrstd)
    tol = BF16_REL if mode == 1 else 1e-5
    assert_close(host(y), ry, tol, atol_frac=1e-3 if mode == 1 else 1e-6, what="y")
    rres = rdx + (dres0.astype(np.float64) if accumulate else 0.0)
    assert_close(host(dres), rres, 2 * tol, atol_frac=2e-3 if mode == 1 else 1e-6, what="dres")
    assert_close(host(dgam), rdg, 1e-4, atol_frac=1e-5, what="dgamma")
    assert_close(host(dbet), rdb, 1e-4, atol_frac=1e-5, what="dbeta")
    # column sums of what was stored (fp32 accumulation of N terms) ...
    assert_close(host(dbias), host(dres).sum(axis=0), 1e-5, atol=N * 2.0 ** -23 * float(np.abs(host(dres)).max()),
                 what="dres column sums")
    # ... and of the exact result: at most the sum over rows of the per-element
    # bounds checked above
    rms = float(np.sqrt(np.mean(rres * rres)))
    col_bound = (2 * tol * np.abs(rres) + (2e-3 if mode == 1 else 1e-6) * rms).sum(axis=0)
    assert np.all(np.abs(host(dbias) - rres.sum(axis=0)) <= col_bound * 1.001), "dres column sums vs oracle"


@pytest.mark.parametrize("mode", [1, 0])
def test_gelu(torch_cuda, mode):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_gelu_backward, gpt2_op_gelu_forward
    u = np.concatenate([np.linspace(-12, 12, 4000, dtype=np.float32), inputs(20, (4000,), 3.0, 0)])
    u = data.round_to_bf16(u) if mode == 1 else u
    dg = inputs(21, u.shape, 1.0, mode)
    du_, ddg = dev(u, mode), dev(dg, mode)
    g = torch.empty_like(du_)
    gpt2_op_gelu_forward(g, du_)
    dd = torch.empty_like(du_)
    gpt2_op_gelu_backward(dd, du_, ddg)
    torch.cuda.synchronize()
    tol = BF16_REL if mode == 1 else 1e-5
    rg = R.gelu_forward(u.astype(np.float64))
    rdu = R.gelu_backward(u.astype(np.float64), dg.astype(np.float64))
    # The float64 oracle evaluates the tanh form, whose 1 + tanh(y) cancels on the
    # negative tail: its absolute error there is about |u| * 1e-16, hence the floor.
    assert_close(host(g), rg, tol, atol=2e-15, what="gelu")
    assert_close(host(dd), rdu, tol, atol=1e-6, what="gelu backward")
    # in place, as the step uses it
    gpt2_op_gelu_backward(ddg, du_, ddg)
    torch.cuda.synchronize()
    assert_close(host(ddg), rdu, tol, atol=1e-6, what="gelu backward in place")


@pytest.mark.parametrize("mode", [1, 0])
@pytest.mark.parametrize("shape", [(300, 776, 256), (1000, 3072, 768)])
def test_matmul_gelu(torch_cuda, mode, shape):
    """Linear + GELU with the GELU in the GEMM epilogue (which keeps gelu' for
    the backward), and the input gradient through the GELU, against the oracle;
    the GELU output bit for bit against the separate matmul and GELU kernels."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import (gpt2_op_gelu_forward, gpt2_op_matmul, gpt2_op_matmul_gelu,
                                           gpt2_op_matmul_gelu_backward, gpt2_op_matmul_gelu_backward_bias)
    M, N, K = shape  # 300 rows: a ragged 128-row tile; N = 776: a ragged column tile
    A = inputs(60, (M, K), 1.0, mode)
    W = inputs(61, (N, K), K ** -0.5, mode)
    b = inputs(62, (N,), 0.5, mode)
    dA, dW, db = dev(A, mode), dev(W, mode), dev(b, mode)
    dgelu = torch.empty(M, N, dtype=torch_dtype(mode), device="cuda")
    out = torch.empty_like(dgelu)
    gpt2_op_matmul_gelu(dgelu, out, dA, dW, db)
    # the separate kernels: u = the linear output as stored, then its GELU
    u, out2 = torch.empty_like(dgelu), torch.empty_like(dgelu)
    gpt2_op_matmul(u, dA, 0, dW, 0, M, N, K, bias=db)
    gpt2_op_gelu_forward(out2, u)
    # backward: du = (dY W) gelu'(u), W [K2, N] (the weight of the next linear)
    K2 = 512
    dY = inputs(63, (M, K2), 1.0, mode)
    W2 = inputs(64, (K2, N), K2 ** -0.5, mode)
    du = torch.empty_like(dgelu)
    gpt2_op_matmul_gelu_backward(du, dev(dY, mode), dev(W2, mode), dgelu)
    dg = torch.empty_like(dgelu)
    gpt2_op_matmul(dg, dev(dY, mode), 0, dev(W2, mode), 1, M, N, K2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2), "fused GELU differs from matmul + gelu"
    tol = BF16_REL if mode == 1 else 1e-5
    rpre = R.linear_forward(A.astype(np.float64), W.astype(np.float64), b.astype(np.float64))
    # as for the plain matmul: fp32 accumulation over K, relative to the output's rms
    assert_close(host(u), rpre, tol, atol_frac=1e-3 if mode == 1 else 1e-5, what="pre-activation")
    hu = host(u)
    assert_close(host(out), R.gelu_forward(hu), tol, atol=2e-15, what="gelu(u)")
    # gelu'(u) sums O(1) terms that cancel near its zero (u ~ -0.75): a few fp32
    # ulps of 1 in absolute terms
    rd = R.gelu_backward(hu, np.ones_like(hu))
    assert_close(host(dgelu), rd, tol, atol=8 * 2.0 ** -23, what="gelu'(u)")
    # du = dtype(dY W) * dgelu exactly as formed, and against the oracle end to end
    # (one more rounding: gelu' as stored)
    assert_close(host(du), host(dg) * host(dgelu), tol, atol=1e-30, what="du = (dY W) dgelu")
    rdg = dY.astype(np.float64) @ W2.astype(np.float64)
    floor = 8 * 2.0 ** -23 * float(np.abs(rdg).max())
    assert_close(host(du), R.gelu_backward(hu, rdg), 3 * tol, atol_frac=2e-3 if mode == 1 else 1e-6, atol=floor,
                 what="du vs oracle")
    # with the bias gradient of the first linear (column sums of du; bf16: from
    # the matmul's epilogue): du bit for bit as without, dbias = the float64
    # column sums of du as stored, to fp32 summation error
    du2 = torch.full_like(dgelu, float("nan"))
    dbias = torch.full((N,), float("nan"), device="cuda")
    gpt2_op_matmul_gelu_backward_bias(du2, dbias, dev(dY, mode), dev(W2, mode), dgelu)
    torch.cuda.synchronize()
    assert torch.equal(du2, du)
    hdu = host(du).astype(np.float64)
    assert_close(host(dbias), hdu.sum(0), 0, atol=1e-5 * float(np.abs(hdu).sum(0).max()), what="dbias = colsum(du)")


@pytest.mark.parametrize("mode", [1, 0])
def test_residual(torch_cuda, mode):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_residual_backward, gpt2_op_residual_forward
    a = inputs(30, (1000, 24), 1.0, mode)
    b = inputs(31, (1000, 24), 1.0, mode)
    da, db = dev(a, mode), dev(b, mode)
    out = torch.empty_like(da)
    gpt2_op_residual_forward(out, da, db)
    gpt2_op_residual_backward(da, db)  # da += db
    torch.cuda.synchronize()
    ref = a.astype(np.float64) + b.astype(np.float64)
    ref = data.round_to_bf16(ref.astype(np.float32)) if mode == 1 else ref
    assert_close(host(out), ref, 1e-7 if mode == 1 else 1e-7, what="residual")
    assert_close(host(da), ref, 1e-7, what="residual backward")


@pytest.mark.parametrize("mode", [1, 0])
@pytest.mark.parametrize("C", [200, 3072])
def test_bias_backward(torch_cuda, mode, C):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_bias_backward
    dy = inputs(40, (1000, C), 1.0, mode)
    out = torch.full((C,), float("nan"), device="cuda")
    gpt2_op_bias_backward(out, dev(dy, mode))
    torch.cuda.synchronize()
    assert_close(host(out), dy.astype(np.float64).sum(0), 1e-5, atol=1e-4, what="bias grad")


# (mode, B, T, H). The last three bf16 cases have more (query tile, batch-head)
# work items than the persistent grids have CTAs (B=4, H=12, T=1024: 384
# items of 128 queries; B=3, T=1000: ragged last tile), so every CTA runs
# several items and the item-ahead loads and deferred accumulator stores of
# the backward are exercised as in the 124M step; at B=16 (1536 items) the
# kernels' schedules start with rounds of paired long and short tiles of one
# batch-head before their longest-first tail, as at B=32.
ATT_CASES = [(1, 2, 64, 3), (1, 2, 200, 2), (1, 1, 1024, 2), (1, 4, 1024, 12), (1, 3, 1000, 12), (1, 16, 1024, 12),
             (0, 2, 64, 4), (0, 3, 37, 4)]

# Element-wise bound on bf16 attention outputs: |got - ref| <= 2^-8 |ref| +
# ATT_BF16_ABS * rms(ref), per output block (o, dq, dk, dv). The kernels round
# P (into PV and dV) and dS (into dQ and dK) to bf16, and every output once
# more. Those roundings, emulated in float64 on q, k, v, dO ~ N(0, 1) at
# T = 1024, hd = 64, give at most 0.093 rms beyond 2^-8 |ref| (dq; 0.058 dk,
# 0.042 dv, 0.026 o); the bound allows about 2.7 times that.
ATT_BF16_ABS = 0.25


@pytest.mark.parametrize("case", ATT_CASES)
def test_attention(torch_cuda, case):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_attention_backward, gpt2_op_attention_forward
    mode, B, T, H = case
    hd = 64 if mode == 1 else 16
    C = H * hd
    qkv = inputs(50, (B, T, 3 * C), 1.0, mode)
    dout = inputs(51, (B, T, C), 1.0, mode)
    dq = dev(qkv, mode)
    o = torch.empty(B, T, C, dtype=dq.dtype, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    gpt2_op_attention_forward(o, lse, dq, B, T, H)
    dqkv = torch.full_like(dq, float("nan"))
    gpt2_op_attention_backward(dqkv, dev(dout, mode), dq, o, lse, B, T, H)
    torch.cuda.synchronize()
    ro, rlse = R.attention_forward(qkv.astype(np.float64), H)
    rd = R.attention_backward(dout.astype(np.float64), qkv.astype(np.float64), rlse, H)
    assert_close(host(lse), rlse, 1e-5, atol=1e-4, what="lse")
    if mode == 1:
        assert rel_l2(host(o), ro) < 1e-2
        assert_close(host(o), ro, 2.0 ** -8, atol_frac=ATT_BF16_ABS, what="o")
        for k, part in enumerate("qkv"):
            sl = slice(k * C, (k + 1) * C)
            assert rel_l2(host(dqkv)[..., sl], rd[..., sl]) < 1e-2, part
            assert_close(host(dqkv)[..., sl], rd[..., sl], 2.0 ** -8, atol_frac=ATT_BF16_ABS, what="d" + part)
    else:
        assert_close(host(o), ro, 1e-4, atol_frac=1e-5, what="o")
        assert_close(host(dqkv), rd, 1e-4, atol_frac=1e-5, what="dqkv")
    # deterministic: the backward run again gives identical bits
    again = torch.full_like(dq, float("nan"))
    gpt2_op_attention_backward(again, dev(dout, mode), dq, o, lse, B, T, H)
    torch.cuda.synchronize()
    assert torch.equal(again, dqkv)


# (mode, rows, V, Vp). The 1024-row cases give each of the persistent bf16
# kernel's CTAs (two per SM) more than one row, as the 124M step does.
CLS_CASES = [(1, 77, 1000, 1024), (0, 77, 1000, 1024), (1, 64, 50257, 50304), (0, 16, 50257, 50304),
             (1, 1024, 50257, 50304), (0, 1024, 50257, 50304)]


@pytest.mark.parametrize("case", CLS_CASES)
def test_classifier(torch_cuda, case):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_classifier, gpt2_op_mean_loss
    mode, N, V, Vp = case
    z = inputs(60, (N, Vp), 2.0, mode)
    z[:, V:] = 7.0  # padded columns must be ignored
    tgt = data.token_stream("uniform", N, 61, vocab=V)
    tgt[0] = V - 1
    dz = dev(z, mode)
    losses = torch.empty(N, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpt2_op_classifier(dz, losses, dev(tgt), V, 1.0 / N, status=status)
    mean = torch.empty(1, device="cuda")
    gpt2_op_mean_loss(mean, losses)
    torch.cuda.synchronize()
    rl, rd = R.classifier(z.astype(np.float64), tgt, V)
    assert int(status.item()) == 0
    assert_close(host(losses), rl, 1e-5, atol=2e-5, what="losses")
    assert abs(float(mean.item()) - rl.mean()) < 1e-5
    got = host(dz)
    assert np.all(got[:, V:] == 0.0)
    tol = BF16_REL if mode == 1 else 1e-5
    assert_close(got, rd, tol, atol=1e-7 / N, what="dlogits")
    # a target outside [0, V) is reported, not trapped
    bad = tgt.copy()
    bad[3] = V + 5
    status.zero_()
    gpt2_op_classifier(dev(z, mode), losses, dev(bad), V, 1.0 / N, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4


@pytest.mark.parametrize("mode", [1, 0])
def test_encoder_forward(torch_cuda, mode):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_encoder_forward
    V, C, B, T = (256, 64, 3, 100) if mode == 1 else (50257, 64, 3, 100)
    wte = inputs(70, (V, C), 0.5, mode)
    wpe = inputs(71, (T, C), 0.5, mode)
    wte[:, 0] = np.arange(V)  # integer ids, exact in bf16 up to 256
    wpe[:, 0] = 0
    wpe[:, 1] = np.arange(T) if mode == 0 else np.arange(T) % 128
    wte[:, 1] = 0
    tok = data.token_stream("uniform" if mode == 1 else "zipf", B * T, 72, vocab=V).reshape(B, T)
    x0 = torch.empty(B * T, C, dtype=torch.bfloat16 if mode == 1 else torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpt2_op_encoder_forward(x0, dev(tok), dev(wte, mode), dev(wpe, mode), V, status=status)
    torch.cuda.synchronize()
    got = host(x0).reshape(B, T, C)
    assert np.array_equal(got[..., 0].astype(np.int64), tok)  # bit-exact indexing
    assert np.array_equal(got[..., 1], np.broadcast_to(wpe[:T, 1], (B, T)))
    ref = R.encoder_forward(wte.astype(np.float64), wpe.astype(np.float64), tok)
    if mode == 1:
        ref = data.round_to_bf16(ref.astype(np.float32))
    assert_close(got, ref, 1e-7, what="x0")
    assert int(status.item()) == 0
    tok[1, 5] = V
    gpt2_op_encoder_forward(x0, dev(tok), dev(wte, mode), dev(wpe, mode), V, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1


ENC_BWD_CASES = [(1, "zipf", 4, 300, 768), (0, "zipf", 2, 64, 64), (1, "same", 2, 1024, 128),
                 (1, "zipf", 32, 1024, 768)]


@pytest.mark.parametrize("case", ENC_BWD_CASES)
def test_encoder_backward(torch_cuda, case):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_encoder_backward
    mode, kind, B, T, C = case
    Vp = 50304
    if kind == "same":
        tok = np.full((B, T), 7, dtype=np.int32)
        tok[0, :5] = [3, 7, 7, 9, 7]
    else:
        tok = data.token_stream("zipf", B * T, 80).reshape(B, T)
    dx0 = inputs(81, (B * T, C), 1.0, mode)
    base = data.normal(82, (Vp, C), 1.0)  # dwte already holds the LM-head part
    dwte = dev_f32(base)
    dwpe = torch.full((T, C), float("nan"), device="cuda")
    dtok = dev(tok)
    gpt2_op_encoder_backward(dwte, dwpe, dev(dx0, mode), dtok)
    torch.cuda.synchronize()
    rwte, rwpe = R.encoder_backward(dx0.astype(np.float64).reshape(B, T, C), tok, Vp, T)
    assert_close(host(dwpe), rwpe, 1e-5, atol=1e-5, what="dwpe")
    assert_close(host(dwte), rwte + base, 1e-5, atol=2e-5 * math.sqrt(B * T), what="dwte")
    # deterministic
    dwte2 = dev_f32(base)
    gpt2_op_encoder_backward(dwte2, dwpe, dev(dx0, mode), dtok)
    torch.cuda.synchronize()
    assert torch.equal(dwte, dwte2)


def test_adamw(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_adamw
    n = 40004
    theta = data.normal(90, (n,), 1.0)
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    th = dev_f32(theta)
    pbf = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    rt, rm, rv = theta.astype(np.float64), np.zeros(n), np.zeros(n)
    hp = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    for t in range(1, 4):
        g = data.normal(91 + t, (n,), 1.0)
        g[:10] = 0.0
        gpt2_op_adamw(th, pbf, dev_f32(g), m, v, t=t, **hp)
        rt, rm, rv = R.adamw_update(rt, g.astype(np.float64), rm, rv, hp["lr"], hp["beta1"], hp["beta2"],
                                    hp["eps"], hp["weight_decay"], t)
    torch.cuda.synchronize()
    assert_close(host(th), rt, 1e-6, atol=1e-7, what="theta")
    assert_close(host(m), rm, 1e-5, atol=1e-7, what="m")
    assert_close(host(v), rv, 1e-5, atol=1e-8, what="v")
    # the bf16 copy is the round-to-nearest-even of the fp32 master, bit for bit
    master = th.cpu().numpy()
    assert np.array_equal(host(pbf), data.round_to_bf16(master).astype(np.float64))


# ------------------------------------------------------------------ FP8 linear

@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("n, std", [(8 * 1000 + 5, 1.0), (1 << 20, 0.02), (37, 3.0)])
def test_quantize_fp8_bit_exact(torch_cuda, n, std, fmt):
    """Per-tensor FP8 codes and scales equal the oracle's bit for bit (the
    scale and the scaled value are fp32 on both sides), ragged tails included,
    in both formats."""
    torch = torch_cuda
    from oracle import fp8_ref as F
    from step_gpt_train_gb300.gpt2 import FP8_E4M3, FP8_E5M2, gpt2_op_quantize_fp8
    x = inputs(61, (n,), std)
    x[::97] *= 40.0  # a heavy tail: most values land in subnormal and low-exponent codes
    if fmt == "e5m2":
        x[::1013] *= 1e4  # a wider range still: e5m2 spans 2^-16 .. 57344
    x = inputs_from_f32(x)
    q = torch.full((n,), 0xAA, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(2, dtype=torch.float32, device="cuda")
    gpt2_op_quantize_fp8(q, scales, dev(x), FP8_E4M3 if fmt == "e4m3" else FP8_E5M2)
    torch.cuda.synchronize()
    ref_q, ref_si = F.quantize(x, fmt)
    fmax = np.float32(F.FORMATS[fmt][3])
    s = scales.cpu().numpy()
    assert s[1] == ref_si and s[0] == fmax / np.float32(np.max(np.abs(x)))
    got = q.cpu().numpy()
    bad = np.nonzero(got != ref_q)[0]
    assert bad.size == 0, (bad[:5], got[bad[:5]], ref_q[bad[:5]], x[bad[:5]])


def inputs_from_f32(x):
    from step_gpt_train_gb300 import data
    return data.round_to_bf16(np.asarray(x, dtype=np.float32))


FP8_CASES = [
    # M, N, K, bias, A format, B format
    (300, 200, 272, True, "e4m3", "e4m3"),      # ragged M and N, K not a multiple of the 128-value k-block
    (256, 256, 128, False, "e4m3", "e4m3"),
    (1024, 3072, 768, True, "e4m3", "e4m3"),    # GPT-2 124M MLP up-projection shape (1024 rows)
    (512, 768, 3072, True, "e4m3", "e4m3"),     # MLP down-projection shape
    (300, 200, 272, False, "e5m2", "e4m3"),     # an e5m2 gradient times an e4m3 weight, ragged
    (1024, 3072, 768, False, "e5m2", "e4m3"),   # input gradient of the MLP down-projection: dY [rows, C], W^T [4C, C]
    (256, 392, 400, True, "e4m3", "e5m2"),
    (512, 768, 1024, False, "e5m2", "e5m2"),
]


@pytest.mark.parametrize("case", FP8_CASES)
def test_matmul_fp8(torch_cuda, case):
    """The FP8 product against the oracle on the same codes and scales: exact
    products, fp32 accumulation (the tensor-core bound) and one bf16 rounding;
    and, as a sanity bound, close to the unquantized product (a few percent
    for e4m3's 3 mantissa bits, more for e5m2's 2)."""
    torch = torch_cuda
    from oracle import fp8_ref as F
    from step_gpt_train_gb300.gpt2 import FP8_E4M3, FP8_E5M2, gpt2_op_matmul_fp8, gpt2_op_quantize_fp8
    M, N, K, use_bias, fa, fb = case
    code = {"e4m3": FP8_E4M3, "e5m2": FP8_E5M2}
    A = inputs(71, (M, K), 1.0)
    if fa == "e5m2":
        A[:, ::31] *= 300.0  # gradient-like: a few columns far larger than the rest
    W = inputs(72, (N, K), 0.02)
    bias = inputs(73, (N,), 0.1) if use_bias else None
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    qw = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sa = torch.zeros(2, dtype=torch.float32, device="cuda")
    sw = torch.zeros(2, dtype=torch.float32, device="cuda")
    gpt2_op_quantize_fp8(qa, sa, dev(A), code[fa])
    gpt2_op_quantize_fp8(qw, sw, dev(W), code[fb])
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    gpt2_op_matmul_fp8(D, qa, sa, qw, sw, bias=dev(bias) if use_bias else None, a_fmt=code[fa], b_fmt=code[fb])
    torch.cuda.synchronize()
    got = host(D)
    assert np.all(np.isfinite(got))
    ca, cw = qa.cpu().numpy(), qw.cpu().numpy()
    si_a, si_w = sa.cpu().numpy()[1], sw.cpu().numpy()[1]
    ref = F.matmul_fp8(ca, si_a, cw, si_w, bias, a_fmt=fa, b_fmt=fb)
    # fp32 accumulation over K (one rounding per 32-deep step at most) plus the bf16 output rounding
    atol = (K / 32) * 2.0 ** -23 * 4 * float(np.abs(ref).max()) * 2
    assert_close(got, ref, BF16_REL, atol=atol, atol_frac=1e-3, what="fp8 matmul")
    exact = A.astype(np.float64) @ W.astype(np.float64).T + (bias if use_bias else 0.0)
    assert rel_l2(got, exact) < (0.08 if fa == fb == "e4m3" else 0.15)
    if fa != fb:
        # the formats are honoured: the same codes read as the other pair of formats give another
        # product (where it is finite: e4m3's top codes are infinities and NaNs in e5m2)
        with np.errstate(invalid="ignore", over="ignore"):
            other = F.matmul_fp8(ca, si_a, cw, si_w, bias, a_fmt=fb, b_fmt=fa)
        fin = np.isfinite(other)
        assert fin.mean() > 0.5 and rel_l2(got[fin], other[fin]) > 0.1


def test_fp8_format_checked(torch_cuda):
    """An unknown FP8 format is an argument error, reported before any launch."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import GPT2Error, gpt2_op_matmul_fp8, gpt2_op_quantize_fp8
    q = torch.empty(64, dtype=torch.uint8, device="cuda")
    sc = torch.ones(2, dtype=torch.float32, device="cuda")
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(GPT2Error):
        gpt2_op_quantize_fp8(q, sc, x, 2)
    D = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((16, 32), dtype=torch.uint8, device="cuda")
    with pytest.raises(GPT2Error):
        gpt2_op_matmul_fp8(D, A, sc, A, sc, a_fmt=7)
    with pytest.raises(GPT2Error):
        gpt2_op_matmul_fp8(D, A, sc, A, sc, b_fmt=-1)

