"""The quantizer fused with the preceding RMSNorm (QServe explainer, "运行时设计": activation
quantization fused into the layer norm before the QKV projection and the first FFN layer).

CPU: the oracle's RMSNorm pinned to closed forms. GPU: fmpq_rmsnorm_quantize bit-exact against
the oracle's RMSNorm followed by the oracle's quantizer."""
import math

import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl

TINY_EPS = 2.0 ** -40   # below the rounding unit of the mean square in these pins: ms + eps == ms


# ---------------------------------------------------------------------- oracle pins (CPU)

def test_oracle_rmsnorm_worked_example(oracle_mod):
    """K=128, x = (3, 4, 0, ...), gamma = 1: T = 25, r = sqrt(128)/5, y = fp16(3r), fp16(4r)."""
    x = np.zeros((1, 128), dtype=np.float16)
    x[0, 0], x[0, 1] = 3, 4
    y = oracle_mod.rmsnorm(x, np.ones(128, dtype=np.float16), TINY_EPS)
    r = math.sqrt(128) / 5
    assert y[0, 0] == np.float16(3 * r) == np.float16(6.7890625)
    assert y[0, 1] == np.float16(4 * r) == np.float16(9.0546875)
    assert np.all(y[0, 2:] == 0)


def test_oracle_rmsnorm_constant_row(oracle_mod):
    """Every channel 0.5 (every partial sum exact): mean square 0.25, r = 2, y = gamma."""
    x = np.full((2, 1024), 0.5, dtype=np.float16)
    g = np.linspace(0.25, 2.0, 1024).astype(np.float16)
    y = oracle_mod.rmsnorm(x, g, TINY_EPS)
    assert np.array_equal(y.view(np.uint16), np.broadcast_to(g, (2, 1024)).view(np.uint16))


def test_oracle_rmsnorm_scale_invariance(oracle_mod):
    """x * 4: every partial sum scales by 16 exactly, r by 1/4 exactly, y is unchanged."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((5, 2048)) * 0.5).astype(np.float16)
    g = rng.uniform(0.5, 1.5, 2048).astype(np.float16)
    y1 = oracle_mod.rmsnorm(x, g, TINY_EPS)
    y4 = oracle_mod.rmsnorm((x.astype(np.float32) * 4).astype(np.float16), g, TINY_EPS)
    assert np.array_equal(y1.view(np.uint16), y4.view(np.uint16))


def _exact_sumsq_f32(row):
    """The exact sum of squares of an fp16 row, rounded to fp32 by mpmath at 24-bit precision
    (round to nearest, ties to even). fp16 values times 2^24 are integers, so the sum is the
    exact integer sum of their squares times 2^-48 (Python integers, no rounding)."""
    mpmath = pytest.importorskip("mpmath")
    n = (np.asarray(row, dtype=np.float16).astype(np.float64) * 2.0 ** 24).astype(np.int64)
    total = sum(int(v) * int(v) for v in n)
    with mpmath.workprec(24):
        t = mpmath.ldexp(mpmath.mpf(total), -48)   # mpf() of an int rounds once to 24 bits
    return np.float32(float(t))


def _rows_that_round(K, count, seed):
    """Rows whose squares span a wide range (Laplace bulk, a few large outliers, tiny values)
    so that partial sums round in fp32."""
    rng = np.random.default_rng(seed)
    X = rng.laplace(0.0, 1.0, (count, K)).astype(np.float32)
    X[:, rng.choice(K, K // 10, replace=False)] *= rng.uniform(20, 100, K // 10).astype(np.float32)
    X[:, rng.choice(K, K // 8, replace=False)] *= np.float32(1e-3)
    return X.astype(np.float16)


def test_oracle_rmsnorm_sumsq_is_exact_then_rounded(oracle_mod):
    """T equals the exact sum rounded once (mpmath), on rows where fp32 summation in any fixed
    order visibly rounds: the pin fails for a sequential or a pairwise fp32 sum (both checked
    to differ from the exact result on some of these rows)."""
    for K, count, seed in ((4096, 24, 1), (28672, 6, 2)):
        X = _rows_that_round(K, count, seed)
        T = oracle_mod.rmsnorm_sumsq(X)
        exact = np.array([_exact_sumsq_f32(r) for r in X], dtype=np.float32)
        assert np.array_equal(T.view(np.uint32), exact.view(np.uint32))
        sq = X.astype(np.float32) ** 2                       # exact squares
        sequential = np.cumsum(sq, axis=1, dtype=np.float32)[:, -1]
        pairwise = np.sum(sq, axis=1, dtype=np.float32)
        assert np.any(sequential != exact), "rows too benign: a sequential fp32 sum would pass"
        assert np.any(pairwise != exact), "rows too benign: a pairwise fp32 sum would pass"


def test_oracle_rmsnorm_from_exact_sumsq(oracle_mod):
    """y = fp16(fp32(x) * r * gamma), r = 1/sqrt(T/K + eps), each an IEEE fp32 step (numpy
    float32), from the exactly rounded T."""
    X = _rows_that_round(2048, 8, 3)
    g = np.random.default_rng(4).uniform(0.5, 1.5, 2048).astype(np.float16)
    eps = np.float32(1e-5)
    Y = oracle_mod.rmsnorm(X, g, float(eps))
    for m in range(X.shape[0]):
        t = _exact_sumsq_f32(X[m])
        r = np.float32(1.0) / np.sqrt(t / np.float32(2048) + eps)
        y = ((X[m].astype(np.float32) * r) * g.astype(np.float32)).astype(np.float16)
        assert np.array_equal(Y[m].view(np.uint16), y.view(np.uint16))


def test_oracle_rmsnorm_order_free(oracle_mod):
    """The exact sum does not depend on the channel order: permuting a row's channels leaves T
    unchanged bit for bit."""
    X = _rows_that_round(8192, 4, 5)
    perm = np.random.default_rng(6).permutation(8192)
    assert np.array_equal(oracle_mod.rmsnorm_sumsq(X).view(np.uint32),
                          oracle_mod.rmsnorm_sumsq(X[:, perm]).view(np.uint32))


def test_oracle_rmsnorm_zero_row(oracle_mod):
    x = np.zeros((1, 256), dtype=np.float16)
    y = oracle_mod.rmsnorm(x, np.ones(256, dtype=np.float16), 1e-5)
    assert np.all(y == 0)


# ---------------------------------------------------------------------- GPU parity

@pytest.fixture(scope="module")
def fmpq_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_gemm_fmpq_gb300 import build, fmpq
    build.build()
    fmpq.load_library()
    return fmpq


def _check(fmpq_gpu, oracle_mod, w, gamma, eps, pad=0):
    import torch
    layout = fmpq_gpu.Layout(w.K, w.perm, w.mask)
    big = np.zeros((w.M, w.K + pad), dtype=np.float16)
    big[:, :w.K] = w.X
    Xd = torch.from_numpy(big).cuda()[:, :w.K]
    gperm = torch.from_numpy(np.ascontiguousarray(gamma[w.perm])).cuda()
    A, sx = fmpq_gpu.fmpq_rmsnorm_quantize(layout, Xd, gperm, eps)
    Y = oracle_mod.rmsnorm(w.X, gamma, eps)
    A_ref, sx_ref, _ = oracle_mod.quantize_activations(Y, w.perm, w.mask)
    assert np.array_equal(sx.cpu().numpy().view(np.uint16), sx_ref), "scales differ"
    assert np.array_equal(A.cpu().numpy(), A_ref), "code planes differ"
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.gpu
@pytest.mark.parametrize("M,K,n8,pad", [(1, 128, 0, 0), (16, 512, 1, 8), (300, 4096, 4, 0), (64, 28672, 27, 16)])
def test_rmsnorm_quantize_matches_oracle(fmpq_gpu, oracle_mod, M, K, n8, pad):
    w = wl.synthetic(M, 256, K, n8=n8, seed=M + K, dist="laplace")
    rng = np.random.default_rng(K)
    gamma = rng.uniform(0.5, 1.5, K).astype(np.float16)
    X = w.X.copy()
    if M > 3:
        X[2] = 0                                   # an all-zero token: y = 0
    w.X = X
    _check(fmpq_gpu, oracle_mod, w, gamma, 1e-5, pad)


@pytest.mark.gpu
def test_rmsnorm_quantize_argument_errors(fmpq_gpu):
    import torch
    w = wl.synthetic(8, 256, 256, n8=1, seed=1)
    layout = fmpq_gpu.Layout(w.K, w.perm, w.mask)
    X = torch.from_numpy(w.X).cuda()
    g = torch.ones(w.K, dtype=torch.float16, device="cuda")
    for bad_eps in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(fmpq_gpu.FmpqError):
            fmpq_gpu.fmpq_rmsnorm_quantize(layout, X, g, bad_eps)
    layout.close()
