"""Offline layout derivation from calibration activations (COMET news article, section 1:
the outliers sit in about 10% of the channels and a permutation gathers them into the same
blocks; QUIK explainer, "第一步: 识别与重排": outlier columns found offline and moved to the end).

CPU: the oracle pinned to worked examples and invariants, and the library's host planner
(C ABI, no GPU needed) bit-exact against the oracle. GPU: the channel-absmax kernel bit-exact
against the oracle, and an end-to-end run: calibrate, plan, quantize and GEMM with the derived
layout against the oracle."""
import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl

BLOCK = 128


# ---------------------------------------------------------------------- error budget (CPU)

def _calib_batch(T, K, seed):
    """Laplace tokens with 10% outlier channels (x U(20, 100)), the workloads' statistics."""
    rng = np.random.default_rng(seed)
    X = rng.laplace(0.0, 1.0, (T, K)).astype(np.float32)
    cols = rng.choice(K, K // 10, replace=False)
    X[:, cols] *= rng.uniform(20.0, 100.0, cols.size).astype(np.float32)
    return X.astype(np.float16)


def test_oracle_layout_error_closed_form(oracle_mod):
    """A block of ones: s = fp16(1/7) = 585 * 2^-12, so every code is 1 and x - q*s = 2^-12
    (INT4); s = fp16(1/127) = 1032 * 2^-17 gives 2^-14 (INT8). The relative error of the token
    is that difference, exactly."""
    s4 = np.float16(np.float32(1) / np.float32(7))
    s8 = np.float16(np.float32(1) / np.float32(127))
    assert 1.0 - 7 * float(s4) == 2.0 ** -12 and 1.0 - 127 * float(s8) == 2.0 ** -14
    X = np.ones((3, 128), dtype=np.float16)
    ident = np.arange(128, dtype=np.int32)
    assert oracle_mod.layout_error(X, ident, np.array([0], np.uint8)) == 2.0 ** -12
    assert oracle_mod.layout_error(X, ident, np.array([1], np.uint8)) == 2.0 ** -14
    X[1] = 0                                             # an all-zero token counts as 0
    assert oracle_mod.layout_error(X, ident, np.array([0], np.uint8)) == 2.0 ** -12


def test_oracle_layout_error_exact_codes(oracle_mod):
    """Tokens whose blocks hold integers in [-7, 7] with a 7 in each block are represented
    exactly by INT4 codes (s = 1): the error is 0 and the planner takes no INT8 block even for
    eps = 0."""
    rng = np.random.default_rng(3)
    X = rng.integers(-7, 8, size=(5, 512)).astype(np.float16)
    X[:, ::BLOCK] = 7
    ident = np.arange(512, dtype=np.int32)
    assert oracle_mod.layout_error(X, ident, np.zeros(4, np.uint8)) == 0.0
    stat = oracle_mod.channel_absmax(X)
    n8, err, perm, mask = oracle_mod.plan_layout_budget(stat, X, 0.0)
    assert (n8, err) == (0, 0.0) and perm.tolist() == list(range(512))


def test_oracle_layout_error_against_numpy(oracle_mod):
    """The error equals the ratio of norms computed in numpy from the oracle quantizer's codes
    and scales (dequantized q * s, fp64 norms), within fp64 summation error."""
    X = _calib_batch(12, 2048, 4)
    stat = oracle_mod.channel_absmax(X)
    perm, mask = oracle_mod.plan_layout(stat, 2)
    _, sx, Aq = oracle_mod.quantize_activations(X, perm, mask)
    s = sx.view(np.float16).astype(np.float64)                 # [nb][T]
    xhat = Aq.astype(np.float64) * np.repeat(s.T, BLOCK, axis=1)
    xp = X[:, perm].astype(np.float64)
    want = np.max(np.linalg.norm(xp - xhat, axis=1) / np.linalg.norm(xp, axis=1))
    assert abs(oracle_mod.layout_error(X, perm, mask) - want) <= 1e-12 * want


def test_oracle_budget_decisions(oracle_mod):
    """One block of ones: errors 2^-12 (INT4) and 2^-14 (INT8). A budget of 2^-13 needs the INT8
    block; 2^-12 does not; 2^-15 cannot be met, so every block is INT8 and err > eps."""
    X = np.ones((2, 128), dtype=np.float16)
    stat = oracle_mod.channel_absmax(X)
    assert oracle_mod.plan_layout_budget(stat, X, 2.0 ** -13)[:2] == (1, 2.0 ** -14)
    assert oracle_mod.plan_layout_budget(stat, X, 2.0 ** -12)[:2] == (0, 2.0 ** -12)
    assert oracle_mod.plan_layout_budget(stat, X, 2.0 ** -15)[:2] == (1, 2.0 ** -14)


@pytest.mark.parametrize("eps", [0.02, 0.05, 0.1])
def test_oracle_budget_is_the_smallest(oracle_mod, eps):
    """Brute force: the chosen n8 meets the budget and n8 - 1 does not."""
    X = _calib_batch(16, 2048, 5)
    stat = oracle_mod.channel_absmax(X)
    n8, err, perm, mask = oracle_mod.plan_layout_budget(stat, X, eps)
    assert err <= eps and err == oracle_mod.layout_error(X, perm, mask)
    assert np.array_equal(oracle_mod.plan_layout(stat, n8)[0], perm)
    if n8 > 0:
        p0, m0 = oracle_mod.plan_layout(stat, n8 - 1)
        assert oracle_mod.layout_error(X, p0, m0) > eps


@pytest.mark.parametrize("T,K,eps", [(32, 8192, 0.03), (32, 8192, 0.06), (8, 4096, 0.0), (64, 1024, 0.08)])
def test_library_budget_planner_matches_oracle(T, K, eps, oracle_mod):
    """The library's host planner (C ABI, no GPU needed) bit-exact against the oracle: n8, the
    error (the same fp64 value), the permutation and the mask."""
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    fmpq.load_library()
    X = _calib_batch(T, K, T + K)
    stat = oracle_mod.channel_absmax(X)
    want = oracle_mod.plan_layout_budget(stat, X, eps)
    got = fmpq.fmpq_plan_layout_budget(stat, X, eps)
    assert got[:2] == want[:2]
    assert np.array_equal(got[2], want[2]) and np.array_equal(got[3], want[3])


def test_library_budget_planner_closed_form():
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    fmpq.load_library()
    X = np.ones((2, 128), dtype=np.float16)
    stat = np.full(128, 0x3C00, dtype=np.uint32)
    assert fmpq.fmpq_plan_layout_budget(stat, X, 2.0 ** -13)[:2] == (1, 2.0 ** -14)
    assert fmpq.fmpq_plan_layout_budget(stat, X, 2.0 ** -12)[:2] == (0, 2.0 ** -12)
    with pytest.raises(fmpq.FmpqError):
        fmpq.fmpq_plan_layout_budget(stat, X, -1.0)


# ---------------------------------------------------------------------- oracle pins (CPU)

def test_oracle_absmax_planted_maxima(oracle_mod):
    """Each column's maximum magnitude is planted at a known row, sign included."""
    rng = np.random.default_rng(1)
    T, K = 37, 256
    X = rng.uniform(-1.0, 1.0, size=(T, K)).astype(np.float16)
    want = rng.uniform(2.0, 9.0, size=K).astype(np.float16)
    rows = rng.integers(0, T, size=K)
    signs = np.where(rng.integers(0, 2, size=K) == 1, -1, 1).astype(np.float16)
    X[rows, np.arange(K)] = want * signs
    assert np.array_equal(oracle_mod.channel_absmax(X), want.view(np.uint16))


def test_oracle_plan_worked_example(oracle_mod):
    """K=256, two large channels (130 above 7), the rest equal: the ranking is 130, 7, then
    channels by index, so block 1 (INT8) holds 130, 7, 0..6, 8..126 and block 0 holds
    127..255 without 130, in order."""
    stat = np.ones(256, dtype=np.uint32)
    stat[7], stat[130] = 50, 60
    perm, mask = oracle_mod.plan_layout(stat, 1)
    top = [130, 7] + list(range(0, 7)) + list(range(8, 127))
    rest = [c for c in range(127, 256) if c != 130]
    assert len(top) == 128 and len(rest) == 128
    assert perm.tolist() == rest + top
    assert mask.tolist() == [0, 1]


def test_oracle_plan_boundaries(oracle_mod):
    rng = np.random.default_rng(2)
    stat = rng.integers(0, 1000, size=512).astype(np.uint32)
    perm, mask = oracle_mod.plan_layout(stat, 0)
    assert perm.tolist() == list(range(512)) and mask.tolist() == [0] * 4      # no INT8 block: identity
    perm, mask = oracle_mod.plan_layout(stat, 4)
    ranking = sorted(range(512), key=lambda c: (-int(stat[c]), c))
    assert perm.tolist() == ranking and mask.tolist() == [1] * 4               # all INT8: the ranking


@pytest.mark.parametrize("n8", [1, 3, 7])
def test_oracle_plan_invariants(oracle_mod, n8):
    rng = np.random.default_rng(n8)
    K = 1024
    stat = rng.integers(0, 50, size=K).astype(np.uint32)       # many ties
    perm, mask = oracle_mod.plan_layout(stat, n8)
    assert sorted(perm.tolist()) == list(range(K))
    cut = K - BLOCK * n8
    assert mask.tolist() == [0] * (K // BLOCK - n8) + [1] * n8
    assert stat[perm[cut:]].min() >= stat[perm[:cut]].max()    # INT8 blocks hold the largest
    assert np.all(np.diff(perm[:cut]) > 0)                     # INT4 part keeps channel order
    top = perm[cut:]
    assert all((stat[a] > stat[b]) or (stat[a] == stat[b] and a < b) for a, b in zip(top[:-1], top[1:]))


def test_oracle_outlier_blocks(oracle_mod):
    assert oracle_mod.outlier_blocks(28672, 0.10) == 23     # 2867 channels -> 23 blocks
    assert oracle_mod.outlier_blocks(4096, 0.10) == 4       # 410 -> 4
    assert oracle_mod.outlier_blocks(256, 0.0) == 0
    assert oracle_mod.outlier_blocks(256, 1.0) == 2
    assert oracle_mod.outlier_blocks(1280, 0.1) == 1        # 128 exactly -> 1
    assert oracle_mod.outlier_blocks(256, 0.5 / 256) == 1   # round(0.5) = 1 (half away from zero)


# ---------------------------------------------------------------------- library host planner (CPU)

def test_library_planner_matches_oracle(oracle_mod):
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    rng = np.random.default_rng(7)
    for K, n8, hi in [(128, 0, 5), (128, 1, 5), (4096, 4, 3), (8192, 8, 1000), (28672, 23, 0x7C00), (32768, 256, 2)]:
        stat = rng.integers(0, hi, size=K).astype(np.uint32)
        got = fmpq.fmpq_plan_layout(stat, n8)
        want = oracle_mod.plan_layout(stat, n8)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]), (K, n8)


def test_library_outlier_blocks_matches_oracle(oracle_mod):
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    for K in (128, 256, 4096, 8192, 28672, 32768):
        for f in (0.0, 0.01, 0.05, 0.1, 0.125, 0.2, 0.5, 0.99, 1.0, 64.5 / K, 127.5 / K):
            assert fmpq.fmpq_outlier_blocks(K, f) == oracle_mod.outlier_blocks(K, f), (K, f)
    with pytest.raises(ValueError):
        fmpq.fmpq_outlier_blocks(100, 0.1)
    with pytest.raises(ValueError):
        fmpq.fmpq_outlier_blocks(256, 1.5)


def test_library_planner_argument_errors():
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    with pytest.raises(fmpq.FmpqError):
        fmpq.fmpq_plan_layout(np.zeros(256, dtype=np.uint32), 3)     # more INT8 blocks than blocks
    with pytest.raises(fmpq.FmpqError):
        fmpq.fmpq_plan_layout(np.zeros(200, dtype=np.uint32), 0)     # K % 128


# ---------------------------------------------------------------------- GPU

@pytest.fixture(scope="module")
def fmpq_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_gemm_fmpq_gb300 import build, fmpq
    build.build()
    fmpq.load_library()
    return fmpq


@pytest.mark.gpu
@pytest.mark.parametrize("T,K,pad", [(1, 128, 0), (3, 256, 8), (300, 1024, 24), (1000, 4096, 0), (64, 28672, 16)])
def test_channel_absmax_kernel(fmpq_gpu, oracle_mod, T, K, pad):
    import torch
    rng = np.random.default_rng(T + K)
    X = (rng.standard_normal((T, K)) * rng.uniform(0.1, 50.0, size=K)).astype(np.float16)
    X[:, rng.integers(0, K, size=3)] = 0                          # zero channels
    big = np.zeros((T, K + pad), dtype=np.float16)
    big[:, :K] = X
    Xd = torch.from_numpy(big).cuda()[:, :K]
    got = fmpq_gpu.fmpq_channel_absmax(Xd).cpu().numpy().astype(np.uint32)
    assert np.array_equal(got, oracle_mod.channel_absmax(X).astype(np.uint32))


@pytest.mark.gpu
def test_calibrated_layout_end_to_end(fmpq_gpu, oracle_mod):
    """Outlier channels at unknown positions: calibrate on the first tokens, plan the layout
    (10% outliers), check that every outlier channel lands in an INT8 block, then quantize and
    run the GEMM with that layout against the oracle."""
    import torch
    from tests.gpu_helpers import Y_TOL, run_gpu, y_error
    M, N, K = 384, 512, 2048
    rng = np.random.default_rng(11)
    outliers = np.sort(rng.choice(K, size=int(0.1 * K), replace=False))
    X32 = rng.standard_normal((M, K)).astype(np.float32)
    X32[:, outliers] *= rng.uniform(20.0, 100.0, size=outliers.size).astype(np.float32)
    X = X32.astype(np.float16)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    stat = fmpq_gpu.fmpq_channel_absmax(torch.from_numpy(X[:128]).cuda()).cpu().numpy().astype(np.uint32)
    n8 = fmpq_gpu.fmpq_outlier_blocks(K, 0.10)
    perm, mask = fmpq_gpu.fmpq_plan_layout(stat, n8)
    assert n8 == 2
    int8_channels = set(perm[K - BLOCK * n8:].tolist())
    assert set(outliers.tolist()) <= int8_channels
    layout = fmpq_gpu.Layout(K, perm, mask)
    got, _ = run_gpu(layout, X, W)
    ref = oracle_mod.reference(X, W, perm, mask)
    assert np.array_equal(got["A"], ref["A_packed"])
    assert y_error(got["Y"], ref["Y"]) <= Y_TOL
    layout.close()
