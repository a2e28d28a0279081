"""Outlier split (QUIK explainer, "第二步: 前向传播"): the base columns through the INT4 path
(a layout selecting them from the full rows), the outlier columns in FP16 (gathered, or split off
by the quantizer in its one pass over the input as in the QUIK explainer's "核融合", then the
library's FP16 tensor-core GEMM added to the output).

CPU: the reference pinned against the full-layout reference. GPU: the selected-layout quantizer
bit-exact against the oracle on the gathered base columns, and its split-off outlier columns
bit-exact against X[:, cols]; the INT4 path's output against its exact value within the output
tolerance; the FP16 outlier product alone, and the merged output (the INT4 output in fp16 plus
the FP16 outlier result, added in fp16 as the pages merge them), against the oracle's exact
product element by element, within the fp16 roundings and the FP32 summation bound."""
import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl

BLOCK = 128


def _problem(M, K_base, n_out, N, seed):
    rng = np.random.default_rng(seed)
    K_in = K_base + n_out
    out_cols = np.sort(rng.choice(K_in, size=n_out, replace=False)).astype(np.int32)
    base_cols = np.setdiff1d(np.arange(K_in), out_cols).astype(np.int32)
    X32 = rng.standard_normal((M, K_in)).astype(np.float32)
    X32[:, out_cols] *= rng.uniform(20.0, 80.0, size=n_out).astype(np.float32)
    W = (rng.standard_normal((N, K_in)) * 0.02).astype(np.float16)
    return X32.astype(np.float16), W, base_cols, out_cols


def test_reference_base_part_is_the_int4_gemm_of_the_base_columns(oracle_mod):
    """With the outlier columns of X zeroed the outlier part is 0, and the base part is the
    full reference of the gathered base problem with every block INT4."""
    X, W, base, out = _problem(24, 256, 16, 64, 3)
    X[:, out] = 0
    yb, yo = oracle_mod.quik_reference(X, W, base, out)
    assert np.all(yo == 0)
    Xb, Wb = np.ascontiguousarray(X[:, base]), np.ascontiguousarray(W[:, base])
    ref = oracle_mod.reference(Xb, Wb, np.arange(base.size, dtype=np.int32), np.zeros(base.size // BLOCK, np.uint8))
    assert np.array_equal(yb, ref["Y"])


def test_reference_outlier_part_selects_the_weight_columns(oracle_mod):
    """Unit outlier activations (token m holds 1 in outlier column m, 0 elsewhere) give back
    the outlier weights: yo[m][n] = W[n][out[m]], exactly, and the base part is 0."""
    X, W, base, out = _problem(16, 256, 16, 48, 5)
    X[:] = 0
    X[np.arange(16), out] = 1.0
    yb, yo = oracle_mod.quik_reference(X, W, base, out)
    assert np.all(yb == 0)
    assert np.array_equal(yo, W[:, out].T.astype(np.float64))


@pytest.fixture(scope="module")
def fmpq_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_gemm_fmpq_gb300 import build, fmpq
    build.build()
    fmpq.load_library()
    return fmpq


def _fp32_sum_bound(X, W, out):
    """A bound on the FP32 accumulation error of the outlier product: each of the n_out
    additions errs by at most 2^-24 of the running magnitude, at most sum_j |x_j w_j|."""
    Xo = np.abs(X[:, out].astype(np.float64))
    Wo = np.abs(W[:, out].astype(np.float64))
    return out.size * 2.0 ** -24 * (Xo @ Wo.T)


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,n_out,presplit", [(256, 512, 128, False), (37, 272, 256, False), (1, 1024, 64, False),
                                                (130, 200, 72, False), (130, 200, 264, True),
                                                (2048, 2560, 192, False), (2048, 2560, 320, True)])
def test_outlier_product_matches_oracle(fmpq_gpu, oracle_mod, M, N, n_out, presplit):
    """The FP16 outlier product alone (Y starts at 0) against the oracle's exact product, element
    by element: one fp16 rounding of the FP32 sum. Ragged M, N and outlier counts that leave
    partial 128-row, 128-column and 64-channel boxes. n_out <= 256 keeps each CTA's W_out rows
    resident across its tiles, more streams them with X_out; the 2048 x 2560 cases give the
    persistent CTAs several tiles each, with ranges that cross into a new W_out panel. presplit:
    the product-only entry point on X[:, cols] given as X_out."""
    import torch
    X, W, base, out = _problem(M, 256, n_out, N, M + 3 * N)
    layout = fmpq_gpu.select_layout(256, 256 + n_out, base, np.zeros(2, np.uint8))
    _, yo = oracle_mod.quik_reference(X, W, base, out)
    Y = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    W_out = torch.from_numpy(np.ascontiguousarray(W[:, out])).cuda()
    if presplit:
        fmpq_gpu.fmpq_outlier_product_fp16(layout, torch.from_numpy(np.ascontiguousarray(X[:, out])).cuda(), W_out, Y)
    else:
        fmpq_gpu.fmpq_outlier_gemm_fp16(layout, torch.from_numpy(X).cuda(), torch.from_numpy(out).cuda(), W_out, Y)
    Yg = Y.cpu().numpy().astype(np.float64)
    half_ulp = 0.5 * np.spacing(np.abs(Yg).astype(np.float16)).astype(np.float64)
    err = np.abs(Yg - yo)
    assert np.all(err <= half_ulp + _fp32_sum_bound(X, W, out)), f"product error {err.max():.3e}"
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.gpu
@pytest.mark.parametrize("M,K_base,n_out,N", [(256, 1024, 128, 512), (37, 512, 256, 272), (1, 384, 64, 1024)])
def test_outlier_split_end_to_end(fmpq_gpu, oracle_mod, M, K_base, n_out, N):
    import torch
    from tests.gpu_helpers import Y_TOL, y_error
    X, W, base, out = _problem(M, K_base, n_out, N, M + N)
    layout = fmpq_gpu.select_layout(K_base, K_base + n_out, base, np.zeros(K_base // BLOCK, np.uint8))
    Xd = torch.from_numpy(X).cuda()
    A, sx = fmpq_gpu.fmpq_quantize(layout, Xd)
    A_ref, sx_ref, _ = oracle_mod.quantize_activations(np.ascontiguousarray(X[:, base]),
                                                      np.arange(K_base, dtype=np.int32), np.zeros(K_base // BLOCK, np.uint8))
    assert np.array_equal(A.cpu().numpy(), A_ref) and np.array_equal(sx.cpu().numpy().view(np.uint16), sx_ref)
    Wp, sw = fmpq_gpu.w4_pack_weights(layout, torch.from_numpy(W).cuda())
    Y = fmpq_gpu.w4ax_gemm(layout, A, sx, Wp, sw, M, N)
    yb, yo = oracle_mod.quik_reference(X, W, base, out)
    # the pages' merge: the INT4 result is brought back to FP16, then the FP16 outlier result is
    # added. Each part is checked against its exact value (cancellation between the parts makes
    # the fp16 rounding of the base part large relative to the merged output).
    Y_base = Y.cpu().numpy()
    err = y_error(Y_base, yb)
    assert err <= Y_TOL, f"INT4 path relative error {err:.3e}"
    cols = torch.from_numpy(out).cuda()
    W_out = torch.from_numpy(np.ascontiguousarray(W[:, out])).cuda()
    fmpq_gpu.fmpq_outlier_gemm_fp16(layout, Xd, cols, W_out, Y)
    # merge, element by element against the oracle's exact outlier product. The pages' order: the
    # FP16 outlier result (the FP32 sum rounded to fp16) is added to the fp16 base output in fp16
    # (one more rounding), so the error is half an fp16 ulp of the result plus half an fp16 ulp of
    # the product (taken one binade up, so that an FP32 sum just above a power of two is covered)
    # plus the FP32 summation bound
    Ym = Y.cpu().numpy().astype(np.float64)
    half_ulp = 0.5 * np.spacing(np.abs(Ym).astype(np.float16)).astype(np.float64)
    prod_half_ulp = 0.5 * np.spacing((np.abs(yo) * (1 + 2.0 ** -9)).astype(np.float16)).astype(np.float64)
    bound = half_ulp + prod_half_ulp + _fp32_sum_bound(X, W, out)
    err = np.abs(Ym - (Y_base.astype(np.float64) + yo))
    assert np.all(err <= bound), f"merge error {err.max():.3e}"
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.gpu
@pytest.mark.parametrize("M,K_base,n_out,asym,n8", [(300, 1024, 128, False, 2), (37, 512, 256, False, 1),
                                                    (5, 384, 264, False, 0), (200, 2048, 136, True, 0),
                                                    (160, 1280, 520, True, 0)])
def test_quantize_split_codes_and_outlier_columns(fmpq_gpu, oracle_mod, M, K_base, n_out, asym, n8):
    """The quantizer with the input split (QUIK explainer, "核融合"): the codes and scales (and
    zero points) are the oracle's for the base columns, bit for bit, and X_out is X[:, cols] bit
    for bit, 0 for an index outside [0, K_in). Fewer tokens than SMs take the per-warp kernel,
    more the row-pipelined one; n_out spans one to three 256-column chunks."""
    import torch
    X, _, base, out = _problem(M, K_base, n_out, 8, 7 * M + n_out)
    K_in = K_base + n_out
    cols = out.copy()
    cols[3], cols[-2] = -1, K_in + 8   # outside the row: read as 0
    mask = np.zeros(K_base // BLOCK, np.uint8)
    mask[K_base // BLOCK - n8:] = 1
    layout = fmpq_gpu.select_layout(K_base, K_in, base, mask)
    A, sx, z, X_out = fmpq_gpu.fmpq_quantize_split(layout, torch.from_numpy(X).cuda(), torch.from_numpy(cols).cuda(),
                                                   asym=asym)
    Xb = np.ascontiguousarray(X[:, base])
    if asym:
        A_ref, sx_ref, z_ref, _ = oracle_mod.quantize_activations_asym(Xb, np.arange(K_base, dtype=np.int32))
        assert np.array_equal(z.cpu().numpy().view(np.uint16), z_ref)
    else:
        A_ref, sx_ref, _ = oracle_mod.quantize_activations(Xb, np.arange(K_base, dtype=np.int32), mask)
    assert np.array_equal(A.cpu().numpy(), A_ref) and np.array_equal(sx.cpu().numpy().view(np.uint16), sx_ref)
    expect = np.where((cols >= 0) & (cols < K_in), X[:, np.clip(cols, 0, K_in - 1)], np.float16(0))
    assert np.array_equal(X_out.cpu().numpy().view(np.uint16), expect.view(np.uint16))
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.gpu
@pytest.mark.parametrize("M,K_base,n_out,N", [(256, 1024, 128, 512), (9, 512, 264, 272)])
def test_outlier_split_fused_path(fmpq_gpu, oracle_mod, M, K_base, n_out, N):
    """The QUIK forward pass with the split fused into the quantizer: quantize + split, INT4 GEMM,
    FP16 product on the split columns added in fp16. The merged output against the oracle's
    exact parts within the fp16 roundings and the FP32 summation bound; the merged output equals
    the unfused path's (gather kernel) bit for bit."""
    import torch
    from tests.gpu_helpers import Y_TOL, y_error
    X, W, base, out = _problem(M, K_base, n_out, N, 11 * M + N)
    layout = fmpq_gpu.select_layout(K_base, K_base + n_out, base, np.zeros(K_base // BLOCK, np.uint8))
    Xd, cols = torch.from_numpy(X).cuda(), torch.from_numpy(out).cuda()
    A, sx, _, X_out = fmpq_gpu.fmpq_quantize_split(layout, Xd, cols)
    Wp, sw = fmpq_gpu.w4_pack_weights(layout, torch.from_numpy(W).cuda())
    Y = fmpq_gpu.w4ax_gemm(layout, A, sx, Wp, sw, M, N)
    Y_base = Y.cpu().numpy().astype(np.float64)
    Y2 = Y.clone()
    W_out = torch.from_numpy(np.ascontiguousarray(W[:, out])).cuda()
    fmpq_gpu.fmpq_outlier_product_fp16(layout, X_out, W_out, Y)
    fmpq_gpu.fmpq_outlier_gemm_fp16(layout, Xd, cols, W_out, Y2)
    yb, yo = oracle_mod.quik_reference(X, W, base, out)
    assert y_error(Y_base, yb) <= Y_TOL
    Ym = Y.cpu().numpy().astype(np.float64)
    bound = (0.5 * np.spacing(np.abs(Ym).astype(np.float16)).astype(np.float64)
             + 0.5 * np.spacing((np.abs(yo) * (1 + 2.0 ** -9)).astype(np.float16)).astype(np.float64)
             + _fp32_sum_bound(X, W, out))
    err = np.abs(Ym - (Y_base + yo))
    assert np.all(err <= bound), f"merge error {err.max():.3e}"
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.gpu
def test_outlier_split_argument_errors(fmpq_gpu):
    import torch
    X = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    Y = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    W_out = torch.zeros((64, 16), dtype=torch.float16, device="cuda")
    layout = fmpq_gpu.select_layout(128, 256, np.arange(128, dtype=np.int32), np.zeros(1, np.uint8))
    with pytest.raises(fmpq_gpu.FmpqError):       # 12 outlier columns: not a multiple of 8
        fmpq_gpu.fmpq_outlier_gemm_fp16(layout, X, torch.zeros(12, dtype=torch.int32, device="cuda"), W_out, Y)
    with pytest.raises(fmpq_gpu.FmpqError):       # the same for the split quantizer
        fmpq_gpu.fmpq_quantize_split(layout, X, torch.zeros(12, dtype=torch.int32, device="cuda"))
    with pytest.raises(fmpq_gpu.FmpqError):       # the product alone: 12 columns, not a multiple of 8
        fmpq_gpu.fmpq_outlier_product_fp16(layout, torch.zeros((4, 12), dtype=torch.float16, device="cuda"),
                                           torch.zeros((64, 12), dtype=torch.float16, device="cuda"), Y)
    layout.close()
    with pytest.raises(fmpq_gpu.FmpqError):       # a selection with a repeated channel
        fmpq_gpu.select_layout(128, 256, np.zeros(128, np.int32), np.zeros(1, np.uint8))
