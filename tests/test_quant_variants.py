"""Quantization variants beside FMPQ's symmetric blocks.

- QUIK asymmetric activations (QUIK explainer, "反量化背后的数学"): activations take a scale and
  a zero point, weights a scale only, and the zero point's term needs only the weights' sums,
  precomputed offline.
- QoQ progressive group quantization (QServe explainer, "渐进式分组量化"): per-channel INT8
  weights in the protective range [-119, 119], then per-group asymmetric UINT4; W4A8 with
  per-token INT8 activations ("运行时设计"), the group zero point subtracted after the
  multiplication ("W4A8逐组快速反量化").

CPU: the oracle pinned to worked examples, closed forms, invariants and an exhaustive check of
the protective range. GPU: the library's kernels bit-exact against the oracle (codes, scales,
zero points, sums, partial sums) and Y within the output tolerance.
"""
import numpy as np
import pytest

BLOCK = 128


def f16(v):
    return np.asarray(v, dtype=np.float16)


# ---------------------------------------------------------------------- QUIK asymmetric: oracle pins

def test_asym_worked_example(oracle_mod):
    """min -1, max 14: s = fp16(15 / 15) = 1, z = -1; (x - z) / s = x + 1 rounded half to even."""
    x = np.zeros((1, BLOCK), dtype=np.float16)
    vals = {0: -1.0, 1: 14.0, 2: 0.5, 3: 1.5, 4: 2.5, 5: -0.5, 6: 3.25}
    for j, v in vals.items():
        x[0, j] = v
    A, s, z, Aq = oracle_mod.quantize_activations_asym(x, np.arange(BLOCK, dtype=np.int32))
    assert s[0, 0] == f16(1.0).view(np.uint16)
    assert z[0, 0] == f16(-1.0).view(np.uint16)
    want = {0: 0, 1: 15, 2: 2, 3: 2, 4: 4, 5: 0, 6: 4}     # 1.5 -> 2, 2.5 -> 2, 3.5 -> 4, 0.5 -> 0, 4.25 -> 4
    for j, q in want.items():
        assert Aq[0, j] == q, (j, Aq[0, j], q)
    assert np.all(Aq[0, 7:] == 1)                           # x = 0 -> 1
    # packed: one plane, byte = E4M3 of q * 2^-9 with the sign bit clear; row 0 is unrotated
    for j in range(BLOCK):
        assert oracle_mod.e4m3_value(int(A[j])) == Aq[0, j] * 2.0 ** -9


def test_asym_constant_and_signed_zero_blocks(oracle_mod):
    x = np.full((2, 2 * BLOCK), 3.0, dtype=np.float16)
    x[1, :BLOCK] = 0.0
    x[1, 5] = -0.0                                          # -0 orders below +0: it is the zero point
    A, s, z, Aq = oracle_mod.quantize_activations_asym(x, np.arange(2 * BLOCK, dtype=np.int32))
    assert np.all(s == 0) and np.all(Aq == 0)
    assert z[0, 0] == f16(3.0).view(np.uint16) and z[1, 0] == f16(3.0).view(np.uint16)
    assert z[0, 1] == np.uint16(0x8000)


@pytest.mark.parametrize("dist", ["normal", "positive", "outliers"])
def test_asym_invariants(oracle_mod, dist):
    """Per block: codes in [0, 15]; the minimum maps to 0 and the maximum to 15 (normal scale);
    |x - (z + q s)| <= s / 2 up to the fp32 roundings of the difference and the quotient."""
    rng = np.random.default_rng(5)
    M, K = 16, 1024
    if dist == "normal":
        x = rng.standard_normal((M, K))
    elif dist == "positive":
        x = rng.uniform(2.0, 3.0, (M, K))                   # far from zero: the zero point matters
    else:
        x = rng.standard_normal((M, K))
        x[:, rng.integers(0, K, 20)] *= 60.0
    X = x.astype(np.float16)
    perm = rng.permutation(K).astype(np.int32)
    _, s, z, Aq = oracle_mod.quantize_activations_asym(X, perm)
    Xp = X[:, perm].astype(np.float64)
    sv = oracle_mod.f16_bits_to_f32(s).reshape(s.shape).astype(np.float64)
    zv = oracle_mod.f16_bits_to_f32(z).reshape(z.shape).astype(np.float64)
    for b in range(K // BLOCK):
        blk = Xp[:, b * BLOCK:(b + 1) * BLOCK]
        q = Aq[:, b * BLOCK:(b + 1) * BLOCK].astype(np.float64)
        assert q.min() >= 0 and q.max() <= 15
        assert np.array_equal(zv[b], blk.min(axis=1))
        rows = np.arange(M)
        assert np.all(q[rows, blk.argmin(axis=1)] == 0)
        assert np.all(q[rows, blk.argmax(axis=1)] == 15)
        err = np.abs(blk - (zv[b][:, None] + q * sv[b][:, None]))
        assert np.all(err <= 0.5 * sv[b][:, None] * (1 + 1e-5) + 1e-6 * np.abs(blk - zv[b][:, None]))


def test_asym_scale_invariance(oracle_mod):
    """X * 2^k: scale and zero point scale by 2^k exactly, the codes are unchanged."""
    rng = np.random.default_rng(8)
    X = (rng.standard_normal((8, 512)) * 0.5).astype(np.float16)
    perm = rng.permutation(512).astype(np.int32)
    _, s1, z1, q1 = oracle_mod.quantize_activations_asym(X, perm)
    X8 = (X.astype(np.float32) * 8).astype(np.float16)
    _, s8, z8, q8 = oracle_mod.quantize_activations_asym(X8, perm)
    assert np.array_equal(q1, q8)
    f = lambda h: oracle_mod.f16_bits_to_f32(h).reshape(h.shape)
    assert np.array_equal(f(s1) * 8, f(s8)) and np.array_equal(f(z1) * 8, f(z8))


def test_asym_epilogue_closed_form(oracle_mod):
    """The epilogue with the offline weight sums equals dequantize-then-multiply:
    sum_k (s_x q_x + z) (s_w q_w), evaluated in fp64."""
    rng = np.random.default_rng(9)
    M, N, K = 6, 10, 512
    X = (rng.standard_normal((M, K)) + 1.5).astype(np.float16)
    W = (rng.standard_normal((N, K)) * 0.03).astype(np.float16)
    perm = rng.permutation(K).astype(np.int32)
    r = oracle_mod.asym_reference(X, W, perm)
    f = lambda h: oracle_mod.f16_bits_to_f32(h).reshape(h.shape).astype(np.float64)
    sx, z, sw = f(r["a_scales"]), f(r["a_zeros"]), f(r["w_scales"])
    blk = np.arange(K) // BLOCK
    Xd = r["Aq"].astype(np.float64) * sx[blk, :].T + z[blk, :].T
    Wd = r["Wq"].astype(np.float64) * sw[blk, :].T
    Y = Xd @ Wd.T
    assert np.allclose(r["Y"], Y, rtol=1e-12, atol=1e-12 * np.abs(Y).max())
    # the weight sums are the block sums of the dequantized weights
    assert np.array_equal(r["wsum"].astype(np.float64), Wd.reshape(N, K // BLOCK, BLOCK).sum(axis=2).T)


# ---------------------------------------------------------------------- QoQ: oracle pins

def test_qoq_group_worked_examples(oracle_mod):
    """Range [-119, 119]: s2 = ceil(238 / 15) = 16, z2 = rne(119 / 16 = 7.4375) = 7."""
    g = np.zeros(BLOCK, dtype=np.int8)
    g[:7] = [-119, 119, 8, 24, -8, -24, 40]
    s2, z2, q4 = oracle_mod.qoq_group(g)
    assert s2[0] == 16 and z2[0] == 7
    # q8 / 16 rounded half to even, plus 7: 119 -> 7 + 7, 8 -> 0.5 -> 0, 24 -> 1.5 -> 2,
    # -8 -> -0.5 -> 0, -24 -> -1.5 -> -2, 40 -> 2.5 -> 2
    assert q4[0, :7].tolist() == [0, 14, 7, 9, 7, 5, 9]
    assert np.all(q4[0, 7:] == 7)
    # a positive group: the range is extended to 0, so z2 = 0 and 0 stays exact
    g = np.full(BLOCK, 3, dtype=np.int8)
    g[0] = 40
    s2, z2, q4 = oracle_mod.qoq_group(g)
    assert s2[0] == 3 and z2[0] == 0 and q4[0, 0] == 13 and q4[0, 1] == 1
    # all zero: s2 = 1, z2 = 0
    s2, z2, q4 = oracle_mod.qoq_group(np.zeros(BLOCK, dtype=np.int8))
    assert s2[0] == 1 and z2[0] == 0 and np.all(q4 == 0)


def test_qoq_protective_range_exhaustive(oracle_mod):
    """For every group range [mn, mx] inside [-119, 119] and every INT8 value in it, the code is
    in [0, 15] and the dequantized (q4 - z2) * s2 is in [-127, 127] (the protective range's
    purpose), within s2 of the INT8 value."""
    lo, hi = np.meshgrid(np.arange(-119, 120), np.arange(-119, 120), indexing="ij")
    sel = lo <= hi
    lo, hi = lo[sel], hi[sel]
    G = lo.size
    # fill each group with mn, mx and values spread over [mn, mx]; two offsets of the fill
    # cover every value of ranges wider than the group
    for phase in range(2):
        t = (np.arange(BLOCK - 2)[None, :] * 2 + phase) / (2 * (BLOCK - 2) - 1)
        fill = np.rint(lo[:, None] + t * (hi - lo)[:, None]).astype(np.int64)
        q8 = np.concatenate([lo[:, None], hi[:, None], fill], axis=1).astype(np.int8)
        s2, z2, q4 = oracle_mod.qoq_group(q8)
        deq = (q4.astype(np.int64) - z2[:, None]) * s2[:, None]
        assert q4.max() <= 15
        assert np.abs(deq).max() <= 127
        assert np.all(np.abs(deq - q8) <= s2[:, None])
        assert s2.max() == 16
    # every value of [-119, 119] occurs in some group of the sweep
    assert G == 239 * 240 // 2


def test_qoq_weight_rule_worked_example(oracle_mod):
    """Row absmax 119 -> s1 = 1, q8 = rne(w) (ties to even), then the group rule."""
    W = np.zeros((1, BLOCK), dtype=np.float16)
    W[0, :5] = [119.0, -2.5, 3.5, 0.5, -60.0]
    r = oracle_mod.qoq_quantize_weights(W, np.arange(BLOCK, dtype=np.int32))
    assert r["s1"][0] == f16(1.0).view(np.uint16)
    assert r["q8"][0, :5].tolist() == [119, -2, 4, 0, -60]
    s2, z2, q4 = oracle_mod.qoq_group(r["q8"][0])
    assert r["s2"][0, 0] == s2[0] and r["z2"][0, 0] == z2[0] and np.array_equal(r["q4"][0], q4[0])


def test_qoq_activation_worked_example(oracle_mod):
    """Per-token scale from the row's absmax (127 -> s = 1), codes rne(x), block sums."""
    X = np.zeros((1, 2 * BLOCK), dtype=np.float16)
    X[0, 0], X[0, 1], X[0, 130], X[0, 131] = 127.0, 2.5, -3.5, 1.5
    A, s, sums, Aq = oracle_mod.qoq_quantize_activations(X, np.arange(2 * BLOCK, dtype=np.int32))
    assert s[0] == f16(1.0).view(np.uint16)
    assert Aq[0, 0] == 127 and Aq[0, 1] == 2 and Aq[0, 130] == -4 and Aq[0, 131] == 2
    assert sums[:, 0].tolist() == [129, -2]
    # every block is packed as an INT8 block (two planes)
    assert np.array_equal(oracle_mod.unpack_activations(A, np.ones(2, np.uint8), 1, 2 * BLOCK), Aq)


def test_qoq_epilogue_closed_form(oracle_mod):
    """Zero point subtracted after the multiplication == dequantize-then-multiply in fp64:
    sum_k (s_x q_x) (s1 s2 (q4 - z2))."""
    rng = np.random.default_rng(12)
    M, N, K = 5, 9, 512
    X = rng.standard_normal((M, K)).astype(np.float16)
    W = (rng.standard_normal((N, K)) * 0.03 + 0.01).astype(np.float16)
    perm = rng.permutation(K).astype(np.int32)
    r = oracle_mod.qoq_reference(X, W, perm)
    f = lambda h: oracle_mod.f16_bits_to_f32(h).reshape(h.shape).astype(np.float64)
    blk = np.arange(K) // BLOCK
    Xd = r["Aq"].astype(np.float64) * f(r["a_scales"])[:, None]
    Wd = ((r["q4"].astype(np.float64) - r["z2"][blk, :].T) * r["s2"][blk, :].T) * f(r["s1"])[:, None]
    Y = Xd @ Wd.T
    assert np.allclose(r["Y"], Y, rtol=1e-12, atol=1e-12 * np.abs(Y).max())
    # the INT8 intermediate is reproduced by the group codes within s2 / 2 except where clipped
    deq8 = (r["q4"].astype(np.int64) - r["z2"][blk, :].T) * r["s2"][blk, :].T
    assert np.all(np.abs(deq8 - r["q8"]) <= r["s2"][blk, :].T)


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


def _inputs(M, N, K, seed, offset=0.0, pad=0):
    """Seeded activations (normal, 10% outlier channels x U(20, 100), optional offset) with a
    row stride of K + pad, and weights; row 0 holds the asymmetric worked example's block."""
    from bit_quantized_gemm_fmpq_gb300 import workloads as wl
    w = wl.synthetic(M, N, K, n8=0, seed=seed, outlier_frac=0.0)
    rng = np.random.default_rng(seed + 7)
    X = w.X.astype(np.float32) + offset
    X[:, rng.choice(K, size=max(1, K // 10), replace=False)] *= rng.uniform(20, 100)
    X = X.astype(np.float16)
    ex = np.zeros(BLOCK, dtype=np.float16)
    ex[:7] = [-1.0, 14.0, 0.5, 1.5, 2.5, -0.5, 3.25]      # exact ties of (x - z) / s
    X[0, w.perm[:BLOCK]] = ex
    big = np.zeros((M, K + pad), dtype=np.float16)
    big[:, :K] = X
    return X, big, w.W, w.perm


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,offset,pad", [(1, 256, 128, 0.0, 0), (37, 512, 1024, 0.0, 8),
                                              (300, 768, 4096, 2.0, 0), (1024, 1024, 8192, 0.0, 16)])
def test_asym_matches_oracle(fmpq_gpu, oracle_mod, M, N, K, offset, pad):
    from tests.gpu_helpers import Y_TOL, to_dev, y_error
    X, big, W, perm = _inputs(M, N, K, seed=M + K, offset=offset, pad=pad)
    layout = fmpq_gpu.Layout(K, perm, np.zeros(K // BLOCK, np.uint8))
    Xd = to_dev(big)[:, :K]
    A, sx, z = fmpq_gpu.fmpq_quantize_asym(layout, Xd)
    Wp, sw = fmpq_gpu.w4_pack_weights(layout, to_dev(W))
    wsum = fmpq_gpu.w4_weight_sums(layout, Wp, sw, N)
    Y = fmpq_gpu.w4ax_gemm_asym(layout, A, sx, z, Wp, sw, wsum, M, N)
    mc, nc = min(M, 48), min(N, 64)
    m0, n0 = M - mc, N - nc
    P = fmpq_gpu.w4ax_gemm_partials(layout, A, Wp, M, N, m0, mc, n0, nc)
    ref = oracle_mod.asym_reference(X, W, perm)
    assert np.array_equal(sx.cpu().numpy().view(np.uint16), ref["a_scales"]), "scales differ"
    assert np.array_equal(z.cpu().numpy().view(np.uint16), ref["a_zeros"]), "zero points differ"
    assert np.array_equal(A.cpu().numpy(), ref["A_packed"]), "codes differ"
    assert np.array_equal(wsum.cpu().numpy(), ref["wsum"]), "weight sums differ"
    assert np.array_equal(P.cpu().numpy(), ref["P"][m0:, n0:]), "partial sums differ"
    err = y_error(Y.cpu().numpy(), ref["Y"])
    assert err <= Y_TOL, err
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.gpu
def test_asym_select_layout(fmpq_gpu, oracle_mod):
    """QUIK's base part: 896 channels selected from rows of 1024 (the outliers left to FP16)."""
    from tests.gpu_helpers import Y_TOL, to_dev, y_error
    M, N, K_in, K = 64, 256, 1024, 896
    X, _, W, _ = _inputs(M, N, K_in, seed=3)
    rng = np.random.default_rng(4)
    base = np.sort(rng.choice(K_in, size=K, replace=False)).astype(np.int32)
    layout = fmpq_gpu.select_layout(K, K_in, base, np.zeros(K // BLOCK, np.uint8))
    A, sx, z = fmpq_gpu.fmpq_quantize_asym(layout, to_dev(X))
    Wp, sw = fmpq_gpu.w4_pack_weights(layout, to_dev(W))
    wsum = fmpq_gpu.w4_weight_sums(layout, Wp, sw, N)
    Y = fmpq_gpu.w4ax_gemm_asym(layout, A, sx, z, Wp, sw, wsum, M, N)
    ref = oracle_mod.asym_reference(X[:, base], W[:, base], np.arange(K, dtype=np.int32))
    assert np.array_equal(A.cpu().numpy(), ref["A_packed"])
    assert np.array_equal(z.cpu().numpy().view(np.uint16), ref["a_zeros"])
    assert y_error(Y.cpu().numpy(), ref["Y"]) <= Y_TOL
    layout.close()


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,pad", [(1, 256, 128, 0), (45, 512, 1024, 8), (300, 768, 4096, 0),
                                       (1024, 1024, 8192, 16)])
def test_qoq_matches_oracle(fmpq_gpu, oracle_mod, M, N, K, pad):
    from tests.gpu_helpers import Y_TOL, to_dev, y_error
    X, big, W, perm = _inputs(M, N, K, seed=2 * M + K, pad=pad)
    Wb = (W.astype(np.float32) + np.float32(0.01)).astype(np.float16)   # groups off-centre: non-trivial zero points
    layout = fmpq_gpu.Layout(K, perm, np.ones(K // BLOCK, np.uint8))
    A, sx, sums = fmpq_gpu.qoq_quantize(layout, to_dev(big)[:, :K])
    Wp, s1, s2, z2 = fmpq_gpu.qoq_pack_weights(layout, to_dev(Wb))
    q4 = fmpq_gpu.qoq_unpack_weights(layout, Wp, N)
    Y = fmpq_gpu.qoq_gemm(layout, A, sx, sums, Wp, s1, s2, z2, M, N)
    mc, nc = min(M, 40), min(N, 72)
    P = fmpq_gpu.qoq_gemm_partials(layout, A, Wp, M, N, 0, mc, 0, nc)
    ref = oracle_mod.qoq_reference(X, Wb, perm)
    assert np.array_equal(s1.cpu().numpy().view(np.uint16), ref["s1"]), "channel scales differ"
    assert np.array_equal(s2.cpu().numpy(), ref["s2"]), "group scales differ"
    assert np.array_equal(z2.cpu().numpy(), ref["z2"]), "group zero points differ"
    assert np.array_equal(q4.cpu().numpy(), ref["q4"]), "weight codes differ"
    assert np.array_equal(sx.cpu().numpy().view(np.uint16), ref["a_scales"]), "token scales differ"
    assert np.array_equal(sums.cpu().numpy(), ref["a_sums"]), "code sums differ"
    assert np.array_equal(A.cpu().numpy(), ref["A_packed"]), "activation codes differ"
    assert np.array_equal(P.cpu().numpy(), ref["P"][:mc, :nc]), "partial sums differ"
    err = y_error(Y.cpu().numpy(), ref["Y"])
    assert err <= Y_TOL, err
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.gpu
def test_variant_argument_errors(fmpq_gpu):
    """Layouts that do not fit the variant are refused before any launch."""
    from tests.gpu_helpers import to_dev
    K, M, N = 256, 8, 256
    X = to_dev(np.zeros((M, K), np.float16))
    mixed = fmpq_gpu.Layout(K, np.arange(K, dtype=np.int32), np.array([0, 1], np.uint8))
    with pytest.raises(fmpq_gpu.FmpqError):
        fmpq_gpu.fmpq_quantize_asym(mixed, X)             # an INT8 block in an asymmetric layout
    with pytest.raises(fmpq_gpu.FmpqError):
        fmpq_gpu.qoq_quantize(mixed, X)                   # QoQ needs every block INT8
    sel = fmpq_gpu.select_layout(128, 256, np.arange(128, dtype=np.int32), np.ones(1, np.uint8))
    with pytest.raises(fmpq_gpu.FmpqError):
        fmpq_gpu.qoq_quantize(sel, X)                     # per-token scale over the whole row only
    mixed.close()
    sel.close()
    # the variants' workspace holds their zero-point term: never empty, and required
    import torch
    asym = fmpq_gpu.Layout(K, np.arange(K, dtype=np.int32), np.zeros(2, np.uint8))
    assert int(asym._lib.fmpq_variant_gemm_workspace_bytes(asym.handle, M, N)) > 0
    A, sx, z = fmpq_gpu.fmpq_quantize_asym(asym, X)
    Wp, sw = fmpq_gpu.w4_pack_weights(asym, to_dev(np.zeros((N, K), np.float16)))
    wsum = fmpq_gpu.w4_weight_sums(asym, Wp, sw, N)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fmpq_gpu.FmpqError) as e:
        fmpq_gpu.w4ax_gemm_asym(asym, A, sx, z, Wp, sw, wsum, M, N, Y, workspace=small)
    assert e.value.code == 7                              # FMPQ_ERR_WORKSPACE
    asym.close()


def test_variant_samples_agree_with_whole_reference(oracle_mod):
    """The sampled forms used at full size give the whole-matrix references' values."""
    rng = np.random.default_rng(21)
    M, N, K = 7, 11, 384
    X = (rng.standard_normal((M, K)) + 0.5).astype(np.float16)
    W = (rng.standard_normal((N, K)) * 0.03 + 0.005).astype(np.float16)
    perm = rng.permutation(K).astype(np.int32)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    r = oracle_mod.asym_reference(X, W, perm)
    P, Y = oracle_mod.gemm_sample_asym(r["Aq"], r["Wq"], r["a_scales"], r["a_zeros"], r["w_scales"], r["wsum"],
                                       ms.ravel(), ns.ravel())
    assert np.array_equal(P.reshape(M, N, -1), r["P"]) and np.array_equal(Y.reshape(M, N), r["Y"])
    q = oracle_mod.qoq_reference(X, W, perm)
    P, Y = oracle_mod.gemm_sample_qoq(q["Aq"], q["q4"], q["a_scales"], q["a_sums"], q["s1"], q["s2"], q["z2"],
                                      ms.ravel(), ns.ravel())
    assert np.array_equal(P.reshape(M, N, -1), q["P"]) and np.array_equal(Y.reshape(M, N), q["Y"])


def _sampled_y_error(Yg, Ys):
    floor = 1e-2 * np.sqrt(np.mean(Ys ** 2))
    return float(np.max(np.abs(Yg - Ys) / np.maximum(np.abs(Ys), floor)))


@pytest.mark.gpu
def test_asym_full_size(fmpq_gpu, oracle_mod):
    """The benchmark's LLaMA-70B down-projection shape (4096 x 28672 -> 8192), every block 4-bit:
    codes, scales, zero points and weight sums bit-exact, a window of partial sums, Y sampled."""
    import torch
    from bit_quantized_gemm_fmpq_gb300 import workloads as wl
    from tests.gpu_helpers import Y_TOL, to_dev
    w = wl.llama70b_down()
    layout = fmpq_gpu.Layout(w.K, w.perm, np.zeros(w.K // BLOCK, np.uint8))
    A, sx, z = fmpq_gpu.fmpq_quantize_asym(layout, to_dev(w.X))
    Wp, sw = fmpq_gpu.w4_pack_weights(layout, to_dev(w.W))
    wsum = fmpq_gpu.w4_weight_sums(layout, Wp, sw, w.N)
    Y = fmpq_gpu.w4ax_gemm_asym(layout, A, sx, z, Wp, sw, wsum, w.M, w.N)
    m0, mc, n0, nc = 4000, 96, 8000, 192
    P = fmpq_gpu.w4ax_gemm_partials(layout, A, Wp, w.M, w.N, m0, mc, n0, nc).cpu().numpy()
    A_ref, sx_ref, z_ref, Aq = oracle_mod.quantize_activations_asym(w.X, w.perm)
    assert np.array_equal(A.cpu().numpy(), A_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint16), sx_ref)
    assert np.array_equal(z.cpu().numpy().view(np.uint16), z_ref)
    del A_ref
    Wq, sw_ref = oracle_mod.quantize_weights(w.W, w.perm)
    wsum_ref = oracle_mod.weight_sums(Wq, sw_ref)
    assert np.array_equal(wsum.cpu().numpy(), wsum_ref)
    ms, ns = np.meshgrid(np.arange(m0, m0 + mc), np.arange(n0, n0 + nc), indexing="ij")
    Pw, _ = oracle_mod.gemm_sample_asym(Aq, Wq, sx_ref, z_ref, sw_ref, wsum_ref, ms.ravel(), ns.ravel())
    assert np.array_equal(P.reshape(-1, w.K // BLOCK), Pw)
    rng = np.random.default_rng(0)
    sm = np.concatenate([rng.integers(0, w.M, 4096), [0, w.M - 1]]).astype(np.int32)
    sn = np.concatenate([rng.integers(0, w.N, 4096), [0, w.N - 1]]).astype(np.int32)
    _, Ys = oracle_mod.gemm_sample_asym(Aq, Wq, sx_ref, z_ref, sw_ref, wsum_ref, sm, sn)
    err = _sampled_y_error(Y.cpu().numpy()[sm, sn].astype(np.float64), Ys)
    assert err <= Y_TOL, err
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_qoq_full_size(fmpq_gpu, oracle_mod):
    """The same shape through QoQ: per-token INT8 codes and sums, progressive weights (s1, s2,
    z2, codes) bit-exact, a window of partial sums, Y sampled."""
    import torch
    from bit_quantized_gemm_fmpq_gb300 import workloads as wl
    from tests.gpu_helpers import Y_TOL, to_dev
    w = wl.llama70b_down()
    layout = fmpq_gpu.Layout(w.K, w.perm, np.ones(w.K // BLOCK, np.uint8))
    A, sx, sums = fmpq_gpu.qoq_quantize(layout, to_dev(w.X))
    Wp, s1, s2, z2 = fmpq_gpu.qoq_pack_weights(layout, to_dev(w.W))
    Y = fmpq_gpu.qoq_gemm(layout, A, sx, sums, Wp, s1, s2, z2, w.M, w.N)
    m0, mc, n0, nc = 0, 64, 8192 - 128, 128
    P = fmpq_gpu.qoq_gemm_partials(layout, A, Wp, w.M, w.N, m0, mc, n0, nc).cpu().numpy()
    q4 = fmpq_gpu.qoq_unpack_weights(layout, Wp, w.N).cpu().numpy()
    A_ref, sx_ref, sums_ref, Aq = oracle_mod.qoq_quantize_activations(w.X, w.perm)
    assert np.array_equal(A.cpu().numpy(), A_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint16), sx_ref)
    assert np.array_equal(sums.cpu().numpy(), sums_ref)
    del A_ref
    r = oracle_mod.qoq_quantize_weights(w.W, w.perm)
    assert np.array_equal(q4, r["q4"])
    assert np.array_equal(s1.cpu().numpy().view(np.uint16), r["s1"])
    assert np.array_equal(s2.cpu().numpy(), r["s2"]) and np.array_equal(z2.cpu().numpy(), r["z2"])
    ms, ns = np.meshgrid(np.arange(m0, m0 + mc), np.arange(n0, n0 + nc), indexing="ij")
    Pw, _ = oracle_mod.gemm_sample_qoq(Aq, r["q4"], sx_ref, sums_ref, r["s1"], r["s2"], r["z2"], ms.ravel(), ns.ravel())
    assert np.array_equal(P.reshape(-1, w.K // BLOCK), Pw)
    rng = np.random.default_rng(1)
    sm = np.concatenate([rng.integers(0, w.M, 4096), [0, w.M - 1]]).astype(np.int32)
    sn = np.concatenate([rng.integers(0, w.N, 4096), [0, w.N - 1]]).astype(np.int32)
    _, Ys = oracle_mod.gemm_sample_qoq(Aq, r["q4"], sx_ref, sums_ref, r["s1"], r["s2"], r["z2"], sm, sn)
    err = _sampled_y_error(Y.cpu().numpy()[sm, sn].astype(np.float64), Ys)
    assert err <= Y_TOL, err
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_quik_whole_path(fmpq_gpu, oracle_mod):
    """QUIK end to end (QUIK explainer, "第二步: 前向传播" and "反量化背后的数学"): base columns
    through asymmetric INT4 (a layout selecting them from the full rows), outlier columns in
    FP16, the two results added in Y. Each part against its exact value: the INT4 output within
    the output tolerance; the merge (the FP16 outlier result added to the fp16 base output in
    fp16) within half an fp16 ulp of the result and of the product plus the FP32 summation
    bound."""
    import torch
    from tests.gpu_helpers import Y_TOL, to_dev, y_error
    M, N, K_in, n_out = 200, 512, 2048, 128
    rng = np.random.default_rng(31)
    X = (rng.standard_normal((M, K_in)) + 0.3).astype(np.float32)
    out_cols = np.sort(rng.choice(K_in, size=n_out, replace=False)).astype(np.int32)
    X[:, out_cols] *= rng.uniform(20, 100, size=n_out).astype(np.float32)
    X = X.astype(np.float16)
    W = (rng.standard_normal((N, K_in)) * 0.02).astype(np.float16)
    base = np.setdiff1d(np.arange(K_in), out_cols).astype(np.int32)
    K = base.size
    layout = fmpq_gpu.select_layout(K, K_in, base, np.zeros(K // BLOCK, np.uint8))
    Xd, Wd = to_dev(X), to_dev(W)
    A, sx, z = fmpq_gpu.fmpq_quantize_asym(layout, Xd)
    Wp, sw = fmpq_gpu.w4_pack_weights(layout, Wd)
    wsum = fmpq_gpu.w4_weight_sums(layout, Wp, sw, N)
    Y = fmpq_gpu.w4ax_gemm_asym(layout, A, sx, z, Wp, sw, wsum, M, N)
    Y_base = Y.cpu().numpy().astype(np.float64)
    W_out = Wd[:, torch.from_numpy(out_cols).long().cuda()].contiguous()
    fmpq_gpu.fmpq_outlier_gemm_fp16(layout, Xd, to_dev(out_cols), W_out, Y)
    Ym = Y.cpu().numpy().astype(np.float64)
    ref = oracle_mod.asym_reference(X[:, base], W[:, base], np.arange(K, dtype=np.int32))
    assert y_error(Y_base, ref["Y"]) <= Y_TOL
    _, yo = oracle_mod.quik_reference(X, W, base, out_cols)
    # fp16 rounding of the FP32 sum of the outlier products (ulp taken one binade up), then of its
    # sum with the fp16 base output
    Xo, Wo = np.abs(X[:, out_cols].astype(np.float64)), np.abs(W[:, out_cols].astype(np.float64))
    bound = (0.5 * np.spacing(np.abs(Ym).astype(np.float16)).astype(np.float64)
             + 0.5 * np.spacing((np.abs(yo) * (1 + 2.0 ** -9)).astype(np.float16)).astype(np.float64)
             + n_out * 2.0 ** -24 * (Xo @ Wo.T))
    assert np.all(np.abs(Ym - (Y_base + yo)) <= bound)
    layout.close()


def test_qoq_group_codes_are_the_nearest_level(oracle_mod):
    """Brute force over the 16 levels (q4 - z2) * s2 of each group: the oracle's code is the
    level nearest to the INT8 value, ties to the even multiple of s2 (round half to even of
    q8 / s2), for every range inside [-119, 119] and the values of the range."""
    rng = np.random.default_rng(13)
    lo = rng.integers(-119, 120, 3000)
    hi = rng.integers(-119, 120, 3000)
    lo, hi = np.minimum(lo, hi), np.maximum(lo, hi)
    q8 = np.stack([rng.integers(l, h + 1, BLOCK) for l, h in zip(lo, hi)]).astype(np.int64)
    q8[:, 0], q8[:, 1] = lo, hi
    s2, z2, q4 = oracle_mod.qoq_group(q8.astype(np.int8))
    levels = (np.arange(16)[None, :] - z2[:, None]) * s2[:, None]          # [G, 16]
    dist = np.abs(q8[:, :, None] - levels[:, None, :])                     # [G, 128, 16]
    best = dist.min(axis=2, keepdims=True)
    cand = dist == best
    k = np.arange(16)[None, None, :] - z2[:, None, None]                   # multiple of s2
    # among equally near levels prefer the even multiple
    pref = np.where(cand & (k % 2 == 0), 0, np.where(cand, 1, 2))
    want = np.argmin(pref * 1000 + np.arange(16)[None, None, :], axis=2)
    assert np.array_equal(q4.astype(np.int64), want)


def test_asym_codes_are_the_nearest_level_on_dyadic_inputs(oracle_mod):
    """Inputs on a grid of 1/16 in [-4, 4) with max - min = 15 * 2^-k: the scale is exact, every
    difference and quotient is exact in fp32, so the code is the nearest of the 16 levels
    z + q s (ties to even q), found by brute force."""
    rng = np.random.default_rng(17)
    M = 64
    X = np.zeros((M, BLOCK), dtype=np.float32)
    for m in range(M):
        s = 2.0 ** -int(rng.integers(1, 5))                 # 1/2 .. 1/16
        z = float(rng.integers(-64, 0)) / 16.0
        v = z + rng.integers(0, 15 * 16, BLOCK) / 16.0 * s   # multiples of s/16 inside [z, z + 15 s)
        v[0], v[1] = z, z + 15 * s
        X[m] = v
    X16 = X.astype(np.float16)
    assert np.array_equal(X16.astype(np.float32), X)          # exactly representable
    _, sv, zv, Aq = oracle_mod.quantize_activations_asym(X16, np.arange(BLOCK, dtype=np.int32))
    s = oracle_mod.f16_bits_to_f32(sv).astype(np.float64)
    z = oracle_mod.f16_bits_to_f32(zv).astype(np.float64)
    levels = z[:, None] + np.arange(16)[None, :] * s[:, None]
    dist = np.abs(X.astype(np.float64)[:, :, None] - levels[:, None, :])
    best = dist.min(axis=2, keepdims=True)
    cand = dist == best
    pref = np.where(cand & (np.arange(16) % 2 == 0)[None, None, :], 0, np.where(cand, 1, 2))
    want = np.argmin(pref * 1000 + np.arange(16)[None, None, :], axis=2)
    assert np.array_equal(Aq.astype(np.int64), want)
