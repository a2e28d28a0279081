"""Pins for the CPU oracle: each test checks it against something other than itself.

- fp16 conversion: numpy's independent float16 cast (structured near-exhaustive sweep);
- quantizer: hand-derived worked examples (tests/golden) and invariants that follow from
  the definition (symmetric range, |x - q*s| <= s/2, sign symmetry, power-of-two scaling,
  joint channel permutation);
- partials: brute force in numpy integer matmul, the zero-extension identity, closed forms,
  intra-block reordering, the all-INT8 / all-INT4 special cases;
- epilogue: exact rational evaluation (Python Fractions), the fp64 summation bound, the
  dequantised-product closed form, and the quantization error bound against X W^T.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantizer_worked_examples.json")


# ----------------------------------------------------------------------------- fp16

def test_f16_to_f32_exhaustive(oracle_mod):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.f16_bits_to_f32(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _f32_sweep():
    """Every fp32 whose dropped mantissa bits sit at a rounding boundary or next to one,
    for every sign/exponent/kept-mantissa combination that matters to fp16, plus the
    subnormal range's half-quantum points, plus random values."""
    parts = []
    # normal fp16 range: exponents covering [2^-15, 2^16]; kept 10 mantissa bits x low patterns
    low = np.array([0, 1, 0xFFF, 0x1000, 0x1001, 0x1FFF, 0x0800, 0x17FF], dtype=np.uint32)
    hi10 = np.arange(1024, dtype=np.uint32) << 13
    for e in range(127 - 15, 127 + 17):
        base = (np.uint32(e) << 23) | hi10
        v = (base[:, None] | low[None, :]).ravel()
        parts += [v, v | np.uint32(0x80000000)]
    # subnormal fp16 range: k * 2^-25 and neighbours (ties and near-ties of the 2^-24 quantum)
    k = np.arange(1, 2 ** 12, dtype=np.float64)
    v = (k * 2.0 ** -25).astype(np.float32)
    vb = v.view(np.uint32)
    parts += [vb, vb + 1, vb - 1, vb | np.uint32(0x80000000)]
    rng = np.random.default_rng(7)
    parts.append(rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32))
    parts.append(np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x477FE000, 0x477FEFFF, 0x477FF000,
                           0x477FF001, 0x387FC000, 0x33000000, 0x33000001, 0x32FFFFFF], dtype=np.uint32))
    return np.concatenate(parts)


def test_f32_to_f16_against_numpy(oracle_mod):
    bits = _f32_sweep()
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    got = oracle_mod.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [(hex(x[i:i+1].view(np.uint32)[0]), hex(got[i]), hex(want[i])) for i in bad[:5]]


# ----------------------------------------------------------------------------- quantizer

def _block_from_example(ex, oracle_mod):
    xs = np.zeros(128, dtype=np.float64)
    if "x" in ex:
        xs[: len(ex["x"])] = ex["x"]
    else:
        u = np.asarray(ex["x_units_2^-24"], dtype=np.float64)
        xs[: len(u)] = u * 2.0 ** -24
    return xs.astype(np.float16)


@pytest.mark.parametrize("idx", range(6))
def test_worked_examples(oracle_mod, idx):
    ex = json.load(open(GOLDEN))["examples"][idx]
    xs = _block_from_example(ex, oracle_mod)
    assert np.array_equal(xs.astype(np.float64), np.asarray(xs, dtype=np.float64))  # fp16-exact inputs
    X = xs[None, :]
    perm = np.arange(128, dtype=np.int32)
    mask = np.array([1 if ex["qmax"] == 127 else 0], dtype=np.uint8)
    _, s, Aq = oracle_mod.quantize_activations(X, perm, mask)
    assert int(s[0, 0]) == int(ex["scale_bits"], 16), ex["name"]
    q = np.zeros(128, dtype=np.int64)
    q[: len(ex["q"])] = ex["q"]
    assert np.array_equal(Aq[0].astype(np.int64), q), ex["name"]


def test_weight_quantizer_is_int4_rule(oracle_mod):
    ex = json.load(open(GOLDEN))["examples"][3]  # INT4 example with scale 0x3092
    xs = _block_from_example(ex, oracle_mod)
    Wq, sw = oracle_mod.quantize_weights(xs[None, :], np.arange(128, dtype=np.int32))
    assert int(sw[0, 0]) == int(ex["scale_bits"], 16)
    q = np.zeros(128, dtype=np.int64)
    q[: len(ex["q"])] = ex["q"]
    assert np.array_equal(Wq[0].astype(np.int64), q)


def _rand_case(seed, M=24, K=512, n8=2, scale=1.0):
    rng = np.random.default_rng(seed)
    X = (rng.standard_normal((M, K)) * scale).astype(np.float16)
    X[:, rng.choice(K, 20, replace=False)] *= np.float16(40)
    perm = rng.permutation(K).astype(np.int32)
    mask = np.zeros(K // 128, dtype=np.uint8)
    mask[rng.choice(K // 128, n8, replace=False)] = 1
    return X, perm, mask


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_quantizer_invariants(oracle_mod, seed):
    X, perm, mask = _rand_case(seed)
    M, K = X.shape
    _, s, Aq = oracle_mod.quantize_activations(X, perm, mask)
    sf = s.view(np.float16).astype(np.float64)                     # [nb, M]
    Xp = X[:, perm].astype(np.float64)
    for b in range(K // 128):
        qmax = 127 if mask[b] else 7
        q = Aq[:, b * 128:(b + 1) * 128].astype(np.int64)
        xb = Xp[:, b * 128:(b + 1) * 128]
        sb = sf[b][:, None]
        assert np.all(np.abs(q) <= qmax)
        nz = sf[b] > 2.0 ** -14                                    # normal scales
        assert np.all(np.abs(q[nz]).max(axis=1) == qmax)           # the absmax lands on +-qmax
        assert np.all(np.abs(xb - q * sb)[nz] <= sb[nz] / 2 + 0)   # round-to-nearest error bound
    # sign symmetry
    _, s2, Aq2 = oracle_mod.quantize_activations(-X, perm, mask)
    assert np.array_equal(s2, s) and np.array_equal(Aq2, -Aq)
    # power-of-two scaling: X * 2^-3 -> scales * 2^-3, same codes (stays in the normal range)
    _, s3, Aq3 = oracle_mod.quantize_activations((X.astype(np.float32) / 8).astype(np.float16), perm, mask)
    assert np.array_equal(Aq3, Aq)
    assert np.array_equal(s3.view(np.float16).astype(np.float64), sf / 8)


def test_joint_permutation_invariance(oracle_mod):
    """Relabelling the input channels by Pi and the permutation by Pi^-1 o perm gives
    bit-identical packed activations and scales."""
    X, perm, mask = _rand_case(5)
    K = X.shape[1]
    rng = np.random.default_rng(11)
    pi = rng.permutation(K)
    Xr = X[:, pi]                       # Xr[:, c] = X[:, pi[c]]
    inv = np.argsort(pi)
    perm_r = inv[perm].astype(np.int32)  # Xr[:, perm_r[j]] = X[:, perm[j]]
    A1, s1, _ = oracle_mod.quantize_activations(X, perm, mask)
    A2, s2, _ = oracle_mod.quantize_activations(Xr, perm_r, mask)
    assert np.array_equal(A1, A2) and np.array_equal(s1, s2)


def test_gather_direction(oracle_mod):
    """perm is a gather: permuted position j takes input channel perm[j]."""
    K = 256
    X = np.zeros((1, K), dtype=np.float16)
    X[0, 5] = 7.0
    perm = np.arange(K, dtype=np.int32)
    perm[130], perm[5] = 5, 130          # channel 5 moves to position 130 (block 1)
    _, s, Aq = oracle_mod.quantize_activations(X, perm, np.array([0, 0], np.uint8))
    assert Aq[0, 130] == 7 and Aq[0, 5] == 0
    assert s[0, 0] == 0 and s[1, 0] == 0x3C00


def test_packed_layout_example(oracle_mod):
    ex = json.load(open(GOLDEN))["packed_layout_example"]
    M = ex["M"]
    X = np.zeros((M, 256), dtype=np.float16)
    X[0, : len(ex["row0_block0_x"])] = ex["row0_block0_x"]
    X[0, 128: 128 + len(ex["row0_block1_x"])] = ex["row0_block1_x"]
    for c, v in ex["row3_x_at"].items():
        X[3, int(c)] = v
    mask = np.array(ex["mask"], dtype=np.uint8)
    A, s, Aq = oracle_mod.quantize_activations(X, np.arange(256, dtype=np.int32), mask)
    assert A.size == ex["total_bytes"]
    want = np.zeros(ex["total_bytes"], dtype=np.uint8)
    for pos, v in ex["expected_nonzero"]:
        want[pos] = int(v, 16)
    assert np.array_equal(A, want), np.nonzero(A != want)
    assert [int(v, 16) for v in ex["expected_scales_bits"]["row0"]] == list(s[:, 0])
    assert [int(v, 16) for v in ex["expected_scales_bits"]["row3"]] == list(s[:, 3])


def test_e4m3_decoder_against_torch(oracle_mod):
    """The oracle's E4M3 decoder (written from the format's definition) against torch's
    float8_e4m3fn conversion, on all 256 encodings."""
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_value(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_plane_bytes_decode_to_code_parts(oracle_mod):
    """Every code in [-127, 127] of an INT8 block and [-7, 7] of an INT4 block: its plane
    bytes decode (E4M3 definition) to parts that sum to |q| * 2^-9, with the code's sign."""
    K, M = 256, 255
    X = np.zeros((M, K), dtype=np.float16)
    q = np.arange(-127, 128)
    # one token per code: channel 128 holds the code, channel 129 pins absmax at 127
    X[:, 128] = q.astype(np.float16)
    X[:, 129] = np.float16(127)
    X[:, 0] = np.clip(q, -7, 7).astype(np.float16)
    X[:, 1] = np.float16(7)
    mask = np.array([0, 1], np.uint8)
    A, s, Aq = oracle_mod.quantize_activations(X, np.arange(K, dtype=np.int32), mask)
    assert np.array_equal(Aq[:, 128], q) and np.array_equal(Aq[:, 0], np.clip(q, -7, 7))
    planes = A.reshape(3, M, 128)
    for m in range(M):
        pos = 16 * ((128 // 16 - 8) ^ (m % 8))          # channel 128 = chunk 0 of block 1
        lo, hi = planes[1, m, pos], planes[2, m, pos]
        v = abs(oracle_mod.e4m3_value(lo)) + abs(oracle_mod.e4m3_value(hi))
        assert v * 512 == abs(q[m])
        assert (lo >> 7) == (q[m] < 0) and (hi >> 7) == (q[m] < 0)
        assert abs(oracle_mod.e4m3_value(lo)) * 512 == abs(q[m]) % 16
        b4 = planes[0, m, 16 * (0 ^ (m % 8))]             # channel 0 = chunk 0 of block 0
        assert abs(oracle_mod.e4m3_value(b4)) * 512 == min(abs(q[m]), 7)
        assert (b4 >> 7) == (q[m] < 0)


@pytest.mark.parametrize("seed", [0, 3])
def test_pack_unpack_roundtrip(oracle_mod, seed):
    X, perm, mask = _rand_case(seed, M=7)
    A, _, Aq = oracle_mod.quantize_activations(X, perm, mask)
    assert A.size == 7 * 128 * sum(2 if m else 1 for m in mask)
    assert np.array_equal(oracle_mod.unpack_activations(A, mask, 7, X.shape[1]), Aq)


# ----------------------------------------------------------------------------- partials

def _codes(seed, M, N, K, n8):
    X, perm, mask = _rand_case(seed, M=M, K=K, n8=n8)
    rng = np.random.default_rng(seed + 100)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    _, sx, Aq = oracle_mod_q(X, perm, mask)
    return X, W, perm, mask


def oracle_mod_q(X, perm, mask):
    import oracle
    return oracle.quantize_activations(X, perm, mask)


def test_partials_brute_force_numpy(oracle_mod):
    rng = np.random.default_rng(3)
    M, N, K = 5, 9, 384
    Aq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    Wq = rng.integers(-7, 8, size=(N, K)).astype(np.int8)
    P = oracle_mod.partials(Aq, Wq)
    for b in range(K // 128):
        sl = slice(b * 128, (b + 1) * 128)
        want = Aq[:, sl].astype(np.int64) @ Wq[:, sl].astype(np.int64).T
        assert np.array_equal(P[:, :, b].astype(np.int64), want)


def test_partials_zero_extension_identity(oracle_mod):
    rng = np.random.default_rng(4)
    Aq = rng.integers(-127, 128, size=(6, 256)).astype(np.int8)
    Wq = rng.integers(-7, 8, size=(7, 256)).astype(np.int8)
    assert np.array_equal(oracle_mod.partials(Aq, Wq, zero_ext=True), oracle_mod.partials(Aq, Wq))


def test_partials_closed_forms(oracle_mod):
    rng = np.random.default_rng(5)
    Wq = rng.integers(-7, 8, size=(4, 256)).astype(np.int8)
    ones = np.ones((3, 256), dtype=np.int8)
    P = oracle_mod.partials(ones, Wq)
    for b in range(2):
        assert np.array_equal(P[0, :, b], Wq[:, b * 128:(b + 1) * 128].sum(axis=1))
    ext = np.full((1, 128), 127, dtype=np.int8)
    w7 = np.full((1, 128), -7, dtype=np.int8)
    assert oracle_mod.partials(ext, w7)[0, 0, 0] == -113792


def test_partials_intra_block_reorder(oracle_mod):
    rng = np.random.default_rng(6)
    Aq = rng.integers(-127, 128, size=(4, 256)).astype(np.int8)
    Wq = rng.integers(-7, 8, size=(5, 256)).astype(np.int8)
    sigma = np.concatenate([rng.permutation(128), 128 + rng.permutation(128)])
    assert np.array_equal(oracle_mod.partials(Aq[:, sigma], Wq[:, sigma]), oracle_mod.partials(Aq, Wq))


def test_all_int8_and_all_int4_masks(oracle_mod):
    """All-INT8 mask = per-token per-block symmetric W4A8; all-INT4 = W4A4 (codes in range,
    scales follow qmax)."""
    X, perm, _ = _rand_case(8, M=6, K=256)
    for val, qmax in ((1, 127), (0, 7)):
        mask = np.full(2, val, dtype=np.uint8)
        _, s, Aq = oracle_mod.quantize_activations(X, perm, mask)
        Xp = X[:, perm].astype(np.float32)
        for b in range(2):
            amax = np.abs(Xp[:, b * 128:(b + 1) * 128]).max(axis=1)
            want = (amax / np.float32(qmax)).astype(np.float16).view(np.uint16)
            assert np.array_equal(s[b], want)
        assert np.abs(Aq).max() == qmax


# ----------------------------------------------------------------------------- epilogue

def _small_reference(oracle_mod, seed=0, M=6, N=5, K=384, n8=1):
    X, perm, mask = _rand_case(seed, M=M, K=K, n8=n8)
    rng = np.random.default_rng(seed + 50)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    return X, W, perm, mask, oracle_mod.reference(X, W, perm, mask)


def test_epilogue_exact_rational(oracle_mod):
    X, W, perm, mask, r = _small_reference(oracle_mod)
    P, sx, sw = r["P"], r["a_scales"], r["w_scales"]
    Yx = oracle_mod.epilogue(P, sx, sw, exact=True)
    sxf = [[Fraction(float(v)) for v in row] for row in sx.view(np.float16)]
    swf = [[Fraction(float(v)) for v in row] for row in sw.view(np.float16)]
    M, N, nb = P.shape
    for m in range(M):
        for n in range(N):
            exact = sum(sxf[b][m] * swf[b][n] * int(P[m, n, b]) for b in range(nb))
            assert Yx[m, n] == float(exact)          # Python rounds Fractions correctly


def test_epilogue_f64_within_summation_bound(oracle_mod):
    _, _, _, _, r = _small_reference(oracle_mod, seed=1, M=8, N=8, K=1024, n8=2)
    P, sx, sw = r["P"], r["a_scales"], r["w_scales"]
    Y64 = oracle_mod.epilogue(P, sx, sw)
    Yx = oracle_mod.epilogue(P, sx, sw, exact=True)
    terms = np.abs(sx.view(np.float16).astype(np.float64).T[:, None, :] *
                   sw.view(np.float16).astype(np.float64).T[None, :, :] * P)
    bound = P.shape[2] * 2.0 ** -53 * terms.sum(axis=2)
    assert np.all(np.abs(Y64 - Yx) <= bound)


def test_dequantised_product_closed_form(oracle_mod):
    """Y = sum_k (q_x s_x)(q_w s_w), the dequantised product, in fp64 via numpy."""
    _, _, _, mask, r = _small_reference(oracle_mod, seed=2, M=7, N=6, K=512, n8=1)
    sx = r["a_scales"].view(np.float16).astype(np.float64)
    sw = r["w_scales"].view(np.float16).astype(np.float64)
    Xd = r["Aq"].astype(np.float64) * np.repeat(sx.T, 128, axis=1)
    Wd = r["Wq"].astype(np.float64) * np.repeat(sw.T, 128, axis=1)
    Yd = Xd @ Wd.T
    Yx = oracle_mod.epilogue(r["P"], r["a_scales"], r["w_scales"], exact=True)
    scale = np.abs(Xd) @ np.abs(Wd).T
    assert np.all(np.abs(Yd - Yx) <= 1e-12 * scale + 1e-300)


def test_close_to_unquantised_product(oracle_mod):
    """|Y - Xp Wp^T| <= sum_k (|x||dw| + |w||dx| + |dx||dw|), with |dx| <= s_x/2, |dw| <= s_w/2:
    catches transposed operands or scales applied to the wrong block."""
    X, W, perm, mask, r = _small_reference(oracle_mod, seed=3, M=6, N=7, K=512, n8=1)
    Xp = X[:, perm].astype(np.float64)
    Wp = W[:, perm].astype(np.float64)
    sx = np.repeat(r["a_scales"].view(np.float16).astype(np.float64).T, 128, axis=1)
    sw = np.repeat(r["w_scales"].view(np.float16).astype(np.float64).T, 128, axis=1)
    bound = np.abs(Xp) @ (sw / 2).T + (sx / 2) @ np.abs(Wp).T + (sx / 2) @ (sw / 2).T
    err = np.abs(r["Y"] - Xp @ Wp.T)
    assert np.all(err <= bound * (1 + 1e-9))
    # ... and the bound is not vacuous: the result is much closer than |X||W|
    assert np.all(err <= 0.5 * (np.abs(Xp) @ np.abs(Wp).T))


def test_joint_permutation_of_x_and_w_leaves_y(oracle_mod):
    """Y depends on X and W only through the permuted channels."""
    X, W, perm, mask, r = _small_reference(oracle_mod, seed=4, M=5, N=6, K=384, n8=1)
    rng = np.random.default_rng(12)
    pi = rng.permutation(X.shape[1])
    inv = np.argsort(pi)
    r2 = oracle_mod.reference(X[:, pi], W[:, pi], inv[perm].astype(np.int32), mask)
    assert np.array_equal(r2["Y"], r["Y"])


def test_gemm_sample_matches_full(oracle_mod):
    _, _, _, _, r = _small_reference(oracle_mod, seed=5, M=9, N=11, K=512, n8=2)
    ms = np.array([0, 3, 8, 8], dtype=np.int32)
    ns = np.array([0, 10, 5, 0], dtype=np.int32)
    P, Y = oracle_mod.gemm_sample(r["Aq"], r["Wq"], r["a_scales"], r["w_scales"], ms, ns)
    assert np.array_equal(P, r["P"][ms, ns])
    assert np.array_equal(Y, r["Y"][ms, ns])


def test_tiny_workload_structure(oracle_mod):
    w = wl.tiny()
    assert w.X.shape == (16, 512) and w.W.shape == (512, 512)
    # both outlier channels land in the INT8 block (positions 256..383)
    pos = np.argsort(w.perm)
    assert 256 <= pos[37] < 384 and 256 <= pos[300] < 384 and w.mask[2] == 1
    r = oracle_mod.reference(w.X, w.W, w.perm, w.mask)
    assert np.abs(r["Aq"][:, 256:384]).max() == 127
