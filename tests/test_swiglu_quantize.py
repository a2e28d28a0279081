"""The quantizer fused with the SwiGLU activation (QServe explainer, "运行时设计": the activation
quantization of the second FFN layer is fused into the activation kernel before it).

h = fp16_rn(g * u / (1 + e^-g)) for the gate and up projections' outputs g, u, then the FMPQ
quantizer on h. CPU: the oracle's SwiGLU pinned against mpmath's exact value rounded to fp16.
GPU: fmpq_swiglu_quantize (inputs in the layout's permuted channel order) bit-exact against the
oracle's SwiGLU followed by the oracle's quantizer."""
import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl


def _round_f16(v, sign_if_zero):
    """An mpmath value rounded to fp16 (ties to even), as a float16; exact zero takes the given
    sign (the IEEE sign of g * u)."""
    mpmath = pytest.importorskip("mpmath")
    if v == 0:
        return np.float16(-0.0) if sign_if_zero else np.float16(0.0)
    neg = v < 0
    a = -v if neg else v

    def rhe(q):   # round half to even of a positive mpf
        fl = mpmath.floor(q)
        d = q - fl
        if d > 0.5 or (d == 0.5 and int(fl) % 2 == 1):
            fl += 1
        return fl

    if a >= 65520:
        r = np.float16(np.inf)
    elif a < mpmath.mpf(2) ** -14:
        r = np.float16(float(rhe(a * mpmath.mpf(2) ** 24)) * 2.0 ** -24)
    else:
        e = int(mpmath.floor(mpmath.log(a, 2)))
        if mpmath.mpf(2) ** e > a:                 # guard the logarithm's rounding
            e -= 1
        elif mpmath.mpf(2) ** (e + 1) <= a:
            e += 1
        q = mpmath.mpf(2) ** (e - 10)
        r = np.float16(float(rhe(a / q) * q))
    return -r if neg else r


def _exact_swiglu(g, u):
    mpmath = pytest.importorskip("mpmath")
    out = np.empty(g.size, dtype=np.float16)
    with mpmath.workdps(50):
        for i, (gi, ui) in enumerate(zip(g.astype(np.float64), u.astype(np.float64))):
            v = mpmath.mpf(gi) * mpmath.mpf(ui) / (1 + mpmath.exp(-mpmath.mpf(gi)))
            out[i] = _round_f16(v, bool(np.signbit(gi)) != bool(np.signbit(ui)))
    return out


def _inputs(n, seed):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal(n) * 2.5).astype(np.float16)
    u = (rng.standard_normal(n) * rng.choice([0.01, 1.0, 30.0], n)).astype(np.float16)
    g[:8] = np.array([0.0, -0.0, 20.0, -20.0, 80.0, -80.0, 11.0, -11.0], dtype=np.float16)
    u[:8] = np.array([1.0, 2.0, 1.0, 1.0, -3.0, 3.0, 0.0, -0.0], dtype=np.float16)
    return g, u


def test_oracle_swiglu_is_the_exact_value_rounded(oracle_mod):
    """Against mpmath at 50 digits rounded to fp16 (ties to even), element for element,
    including signed zeros, large negative gates (results that underflow to subnormals or
    zero) and large positive gates (results equal to g * u up to e^-g)."""
    g, u = _inputs(6000, 1)
    got = oracle_mod.swiglu(g, u)
    want = _exact_swiglu(g, u)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_oracle_swiglu_pins_catch_fp32_evaluation(oracle_mod):
    """The pin has teeth: evaluating in fp32 (numpy) and rounding to fp16 differs from the
    oracle's rounding on some elements (about one in ten thousand) of a larger random batch."""
    g, u = _inputs(400000, 2)
    g32, u32 = g.astype(np.float32), u.astype(np.float32)
    with np.errstate(over="ignore"):
        naive = ((g32 * u32) / (np.float32(1) + np.exp(-g32))).astype(np.float16)
    assert np.any(naive.view(np.uint16) != oracle_mod.swiglu(g, u).view(np.uint16))


def test_oracle_swiglu_closed_forms(oracle_mod):
    """silu(0) = 0 with the sign of g * u; silu(g) * u for g = 2^k with e^-g negligible is g * u
    rounded; u = 1 and g = -2^k: the exact tiny value rounds to the nearest subnormal."""
    g = np.array([0.0, -0.0, 0.0, 64.0, 64.0], dtype=np.float16)
    u = np.array([3.0, 3.0, -3.0, 1.5, -0.25], dtype=np.float16)
    h = oracle_mod.swiglu(g, u)
    assert h.view(np.uint16).tolist()[:3] == [0x0000, 0x8000, 0x8000]
    assert h[3] == np.float16(96.0) and h[4] == np.float16(-16.0)


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
@pytest.mark.parametrize("M,K,n8,pad", [(1, 128, 0, 0), (16, 512, 1, 8), (300, 4096, 4, 0), (64, 28672, 27, 16),
                                        (4096, 28672, 27, 0)])
def test_swiglu_quantize_matches_oracle(fmpq_gpu, oracle_mod, M, K, n8, pad):
    """Codes and scales bit-exact; the last case is the LLaMA-70B down projection's activations."""
    import torch
    w = wl.synthetic(M, 256, K, n8=n8, seed=M + K, dist="laplace")
    rng = np.random.default_rng(K + 1)
    G = (rng.standard_normal((M, K)) * 2.0).astype(np.float16)
    U = w.X                                   # Laplace activations with the outlier channels
    layout = fmpq_gpu.Layout(w.K, w.perm, w.mask)
    Gp = np.zeros((M, K + pad), dtype=np.float16)
    Up = np.zeros((M, K + pad), dtype=np.float16)
    Gp[:, :K] = G[:, w.perm]
    Up[:, :K] = U[:, w.perm]
    Gd = torch.from_numpy(Gp).cuda()[:, :K]
    Ud = torch.from_numpy(Up).cuda()[:, :K]
    A, sx = fmpq_gpu.fmpq_swiglu_quantize(layout, Gd, Ud)
    H = oracle_mod.swiglu(G, U)
    A_ref, sx_ref, _ = oracle_mod.quantize_activations(H, w.perm, w.mask, want_codes=False)
    assert np.array_equal(sx.cpu().numpy().view(np.uint16), sx_ref), "scales differ"
    assert np.array_equal(A.cpu().numpy(), A_ref), "code planes differ"
    assert fmpq_gpu.fmpq_device_status(layout) == 0
    layout.close()
