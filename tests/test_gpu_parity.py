"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded
inputs. Integers (packed codes, scales, unpacked weights, per-block partial sums) must be
bit-exact; Y must be within 2e-3 floored relative error of the oracle's fp64 epilogue."""
import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl
from tests.gpu_helpers import Y_TOL, run_gpu, to_dev, y_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fmpq_mod():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_gemm_fmpq_gb300 import build, fmpq
    build.build()
    fmpq.load_library()
    return fmpq


def _check_all(fmpq_mod, oracle_mod, w, partial_window=None):
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    M, N, K = w.M, w.N, w.K
    if partial_window is None:
        partial_window = (0, M, 0, N)
    got, _ = run_gpu(layout, w.X, w.W, want_partials=partial_window)
    ref = oracle_mod.reference(w.X, w.W, w.perm, w.mask)
    assert np.array_equal(got["A"], ref["A_packed"]), "packed activations differ"
    assert np.array_equal(got["sx"].view(np.uint16), ref["a_scales"]), "activation scales differ"
    assert np.array_equal(got["sw"].view(np.uint16), ref["w_scales"]), "weight scales differ"
    Wq = fmpq_mod.w4_unpack_weights(layout, to_dev(got["Wp"]), N).cpu().numpy()
    assert np.array_equal(Wq, ref["Wq"]), "packed weights differ"
    m0, mc, n0, nc = partial_window
    assert np.array_equal(got["P"], ref["P"][m0:m0 + mc, n0:n0 + nc]), "partial sums differ"
    err = y_error(got["Y"], ref["Y"])
    assert err <= Y_TOL, f"Y relative error {err:.3e}"
    assert fmpq_mod.fmpq_device_status(layout) == 0
    layout.close()
    return err


def test_tiny_config(fmpq_mod, oracle_mod):
    _check_all(fmpq_mod, oracle_mod, wl.tiny())


@pytest.mark.parametrize("M,N,K,n8", [
    (300, 784, 1024, 2),     # 3 M-tiles (ragged 44) x 4 N-tiles (ragged 16), 8 blocks
    (128, 256, 512, 1),      # exactly one tile
    (1, 512, 2048, 3),       # one token: split-K path
    (129, 272, 384, 1),      # ragged by one in both dimensions
    (64, 1024, 4096, 4),     # decode-like, split-K
    (200, 512, 1024, 8),     # all INT8
    (200, 512, 1024, 0),     # all INT4
    (40, 256, 128, 0),       # single block
    # few tokens (the operand-swapped GEMM, M <= 64): token tiles of 16/32/64, ragged N
    (5, 272, 384, 1),        # 16-token tile, last channel tile 16 wide
    (17, 528, 1024, 2),      # 32-token tile with 17 tokens
    (33, 256, 256, 0),       # all INT4, 64-token tile
    (64, 400, 640, 5),       # all INT8, full 64-token tile
    # 65-128 tokens: the main GEMM with one partly filled 256-token tile
    (100, 784, 2048, 3),     # 100 tokens, ragged N
    (128, 400, 640, 5),      # all INT8, 128 tokens
])
def test_shapes(fmpq_mod, oracle_mod, M, N, K, n8):
    w = wl.synthetic(M, N, K, n8=n8, seed=M + N + K)
    _check_all(fmpq_mod, oracle_mod, w)


def test_zero_rows_blocks_and_extreme_values(fmpq_mod, oracle_mod):
    w = wl.synthetic(150, 512, 1024, n8=2, seed=9)
    X = w.X.copy()
    X[3] = 0                                   # an all-zero token
    X[5, :300] = 0                             # zero channels -> some zero blocks after perm
    X[7] = (X[7].astype(np.float32) * 1e-6).astype(np.float16)     # subnormal scales
    X[8] = np.clip(X[8].astype(np.float32) * 600, -65000, 65000).astype(np.float16)  # near fp16 max
    X[9, ::7] = np.float16(2.5)                # ties
    w.X = X
    W = w.W.copy()
    W[11] = 0
    W[12] = (W[12].astype(np.float32) * 1e-3).astype(np.float16)
    w.W = W
    _check_all(fmpq_mod, oracle_mod, w)


def test_strided_inputs_and_outputs(fmpq_mod, oracle_mod):
    import torch
    w = wl.synthetic(100, 512, 768, n8=1, seed=3)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    Xbig = np.zeros((w.M, w.K + 64), dtype=np.float16)
    Xbig[:, :w.K] = w.X
    Wbig = np.zeros((w.N, w.K + 8), dtype=np.float16)
    Wbig[:, :w.K] = w.W
    Xd = to_dev(Xbig)[:, :w.K]
    Wd = to_dev(Wbig)[:, :w.K]
    A, sx = fmpq_mod.fmpq_quantize(layout, Xd)
    Wp, sw = fmpq_mod.w4_pack_weights(layout, Wd)
    Ybig = torch.full((w.M, w.N + 24), 7.0, dtype=torch.float16, device="cuda")
    fmpq_mod.w4ax_gemm(layout, A, sx, Wp, sw, w.M, w.N, Y=Ybig[:, :w.N])
    ref = oracle_mod.reference(w.X, w.W, w.perm, w.mask)
    Yh = Ybig.cpu().numpy()
    assert np.all(Yh[:, w.N:] == 7.0), "wrote past N"
    assert y_error(Yh[:, :w.N], ref["Y"]) <= Y_TOL
    assert np.array_equal(A.cpu().numpy(), ref["A_packed"])
    layout.close()


@pytest.mark.parametrize("M,uses_workspace", [
    (16, False),    # few tokens: the splits of a tile meet in a cluster's shared memory
    (256, True),    # the main GEMM's split-K: workspace counters return to zero
])
def test_repeated_calls_and_workspace_reuse(fmpq_mod, oracle_mod, M, uses_workspace):
    """Split-K in both GEMMs: repeated calls give identical output."""
    w = wl.synthetic(M, 512, 2048, n8=2, seed=21)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    assert (layout.workspace_bytes(w.M, w.N) > 0) == uses_workspace
    Xd, Wd = to_dev(w.X), to_dev(w.W)
    A, sx = fmpq_mod.fmpq_quantize(layout, Xd)
    Wp, sw = fmpq_mod.w4_pack_weights(layout, Wd)
    Ys = [fmpq_mod.w4ax_gemm(layout, A, sx, Wp, sw, w.M, w.N).cpu().numpy() for _ in range(4)]
    for Y in Ys[1:]:
        assert np.array_equal(Y.view(np.uint16), Ys[0].view(np.uint16))
    ref = oracle_mod.reference(w.X, w.W, w.perm, w.mask)
    assert y_error(Ys[0], ref["Y"]) <= Y_TOL
    layout.close()


def test_argument_errors(fmpq_mod):
    import torch
    K = 256
    perm = np.arange(K, dtype=np.int32)
    with pytest.raises(fmpq_mod.FmpqError):
        fmpq_mod.Layout(K, np.zeros(K, dtype=np.int32), np.zeros(2, np.uint8))   # not a permutation
    with pytest.raises(fmpq_mod.FmpqError):
        fmpq_mod.Layout(K, perm, np.array([0, 2], np.uint8))                     # bad mask value
    layout = fmpq_mod.Layout(K, perm, np.zeros(2, np.uint8))
    X = torch.zeros((4, K), dtype=torch.float16, device="cuda")
    W = torch.zeros((24, K), dtype=torch.float16, device="cuda")
    with pytest.raises(fmpq_mod.FmpqError) as e:
        fmpq_mod.w4_pack_weights(layout, W)                                      # N % 16 != 0
    assert e.value.code == 2
    Xo = torch.zeros((4, K + 4), dtype=torch.float16, device="cuda")[:, :K]
    with pytest.raises(fmpq_mod.FmpqError) as e:
        fmpq_mod.fmpq_quantize(layout, Xo)                                      # ldx % 8 != 0
    assert e.value.code == 3
    A, sx = fmpq_mod.fmpq_quantize(layout, X)
    assert fmpq_mod.fmpq_device_status(layout) == 0
    layout.close()


# --------------------------------------------------------------------- full-size configs

def _sampled_check(fmpq_mod, oracle_mod, w, n_samples=4096, window=(0, 16, 0, 32), seed=0, full_y=False):
    """Full-size run in the benchmark's launch configuration; bit-exact quantizer, weights and
    a window of partial sums; Y at sampled positions against the oracle's fp64 epilogue (every
    position when full_y)."""
    import torch
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    got, dev = run_gpu(layout, w.X, w.W, want_partials=window)
    A_ref, sx_ref, Aq = oracle_mod.quantize_activations(w.X, w.perm, w.mask)
    assert np.array_equal(got["A"], A_ref), "packed activations differ"
    assert np.array_equal(got["sx"].view(np.uint16), sx_ref)
    Wq_ref, sw_ref = oracle_mod.quantize_weights(w.W, w.perm)
    assert np.array_equal(got["sw"].view(np.uint16), sw_ref)
    Wq = fmpq_mod.w4_unpack_weights(layout, dev["Wp"], w.N).cpu().numpy()
    assert np.array_equal(Wq, Wq_ref), "packed weights differ"
    del Wq
    m0, mc, n0, nc = window
    ms, ns = np.meshgrid(np.arange(m0, m0 + mc), np.arange(n0, n0 + nc), indexing="ij")
    Pw, _ = oracle_mod.gemm_sample(Aq, Wq_ref, sx_ref, sw_ref, ms.ravel(), ns.ravel())
    assert np.array_equal(got["P"].reshape(-1, w.K // 128), Pw), "partial sums differ"
    rng = np.random.default_rng(seed)
    if full_y:
        gm, gn = np.meshgrid(np.arange(w.M), np.arange(w.N), indexing="ij")
        sm, sn = gm.ravel().astype(np.int32), gn.ravel().astype(np.int32)
    else:
        sm = np.concatenate([rng.integers(0, w.M, n_samples), [0, w.M - 1, w.M - 1]]).astype(np.int32)
        sn = np.concatenate([rng.integers(0, w.N, n_samples), [0, 0, w.N - 1]]).astype(np.int32)
    _, Ys = oracle_mod.gemm_sample(Aq, Wq_ref, sx_ref, sw_ref, sm, sn, want_partials=False)
    Yg = got["Y"][sm, sn].astype(np.float64)
    # the floor uses the rms of the sampled reference values
    floor = 1e-2 * np.sqrt(np.mean(Ys ** 2))
    err = float(np.max(np.abs(Yg - Ys) / np.maximum(np.abs(Ys), floor)))
    assert err <= Y_TOL, f"Y relative error {err:.3e}"
    assert fmpq_mod.fmpq_device_status(layout) == 0
    layout.close()
    torch.cuda.empty_cache()
    return err


def test_config_llama7b_qkv(fmpq_mod, oracle_mod):
    _sampled_check(fmpq_mod, oracle_mod, wl.llama7b_qkv())


def test_config_llama70b_down(fmpq_mod, oracle_mod):
    _sampled_check(fmpq_mod, oracle_mod, wl.llama70b_down(), window=(4000, 96, 8000, 192))


@pytest.mark.parametrize("M", wl.DECODE_MS)
def test_config_decode(fmpq_mod, oracle_mod, M):
    """Decode shapes (the few-token kernel): every output element against the oracle, and the
    per-block partial sums of a 300-channel window bit-exact through the same kernel."""
    _sampled_check(fmpq_mod, oracle_mod, wl.decode(M), window=(0, M, 100, 300), full_y=True)


@pytest.mark.parametrize("frac", wl.LOAD_BALANCE_FRACS)
def test_config_load_balance(fmpq_mod, oracle_mod, frac):
    _sampled_check(fmpq_mod, oracle_mod, wl.load_balance(frac), window=(1000, 40, 28672 - 80, 80))


def test_scale_every_fp16_absmax(fmpq_mod, oracle_mod):
    """Every finite non-negative fp16 value as the absmax of an INT4 and of an INT8 block
    (one token each), the other channels random fractions of it: scales and code planes
    bit-exact against the oracle."""
    rng = np.random.default_rng(5)
    amax = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)
    M, K = amax.size, 256
    frac = rng.uniform(-1.0, 1.0, size=(M, K)).astype(np.float32)
    X = (frac * amax[:, None]).astype(np.float16)
    X[:, 0] = amax.astype(np.float16)
    X[:, 128] = (-amax).astype(np.float16)
    perm = np.arange(K, dtype=np.int32)
    mask = np.array([0, 1], np.uint8)
    layout = fmpq_mod.Layout(K, perm, mask)
    A, sx = fmpq_mod.fmpq_quantize(layout, to_dev(X))
    A_ref, sx_ref, _ = oracle_mod.quantize_activations(X, perm, mask, want_codes=False)
    assert np.array_equal(sx.cpu().numpy().view(np.uint16), sx_ref)
    assert np.array_equal(A.cpu().numpy(), A_ref)
    assert fmpq_mod.fmpq_device_status(layout) == 0
    layout.close()


@pytest.mark.parametrize("M", [16, 32, 64])
@pytest.mark.parametrize("one_call", [False, True])
def test_back_to_back_steps(fmpq_mod, M, one_call):
    """Few-token GEMM (K = N = 8192) in 20 back-to-back steps, each with its own Y, captured in a
    CUDA graph and replayed 100 times: every step's Y is bit-identical to a single eager call.
    The activation copies' slots are refilled only after every block reading them is done,
    including blocks of the other MMA issuer that finish after a later block; a refill that
    waited for the last reader alone corrupted ~1% of the steps at 64 tokens."""
    import torch
    w = wl.decode(M)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    X = to_dev(w.X)
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    A0, sx0 = fmpq_mod.fmpq_quantize(layout, X)
    Yref = fmpq_mod.w4ax_gemm(layout, A0, sx0, Wp, sw, M, w.N)
    Wc = [Wp] + [Wp.clone() for _ in range(4)]
    A, sx = torch.empty_like(A0), torch.empty_like(sx0)
    Ys = [torch.empty_like(Yref) for _ in range(20)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in range(20):
            if one_call:
                fmpq_mod.fmpq_quantize_gemm(layout, X, Wc[r % 5], sw, w.N, A_packed=A, a_scales=sx, Y=Ys[r])
            else:
                fmpq_mod.fmpq_quantize(layout, X, A, sx)
                fmpq_mod.w4ax_gemm(layout, A, sx, Wc[r % 5], sw, M, w.N, Ys[r])
    bad = 0
    for _ in range(100):
        for Y in Ys:
            Y.fill_(1.0)
        g.replay()
        torch.cuda.synchronize()
        bad += sum(0 if torch.equal(Y.view(torch.int16), Yref.view(torch.int16)) else 1 for Y in Ys)
    assert bad == 0, f"{bad} of 2000 steps differ"
    assert fmpq_mod.fmpq_device_status(layout) == 0
    del g
    layout.close()
