"""GPU: the one-call quantize + GEMM (the GEMM launched as the quantizer's programmatic
dependent) gives the same codes, scales and Y, bit for bit, as the two separate calls, and Y
within tolerance of the oracle, in both GEMM kernels (few tokens and the main one) and at the
full LLaMA-70B down-projection shape."""
import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl
from tests.gpu_helpers import Y_TOL, to_dev, y_error

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


def _both(fmpq_mod, layout, Xd, Wp, sw, N, reps=1):
    import torch
    M = Xd.shape[0]
    A, sx = fmpq_mod.fmpq_quantize(layout, Xd)
    Y = fmpq_mod.w4ax_gemm(layout, A, sx, Wp, sw, M, N)
    A2 = torch.empty_like(A)
    sx2 = torch.empty_like(sx)
    Y2 = torch.empty_like(Y)
    for _ in range(reps):   # back to back: each call's GEMM overlaps its own quantizer only
        fmpq_mod.fmpq_quantize_gemm(layout, Xd, Wp, sw, N, A_packed=A2, a_scales=sx2, Y=Y2)
    torch.cuda.synchronize()
    assert torch.equal(A2, A), "codes differ"
    assert torch.equal(sx2.view(torch.int16), sx.view(torch.int16)), "activation scales differ"
    assert torch.equal(Y2.view(torch.int16), Y.view(torch.int16)), "Y differs from the two calls"
    assert fmpq_mod.fmpq_device_status(layout) == 0
    return Y2


@pytest.mark.parametrize("M,N,K,n8", [
    (1, 512, 2048, 3),       # few-token kernel, 16-token tile
    (17, 528, 1024, 2),      # 32-token tile, ragged N
    (64, 400, 640, 5),       # full 64-token tile
    (100, 784, 2048, 3),     # main kernel, one partly filled tile
    (300, 784, 1024, 2),     # main kernel, ragged M and N
    (512, 512, 4096, 4),     # main kernel with split-K (workspace)
])
def test_matches_separate_calls_and_oracle(fmpq_mod, oracle_mod, M, N, K, n8):
    w = wl.synthetic(M, N, K, n8=n8, seed=7 * M + N + K)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    Y = _both(fmpq_mod, layout, to_dev(w.X), Wp, sw, w.N, reps=3)
    ref = oracle_mod.reference(w.X, w.W, w.perm, w.mask)
    err = y_error(Y.cpu().numpy(), ref["Y"])
    assert err <= Y_TOL, f"Y relative error {err:.3e}"
    layout.close()


@pytest.mark.parametrize("make", [lambda: wl.decode(16), wl.llama70b_down])
def test_full_size(fmpq_mod, make):
    """Decode (16 tokens, 8192 x 8192) and the 4096 x 28672 -> 8192 step: identical to the two
    calls (which the sampled oracle checks of the configuration tests cover)."""
    w = make()
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    _both(fmpq_mod, layout, to_dev(w.X), Wp, sw, w.N, reps=2)
    layout.close()


def test_argument_errors(fmpq_mod):
    """Every argument is checked before either kernel is launched: a bad GEMM argument leaves
    the activation buffers untouched."""
    import torch
    w = wl.synthetic(32, 256, 512, n8=1, seed=3)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    Xd = to_dev(w.X)
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    A = torch.zeros(layout.packed_a_bytes(w.M), dtype=torch.uint8, device="cuda")
    sx = torch.zeros((layout.nb, w.M), dtype=torch.float16, device="cuda")
    with pytest.raises(fmpq_mod.FmpqError):
        fmpq_mod.fmpq_quantize_gemm(layout, Xd, Wp, sw, 250, A_packed=A, a_scales=sx)   # N % 16
    Ynarrow = torch.empty((w.M, w.N - 16), dtype=torch.float16, device="cuda")
    with pytest.raises(fmpq_mod.FmpqError):
        fmpq_mod.fmpq_quantize_gemm(layout, Xd, Wp, sw, w.N, A_packed=A, a_scales=sx, Y=Ynarrow)   # ldy < N
    torch.cuda.synchronize()
    assert int(A.count_nonzero()) == 0 and int(sx.count_nonzero()) == 0
    layout.close()


@pytest.mark.parametrize("M", [16, 256])
def test_inside_cuda_graph(fmpq_mod, M):
    """Captured in a CUDA graph (the programmatic dependency becomes a graph edge) and replayed
    with a new input: the same Y as the two separate calls on that input."""
    import torch
    w = wl.synthetic(M, 1024, 2048, n8=2, seed=40 + M)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    X = to_dev(w.X)
    A = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device="cuda")
    sx = torch.empty((layout.nb, M), dtype=torch.float16, device="cuda")
    Y = torch.empty((M, w.N), dtype=torch.float16, device="cuda")
    ws = layout.workspace(M, w.N)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fmpq_mod.fmpq_quantize_gemm(layout, X, Wp, sw, w.N, A_packed=A, a_scales=sx, Y=Y, workspace=ws, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                fmpq_mod.fmpq_quantize_gemm(layout, X, Wp, sw, w.N, A_packed=A, a_scales=sx, Y=Y, workspace=ws,
                                            stream=s)
    torch.cuda.synchronize()
    X.copy_(to_dev(wl.synthetic(M, 1024, 2048, n8=2, seed=41 + M).X))
    g.replay()
    torch.cuda.synchronize()
    A2, sx2 = fmpq_mod.fmpq_quantize(layout, X)
    Yref = fmpq_mod.w4ax_gemm(layout, A2, sx2, Wp, sw, M, w.N)
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), Yref.view(torch.int16))
    assert fmpq_mod.fmpq_device_status(layout) == 0
    del g
    layout.close()
