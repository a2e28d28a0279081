"""GPU test of w4ax_gemm_noalloc, the GEMM entry point for callers that cannot allocate
device memory (the library supplies the split-K workspace from its own fixed device array).

Both entry points run the same deterministic kernel, so w4ax_gemm_noalloc must reproduce
w4ax_gemm's output bit for bit, on two calls in a row (the second call reuses the array the
first one left behind), and both must agree with the oracle within the parity tolerance. This
file is collected last so a run that stops at the first failure has already run every other
test."""
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


@pytest.mark.parametrize("M,N,K,n8,split", [
    (16, 512, 2048, 2, False),    # few tokens, few output tiles: split-K inside a cluster, no workspace
    (1, 1024, 4096, 3, False),    # one token, the same
    (300, 784, 1024, 2, True),    # 8 output tiles: split-K
    (1024, 2560, 512, 1, False),  # 40 output tiles: no workspace needed
])
def test_noalloc_matches_gemm(fmpq_mod, oracle_mod, M, N, K, n8, split):
    w = wl.synthetic(M, N, K, n8=n8, seed=M * 7 + N + K)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    # the split-K cases must really go through the library's fixed array
    assert (layout.workspace_bytes(M, N) > 0) == split
    A, sx = fmpq_mod.fmpq_quantize(layout, to_dev(w.X))
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    ref = fmpq_mod.w4ax_gemm(layout, A, sx, Wp, sw, M, N).cpu().numpy()
    oracle_y = oracle_mod.reference(w.X, w.W, w.perm, w.mask)["Y"]
    assert y_error(ref, oracle_y) <= Y_TOL
    for _ in range(2):
        Y = fmpq_mod.w4ax_gemm_noalloc(layout, A, sx, Wp, sw, M, N).cpu().numpy()
        assert np.array_equal(Y.view(np.uint16), ref.view(np.uint16))
        assert y_error(Y, oracle_y) <= Y_TOL
    assert fmpq_mod.fmpq_device_status(layout) == 0
    layout.close()
