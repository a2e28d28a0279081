"""Failure detection without a GPU fault: every device-side wait of the GEMM is bounded, and a
wait that runs out ends the kernel with FMPQ_ERR_TIMEOUT in the layout's device status word.

The test makes one wait run out on purpose through the library's test hook: the first CTA's
weight producer never issues one packed weight copy, so the converters' wait on it cannot
complete (a flag that nothing sets), and every wait is limited to a few thousand polls. The
call must return, the status must read FMPQ_ERR_TIMEOUT, the context must stay usable, and the
next normal call must be correct, including reuse of a split-K workspace whose counters the
aborted call touched."""
import time

import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl
from tests.gpu_helpers import Y_TOL, to_dev, y_error

pytestmark = pytest.mark.gpu

FMPQ_ERR_TIMEOUT = 5


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
    (1024, 2560, 512, 1, False),   # 40 output tiles: every pair runs one whole tile
    (256, 512, 2048, 2, True),     # 2 output tiles: split-K with a workspace
])
def test_withheld_copy_times_out_and_recovers(fmpq_mod, oracle_mod, M, N, K, n8, split):
    import torch
    w = wl.synthetic(M, N, K, n8=n8, seed=M + N + K)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    assert (layout.workspace_bytes(M, N) > 0) == split
    A, sx = fmpq_mod.fmpq_quantize(layout, to_dev(w.X))
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    torch.cuda.synchronize()
    assert fmpq_mod.fmpq_device_status(layout, clear=True) == 0
    t0 = time.perf_counter()
    fmpq_mod.w4ax_gemm_fault_test(layout, A, sx, Wp, sw, M, N, withhold_copy=0, poll_limit=1 << 14)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert fmpq_mod.fmpq_device_status(layout, clear=True) == FMPQ_ERR_TIMEOUT
    assert elapsed < 30.0, f"the aborted call took {elapsed:.1f} s"
    # the context is usable and the next normal call (same workspace) is correct
    ref = oracle_mod.reference(w.X, w.W, w.perm, w.mask)["Y"]
    for _ in range(2):
        Y = fmpq_mod.w4ax_gemm(layout, A, sx, Wp, sw, M, N).cpu().numpy()
        assert y_error(Y, ref) <= Y_TOL
    assert fmpq_mod.fmpq_device_status(layout, clear=True) == 0
    layout.close()


@pytest.mark.parametrize("M,N,K,n8", [
    (16, 2048, 8192, 2),    # 16 channel tiles: K split across the CTAs of a cluster
    (5, 20480, 1024, 1),    # 160 tiles, more than the CTAs: the aborted CTA also skips its later units
])
def test_few_tokens_withheld_copy_times_out_and_recovers(fmpq_mod, oracle_mod, M, N, K, n8):
    """The few-token kernel: the first CTA's first weight copy is withheld, its converters' wait
    runs out, the CTA stops before any exchange with the other splits of its cluster (whose
    waits for it run out in turn), and the next normal call is correct."""
    import torch
    w = wl.synthetic(M, N, K, n8=n8, seed=M + N + K)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    A, sx = fmpq_mod.fmpq_quantize(layout, to_dev(w.X))
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    torch.cuda.synchronize()
    assert fmpq_mod.fmpq_device_status(layout, clear=True) == 0
    t0 = time.perf_counter()
    fmpq_mod.w4ax_gemm_fault_test(layout, A, sx, Wp, sw, M, N, withhold_copy=0, poll_limit=1 << 14)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert fmpq_mod.fmpq_device_status(layout, clear=True) == FMPQ_ERR_TIMEOUT
    assert elapsed < 30.0, f"the aborted call took {elapsed:.1f} s"
    ref = oracle_mod.reference(w.X, w.W, w.perm, w.mask)["Y"]
    for _ in range(2):
        Y = fmpq_mod.w4ax_gemm(layout, A, sx, Wp, sw, M, N).cpu().numpy()
        assert y_error(Y, ref) <= Y_TOL
    assert fmpq_mod.fmpq_device_status(layout, clear=True) == 0
    layout.close()


def test_fault_test_argument_errors(fmpq_mod):
    import torch
    w = wl.synthetic(256, 256, 256, n8=0, seed=3)
    layout = fmpq_mod.Layout(w.K, w.perm, w.mask)
    A, sx = fmpq_mod.fmpq_quantize(layout, to_dev(w.X))
    Wp, sw = fmpq_mod.w4_pack_weights(layout, to_dev(w.W))
    for kwargs in (dict(withhold_copy=2, poll_limit=1 << 14),    # copy index past K/128
                   dict(withhold_copy=0, poll_limit=16)):         # too few polls
        with pytest.raises(fmpq_mod.FmpqError):
            fmpq_mod.w4ax_gemm_fault_test(layout, A, sx, Wp, sw, 256, 256, **kwargs)
    with pytest.raises(fmpq_mod.FmpqError):                     # no tokens
        fmpq_mod.w4ax_gemm_fault_test(layout, A, sx, Wp, sw, 0, 256, withhold_copy=0, poll_limit=1 << 14)
    torch.cuda.synchronize()
    assert fmpq_mod.fmpq_device_status(layout, clear=True) == 0
    layout.close()
