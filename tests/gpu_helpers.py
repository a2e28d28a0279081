"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI binding and
the oracle on the same seeded inputs, and compare."""
import numpy as np

Y_TOL = 2e-3  # max relative error of Y against the oracle's fp64 epilogue (floored)


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def run_gpu(layout, X, W, want_partials=None):
    """Quantize X, pack W, run the GEMM; return host copies of every output."""
    import torch
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    Xd = to_dev(X)
    Wd = to_dev(W)
    A, sx = fmpq.fmpq_quantize(layout, Xd)
    Wp, sw = fmpq.w4_pack_weights(layout, Wd)
    M, N = X.shape[0], W.shape[0]
    Y = fmpq.w4ax_gemm(layout, A, sx, Wp, sw, M, N)
    out = dict(A=A, sx=sx, Wp=Wp, sw=sw, Y=Y)
    if want_partials is not None:
        m0, mc, n0, nc = want_partials
        out["P"] = fmpq.w4ax_gemm_partials(layout, A, Wp, M, N, m0, mc, n0, nc)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, dict(A=A, sx=sx, Wp=Wp, sw=sw)


def y_error(Y, Yref):
    """max |Y - Yref| / max(|Yref|, 1e-2 * rms(Yref)) -- elementwise relative error with a floor
    (pure elementwise relative error is undefined where Yref cancels to ~0)."""
    Y = Y.astype(np.float64)
    floor = 1e-2 * np.sqrt(np.mean(Yref ** 2)) + 1e-30
    return float(np.max(np.abs(Y - Yref) / np.maximum(np.abs(Yref), floor)))
