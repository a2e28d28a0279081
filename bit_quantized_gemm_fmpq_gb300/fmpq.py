"""Thin Python binding of the C ABI in include/fmpq.h (argument marshalling only).

Every function here forwards to the CUDA library built in-tree
(bit_quantized_gemm_fmpq_gb300/_build/libfmpq_gb300.so); all the arithmetic runs in its
kernels. Torch is used only to own device memory and to supply the current CUDA stream.
If the library is missing, the first call raises ``FmpqLibraryMissing``: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfmpq_gb300.so")
BLOCK = 128
TILE_N = 256

_lib = None
_lock = threading.Lock()

STATUS = {
    0: "FMPQ_OK", 1: "FMPQ_ERR_INVALID_ARG", 2: "FMPQ_ERR_UNSUPPORTED_SHAPE", 3: "FMPQ_ERR_MISALIGNED",
    4: "FMPQ_ERR_CUDA", 5: "FMPQ_ERR_TIMEOUT", 6: "FMPQ_ERR_DEVICE", 7: "FMPQ_ERR_WORKSPACE",
}

# C-ABI symbols and their ctypes signatures (restype, argtypes)
_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "fmpq_layout_create": (_I32, [_I32, _P, _P, ctypes.POINTER(_P)]),
    "fmpq_layout_destroy": (None, [_P]),
    "fmpq_layout_k": (_I32, [_P]),
    "fmpq_layout_num_blocks": (_I32, [_P]),
    "fmpq_layout_num_int8_blocks": (_I32, [_P]),
    "fmpq_packed_a_bytes": (_SZ, [_P, _I64]),
    "fmpq_packed_w_bytes": (_SZ, [_P, _I64]),
    "fmpq_quantize": (_I32, [_P, _P, _I64, _I64, _P, _P, _P]),
    "w4_pack_weights": (_I32, [_P, _P, _I64, _I64, _P, _P, _P]),
    "w4_unpack_weights": (_I32, [_P, _P, _I64, _P, _P]),
    "w4ax_gemm_workspace_bytes": (_SZ, [_P, _I64, _I64]),
    "w4ax_gemm": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _P, _I64, _P, _SZ, _P]),
    "w4ax_gemm_noalloc": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _P, _I64, _P]),
    "w4ax_gemm_fault_test": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _P, _I64, _P, _SZ, _I32, ctypes.c_uint32, _P]),
    "w4ax_gemm_partials": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P, _P]),
    "fmpq_device_status": (_I32, [_P, ctypes.POINTER(_I32), _I32]),
    "fmpq_rmsnorm_quantize": (_I32, [_P, _P, _I64, _I64, _P, ctypes.c_float, _P, _P, _P]),
    "fmpq_swiglu_quantize": (_I32, [_P, _P, _I64, _P, _I64, _I64, _P, _P, _P]),
    "fmpq_variant_gemm_workspace_bytes": (_SZ, [_P, _I64, _I64]),
    "fmpq_quantize_asym": (_I32, [_P, _P, _I64, _I64, _P, _P, _P, _P]),
    "w4_weight_sums": (_I32, [_P, _P, _P, _I64, _P, _P]),
    "w4ax_gemm_asym": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _I64, _P, _SZ, _P]),
    "qoq_pack_weights": (_I32, [_P, _P, _I64, _I64, _P, _P, _P, _P, _P]),
    "qoq_unpack_weights": (_I32, [_P, _P, _I64, _P, _P]),
    "qoq_quantize": (_I32, [_P, _P, _I64, _I64, _P, _P, _P, _P]),
    "qoq_gemm": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _I64, _P, _SZ, _P]),
    "qoq_gemm_partials": (_I32, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P, _P]),
    "fmpq_layout_create_select": (_I32, [_I32, _I32, _P, _P, ctypes.POINTER(_P)]),
    "fmpq_outlier_gemm_fp16": (_I32, [_P, _P, _I64, _I64, _P, _I32, _P, _I64, _I64, _P, _P, _I64, _P]),
    "fmpq_quantize_split": (_I32, [_P, _P, _I64, _I64, _P, _I32, _I32, _P, _P, _P, _P, _P]),
    "fmpq_quantize_gemm": (_I32, [_P, _P, _I64, _I64, _P, _P, _P, _P, _I64, _P, _I64, _P, _I64, _P]),
    "fmpq_outlier_product_fp16": (_I32, [_P, _P, _I64, _I32, _P, _I64, _I64, _P, _I64, _P]),
    "fmpq_channel_absmax": (_I32, [_P, _I64, _I64, _I32, _P, _P]),
    "fmpq_plan_layout": (_I32, [_I32, _P, _I32, _P, _P]),
    "fmpq_plan_layout_budget": (_I32, [_I32, _P, _P, _I64, _I64, ctypes.c_double, _P, _P, _P, _P]),
    "fmpq_outlier_blocks": (_I32, [_I32, ctypes.c_double]),
    "fmpq_status_string": (ctypes.c_char_p, [_I32]),
    "fmpq_version": (_I32, []),
}


class FmpqLibraryMissing(RuntimeError):
    pass


class FmpqError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


def load_library():
    """Load the in-tree CUDA library (raises FmpqLibraryMissing when it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise FmpqLibraryMissing(
                    f"{LIB_PATH} is missing: build it with `python -m bit_quantized_gemm_fmpq_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _check(fn: str, code: int):
    if code != 0:
        raise FmpqError(fn, code)


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


class Layout:
    """Owns an fmpq_layout* (channel permutation + outlier-block mask) on the current device."""

    def __init__(self, K: int, perm, mask):
        lib = load_library()
        perm = np.ascontiguousarray(perm, dtype=np.int32)
        mask = np.ascontiguousarray(mask, dtype=np.uint8)
        if perm.shape != (K,) or mask.shape != (K // BLOCK,):
            raise ValueError("perm must have K entries and mask K/128 entries")
        h = ctypes.c_void_p()
        _check("fmpq_layout_create", lib.fmpq_layout_create(K, perm.ctypes.data, mask.ctypes.data, ctypes.byref(h)))
        self._h = h
        self._lib = lib
        self.K = K
        self.nb = K // BLOCK
        self.mask = mask.copy()
        self.perm = perm.copy()
        self._workspaces = {}

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.fmpq_layout_destroy(self._h)
            self._h = ctypes.c_void_p()
        self._workspaces = {}

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def n8(self) -> int:
        return int(self._lib.fmpq_layout_num_int8_blocks(self._h))

    def packed_a_bytes(self, M: int) -> int:
        return int(self._lib.fmpq_packed_a_bytes(self._h, M))

    def packed_w_bytes(self, N: int) -> int:
        return int(self._lib.fmpq_packed_w_bytes(self._h, N))

    def workspace_bytes(self, M: int, N: int) -> int:
        return int(self._lib.w4ax_gemm_workspace_bytes(self._h, M, N))

    def workspace(self, M: int, N: int, variant: bool = False):
        """A zero-initialised, reusable workspace tensor for (M, N) (cached per size); variant:
        for the quantization variants' GEMMs."""
        import torch
        nbytes = (int(self._lib.fmpq_variant_gemm_workspace_bytes(self._h, M, N)) if variant
                  else self.workspace_bytes(M, N))
        if nbytes == 0:
            return None
        ws = self._workspaces.get(nbytes)
        if ws is None:
            ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
            self._workspaces[nbytes] = ws
        return ws


# ---- the C-ABI entry points, same names ---------------------------------------------------

def fmpq_layout_create(K: int, perm, mask) -> Layout:
    return Layout(K, perm, mask)


def fmpq_quantize(layout: Layout, X, A_packed=None, a_scales=None, stream=None):
    """X: fp16 CUDA tensor [M, >=K] (row stride multiple of 8). Returns (A_packed u8, a_scales fp16 [nb, M])."""
    import torch
    M = X.shape[0]
    if A_packed is None:
        A_packed = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty((layout.nb, M), dtype=torch.float16, device=X.device)
    _check("fmpq_quantize", layout._lib.fmpq_quantize(layout.handle, _ptr(X), X.stride(0), M, _ptr(A_packed),
                                                        _ptr(a_scales), _stream(stream)))
    return A_packed, a_scales


def fmpq_swiglu_quantize(layout: Layout, G_perm, U_perm, A_packed=None, a_scales=None, stream=None):
    """SwiGLU (silu(g) * u, rounded once to fp16) fused with the activation quantizer; G_perm and
    U_perm fp16 [M, >=K] in the layout's permuted channel order."""
    import torch
    M = G_perm.shape[0]
    if A_packed is None:
        A_packed = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device=G_perm.device)
    if a_scales is None:
        a_scales = torch.empty((layout.nb, M), dtype=torch.float16, device=G_perm.device)
    _check("fmpq_swiglu_quantize", load_library().fmpq_swiglu_quantize(
        layout.handle, _ptr(G_perm), G_perm.stride(0), _ptr(U_perm), U_perm.stride(0), M, _ptr(A_packed),
        _ptr(a_scales), _stream(stream)))
    return A_packed, a_scales


def fmpq_rmsnorm_quantize(layout: Layout, X, gamma_perm, eps: float, A_packed=None, a_scales=None, stream=None):
    """RMSNorm of X fused with the activation quantizer (gamma in the permuted channel order)."""
    import torch
    M = X.shape[0]
    if A_packed is None:
        A_packed = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty((layout.nb, M), dtype=torch.float16, device=X.device)
    _check("fmpq_rmsnorm_quantize", load_library().fmpq_rmsnorm_quantize(
        layout.handle, _ptr(X), X.stride(0), M, _ptr(gamma_perm), ctypes.c_float(eps), _ptr(A_packed),
        _ptr(a_scales), _stream(stream)))
    return A_packed, a_scales


def w4_pack_weights(layout: Layout, W, W_packed=None, w_scales=None, stream=None):
    """W: fp16 CUDA tensor [N, >=K]. Returns (W_packed u8, w_scales fp16 [nb, N])."""
    import torch
    N = W.shape[0]
    if W_packed is None:
        W_packed = torch.empty(layout.packed_w_bytes(N), dtype=torch.uint8, device=W.device)
    if w_scales is None:
        w_scales = torch.empty((layout.nb, N), dtype=torch.float16, device=W.device)
    _check("w4_pack_weights", layout._lib.w4_pack_weights(layout.handle, _ptr(W), W.stride(0), N, _ptr(W_packed),
                                                            _ptr(w_scales), _stream(stream)))
    return W_packed, w_scales


def w4_unpack_weights(layout: Layout, W_packed, N: int, stream=None):
    import torch
    Wq = torch.empty((N, layout.K), dtype=torch.int8, device=W_packed.device)
    _check("w4_unpack_weights", layout._lib.w4_unpack_weights(layout.handle, _ptr(W_packed), N, _ptr(Wq),
                                                                _stream(stream)))
    return Wq


def w4ax_gemm(layout: Layout, A_packed, a_scales, W_packed, w_scales, M: int, N: int, Y=None, workspace=None,
              stream=None):
    """Returns Y fp16 [M, N] (or writes into the given Y [M, >=N])."""
    import torch
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=A_packed.device)
    if workspace is None:
        workspace = layout.workspace(M, N)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check("w4ax_gemm", layout._lib.w4ax_gemm(layout.handle, _ptr(A_packed), _ptr(a_scales), _ptr(W_packed),
                                                _ptr(w_scales), M, N, _ptr(Y), Y.stride(0), _ptr(workspace),
                                                ws_bytes, _stream(stream)))
    return Y


def fmpq_quantize_gemm(layout: Layout, X, W_packed, w_scales, N: int, A_packed=None, a_scales=None, Y=None,
                       workspace=None, stream=None):
    """fmpq_quantize then w4ax_gemm in one call (the GEMM's prologue and weight stream overlap the
    quantizer). Returns Y (fp16 [M, N])."""
    import torch
    M = X.shape[0]
    if A_packed is None:
        A_packed = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty((layout.nb, M), dtype=torch.float16, device=X.device)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = layout.workspace(M, N)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check("fmpq_quantize_gemm", layout._lib.fmpq_quantize_gemm(
        layout.handle, _ptr(X), X.stride(0), M, _ptr(A_packed), _ptr(a_scales), _ptr(W_packed), _ptr(w_scales), N,
        _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, _stream(stream)))
    return Y


def w4ax_gemm_fault_test(layout: Layout, A_packed, a_scales, W_packed, w_scales, M: int, N: int, withhold_copy: int,
                         poll_limit: int, Y=None, workspace=None, stream=None):
    """Debug/test of failure detection: w4ax_gemm with one packed weight copy of the first CTA
    withheld and every device wait bounded by poll_limit polls; records FMPQ_ERR_TIMEOUT."""
    import torch
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=A_packed.device)
    if workspace is None:
        workspace = layout.workspace(M, N)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check("w4ax_gemm_fault_test", layout._lib.w4ax_gemm_fault_test(
        layout.handle, _ptr(A_packed), _ptr(a_scales), _ptr(W_packed), _ptr(w_scales), M, N, _ptr(Y), Y.stride(0),
        _ptr(workspace), ws_bytes, int(withhold_copy), int(poll_limit), _stream(stream)))
    return Y


def w4ax_gemm_noalloc(layout: Layout, A_packed, a_scales, W_packed, w_scales, M: int, N: int, Y=None,
                      stream=None):
    """w4ax_gemm without a workspace argument: for callers that cannot allocate device memory,
    the library's own fixed device array serves as the split-K workspace."""
    import torch
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=A_packed.device)
    _check("w4ax_gemm_noalloc", layout._lib.w4ax_gemm_noalloc(layout.handle, _ptr(A_packed), _ptr(a_scales),
                                                                _ptr(W_packed), _ptr(w_scales), M, N, _ptr(Y),
                                                                Y.stride(0), _stream(stream)))
    return Y


def w4ax_gemm_partials(layout: Layout, A_packed, W_packed, M: int, N: int, m0: int, mcount: int, n0: int,
                       ncount: int, stream=None):
    """Exact per-block integer partial sums P int32 [mcount, ncount, nb] from the GEMM's tensor-core path."""
    import torch
    P = torch.zeros((mcount, ncount, layout.nb), dtype=torch.int32, device=A_packed.device)
    _check("w4ax_gemm_partials", layout._lib.w4ax_gemm_partials(layout.handle, _ptr(A_packed), _ptr(W_packed), M, N,
                                                                  m0, mcount, n0, ncount, _ptr(P), _stream(stream)))
    return P


def fmpq_device_status(layout: Layout, clear: bool = True) -> int:
    code = ctypes.c_int32(0)
    _check("fmpq_device_status", layout._lib.fmpq_device_status(layout.handle, ctypes.byref(code), int(clear)))
    return int(code.value)


def fmpq_version() -> int:
    return int(load_library().fmpq_version())


# ---------------------------------------------------------------------- calibration (offline)

def fmpq_channel_absmax(X, out=None, stream=None):
    """Per-channel absolute maximum of fp16 X [T][K] (rows may be strided): uint32 [K] of fp16
    bit patterns, computed on the GPU."""
    import torch
    T, K = X.shape
    if out is None:
        out = torch.empty(K, dtype=torch.int32, device=X.device)
    _check("fmpq_channel_absmax", load_library().fmpq_channel_absmax(_ptr(X), X.stride(0), T, K, _ptr(out),
                                                                         _stream(stream)))
    return out


def fmpq_plan_layout(absmax, n8: int):
    """Host planner: (perm int32 [K], mask uint8 [K/128]) from per-channel statistics."""
    a = np.ascontiguousarray(np.asarray(absmax).astype(np.uint32))
    K = a.size
    perm = np.empty(K, dtype=np.int32)
    mask = np.empty(K // BLOCK, dtype=np.uint8)
    _check("fmpq_plan_layout", load_library().fmpq_plan_layout(K, a.ctypes.data, n8, perm.ctypes.data,
                                                                   mask.ctypes.data))
    return perm, mask


def fmpq_plan_layout_budget(absmax, X_calib, eps: float):
    """Host planner with an error budget: the fewest INT8 blocks whose layout keeps the largest
    relative quantization error of the calibration tokens X_calib (fp16 [T, K], host) within
    eps. Returns (n8, err, perm int32 [K], mask uint8 [K/128])."""
    a = np.ascontiguousarray(np.asarray(absmax).astype(np.uint32))
    Xc = np.ascontiguousarray(np.asarray(X_calib, dtype=np.float16))
    T, K = Xc.shape
    perm = np.empty(K, dtype=np.int32)
    mask = np.empty(K // BLOCK, dtype=np.uint8)
    n8 = np.zeros(1, dtype=np.int32)
    err = np.zeros(1, dtype=np.float64)
    _check("fmpq_plan_layout_budget", load_library().fmpq_plan_layout_budget(
        K, a.ctypes.data, Xc.ctypes.data, T, K, float(eps), n8.ctypes.data, err.ctypes.data, perm.ctypes.data,
        mask.ctypes.data))
    return int(n8[0]), float(err[0]), perm, mask


def fmpq_outlier_blocks(K: int, fraction: float) -> int:
    n8 = int(load_library().fmpq_outlier_blocks(K, fraction))
    if n8 < 0:
        raise ValueError("K must be a multiple of 128 in [128, 32768] and fraction in [0, 1]")
    return n8


# ---------------------------------------------------------------------- outlier split (QUIK)

def select_layout(K: int, K_in: int, select, mask) -> "Layout":
    """A Layout over K channels selected (distinct indices < K_in) from rows of K_in channels."""
    lib = load_library()
    sel = np.ascontiguousarray(select, dtype=np.int32)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    if sel.shape != (K,) or mask.shape != (K // BLOCK,):
        raise ValueError("select must have K entries and mask K/128 entries")
    h = ctypes.c_void_p()
    _check("fmpq_layout_create_select",
           lib.fmpq_layout_create_select(K, K_in, sel.ctypes.data, mask.ctypes.data, ctypes.byref(h)))
    lay = Layout.__new__(Layout)
    lay._h = h
    lay._lib = lib
    lay.K = K
    lay.nb = K // BLOCK
    lay.mask = mask.copy()
    lay.perm = sel.copy()
    lay._workspaces = {}
    return lay


def fmpq_outlier_gemm_fp16(layout: "Layout", X, cols, W_out, Y, X_out=None, stream=None):
    """Y += X[:, cols] @ W_out^T in FP16 (the outlier path of an outlier split); `layout` is the
    base part's layout (its device status word records device-side timeouts)."""
    import torch
    M = X.shape[0]
    n_out = cols.numel()
    N = W_out.shape[0]
    if X_out is None:
        X_out = torch.empty((M, n_out), dtype=torch.float16, device=X.device)
    _check("fmpq_outlier_gemm_fp16", load_library().fmpq_outlier_gemm_fp16(
        layout.handle, _ptr(X), X.stride(0), M, _ptr(cols), n_out, _ptr(W_out), W_out.stride(0), N, _ptr(X_out), _ptr(Y),
        Y.stride(0), _stream(stream)))
    return Y


def fmpq_quantize_split(layout: "Layout", X, cols, asym: bool = False, A_packed=None, a_scales=None, a_zeros=None,
                        X_out=None, stream=None):
    """The quantizer (symmetric, or asymmetric with asym=True) that also splits off X[:, cols]
    into X_out in the same pass. Returns (A_packed, a_scales, a_zeros or None, X_out)."""
    import torch
    M = X.shape[0]
    n_out = cols.numel()
    if A_packed is None:
        A_packed = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty((layout.nb, M), dtype=torch.float16, device=X.device)
    if asym and a_zeros is None:
        a_zeros = torch.empty((layout.nb, M), dtype=torch.float16, device=X.device)
    if X_out is None:
        X_out = torch.empty((M, n_out), dtype=torch.float16, device=X.device)
    _check("fmpq_quantize_split", layout._lib.fmpq_quantize_split(
        layout.handle, _ptr(X), X.stride(0), M, _ptr(cols), n_out, 1 if asym else 0, _ptr(A_packed), _ptr(a_scales),
        _ptr(a_zeros if asym else None), _ptr(X_out), _stream(stream)))
    return A_packed, a_scales, (a_zeros if asym else None), X_out


def fmpq_outlier_product_fp16(layout: "Layout", X_out, W_out, Y, stream=None):
    """Y = fp16(Y + fp16(X_out @ W_out^T)) with X_out already split off (fmpq_quantize_split)."""
    M, n_out = X_out.shape
    N = W_out.shape[0]
    _check("fmpq_outlier_product_fp16", load_library().fmpq_outlier_product_fp16(
        layout.handle, _ptr(X_out), M, n_out, _ptr(W_out), W_out.stride(0), N, _ptr(Y), Y.stride(0), _stream(stream)))
    return Y


# ---- quantization variants: QUIK asymmetric activations, QoQ progressive group quantization

def _gemm_ws(layout: Layout, M: int, N: int, workspace):
    if workspace is None:
        workspace = layout.workspace(M, N, variant=True)
    return workspace, (workspace.numel() if workspace is not None else 0)


def fmpq_quantize_asym(layout: Layout, X, A_packed=None, a_scales=None, a_zeros=None, stream=None):
    """Asymmetric 4-bit activations. Returns (A_packed u8, a_scales fp16 [nb, M], a_zeros fp16 [nb, M])."""
    import torch
    M = X.shape[0]
    if A_packed is None:
        A_packed = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty((layout.nb, M), dtype=torch.float16, device=X.device)
    if a_zeros is None:
        a_zeros = torch.empty((layout.nb, M), dtype=torch.float16, device=X.device)
    _check("fmpq_quantize_asym", layout._lib.fmpq_quantize_asym(layout.handle, _ptr(X), X.stride(0), M, _ptr(A_packed),
                                                                  _ptr(a_scales), _ptr(a_zeros), _stream(stream)))
    return A_packed, a_scales, a_zeros


def w4_weight_sums(layout: Layout, W_packed, w_scales, N: int, out=None, stream=None):
    """w_sums fp32 [nb, N] = w_scales * (sum of each block's weight codes)."""
    import torch
    if out is None:
        out = torch.empty((layout.nb, N), dtype=torch.float32, device=W_packed.device)
    _check("w4_weight_sums", layout._lib.w4_weight_sums(layout.handle, _ptr(W_packed), _ptr(w_scales), N, _ptr(out),
                                                          _stream(stream)))
    return out


def w4ax_gemm_asym(layout: Layout, A_packed, a_scales, a_zeros, W_packed, w_scales, w_sums, M: int, N: int,
                   Y=None, workspace=None, stream=None):
    import torch
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=A_packed.device)
    workspace, ws_bytes = _gemm_ws(layout, M, N, workspace)
    _check("w4ax_gemm_asym", layout._lib.w4ax_gemm_asym(
        layout.handle, _ptr(A_packed), _ptr(a_scales), _ptr(a_zeros), _ptr(W_packed), _ptr(w_scales), _ptr(w_sums),
        M, N, _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, _stream(stream)))
    return Y


def qoq_pack_weights(layout: Layout, W, W_packed=None, stream=None):
    """Returns (W_packed u8, ch_scales fp16 [N], grp_scales u8 [nb, N], grp_zeros u8 [nb, N])."""
    import torch
    N = W.shape[0]
    if W_packed is None:
        W_packed = torch.empty(layout.packed_w_bytes(N), dtype=torch.uint8, device=W.device)
    s1 = torch.empty(N, dtype=torch.float16, device=W.device)
    s2 = torch.empty((layout.nb, N), dtype=torch.uint8, device=W.device)
    z2 = torch.empty((layout.nb, N), dtype=torch.uint8, device=W.device)
    _check("qoq_pack_weights", layout._lib.qoq_pack_weights(layout.handle, _ptr(W), W.stride(0), N, _ptr(W_packed),
                                                              _ptr(s1), _ptr(s2), _ptr(z2), _stream(stream)))
    return W_packed, s1, s2, z2


def qoq_unpack_weights(layout: Layout, W_packed, N: int, stream=None):
    import torch
    q4 = torch.empty((N, layout.K), dtype=torch.uint8, device=W_packed.device)
    _check("qoq_unpack_weights", layout._lib.qoq_unpack_weights(layout.handle, _ptr(W_packed), N, _ptr(q4),
                                                                  _stream(stream)))
    return q4


def qoq_quantize(layout: Layout, X, A_packed=None, a_scales=None, a_sums=None, stream=None):
    """Per-token INT8 activations. Returns (A_packed u8, a_scales fp16 [M], a_sums int32 [nb, M])."""
    import torch
    M = X.shape[0]
    if A_packed is None:
        A_packed = torch.empty(layout.packed_a_bytes(M), dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty(M, dtype=torch.float16, device=X.device)
    if a_sums is None:
        a_sums = torch.empty((layout.nb, M), dtype=torch.int32, device=X.device)
    _check("qoq_quantize", layout._lib.qoq_quantize(layout.handle, _ptr(X), X.stride(0), M, _ptr(A_packed),
                                                      _ptr(a_scales), _ptr(a_sums), _stream(stream)))
    return A_packed, a_scales, a_sums


def qoq_gemm(layout: Layout, A_packed, a_scales, a_sums, W_packed, ch_scales, grp_scales, grp_zeros, M: int,
             N: int, Y=None, workspace=None, stream=None):
    import torch
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float16, device=A_packed.device)
    workspace, ws_bytes = _gemm_ws(layout, M, N, workspace)
    _check("qoq_gemm", layout._lib.qoq_gemm(
        layout.handle, _ptr(A_packed), _ptr(a_scales), _ptr(a_sums), _ptr(W_packed), _ptr(ch_scales),
        _ptr(grp_scales), _ptr(grp_zeros), M, N, _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, _stream(stream)))
    return Y


def qoq_gemm_partials(layout: Layout, A_packed, W_packed, M: int, N: int, m0: int, mcount: int, n0: int,
                      ncount: int, stream=None):
    import torch
    P = torch.zeros((mcount, ncount, layout.nb), dtype=torch.int32, device=A_packed.device)
    _check("qoq_gemm_partials", layout._lib.qoq_gemm_partials(layout.handle, _ptr(A_packed), _ptr(W_packed), M, N,
                                                                m0, mcount, n0, ncount, _ptr(P), _stream(stream)))
    return P
