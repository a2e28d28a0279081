"""CPU oracle for the FMPQ W4Ax path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py``
may import this package. The product library never does, and shares no code with it.

The arithmetic lives in ``fmpq_oracle.c`` (plain C, compiled with gcc, no fast-math,
no FMA contraction); this module only builds it and marshals numpy arrays. See the C
file's header for the steps it follows and the readings it takes where the pages are
silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fmpq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
BLOCK = 128

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/liboracle.so (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=gnu11", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            lib.oracle_f32_to_f16_array.argtypes = [P, i64, P]
            lib.oracle_f16_to_f32_array.argtypes = [P, i64, P]
            lib.oracle_rmsnorm.argtypes = [P, i64, i32, i32, P, ctypes.c_float, P]
            lib.oracle_rmsnorm_sumsq.argtypes = [P, i64, i32, i32, P]
            lib.oracle_swiglu.argtypes = [P, P, i64, P]
            lib.oracle_channel_absmax.argtypes = [P, i64, i32, P]
            lib.oracle_plan_layout.argtypes = [i32, P, i32, P, P]
            lib.oracle_plan_layout.restype = i32
            lib.oracle_layout_error.argtypes = [P, i64, i32, P, P, P]
            lib.oracle_layout_error.restype = i32
            lib.oracle_plan_layout_budget.argtypes = [i32, P, P, i64, ctypes.c_double, P, P, P, P]
            lib.oracle_plan_layout_budget.restype = i32
            lib.oracle_quantize_activations.argtypes = [P, i64, i32, i32, P, P, P, P, P]
            lib.oracle_quantize_activations.restype = i32
            lib.oracle_unpack_activations.argtypes = [P, P, i32, i32, P]
            lib.oracle_unpack_activations.restype = i32
            lib.oracle_quantize_weights.argtypes = [P, i64, i32, i32, P, P, P]
            lib.oracle_quantize_weights.restype = i32
            lib.oracle_partials.argtypes = [P, P, i32, i32, i32, P]
            lib.oracle_partials_zero_ext.argtypes = [P, P, i32, i32, i32, P]
            lib.oracle_epilogue_f64.argtypes = [P, P, P, i32, i32, i32, P]
            lib.oracle_epilogue_exact.argtypes = [P, P, P, i32, i32, i32, P]
            lib.oracle_gemm_sample.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, P, P]
            lib.oracle_plane_offset.argtypes = [P, i32]
            lib.oracle_plane_offset.restype = i64
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_packed_a_bytes.argtypes = [P, i32, i32]
            lib.oracle_packed_a_bytes.restype = i64
            lib.oracle_num_threads.restype = i32
            lib.oracle_quantize_activations_asym.argtypes = [P, i64, i32, i32, P, P, P, P, P]
            lib.oracle_quantize_activations_asym.restype = i32
            lib.oracle_weight_sums.argtypes = [P, P, i32, i32, P]
            lib.oracle_epilogue_asym_f64.argtypes = [P, P, P, P, P, i32, i32, i32, P]
            lib.oracle_qoq_group_batch.argtypes = [P, i32, P, P, P]
            lib.oracle_qoq_quantize_weights.argtypes = [P, i64, i32, i32, P, P, P, P, P, P]
            lib.oracle_qoq_quantize_weights.restype = i32
            lib.oracle_qoq_quantize_activations.argtypes = [P, i64, i32, i32, P, P, P, P, P]
            lib.oracle_qoq_quantize_activations.restype = i32
            lib.oracle_epilogue_qoq_f64.argtypes = [P, P, P, P, P, P, i32, i32, i32, P]
            lib.oracle_gemm_sample_asym.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, P, P, P, P]
            lib.oracle_gemm_sample_qoq.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, P, P, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---- fp16 ----------------------------------------------------------------------------

def f32_to_f16_bits(x) -> np.ndarray:
    x = _c(x, np.float32).ravel()
    out = np.empty(x.size, dtype=np.uint16)
    _load().oracle_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16).ravel()
    out = np.empty(h.size, dtype=np.float32)
    _load().oracle_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out


# ---- quantizer -----------------------------------------------------------------------

def packed_a_bytes(mask, K: int, M: int) -> int:
    mask = _c(mask, np.uint8)
    return int(_load().oracle_packed_a_bytes(_ptr(mask), K, M))


def plane_offsets(mask) -> np.ndarray:
    """Per-block plane offset of the packed activation layout (a plane is M x 128 bytes)."""
    mask = _c(mask, np.uint8)
    return np.array([_load().oracle_plane_offset(_ptr(mask), b) for b in range(mask.size)], dtype=np.int64)


def e4m3_value(byte: int) -> float:
    """Value of an E4M3 byte, decoded from the format's definition."""
    return float(_load().oracle_e4m3_value(int(byte) & 0xFF))


def quantize_activations(X, perm, mask, want_codes: bool = True):
    """X fp16 [M, K] -> (A_packed uint8, a_scales fp16-bits uint16 [nb, M], Aq int8 [M, K] or None)."""
    Xb = _c(np.asarray(X, dtype=np.float16).view(np.uint16), np.uint16)
    M, K = Xb.shape
    perm = _c(perm, np.int32)
    mask = _c(mask, np.uint8)
    nb = K // BLOCK
    A = np.zeros(packed_a_bytes(mask, K, M), dtype=np.uint8)
    s = np.zeros((nb, M), dtype=np.uint16)
    Aq = np.zeros((M, K), dtype=np.int8) if want_codes else None
    rc = _load().oracle_quantize_activations(_ptr(Xb), K, M, K, _ptr(perm), _ptr(mask), _ptr(A), _ptr(s),
                                             _ptr(Aq) if want_codes else None)
    if rc != 0:
        raise ValueError(f"oracle_quantize_activations failed ({rc})")
    return A, s, Aq


def unpack_activations(A_packed, mask, M: int, K: int) -> np.ndarray:
    A_packed = _c(A_packed, np.uint8)
    mask = _c(mask, np.uint8)
    Aq = np.zeros((M, K), dtype=np.int8)
    rc = _load().oracle_unpack_activations(_ptr(A_packed), _ptr(mask), M, K, _ptr(Aq))
    if rc != 0:
        raise ValueError("oracle_unpack_activations failed")
    return Aq


def quantize_weights(W, perm):
    """W fp16 [N, K] -> (Wq int8 [N, K] permuted order, w_scales fp16-bits uint16 [nb, N])."""
    Wb = _c(np.asarray(W, dtype=np.float16).view(np.uint16), np.uint16)
    N, K = Wb.shape
    perm = _c(perm, np.int32)
    Wq = np.zeros((N, K), dtype=np.int8)
    s = np.zeros((K // BLOCK, N), dtype=np.uint16)
    rc = _load().oracle_quantize_weights(_ptr(Wb), K, N, K, _ptr(perm), _ptr(Wq), _ptr(s))
    if rc != 0:
        raise ValueError("oracle_quantize_weights failed")
    return Wq, s


# ---- partials and epilogue -------------------------------------------------------------

def partials(Aq, Wq, zero_ext: bool = False) -> np.ndarray:
    """P int32 [M, N, nb], exact per-block integer partial sums."""
    Aq = _c(Aq, np.int8)
    Wq = _c(Wq, np.int8)
    M, K = Aq.shape
    N = Wq.shape[0]
    P = np.zeros((M, N, K // BLOCK), dtype=np.int32)
    fn = _load().oracle_partials_zero_ext if zero_ext else _load().oracle_partials
    fn(_ptr(Aq), _ptr(Wq), M, N, K, _ptr(P))
    return P


def epilogue(P, a_scales, w_scales, exact: bool = False) -> np.ndarray:
    """Y fp64 [M, N] = sum_b sx[b, m] * sw[b, n] * P[m, n, b] (fp64 block order, or exact)."""
    P = _c(P, np.int32)
    M, N, nb = P.shape
    sx = _c(a_scales, np.uint16)
    sw = _c(w_scales, np.uint16)
    Y = np.zeros((M, N), dtype=np.float64)
    fn = _load().oracle_epilogue_exact if exact else _load().oracle_epilogue_f64
    fn(_ptr(P), _ptr(sx), _ptr(sw), M, N, nb, _ptr(Y))
    return Y


def gemm_sample(Aq, Wq, a_scales, w_scales, ms, ns, want_partials=True):
    """Per-block partials P [S, nb] (None unless want_partials) and Y [S] at output positions
    (ms[s], ns[s])."""
    Aq = _c(Aq, np.int8)
    Wq = _c(Wq, np.int8)
    M, K = Aq.shape
    N = Wq.shape[0]
    ms = _c(ms, np.int32)
    ns = _c(ns, np.int32)
    S = ms.size
    P = np.zeros((S, K // BLOCK), dtype=np.int32) if want_partials else None
    Y = np.zeros(S, dtype=np.float64)
    _load().oracle_gemm_sample(_ptr(Aq), _ptr(Wq), _ptr(_c(a_scales, np.uint16)), _ptr(_c(w_scales, np.uint16)),
                               M, N, K, S, _ptr(ms), _ptr(ns), _ptr(P) if P is not None else None, _ptr(Y))
    return P, Y


def reference(X, W, perm, mask):
    """Whole path on the CPU for small shapes: returns a dict of every intermediate."""
    A, sx, Aq = quantize_activations(X, perm, mask)
    Wq, sw = quantize_weights(W, perm)
    P = partials(Aq, Wq)
    Y = epilogue(P, sx, sw)
    return dict(A_packed=A, a_scales=sx, Aq=Aq, Wq=Wq, w_scales=sw, P=P, Y=Y)


# ---------------------------------------------------------------------- calibration (offline)

def channel_absmax(X) -> np.ndarray:
    """fp16 bits of each channel's absolute maximum over the rows of X [T][K] (float16)."""
    X = np.ascontiguousarray(np.asarray(X, dtype=np.float16)).view(np.uint16)
    T, K = X.shape
    out = np.empty(K, dtype=np.uint16)
    _load().oracle_channel_absmax(_ptr(X), T, K, _ptr(out))
    return out


def plan_layout(stat, n8: int):
    """(perm int32 [K], mask uint8 [K/128]) from per-channel statistics; see fmpq_oracle.c."""
    stat = np.ascontiguousarray(np.asarray(stat).astype(np.uint32))
    K = stat.size
    perm = np.empty(K, dtype=np.int32)
    mask = np.empty(K // BLOCK, dtype=np.uint8)
    if _load().oracle_plan_layout(K, _ptr(stat), int(n8), _ptr(perm), _ptr(mask)) != 0:
        raise ValueError("bad calibration arguments")
    return perm, mask


def layout_error(Xc, perm, mask) -> float:
    """Largest relative quantization error ||x - xhat|| / ||x|| over calibration tokens Xc
    (fp16 [T, K], input channel order) under the layout (perm, mask)."""
    Xc = _c(np.asarray(Xc, dtype=np.float16).view(np.uint16), np.uint16)
    T, K = Xc.shape
    err = np.zeros(1, dtype=np.float64)
    if _load().oracle_layout_error(_ptr(Xc), T, K, _ptr(_c(perm, np.int32)), _ptr(_c(mask, np.uint8)), _ptr(err)) != 0:
        raise ValueError("bad layout")
    return float(err[0])


def plan_layout_budget(stat, Xc, eps: float):
    """The smallest n8 whose planned layout keeps layout_error within eps on Xc (n8 = K/128
    when none does): returns (n8, err, perm, mask)."""
    stat = _c(stat, np.uint32)
    Xc = _c(np.asarray(Xc, dtype=np.float16).view(np.uint16), np.uint16)
    T, K = Xc.shape
    perm = np.empty(K, dtype=np.int32)
    mask = np.empty(K // BLOCK, dtype=np.uint8)
    n8 = np.zeros(1, dtype=np.int32)
    err = np.zeros(1, dtype=np.float64)
    if _load().oracle_plan_layout_budget(K, _ptr(stat), _ptr(Xc), T, ctypes.c_double(eps), _ptr(n8), _ptr(err),
                                         _ptr(perm), _ptr(mask)) != 0:
        raise ValueError("bad arguments")
    return int(n8[0]), float(err[0]), perm, mask

def outlier_blocks(K: int, fraction: float) -> int:
    """ceil(round(fraction*K) / 128), halves rounded away from zero, at most K/128."""
    n_out = int(np.floor(fraction * K + 0.5))
    return min((n_out + BLOCK - 1) // BLOCK, K // BLOCK)


def rmsnorm_sumsq(X) -> np.ndarray:
    """T[m] = the exact sum of the squares of fp16 row X[m], rounded once to fp32 (nearest,
    ties to even); float32 [M]."""
    X = np.ascontiguousarray(np.asarray(X, dtype=np.float16)).view(np.uint16)
    M, K = X.shape
    T = np.empty(M, dtype=np.float32)
    _load().oracle_rmsnorm_sumsq(_ptr(X), K, M, K, _ptr(T))
    return T


def rmsnorm(X, gamma, eps: float) -> np.ndarray:
    """RMSNorm of fp16 X [M][K] with fp16 gamma [K] (input channel order): r = 1/sqrt(T/K + eps)
    with T the exact sum of squares rounded once to fp32; returns float16 [M][K]."""
    X = np.ascontiguousarray(np.asarray(X, dtype=np.float16)).view(np.uint16)
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float16)).view(np.uint16)
    M, K = X.shape
    Y = np.empty((M, K), dtype=np.uint16)
    _load().oracle_rmsnorm(_ptr(X), K, M, K, _ptr(g), ctypes.c_float(eps), _ptr(Y))
    return Y.view(np.float16)


def swiglu(G, U) -> np.ndarray:
    """h = fp16_rn(g * u / (1 + e^-g)) elementwise for fp16 arrays G, U of one shape."""
    G = np.ascontiguousarray(np.asarray(G, dtype=np.float16)).view(np.uint16)
    U = np.ascontiguousarray(np.asarray(U, dtype=np.float16)).view(np.uint16)
    assert G.shape == U.shape
    H = np.empty(G.shape, dtype=np.uint16)
    _load().oracle_swiglu(_ptr(G), _ptr(U), G.size, _ptr(H))
    return H.view(np.float16)


# ---------------------------------------------------------------------- outlier split (QUIK)

def quik_reference(X, W, base_cols, out_cols):
    """QUIK explainer, "第二步: 前向传播": the base columns go through the INT4 path (all blocks
    INT4, channels in the given order), the outlier columns stay FP16; Y is the sum. Returns
    (Y_base, Y_outlier) in float64."""
    base_cols = np.asarray(base_cols, dtype=np.int64)
    out_cols = np.asarray(out_cols, dtype=np.int64)
    Xb = np.ascontiguousarray(np.asarray(X, dtype=np.float16)[:, base_cols])
    Wb = np.ascontiguousarray(np.asarray(W, dtype=np.float16)[:, base_cols])
    K = base_cols.size
    ident = np.arange(K, dtype=np.int32)
    mask = np.zeros(K // BLOCK, dtype=np.uint8)
    _, sx, Aq = quantize_activations(Xb, ident, mask)
    Wq, sw = quantize_weights(Wb, ident)
    Y_base = epilogue(partials(Aq, Wq), sx, sw)
    Xo = np.asarray(X, dtype=np.float16)[:, out_cols].astype(np.float64)
    Wo = np.asarray(W, dtype=np.float16)[:, out_cols].astype(np.float64)
    return Y_base, Xo @ Wo.T


# ---------------------------------------------------------------------- QUIK asymmetric activations

def quantize_activations_asym(X, perm):
    """QUIK explainer, "反量化背后的数学": X fp16 [M, K] -> (A_packed uint8 (one plane per block),
    a_scales, a_zeros (fp16 bits uint16 [nb, M]), Aq int8 [M, K] codes 0..15, permuted order)."""
    Xb = _c(np.asarray(X, dtype=np.float16).view(np.uint16), np.uint16)
    M, K = Xb.shape
    perm = _c(perm, np.int32)
    nb = K // BLOCK
    A = np.zeros(nb * M * BLOCK, dtype=np.uint8)
    s = np.zeros((nb, M), dtype=np.uint16)
    z = np.zeros((nb, M), dtype=np.uint16)
    Aq = np.zeros((M, K), dtype=np.int8)
    if _load().oracle_quantize_activations_asym(_ptr(Xb), K, M, K, _ptr(perm), _ptr(A), _ptr(s), _ptr(z), _ptr(Aq)):
        raise ValueError("oracle_quantize_activations_asym failed")
    return A, s, z, Aq


def weight_sums(Wq, w_scales) -> np.ndarray:
    """wsum float32 [nb, N] = sw[b, n] * sum of the block's weight codes."""
    Wq = _c(Wq, np.int8)
    N, K = Wq.shape
    out = np.zeros((K // BLOCK, N), dtype=np.float32)
    _load().oracle_weight_sums(_ptr(Wq), _ptr(_c(w_scales, np.uint16)), N, K, _ptr(out))
    return out


def epilogue_asym(P, a_scales, a_zeros, w_scales, wsum) -> np.ndarray:
    """Y fp64 [M, N] = sum_b (sx sw P + z wsum), block order."""
    P = _c(P, np.int32)
    M, N, nb = P.shape
    Y = np.zeros((M, N), dtype=np.float64)
    _load().oracle_epilogue_asym_f64(_ptr(P), _ptr(_c(a_scales, np.uint16)), _ptr(_c(a_zeros, np.uint16)),
                                     _ptr(_c(w_scales, np.uint16)), _ptr(_c(wsum, np.float32)), M, N, nb, _ptr(Y))
    return Y


def asym_reference(X, W, perm):
    """Whole QUIK-asymmetric path on the CPU (every block 4-bit): dict of every intermediate."""
    A, sx, z, Aq = quantize_activations_asym(X, perm)
    Wq, sw = quantize_weights(W, perm)
    wsum = weight_sums(Wq, sw)
    P = partials(Aq, Wq)
    Y = epilogue_asym(P, sx, z, sw, wsum)
    return dict(A_packed=A, a_scales=sx, a_zeros=z, Aq=Aq, Wq=Wq, w_scales=sw, wsum=wsum, P=P, Y=Y)


# ---------------------------------------------------------------------- QoQ progressive group quantization

def qoq_group(q8):
    """One or more groups of 128 INT8 values [G, 128] -> (s2 [G], z2 [G], q4 uint8 [G, 128])."""
    q8 = _c(np.atleast_2d(q8), np.int8)
    G = q8.shape[0]
    s2 = np.zeros(G, dtype=np.int32)
    z2 = np.zeros(G, dtype=np.int32)
    q4 = np.zeros((G, BLOCK), dtype=np.uint8)
    _load().oracle_qoq_group_batch(_ptr(q8), G, _ptr(s2), _ptr(z2), _ptr(q4))
    return s2, z2, q4


def qoq_quantize_weights(W, perm):
    """W fp16 [N, K] -> dict(q8 int8 [N, K], q4 uint8 [N, K] (permuted order), s1 fp16 bits [N],
    s2 uint8 [nb, N], z2 uint8 [nb, N])."""
    Wb = _c(np.asarray(W, dtype=np.float16).view(np.uint16), np.uint16)
    N, K = Wb.shape
    nb = K // BLOCK
    out = dict(q8=np.zeros((N, K), np.int8), q4=np.zeros((N, K), np.uint8), s1=np.zeros(N, np.uint16),
               s2=np.zeros((nb, N), np.uint8), z2=np.zeros((nb, N), np.uint8))
    if _load().oracle_qoq_quantize_weights(_ptr(Wb), K, N, K, _ptr(_c(perm, np.int32)), _ptr(out["q8"]),
                                           _ptr(out["q4"]), _ptr(out["s1"]), _ptr(out["s2"]), _ptr(out["z2"])):
        raise ValueError("oracle_qoq_quantize_weights failed")
    return out


def qoq_quantize_activations(X, perm):
    """X fp16 [M, K] -> (A_packed uint8 (two planes per block), a_scales fp16 bits [M],
    a_sums int32 [nb, M], Aq int8 [M, K])."""
    Xb = _c(np.asarray(X, dtype=np.float16).view(np.uint16), np.uint16)
    M, K = Xb.shape
    nb = K // BLOCK
    A = np.zeros(2 * nb * M * BLOCK, dtype=np.uint8)
    s = np.zeros(M, dtype=np.uint16)
    sums = np.zeros((nb, M), dtype=np.int32)
    Aq = np.zeros((M, K), dtype=np.int8)
    if _load().oracle_qoq_quantize_activations(_ptr(Xb), K, M, K, _ptr(_c(perm, np.int32)), _ptr(A), _ptr(s),
                                               _ptr(sums), _ptr(Aq)):
        raise ValueError("oracle_qoq_quantize_activations failed")
    return A, s, sums, Aq


def partials_u4(Aq, q4) -> np.ndarray:
    """P int32 [M, N, nb] with unsigned 4-bit weight codes."""
    Aq = _c(Aq, np.int8)
    M, K = Aq.shape
    N = q4.shape[0]
    Wq = _c(np.asarray(q4).astype(np.int8), np.int8)    # 0..15 fits int8
    P = np.zeros((M, N, K // BLOCK), dtype=np.int32)
    _load().oracle_partials(_ptr(Aq), _ptr(Wq), M, N, K, _ptr(P))
    return P


def epilogue_qoq(P, a_scales, a_sums, s1, s2, z2) -> np.ndarray:
    P = _c(P, np.int32)
    M, N, nb = P.shape
    Y = np.zeros((M, N), dtype=np.float64)
    _load().oracle_epilogue_qoq_f64(_ptr(P), _ptr(_c(a_scales, np.uint16)), _ptr(_c(a_sums, np.int32)),
                                    _ptr(_c(s1, np.uint16)), _ptr(_c(s2, np.uint8)), _ptr(_c(z2, np.uint8)),
                                    M, N, nb, _ptr(Y))
    return Y


def qoq_reference(X, W, perm):
    """Whole QoQ W4A8 path on the CPU: dict of every intermediate."""
    A, sx, sums, Aq = qoq_quantize_activations(X, perm)
    w = qoq_quantize_weights(W, perm)
    P = partials_u4(Aq, w["q4"])
    Y = epilogue_qoq(P, sx, sums, w["s1"], w["s2"], w["z2"])
    return dict(A_packed=A, a_scales=sx, a_sums=sums, Aq=Aq, P=P, Y=Y, **w)


def gemm_sample_asym(Aq, Wq, a_scales, a_zeros, w_scales, wsum, ms, ns):
    """QUIK asymmetric GEMM at sampled positions: (P [S, nb], Y [S])."""
    Aq, Wq = _c(Aq, np.int8), _c(Wq, np.int8)
    M, K = Aq.shape
    N = Wq.shape[0]
    ms, ns = _c(ms, np.int32), _c(ns, np.int32)
    P = np.zeros((ms.size, K // BLOCK), dtype=np.int32)
    Y = np.zeros(ms.size, dtype=np.float64)
    _load().oracle_gemm_sample_asym(_ptr(Aq), _ptr(Wq), _ptr(_c(a_scales, np.uint16)), _ptr(_c(a_zeros, np.uint16)),
                                    _ptr(_c(w_scales, np.uint16)), _ptr(_c(wsum, np.float32)), M, N, K, ms.size,
                                    _ptr(ms), _ptr(ns), _ptr(P), _ptr(Y))
    return P, Y


def gemm_sample_qoq(Aq, q4, a_scales, a_sums, s1, s2, z2, ms, ns):
    """QoQ W4A8 GEMM at sampled positions: (P [S, nb], Y [S])."""
    Aq, q4 = _c(Aq, np.int8), _c(q4, np.uint8)
    M, K = Aq.shape
    N = q4.shape[0]
    ms, ns = _c(ms, np.int32), _c(ns, np.int32)
    P = np.zeros((ms.size, K // BLOCK), dtype=np.int32)
    Y = np.zeros(ms.size, dtype=np.float64)
    _load().oracle_gemm_sample_qoq(_ptr(Aq), _ptr(q4), _ptr(_c(a_scales, np.uint16)), _ptr(_c(a_sums, np.int32)),
                                   _ptr(_c(s1, np.uint16)), _ptr(_c(s2, np.uint8)), _ptr(_c(z2, np.uint8)), M, N, K,
                                   ms.size, _ptr(ms), _ptr(ns), _ptr(P), _ptr(Y))
    return P, Y
