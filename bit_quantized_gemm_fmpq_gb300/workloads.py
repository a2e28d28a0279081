"""Seeded synthetic inputs for the FMPQ W4Ax path (no quantization arithmetic here).

This module only draws activations ``X`` (fp16 [M, K]), weights ``W`` (fp16 [N, K]),
the channel permutation ``perm`` (int32 [K], gather form: permuted channel ``j`` is
input channel ``perm[j]``) and the outlier-block mask (uint8 [K/128], 1 = INT8 block).
Both the CUDA path and the CPU oracle consume what it returns; it holds none of the
method's arithmetic.

The recipes restate the LLM-layer workloads the COMET/FMPQ pages evaluate on
(LLaMA-family linear layers whose activations carry outliers concentrated in roughly
10% of channels -- "COMET" news page, section 1 on outlier distribution), using
synthetic data of the same shapes because no model weights or datasets are used:

* ``tiny``          16 x 512 x 512, N(0,1), channels 37 and 300 scaled x50, one INT8 block
* ``llama7b_qkv``   2048 x 4096 x 12288, 10% outlier channels x U(20,100), 4/32 INT8 blocks
* ``llama70b_down`` 4096 x 28672 x 8192, Laplace(0,1), 10% outliers x U(20,100), 27/224 INT8
* ``decode``        M in {1,8,16,32,64,128}, K = N = 8192, 10% outliers x50, block 8g+7 INT8
* ``load_balance``  4096 x 8192 x 28672, INT8 fraction in {0, .1, .25, .5}, random positions

Values are drawn in fp32 and rounded to fp16 (numpy's round-to-nearest-even cast).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK = 128  # channels per quantization block (COMET news page, section 1)

DECODE_MS = (1, 8, 16, 32, 64, 128)
LOAD_BALANCE_FRACS = (0.0, 0.10, 0.25, 0.50)


@dataclass
class Workload:
    name: str
    X: np.ndarray          # fp16 [M, K]
    W: np.ndarray          # fp16 [N, K]
    perm: np.ndarray       # int32 [K]
    mask: np.ndarray       # uint8 [K // 128]
    meta: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return int(self.X.shape[0])

    @property
    def K(self) -> int:
        return int(self.X.shape[1])

    @property
    def N(self) -> int:
        return int(self.W.shape[0])


def _normal_fp16(rng: np.random.Generator, rows: int, cols: int, std: float,
                 chunk_rows: int = 1024) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.float16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        v = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[r0:r1] = v.astype(np.float16)
    return out


def _activations(rng: np.random.Generator, M: int, K: int, dist: str,
                 outliers: np.ndarray, factors: np.ndarray, chunk_rows: int = 512) -> np.ndarray:
    """X[m, c] ~ dist, with column ``outliers[i]`` multiplied by ``factors[i]`` (fp32), then fp16."""
    X = np.empty((M, K), dtype=np.float16)
    f = np.ones(K, dtype=np.float32)
    f[outliers] = factors.astype(np.float32)
    for r0 in range(0, M, chunk_rows):
        r1 = min(M, r0 + chunk_rows)
        if dist == "normal":
            v = rng.standard_normal((r1 - r0, K), dtype=np.float32)
        elif dist == "laplace":
            v = rng.laplace(0.0, 1.0, size=(r1 - r0, K)).astype(np.float32)
        else:
            raise ValueError(dist)
        v *= f[None, :]
        X[r0:r1] = v.astype(np.float16)
    return X


def _perm_gathering(rng: np.random.Generator, K: int, outliers: np.ndarray,
                    int8_blocks: np.ndarray) -> np.ndarray:
    """Random gather permutation that places every outlier channel inside an INT8 block."""
    slots8 = np.concatenate([np.arange(b * BLOCK, (b + 1) * BLOCK) for b in np.sort(int8_blocks)]) \
        if len(int8_blocks) else np.zeros(0, dtype=np.int64)
    if len(outliers) > len(slots8):
        raise ValueError("more outlier channels than INT8 slots")
    is_out = np.zeros(K, dtype=bool)
    is_out[outliers] = True
    normal = np.flatnonzero(~is_out)
    normal = rng.permutation(normal)
    fill8 = np.concatenate([rng.permutation(outliers), normal[: len(slots8) - len(outliers)]])
    fill8 = rng.permutation(fill8)
    rest = normal[len(slots8) - len(outliers):]
    perm = np.empty(K, dtype=np.int64)
    slots4 = np.setdiff1d(np.arange(K), slots8, assume_unique=True)
    perm[slots8] = fill8
    perm[slots4] = rest
    return perm.astype(np.int32)


def synthetic(M: int, N: int, K: int, *, n8: int, outlier_frac: float = 0.10,
              outlier_lo: float = 20.0, outlier_hi: float = 100.0, dist: str = "normal",
              w_std: float = 0.02, seed: int = 0, int8_blocks=None, name: str = "synthetic",
              outliers_fill_int8: bool = False) -> Workload:
    """General recipe: outlier channels scaled by U(lo, hi) and gathered into ``n8`` INT8 blocks.

    ``outliers_fill_int8``: every channel permuted into an INT8 block is an outlier
    (the load-balance recipe); otherwise ``round(outlier_frac*K)`` fixed random channels are.
    """
    if K % BLOCK:
        raise ValueError("K must be a multiple of 128")
    nb = K // BLOCK
    srng = np.random.default_rng(seed + 1000)   # structure: outlier set, mask, perm
    vrng = np.random.default_rng(seed)          # values
    if int8_blocks is None:
        int8_blocks = np.sort(srng.choice(nb, size=n8, replace=False)) if n8 else np.zeros(0, np.int64)
    int8_blocks = np.asarray(int8_blocks, dtype=np.int64)
    mask = np.zeros(nb, dtype=np.uint8)
    mask[int8_blocks] = 1
    if outliers_fill_int8:
        perm = srng.permutation(K).astype(np.int32)
        slots8 = np.concatenate([np.arange(b * BLOCK, (b + 1) * BLOCK) for b in int8_blocks]) \
            if len(int8_blocks) else np.zeros(0, np.int64)
        outliers = np.sort(perm[slots8]).astype(np.int64)
    else:
        n_out = int(round(outlier_frac * K))
        n_out = min(n_out, len(int8_blocks) * BLOCK)
        outliers = np.sort(srng.choice(K, size=n_out, replace=False)) if n_out else np.zeros(0, np.int64)
        perm = _perm_gathering(srng, K, outliers, int8_blocks)
    if outlier_lo == outlier_hi:
        factors = np.full(len(outliers), outlier_lo, dtype=np.float32)
    else:
        factors = srng.uniform(outlier_lo, outlier_hi, size=len(outliers)).astype(np.float32)
    X = _activations(vrng, M, K, dist, outliers, factors)
    W = _normal_fp16(vrng, N, K, w_std)
    meta = dict(n8=int(mask.sum()), outliers=int(len(outliers)), dist=dist, w_std=w_std, seed=seed)
    return Workload(name, X, W, perm, mask, meta)


def tiny(seed: int = 0) -> Workload:
    """16 x 512 x 512: channels 37 and 300 scaled x50; the permutation swaps channel 37
    into block 2 (positions 256..383, which already hold channel 300) and marks block 2 INT8."""
    M, N, K = 16, 512, 512
    vrng = np.random.default_rng(seed)
    X32 = vrng.standard_normal((M, K), dtype=np.float32)
    X32[:, 37] *= np.float32(50.0)
    X32[:, 300] *= np.float32(50.0)
    X = X32.astype(np.float16)
    W = _normal_fp16(vrng, N, K, 0.02)
    perm = np.arange(K, dtype=np.int32)
    perm[37], perm[293] = 293, 37
    mask = np.array([0, 0, 1, 0], dtype=np.uint8)
    return Workload("tiny", X, W, perm, mask, dict(n8=1, outliers=2, dist="normal", w_std=0.02, seed=seed))


def llama7b_qkv(seed: int = 1, M: int = 2048) -> Workload:
    return synthetic(M, 12288, 4096, n8=4, outlier_frac=0.10, dist="normal", w_std=0.02,
                     seed=seed, name="llama7b_qkv")


def llama70b_down(seed: int = 2, M: int = 4096) -> Workload:
    return synthetic(M, 8192, 28672, n8=27, outlier_frac=0.10, dist="laplace", w_std=0.015,
                     seed=seed, name="llama70b_down")


def decode(M: int, seed: int = 3) -> Workload:
    K = N = 8192
    blocks = np.arange(7, K // BLOCK, 8)
    return synthetic(M, N, K, n8=len(blocks), outlier_frac=0.10, outlier_lo=50.0, outlier_hi=50.0,
                     dist="normal", w_std=0.02, seed=seed, int8_blocks=blocks, name=f"decode_m{M}")


def load_balance(frac: float, seed: int = 4, M: int = 4096) -> Workload:
    K, N = 8192, 28672
    n8 = int(round(frac * (K // BLOCK)))
    return synthetic(M, N, K, n8=n8, dist="normal", w_std=0.02, seed=seed,
                     outliers_fill_int8=True, name=f"load_balance_{int(round(frac * 100))}pct")
