"""GPU: every kernel family run back to back. Ten steps are captured in a CUDA graph, each with
its own output buffers, and replayed 30 times. Every output must be bit-identical to one eager
call on the same inputs. A step may start while its predecessor's last CTAs drain, and ring
slots turn over many times per launch, so this catches races that single calls do not show.
Covered: the main GEMM (with and without split-K, ragged), the few-token GEMM, the quantizer
(row and per-token kernels), the no-alloc GEMM, QUIK asymmetric and QoQ GEMMs, and the FP16
outlier product merging into Y."""
import numpy as np
import pytest

from bit_quantized_gemm_fmpq_gb300 import workloads as wl
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu
STEPS, REPS = 10, 30


@pytest.fixture(scope="module")
def fmpq_mod():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_gemm_fmpq_gb300 import build, fmpq
    build.build()
    fmpq.load_library()
    return fmpq


def _replay_check(fmpq_mod, layout, ref, body, prep=None):
    import torch
    outs = [[torch.empty_like(t) for t in ref] for _ in range(STEPS)]

    def reset():
        if prep is not None:
            prep(outs)
        else:
            for o in outs:
                for t in o:
                    t.fill_(1)

    torch.cuda.synchronize()
    reset()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in range(STEPS):
            body(r, outs[r])
    bad = 0
    for _ in range(REPS):
        reset()
        g.replay()
        torch.cuda.synchronize()
        for o in outs:
            bad += sum(0 if torch.equal(a.view(torch.int16) if a.dtype == torch.float16 else a,
                                        b.view(torch.int16) if b.dtype == torch.float16 else b)
                       else 1 for a, b in zip(o, ref))
    del g
    assert bad == 0, f"{bad} of {REPS * STEPS * len(ref)} outputs differ"
    assert fmpq_mod.fmpq_device_status(layout) == 0


@pytest.mark.parametrize("M,N,K,n8", [(128, 8192, 8192, 8), (512, 2048, 4096, 4), (300, 784, 1024, 2),
                                      (48, 4096, 4096, 4)])
def test_fmpq_steps(fmpq_mod, M, N, K, n8):
    import torch
    w = wl.synthetic(M, N, K, n8=n8, seed=M + N)
    L = fmpq_mod.Layout(K, w.perm, w.mask)
    X = to_dev(w.X)
    Wp, sw = fmpq_mod.w4_pack_weights(L, to_dev(w.W))
    A0, s0 = fmpq_mod.fmpq_quantize(L, X)
    Y0 = fmpq_mod.w4ax_gemm(L, A0, s0, Wp, sw, M, N)
    Wc = [Wp, Wp.clone(), Wp.clone()]
    A, s = torch.empty_like(A0), torch.empty_like(s0)
    ws = L.workspace(M, N)
    _replay_check(fmpq_mod, L, [Y0], lambda r, o: (fmpq_mod.fmpq_quantize(L, X, A, s),
                                                   fmpq_mod.w4ax_gemm(L, A, s, Wc[r % 3], sw, M, N, o[0], workspace=ws)))
    _replay_check(fmpq_mod, L, [A0, s0], lambda r, o: fmpq_mod.fmpq_quantize(L, X, o[0], o[1]))
    Yn = fmpq_mod.w4ax_gemm_noalloc(L, A0, s0, Wp, sw, M, N)
    assert torch.equal(Yn.view(torch.int16), Y0.view(torch.int16))
    _replay_check(fmpq_mod, L, [Y0], lambda r, o: fmpq_mod.w4ax_gemm_noalloc(L, A0, s0, Wc[r % 3], sw, M, N, o[0]))
    L.close()


@pytest.mark.parametrize("M,N,K", [(256, 1024, 2048), (40, 2048, 4096)])
def test_variant_steps(fmpq_mod, M, N, K):
    import torch
    w = wl.synthetic(M, N, K, n8=0, seed=7 + M)
    X = to_dev(w.X)
    L = fmpq_mod.Layout(K, w.perm, np.zeros(K // 128, np.uint8))
    Wp, sw = fmpq_mod.w4_pack_weights(L, to_dev(w.W))
    wsum = fmpq_mod.w4_weight_sums(L, Wp, sw, N)
    A0, s0, z0 = fmpq_mod.fmpq_quantize_asym(L, X)
    Y0 = fmpq_mod.w4ax_gemm_asym(L, A0, s0, z0, Wp, sw, wsum, M, N)
    A, s, z = torch.empty_like(A0), torch.empty_like(s0), torch.empty_like(z0)
    ws = L.workspace(M, N, variant=True)
    _replay_check(fmpq_mod, L, [Y0], lambda r, o: (fmpq_mod.fmpq_quantize_asym(L, X, A, s, z),
                                                   fmpq_mod.w4ax_gemm_asym(L, A, s, z, Wp, sw, wsum, M, N, o[0],
                                                                           workspace=ws)))
    L.close()
    L = fmpq_mod.Layout(K, w.perm, np.ones(K // 128, np.uint8))
    Wq, s1, s2, z2 = fmpq_mod.qoq_pack_weights(L, to_dev(w.W))
    A0, s0, u0 = fmpq_mod.qoq_quantize(L, X)
    Y0 = fmpq_mod.qoq_gemm(L, A0, s0, u0, Wq, s1, s2, z2, M, N)
    A, s, u = torch.empty_like(A0), torch.empty_like(s0), torch.empty_like(u0)
    ws = L.workspace(M, N, variant=True)
    _replay_check(fmpq_mod, L, [Y0], lambda r, o: (fmpq_mod.qoq_quantize(L, X, A, s, u),
                                                   fmpq_mod.qoq_gemm(L, A, s, u, Wq, s1, s2, z2, M, N, o[0],
                                                                     workspace=ws)))
    L.close()


@pytest.mark.parametrize("M,N,n_out", [(2048, 2560, 256), (512, 1024, 384)])
def test_outlier_product_steps(fmpq_mod, M, N, n_out):
    """The product adds into Y (a TMA reduce-add at the L2): every step's Y starts from the same
    values and must end bit-identical to one eager merge."""
    rng = np.random.default_rng(M)
    K_base = 512
    L = fmpq_mod.select_layout(K_base, K_base + n_out, np.arange(K_base, dtype=np.int32),
                               np.zeros(K_base // 128, np.uint8))
    Xo = to_dev(rng.standard_normal((M, n_out)).astype(np.float16))
    Wo = to_dev((0.05 * rng.standard_normal((N, n_out))).astype(np.float16))
    Yin = to_dev(rng.standard_normal((M, N)).astype(np.float16))
    Y0 = Yin.clone()
    fmpq_mod.fmpq_outlier_product_fp16(L, Xo, Wo, Y0)

    def prep(outs):
        for o in outs:
            o[0].copy_(Yin)

    _replay_check(fmpq_mod, L, [Y0], lambda r, o: fmpq_mod.fmpq_outlier_product_fp16(L, Xo, Wo, o[0]), prep)
    L.close()
