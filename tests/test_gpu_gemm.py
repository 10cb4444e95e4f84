"""Tensor-core GEMM (tcgen05, TMA, stream-K) against a float64 matrix product.

Shapes cover every token-tile width (M = 1..300), ragged feature counts, the
K-split A operand of the fc step, paired SwiGLU tiles and the argmax
epilogue.  Tolerance: fp32 accumulation of exact bf16 products, so the error
is a few fp32 ulps times sqrt(K); 1e-5 relative is ample.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import block_diffusion_speculative_fc_gb300 as pkg  # noqa: E402


def _lib():
    lib = pkg.load_library()
    lib.dflash_test_gemm_scratch.restype = ctypes.c_size_t
    lib.dflash_test_gemm_scratch.argtypes = [ctypes.c_int32, ctypes.c_int32]
    lib.dflash_test_gemm.argtypes = [ctypes.c_int32] * 4 + [ctypes.POINTER(ctypes.c_void_p),
                                                           ctypes.c_int32, ctypes.c_void_p,
                                                           ctypes.c_int32, ctypes.c_int32,
                                                           ctypes.c_void_p, ctypes.c_void_p,
                                                           ctypes.c_void_p, ctypes.c_size_t,
                                                           ctypes.c_void_p]
    return lib


def run_gemm(A_parts, W, op, M, N):
    lib = _lib()
    K = sum(a.shape[1] for a in A_parts)
    scratch_n = lib.dflash_test_gemm_scratch(M, N)
    scratch = torch.empty(scratch_n, dtype=torch.uint8, device="cuda")
    ptrs = (ctypes.c_void_p * len(A_parts))(*[a.data_ptr() for a in A_parts])
    out = act = None
    if op == 0:
        out = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    elif op == 2:
        act = torch.zeros((M, N // 2), dtype=torch.bfloat16, device="cuda")
    else:
        out = torch.zeros(M, dtype=torch.int64, device="cuda")
    st = lib.dflash_test_gemm(M, N, K, len(A_parts), ptrs, A_parts[0].shape[1], W.data_ptr(), K, op,
                              out.data_ptr() if out is not None else None,
                              act.data_ptr() if act is not None else None, scratch.data_ptr(),
                              scratch_n, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return out, act


def reference(A_parts, W):
    A = np.concatenate([a.float().cpu().numpy().astype(np.float64) for a in A_parts], axis=1)
    return A @ W.float().cpu().numpy().astype(np.float64).T


@pytest.mark.parametrize("M", [1, 5, 16, 17, 33, 64, 100, 128, 200, 300])
@pytest.mark.parametrize("N,K", [(128, 128), (384, 1024), (3000, 512), (4096, 4096)])
def test_gemm_store_f32(M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7919 + N + K)
    A = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    W = torch.randn((N, K), generator=g, device="cuda").to(torch.bfloat16)
    out, _ = run_gemm([A], W, 0, M, N)
    ref = reference([A], W)
    err = np.abs(out.cpu().numpy() - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


@pytest.mark.parametrize("M", [16, 70])
def test_gemm_k_split_sources(M):
    g = torch.Generator(device="cuda").manual_seed(M)
    parts = [torch.randn((M, 256), generator=g, device="cuda").to(torch.bfloat16) for _ in range(5)]
    W = torch.randn((512, 1280), generator=g, device="cuda").to(torch.bfloat16)
    out, _ = run_gemm(parts, W, 0, M, 512)
    ref = reference(parts, W)
    assert np.abs(out.cpu().numpy() - ref).max() / np.abs(ref).max() < 1e-5


@pytest.mark.parametrize("M", [16, 48, 130, 385])
def test_gemm_swiglu_pairs(M):
    g = torch.Generator(device="cuda").manual_seed(100 + M)
    I, K = 768, 1024
    A = (0.05 * torch.randn((M, K), generator=g, device="cuda")).to(torch.bfloat16)
    W = torch.randn((2 * I, K), generator=g, device="cuda").to(torch.bfloat16)
    _, act = run_gemm([A], W, 2, M, 2 * I)
    y = reference([A], W)
    gate, up = y[:, :I], y[:, I:]
    ref = gate / (1 + np.exp(-gate)) * up
    got = act.float().cpu().numpy()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 5e-3


@pytest.mark.parametrize("M,V", [(16, 151936 // 8), (24, 3000)])
def test_gemm_argmax(M, V):
    g = torch.Generator(device="cuda").manual_seed(V)
    K = 1024
    A = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    W = torch.randn((V, K), generator=g, device="cuda").to(torch.bfloat16)
    keys, _ = run_gemm([A], W, 3, M, V)
    ids = (~(keys.cpu().numpy() & 0xffffffff)) & 0xffffffff
    logits = reference([A], W)
    top = np.argmax(logits, axis=1)
    srt = np.sort(logits, axis=1)
    for m in range(M):
        assert ids[m] == top[m] or srt[m, -1] - srt[m, -2] < 1e-3 * abs(srt[m, -1])


def _lib_program():
    lib = pkg.load_library()
    I32P = ctypes.POINTER(ctypes.c_int32)
    VP = ctypes.POINTER(ctypes.c_void_p)
    lib.dflash_test_program_scratch.restype = ctypes.c_size_t
    lib.dflash_test_program_scratch.argtypes = [ctypes.c_int32, ctypes.c_int32, I32P, I32P]
    lib.dflash_test_gemm_program.argtypes = [ctypes.c_int32, ctypes.c_int32, I32P, I32P, VP, VP,
                                             I32P, VP, ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_void_p]
    return lib


def run_program(M, phases):
    """phases: list of (A, W, op, out) with device tensors; one fused launch."""
    lib = _lib_program()
    n = len(phases)
    arr_i = lambda v: (ctypes.c_int32 * n)(*v)  # noqa: E731
    arr_p = lambda v: (ctypes.c_void_p * n)(*v)  # noqa: E731
    N = arr_i([ph[1].shape[0] for ph in phases])
    K = arr_i([ph[1].shape[1] for ph in phases])
    op = arr_i([ph[2] for ph in phases])
    nbytes = lib.dflash_test_program_scratch(n, M, N, op)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    st = lib.dflash_test_gemm_program(n, M, N, K, arr_p([ph[0].data_ptr() for ph in phases]),
                                      arr_p([ph[1].data_ptr() for ph in phases]), op,
                                      arr_p([ph[3].data_ptr() for ph in phases]),
                                      scratch.data_ptr(), nbytes,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return scratch[:4].view(torch.int32).item()


def _rel(got, ref):
    return np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)


@pytest.mark.parametrize("M", [1, 16, 37, 130, 300, 600])
def test_program_four_dependent_phases(M):
    """x -> bf16 y1 -> swiglu act -> bf16 y3 -> fp32 out, one cooperative launch;
    each phase is checked against a float64 product of the GPU's own input of
    that phase, so a phase that read its input too early shows at once."""
    g = torch.Generator(device="cuda").manual_seed(500 + M)
    K0, N0, I, N2, N3 = 512, 768, 640, 384, 1000
    rnd = lambda *s, sc=1.0: (sc * torch.randn(s, generator=g, device="cuda")).to(torch.bfloat16)  # noqa: E731
    x = rnd(M, K0)
    W0, W1 = rnd(N0, K0, sc=0.05), rnd(2 * I, N0, sc=0.05)
    W2, W3 = rnd(N2, I, sc=0.05), rnd(N3, N2, sc=0.05)
    y1 = torch.zeros((M, N0), dtype=torch.bfloat16, device="cuda")
    act = torch.zeros((M, I), dtype=torch.bfloat16, device="cuda")
    y3 = torch.zeros((M, N2), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((M, N3), dtype=torch.float32, device="cuda")
    err = run_program(M, [(x, W0, 1, y1), (y1, W1, 2, act), (act, W2, 1, y3), (y3, W3, 0, out)])
    assert err == 0
    r1 = reference([x], W0)
    assert _rel(y1.float().cpu().numpy(), r1) < 5e-3
    gu = reference([y1], W1)
    ra = gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]
    assert _rel(act.float().cpu().numpy(), ra) < 5e-3
    assert _rel(y3.float().cpu().numpy(), reference([act], W2)) < 5e-3
    r4 = reference([y3], W3)
    assert np.abs(out.cpu().numpy() - r4).max() / np.abs(r4).max() < 1e-5


def test_program_repeated_launches_reset_barrier():
    """Back-to-back fused launches on one scratch: the grid barrier words must
    be back at zero after each launch."""
    M = 16
    g = torch.Generator(device="cuda").manual_seed(9)
    x = torch.randn((M, 256), generator=g, device="cuda").to(torch.bfloat16)
    W0 = (0.05 * torch.randn((512, 256), generator=g, device="cuda")).to(torch.bfloat16)
    W1 = (0.05 * torch.randn((256, 512), generator=g, device="cuda")).to(torch.bfloat16)
    lib = _lib_program()
    N = (ctypes.c_int32 * 2)(512, 256)
    K = (ctypes.c_int32 * 2)(256, 512)
    op = (ctypes.c_int32 * 2)(1, 0)
    nbytes = lib.dflash_test_program_scratch(2, M, N, op)
    scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        y = torch.zeros((M, 512), dtype=torch.bfloat16, device="cuda")
        o = torch.zeros((M, 256), dtype=torch.float32, device="cuda")
        st = lib.dflash_test_gemm_program(
            2, M, N, K, (ctypes.c_void_p * 2)(x.data_ptr(), y.data_ptr()),
            (ctypes.c_void_p * 2)(W0.data_ptr(), W1.data_ptr()), op,
            (ctypes.c_void_p * 2)(y.data_ptr(), o.data_ptr()), scratch.data_ptr(), nbytes,
            torch.cuda.current_stream().cuda_stream)
        assert st == 0
        outs.append(o)
    torch.cuda.synchronize()
    ref = reference([y], W1)
    for o in outs:
        assert np.abs(o.cpu().numpy() - ref).max() / np.abs(ref).max() < 1e-5
