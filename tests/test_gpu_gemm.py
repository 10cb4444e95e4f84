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


@pytest.mark.parametrize("M", [16, 48, 130])
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
