"""The QKV projection of a draft layer (tensor-core GEMM + EPI_QKV epilogue)
against the oracle's per-head RMSNorm and rotate-half RoPE in float64.

Both tilings of the GEMM run: head pairs (two consecutive heads by 128
tokens, the epilogue reading whole head rows from the TMEM accumulator; the
default at more than 128 rows) and 128-feature tiles with the staged
epilogue.  Head counts put a pair across the k/v boundary, row
counts span one token tile, several, and ragged tails, and the deferred
input RMSNorm (row scales from per-part sums of squares) is on or off.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import block_diffusion_speculative_fc_gb300 as pkg  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402

THETA, EPS, MAXPOS = 1.0e6, 1e-6, 40000


def _lib():
    lib = pkg.load_library()
    lib.dflash_test_qkv_scratch.argtypes = [ctypes.c_int32] * 3
    lib.dflash_test_qkv_scratch.restype = ctypes.c_size_t
    lib.dflash_test_qkv.argtypes = ([ctypes.c_int32] * 6 + [ctypes.c_float] * 2 +
                                    [ctypes.c_void_p] * 10 + [ctypes.c_size_t, ctypes.c_void_p])
    lib.dflash_test_qkv.restype = ctypes.c_int
    lib.dflash_test_set_head_pairs.argtypes = [ctypes.c_int32]
    lib.dflash_test_set_head_pairs.restype = ctypes.c_int
    return lib


class Case:
    def __init__(self, M, K, H, kvh, D=128, deferred=False, seed=0):
        g = torch.Generator(device="cpu").manual_seed(seed)
        self.M, self.K, self.H, self.kvh, self.D = M, K, H, kvh, D
        self.N = (H + 2 * kvh) * D
        rnd = lambda *s: torch.randn(*s, generator=g)  # noqa: E731
        x = rnd(M, K) * 1.5
        self.ssq = None
        if deferred:
            # the deferred input norm: A = x * g, ssq[t, m] = sum of x^2 over part t
            gain = (1.0 + 0.2 * rnd(K)).to(torch.bfloat16)
            self.A = (x * gain.float()).to(torch.bfloat16)
            self.ssq = (x.double() ** 2).reshape(M, K // 128, 128).sum(-1).T.contiguous().float()
        else:
            self.A = x.to(torch.bfloat16)
        self.W = (rnd(self.N, K) / np.sqrt(K)).to(torch.bfloat16)
        self.q_gain = (1.0 + 0.3 * rnd(D)).to(torch.bfloat16)
        self.k_gain = (1.0 + 0.3 * rnd(D)).to(torch.bfloat16)
        pos = torch.randint(0, MAXPOS, (M,), generator=g, dtype=torch.int32)
        pos[0] = 0
        pos[-1] = MAXPOS - 1
        self.pos = pos

    def run(self, head_pairs):
        lib = _lib()
        assert lib.dflash_test_set_head_pairs(1 if head_pairs else 0) == 0
        try:
            dev = lambda t: t.cuda().contiguous()  # noqa: E731
            A, W, qg, kg, pos = dev(self.A), dev(self.W), dev(self.q_gain), dev(self.k_gain), dev(self.pos)
            ssq = dev(self.ssq) if self.ssq is not None else None
            q = torch.full((self.M, self.H * self.D), float("nan"), dtype=torch.bfloat16, device="cuda")
            k = torch.full((self.M, self.kvh * self.D), float("nan"), dtype=torch.bfloat16, device="cuda")
            v = torch.full_like(k, float("nan"))
            nbytes = lib.dflash_test_qkv_scratch(self.M, self.N, MAXPOS)
            scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
            st = lib.dflash_test_qkv(self.M, self.K, self.H, self.kvh, self.D, MAXPOS, THETA, EPS,
                                     A.data_ptr(), W.data_ptr(),
                                     ssq.data_ptr() if ssq is not None else None, qg.data_ptr(),
                                     kg.data_ptr(), pos.data_ptr(), q.data_ptr(), k.data_ptr(),
                                     v.data_ptr(), scratch.data_ptr(), nbytes,
                                     torch.cuda.current_stream().cuda_stream)
            assert st == 0, st
            torch.cuda.synchronize()
            assert int(scratch[:4].view(torch.int32).item()) == 0
        finally:
            lib.dflash_test_set_head_pairs(1)
        f = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
        return f(q), f(k), f(v)

    def oracle(self):
        """Y = r * A W^T, then the oracle's head RMSNorm and RoPE on q and k."""
        y = O.linear(self.A.float().numpy(), self.W.float().numpy())
        if self.ssq is not None:
            ms = self.ssq.double().numpy().sum(0) / self.K
            y = y / np.sqrt(ms + EPS)[:, None]
        M, D, H, kvh = self.M, self.D, self.H, self.kvh
        q = y[:, :H * D].reshape(M, H, D)
        k = y[:, H * D:(H + kvh) * D].reshape(M, kvh, D)
        v = y[:, (H + kvh) * D:].reshape(M, kvh, D)
        pos = self.pos.numpy().astype(np.int64)
        q = O.rope_neox(O.head_rms_norm(q, self.q_gain.float().numpy(), EPS), pos, THETA)
        k = O.rope_neox(O.head_rms_norm(k, self.k_gain.float().numpy(), EPS), pos, THETA)
        return q.reshape(M, -1), k.reshape(M, -1), v.reshape(M, -1)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


# bf16 outputs (relative rounding 2^-9 per element), fp32 accumulation and
# an fp32 RoPE table: the error per head row stays well under 1e-2 of its norm
TOL_ROW = 1e-2
TOL_ALL = 5e-3


def _check(out, ref, D):
    for name, o, r in zip("qkv", out, ref):
        assert np.isfinite(o).all(), name
        M = o.shape[0]
        oh, rh = o.reshape(M, -1, D), r.reshape(M, -1, D)
        row = np.linalg.norm(oh - rh, axis=-1) / np.maximum(np.linalg.norm(rh, axis=-1), 1e-30)
        assert row.max() <= TOL_ROW, (name, float(row.max()), np.unravel_index(row.argmax(), row.shape))
        assert _rel(o, r) <= TOL_ALL, (name, _rel(o, r))


@pytest.mark.parametrize("H,kvh", [(32, 8), (4, 3), (6, 1), (8, 2)])
@pytest.mark.parametrize("M", [1, 100, 129, 300, 640])
def test_qkv_heads(M, H, kvh):
    """(4, 3) and (6, 1): a head pair straddles the k/v boundary (the q/k
    boundary falls between pairs whenever the head total is even)."""
    case = Case(M, 512, H, kvh, seed=M * 7 + H)
    ref = case.oracle()
    outs = [case.run(hp) for hp in (True, False)]
    for out in outs:
        _check(out, ref, 128)
    for a, b in zip(*outs):
        assert _rel(a, b) <= 4e-3


@pytest.mark.parametrize("M", [64, 300, 2048])
def test_qkv_deferred_input_norm(M):
    case = Case(M, 1024, 32, 8, deferred=True, seed=M)
    ref = case.oracle()
    for hp in (True, False):
        _check(case.run(hp), ref, 128)


def test_qkv_odd_head_total_keeps_feature_tiles():
    """5 + 2*2 = 9 heads: no head-pair tiling (N is not a multiple of 256)."""
    case = Case(300, 256, 5, 2, seed=5)
    _check(case.run(True), case.oracle(), 128)


def test_qkv_head_dim_64():
    case = Case(300, 256, 8, 4, D=64, seed=9)
    _check(case.run(True), case.oracle(), 64)


def test_qkv_full_stress_shape():
    """2048 rows x 4096 inputs, 32 + 2*8 heads: the stress workload's layer
    QKV (stream-K tail tiles merged in TMEM)."""
    case = Case(2048, 4096, 32, 8, deferred=True, seed=21)
    ref = case.oracle()
    _check(case.run(True), ref, 128)
