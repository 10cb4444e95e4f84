"""The bf16 attention kernels on their own against the oracle's block attention.

dflash_test_attention runs one attention launch (the tcgen05 kernel or the
mma.sync kernels) on random paged K/V; every checked request is compared
with oracle.block_attention in float64 on the same bf16 values: context keys
gathered through the page table (the ring for a draft window), the S block
keys, the layer's sliding window.  Shapes cover every query-row padding of
the tcgen05 kernel (R = 8..64 rows per (request, KV head)), ragged and empty
contexts, contexts cut into many splits (the ticketed merge), windows, and
the stress workload's full size on sampled requests.
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

D, PAGE = 128, 64


def _lib():
    lib = pkg.load_library()
    lib.dflash_test_attention_scratch.argtypes = [ctypes.c_int32] * 4
    lib.dflash_test_attention_scratch.restype = ctypes.c_size_t
    lib.dflash_test_attention.argtypes = ([ctypes.c_int32] * 9 + [ctypes.c_void_p] * 8 +
                                          [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                           ctypes.c_void_p])
    lib.dflash_test_attention.restype = ctypes.c_int
    return lib


class Case:
    def __init__(self, B, S, H, kvh, ctx, window=0, draft_window=0, seed=0, q_scale=2.0,
                 extra_pages=1):
        g = torch.Generator(device="cpu").manual_seed(seed)
        self.B, self.S, self.H, self.kvh = B, S, H, kvh
        self.window, self.draft_window = window, draft_window
        self.kv = np.asarray(ctx, dtype=np.int64)
        if draft_window > 0:
            self.ppr = (draft_window + PAGE - 1) // PAGE + 1 + extra_pages
            used = np.full(B, self.ppr)
        else:
            self.ppr = int(max(1, (self.kv.max() + PAGE - 1) // PAGE)) + extra_pages
            used = (self.kv + PAGE - 1) // PAGE
        # the pages a request uses, drawn at random from one pool; unused
        # table entries point at page 0 (never read)
        self.n_pages = int(max(1, used.sum()))
        perm = torch.randperm(self.n_pages, generator=g).to(torch.int32)
        table = torch.zeros(B, self.ppr, dtype=torch.int32)
        at = 0
        for b in range(B):
            table[b, :used[b]] = perm[at:at + used[b]]
            at += int(used[b])
        self.page_table = table
        rnd = lambda *shape: torch.randn(*shape, generator=g)  # noqa: E731
        self.q = (rnd(B * S, H, D) * q_scale).to(torch.bfloat16)
        self.kb = rnd(B * S, kvh, D).to(torch.bfloat16)
        self.vb = rnd(B * S, kvh, D).to(torch.bfloat16)
        self.kc = rnd(self.n_pages * PAGE, kvh, D).to(torch.bfloat16)
        self.vc = rnd(self.n_pages * PAGE, kvh, D).to(torch.bfloat16)

    def run(self, kernel):
        lib = _lib()
        dev = lambda t: t.cuda().contiguous()  # noqa: E731
        q, kb, vb, kc, vc = dev(self.q), dev(self.kb), dev(self.vb), dev(self.kc), dev(self.vc)
        pt = dev(self.page_table.reshape(-1))
        kvl = torch.as_tensor(self.kv, dtype=torch.int32).cuda()
        out = torch.full_like(q, float("nan"))
        nbytes = lib.dflash_test_attention_scratch(self.B, self.H, self.kvh, self.S)
        scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = lib.dflash_test_attention(
            kernel, self.B, self.S, self.H, self.kvh, self.ppr, self.n_pages, self.window,
            self.draft_window, q.data_ptr(), kb.data_ptr(), vb.data_ptr(), kc.data_ptr(),
            vc.data_ptr(), pt.data_ptr(), kvl.data_ptr(), out.data_ptr(), scratch.data_ptr(),
            nbytes, err.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0, st
        torch.cuda.synchronize()
        assert int(err.item()) == 0, hex(int(err.item()))
        return out.float().cpu().numpy().reshape(self.B, self.S, self.H, D)

    def oracle(self, b):
        """oracle.block_attention of request b over the rows the cache keeps."""
        kv = int(self.kv[b])
        lo = max(0, kv - self.draft_window) if self.draft_window > 0 else 0
        pos = np.arange(lo, kv)
        lp = pos // PAGE
        if self.draft_window > 0:
            lp = lp % self.ppr
        pages = self.page_table[b].numpy()[lp]
        rows = pages.astype(np.int64) * PAGE + pos % PAGE
        kc = self.kc.float().numpy()[rows]
        vc = self.vc.float().numpy()[rows]
        sl = slice(b * self.S, (b + 1) * self.S)
        q = self.q.float().numpy()[sl]
        kbb, vbb = self.kb.float().numpy()[sl], self.vb.float().numpy()[sl]
        q_pos = kv + np.arange(self.S)
        return O.block_attention(q, kc, vc, kbb, vbb, q_pos, pos, self.window)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


# bf16 output (2^-9 relative) and P rounded to bf16 before P.V; fp32 sums
TOL = 1e-2


def _check(case, kernels=(0, 1), check=None):
    outs = {k: case.run(k) for k in kernels}
    rows = range(case.B) if check is None else check
    worst = {}
    for b in rows:
        ref = case.oracle(b)
        for k, out in outs.items():
            assert np.isfinite(out[b]).all(), (k, b)
            r = _rel(out[b], ref)
            worst[k] = max(worst.get(k, 0.0), r)
            assert r <= TOL, (k, b, r)
    if len(outs) == 2:
        between = _rel(outs[0], outs[1])
        assert between <= TOL, between
        worst["tc_vs_mma"] = between
    print(worst)
    return outs


@pytest.mark.parametrize("H,kvh,S", [(32, 8, 16), (32, 8, 8), (8, 2, 8), (8, 4, 4), (12, 4, 16),
                                     (12, 4, 8), (6, 2, 4), (16, 8, 1)])
def test_query_row_paddings(H, kvh, S):
    """R = (H/kvh)*S rows per (request, KV head): 64, 32, 32, 8, 48, 24, 12, 2."""
    rng = np.random.default_rng(H * 100 + S)
    B = max(12, 80 // kvh + 1)
    ctx = rng.integers(0, 700, B)
    ctx[0], ctx[1], ctx[2] = 0, 64, 128     # empty, whole pages
    _check(Case(B, S, H, kvh, ctx, seed=H + S), check=[0, 1, 2, 3, B - 1])


def test_long_contexts_many_splits():
    """Few requests with long contexts: up to 16 splits per (request, head),
    merged by the last split to finish."""
    ctx = [9000, 5123, 64 * 70, 7777, 1]
    _check(Case(5, 16, 32, 8, ctx, seed=3))


def test_sliding_window():
    rng = np.random.default_rng(7)
    ctx = rng.integers(50, 900, 24)
    _check(Case(24, 16, 32, 8, ctx, window=100, seed=7), check=[0, 5, 23])


def test_draft_window_ring():
    """Draft window 200: the page table is a ring of 5 pages per request; only
    the newest 200 context rows are visible."""
    ctx = [1000, 199, 200, 4096 + 37, 64 * 9, 5000, 0, 333] * 3
    _check(Case(24, 16, 32, 8, ctx, draft_window=200, seed=11), check=[0, 1, 2, 3, 4, 5, 6, 7])


def test_draft_window_and_sliding_window():
    ctx = [1000, 300, 2000, 64]
    _check(Case(4, 8, 32, 8, ctx, window=150, draft_window=256, seed=13))


def test_peaked_logits():
    """Large logits (q scaled by 12): the running maximum moves across tiles
    and the rescaling of the partial sums matters."""
    rng = np.random.default_rng(17)
    ctx = rng.integers(100, 3000, 12)
    _check(Case(12, 16, 32, 8, ctx, seed=17, q_scale=12.0), check=[0, 6, 11])


@pytest.mark.slow
def test_stress_full_size_sampled():
    """stress-b128-s16's attention shape at full size (128 requests, lognormal
    contexts up to 32768): every request of the tcgen05 kernel against the
    mma.sync kernel, eight sampled requests against the oracle."""
    from synth import WORKLOADS, make_context_lengths
    wl = WORKLOADS["stress-b128-s16"]
    ctx = make_context_lengths(wl, 0)
    case = Case(wl.batch, wl.cfg.block_size, wl.cfg.n_heads, wl.cfg.n_kv_heads, ctx, seed=23)
    order = np.argsort(ctx)
    check = sorted(set([int(order[0]), int(order[-1]), int(order[len(order) // 2])] +
                       list(range(0, 128, 25))))
    _check(case, check=check)
