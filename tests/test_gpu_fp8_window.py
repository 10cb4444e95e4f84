"""FP8 draft KV cache and draft KV windowing on the GPU against the oracle.

FP8 (CSDN article, Kimi-K2.6 draft card: "KV cache per token (FP8)" of one
byte per element):
  * the encoder the injection epilogue uses is bit-exact against the
    oracle's E4M3 encoder on the same float32 quotients x / scale (values
    across the whole range, exact midpoints, saturation, signed zeros,
    subnormals);
  * in full draft-verify cycles every stored code is the code of a value
    within the bf16 path's error of the oracle's x / scale, and the decoded
    cache is within rel-L2 2e-2 of the oracle's own FP8 cache (DraftContext.
    layers_fp8);
  * a code is an integer decided by floating point, so the hidden states are
    compared (rel-L2 2e-2) with the oracle's draft over the GPU's own codes;
    against the oracle's own codes the difference is reported: about 6% of
    the codes sit one step apart where the two sides' values straddle a
    rounding boundary, which moves the hidden states by about 2e-2;
    drafted ids follow the parity tests' rule.
Draft KV windowing ("Inside SGLang", worker/memory section: the draft's
private compact mapping; CSDN article, --speculative-dflash-draft-window-size):
the cache is a ring of ceil(W/64)+1 pages per request; contexts run to
several times W; the kept rows are compared with the oracle's rows at the
same positions and the draft with draft_block_windowed.
"""
import ctypes

import numpy as np
import pytest

from synth import WORKLOADS, make_context_lengths
from synth.configs import shrink

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import block_diffusion_speculative_fc_gb300 as pkg  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402
from tests.harness import CycleRun  # noqa: E402

TINY = WORKLOADS["tiny"].cfg
QWEN = WORKLOADS["qwen8b-b1"].cfg
KIMI = WORKLOADS["kimi-b8"].cfg
QWEN_MINI = shrink(QWEN, name="qwen-mini", target_hidden=256, hidden=512, n_layers=2, n_heads=8,
                   n_kv_heads=2, intermediate=1024, vocab=4096, mask_token_id=4095)
KIMI_MINI = shrink(KIMI, name="kimi-mini", target_hidden=256, target_layer_ids=(1, 12, 24),
                   hidden=512, n_layers=3, n_heads=8, n_kv_heads=1, intermediate=768,
                   vocab=3000, mask_token_id=2998, sliding_window=(64, 64, 0))


def _report(run, st):
    flips = st["e2e_flips"]
    print(f"hidden_rel {max(st['hidden_rel']):.3e} kv_rel {max(st['kv_rel']):.3e} "
          f"ids {st['ids']} near-tie {st['id_near_tie']} e2e flips {len(flips)}"
          + (f" fp8 codes off the oracle's {max(run.stats_fp8):.3%}" if run.stats_fp8 else "")
          + (f" hidden_rel vs the oracle's own codes {max(st['hidden_rel_own_fp8']):.3e}"
             if st.get("hidden_rel_own_fp8") else ""))


# ---------------------------------------------------------------- FP8 encoder
def _encode_gpu(x, scale):
    lib = pkg.load_library()
    lib.dflash_test_e4m3_encode.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                            ctypes.c_void_p, ctypes.c_void_p]
    lib.dflash_test_e4m3_encode.restype = ctypes.c_int
    xd = torch.as_tensor(np.asarray(x, dtype=np.float32), device="cuda")
    codes = torch.zeros(xd.numel(), dtype=torch.uint8, device="cuda")
    st = lib.dflash_test_e4m3_encode(xd.data_ptr(), xd.numel(), scale, codes.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return codes.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("scale", [1.0, 0.37, 3.0e-3, 250.0])
def test_e4m3_encoder_is_bit_exact(scale):
    rng = np.random.default_rng(int(scale * 1000) % 97)
    pos = O.e4m3_decode(np.arange(0x7F))                    # every finite positive code value
    mids = (pos[:-1] + pos[1:]) / 2                          # exact ties
    vals = np.concatenate([
        rng.normal(size=20000) * 3.0,
        rng.uniform(-448.0, 448.0, 5000),
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), 5000)) * rng.choice([-1, 1], 5000),
        pos, -pos, mids, -mids, [0.0, -0.0, 448.0, 464.0, 1e6, -1e6, 2.0 ** -10, 2.0 ** -9],
    ])
    # values that are already the quotients the hardware rounds: x = q * scale
    # with q chosen above, so x / scale in float32 lands on them (or next to them)
    x = (vals.astype(np.float32) * np.float32(scale)).astype(np.float32)
    q = (x / np.float32(scale)).astype(np.float32)           # the kernel's float32 division
    want = O.e4m3_encode(q.astype(np.float64))
    got = _encode_gpu(x, scale)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(q[i]), int(got[i]), int(want[i])) for i in bad[:8]]


# ----------------------------------------------------------------- FP8 cycles
def test_fp8_cache_qwen_mini_cycles():
    run = CycleRun(QWEN_MINI, 3, [100, 300, 37], cycles=3, gains="random", permuted=True, fp8=True)
    _report(run, run.run())


def test_fp8_cache_kimi_mini_sliding_layers():
    run = CycleRun(KIMI_MINI, 3, [150, 40, 700], cycles=3, permuted=True, fp8=True)
    _report(run, run.run())


def test_fp8_cache_split_attention_many_requests():
    """48 (request, KV head) pairs and more: the persistent split kernel."""
    lens = np.random.default_rng(8).integers(20, 900, 48)
    run = CycleRun(QWEN_MINI, 48, lens, cycles=2, permuted=True, check=[0, 21, 47], fp8=True)
    _report(run, run.run())


def test_fp8_cache_block8_geometric_commits():
    cfg = shrink(QWEN_MINI, name="stress-mini-fp8", block_size=8)
    run = CycleRun(cfg, 16, np.random.default_rng(4).integers(8, 400, 16), cycles=3,
                   permuted=True, match=("geometric", 6.4), check=[0, 9, 15], fp8=True)
    _report(run, run.run())


@pytest.mark.slow
def test_fp8_cache_stress_b128_s8_full():
    wl = WORKLOADS["stress-b128-s8"]
    T = make_context_lengths(wl, 0)
    check = sorted({0, wl.batch - 1, int(np.argmax(T)), wl.batch // 2})
    run = CycleRun(wl.cfg, wl.batch, T, cycles=1, permuted=True, check=check, match=wl.match,
                   max_rows=65536, pool=64, fp8=True)
    _report(run, run.run())


def test_fp8_cache_refuses_fp32():
    with pytest.raises(pkg.DFlashError):
        pkg.DraftSession(TINY, _weights(TINY), max_batch=1, max_rows=64, max_position=256,
                         kv_fp8=True)


def _weights(cfg):
    from synth import make_weights
    return make_weights(cfg, seed=0, device="cuda")


# ---------------------------------------------------------- draft KV window
def test_window_qwen_mini_contexts_several_times_the_window():
    run = CycleRun(QWEN_MINI, 3, [1000, 450, 90], cycles=3, gains="random", permuted=True,
                   draft_window=200)
    _report(run, run.run())


def test_window_kimi_mini_with_layer_windows():
    """Layer windows of 64 inside a draft window of 150, and a full layer."""
    run = CycleRun(KIMI_MINI, 2, [800, 130], cycles=3, permuted=True, draft_window=150)
    _report(run, run.run())


def test_window_with_fp8_cache():
    run = CycleRun(QWEN_MINI, 2, [900, 260], cycles=3, permuted=True, draft_window=256, fp8=True)
    _report(run, run.run())


def test_window_split_attention_many_requests():
    lens = np.random.default_rng(9).integers(100, 1500, 44)
    run = CycleRun(QWEN_MINI, 44, lens, cycles=2, permuted=True, check=[0, 30, 43],
                   draft_window=300)
    _report(run, run.run())


def test_window_chunked_prefill():
    """Prefill rows in chunks smaller than the prefill: rows that fall out of
    the window before the call ends are skipped in every chunk."""
    run = CycleRun(QWEN_MINI, 2, [700, 333], cycles=2, permuted=True, max_rows=128,
                   draft_window=180)
    _report(run, run.run())


def test_window_fp32_cuda_core_path():
    run = CycleRun(TINY, 2, [70, 33], cycles=4, permuted=True, draft_window=20)
    _report(run, run.run())


def test_window_ring_too_small_is_refused():
    run = CycleRun(QWEN_MINI, 1, [50], cycles=1, draft_window=200)
    kv = run.sess.new_kv(1, 3, np.arange(3, dtype=np.int32)[None], draft_window=200)
    feats = torch.zeros((QWEN_MINI.n_sel, 4, QWEN_MINI.target_hidden), dtype=torch.bfloat16,
                        device="cuda")
    i32 = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device="cuda")  # noqa: E731
    with pytest.raises(pkg.DFlashError):
        run.sess.inject(kv, feats, i32([0]), i32([4]))
