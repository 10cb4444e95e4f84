"""DFlash 2 candidate selector on the GPU against the oracle.

The backbone is the draft pass the other parity tests already check; here the
selector is compared with the oracle fed the GPU's own final-normed hidden
states (``hidden_out`` of a plain draft call on the same inputs), so the
check is tight:
  * candidates: the k-th GPU candidate's logit equals the oracle's k-th best
    logit within the rounding of the hidden state (ids identical except
    where logits tie within that bound);
  * the walk, in lock-step with the GPU's choices: q_rows within tolerance of
    the oracle's softmax of the chosen predecessor's scores, and every choice
    the oracle's (greedy: the best score; sampled: the race winner) unless
    two candidates are within the rounding bound of each other -- and such
    choices are rare (at most one position in eight).
Exact checks: K = 1, and A = 0 with the greedy walk, reproduce the argmax
draft bit for bit.
"""
import numpy as np
import pytest

from synth import WORKLOADS, make_anchor
from synth.configs import shrink

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import block_diffusion_speculative_fc_gb300 as pkg  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402
from tests.harness import CycleRun, i32  # noqa: E402

TINY = WORKLOADS["tiny"].cfg
QWEN = WORKLOADS["qwen8b-b1"].cfg
QWEN_MINI = shrink(QWEN, name="qwen-mini", target_hidden=256, hidden=512, n_layers=2, n_heads=8,
                   n_kv_heads=2, intermediate=1024, vocab=4096, mask_token_id=4095)
QWEN_VOCAB = shrink(QWEN, name="qwen-vocab", target_hidden=256, hidden=512, n_layers=1, n_heads=8,
                    n_kv_heads=2, intermediate=1024)


def _sel_weights(cfg, r, seed, zero_A=False):
    g = torch.Generator(device="cuda").manual_seed(seed)
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    H, V = cfg.hidden, cfg.vocab
    W_h = (torch.randn((r, H), generator=g, device="cuda") / np.sqrt(H)).to(dt)
    s = r ** -0.25
    A = (s * torch.randn((V, r), generator=g, device="cuda")).to(dt)
    if zero_A:
        A.zero_()
    B = (s * torch.randn((V, r), generator=g, device="cuda")).to(dt)
    return W_h, A, B


def _setup(cfg, batch, ctx_lens, seed):
    run = CycleRun(cfg, batch, ctx_lens, cycles=1, seed=seed, gains="random", permuted=True)
    run.prefill()
    anchor = make_anchor(batch, cfg, seed)
    return run, anchor


def _plain(run, anchor):
    cfg, B, S = run.cfg, run.B, run.cfg.block_size
    draft = torch.zeros((B, S), dtype=torch.int32, device="cuda")
    hid = torch.zeros((B, S, cfg.hidden), dtype=run.sess.dtype, device="cuda")
    run.sess.draft(run.kv, i32(anchor), draft, hid)
    return draft, hid


def _selector(run, anchor, K, noise):
    B, S = run.B, run.cfg.block_size
    draft = torch.zeros((B, S), dtype=torch.int32, device="cuda")
    cand = torch.full((B, S - 1, K), -7, dtype=torch.int32, device="cuda")
    q = torch.full((B, S - 1, K), -1.0, dtype=torch.float32, device="cuda")
    run.sess.draft_selector(run.kv, i32(anchor), draft, noise, cand, q)
    torch.cuda.synchronize()
    assert run.sess.error() == 0
    return draft.cpu().numpy(), cand.cpu().numpy(), q.cpu().numpy()


def _check_against_oracle(run, anchor, hid, W_h, A, Bm, K, got, noise):
    cfg, S = run.cfg, run.cfg.block_size
    bf16 = cfg.dtype != "f32"
    draft_s, cand, q = got
    lm = run.Wn["lm_head"].astype(np.float64)
    Whn, An, Bn = (t.float().cpu().numpy().astype(np.float64) for t in (W_h, A, Bm))
    e_all = noise.cpu().numpy() if noise is not None else None
    h_all = hid.double().cpu().numpy()
    wnorm = float(np.linalg.norm(lm, axis=1).max())
    ties = 0
    for b in range(run.B):
        h = h_all[b, 1:]
        assert draft_s[b, 0] == anchor[b]
        logits = h @ lm.T
        _, ref_u = O.compute_candidates(h, lm, K)
        wh = h @ Whn.T
        # rounding of the hidden state the lm_head reads (x*g in bf16, then the
        # row scale) against hidden_out (bf16 of the normalised row)
        rel = 2.0 ** -7 if bf16 else 1e-5
        for j in range(S - 1):
            tol = rel * float(np.linalg.norm(h[j])) * wnorm / np.sqrt(cfg.hidden) * 4 + 1e-6
            c = cand[b, j]
            assert len(set(c.tolist())) == K and c.min() >= 0 and c.max() < cfg.vocab
            # ids may differ only where logits tie within tol (mostly the K-th
            # against the (K+1)-th best): the values rank by rank agree
            assert np.all(np.abs(logits[j, c] - ref_u[j]) <= tol), (b, j, logits[j, c], ref_u[j], tol)
        # the walk in lock-step with the GPU's choices
        pred = int(anchor[b])
        for j in range(S - 1):
            c = cand[b, j]
            sc = logits[j, c] + (An[pred] * wh[j]) @ Bn[c].T
            qr = O.softmax(sc)
            comp = np.abs(An[pred] * wh[j] * Bn[c]).sum(axis=1)
            stol = (2.0 ** -7 if bf16 else 1e-5) * (np.abs(logits[j, c]) + comp).max() * 4 + 1e-6
            assert np.allclose(q[b, j], qr, atol=4 * stol + 1e-6), (b, j, q[b, j], qr)
            y = int(draft_s[b, 1 + j])
            slot = np.nonzero(c == y)[0]
            assert len(slot) == 1, (b, j, y, c)
            k = int(slot[0])
            if e_all is None:
                best = int(np.argmax(sc))
                if k != best:
                    assert sc[best] - sc[k] <= 2 * stol, (b, j, sc, k)
                    ties += 1
            else:
                keys = qr / e_all[b, j]
                best = int(np.argmax(keys))
                if k != best:
                    assert keys[best] - keys[k] <= 4 * stol / e_all[b, j].min(), (b, j, keys, k)
                    ties += 1
            pred = y
    return ties


@pytest.mark.parametrize("cfg,batch,ctx,K,r,sampled", [
    (QWEN_MINI, 1, [100], 8, 128, False),
    (QWEN_MINI, 3, [100, 37, 260], 5, 64, True),
    (QWEN_MINI, 2, [64, 129], 8, 200, False),
    (TINY, 3, [32, 5, 70], 4, 16, True),
    (TINY, 1, [32], 8, 8, False),
])
def test_selector_matches_oracle(cfg, batch, ctx, K, r, sampled):
    run, anchor = _setup(cfg, batch, ctx, seed=31 + K)
    W_h, A, Bm = _sel_weights(cfg, r, seed=7 + r)
    run.sess.set_selector(K, W_h, A, Bm)
    _, hid = _plain(run, anchor)
    noise = None
    if sampled:
        g = torch.Generator(device="cuda").manual_seed(5)
        noise = torch.empty((batch, cfg.block_size - 1, K), device="cuda").exponential_(generator=g)
    got = _selector(run, anchor, K, noise)
    ties = _check_against_oracle(run, anchor, hid, W_h, A, Bm, K, got, noise)
    assert ties <= max(2, batch * (cfg.block_size - 1) // 8), ties   # walk choices within rounding


def test_selector_full_qwen_vocabulary():
    """151,936 tokens: 1,187 vocabulary tiles, the skip of tiles that cannot
    reach a row's top K, ragged last tile."""
    cfg = QWEN_VOCAB
    run, anchor = _setup(cfg, 2, [80, 150], seed=3)
    W_h, A, Bm = _sel_weights(cfg, 128, seed=4)
    run.sess.set_selector(8, W_h, A, Bm)
    _, hid = _plain(run, anchor)
    got = _selector(run, anchor, 8, None)
    ties = _check_against_oracle(run, anchor, hid, W_h, A, Bm, 8, got, None)
    assert ties <= 3, ties


@pytest.mark.parametrize("cfg", [QWEN_MINI, TINY])
def test_selector_k1_and_zero_compatibility_are_the_argmax_draft(cfg):
    run, anchor = _setup(cfg, 3, [40, 90, 17], seed=11)
    plain, _ = _plain(run, anchor)
    plain = plain.cpu().numpy()
    W_h, A, Bm = _sel_weights(cfg, 32, seed=12)
    run.sess.set_selector(1, W_h, A, Bm)
    d, c, q = _selector(run, anchor, 1, None)
    assert np.array_equal(d, plain) and np.array_equal(c[:, :, 0], plain[:, 1:])
    assert np.all(q == 1.0)
    W_h, A0, Bm = _sel_weights(cfg, 32, seed=13, zero_A=True)
    run.sess.set_selector(6, W_h, A0, Bm)
    d, c, _ = _selector(run, anchor, 6, None)
    assert np.array_equal(d, plain) and np.array_equal(c[:, :, 0], plain[:, 1:])


def test_selector_repeated_calls_reset_the_bounds():
    """Two calls in a row with different anchors: the second must not inherit
    the first call's per-row bounds (cleared by the embedding)."""
    cfg = QWEN_MINI
    run, anchor = _setup(cfg, 2, [70, 33], seed=17)
    W_h, A, Bm = _sel_weights(cfg, 64, seed=18)
    run.sess.set_selector(8, W_h, A, Bm)
    _selector(run, anchor, 8, None)
    anchor2 = (anchor + 1234) % (cfg.vocab - 1)
    _, hid2 = _plain(run, anchor2)
    got = _selector(run, anchor2, 8, None)
    _check_against_oracle(run, anchor2, hid2, W_h, A, Bm, 8, got, None)


def test_selector_host_checks():
    cfg = QWEN_MINI
    run, anchor = _setup(cfg, 1, [20], seed=19)
    B, S = 1, cfg.block_size
    draft = torch.zeros((B, S), dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        run.sess.draft_selector(run.kv, i32(anchor), draft)      # no selector set
    W_h, A, Bm = _sel_weights(cfg, 32, seed=20)
    with pytest.raises(RuntimeError):
        run.sess.set_selector(9, W_h, A, Bm)                     # K above 8
    big = torch.zeros((300, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        run.sess.set_selector(4, big, A, Bm)                     # rank above 256
    run.sess.set_selector(4, W_h, A, Bm)
    run.sess.set_selector(0, None, None, None)                   # removed again
    with pytest.raises(RuntimeError):
        run.sess.draft_selector(run.kv, i32(anchor), draft)
