"""DFlash 2 candidate selector on the GPU against the oracle.

The backbone is the draft pass the other parity tests already check; here the
selector is compared with the oracle fed the GPU's own final-normed hidden
states (``hidden_out`` of a plain draft call on the same inputs -- exactly the
rows the GPU's lm_head reads), so the only differences left are the GPU's
fp32 dot products.  Every score, softmax and choice on the oracle side comes
from the oracle's own functions (compute_candidates, selector_walk); a GPU
choice may differ from the oracle's only where the two competing scores are
within the a-priori rounding bound of fp32 dot products,
gamma_n * sum |x_i y_i| with gamma_n = n u / (1 - n u), u = 2^-24, summed over
the terms of each score; the walk then continues from the GPU's choice.
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


def _gamma(n):
    u = 2.0 ** -24
    return n * u / (1 - n * u)


def _check_against_oracle(run, anchor, hid, W_h, A, Bm, K, got, noise):
    """Returns the number of choices (candidates or walk steps) that differ
    from the oracle's within their rounding bound."""
    cfg, S = run.cfg, run.cfg.block_size
    H = cfg.hidden
    draft_s, cand, q = got
    lm = run.Wn["lm_head"].astype(np.float64)
    Whn, An, Bn = (t.float().cpu().numpy().astype(np.float64) for t in (W_h, A, Bm))
    r = Whn.shape[0]
    e_all = noise.cpu().numpy().astype(np.float64) if noise is not None else None
    h_all = hid.double().cpu().numpy()
    gH, gr = _gamma(H), _gamma(r)
    near = 0
    for b in range(run.B):
        h = h_all[b, 1:]
        assert draft_s[b, 0] == anchor[b]
        # oracle candidates, with a few more ranks to look the GPU's ids up in
        extra = min(K + 8, cfg.vocab)
        ids_o, logit_o = O.compute_candidates(h, lm, extra)
        wh = O.linear(h, Whn)                       # W_h h of the same rows
        # bound of |fp32 - exact| of each logit and of each W_h h entry
        err_wh = gH * (np.abs(h) @ np.abs(Whn).T)   # [S-1, r]
        unary = np.zeros((S - 1, K))
        err_u = np.zeros((S - 1, K))
        for j in range(S - 1):
            c = cand[b, j]
            assert len(set(c.tolist())) == K and c.min() >= 0 and c.max() < cfg.vocab
            eu = gH * (np.abs(h[j]) @ np.abs(lm[c]).T)
            for k in range(K):
                hit = np.nonzero(ids_o[j] == c[k])[0]
                assert len(hit) == 1, ("GPU candidate outside the oracle's top ranks", b, j, k)
                unary[j, k] = logit_o[j, hit[0]]
                err_u[j, k] = eu[k]
                if c[k] != ids_o[j, k]:
                    # rank k holds another id only when its logit ties the
                    # oracle's k-th best within both rounding bounds
                    e_ref = gH * float(np.abs(h[j]) @ np.abs(lm[ids_o[j, k]]))
                    assert abs(unary[j, k] - logit_o[j, k]) <= err_u[j, k] + e_ref, (b, j, k)
                    near += 1
        # the oracle's walk over the GPU's candidates, restarted from the
        # GPU's choice after a choice within rounding
        y_gpu = draft_s[b, 1:].astype(np.int64)
        j0, pred = 0, int(anchor[b])
        while j0 < S - 1:
            ids_w, slots_w, q_w = O.selector_walk(
                pred, cand[b, j0:], unary[j0:], wh[j0:], An, Bn,
                None if e_all is None else e_all[b, j0:])
            for t in range(S - 1 - j0):
                j = j0 + t
                c = cand[b, j]
                # rounding bound of each score: its logit, the W_h h entries
                # it uses, and the fp32 sum over the rank
                ab = np.abs(An[pred])[None, :] * np.abs(Bn[c])        # [K, r]
                d = err_u[j] + ab @ err_wh[j] + gr * (ab @ np.abs(wh[j]))
                assert np.all(np.abs(q[b, j] - q_w[t]) <= q_w[t] * np.expm1(4 * d.max()) + 1e-5), \
                    (b, j, q[b, j], q_w[t])
                slot = np.nonzero(c == y_gpu[j])[0]
                assert len(slot) == 1, (b, j, y_gpu[j], c)
                k = int(slot[0])
                if k != slots_w[t]:
                    kw = int(slots_w[t])
                    if e_all is None:
                        sc = np.log(q_w[t])            # scores up to a common shift
                        assert sc[kw] - sc[k] <= d[kw] + d[k] + 1e-6, (b, j, k, kw)
                    else:
                        key = np.log(q_w[t]) - np.log(e_all[b, j])
                        assert key[kw] - key[k] <= 2 * (d[kw] + d[k]) + 1e-5, (b, j, k, kw)
                    near += 1
                    j0, pred = j + 1, int(y_gpu[j])
                    break
                pred = int(ids_w[t])
            else:
                j0 = S - 1
    return near


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
    near = _check_against_oracle(run, anchor, hid, W_h, A, Bm, K, got, noise)
    print("choices within rounding of the oracle's:", near)


def test_selector_full_qwen_vocabulary():
    """151,936 tokens: 1,187 vocabulary tiles, the skip of tiles that cannot
    reach a row's top K, ragged last tile."""
    cfg = QWEN_VOCAB
    run, anchor = _setup(cfg, 2, [80, 150], seed=3)
    W_h, A, Bm = _sel_weights(cfg, 128, seed=4)
    run.sess.set_selector(8, W_h, A, Bm)
    _, hid = _plain(run, anchor)
    got = _selector(run, anchor, 8, None)
    near = _check_against_oracle(run, anchor, hid, W_h, A, Bm, 8, got, None)
    print("choices within rounding of the oracle's:", near)


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
