"""Seeded random draws for weights, target features, lengths and posteriors.

Every tensor gets its own generator seeded from (seed, tag...) through a
stable hash, so any tensor can be regenerated on its own.  Floating-point
tensors are drawn with torch on the requested device (CPU draws and CUDA
draws differ, but one run always feeds the same tensors to both sides).
Integer workload structure (lengths, page tables, commit lengths) is drawn on
the host with numpy and is identical on every machine.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch


def tensor_seed(seed, *tags) -> int:
    h = hashlib.sha256(repr((int(seed),) + tuple(str(t) for t in tags)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed, *tags):
    g = torch.Generator(device=device)
    g.manual_seed(tensor_seed(seed, *tags))
    return g


def _rng(seed, *tags):
    return np.random.default_rng(tensor_seed(seed, *tags))


def torch_dtype(cfg):
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def _normal(shape, std, cfg, device, seed, *tags):
    g = _gen(device, seed, *tags)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(torch_dtype(cfg))


def _gain(n, cfg, device, seed, gains, *tags):
    if gains == "unit":
        return torch.ones(n, dtype=torch_dtype(cfg), device=device)
    g = _gen(device, seed, *tags)
    t = torch.empty(n, dtype=torch.float32, device=device).uniform_(0.5, 1.5, generator=g)
    return t.to(torch_dtype(cfg))


def make_weights(cfg, seed=0, device="cpu", gains="unit", std=0.02):
    """Draft weights in [out, in] layout; embed/lm_head stand in for the target's.

    gains="unit" gives RMSNorm gains of 1 (the workloads' setting);
    gains="random" draws them from U[0.5, 1.5] so that a dropped gain shows.
    """
    H, D = cfg.hidden, cfg.head_dim
    W = {
        "fc": _normal((H, cfg.n_sel * cfg.target_hidden), std, cfg, device, seed, "fc"),
        "hidden_norm": _gain(H, cfg, device, seed, gains, "hidden_norm"),
        "final_norm": _gain(H, cfg, device, seed, gains, "final_norm"),
        "embed": _normal((cfg.vocab, H), std, cfg, device, seed, "embed"),
        "lm_head": _normal((cfg.vocab, H), std, cfg, device, seed, "lm_head"),
        "layers": [],
    }
    for l in range(cfg.n_layers):
        W["layers"].append({
            "qkv": _normal((cfg.qkv_rows, H), std, cfg, device, seed, "qkv", l),
            "o": _normal((H, cfg.n_heads * D), std, cfg, device, seed, "o", l),
            "gate_up": _normal((2 * cfg.intermediate, H), std, cfg, device, seed, "gate_up", l),
            "down": _normal((H, cfg.intermediate), std, cfg, device, seed, "down", l),
            "in_norm": _gain(H, cfg, device, seed, gains, "in_norm", l),
            "post_norm": _gain(H, cfg, device, seed, gains, "post_norm", l),
            "q_norm": _gain(D, cfg, device, seed, gains, "q_norm", l),
            "k_norm": _gain(D, cfg, device, seed, gains, "k_norm", l),
        })
    return W


def make_features(cfg, rows, seed, tag, device="cpu"):
    """Target features of the selected layers: [n_sel, rows, H_t], N(0, 1)."""
    return _normal((cfg.n_sel, rows, cfg.target_hidden), 1.0, cfg, device, seed, "feat", tag)


def make_pooled_features(cfg, rows, pool, seed, tag, device="cpu"):
    """Target features whose rows are drawn (seeded, uniformly) from `pool`
    distinct N(0, 1) rows: [n_sel, rows, H_t] and the row -> pool index map.
    Long contexts keep their full size on the device while a row-wise checker
    only has to project each distinct row once."""
    base = _normal((cfg.n_sel, pool, cfg.target_hidden), 1.0, cfg, device, seed, "pool", tag)
    idx = _rng(seed, "pool_idx", tag).integers(0, pool, size=rows)
    return base[:, torch.as_tensor(idx, device=device)], base, idx


def make_context_lengths(wl, seed=0):
    kind = wl.context[0]
    B = wl.batch
    if kind == "fixed":
        return np.full(B, wl.context[1], dtype=np.int64)
    r = _rng(seed, "ctx", wl.name)
    if kind == "uniform":
        lo, hi = wl.context[1], wl.context[2]
        return r.integers(lo, hi + 1, size=B).astype(np.int64)
    if kind == "lognormal":
        med, sigma, lo, hi = wl.context[1:]
        t = np.exp(np.log(med) + sigma * r.standard_normal(B))
        return np.clip(np.round(t), lo, hi).astype(np.int64)
    raise ValueError(kind)


def make_match_probs(wl, seed=0):
    kind = wl.match[0]
    if kind == "bernoulli":
        return np.full(wl.batch, wl.match[1])
    if kind == "bernoulli_per_req":
        return _rng(seed, "match", wl.name).uniform(wl.match[1], wl.match[2], size=wl.batch)
    return None


def make_page_table(B, pages_per_req, permuted, seed=0):
    """int32 [B, pages_per_req] over a pool of B * pages_per_req pages."""
    n = B * pages_per_req
    ids = np.arange(n, dtype=np.int32)
    if permuted:
        ids = _rng(seed, "pages").permutation(n).astype(np.int32)
    return ids.reshape(B, pages_per_req)


def make_anchor(B, cfg, seed, tag=0):
    return _rng(seed, "anchor", tag).integers(0, cfg.vocab, size=B).astype(np.int64)


def make_posterior(draft, match_p, vocab, seed, tag):
    """Synthetic target choices for a drafted block (stand-in for the target
    verify pass).  draft [B, S] int64 host array; position i < S-1 repeats
    draft[i+1] with probability match_p[b], every other entry is uniform."""
    draft = np.asarray(draft, dtype=np.int64)
    B, S = draft.shape
    r = _rng(seed, "posterior", tag)
    post = r.integers(0, vocab, size=(B, S)).astype(np.int64)
    hit = r.random((B, S - 1)) < np.asarray(match_p, dtype=np.float64)[:, None]
    post[:, :-1] = np.where(hit, draft[:, 1:], post[:, :-1])
    return post


def make_commit_lengths(B, S, mean, seed, tag):
    """Commit lengths ~ Geometric(1/mean) on {1, 2, ...}, clipped to S."""
    r = _rng(seed, "commit", tag)
    return np.minimum(r.geometric(1.0 / mean, size=B), S).astype(np.int64)


def make_posterior_with_commit(draft, commit, vocab, seed, tag):
    """Posterior whose greedy acceptance gives exactly accept = commit - 1."""
    draft = np.asarray(draft, dtype=np.int64)
    B, S = draft.shape
    r = _rng(seed, "posterior_commit", tag)
    post = r.integers(0, vocab, size=(B, S)).astype(np.int64)
    for b in range(B):
        a = int(commit[b]) - 1
        post[b, :a] = draft[b, 1:a + 1]
        if a < S - 1:
            post[b, a] = (draft[b, a + 1] + 1 + r.integers(0, vocab - 1)) % vocab
    return post
