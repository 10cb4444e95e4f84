"""Draft-model shapes and workload descriptions.

Shapes follow the draft configurations named by the pages: the Kimi-K2.6
DFlash draft card quoted in the CSDN article (block 8, mask id 163838,
target_layer_ids [1,12,24,35,47,58], five sliding layers of window 2048 then
one full layer, 64 heads x 128, 8 KV heads) and the Qwen3-8B target / b16
draft of the SGLang PR benchmark.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class DraftConfig:
    name: str
    dtype: str                      # "f32" or "bf16": storage and arithmetic type of inputs
    target_hidden: int
    target_layer_ids: tuple
    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    mask_token_id: int
    block_size: int
    sliding_window: tuple           # per draft layer; 0 = full attention
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    page_size: int = 64

    @property
    def n_sel(self):
        return len(self.target_layer_ids)

    @property
    def qkv_rows(self):
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def weight_bytes(self):
        es = 4 if self.dtype == "f32" else 2
        per_layer = (self.qkv_rows * self.hidden + self.hidden * self.n_heads * self.head_dim
                     + 3 * self.hidden * self.intermediate)
        return es * (self.n_layers * per_layer + 2 * self.vocab * self.hidden
                     + self.hidden * self.n_sel * self.target_hidden)


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: DraftConfig
    batch: int
    # context lengths: ("fixed", T) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    context: tuple
    # match model: ("bernoulli", p) | ("bernoulli_per_req", lo, hi) | ("geometric", mean)
    match: tuple
    cycles: int = 8
    permuted_pages: bool = False
    extra: dict = field(default_factory=dict)


TINY = DraftConfig(
    name="tiny-f32", dtype="f32", target_hidden=256, target_layer_ids=(0, 2, 4),
    hidden=256, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64, intermediate=512,
    vocab=1024, mask_token_id=1023, block_size=4, sliding_window=(0, 0))

# Qwen3-8B-shaped draft.  The pages give no mask id or layer ids for it: the
# mask id is the last vocabulary row and the five layer ids are labels only.
QWEN8B = DraftConfig(
    name="qwen3-8b-b16", dtype="bf16", target_hidden=4096, target_layer_ids=(1, 9, 17, 25, 33),
    hidden=4096, n_layers=5, n_heads=32, n_kv_heads=8, head_dim=128, intermediate=12288,
    vocab=151936, mask_token_id=151935, block_size=16, sliding_window=(0,) * 5)

KIMI = DraftConfig(
    name="kimi-k2-b8", dtype="bf16", target_hidden=7168,
    target_layer_ids=(1, 12, 24, 35, 47, 58), hidden=7168, n_layers=6, n_heads=64,
    n_kv_heads=8, head_dim=128, intermediate=18432, vocab=163840, mask_token_id=163838,
    block_size=8, sliding_window=(2048, 2048, 2048, 2048, 2048, 0))


def _qwen_bs(s):
    return DraftConfig(**{**QWEN8B.__dict__, "name": f"qwen3-8b-b{s}", "block_size": s})


WORKLOADS = {
    "tiny": Workload("tiny", TINY, batch=1, context=("fixed", 32), match=("bernoulli", 0.8)),
    "qwen8b-b1": Workload("qwen8b-b1", QWEN8B, batch=1, context=("fixed", 1024),
                          match=("bernoulli", 0.85)),
    "qwen8b-b32": Workload("qwen8b-b32", QWEN8B, batch=32, context=("uniform", 256, 4096),
                           match=("bernoulli_per_req", 0.6, 0.95), permuted_pages=True),
    "kimi-b8": Workload("kimi-b8", KIMI, batch=8, context=("fixed", 8192),
                        match=("bernoulli", 0.85)),
}
for _b in (64, 128):
    for _s in (8, 16):
        WORKLOADS[f"stress-b{_b}-s{_s}"] = Workload(
            f"stress-b{_b}-s{_s}", _qwen_bs(_s), batch=_b,
            context=("lognormal", 2048, 1.0, _s, 32768), match=("geometric", 6.4),
            permuted_pages=True)


def get_workload(name):
    return WORKLOADS[name]


def shrink(cfg: DraftConfig, **over) -> DraftConfig:
    """A smaller variant of a config (same structure, fewer features).  With
    fewer layers and no explicit windows, the per-layer windows are cut to
    the new layer count."""
    d = {**cfg.__dict__, **over}
    if "sliding_window" not in over and len(d["sliding_window"]) != d["n_layers"]:
        w = tuple(d["sliding_window"])
        d["sliding_window"] = (w + (0,) * d["n_layers"])[:d["n_layers"]]
    return DraftConfig(**d)
