#!/usr/bin/env python
"""Throughput of the DFlash draft pass on one GB300: drafted tokens/s.

One step = one draft-verify cycle of the whole hot path on one batch:
  dflash_draft_block -> (synthetic target verify) -> dflash_accept_commit
  -> dflash_inject_context(commit rows)
metric = batch * (block_size - 1) / (device time of the three calls), the
synthetic verify (a torch.where over pre-drawn randoms) being excluded.
Before every cycle kv_len / seq_len are restored to the workload's context
length, so every timed cycle drafts against exactly that context.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                  [--verify greedy|sampled]

The default workload is the largest one that fits one GPU, the stress sweep
point stress-b128-s16 (Qwen3-8B-shaped bf16 draft, batch 128, block 16,
lognormal contexts with median 2048 up to 32768, paged KV); the other named
workloads (qwen8b-b1, qwen8b-b32, kimi-b8, stress-b{64,128}-s{8,16}) are
selected with --workload.

--verify sampled replaces the greedy acceptance with dflash_accept_commit_sampled
(lossless rejection sampling): synthetic target rows (softmax of random
logits, the proposed tokens given the workload's match probability, built
outside the timed region) and per-step Exp(1) race noise.

Under torchrun (N > 1) each rank runs an independent replica (requests are
independent; no collective is on the path) and rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import WORKLOADS, make_anchor, make_context_lengths, make_features, \
    make_page_table, make_weights  # noqa: E402

METRIC = "DFlash draft-pass drafted tokens/s on 1 GB300; % of BF16/HBM roofline"
UNIT = "drafted tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="stress-b128-s16")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--draft", default="plain", choices=["plain", "selector"],
                    help="plain: argmax drafter; selector: DFlash 2 candidate selector "
                         "(K=8 candidates, rank 128, greedy walk, random factors)")
    ap.add_argument("--verify", default="greedy", choices=["greedy", "sampled"],
                    help="greedy: dflash_accept_commit; sampled: dflash_accept_commit_sampled "
                         "(lossless rejection sampling against synthetic target rows)")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="draft KV cache: bf16, or one-byte FP8 E4M3 codes with per-layer scales")
    ap.add_argument("--draft-window", type=int, default=0,
                    help="draft KV windowing: keep the newest W committed rows per request "
                         "(a ring of ceil(W/64)+1 pages); 0 = off")
    ap.add_argument("--profile-case", action="store_true",
                    help="counter captures only: two layers and a 32,768-token vocabulary "
                         "(same per-layer kernels and batch shape); not a benchmark value")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-cycles", type=int, default=2)
    ap.add_argument("--reference-budget-s", type=float, default=120.0)
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------- roofline model
def visible_keys(cfg, ctx, draft_window=0):
    """Context keys one attention launch reads, summed over the requests and
    averaged over the layers: min(T_b, the layer's sliding window, the draft
    window) -- the pages the kernel stages (a window's first page may be
    partial; that slack is not counted)."""
    T = np.atleast_1d(np.asarray(ctx, dtype=np.float64))
    per_layer = []
    for w in cfg.sliding_window:
        v = T.copy()
        if w:
            v = np.minimum(v, w)
        if draft_window:
            v = np.minimum(v, draft_window)
        per_layer.append(v.sum())
    return float(np.mean(per_layer))


def algorithmic(cfg, B, ctx, commit_mean, kv_fp8=False, draft_window=0):
    """Per-launch algorithmic bytes and flops of each kernel family; ctx is
    the mean context length or the per-request lengths."""
    S, H, D = cfg.block_size, cfg.hidden, cfg.head_dim
    M = B * S
    es = 2 if cfg.dtype == "bf16" else 4
    kvb = 1 if kv_fp8 else es             # bytes per cached K/V element
    qkv = cfg.qkv_rows
    qd, kvd, I, V = cfg.n_heads * D, cfg.n_kv_heads * D, cfg.intermediate, cfg.vocab
    K_fc = cfg.n_sel * cfg.target_hidden
    rows = B * commit_mean  # the committed rows are projected and written
    if np.ndim(ctx) == 0:
        ctx = np.full(B, float(ctx))
    ctx_keys = visible_keys(cfg, ctx, draft_window)          # summed over the batch
    fam = {
        "gemm_qkv": (es * (qkv * H + M * H + M * qkv), 2 * M * qkv * H),
        "gemm_o": (es * (H * qd + M * qd) + 8 * M * H, 2 * M * H * qd),
        "gemm_gate_up": (es * (2 * I * H + M * H + M * I), 2 * M * 2 * I * H),
        "gemm_down": (es * (H * I + M * I) + 8 * M * H, 2 * M * H * I),
        "gemm_lm_head_argmax": (es * (V * H + M * H) + 8 * M, 2 * M * V * H),
        "attention": (kvb * 2 * ctx_keys * kvd + es * (2 * B * S * kvd + 2 * M * qd),
                      4 * S * qd * (ctx_keys + B * S)),
        "gemm_fc": (es * (H * K_fc + rows * K_fc) + 4 * rows * H, 2 * rows * H * K_fc),
        "gemm_kv_inject": (es * (cfg.n_layers * 2 * kvd * H + rows * H)
                           + kvb * rows * cfg.n_layers * 2 * kvd,
                           2 * rows * cfg.n_layers * 2 * kvd * H),
        # the final RMSNorm phase: x (fp32) read, the normalised rows written
        "final_norm": ((4 + es) * M * H + 4 * M * (H // 128), 0),
        "accept": (4 * (2 * B * S + B * (S + 4)), 0),
        # target row at the stop position and the race noise, read once each
        "accept_sampled": (4 * (2 * B * V + 2 * B * S + B * (S + 4)), 0),
    }
    add = lambda *names: tuple(sum(fam[n][i] for n in names) for i in range(2))  # noqa: E731
    fam["gemm_layer_program"] = add("gemm_o", "gemm_gate_up", "gemm_down", "gemm_qkv")
    fam["gemm_last_program"] = add("gemm_o", "gemm_gate_up", "gemm_down", "final_norm",
                                   "gemm_lm_head_argmax")
    fam["gemm_inject_program"] = add("gemm_fc", "gemm_kv_inject")
    # block embedding (table rows read; x fp32, x*g bf16 and row sums of squares written)
    fam["embed"] = (es * M * H + (4 + es) * M * H + 4 * M * (H // 128), 0)
    fam["gemm_embed_qkv_program"] = add("embed", "gemm_qkv")
    return fam


# the sources a kernel family's launches are built from (its kernels, the
# headers they include, and the host code that sets the launches up)
KERNEL_SOURCES = {
    "gemm": ("gemm_tc.cu", "epilogue.cuh", "inject_rows.cuh", "common.cuh", "kernels.h",
             "dflash_api.cu"),
    "attention": ("attention_tc.cu", "attention_mma.cu", "attention_simt.cu", "common.cuh",
                  "kernels.h", "dflash_api.cu"),
}


def source_hash(kernel=None):
    """Hash of the sources of a kernel family (launch names starting with
    "gemm" or "attention"); of every source file when kernel is None."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_diffusion_speculative_fc_gb300", "csrc")
    fam = next((v for k, v in KERNEL_SOURCES.items() if kernel and kernel.startswith(k)), None)
    for f in sorted(fam if fam else os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the
    source (workload keys carry "+fp8" / "+w<W>" for the cache options)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
    except Exception:
        return None
    e = t.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------- clock sampling
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        time.sleep(0.3)

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- our arm
class Bench:
    def __init__(self, wl, seed=0, verify="greedy", draft="plain", kv="bf16", draft_window=0):
        import torch
        import block_diffusion_speculative_fc_gb300 as pkg
        self.torch, self.pkg = torch, pkg
        self.wl, self.cfg = wl, wl.cfg
        cfg = self.cfg
        B, S = wl.batch, cfg.block_size
        self.B, self.S = B, S
        self.T = make_context_lengths(wl, seed)
        self.W = make_weights(cfg, seed=seed, device="cuda")
        self.kv_fp8 = kv == "fp8"
        self.draft_window = int(draft_window)
        full_ppr = (int(self.T.max()) + 2 * S + 63) // 64 + 1
        # a draft window keeps a ring of ceil(W / 64) + 1 pages per request
        self.ppr = (self.draft_window + 63) // 64 + 1 if self.draft_window else full_ppr
        self.page_table = make_page_table(B, self.ppr, wl.permuted_pages, seed)
        self.sess = pkg.DraftSession(cfg, self.W, max_batch=B,
                                     max_rows=max(B * S, min(int(self.T.sum()), 65536)),
                                     max_position=full_ppr * 64 + S, kv_fp8=self.kv_fp8)
        # FP8 scales: the magnitude k-normed K and hidden_norm(y) W_v^T reach, over 448
        ks = [4.5 / 448.0] * cfg.n_layers if self.kv_fp8 else None
        vs = [4.0 * 0.02 * cfg.hidden ** 0.5 / 448.0] * cfg.n_layers if self.kv_fp8 else None
        self.kv = self.sess.new_kv(B, self.ppr, self.page_table, ks, vs,
                                   draft_window=self.draft_window)
        i32 = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device="cuda")  # noqa
        self.i32 = i32
        offs = np.concatenate([[0], np.cumsum(self.T)[:-1]])
        # prefill in slices so that feature buffers stay moderate
        for b0 in range(0, B, 8):
            bs = list(range(b0, min(B, b0 + 8)))
            rows = int(self.T[bs].sum())
            feats = make_features(cfg, rows, seed, ("prefill", b0), device="cuda")
            ro = np.zeros(B, dtype=np.int64)
            nr = np.zeros(B, dtype=np.int64)
            acc = 0
            for b in bs:
                ro[b] = acc
                nr[b] = self.T[b]
                acc += self.T[b]
            self.sess.inject(self.kv, feats, i32(ro), i32(nr))
            del feats
        torch.cuda.synchronize()
        assert self.sess.error() == 0
        self.base_len = i32(self.T)
        self.anchor = i32(make_anchor(B, cfg, seed))
        self.draft = torch.zeros((B, S), dtype=torch.int32, device="cuda")
        # a step's results in one contiguous block (committed tokens [B, S], then
        # accept length, bonus id and sequence length [B] each), so the end-to-end
        # loop reads them back with a single copy
        self.results = torch.zeros(B * (S + 3), dtype=torch.int32, device="cuda")
        self.tok = self.results[:B * S].view(B, S)
        self.acc = self.results[B * S:B * S + B]
        self.bon = self.results[B * S + B:B * S + 2 * B]
        self.seq = self.results[B * S + 2 * B:]
        self.seq.copy_(i32(self.T))
        self.com = torch.zeros(B, dtype=torch.int32, device="cuda")
        self.row_off = i32(np.arange(B) * S)
        self.pool = [make_features(cfg, B * S, seed, ("verify", i), device="cuda") for i in range(4)]
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 17)
        self.gen = g
        if wl.match[0] == "bernoulli":
            self.p = torch.full((B, 1), wl.match[1], device="cuda")
        elif wl.match[0] == "bernoulli_per_req":
            r = np.random.default_rng(seed).uniform(wl.match[1], wl.match[2], B)
            self.p = torch.as_tensor(r, dtype=torch.float32, device="cuda")[:, None]
        else:
            self.p = None
        self.verify = verify
        self.selector = draft == "selector"
        if self.selector:
            g2 = torch.Generator(device="cuda")
            g2.manual_seed(seed + 29)
            dt = torch.bfloat16 if cfg.dtype != "f32" else torch.float32
            r = 128
            self.sel_w = ((torch.randn((r, cfg.hidden), generator=g2, device="cuda") /
                           cfg.hidden ** 0.5).to(dt),
                          (r ** -0.25 * torch.randn((cfg.vocab, r), generator=g2, device="cuda")).to(dt),
                          (r ** -0.25 * torch.randn((cfg.vocab, r), generator=g2, device="cuda")).to(dt))
            self.sess.set_selector(8, *self.sel_w)
        if verify == "sampled":
            # target rows: softmax of random logits; each cycle the proposed
            # tokens get the workload's match probability (outside the timed region)
            V = cfg.vocab
            logits = torch.randn((B, S, V), generator=g, device="cuda")
            self.probs_base = torch.softmax(logits, dim=-1).contiguous()
            del logits
            self.probs = torch.empty_like(self.probs_base)
            self.noise = [torch.empty((B, V), device="cuda").exponential_(generator=g) for _ in range(4)]
            m = self.p if self.p is not None else torch.full((B, 1), 0.84, device="cuda")
            self.match_val = m.expand(B, S - 1).contiguous().float()

    def posterior_randoms(self, n):
        torch, B, S, V = self.torch, self.B, self.S, self.cfg.vocab
        u = torch.rand((n, B, S - 1), generator=self.gen, device="cuda")
        r = torch.randint(0, V, (n, B, S), generator=self.gen, device="cuda", dtype=torch.int32)
        if self.p is None:  # geometric commit lengths: accept = commit - 1
            c = torch.distributions.Geometric(probs=torch.tensor(1.0 / self.wl.match[1]))
            k = c.sample((n, B)).to("cuda").clamp(max=S - 1)       # failures before success
            return u, r, k
        return u, r, None

    def make_post(self, u, r, k):
        torch = self.torch
        post = r.clone()
        nxt = self.draft[:, 1:]
        if k is None:
            post[:, :-1] = torch.where(u < self.p, nxt, r[:, :-1])
        else:
            idx = torch.arange(self.S - 1, device="cuda")[None, :]
            take = idx < k[:, None]
            miss = (nxt + 1) % self.cfg.vocab
            post[:, :-1] = torch.where(take, nxt, torch.where(idx == k[:, None], miss, r[:, :-1]))
        return post

    def draft_call(self, anchor):
        if self.selector:
            self.sess.draft_selector(self.kv, anchor, self.draft)
        else:
            self.sess.draft(self.kv, anchor, self.draft)

    def cycle(self, c, u, r, k, ev=None):
        torch = self.torch
        self.kv.kv_len.copy_(self.base_len)
        self.seq.copy_(self.base_len)
        anchor = self.anchor if c == 0 else self.bon
        if ev:
            ev[0].record()
        self.draft_call(anchor)
        if ev:
            ev[1].record()
        if self.verify == "sampled":
            self.probs.copy_(self.probs_base)
            self.probs[:, :-1].scatter_(2, self.draft[:, 1:].long().unsqueeze(-1),
                                        self.match_val.unsqueeze(-1))
        else:
            post = self.make_post(u, r, k)
        if ev:
            ev[2].record()
        if self.verify == "sampled":
            self.sess.accept_sampled(self.B, self.draft, self.probs, u, self.noise[c % 4], self.seq,
                                     self.acc, self.com, self.bon, self.tok)
        else:
            self.sess.accept(self.B, self.draft, post, self.seq, self.acc, self.com, self.bon,
                             self.tok)
        self.sess.inject(self.kv, self.pool[c % len(self.pool)], self.row_off, self.com)
        if ev:
            ev[3].record()

    def run(self, warmup, steps, prof_steps):
        """Timed pass (events around the three calls only), then a separate
        profiled pass with per-kernel events recorded by the library."""
        torch = self.torch
        u, r, k = self.posterior_randoms(warmup + steps + prof_steps)
        kk = lambda c: None if k is None else k[c]  # noqa: E731
        for c in range(warmup):
            self.cycle(c, u[c], r[c], kk(c))
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        acc_sum = torch.zeros((), dtype=torch.int64, device="cuda")
        for i in range(steps):
            c = warmup + i
            self.cycle(c, u[c], r[c], kk(c), evs[i])
            acc_sum += self.com.sum()
        torch.cuda.synchronize()
        ms = [e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in evs]
        mean_commit = float(acc_sum.item()) / (steps * self.B)
        # profiled pass: same cycles, one event pair per kernel launch
        per_cycle_launches = 12 * self.cfg.n_layers + 16
        self.pkg.dflash_profile_enable(self.sess.h, prof_steps * per_cycle_launches + 64)
        for i in range(prof_steps):
            c = warmup + steps + i
            self.cycle(c, u[c], r[c], kk(c))
        torch.cuda.synchronize()
        prof = self.pkg.dflash_profile_collect(self.sess.h)
        self.pkg.dflash_profile_disable(self.sess.h)
        assert self.sess.error() == 0
        prof = {n: (v[0] / prof_steps, v[1] / prof_steps) for n, v in prof.items()}  # per cycle
        return sum(ms), ms, prof, mean_commit

    def run_e2e(self, steps):
        """Same cycles through the public API with host buffers: verify features
        and verify randoms copied host->device each step, results device->host.
        The host->device copies of a step run on a second stream while that
        step's draft block computes (only the acceptance and the injection read
        them; the main stream waits on their event before the acceptance), and
        the next step's copies wait for this step's injection to finish reading
        the buffers.  The results come back with one device->host copy."""
        torch, B, S, cfg = self.torch, self.B, self.S, self.cfg
        u, r, k = self.posterior_randoms(steps)
        u_h, r_h = u.cpu().pin_memory(), r.cpu().pin_memory()
        k_h = k.cpu().pin_memory() if k is not None else None
        feats_h = [p.cpu().pin_memory() for p in self.pool]
        feat_d = torch.empty_like(self.pool[0])
        u_d, r_d = torch.empty_like(u[0]), torch.empty_like(r[0])
        k_d = torch.empty_like(k[0]) if k is not None else None
        out_h = torch.empty(B * (S + 3), dtype=torch.int32).pin_memory()
        h2d = feats_h[0].numel() * feats_h[0].element_size() + u_h[0].numel() * 4 + r_h[0].numel() * 4
        if k_h is not None:
            h2d += k_h[0].numel() * k_h.element_size()
        sampled = self.verify == "sampled"
        if sampled:   # the race noise of each step comes from the host as well
            noise_h = [n.cpu().pin_memory() for n in self.noise]
            noise_d = torch.empty_like(self.noise[0])
            h2d += noise_h[0].numel() * 4
        d2h = out_h.numel() * 4
        main = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        copied = torch.cuda.Event()
        consumed = torch.cuda.Event()
        consumed.record(main)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for c in range(steps):
            with torch.cuda.stream(side):
                side.wait_event(consumed)      # the previous step's injection has read them
                feat_d.copy_(feats_h[c % len(feats_h)], non_blocking=True)
                u_d.copy_(u_h[c], non_blocking=True)
                r_d.copy_(r_h[c], non_blocking=True)
                if k_d is not None:
                    k_d.copy_(k_h[c], non_blocking=True)
                if sampled:
                    noise_d.copy_(noise_h[c % len(noise_h)], non_blocking=True)
                copied.record(side)
            self.kv.kv_len.copy_(self.base_len)
            self.seq.copy_(self.base_len)
            anchor = self.anchor if c == 0 else self.bon
            self.draft_call(anchor)
            main.wait_event(copied)
            if sampled:
                self.probs.copy_(self.probs_base)
                self.probs[:, :-1].scatter_(2, self.draft[:, 1:].long().unsqueeze(-1),
                                            self.match_val.unsqueeze(-1))
                self.sess.accept_sampled(B, self.draft, self.probs, u_d, noise_d, self.seq,
                                         self.acc, self.com, self.bon, self.tok)
            else:
                post = self.make_post(u_d, r_d, k_d)
                self.sess.accept(B, self.draft, post, self.seq, self.acc, self.com, self.bon,
                                 self.tok)
            self.sess.inject(self.kv, feat_d, self.row_off, self.com)
            consumed.record(main)
            out_h.copy_(self.results, non_blocking=True)
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1)
        return ms, h2d, d2h


def host_weights(W):
    """float32 numpy copies of a weight dict (every bf16 value is exact in float32)."""
    f = lambda t: t.float().cpu().numpy()  # noqa: E731
    out = {k: f(v) for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: f(v) for k, v in L.items()} for L in W["layers"]]
    return out


def cpu_baseline(cfg, T, W, cycles):
    """The oracle, as it stands, timed on this host's cores for `cycles` cycles
    of the same workload (one request at context T; W: host weights).  Its
    inputs come from synth on the host: nothing here touches the GPU library."""
    from oracle import dflash_oracle as O
    from synth import make_posterior
    T = int(T)
    feats = make_features(cfg, T, 99, "cpu-prefill", device="cpu")
    ctx = O.DraftContext(cfg)
    ctx.inject([feats[j].double().numpy() for j in range(cfg.n_sel)], W)
    vfe = make_features(cfg, cfg.block_size, 99, "cpu-verify", device="cpu")
    vf = [vfe[j].double().numpy() for j in range(cfg.n_sel)]
    anchor = 5
    t0 = time.perf_counter()
    for c in range(cycles):
        ids, hid, margin = O.draft_block(cfg, W, anchor, ctx.layers(), ctx.kv_len)
        post = make_posterior(ids[None], [0.85], cfg.vocab, 0, c)[0]
        acc, bonus, commit, out = O.accept_block(ids, post)
        ctx.inject([v[:commit] for v in vf], W)
        anchor = bonus
    dt = time.perf_counter() - t0
    try:
        import threadpoolctl
        blas = max((p.get("num_threads", 0) for p in threadpoolctl.threadpool_info()), default=None)
    except Exception:
        blas = None
    cores = len(os.sched_getaffinity(0))
    value = cycles * (cfg.block_size - 1) / dt      # one request's drafted tokens per second
    return {"value": value, "unit": UNIT, "cores": blas or cores, "kind": "oracle",
            "sample": f"{cycles} full cycles (draft_block + accept + inject of the commit rows) "
                      f"of request 0 at context {T}, float64 numpy, {cores} host cores"}


def dominant_roofline(bench, prof, mean_commit, wl_name):
    hbm, tf, tf_sus, src = peaks()
    fam = algorithmic(bench.cfg, bench.B, bench.T, mean_commit, getattr(bench, "kv_fp8", False),
                      getattr(bench, "draft_window", 0))
    total = sum(v[1] for v in prof.values())
    name = max(prof, key=lambda n: prof[n][1])
    launches, ms = prof[name]          # per cycle
    avg_s = ms / launches / 1e3
    bytes_, flops = fam.get(name, (0, 0))
    ai = flops / bytes_ if bytes_ else 0
    ridge = tf * 1e12 / (hbm * 1e9)
    if ai > ridge:
        out = {"bound": "tensor", "achieved": flops / avg_s / 1e12, "peak": tf_sus,
               "unit": "TFLOP/s"}
    else:
        out = {"bound": "hbm", "achieved": bytes_ / avg_s / 1e9, "peak": hbm, "unit": "GB/s"}
    out["frac"] = out["achieved"] / out["peak"]
    key = wl_name + ("+fp8" if getattr(bench, "kv_fp8", False) else "") + \
        (f"+w{bench.draft_window}" if getattr(bench, "draft_window", 0) else "")
    out["traffic"] = traffic_for(name, key)
    out["kernel"] = name
    out["share"] = ms / total if total else None
    out["peak_source"] = src
    return out


def job_rate(ms, units, dist=None, device="cpu"):
    """Whole-job rate of independent replicas: the units every rank processed,
    summed, over the slowest rank's time (the job ends when its last replica
    does).  Returns (units per second, max ms, total units); every rank gets
    the same answer."""
    if dist is None:
        return units / (ms / 1e3), ms, units
    import torch
    t_max = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    t_sum = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    dist.all_reduce(t_sum, op=dist.ReduceOp.SUM)
    ms_max, total = float(t_max.item()), float(t_sum.item())
    return total / (ms_max / 1e3), ms_max, total


def main():
    a = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = WORKLOADS[a.workload]
    if a.profile_case:
        # for counter captures only: the same per-layer kernels and batch
        # shape on two layers and a 32,768-token vocabulary, so the capture
        # holds a few GB; the line is marked and is not a benchmark value
        from dataclasses import replace
        from synth.configs import shrink
        cfg = shrink(wl.cfg, name=wl.cfg.name + "-profile-case", n_layers=2,
                     vocab=32768, mask_token_id=32767)
        wl = replace(wl, cfg=cfg)   # same name: the same seeded context lengths
    if a.impl == "reference":
        return reference_arm(a, wl, rank, world)
    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    bench = Bench(wl, verify=a.verify, draft=a.draft, kv=a.kv, draft_window=a.draft_window)
    cs = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    cs.start()
    total_ms, ms, prof, mean_commit = bench.run(a.warmup, a.steps, min(a.steps, 50))
    clocks = cs.stop()
    tokens_here = a.steps * bench.B * (bench.S - 1)
    value, total_ms, _ = job_rate(total_ms, tokens_here, dist, "cuda")
    e2e = None
    if not a.no_e2e:
        e_ms, h2d, d2h = bench.run_e2e(a.steps)
        e_value, _, _ = job_rate(e_ms, tokens_here, dist, "cuda")
        e2e = {"value": e_value, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    roof = dominant_roofline(bench, prof, mean_commit,
                             a.workload + ("+profile-case" if a.profile_case else ""))
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(bench.cfg, bench.T[0], host_weights(bench.W), a.cpu_cycles)
    launches = int(round(sum(v[0] for v in prof.values()) * a.steps))
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": total_ms / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": bench.cfg.dtype, "data": "synthetic",
            "config": {"workload": a.workload, "batch": bench.B, "block_size": bench.S,
                       "context": int(bench.T[0]) if len(set(bench.T.tolist())) == 1 else
                       f"{int(bench.T.min())}..{int(bench.T.max())}",
                       "layers": bench.cfg.n_layers, "hidden": bench.cfg.hidden,
                       "vocab": bench.cfg.vocab, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (weights streamed every step)",
                       "kv_len_reset_each_cycle": True, "verify": a.verify, "draft": a.draft,
                       "kv_cache": a.kv, "draft_window": a.draft_window,
                       "profile_case": bool(a.profile_case),
                       "mean_commit_len": mean_commit},
            "clocks": clocks, "e2e": e2e, "gpu_launches": launches,
            "roofline": roof, "cpu_baseline": cpu,
            "kernels_ms_per_step": {k: v[1] for k, v in sorted(prof.items())},
            "kernel_profile": "separate pass of min(steps, 50) cycles with one CUDA event pair "
                              "per launch; the timed pass records only per-call events",
        }
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def reference_arm(a, wl, rank, world):
    """The oracle as it stands on the host cores: same workload, metric, unit."""
    if rank != 0:
        return
    # host-only inputs: the same workload drawn by synth on the CPU; no
    # session, no device memory and no library call in this process
    T = make_context_lengths(wl, 0)
    W = host_weights(make_weights(wl.cfg, seed=0, device="cpu"))
    steps = max(1, a.steps)
    per = []
    t_start = time.perf_counter()
    cb = cpu_baseline(wl.cfg, T[0], W, 1)       # warm-up / setup sample
    done = 0
    for _ in range(steps):
        r = cpu_baseline(wl.cfg, T[0], W, 1)
        per.append(r["value"])
        done += 1
        if time.perf_counter() - t_start > a.reference_budget_s:
            break
    # The oracle drafts one request per call, so a batch of B requests takes
    # about B times one request's time: the batch rate is one request's rate.
    value = float(np.mean(per))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": done,
            "steps_requested": a.steps, "warmup": a.warmup, "higher_is_better": True,
            "impl": "reference", "dtype": "f64", "data": "synthetic",
            "config": {"workload": a.workload, "batch": wl.batch,
                       "block_size": wl.cfg.block_size},
            "cpu_baseline": {"kind": "oracle", "cores": cb["cores"], "sample": cb["sample"]
                             + f"; request 0 timed: the oracle drafts one request per call, "
                               f"so the batch of {wl.batch} runs at one request's rate",
                             "value": value},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
