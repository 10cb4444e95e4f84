"""Owner of one libdflash handle and its torch-allocated device buffers.

PyTorch only provides device memory and the current CUDA stream here; every
computation is a call into libdflash.
"""
from __future__ import annotations

import ctypes

import torch

from . import (DFLASH_BF16, DFLASH_F32, DflashConfig, DflashKV, DflashWeights, _ptr_array,
               dflash_accept_commit, dflash_bind_workspace, dflash_create, dflash_destroy,
               dflash_accept_commit_sampled, dflash_draft_block, dflash_get_error,
               dflash_inject_context, dflash_workspace_size, DflashSelector,
               dflash_selector_workspace_size, dflash_set_selector, dflash_draft_block_selector,
               dflash_accept_commit_sampled_q,
               _check, load_library)


def _stream():
    return torch.cuda.current_stream().cuda_stream


class KVCache:
    """Paged draft KV cache: per layer K and V pages [n_pages, 64, KVH, D].

    fp8: the pages hold one-byte E4M3 codes (uint8 tensors) with the per-layer
    scales k_scale / v_scale (sequences of n_layers floats).  draft_window W >
    0: the page table is a ring of pages_per_req pages keeping the newest W
    committed rows of each request (include/dflash.h, dflash_kv).
    """

    def __init__(self, cfg, batch, pages_per_req, page_table, dtype, device="cuda", fp8=False,
                 k_scale=None, v_scale=None, draft_window=0):
        self.batch = batch
        self.pages_per_req = pages_per_req
        self.page_table = torch.as_tensor(page_table, dtype=torch.int32).to(device).contiguous()
        self.n_pages = int(self.page_table.max().item()) + 1 if self.page_table.numel() else 1
        self.fp8 = bool(fp8)
        self.draft_window = int(draft_window)
        shape = (self.n_pages, cfg.page_size, cfg.n_kv_heads, cfg.head_dim)
        dt = torch.uint8 if self.fp8 else dtype
        self.k = [torch.zeros(shape, dtype=dt, device=device) for _ in range(cfg.n_layers)]
        self.v = [torch.zeros(shape, dtype=dt, device=device) for _ in range(cfg.n_layers)]
        self.kv_len = torch.zeros(batch, dtype=torch.int32, device=device)
        self._kp = _ptr_array(self.k)
        self._vp = _ptr_array(self.v)
        n = cfg.n_layers
        self.k_scale = list(k_scale) if k_scale is not None else [1.0] * n
        self.v_scale = list(v_scale) if v_scale is not None else [1.0] * n
        self._ks = (ctypes.c_float * n)(*self.k_scale)
        self._vs = (ctypes.c_float * n)(*self.v_scale)
        self.struct = DflashKV(ctypes.cast(self._kp, ctypes.POINTER(ctypes.c_void_p)),
                               ctypes.cast(self._vp, ctypes.POINTER(ctypes.c_void_p)),
                               self.page_table.data_ptr(), pages_per_req, self.n_pages,
                               self.kv_len.data_ptr(), self.draft_window,
                               ctypes.cast(self._ks, ctypes.POINTER(ctypes.c_float)),
                               ctypes.cast(self._vs, ctypes.POINTER(ctypes.c_float)))


class DraftSession:
    """One draft model bound to libdflash.

    cfg: object with the DraftConfig attributes; W: dict of device tensors in
    the layout of include/dflash.h (see synth.make_weights).
    """

    def __init__(self, cfg, W, max_batch, max_rows, max_position, kv_fp8=False):
        self.cfg = cfg
        self.W = W
        self.kv_fp8 = bool(kv_fp8)
        self.dtype = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
        self._win = (ctypes.c_int32 * cfg.n_layers)(*cfg.sliding_window)
        self.c = DflashConfig(DFLASH_F32 if cfg.dtype == "f32" else DFLASH_BF16, cfg.target_hidden,
                              cfg.n_sel, cfg.hidden, cfg.n_layers, cfg.n_heads, cfg.n_kv_heads,
                              cfg.head_dim, cfg.intermediate, cfg.vocab, cfg.mask_token_id,
                              cfg.block_size, cfg.page_size,
                              ctypes.cast(self._win, ctypes.POINTER(ctypes.c_int32)),
                              cfg.rms_eps, cfg.rope_theta, max_batch, max_rows, max_position,
                              1 if self.kv_fp8 else 0)
        Ls = W["layers"]
        self._arrs = {k: _ptr_array([L[k] for L in Ls]) for k in
                      ["qkv", "o", "gate_up", "down", "in_norm", "post_norm", "q_norm", "k_norm"]}
        cast = lambda a: ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p))  # noqa: E731
        A = self._arrs
        self.w = DflashWeights(W["fc"].data_ptr(), W["hidden_norm"].data_ptr(),
                               W["final_norm"].data_ptr(), W["embed"].data_ptr(),
                               W["lm_head"].data_ptr(), cast(A["qkv"]), cast(A["o"]),
                               cast(A["gate_up"]), cast(A["down"]), cast(A["in_norm"]),
                               cast(A["post_norm"]), cast(A["q_norm"]), cast(A["k_norm"]))
        self.h = dflash_create(self.c, self.w)
        self.ws_bytes = dflash_workspace_size(self.h)
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device="cuda")
        base = self.ws.data_ptr()
        self.ws_ptr = (base + 255) // 256 * 256
        dflash_bind_workspace(self.h, self.ws_ptr, self.ws_bytes, _stream())

    def close(self):
        if self.h is not None:
            dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_kv(self, batch, pages_per_req, page_table, k_scale=None, v_scale=None,
               draft_window=0):
        return KVCache(self.cfg, batch, pages_per_req, page_table, self.dtype, fp8=self.kv_fp8,
                       k_scale=k_scale, v_scale=v_scale, draft_window=draft_window)

    def inject(self, kv, feats, row_offset, n_rows, batch=None):
        """feats: [n_sel, rows, H_t] device tensor (or a list of n_sel [rows, H_t])."""
        batch = kv.batch if batch is None else batch
        fl = [feats[j] for j in range(self.cfg.n_sel)]
        rows = fl[0].shape[0]
        dflash_inject_context(self.h, kv.struct, batch, rows, fl, row_offset, n_rows, _stream())

    def draft(self, kv, anchor, draft_ids, hidden_out=None, batch=None):
        batch = kv.batch if batch is None else batch
        dflash_draft_block(self.h, kv.struct, batch, anchor, draft_ids, hidden_out, _stream())

    def accept(self, batch, draft_ids, posterior, seq_len, accept_len, commit_len, bonus,
               out_tokens, output_ids=None):
        stride = output_ids.shape[1] if output_ids is not None else 0
        dflash_accept_commit(self.h, batch, draft_ids, posterior, seq_len, accept_len, commit_len,
                             bonus, out_tokens, output_ids, stride, _stream())

    def accept_sampled(self, batch, draft_ids, probs, accept_u, exp_noise, seq_len, accept_len,
                       commit_len, bonus, out_tokens, output_ids=None):
        """Lossless sampled verification (include/dflash.h); probs [B, S, V],
        accept_u [B, S-1], exp_noise [B, V] float32 device tensors."""
        stride = output_ids.shape[1] if output_ids is not None else 0
        dflash_accept_commit_sampled(self.h, batch, draft_ids, probs, accept_u, exp_noise, seq_len,
                                     accept_len, commit_len, bonus, out_tokens, output_ids, stride,
                                     _stream())

    def accept_sampled_q(self, batch, draft_ids, probs, cand_ids, q_rows, accept_u, exp_noise,
                         seq_len, accept_len, commit_len, bonus, out_tokens, output_ids=None):
        """Sampled verification against a real proposal: cand_ids [B, S-1, K]
        int32 with q_rows [B, S-1, K] float32 (e.g. the selector's)."""
        stride = output_ids.shape[1] if output_ids is not None else 0
        dflash_accept_commit_sampled_q(self.h, batch, draft_ids, probs, cand_ids.shape[-1],
                                       cand_ids, q_rows, accept_u, exp_noise, seq_len, accept_len,
                                       commit_len, bonus, out_tokens, output_ids, stride,
                                       _stream())

    def set_selector(self, K, W_h, A, B):
        """DFlash 2 candidate selector (include/dflash.h): K candidates per
        position; W_h [rank, hidden], A and B [vocab, rank] device tensors in
        the model dtype (kept referenced here).  None for W_h removes it."""
        if W_h is None:
            dflash_set_selector(self.h, None, None, 0)
            self._sel = None
            return
        rank = W_h.shape[0]
        n = dflash_selector_workspace_size(self.h, K, rank)
        ws = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
        ptr = (ws.data_ptr() + 255) // 256 * 256
        sel = DflashSelector(K, rank, W_h.data_ptr(), A.data_ptr(), B.data_ptr())
        dflash_set_selector(self.h, sel, ptr, n)
        self._sel = (sel, ws, W_h, A, B)

    def draft_selector(self, kv, anchor, draft_ids, exp_noise=None, cand_ids=None, q_rows=None,
                       batch=None):
        """Draft block with the selector walk: greedy (exp_noise None) or
        sampled with exp_noise [B, S-1, K] Exp(1) float32."""
        batch = kv.batch if batch is None else batch
        dflash_draft_block_selector(self.h, kv.struct, batch, anchor, exp_noise, draft_ids,
                                    cand_ids, q_rows, _stream())

    def set_fusion(self, on):
        """Dependent GEMMs as one fused launch (True) or one launch each (False)."""
        lib = load_library()
        lib.dflash_test_set_fusion.argtypes = [ctypes.c_void_p, ctypes.c_int32]
        lib.dflash_test_set_fusion.restype = ctypes.c_int
        _check(lib.dflash_test_set_fusion(self.h, 1 if on else 0))

    def set_attention(self, kernel):
        """Attention kernel: "tc" (tcgen05 where it applies, the default) or
        "mma" (the mma.sync kernels only)."""
        lib = load_library()
        lib.dflash_test_set_attention.argtypes = [ctypes.c_void_p, ctypes.c_int32]
        lib.dflash_test_set_attention.restype = ctypes.c_int
        _check(lib.dflash_test_set_attention(self.h, {"tc": 0, "mma": 1}[kernel]))

    def error(self):
        return dflash_get_error(self.h, _stream())
