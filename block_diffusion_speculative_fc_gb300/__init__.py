"""Python binding of libdflash (the GB300 DFlash draft-pass library).

Argument marshalling only: every step of the draft pass runs in the CUDA
kernels behind the C ABI declared in include/dflash.h.  The functions below
carry the C names; `DraftSession` is a convenience owner of the ctypes
structures and of torch-allocated device buffers (weights, KV pages,
workspace).  There is no fallback: if the library is missing or no CUDA
device is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")

c_int32, c_float, c_void_p, c_size_t = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
P_VOID = ctypes.POINTER(c_void_p)

DFLASH_F32, DFLASH_BF16 = 0, 1
DERR_BITS = {0x1: "KV_CAPACITY", 0x2: "PAGE_RANGE", 0x4: "TOKEN_RANGE", 0x8: "POSITION",
             0x10: "OUTPUT_ROW", 0x20: "TIMEOUT", 0x40: "ROW_RANGE"}
EXPORTED = ["dflash_create", "dflash_destroy", "dflash_workspace_size", "dflash_bind_workspace",
            "dflash_inject_context", "dflash_draft_block", "dflash_accept_commit",
            "dflash_accept_commit_sampled",
            "dflash_selector_workspace_size", "dflash_set_selector", "dflash_draft_block_selector",
            "dflash_accept_commit_sampled_q",
            "dflash_get_error", "dflash_status_string", "dflash_last_error",
            "dflash_profile_enable", "dflash_profile_disable", "dflash_profile_collect"]


class DflashConfig(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("target_hidden", c_int32), ("n_sel", c_int32),
                ("hidden", c_int32), ("n_layers", c_int32), ("n_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("intermediate", c_int32),
                ("vocab", c_int32), ("mask_token_id", c_int32), ("block_size", c_int32),
                ("page_size", c_int32), ("sliding_window", ctypes.POINTER(c_int32)),
                ("rms_eps", c_float), ("rope_theta", c_float), ("max_batch", c_int32),
                ("max_rows", c_int32), ("max_position", c_int32), ("kv_fp8", c_int32)]


class DflashWeights(ctypes.Structure):
    _fields_ = [("fc_w", c_void_p), ("hidden_norm_g", c_void_p), ("final_norm_g", c_void_p),
                ("embed", c_void_p), ("lm_head", c_void_p), ("qkv_w", P_VOID), ("o_w", P_VOID),
                ("gate_up_w", P_VOID), ("down_w", P_VOID), ("in_norm_g", P_VOID),
                ("post_norm_g", P_VOID), ("q_norm_g", P_VOID), ("k_norm_g", P_VOID)]


class DflashKV(ctypes.Structure):
    _fields_ = [("k_pages", P_VOID), ("v_pages", P_VOID), ("page_table", c_void_p),
                ("pages_per_req", c_int32), ("n_pages", c_int32), ("kv_len", c_void_p),
                ("draft_window", c_int32), ("k_scale", ctypes.POINTER(c_float)),
                ("v_scale", ctypes.POINTER(c_float))]


class DflashSelector(ctypes.Structure):
    _fields_ = [("K", c_int32), ("rank", c_int32), ("W_h", c_void_p), ("A", c_void_p),
                ("B", c_void_p)]


class DflashProfileEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", c_int32), ("total_ms", c_float)]


class DFlashError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lib = None


def load_library(path=LIB_PATH):
    """Load libdflash.so (build it with __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libdflash.so not built at {path}; run block_diffusion_speculative_fc_gb300._build.build()")
    lib = ctypes.CDLL(path)
    lib.dflash_create.argtypes = [ctypes.POINTER(DflashConfig), ctypes.POINTER(DflashWeights),
                                  ctypes.POINTER(c_void_p)]
    lib.dflash_destroy.argtypes = [c_void_p]
    lib.dflash_destroy.restype = None
    lib.dflash_workspace_size.argtypes = [c_void_p, ctypes.POINTER(c_size_t)]
    lib.dflash_bind_workspace.argtypes = [c_void_p, c_void_p, c_size_t, c_void_p]
    lib.dflash_inject_context.argtypes = [c_void_p, ctypes.POINTER(DflashKV), c_int32, c_int32,
                                          P_VOID, c_void_p, c_void_p, c_void_p]
    lib.dflash_draft_block.argtypes = [c_void_p, ctypes.POINTER(DflashKV), c_int32, c_void_p,
                                       c_void_p, c_void_p, c_void_p]
    lib.dflash_accept_commit.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_void_p]
    lib.dflash_accept_commit_sampled.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                 c_void_p, c_void_p, c_int32, c_void_p]
    lib.dflash_selector_workspace_size.argtypes = [c_void_p, c_int32, c_int32, ctypes.POINTER(c_size_t)]
    lib.dflash_set_selector.argtypes = [c_void_p, ctypes.POINTER(DflashSelector), c_void_p, c_size_t]
    lib.dflash_draft_block_selector.argtypes = [c_void_p, ctypes.POINTER(DflashKV), c_int32, c_void_p,
                                                c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    lib.dflash_accept_commit_sampled_q.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_int32,
                                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                   c_int32, c_void_p]
    lib.dflash_get_error.argtypes = [c_void_p, c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    lib.dflash_profile_enable.argtypes = [c_void_p, c_int32]
    lib.dflash_profile_disable.argtypes = [c_void_p]
    lib.dflash_profile_collect.argtypes = [c_void_p, ctypes.POINTER(DflashProfileEntry), c_int32,
                                           ctypes.POINTER(c_int32)]
    lib.dflash_status_string.argtypes = [ctypes.c_int]
    lib.dflash_status_string.restype = ctypes.c_char_p
    lib.dflash_last_error.argtypes = []
    lib.dflash_last_error.restype = ctypes.c_char_p
    for name in ["dflash_create", "dflash_workspace_size", "dflash_bind_workspace",
                 "dflash_inject_context", "dflash_draft_block", "dflash_accept_commit",
                 "dflash_accept_commit_sampled", "dflash_selector_workspace_size",
                 "dflash_set_selector", "dflash_draft_block_selector",
                 "dflash_accept_commit_sampled_q", "dflash_get_error", "dflash_profile_enable", "dflash_profile_disable",
                 "dflash_profile_collect"]:
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(st):
    if st != 0:
        lib = load_library()
        msg = lib.dflash_last_error().decode() or lib.dflash_status_string(st).decode()
        raise DFlashError(st, msg)
    return st


def _p(x):
    """Device pointer of a torch tensor, an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptr_array(ptrs):
    return (c_void_p * len(ptrs))(*[_p(t) for t in ptrs])


# ------------------------------------------------------------- C entry points
def dflash_create(cfg: DflashConfig, weights: DflashWeights):
    h = c_void_p()
    _check(load_library().dflash_create(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(h)))
    return h


def dflash_destroy(h):
    load_library().dflash_destroy(h)


def dflash_workspace_size(h):
    n = c_size_t()
    _check(load_library().dflash_workspace_size(h, ctypes.byref(n)))
    return n.value


def dflash_bind_workspace(h, ws, nbytes, stream):
    _check(load_library().dflash_bind_workspace(h, _p(ws), nbytes, stream))


def dflash_inject_context(h, kv: DflashKV, batch, total_rows, target_feats, row_offset, n_rows, stream):
    feats = _ptr_array(target_feats)
    _check(load_library().dflash_inject_context(h, ctypes.byref(kv), batch, total_rows, feats,
                                                _p(row_offset), _p(n_rows), stream))


def dflash_draft_block(h, kv: DflashKV, batch, anchor, draft_ids, hidden_out, stream):
    _check(load_library().dflash_draft_block(h, ctypes.byref(kv), batch, _p(anchor), _p(draft_ids),
                                             _p(hidden_out), stream))


def dflash_accept_commit(h, batch, draft_ids, posterior, seq_len, accept_len, commit_len, bonus,
                         out_tokens, output_ids, out_stride, stream):
    _check(load_library().dflash_accept_commit(h, batch, _p(draft_ids), _p(posterior), _p(seq_len),
                                               _p(accept_len), _p(commit_len), _p(bonus),
                                               _p(out_tokens), _p(output_ids), out_stride, stream))


def dflash_accept_commit_sampled(h, batch, draft_ids, probs, accept_u, exp_noise, seq_len,
                                 accept_len, commit_len, bonus, out_tokens, output_ids, out_stride,
                                 stream):
    _check(load_library().dflash_accept_commit_sampled(
        h, batch, _p(draft_ids), _p(probs), _p(accept_u), _p(exp_noise), _p(seq_len),
        _p(accept_len), _p(commit_len), _p(bonus), _p(out_tokens), _p(output_ids), out_stride,
        stream))


def dflash_selector_workspace_size(h, K, rank):
    n = c_size_t()
    _check(load_library().dflash_selector_workspace_size(h, K, rank, ctypes.byref(n)))
    return n.value


def dflash_set_selector(h, sel, workspace, nbytes):
    """sel: DflashSelector or None (removes the selector)."""
    _check(load_library().dflash_set_selector(h, ctypes.byref(sel) if sel is not None else None,
                                              _p(workspace), nbytes))


def dflash_draft_block_selector(h, kv: DflashKV, batch, anchor, exp_noise, draft_ids, cand_ids,
                                q_rows, stream):
    _check(load_library().dflash_draft_block_selector(h, ctypes.byref(kv), batch, _p(anchor),
                                                      _p(exp_noise), _p(draft_ids), _p(cand_ids),
                                                      _p(q_rows), stream))


def dflash_accept_commit_sampled_q(h, batch, draft_ids, probs, K, cand_ids, q_rows, accept_u,
                                   exp_noise, seq_len, accept_len, commit_len, bonus, out_tokens,
                                   output_ids, out_stride, stream):
    _check(load_library().dflash_accept_commit_sampled_q(
        h, batch, _p(draft_ids), _p(probs), K, _p(cand_ids), _p(q_rows), _p(accept_u),
        _p(exp_noise), _p(seq_len), _p(accept_len), _p(commit_len), _p(bonus), _p(out_tokens),
        _p(output_ids), out_stride, stream))


def dflash_get_error(h, stream):
    """Returns the device error word (0 = clean) after synchronising the stream."""
    w = ctypes.c_uint32()
    st = load_library().dflash_get_error(h, stream, ctypes.byref(w))
    if st not in (0, -5):
        _check(st)
    return w.value


def dflash_profile_enable(h, max_records):
    _check(load_library().dflash_profile_enable(h, max_records))


def dflash_profile_disable(h):
    _check(load_library().dflash_profile_disable(h))


def dflash_profile_collect(h, cap=64):
    """{kernel name: (launches, total_ms)} of the launches recorded since enable."""
    arr = (DflashProfileEntry * cap)()
    n = c_int32()
    _check(load_library().dflash_profile_collect(h, arr, cap, ctypes.byref(n)))
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n.value)}


def decode_error(word):
    return [name for bit, name in DERR_BITS.items() if word & bit]


from .session import DraftSession  # noqa: E402,F401
