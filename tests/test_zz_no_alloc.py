"""The allocation-free token selection entry point.

dflash_select_tokens_noalloc is for callers that cannot give the library
device memory (its scratch is a static device array of the library).  Its ids
must be the oracle's lm_head argmax of the same bf16 rows (identical except
where the oracle's top-2 margin is below 1e-2), call after call, with a zero
status word; they must also agree with dflash_draft_block's own lm_head +
argmax.  This file is collected last so that a failure here never hides the
other GPU tests.
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
from synth import WORKLOADS, make_features, make_weights  # noqa: E402
from synth.configs import shrink  # noqa: E402

# the near-tie margin the parity tests use for drafted ids
MARGIN = 1e-2

CFG = shrink(WORKLOADS["qwen8b-b1"].cfg, name="noalloc-mini", target_hidden=256, hidden=512,
             n_layers=2, n_heads=8, n_kv_heads=2, intermediate=1024, vocab=4096,
             mask_token_id=4095)


def _lib():
    lib = pkg.load_library()
    lib.dflash_select_tokens_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.dflash_select_tokens_noalloc.restype = ctypes.c_int
    return lib


def test_select_tokens_noalloc_matches_draft_block():
    lib = _lib()
    W = make_weights(CFG, seed=3, device="cuda", gains="random")
    S, H = CFG.block_size, CFG.hidden
    sess = pkg.DraftSession(CFG, W, max_batch=2, max_rows=256, max_position=1024)
    kv = sess.new_kv(2, 4, np.arange(8, dtype=np.int32).reshape(2, 4))
    i32 = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device="cuda")  # noqa: E731
    feats = make_features(CFG, 150, 3, "noalloc", device="cuda")
    sess.inject(kv, feats, i32([0, 100]), i32([100, 50]))
    draft = torch.zeros((2, S), dtype=torch.int32, device="cuda")
    hid = torch.zeros((2, S, H), dtype=torch.bfloat16, device="cuda")
    sess.draft(kv, i32([7, 11]), draft, hid)
    assert sess.error() == 0
    # rows 1..S-1 of each request, as the draft block scored them
    rows = hid[:, 1:, :].reshape(-1, H).contiguous()
    ref = draft[:, 1:].reshape(-1).cpu().numpy()
    n = rows.shape[0]
    assert n <= 32
    # the oracle's greedy choice on exactly the rows the call reads
    want, margin = O.lm_head_argmax(rows.double().cpu().numpy(), W["lm_head"].double().cpu().numpy())
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.full((1,), 0xDEAD, dtype=torch.int32, device="cuda")
    for call in range(2):     # the static scratch keeps the last call's contents
        ids = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        st = lib.dflash_select_tokens_noalloc(sess.h, n, rows.data_ptr(), ids.data_ptr(),
                                              status.data_ptr(), stream)
        assert st == 0, pkg.load_library().dflash_last_error()
        got = ids.cpu().numpy()
        assert status.item() == 0, (call, status.item())
        off = [r for r in range(n) if got[r] != want[r]]
        assert all(margin[r] < MARGIN for r in off), (call, [(r, got[r], want[r], margin[r]) for r in off])
        # and the draft block's own lm_head + argmax on the same rows
        off_draft = [r for r in range(n) if got[r] != ref[r]]
        assert all(margin[r] < MARGIN for r in off_draft), (call, off_draft)
        assert np.all(got >= 0) and np.all(got < CFG.vocab)
        status.fill_(0xDEAD)
    sess.close()


def test_select_tokens_noalloc_refuses_too_many_rows():
    lib = _lib()
    W = make_weights(CFG, seed=4, device="cuda")
    sess = pkg.DraftSession(CFG, W, max_batch=1, max_rows=64, max_position=256)
    x = torch.zeros((33, CFG.hidden), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(33, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.dflash_select_tokens_noalloc(sess.h, 33, x.data_ptr(), ids.data_ptr(), None, stream)
    assert st == -3
    # a hidden pointer off the 16-byte grid is refused on the host
    st = lib.dflash_select_tokens_noalloc(sess.h, 4, x.data_ptr() + 2, ids.data_ptr(), None, stream)
    assert st == -1
    sess.close()
