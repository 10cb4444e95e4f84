"""CPU-only checks of the C-ABI library: it loads, exports every declared
symbol, and its host-side validation refuses bad arguments without touching
a GPU (dflash_create and dflash_workspace_size make no CUDA call)."""
import ctypes
import os
import re

import pytest

import block_diffusion_speculative_fc_gb300 as pkg
from block_diffusion_speculative_fc_gb300 import _build
from synth import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkg.load_library()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(dflash_\w+)\s*\(", src, re.M))
    return sorted(names)


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"dflash_inject_context", "dflash_draft_block", "dflash_accept_commit"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(pkg.EXPORTED) <= set(names)
    assert "dflash_test_gemm" in names


def _session_structs(cfg, **over):
    win = (ctypes.c_int32 * cfg.n_layers)(*cfg.sliding_window)
    c = pkg.DflashConfig(pkg.DFLASH_F32 if cfg.dtype == "f32" else pkg.DFLASH_BF16,
                         cfg.target_hidden, cfg.n_sel, cfg.hidden, cfg.n_layers, cfg.n_heads,
                         cfg.n_kv_heads, cfg.head_dim, cfg.intermediate, cfg.vocab,
                         cfg.mask_token_id, cfg.block_size, cfg.page_size,
                         ctypes.cast(win, ctypes.POINTER(ctypes.c_int32)), cfg.rms_eps,
                         cfg.rope_theta, 4, 256, 4096)
    for k, v in over.items():
        setattr(c, k, v)
    fake = 0x10000  # never dereferenced by host-side code
    arr = (ctypes.c_void_p * cfg.n_layers)(*([fake] * cfg.n_layers))
    P = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    w = pkg.DflashWeights(fake, fake, fake, fake, fake, P, P, P, P, P, P, P, P)
    return c, w, (win, arr)


def test_create_validates_config(lib):
    cfg = WORKLOADS["tiny"].cfg
    c, w, keep = _session_structs(cfg)
    h = pkg.dflash_create(c, w)
    n = pkg.dflash_workspace_size(h)
    assert n > 0
    pkg.dflash_destroy(h)
    for field, bad in [("head_dim", 96), ("page_size", 32), ("block_size", 1), ("block_size", 40),
                       ("n_kv_heads", 3), ("hidden", 200), ("mask_token_id", 5000),
                       ("max_batch", 0), ("dtype", 7), ("n_sel", 9)]:
        c2, w2, keep2 = _session_structs(cfg, **{field: bad})
        with pytest.raises(pkg.DFlashError) as ei:
            pkg.dflash_create(c2, w2)
        assert ei.value.status in (-1, -2), (field, ei.value.status)


def test_calls_before_workspace_are_refused(lib):
    cfg = WORKLOADS["tiny"].cfg
    c, w, keep = _session_structs(cfg)
    h = pkg.dflash_create(c, w)
    kvarr = (ctypes.c_void_p * cfg.n_layers)(*([0x10000] * cfg.n_layers))
    P = ctypes.cast(kvarr, ctypes.POINTER(ctypes.c_void_p))
    kv = pkg.DflashKV(P, P, 0x10000, 4, 16, 0x10000)
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_draft_block(h, kv, 1, 0x10000, 0x10000, None, None)
    assert ei.value.status == -6
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_accept_commit(h, 1, 1, 1, 1, 1, 1, 1, 1, None, 0, None)
    assert ei.value.status == -6
    with pytest.raises(pkg.DFlashError):
        pkg.dflash_bind_workspace(h, None, 1 << 20, None)
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_bind_workspace(h, 0x10001, 1 << 40, None)   # misaligned
    assert ei.value.status == -1
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_bind_workspace(h, 0x10000, 16, None)        # too small
    assert ei.value.status == -3
    pkg.dflash_destroy(h)


def test_null_arguments_are_refused(lib):
    with pytest.raises(pkg.DFlashError):
        pkg.dflash_create(pkg.DflashConfig(), pkg.DflashWeights())
    assert lib.dflash_status_string(-3) == b"capacity exceeded"
    assert lib.dflash_workspace_size(None, None) == -1
    assert lib.dflash_inject_context(None, None, 0, 0, None, None, None, None) == -1
    pkg.dflash_destroy(None)


def test_selector_host_checks(lib):
    """Selector sizes, workspace and state checks are host-side (no CUDA)."""
    cfg = WORKLOADS["tiny"].cfg
    c, w, keep = _session_structs(cfg)
    h = pkg.dflash_create(c, w)
    for K, r in [(0, 16), (9, 16), (4, 0), (4, 257)]:
        with pytest.raises(pkg.DFlashError) as ei:
            pkg.dflash_selector_workspace_size(h, K, r)
        assert ei.value.status == -2, (K, r)
    rows, n_vt = 4 * cfg.block_size, (cfg.vocab + 127) // 128   # max_batch 4
    n1 = pkg.dflash_selector_workspace_size(h, 1, 16)
    n8 = pkg.dflash_selector_workspace_size(h, 8, 16)
    nr = pkg.dflash_selector_workspace_size(h, 8, 256)
    # per-tile keys, K bound slots per row, W_h h rows, merged candidates
    assert n8 >= n_vt * rows * 8 * 8 + rows * 8 * 8 + rows * 16 * 4 + rows * 8 * 8
    assert n1 < n8 < nr
    kvarr = (ctypes.c_void_p * cfg.n_layers)(*([0x10000] * cfg.n_layers))
    P = ctypes.cast(kvarr, ctypes.POINTER(ctypes.c_void_p))
    kv = pkg.DflashKV(P, P, 0x10000, 4, 16, 0x10000)
    with pytest.raises(pkg.DFlashError) as ei:      # no selector set
        pkg.dflash_draft_block_selector(h, kv, 1, 0x10000, None, 0x10000, None, None, None)
    assert ei.value.status == -6
    need = pkg.dflash_selector_workspace_size(h, 4, 16)
    sel = pkg.DflashSelector(4, 16, 0x10000, 0x10000, 0x10000)
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_set_selector(h, sel, 0x10000, need - 1)           # too small
    assert ei.value.status == -3
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_set_selector(h, sel, 0x10010, need)               # not 256-byte aligned
    assert ei.value.status == -1
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_set_selector(h, pkg.DflashSelector(4, 16, None, 0x10000, 0x10000), 0x10000, need)
    assert ei.value.status == -1
    pkg.dflash_set_selector(h, sel, 0x10000, need)
    with pytest.raises(pkg.DFlashError) as ei:      # selector set, but no workspace bound
        pkg.dflash_draft_block_selector(h, kv, 1, 0x10000, None, 0x10000, None, None, None)
    assert ei.value.status == -6
    pkg.dflash_set_selector(h, None, None, 0)       # removed again
    with pytest.raises(pkg.DFlashError) as ei:
        pkg.dflash_accept_commit_sampled_q(h, 1, 1, 1, 4, 1, 1, 1, 1, 1, 1, 1, 1, 1, None, 0, None)
    assert ei.value.status == -6                    # no workspace
    pkg.dflash_destroy(h)


def test_public_headers_compile_as_c_and_cpp():
    """The boundary is a C ABI: its headers must compile as plain C99
    (pedantic) and as C++, with no CUDA compiler involved."""
    import shutil
    import subprocess
    cc, cxx = shutil.which("gcc"), shutil.which("g++")
    if not cc or not cxx:
        pytest.skip("no host C/C++ compiler")
    inc = os.path.join(ROOT, "include")
    cuda_inc = "/usr/local/cuda/include"
    for h in sorted(f for f in os.listdir(inc) if f.endswith(".h")):
        path = os.path.join(inc, h)
        for cmd in ([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                     "-x", "c", "-I", cuda_inc, path],
                    [cxx, "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++", "-I",
                     cuda_inc, path]):
            r = subprocess.run(cmd, capture_output=True, text=True)
            assert r.returncode == 0, (h, r.stderr)


def test_plain_c_caller_links_and_runs(lib, tmp_path):
    """tests/abi_example.c: a C program built with gcc against include/ and
    linked to libdflash.so uses the host-side ABI (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc")
    if not cc:
        pytest.skip("no host C compiler")
    libdir = os.path.dirname(pkg.LIB_PATH)
    exe = str(tmp_path / "abi_example")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "abi_example.c"), "-L", libdir, "-ldflash",
                        "-Wl,-rpath," + libdir, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok workspace="), r.stdout
