"""The C-ABI library loads, exports every symbol include/spec_verify.h declares, and rejects bad
arguments on the host before any CUDA call.  The argument checks pass placeholder device
addresses, so they run only where no GPU is visible: should a regression let one of those calls
reach a launch, nothing would read the addresses."""

import ctypes
import os
import re

import pytest

from speculative_decoding_verification_82_gb300 import binding
from speculative_decoding_verification_82_gb300.build import INCLUDE, build

HEADER = os.path.join(INCLUDE, "spec_verify.h")


def _gpu_visible() -> bool:
    try:
        import torch
    except ImportError:
        return False
    return torch.cuda.is_available()


host_only = pytest.mark.skipif(_gpu_visible(), reason="placeholder device addresses: run without a GPU")


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_workspace_size(lib):
    # V = 128256 fp32 spans at most 32064 16-byte vectors: 16 stats chunks of 2048 vectors and 32
    # residual chunks of 1024.  Layout: counters (two 128-byte lines, 2 * B * rows u32 counts,
    # padded to 16 B), request states (32 B each) and the residual queue (five 8-byte words per
    # request), together padded to 256 B; then chunk stats, sub-chunk stats (8 per chunk), row stats
    # and residual sub-sums (8 per residual chunk; 8 bytes each: the value and the call's tag), each
    # padded to 256 B.
    def up(x, a=256):
        return (x + a - 1) // a * a

    B, rows, n, nr = 64, 11, 16, 32
    want = (up(up(256 + 2 * B * rows * 4, 16) + B * 32 + B * 40) + up(B * rows * n * 16)
            + up(B * rows * n * 8 * 16) + up(B * rows * 32) + up(B * rows * nr * 8 * 8))
    assert lib.spec_verify_workspace_bytes(B, rows, 128256, 0) == want
    assert lib.spec_verify_workspace_bytes(-1, 6, 100, 0) == 0
    assert lib.spec_verify_workspace_bytes(4, 0, 100, 0) == 0
    assert lib.spec_verify_workspace_bytes(4, 6, 0, 0) == 0
    assert lib.spec_verify_workspace_bytes(4, 6, 100, 7) == 0
    # bf16 halves the bytes per element: 128256 bf16 rows are 8 chunks
    assert lib.spec_verify_workspace_bytes(64, 11, 128256, 1) < lib.spec_verify_workspace_bytes(64, 11, 128256, 0)


def test_status_strings(lib):
    assert lib.spec_status_string(0) == b"SPEC_OK"
    assert lib.spec_status_string(3) == b"SPEC_ERR_WORKSPACE"


def _chain(lib, **kw):
    a = dict(target=1 << 20, draft=2 << 20, dtype=0, B=2, K=3, V=100, T=1.0, temps=0, x=3 << 20, r=4 << 20,
             u=5 << 20, na=6 << 20, ot=7 << 20, ws=1 << 30, wsb=10 ** 6)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.spec_verify_chain(P(a["target"]), P(a["draft"]), a["dtype"], a["B"], a["K"], a["V"],
                                 a["T"], P(a["temps"]), P(a["x"]), P(a["r"]), P(a["u"]), P(a["na"]),
                                 P(a["ot"]), None, None, None, None, None, None, None, P(a["ws"]), a["wsb"],
                                 None)


@host_only
def test_host_validation_rejects_before_launch(lib):
    # Each call fails its checks on the host, so no device pointer is ever touched.
    assert _chain(lib, B=0) == binding.SPEC_OK  # empty batch: nothing to do
    assert _chain(lib, V=0) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, K=-1) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, dtype=9) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, T=-0.5) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, T=float("nan")) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, T=float("inf")) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, K=300) == binding.SPEC_ERR_UNSUPPORTED  # beyond SPEC_MAX_K
    assert _chain(lib, draft=0) == binding.SPEC_ERR_INVALID_ARG  # T > 0 needs draft logits
    assert _chain(lib, r=0) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, target=0) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, target=(1 << 20) + 2) == binding.SPEC_ERR_INVALID_ARG  # misaligned fp32
    assert _chain(lib, ws=0) == binding.SPEC_ERR_WORKSPACE
    assert _chain(lib, wsb=100) == binding.SPEC_ERR_WORKSPACE
    assert _chain(lib, ws=(1 << 30) + 16) == binding.SPEC_ERR_WORKSPACE  # workspace 256-B aligned
    assert _chain(lib, wsb=20000, V=10 ** 6) == binding.SPEC_ERR_WORKSPACE  # too small for this V
    # per-request temperatures: any request may sample, so draft logits, r and u are required even
    # when the call's own temperature is 0, and the workspace holds 2K + 1 rows per request
    assert _chain(lib, T=0.0, temps=8 << 20, draft=0) == binding.SPEC_ERR_INVALID_ARG
    assert _chain(lib, T=0.0, temps=8 << 20, u=0) == binding.SPEC_ERR_INVALID_ARG
    need = lib.spec_verify_workspace_bytes(2, 7, 100, 0)
    assert _chain(lib, T=0.0, temps=8 << 20, wsb=lib.spec_verify_workspace_bytes(2, 4, 100, 0)) == \
        binding.SPEC_ERR_WORKSPACE and need > lib.spec_verify_workspace_bytes(2, 4, 100, 0)


@host_only
def test_tree_validation(lib):
    P = ctypes.c_void_p
    f = lib.spec_verify_tree_greedy
    ok = dict(t=1 << 20, dt=1, B=2, N=5, V=64, tok=2 << 20, par=3 << 20, al=4 << 20, pn=5 << 20,
              ot=6 << 20, ws=1 << 30, wsb=10 ** 6)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(P(a["t"]), a["dt"], a["B"], a["N"], a["V"], P(a["tok"]), P(a["par"]), P(a["al"]),
                 P(a["pn"]), P(a["ot"]), None, None, P(a["ws"]), a["wsb"], None)

    assert call(B=0) == binding.SPEC_OK
    assert call(N=-1) == binding.SPEC_ERR_INVALID_ARG
    assert call(N=5000) == binding.SPEC_ERR_UNSUPPORTED
    assert call(par=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(wsb=10) == binding.SPEC_ERR_WORKSPACE


def test_workspace_reset_is_host_only(lib):
    # marks a pointer for clearing at its next call; touches no memory, so any pointer is fine
    lib.spec_verify_workspace_reset(None)
    lib.spec_verify_workspace_reset(ctypes.c_void_p(0x1000))
    lib.spec_verify_workspace_reset(ctypes.c_void_p(0x1000))


@host_only
def test_tree_walk_validation(lib):
    P = ctypes.c_void_p
    f = lib.spec_verify_tree_walk
    ok = dict(t=1 << 20, d=7 << 20, dt=1, B=2, N=5, V=64, T=1.0, tok=2 << 20, par=3 << 20,
              r=8 << 20, u=9 << 20, al=4 << 20, pn=5 << 20, ot=6 << 20)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(P(a["t"]), P(a["d"]), a["dt"], a["B"], a["N"], a["V"], a["T"], P(a.get("temps", 0)), P(a["tok"]),
                 P(a["par"]), P(a["r"]), P(a["u"]), P(a["al"]), P(a["pn"]), P(a["ot"]), None, None,
                 None, None)

    assert call(B=0) == binding.SPEC_OK
    assert call(dt=5) == binding.SPEC_ERR_INVALID_ARG
    assert call(N=-1) == binding.SPEC_ERR_INVALID_ARG
    assert call(V=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(T=-1.0) == binding.SPEC_ERR_INVALID_ARG
    assert call(T=float("nan")) == binding.SPEC_ERR_INVALID_ARG
    assert call(N=binding.MAX_WALK_NODES) == binding.SPEC_ERR_UNSUPPORTED
    assert call(V=binding.MAX_WALK_VOCAB + 1) == binding.SPEC_ERR_UNSUPPORTED
    assert call(par=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(d=0) == binding.SPEC_ERR_INVALID_ARG        # T > 0 needs draft logits
    assert call(r=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(t=(1 << 20) + 1) == binding.SPEC_ERR_INVALID_ARG  # misaligned bf16
    assert call(T=0.0, temps=9 << 20, d=0) == binding.SPEC_ERR_INVALID_ARG  # per-request T needs the draft


@host_only
def test_ngram_draft_validation(lib):
    P = ctypes.c_void_p
    f = lib.spec_ngram_draft
    ok = dict(ctx=1 << 20, cl=2 << 20, B=4, Lmax=100, nmax=4, nmin=1, K=5, d=3 << 20, dl=4 << 20)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(P(a["ctx"]), P(a["cl"]), a["B"], a["Lmax"], a["nmax"], a["nmin"], a["K"], P(a["d"]),
                 P(a["dl"]), None, None, None, None)

    assert call(B=0) == binding.SPEC_OK
    assert call(B=-1) == binding.SPEC_ERR_INVALID_ARG
    assert call(K=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(nmin=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(nmin=5) == binding.SPEC_ERR_INVALID_ARG      # n_min > n_max
    assert call(nmax=binding.MAX_NGRAM + 1) == binding.SPEC_ERR_UNSUPPORTED
    assert call(K=binding.MAX_K + 1) == binding.SPEC_ERR_UNSUPPORTED
    assert call(ctx=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(d=0) == binding.SPEC_ERR_INVALID_ARG


@host_only
def test_kv_compact_validation(lib):
    P = ctypes.c_void_p
    f = lib.spec_kv_compact
    arr = (P * 2)(P(1 << 20), P(2 << 20))
    ok = dict(C=2, S=100, W=64, B=3, N=5, sl=3 << 20, pa=4 << 20, al=5 << 20, pn=6 << 20)

    def call(caches=arr, **kw):
        a = dict(ok)
        a.update(kw)
        return f(caches, a["C"], a["S"], a["W"], a["B"], a["N"], P(a["sl"]), P(a["pa"]), P(a["al"]), P(a["pn"]),
                 None, None)

    assert call(B=0) == binding.SPEC_OK
    assert call(C=0) == binding.SPEC_OK
    assert call(W=24) == binding.SPEC_ERR_INVALID_ARG           # rows a multiple of 16 bytes
    assert call(B=-1) == binding.SPEC_ERR_INVALID_ARG
    assert call(N=binding.MAX_WALK_NODES) == binding.SPEC_ERR_UNSUPPORTED
    assert call(C=binding.MAX_KV_CACHES + 1) == binding.SPEC_ERR_UNSUPPORTED
    assert call(sl=0) == binding.SPEC_ERR_INVALID_ARG
    assert call(caches=(P * 2)(P(1 << 20), P((2 << 20) + 8))) == binding.SPEC_ERR_INVALID_ARG  # misaligned
    assert call(caches=(P * 2)(P(1 << 20), None)) == binding.SPEC_ERR_INVALID_ARG


def test_header_is_plain_c(tmp_path):
    """The ABI header compiles as strict C99 (no C++ or CUDA types in the signatures)."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        import pytest

        pytest.skip("gcc not found")
    src = tmp_path / "use.c"
    src.write_text('#include "spec_verify.h"\nint main(void) { return spec_status_string(SPEC_OK) == 0; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
