"""spec_verify_chain_static: the entry point for callers that cannot allocate device memory.

Such callers (a plugin inside an engine that keeps all GPU memory in its own pool, a hook that
must not call cudaMalloc because it can synchronise the device) pass only inputs and outputs; the
library's scratch is a fixed device array inside the library.  These tests call it through the
C ABI and check it against spec_verify_chain with a caller-provided workspace, on two calls in a
row with different inputs, so results left in the shared array by one call cannot leak into the
next.  The file is named to run last.
"""

import ctypes

import numpy as np
import pytest
import torch

import parity
from speculative_decoding_verification_82_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return binding.library()


def _static_call(lib, ci):
    dev = "cuda"
    greedy = float(ci.temperature) == 0.0
    tl = parity.to_device(ci.target, ci.dtype)
    dl = None if greedy else parity.to_device(ci.draft, ci.dtype)
    x, r, u = parity.i32(ci.draft_tokens), parity.f32(ci.r), parity.f32(ci.u)
    na = torch.full((ci.B,), -9, dtype=torch.int32, device=dev)
    ot = torch.full((ci.B, ci.K + 1), -9, dtype=torch.int32, device=dev)
    rm = torch.full((ci.B,), -9.0, device=dev)
    ef = torch.full((ci.B,), -9, dtype=torch.int32, device=dev)
    P = ctypes.c_void_p
    ptr = lambda t: P(t.data_ptr()) if t is not None else None  # noqa: E731
    st = lib.spec_verify_chain_static(ptr(tl), ptr(dl), binding.DTYPE_CODE[tl.dtype],
                                      ci.B, ci.K, ci.V, float(ci.temperature), ptr(x),
                                      ptr(r), ptr(u), ptr(na), ptr(ot), ptr(rm), ptr(ef),
                                      P(torch.cuda.current_stream().cuda_stream))
    assert st == binding.SPEC_OK, lib.spec_status_string(st)
    torch.cuda.synchronize()
    return dict(num_accepted=na.cpu().numpy(), out_tokens=ot.cpu().numpy(),
                residual_mass=rm.cpu().numpy(), err_flags=ef.cpu().numpy())


def _check(lib, ci):
    got = _static_call(lib, ci)
    ref = parity.run_gpu_chain(ci, diag=False)
    for key in ("num_accepted", "out_tokens", "err_flags"):
        assert np.array_equal(got[key], ref[key]), key
    assert np.abs(got["residual_mass"] - ref["residual_mass"]).max() <= parity.PROB_TOL
    parity.compare_chain(dict(ref, **got), parity.run_oracle_chain(ci, threads=16), ci)


def test_static_scratch_matches_workspace_entry_point(lib):
    for seed, dtype in ((21, "f32"), (22, "bf16")):  # two calls in a row share the array
        _check(lib, synth.chain_batched(seed=seed, B=8, V=20011, dtype=dtype))


def test_static_scratch_greedy_and_headline_size(lib):
    """Greedy verification (K + 1 rows of scratch per request) and the largest headline batch that
    the array holds (B = 64, K = 5, V = 128256, fp32 with draft logits: 2K + 1 rows)."""
    ci = synth.chain_small_vocab(seed=3, B=16, temperature=0.0)
    _check(lib, ci)
    full = synth.chain_batched(seed=4)
    need = lib.spec_verify_workspace_bytes(full.B, 2 * full.K + 1, full.V, 0)
    assert need <= binding.STATIC_WORKSPACE_BYTES
    _check(lib, full)


def test_static_scratch_rejects_too_large_a_call(lib):
    # The smallest batch of 11-row requests at V = 128256 whose scratch exceeds the fixed array is
    # rejected before anything is launched; every pointer is NULL, so a call that got past the size
    # check would fail on the pointers (SPEC_ERR_INVALID_ARG) instead of reaching a kernel.
    B = 1
    while lib.spec_verify_workspace_bytes(B, 11, 128256, 0) <= binding.STATIC_WORKSPACE_BYTES:
        B += 1
    for b in (B, 4096):
        st = lib.spec_verify_chain_static(None, None, 0, b, 5, 128256, ctypes.c_float(1.0), None, None,
                                          None, None, None, None, None, None)
        assert st == binding.SPEC_ERR_UNSUPPORTED
    # a draft length beyond SPEC_MAX_K: the same status as spec_verify_chain gives
    st = lib.spec_verify_chain_static(None, None, 0, 1, 1 << 30, 16, ctypes.c_float(1.0), None, None,
                                      None, None, None, None, None, None)
    assert st == binding.SPEC_ERR_UNSUPPORTED
