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
    tl, dl = parity.to_device(ci.target, ci.dtype), parity.to_device(ci.draft, ci.dtype)
    x, r, u = parity.i32(ci.draft_tokens), parity.f32(ci.r), parity.f32(ci.u)
    na = torch.full((ci.B,), -9, dtype=torch.int32, device=dev)
    ot = torch.full((ci.B, ci.K + 1), -9, dtype=torch.int32, device=dev)
    rm = torch.full((ci.B,), -9.0, device=dev)
    ef = torch.full((ci.B,), -9, dtype=torch.int32, device=dev)
    P = ctypes.c_void_p
    st = lib.spec_verify_chain_static(P(tl.data_ptr()), P(dl.data_ptr()), binding.DTYPE_CODE[tl.dtype],
                                      ci.B, ci.K, ci.V, float(ci.temperature), P(x.data_ptr()),
                                      P(r.data_ptr()), P(u.data_ptr()), P(na.data_ptr()),
                                      P(ot.data_ptr()), P(rm.data_ptr()), P(ef.data_ptr()),
                                      P(torch.cuda.current_stream().cuda_stream))
    assert st == binding.SPEC_OK, lib.spec_status_string(st)
    torch.cuda.synchronize()
    return dict(num_accepted=na.cpu().numpy(), out_tokens=ot.cpu().numpy(),
                residual_mass=rm.cpu().numpy(), err_flags=ef.cpu().numpy())


def test_static_scratch_matches_workspace_entry_point(lib):
    for seed, dtype in ((21, "f32"), (22, "bf16")):  # two calls in a row share the array
        ci = synth.chain_batched(seed=seed, B=8, V=20011, dtype=dtype)
        got = _static_call(lib, ci)
        ref = parity.run_gpu_chain(ci, diag=False)
        for key in ("num_accepted", "out_tokens", "err_flags"):
            assert np.array_equal(got[key], ref[key]), (seed, key)
        assert np.abs(got["residual_mass"] - ref["residual_mass"]).max() <= parity.PROB_TOL
        parity.compare_chain(dict(ref, **got), parity.run_oracle_chain(ci), ci)


def test_static_scratch_rejects_too_large_a_call(lib):
    # 4096 requests of 11 rows at V = 128256 need more scratch than the fixed array holds; the
    # host rejects the call before touching any pointer.
    need = lib.spec_verify_workspace_bytes(4096, 11, 128256, 0)
    assert need > binding.STATIC_WORKSPACE_BYTES
    P = ctypes.c_void_p
    st = lib.spec_verify_chain_static(P(1 << 20), P(2 << 20), 0, 4096, 5, 128256, 1.0, P(3 << 20),
                                      P(4 << 20), P(5 << 20), P(6 << 20), P(7 << 20), None, None, None)
    assert st == binding.SPEC_ERR_UNSUPPORTED
