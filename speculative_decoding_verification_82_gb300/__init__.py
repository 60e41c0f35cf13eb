"""GB300 (sm_103a) kernels for the target-side verification step of speculative decoding.

The compute path is the C-ABI library built from csrc/ (declared in include/spec_verify.h);
`binding` exposes its entry points under the same names for torch CUDA tensors.
"""

from .binding import (  # noqa: F401
    SpecVerifyError,
    library,
    make_workspace,
    workspace_reset,
    spec_kv_compact,
    spec_ngram_draft,
    spec_verify_chain,
    spec_verify_ngram,
    spec_verify_tree_greedy,
    spec_verify_tree_walk,
    workspace_bytes,
)
