"""Thin ctypes binding of the C ABI declared in include/spec_verify.h.

Argument marshalling only: the functions take torch CUDA tensors, check their shape, dtype and
device, allocate outputs and the workspace when the caller did not supply them, and pass raw
pointers and the current CUDA stream to the library.  Every step of the verification runs in the
library's kernels; there is no other implementation to fall back on, so a missing library raises.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int, c_size_t, c_void_p

import torch

from .build import LIB_PATH

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_CUDA, SPEC_ERR_WORKSPACE, SPEC_ERR_UNSUPPORTED = range(5)
ERRF_BAD_TOKEN, ERRF_NONFINITE, ERRF_TIMEOUT, ERRF_BAD_TREE, ERRF_BAD_TEMPERATURE = 1, 2, 4, 8, 16
MAX_K, MAX_TREE_NODES, MAX_WALK_NODES, MAX_WALK_VOCAB, MAX_NGRAM = 256, 4096, 1024, 262144, 32
MAX_KV_CACHES = 1024
DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}

EXPORTED = ("spec_verify_workspace_bytes", "spec_verify_workspace_reset", "spec_verify_chain",
            "spec_verify_ngram", "spec_verify_tree_greedy", "spec_verify_tree_walk", "spec_ngram_draft",
            "spec_kv_compact",
            "spec_verify_chain_static", "spec_status_string")
STATIC_WORKSPACE_BYTES = 4 << 20

_lib = None


class SpecVerifyError(RuntimeError):
    pass


def library(path: str | None = None) -> ctypes.CDLL:
    """Load libspecverify.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise SpecVerifyError(f"CUDA library not built: {p} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    P, I, F, Z = c_void_p, c_int, c_float, c_size_t
    lib.spec_verify_workspace_bytes.argtypes = [I, I, I, I]
    lib.spec_verify_workspace_bytes.restype = Z
    lib.spec_verify_workspace_reset.argtypes = [P]
    lib.spec_verify_workspace_reset.restype = None
    lib.spec_verify_chain.argtypes = [P, P, I, I, I, I, F, P, P, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_chain.restype = I
    lib.spec_verify_ngram.argtypes = [P, I, I, I, I, F, P, P, P, P, P, P, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_ngram.restype = I
    lib.spec_verify_tree_greedy.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, P, Z, P]
    lib.spec_verify_tree_greedy.restype = I
    lib.spec_verify_tree_walk.argtypes = [P, P, I, I, I, I, F, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.spec_verify_tree_walk.restype = I
    lib.spec_ngram_draft.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P, P]
    lib.spec_ngram_draft.restype = I
    lib.spec_kv_compact.argtypes = [ctypes.POINTER(c_void_p), I, ctypes.c_longlong, I, I, I, P, P, P, P, P, P]
    lib.spec_kv_compact.restype = I
    lib.spec_verify_chain_static.argtypes = [P, P, I, I, I, I, F, P, P, P, P, P, P, P, P]
    lib.spec_verify_chain_static.restype = I
    lib.spec_status_string.argtypes = [I]
    lib.spec_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _check(status: int) -> None:
    if status != SPEC_OK:
        name = library().spec_status_string(status).decode()
        raise SpecVerifyError(f"{name} ({status})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(device) -> c_void_p:
    return c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name: str, dtype, shape, device) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def workspace_bytes(B: int, rows_per_request: int, V: int, dtype: torch.dtype) -> int:
    """Workspace bytes for B requests reading `rows_per_request` logits rows of V elements each
    (draft-model chain: 2K+1, greedy chain / n-gram: K+1, tree: N+1)."""
    return int(library().spec_verify_workspace_bytes(B, rows_per_request, V, DTYPE_CODE[dtype]))


def make_workspace(B: int, rows_per_request: int, V: int, dtype: torch.dtype, device) -> torch.Tensor:
    """A workspace for such calls (new memory: its first call clears it)."""
    n = max(256, workspace_bytes(B, rows_per_request, V, dtype))
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    workspace_reset(ws)  # the caching allocator may hand out the block of an earlier workspace
    return ws


def workspace_reset(workspace: torch.Tensor) -> None:
    """Tells the library that something other than its calls wrote to `workspace` (see
    spec_verify_workspace_reset): the next call clears it first."""
    library().spec_verify_workspace_reset(ctypes.c_void_p(workspace.data_ptr()))


def _out(given, name, dtype, shape, device):
    if given is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _need(given, name, dtype, shape, device)


def _opt(given, name, dtype, shape, device):
    return None if given is None else _need(given, name, dtype, shape, device)


def _chain_like(ngram: bool, target_logits, draft_logits, draft_tokens, r, u, temperature,
                workspace, out, accept_prob, cand_tokens, pos_mass, target_probs, draft_probs,
                temperatures=None):
    lib = library()
    dev = target_logits.device
    if target_logits.dtype not in DTYPE_CODE or target_logits.dim() != 3:
        raise TypeError("target_logits must be a [B][K+1][V] float32/bfloat16/float16 tensor")
    B, K1, V = target_logits.shape
    K = K1 - 1
    T = float(temperature)
    _need(target_logits, "target_logits", None, (B, K1, V), dev)
    if draft_tokens is None:
        draft_tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, K), dev)
    sampled = T > 0 or temperatures is not None  # per-request temperatures: any request may sample
    if temperatures is not None:
        _need(temperatures, "temperatures", torch.float32, (B,), dev)
    if not ngram and sampled and K > 0:
        _need(draft_logits, "draft_logits", target_logits.dtype, (B, K, V), dev)
    if sampled:
        _need(r, "r", torch.float32, (B, K), dev)
        _need(u, "u", torch.float32, (B,), dev)
    if workspace is None:
        rows = 2 * K + 1 if (not ngram and sampled and K > 0) else K1
        workspace = make_workspace(B, rows, V, target_logits.dtype, dev)
    out = dict(out or {})
    na = _out(out.get("num_accepted"), "num_accepted", torch.int32, (B,), dev)
    ot = _out(out.get("out_tokens"), "out_tokens", torch.int32, (B, K1), dev)
    rm = _out(out.get("residual_mass"), "residual_mass", torch.float32, (B,), dev)
    ef = _out(out.get("err_flags"), "err_flags", torch.int32, (B,), dev)
    ap = _opt(accept_prob, "accept_prob", torch.float32, (B, K), dev)
    ct = _opt(cand_tokens, "cand_tokens", torch.int32, (B, K1), dev)
    pm = _opt(pos_mass, "pos_mass", torch.float32, (B, K1), dev)
    tp = _opt(target_probs, "target_probs", torch.float32, (B, K1, V), dev)
    tail = (_ptr(na), _ptr(ot), _ptr(rm), _ptr(ef), _ptr(ap), _ptr(ct), _ptr(pm), _ptr(tp))
    if ngram:
        st = lib.spec_verify_ngram(_ptr(target_logits), DTYPE_CODE[target_logits.dtype], B, K, V, T,
                                   _ptr(temperatures), _ptr(draft_tokens), _ptr(r), _ptr(u), *tail, _ptr(workspace),
                                   workspace.numel(), _stream(dev))
    else:
        dp = _opt(draft_probs, "draft_probs", torch.float32, (B, K, V), dev)
        st = lib.spec_verify_chain(_ptr(target_logits), _ptr(draft_logits),
                                   DTYPE_CODE[target_logits.dtype], B, K, V, T, _ptr(temperatures),
                                   _ptr(draft_tokens),
                                   _ptr(r), _ptr(u), *tail, _ptr(dp), _ptr(workspace),
                                   workspace.numel(), _stream(dev))
    _check(st)
    return dict(num_accepted=na, out_tokens=ot, residual_mass=rm, err_flags=ef)


def spec_verify_chain(target_logits, draft_logits, draft_tokens, r, u, temperature, *,
                      workspace=None, out=None, accept_prob=None, cand_tokens=None, pos_mass=None,
                      target_probs=None, draft_probs=None, temperatures=None) -> dict:
    """Chain verification with draft logits (draft model / EAGLE head); `temperatures` [B] gives
    each request its own T.  See spec_verify.h."""
    return _chain_like(False, target_logits, draft_logits, draft_tokens, r, u, temperature,
                       workspace, out, accept_prob, cand_tokens, pos_mass, target_probs,
                       draft_probs, temperatures)


def spec_verify_ngram(target_logits, draft_tokens, r, u, temperature, *, workspace=None, out=None,
                      accept_prob=None, cand_tokens=None, pos_mass=None,
                      target_probs=None, temperatures=None) -> dict:
    """Chain verification with a one-hot (prompt n-gram lookup) draft; `temperatures` [B] gives
    each request its own T.  See spec_verify.h."""
    return _chain_like(True, target_logits, None, draft_tokens, r, u, temperature, workspace, out,
                       accept_prob, cand_tokens, pos_mass, target_probs, None, temperatures)


def spec_verify_tree_greedy(target_logits, node_tokens, parents, *, workspace=None, out=None,
                            node_argmax=None) -> dict:
    """Greedy verification of a draft tree.  See spec_verify.h."""
    lib = library()
    dev = target_logits.device
    if target_logits.dtype not in DTYPE_CODE or target_logits.dim() != 3:
        raise TypeError("target_logits must be a [B][N+1][V] float32/bfloat16/float16 tensor")
    B, N1, V = target_logits.shape
    _need(target_logits, "target_logits", None, (B, N1, V), dev)
    _need(node_tokens, "node_tokens", torch.int32, (B, N1), dev)
    _need(parents, "parents", torch.int32, (B, N1), dev)
    if workspace is None:
        workspace = make_workspace(B, N1, V, target_logits.dtype, dev)
    out = dict(out or {})
    al = _out(out.get("accept_len"), "accept_len", torch.int32, (B,), dev)
    pn = _out(out.get("path_nodes"), "path_nodes", torch.int32, (B, N1), dev)
    ot = _out(out.get("out_tokens"), "out_tokens", torch.int32, (B, N1), dev)
    ef = _out(out.get("err_flags"), "err_flags", torch.int32, (B,), dev)
    am = _opt(node_argmax, "node_argmax", torch.int32, (B, N1), dev)
    st = lib.spec_verify_tree_greedy(_ptr(target_logits), DTYPE_CODE[target_logits.dtype], B, N1 - 1,
                                     V, _ptr(node_tokens), _ptr(parents), _ptr(al), _ptr(pn),
                                     _ptr(ot), _ptr(ef), _ptr(am), _ptr(workspace),
                                     workspace.numel(), _stream(dev))
    _check(st)
    return dict(accept_len=al, path_nodes=pn, out_tokens=ot, err_flags=ef)


def spec_verify_tree_walk(target_logits, draft_logits, node_tokens, parents, r, u, temperature, *,
                          out=None, accept_prob=None, temperatures=None) -> dict:
    """Verification of a draft tree by walking it (stochastic for T > 0, greedy for T == 0),
    reading only the visited rows; `temperatures` [B] gives each request its own T.  See
    spec_verify.h."""
    lib = library()
    dev = target_logits.device
    if target_logits.dtype not in DTYPE_CODE or target_logits.dim() != 3:
        raise TypeError("target_logits must be a [B][N+1][V] float32/bfloat16/float16 tensor")
    B, N1, V = target_logits.shape
    T = float(temperature)
    _need(target_logits, "target_logits", None, (B, N1, V), dev)
    _need(node_tokens, "node_tokens", torch.int32, (B, N1), dev)
    _need(parents, "parents", torch.int32, (B, N1), dev)
    if temperatures is not None:
        _need(temperatures, "temperatures", torch.float32, (B,), dev)
    sampled = T > 0 or temperatures is not None
    if sampled:
        _need(draft_logits, "draft_logits", target_logits.dtype, (B, N1, V), dev)
        _need(r, "r", torch.float32, (B, N1), dev)
        _need(u, "u", torch.float32, (B,), dev)
    out = dict(out or {})
    al = _out(out.get("accept_len"), "accept_len", torch.int32, (B,), dev)
    pn = _out(out.get("path_nodes"), "path_nodes", torch.int32, (B, N1), dev)
    ot = _out(out.get("out_tokens"), "out_tokens", torch.int32, (B, N1), dev)
    rm = _out(out.get("residual_mass"), "residual_mass", torch.float32, (B,), dev)
    ef = _out(out.get("err_flags"), "err_flags", torch.int32, (B,), dev)
    ap = _opt(accept_prob, "accept_prob", torch.float32, (B, N1), dev)
    st = lib.spec_verify_tree_walk(_ptr(target_logits), _ptr(draft_logits) if sampled else None,
                                   DTYPE_CODE[target_logits.dtype], B, N1 - 1, V, T, _ptr(temperatures),
                                   _ptr(node_tokens), _ptr(parents), _ptr(r) if sampled else None,
                                   _ptr(u) if sampled else None, _ptr(al), _ptr(pn), _ptr(ot),
                                   _ptr(rm), _ptr(ef), _ptr(ap), _stream(dev))
    _check(st)
    return dict(accept_len=al, path_nodes=pn, out_tokens=ot, residual_mass=rm, err_flags=ef)


def spec_ngram_draft(context, context_len, K: int, *, n_max: int = 4, n_min: int = 1, out=None) -> dict:
    """Prompt n-gram lookup drafts of B contexts [B][Lmax] (int32) with lengths [B].  See
    spec_verify.h."""
    lib = library()
    dev = context.device
    if context.dim() != 2:
        raise ValueError("context must be [B][Lmax]")
    B, Lmax = context.shape
    _need(context, "context", torch.int32, (B, Lmax), dev)
    _need(context_len, "context_len", torch.int32, (B,), dev)
    out = dict(out or {})
    d = _out(out.get("draft_tokens"), "draft_tokens", torch.int32, (B, K), dev)
    dl = _out(out.get("draft_len"), "draft_len", torch.int32, (B,), dev)
    mn = _out(out.get("match_n"), "match_n", torch.int32, (B,), dev)
    me = _out(out.get("match_end"), "match_end", torch.int32, (B,), dev)
    ef = _out(out.get("err_flags"), "err_flags", torch.int32, (B,), dev)
    st = lib.spec_ngram_draft(_ptr(context), _ptr(context_len), B, Lmax, n_max, n_min, K, _ptr(d),
                              _ptr(dl), _ptr(mn), _ptr(me), _ptr(ef), _stream(dev))
    _check(st)
    return dict(draft_tokens=d, draft_len=dl, match_n=mn, match_end=me, err_flags=ef)


def spec_kv_compact(caches, slots, parents, accept_len, path_nodes, *, err_flags=None) -> torch.Tensor:
    """Moves the accepted path's KV rows into the request's first slots, in place, in every cache
    of `caches` (CUDA tensors whose first dimension is the slot).  See spec_verify.h."""
    lib = library()
    caches = list(caches)
    if not caches:
        raise ValueError("no caches")
    dev = caches[0].device
    S = caches[0].shape[0]
    row = caches[0].numel() // max(S, 1) * caches[0].element_size()
    for i, c in enumerate(caches):
        if c.device != dev or c.shape[0] != S or not c.is_contiguous():
            raise ValueError(f"cache {i}: every cache must be contiguous on {dev} with {S} slots")
        if c.numel() // max(S, 1) * c.element_size() != row:
            raise ValueError(f"cache {i}: rows of {row} bytes expected")
    B, N1 = slots.shape
    for name, t, shp in (("slots", slots, (B, N1)), ("parents", parents, (B, N1)), ("accept_len", accept_len, (B,)),
                         ("path_nodes", path_nodes, (B, N1))):
        _need(t, name, torch.int32, shp, dev)
    ef = _out(err_flags, "err_flags", torch.int32, (B,), dev)
    arr = (c_void_p * len(caches))(*[c.data_ptr() for c in caches])
    st = lib.spec_kv_compact(arr, len(caches), S, row, B, N1 - 1, _ptr(slots), _ptr(parents), _ptr(accept_len),
                             _ptr(path_nodes), _ptr(ef), _stream(dev))
    _check(st)
    return ef
