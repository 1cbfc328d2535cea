"""fp64 CPU oracle for the speculative-decoding verify step (ctypes wrapper).

TEST INFRASTRUCTURE.  Only `tests/`, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library and its binding) never imports or calls it.

The arithmetic lives in spec_oracle.c; this module only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
_lib = None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bind(lib):
    vp, ip = ctypes.c_void_p, ctypes.c_int
    lib.oracle_verify.restype = ip
    lib.oracle_verify.argtypes = [vp, vp, ip, vp, vp, vp, vp, ip, vp, ip, vp, vp,
                                  vp, vp, vp, vp, vp, vp, ip, ip]
    lib.oracle_draft_sample.restype = ip
    lib.oracle_draft_sample.argtypes = [vp, ip, vp, vp, ip, vp, ip, vp, vp, vp, ip]
    lib.oracle_tree_verify.restype = ip
    lib.oracle_tree_verify.argtypes = [vp, vp, ip, vp, vp, vp, vp, vp, vp, ip, ip, vp, vp, vp, vp, ip]
    lib.oracle_tree_draft_sample.restype = ip
    lib.oracle_tree_draft_sample.argtypes = [vp, ip, vp, vp, vp, vp, ip, ip, vp, vp, ip]
    lib.oracle_softmax_row.restype = ip
    lib.oracle_softmax_row.argtypes = [vp, ip, ip, ctypes.c_double, vp, vp]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  A custom path
    loads another build of the same source (the mutation tests use this)."""
    global _lib
    if path is None:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(_build.build()))
        return _lib
    return _bind(ctypes.CDLL(path))


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {arr.dtype}")


class VerifyResult(dict):
    __getattr__ = dict.__getitem__


def verify(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
           temperature, k_offsets, seq_list=None, nthreads: int = 1, lib=None):
    """Run the oracle verify step.  Logits: float32 or uint16 bf16 bits,
    [R_t, V] and [R_d, V].  Returns tokens [R_t], num_accepted [B] and the aux
    arrays accept_prob [R_d], residual_mass [B], lse_target [R_t],
    lse_draft [R_d], margin [B]."""
    lib = lib or load()
    tl = np.ascontiguousarray(target_logits)
    dl = np.ascontiguousarray(draft_logits)
    dt = _dtype_code(tl)
    assert _dtype_code(dl) == dt if dl.size else True
    k_offsets = _c(k_offsets, np.int32)
    B = len(k_offsets) - 1
    V = tl.shape[-1]
    R_d = int(k_offsets[-1]) if B > 0 else 0
    R_t = R_d + B
    out_tokens = np.full(R_t, -7, dtype=np.int32)
    out_num = np.full(B, -7, dtype=np.int32)
    accept_prob = np.full(R_d, np.nan)
    residual_mass = np.full(B, np.nan)
    lse_t = np.full(R_t, np.nan)
    lse_d = np.full(R_d, np.nan)
    margin = np.full(B, np.inf)
    sl = None if seq_list is None else _c(seq_list, np.int32)
    toks = _c(draft_tokens, np.int32)
    ua, ur, tp = _c(u_accept, np.float32), _c(u_resample, np.float32), _c(temperature, np.float32)
    rc = lib.oracle_verify(_ptr(tl), _ptr(dl), dt, _ptr(toks), _ptr(ua), _ptr(ur), _ptr(tp),
                           B, _ptr(k_offsets), V, _ptr(out_tokens), _ptr(out_num),
                           _ptr(accept_prob), _ptr(residual_mass), _ptr(lse_t), _ptr(lse_d),
                           _ptr(margin), _ptr(sl), 0 if sl is None else len(sl), nthreads)
    return VerifyResult(rc=rc, tokens=out_tokens, num_accepted=out_num,
                        accept_prob=accept_prob, residual_mass=residual_mass,
                        lse_target=lse_t, lse_draft=lse_d, margin=margin)


def draft_sample(draft_logits, temperature, u_draft, k_offsets, nthreads: int = 1, lib=None):
    """Oracle draft-side sampling: argmax for T=0 rows, inverse CDF of
    softmax(z/T) at u_draft otherwise.  Returns tokens [R_d], margin [R_d],
    lse [R_d]."""
    lib = lib or load()
    dl = np.ascontiguousarray(draft_logits)
    dt = _dtype_code(dl)
    k_offsets = _c(k_offsets, np.int32)
    B = len(k_offsets) - 1
    V = dl.shape[-1]
    R = int(k_offsets[-1]) if B > 0 else 0
    out = np.full(R, -7, dtype=np.int32)
    margin = np.full(R, np.inf)
    lse = np.full(R, np.nan)
    tp, ud = _c(temperature, np.float32), _c(u_draft, np.float32)
    rc = lib.oracle_draft_sample(_ptr(dl), dt, _ptr(tp), _ptr(ud), B, _ptr(k_offsets), V,
                                 _ptr(out), _ptr(margin), _ptr(lse), nthreads)
    return VerifyResult(rc=rc, tokens=out, margin=margin, lse=lse)


def tree_verify(target_logits, draft_logits, node_offsets, parent, tokens, u_accept, u_resample,
                temperature, nthreads: int = 1, lib=None):
    """Oracle tree (multi-candidate) verify.  Logits [N, V] (float32 or uint16
    bf16 bits), one target and one draft row per node.  Returns tokens [N],
    num_accepted [B], last_node [B], margin [B]."""
    lib = lib or load()
    tl = np.ascontiguousarray(target_logits)
    dl = np.ascontiguousarray(draft_logits)
    dt = _dtype_code(tl)
    no = _c(node_offsets, np.int32)
    B = len(no) - 1
    V = tl.shape[-1]
    N = int(no[-1]) if B > 0 else 0
    out_tokens = np.full(N, -7, dtype=np.int32)
    out_num = np.full(B, -7, dtype=np.int32)
    out_last = np.full(B, -7, dtype=np.int32)
    margin = np.full(B, np.inf)
    pa, tk = _c(parent, np.int32), _c(tokens, np.int32)
    ua, ur, tp = _c(u_accept, np.float32), _c(u_resample, np.float32), _c(temperature, np.float32)
    rc = lib.oracle_tree_verify(_ptr(tl), _ptr(dl), dt, _ptr(no), _ptr(pa), _ptr(tk), _ptr(ua), _ptr(ur),
                                _ptr(tp), B, V, _ptr(out_tokens), _ptr(out_num), _ptr(out_last),
                                _ptr(margin), nthreads)
    return VerifyResult(rc=rc, tokens=out_tokens, num_accepted=out_num, last_node=out_last,
                        margin=margin)


def tree_draft_sample(draft_logits, node_offsets, parent, temperature, u_draft, nthreads: int = 1,
                      lib=None):
    """Oracle tree drafting: each non-root node's token from its parent's
    draft row.  Returns tokens [N] (-1 for roots) and margin [N]."""
    lib = lib or load()
    dl = np.ascontiguousarray(draft_logits)
    dt = _dtype_code(dl)
    no = _c(node_offsets, np.int32)
    B = len(no) - 1
    V = dl.shape[-1]
    N = int(no[-1]) if B > 0 else 0
    out = np.full(N, -7, dtype=np.int32)
    margin = np.full(N, np.inf)
    pa = _c(parent, np.int32)
    tp, ud = _c(temperature, np.float32), _c(u_draft, np.float32)
    rc = lib.oracle_tree_draft_sample(_ptr(dl), dt, _ptr(no), _ptr(pa), _ptr(tp), _ptr(ud), B, V,
                                      _ptr(out), _ptr(margin), nthreads)
    return VerifyResult(rc=rc, tokens=out, margin=margin)


def softmax_row(logits_row, T: float, lib=None):
    """(p, lse) of one row of logits at temperature T; None if invalid."""
    lib = lib or load()
    z = np.ascontiguousarray(logits_row)
    dt = _dtype_code(z)
    V = z.shape[-1]
    p = np.zeros(V)
    lse = np.zeros(1)
    rc = lib.oracle_softmax_row(_ptr(z), dt, V, float(T), _ptr(p), _ptr(lse))
    return None if rc != 0 else (p, float(lse[0]))


def cores() -> int:
    return os.cpu_count() or 1
