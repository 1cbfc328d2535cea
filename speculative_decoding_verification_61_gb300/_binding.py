"""ctypes marshalling for libspecverify.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(PKG, "_build", "libspecverify.so")

F32, BF16 = 0, 1
MAX_K, MAX_B, MAX_V = 32, 4096, 1 << 24
MAX_TREE_NODES = 64
MAX_SHARDS = 64
NOALLOC_SCRATCH_BYTES = 48 << 20  # spec_verify_noalloc's fixed scratch array
ABI_VERSION = 1
SPEC_ERRORS = {0: "SPEC_OK", -1: "SPEC_ERR_INVALID_ARG", -2: "SPEC_ERR_ALIGNMENT",
               -3: "SPEC_ERR_CUDA", -4: "SPEC_ERR_TIMEOUT", -5: "SPEC_ERR_WORKSPACE"}

# every symbol include/spec_verify.h declares
EXPORTS = ("spec_verify", "spec_verify_ex", "spec_draft_sample", "spec_draft_sample_ex",
           "spec_round_host", "spec_workspace_bytes", "spec_workspace_status",
           "spec_status_string", "spec_abi_version", "spec_last_error", "spec_verify_noalloc",
           "spec_noalloc_bytes", "spec_adapt_state_bytes", "spec_adapt_init", "spec_adapt_update",
           "spec_draft_sample_lse", "spec_verify_lse", "spec_round", "spec_tree_verify",
           "spec_tree_draft_sample", "spec_shard_workspace_bytes", "spec_shard_stats",
           "spec_shard_decide", "spec_shard_draw", "spec_shutdown", "spec_selfcheck_wait_timeout")


class SpecError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {SPEC_ERRORS.get(code, code)}")
        self.code = code


class _Aux(ctypes.Structure):
    _fields_ = [("accept_prob", ctypes.c_void_p), ("residual_mass", ctypes.c_void_p),
                ("lse_target", ctypes.c_void_p), ("lse_draft", ctypes.c_void_p)]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {_LIB_PATH} is missing "
                           "(run __graft_entry__.build() or python -m "
                           "speculative_decoding_verification_61_gb300.build)")
    L = ctypes.CDLL(_LIB_PATH)
    vp, ip, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.spec_verify.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, ip, ip, vp, vp, vp]
    L.spec_verify_ex.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, ip, ip, vp, vp,
                                 ctypes.POINTER(_Aux), vp, sz, vp]
    L.spec_draft_sample.argtypes = [vp, vp, vp, ip, vp, ip, ip, vp, vp]
    L.spec_draft_sample_ex.argtypes = [vp, vp, vp, ip, vp, ip, ip, vp, vp, sz, vp]
    L.spec_round_host.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, ip, ip, vp, vp, vp, vp]
    L.spec_draft_sample_lse.argtypes = [vp, vp, vp, ip, vp, ip, ip, vp, vp, vp, sz, vp]
    L.spec_verify_lse.argtypes = [vp, vp, vp, vp, vp, vp, vp, ip, vp, ip, ip, vp, vp,
                                  ctypes.POINTER(_Aux), vp, sz, vp]
    L.spec_round.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, ip, ip, vp, vp, vp, vp]
    L.spec_tree_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ip, ip, ip, ip, vp, vp, vp, vp]
    L.spec_tree_draft_sample.argtypes = [vp, vp, vp, vp, vp, ip, ip, ip, ip, vp, vp]
    L.spec_shard_workspace_bytes.argtypes = [ip, ip, ip]
    L.spec_shard_workspace_bytes.restype = sz
    L.spec_shard_stats.argtypes = [vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, vp, vp, sz, vp]
    L.spec_shard_decide.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, vp, vp, vp, vp, sz, vp]
    L.spec_shard_draw.argtypes = [vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, vp, vp, sz, vp]
    L.spec_workspace_bytes.argtypes = [ip, ip, ip]
    L.spec_workspace_bytes.restype = sz
    L.spec_noalloc_bytes.argtypes = [ip, ip, ip]
    L.spec_noalloc_bytes.restype = sz
    L.spec_workspace_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int), ip]
    L.spec_status_string.argtypes = [ip]
    L.spec_status_string.restype = ctypes.c_char_p
    L.spec_abi_version.argtypes = []
    L.spec_shutdown.argtypes = []
    L.spec_shutdown.restype = ip
    L.spec_selfcheck_wait_timeout.argtypes = [vp, sz, vp]
    L.spec_selfcheck_wait_timeout.restype = ip
    L.spec_verify_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, ip, ip, vp, vp, vp]
    L.spec_verify_noalloc.restype = ip
    L.spec_last_error.argtypes = []
    L.spec_last_error.restype = ctypes.c_char_p
    L.spec_adapt_state_bytes.argtypes = [ip]
    L.spec_adapt_state_bytes.restype = sz
    L.spec_adapt_init.argtypes = [vp, ip, ip, ip, vp, vp]
    L.spec_adapt_init.restype = ip
    L.spec_adapt_update.argtypes = [vp, vp, ip, ip, ip, vp, vp]
    L.spec_adapt_update.restype = ip
    for name in ("spec_verify", "spec_verify_ex", "spec_draft_sample", "spec_draft_sample_ex",
                 "spec_round_host", "spec_workspace_status", "spec_abi_version",
                 "spec_draft_sample_lse", "spec_verify_lse", "spec_round", "spec_tree_verify",
                 "spec_tree_draft_sample", "spec_shard_stats", "spec_shard_decide", "spec_shard_draw"):
        getattr(L, name).restype = ip
    _lib = L
    return L


def exported_symbols():
    L = lib()
    return {name: hasattr(L, name) for name in EXPORTS}


# ----------------------------------------------------------------- helpers
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_dev(name, t, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _raise(rc, what):
    if rc != 0:
        detail = lib().spec_last_error().decode() if rc == -3 else ""
        raise SpecError(rc, f"{what} [{detail}]" if detail else what)


# ----------------------------------------------------------------- API
def spec_verify(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                temperature, k_offsets, out_tokens=None, out_num_accepted=None,
                aux: bool = False, workspace=None, stream=None):
    """Verify-and-resample (device tensors).  Returns (out_tokens [R_t] int32,
    out_num_accepted [B] int32) and, with aux=True, a dict of accept_prob,
    residual_mass, lse_target, lse_draft (float32)."""
    import torch
    B = temperature.numel()
    V = target_logits.shape[-1]
    dt = _dtype_code(target_logits)
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits)):
        _check_dev(name, t, target_logits.dtype)
    _check_dev("draft_tokens", draft_tokens, torch.int32)
    _check_dev("u_accept", u_accept, torch.float32)
    _check_dev("u_resample", u_resample, torch.float32)
    _check_dev("temperature", temperature, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    if k_offsets.numel() != B + 1:
        raise ValueError("k_offsets must have B + 1 entries")
    R_t = u_resample.numel()
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty(R_t, dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    L = lib()
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_p(workspace), workspace.numel() * workspace.element_size())
    aux_out, ax = _aux_buffers(B, R_t, draft_tokens.numel(), dev) if aux else (None, None)
    if ax is None and workspace is None:
        rc = L.spec_verify(_p(target_logits), _p(draft_logits), _p(draft_tokens), _p(u_accept),
                           _p(u_resample), _p(temperature), B, _p(k_offsets), V, dt,
                           _p(out_tokens), _p(out_num_accepted), _stream(stream))
    else:
        rc = L.spec_verify_ex(_p(target_logits), _p(draft_logits), _p(draft_tokens), _p(u_accept),
                              _p(u_resample), _p(temperature), B, _p(k_offsets), V, dt,
                              _p(out_tokens), _p(out_num_accepted),
                              ctypes.byref(ax) if ax is not None else None, ws_ptr, ws_bytes,
                              _stream(stream))
    _raise(rc, "spec_verify")
    if aux:
        return out_tokens, out_num_accepted, aux_out
    return out_tokens, out_num_accepted


def spec_draft_sample(draft_logits, temperature, u_draft, k_offsets, out_draft_tokens=None,
                      workspace=None, stream=None):
    """Draft-side softmax + multinomial (argmax for T = 0).  Returns int32 [R_d]."""
    import torch
    B = temperature.numel()
    V = draft_logits.shape[-1]
    dt = _dtype_code(draft_logits)
    _check_dev("draft_logits", draft_logits)
    _check_dev("temperature", temperature, torch.float32)
    _check_dev("u_draft", u_draft, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    if out_draft_tokens is None:
        out_draft_tokens = torch.empty(u_draft.numel(), dtype=torch.int32, device=draft_logits.device)
    L = lib()
    if workspace is None:
        rc = L.spec_draft_sample(_p(draft_logits), _p(temperature), _p(u_draft), B, _p(k_offsets), V,
                                 dt, _p(out_draft_tokens), _stream(stream))
    else:
        rc = L.spec_draft_sample_ex(_p(draft_logits), _p(temperature), _p(u_draft), B, _p(k_offsets),
                                    V, dt, _p(out_draft_tokens), _p(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(rc, "spec_draft_sample")
    return out_draft_tokens


def _aux_buffers(B, R_t, R_d, dev):
    import torch
    out = dict(accept_prob=torch.full((R_d,), float("nan"), device=dev),
               residual_mass=torch.full((B,), float("nan"), device=dev),
               lse_target=torch.full((R_t,), float("nan"), device=dev),
               lse_draft=torch.full((R_d,), float("nan"), device=dev))
    ax = _Aux(*(ctypes.c_void_p(out[k].data_ptr()) for k in
                ("accept_prob", "residual_mass", "lse_target", "lse_draft")))
    return out, ax


def spec_draft_sample_lse(draft_logits, temperature, u_draft, k_offsets, out_draft_tokens=None,
                          out_draft_lse2=None, workspace=None, stream=None):
    """Draft sampling that also returns each draft row's log2-domain
    log-sum-exp (float64 [R_d], NaN for greedy/invalid rows), for
    spec_verify_lse.  Returns (draft_tokens int32 [R_d], draft_lse2)."""
    import torch
    B = temperature.numel()
    V = draft_logits.shape[-1]
    dt = _dtype_code(draft_logits)
    _check_dev("draft_logits", draft_logits)
    _check_dev("temperature", temperature, torch.float32)
    _check_dev("u_draft", u_draft, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    R_d = u_draft.numel()
    dev = draft_logits.device
    if out_draft_tokens is None:
        out_draft_tokens = torch.empty(R_d, dtype=torch.int32, device=dev)
    if out_draft_lse2 is None:
        out_draft_lse2 = torch.empty(max(R_d, 1), dtype=torch.float64, device=dev)
    _check_dev("out_draft_lse2", out_draft_lse2, torch.float64)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_p(workspace), workspace.numel() * workspace.element_size())
    rc = lib().spec_draft_sample_lse(_p(draft_logits), _p(temperature), _p(u_draft), B, _p(k_offsets), V, dt,
                                     _p(out_draft_tokens), _p(out_draft_lse2), ws_ptr, ws_bytes, _stream(stream))
    _raise(rc, "spec_draft_sample_lse")
    return out_draft_tokens, out_draft_lse2[:R_d]


def spec_verify_lse(target_logits, draft_logits, draft_lse2, draft_tokens, u_accept, u_resample,
                    temperature, k_offsets, out_tokens=None, out_num_accepted=None, aux: bool = False,
                    workspace=None, stream=None):
    """spec_verify with the draft rows' normalisers given (from
    spec_draft_sample_lse): only the target rows are streamed.  Same
    returns as spec_verify."""
    import torch
    B = temperature.numel()
    V = target_logits.shape[-1]
    dt = _dtype_code(target_logits)
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits)):
        _check_dev(name, t, target_logits.dtype)
    _check_dev("draft_lse2", draft_lse2, torch.float64)
    _check_dev("draft_tokens", draft_tokens, torch.int32)
    _check_dev("u_accept", u_accept, torch.float32)
    _check_dev("u_resample", u_resample, torch.float32)
    _check_dev("temperature", temperature, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    if k_offsets.numel() != B + 1:
        raise ValueError("k_offsets must have B + 1 entries")
    R_t, R_d = u_resample.numel(), draft_tokens.numel()
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty(R_t, dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    aux_out, ax = _aux_buffers(B, R_t, R_d, dev) if aux else (None, None)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_p(workspace), workspace.numel() * workspace.element_size())
    rc = lib().spec_verify_lse(_p(target_logits), _p(draft_logits), _p(draft_lse2), _p(draft_tokens),
                               _p(u_accept), _p(u_resample), _p(temperature), B, _p(k_offsets), V, dt,
                               _p(out_tokens), _p(out_num_accepted),
                               ctypes.byref(ax) if ax is not None else None, ws_ptr, ws_bytes, _stream(stream))
    _raise(rc, "spec_verify_lse")
    if aux:
        return out_tokens, out_num_accepted, aux_out
    return out_tokens, out_num_accepted


def spec_round(target_logits, draft_logits, u_draft, u_accept, u_resample, temperature, k_offsets,
               out_draft_tokens=None, out_tokens=None, out_num_accepted=None, stream=None):
    """One sampling round on device tensors: draft sampling, then verify
    with the draft rows' normalisers kept between the passes (every row
    read once).  Returns (draft_tokens [R_d], out_tokens [R_t],
    out_num_accepted [B])."""
    import torch
    B = temperature.numel()
    V = target_logits.shape[-1]
    dt = _dtype_code(target_logits)
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits)):
        _check_dev(name, t, target_logits.dtype)
    for name, t in (("u_draft", u_draft), ("u_accept", u_accept), ("u_resample", u_resample),
                    ("temperature", temperature)):
        _check_dev(name, t, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    if k_offsets.numel() != B + 1:
        raise ValueError("k_offsets must have B + 1 entries")
    R_t, R_d = u_resample.numel(), u_accept.numel()
    dev = target_logits.device
    if out_draft_tokens is None:
        out_draft_tokens = torch.empty(R_d, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(R_t, dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    rc = lib().spec_round(_p(target_logits), _p(draft_logits), _p(u_draft), _p(u_accept), _p(u_resample),
                          _p(temperature), B, _p(k_offsets), V, dt, _p(out_draft_tokens), _p(out_tokens),
                          _p(out_num_accepted), _stream(stream))
    _raise(rc, "spec_round")
    return out_draft_tokens, out_tokens, out_num_accepted


def spec_tree_verify(target_logits, draft_logits, node_offsets, parent, tokens, u_accept, u_resample,
                     temperature, out_tokens=None, out_num_accepted=None, out_last_node=None,
                     stream=None):
    """Tree (multi-candidate) verify (device tensors, one target and one
    draft row per node).  Returns (out_tokens [N] int32, out_num_accepted [B]
    int32, out_last_node [B] int32)."""
    import torch
    B = temperature.numel()
    N = parent.numel()
    V = target_logits.shape[-1]
    dt = _dtype_code(target_logits)
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits)):
        _check_dev(name, t, target_logits.dtype)
    for name, t in (("node_offsets", node_offsets), ("parent", parent), ("tokens", tokens)):
        _check_dev(name, t, torch.int32)
    for name, t in (("u_accept", u_accept), ("u_resample", u_resample), ("temperature", temperature)):
        _check_dev(name, t, torch.float32)
    if node_offsets.numel() != B + 1:
        raise ValueError("node_offsets must have B + 1 entries")
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty(N, dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if out_last_node is None:
        out_last_node = torch.empty(B, dtype=torch.int32, device=dev)
    rc = lib().spec_tree_verify(_p(target_logits), _p(draft_logits), _p(node_offsets), _p(parent), _p(tokens),
                                _p(u_accept), _p(u_resample), _p(temperature), B, N, V, dt, _p(out_tokens),
                                _p(out_num_accepted), _p(out_last_node), _stream(stream))
    _raise(rc, "spec_tree_verify")
    return out_tokens, out_num_accepted, out_last_node


def spec_tree_draft_sample(draft_logits, node_offsets, parent, temperature, u_draft, out_tokens=None,
                           stream=None):
    """Tree drafting: each non-root node's token from its parent's draft
    row.  Returns int32 [N] (-1 for roots)."""
    import torch
    B = temperature.numel()
    N = parent.numel()
    V = draft_logits.shape[-1]
    dt = _dtype_code(draft_logits)
    _check_dev("draft_logits", draft_logits)
    for name, t in (("node_offsets", node_offsets), ("parent", parent)):
        _check_dev(name, t, torch.int32)
    _check_dev("temperature", temperature, torch.float32)
    _check_dev("u_draft", u_draft, torch.float32)
    if out_tokens is None:
        out_tokens = torch.empty(N, dtype=torch.int32, device=draft_logits.device)
    rc = lib().spec_tree_draft_sample(_p(draft_logits), _p(node_offsets), _p(parent), _p(temperature), _p(u_draft),
                                      B, N, V, dt, _p(out_tokens), _stream(stream))
    _raise(rc, "spec_tree_draft_sample")
    return out_tokens


def spec_round_host(target_logits, draft_logits, u_draft, u_accept, u_resample, temperature,
                    k_offsets, out_draft_tokens=None, out_tokens=None, out_num_accepted=None,
                    stream=None):
    """One sampling round from host (CPU, ideally pinned) tensors: draft
    sampling then verify on the GPU, results copied back to host tensors."""
    import torch
    B = temperature.numel()
    V = target_logits.shape[-1]
    dt = _dtype_code(target_logits)
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits),
                    ("u_draft", u_draft), ("u_accept", u_accept), ("u_resample", u_resample),
                    ("temperature", temperature), ("k_offsets", k_offsets)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    R_d, R_t = u_accept.numel(), u_resample.numel()
    if out_draft_tokens is None:
        out_draft_tokens = torch.empty(R_d, dtype=torch.int32)
    if out_tokens is None:
        out_tokens = torch.empty(R_t, dtype=torch.int32)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32)
    rc = lib().spec_round_host(_p(target_logits), _p(draft_logits), _p(u_draft), _p(u_accept),
                               _p(u_resample), _p(temperature), B, _p(k_offsets), V, dt,
                               _p(out_draft_tokens), _p(out_tokens), _p(out_num_accepted),
                               _stream(stream))
    _raise(rc, "spec_round_host")
    return out_draft_tokens, out_tokens, out_num_accepted


# ------------------------------------------------------- vocab-sharded verify
def _bounds(shard_bounds):
    b = [int(x) for x in shard_bounds]
    return (ctypes.c_int32 * len(b))(*b), len(b) - 1


def _ws_args(workspace):
    _check_dev("workspace", workspace)
    return _p(workspace), workspace.numel() * workspace.element_size()


def shard_workspace_bytes(B: int, Vs: int, dtype: int) -> int:
    """Workspace bytes of one rank's vocab-sharded verify (Vs columns)."""
    return int(lib().spec_shard_workspace_bytes(B, Vs, dtype))


def shard_workspace(B: int, Vs: int, dtype: int, device="cuda"):
    """A zero-filled workspace tensor for spec_shard_* (the caching
    allocator's blocks are 512-byte aligned; the zeros clear the status
    word that workspace_status reads)."""
    import torch
    n = shard_workspace_bytes(B, Vs, dtype)
    if n == 0:
        raise ValueError(f"invalid shard workspace arguments B={B}, Vs={Vs}, dtype={dtype}")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def spec_shard_stats(target_shard, draft_shard, draft_tokens, temperature, k_offsets, shard_bounds, rank,
                     workspace, out_stats=None, stream=None):
    """Step 1 of the vocab-sharded verify on this rank's columns.  Returns
    the row records as int32 [R_t + R_d, 4] (fields m, s, zx as float bits,
    then arg)."""
    import torch
    B = temperature.numel()
    dt = _dtype_code(target_shard)
    for name, t in (("target_shard", target_shard), ("draft_shard", draft_shard)):
        _check_dev(name, t, target_shard.dtype)
    _check_dev("draft_tokens", draft_tokens, torch.int32)
    _check_dev("temperature", temperature, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    rows = target_shard.shape[0] + draft_shard.shape[0]
    if out_stats is None:
        out_stats = torch.empty((rows, 4), dtype=torch.int32, device=target_shard.device)
    bounds, G = _bounds(shard_bounds)
    wp, wb = _ws_args(workspace)
    rc = lib().spec_shard_stats(_p(target_shard), _p(draft_shard), _p(draft_tokens), _p(temperature), B,
                                _p(k_offsets), bounds, G, rank, dt, _p(out_stats), wp, wb, _stream(stream))
    _raise(rc, "spec_shard_stats")
    return out_stats


def spec_shard_decide(target_shard, draft_shard, all_stats, draft_tokens, u_accept, temperature, k_offsets,
                      shard_bounds, rank, workspace, out_tokens=None, out_num_accepted=None, out_mass=None,
                      stream=None):
    """Step 2: the decision from the gathered records (all_stats: the G
    ranks' records, rank-major).  Returns (out_tokens [R_t] int32,
    out_num_accepted [B] int32, out_mass [B, 2] float64)."""
    import torch
    B = temperature.numel()
    dt = _dtype_code(target_shard)
    bounds, G = _bounds(shard_bounds)
    R_t, R_d = target_shard.shape[0], draft_shard.shape[0]
    _check_dev("all_stats", all_stats, torch.int32)
    if all_stats.numel() != G * (R_t + R_d) * 4:
        raise ValueError("all_stats must hold G * (R_t + R_d) records")
    for name, t in (("draft_tokens", draft_tokens), ("k_offsets", k_offsets)):
        _check_dev(name, t, torch.int32)
    for name, t in (("u_accept", u_accept), ("temperature", temperature)):
        _check_dev(name, t, torch.float32)
    dev = target_shard.device
    if out_tokens is None:
        out_tokens = torch.empty(R_t, dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if out_mass is None:
        out_mass = torch.empty((B, 2), dtype=torch.float64, device=dev)
    wp, wb = _ws_args(workspace)
    rc = lib().spec_shard_decide(_p(target_shard), _p(draft_shard), _p(all_stats), _p(draft_tokens), _p(u_accept),
                                 _p(temperature), B, _p(k_offsets), bounds, G, rank, dt, _p(out_tokens),
                                 _p(out_num_accepted), _p(out_mass), wp, wb, _stream(stream))
    _raise(rc, "spec_shard_decide")
    return out_tokens, out_num_accepted, out_mass


def spec_shard_draw(target_shard, draft_shard, all_mass, u_resample, k_offsets, shard_bounds, rank, workspace,
                    out_tokens, stream=None):
    """Step 3: the draw by the rank owning the crossing (all_mass: the G
    ranks' out_mass, rank-major).  Writes the drawn token into out_tokens
    on that rank; returns out_tokens."""
    import torch
    B = k_offsets.numel() - 1
    dt = _dtype_code(target_shard)
    bounds, G = _bounds(shard_bounds)
    _check_dev("all_mass", all_mass, torch.float64)
    if all_mass.numel() != G * B * 2:
        raise ValueError("all_mass must hold G * B * 2 values")
    _check_dev("u_resample", u_resample, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    _check_dev("out_tokens", out_tokens, torch.int32)
    wp, wb = _ws_args(workspace)
    rc = lib().spec_shard_draw(_p(target_shard), _p(draft_shard), _p(all_mass), _p(u_resample), B, _p(k_offsets),
                               bounds, G, rank, dt, _p(out_tokens), wp, wb, _stream(stream))
    _raise(rc, "spec_shard_draw")
    return out_tokens


def selfcheck_wait_timeout(workspace, stream=None):
    """Run the device-side bounded waits until they give up (about 4 s);
    afterwards workspace_status(workspace) is SPEC_ERR_TIMEOUT."""
    wp, wb = _ws_args(workspace)
    _raise(lib().spec_selfcheck_wait_timeout(wp, wb, _stream(stream)), "spec_selfcheck_wait_timeout")


def shutdown():
    """Free the library-owned device buffers (they are allocated again on
    the next call that needs them)."""
    _raise(lib().spec_shutdown(), "spec_shutdown")


def workspace_bytes(B: int, V: int, dtype: int) -> int:
    return int(lib().spec_workspace_bytes(B, V, dtype))


def noalloc_bytes(B: int, V: int, dtype: int) -> int:
    """Scratch a spec_verify_noalloc call uses (refused above NOALLOC_SCRATCH_BYTES)."""
    return int(lib().spec_noalloc_bytes(B, V, dtype))


def workspace_status(workspace=None, clear: bool = False) -> int:
    """Device status word of a workspace tensor (None: the library-owned one)."""
    v = ctypes.c_int(0)
    rc = lib().spec_workspace_status(None if workspace is None else _p(workspace), ctypes.byref(v),
                                     1 if clear else 0)
    _raise(rc, "spec_workspace_status")
    return v.value


def spec_verify_noalloc(target_logits, draft_logits, draft_tokens, u_accept, u_resample,
                        temperature, k_offsets, out_tokens=None, out_num_accepted=None,
                        stream=None):
    """spec_verify without any device allocation inside the call, for callers
    that cannot allocate while they verify (a serving loop that keeps
    allocation off its hot path, a runtime whose memory pool owns the
    device).  Scratch comes from a fixed array in the library (48 MiB);
    larger batches raise SpecError (SPEC_ERR_WORKSPACE).  Calls share that
    array, so keep them ordered on one stream.  Pass out_tokens and
    out_num_accepted to keep this wrapper from allocating them; the inputs
    are checked as spec_verify checks them."""
    import torch
    B = temperature.numel()
    V = target_logits.shape[-1]
    dt = _dtype_code(target_logits)
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits)):
        _check_dev(name, t, target_logits.dtype)
    _check_dev("draft_tokens", draft_tokens, torch.int32)
    _check_dev("u_accept", u_accept, torch.float32)
    _check_dev("u_resample", u_resample, torch.float32)
    _check_dev("temperature", temperature, torch.float32)
    _check_dev("k_offsets", k_offsets, torch.int32)
    if k_offsets.numel() != B + 1:
        raise ValueError("k_offsets must have B + 1 entries")
    R_t = u_resample.numel()
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty(R_t, dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    _check_dev("out_tokens", out_tokens, torch.int32)
    _check_dev("out_num_accepted", out_num_accepted, torch.int32)
    if out_tokens.numel() < R_t or out_num_accepted.numel() < B:
        raise ValueError("out_tokens needs R_t = u_resample.numel() entries and out_num_accepted B")
    rc = lib().spec_verify_noalloc(_p(target_logits), _p(draft_logits), _p(draft_tokens), _p(u_accept),
                                   _p(u_resample), _p(temperature), B, _p(k_offsets), V, dt,
                                   _p(out_tokens), _p(out_num_accepted), _stream(stream))
    _raise(rc, "spec_verify_noalloc")
    return out_tokens, out_num_accepted


class AdaptiveK:
    """Device-side adaptive draft length for a batch of B sequences (the
    spec_adapt_* entry points): holds the state buffer and the next round's
    k_offsets on the device."""

    def __init__(self, B: int, min_k: int = 1, max_k: int = 10, device="cuda", stream=None):
        import torch
        nbytes = int(lib().spec_adapt_state_bytes(B))
        if nbytes == 0:
            raise SpecError(-1, "spec_adapt_state_bytes")
        self.B, self.min_k, self.max_k = B, min_k, max_k
        self.state = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.k_offsets = torch.empty(B + 1, dtype=torch.int32, device=device)
        _raise(lib().spec_adapt_init(_p(self.state), B, min_k, max_k, _p(self.k_offsets), _stream(stream)),
               "spec_adapt_init")

    def update(self, num_accepted, stream=None):
        """Feed one round's out_num_accepted ([B] int32, device); returns the
        next round's k_offsets ([B+1] int32, device, updated in place)."""
        import torch
        _check_dev("num_accepted", num_accepted, torch.int32)
        _raise(lib().spec_adapt_update(_p(self.state), _p(num_accepted), self.B, self.min_k, self.max_k,
                                       _p(self.k_offsets), _stream(stream)), "spec_adapt_update")
        return self.k_offsets
