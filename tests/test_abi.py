"""CPU checks of the C-ABI library: it builds for sm_103a, loads without a
GPU, exports every symbol include/spec_verify.h declares, and rejects bad
arguments on the host (no compute call needs a GPU for these)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_61_gb300 import build
    build.build()
    import speculative_decoding_verification_61_gb300 as sv
    return sv.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", src)))


def test_binding_constants_match_the_header():
    """The binding's limits are the header's #defines (the library checks
    arguments against the latter)."""
    import speculative_decoding_verification_61_gb300 as sv
    src = open(HEADER).read()

    def define(name):
        m = re.search(r"#define\s+" + name + r"\s+(.+?)\s*(/\*|$)", src, flags=re.M)
        assert m, name
        return int(eval(m.group(1).replace("(size_t)", ""), {}))  # integer arithmetic only

    assert define("SPEC_MAX_K") == sv.MAX_K
    assert define("SPEC_MAX_B") == sv.MAX_B
    assert define("SPEC_MAX_V") == sv.MAX_V
    assert define("SPEC_MAX_TREE_NODES") == sv.MAX_TREE_NODES
    assert define("SPEC_MAX_SHARDS") == sv.MAX_SHARDS
    assert define("SPEC_NOALLOC_SCRATCH_BYTES") == sv.NOALLOC_SCRATCH_BYTES
    assert define("SPEC_VERIFY_ABI_VERSION") == sv.ABI_VERSION


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("spec_verify", "spec_verify_ex", "spec_draft_sample", "spec_draft_sample_ex",
              "spec_round_host", "spec_workspace_bytes", "spec_workspace_status",
              "spec_status_string", "spec_abi_version", "spec_draft_sample_lse", "spec_verify_lse",
              "spec_round", "spec_tree_verify", "spec_tree_draft_sample", "spec_shard_workspace_bytes",
              "spec_shard_stats", "spec_shard_decide", "spec_shard_draw", "spec_shutdown",
              "spec_selfcheck_wait_timeout"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in spec_verify.h but not exported"


def test_binding_covers_every_declared_symbol():
    from speculative_decoding_verification_61_gb300 import _binding
    assert set(declared_functions()) <= set(_binding.EXPORTS)


def test_abi_version_and_status_strings(lib):
    assert lib.spec_abi_version() == 1
    assert lib.spec_status_string(0) == b"SPEC_OK"
    assert lib.spec_status_string(-2) == b"SPEC_ERR_ALIGNMENT"
    assert lib.spec_status_string(12345) == b"SPEC_ERR_UNKNOWN"


def test_workspace_bytes_host_only(lib):
    import speculative_decoding_verification_61_gb300 as sv
    a = sv.workspace_bytes(512, 128256, sv.BF16)
    b = sv.workspace_bytes(64, 128256, sv.BF16)
    assert a > b > 0 and a % 256 == 0
    assert sv.noalloc_bytes(512, 128256, sv.BF16) == a   # the same kernels, the same scratch
    assert sv.noalloc_bytes(4, 1001, sv.BF16) == 0
    assert sv.workspace_bytes(4, 1001, sv.BF16) == 0      # V * 2 not a multiple of 16
    assert sv.workspace_bytes(-1, 1000, sv.F32) == 0
    assert sv.workspace_bytes(4, 1000, 7) == 0
    assert sv.workspace_bytes(sv.MAX_B + 1, 1000, sv.F32) == 0


def test_host_argument_errors_launch_nothing(lib):
    """Errors the host can see are returned before any CUDA call."""
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: validation fails first
    # bad dtype
    assert lib.spec_verify(fake, fake, fake, fake, fake, fake, 4, fake, 1000, 9, fake, fake, None) == -1
    # negative B, oversized B
    assert lib.spec_verify(fake, fake, fake, fake, fake, fake, -1, fake, 1000, 0, fake, fake, None) == -1
    assert lib.spec_verify(fake, fake, fake, fake, fake, fake, 5000, fake, 1000, 0, fake, fake, None) == -1
    # V not a multiple of 16 bytes
    assert lib.spec_verify(fake, fake, fake, fake, fake, fake, 4, fake, 1001, 1, fake, fake, None) == -2
    # null pointer
    assert lib.spec_verify(None, fake, fake, fake, fake, fake, 4, fake, 1000, 0, fake, fake, None) == -1
    # misaligned logits pointer
    assert lib.spec_verify(vp((1 << 20) + 4), fake, fake, fake, fake, fake, 4, fake, 1000, 0, fake,
                           fake, None) == -2
    # B == 0 is a no-op
    assert lib.spec_verify(None, None, None, None, None, None, 0, None, 1000, 0, None, None, None) == 0
    assert lib.spec_draft_sample(None, None, None, 0, None, 1000, 0, None, None) == 0
    assert lib.spec_draft_sample(fake, fake, fake, 4, fake, 1000, 3, fake, None) == -1


def test_fused_round_host_argument_errors(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: validation fails first
    # the normaliser arrays of the fused path are required
    assert lib.spec_verify_lse(fake, fake, None, fake, fake, fake, fake, 4, fake, 1000, 0, fake, fake,
                               None, None, 0, None) == -1
    assert lib.spec_draft_sample_lse(fake, fake, fake, 4, fake, 1000, 0, fake, None, None, 0, None) == -1
    # spec_round: null output, bad dtype, V not a multiple of 16 bytes, B == 0 no-op
    assert lib.spec_round(fake, fake, fake, fake, fake, fake, 4, fake, 1000, 0, fake, None, fake, None) == -1
    assert lib.spec_round(fake, fake, fake, fake, fake, fake, 4, fake, 1000, 5, fake, fake, fake, None) == -1
    assert lib.spec_round(fake, fake, fake, fake, fake, fake, 4, fake, 1001, 1, fake, fake, fake, None) == -2
    assert lib.spec_round(None, None, None, None, None, None, 0, None, 1000, 0, None, None, None, None) == 0


def test_round_host_argument_errors(lib):
    """spec_round_host reads k_offsets on the host to size its copies: a bad
    array, a null pointer or a bad dtype is refused before any CUDA call."""
    import numpy as np
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: validation fails first

    def call(ko, B=3, V=1000, dtype=0, first=fake):
        k = np.ascontiguousarray(ko, dtype=np.int32)
        return lib.spec_round_host(first, fake, fake, fake, fake, fake, B, k.ctypes.data_as(vp), V, dtype,
                                   fake, fake, fake, None)
    assert call([1, 2, 3, 4]) == -1        # k_offsets[0] != 0
    assert call([0, 2, 1, 4]) == -1        # a negative k_b
    assert call([0, 2, 40, 41]) == -1      # k_b = 38 > MAX_K
    assert call([0, 1, 2, 3], first=None) == -1
    assert call([0, 1, 2, 3], dtype=7) == -1
    assert call([0, 1, 2, 3], V=1001, dtype=1) == -2
    assert lib.spec_round_host(None, None, None, None, None, None, 0, None, 1000, 0, None, None, None, None) == 0


def test_tree_host_argument_errors(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: validation fails first
    # N outside [B, 64 B], null pointer, bad dtype; B == 0 is a no-op
    assert lib.spec_tree_verify(fake, fake, fake, fake, fake, fake, fake, fake, 4, 3, 1000, 0, fake, fake,
                                None, None) == -1
    assert lib.spec_tree_verify(fake, fake, fake, fake, fake, fake, fake, fake, 4, 257, 1000, 0, fake, fake,
                                None, None) == -1
    assert lib.spec_tree_verify(fake, fake, None, fake, fake, fake, fake, fake, 4, 8, 1000, 0, fake, fake,
                                None, None) == -1
    assert lib.spec_tree_verify(fake, fake, fake, fake, fake, fake, fake, fake, 4, 8, 1000, 7, fake, fake,
                                None, None) == -1
    assert lib.spec_tree_verify(None, None, None, None, None, None, None, None, 0, 0, 1000, 0, None, None,
                                None, None) == 0
    assert lib.spec_tree_draft_sample(fake, fake, fake, fake, fake, 4, 3, 1000, 0, fake, None) == -1
    assert lib.spec_tree_draft_sample(fake, fake, fake, fake, fake, 4, 8, 1001, 1, fake, None) == -2


def test_shard_host_argument_errors(lib):
    """The vocab-sharded calls check bounds, G, rank, widths and the
    workspace on the host before touching the device."""
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: validation fails first

    def bounds(*b):
        return (ctypes.c_int32 * len(b))(*b)

    ws_need = lib.spec_shard_workspace_bytes(4, 504, 1)
    assert ws_need > 0 and ws_need % 256 == 0
    assert lib.spec_shard_workspace_bytes(4, 501, 1) == 0   # bf16 width not a multiple of 8
    assert lib.spec_shard_workspace_bytes(4, 0, 1) == 0
    ok = bounds(0, 496, 1000)
    ws = vp(1 << 24)  # 256-byte aligned, never dereferenced here

    def stats(b, G, rank, dtype=1, ws_ptr=ws, ws_bytes=1 << 30, first=fake):
        return lib.spec_shard_stats(first, fake, fake, fake, 4, fake, b, G, rank, dtype, fake, ws_ptr, ws_bytes,
                                    None)

    assert stats(None, 2, 0) == -1                      # no bounds
    assert stats(ok, 0, 0) == -1 and stats(ok, 65, 0) == -1   # G outside [1, 64]
    assert stats(ok, 2, 2) == -1 and stats(ok, 2, -1) == -1   # rank outside [0, G)
    assert stats(bounds(8, 496, 1000), 2, 0) == -1      # must start at 0
    assert stats(bounds(0, 496, 496), 2, 0) == -1       # an empty shard
    assert stats(bounds(0, 500, 1000), 2, 0) == -2      # width 500: not a multiple of 8 (bf16)
    assert stats(bounds(0, 500, 1000), 2, 0, dtype=0) != -2   # ... but of 4 (fp32): passes that check
    assert stats(ok, 2, 0, dtype=3) == -1               # bad dtype
    assert stats(ok, 2, 0, ws_ptr=None) == -1           # the workspace is required
    assert stats(ok, 2, 0, ws_bytes=16) == -5           # too small
    assert stats(ok, 2, 0, ws_ptr=vp((1 << 24) + 16)) == -2   # not 256-byte aligned
    assert stats(ok, 2, 0, first=None) == -1            # a null logit pointer
    assert stats(ok, 2, 0, first=vp((1 << 20) + 4)) == -2     # unaligned logits
    assert lib.spec_shard_decide(fake, fake, None, fake, fake, fake, 4, fake, ok, 2, 0, 1, fake, fake, fake, ws,
                                 1 << 30, None) == -1   # no gathered records
    assert lib.spec_shard_draw(fake, fake, None, fake, 4, fake, ok, 2, 1, 1, fake, ws, 1 << 30, None) == -1
    assert lib.spec_shard_draw(fake, fake, fake, fake, 4, fake, ok, 2, 1, 1, fake, ws, 16, None) == -5
    # B = 0 is a no-op that still checks the shard arguments
    assert lib.spec_shard_draw(None, None, None, None, 0, None, ok, 2, 1, 1, None, None, 0, None) == 0
    assert lib.spec_shard_draw(None, None, None, None, 0, None, ok, 2, 2, 1, None, None, 0, None) == -1


def test_selfcheck_host_argument_errors(lib):
    vp = ctypes.c_void_p
    assert lib.spec_selfcheck_wait_timeout(None, 256, None) == -1
    assert lib.spec_selfcheck_wait_timeout(vp(1 << 20), 64, None) == -5
    assert lib.spec_selfcheck_wait_timeout(vp((1 << 20) + 4), 256, None) == -2


def test_noalloc_wrapper_refuses_host_tensors(lib):
    """The allocation-free wrapper checks its tensors before it hands any
    pointer to the library: host (CPU) tensors are refused on the host."""
    torch = pytest.importorskip("torch")
    import speculative_decoding_verification_61_gb300 as sv
    B, V, R_d = 2, 64, 4
    z = torch.zeros((R_d + B, V), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sv.spec_verify_noalloc(z, z[:R_d], torch.zeros(R_d, dtype=torch.int32), torch.zeros(R_d),
                               torch.zeros(R_d + B), torch.ones(B), torch.tensor([0, 2, 4], dtype=torch.int32))
