"""The C-ABI library builds, loads without a GPU, and exports every function
include/dflash.h declares; the binding wraps each of them.  No compute calls."""
import ctypes
import os
import re

import pytest

from block_diffusion_speculative_kv_gb300 import binding, build

HEADER = os.path.join(build.ROOT, "include", "dflash.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keep = [n for n in names if n.startswith(("dflash_", "ddtree_"))]
    return sorted(set(keep))


@pytest.fixture(scope="module")
def libpath():
    return build.build()


def test_header_declares_the_path_calls():
    d = _declared()
    for name in ("dflash_inject_kv", "dflash_draft_block", "ddtree_build", "ddtree_accept",
                 "dflash_logits_topk", "dflash_model_create", "dflash_workspace_bytes"):
        assert name in d


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(libpath):
    assert sorted(binding.exported_symbols()) == _declared()
    lib = binding.lib()
    assert lib.dflash_abi_version() == 2


def test_host_validation_needs_no_gpu(libpath):
    lib = binding.lib()
    # invalid budget and depth are rejected before anything touches the device
    assert lib.ddtree_build(1, 0, 8, 64, *([None] * 9), None) == 1
    assert lib.ddtree_build(1, 8, 8, 2000, *([None] * 9), None) == 1
    assert lib.ddtree_build(1, 8, 1025, 64, *([None] * 9), None) == 1
    assert b"K" in lib.dflash_last_error()
    assert lib.dflash_logits_topk(4, 100, 50, 1, None, 8, None, None, None, 0, None) == 1
    assert lib.dflash_topk_workspace_bytes(4, 100, 0) == 0
    assert lib.dflash_topk_workspace_bytes(4, 100000, 1025) == 0
    assert lib.dflash_topk_workspace_bytes(4, 100000, 1024) > 4 * 1024 * 8
    assert lib.dflash_logits_topk(4, 2000, 2000, 0, None, 1025, None, None, None, 0, None) == 1
    # sampling draws at most 32 tokens
    s1 = ctypes.byref(binding.Sampling(1.0, 1, 0))
    assert lib.dflash_logits_sample(4, 2000, 2000, 0, None, s1, 64, None, None, None, 0,
                                    None) == 2
    # zero-sized requests are valid no-ops
    assert lib.ddtree_build(0, 8, 8, 64, *([None] * 9), None) == 0
    assert lib.dflash_chain_tree(1, 0, 1, 64, *([None] * 8), None) == 1
    assert lib.dflash_chain_tree(0, 4, 1, 64, *([None] * 8), None) == 0
    # a negative or huge temperature is rejected on the host; 0 is the top-K
    for t in (-1.0, 1e-9, 1e9, float("nan")):
        s = ctypes.byref(binding.Sampling(t, 1, 0))
        assert lib.dflash_logits_sample(0, 100, 100, 0, None, s, 1, None, None, None, 0,
                                        None) == 1, t
    s = ctypes.byref(binding.Sampling(0.0, 1, 0))
    assert lib.dflash_logits_sample(0, 100, 100, 0, None, s, 1, None, None, None, 0, None) == 0


def test_sampling_struct_layout_matches_the_header():
    # typedef struct { float temperature; uint64_t seed; int64_t row_offset; }
    S = binding.Sampling
    assert ctypes.sizeof(S) == 24
    assert S.temperature.offset == 0 and S.seed.offset == 8 and S.row_offset.offset == 16
    assert binding.sampling_arg(None) is None
    a = binding.sampling_arg((0.5, -1, 7))._obj
    assert a.temperature == 0.5 and a.seed == 2 ** 64 - 1 and a.row_offset == 7


def test_commit_host_validation_needs_no_gpu(libpath):
    lib = binding.lib()
    f = lib.dflash_commit_accepted
    # depth, budget, dtype and feature-row size are checked before any launch
    assert f(1, 0, 8, 64, 1, None, 64, *([None] * 8), None) == 1          # D = 0
    assert f(1, 4, 2000, 64, 1, None, 64, *([None] * 8), None) == 1       # B > 1024
    assert f(1, 4, 8, 63, 1, None, 64, *([None] * 8), None) == 1          # 126-byte rows
    assert f(1, 4, 8, 64, 7, None, 64, *([None] * 8), None) == 1          # bad dtype
    assert f(1, 4, 8, 64, 1, None, 32, *([None] * 8), None) == 1          # tree_ld < feat_dim
    assert f(1, 4, 8, 64, 1, None, 64, *([None] * 8), None) == 1          # null pointers
    assert f(0, 4, 8, 64, 1, None, 64, *([None] * 8), None) == 0          # nothing to do


def test_verify_and_linear_host_validation_needs_no_gpu(libpath):
    lib = binding.lib()
    N = None
    ws = lib.dflash_tree_attention_workspace_bytes
    assert ws(1, 32, 8, 128, 256, 8192) > 0
    assert ws(1, 32, 8, 64, 256, 8192) == 0          # head_dim 128 only
    assert ws(1, 30, 8, 128, 256, 8192) == 0         # n_q not a multiple of n_kv
    ta = lib.dflash_tree_attention
    p = ctypes.c_void_p(16)                          # never dereferenced: rejected first
    args = lambda n_q, n_kv, hd, B, max_ctx, cap, ld: (
        1, n_q, n_kv, hd, B, p, max_ctx, cap, p, p, p, ld, p, p, ld, p, p, p, ld, N, 0, N)
    assert ta(*args(32, 8, 64, 256, 100, 100, 4096)) == 1     # head_dim
    assert ta(*args(40, 8, 128, 256, 100, 100, 5120)) == 1    # 5 query heads per KV head
    assert ta(*args(32, 8, 128, 2000, 100, 100, 4096)) == 1   # B > 1024
    assert ta(*args(32, 8, 128, 256, 200, 100, 4096)) == 1    # max_ctx > cap
    assert ta(*args(32, 8, 128, 256, 100, 100, 4000)) == 1    # strides
    assert ta(*args(32, 8, 128, 256, 100, 100, 4096)) == 3    # workspace missing
    tr = lib.dflash_tree_rope
    assert tr(1, 8, 2, 127, 1e6, p, p, p, 256, 1, N) == 1     # odd head_dim
    assert tr(1, 8, 2, 128, 0.0, p, p, p, 256, 1, N) == 1     # theta
    assert tr(1, 8, 2, 128, 1e6, p, p, p, 200, 1, N) == 1     # row stride
    assert lib.dflash_linear_workspace_bytes(16, 100, 64) == 0
    assert lib.dflash_linear_bf16(16, 100, 64, p, p, p, N, 0, N) == 1
    assert lib.dflash_linear_bf16(0, 128, 64, N, N, N, N, 0, N) == 0
    assert lib.dflash_workspace_bytes(N, 1, 16, 16, 8) == 0

