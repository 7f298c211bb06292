"""Thin ctypes binding of libdflash.so (include/dflash.h).

Argument marshalling only: every function passes PyTorch CUDA tensors' device
pointers and sizes to the C ABI call of the same name, on the current CUDA
stream.  There is no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdflash.so")

DFLASH_OK = 0
DFLASH_F32, DFLASH_BF16 = 0, 1
MAX_LAYERS = 16

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA",
                5: "TIMEOUT"}


class DflashError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


# ---------------------------------------------------------------------------
# Structs mirroring include/dflash.h
# ---------------------------------------------------------------------------

class Dims(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d", C.c_int), ("n_q", C.c_int), ("n_kv", C.c_int),
                ("head_dim", C.c_int), ("d_ff", C.c_int), ("vocab", C.c_int),
                ("n_feat", C.c_int), ("d_feat", C.c_int), ("dtype", C.c_int),
                ("rope_theta", C.c_float), ("rms_eps", C.c_float), ("mask_id", C.c_int),
                ("anchor_sees_block", C.c_int)]


class Weights(C.Structure):
    _fields_ = [("w_proj", C.c_void_p), ("embed", C.c_void_p), ("lm_head", C.c_void_p),
                ("final_norm", C.c_void_p), ("u_kv", C.c_void_p),
                ("attn_norm", C.c_void_p * MAX_LAYERS), ("w_qkv", C.c_void_p * MAX_LAYERS),
                ("wo", C.c_void_p * MAX_LAYERS), ("mlp_norm", C.c_void_p * MAX_LAYERS),
                ("w_gate_up", C.c_void_p * MAX_LAYERS), ("w_down", C.c_void_p * MAX_LAYERS)]


class Cache(C.Structure):
    _fields_ = [("k", C.c_void_p * MAX_LAYERS), ("v", C.c_void_p * MAX_LAYERS),
                ("n_req", C.c_int), ("cap", C.c_int)]


class Sampling(C.Structure):
    """Temperature sampling of a top-K pass (temperature 0: plain top-K)."""
    _fields_ = [("temperature", C.c_float), ("seed", C.c_uint64), ("row_offset", C.c_int64)]


def sampling_arg(sampling):
    """None, or (temperature, seed[, row_offset]) -> a Sampling pointer argument."""
    if sampling is None:
        return None
    t, seed, *rest = sampling
    return C.byref(Sampling(float(t), int(seed) & (2 ** 64 - 1), int(rest[0]) if rest else 0))


_lib = None

_vp, _i, _sz = C.c_void_p, C.c_int, C.c_size_t
_SIGS = {
    "dflash_last_error": (C.c_char_p, []),
    "dflash_abi_version": (_i, []),
    "dflash_model_create": (_i, [C.POINTER(Dims), C.POINTER(Weights), C.POINTER(_vp)]),
    "dflash_model_destroy": (None, [_vp]),
    "dflash_workspace_bytes": (_sz, [_vp, _i, _i, _i, _i]),
    "dflash_workspace_init": (_i, [_vp, _sz, _vp]),
    "dflash_read_status": (_i, [_vp, C.POINTER(_i), _vp]),
    "dflash_workspace_set_wait_limit": (_i, [_vp, _sz, C.c_uint64, _vp]),
    "dflash_inject_kv": (_i, [_vp, C.POINTER(Cache), _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dflash_draft_block": (_i, [_vp, C.POINTER(Cache), _i, _vp, _vp, _i, _i, _i,
                                C.POINTER(Sampling), _vp, _vp, _vp, _vp, _sz, _vp]),
    "dflash_draft_cycle": (_i, [_vp, C.POINTER(Cache), _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _i,
                                _i, C.POINTER(Sampling), _vp, _vp, _vp, _vp, _sz, _vp]),
    "dflash_tree_attention_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "dflash_tree_attention": (_i, [_i, _i, _i, _i, _i, _vp, _i, _i, _vp, _vp, _vp, C.c_longlong,
                                   _vp, _vp, C.c_longlong, _vp, _vp, _vp, C.c_longlong, _vp,
                                   _sz, _vp]),
    "dflash_tree_rope": (_i, [_i, _i, _i, _i, C.c_float, _vp, _vp, _vp, C.c_longlong, _i,
                              _vp]),
    "dflash_topk_workspace_bytes": (_sz, [_i, _i, _i]),
    "dflash_logits_topk": (_i, [_i, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
    "dflash_logits_sample": (_i, [_i, _i, _i, _i, _vp, C.POINTER(Sampling), _i, _vp, _vp, _vp,
                                  _sz, _vp]),
    "dflash_chain_tree": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ddtree_build": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ddtree_accept": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "dflash_commit_accepted": (_i, [_i, _i, _i, _i, _i, _vp, C.c_longlong, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _vp]),
    "dflash_linear_workspace_bytes": (_sz, [_i, _i, _i]),
    "dflash_linear_bf16": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dflash_set_trace_hook": (None, [_vp, _vp]),
    "dflash_logits_topk_noalloc": (_i, [_i, _i, _i, _i, _vp, _i, _vp, _vp, _vp]),
}

TRACE_FN = C.CFUNCTYPE(None, C.c_void_p, C.c_char_p, C.c_int, C.c_void_p)


def lib():
    """Load libdflash.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
        l = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def set_trace_hook(fn) -> None:
    """Install fn(name: str, phase: int, stream_ptr: int) around every kernel
    launch (None removes it).  Keeps a reference to the ctypes thunk."""
    global _trace_thunk
    if fn is None:
        lib().dflash_set_trace_hook(None, None)
        _trace_thunk = None
        return

    def _cb(user, name, phase, stream):
        fn(name.decode(), phase, stream or 0)

    _trace_thunk = TRACE_FN(_cb)
    lib().dflash_set_trace_hook(C.cast(_trace_thunk, C.c_void_p), None)


_trace_thunk = None


def exported_symbols() -> List[str]:
    return list(_SIGS)


def _check(status: int):
    if status != DFLASH_OK:
        raise DflashError(status, lib().dflash_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DFLASH_F32
    if t.dtype == torch.bfloat16:
        return DFLASH_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


# ---------------------------------------------------------------------------
# Workspace and status
# ---------------------------------------------------------------------------

def workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().dflash_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def workspace_set_wait_limit(ws: torch.Tensor, limit_ns: int, stream=None):
    _check(lib().dflash_workspace_set_wait_limit(_ptr(ws), ws.numel() * ws.element_size(),
                                                 int(limit_ns), _stream(stream)))


def read_status(ws: torch.Tensor, stream=None) -> int:
    out = C.c_int(0)
    _check(lib().dflash_read_status(_ptr(ws), C.byref(out), _stream(stream)))
    return out.value


# ---------------------------------------------------------------------------
# Step a6 standalone
# ---------------------------------------------------------------------------

def topk_workspace_bytes(rows: int, vocab: int, K: int) -> int:
    return int(lib().dflash_topk_workspace_bytes(rows, vocab, K))


def logits_topk(logits: torch.Tensor, K: int, ids: torch.Tensor, logp: torch.Tensor,
                ws: torch.Tensor, vocab: Optional[int] = None, stream=None):
    rows, ld = logits.shape
    vocab = ld if vocab is None else vocab
    _check(lib().dflash_logits_topk(rows, vocab, ld, _dtype_code(logits), _ptr(logits), K,
                                    _ptr(ids), _ptr(logp), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)))


def logits_sample(logits: torch.Tensor, sampling, K: int, ids: torch.Tensor,
                  logq: torch.Tensor, ws: torch.Tensor, vocab: Optional[int] = None, stream=None):
    """Gumbel-max draw of K tokens per row at sampling = (temperature, seed[,
    row_offset]); ids[:, 0] is a sample from softmax(logits / temperature)."""
    rows, ld = logits.shape
    vocab = ld if vocab is None else vocab
    _check(lib().dflash_logits_sample(rows, vocab, ld, _dtype_code(logits), _ptr(logits),
                                      sampling_arg(sampling), K, _ptr(ids), _ptr(logq), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)))


def logits_topk_noalloc(logits: torch.Tensor, K: int, ids: torch.Tensor, logp: torch.Tensor,
                        vocab: Optional[int] = None, stream=None):
    """Step a6 without a workspace, for callers that cannot allocate device
    memory at this point (the library keeps a fixed scratch array per device)."""
    rows, ld = logits.shape
    vocab = ld if vocab is None else vocab
    _check(lib().dflash_logits_topk_noalloc(rows, vocab, ld, _dtype_code(logits), _ptr(logits),
                                            K, _ptr(ids), _ptr(logp), _stream(stream)))


# ---------------------------------------------------------------------------
# The dense contraction on its own
# ---------------------------------------------------------------------------

def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().dflash_linear_workspace_bytes(M, N, K))


def linear_bf16(X: torch.Tensor, W: torch.Tensor, Y: torch.Tensor, ws: torch.Tensor, stream=None):
    """Y = X . W^T (bf16 in, fp32 out) on the tensor cores."""
    M, K = X.shape
    N = W.shape[0]
    _check(lib().dflash_linear_bf16(M, N, K, _ptr(X), _ptr(W), _ptr(Y), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)))


# ---------------------------------------------------------------------------
# Steps a7, a8
# ---------------------------------------------------------------------------

def ddtree_build(topk_logp: torch.Tensor, topk_ids: torch.Tensor, root_tok: torch.Tensor, B: int,
                 n_nodes, tok, parent, depth, rank, mask, stream=None):
    n_req, D, K = topk_logp.shape
    _check(lib().ddtree_build(n_req, D, K, B, _ptr(topk_logp), _ptr(topk_ids), _ptr(root_tok),
                              _ptr(n_nodes), _ptr(tok), _ptr(parent), _ptr(depth), _ptr(rank),
                              _ptr(mask), _stream(stream)))


def chain_tree(topk_ids: torch.Tensor, root_tok: torch.Tensor, B: int, n_nodes, tok, parent,
               depth, rank, mask, stream=None):
    """The vanilla DFlash chain of topk_ids[:, :, 0] in ddtree_build's layout."""
    n_req, D, K = topk_ids.shape
    _check(lib().dflash_chain_tree(n_req, D, K, B, _ptr(topk_ids), _ptr(root_tok), _ptr(n_nodes),
                                   _ptr(tok), _ptr(parent), _ptr(depth), _ptr(rank), _ptr(mask),
                                   _stream(stream)))


def ddtree_accept(D: int, B: int, n_nodes, tok, parent, target_tok, accept_len, accepted, bonus,
                  stream=None):
    n_req = n_nodes.shape[0]
    _check(lib().ddtree_accept(n_req, D, B, _ptr(n_nodes), _ptr(tok), _ptr(parent),
                               _ptr(target_tok), _ptr(accept_len), _ptr(accepted), _ptr(bonus),
                               _stream(stream)))


def commit_accepted(D: int, tree_feats: torch.Tensor, accept_len, accepted, bonus, ctx_len,
                    anchor, row_off, pos0, feats, stream=None):
    """The accepted path into the next cycle's injection inputs (in place):
    tree_feats [n_req, B+1, feat_dim], feats [n_req*(D+1), feat_dim]."""
    n_req, B1, fd = tree_feats.shape
    _check(lib().dflash_commit_accepted(n_req, D, B1 - 1, fd, _dtype_code(tree_feats),
                                        _ptr(tree_feats), tree_feats.stride(1), _ptr(accept_len),
                                        _ptr(accepted), _ptr(bonus), _ptr(ctx_len), _ptr(anchor),
                                        _ptr(row_off), _ptr(pos0), _ptr(feats), _stream(stream)))


def tree_buffers(n_req: int, B: int, device="cuda"):
    """Output tensors for ddtree_build: n_nodes, tok, parent, depth, rank, mask."""
    W = (B + 1 + 31) // 32
    i32 = dict(dtype=torch.int32, device=device)
    return (torch.empty(n_req, **i32), torch.empty(n_req, B + 1, **i32),
            torch.empty(n_req, B + 1, **i32), torch.empty(n_req, B + 1, **i32),
            torch.empty(n_req, B + 1, **i32), torch.empty(n_req, B + 1, W, **i32))


# ---------------------------------------------------------------------------
# Verification-side tree attention (DDTree page, 3.4.5)
# ---------------------------------------------------------------------------

def tree_attention_workspace_bytes(n_req: int, n_q: int, n_kv: int, head_dim: int, B: int,
                                   max_ctx: int) -> int:
    return int(lib().dflash_tree_attention_workspace_bytes(n_req, n_q, n_kv, head_dim, B,
                                                           max_ctx))


def tree_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cache_k: torch.Tensor,
                   cache_v: torch.Tensor, ctx_len: torch.Tensor, max_ctx: int,
                   mask: torch.Tensor, n_nodes: torch.Tensor, out: torch.Tensor,
                   ws: torch.Tensor, stream=None):
    """q [n_req, B+1, n_q*hd], k/v [n_req, B+1, n_kv*hd], cache [n_req, n_kv, cap, hd]
    (bf16), mask [n_req, B+1, W] (int32 view of the uint32 words), out like q."""
    n_req, B1, qw = q.shape
    _, n_kv, cap, hd = cache_k.shape
    n_q = qw // hd
    _check(lib().dflash_tree_attention(
        n_req, n_q, n_kv, hd, B1 - 1, _ptr(ctx_len), max_ctx, cap, _ptr(cache_k),
        _ptr(cache_v), _ptr(q), q.stride(1), _ptr(k), _ptr(v), k.stride(1), _ptr(mask),
        _ptr(n_nodes), _ptr(out), out.stride(1), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def tree_rope(x: torch.Tensor, n_heads: int, head_dim: int, theta: float, ctx_len: torch.Tensor,
              depth: torch.Tensor, stream=None):
    """Rotate heads 0..n_heads-1 of x [n_req, B+1, ld] in place at ctx_len + depth."""
    n_req, B1, ld = x.shape
    _check(lib().dflash_tree_rope(n_req, B1 - 1, n_heads, head_dim, theta, _ptr(ctx_len),
                                  _ptr(depth), _ptr(x), x.stride(1), _dtype_code(x),
                                  _stream(stream)))
