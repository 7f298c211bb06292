"""PyTorch-facing wrapper of the drafter calls of libdflash.so.

Marshalling only: it packs natural-layout weights ([out, in] matrices per
layer) into the layouts include/dflash.h documents (W_q|W_k|W_v stacked,
gate/up rows interleaved, U_K|U_V of every layer stacked), allocates the KV
cache and the workspace as PyTorch CUDA tensors, and forwards each call to
the C ABI function of the same name.  All arithmetic runs in the library.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, List, Optional

import torch

from . import binding as bd
from .configs import DrafterShape


def pack_weights(shape: DrafterShape, w: Dict) -> Dict[str, object]:
    """Copy natural-layout weights into the packed device layouts."""
    s = shape
    packed = {
        "w_proj": w["w_proj"].contiguous(),
        "embed": w["embed"].contiguous(),
        "lm_head": w["lm_head"].contiguous(),
        "final_norm": w["final_norm"].contiguous(),
        "u_kv": torch.stack([torch.cat([w["uk"][l], w["uv"][l]], 0)
                             for l in range(s.n_layers)], 0).contiguous(),
        "attn_norm": [t.contiguous() for t in w["attn_norm"]],
        "mlp_norm": [t.contiguous() for t in w["mlp_norm"]],
        "w_qkv": [torch.cat([w["wq"][l], w["wk"][l], w["wv"][l]], 0).contiguous()
                  for l in range(s.n_layers)],
        "wo": [t.contiguous() for t in w["wo"]],
        "w_gate_up": [torch.stack([w["w_gate"][l], w["w_up"][l]], 1)
                      .reshape(2 * s.d_ff, s.d).contiguous() for l in range(s.n_layers)],
        "w_down": [t.contiguous() for t in w["w_down"]],
    }
    return packed


class Drafter:
    """One drafter model with its KV cache and workspace on the current device."""

    def __init__(self, shape: DrafterShape, weights: Dict, n_req: int, cap: int,
                 max_inject_rows: int, L: int, K: int, anchor_sees_block: bool = True,
                 packed: Optional[Dict] = None):
        self.shape = shape
        self.n_req, self.cap, self.L, self.K = n_req, cap, L, K
        self.max_inject_rows = max_inject_rows
        self.packed = packed if packed is not None else pack_weights(shape, weights)
        p = self.packed
        dt = bd.DFLASH_BF16 if shape.dtype == "bf16" else bd.DFLASH_F32
        self.dims = bd.Dims(shape.n_layers, shape.d, shape.n_q, shape.n_kv, shape.head_dim,
                            shape.d_ff, shape.vocab, shape.n_feat, shape.d_feat, dt,
                            shape.rope_theta, shape.rms_eps, shape.mask_id,
                            1 if anchor_sees_block else 0)
        wt = bd.Weights()
        wt.w_proj = p["w_proj"].data_ptr()
        wt.embed = p["embed"].data_ptr()
        wt.lm_head = p["lm_head"].data_ptr()
        wt.final_norm = p["final_norm"].data_ptr()
        wt.u_kv = p["u_kv"].data_ptr()
        for l in range(shape.n_layers):
            wt.attn_norm[l] = p["attn_norm"][l].data_ptr()
            wt.w_qkv[l] = p["w_qkv"][l].data_ptr()
            wt.wo[l] = p["wo"][l].data_ptr()
            wt.mlp_norm[l] = p["mlp_norm"][l].data_ptr()
            wt.w_gate_up[l] = p["w_gate_up"][l].data_ptr()
            wt.w_down[l] = p["w_down"][l].data_ptr()
        self._weights_struct = wt
        h = C.c_void_p()
        bd._check(bd.lib().dflash_model_create(C.byref(self.dims), C.byref(wt), C.byref(h)))
        self.handle = h
        tdt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
        dev = torch.device("cuda", torch.cuda.current_device())
        self.cache_k: List[torch.Tensor] = [
            torch.zeros(n_req, shape.n_kv, cap, shape.head_dim, dtype=tdt, device=dev)
            for _ in range(shape.n_layers)]
        self.cache_v: List[torch.Tensor] = [torch.zeros_like(t) for t in self.cache_k]
        cs = bd.Cache()
        for l in range(shape.n_layers):
            cs.k[l] = self.cache_k[l].data_ptr()
            cs.v[l] = self.cache_v[l].data_ptr()
        cs.n_req, cs.cap = n_req, cap
        self.cache_struct = cs
        nbytes = int(bd.lib().dflash_workspace_bytes(h, n_req, max_inject_rows, L, K))
        if nbytes == 0:
            raise bd.DflashError(1, "dflash_workspace_bytes rejected the sizes")
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.logits = None

    # -- the path ----------------------------------------------------------
    def inject_kv(self, feats: torch.Tensor, row_off: torch.Tensor, pos0: torch.Tensor,
                  n_req: Optional[int] = None, stream=None):
        n_req = self.n_req if n_req is None else n_req
        bd._check(bd.lib().dflash_inject_kv(
            self.handle, C.byref(self.cache_struct), n_req, feats.shape[0], bd._ptr(row_off),
            bd._ptr(pos0), bd._ptr(feats), bd._ptr(self.ws), self.ws.numel(),
            bd._stream(stream)))

    def draft_block(self, anchor: torch.Tensor, ctx_len: torch.Tensor, max_ctx: int,
                    topk_ids: torch.Tensor, topk_logp: torch.Tensor,
                    logits: Optional[torch.Tensor] = None, n_req: Optional[int] = None,
                    L: Optional[int] = None, K: Optional[int] = None, sampling=None,
                    stream=None):
        """sampling: None (top-K by logit) or (temperature, seed[, row_offset])."""
        n_req = self.n_req if n_req is None else n_req
        L = self.L if L is None else L
        K = self.K if K is None else K
        bd._check(bd.lib().dflash_draft_block(
            self.handle, C.byref(self.cache_struct), n_req, bd._ptr(anchor), bd._ptr(ctx_len),
            max_ctx, L, K, bd.sampling_arg(sampling), bd._ptr(topk_ids), bd._ptr(topk_logp),
            bd._ptr(logits), bd._ptr(self.ws), self.ws.numel(), bd._stream(stream)))

    def draft_cycle(self, feats: torch.Tensor, row_off: torch.Tensor, pos0: torch.Tensor,
                    anchor: torch.Tensor, ctx_len: torch.Tensor, max_ctx: int,
                    topk_ids: torch.Tensor, topk_logp: torch.Tensor,
                    logits: Optional[torch.Tensor] = None, n_req: Optional[int] = None,
                    L: Optional[int] = None, K: Optional[int] = None, sampling=None,
                    stream=None):
        """inject_kv followed by draft_block, as one call (same results)."""
        n_req = self.n_req if n_req is None else n_req
        L = self.L if L is None else L
        K = self.K if K is None else K
        bd._check(bd.lib().dflash_draft_cycle(
            self.handle, C.byref(self.cache_struct), n_req, feats.shape[0], bd._ptr(row_off),
            bd._ptr(pos0), bd._ptr(feats), bd._ptr(anchor), bd._ptr(ctx_len), max_ctx, L, K,
            bd.sampling_arg(sampling), bd._ptr(topk_ids), bd._ptr(topk_logp), bd._ptr(logits),
            bd._ptr(self.ws), self.ws.numel(), bd._stream(stream)))

    def read_status(self) -> int:
        return bd.read_status(self.ws)

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            bd.lib().dflash_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
