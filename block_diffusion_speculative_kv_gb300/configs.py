"""The five synthetic workloads the drafter cycle is tested and measured on.

Shapes follow the workloads the DFlash and DDTree pages evaluate: Qwen3-4B/8B
shaped five-layer drafters with a ~152k vocabulary, blocks of 16 (anchor plus
15 masks), five fused target layers, DDTree budgets between 16 and 1024 nodes,
and serving concurrency up to 32 ("DFlash" page, sections 3.4.3-3.4.4 and 4;
"DDTree" page, sections 3.4.3-3.4.6 and 5).  All tensors are seeded synthetic
data: the pages' datasets and trained checkpoints are not available.
"""
from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class DrafterShape:
    n_layers: int
    d: int            # drafter hidden size (also the fused feature size)
    n_q: int          # query heads
    n_kv: int         # key/value heads (GQA groups)
    head_dim: int
    d_ff: int         # SwiGLU inner size
    vocab: int
    n_feat: int       # number of target layers whose hidden states are fused
    d_feat: int       # target hidden size
    dtype: str        # "fp32" or "bf16": weights, KV cache and GEMM operands
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6

    @property
    def mask_id(self) -> int:
        # The pages never name the mask token; the last vocabulary id is used.
        return self.vocab - 1

    @property
    def qkv_dim(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv * self.head_dim


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Optional[DrafterShape]   # None for the logits-only stress workload
    n_req: int
    L: int                          # block length: anchor + L-1 masks
    D: int                          # draft depth (rows of marginals per request)
    K: int                          # top-K per draft position
    B: int                          # DDTree node budget (non-root nodes)
    ctx: Tuple[int, int]            # context length (fixed, or inclusive U[lo, hi])
    cap: int                        # KV-cache capacity per request
    target_agree: float             # p in p**(depth+1): chance target agrees with top-1
    temperatures: Tuple[float, ...] = (0.0,)
    seed: int = 0
    vocab: int = 0                  # logits-only workload vocabulary


QWEN3_4B_DRAFTER = DrafterShape(5, 2560, 32, 8, 128, 9728, 151936, 5, 2560, "bf16")
QWEN3_8B_DRAFTER = DrafterShape(5, 4096, 32, 8, 128, 12288, 151936, 5, 4096, "bf16")
TINY_DRAFTER = DrafterShape(1, 256, 4, 2, 64, 688, 1024, 3, 256, "fp32")

WORKLOADS = {
    0: Workload("tiny-fp32", TINY_DRAFTER, n_req=1, L=8, D=7, K=4, B=16,
                ctx=(64, 64), cap=64, target_agree=0.9, seed=0),
    1: Workload("qwen3-4b-drafter-b1", QWEN3_4B_DRAFTER, n_req=1, L=16, D=15, K=8,
                B=64, ctx=(2048, 2048), cap=2048, target_agree=0.9, seed=1),
    2: Workload("qwen3-8b-drafter-b1", QWEN3_8B_DRAFTER, n_req=1, L=16, D=15, K=8,
                B=256, ctx=(8192, 8192), cap=8192, target_agree=0.9,
                temperatures=(0.0, 1.0), seed=2),
    3: Workload("qwen3-8b-drafter-batch32", QWEN3_8B_DRAFTER, n_req=32, L=16, D=15,
                K=8, B=64, ctx=(512, 8192), cap=8192, target_agree=0.9, seed=3),
    4: Workload("topk-ddtree-stress", None, n_req=256, L=16, D=16, K=8, B=512,
                ctx=(0, 0), cap=0, target_agree=0.95, seed=4, vocab=151936),
}
