"""The allocation-free top-K entry point (for callers that cannot allocate
device memory when they run this step, e.g. a serving loop that must not call
cudaMalloc after start-up) gives the same results as the workspace variant,
on two calls in a row, through the C ABI.

This file sorts last so that a run stopping at the first failure has already
run every other test."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import binding as bd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,V,K,dtype", [
    (15, 151936, 8, torch.float32),     # the drafter's rows: split rows, partial records
    (300, 4099, 5, torch.bfloat16),     # one CTA per row, ragged vocabulary
])
def test_noalloc_topk_matches_workspace_variant(rows, V, K, dtype):
    g = torch.Generator(device="cuda").manual_seed(rows + K)
    x = (torch.randn(rows, V, generator=g, device="cuda") * 2.0).to(dtype)
    ids_ref = torch.empty(rows, K, dtype=torch.int32, device="cuda")
    lp_ref = torch.empty(rows, K, dtype=torch.float32, device="cuda")
    ws = torch.zeros(bd.topk_workspace_bytes(rows, V, K), dtype=torch.uint8, device="cuda")
    bd.logits_topk(x, K, ids_ref, lp_ref, ws)
    for _ in range(2):
        ids = torch.full((rows, K), -1, dtype=torch.int32, device="cuda")
        lp = torch.full((rows, K), float("nan"), dtype=torch.float32, device="cuda")
        bd.logits_topk_noalloc(x, K, ids, lp)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_ref)
        assert np.allclose(lp.cpu().numpy(), lp_ref.cpu().numpy(), atol=1e-5, rtol=0)


def test_noalloc_topk_rejects_too_many_rows():
    x = torch.zeros(4097, 16, device="cuda")
    ids = torch.empty(4097, 4, dtype=torch.int32, device="cuda")
    lp = torch.empty(4097, 4, device="cuda")
    with pytest.raises(bd.DflashError) as ei:
        bd.logits_topk_noalloc(x, 4, ids, lp)
    assert ei.value.status == 2
