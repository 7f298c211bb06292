"""The tensor-core GEMM (tcgen05 + TMEM + TMA, stream-K with last-arriver
reduction) through its C ABI entry point, against a float64 product of the
same bf16 values.  Bound: |Y - ref| <= 5e-4 * (|X| . |W|^T), the fp32
accumulation bound over K <= 20480 with margin."""
import numpy as np
import pytest
import torch

from block_diffusion_speculative_kv_gb300 import binding as bd

pytestmark = pytest.mark.gpu


def _run(M, N, K, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    X = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    Y = torch.full((M, N), float("nan"), device="cuda")
    ws = torch.zeros(bd.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    bd.linear_bf16(X, W, Y, ws)
    Y2 = torch.empty_like(Y)
    bd.linear_bf16(X, W, Y2, ws)          # counters must have been left at zero
    torch.cuda.synchronize()
    assert bd.read_status(ws) == 0
    x = X.double().cpu().numpy()
    w = W.double().cpu().numpy()
    ref = x @ w.T
    bound = 5e-4 * (np.abs(x) @ np.abs(w).T) + 1e-30
    y = Y.cpu().numpy()
    assert np.all(np.isfinite(y))
    assert np.all(np.abs(y - ref) <= bound), float(np.max(np.abs(y - ref) / bound))
    assert torch.equal(Y, Y2), "two runs differ: the reduction order is not fixed"


@pytest.mark.parametrize("M,N,K", [
    (16, 128, 64),        # one tile, one K block
    (16, 4096, 4096),     # batch-1 square layer: split tiles, several slots
    (15, 6144, 4096),     # ragged rows (TMA zero fill), QKV shape
    (1, 256, 1024),       # a single activation row
    (16, 4096, 12288),    # down projection shape
    (16, 24576, 4096),    # gate/up shape
    (40, 1024, 640),      # 64-row tile
    (200, 512, 1024),     # 256-row tile, ragged
    (512, 1024, 4096),    # two 256-row tiles (batched workload)
    (700, 384, 256),      # three row tiles, few units per CTA
])
def test_linear_matches_float64(M, N, K):
    _run(M, N, K, seed=M + N + K)


def test_linear_unaligned_output_rows():
    # an output 4 bytes off a 16-byte boundary: the 32..256-row tiles' epilogues
    # take their element-wise paths (the split-tile shares from registers, one
    # column per thread), with split tiles of many contributors (16 tiles of
    # 256 rows for 152 SMs)
    M, N, K = 512, 1024, 4096
    g = torch.Generator(device="cuda").manual_seed(11)
    X = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    buf = torch.full((M * N + 1,), float("nan"), device="cuda")
    Y = buf[1:].view(M, N)
    assert Y.data_ptr() % 16 == 4
    ws = torch.zeros(bd.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    bd.linear_bf16(X, W, Y, ws)
    torch.cuda.synchronize()
    assert bd.read_status(ws) == 0
    x = X.double().cpu().numpy()
    w = W.double().cpu().numpy()
    ref = x @ w.T
    bound = 5e-4 * (np.abs(x) @ np.abs(w).T) + 1e-30
    y = Y.cpu().numpy()
    assert np.all(np.isfinite(y))
    assert np.all(np.abs(y - ref) <= bound), float(np.max(np.abs(y - ref) / bound))
    assert np.isnan(buf[0].item())      # nothing written before the output
    # and the same values as through an aligned output (the same sum order)
    Y2 = torch.empty(M, N, device="cuda")
    bd.linear_bf16(X, W, Y2, ws)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2)


def test_linear_lm_head_shape():
    # vocab-sized output: 1187 column tiles streamed by one CTA per SM
    _run(16, 151936, 256, seed=7)


def test_linear_rejects_bad_shapes():
    lib = bd.lib()
    assert lib.dflash_linear_bf16(16, 100, 64, None, None, None, None, 0, None) == 1
    assert lib.dflash_linear_bf16(16, 128, 100, None, None, None, None, 0, None) == 1
