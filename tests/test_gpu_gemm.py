"""The tensor-core GEMM engine (TMA + tcgen05 + TMEM) against a float64 matmul.

The engine computes X0 W0^T (+ X1 W0^T when X has a second plane, + X0 W1^T
when W has one); the reference forms exactly those products in float64 from
the same bf16 values, so the only difference is fp32 accumulation order.
"""
import numpy as np
import pytest
import torch

from history_free_speculative_gb300 import binding

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # rows, outs, K, xplanes, wplanes
    (8, 6144, 4096, 1, 1),      # B=1 QKV-like: split-K over many CTAs
    (14, 2048, 4096, 1, 1),     # context K/V rows
    (1, 64, 64, 2, 2),          # smallest: one row, one k block, all plane products
    (7, 4096, 512, 2, 1),       # head output map P (k = padded rank)
    (224, 1216, 4096, 2, 1),    # LM-head-like rows (2 M-tiles), two activation planes
    (256, 2048, 1024, 1, 1),    # B=32 local rows
    (448, 512, 256, 1, 1),      # 4 M-tiles in one CTA
    (600, 264, 128, 1, 1),      # 5 M-tiles: two row groups; outs not a multiple of 16
    (129, 200, 192, 2, 2),      # ragged rows / outs, k = 3 blocks, two planes on both sides
]


def _tiled(w):
    """The library's tiled weight layout: rows padded to 64, 64 x 64 row-major tiles."""
    rows, K = w.shape
    rp = (rows + 63) // 64 * 64
    wp = torch.zeros(rp, K, dtype=w.dtype, device=w.device)
    wp[:rows] = w
    return wp.view(rp // 64, 64, K // 64, 64).permute(0, 2, 1, 3).contiguous().view(rp, K)


def _planes(x, n):
    hi = x.to(torch.bfloat16)
    if n == 1:
        return [hi]
    lo = (x - hi.float()).to(torch.bfloat16)
    return [hi, lo]


@pytest.mark.parametrize("rows,outs,K,xp,wp", CASES)
def test_engine_matches_float64(rows, outs, K, xp, wp):
    g = torch.Generator().manual_seed(rows * 7 + outs + K)
    x_rows = (rows + 127) // 128 * 128
    X = torch.randn(x_rows, K, generator=g)
    X[rows:] = float("nan")          # rows past `rows` must not leak into the result
    W = torch.randn(outs, K, generator=g) * 0.05
    Xp = [p.to(DEV) for p in _planes(X, xp)]
    Wp = [p.to(DEV) for p in _planes(W, wp)]
    got, st = binding.selftest_gemm(Xp, [_tiled(p) for p in Wp], rows=rows, outs=outs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x64 = [p[:rows].double().cpu().numpy() for p in Xp]
    w64 = [p.double().cpu().numpy() for p in Wp]
    ref = x64[0] @ w64[0].T
    if xp == 2:
        ref += x64[1] @ w64[0].T
    if wp == 2:
        ref += x64[0] @ w64[1].T
    got = got.double().cpu().numpy()
    scale = np.sqrt(K) * np.abs(w64[0]).max() * np.abs(x64[0]).max()
    err = np.abs(got - ref).max()
    assert np.isfinite(got).all()
    assert err <= 1e-5 * scale, (err, scale)


@pytest.mark.parametrize("N", [64, 128, 192, 256])
@pytest.mark.parametrize("S", [1, 2, 4])
@pytest.mark.parametrize("rows", [256, 100])
def test_engine_plans_match_float64(N, S, rows):
    """Every slab width and k split the create-time plan timing may pick, on a
    two-tile and a one-tile row count: the same product as the float64 one."""
    outs, K = 768, 512
    g = torch.Generator().manual_seed(N * 31 + S * 7 + rows)
    x_rows = (rows + 127) // 128 * 128
    X = torch.randn(x_rows, K, generator=g)
    X[rows:] = float("nan")
    W = torch.randn(outs, K, generator=g) * 0.05
    Xp = [p.to(DEV) for p in _planes(X, 1)]
    Wp = [p.to(DEV) for p in _planes(W, 1)]
    got, st = binding.selftest_gemm(Xp, [_tiled(p) for p in Wp], rows=rows, outs=outs, plan=(N, S, 0))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x64 = Xp[0][:rows].double().cpu().numpy()
    w64 = Wp[0].double().cpu().numpy()
    ref = x64 @ w64.T
    got = got.double().cpu().numpy()
    scale = np.sqrt(K) * np.abs(w64).max() * np.abs(x64).max()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 1e-5 * scale



@pytest.mark.parametrize("rows,K,N,S", [(8, 4096, 256, 8), (8, 12288, 192, 16), (21, 4096, 128, 6), (64, 2048, 256, 12)])
def test_engine_few_rows_many_splits_match_float64(rows, K, N, S):
    """Few-row products take up to 16 k splits (wide slabs over all SMs): the planes
    of every split count sum to the float64 product."""
    outs = 1000 if N != 256 else 4096
    g = torch.Generator().manual_seed(rows * 5 + K + N + S)
    x_rows = 128
    X = torch.randn(x_rows, K, generator=g)
    X[rows:] = float("nan")
    W = torch.randn(outs, K, generator=g) * 0.05
    Xp = [p.to(DEV) for p in _planes(X, 1)]
    Wp = [p.to(DEV) for p in _planes(W, 1)]
    got, st = binding.selftest_gemm(Xp, [_tiled(p) for p in Wp], rows=rows, outs=outs, plan=(N, S, 0))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x64 = Xp[0][:rows].double().cpu().numpy()
    w64 = Wp[0].double().cpu().numpy()
    ref = x64 @ w64.T
    got = got.double().cpu().numpy()
    scale = np.sqrt(K) * np.abs(w64).max() * np.abs(x64).max()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 1e-5 * scale
