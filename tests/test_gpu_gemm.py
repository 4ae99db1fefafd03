"""tcgen05 GEMM and fused LM-head argmax against plain float64 matmuls.

The reference is numpy's float64 matrix product of the same bf16 inputs (a
library primitive, independent of the CUDA path).  The GEMM accumulates in
fp32, so each output may differ from the float64 value by a few fp32 ulps of
the sum of |x||w| terms: the bound used is 1e-5 of that sum.  Argmax must
pick the float64 argmax wherever the float64 top-2 margin exceeds that bound,
and otherwise an index whose float64 logit is within it of the maximum.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import synthetic as syn

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dfl():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as m
    return m


def bf16(a: np.ndarray) -> np.ndarray:
    """Round to bf16; return float32 holding the rounded values."""
    return syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(a))


def dev_bf16(a: np.ndarray):
    return torch.from_numpy(syn.f32_to_bf16_bits(a).view(np.int16)).cuda().view(torch.bfloat16)


def inputs(M, N, K, seed):
    x = bf16(syn.make_normal((M, K), 1.0, seed=seed, stream=0))
    w = bf16(syn.make_normal((N, K), 0.02, seed=seed, stream=1))
    return x, w


def check_close(y, x, w, cols=None):
    x64 = x.astype(np.float64)
    w64 = w.astype(np.float64) if cols is None else w[cols].astype(np.float64)
    ref = x64 @ w64.T
    bound = np.abs(x64) @ np.abs(w64).T
    got = y if cols is None else y[:, cols]
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= 1e-5 * bound + 1e-30), float((err / (bound + 1e-30)).max())


CASES = [
    # (M, N, K, splits, token_tile): ragged rows, several tiles, split-K
    (1, 256, 128, 1, 16),
    (5, 384, 256, 2, 16),
    (16, 512, 4096, 0, 0),
    (17, 1024, 512, 3, 32),
    (40, 256, 1024, 4, 64),
    (100, 512, 1024, 0, 0),
    (300, 256, 640, 0, 0),
    (512, 384, 320, 5, 256),
]


@pytest.mark.parametrize("M,N,K,splits,nt", CASES)
def test_gemm_matches_float64(dfl, M, N, K, splits, nt):
    x, w = inputs(M, N, K, seed=100 + M)
    y = dfl.gemm_bf16(dev_bf16(x), dev_bf16(w), splits=splits, token_tile=nt)
    torch.cuda.synchronize()
    check_close(y.cpu().numpy(), x, w)


# The decode-cycle shapes of the Qwen3-8B-shaped model (d=4096, GQA 32/8 x 128,
# SwiGLU 12288) at 16 token rows, in the launch configuration the engine uses.
FULL = [
    (16, 6144, 4096),    # fused q|k|v
    (16, 4096, 4096),    # o
    (16, 24576, 4096),   # gate|up
    (16, 4096, 12288),   # down
    (16, 4096, 20480),   # feature fusion FC
    (16, 10240, 4096),   # K/V injection, 5 drafter layers
    (512, 6144, 4096),   # prefill rows
]


@pytest.mark.parametrize("M,N,K", FULL)
def test_gemm_full_shapes_sampled(dfl, M, N, K):
    x, w = inputs(M, N, K, seed=7)
    y = dfl.gemm_bf16(dev_bf16(x), dev_bf16(w)).cpu().numpy()
    cols = np.random.default_rng(0).choice(N, size=min(N, 384), replace=False)
    check_close(y, x, w, cols)
    assert np.isfinite(y).all()


def test_gemm_rows_independent_of_M(dfl):
    # A row's result is bitwise the same whatever the number of token rows.
    M, N, K = 16, 1024, 4096
    x, w = inputs(M, N, K, seed=11)
    xd, wd = dev_bf16(x), dev_bf16(w)
    full = dfl.gemm_bf16(xd, wd).cpu().numpy()
    for j in [0, 3, 15]:
        one = dfl.gemm_bf16(xd[j:j + 1].contiguous(), wd).cpu().numpy()
        np.testing.assert_array_equal(one[0], full[j])
    part = dfl.gemm_bf16(xd[:7].contiguous(), wd).cpu().numpy()
    np.testing.assert_array_equal(part, full[:7])


@pytest.mark.parametrize("nt", [32, 64, 128, 256])
def test_gemm_rows_independent_of_token_tile(dfl, nt):
    M, N, K = 16, 512, 2048
    x, w = inputs(M, N, K, seed=12)
    xd, wd = dev_bf16(x), dev_bf16(w)
    a = dfl.gemm_bf16(xd, wd, token_tile=16).cpu().numpy()
    b = dfl.gemm_bf16(xd, wd, token_tile=nt).cpu().numpy()
    np.testing.assert_array_equal(a, b)


# The serial-split form (token_tile -64 / -128; the engine's choice beyond 128
# token rows): one CTA runs every K range of its tile and adds the partials in
# split order, so it must equal the split-K form bit for bit.
WIDE = [
    # (M, N, K, splits, token_tile)
    (129, 256, 512, 1, -64),
    (200, 384, 1024, 3, -64),
    (256, 512, 4096, 8, -128),
    (300, 256, 640, 5, -128),
    (512, 1024, 2048, 4, -64),
    (77, 128, 256, 2, -128),
]


@pytest.mark.parametrize("M,N,K,splits,nt", WIDE)
def test_gemm_wide_matches_float64_and_split_k(dfl, M, N, K, splits, nt):
    x, w = inputs(M, N, K, seed=300 + M)
    xd, wd = dev_bf16(x), dev_bf16(w)
    y = dfl.gemm_bf16(xd, wd, splits=splits, token_tile=nt).cpu().numpy()
    check_close(y, x, w)
    ref = dfl.gemm_bf16(xd, wd, splits=splits, token_tile=16).cpu().numpy()
    np.testing.assert_array_equal(y, ref)


@pytest.mark.parametrize("M,N,K", [(256, 6144, 4096), (256, 4096, 4096), (256, 4096, 12288), (144, 24576, 4096)])
def test_gemm_wide_engine_shapes_bitwise(dfl, M, N, K):
    # the engine's own choice (token_tile 0: the serial-split form for the first two
    # shapes, the split-K form with 256-token tiles for the others) against the
    # split-K form with 16-token tiles, on the verify pass shapes of a 16-sequence batch
    x, w = inputs(M, N, K, seed=17)
    xd, wd = dev_bf16(x), dev_bf16(w)
    a = dfl.gemm_bf16(xd, wd).cpu().numpy()
    b = dfl.gemm_bf16(xd, wd, token_tile=16).cpu().numpy()
    np.testing.assert_array_equal(a, b)
    cols = np.random.default_rng(1).choice(N, size=256, replace=False)
    check_close(a, x, w, cols)


def check_argmax(ids, x, w):
    x64, w64 = x.astype(np.float64), w.astype(np.float64)
    logits = x64 @ w64.T
    bound = 1e-5 * (np.abs(x64) @ np.abs(w64).T).max(axis=1)
    srt = np.sort(logits, axis=1)
    margin = srt[:, -1] - srt[:, -2]
    want = np.argmax(logits, axis=1)
    for m in range(len(ids)):
        if margin[m] > 2 * bound[m]:
            assert ids[m] == want[m], (m, ids[m], want[m])
        else:
            assert logits[m, ids[m]] >= srt[m, -1] - 2 * bound[m]


@pytest.mark.parametrize("M,V,K", [(1, 1024, 256), (15, 2048, 512), (16, 151936, 4096), (33, 4096, 1024),
                                   (160, 8192, 1024), (256, 16384, 4096)])
def test_lmhead_argmax(dfl, M, V, K):
    x, w = inputs(M, V, K, seed=21 + M)
    ids = dfl.lmhead_argmax_bf16(dev_bf16(x), dev_bf16(w)).cpu().numpy()
    check_argmax(ids, x, w)


def test_lmhead_argmax_ties_pick_lowest_index(dfl):
    # Duplicate the winning row at a higher and at a lower index: the lowest wins.
    M, V, K = 4, 1024, 256
    x, w = inputs(M, V, K, seed=31)
    logits = x.astype(np.float64) @ w.astype(np.float64).T
    win = np.argmax(logits, axis=1)
    w2 = w.copy()
    for m in range(M):
        w2[1000 - m] = w[win[m]]
        w2[3 + m] = w[win[m]]
    ids = dfl.lmhead_argmax_bf16(dev_bf16(x), dev_bf16(w2)).cpu().numpy()
    for m in range(M):
        assert ids[m] == min(3 + m, win[m])


# Split-K through the cluster (each CTA reads its rows of the other CTAs'
# partials from their shared memory) against split-K through a global
# workspace (DF_NO_CLUSTER=1, in a child process): both add the partials in
# split order, so the results are the same bits.
SPLIT_K = [(16, 1024, 4096, 8, 16), (13, 640, 2560, 5, 16), (40, 256, 1024, 4, 64), (256, 384, 320, 5, 256)]

_WORKSPACE_CHILD = """
import sys
import numpy as np
import torch
sys.path[:0] = [sys.argv[2], sys.argv[3]]
import block_diffusion_speculative_layer_gb300 as dfl
import test_gpu_gemm as t
for i, (M, N, K, splits, nt) in enumerate(t.SPLIT_K):
    x, w = t.inputs(M, N, K, seed=30 + i)
    y = dfl.gemm_bf16(t.dev_bf16(x), t.dev_bf16(w), splits=splits, token_tile=nt).cpu().numpy()
    np.save(sys.argv[1] + "/y%d.npy" % i, y)
"""


def test_cluster_split_k_equals_workspace_split_k(dfl, tmp_path):
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, DF_NO_CLUSTER="1")
    subprocess.run([sys.executable, "-c", _WORKSPACE_CHILD, str(tmp_path), os.path.dirname(here), here], env=env,
                   check=True, timeout=600)
    for i, (M, N, K, splits, nt) in enumerate(SPLIT_K):
        x, w = inputs(M, N, K, seed=30 + i)
        got = dfl.gemm_bf16(dev_bf16(x), dev_bf16(w), splits=splits, token_tile=nt).cpu().numpy()
        check_close(got, x, w)
        np.testing.assert_array_equal(got, np.load(tmp_path / ("y%d.npy" % i)))
