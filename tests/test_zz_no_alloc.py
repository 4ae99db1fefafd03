"""df_op_gemm_bf16_noalloc: the split-K GEMM without device allocation.

Some callers may not allocate device memory while they run (a process whose
memory is reserved up front by its own pool, a latency-critical loop).  The
no-alloc entry point runs the same tcgen05 GEMM with fixed scratch compiled
into the library.  Its output must match the allocating entry point's within
the GEMM tests' bound (1e-5 of the sum of |x||w| terms), on calls made one
after another that share the scratch, and shapes too large for the scratch
must be refused before anything is launched.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import synthetic as syn

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__ as g
    g.build()
    import block_diffusion_speculative_layer_gb300 as dfl
    return dfl.lib()


def dev_bf16(a):
    return torch.from_numpy(syn.f32_to_bf16_bits(a).view(np.int16)).cuda().view(torch.bfloat16)


def run(L, fn, x, w, splits, nt):
    M, K = x.shape
    N = w.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = fn(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(y.data_ptr()),
            M, N, K, splits, nt, ctypes.c_void_p(s))
    assert st == 0, st
    torch.cuda.synchronize()
    return y.cpu().numpy()


def bound(x, w):
    x64 = syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(x)).astype(np.float64)
    w64 = syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(w)).astype(np.float64)
    return 1e-5 * (np.abs(x64) @ np.abs(w64).T) + 1e-30


# (M, N, K, splits, token tile): split-K shapes of the decode cycle, one ragged
CASES = [(16, 4096, 4096, 5, 16), (5, 6144, 4096, 3, 16), (16, 4096, 12288, 5, 16), (40, 1024, 2048, 4, 64)]


def test_noalloc_matches_allocating_gemm_on_consecutive_calls(L):
    for rep in range(2):                      # two passes: the scratch keeps the last call's contents
        for i, (M, N, K, sp, nt) in enumerate(CASES):
            x = syn.make_normal((M, K), 1.0, seed=300 + i, stream=rep)
            w = syn.make_normal((N, K), 0.02, seed=300 + i, stream=10 + rep)
            xd, wd = dev_bf16(x), dev_bf16(w)
            ref = run(L, L.df_op_gemm_bf16, xd, wd, sp, nt)
            got = run(L, L.df_op_gemm_bf16_noalloc, xd, wd, sp, nt)
            assert np.isfinite(got).all()
            assert np.all(np.abs(got.astype(np.float64) - ref) <= bound(x, w))


def test_noalloc_rejects_shapes_beyond_its_scratch(L):
    # 512 rows in 256-row token tiles, 32 weight tiles, 5 splits: 10.5 M partial
    # floats, more than the fixed scratch holds; refused before any launch.
    M, N, K = 512, 4096, 4096
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    st = L.df_op_gemm_bf16_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                   ctypes.c_void_p(y.data_ptr()), M, N, K, 5, 256, None)
    assert st == 1  # DF_EINVAL
    assert float(y.abs().max()) == 0.0
