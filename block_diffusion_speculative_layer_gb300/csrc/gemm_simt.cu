// fp32 GEMM on the CUDA cores for the fp32 engine: plain FMA, no TF32, so
// that the tiny fp32 decoder reproduces a float64 reference's token stream.
// One warp per output; lane l sums k = l, l+32, ... in order and the lanes
// meet in a fixed xor-shuffle tree, so each output is independent of M.
// The fused epilogues are the same ones the tensor-core GEMM runs.
#include "common.cuh"
#include "internal.h"

namespace dfk {

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                       float* __restrict__ y, int M, int N, int K) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  const int m = blockIdx.y;
  if (n >= N || m >= M) return;
  const float* xr = x + (size_t)m * K;
  const float* wr = w + (size_t)n * K;
  float s = 0.f;
  for (int k = lane; k < K; k += 32) s = fmaf(xr[k], wr[k], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) y[(size_t)m * N + n] = s;
}

constexpr int EPI_ROWS = 16;
constexpr int EPI_LD = 129;

__global__ void __launch_bounds__(128) epilogue_f32_kernel(const float* __restrict__ y, int N, int M, EpiParams ep) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[EPI_ROWS * EPI_LD];
  __shared__ RowMeta meta[EPI_ROWS];
  __shared__ float red[EPI_ROWS * 4];
  const int n0 = blockIdx.x * 128, m0 = blockIdx.y * EPI_ROWS;
  const int rows = min(EPI_ROWS, M - m0);
  for (int r = 0; r < rows; ++r) tile[r * EPI_LD + threadIdx.x] = y[(size_t)(m0 + r) * N + n0 + threadIdx.x];
  __syncthreads();
  epilogue_tile<float>(ep, tile, EPI_LD, n0, m0, rows, M, meta, red);
}

cudaError_t launch_gemm_f32(const float* x, const float* w, float* tmp, int M, int N, int K, const EpiParams& ep,
                            cudaStream_t st) {
  if (N % 128 || M < 1) return cudaErrorInvalidValue;
  cudaError_t e = launch_k(gemm_f32_kernel, dim3((N + 7) / 8, M), dim3(256), 0, st, x, w, tmp, M, N, K);
  if (e != cudaSuccess) return e;
  return launch_k(epilogue_f32_kernel, dim3(N / 128, (M + EPI_ROWS - 1) / EPI_ROWS), dim3(128), 0, st, tmp, N, M, ep);
}

}  // namespace dfk
