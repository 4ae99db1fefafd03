// Small kernels of the draft-and-verify cycle: embedding gather, RMSNorm
// (with the feature-layer tap), block preparation, argmax finalisation,
// greedy acceptance with rollback bookkeeping, and the greedy decode step.
#include "common.cuh"
#include "internal.h"

#include <stdlib.h>

namespace dfk {

bool pdl_enabled() {
  static int on = -1;
  if (on < 0) {
    const char* e = getenv("DF_NO_PDL");
    on = (e && e[0] == '1') ? 0 : 1;
  }
  return on != 0;
}

// Embedding gather for the rows of a pass: h[m] = embed[tok[m]] (fp32), the
// same row in the model dtype for the first layer's GEMM, and its sum of
// squares per 128-feature tile (the folded RMSNorm of that GEMM).  128 threads.
constexpr int EMBED_MAX_TILES = 128;  // model width up to 16384

template <typename T>
__global__ void __launch_bounds__(128) embed_kernel(const T* __restrict__ embed, const int* __restrict__ tok,
                                                    float* __restrict__ h, T* __restrict__ xraw,
                                                    float* __restrict__ ss, int d, int vocab, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[EMBED_MAX_TILES * 4];  // per 128-feature tile, one partial per warp
  const int m = blockIdx.x;
  const int t = tok[m];
  const bool ok = t >= 0 && t < vocab;
  if (!ok && threadIdx.x == 0 && t >= vocab) flag_error(err, ERR_BOUNDS);
  const int tiles = d >> 7;
  const int warp = threadIdx.x >> 5;
  for (int tb = 0; tb < tiles; tb += 32) {
    // 32 tiles' loads in flight together
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int i = (tb + j) * 128 + threadIdx.x;
      v[j] = (ok && tb + j < tiles) ? Cvt<T>::to_f(embed[(size_t)t * d + i]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (tb + j >= tiles) break;
      const int i = (tb + j) * 128 + threadIdx.x;
      h[(size_t)m * d + i] = v[j];
      xraw[(size_t)m * d + i] = Cvt<T>::from_f(v[j]);
      float q = v[j] * v[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
      if ((threadIdx.x & 31) == 0) red[(tb + j) * 4 + warp] = q;
    }
  }
  __syncthreads();
  for (int tl = threadIdx.x; tl < tiles; tl += 128)
    ss[(size_t)m * tiles + tl] = ((red[tl * 4 + 0] + red[tl * 4 + 1]) + red[tl * 4 + 2]) + red[tl * 4 + 3];
}

cudaError_t launch_embed(const void* embed, bool bf16, const int* tok, float* h, void* xraw, float* ss, int M, int d,
                         int vocab, int* err, cudaStream_t st) {
  if (d % 128 || d / 128 > EMBED_MAX_TILES) return cudaErrorInvalidValue;
  if (bf16)
    return launch_k(embed_kernel<__nv_bfloat16>, dim3(M), dim3(128), 0, st,
                    reinterpret_cast<const __nv_bfloat16*>(embed), tok, h, reinterpret_cast<__nv_bfloat16*>(xraw), ss, d,
                    vocab, err);
  return launch_k(embed_kernel<float>, dim3(M), dim3(128), 0, st, reinterpret_cast<const float*>(embed), tok, h,
                  reinterpret_cast<float*>(xraw), ss, d, vocab, err);
}

// W[n][k] *= gain[k] for a [rows][cols] matrix (a norm's gain folded into the
// weight that consumes the normalised rows).
template <typename T>
__global__ void scale_cols_kernel(T* __restrict__ w, long long rows, int cols, const float* __restrict__ gain) {
  const long long n = rows * cols;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    w[i] = Cvt<T>::from_f(Cvt<T>::to_f(w[i]) * gain[i % cols]);
}

cudaError_t launch_scale_cols(void* w, bool bf16, long long rows, int cols, const float* gain, cudaStream_t st) {
  if (bf16)
    scale_cols_kernel<__nv_bfloat16><<<1024, 256, 0, st>>>(reinterpret_cast<__nv_bfloat16*>(w), rows, cols, gain);
  else
    scale_cols_kernel<float><<<1024, 256, 0, st>>>(reinterpret_cast<float*>(w), rows, cols, gain);
  return cudaGetLastError();
}

// One block per row; the sum of squares is reduced in a fixed order
// (thread-strided partial sums, then a fixed tree), so a row's result never
// depends on the other rows.
template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ h, int ldh,
                                                      const float* __restrict__ gain, T* __restrict__ out, int ldo,
                                                      int d, float eps, T* __restrict__ taps, int tap_index,
                                                      const int* __restrict__ row_pos) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  if (row_pos && row_pos[m] < 0) return;
  const float* x = h + (size_t)m * ldh;
  __shared__ float red[256];
  float s = 0.f;
  for (int i = threadIdx.x; i < d; i += 256) s = fmaf(x[i], x[i], s);
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  const float inv = rsqrtf(red[0] / (float)d + eps);
  for (int i = threadIdx.x; i < d; i += 256) {
    const float v = x[i];
    out[(size_t)m * ldo + i] = Cvt<T>::from_f(v * inv * gain[i]);
    if (taps) taps[((size_t)m * 5 + tap_index) * d + i] = Cvt<T>::from_f(v);
  }
}

cudaError_t launch_rmsnorm(const float* h, int ldh, const float* gain, void* out, int ldo, bool bf16, int M, int d,
                           float eps, void* taps, int tap_index, const int* row_pos, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (bf16)
    return launch_k(rmsnorm_kernel<__nv_bfloat16>, dim3(M), dim3(256), 0, st, h, ldh, gain, reinterpret_cast<__nv_bfloat16*>(out), ldo, d, eps,
                                                     reinterpret_cast<__nv_bfloat16*>(taps), tap_index, row_pos);
  else
    return launch_k(rmsnorm_kernel<float>, dim3(M), dim3(256), 0, st, h, ldh, gain, reinterpret_cast<float*>(out), ldo, d, eps,
                                             reinterpret_cast<float*>(taps), tap_index, row_pos);
}

__global__ void fill_u64_kernel(unsigned long long* p, unsigned long long v, int n) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}
cudaError_t launch_fill_u64(unsigned long long* p, unsigned long long v, int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  return launch_k(fill_u64_kernel, dim3((n + 255) / 256), dim3(256), 0, st, p, v, n);
}

__global__ void argmax_finalize_kernel(const unsigned long long* amax, int* ids, int M) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < M) ids[i] = argmax_key_index(amax[i]);
}
cudaError_t launch_argmax_finalize(const unsigned long long* amax, int* ids, int M, cudaStream_t st) {
  return launch_k(argmax_finalize_kernel, dim3((M + 127) / 128), dim3(128), 0, st, amax, ids, M);
}

// Row b*B + i of a block: token (bonus, then MASK or draft i), absolute
// position bonus_pos + i, sequence slot.  The block starts at the bonus token
// the last verification produced.
__global__ void prep_block_kernel(const int* slots, int B, const int* bonus, const int* bonus_pos, const int* drafts,
                                  int mask_id, int verify, int* row_tok, int* row_pos, int* row_seq) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, i = threadIdx.x;
  if (i >= B) return;
  const int s = slots[b];
  const int m = b * B + i;
  int t;
  if (i == 0) t = bonus[s];
  else t = verify ? drafts[s * (B - 1) + i - 1] : mask_id;
  row_tok[m] = t;
  row_pos[m] = bonus_pos[s] + i;
  row_seq[m] = s;
}
cudaError_t launch_prep_block(const int* batch_slots, int nseq, int B, const int* bonus, const int* bonus_pos,
                              const int* drafts, int mask_id, int verify, int* row_tok, int* row_pos, int* row_seq,
                              cudaStream_t st) {
  return launch_k(prep_block_kernel, dim3(nseq), dim3(((B + 31) / 32) * 32), 0, st, batch_slots, B, bonus, bonus_pos, drafts, mask_id, verify,
                                                            row_tok, row_pos, row_seq);
}

// Greedy acceptance for one sequence per warp.  Slot i of the block holds
// token t_i (t_0 = bonus, t_i = draft d_i); g_i = target argmax at slot i.
// d_i is accepted while d_i == g_{i-1} for all i up to it; k = accepted count.
// Emits d_1..d_k, g_k; the next bonus is g_k at position p + k + 1; rows
// 0..k become context positions p..p+k for injection, the rest are inactive.
__global__ void accept_kernel(const int* slots, int B, const int* row_tok, const int* ids, int* bonus, int* bonus_pos,
                              int* acc_out, int* n_out, int* inj_pos) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int lane = threadIdx.x;  // one warp; B <= 32
  const int s = slots[b];
  const int base = b * B;
  // lane i (1 <= i < B) checks draft d_i against g_{i-1}
  const bool mismatch = (lane >= 1 && lane < B) && (row_tok[base + lane] != ids[base + lane - 1]);
  const unsigned bad = __ballot_sync(0xffffffffu, mismatch);
  const int k = bad ? (__ffs(bad) - 2) : (B - 1);
  const int p = bonus_pos[s];
  if (lane < B) {
    int v = -1;
    if (lane < k) v = row_tok[base + lane + 1];
    else if (lane == k) v = ids[base + k];
    acc_out[b * B + lane] = v;
    inj_pos[base + lane] = (lane <= k) ? p + lane : -1;
  }
  __syncwarp();
  if (lane == 0) {
    n_out[b] = k + 1;
    bonus[s] = ids[base + k];
    bonus_pos[s] = p + k + 1;
  }
}
cudaError_t launch_accept(const int* batch_slots, int nseq, int B, const int* row_tok, const int* ids, int* bonus,
                          int* bonus_pos, int* acc_out, int* n_out, int* inj_pos, cudaStream_t st) {
  if (B > 32) return cudaErrorInvalidValue;
  return launch_k(accept_kernel, dim3(nseq), dim3(32), 0, st, batch_slots, B, row_tok, ids, bonus, bonus_pos, acc_out, n_out, inj_pos);
}

__global__ void collect_drafts_kernel(const int* ids, int B, const int* slots, int* drafts) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, i = threadIdx.x;
  if (i < B - 1) drafts[slots[b] * (B - 1) + i] = ids[b * B + 1 + i];
}
cudaError_t launch_collect_drafts(const int* ids, int nseq, int B, const int* batch_slots, int* drafts,
                                  cudaStream_t st) {
  return launch_k(collect_drafts_kernel, dim3(nseq), dim3(32), 0, st, ids, B, batch_slots, drafts);
}

__global__ void greedy_step_kernel(const int* ids, int nseq, int t, int n_new, int* out, int* row_tok, int* row_pos) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nseq) return;
  const int tok = ids[b];
  out[(size_t)b * n_new + t] = tok;
  row_tok[b] = tok;
  row_pos[b] += 1;
}
cudaError_t launch_greedy_step(const int* ids, int nseq, int t, int n_new, int* out, int* row_tok, int* row_pos,
                               cudaStream_t st) {
  return launch_k(greedy_step_kernel, dim3((nseq + 127) / 128), dim3(128), 0, st, ids, nseq, t, n_new, out, row_tok, row_pos);
}

__global__ void copy_rows_kernel(const float* src, int lds, float* dst, int ldd, int cols) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  for (int i = threadIdx.x; i < cols; i += blockDim.x) dst[(size_t)r * ldd + i] = src[(size_t)r * lds + i];
}
cudaError_t launch_copy_row_f32(const float* src, int lds, float* dst, int ldd, int rows, int cols, cudaStream_t st) {
  return launch_k(copy_rows_kernel, dim3(rows), dim3(256), 0, st, src, lds, dst, ldd, cols);
}

}  // namespace dfk
