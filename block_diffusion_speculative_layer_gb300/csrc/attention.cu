// Attention over a paged KV cache, split along the keys.
//
// Two masks share one kernel:
//   causal (target prefill / verification / greedy decode): row m at
//     position p sees cache positions [0, p]; the block's own keys were
//     written to the cache by the QKV epilogue before this runs.
//   block (drafter): row m in slot i of a block anchored at position a sees
//     the injected context [0, a) and every slot of its own block, which
//     lives in a separate row buffer, and nothing of any other block
//     (bidirectional inside the block, no flow between blocks).
//
// Keys are cut into fixed chunks of `chunk` positions counted from 0 (the
// block rows form one extra chunk).  A CTA takes one (chunk, KV head, 16-row
// query tile) and runs an online softmax for each query vector (row x
// grouped query head) with one warp per vector: lane l scores key l of a
// 32-key tile, then accumulates head dims l, l+32, ... .  Partials (max,
// sum, weighted values) are merged by a second kernel in chunk order.  A
// row's arithmetic depends only on its own position, never on how many
// rows share the pass, so verification reproduces greedy decoding bitwise.
#include "common.cuh"
#include "internal.h"

namespace dfk {

constexpr int QROWS = 16;   // query rows per CTA
constexpr int KT = 32;      // keys per inner tile
constexpr int ATT_THREADS = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Number of context keys row m sees.
__device__ __forceinline__ int ctx_len_of(const AttnParams& p, int m) {
  const int pos = p.row_pos[m];
  if (p.causal) return pos + 1;
  const int slot = m % p.rows_per_seq;
  return pos - slot;
}

template <typename T, int HD, int MAXQ>
__global__ void __launch_bounds__(ATT_THREADS) attn_partial_kernel(AttnParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int DPL = HD / 32;  // head dims per lane
  // MAXQ: query vectors per warp (16 rows x group size / 8 warps, rounded up)
  extern __shared__ float sm[];
  const int G = p.Hq / p.Hkv;
  const int nq_max = QROWS * G;
  float* qs = sm;                          // [QROWS*G][HD]
  float* ks = qs + nq_max * HD;            // [KT][HD+1]
  float* vs = ks + KT * (HD + 1);          // [KT][HD]

  const int c = blockIdx.x;
  const int h = blockIdx.y;
  const int qtiles = (p.rows_per_seq + QROWS - 1) / QROWS;
  const int z = blockIdx.z / qtiles;
  const int qt = blockIdx.z % qtiles;
  const int r0 = z * p.rows_per_seq + qt * QROWS;
  const int nrows = min(QROWS, p.rows_per_seq - qt * QROWS);
  const bool blk_chunk = (!p.causal && c == p.grid_chunks);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Key range of this chunk and the largest visible length among the rows
  // (one row per lane of the first warp).
  int key0, key1;
  __shared__ int s_max_len;
  if (warp == 0) {
    int l = 0;
    if (lane < nrows && p.row_pos[r0 + lane] >= 0) l = ctx_len_of(p, r0 + lane);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l = max(l, __shfl_xor_sync(0xffffffffu, l, o));
    if (lane == 0) s_max_len = l;
  }
  __syncthreads();
  const int max_len = s_max_len;
  if (blk_chunk) {
    key0 = 0;
    key1 = p.rows_per_seq;
  } else {
    key0 = c * p.chunk;
    key1 = min(key0 + p.chunk, max_len);
    if (key0 >= key1) return;  // no row of this tile reaches the chunk
  }

  const int nq = nrows * G;
  const size_t q_ld = (size_t)p.Hq * HD;
  for (int i = threadIdx.x; i < nq * HD; i += ATT_THREADS) {
    const int qi = i / HD, d = i % HD;
    const int r = qi / G, g = qi % G;
    const T* qp = reinterpret_cast<const T*>(p.q) + (size_t)(r0 + r) * q_ld + (size_t)(h * G + g) * HD + d;
    qs[qi * HD + d] = Cvt<T>::to_f(*qp) * p.scale_log2;
  }

  float m_i[MAXQ], l_i[MAXQ], acc[MAXQ][DPL];
#pragma unroll
  for (int j = 0; j < MAXQ; ++j) {
    m_i[j] = -INFINITY;
    l_i[j] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[j][d] = 0.f;
  }

  const T* cache = reinterpret_cast<const T*>(p.cache);
  const size_t page_elems = (size_t)2 * p.Hkv * p.page_tokens * HD;
  const int seq_slot = (p.row_seq != nullptr) ? p.row_seq[r0] : 0;

  for (int t0 = key0; t0 < key1; t0 += KT) {
    __syncthreads();
    // Stage KT keys and values of head h (fp32 in shared memory).
    for (int i = threadIdx.x; i < KT * HD; i += ATT_THREADS) {
      const int j = i / HD, d = i % HD;
      const int key = t0 + j;
      float kv = 0.f, vv = 0.f;
      if (key < key1) {
        if (blk_chunk) {
          const T* b = reinterpret_cast<const T*>(p.blk);
          const int row = z * p.rows_per_seq + key;
          kv = Cvt<T>::to_f(b[((size_t)(0 * p.Hkv + h) * p.rows_cap + row) * HD + d]);
          vv = Cvt<T>::to_f(b[((size_t)(1 * p.Hkv + h) * p.rows_cap + row) * HD + d]);
        } else {
          const int page = p.page_table[(size_t)seq_slot * p.pt_stride + key / p.page_tokens];
          if (page >= 0 && page < p.n_pages) {
            const size_t base = (size_t)page * page_elems + (size_t)(key % p.page_tokens) * HD + d;
            kv = Cvt<T>::to_f(cache[base + (size_t)(0 * p.Hkv + h) * p.page_tokens * HD]);
            vv = Cvt<T>::to_f(cache[base + (size_t)(1 * p.Hkv + h) * p.page_tokens * HD]);
          } else if (d == 0) {
            flag_error(p.err, ERR_BOUNDS);
          }
        }
      }
      ks[j * (HD + 1) + d] = kv;
      vs[j * HD + d] = vv;
    }
    __syncthreads();

#pragma unroll
    for (int j = 0; j < MAXQ; ++j) {
      const int qi = warp + j * 8;
      if (qi >= nq) break;
      const int m = r0 + qi / G;
      if (p.row_pos[m] < 0) continue;
      const int len = blk_chunk ? key1 : ctx_len_of(p, m);
      const int key = t0 + lane;
      const bool valid = key < key1 && key < len;
      float s = -INFINITY;
      if (valid) {
        const float* qv = qs + qi * HD;
        const float* kr = ks + lane * (HD + 1);
        float a = 0.f;
#pragma unroll 16
        for (int d = 0; d < HD; ++d) a = fmaf(qv[d], kr[d], a);
        s = a;
      }
      const float mt = warp_max(s);
      const float m_new = fmaxf(m_i[j], mt);
      if (m_new == -INFINITY) continue;  // nothing visible yet
      const float pr = valid ? exp2f(s - m_new) : 0.f;
      const float alpha = (m_i[j] == -INFINITY) ? 0.f : exp2f(m_i[j] - m_new);
      l_i[j] = l_i[j] * alpha + warp_sum(pr);
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[j][d] *= alpha;
      for (int kk = 0; kk < KT; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, pr, kk);
        const float* vr = vs + kk * HD + lane;
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[j][d] = fmaf(pk, vr[32 * d], acc[j][d]);
      }
      m_i[j] = m_new;
    }
  }

  // Write this chunk's partials.
  const int slot = blk_chunk ? p.n_chunk_slots - 1 : c;
#pragma unroll
  for (int j = 0; j < MAXQ; ++j) {
    const int qi = warp + j * 8;
    if (qi >= nq) break;
    const int m = r0 + qi / G;
    const int head = h * G + qi % G;
    const size_t idx = ((size_t)m * p.Hq + head) * p.n_chunk_slots + slot;
    if (lane == 0) p.part_ml[idx] = make_float2(m_i[j], l_i[j]);
#pragma unroll
    for (int d = 0; d < DPL; ++d) p.part_acc[idx * HD + lane + 32 * d] = acc[j][d];
  }
}

// Merge chunk partials in chunk order: out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
// Loads are issued eight chunks at a time; the sums still run in chunk order.
template <typename T, int HD>
__global__ void attn_combine_kernel(AttnParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int CB = 8;
  const int m = blockIdx.x, head = blockIdx.y, d = threadIdx.x;
  if (p.row_pos[m] < 0) return;
  const int len = ctx_len_of(p, m);
  const int nA = (len + p.chunk - 1) / p.chunk;
  const size_t base = ((size_t)m * p.Hq + head) * p.n_chunk_slots;
  const bool has_blk = !p.causal;
  const int nc = nA + (has_blk ? 1 : 0);  // partial c: context chunk c, or the block slot last
  auto slot = [&](int c) { return (c < nA) ? base + c : base + p.n_chunk_slots - 1; };
  float M_ = -INFINITY;
  for (int c0 = 0; c0 < nc; c0 += CB) {
    float mv[CB];
#pragma unroll
    for (int i = 0; i < CB; ++i) mv[i] = (c0 + i < nc) ? __ldcg(&p.part_ml[slot(c0 + i)].x) : -INFINITY;
#pragma unroll
    for (int i = 0; i < CB; ++i) M_ = fmaxf(M_, mv[i]);
  }
  float L = 0.f, a = 0.f;
  for (int c0 = 0; c0 < nc; c0 += CB) {
    float2 ml[CB];
    float av[CB];
#pragma unroll
    for (int i = 0; i < CB; ++i) {
      const bool ok = c0 + i < nc;
      ml[i] = ok ? __ldcg(&p.part_ml[slot(c0 + i)]) : make_float2(-INFINITY, 0.f);
      av[i] = ok ? __ldcg(&p.part_acc[slot(c0 + i) * HD + d]) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < CB; ++i) {
      if (c0 + i >= nc) break;
      const float w = (ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - M_);
      L = fmaf(ml[i].y, w, L);
      a = fmaf(av[i], w, a);
    }
  }
  T* out = reinterpret_cast<T*>(p.out);
  out[(size_t)m * p.Hq * HD + (size_t)head * HD + d] = Cvt<T>::from_f(L > 0.f ? a / L : 0.f);
}

template <typename T, int HD, int MAXQ>
static cudaError_t launch_partial(const AttnParams& p, dim3 grid, size_t smem, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<T, HD, MAXQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 112 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_k(attn_partial_kernel<T, HD, MAXQ>, grid, dim3(ATT_THREADS), smem, st, p);
}

template <typename T, int HD, int MAXQ>
static cudaError_t set_attn_attr() {
  return cudaFuncSetAttribute(attn_partial_kernel<T, HD, MAXQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              112 * 1024);
}

// Set the CUDA-core attention kernels' shared-memory limits up front (before
// any stream capture).
cudaError_t attention_prepare() {
  cudaError_t e = attention_cluster_prepare();
  if (e != cudaSuccess) return e;
  if ((e = attention_tp_prepare()) != cudaSuccess) return e;
#define DF_ATTR(T, HD, Q) \
  if ((e = set_attn_attr<T, HD, Q>()) != cudaSuccess) return e;
  DF_ATTR(float, 64, 2) DF_ATTR(float, 64, 4) DF_ATTR(float, 64, 8) DF_ATTR(float, 64, 16)
  DF_ATTR(float, 128, 2) DF_ATTR(float, 128, 4) DF_ATTR(float, 128, 8) DF_ATTR(float, 128, 16)
  DF_ATTR(__nv_bfloat16, 64, 2) DF_ATTR(__nv_bfloat16, 64, 4) DF_ATTR(__nv_bfloat16, 64, 8)
  DF_ATTR(__nv_bfloat16, 64, 16)
#undef DF_ATTR
  return e;
}

template <typename T, int HD>
static cudaError_t launch_t(const AttnParams& p, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  const size_t smem = ((size_t)QROWS * G * HD + (size_t)KT * (HD + 1) + (size_t)KT * HD) * sizeof(float);
  const int qtiles = (p.rows_per_seq + QROWS - 1) / QROWS;
  dim3 grid(p.grid_chunks + (p.causal ? 0 : 1), p.Hkv, p.n_seqs * qtiles);
  cudaError_t e;
  if (G <= 1) e = launch_partial<T, HD, 2>(p, grid, smem, st);
  else if (G <= 2) e = launch_partial<T, HD, 4>(p, grid, smem, st);
  else if (G <= 4) e = launch_partial<T, HD, 8>(p, grid, smem, st);
  else e = launch_partial<T, HD, 16>(p, grid, smem, st);
  if (e != cudaSuccess) return e;
  return launch_k(attn_combine_kernel<T, HD>, dim3(p.M, p.Hq), dim3(HD), 0, st, p);
}

static bool attn_split() {
  static const bool split = [] {
    const char* e = getenv("DF_ATTN_SPLIT");
    return e && e[0] == '1';
  }();
  return split;
}

int attention_launches(const AttnParams& p, bool bf16) {
  return (bf16 && !attn_split() && attention_cluster_fits(p)) ? 1 : 2;  // either cluster form: one kernel
}

cudaError_t launch_attention(const AttnParams& p, bool bf16, cudaStream_t st) {
  if (p.Hq % p.Hkv || p.Hq / p.Hkv > 8 || p.M != p.rows_per_seq * p.n_seqs) return cudaErrorInvalidValue;
  if (bf16 && p.hd == 128) {
    // tensor cores, chunk partials merged inside a cluster (attention_mma.cu);
    // DF_ATTN_SPLIT=1: partials to global memory and the ordered merge kernel
    // DF_ATTN_TC=1: the tcgen05 form of the cluster kernel (other rounding)
    static const bool use_tc = [] {
      const char* e = getenv("DF_ATTN_TC");
      return e && e[0] == '1';
    }();
    if (p.pipelined && !attn_split() && attention_cluster_fits(p)) return launch_attention_tp(p, st);
    if (use_tc && !attn_split() && attention_cluster_fits(p) && p.Hq / p.Hkv <= 4) return launch_attention_tc(p, st);
    if (!attn_split() && attention_cluster_fits(p)) return launch_attention_cluster(p, st);
    cudaError_t e = launch_attention_mma(p, st);
    if (e != cudaSuccess) return e;
    return launch_k(attn_combine_kernel<__nv_bfloat16, 128>, dim3(p.M, p.Hq), dim3(128), 0, st, p);
  }
  if (p.hd == 128) return bf16 ? launch_t<__nv_bfloat16, 128>(p, st) : launch_t<float, 128>(p, st);
  if (p.hd == 64) return bf16 ? launch_t<__nv_bfloat16, 64>(p, st) : launch_t<float, 64>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace dfk
