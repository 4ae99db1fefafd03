// Speculative sampling on the GPU ([ABS] 实践 4: temperature and top-p with
// the drafter and the target aligned; 核心思想 step 3: verification keeps the
// target's output distribution).
//
// The sampling distribution of a row of fp32 logits is softmax(logits / T)
// restricted to the nucleus (the fewest most probable tokens whose mass
// reaches top_p, tokens of equal logit in index order) and renormalised;
// T = 0 is the argmax (lowest index on ties).  A row is held as its logits
// plus a SampleRow (largest logit, 1/T, where the nucleus ends, kept mass):
// the mass of token i is recomputed from its logit whenever it is needed, as
// a fixed-point integer, exp((l_i - max) / T) in units of 2^-44.  Every sum,
// prefix sum and nucleus cut is then exact integer arithmetic: a row's result
// does not depend on the order of additions, the launch shape or the other
// rows of the batch.  Masses below 2^-45 of the row's largest round to zero.
//
// A draw with uniform u picks the lowest index j whose cumulative mass
// exceeds u x (total mass).  The rejection test of a drafted block keeps
// draft d_i while u_i * q_i(d_i) < p_i(d_i); at the first rejection the token
// is drawn from max(0, p_i - q_i) (from p_i if that is zero everywhere), and
// after a fully kept block from the target's distribution after the block.
//
// Uniforms are Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): uniform j of (seed, stream) is word
// j mod 4 of the block for counter (j / 4 as two 32-bit words, stream, 0) and
// key (seed as two 32-bit words), taken as (word >> 8) * 2^-24.
#include "dflash.h"
#include "internal.h"

#include <math.h>

#include <algorithm>

namespace dfk {

namespace {

constexpr uint32_t PH_M0 = 0xD2511F53u, PH_M1 = 0xCD9E8D57u;  // round multipliers
constexpr uint32_t PH_W0 = 0x9E3779B9u, PH_W1 = 0xBB67AE85u;  // key schedule increments

// A row's columns are split over a thread-block cluster of CS CTAs of SB
// threads (CTA q takes columns [V q / CS, V (q + 1) / CS)); the CTAs combine
// their maxima, sums, histograms and counts through distributed shared
// memory.  Masses are exact integers, so every result is the same for any
// split.
constexpr int SB = 256;      // threads per CTA
constexpr int SW = SB / 32;  // warps per CTA
constexpr int CS = 8;        // CTAs per row
constexpr unsigned long long WONE = 1ull << 44;   // fixed-point unit of mass
constexpr float WONE_F = 17592186044416.0f;       // 2^44
constexpr double WONE_D = 17592186044416.0;

}  // namespace

// Ten rounds of Philox4x32 on counter c with key (k0, k1), in place.
__host__ __device__ inline void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
  for (int r = 0; r < 10; ++r) {
    const uint64_t a = (uint64_t)PH_M0 * c[0];
    const uint64_t b = (uint64_t)PH_M1 * c[2];
    const uint32_t n0 = (uint32_t)(b >> 32) ^ c[1] ^ k0;
    const uint32_t n2 = (uint32_t)(a >> 32) ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = (uint32_t)b;
    c[2] = n2;
    c[3] = (uint32_t)a;
    k0 += PH_W0;
    k1 += PH_W1;
  }
}

__device__ __forceinline__ float philox_uniform(unsigned long long seed, uint32_t stream, unsigned long long j) {
  const unsigned long long blk = j >> 2;
  uint32_t c[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), stream, 0u};
  philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t w = (j & 3) == 0 ? c[0] : (j & 3) == 1 ? c[1] : (j & 3) == 2 ? c[2] : c[3];
  return (float)(w >> 8) * (1.0f / 16777216.0f);
}

namespace {

// Order key of a logit (larger logit -> larger key); -0 and +0 are one value;
// NaN orders below every number.
__device__ __forceinline__ uint32_t logit_key(float x) { return x != x ? 0u : ordered_bits(x == 0.f ? 0.f : x); }
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// exp((l - m) / T) in units of 2^-44 (l <= m).
__device__ __forceinline__ unsigned long long raw_weight(float l, float m, float inv_t) {
  return __float2ull_rn(expf((l - m) * inv_t) * WONE_F);
}

// Mass of token i (logit l) under a row's sampling distribution.
__device__ __forceinline__ unsigned long long kept_weight(const SampleRow& s, float l, int i) {
  const uint32_t k = logit_key(l);
  if (k < s.cut_key || (k == s.cut_key && i > s.cut_idx)) return 0ull;
  if (s.inv_t == 0.f) return WONE;  // greedy: the one kept token
  return raw_weight(l, s.m, s.inv_t);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, v, o);
    v = y > v ? y : v;
  }
  return v;
}
// Inclusive prefix sum over the lanes of a warp.
__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Block-wide sum / max over SB threads; every thread receives the result.
__device__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* sh) {
  v = warp_sum_u64(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < SW; ++w) t += sh[w];
  return t;
}
__device__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* sh) {
  v = warp_max_u64(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < SW; ++w) t = sh[w] > t ? sh[w] : t;
  return t;
}

// ---- the row's cluster
__device__ __forceinline__ uint32_t cs_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Barrier of the cluster's threads: shared-memory writes before it are
// visible to every CTA of the cluster after it.
__device__ __forceinline__ void cs_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The u64 at `p` in the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ unsigned long long cs_ld_u64(const unsigned long long* p, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(p), b;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(b) : "r"(a), "r"(rank));
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(b) : "memory");
  return v;
}
// Every CTA's value v, published in slot (a shared variable used for this
// step only), gathered: *before = the sum over ranks below this CTA's, the
// return value the sum (or, with take_max, the maximum) over all ranks.
__device__ unsigned long long cs_gather(unsigned long long v, unsigned long long* slot, uint32_t rank,
                                        unsigned long long* before, bool take_max = false) {
  if (threadIdx.x == 0) *slot = v;
  cs_sync();
  unsigned long long x[CS];
#pragma unroll
  for (int q = 0; q < CS; ++q) x[q] = cs_ld_u64(slot, (uint32_t)q);  // every load in flight before any is used
  unsigned long long t = 0, b = 0;
#pragma unroll
  for (int q = 0; q < CS; ++q) {
    if ((uint32_t)q < rank) b += x[q];
    t = take_max ? (x[q] > t ? x[q] : t) : t + x[q];
  }
  if (before) *before = b;
  return t;
}

// The lowest j in [lo, hi) with wfn(lo) + ... + wfn(j) > t (wfn >= 0), or -1
// if the range's total does not exceed t.  Called by every thread of the
// CTA; every thread receives the result.  Each warp sums its chunk of the
// range; the one warp whose chunk holds the crossing walks it 32 columns at a
// time.
template <typename WF>
__device__ int block_find(int lo, int hi, unsigned long long t, WF wfn, unsigned long long* sh, int* shi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = ((hi - lo + SB - 1) / SB) * 32;  // SW chunks cover the range
  const int a = lo + warp * chunk;
  const int b = min(hi, a + chunk);
  unsigned long long s = 0;
  for (int i = a + lane; i < b; i += 32) s += wfn(i);
  s = warp_sum_u64(s);
  __syncthreads();
  if (lane == 0) sh[warp] = s;
  if (threadIdx.x == 0) *shi = -1;
  __syncthreads();
  unsigned long long before = 0;
  for (int w = 0; w < warp; ++w) before += sh[w];
  if (before <= t && t - before < s) {  // warp-uniform: at most one warp enters
    unsigned long long seen = before;
    for (int base = a; base < b; base += 32) {
      const int i = base + lane;
      const unsigned long long x = warp_incl_u64(i < b ? wfn(i) : 0ull, lane);
      const unsigned hit = __ballot_sync(0xffffffffu, x > t - seen);
      if (hit) {
        if (lane == 0) *shi = base + __ffs(hit) - 1;
        break;
      }
      seen += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  __syncthreads();
  return *shi;
}

// floor(u * total), kept below total (u in [0, 1)).
__device__ __forceinline__ unsigned long long draw_target(float u, unsigned long long total) {
  double t = (double)u * (double)total;
  unsigned long long r = t > 0.0 ? (unsigned long long)t : 0ull;
  return r < total ? r : total - 1;
}

// Columns of CTA `rank` of a row's cluster.
__device__ __forceinline__ void cs_range(int V, uint32_t rank, int& lo, int& hi) {
  lo = (int)((long long)V * rank / CS);
  hi = (int)((long long)V * (rank + 1) / CS);
}

// Shared memory for a CTA's slice of a row (or of two rows): up to
// STAGE_FLOATS fp32 values each, staged once so the passes over the slice
// read shared memory; a larger slice is read from global memory instead.
constexpr int STAGE_FLOATS = 20480;  // 80 KB per row slice; V up to 8 x 20480 = 163840 is staged

// Copy columns [lo, hi) of a row into sh (every load issued before any is
// used); returns the row pointer the passes read: sh - lo, or the row itself.
__device__ __forceinline__ const float* stage_slice(const float* __restrict__ row, int lo, int hi, float* sh,
                                                    bool staged) {
  if (!staged) return row;
  for (int i = lo + (int)threadIdx.x; i < hi; i += SB) sh[i - lo] = row[i];
  __syncthreads();
  return sh - lo;
}

}  // namespace

// One cluster per row: the row's largest logit, its total mass and, for
// top_p < 1, the nucleus cut (a radix search over the logits' order keys,
// eight bits per pass, on per-digit masses; then the tied logits at the cut
// in index order).
__global__ void __launch_bounds__(SB) sample_state_kernel(const float* __restrict__ logits, long long ld, int V,
                                                          float inv_t, float top_p, SampleRow* __restrict__ out,
                                                          int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned long long hist[SW][256];     // per-warp digit masses
  __shared__ unsigned long long chist[2][256];     // this CTA's digit masses, read by the cluster (by pass parity)
  __shared__ unsigned long long red[SW];
  __shared__ unsigned long long g_max, g_w, g_ties;  // this CTA's values, read by the cluster
  __shared__ int shi;
  __shared__ uint32_t sel_digit;
  __shared__ unsigned long long sel_above;
  extern __shared__ float sl_dyn[];
  const int r = blockIdx.x / CS;  // one cluster of CS CTAs per row (a 1-D grid: rows may pass 65535)
  const uint32_t rank = cs_rank();
  int lo, hi;
  cs_range(V, rank, lo, hi);
  const float* l = stage_slice(logits + (size_t)r * ld, lo, hi, sl_dyn, (V + CS - 1) / CS <= STAGE_FLOATS);
  const int warp = threadIdx.x >> 5;

  unsigned long long best = 0;
  for (int i = lo + (int)threadIdx.x; i < hi; i += SB) {
    const unsigned long long k = ((unsigned long long)logit_key(l[i]) << 32) | (0xFFFFFFFFu - (uint32_t)i);
    best = k > best ? k : best;
  }
  best = cs_gather(block_max_u64(best, red), &g_max, rank, nullptr, true);
  const int am = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
  const float m = logits[(size_t)r * ld + am];  // may be another CTA's column: read the row itself
  SampleRow s;
  s.m = m;
  s.inv_t = inv_t;
  bool writer = rank == 0;
  if (inv_t == 0.f) {
    s.cut_key = logit_key(m);
    s.cut_idx = am;
    s.w_kept = WONE;
  } else {
    unsigned long long W = 0;
    for (int i = lo + (int)threadIdx.x; i < hi; i += SB) W += raw_weight(l[i], m, inv_t);
    W = cs_gather(block_sum_u64(W, red), &g_w, rank, nullptr);
    s.cut_key = 0;
    s.cut_idx = 0x7FFFFFFF;
    s.w_kept = W;
    if (top_p < 1.f) {
      // the nucleus: the first tokens in descending order whose mass reaches target
      unsigned long long target = (unsigned long long)ceil((double)top_p * (double)W);
      target = target < 1 ? 1 : (target > W ? W : target);
      uint32_t prefix = 0;
      unsigned long long above = 0;  // mass of the tokens ordered before the current prefix
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < SW * 256; i += SB) (&hist[0][0])[i] = 0ull;
        __syncthreads();
        unsigned long long* h = hist[warp];
        for (int i = lo + (int)threadIdx.x; i < hi; i += SB) {
          const float x = l[i];
          const uint32_t k = logit_key(x);
          if (pass > 0 && (k >> (shift + 8)) != prefix) continue;
          const unsigned long long w = raw_weight(x, m, inv_t);
          if (w) atomicAdd(h + ((k >> shift) & 255u), w);
        }
        __syncthreads();
        for (int b = threadIdx.x; b < 256; b += SB) {
          unsigned long long v = 0;
          for (int w = 0; w < SW; ++w) v += hist[w][b];
          chist[pass & 1][b] = v;
        }
        cs_sync();
        // the row's digit masses (every CTA sums the same values in the same order)
        for (int b = threadIdx.x; b < 256; b += SB) {
          unsigned long long x[CS], v = 0;
#pragma unroll
          for (int q = 0; q < CS; ++q) x[q] = cs_ld_u64(&chist[pass & 1][b], (uint32_t)q);
#pragma unroll
          for (int q = 0; q < CS; ++q) v += x[q];
          hist[0][b] = v;
        }
        __syncthreads();
        if (threadIdx.x < 32) {
          // lane j holds digits 255 - 8j down to 248 - 8j
          const int lane = threadIdx.x;
          unsigned long long b8[8], tot = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            b8[q] = hist[0][255 - 8 * lane - q];
            tot += b8[q];
          }
          const unsigned long long incl = warp_incl_u64(tot, lane);
          const unsigned hit = __ballot_sync(0xffffffffu, above + incl >= target);
          const int L = hit ? __ffs(hit) - 1 : 31;
          if (lane == L) {
            unsigned long long c = above + incl - tot;
            int qsel = 7;
            bool found = false;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (!found) {
                if (q == 7 || c + b8[q] >= target) {
                  qsel = q;
                  found = true;
                } else {
                  c += b8[q];
                }
              }
            }
            sel_digit = (uint32_t)(255 - 8 * L - qsel);
            sel_above = c;
          }
        }
        __syncthreads();
        prefix = (prefix << 8) | sel_digit;
        above = sel_above;
      }
      // prefix is the key of the cut logit; take its ties in index order
      const unsigned long long ws = raw_weight(key_logit(prefix), m, inv_t);
      if (ws == 0ull || target <= above) {
        if (rank == 0 && threadIdx.x == 0) flag_error(err, ERR_BOUNDS);
      } else {
        const unsigned long long cnt = (target - above + ws - 1) / ws;  // ties kept, in index order
        unsigned long long mine = 0, before = 0;
        for (int i = lo + (int)threadIdx.x; i < hi; i += SB) mine += logit_key(l[i]) == prefix ? 1ull : 0ull;
        mine = block_sum_u64(mine, red);
        const unsigned long long total = cs_gather(mine, &g_ties, rank, &before);
        if (total < cnt) {
          if (rank == 0 && threadIdx.x == 0) flag_error(err, ERR_BOUNDS);
        } else {
          writer = before <= cnt - 1 && cnt - 1 - before < mine;  // this CTA holds the last kept tie
          if (writer) {
            const int idx = block_find(lo, hi, cnt - 1 - before,
                                       [&](int i) { return logit_key(l[i]) == prefix ? 1ull : 0ull; }, red, &shi);
            if (idx < 0) {
              if (threadIdx.x == 0) flag_error(err, ERR_BOUNDS);
            } else {
              s.cut_key = prefix;
              s.cut_idx = idx;
              s.w_kept = above + cnt * ws;
            }
          }
        }
      }
    }
  }
  if (writer && threadIdx.x == 0) out[r] = s;
  cs_sync();  // no CTA leaves while another may still read its shared memory
}

// One cluster per row: an inverse-CDF draw.  Row r = b * rows_per_seq + i
// draws with u[b * u_ld + i - skip]; rows with i < skip draw nothing.
__global__ void __launch_bounds__(SB) sample_draw_kernel(const float* __restrict__ logits, long long ld, int V,
                                                         const SampleRow* __restrict__ st,
                                                         const float* __restrict__ u, int rows_per_seq, int u_ld,
                                                         int skip, int* __restrict__ out, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned long long red[SW];
  __shared__ unsigned long long g_sum;
  __shared__ int shi;
  const int r = blockIdx.x / CS;  // one cluster of CS CTAs per row (a 1-D grid: rows may pass 65535)
  const int b = r / rows_per_seq, i = r % rows_per_seq;
  if (i < skip) return;  // the whole cluster returns
  const uint32_t rank = cs_rank();
  int lo, hi;
  cs_range(V, rank, lo, hi);
  extern __shared__ float sl_dyn[];
  const SampleRow s = st[r];
  const float* l = stage_slice(logits + (size_t)r * ld, lo, hi, sl_dyn, (V + CS - 1) / CS <= STAGE_FLOATS);
  if (s.w_kept == 0ull) {  // the whole cluster returns
    if (rank == 0 && threadIdx.x == 0) flag_error(err, ERR_BOUNDS);
    return;
  }
  const unsigned long long t = draw_target(u[(size_t)b * u_ld + i - skip], s.w_kept);
  unsigned long long mine = 0, before = 0;
  for (int c = lo + (int)threadIdx.x; c < hi; c += SB) mine += kept_weight(s, l[c], c);
  mine = block_sum_u64(mine, red);
  const unsigned long long total = cs_gather(mine, &g_sum, rank, &before);
  if (before <= t && t - before < mine) {  // the CTA whose columns hold the draw
    const int j = block_find(lo, hi, t - before, [&](int c) { return kept_weight(s, l[c], c); }, red, &shi);
    if (threadIdx.x == 0) {
      if (j < 0) flag_error(err, ERR_BOUNDS);
      out[r] = j < 0 ? 0 : j;
    }
  } else if (rank == 0 && t >= total && threadIdx.x == 0) {
    flag_error(err, ERR_BOUNDS);
    out[r] = 0;
  }
  cs_sync();  // no CTA leaves while another may still read its shared memory
}

// probs[r][i] = the probability of token i in row r's sampling distribution.
__global__ void sample_probs_kernel(const float* __restrict__ logits, long long ld, int V, int rows,
                                    const SampleRow* __restrict__ st, float* __restrict__ probs, long long ldp) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= V) return;
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {  // rows may pass the grid's y limit
    const SampleRow s = st[r];
    const unsigned long long w = kept_weight(s, logits[(size_t)r * ld + i], i);
    probs[(size_t)r * ldp + i] = s.w_kept ? (float)((double)w / (double)s.w_kept) : 0.f;
  }
}

// Uniforms of a cycle: u[b][j] = uniform counts[slot] + j of (seed,
// streams[slot]) for j < n; then counts[slot] += n.  One block per sequence.
__global__ void cycle_uniforms_kernel(const int* __restrict__ slots, int n, unsigned long long seed,
                                      const uint32_t* __restrict__ streams, unsigned long long* counts,
                                      float* __restrict__ u, int u_ld) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int s = slots[b];
  const unsigned long long c0 = counts[s];
  const uint32_t str = streams[s];
  for (int j = threadIdx.x; j < n; j += blockDim.x) u[(size_t)b * u_ld + j] = philox_uniform(seed, str, c0 + j);
  __syncthreads();
  if (threadIdx.x == 0) counts[s] = c0 + (unsigned long long)n;
}

__global__ void philox_uniforms_kernel(unsigned long long seed, uint32_t stream, unsigned long long offset, int n,
                                       float* __restrict__ u) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < n) u[j] = philox_uniform(seed, stream, offset + (unsigned long long)j);
}

// The rejection test of one drafted block per cluster.
// Draft i (1..B-1) of sequence b is drafts[b * d_ld + i - 1], drawn from q row
// b * q_seq_rows + q_row0 + i - 1; the target's row j (0..B-1) is p row
// b * B + j.  Test i uses u[b * u_ld + u0 + i - 1], the final draw
// u[b * u_ld + u0 + B - 1].  With `bonus` given, the engine's per-sequence
// state is advanced exactly as the greedy acceptance does; with k_out given,
// k and the final token are written there.  Every CTA of the cluster runs
// the tests (they read B - 1 masses); the final draw is split over the
// cluster, and the CTA whose columns hold it writes the results.
__global__ void __launch_bounds__(SB) accept_sampled_kernel(
    const int* __restrict__ slots, int B, const int* __restrict__ drafts, int d_ld, const float* __restrict__ qlog,
    long long ldq, const SampleRow* __restrict__ qst, int q_seq_rows, int q_row0, const float* __restrict__ plog,
    long long ldp, const SampleRow* __restrict__ pst, int V, const float* __restrict__ u, int u_ld, int u0,
    int* bonus, int* bonus_pos, int* acc_out, int* n_out, int* inj_pos, int* k_out, int* tok_out, int* err) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned long long red[SW];
  __shared__ unsigned long long g_r, g_p;
  __shared__ int shi, sk, sbad;
  const int b = blockIdx.x / CS;  // one cluster of CS CTAs per sequence
  const uint32_t rank = cs_rank();
  int lo, hi;
  cs_range(V, rank, lo, hi);
  const float* ub = u + (size_t)b * u_ld + u0;
  if (threadIdx.x < 32) {
    // lane i runs test i (the tests are independent); k = the first one that rejects
    const int lane = threadIdx.x;
    bool keep = false, bad = false;
    if (lane < B - 1) {
      const int d = drafts[(size_t)b * d_ld + lane];
      bad = d < 0 || d >= V;
      if (!bad) {
        const int qr = b * q_seq_rows + q_row0 + lane, pr = b * B + lane;
        const SampleRow Q = qst[qr], P = pst[pr];
        const unsigned long long wq = kept_weight(Q, qlog[(size_t)qr * ldq + d], d);
        const unsigned long long wp = kept_weight(P, plog[(size_t)pr * ldp + d], d);
        const double q = Q.w_kept ? (double)wq / (double)Q.w_kept : 0.0;
        const double p = P.w_kept ? (double)wp / (double)P.w_kept : 0.0;
        keep = q > 0.0 && (double)ub[lane] * q < p;
      }
    }
    const unsigned stop = __ballot_sync(0xffffffffu, lane < B - 1 && (bad || !keep));
    const int k = stop ? __ffs(stop) - 1 : B - 1;
    const unsigned badm = __ballot_sync(0xffffffffu, bad);
    if (lane == 0) {
      sk = k;
      sbad = (badm >> k) & 1u;  // a draft outside the vocabulary stopped the block
    }
  }
  __syncthreads();
  const int k = sk;
  if (sbad && rank == 0 && threadIdx.x == 0) flag_error(err, ERR_BOUNDS);
  extern __shared__ float sl_dyn[];
  const bool staged = (V + CS - 1) / CS <= STAGE_FLOATS;
  const int pr = b * B + k;
  const SampleRow P = pst[pr];
  const float* pl = stage_slice(plog + (size_t)pr * ldp, lo, hi, sl_dyn, staged);
  auto pw = [&](int i) { return kept_weight(P, pl[i], i); };
  const bool rejected = k < B - 1;
  const int qr = b * q_seq_rows + q_row0 + (rejected ? k : 0);
  const SampleRow Q = qst[qr];
  const float* ql = rejected ? stage_slice(qlog + (size_t)qr * ldq, lo, hi, sl_dyn + STAGE_FLOATS, staged)
                             : qlog + (size_t)qr * ldq;
  const double ip = P.w_kept ? 1.0 / (double)P.w_kept : 0.0;
  const double iq = Q.w_kept ? 1.0 / (double)Q.w_kept : 0.0;
  auto rw = [&](int i) {
    const double x = (double)kept_weight(P, pl[i], i) * ip - (double)kept_weight(Q, ql[i], i) * iq;
    return x > 0.0 ? __double2ull_rn(x * WONE_D) : 0ull;
  };
  // this CTA's share of the residual max(0, p - q) (after a rejection) and of p
  unsigned long long r_mine = 0, p_mine = 0, r_before = 0, p_before = 0;
  for (int i = lo + (int)threadIdx.x; i < hi; i += SB) {
    if (rejected) r_mine += rw(i);
    p_mine += pw(i);
  }
  r_mine = block_sum_u64(r_mine, red);
  p_mine = block_sum_u64(p_mine, red);
  if (threadIdx.x == 0) {
    g_r = r_mine;
    g_p = p_mine;
  }
  cs_sync();
  unsigned long long R = 0, Ptot = 0, xr[CS], xp[CS];
#pragma unroll
  for (int q = 0; q < CS; ++q) {
    xr[q] = cs_ld_u64(&g_r, (uint32_t)q);
    xp[q] = cs_ld_u64(&g_p, (uint32_t)q);
  }
#pragma unroll
  for (int q = 0; q < CS; ++q) {
    if ((uint32_t)q < rank) {
      r_before += xr[q];
      p_before += xp[q];
    }
    R += xr[q];
    Ptot += xp[q];
  }
  // the final draw: from the residual after a rejection (unless it is zero
  // everywhere), else from the target's distribution after the kept drafts
  const bool from_r = rejected && R > 0ull;
  const unsigned long long total = from_r ? R : Ptot;
  const unsigned long long mine = from_r ? r_mine : p_mine, before = from_r ? r_before : p_before;
  bool writer = false;
  int tok = -1;
  if (total > 0ull) {
    const unsigned long long t = draw_target(ub[B - 1], total);
    if (before <= t && t - before < mine) {
      writer = true;
      tok = from_r ? block_find(lo, hi, t - before, rw, red, &shi) : block_find(lo, hi, t - before, pw, red, &shi);
    }
  } else {
    writer = rank == 0;
  }
  if (writer) {
    if (tok < 0) {
      if (threadIdx.x == 0) flag_error(err, ERR_BOUNDS);
      tok = 0;
    }
    if (bonus) {
      const int s = slots[b];
      const int p0 = bonus_pos[s];
      if (threadIdx.x < B) {
        const int lane = threadIdx.x;
        int v = -1;
        if (lane < k) v = drafts[(size_t)b * d_ld + lane];
        else if (lane == k) v = tok;
        acc_out[b * B + lane] = v;
        inj_pos[b * B + lane] = lane <= k ? p0 + lane : -1;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        n_out[b] = k + 1;
        bonus[s] = tok;
        bonus_pos[s] = p0 + k + 1;
      }
    }
    if (k_out && threadIdx.x == 0) {
      k_out[b] = k;
      tok_out[b] = tok;
    }
  }
  cs_sync();  // no CTA leaves while another may still read its shared memory
}

// ---- launchers

// Dynamic shared memory of a launch: `rows` row slices when a slice fits,
// else none (the kernels then read global memory).
static size_t stage_bytes(int V, int rows) {
  return (V + CS - 1) / CS <= STAGE_FLOATS ? (size_t)rows * STAGE_FLOATS * sizeof(float) : 0;
}

cudaError_t sampling_prepare() {
  const int one = STAGE_FLOATS * (int)sizeof(float), two = 2 * one;
  cudaError_t e = cudaFuncSetAttribute(sample_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, one);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(sample_draw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, one);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(accept_sampled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, two);
  return e;
}

cudaError_t launch_sample_state(const float* logits, long long ld, int rows, int V, float inv_t, float top_p,
                                SampleRow* st, int* err, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (V < 1 || V > SAMPLE_MAX_VOCAB) return cudaErrorInvalidValue;
  if ((long long)rows * CS > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  return launch_kcl(sample_state_kernel, dim3(CS * rows), dim3(SB), stage_bytes(V, 1), s, dim3(CS, 1, 1), logits, ld, V,
                    inv_t, top_p, st, err);
}

cudaError_t launch_sample_draw(const float* logits, long long ld, int rows, int V, const SampleRow* st, const float* u,
                               int rows_per_seq, int u_ld, int skip, int* out, int* err, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (V < 1 || V > SAMPLE_MAX_VOCAB || rows_per_seq < 1) return cudaErrorInvalidValue;
  if ((long long)rows * CS > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  return launch_kcl(sample_draw_kernel, dim3(CS * rows), dim3(SB), stage_bytes(V, 1), s, dim3(CS, 1, 1), logits, ld, V,
                    st, u, rows_per_seq, u_ld, skip, out, err);
}

cudaError_t launch_sample_probs(const float* logits, long long ld, int rows, int V, const SampleRow* st, float* probs,
                                long long ldp, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  return launch_k(sample_probs_kernel, dim3((V + 255) / 256, std::min(rows, 65535)), dim3(256), 0, s, logits, ld, V, rows,
                  st, probs, ldp);
}

cudaError_t launch_cycle_uniforms(const int* slots, int nseq, int n, unsigned long long seed, const uint32_t* streams,
                                  unsigned long long* counts, float* u, int u_ld, cudaStream_t s) {
  if (nseq <= 0 || n <= 0) return cudaSuccess;
  return launch_k(cycle_uniforms_kernel, dim3(nseq), dim3(64), 0, s, slots, n, seed, streams, counts, u, u_ld);
}

cudaError_t launch_accept_sampled(const int* slots, int nseq, int B, const int* drafts, int d_ld, const float* qlog,
                                  long long ldq, const SampleRow* qst, int q_seq_rows, int q_row0, const float* plog,
                                  long long ldp, const SampleRow* pst, int V, const float* u, int u_ld, int u0,
                                  int* bonus, int* bonus_pos, int* acc_out, int* n_out, int* inj_pos, int* k_out,
                                  int* tok_out, int* err, cudaStream_t s) {
  if (nseq <= 0) return cudaSuccess;
  if (B < 1 || B > 32 || V < 1 || V > SAMPLE_MAX_VOCAB) return cudaErrorInvalidValue;
  if ((long long)nseq * CS > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  return launch_kcl(accept_sampled_kernel, dim3(CS * nseq), dim3(SB), stage_bytes(V, 2), s, dim3(CS, 1, 1), slots, B,
                    drafts, d_ld,
                    qlog, ldq, qst, q_seq_rows, q_row0, plog, ldp, pst, V, u, u_ld, u0, bonus, bonus_pos, acc_out, n_out,
                    inj_pos, k_out, tok_out, err);
}

bool sampling_args_ok(float temperature, float top_p) {
  if (!(temperature == 0.f || (temperature >= SAMPLE_MIN_TEMPERATURE && temperature <= SAMPLE_MAX_TEMPERATURE)))
    return false;
  return top_p >= 0.f && top_p <= 1.f;
}
float sampling_inv_t(float temperature) { return temperature == 0.f ? 0.f : 1.0f / temperature; }

}  // namespace dfk

using namespace dfk;

namespace {

// Sampling rows of a temporary SampleRow array on `st` (freed on the stream).
struct RowStates {
  SampleRow* p = nullptr;
  cudaStream_t st;
  explicit RowStates(cudaStream_t s) : st(s) {}
  bool alloc(size_t n) { return cudaMallocAsync(reinterpret_cast<void**>(&p), std::max<size_t>(n, 1) * sizeof(SampleRow), st) == cudaSuccess; }
  ~RowStates() {
    if (p) cudaFreeAsync(p, st);
  }
};

}  // namespace

extern "C" {

df_status df_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  if (!ctr || !key || !out) return DF_EINVAL;
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  philox4x32_10(c, key[0], key[1]);
  for (int i = 0; i < 4; ++i) out[i] = c[i];
  return DF_OK;
}

df_status df_op_philox_uniforms(uint64_t seed, uint32_t stream_id, uint64_t offset, int32_t n, float* u_dev,
                                void* stream) {
  if (n < 0 || (n > 0 && !u_dev)) return DF_EINVAL;
  if (n == 0) return DF_OK;
  philox_uniforms_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(seed, stream_id, offset,
                                                                                            n, u_dev);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ECUDA;
}

df_status df_op_sampling_probs(const float* logits_dev, int32_t rows, int32_t V, float temperature, float top_p,
                               float* probs_dev, int32_t* err_dev, void* stream) {
  if (rows < 0 || V < 1 || V > SAMPLE_MAX_VOCAB || !sampling_args_ok(temperature, top_p)) return DF_EINVAL;
  if (rows == 0) return DF_OK;
  if (!logits_dev || !probs_dev) return DF_EINVAL;
  if (sampling_prepare() != cudaSuccess) return DF_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  RowStates rs(st);
  if (!rs.alloc(rows)) return DF_ENOMEM;
  cudaError_t r = launch_sample_state(logits_dev, V, rows, V, sampling_inv_t(temperature), top_p, rs.p, err_dev, st);
  if (r == cudaSuccess) r = launch_sample_probs(logits_dev, V, rows, V, rs.p, probs_dev, V, st);
  return r == cudaSuccess ? DF_OK : DF_ECUDA;
}

df_status df_op_sample_draw(const float* logits_dev, int32_t rows, int32_t V, float temperature, float top_p,
                            const float* u_dev, int32_t* idx_dev, int32_t* err_dev, void* stream) {
  if (rows < 0 || V < 1 || V > SAMPLE_MAX_VOCAB || !sampling_args_ok(temperature, top_p)) return DF_EINVAL;
  if (rows == 0) return DF_OK;
  if (!logits_dev || !u_dev || !idx_dev) return DF_EINVAL;
  if (sampling_prepare() != cudaSuccess) return DF_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  RowStates rs(st);
  if (!rs.alloc(rows)) return DF_ENOMEM;
  cudaError_t r = launch_sample_state(logits_dev, V, rows, V, sampling_inv_t(temperature), top_p, rs.p, err_dev, st);
  if (r == cudaSuccess) r = launch_sample_draw(logits_dev, V, rows, V, rs.p, u_dev, 1, 1, 0, idx_dev, err_dev, st);
  return r == cudaSuccess ? DF_OK : DF_ECUDA;
}

df_status df_op_accept_sampled(const int32_t* drafts_dev, const float* q_logits_dev, const float* p_logits_dev,
                               int32_t nseq, int32_t B, int32_t V, float temperature, float top_p,
                               const float* u_dev, int32_t* k_dev, int32_t* tok_dev, int32_t* err_dev,
                               void* stream) {
  if (nseq < 0 || B < 2 || B > 32 || V < 1 || V > SAMPLE_MAX_VOCAB || !sampling_args_ok(temperature, top_p))
    return DF_EINVAL;
  if (nseq == 0) return DF_OK;
  if (!drafts_dev || !q_logits_dev || !p_logits_dev || !u_dev || !k_dev || !tok_dev) return DF_EINVAL;
  if (sampling_prepare() != cudaSuccess) return DF_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int qrows = nseq * (B - 1), prows = nseq * B;
  RowStates qs(st), ps(st);
  if (!qs.alloc(qrows) || !ps.alloc(prows)) return DF_ENOMEM;
  const float inv_t = sampling_inv_t(temperature);
  cudaError_t r = launch_sample_state(q_logits_dev, V, qrows, V, inv_t, top_p, qs.p, err_dev, st);
  if (r == cudaSuccess) r = launch_sample_state(p_logits_dev, V, prows, V, inv_t, top_p, ps.p, err_dev, st);
  if (r == cudaSuccess)
    r = launch_accept_sampled(nullptr, nseq, B, drafts_dev, B - 1, q_logits_dev, V, qs.p, B - 1, 0, p_logits_dev, V,
                              ps.p, V, u_dev, B, 0, nullptr, nullptr, nullptr, nullptr, nullptr, k_dev, tok_dev, err_dev,
                              st);
  return r == cudaSuccess ? DF_OK : DF_ECUDA;
}

}  // extern "C"
