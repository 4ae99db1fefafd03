// bf16 attention over the paged caches on the tensor cores (mma.sync m16n8k16).
//
// attn_cl_kernel (the engine's kernel; below): fixed 64-key chunks counted
// from position 0, the drafter's block rows as one extra chunk, chunk
// partials merged inside a thread-block cluster.
// attn_mma_kernel: the same chunks with partials to global memory, merged in
// chunk order by attn_combine (DF_ATTN_SPLIT=1, and shapes the cluster kernel
// does not take).  Either way a row's result does not depend on the other
// rows, so verification and greedy decoding give bitwise the same rows.
//
// One CTA = one (chunk, KV head, 16-token tile); one warp per grouped query
// head, so a warp's 16 token rows form exactly one m16 tile.  The chunk's keys
// and values (64 x 128 bf16 each) are staged with 16-byte cp.async into shared
// memory with the 16-byte column blocks XOR-swizzled by key (conflict-free
// ldmatrix).  S = Q K^T (64 MMAs per warp), masked softmax statistics per row
// (quad shuffles), P kept in registers as the A operand of P V (64 MMAs), fp32
// accumulators.  A row's arithmetic never depends on the other rows.
#include <cuda.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

namespace dfk {

constexpr int MC = 64;         // keys per chunk (the engine's chunk)
constexpr int MHD = 128;       // head dim
constexpr int ROWB = MHD * 2;  // bytes per key row in shared memory

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// 2^x on the special-function unit (ex2.approx, flush to zero): 2^-inf = +0,
// so masked scores need no branch.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Lazy rescale threshold (log2 units): a chunk whose largest scaled score
// exceeds the running maximum by at most this keeps the maximum (its
// probabilities may reach 2^8), so the running output is rescaled only when
// a much larger score appears.  The decision depends on the row alone.
constexpr float ATT_RESCALE = 8.f;

// Byte offset of (key, 16-byte column block) in a swizzled [MC][MHD] tile.
__device__ __forceinline__ uint32_t swz(int key, int blk) { return (uint32_t)(key * ROWB + ((blk ^ (key & 7)) << 4)); }

__device__ __forceinline__ int ctx_len_rows(const AttnParams& p, int m) {
  const int pos = p.row_pos[m];
  return p.causal ? pos + 1 : pos - (m % p.rows_per_seq);
}

__global__ void __launch_bounds__(256) attn_mma_kernel(AttnParams p) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(128) uint8_t sK[MC * ROWB];
  __shared__ __align__(128) uint8_t sV[MC * ROWB];
  const int G = p.Hq / p.Hkv;
  const int c = blockIdx.x;
  const int h = blockIdx.y;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  const int z = blockIdx.z / qtiles;
  const int qt = blockIdx.z % qtiles;
  const int r0 = z * p.rows_per_seq + qt * 16;
  const int nrows = min(16, p.rows_per_seq - qt * 16);
  const bool blk_chunk = (!p.causal && c == p.grid_chunks);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  // the tile's longest visible length: one row per lane of the first warp
  __shared__ int s_max_len;
  if (warp == 0) {
    int l = 0;
    if (lane < nrows && p.row_pos[r0 + lane] >= 0) l = ctx_len_rows(p, r0 + lane);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l = max(l, __shfl_xor_sync(0xffffffffu, l, o));
    if (lane == 0) s_max_len = l;
  }
  __syncthreads();
  const int max_len = s_max_len;
  int key0, nkeys;
  if (blk_chunk) {
    key0 = 0;
    nkeys = p.rows_per_seq;
  } else {
    key0 = c * MC;
    nkeys = min(MC, max_len - key0);
    if (nkeys <= 0) return;  // no row of this tile reaches the chunk
  }

  // ---- stage keys and values (16-byte pieces, swizzled); keys past nkeys are zero
  const __nv_bfloat16* cache = reinterpret_cast<const __nv_bfloat16*>(p.cache);
  const __nv_bfloat16* blk = reinterpret_cast<const __nv_bfloat16*>(p.blk);
  const size_t page_elems = (size_t)2 * p.Hkv * p.page_tokens * MHD;
  const int seq_slot = p.row_seq[r0];
  // The chunk's page ids, one per key, looked up in parallel first so the
  // copies below never wait on a dependent load.
  __shared__ int s_page[MC];
  if (!blk_chunk && threadIdx.x < MC) {
    const int kabs = key0 + threadIdx.x;
    s_page[threadIdx.x] =
        (threadIdx.x < nkeys) ? p.page_table[(size_t)seq_slot * p.pt_stride + kabs / p.page_tokens] : -1;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < MC * (MHD / 8); idx += blockDim.x) {
    const int key = idx >> 4, b = idx & 15;
    bool ok = key < nkeys;
    const __nv_bfloat16 *srck = nullptr, *srcv = nullptr;
    if (ok) {
      if (blk_chunk) {
        const int row = z * p.rows_per_seq + key;
        srck = blk + ((size_t)(0 * p.Hkv + h) * p.rows_cap + row) * MHD + b * 8;
        srcv = blk + ((size_t)(1 * p.Hkv + h) * p.rows_cap + row) * MHD + b * 8;
      } else {
        const int kabs = key0 + key;
        const int page = s_page[key];
        if (page >= 0 && page < p.n_pages) {
          const size_t base = (size_t)page * page_elems + (size_t)(kabs % p.page_tokens) * MHD + b * 8;
          srck = cache + base + (size_t)(0 * p.Hkv + h) * p.page_tokens * MHD;
          srcv = cache + base + (size_t)(1 * p.Hkv + h) * p.page_tokens * MHD;
        } else {
          ok = false;
          if (b == 0) flag_error(p.err, ERR_BOUNDS);
        }
      }
    }
    if (ok) {
      cp_async16(smem_addr(sK) + swz(key, b), srck);
      cp_async16(smem_addr(sV) + swz(key, b), srcv);
    } else {
      *reinterpret_cast<uint4*>(sK + swz(key, b)) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sV + swz(key, b)) = make_uint4(0, 0, 0, 0);
    }
  }

  // ---- this warp's query head and its 16 rows (A fragments straight from global)
  const bool active = warp < G;
  const int head = h * G + warp;
  uint32_t qa[8][4];
  int len_lo = -1, len_hi = -1;  // visible keys of rows gid and gid + 8 (-1: inactive row)
  if (active) {
    const size_t q_ld = (size_t)p.Hq * MHD;
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
    const int rlo = gid, rhi = gid + 8;
    const bool vlo = rlo < nrows && p.row_pos[r0 + rlo] >= 0;
    const bool vhi = rhi < nrows && p.row_pos[r0 + rhi] >= 0;
    if (vlo) len_lo = blk_chunk ? p.rows_per_seq : ctx_len_rows(p, r0 + rlo);
    if (vhi) len_hi = blk_chunk ? p.rows_per_seq : ctx_len_rows(p, r0 + rhi);
    const size_t base_lo = ((size_t)(r0 + rlo) * q_ld + (size_t)head * MHD) / 2;
    const size_t base_hi = ((size_t)(r0 + rhi) * q_ld + (size_t)head * MHD) / 2;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d0 = ks * 16 + tig * 2;
      qa[ks][0] = vlo ? q32[base_lo + d0 / 2] : 0u;
      qa[ks][1] = vhi ? q32[base_hi + d0 / 2] : 0u;
      qa[ks][2] = vlo ? q32[base_lo + (d0 + 8) / 2] : 0u;
      qa[ks][3] = vhi ? q32[base_hi + (d0 + 8) / 2] : 0u;
    }
  }
  cp_async_wait_all();
  __syncthreads();
  if (!active) return;

  // ---- S = Q K^T for 64 keys: 8 n-tiles of 8 keys
  float s[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
  const uint32_t kbase = smem_addr(sK);
  const int lq = lane >> 3, lr = lane & 7;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {  // two k-steps (32 dims) per ldmatrix.x4
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbase + swz(nt * 8 + lr, kp * 4 + lq), b0, b1, b2, b3);
      mma_16816(s[nt], qa[2 * kp], b0, b1);
      mma_16816(s[nt], qa[2 * kp + 1], b2, b3);
    }
  }

  // ---- masked statistics per row (log2 domain)
  float mlo = -INFINITY, mhi = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int kabs = key0 + nt * 8 + tig * 2 + e;
      const float vlo = s[nt][e] * p.scale_log2, vhi = s[nt][2 + e] * p.scale_log2;
      s[nt][e] = (kabs < len_lo) ? vlo : -INFINITY;
      s[nt][2 + e] = (kabs < len_hi) ? vhi : -INFINITY;
      mlo = fmaxf(mlo, s[nt][e]);
      mhi = fmaxf(mhi, s[nt][2 + e]);
    }
  }
  mlo = fmaxf(mlo, __shfl_xor_sync(0xffffffffu, mlo, 1));
  mlo = fmaxf(mlo, __shfl_xor_sync(0xffffffffu, mlo, 2));
  mhi = fmaxf(mhi, __shfl_xor_sync(0xffffffffu, mhi, 1));
  mhi = fmaxf(mhi, __shfl_xor_sync(0xffffffffu, mhi, 2));
  float llo = 0.f, lhi = 0.f;
  uint32_t pa[4][4];  // P as A fragments, 4 k-steps of 16 keys
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const float p0 = (s[nt][0] == -INFINITY) ? 0.f : exp2f(s[nt][0] - mlo);
    const float p1 = (s[nt][1] == -INFINITY) ? 0.f : exp2f(s[nt][1] - mlo);
    const float p2 = (s[nt][2] == -INFINITY) ? 0.f : exp2f(s[nt][2] - mhi);
    const float p3 = (s[nt][3] == -INFINITY) ? 0.f : exp2f(s[nt][3] - mhi);
    llo += p0 + p1;
    lhi += p2 + p3;
    const int kk = nt >> 1;
    if ((nt & 1) == 0) {
      pa[kk][0] = pack_bf16(p0, p1);
      pa[kk][1] = pack_bf16(p2, p3);
    } else {
      pa[kk][2] = pack_bf16(p0, p1);
      pa[kk][3] = pack_bf16(p2, p3);
    }
  }
  llo += __shfl_xor_sync(0xffffffffu, llo, 1);
  llo += __shfl_xor_sync(0xffffffffu, llo, 2);
  lhi += __shfl_xor_sync(0xffffffffu, lhi, 1);
  lhi += __shfl_xor_sync(0xffffffffu, lhi, 2);

  // ---- O = P V: 16 n-tiles of 8 dims, 4 k-steps of 16 keys
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  const uint32_t vbase = smem_addr(sV);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
    for (int np = 0; np < 8; ++np) {  // two n-tiles (16 dims) per ldmatrix.x4.trans
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vbase + swz(kk * 16 + (lq & 1) * 8 + lr, np * 2 + (lq >> 1)), b0, b1, b2, b3);
      mma_16816(o[2 * np], pa[kk], b0, b1);
      mma_16816(o[2 * np + 1], pa[kk], b2, b3);
    }
  }

  // ---- partials of this chunk
  const int slot = blk_chunk ? p.n_chunk_slots - 1 : c;
#pragma unroll
  for (int hl = 0; hl < 2; ++hl) {
    const int rr = gid + hl * 8;
    if (rr >= nrows || (hl ? len_hi : len_lo) < 0) continue;
    const int m = r0 + rr;
    const size_t idx = ((size_t)m * p.Hq + head) * p.n_chunk_slots + slot;
    if (tig == 0) p.part_ml[idx] = make_float2(hl ? mhi : mlo, hl ? lhi : llo);
    float* dst = p.part_acc + idx * MHD;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<float2*>(dst + nt * 8 + tig * 2) = make_float2(o[nt][2 * hl], o[nt][2 * hl + 1]);
  }
}

cudaError_t launch_attention_mma(const AttnParams& p, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  if (p.hd != MHD || p.chunk != MC || G > 8) return cudaErrorInvalidValue;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  dim3 grid(p.grid_chunks + (p.causal ? 0 : 1), p.Hkv, p.n_seqs * qtiles);
  const int threads = ((G * 32 + 127) / 128) * 128;  // at least 128 threads stage the chunk
  return launch_k(attn_mma_kernel, grid, dim3(threads), 0, st, p);
}

// ---------------------------------------------------------------------------
// Cluster variant: partials merged inside the kernel.
//
// A cluster of CLA CTAs (16 where the device can place such clusters, else 8)
// covers one (KV head, 16-token tile).  CTA rank j takes the 64-key context
// chunks c = j, j + CLA, j + 2*CLA, ... (the drafter's block rows, as one more
// chunk, go to rank CLA-1 after its context chunks) and runs an online softmax
// over them.  The chunks' pages come by TMA into CL_NST shared-memory stages,
// so the next chunks' keys and values load while one is computed.  Each CTA
// owns a share of the (head, row) pairs: every CTA writes its partial of a pair
// (running max, sum, unnormalised output) into the owner's receive region
// through distributed shared memory and arrives on the owner's barrier, and
// the owner merges the CLA partials in rank order from its own shared memory.
//
// A row's arithmetic depends only on its own visible length: which CTA takes a
// chunk depends on the chunk index alone, chunks that a row cannot see leave
// its state bit-for-bit unchanged, and the merge order is fixed, so a row gets
// the same bits whatever the other rows of its tile or batch.
constexpr int MAXPG = 2048;                 // page ids a CTA stages for its chunks
constexpr int CL_NST = 2;                   // key/value stages in flight (two CTAs fit on an SM)
// One stage: keys then values, each [2 halves of the head dim][64 keys][128 B]
// in the 128-byte swizzle (16-byte piece b of a row at b ^ (key & 7)).
constexpr int CL_HALF = MC * 128;
constexpr int CL_STAGE = 2 * 2 * CL_HALF;
constexpr unsigned long long CL_WAIT_NS = 2000000000ull;

__host__ __device__ constexpr int cl_pg_off(int G) { return (void)G, CL_NST * CL_STAGE; }
// Receive region of the merge: one region per cluster rank, holding that
// rank's slots of the (query head, token row) pairs this CTA owns, CL_RSLOT
// floats each (the partial output's 128 dims, then the running maximum and
// sum).  A rank stages its own slots of all pairs over the stage buffers.
constexpr int CL_RSLOT = MHD + 4;
__host__ __device__ constexpr int cl_rb_off(int G) { return cl_pg_off(G) + MAXPG * 4; }
__host__ __device__ constexpr int cl_smem_bytes(int G) { return cl_rb_off(G) + G * 16 * CL_RSLOT * 4 + 1024; }
static_assert(8 * 16 * CL_RSLOT * 4 <= cl_rb_off(8), "the partials' staging area ends before the receive area");
static_assert((CL_RSLOT * 4) % 16 == 0 && cl_rb_off(8) % 16 == 0, "bulk copies move whole 16-byte units");

// Byte offset of (key, 16-byte piece b of the 256-byte row) in a stage's key or value tile.
__device__ __forceinline__ uint32_t swz2(int key, int b) {
  return (uint32_t)((b >> 3) * CL_HALF + key * 128 + (((b & 7) ^ (key & 7)) << 4));
}
__device__ __forceinline__ void cl_mbar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cl_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cl_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool cl_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a stage barrier; false (error word set) after about two seconds.
__device__ __noinline__ bool cl_wait_bar(uint32_t bar, uint32_t parity, int* err) {
  if (cl_try_wait(bar, parity)) return true;
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (cl_try_wait(bar, parity)) return true;
    if ((it & 1023u) == 0) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > CL_WAIT_NS) break;
    }
  }
  flag_error(err, ERR_TIMEOUT);
  return false;
}
// One page-half (page_tokens keys x 64 head dims = page_tokens x 128 B) of
// cache slab `slab` = (page * 2 + k|v) * Hkv + head into shared memory.
__device__ __forceinline__ void tma_kv(uint32_t dst, const CUtensorMap* map, uint32_t bar, int half, int slab) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(half), "r"(0), "r"(slab)
      : "memory");
}

__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
// Arrive without ordering this thread's earlier memory operations: for an
// arrival that publishes no data (barrier initialisation is published by
// fence.mbarrier_init), or that follows reads whose values are already used.
// Every thread of the CTA takes the same form: the arrivals of one warp are
// never split between the two.
__device__ __forceinline__ void cl_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 cl_ld2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 cl_ld4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory into another CTA's; the bytes complete that CTA's
// mbarrier at `rbar` (complete-tx).
__device__ __forceinline__ void cl_bulk_push(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t rbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(src), "r"(bytes), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ bool cl_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (acquire at cluster scope) for arrivals from other CTAs of the cluster.
__device__ __noinline__ bool cl_wait_bar_cluster(uint32_t bar, uint32_t parity, int* err) {
  if (cl_try_wait_cluster(bar, parity)) return true;
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (cl_try_wait_cluster(bar, parity)) return true;
    if ((it & 1023u) == 0) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > CL_WAIT_NS) break;
    }
  }
  flag_error(err, ERR_TIMEOUT);
  return false;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// NW warps (one per query head of a group, at least four); two four-warp CTAs
// fit on an SM next to their shared memory.
template <int CLA, int NW>
__device__ __forceinline__ void attn_cl_body(const AttnParams& p, const CUtensorMap& kvmap) {
  // The GEMM before this kernel triggers it only after its own wait (see
  // gemm_tc.cu), so everything older than that GEMM is complete here: the row
  // metadata, the page table and the cache entries of earlier positions are
  // read before the wait; the queries, this pass's keys and values and the
  // drafter's block rows after it.
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smc_raw[];
  // 1024-byte aligned: the TMA's 128-byte swizzle repeats every 1024 bytes
  uint8_t* smc = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smc_raw) + 1023) & ~uintptr_t(1023));
  const int G = p.Hq / p.Hkv;
  const int j = (int)cl_rank();
  const int h = blockIdx.y;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  const int z = blockIdx.z / qtiles;
  const int qt = blockIdx.z % qtiles;
  const int r0 = z * p.rows_per_seq + qt * 16;
  const int nrows = min(16, p.rows_per_seq - qt * 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const bool causal = p.causal != 0;

  // ---- the tile's rows: visible context length (-1: no position), longest
  __shared__ int s_len[16];
  __shared__ int s_first_new;  // cache positions from here on are written by this pass
  if (threadIdx.x < 16) {
    int l = -1;
    if ((int)threadIdx.x < nrows && p.row_pos[r0 + threadIdx.x] >= 0) l = ctx_len_rows(p, r0 + threadIdx.x);
    s_len[threadIdx.x] = l;
  }
  if (threadIdx.x == 32) {
    const int f = p.row_pos[z * p.rows_per_seq];
    s_first_new = causal ? (f >= 0 ? f : 0) : 0x7fffffff;
  }
  const int ppc = MC / p.page_tokens;
  // ---- page ids of this CTA's chunks (every chunk the longest row could need)
  int* s_pg = reinterpret_cast<int*>(smc + cl_pg_off(G));
  const int seq_slot = p.row_seq[r0];
  const int cap_chunks = (p.grid_chunks > j) ? (p.grid_chunks - j + CLA - 1) / CLA : 0;
  for (int t = threadIdx.x; t < cap_chunks * ppc && t < MAXPG; t += blockDim.x) {
    const int pg = (j + CLA * (t / ppc)) * ppc + t % ppc;  // page of the sequence
    s_pg[t] = pg < p.pt_stride ? p.page_table[(size_t)seq_slot * p.pt_stride + pg] : -1;
  }
  __syncthreads();
  int max_len = 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) max_len = max(max_len, s_len[r]);
  const int first_new = s_first_new;
  const int nA = (max_len + MC - 1) / MC;                       // context chunks of the tile
  const int nmine = nA > j ? (nA - j + CLA - 1) / CLA : 0;       // this CTA's context chunks
  const bool has_blk = !causal && j == CLA - 1;
  const int nsteps = nmine + (has_blk ? 1 : 0);

  const __nv_bfloat16* blk = reinterpret_cast<const __nv_bfloat16*>(p.blk);
  const int PT = p.page_tokens;
  __shared__ __align__(8) uint64_t s_full[CL_NST];
  __shared__ __align__(8) uint64_t s_merge;  // complete once every partial of this rank's pairs is here
  __shared__ int s_failed;
  if (threadIdx.x == 0) {
    for (int b2 = 0; b2 < CL_NST; ++b2) cl_mbar_init(smem_addr(&s_full[b2]));
    cl_mbar_init(smem_addr(&s_merge));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the merge barrier's one arrival, with the bytes the holding ranks send
    // here: per pair of this rank, one slot (output row, maximum and sum)
    const int held = min(nA, CLA) + ((!causal && nA < CLA) ? 1 : 0);
    cl_arrive_expect_tx(smem_addr(&s_merge), (uint32_t)(held * (G * 16 / CLA) * CL_RSLOT * 4));
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kvmap)) : "memory");
    s_failed = 0;
  }
  __syncthreads();
  // every rank's merge barrier is initialised before any rank sends into it
  // (the matching wait comes after the chunks).  The arrival is relaxed: the
  // initialisation is published by its fence, and the barrier's own arrival
  // (with the expected bytes) keeps its phase open even if a copy's bytes
  // land first (the transaction count may go below zero meanwhile).  A
  // release arrival here cost about 1.2 us at batch 1.
  cl_arrive_relaxed();
  // Stage step st into buffer buf: part 1 = the pages wholly before first_new
  // (written by earlier passes), 2 = the rest, 3 = all.  Context chunks come
  // by TMA, one 2 KB box per (page, k|v, half row), issued by thread 0; the
  // drafter's block rows by 16-byte cp.async from every thread.  Part 2 (or
  // 3) makes the stage barrier's one arrival.
  auto stage = [&](int st, int buf, int part) {
    uint8_t* sK = smc + buf * CL_STAGE;
    uint8_t* sV = sK + 2 * CL_HALF;
    const uint32_t bar = smem_addr(&s_full[buf]);
    if (st >= nmine) {  // block chunk
      if (!(part & 2)) return;
      for (int idx = threadIdx.x; idx < MC * (MHD / 8); idx += blockDim.x) {
        const int key = idx >> 4, b = idx & 15;
        if (key < p.rows_per_seq) {
          const int row = z * p.rows_per_seq + key;
          cp_async16(smem_addr(sK) + swz2(key, b), blk + ((size_t)(0 * p.Hkv + h) * p.rows_cap + row) * MHD + b * 8);
          cp_async16(smem_addr(sV) + swz2(key, b), blk + ((size_t)(1 * p.Hkv + h) * p.rows_cap + row) * MHD + b * 8);
        } else {
          *reinterpret_cast<uint4*>(sK + swz2(key, b)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(sV + swz2(key, b)) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_commit();
      if (threadIdx.x == 0) cl_arrive_expect_tx(bar, 0);
      return;
    }
    // warp 0: lane 0 keeps the barrier's byte count, lane 4 * pg + 2 * kv + half
    // issues the box of (page pg, k|v, half) itself, so the chunk's boxes go out
    // in parallel rather than one after another from a single thread
    if (threadIdx.x >= 32) return;
    const int ln = threadIdx.x;
    const int key0 = (j + CLA * st) * MC;
    const int npg = (min(MC, max_len - key0) + PT - 1) / PT;  // pages holding a key the tile can see
    auto wanted = [&](int pg) {
      const bool old = key0 + (pg + 1) * PT <= first_new;
      const int page = s_pg[st * ppc + pg];
      return ((old ? 1 : 2) & part) && page >= 0 && page < p.n_pages;
    };
    if (ln == 0) {
      uint32_t bytes = 0;
      for (int pg = 0; pg < npg; ++pg)
        if (wanted(pg)) bytes += 4u * (uint32_t)PT * 128u;
      if (part == 1) {
        if (bytes) cl_expect_tx(bar, bytes);
      } else {
        cl_arrive_expect_tx(bar, bytes);
      }
    }
    const int pg = ln >> 2, kv = (ln >> 1) & 1, half = ln & 1;
    if (pg < npg && wanted(pg)) {
      const int page = s_pg[st * ppc + pg];
      tma_kv(smem_addr((kv ? sV : sK) + half * CL_HALF + pg * PT * 128), &kvmap, bar, half,
             (page * 2 + kv) * p.Hkv + h);
    }
  };
  // Keys and values the staged pages do not cover (past the tile's longest
  // row, or in a page the table does not hold) read as zeros.
  auto fixup = [&](int st, int buf) {
    if (st >= nmine) return;
    uint8_t* sK = smc + buf * CL_STAGE;
    uint8_t* sV = sK + 2 * CL_HALF;
    const int key0 = (j + CLA * st) * MC;
    const int nkeys = min(MC, max_len - key0);
    if (nkeys == MC) {  // a full chunk whose pages are all in the table needs nothing (the usual case)
      bool all = true;
      for (int pg = 0; pg < ppc; ++pg) {
        const int page = s_pg[st * ppc + pg];
        all = all && page >= 0 && page < p.n_pages;
      }
      if (all) return;
    }
    for (int idx = threadIdx.x; idx < MC * (MHD / 8); idx += blockDim.x) {
      const int key = idx >> 4, b = idx & 15;
      const int page = s_pg[st * ppc + key / PT];
      const bool have = key < nkeys && page >= 0 && page < p.n_pages;
      if (!have) {
        if (key < nkeys && b == 0 && (key % PT) == 0) flag_error(p.err, ERR_BOUNDS);
        *reinterpret_cast<uint4*>(sK + swz2(key, b)) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sV + swz2(key, b)) = make_uint4(0, 0, 0, 0);
      }
    }
  };
  // the first stages' earlier-position pages go out before the wait
  for (int st = 0; st < CL_NST && st < nsteps; ++st) stage(st, st, 1);

  pdl_wait();
  // the rest of the first stages (the pages this pass wrote), ahead of the queries
  for (int st = 0; st < CL_NST && st < nsteps; ++st) stage(st, st, 2);
  // ---- this warp's query head and its 16 rows (A fragments straight from global)
  const bool active = warp < G;
  const int head = h * G + warp;
  uint32_t qa[8][4];
  const int len_lo = s_len[gid], len_hi = s_len[gid + 8];
  if (active) {
    const size_t q_ld = (size_t)p.Hq * MHD;
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
    const bool vlo = len_lo >= 0, vhi = len_hi >= 0;
    const size_t base_lo = ((size_t)(r0 + gid) * q_ld + (size_t)head * MHD) / 2;
    const size_t base_hi = ((size_t)(r0 + gid + 8) * q_ld + (size_t)head * MHD) / 2;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d0 = ks * 16 + tig * 2;
      qa[ks][0] = vlo ? q32[base_lo + d0 / 2] : 0u;
      qa[ks][1] = vhi ? q32[base_hi + d0 / 2] : 0u;
      qa[ks][2] = vlo ? q32[base_lo + (d0 + 8) / 2] : 0u;
      qa[ks][3] = vhi ? q32[base_hi + (d0 + 8) / 2] : 0u;
    }
  }

  // ---- online softmax over this CTA's chunks
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  const int lq = lane >> 3, lr = lane & 7;
  int done = 0;  // steps consumed
  for (int st = 0; st < nsteps; ++st) {
    const int buf = st % CL_NST;
    if (st >= nmine) cp_async_wait_0();  // the block rows (this thread's copies)
    if (!cl_try_wait(smem_addr(&s_full[buf]), (uint32_t)(st / CL_NST) & 1u) &&
        !cl_wait_bar(smem_addr(&s_full[buf]), (uint32_t)(st / CL_NST) & 1u, p.err))
      s_failed = 1;
    fixup(st, buf);
    __syncthreads();
    if (s_failed) break;
    done = st + 1;
    if (active) {
      const bool is_blk = st >= nmine;
      const int key0 = is_blk ? 0 : (j + CLA * st) * MC;
      // visible keys of the two rows in this chunk's numbering
      const int vis_lo = len_lo < 0 ? 0 : (is_blk ? p.rows_per_seq : len_lo - key0);
      const int vis_hi = len_hi < 0 ? 0 : (is_blk ? p.rows_per_seq : len_hi - key0);
      const uint32_t kbase = smem_addr(smc + buf * CL_STAGE);
      const uint32_t vbase = kbase + 2 * CL_HALF;
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + swz2(nt * 8 + lr, kp * 4 + lq), b0, b1, b2, b3);
          mma_16816(s[nt], qa[2 * kp], b0, b1);
          mma_16816(s[nt], qa[2 * kp + 1], b2, b3);
        }
      }
      if (vis_lo < MC || vis_hi < MC) {  // keys a row cannot see score -inf (full chunks skip this)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kk = nt * 8 + tig * 2 + e;
            if (kk >= vis_lo) s[nt][e] = -INFINITY;
            if (kk >= vis_hi) s[nt][2 + e] = -INFINITY;
          }
        }
      }
      // raw row maxima (two chains per row), then over the quad, scaled once (scale > 0)
      float ma_lo = fmaxf(s[0][0], s[0][1]), mb_lo = fmaxf(s[1][0], s[1][1]);
      float ma_hi = fmaxf(s[0][2], s[0][3]), mb_hi = fmaxf(s[1][2], s[1][3]);
#pragma unroll
      for (int nt = 2; nt < 8; nt += 2) {
        ma_lo = fmaxf(ma_lo, fmaxf(s[nt][0], s[nt][1]));
        mb_lo = fmaxf(mb_lo, fmaxf(s[nt + 1][0], s[nt + 1][1]));
        ma_hi = fmaxf(ma_hi, fmaxf(s[nt][2], s[nt][3]));
        mb_hi = fmaxf(mb_hi, fmaxf(s[nt + 1][2], s[nt + 1][3]));
      }
      float mc_lo = fmaxf(ma_lo, mb_lo), mc_hi = fmaxf(ma_hi, mb_hi);
      mc_lo = fmaxf(mc_lo, __shfl_xor_sync(0xffffffffu, mc_lo, 1));
      mc_lo = fmaxf(mc_lo, __shfl_xor_sync(0xffffffffu, mc_lo, 2));
      mc_hi = fmaxf(mc_hi, __shfl_xor_sync(0xffffffffu, mc_hi, 1));
      mc_hi = fmaxf(mc_hi, __shfl_xor_sync(0xffffffffu, mc_hi, 2));
      mc_lo *= p.scale_log2;
      mc_hi *= p.scale_log2;
      // lazy rescale: the running maximum moves only for a much larger score
      const bool rs_lo = mc_lo > m_lo + ATT_RESCALE, rs_hi = mc_hi > m_hi + ATT_RESCALE;
      const float mn_lo = rs_lo ? mc_lo : m_lo, mn_hi = rs_hi ? mc_hi : m_hi;
      const float a_lo = rs_lo ? ex2_fast(m_lo - mn_lo) : 1.f;  // 0 for a row's first visible chunk
      const float a_hi = rs_hi ? ex2_fast(m_hi - mn_hi) : 1.f;
      const float ng_lo = (mn_lo == -INFINITY) ? 0.f : -mn_lo, ng_hi = (mn_hi == -INFINITY) ? 0.f : -mn_hi;
      float cs_lo = 0.f, cs_hi = 0.f, cs2_lo = 0.f, cs2_hi = 0.f;
      uint32_t pa[4][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        // P = 2^(s * scale - m): one FFMA and one ex2 per score (2^-inf = 0)
        const float p0 = ex2_fast(fmaf(s[nt][0], p.scale_log2, ng_lo));
        const float p1 = ex2_fast(fmaf(s[nt][1], p.scale_log2, ng_lo));
        const float p2 = ex2_fast(fmaf(s[nt][2], p.scale_log2, ng_hi));
        const float p3 = ex2_fast(fmaf(s[nt][3], p.scale_log2, ng_hi));
        if (nt & 1) {
          cs2_lo += p0 + p1;
          cs2_hi += p2 + p3;
        } else {
          cs_lo += p0 + p1;
          cs_hi += p2 + p3;
        }
        const int kk = nt >> 1;
        if ((nt & 1) == 0) {
          pa[kk][0] = pack_bf16(p0, p1);
          pa[kk][1] = pack_bf16(p2, p3);
        } else {
          pa[kk][2] = pack_bf16(p0, p1);
          pa[kk][3] = pack_bf16(p2, p3);
        }
      }
      cs_lo += cs2_lo;
      cs_hi += cs2_hi;
      cs_lo += __shfl_xor_sync(0xffffffffu, cs_lo, 1);
      cs_lo += __shfl_xor_sync(0xffffffffu, cs_lo, 2);
      cs_hi += __shfl_xor_sync(0xffffffffu, cs_hi, 1);
      cs_hi += __shfl_xor_sync(0xffffffffu, cs_hi, 2);
      l_lo = l_lo * a_lo + cs_lo;
      l_hi = l_hi * a_hi + cs_hi;
      m_lo = mn_lo;
      m_hi = mn_hi;
      if (__any_sync(0xffffffffu, rs_lo || rs_hi)) {  // rows that keep their scale multiply by exactly 1
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          o[nt][0] *= a_lo;
          o[nt][1] *= a_lo;
          o[nt][2] *= a_hi;
          o[nt][3] *= a_hi;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + swz2(kk * 16 + (lq & 1) * 8 + lr, np * 2 + (lq >> 1)), b0, b1, b2, b3);
          mma_16816(o[2 * np], pa[kk], b0, b1);
          mma_16816(o[2 * np + 1], pa[kk], b2, b3);
        }
      }
    }
    __syncthreads();  // this buffer is refilled now, for CL_NST steps on
    if (st + CL_NST < nsteps) stage(st + CL_NST, buf, 3);
  }
  if (s_failed && threadIdx.x == 0) {
    // leave no copy in flight: wait (bounded) for the stages issued but not consumed
    for (int st = done; st < nsteps && st < done + CL_NST; ++st)
      if (st < nmine) cl_wait_bar(smem_addr(&s_full[st % CL_NST]), (uint32_t)(st / CL_NST) & 1u, p.err);
  }
  cp_async_wait_0();
  __syncthreads();

  // ---- the merge.  Pair pp = (query head g, token row r) = g * 16 + r belongs to
  // rank pp / (pairs / CLA).  Every rank leaves its partial of each pair
  // (output, running maximum and sum) in slot pp of a local staging area over
  // the stage buffers, so the pairs of one owner are consecutive slots, and
  // sends each owner its slots with one bulk copy into region j of the
  // owner's receive area; the copies' bytes complete the owner's merge
  // barrier.  Each rank waits for its own barrier and merges its pairs from
  // local shared memory.  A copy reads its source until the destination's
  // barrier completes, so every rank arrives on a cluster barrier once its own
  // merge barrier has completed and waits on it before it leaves.
  const int pairs = G * 16;
  const int per_owner = pairs / CLA;  // G * 16 is a multiple of 16, CLA divides 16
  const uint32_t rb_s = smem_addr(smc + cl_rb_off(G));
  // ranks without a chunk of this tile hold (-inf, 0, 0): their terms are
  // exactly zero, so they are neither sent nor read
  const bool held_me = j < nA || (!causal && j == CLA - 1);
  if (active && held_me) {
    float* stg = reinterpret_cast<float*>(smc);
#pragma unroll
    for (int hl = 0; hl < 2; ++hl) {
      float* slot = stg + (size_t)(warp * 16 + gid + hl * 8) * CL_RSLOT;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2*>(slot + nt * 8 + tig * 2) = make_float2(o[nt][2 * hl], o[nt][2 * hl + 1]);
      if (tig == 0) *reinterpret_cast<float2*>(slot + MHD) = make_float2(hl ? m_hi : m_lo, hl ? l_hi : l_lo);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes, read by the bulk copies
  __syncthreads();
  cl_wait();  // the merge barriers are initialised
  if (held_me && (int)threadIdx.x < CLA) {
    const uint32_t q = threadIdx.x, bytes = (uint32_t)(per_owner * CL_RSLOT * 4);
    cl_bulk_push(cl_map(rb_s + (uint32_t)j * bytes, q), smem_addr(smc) + q * bytes, bytes,
                 cl_map(smem_addr(&s_merge), q));
  }
  const bool merged_in = cl_wait_bar_cluster(smem_addr(&s_merge), 0u, p.err);
  cl_arrive_relaxed();  // every copy into this rank has landed

  // ---- merge this rank's pairs, 32 threads x 4 dims per pair, ranks in order
  for (int lp = warp; merged_in && lp < per_owner; lp += blockDim.x >> 5) {
    const int pp = j * per_owner + lp;
    const int g = pp >> 4, rr = pp & 15;
    if (rr >= nrows || s_len[rr] < 0) continue;
    const float* slot0 = reinterpret_cast<const float*>(smc + cl_rb_off(G)) + (size_t)lp * CL_RSLOT;
    float2 ml[CLA];
    float4 av[CLA];
#pragma unroll
    for (int i = 0; i < CLA; ++i) {
      const bool held = i < nA || (!causal && i == CLA - 1);
      const float* sl = slot0 + (size_t)i * per_owner * CL_RSLOT;
      ml[i] = held ? *reinterpret_cast<const float2*>(sl + MHD) : make_float2(-INFINITY, 0.f);
      av[i] = held ? *reinterpret_cast<const float4*>(sl + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < CLA; ++i) Mx = fmaxf(Mx, ml[i].x);
    float L = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < CLA; ++i) {
      const float w = (ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - Mx);
      L = fmaf(ml[i].y, w, L);
      a.x = fmaf(av[i].x, w, a.x);
      a.y = fmaf(av[i].y, w, a.y);
      a.z = fmaf(av[i].z, w, a.z);
      a.w = fmaf(av[i].w, w, a.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)(r0 + rr) * p.Hq * MHD +
                         (size_t)(h * G + g) * MHD + lane * 4;
    uint2 packed;
    packed.x = pack_bf16(a.x * inv, a.y * inv);
    packed.y = pack_bf16(a.z * inv, a.w * inv);
    *reinterpret_cast<uint2*>(out) = packed;
  }
  cl_wait();  // and every copy out of it has landed
}

template <int CLA, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 4 ? 2 : 1)
    attn_cl_kernel(AttnParams p, const __grid_constant__ CUtensorMap kvmap) {
  trace_entry(p.trace);
  attn_cl_body<CLA, NW>(p, kvmap);
  trace_exit(p.trace);
}


// ---------------------------------------------------------------------------
// tcgen05 form of the cluster attention (DF_ATTN_TC=1, groups of at most four
// query heads).  Same chunks, staging and cluster merge as attn_cl_kernel;
// per chunk, S = Q K^T (M = 128 rows: query head g x token row r at row
// g * 16 + r, rows past 16 G zero; N = 64 keys) and O += P V (V read as an
// MN-major operand) run on tcgen05 with accumulators in tensor memory, and
// thread t runs the softmax of row t.  In this form each chunk is serial
// (S, softmax, O rescale, P V) with one CTA per SM, which measured 2.6-3x
// slower than attn_cl_kernel, so it is not the default.
constexpr int TC_QHALF = 128 * 128;          // one 64-dim half of the 128-row Q tile
constexpr int TC_QOFF = 2 * CL_STAGE;         // after the two key/value stages
constexpr int TC_POFF = TC_QOFF + 2 * TC_QHALF;
constexpr int TC_PGOFF = TC_POFF + 128 * 128;
constexpr int TC_SMEM = TC_PGOFF + MAXPG * 4 + 1024;
constexpr int TC_OLD = 132;                   // row stride (floats) of the partials left for the merge
constexpr uint32_t TC_IDESC_S = (1u << 4) | (1u << 7) | (1u << 10) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t TC_IDESC_PV =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
static_assert(4 * 16 * TC_OLD * 4 + 4 * 16 * 8 <= 2 * CL_STAGE, "partials fit over the stages");

// Shared-memory descriptor, 128-byte swizzle: 8-row groups 1024 bytes apart;
// lbo: K-major 16 (unused), MN-major the byte stride between 64-element column blocks.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];" : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]) : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]) : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])) : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <int CLA>
__global__ void __launch_bounds__(128, 1) attn_tc_kernel(AttnParams p, const __grid_constant__ CUtensorMap kvmap) {
  // The GEMM before this kernel triggers it only after its own wait (see
  // gemm_tc.cu), so everything older than that GEMM is complete here: the row
  // metadata, the page table and the cache entries of earlier positions are
  // read before the wait; the queries, this pass's keys and values and the
  // drafter's block rows after it.
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smc_raw[];
  // 1024-byte aligned: the TMA's 128-byte swizzle repeats every 1024 bytes
  uint8_t* smc = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smc_raw) + 1023) & ~uintptr_t(1023));
  const int G = p.Hq / p.Hkv;
  const int j = (int)cl_rank();
  const int h = blockIdx.y;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  const int z = blockIdx.z / qtiles;
  const int qt = blockIdx.z % qtiles;
  const int r0 = z * p.rows_per_seq + qt * 16;
  const int nrows = min(16, p.rows_per_seq - qt * 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool causal = p.causal != 0;

  // ---- the tile's rows: visible context length (-1: no position), longest
  __shared__ int s_len[16];
  __shared__ int s_first_new;  // cache positions from here on are written by this pass
  if (threadIdx.x < 16) {
    int l = -1;
    if ((int)threadIdx.x < nrows && p.row_pos[r0 + threadIdx.x] >= 0) l = ctx_len_rows(p, r0 + threadIdx.x);
    s_len[threadIdx.x] = l;
  }
  if (threadIdx.x == 32) {
    const int f = p.row_pos[z * p.rows_per_seq];
    s_first_new = causal ? (f >= 0 ? f : 0) : 0x7fffffff;
  }
  const int ppc = MC / p.page_tokens;
  // ---- page ids of this CTA's chunks (every chunk the longest row could need)
  int* s_pg = reinterpret_cast<int*>(smc + TC_PGOFF);
  const int seq_slot = p.row_seq[r0];
  const int cap_chunks = (p.grid_chunks > j) ? (p.grid_chunks - j + CLA - 1) / CLA : 0;
  for (int t = threadIdx.x; t < cap_chunks * ppc && t < MAXPG; t += blockDim.x) {
    const int pg = (j + CLA * (t / ppc)) * ppc + t % ppc;  // page of the sequence
    s_pg[t] = pg < p.pt_stride ? p.page_table[(size_t)seq_slot * p.pt_stride + pg] : -1;
  }
  __syncthreads();
  int max_len = 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) max_len = max(max_len, s_len[r]);
  const int first_new = s_first_new;
  const int nA = (max_len + MC - 1) / MC;                       // context chunks of the tile
  const int nmine = nA > j ? (nA - j + CLA - 1) / CLA : 0;       // this CTA's context chunks
  const bool has_blk = !causal && j == CLA - 1;
  const int nsteps = nmine + (has_blk ? 1 : 0);

  const __nv_bfloat16* blk = reinterpret_cast<const __nv_bfloat16*>(p.blk);
  const int PT = p.page_tokens;
  __shared__ __align__(8) uint64_t s_full[CL_NST];
  __shared__ int s_failed;
  __shared__ __align__(8) uint64_t s_mma[2];  // 0: S complete, 1: P V complete
  __shared__ uint32_t s_tmem;
  if (threadIdx.x == 0) {
    cl_mbar_init(smem_addr(&s_mma[0]));
    cl_mbar_init(smem_addr(&s_mma[1]));
    for (int b2 = 0; b2 < CL_NST; ++b2) cl_mbar_init(smem_addr(&s_full[b2]));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kvmap)) : "memory");
    s_failed = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_addr(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;                    // columns [0, 64): S; [64, 192): O
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t bar_s = smem_addr(&s_mma[0]), bar_o = smem_addr(&s_mma[1]);
  // Stage step st into buffer buf: part 1 = the pages wholly before first_new
  // (written by earlier passes), 2 = the rest, 3 = all.  Context chunks come
  // by TMA, one 2 KB box per (page, k|v, half row), issued by thread 0; the
  // drafter's block rows by 16-byte cp.async from every thread.  Part 2 (or
  // 3) makes the stage barrier's one arrival.
  auto stage = [&](int st, int buf, int part) {
    uint8_t* sK = smc + buf * CL_STAGE;
    uint8_t* sV = sK + 2 * CL_HALF;
    const uint32_t bar = smem_addr(&s_full[buf]);
    if (st >= nmine) {  // block chunk
      if (!(part & 2)) return;
      for (int idx = threadIdx.x; idx < MC * (MHD / 8); idx += blockDim.x) {
        const int key = idx >> 4, b = idx & 15;
        if (key < p.rows_per_seq) {
          const int row = z * p.rows_per_seq + key;
          cp_async16(smem_addr(sK) + swz2(key, b), blk + ((size_t)(0 * p.Hkv + h) * p.rows_cap + row) * MHD + b * 8);
          cp_async16(smem_addr(sV) + swz2(key, b), blk + ((size_t)(1 * p.Hkv + h) * p.rows_cap + row) * MHD + b * 8);
        } else {
          *reinterpret_cast<uint4*>(sK + swz2(key, b)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(sV + swz2(key, b)) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_commit();
      if (threadIdx.x == 0) cl_arrive_expect_tx(bar, 0);
      return;
    }
    // warp 0: lane 0 keeps the barrier's byte count, lane 4 * pg + 2 * kv + half
    // issues the box of (page pg, k|v, half) itself, so the chunk's boxes go out
    // in parallel rather than one after another from a single thread
    if (threadIdx.x >= 32) return;
    const int ln = threadIdx.x;
    const int key0 = (j + CLA * st) * MC;
    const int npg = (min(MC, max_len - key0) + PT - 1) / PT;  // pages holding a key the tile can see
    auto wanted = [&](int pg) {
      const bool old = key0 + (pg + 1) * PT <= first_new;
      const int page = s_pg[st * ppc + pg];
      return ((old ? 1 : 2) & part) && page >= 0 && page < p.n_pages;
    };
    if (ln == 0) {
      uint32_t bytes = 0;
      for (int pg = 0; pg < npg; ++pg)
        if (wanted(pg)) bytes += 4u * (uint32_t)PT * 128u;
      if (part == 1) {
        if (bytes) cl_expect_tx(bar, bytes);
      } else {
        cl_arrive_expect_tx(bar, bytes);
      }
    }
    const int pg = ln >> 2, kv = (ln >> 1) & 1, half = ln & 1;
    if (pg < npg && wanted(pg)) {
      const int page = s_pg[st * ppc + pg];
      tma_kv(smem_addr((kv ? sV : sK) + half * CL_HALF + pg * PT * 128), &kvmap, bar, half,
             (page * 2 + kv) * p.Hkv + h);
    }
  };
  // Keys and values the staged pages do not cover (past the tile's longest
  // row, or in a page the table does not hold) read as zeros.
  auto fixup = [&](int st, int buf) {
    if (st >= nmine) return;
    uint8_t* sK = smc + buf * CL_STAGE;
    uint8_t* sV = sK + 2 * CL_HALF;
    const int key0 = (j + CLA * st) * MC;
    const int nkeys = min(MC, max_len - key0);
    for (int idx = threadIdx.x; idx < MC * (MHD / 8); idx += blockDim.x) {
      const int key = idx >> 4, b = idx & 15;
      const int page = s_pg[st * ppc + key / PT];
      const bool have = key < nkeys && page >= 0 && page < p.n_pages;
      if (!have) {
        if (key < nkeys && b == 0 && (key % PT) == 0) flag_error(p.err, ERR_BOUNDS);
        *reinterpret_cast<uint4*>(sK + swz2(key, b)) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sV + swz2(key, b)) = make_uint4(0, 0, 0, 0);
      }
    }
  };
  // the first stages' earlier-position pages go out before the wait
  for (int st = 0; st < CL_NST && st < nsteps; ++st) stage(st, st, 1);

  pdl_wait();
  // ---- Q as the A operand of S = Q K^T: 128 rows (g * 16 + r = query head g,
  // token row r; rows past 16 G read as zeros), two 64-dim halves, 128-byte swizzle
  uint8_t* sQ = smc + TC_QOFF;
  for (int idx = threadIdx.x; idx < 128 * 16; idx += blockDim.x) {
    const int row = idx >> 4, c = idx & 15;
    const int g = row >> 4, r = row & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (g < G && r < nrows && s_len[r] >= 0)
      v = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + (size_t)(r0 + r) * p.Hq * MHD +
                                          (size_t)(h * G + g) * MHD + c * 8);
    *reinterpret_cast<uint4*>(sQ + (c >> 3) * TC_QHALF + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = v;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  // the rest of the first stages
  for (int st = 0; st < CL_NST && st < nsteps; ++st) stage(st, st, 2);

  // ---- online softmax over this CTA's chunks: thread t owns row t
  const int trow = threadIdx.x, tg = trow >> 4, tr = trow & 15;
  const bool row_ok = tg < G && tr < nrows && s_len[tr] >= 0;
  float m_run = -INFINITY, l_run = 0.f;
  bool pv_issued = false;
  uint32_t ph_s = 0, ph_o = 0;
  const uint32_t qbase = smem_addr(sQ), pbase = smem_addr(smc + TC_POFF);
  int done = 0;  // steps consumed
  for (int st = 0; st < nsteps; ++st) {
    const int buf = st % CL_NST;
    if (st >= nmine) cp_async_wait_0();  // the block rows (this thread's copies)
    if (!cl_wait_bar(smem_addr(&s_full[buf]), (uint32_t)(st / CL_NST) & 1u, p.err)) s_failed = 1;
    fixup(st, buf);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // zero rows and block rows: generic writes
    __syncthreads();
    if (s_failed) break;
    done = st + 1;
    {
      const bool is_blk = st >= nmine;
      const int key0 = is_blk ? 0 : (j + CLA * st) * MC;
      const uint32_t kbase = smem_addr(smc + buf * CL_STAGE);
      const uint32_t vbase = kbase + 2 * CL_HALF;
      // S = Q K^T: M 128 rows, N 64 keys, K 128 dims, into TMEM columns [0, 64)
      if (threadIdx.x == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tmem, tc_desc(qbase + (kk >> 2) * TC_QHALF + (kk & 3) * 32, 16),
                 tc_desc(kbase + (kk >> 2) * CL_HALF + (kk & 3) * 32, 16), TC_IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(bar_s);
      }
      if (!cl_wait_bar(bar_s, ph_s, p.err)) s_failed = 1;
      ph_s ^= 1u;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      float sv[64];
      tc_ld64(tmem + lane_base, sv);
      const int vis = !row_ok ? 0 : (is_blk ? p.rows_per_seq : s_len[tr] - key0);
      float mc = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < 64; ++kk) {
        sv[kk] = (kk < vis) ? sv[kk] * p.scale_log2 : -INFINITY;
        mc = fmaxf(mc, sv[kk]);
      }
      const float mn = fmaxf(m_run, mc);
      const float alpha = (mn == -INFINITY) ? 1.f : exp2f(m_run - mn);
      float cs = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int kk = 0; kk < 64; kk += 2) {
        const float e0 = (sv[kk] == -INFINITY) ? 0.f : exp2f(sv[kk] - mn);
        const float e1 = (sv[kk + 1] == -INFINITY) ? 0.f : exp2f(sv[kk + 1] - mn);
        cs += e0 + e1;
        pk[kk >> 1] = pack_bf16(e0, e1);
      }
      l_run = l_run * alpha + cs;
      m_run = mn;
      // O rows rescaled in tensor memory (the previous P V finished at the end of
      // its step); the loads and stores are warp-wide, rows that keep their
      // scale multiply by exactly 1
      if (__any_sync(0xffffffffu, pv_issued && alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float ov[32];
          tc_ld32(tmem + lane_base + 64u + 32u * c, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= alpha;
          tc_st32(tmem + lane_base + 64u + 32u * c, ov);
        }
      }
      // P row t (64 keys, 128 bytes) as the A operand of P V, 128-byte swizzle
      uint8_t* sP = smc + TC_POFF;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sP + trow * 128 + ((c ^ (trow & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncthreads();
      // O += P V: M 128 rows, N 128 dims (V read MN-major), K 64 keys, into TMEM columns [64, 192)
      if (threadIdx.x == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma(tmem + 64u, tc_desc(pbase + kk * 32, 16), tc_desc(vbase + kk * 2048, CL_HALF), TC_IDESC_PV,
                 (pv_issued || kk > 0) ? 1u : 0u);
        tc_commit(bar_o);
      }
      pv_issued = true;
      if (!cl_wait_bar(bar_o, ph_o, p.err)) s_failed = 1;   // V's stage is refilled below
      ph_o ^= 1u;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    __syncthreads();  // this buffer is refilled now, for CL_NST steps on
    if (st + CL_NST < nsteps) stage(st + CL_NST, buf, 3);
  }
  if (s_failed && threadIdx.x == 0) {
    // leave no copy in flight: wait (bounded) for the stages issued but not consumed
    for (int st = done; st < nsteps && st < done + CL_NST; ++st)
      if (st < nmine) cl_wait_bar(smem_addr(&s_full[st % CL_NST]), (uint32_t)(st / CL_NST) & 1u, p.err);
  }
  cp_async_wait_0();
  __syncthreads();

  // ---- leave the partial in shared memory (over the stage buffers)
  float* sO = reinterpret_cast<float*>(smc);
  float2* sML = reinterpret_cast<float2*>(smc + G * 16 * TC_OLD * 4);
  // (pv_issued is uniform over the CTA, so every warp takes part in the
  // warp-wide loads; only rows of real query heads are stored)
  float* dst = sO + (size_t)(tg * 16 + tr) * TC_OLD;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float ov[32];
    if (pv_issued) {
      tc_ld32(tmem + lane_base + 64u + 32u * c, ov);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) ov[i] = 0.f;
    }
    if (tg < G) {
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + 32 * c + i) = make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]);
    }
  }
  if (tg < G) sML[tg * 16 + tr] = make_float2(m_run, l_run);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
  }
  cl_arrive();
  cl_wait();

  // ---- merge: this CTA's share of the (head, row) pairs, 32 threads x 4 dims per pair
  const int pairs = G * 16;
  const int p0 = j * pairs / CLA, p1 = (j + 1) * pairs / CLA;
  const uint32_t sO_s = smem_addr(sO), sML_s = smem_addr(sML);
  for (int pp = p0 + warp; pp < p1; pp += blockDim.x >> 5) {
    const int g = pp >> 4, rr = pp & 15;
    if (rr >= nrows || s_len[rr] < 0) continue;
    float2 ml[CLA];
    float4 av[CLA];
    // ranks without a chunk of this tile hold (-inf, 0, 0): their terms are
    // exactly zero, so they are not read
#pragma unroll
    for (int i = 0; i < CLA; ++i) {
      const bool held = i < nA || (!causal && i == CLA - 1);
      ml[i] = held ? cl_ld2(cl_map(sML_s + (uint32_t)(g * 16 + rr) * 8u, (uint32_t)i)) : make_float2(-INFINITY, 0.f);
      av[i] = held ? cl_ld4(cl_map(sO_s + (uint32_t)((g * 16 + rr) * TC_OLD + lane * 4) * 4u, (uint32_t)i))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < CLA; ++i) Mx = fmaxf(Mx, ml[i].x);
    float L = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < CLA; ++i) {
      const float w = (ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - Mx);
      L = fmaf(ml[i].y, w, L);
      a.x = fmaf(av[i].x, w, a.x);
      a.y = fmaf(av[i].y, w, a.y);
      a.z = fmaf(av[i].z, w, a.z);
      a.w = fmaf(av[i].w, w, a.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)(r0 + rr) * p.Hq * MHD +
                         (size_t)(h * G + g) * MHD + lane * 4;
    uint2 packed;
    packed.x = pack_bf16(a.x * inv, a.y * inv);
    packed.y = pack_bf16(a.z * inv, a.w * inv);
    *reinterpret_cast<uint2*>(out) = packed;
  }
  cl_arrive_relaxed();  // this CTA's reads of the other partials are done
  cl_wait();    // and nobody leaves while another CTA may still read its partial
}


// ---------------------------------------------------------------------------
// Pipelined tcgen05 attention (attn_tp_kernel): the chunks, staging and
// cluster merge of attn_cl_kernel, with the per-chunk arithmetic on tcgen05
// and the chunks in flight at once.  Warp roles in a CTA of six warps:
//   warps 0-3  softmax: thread t owns tensor-memory lane t, i.e. MMA row t.
//              Query head g, token row r sits at row (g & 3) * 32 + (g >> 2) * 16
//              + r, so each warp holds the rows of one or two heads;
//   warps 4, 6 producers: the chunks' key pages (warp 4) and value pages
//              (warp 6) by TMA into TP_NST stages, each with its own
//              barriers (the drafter's block rows by cp.async);
//   warp 5     MMA issuer (one thread) and tensor-memory owner.
// Per chunk i, the issuer computes S_i = Q K_i^T (M 128 rows, N 64 keys) into
// one of two tensor-memory buffers, then O += P_i V_i once the softmax has
// written P_i; S_{i+2} is issued right after P_i V_i, so the softmax of chunk
// i+1 overlaps the tensor cores' work on chunks i and i+2.  A key tile is
// released when S_i has read it and a value tile when P_i V_i has, so each
// load has about TP_NST chunks' time to land.  The running maximum
// is updated lazily: a chunk whose maximum exceeds it by at most 2^8 keeps it
// (P values up to 256), otherwise O is rescaled in tensor memory once P_{i-1}
// V_{i-1} has finished.  Every decision depends on the row's own scores only,
// and rows that keep their scale multiply by exactly 1, so a row's bits do not
// depend on the other rows of its tile or batch.
constexpr int TP_NST = 4;                          // key/value stages
constexpr int TP_QOFF = TP_NST * CL_STAGE;         // Q tile: two 64-dim halves x 128 rows x 128 B
constexpr int TP_POFF = TP_QOFF + 2 * TC_QHALF;    // P tiles: two buffers x 128 rows x 128 B
constexpr int TP_PGOFF = TP_POFF + 2 * 128 * 128;  // page ids of the CTA's chunks
constexpr int TP_SMEM = TP_PGOFF + MAXPG * 4 + 1024;
constexpr int TP_THREADS = 256;
constexpr float TP_RESCALE = ATT_RESCALE;          // lazy rescale threshold (log2 units)
static_assert(8 * 16 * TC_OLD * 4 + 8 * 16 * 8 <= TP_NST * CL_STAGE, "partials fit over the stages");
static_assert(TP_SMEM <= 227 * 1024, "shared memory of one CTA");

__device__ __forceinline__ void tp_mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void tp_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// A bounded wait whose outcome is the same for every lane of the warp (the
// warp-collective tensor-memory loads after it need all 32 lanes).
// One test inline first: in the pipelined kernel most waits find the phase
// already complete, and the bounded loop is an out-of-line call.
__device__ __forceinline__ bool cl_wait_fast(uint32_t bar, uint32_t parity, int* err) {
  return cl_try_wait(bar, parity) || cl_wait_bar(bar, parity, err);
}
__device__ __forceinline__ bool tp_wait_warp(uint32_t bar, uint32_t parity, int* err) {
  return __all_sync(0xffffffffu, cl_wait_fast(bar, parity, err)) != 0;
}

// DUP (groups of at most four query heads): the 64 real rows of the 128-row
// tile are each held twice, in tensor-memory lanes w*32 + r and w*32 + 16 + r
// of softmax warp w (head w, token row r); the two threads of a row take its
// keys 0..31 and 32..63 and meet through one shuffle for the maximum and the
// sum, so every lane of a softmax warp does useful work.  Otherwise rows
// (g & 3) * 32 + (g >> 2) * 16 + r hold head g, one thread per row.
template <int CLA, bool DUP>
__device__ __forceinline__ void attn_tp_body(const AttnParams& p, const CUtensorMap& kvmap) {
  // Everything older than the key/value GEMM before this kernel is complete
  // here (that GEMM triggers only after its own wait): the row metadata, the
  // page table and older cache entries are read before the wait; the
  // queries, this pass's keys and values and the block rows after it.
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smc_raw[];
  uint8_t* smc = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smc_raw) + 1023) & ~uintptr_t(1023));
  const int G = p.Hq / p.Hkv;
  const int j = (int)cl_rank();
  const int h = blockIdx.y;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  const int z = blockIdx.z / qtiles;
  const int qt = blockIdx.z % qtiles;
  const int r0 = z * p.rows_per_seq + qt * 16;
  const int nrows = min(16, p.rows_per_seq - qt * 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool causal = p.causal != 0;

  // ---- the tile's rows: visible context length (-1: no position), longest
  __shared__ int s_len[16];
  __shared__ int s_first_new;  // cache positions from here on are written by this pass
  if (threadIdx.x < 16) {
    int l = -1;
    if ((int)threadIdx.x < nrows && p.row_pos[r0 + threadIdx.x] >= 0) l = ctx_len_rows(p, r0 + threadIdx.x);
    s_len[threadIdx.x] = l;
  }
  if (threadIdx.x == 32) {
    const int f = p.row_pos[z * p.rows_per_seq];
    s_first_new = causal ? (f >= 0 ? f : 0) : 0x7fffffff;
  }
  const int ppc = MC / p.page_tokens;
  int* s_pg = reinterpret_cast<int*>(smc + TP_PGOFF);
  const int seq_slot = p.row_seq[r0];
  const int cap_chunks = (p.grid_chunks > j) ? (p.grid_chunks - j + CLA - 1) / CLA : 0;
  for (int t = threadIdx.x; t < cap_chunks * ppc && t < MAXPG; t += blockDim.x) {
    const int pg = (j + CLA * (t / ppc)) * ppc + t % ppc;  // page of the sequence
    s_pg[t] = pg < p.pt_stride ? p.page_table[(size_t)seq_slot * p.pt_stride + pg] : -1;
  }

  // full / empty barriers of the key (k) and value (v) tiles of each stage
  __shared__ __align__(8) uint64_t s_fk[TP_NST], s_fv[TP_NST], s_ek[TP_NST], s_ev[TP_NST];
  __shared__ __align__(8) uint64_t s_bs[2], s_bp[2], s_bpv[2], s_sc[2], s_done, s_done_s;
  __shared__ int s_failed;
  __shared__ uint8_t s_part[MAXPG];  // per chunk of this CTA: the value tile needs zeros
  __shared__ uint32_t s_tmem;
  if (threadIdx.x == 0) {
    for (int b = 0; b < TP_NST; ++b) {
      tp_mbar_init(smem_addr(&s_fk[b]), 1);
      tp_mbar_init(smem_addr(&s_fv[b]), 1);
      tp_mbar_init(smem_addr(&s_ek[b]), 1);
      tp_mbar_init(smem_addr(&s_ev[b]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tp_mbar_init(smem_addr(&s_bs[b]), 1);
      tp_mbar_init(smem_addr(&s_bp[b]), 4);  // one arrival per softmax warp
      tp_mbar_init(smem_addr(&s_bpv[b]), 1);
    }
    for (int b = 0; b < 2; ++b) tp_mbar_init(smem_addr(&s_sc[b]), 4);  // S buffer read: one arrival per softmax warp
    tp_mbar_init(smem_addr(&s_done), 1);
    tp_mbar_init(smem_addr(&s_done_s), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kvmap)) : "memory");
    s_failed = 0;
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_addr(&s_tmem))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;  // columns [0, 128): S buffers 0 and 1; [128, 256): O

  int max_len = 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) max_len = max(max_len, s_len[r]);
  const int first_new = s_first_new;
  const int nA = (max_len + MC - 1) / MC;                       // context chunks of the tile
  const int nmine = nA > j ? (nA - j + CLA - 1) / CLA : 0;       // this CTA's context chunks
  const bool has_blk = !causal && j == CLA - 1;
  const int nsteps = nmine + (has_blk ? 1 : 0);
  const int PT = p.page_tokens;
  const __nv_bfloat16* blk = reinterpret_cast<const __nv_bfloat16*>(p.blk);

  if (warp == 4 || warp == 6) {
    // ================================================================ producers
    // warp 4 stages the key tiles, warp 6 the value tiles.  TMA of context
    // chunk st into stage buf: part 1 = pages wholly before first_new (written
    // by earlier passes), 2 = the rest, 3 = all; part 2 or 3 makes the tile
    // barrier's one arrival.
    const int kv = warp == 4 ? 0 : 1;
    uint64_t* fullb = kv ? s_fv : s_fk;
    uint64_t* emptyb = kv ? s_ev : s_ek;
    // Called by the whole warp: lane 0 keeps the barrier's byte count, and
    // lane 2 * pg + half issues the box of (page pg, half) itself, so a
    // chunk's boxes go out in parallel (each issuing thread's TMA copies are
    // served one after another, and a box here is only 2 KB).
    auto stage_tma = [&](int st, int buf, int part) {
      uint8_t* sT = smc + buf * CL_STAGE + kv * 2 * CL_HALF;
      const uint32_t bar = smem_addr(&fullb[buf]);
      const int key0 = (j + CLA * st) * MC;
      const int npg = (min(MC, max_len - key0) + PT - 1) / PT;  // pages holding a key the tile can see
      auto wanted = [&](int pg) {
        const bool old = key0 + (pg + 1) * PT <= first_new;
        const int page = s_pg[st * ppc + pg];
        return ((old ? 1 : 2) & part) && page >= 0 && page < p.n_pages;
      };
      if (lane == 0) {
        uint32_t bytes = 0;
        for (int pg = 0; pg < npg; ++pg)
          if (wanted(pg)) bytes += 2u * (uint32_t)PT * 128u;
        if (part == 1) {
          if (bytes) cl_expect_tx(bar, bytes);
        } else {
          cl_arrive_expect_tx(bar, bytes);
        }
      }
      const int pg = lane >> 1, half = lane & 1;
      if (pg < npg && wanted(pg)) {
        const int page = s_pg[st * ppc + pg];
        tma_kv(smem_addr(sT + half * CL_HALF + pg * PT * 128), &kvmap, bar, half, (page * 2 + kv) * p.Hkv + h);
      }
    };
    for (int st = 0; st < TP_NST && st < nmine; ++st) stage_tma(st, st, 1);
    pdl_wait();
    int issued = 0;
    for (int st = 0; st < nsteps; ++st) {
      const int buf = st % TP_NST;
      if (st >= TP_NST) {
        // the tile is free once chunk st - TP_NST's S (keys) or P V (values) has finished
        bool ok = true;
        if (lane == 0) ok = cl_wait_fast(smem_addr(&emptyb[buf]), (uint32_t)((st / TP_NST) - 1) & 1u, p.err);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok || *reinterpret_cast<volatile int*>(&s_failed)) {
          s_failed = 1;
          break;
        }
      }
      if (st < nmine) {
        stage_tma(st, buf, st < TP_NST ? 2 : 3);
      } else {
        // the drafter's block rows (keys past the block read as zeros)
        uint8_t* sT = smc + buf * CL_STAGE + kv * 2 * CL_HALF;
        for (int idx = lane; idx < MC * (MHD / 8); idx += 32) {
          const int key = idx >> 4, b = idx & 15;
          if (key < p.rows_per_seq) {
            const int row = z * p.rows_per_seq + key;
            cp_async16(smem_addr(sT) + swz2(key, b), blk + ((size_t)(kv * p.Hkv + h) * p.rows_cap + row) * MHD + b * 8);
          } else {
            *reinterpret_cast<uint4*>(sT + swz2(key, b)) = make_uint4(0, 0, 0, 0);
          }
        }
        cp_async_commit();
        cp_async_wait_0();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) tp_arrive(smem_addr(&fullb[buf]));
      }
      issued = st + 1;
    }
    // leave no copy in flight: wait (bounded) for the last tiles issued
    if (lane == 0)
      for (int st = max(0, issued - TP_NST); st < issued; ++st)
        if (st < nmine) cl_wait_bar(smem_addr(&fullb[st % TP_NST]), (uint32_t)(st / TP_NST) & 1u, p.err);
    __syncwarp();
  } else if (warp == 5 || warp == 7) {
    // ================================================================ MMA issuers
    // Warp 7 issues S = Q K^T of every chunk, warp 5 every O += P V: each
    // thread's tcgen05.mma instructions take long to issue, and the two
    // chains are independent (different tensor-memory accumulators).
    // Shared-memory descriptors are computed once: a descriptor's start
    // address field is the byte address / 16, so an operand at a constant
    // offset is the base descriptor plus offset / 16 (no carry: every address
    // is below 256 KB).
    if (warp == 7) asm volatile("bar.sync 1, 160;" ::: "memory");  // the Q tile is in shared memory
    if (lane == 0 && nsteps > 0) {
      bool ok = true;
      if (warp == 7) {
        const uint64_t qd = tc_desc(smem_addr(smc + TP_QOFF), 16);
        const uint64_t kd = tc_desc(smem_addr(smc), 16);
        for (int i = 0; ok && i < nsteps; ++i) {
          const int buf = i % TP_NST;
          // S buffer i & 1 is free once the softmax has read S_{i-2}; the key tile has landed
          if ((i >= 2 && !cl_wait_fast(smem_addr(&s_sc[i & 1]), (uint32_t)((i - 2) >> 1) & 1u, p.err)) ||
              !cl_wait_fast(smem_addr(&s_fk[buf]), (uint32_t)(i / TP_NST) & 1u, p.err)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint64_t kb = kd + (uint64_t)((buf * CL_STAGE) >> 4);
          const uint32_t dst = tmem + (uint32_t)(i & 1) * 64u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma(dst, qd + (uint64_t)(((kk >> 2) * TC_QHALF + (kk & 3) * 32) >> 4),
                   kb + (uint64_t)(((kk >> 2) * CL_HALF + (kk & 3) * 32) >> 4), TC_IDESC_S, kk > 0 ? 1u : 0u);
          tc_commit(smem_addr(&s_bs[i & 1]));
          tc_commit(smem_addr(&s_ek[buf]));  // the key tile is free once S_i has read it
        }
      } else {
        const uint64_t pd = tc_desc(smem_addr(smc + TP_POFF), 16);
        const uint64_t vd = tc_desc(smem_addr(smc + 2 * CL_HALF), CL_HALF);
        for (int i = 0; ok && i < nsteps; ++i) {
          if (!cl_wait_fast(smem_addr(&s_bp[i & 1]), (uint32_t)(i >> 1) & 1u, p.err) ||
              !cl_wait_fast(smem_addr(&s_fv[i % TP_NST]), (uint32_t)(i / TP_NST) & 1u, p.err)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint64_t vb = vd + (uint64_t)(((i % TP_NST) * CL_STAGE) >> 4);
          const uint64_t pb = pd + (uint64_t)(((i & 1) * 128 * 128) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(tmem + 128u, pb + (uint64_t)((kk * 32) >> 4), vb + (uint64_t)((kk * 2048) >> 4), TC_IDESC_PV,
                   (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_addr(&s_bpv[i & 1]));
          tc_commit(smem_addr(&s_ev[i % TP_NST]));  // the value tile is free once P_i V_i has read it
        }
      }
      if (!ok) s_failed = 1;
      // every MMA this thread issued has finished before tensor memory is freed
      const uint32_t done = smem_addr(warp == 7 ? &s_done_s : &s_done);
      tc_commit(done);
      cl_wait_bar(done, 0u, p.err);
    }
    __syncwarp();
  } else {
    // ================================================================ softmax
    pdl_wait();
    // Q as the A operand of S = Q K^T: 128 rows, two 64-dim halves, 128-byte swizzle;
    // rows without a (head, token) read as zeros
    uint8_t* sQ = smc + TP_QOFF;
    for (int idx = threadIdx.x; idx < 128 * 16; idx += 128) {
      const int row = idx >> 4, c = idx & 15;
      const int g = DUP ? (row >> 5) : (row >> 5) + 4 * ((row >> 4) & 1), r = row & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (g < G && r < nrows && s_len[r] >= 0)
        v = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + (size_t)(r0 + r) * p.Hq * MHD +
                                            (size_t)(h * G + g) * MHD + c * 8);
      *reinterpret_cast<uint4*>(sQ + (c >> 3) * TC_QHALF + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = v;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("bar.arrive 1, 160;" ::: "memory");
    // which of this CTA's chunks need zeros in their value tile (keys past the
    // tile's longest row, or a page the table does not hold), once for all
    for (int st = threadIdx.x; st < nmine && st < MAXPG; st += 128) {
      const int nkeys = min(MC, max_len - (j + CLA * st) * MC);
      bool part = nkeys < MC;
      for (int pg = 0; pg < (nkeys + PT - 1) / PT; ++pg) {
        const int page = s_pg[st * ppc + pg];
        part = part || page < 0 || page >= p.n_pages;
      }
      s_part[st] = part ? 1 : 0;
    }
    asm volatile("bar.sync 3, 128;" ::: "memory");

    const int trow = threadIdx.x;  // tensor-memory lane = MMA row
    const int half = lane >> 4;    // DUP: this thread's keys of a chunk are half * 32 + [0, 32)
    const int g = DUP ? warp : warp + 4 * half, r = lane & 15;
    const bool row_ok = g < G && r < nrows && s_len[r] >= 0;
    const int len = row_ok ? s_len[r] : 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    bool failed = false;
    for (int i = 0; i < nsteps; ++i) {
      const int sb = i & 1;
      if (!tp_wait_warp(smem_addr(&s_bs[sb]), (uint32_t)(i >> 1) & 1u, p.err)) {
        failed = true;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      constexpr int NK = DUP ? 32 : 64;  // scores of this thread per chunk
      float sv[NK];
      if constexpr (DUP) {
        float s2[64];
        tc_ld64(tmem + lane_base + (uint32_t)sb * 64u, s2);
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) sv[kk] = half ? s2[32 + kk] : s2[kk];
      } else {
        tc_ld64(tmem + lane_base + (uint32_t)sb * 64u, sv);
      }
      // S_i is in registers: its buffer may take S_{i+2}
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) tp_arrive(smem_addr(&s_sc[sb]));
      const int koff = DUP ? half * 32 : 0;
      const bool is_blk = i >= nmine;
      const int key0 = is_blk ? 0 : (j + CLA * i) * MC;
      const int vis = (!row_ok ? 0 : (is_blk ? p.rows_per_seq : len - key0)) - koff;
      if (vis < NK) {  // keys the row cannot see score -inf (full chunks skip this)
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) sv[kk] = (kk < vis) ? sv[kk] : -INFINITY;
      }
      // the raw maximum in four independent chains, scaled once (scale > 0)
      float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
      for (int kk = 4; kk < NK; kk += 4) {
        mx0 = fmaxf(mx0, sv[kk]);
        mx1 = fmaxf(mx1, sv[kk + 1]);
        mx2 = fmaxf(mx2, sv[kk + 2]);
        mx3 = fmaxf(mx3, sv[kk + 3]);
      }
      float mraw = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      if constexpr (DUP) mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, 16));
      const float mc = mraw * p.scale_log2;
      const bool resc = mc > m_run + TP_RESCALE;
      const float m_new = resc ? mc : m_run;
      const float alpha = resc ? ex2_fast(m_run - m_new) : 1.f;  // 0 for a row's first visible chunk
      const float mneg = (m_new == -INFINITY) ? 0.f : -m_new;
      // P = 2^(s * scale - m): one FFMA and one ex2 per score, sums in four chains
      float cs0 = 0.f, cs1 = 0.f, cs2 = 0.f, cs3 = 0.f;
      uint32_t pk[NK / 2];
#pragma unroll
      for (int kk = 0; kk < NK; kk += 4) {
        const float e0 = ex2_fast(fmaf(sv[kk], p.scale_log2, mneg));
        const float e1 = ex2_fast(fmaf(sv[kk + 1], p.scale_log2, mneg));
        const float e2 = ex2_fast(fmaf(sv[kk + 2], p.scale_log2, mneg));
        const float e3 = ex2_fast(fmaf(sv[kk + 3], p.scale_log2, mneg));
        cs0 += e0;
        cs1 += e1;
        cs2 += e2;
        cs3 += e3;
        pk[kk >> 1] = pack_bf16(e0, e1);
        pk[(kk >> 1) + 1] = pack_bf16(e2, e3);
      }
      float cs = (cs0 + cs1) + (cs2 + cs3);
      if constexpr (DUP) cs += __shfl_xor_sync(0xffffffffu, cs, 16);
      l_run = l_run * alpha + cs;
      m_run = m_new;
      // values of keys the staged pages do not cover (past the tile's longest
      // row, or a page the table does not hold) read as zeros in P V
      if (!is_blk) {
        const int nkeys = min(MC, max_len - key0);
        if (s_part[i]) {
          // the value tile has landed (its barrier cannot run ahead: the tile is refilled only after P_i V_i)
          if (!tp_wait_warp(smem_addr(&s_fv[i % TP_NST]), (uint32_t)(i / TP_NST) & 1u, p.err)) {
            failed = true;
            break;
          }
          uint8_t* sV = smc + (i % TP_NST) * CL_STAGE + 2 * CL_HALF;
          for (int idx = threadIdx.x; idx < MC * (MHD / 8); idx += 128) {
            const int key = idx >> 4, b = idx & 15;
            const int page = s_pg[i * ppc + key / PT];
            const bool have = key < nkeys && page >= 0 && page < p.n_pages;
            if (!have) {
              if (key < nkeys && b == 0 && (key % PT) == 0) flag_error(p.err, ERR_BOUNDS);
              *reinterpret_cast<uint4*>(sV + swz2(key, b)) = make_uint4(0, 0, 0, 0);
            }
          }
        }
      }
      // the P buffer is free once P V of chunk i - 2 has finished
      if (i >= 2 && !tp_wait_warp(smem_addr(&s_bpv[sb]), (uint32_t)((i - 2) >> 1) & 1u, p.err)) {
        failed = true;
        break;
      }
      // O rows rescaled in tensor memory (P V of chunk i - 1 finished first);
      // warp-wide loads and stores, rows that keep their scale multiply by 1
      if (i >= 1 && __any_sync(0xffffffffu, resc)) {
        if (!tp_wait_warp(smem_addr(&s_bpv[(i - 1) & 1]), (uint32_t)((i - 1) >> 1) & 1u, p.err)) {
          failed = true;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float ov[32];
          tc_ld32(tmem + lane_base + 128u + 32u * c, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= alpha;
          tc_st32(tmem + lane_base + 128u + 32u * c, ov);
        }
      }
      uint8_t* sP = smc + TP_POFF + sb * 128 * 128;
      if constexpr (DUP) {
        // this thread's 32 keys into both copies of its row (lanes r and 16 + r of the warp)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          const int cc = half * 4 + c;
          *reinterpret_cast<uint4*>(sP + (trow & ~16) * 128 + ((cc ^ (trow & 7)) << 4)) = v;
          *reinterpret_cast<uint4*>(sP + (trow | 16) * 128 + ((cc ^ (trow & 7)) << 4)) = v;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(sP + trow * 128 + ((c ^ (trow & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) tp_arrive(smem_addr(&s_bp[sb]));
    }
    if (failed) s_failed = 1;
    // the last P V
    bool have_o = nsteps > 0 && !failed;
    if (have_o && !tp_wait_warp(smem_addr(&s_bpv[(nsteps - 1) & 1]), (uint32_t)((nsteps - 1) >> 1) & 1u, p.err)) {
      have_o = false;
      s_failed = 1;
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // the partial (running max, sum, unnormalised output) for the merge: wait
    // until every warp's stages are consumed before writing over them
    asm volatile("bar.sync 2, 128;" ::: "memory");
    float* sO = reinterpret_cast<float*>(smc);
    float2* sML = reinterpret_cast<float2*>(smc + 8 * 16 * TC_OLD * 4);
    float* dst = sO + (size_t)(g * 16 + r) * TC_OLD;
    const bool any_o = __any_sync(0xffffffffu, have_o);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float ov[32];
      if (any_o) {
        tc_ld32(tmem + lane_base + 128u + 32u * c, ov);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0.f;
      }
      // DUP: the two copies of a row write the output's dims 0..63 and 64..127
      if (row_ok && (!DUP || (c >> 1) == half)) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dst + 32 * c + e) = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
      }
    }
    if (row_ok && (!DUP || half == 0)) sML[g * 16 + r] = make_float2(m_run, l_run);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 5) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
  }
  cl_arrive();
  cl_wait();

  // ---- merge: this CTA's share of the (head, row) pairs, 32 threads x 4 dims per pair
  const float* sO = reinterpret_cast<const float*>(smc);
  const float2* sML = reinterpret_cast<const float2*>(smc + 8 * 16 * TC_OLD * 4);
  const int pairs = G * 16;
  const int p0 = j * pairs / CLA, p1 = (j + 1) * pairs / CLA;
  const uint32_t sO_s = smem_addr(sO), sML_s = smem_addr(sML);
  for (int pp = p0 + warp; pp < p1; pp += TP_THREADS / 32) {
    const int g = pp >> 4, rr = pp & 15;
    if (rr >= nrows || s_len[rr] < 0) continue;
    float2 ml[CLA];
    float4 av[CLA];
    // ranks without a chunk of this tile hold (-inf, 0, 0): their terms are
    // exactly zero, so they are not read
#pragma unroll
    for (int i = 0; i < CLA; ++i) {
      const bool held = i < nA || (!causal && i == CLA - 1);
      ml[i] = held ? cl_ld2(cl_map(sML_s + (uint32_t)(g * 16 + rr) * 8u, (uint32_t)i)) : make_float2(-INFINITY, 0.f);
      av[i] = held ? cl_ld4(cl_map(sO_s + (uint32_t)((g * 16 + rr) * TC_OLD + lane * 4) * 4u, (uint32_t)i))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < CLA; ++i) Mx = fmaxf(Mx, ml[i].x);
    float L = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < CLA; ++i) {
      const float w = (ml[i].x == -INFINITY) ? 0.f : exp2f(ml[i].x - Mx);
      L = fmaf(ml[i].y, w, L);
      a.x = fmaf(av[i].x, w, a.x);
      a.y = fmaf(av[i].y, w, a.y);
      a.z = fmaf(av[i].z, w, a.z);
      a.w = fmaf(av[i].w, w, a.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)(r0 + rr) * p.Hq * MHD +
                         (size_t)(h * G + g) * MHD + lane * 4;
    uint2 packed;
    packed.x = pack_bf16(a.x * inv, a.y * inv);
    packed.y = pack_bf16(a.z * inv, a.w * inv);
    *reinterpret_cast<uint2*>(out) = packed;
  }
  cl_arrive_relaxed();  // this CTA's reads of the other partials are done
  cl_wait();    // and nobody leaves while another CTA may still read its partial
}

template <int CLA, bool DUP>
__global__ void __launch_bounds__(TP_THREADS, 1)
    attn_tp_kernel(AttnParams p, const __grid_constant__ CUtensorMap kvmap) {
  trace_entry(p.trace);
  attn_tp_body<CLA, DUP>(p, kvmap);
  trace_exit(p.trace);
}

static int g_cla_tp = 0;         // default CTAs per cluster of the pipelined kernel (0: not prepared)
static bool g_tp16_ok = false;  // clusters of 16 can be placed

template <bool DUP>
static cudaError_t launch_tp(const AttnParams& p, int cla, int qtiles, const CUtensorMap& map, cudaStream_t st) {
  const dim3 grid(cla, p.Hkv, p.n_seqs * qtiles);
  switch (cla) {
    case 16:
      return launch_kcl(attn_tp_kernel<16, DUP>, grid, dim3(TP_THREADS), (size_t)TP_SMEM, st, dim3(16, 1, 1), p, map);
    case 8:
      return launch_kcl(attn_tp_kernel<8, DUP>, grid, dim3(TP_THREADS), (size_t)TP_SMEM, st, dim3(8, 1, 1), p, map);
    case 4:
      return launch_kcl(attn_tp_kernel<4, DUP>, grid, dim3(TP_THREADS), (size_t)TP_SMEM, st, dim3(4, 1, 1), p, map);
    default:
      return launch_kcl(attn_tp_kernel<2, DUP>, grid, dim3(TP_THREADS), (size_t)TP_SMEM, st, dim3(2, 1, 1), p, map);
  }
}

template <bool DUP>
static cudaError_t tp_attrs() {
  cudaError_t e = cudaFuncSetAttribute(attn_tp_kernel<8, DUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, TP_SMEM);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_tp_kernel<16, DUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, TP_SMEM);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_tp_kernel<4, DUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, TP_SMEM);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_tp_kernel<2, DUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, TP_SMEM);
  return e;
}

cudaError_t launch_attention_tp(const AttnParams& p, cudaStream_t st) {
  if (!attention_cluster_fits(p)) return cudaErrorInvalidValue;
  cudaError_t e = attention_tp_prepare();
  if (e != cudaSuccess) return e;
  // CTAs per cluster: the launch's choice (2, 4, 8 or 16), else the process default
  const int cla = (p.cla == 2 || p.cla == 4 || p.cla == 8 || (p.cla == 16 && g_tp16_ok)) ? p.cla : g_cla_tp;
  // page ids a CTA stages for its chunks (the cluster's ranks take every cla-th chunk)
  const int per_cta = (p.grid_chunks + cla - 1) / cla;
  if (per_cta * (MC / p.page_tokens) > MAXPG) return cudaErrorInvalidValue;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(p.kv_map);
  return p.Hq / p.Hkv <= 4 ? launch_tp<true>(p, cla, qtiles, map, st) : launch_tp<false>(p, cla, qtiles, map, st);
}

cudaError_t attention_tp_prepare() {
  if (g_cla_tp) return cudaSuccess;
  cudaError_t e = tp_attrs<true>();
  if (e == cudaSuccess) e = tp_attrs<false>();
  if (e != cudaSuccess) return e;
  // clusters of 16 need the non-portable size and a device that can place them
  bool big = cudaFuncSetAttribute(attn_tp_kernel<16, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                 cudaSuccess &&
             cudaFuncSetAttribute(attn_tp_kernel<16, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                 cudaSuccess;
  if (big) {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(16, 1, 1);
    c.blockDim = dim3(TP_THREADS);
    c.dynamicSmemBytes = TP_SMEM;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = 16;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    c.attrs = a;
    c.numAttrs = 1;
    int n = 0;
    big = cudaOccupancyMaxActiveClusters(&n, attn_tp_kernel<16, true>, &c) == cudaSuccess && n > 0;
  }
  cudaGetLastError();
  g_tp16_ok = big;
  // the process default when a launch names no cluster size: DF_ATTN_PIPE_CLA (2, 4, 8 or 16), else 4
  // (one CTA per SM: small clusters place on every SM and give each CTA a long chunk pipeline)
  const char* env = getenv("DF_ATTN_PIPE_CLA");
  const int want = env ? atoi(env) : 4;
  g_cla_tp = (want == 2 || want == 4 || want == 8 || (want == 16 && big)) ? want : 4;
  return cudaSuccess;
}

static int g_cla_tc = 0;

cudaError_t launch_attention_tc(const AttnParams& p, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  if (!attention_cluster_fits(p) || G > 4) return cudaErrorInvalidValue;
  if (!g_cla_tc) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    if (e != cudaSuccess) return e;
    const bool big = cudaFuncSetAttribute(attn_tc_kernel<16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    cudaGetLastError();
    g_cla_tc = big ? 16 : 8;
  }
  const int per_cta = (p.grid_chunks + g_cla_tc - 1) / g_cla_tc;  // page ids a CTA stages
  if (per_cta * (MC / p.page_tokens) > MAXPG) return cudaErrorInvalidValue;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(p.kv_map);
  if (g_cla_tc == 16)
    return launch_kcl(attn_tc_kernel<16>, dim3(16, p.Hkv, p.n_seqs * qtiles), dim3(128), (size_t)TC_SMEM, st, dim3(16, 1, 1), p, map);
  return launch_kcl(attn_tc_kernel<8>, dim3(8, p.Hkv, p.n_seqs * qtiles), dim3(128), (size_t)TC_SMEM, st, dim3(8, 1, 1), p, map);
}

// TMA map of one layer of the paged cache (declared in internal.h).
typedef CUresult (*PFN_kvEncodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                        const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                        CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_tmap_kvcache(void* map_out, const void* base, int n_pages, int n_kv_heads, int page_tokens) {
  static PFN_kvEncodeTiled_t enc = nullptr;
  if (!enc) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<PFN_kvEncodeTiled_t>(fn);
  }
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) || page_tokens <= 0 || page_tokens > 256) return false;
  cuuint64_t gdim[4] = {64, 2, (cuuint64_t)page_tokens, (cuuint64_t)n_pages * 2 * n_kv_heads};
  cuuint64_t gstride[3] = {128, (cuuint64_t)MHD * 2, (cuuint64_t)page_tokens * MHD * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)page_tokens, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = enc(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
                   gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int CLA>
static bool cluster_placeable() {
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3(CLA, 1, 1);
  c.blockDim = dim3(256);
  c.dynamicSmemBytes = cl_smem_bytes(8);
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = CLA;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  c.attrs = a;
  c.numAttrs = 1;
  int n = 0;
  const bool ok = cudaOccupancyMaxActiveClusters(&n, attn_cl_kernel<CLA, 8>, &c) == cudaSuccess && n > 0;
  cudaGetLastError();
  return ok;
}

static int g_cla = 0;  // cluster size in use (0: not chosen yet)

// Kernel attributes and the cluster size, once, before any stream capture.
template <int CLA, int NW>
static cudaError_t cl_attrs() {
  return cudaFuncSetAttribute(attn_cl_kernel<CLA, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, cl_smem_bytes(8));
}

// Failure-detection check: one bounded wait on a barrier that nothing
// completes.  The wait the attention kernels use runs out after its limit,
// records ERR_TIMEOUT in `err`, and the kernel returns normally.
__global__ void wait_probe_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) cl_mbar_init(smem_addr(&bar));
  __syncthreads();
  if (threadIdx.x == 0) (void)cl_wait_bar(smem_addr(&bar), 0u, err);
}
cudaError_t launch_wait_probe(int* err, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(err);
  return cudaGetLastError();
}

cudaError_t attention_cluster_prepare() {
  if (g_cla) return cudaSuccess;
  cudaError_t e;
  if ((e = cl_attrs<4, 4>()) != cudaSuccess || (e = cl_attrs<4, 8>()) != cudaSuccess ||
      (e = cl_attrs<8, 4>()) != cudaSuccess || (e = cl_attrs<8, 8>()) != cudaSuccess ||
      (e = cl_attrs<16, 4>()) != cudaSuccess || (e = cl_attrs<16, 8>()) != cudaSuccess)
    return e;
  const bool big =
      cudaFuncSetAttribute(attn_cl_kernel<16, 4>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
      cudaFuncSetAttribute(attn_cl_kernel<16, 8>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
      cluster_placeable<16>();
  cudaGetLastError();
  // DF_ATTN_CLA=4|8|16 in the environment picks the cluster size; otherwise 16 where it can be placed
  const char* env = getenv("DF_ATTN_CLA");
  const int want = env ? atoi(env) : 16;
  g_cla = (want == 4 || want == 8) ? want : (big ? 16 : 8);
  return cudaSuccess;
}

template <int CLA>
static cudaError_t launch_cl(const AttnParams& p, cudaStream_t st) {
  const int G = p.Hq / p.Hkv;
  const int per_cta = (p.grid_chunks + CLA - 1) / CLA;
  if (per_cta * (MC / p.page_tokens) > MAXPG) return cudaErrorInvalidValue;
  const int qtiles = (p.rows_per_seq + 15) / 16;
  dim3 grid(CLA, p.Hkv, p.n_seqs * qtiles);
  const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(p.kv_map);
  if (G <= 4)
    return launch_kcl(attn_cl_kernel<CLA, 4>, grid, dim3(128), (size_t)cl_smem_bytes(G), st, dim3(CLA, 1, 1), p, map);
  return launch_kcl(attn_cl_kernel<CLA, 8>, grid, dim3(256), (size_t)cl_smem_bytes(G), st, dim3(CLA, 1, 1), p, map);
}

bool attention_cluster_fits(const AttnParams& p) {
  const int G = p.Hq / p.Hkv;
  return p.hd == MHD && p.chunk == MC && G <= 8 && p.page_tokens > 0 && MC % p.page_tokens == 0 &&
         p.page_tokens % 8 == 0 && p.kv_map != nullptr && (p.causal || p.rows_per_seq <= MC);
}

cudaError_t launch_attention_cluster(const AttnParams& p, cudaStream_t st) {
  if (!attention_cluster_fits(p)) return cudaErrorInvalidValue;
  cudaError_t e = attention_cluster_prepare();
  if (e != cudaSuccess) return e;
  return g_cla == 16 ? launch_cl<16>(p, st) : g_cla == 8 ? launch_cl<8>(p, st) : launch_cl<4>(p, st);
}
}  // namespace dfk
