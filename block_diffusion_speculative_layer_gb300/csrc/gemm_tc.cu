// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Computes acc[m][n] = sum_k X[m][k] * W[n][k] for a weight matrix W
// [N][K] (a linear layer's [out, in] layout) and activations X [M][K], both
// bf16 and K-contiguous, accumulating in fp32.  Decode-shaped calls have few
// token rows (M = block size x batch), so the roles are swapped: 128 weight
// rows form the MMA's M side and the token rows its N side (16..256).  Each
// CTA owns one 128-row weight tile, one token tile and one K range (split-K);
// the weight stream is what bounds the kernel, so the pipeline only has to
// keep enough TMA loads in flight.
//
// Roles (128 threads): warp 0 lane 0 issues TMA loads into a STAGES-deep ring
// of shared-memory stages; warp 1 lane 0 issues tcgen05.mma (kind::f16, bf16 in,
// fp32 accumulate in tensor memory) and releases stages with tcgen05.commit;
// warp 2 owns the TMEM allocation; all four warps drain the accumulator with
// tcgen05.ld (thread t holds weight row n0+t for every token) into a shared
// tile on which the fused epilogue runs.
//
// Split-K: the `splits` CTAs of a tile form a thread-block cluster.  Each
// leaves its fp32 partial tile in its own shared memory; after a cluster
// barrier, CTA q sums rows [rows*q/splits, rows*(q+1)/splits) of all partials
// through distributed shared memory, in split order 0,1,2,..., and runs the
// epilogue on those rows; a second barrier keeps every CTA's shared memory
// alive until the reads are done.  (Without clusters the partials go to a
// workspace instead and the CTA that finishes a tile last, by an atomic
// ticket, adds them in the same order.)  The split count depends only on
// (N, K), and the MMA sequence of one output does not depend on M, so every
// output is bitwise the same whatever the number of token rows.
//
// Launched with programmatic dependent launch: the producer streams the first
// STAGES weight tiles before waiting for the previous kernel's outputs.
//
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel
// records ERR_TIMEOUT, waits (bounded) for the TMA loads it issued, frees its
// tensor memory and returns.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace dfk {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K elements per stage: 128 bytes, one swizzle row
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait on an mbarrier phase.  Returns false (and flags the error word)
// when the phase has not completed within the limit.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 1023u) == 0 && global_ns() - t0 > kWaitLimitNs) break;
  }
  flag_error(err, ERR_TIMEOUT);
  return false;
}

// One test inline first; the bounded loop is an out-of-line call.
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity, int* err) {
  return mbar_try_wait(bar, parity) || mbar_wait(bar, parity, err);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// L2 prefetch of one tile of a tensor map (a hint: no data reaches shared memory).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}

// Thread-block cluster helpers (all threads of every CTA execute the barriers).
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
// For an arrival that follows reads whose values are already used (it
// publishes nothing); every thread of the CTA takes the same form.
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 dsmem_ld4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                     // leading-dimension offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride between 8-row groups
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <int NT, int ST = 0>
struct TcCfg {
  static constexpr int STAGES = ST ? ST : NT <= 16 ? 6 : NT <= 32 ? 5 : 4;
  static constexpr int W_BYTES = BM * BK * 2;
  static constexpr int X_BYTES = NT * BK * 2;
  static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
  static constexpr int TMEM_COLS = NT < 32 ? 32 : NT;
  static constexpr int TLD = BM + 4;  // epilogue tile row stride (floats)
  static constexpr int META_OFF = STAGES * STAGE_BYTES + 256;   // row facts staged during the mainloop
  static constexpr int SMEM = 1024 + META_OFF + NT * (int)sizeof(RowMeta);
  static constexpr int PRE_OFF = NT * TLD * 4 + NT * 16;  // the epilogue's operand copies, after tile and row sums
  static_assert(PRE_OFF + EPI_PRE_FLOATS * 4 <= STAGES * STAGE_BYTES, "epilogue tile, row sums and copies fit in the ring");
  static_assert((TLD * 4) % 16 == 0, "tile rows must stay 16-byte aligned for vector copies");
};

template <int NT, int ST>
__device__ __forceinline__ void gemm_tc_body(const CUtensorMap& tmW, const CUtensorMap& tmX, int M, int N, int K,
                                             int splits, float* __restrict__ ws, int* __restrict__ counters,
                                             int creduce, const EpiParams& ep) {
  using C = TcCfg<NT, ST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sX = smem + C::STAGES * C::W_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // 0 last-CTA, 1 consumed, 2 failed, 3 issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, tile_m = blockIdx.y, split = blockIdx.z;
  const int n0 = tile_n * BM, m0 = tile_m * NT;
  const int nkb = K / BK;
  const int kb0 = (int)((long long)nkb * split / splits);
  const int kb1 = (int)((long long)nkb * (split + 1) / splits);
  const int nk = kb1 - kb0;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + C::STAGES);
  const uint32_t accum_bar = smem_u32(bars + 2 * C::STAGES);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accum_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    flags[0] = 0; flags[1] = 0; flags[2] = 0; flags[3] = 0;
  }
  if (threadIdx.x == 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  // A GEMM that writes keys and values triggers its dependent (the attention)
  // only once its own wait has returned: every kernel before this one is then
  // complete, so the attention may read the older cache entries and the row
  // metadata before its own wait.  Every other GEMM lets its dependent start
  // at once.
  const bool late_trigger = ep.kind == EPI_QKV;
  if (!late_trigger) pdl_trigger();
  if (warp == 0 && lane < 2) {
    // ---- TMA producers: lane 0 the weight tiles (and each stage's byte count),
    // lane 1 the token tiles, so the two copies of a stage are issued in
    // parallel (one thread's TMA copies are served one after another)
    const uint64_t pol_w = policy_evict_first();  // weights are read once per launch
    const uint64_t pol_x = policy_evict_last();   // activations are re-read by every weight tile
    // The weights do not depend on the kernel before this one: fill the first
    // stages with weight tiles while it drains, then wait for its outputs.
    const int pre = nk < C::STAGES ? nk : C::STAGES;
    if (lane == 0) {
      for (int i = 0; i < pre; ++i) {
        mbar_expect_tx(full0 + 8 * i, C::STAGE_BYTES);
        tma_load_2d(smem_u32(sW + i * C::W_BYTES), &tmW, full0 + 8 * i, (kb0 + i) * BK, n0, pol_w);
      }
      // and up to ep.l2_prefetch further weight tiles into L2 while the kernel before drains
      const int pf_end = min(nk, pre + ep.l2_prefetch);
      for (int i = pre; i < pf_end; ++i) tma_prefetch_2d(&tmW, (kb0 + i) * BK, n0);
    }
    pdl_wait();
    if (late_trigger) pdl_trigger();
    if (lane == 1)
      for (int i = 0; i < pre; ++i)
        tma_load_2d(smem_u32(sX + i * C::X_BYTES), &tmX, full0 + 8 * i, (kb0 + i) * BK, m0, pol_x);
    int i = pre;
    for (; i < nk; ++i) {
      const int s = i % C::STAGES;
      const uint32_t ph = (uint32_t)(i / C::STAGES) & 1u;
      int ok = 1;
      if (lane == 0) ok = (i < C::STAGES || mbar_wait_fast(empty0 + 8 * s, ph ^ 1u, ep.err)) ? 1 : 0;
      ok = __shfl_sync(0x3u, ok, 0);
      if (!ok) {
        flags[2] = 1;
        break;
      }
      const int kc = (kb0 + i) * BK;
      if (lane == 0) {
        mbar_expect_tx(full0 + 8 * s, C::STAGE_BYTES);
        tma_load_2d(smem_u32(sW + s * C::W_BYTES), &tmW, full0 + 8 * s, kc, n0, pol_w);
      } else {
        tma_load_2d(smem_u32(sX + s * C::X_BYTES), &tmX, full0 + 8 * s, kc, m0, pol_x);
      }
    }
    if (lane == 0) flags[3] = i;
  } else {
    pdl_wait();
    if (late_trigger) pdl_trigger();
  }
  if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(BM, NT);
    // descriptors computed once: an operand at a constant offset is the base
    // descriptor plus offset / 16 (the start-address field; addresses < 256 KB)
    const uint64_t dw0 = desc_sw128(smem_u32(sW)), dx0 = desc_sw128(smem_u32(sX));
    int i = 0;
    for (; i < nk; ++i) {
      const int s = i % C::STAGES;
      const uint32_t ph = (uint32_t)(i / C::STAGES) & 1u;
      if (!mbar_wait_fast(full0 + 8 * s, ph, ep.err)) {
        flags[2] = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t dw = dw0 + (uint64_t)((s * C::W_BYTES) >> 4), dx = dx0 + (uint64_t)((s * C::X_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        mma_bf16(tmem, dw + (uint64_t)(kk * 2), dx + (uint64_t)(kk * 2), idesc, (i > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(empty0 + 8 * s);
    }
    flags[1] = i;
    mma_commit(accum_bar);  // arrives once every MMA issued above has completed
  }
  // Warps 2 and 3 are idle during the mainloop: they stage the epilogue's
  // row facts (positions, KV pages, folded-norm scales) now, so the tail after
  // the last MMA does no dependent global loads of its own.
  RowMeta* meta = reinterpret_cast<RowMeta*>(smem + C::META_OFF);
  if (warp >= 2) epilogue_stage(ep, m0, NT, M, meta, threadIdx.x - 64, 64);
  __syncwarp();

  // ---- drain the accumulator: thread t holds weight row n0 + t for all NT tokens
  if (!mbar_wait(accum_bar, 0, ep.err)) flags[2] = 1;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  __syncthreads();
  // The rows whose epilogue this CTA runs; the copies of their global
  // operands start now (into the ring, which no MMA or load uses any more),
  // ahead of the drain and the split-K reduction.
  const int rows = min(NT, M - m0);
  const bool cl = creduce && splits > 1;
  const int q = cl ? (int)cluster_rank() : 0;
  const int r0 = cl ? rows * q / splits : 0, r1 = cl ? rows * (q + 1) / splits : rows;
  const bool failed = flags[2] != 0;
  const EpiPre pre{reinterpret_cast<float*>(smem + C::PRE_OFF)};
  const bool have_pre =
      !failed && (cl || splits == 1) && epilogue_preload(ep, n0, m0 + r0, r1 - r0, M, meta + r0, pre);
  float* tile = reinterpret_cast<float*>(smem);
  const int f = threadIdx.x;
  if (!failed) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
    for (int c = 0; c < NT; c += 16) {
      float v[16];
      tmem_ld16(tmem + lane_base + (uint32_t)c, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) tile[(c + j) * C::TLD + f] = v[j];
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 2) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
  }
  if (failed) {
    // Wait (bounded) for loads that were issued but never consumed.
    if (threadIdx.x == 0) {
      const int consumed = flags[1], issued = flags[3];
      for (int i = consumed; i < issued; ++i) {
        if (!mbar_wait(full0 + 8 * (i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u, ep.err)) break;
      }
    }
    __syncthreads();
    // A cluster member still takes part in both cluster barriers below (its
    // partial is garbage then, and the error word is already set).
    if (!cl) return;
  }

  float* red = reinterpret_cast<float*>(smem + (size_t)NT * C::TLD * 4);
  if (cl) {
    // ---- split-K through distributed shared memory: every partial is in its CTA's `tile`
    cluster_arrive();
    cluster_wait();
    const uint32_t tile_s = smem_u32(tile);
    const int c4 = threadIdx.x & 31, rl = threadIdx.x >> 5;  // 4 columns x 1 row per thread and pass
    for (int rb = r0; rb < r1; rb += 8) {
      // the loads of two 4-row passes first, then the sums in split order
      float4 v[2][8];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = rb + 4 * i + rl;
        const uint32_t off = (uint32_t)(r * C::TLD + 4 * c4) * 4u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[i][j] = (r < r1 && j < splits) ? dsmem_ld4(dsmem_map(tile_s + off, (uint32_t)j)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = rb + 4 * i + rl;
        float4 acc = v[i][0];
#pragma unroll
        for (int j = 1; j < 8; ++j)
          if (j < splits) {
            acc.x += v[i][j].x;
            acc.y += v[i][j].y;
            acc.z += v[i][j].z;
            acc.w += v[i][j].w;
          }
        if (r < r1) *reinterpret_cast<float4*>(tile + r * C::TLD + 4 * c4) = acc;
      }
    }
    cluster_arrive_relaxed();  // this CTA's reads of the other partials are done
    __syncthreads();
    if (!failed)
      epilogue_tile<__nv_bfloat16>(ep, tile + (size_t)r0 * C::TLD, C::TLD, n0, m0 + r0, r1 - r0, M, meta + r0, red,
                                   /*staged=*/true, have_pre ? &pre : nullptr);
    cp_async_wait_own();  // no copy into this CTA's memory outlives it
    cluster_wait();    // nobody leaves while another CTA may still read its tile
    return;
  }
  if (splits > 1) {
    const int tile_id = tile_m * gridDim.x + tile_n;
    float* part = ws + (size_t)tile_id * splits * NT * BM;
    float* mine = part + (size_t)split * NT * BM;
    for (int r = 0; r < rows; ++r) mine[r * BM + f] = tile[r * C::TLD + f];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int prev = atomicAdd(counters + tile_id, 1);
      flags[0] = (prev == splits - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!flags[0]) return;
    __threadfence();
    // Sum the partials in split order 0, 1, 2, ... (a fixed order, whoever
    // arrives last); the loads of a batch of rows are issued together.
    for (int rb = 0; rb < rows; rb += 16) {
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = rb + i;
        acc[i] = (r < rows) ? ((split == 0) ? tile[r * C::TLD + f] : __ldcg(part + r * BM + f)) : 0.f;
      }
      for (int q = 1; q < splits; ++q) {
        float pv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = rb + i;
          pv[i] = (r < rows) ? ((q == split) ? tile[r * C::TLD + f] : __ldcg(part + (size_t)q * NT * BM + r * BM + f))
                             : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] += pv[i];
      }
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (rb + i < rows) tile[(rb + i) * C::TLD + f] = acc[i];
    }
    if (threadIdx.x == 0) counters[tile_id] = 0;
    __syncthreads();
  }
  epilogue_tile<__nv_bfloat16>(ep, tile, C::TLD, n0, m0, rows, M, meta, red, /*staged=*/true,
                               (have_pre && splits == 1) ? &pre : nullptr);
}

template <int NT, int ST = 0>
__global__ void __launch_bounds__(128, 1) gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                                                      const __grid_constant__ CUtensorMap tmX, int M, int N, int K,
                                                      int splits, float* __restrict__ ws, int* __restrict__ counters,
                                                      int creduce, EpiParams ep) {
  trace_entry(ep.trace);
  gemm_tc_body<NT, ST>(tmW, tmX, M, N, K, splits, ws, counters, creduce, ep);
  trace_exit(ep.trace);
}

// ----------------------------------------------------------------------------
// Serial-split form for many token rows.  With hundreds of token rows a
// split-K tile is large (up to 128 x 256 fp32), one CTA fills an SM, and the
// splits' clusters cannot all be resident at once: the launch runs in waves
// with idle SMs.  Here one CTA per (weight tile, token tile) runs every K
// range of its tile in order, each range into its own tensor-memory
// accumulator (two, alternating, so the next range's MMAs overlap the fold of
// the last), and four fold warps add the finished partials in split order
// 0, 1, 2, ... in registers.  The split count, each partial's MMA sequence and
// the fp32 additions and their order are those of the split-K form, so every
// output is bitwise the same as there; no cluster and no workspace.
//
// Roles (192 threads): warps 0-3 fold (warp w reads tensor-memory lanes
// 32w..32w+31, thread f holds weight row n0 + f for every token) and then run
// the fused epilogue; warp 4 lane 0 issues the TMA loads; warp 5 lane 0 issues
// the MMAs.  The token tile is the fastest grid index, so the CTAs that share
// a weight tile run together and read it from DRAM once.
constexpr int TW_THREADS = 192;

// Stages and where the running sums live.  64-token tiles: 4 stages of 24 KB,
// two CTAs per SM, sums in registers.  128-token tiles: 6 stages of 32 KB, one
// CTA per SM, sums in a third tensor-memory accumulator (128 floats a thread
// would spill).  (Measured at 256 and 512 token rows on the Qwen3-8B shapes:
// 64-token tiles at two CTAs per SM are the fastest or equal in every case;
// 8 stages at one CTA per SM gained nothing where the grid fits one wave and
// lost up to 2x where it does not.)
template <int NT>
struct TwCfg {
  using C = TcCfg<NT>;
  static constexpr int STAGES = NT == 64 ? 4 : 6;
  static constexpr bool RTMEM = NT > 64;
  static constexpr int TCOLS = RTMEM ? 512 : 2 * NT;  // accumulators 0 and 1 (and the sums at 2 NT)
  static constexpr int META_OFF = STAGES * C::STAGE_BYTES + 256;
  static constexpr int SMEM = 1024 + META_OFF + NT * (int)sizeof(RowMeta);
  static_assert(NT * C::TLD * 4 + NT * 16 <= STAGES * C::STAGE_BYTES, "epilogue tile and row sums fit in the ring");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <int NT>
__device__ __forceinline__ void gemm_tcw_body(const CUtensorMap& tmW, const CUtensorMap& tmX, int M, int N, int K,
                                              int splits, const EpiParams& ep) {
  using C = TcCfg<NT>;
  using W = TwCfg<NT>;
  constexpr int STAGES = W::STAGES;
  constexpr int TCOLS = W::TCOLS;
  static_assert(TCOLS >= 32 && TCOLS <= 512 && (TCOLS & (TCOLS - 1)) == 0, "tensor-memory allocation");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sX = smem + STAGES * C::W_BYTES;
  // barriers: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], done
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // 0 failed, 1 consumed, 2 issued
  RowMeta* meta = reinterpret_cast<RowMeta*>(smem + W::META_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * NT, n0 = blockIdx.y * BM;
  const int nkb = K / BK;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t afull0 = smem_u32(bars + 2 * STAGES), aempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t done_bar = smem_u32(bars + 2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(afull0 + 8 * b, 1);
      mbar_init(aempty0 + 8 * b, 4);  // one arrival per fold warp
    }
    mbar_init(done_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    flags[0] = 0; flags[1] = 0; flags[2] = 0;
  }
  if (threadIdx.x == 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  // as in the split-K form: a GEMM that writes keys and values lets its
  // dependent start only after its own wait
  const bool late_trigger = ep.kind == EPI_QKV;
  if (!late_trigger) pdl_trigger();
  // fold warps: the running sum of weight row n0 + threadIdx.x over the tile's tokens, in
  // registers (R) or in tensor-memory columns [2 NT, 3 NT) of the thread's lane
  constexpr bool RTMEM = W::RTMEM;
  float R[RTMEM ? 1 : NT];
  if (warp == 4) {
    if (lane < 2) {
      // ---- TMA producers, the tile's whole K: lane 0 the weight tiles (of the
      // first stages before the wait) and the byte counts, lane 1 the token tiles
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int pre = nkb < STAGES ? nkb : STAGES;
      if (lane == 0)
        for (int i = 0; i < pre; ++i) {
          mbar_expect_tx(full0 + 8 * i, C::STAGE_BYTES);
          tma_load_2d(smem_u32(sW + i * C::W_BYTES), &tmW, full0 + 8 * i, i * BK, n0, pol_w);
        }
      pdl_wait();
      if (late_trigger) pdl_trigger();
      if (lane == 1)
        for (int i = 0; i < pre; ++i)
          tma_load_2d(smem_u32(sX + i * C::X_BYTES), &tmX, full0 + 8 * i, i * BK, m0, pol_x);
      int i = pre;
      for (; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
        int ok = 1;
        if (lane == 0) ok = (mbar_wait_fast(empty0 + 8 * s, ph ^ 1u, ep.err) && !flags[0]) ? 1 : 0;
        ok = __shfl_sync(0x3u, ok, 0);
        if (!ok) {
          flags[0] = 1;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(full0 + 8 * s, C::STAGE_BYTES);
          tma_load_2d(smem_u32(sW + s * C::W_BYTES), &tmW, full0 + 8 * s, i * BK, n0, pol_w);
        } else {
          tma_load_2d(smem_u32(sX + s * C::X_BYTES), &tmX, full0 + 8 * s, i * BK, m0, pol_x);
        }
      }
      if (lane == 0) flags[2] = i;
    } else {
      pdl_wait();
      if (late_trigger) pdl_trigger();
    }
  } else if (warp == 5) {
    pdl_wait();
    if (late_trigger) pdl_trigger();
    if (lane == 0) {
      // ---- MMA issuer: split q into accumulator q & 1, reused once the fold of split q - 2 is done
      constexpr uint32_t idesc = idesc_bf16(BM, NT);
      const uint64_t dw0 = desc_sw128(smem_u32(sW)), dx0 = desc_sw128(smem_u32(sX));
      int i = 0;
      bool ok = true;
      for (int q = 0; q < splits && ok; ++q) {
        const int kb0 = (int)((long long)nkb * q / splits), kb1 = (int)((long long)nkb * (q + 1) / splits);
        const int b = q & 1;
        if (q >= 2 && !mbar_wait_fast(aempty0 + 8 * b, (uint32_t)((q - 2) >> 1) & 1u, ep.err)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        for (int kb = kb0; kb < kb1; ++kb, ++i) {
          const int s = i % STAGES;
          const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
          if (!mbar_wait_fast(full0 + 8 * s, ph, ep.err)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint64_t dw = dw0 + (uint64_t)((s * C::W_BYTES) >> 4), dx = dx0 + (uint64_t)((s * C::X_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(tmem + (uint32_t)(b * NT), dw + (uint64_t)(kk * 2), dx + (uint64_t)(kk * 2), idesc,
                     (kb > kb0 || kk > 0) ? 1u : 0u);
          mma_commit(empty0 + 8 * s);
        }
        if (ok) mma_commit(afull0 + 8 * b);
      }
      if (!ok) flags[0] = 1;
      flags[1] = i;
      mma_commit(done_bar);  // arrives once every MMA issued above has completed
    }
  } else {
    // ---- fold warps: stage the epilogue's row facts, then add the partials in split order
    pdl_wait();
    if (late_trigger) pdl_trigger();
    epilogue_stage(ep, m0, NT, M, meta, threadIdx.x, 128);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int q = 0; q < splits; ++q) {
      const int b = q & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_fast(afull0 + 8 * b, (uint32_t)(q >> 1) & 1u, ep.err))) {
        flags[0] = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
      for (int c = 0; c < NT; c += 16) {
        float v[16];
        tmem_ld16(tmem + lane_base + (uint32_t)(b * NT + c), v);
        if constexpr (RTMEM) {
          const uint32_t ra = tmem + lane_base + (uint32_t)(2 * NT + c);
          if (q > 0) {
            float r[16];
            tmem_ld16(ra, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = r[j] + v[j];
          }
          tmem_st16(ra, v);
        } else if (q == 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) R[c + j] = v[j];
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) R[c + j] += v[j];
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty0 + 8 * b);
      if (flags[0]) break;
    }
    if (threadIdx.x == 0) mbar_wait(done_bar, 0, ep.err);  // every MMA has finished
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  const bool failed = flags[0] != 0;
  auto free_tmem = [&]() {
    if (warp == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TCOLS) : "memory");
    }
  };
  if (failed) {
    free_tmem();
    // wait (bounded) for loads that were issued but never consumed, then leave
    if (threadIdx.x == 0) {
      const int consumed = flags[1], issued = flags[2];
      for (int i = consumed; i < issued; ++i)
        if (!mbar_wait(full0 + 8 * (i % STAGES), (uint32_t)(i / STAGES) & 1u, ep.err)) break;
    }
    return;
  }
  if (warp >= 4) return;
  // ---- the sums into a shared tile over the (now idle) stages, then the epilogue
  float* tile = reinterpret_cast<float*>(smem);
  if constexpr (RTMEM) {
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
    for (int c = 0; c < NT; c += 16) {
      float v[16];
      tmem_ld16(tmem + lane_base + (uint32_t)(2 * NT + c), v);
#pragma unroll
      for (int j = 0; j < 16; ++j) tile[(c + j) * C::TLD + threadIdx.x] = v[j];
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  } else {
#pragma unroll
    for (int t = 0; t < NT; ++t) tile[t * C::TLD + threadIdx.x] = R[t];
  }
  epi_sync();
  free_tmem();  // every fold warp's last tensor-memory read is done
  float* red = tile + (size_t)NT * C::TLD;
  epilogue_tile<__nv_bfloat16>(ep, tile, C::TLD, n0, m0, min(NT, M - m0), M, meta, red, /*staged=*/true, nullptr);
}

template <int NT>
__global__ void __launch_bounds__(TW_THREADS, 1) gemm_tcw_kernel(const __grid_constant__ CUtensorMap tmW,
                                                              const __grid_constant__ CUtensorMap tmX, int M, int N,
                                                              int K, int splits, EpiParams ep) {
  trace_entry(ep.trace);
  gemm_tcw_body<NT>(tmW, tmX, M, N, K, splits, ep);
  trace_exit(ep.trace);
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled_t encode_fn() {
  static PFN_encodeTiled_t fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled_t>(p);
  }
  return fn;
}

bool make_tmap_bf16(void* map_out, const void* ptr, long long rows, long long cols, int box_rows) {
  PFN_encodeTiled_t enc = encode_fn();
  if (!enc) return false;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (cols * 2) % 16 || cols % BK || box_rows > 256) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                   gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static_assert(sizeof(CUtensorMap) == TMAP_BYTES, "tensor map size");

int tc_token_tile(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

// CTAs a split-K launch aims for: two of these CTAs fit on an SM, and about a
// sixth of those slots stay free so that the next kernel's CTAs can become
// resident early (programmatic dependent launch) and start their weight loads.
// (Measured on the Qwen3-8B decode cycle: 1x, 1.3x, 1.5x, 1.7x, 1.85x, 2x the
// SM count gave 232, 236, 240-243, 242, 229, 215 tokens/s.)
int tc_split_target(int sm_count) { return sm_count * 5 / 3; }

int tc_splits(int N, int K, int target_ctas) {
  const int tiles = N / BM;
  const int nkb = K / BK;
  int s = (target_ctas + tiles / 2) / tiles;
  if (s < 1) s = 1;
  if (s > 8) s = 8;
  if (s > nkb / 4) s = nkb / 4 > 0 ? nkb / 4 : 1;
  return s;
}

size_t tc_workspace_floats(int M, int N, int splits, int nt) {
  if (splits <= 1) return 0;
  const size_t tiles = (size_t)(N / BM) * ((M + nt - 1) / nt);
  return tiles * splits * nt * BM;
}
size_t tc_counter_ints(int M, int N, int nt) { return (size_t)(N / BM) * ((M + nt - 1) / nt); }

bool tc_cluster_reduce(int nt, int splits);
static bool tc_cluster_reduce_qkv16(int splits);

template <int NT, int ST = 0>
static cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_tc_kernel<NT, ST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcCfg<NT, ST>::SMEM);
}

// Stages of the 16-token GEMMs: 6 (108 KB, two CTAs per SM), or 4 (73 KB, three
// CTAs per SM) with DF_GEMM16_STAGES=4 in the environment, so that a GEMM's
// CTAs can become resident (and prefetch their weights) next to the CTAs of
// the GEMM before it; DF_QKV_STAGES=4 applies the 4-stage ring to the
// key/value GEMM alone (measured slower in the decode chain: q|k|v 14.5
// against 13.8 us).  Same splits and MMA order either way: the same bits.
constexpr int QKV_LEAN_STAGES = 4;
static int lean16_mode() {  // 0: 6 stages; 1: 4 for the key/value GEMM; 2: 4 for every 16-token GEMM
  static int v = -1;
  if (v < 0) {
    const char* a = getenv("DF_GEMM16_STAGES");
    const char* q = getenv("DF_QKV_STAGES");
    v = (a && atoi(a) == 4) ? 2 : (q && atoi(q) == 4) ? 1 : 0;
  }
  return v;
}

// Set every token-tile variant's shared-memory limit up front (before any
// stream capture).
cudaError_t tc_prepare() {
  for (int nt = 16; nt <= 256; nt *= 2)
    for (int cz = 2; cz <= 8; ++cz) tc_cluster_reduce(nt, cz);
  cudaError_t e;
  for (int cz = 2; cz <= 8; ++cz) tc_cluster_reduce_qkv16(cz);
  if ((e = set_smem_attr<16>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<16, QKV_LEAN_STAGES>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<32>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<64>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<128>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<256>()) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(gemm_tcw_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, TwCfg<64>::SMEM)) !=
      cudaSuccess)
    return e;
  return cudaFuncSetAttribute(gemm_tcw_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, TwCfg<128>::SMEM);
}

// Whether clusters of cz CTAs of this token-tile variant can be resident
// (asked once per variant and size; DF_NO_CLUSTER=1 in the environment
// turns cluster reduction off).
template <int NT, int ST = 0>
static bool cluster_fits(int cz) {
  static int known[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};  // 0 unknown, 1 yes, 2 no
  if (cz < 2 || cz > 8) return false;
  if (!known[cz]) {
    const char* env = getenv("DF_NO_CLUSTER");
    bool ok = !(env && env[0] == '1');
    if (ok) {
      ok = set_smem_attr<NT, ST>() == cudaSuccess;
      cudaLaunchConfig_t c = {};
      c.gridDim = dim3(1, 1, cz);
      c.blockDim = dim3(128);
      c.dynamicSmemBytes = TcCfg<NT, ST>::SMEM;
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = 1;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = (unsigned)cz;
      c.attrs = a;
      c.numAttrs = 1;
      int n = 0;
      ok = ok && cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<NT, ST>, &c) == cudaSuccess && n > 0;
      cudaGetLastError();
    }
    known[cz] = ok ? 1 : 2;
  }
  return known[cz] == 1;
}

static bool tc_cluster_reduce_qkv16(int splits) { return cluster_fits<16, QKV_LEAN_STAGES>(splits); }

bool tc_cluster_reduce(int nt, int splits) {
  switch (nt) {
    case 16: return cluster_fits<16>(splits);
    case 32: return cluster_fits<32>(splits);
    case 64: return cluster_fits<64>(splits);
    case 128: return cluster_fits<128>(splits);
    case 256: return cluster_fits<256>(splits);
    default: return false;
  }
}

template <int NT, int ST = 0>
static cudaError_t launch_nt(const void* tmW, const void* tmX, int M, int N, int K, int splits, float* ws,
                             int* counters, const EpiParams& ep, bool creduce, cudaStream_t st) {
  using C = TcCfg<NT, ST>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<NT, ST>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(N / BM, (M + NT - 1) / NT, splits);
  const int cz = (creduce && splits > 1) ? splits : 1;
  return launch_kc(gemm_tc_kernel<NT, ST>, grid, dim3(128), (size_t)C::SMEM, st, cz,
                   *reinterpret_cast<const CUtensorMap*>(tmW), *reinterpret_cast<const CUtensorMap*>(tmX), M, N, K,
                   splits, ws, counters, cz > 1 ? 1 : 0, ep);
}

// Token tile of the serial-split form for an M-row GEMM of an N x K weight
// cut into `splits` K ranges (0: the split-K form).  Beyond 128 token rows
// the split-K form's 256-token tiles fill an SM each and its clusters run in
// waves; where the K ranges are short (K / splits <= 1024) that wave and
// reduction overhead dominates and the serial-split form with 64-token tiles
// is faster (at 256 rows: o projection 37.6 -> 28.8 us, q|k|v 31.0 -> 27.5);
// with long ranges (the down projection, 1536 per range: 56.2 against
// 69.4 us) or a single range (gate|up, the LM head: no cluster at all) the
// split-K form reads each weight tile once per 256 tokens and stays.  At 128
// rows the split-K form is as fast or faster everywhere.  DF_GEMM_WIDE=0 in
// the environment turns the serial-split form off; DF_GEMM_WIDE_MIN=m moves
// the row threshold.
int tc_wide_tile(int M, int N, int K, int splits) {
  static int min_m = -1;
  if (min_m < 0) {
    const char* off = getenv("DF_GEMM_WIDE");
    const char* mm = getenv("DF_GEMM_WIDE_MIN");
    min_m = (off && off[0] == '0') ? (1 << 30) : (mm ? atoi(mm) : 129);
    if (min_m < 1) min_m = 1;
  }
  (void)N;
  return (M >= min_m && splits > 1 && K / splits <= 1024) ? 64 : 0;
}

template <int NT>
static cudaError_t launch_nt_wide(const void* tmW, const void* tmX, int M, int N, int K, int splits,
                                  const EpiParams& ep, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tcw_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, TwCfg<NT>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((M + NT - 1) / NT, N / BM);
  return launch_k(gemm_tcw_kernel<NT>, grid, dim3(TW_THREADS), (size_t)TwCfg<NT>::SMEM, st,
                  *reinterpret_cast<const CUtensorMap*>(tmW), *reinterpret_cast<const CUtensorMap*>(tmX), M, N, K,
                  splits, ep);
}

cudaError_t launch_gemm_tcw(const void* tmW, const void* tmX, int nt, int M, int N, int K, int splits,
                            const EpiParams& ep, cudaStream_t st) {
  if (N % BM || K % BK || M < 1 || splits < 1 || splits > K / BK) return cudaErrorInvalidValue;
  switch (nt) {
    case 64: return launch_nt_wide<64>(tmW, tmX, M, N, K, splits, ep, st);
    case 128: return launch_nt_wide<128>(tmW, tmX, M, N, K, splits, ep, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_tc(const void* tmW, const void* tmX, int nt, int M, int N, int K, int splits, float* ws,
                           int* counters, const EpiParams& ep, cudaStream_t st, bool creduce) {
  if (N % BM || K % BK || M < 1 || splits < 1 || splits > K / BK) return cudaErrorInvalidValue;
  if (creduce && splits > 8) return cudaErrorInvalidValue;  // a portable cluster holds at most 8 CTAs
  switch (nt) {
    case 16:
      if (lean16_mode() == 2 || (lean16_mode() == 1 && ep.kind == EPI_QKV))  // same split and MMA order
        return launch_nt<16, QKV_LEAN_STAGES>(tmW, tmX, M, N, K, splits, ws, counters, ep,
                                              creduce && tc_cluster_reduce_qkv16(splits), st);
      return launch_nt<16>(tmW, tmX, M, N, K, splits, ws, counters, ep, creduce, st);
    case 32: return launch_nt<32>(tmW, tmX, M, N, K, splits, ws, counters, ep, creduce, st);
    case 64: return launch_nt<64>(tmW, tmX, M, N, K, splits, ws, counters, ep, creduce, st);
    case 128: return launch_nt<128>(tmW, tmX, M, N, K, splits, ws, counters, ep, creduce, st);
    case 256: return launch_nt<256>(tmW, tmX, M, N, K, splits, ws, counters, ep, creduce, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfk
