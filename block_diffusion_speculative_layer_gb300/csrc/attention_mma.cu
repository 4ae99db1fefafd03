// bf16 attention over the paged caches on the tensor cores (mma.sync m16n8k16).
//
// Same split and masks as the CUDA-core kernel in attention.cu (fixed 64-key
// chunks counted from position 0, the drafter's block rows as one extra chunk,
// partials merged in chunk order by attn_combine), so verification and greedy
// decoding give bitwise the same rows.
//
// One CTA = one (chunk, KV head, 16-token tile); one warp per grouped query
// head, so a warp's 16 token rows form exactly one m16 tile.  The chunk's keys
// and values (64 x 128 bf16 each) are staged with 16-byte cp.async into shared
// memory with the 16-byte column blocks XOR-swizzled by key (conflict-free
// ldmatrix).  S = Q K^T (64 MMAs per warp), masked softmax statistics per row
// (quad shuffles), P kept in registers as the A operand of P V (64 MMAs), fp32
// accumulators.  A row's arithmetic never depends on the other rows.
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

}  // namespace dfk
