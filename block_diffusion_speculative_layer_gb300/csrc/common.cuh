// Shared device-side definitions of the DFlash engine (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfk {

// Bits of the sticky device error word.
enum : int {
  ERR_TIMEOUT = 1,     // a bounded mbarrier wait ran out
  ERR_BOUNDS = 2,      // an index fell outside its buffer; the access was skipped
  ERR_TMEM = 4,        // tensor-memory allocation returned an unexpected address
};

__device__ __forceinline__ void flag_error(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

// Programmatic dependent launch.  Every kernel of the engine is launched so
// that it may start while the kernel before it drains: pdl_wait() blocks until
// that kernel has finished and its writes are visible (a no-op when launched
// normally); pdl_trigger() lets the next kernel start its own prologue.
// Kernels trigger first and then wait: a kernel launched early does nothing
// before its own wait but read constant weights, and a kernel can only be
// launched once every CTA of the one before it is resident, so a chain of
// early launches never holds back a kernel it depends on.  (The GEMM lets its
// weight loads run ahead of the wait.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// In-situ launch timing: each CTA's thread 0 folds its entry and exit times
// (the %globaltimer, ns) into trace[0] = max ~entry (so ~trace[0] is the
// first CTA's entry) and trace[1] = max exit.  trace null: off.
__device__ __forceinline__ unsigned long long device_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace_entry(unsigned long long* trace) {
  if (trace && threadIdx.x == 0) atomicMax(trace, ~device_ns());
}
__device__ __forceinline__ void trace_exit(unsigned long long* trace) {
  if (trace && threadIdx.x == 0) atomicMax(trace + 1, device_ns());
}

template <typename T> struct Cvt;
template <> struct Cvt<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Cvt<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Monotonic map of an fp32 value to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Packed (value, index) key: max picks the largest value, then the lowest index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  return ((unsigned long long)ordered_bits(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

// What a GEMM does with its fp32 result tile.
enum EpiKind : int {
  EPI_STORE = 0,   // out[m][n] = acc (out type = T)
  EPI_STORE_F32,   // out_f32[m][n] = acc
  EPI_RESID,       // resid[m][n] += acc (fp32 residual stream)
  EPI_SWIGLU,      // tiles hold 64 gate rows then the 64 matching up rows:
                   // out[m][n/2 + f] = silu(gate) * up
  EPI_QKV,         // rotary embedding + scatter of q / k / v
  EPI_ARGMAX,      // per-row packed max over the tile's logits (+ optional store)
  EPI_STORE_SS,    // out[m][n] = acc (type T) and this tile's partial sum of acc^2 per row
};

// Where K/V rows of EPI_QKV go.
enum KvDest : int {
  KV_PAGED = 0,  // paged cache: [layer][page][k|v][head][page_tokens][hd]
  KV_ROWS = 1,   // row buffer:  [k|v][head][row][hd] (drafter block keys/values)
};

struct EpiParams {
  int kind;
  void* out;          // EPI_STORE / EPI_SWIGLU / EPI_QKV (q) / EPI_ARGMAX (debug logits, fp32)
  int ldo;            // row stride of out (elements)
  float* resid;       // EPI_RESID
  int ldr;
  // EPI_QKV
  int q_dim;          // features [0, q_dim) are queries (0 for pure K/V injection)
  int kv_dim;         // features per K (and per V) block
  int head_dim;
  int n_kv_heads;
  int kv_dest;        // KvDest
  void* kv_base;      // cache base (KV_PAGED) or row buffer (KV_ROWS)
  long long layer_stride;   // elements between layers of the paged cache
  int layer0;         // first cache layer written (injection spans several)
  const int* page_table;    // [seq][pt_stride]
  int pt_stride;
  int page_tokens;
  int n_pages;        // bounds check on page ids
  int rows_cap;       // KV_ROWS: rows per (k|v, head) plane
  const int* row_pos; // [M] absolute position of row m; < 0 = row is inactive
  const int* row_seq; // [M] sequence slot of row m
  const float2* rope; // [pos][hd/2] (cos, sin)
  int rope_rows;      // positions in the table (bounds check)
  // EPI_ARGMAX
  unsigned long long* amax;  // [M]
  // RMSNorm folded into the GEMM: the input rows were not normalised; each
  // output row is scaled by rsqrt(sum(ss_in[m][:]) / d + eps) (the norm's
  // gain is folded into the weight's columns).
  const float* ss_in;        // [M][ss_tiles] partial sums of squares of the input rows; null: no scaling
  int ss_tiles;
  float inv_d;
  float eps;
  // EPI_RESID / EPI_STORE_SS: what the next (normalising) GEMM reads
  void* xraw;                // [M][ldx] the new rows in the model dtype; null: none
  int ldx;
  float* ss_out;             // [M][ss_tiles] this tile's partial sum of squares; null: none
  void* tap;                 // [M][5][N] feature-layer tap of the new rows; null: none
  int tap_index;
  int* err;
  // In-situ timing (null: off): trace[0] = max over CTAs of ~(entry time),
  // trace[1] = max over CTAs of the exit time, in device-timer nanoseconds.
  unsigned long long* trace;
  // weight tiles past the shared-memory ring prefetched into L2 before the
  // programmatic wait (split-K form; 0 = none)
  int l2_prefetch;
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Per-row facts an epilogue needs, staged in shared memory once per tile so
// that the element loops never wait on a chain of dependent global loads.
struct RowMeta {
  int pos;      // absolute position (< 0: inactive row)
  int page;     // KV page of that position (paged K/V destinations), else -1
  float scale;  // 1/rms of the input row (folded RMSNorm), else unused
};

// Partial sum of squares of one row's 128 tile values: each warp reduces its
// 32 lanes in a fixed xor tree, then the four warp sums add in warp order.
__device__ __forceinline__ void row_sumsq(float v, int r, float* red) {
  float q = v * v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  if ((threadIdx.x & 31) == 0) red[r * 4 + (threadIdx.x >> 5)] = q;
}

constexpr int EPI_BATCH = 16;  // rows whose global loads are issued together

// The epilogue's barrier: named barrier 1 over its 128 threads (the first four
// warps), so that a kernel with further warps (producer, MMA issuer) can run
// the epilogue on its first four warps alone.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Stage the per-row facts the epilogue needs (positions, KV pages, 1/rms of
// folded norms) into meta.  Run by `nthr` threads (whole warps) with index
// `tid`; the caller synchronises before epilogue_tile reads meta.
__device__ __forceinline__ void epilogue_stage(const EpiParams& ep, int m0, int rows, int M, RowMeta* meta, int tid,
                                               int nthr) {
  rows = min(rows, M - m0);
  const bool need_meta = ep.kind == EPI_QKV || (ep.kind == EPI_RESID && ep.row_pos);
  if (need_meta) {
    for (int r = tid; r < rows; r += nthr) {
      const int m = m0 + r;
      const int pos = ep.row_pos[m];
      meta[r].pos = pos;
      meta[r].page = (ep.kind == EPI_QKV && ep.kv_dest == KV_PAGED && pos >= 0)
                         ? ep.page_table[(size_t)ep.row_seq[m] * ep.pt_stride + pos / ep.page_tokens]
                         : -1;
    }
  }
  if (ep.ss_in) {
    // 1/rms per row: 8 threads per row each add every 8th tile partial, then a
    // fixed xor tree joins them (the same order for every row and batch).
    const int per_pass = nthr >> 3;
    for (int rb = 0; rb < rows; rb += per_pass) {
      const int r = rb + (tid >> 3), j = tid & 7;
      float part = 0.f;
      if (r < rows) {
        const float* sp = ep.ss_in + (size_t)(m0 + r) * ep.ss_tiles;
        for (int t = j; t < ep.ss_tiles; t += 8) part += sp[t];
      }
      part += __shfl_xor_sync(0xffffffffu, part, 4);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      if (r < rows && j == 0) meta[r].scale = rsqrtf(part * ep.inv_d + ep.eps);
    }
  }
}

// Global operands of the epilogue that do not depend on the accumulator (the
// residual rows, the rotary factors), copied into shared memory with cp.async
// as soon as the accumulator is complete: the copies' latency overlaps the
// accumulator drain and the split-K reduction, and each thread waits for its
// own copies only when the epilogue reads them.  (Loads into a register array
// that the epilogue indexes by a run-time row would live in local memory, and
// storing them there waits for the loads at once.)  Only for tiles of at most
// EPI_BATCH rows.  `buf` holds EPI_PRE_FLOATS floats of shared memory: thread
// f keeps row r's residual at buf[r * 128 + f] (EPI_RESID), or its (cosine,
// sine) at ((float2*)buf)[r * 128 + f] (EPI_QKV).
constexpr int EPI_PRE_FLOATS = 2 * EPI_BATCH * 128;
struct EpiPre {
  float* buf;
};
__device__ __forceinline__ void cp_async_f1(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_f2(float2* dst, const float2* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_own() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Start the copies for rows [0, rows) of the tile at (m0, n0); all 128 threads
// call it, thread f for feature n0 + f.  Returns whether `pre` will be filled.
__device__ __forceinline__ bool epilogue_preload(const EpiParams& ep, int n0, int m0, int rows, int M,
                                                 const RowMeta* meta, const EpiPre& pre) {
  rows = min(rows, M - m0);
  if (rows > EPI_BATCH) return false;
  const int f = threadIdx.x & 127;
  const int n = n0 + f;
  if (ep.kind == EPI_RESID) {
    for (int i = 0; i < rows; ++i) cp_async_f1(pre.buf + i * 128 + f, ep.resid + (size_t)(m0 + i) * ep.ldr + n);
    return true;
  }
  if (ep.kind == EPI_QKV) {
    const int hd = ep.head_dim, half = hd >> 1;
    const int dim = n & (hd - 1);
    bool rotated = true;  // queries and keys; values are not rotated
    if (n >= ep.q_dim) {
      const int r2 = (n - ep.q_dim) % (2 * ep.kv_dim);
      rotated = r2 < ep.kv_dim;
    }
    float2* cs = reinterpret_cast<float2*>(pre.buf);
    for (int i = 0; i < rows; ++i) {
      const int pos = meta[i].pos;
      if (rotated && pos >= 0 && pos < ep.rope_rows)
        cp_async_f2(cs + i * 128 + f, ep.rope + (size_t)pos * half + (dim & (half - 1)));
      else
        cs[i * 128 + f] = make_float2(1.f, 0.f);
    }
    return true;
  }
  return false;
}

// Apply the epilogue to one result tile held in shared memory.
//   tile[r * ld + f] = acc for row m0 + r, feature n0 + f, f in [0, 128),
//   r in [0, rows), rows <= M - m0.  Called by exactly the 128 threads of
//   warps 0-3 (one per feature column).  meta has room for `rows` entries;
//   if `staged`, the caller already ran epilogue_stage into it and
//   synchronised.  red holds 4 floats per row.  Synchronises those 128
//   threads (epi_sync), so all of them call it.
template <typename T>
__device__ void epilogue_tile(const EpiParams& ep, const float* tile, int ld, int n0, int m0, int rows, int M,
                              RowMeta* meta, float* red, bool staged = false, const EpiPre* pre = nullptr) {
  const int f = threadIdx.x & 127;
  const int n = n0 + f;
  rows = min(rows, M - m0);
  if (!staged) {
    epilogue_stage(ep, m0, rows, M, meta, threadIdx.x & 127, 128);
    epi_sync();
  }
  const bool scaled = ep.ss_in != nullptr;
  switch (ep.kind) {
    case EPI_STORE: {
      T* out = reinterpret_cast<T*>(ep.out);
      for (int r = 0; r < rows; ++r) out[(size_t)(m0 + r) * ep.ldo + n] = Cvt<T>::from_f(tile[r * ld + f]);
    } break;
    case EPI_STORE_F32: {
      float* out = reinterpret_cast<float*>(ep.out);
      for (int r = 0; r < rows; ++r) out[(size_t)(m0 + r) * ep.ldo + n] = tile[r * ld + f];
    } break;
    case EPI_RESID: {
      // Add the residual and store it; also write the new rows for the next
      // normalising GEMM (model dtype, tap, sum of squares).
      auto row = [&](int r, float old) {
        const int m = m0 + r;
        const bool live = !(ep.row_pos && meta[r].pos < 0);
        const float nv = live ? old + tile[r * ld + f] : old;
        if (live) ep.resid[(size_t)m * ep.ldr + n] = nv;
        if (ep.xraw) reinterpret_cast<T*>(ep.xraw)[(size_t)m * ep.ldx + n] = Cvt<T>::from_f(nv);
        if (ep.tap) reinterpret_cast<T*>(ep.tap)[((size_t)m * 5 + ep.tap_index) * ep.ldr + n] = Cvt<T>::from_f(nv);
        if (ep.ss_out) row_sumsq(nv, r, red);
      };
      if (pre) {
        // residuals already on their way to shared memory: a compact row loop
        cp_async_wait_own();
#pragma unroll 1
        for (int r = 0; r < rows; ++r) row(r, pre->buf[r * 128 + f]);
      } else {
        // issue EPI_BATCH residual loads together, then the rows
        for (int rb = 0; rb < rows; rb += EPI_BATCH) {
          float old[EPI_BATCH];
#pragma unroll
          for (int i = 0; i < EPI_BATCH; ++i) {
            const int r = rb + i;
            old[i] = (r < rows) ? ep.resid[(size_t)(m0 + r) * ep.ldr + n] : 0.f;
          }
#pragma unroll
          for (int i = 0; i < EPI_BATCH; ++i) {
            if (rb + i >= rows) break;
            row(rb + i, old[i]);
          }
        }
      }
      if (ep.ss_out) {
        epi_sync();
        for (int r = threadIdx.x; r < rows; r += 128)
          ep.ss_out[(size_t)(m0 + r) * ep.ss_tiles + (n0 >> 7)] =
              ((red[r * 4 + 0] + red[r * 4 + 1]) + red[r * 4 + 2]) + red[r * 4 + 3];
      }
    } break;
    case EPI_STORE_SS: {
      T* out = reinterpret_cast<T*>(ep.out);
      for (int r = 0; r < rows; ++r) {
        const float v = tile[r * ld + f];
        out[(size_t)(m0 + r) * ep.ldo + n] = Cvt<T>::from_f(v);
        row_sumsq(v, r, red);
      }
      epi_sync();
      for (int r = threadIdx.x; r < rows; r += 128)
        ep.ss_out[(size_t)(m0 + r) * ep.ss_tiles + (n0 >> 7)] =
            ((red[r * 4 + 0] + red[r * 4 + 1]) + red[r * 4 + 2]) + red[r * 4 + 3];
    } break;
    case EPI_SWIGLU: {
      // 128 threads handle (row, gate feature) pairs: 64 features x 2 rows per pass.
      T* out = reinterpret_cast<T*>(ep.out);
      const int g = f & 63;
      const int rsub = f >> 6;
      for (int r = rsub; r < rows; r += 2) {
        const float sc = scaled ? meta[r].scale : 1.f;
        const float gate = tile[r * ld + g] * sc;
        const float up = tile[r * ld + 64 + g] * sc;
        out[(size_t)(m0 + r) * ep.ldo + (n0 >> 1) + g] = Cvt<T>::from_f(silu_f(gate) * up);
      }
    } break;
    case EPI_QKV: {
      const int hd = ep.head_dim;
      const int half = hd >> 1;
      const int dim = n & (hd - 1);
      const int partner = f ^ half;
      int kind;  // 0 = q, 1 = k, 2 = v
      int layer = 0, head = 0;
      if (n < ep.q_dim) {
        kind = 0;
      } else {
        int r2 = n - ep.q_dim;
        const int per_layer = 2 * ep.kv_dim;
        layer = r2 / per_layer;
        r2 -= layer * per_layer;
        kind = 1 + r2 / ep.kv_dim;
        head = (r2 % ep.kv_dim) / hd;
      }
      const size_t page_elems = (size_t)2 * ep.n_kv_heads * ep.page_tokens * hd;
      // the (scaled, rotated) value of row r, given its rotary factors
      auto value = [&](int r, float2 cs) {
        const float sc = scaled ? meta[r].scale : 1.f;
        float v = tile[r * ld + f] * sc;
        if (kind < 2) {
          const float p = tile[r * ld + partner] * sc;
          v = (dim < half) ? (v * cs.x - p * cs.y) : (v * cs.x + p * cs.y);
        }
        return v;
      };
      // store row r: queries to `out`, keys and values to the cache
      auto store = [&](int r, float v) {
        const int m = m0 + r;
        const int pos = meta[r].pos;
        if (kind == 0) {
          reinterpret_cast<T*>(ep.out)[(size_t)m * ep.ldo + n] = Cvt<T>::from_f(v);
          return;
        }
        T* base = reinterpret_cast<T*>(ep.kv_base);
        const int kv = kind - 1;
        size_t off;
        if (ep.kv_dest == KV_PAGED) {
          const int page = meta[r].page;
          if (page < 0 || page >= ep.n_pages) {
            flag_error(ep.err, ERR_BOUNDS);
            return;
          }
          off = (size_t)(ep.layer0 + layer) * ep.layer_stride + (size_t)page * page_elems +
                ((size_t)(kv * ep.n_kv_heads + head) * ep.page_tokens + (pos % ep.page_tokens)) * hd + dim;
        } else {
          if (m >= ep.rows_cap) {
            flag_error(ep.err, ERR_BOUNDS);
            return;
          }
          off = ((size_t)(kv * ep.n_kv_heads + head) * ep.rows_cap + m) * hd + dim;
        }
        base[off] = Cvt<T>::from_f(v);
      };
      // rows without a position are skipped; a rotated row past the table is an error
      auto usable = [&](int r) {
        const int pos = meta[r].pos;
        if (pos < 0) return false;
        if (kind < 2 && pos >= ep.rope_rows) {
          flag_error(ep.err, ERR_BOUNDS);
          return false;
        }
        return true;
      };
      if (pre) {
        // rotary factors already on their way to shared memory: a compact row loop
        cp_async_wait_own();
        const float2* cs = reinterpret_cast<const float2*>(pre->buf);
#pragma unroll 1
        for (int r = 0; r < rows; ++r)
          if (usable(r)) store(r, value(r, cs[r * 128 + f]));
      } else {
        for (int rb = 0; rb < rows; rb += EPI_BATCH) {
          // the batch's rotary factors first (independent read-only loads)
          float2 cs[EPI_BATCH];
#pragma unroll
          for (int i = 0; i < EPI_BATCH; ++i) {
            const int r = rb + i;
            cs[i] = make_float2(1.f, 0.f);
            if (r >= rows || kind == 2) continue;
            const int pos = meta[r].pos;
            if (pos >= 0 && pos < ep.rope_rows) cs[i] = __ldg(ep.rope + (size_t)pos * half + (dim & (half - 1)));
          }
#pragma unroll
          for (int i = 0; i < EPI_BATCH; ++i) {
            const int r = rb + i;
            if (r >= rows) break;
            if (usable(r)) store(r, value(r, cs[i]));
          }
        }
      }
    } break;
    case EPI_ARGMAX: {
      // One warp reduces 32 features of a row; four keys per row meet in one atomicMax each.
      float* dbg = reinterpret_cast<float*>(ep.out);
      for (int r = 0; r < rows; ++r) {
        const int m = m0 + r;
        const float v = tile[r * ld + f];
        if (dbg) dbg[(size_t)m * ep.ldo + n] = v;
        unsigned long long key = argmax_key(v, n);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
          key = other > key ? other : key;
        }
        if ((threadIdx.x & 31) == 0) atomicMax(ep.amax + m, key);
      }
    } break;
  }
}

}  // namespace dfk
