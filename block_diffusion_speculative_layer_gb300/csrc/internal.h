// Internal launch interface between the engine and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace dfk {

constexpr int TMAP_BYTES = 128;  // sizeof(CUtensorMap)

// Whether launches carry the programmatic-stream-serialization attribute
// (on by default; DF_NO_PDL=1 in the environment turns it off).
bool pdl_enabled();

// Launch a kernel with programmatic dependent launch allowed and, when the
// cluster shape has more than one CTA, thread-block clusters of that shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_kcl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, dim3 cluster,
                       Args... args) {
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = st;
  cudaLaunchAttribute a[2];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  int n = 1;
  if (cluster.x * cluster.y * cluster.z > 1) {
    a[1].id = cudaLaunchAttributeClusterDimension;
    a[1].val.clusterDim.x = cluster.x;
    a[1].val.clusterDim.y = cluster.y;
    a[1].val.clusterDim.z = cluster.z;
    n = 2;
  }
  c.attrs = a;
  c.numAttrs = n;
  return cudaLaunchKernelEx(&c, kernel, static_cast<KArgs>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_kc(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_z,
                      Args... args) {
  return launch_kcl(kernel, grid, block, smem, st, dim3(1, 1, cluster_z > 1 ? cluster_z : 1), args...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  return launch_kc(kernel, grid, block, smem, st, 1, args...);
}

// ---- tcgen05 GEMM (gemm_tc.cu)
bool make_tmap_bf16(void* map_out, const void* ptr, long long rows, long long cols, int box_rows);
// TMA map of one layer of a paged bf16 cache [page][k|v][Hkv][page_tokens][128]:
// 4-D (64 head dims, 2 halves, page_tokens, page x k|v x head), boxes of one
// page-half (page_tokens x 128 B), 128-byte swizzle.
bool make_tmap_kvcache(void* map_out, const void* base, int n_pages, int n_kv_heads, int page_tokens);
int tc_token_tile(int M);
cudaError_t tc_prepare();         // kernel attributes, once, before any stream capture
int tc_split_target(int sm_count);  // CTA count split-K aims for
int tc_splits(int N, int K, int target_ctas);  // split count for a target CTA count
size_t tc_workspace_floats(int M, int N, int splits, int nt);
bool tc_cluster_reduce(int nt, int splits);  // split-K by clusters for this variant and split count
size_t tc_counter_ints(int M, int N, int nt);
// Split-K partials are reduced across a cluster of the tile's `splits` CTAs
// through distributed shared memory (cluster_reduce) or, otherwise, through
// the workspace `ws` and the tile tickets `counters` (splits > 1 only).
cudaError_t launch_gemm_tc(const void* tmW, const void* tmX, int nt, int M, int N, int K, int splits, float* ws,
                           int* counters, const EpiParams& ep, cudaStream_t st, bool cluster_reduce = false);
// Serial-split form (one CTA per weight tile and token tile runs all `splits`
// K ranges and adds them in split order: bitwise the split-K form's result).
// nt is 64 or 128; the X map's box has nt rows.  tc_wide_tile(M, N, K,
// splits) is the engine's choice of nt for M token rows, 0 for the split-K form.
int tc_wide_tile(int M, int N, int K, int splits);
cudaError_t launch_gemm_tcw(const void* tmW, const void* tmX, int nt, int M, int N, int K, int splits,
                            const EpiParams& ep, cudaStream_t st);

// ---- fp32 SIMT GEMM + epilogue (gemm_simt.cu)
cudaError_t launch_gemm_f32(const float* x, const float* w, float* tmp, int M, int N, int K, const EpiParams& ep,
                            cudaStream_t st);

// ---- attention (attention.cu)
struct AttnParams {
  const void* q;          // [M][Hq*hd]
  void* out;              // [M][Hq*hd]
  int M;                  // rows
  int rows_per_seq;       // rows of one sequence (block size, or a prefill chunk)
  int n_seqs;             // sequences in this pass (rows are sequence-major)
  int Hq, Hkv, hd;
  const int* row_pos;     // [M] absolute positions
  const int* row_seq;     // [M] sequence slots
  int causal;             // 1: keys [0, pos]; 0: context [0, pos - slot) plus the whole block
  const void* cache;      // paged cache of this layer: [page][k|v][Hkv][page_tokens][hd]
  const int* page_table;  // [slot][pt_stride]
  int pt_stride, page_tokens, n_pages;
  const void* blk;        // block rows [k|v][Hkv][rows_cap][hd] (causal == 0)
  int rows_cap;
  int chunk;              // keys per split-KV chunk
  int n_chunk_slots;      // chunk slots per (row, head) in the partial buffers
  int grid_chunks;        // context chunks launched
  float* part_acc;        // [M][Hq][n_chunk_slots][hd]
  float2* part_ml;        // [M][Hq][n_chunk_slots]
  float scale_log2;       // log2(e) / sqrt(hd)
  int* err;
  const void* kv_map;     // host copy of a TMA map of `cache` (make_tmap_kvcache), or null
  unsigned long long* trace;  // in-situ timing of the launch (see trace_entry), or null
  int pipelined;          // bf16: the pipelined tcgen05 kernel (attn_tp_kernel) instead of attn_cl_kernel
  int cla;                // pipelined kernel: CTAs per cluster (2, 4, 8, 16; 0: the process default)
};
cudaError_t launch_attention(const AttnParams& p, bool bf16, cudaStream_t st);
int attention_launches(const AttnParams& p, bool bf16);  // kernels one launch_attention call makes
cudaError_t attention_prepare();  // kernel attributes, once, before any stream capture
// bf16, head_dim 128 (attention_mma.cu): tensor-core chunk partials for
// attn_combine, or (cluster) one kernel that also merges them in a cluster.
cudaError_t launch_attention_mma(const AttnParams& p, cudaStream_t st);
cudaError_t launch_attention_cluster(const AttnParams& p, cudaStream_t st);
cudaError_t launch_attention_tc(const AttnParams& p, cudaStream_t st);
// The pipelined tcgen05 cluster kernel (warp-specialised: TMA producer, MMA
// issuer, four softmax warps; S double-buffered in tensor memory).
cudaError_t launch_attention_tp(const AttnParams& p, cudaStream_t st);
cudaError_t attention_tp_prepare();  // kernel attributes, once, before any stream capture
bool attention_cluster_fits(const AttnParams& p);  // shapes the cluster kernel takes
cudaError_t attention_cluster_prepare();  // kernel attributes, once, before any stream capture
// One kernel whose bounded wait on a barrier nothing completes runs out and
// sets ERR_TIMEOUT in err (about two seconds); it returns normally.
cudaError_t launch_wait_probe(int* err, cudaStream_t st);

// ---- small kernels (misc.cu)
// h[m] = embed[tok[m]] (fp32), xraw[m] = the same row in the model dtype,
// ss[m][tile] = its sum of squares per 128-feature tile.
cudaError_t launch_embed(const void* embed, bool bf16, const int* tok, float* h, void* xraw, float* ss, int M, int d,
                         int vocab, int* err, cudaStream_t st);
// W[n][k] *= gain[k] (init only).
cudaError_t launch_scale_cols(void* w, bool bf16, long long rows, int cols, const float* gain, cudaStream_t st);
// out[m] = T(h[m] * rsqrt(mean(h[m]^2) + eps) * gain); optionally taps[m][tap][:] = T(h[m]).
// rows with row_pos[m] < 0 (if row_pos given) are skipped.
cudaError_t launch_rmsnorm(const float* h, int ldh, const float* gain, void* out, int ldo, bool bf16, int M, int d,
                           float eps, void* taps, int tap_index, const int* row_pos, cudaStream_t st);
cudaError_t launch_fill_u64(unsigned long long* p, unsigned long long v, int n, cudaStream_t st);
cudaError_t launch_argmax_finalize(const unsigned long long* amax, int* ids, int M, cudaStream_t st);
// Block rows for drafting (verify = 0: [bonus, MASK...]) or verification (verify = 1: [bonus, drafts...]);
// drafts are per slot: drafts[slot][B-1].
cudaError_t launch_prep_block(const int* batch_slots, int nseq, int B, const int* bonus, const int* bonus_pos,
                              const int* drafts, int mask_id, int verify, int* row_tok, int* row_pos, int* row_seq,
                              cudaStream_t st);
// Greedy acceptance: one warp per sequence.
cudaError_t launch_accept(const int* batch_slots, int nseq, int B, const int* row_tok, const int* ids, int* bonus,
                          int* bonus_pos, int* acc_out, int* n_out, int* inj_pos, cudaStream_t st);
// Drafts for the next verification, per slot: drafts[slot_b][i] = ids[b*B + 1 + i].
cudaError_t launch_collect_drafts(const int* ids, int nseq, int B, const int* batch_slots, int* drafts,
                                  cudaStream_t st);
// One greedy decode step: out[b][t] = ids[b]; row_tok[b] = ids[b]; row_pos[b] += 1.
cudaError_t launch_greedy_step(const int* ids, int nseq, int t, int n_new, int* out, int* row_tok, int* row_pos,
                               cudaStream_t st);
cudaError_t launch_copy_row_f32(const float* src, int lds, float* dst, int ldd, int rows, int cols, cudaStream_t st);

// ---- speculative sampling (sampling.cu)
// A row's sampling distribution over its fp32 logits: token i is kept when
// its logit's order key is above cut_key, or equal to it with i <= cut_idx;
// a kept token's mass is exp((l_i - m) * inv_t) in units of 2^-44 (inv_t = 0:
// greedy, the one kept token has mass 2^44); w_kept is the kept total.
struct SampleRow {
  float m;
  float inv_t;
  uint32_t cut_key;
  int cut_idx;
  unsigned long long w_kept;
};
constexpr int SAMPLE_MAX_VOCAB = 1 << 19;  // keeps a row's total mass below 2^63
constexpr float SAMPLE_MIN_TEMPERATURE = 1e-3f, SAMPLE_MAX_TEMPERATURE = 1e3f;
cudaError_t sampling_prepare();  // kernel attributes (staged shared memory), once, before any stream capture
bool sampling_args_ok(float temperature, float top_p);  // temperature 0 or in [1e-3, 1e3]; top_p in [0, 1]
float sampling_inv_t(float temperature);                // 0 for temperature 0
// st[r] for rows r of logits (row stride ld floats): largest logit, total
// mass and the nucleus for top_p < 1.  One 1024-thread block per row.
cudaError_t launch_sample_state(const float* logits, long long ld, int rows, int V, float inv_t, float top_p,
                                SampleRow* st, int* err, cudaStream_t s);
// out[r] = inverse-CDF draw from row r with u[b * u_ld + i - skip], where
// r = b * rows_per_seq + i; rows with i < skip are left alone.
cudaError_t launch_sample_draw(const float* logits, long long ld, int rows, int V, const SampleRow* st, const float* u,
                               int rows_per_seq, int u_ld, int skip, int* out, int* err, cudaStream_t s);
// probs[r][i] = probability of token i in row r (tests and the single-op entry point).
cudaError_t launch_sample_probs(const float* logits, long long ld, int rows, int V, const SampleRow* st, float* probs,
                                long long ldp, cudaStream_t s);
// u[b][j] = Philox uniform counts[slots[b]] + j of (seed, streams[slots[b]]), j < n; counts advance by n.
cudaError_t launch_cycle_uniforms(const int* slots, int nseq, int n, unsigned long long seed, const uint32_t* streams,
                                  unsigned long long* counts, float* u, int u_ld, cudaStream_t s);
// The speculative-sampling test of nseq drafted blocks (one block of threads each).
cudaError_t launch_accept_sampled(const int* slots, int nseq, int B, const int* drafts, int d_ld, const float* qlog,
                                  long long ldq, const SampleRow* qst, int q_seq_rows, int q_row0, const float* plog,
                                  long long ldp, const SampleRow* pst, int V, const float* u, int u_ld, int u0,
                                  int* bonus, int* bonus_pos, int* acc_out, int* n_out, int* inj_pos, int* k_out,
                                  int* tok_out, int* err, cudaStream_t s);

}  // namespace dfk
