/*
 * dflash.h - C ABI of the GB300 DFlash draft-and-verify engine.
 *
 * The engine runs DFlash speculative decoding on one GPU: a target decoder
 * (RMSNorm, RoPE, grouped-query attention, SwiGLU) verifies blocks that a
 * small block-diffusion drafter proposes in one forward pass.  The drafter
 * is conditioned on hidden states of five target layers, fused by a light FC
 * + RMSNorm and injected as K/V into every drafter layer.
 *
 * Sources (web pages, by title and section):
 *   [ARCH]  "DFlash 的架构密码——扩散模型如何「寄生」在自回归模型上"
 *           (zhichai.net): 第一层 Feature Fusion, 第二层 KV Injection,
 *           第三层 Block Diffusion, 训练策略 (bonus-token anchors, shared
 *           embedding & LM head), 技术细节补充 (提取层数, 投影层, 稀疏注意力训练).
 *   [ABS]   "DFlash：基于块扩散的闪存推测解码方法" (ai-stack.site): 摘要
 *           (single forward pass, feature conditioning, lossless);
 *           实践 2 (block verification, keep up to the last correct token);
 *           实践 3 (the drafter never modifies the target's KV cache);
 *           实践 4 (temperature and top-p sampling, drafter and target aligned);
 *           实践 5 (pre-allocated activation pool, verification fused on the GPU);
 *           核心思想 step 3 (verification keeps the target's output distribution).
 *   [PRESS] DFlash press repost (zaocj.com): a single forward pass with
 *           bidirectional attention fills the 8-16 slots after the verified token.
 *
 * Conventions shared by every call
 *   - All sizes are explicit int32/int64.  Token ids are int32.
 *   - Weights are passed as DEVICE pointers in the canonical order given by
 *     df_weight_info(); df_init copies them into a library-owned arena, so the
 *     caller may free its copies once df_init returns.
 *   - Every other pointer named *_host is caller-owned HOST memory; pointers
 *     named *_dev are caller-owned DEVICE memory.
 *   - All GPU work is ordered on the stream passed to df_init (a cudaStream_t,
 *     or NULL for the legacy default stream).  Calls that return host-visible
 *     results synchronise that stream before returning.
 *   - Errors: every call returns a df_status; df_last_error() gives a message.
 *     Kernels report device-side failures (a bounded wait that ran out, an
 *     index outside its buffer) in a sticky error word; once set, later calls
 *     on the handle return DF_ECUDA or DF_ETIMEOUT.
 *   - The library never prints, never aborts and never falls back to the CPU.
 *
 * Environment switches (read once per process; each keeps the results
 * correct and exists to compare an implementation choice):
 *   DF_NO_PDL=1      launch kernels without programmatic dependent launch
 *   DF_NO_GRAPH=1    df_generate launches each cycle's kernels directly
 *                    instead of replaying captured CUDA graphs
 *   DF_GRAPH_CYCLES=k  draft+verify cycles per captured graph (1..8, default 4)
 *   DF_NO_CLUSTER=1  split-K partials through a workspace, not a cluster
 *   DF_ATTN_SPLIT=1  attention partials through global memory and a merge
 *                    kernel instead of the cluster kernel (other rounding)
 *   DF_ATTN_TC=1     attention math on tcgen05 (groups of <= 4 query heads;
 *                    other rounding; slower in its present serial form)
 *   DF_SPLIT_CTAS=n  the CTA count the engine's split-K choice aims for
 *                    (other rounding: the split counts change)
 * The switches marked "other rounding" change the fp32 summation order, so
 * results may differ in the last bits; verification and greedy decoding
 * under the same switches still agree bitwise.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct df_handle df_handle; /* opaque; owned by the library */

typedef enum {
  DF_OK = 0,
  DF_EINVAL = 1,   /* bad argument or unsupported shape */
  DF_ENOMEM = 2,   /* device allocation or page pool exhausted */
  DF_ECUDA = 3,    /* a CUDA call failed or a kernel flagged an error */
  DF_ETIMEOUT = 4, /* a bounded device-side wait ran out */
  DF_ESTATE = 5    /* call made in the wrong sequence state */
} df_status;

typedef enum { DF_FP32 = 0, DF_BF16 = 1 } df_dtype;

/* Model and capacity description.
 *   n_layers .. vocab : target decoder shape (head_dim 64 or 128).
 *   draft_layers      : drafter depth (same width as the target).
 *   block_size B      : slots per draft block, the bonus slot included, so a
 *                       cycle proposes B-1 drafts ([PRESS]: 8-16 slots).
 *   feat_layers[5]    : 1-based target layers whose outputs are fused; fill
 *                       with df_default_feat_layers() ([ARCH] 提取层数).
 *   max_batch         : sequences held at once; max_ctx: positions per sequence.
 *   page_tokens       : tokens per KV page (16).
 *   dtype             : DF_FP32 (plain fp32 FMA everywhere) or DF_BF16 (bf16
 *                       weights and GEMM operands, fp32 accumulation,
 *                       fp32 residual stream).
 *   mask_token_id     : id embedded into the drafter's masked slots (vocab-1).
 *   attn_kernel       : bf16 attention kernel for the whole handle (fixed, with
 *                       its cluster size, so that verification and greedy
 *                       decoding stay bitwise equal and a sequence decodes the
 *                       same alone or in a batch): DF_ATTN_MMA (1) the mma.sync
 *                       cluster kernel (lowest latency for one sequence up to
 *                       8K positions), DF_ATTN_PIPE (2) the warp-specialised
 *                       tcgen05 kernel (streams long contexts and batches
 *                       fastest) in clusters of DF_ATTN_PIPE_CLUSTER CTAs, or
 *                       DF_ATTN_PIPE_CLUSTER_ONE for a handle with max_batch 1,
 *                       DF_ATTN_AUTO (0) the pipelined kernel when max_batch >=
 *                       DF_ATTN_PIPE_MIN_BATCH or max_ctx > DF_ATTN_PIPE_MIN_CTX,
 *                       else the mma.sync kernel.  The two round differently.
 */
typedef struct {
  int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn, vocab;
  int32_t draft_layers, block_size;
  int32_t feat_layers[5];
  int32_t max_batch, max_ctx, page_tokens;
  int32_t dtype;
  int32_t mask_token_id;
  float rms_eps, rope_theta;
  int32_t attn_kernel;
} df_config;

enum { DF_ATTN_AUTO = 0, DF_ATTN_MMA = 1, DF_ATTN_PIPE = 2 };
#define DF_ATTN_PIPE_MIN_BATCH 2    /* DF_ATTN_AUTO: the pipelined kernel from this max_batch on, */
#define DF_ATTN_PIPE_MIN_CTX 8192   /* or for one sequence beyond this max_ctx */
#define DF_ATTN_PIPE_CLUSTER 4      /* the pipelined kernel's cluster size (CTAs) */
#define DF_ATTN_PIPE_CLUSTER_ONE 8  /* ... for a handle with max_batch 1 */

/* Per-handle counters.  k = accepted drafts in a cycle; a cycle emits k+1
 * tokens, so the mean accepted length is (accepted_drafts + cycles) / cycles. */
typedef struct {
  int64_t cycles;
  int64_t accepted_drafts;
  int64_t emitted_tokens;
  int64_t accept_hist[65]; /* histogram of k, k <= 64 */
  double draft_us;         /* summed device time of draft passes (CUDA events) */
  double verify_us;        /* summed device time of verify+accept+inject */
  double prefill_us;
  int64_t kernel_launches; /* this library's kernels launched */
  int64_t h2d_bytes;       /* host-to-device bytes copied by the engine */
  int64_t d2h_bytes;       /* device-to-host bytes copied by the engine */
  int64_t block_hist[33];  /* cycles run at each block size (df_set_block_range) */
} df_stats;

/* Device time per kernel class while profiling is on (df_profile_enable:
 * CUDA events around every launch, or the in-situ device-timer stamps).
 * bytes / flops are ALGORITHMIC: weights + inputs + outputs each counted once
 * (for a GEMM: N*K weights, M*K inputs, M*N outputs; for attention: the
 * visible keys and values plus queries and outputs), not measured traffic. */
typedef struct {
  char name[32];
  int64_t launches;
  double total_us;
  double bytes;
  double flops;
} df_kernel_stat;

/* Five feature layers sampled uniformly from layer 2 to the third-from-last
 * ([ARCH] 技术细节补充, 提取层数): s_i = 2 + round_half_up(i (L-4) / 4), 1-based.
 * DF_EINVAL if n_layers < 8 (five distinct layers need L >= 8). */
df_status df_default_feat_layers(int32_t n_layers, int32_t out[5]);

/* Number of weight tensors df_init expects for cfg. */
int32_t df_num_weights(const df_config* cfg);

/* Canonical weight list.  For index i fills a NUL-terminated name (<= 31
 * chars), the number of dims (1 or 2) and the shape.  Matrices are
 * [out_features, in_features] row-major; vectors are RMSNorm gains.  Order:
 * embed[V,d]; per target layer: attn_norm, wq, wk, wv, wo, mlp_norm, w_gate,
 * w_up, w_down; final_norm; lm_head[V,d]; fc[d,5d]; fc_norm; per drafter
 * layer the same nine; d_final_norm.  The drafter has no embedding or LM head
 * of its own: it reuses the target's ([ARCH] Shared Embedding & LM Head). */
df_status df_weight_info(const df_config* cfg, int32_t index, char name[32], int32_t* ndim, int64_t shape[2]);

/* Create an engine.  weights: n_weights DEVICE pointers in canonical order,
 * each dense row-major in cfg->dtype (fp32, or bf16 bit patterns).  stream: a
 * cudaStream_t (may be NULL).  Allocates the weight arena, both paged KV caches
 * (target, and the drafter's injected context cache, kept apart per [ABS]
 * 实践 3) and every activation buffer up front ([ABS] 实践 5).  *out receives
 * the handle; on failure *out is NULL and the status says why. */
df_status df_init(const df_config* cfg, const void* const* weights, int32_t n_weights, void* stream,
                  df_handle** out);

/* Prefill sequence slot seq (0 <= seq < max_batch, slot must be empty):
 * run the target over prompt_host[0..len), write its KV pages, take the argmax
 * at the last position as the first bonus token (*bonus_out), fuse the prompt's
 * feature-layer states and inject them into the drafter's context cache
 * ([ARCH] 第一层: after the target's prefill). */
df_status df_prefill(df_handle* h, int32_t seq, const int32_t* prompt_host, int32_t len, int32_t* bonus_out);

/* Draft one block for each listed sequence: one drafter forward pass over
 * [bonus, MASK x (B-1)] at the bonus position, attending to the injected
 * context and bidirectionally inside the block, nothing across blocks
 * ([ARCH] 第三层, 稀疏注意力训练).  Slot i (1..B-1) gives draft i by argmax
 * through the shared LM head.  drafts_host: [nseq][B-1] (may be NULL). */
df_status df_draft_block(df_handle* h, const int32_t* seqs_host, int32_t nseq, int32_t* drafts_host);

/* Verify and accept.  The target runs once over [bonus, d_1..d_{B-1}] for each
 * sequence; k = the longest prefix with d_i equal to the target's greedy token
 * before it; the cycle emits d_1..d_k and the target's token after them (the
 * next bonus), rolls the target KV cache back to the verified length and
 * injects the fused features of the k+1 verified positions into the drafter's
 * context cache ([ABS] 实践 2; [ARCH] bonus-token anchors).
 * drafts_host: [nseq][B-1] drafts to verify, or NULL to verify the drafts of
 * the last df_draft_block for these sequences.
 * accepted_host: [nseq][B] emitted tokens (first n_host[i] valid);
 * n_host: [nseq] = k+1.  Either output may be NULL. */
df_status df_verify_accept(df_handle* h, const int32_t* seqs_host, int32_t nseq, const int32_t* drafts_host,
                           int32_t* accepted_host, int32_t* n_host);

/* Whole speculative generation for nseq prompts (packed back to back in
 * prompts_host, lengths lens_host): prefill each into slots 0..nseq-1, then
 * draft/verify cycles until n_new tokens per sequence; tokens past n_new are
 * dropped.  Cycles run in groups replayed from captured CUDA graphs and
 * chained on the device, with one host synchronisation per group.  A
 * sequence that reaches n_new inside a group still runs that group's
 * remaining cycles, and they count in the stats.
 * out_host: [nseq][n_new].  stats (may be NULL) receives this call's
 * counters.  Slots are released at the end. */
df_status df_generate(df_handle* h, const int32_t* prompts_host, const int32_t* lens_host, int32_t nseq,
                      int32_t n_new, int32_t* out_host, df_stats* stats);

/* Block size of df_generate / df_generate_sampled's cycles ([ABS] 实践 2:
 * a long block rolls back more often, so the block size may follow how
 * predictable the text is).  With b_min == b_max every cycle drafts and
 * verifies b_max slots (b_max - 1 drafts); with b_min < b_max the first
 * group of cycles uses b_max and each later group df_block_size_for() of the
 * tokens per cycle seen so far (an average over the groups, each weighted
 * half as much as the one after it).  A cycle of b slots verifies b rows per
 * sequence, so the target's GEMMs and attention shrink with it; the output
 * is the target's greedy (or sampled) stream whatever the block sizes.
 * 2 <= b_min <= b_max <= the configured block size; default: both equal to
 * it.  Stays in force for the handle until changed. */
df_status df_set_block_range(df_handle* h, int32_t b_min, int32_t b_max);

/* The block-size rule on the host: the smallest power of two that is at
 * least 2 x tokens_per_cycle, clamped to [b_min, b_max] (b_max itself where
 * the power of two passes it).  -1 for arguments outside 2 <= b_min <= b_max
 * <= 32 or a negative rate. */
int32_t df_block_size_for(double tokens_per_cycle, int32_t b_min, int32_t b_max);

/* df_generate with sampling instead of greedy decoding ([ABS] 实践 4; 核心思想
 * step 3).  A token's sampling distribution is softmax(logits / temperature)
 * over the fp32 logits of the shared LM head, restricted to the nucleus (the
 * fewest most probable tokens whose mass reaches top_p; tokens of equal logit
 * in index order) and renormalised; temperature 0 is the greedy argmax, and
 * then the output equals df_generate's.  The drafter and the target use the
 * same temperature and top_p.  Each cycle draws draft i from the drafter's
 * distribution at slot i, keeps d_i while u_i * q_i(d_i) < p_i(d_i) (q the
 * drafter's, p the target's distribution before d_i), and draws the token
 * after the kept drafts from max(0, p - q) renormalised at the first
 * rejection (from p where that is zero), or from the target's distribution
 * after a fully kept block: the standard speculative-sampling test, under
 * which the output follows the target's own sampling distribution.
 * Masses are fixed-point integers (units of 2^-44 of the row's largest
 * exp((l - max) / T)), so every draw is exact integer arithmetic and does
 * not depend on the batch; masses below 2^-45 of the largest are zero.
 * Uniforms: sequence i of the call uses Philox4x32-10 stream i of `seed`
 * (df_op_philox_uniforms), one uniform for the first token after its prompt,
 * then 2B - 1 per cycle (B - 1 draft draws, B - 1 tests, the final draw).
 * temperature: 0, or in [1e-3, 1e3]; top_p in [0, 1] (1: no nucleus);
 * vocab <= 2^19.  DF_EINVAL otherwise.  The first call allocates two fp32
 * logit buffers of max_batch * B rows.  Other arguments as df_generate. */
df_status df_generate_sampled(df_handle* h, const int32_t* prompts_host, const int32_t* lens_host, int32_t nseq,
                              int32_t n_new, float temperature, float top_p, uint64_t seed, int32_t* out_host,
                              df_stats* stats);

/* Failure-detection check.  Launches one kernel whose bounded wait on a
 * barrier that nothing completes runs out after the limit every wait of the
 * engine's kernels has (about two seconds), records the timeout in the
 * handle's error word and returns.  The call returns DF_ETIMEOUT and leaves
 * the handle failed (later calls return DF_ECUDA); the CUDA context stays
 * usable, so a new handle works.  For tests of the error path only. */
df_status df_debug_wait_probe(df_handle* h);

/* Per-sequence acceptance of the last df_generate / df_generate_sampled
 * call: out[k] = cycles of sequence `seq` (its index in that call) that kept
 * k drafts (k >= 32 counted at 32), over the cycles that emitted its tokens
 * (a group's cycles after a sequence reached n_new are not counted here).
 * DF_EINVAL if seq is outside the last call's sequences. */
df_status df_generate_accept_hist(const df_handle* h, int32_t seq, int64_t out[33]);

/* Plain token-by-token greedy decoding of the target on the GPU, with the
 * same kernels as verification: the lossless reference the speculative
 * output must equal bit for bit.  Same arguments as df_generate. */
df_status df_greedy_reference(df_handle* h, const int32_t* prompts_host, const int32_t* lens_host,
                              int32_t nseq, int32_t n_new, int32_t* out_host);

/* Release a sequence slot (its pages return to the pool). */
df_status df_reset_seq(df_handle* h, int32_t seq);

/* Counters accumulated since df_init or the last df_reset_stats. */
df_status df_get_stats(const df_handle* h, df_stats* out);
df_status df_reset_stats(df_handle* h);

/* Current verified length and bonus token of a slot (host mirror). */
df_status df_seq_info(const df_handle* h, int32_t seq, int32_t* length, int32_t* bonus);

void df_destroy(df_handle* h);
const char* df_last_error(const df_handle* h);

/* Kernel-class profiling (off by default), in one of two modes.
 *   on = 1 (serialised): every launch is bracketed by two CUDA events on the
 *     engine's stream (df_generate then launches its cycles directly, without
 *     graphs); the events are read at the next synchronising call.  Launches
 *     no longer overlap, so the times include each launch's ramp and tail.
 *   on = 2 (in situ): df_generate's cycles run as usual (captured graphs,
 *     programmatic dependent launch), and every GEMM and cluster-attention
 *     launch of a cycle stamps the device timer at its first CTA's entry and
 *     its last CTA's exit.  A cycle's timeline is cut at those exit stamps:
 *     each launch is charged the time from the previous stamped exit (the
 *     cycle's first entry for the first) to its own exit, so the classes add
 *     up to the cycles' device time and kernels that are not stamped (norms,
 *     embedding, control) are charged to the launch after them.  Only
 *     draft + verify cycles are recorded (not prefill).
 * on = 0 turns profiling off.  df_profile_read fills up to max entries
 * (classes: gemm (layer GEMMs), lm_head, fuse, inject, attention, rmsnorm,
 * embed, control) and clears them. */
df_status df_profile_enable(df_handle* h, int32_t on);
df_status df_profile_read(df_handle* h, df_kernel_stat* out, int32_t max, int32_t* n);

/* ------------------------------------------------------------------------
 * Inspection (tests).  df_debug_read copies a buffer of the last pass to
 * host memory as float32 (bf16 widened exactly):
 *   DF_DBG_TAPS          [rows][5][d]  feature-layer outputs of the last target pass
 *   DF_DBG_LOGITS        [rows][V]     logits of the last target pass (needs debug on)
 *   DF_DBG_DRAFT_LOGITS  [rows][V]     logits of the last drafter pass (needs debug on)
 *   DF_DBG_DRAFT_HIDDEN  [rows][d]     drafter output before its final norm
 *   DF_DBG_CTX           [rows][d]     fused context features of the last injection
 *   DF_DBG_HIDDEN        [rows][d]     target output before the final norm
 *   DF_DBG_TARGET_LAYERS [L+1][M][d]   fp32 residual rows of the last target pass (M
 *                                      rows) entering each of its L layers, then the
 *                                      last layer's output (needs debug on)
 *   DF_DBG_DRAFT_LAYERS  [Ld+1][M][d]  the same for the last drafter pass
 * rows is the row count of that pass (*rows_out; (layers + 1) x M for the
 * two per-layer buffers).  With debug on, the fused
 * LM-head argmax also stores the logits it reduces; off by default.
 * ------------------------------------------------------------------------ */
enum {
  DF_DBG_TAPS = 1,
  DF_DBG_LOGITS = 2,
  DF_DBG_DRAFT_LOGITS = 3,
  DF_DBG_DRAFT_HIDDEN = 4,
  DF_DBG_CTX = 5,
  DF_DBG_HIDDEN = 6,
  DF_DBG_TARGET_LAYERS = 7,
  DF_DBG_DRAFT_LAYERS = 8
};
df_status df_debug_enable(df_handle* h, int32_t on);
df_status df_debug_read(df_handle* h, int32_t what, float* out_host, int64_t max_floats, int32_t* rows_out);

/* Device address of a weight as the engine holds it (embed, lm_head, ...):
 * lets a test confirm that the drafter and the target share one embedding
 * and one LM head.  which: 0 target embedding, 1 drafter embedding, 2 target
 * LM head, 3 drafter LM head. */
df_status df_debug_weight_ptr(const df_handle* h, int32_t which, uint64_t* addr);

/* ------------------------------------------------------------------------
 * Single operations on caller device buffers (per-kernel tests, microbench).
 * All pointers are *_dev DEVICE pointers; dtype follows the argument's type.
 * Each call is stream-ordered on `stream` and does not synchronise.
 * ------------------------------------------------------------------------ */

/* y[M][N] = x[M][K] . w[N][K]^T, bf16 operands, fp32 accumulation and output
 * (the tcgen05 GEMM the engine uses; fixed K order, so each output does not
 * depend on M).  N % 128 == 0, K % 64 == 0, M >= 1, 16-byte aligned pointers.
 * splits: 0 = the engine's choice for (N, K) (about 5/3 of the SM count in
 * CTAs), else the split-K count.  With 2..8 splits the split CTAs of a tile
 * form a thread-block cluster and add their partials in split order through
 * distributed shared memory; otherwise (or with DF_NO_CLUSTER=1 in the
 * environment) the partials go through a workspace allocated on `stream`
 * for the call.  Both give bitwise the same y.
 * token_tile: 0 = the engine's choice for M; 16, 32, 64, 128 or 256 = the
 * split-K form with that many token rows per tile; -64 or -128 = the
 * serial-split form with 64 or 128 token rows per tile, which the engine
 * uses beyond 128 token rows: one CTA per (weight tile, token tile) runs
 * every K range of its tile in order, each into its own tensor-memory
 * accumulator, and adds the partials in split order (bitwise the split-K
 * form's y, no cluster, no workspace). */
df_status df_op_gemm_bf16(const void* x_dev, const void* w_dev, float* y_dev, int32_t M, int32_t N, int32_t K,
                          int32_t splits, int32_t token_tile, void* stream);

/* One attention launch of the engine on caller-owned device buffers: the
 * causal attention of the target's verify pass or the drafter's block
 * attention ([ARCH] 第三层 Block Diffusion and 稀疏注意力训练: the block sees
 * the injected context before its anchor and, in both directions, its own
 * block rows; nothing of another sequence).  bf16, head_dim 128, 16-token
 * pages, scale 1/sqrt(128), fp32 softmax.
 *   q_dev / out_dev  [nseq * rows_per_seq][n_q_heads * 128] (rows sequence-major)
 *   cache_dev        one layer of the paged cache: [n_pages][k|v][n_kv_heads][16][128]
 *   page_table_dev   [slots][pt_stride]: page ids of each slot's positions 0, 16, 32, ...
 *   row_pos_dev      [rows]: each row's absolute position (< 0: row skipped)
 *   row_seq_dev      [rows]: each row's slot in the page table
 *   blk_dev          causal == 0: the block rows' keys and values
 *                    [k|v][n_kv_heads][rows_cap][128] (rows_cap >= rows); else ignored
 *   causal           1: row at position p sees cache positions 0..p;
 *                    0: row j of a block anchored at a sees cache positions
 *                    0..a-1 and every row of its own block (rows_per_seq <= 64)
 *   max_len          bound on the cache positions any row sees (sets the grid)
 *   kernel           DF_ATTN_MMA or DF_ATTN_PIPE (see df_config.attn_kernel)
 *   cluster_ctas     DF_ATTN_PIPE: CTAs per cluster, 2, 4, 8 or 16 (0: 4,
 *                    or DF_ATTN_PIPE_CLA from the environment); the chunks
 *                    are split over a cluster's CTAs, so the size changes
 *                    the rounding; DF_ATTN_MMA: 0 (16 where placeable)
 *   err_dev          device int receiving the kernels' sticky error bits
 *                    (1: a bounded wait ran out, 2: a page id outside the cache)
 * Query heads per KV head <= 8.  Stream-ordered, no synchronisation, no
 * allocation; DF_EINVAL for shapes the cluster kernels do not take. */
df_status df_op_attention_bf16(const void* q_dev, void* out_dev, const void* cache_dev, int32_t n_pages,
                               const int32_t* page_table_dev, int32_t pt_stride, const int32_t* row_pos_dev,
                               const int32_t* row_seq_dev, const void* blk_dev, int32_t rows_cap, int32_t nseq,
                               int32_t rows_per_seq, int32_t n_q_heads, int32_t n_kv_heads, int32_t causal,
                               int32_t max_len, int32_t kernel, int32_t cluster_ctas, int32_t* err_dev,
                               void* stream);

/* ids[m] = argmax_v (x[m] . w_lm[v]) over V rows of w_lm (bf16 [V][K]),
 * fp32 logits, lowest index on ties; logits are never written.  V % 128 == 0. */
df_status df_op_lmhead_argmax_bf16(const void* x_dev, const void* wlm_dev, int32_t* ids_dev, int32_t M, int32_t V,
                                   int32_t K, void* stream);

/* The GEMM of df_op_gemm_bf16 without any device allocation.  The pages
 * have no counterpart of this call: it serves callers that may not allocate
 * device memory while they run (a process whose memory is reserved up front
 * by its own pool, a latency-critical loop that cannot afford the
 * synchronisation of an allocation and its release).  It always adds the
 * split partials through a workspace (never through a cluster), and instead
 * of a cudaMallocAsync'd one it uses fixed scratch compiled into the library:
 * DF_NOALLOC_WS_FLOATS floats of split-K partial sums and DF_NOALLOC_TICKETS
 * tile tickets, held by every GPU that loads the library until the process
 * exits.  Arguments and result as df_op_gemm_bf16; returns DF_EINVAL, before
 * launching anything, when the shape's split-K scratch (tiles x splits x
 * token tile x 128 floats) or its ticket count exceeds those limits.
 * The first call on a device looks up the scratch's device address with that
 * device current; make that first call before any stream capture.  The
 * address belongs to the device's CUDA context: after that context is reset
 * (cudaDeviceReset) the next call looks it up again, so make that call
 * before any capture too.  All calls
 * on a device share the one scratch, which keeps the last call's contents
 * (the tickets a call uses are cleared on its stream first): calls that can
 * overlap on the GPU (different streams without ordering) race and must not
 * be issued. */
#define DF_NOALLOC_WS_FLOATS (1 << 20)
#define DF_NOALLOC_TICKETS 4096
df_status df_op_gemm_bf16_noalloc(const void* x_dev, const void* w_dev, float* y_dev, int32_t M, int32_t N,
                                  int32_t K, int32_t splits, int32_t token_tile, void* stream);

/* Drafter-step microbenchmark (the drafter's own kernels alone, at a chosen
 * context length and batch).  Uses free slots 0..nseq-1 and releases them:
 * fills the drafter's context cache for positions [0, ctx_len) of each
 * sequence by fusing and injecting the caller's feature rows (taps_host:
 * [taps_rows][5][d] float32, reused cyclically; nseq*B <= taps_rows <= 512),
 * then runs `iters` times: fusion and injection of one block of feature rows
 * per sequence, and one drafter pass over [bonus, MASK x (B-1)] at position
 * ctx_len.  us_out receives the mean device microseconds per iteration of
 * [0] the fusion GEMM (its RMSNorm is folded into the injection), [1] the
 * injection GEMM, [2] block attention summed over the drafter layers, [3] the
 * LM-head argmax, [4] the drafter's layer GEMMs (CUDA events around each
 * launch), and [5] one whole drafter pass timed without per-launch events
 * ([ARCH] 第一层/第二层/第三层 and Shared LM Head). */
df_status df_bench_drafter_step(df_handle* h, int32_t nseq, int32_t ctx_len, const float* taps_host,
                                int32_t taps_rows, int32_t iters, double us_out[6]);

/* Device time of the tcgen05 GEMM alone: y = x . w^T launched `iters` times
 * back to back on `stream` (tensor maps, and a split-K workspace where one is
 * used, made once),
 * timed with CUDA events around the whole run; *us_per_launch receives the
 * mean.  Same shape rules as df_op_gemm_bf16.  Synchronises `stream`. */
df_status df_op_bench_gemm_bf16(const void* x_dev, const void* w_dev, float* y_dev, int32_t M, int32_t N, int32_t K,
                                int32_t splits, int32_t token_tile, int32_t iters, void* stream, float* us_per_launch);

/* ---- speculative sampling, one operation at a time ----------------------
 * The pieces of df_generate_sampled on caller-owned device buffers, for
 * tests and for callers with their own loop.  Logit rows are fp32 [rows][V]
 * (row stride V), V in [1, 2^19]; temperature and top_p as in
 * df_generate_sampled.  err_dev (may be NULL): a device int that receives
 * the sticky error bits of the kernels (2: a draw or a nucleus search found
 * no token, which only invalid input can cause).  Each call is stream-ordered
 * on `stream`, allocates its scratch on that stream and does not synchronise. */

/* The Philox4x32-10 block function on the host (Salmon, Moraes, Dror and
 * Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), from the same
 * source as the device generator: out = philox(counter ctr, key). */
df_status df_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* u_dev[j] = uniform offset + j of (seed, stream_id), j < n: word
 * (offset + j) mod 4 of the Philox4x32-10 block for counter ((offset + j) / 4
 * as two 32-bit words, stream_id, 0) and key (seed as two 32-bit words),
 * taken as (word >> 8) * 2^-24. */
df_status df_op_philox_uniforms(uint64_t seed, uint32_t stream_id, uint64_t offset, int32_t n, float* u_dev,
                                void* stream);

/* probs_dev[r][v] = probability of token v in row r's sampling distribution
 * (the kept fixed-point mass over the row's kept total, rounded to fp32). */
df_status df_op_sampling_probs(const float* logits_dev, int32_t rows, int32_t V, float temperature, float top_p,
                               float* probs_dev, int32_t* err_dev, void* stream);

/* idx_dev[r] = the lowest index j whose cumulative mass in row r exceeds
 * u_dev[r] x (row r's total mass): an inverse-CDF draw; u in [0, 1). */
df_status df_op_sample_draw(const float* logits_dev, int32_t rows, int32_t V, float temperature, float top_p,
                            const float* u_dev, int32_t* idx_dev, int32_t* err_dev, void* stream);

/* The speculative-sampling test of nseq drafted blocks of B slots (2 <= B
 * <= 32).  drafts_dev [nseq][B-1]: d_1..d_{B-1}; q_logits_dev [nseq][B-1][V]:
 * the drafter's logits at slots 1..B-1; p_logits_dev [nseq][B][V]: the
 * target's logits at slots 0..B-1 (row j predicts the token after slot j);
 * u_dev [nseq][B]: B-1 test uniforms then the final draw's.  k_dev[b] = kept
 * drafts, tok_dev[b] = the token after them (see df_generate_sampled). */
df_status df_op_accept_sampled(const int32_t* drafts_dev, const float* q_logits_dev, const float* p_logits_dev,
                               int32_t nseq, int32_t B, int32_t V, float temperature, float top_p,
                               const float* u_dev, int32_t* k_dev, int32_t* tok_dev, int32_t* err_dev,
                               void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
