// Host engine of the DFlash draft-and-verify cycle and its C ABI.
//
// One handle holds one model on one GPU: a weight arena (target, drafter,
// one shared embedding and LM head), a paged target KV cache, a paged drafter
// context cache filled by KV injection, pre-allocated activation buffers,
// the split-K and split-KV workspaces of the non-cluster paths, and the
// per-sequence state (bonus token and its position) on the device.  A cycle
// launches only this library's kernels and reads back one small result
// (accepted tokens and their count); df_generate replays groups of cycles
// from CUDA graphs and reads a group's results after one synchronisation.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <array>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "dflash.h"
#include "internal.h"

using namespace dfk;

namespace {

constexpr int ATTN_CHUNK = 64;
constexpr int PREFILL_CHUNK = 512;

constexpr int KMAX_CYCLES = 8;  // most draft+verify cycles in one captured graph
constexpr size_t MAX_GRAPHS = 8;  // captured cycle graphs kept per handle

struct Tmap {
  alignas(64) uint8_t b[TMAP_BYTES];
};

struct Linear {
  void* ptr = nullptr;  // [N][K] row-major
  int N = 0, K = 0;
  Tmap tm;              // bf16 only: TMA map with 128-row boxes
};

struct Layer {
  float* attn_norm = nullptr;
  Linear qkv, wo;
  float* mlp_norm = nullptr;
  Linear gu, down;  // gu: 64 gate rows then the 64 matching up rows, per 128-row tile
};

struct SeqHost {
  bool active = false;
  int len = 0;    // verified positions = position of the bonus token
  int bonus = -1;
  std::vector<int> pages;  // page ids in position order
};

}  // namespace

struct df_handle {
  df_config cfg{};
  cudaStream_t st = nullptr;
  bool bf16 = false;
  size_t esz = 4;
  int d = 0, hd = 0, Hq = 0, Hkv = 0, F = 0, V = 0, L = 0, Ld = 0, B = 0, qdim = 0, kvdim = 0, qkv_n = 0;
  int sm_count = 152;
  bool attn_pipe = false;  // bf16 attention on the pipelined tcgen05 kernel (df_config.attn_kernel)
  int attn_cla = 4;        // its cluster size (CTAs), fixed for the handle
  int split_target = 253;  // CTAs a split-K GEMM aims for (DF_SPLIT_CTAS overrides tc_split_target)
  int l2_prefetch = 0;     // weight tiles a GEMM prefetches into L2 past its ring before its wait (DF_GEMM_L2PF)
  int tap_of_layer[1024];  // zero-based layer index -> tap slot (or -1)
  int Mmax = 0;

  std::vector<void*> allocs;
  void* arena = nullptr;
  std::vector<Layer> tl, dl;
  void* embed = nullptr;
  Linear lm_head, fc, inj;
  float *final_norm = nullptr, *fc_norm = nullptr, *d_final_norm = nullptr;

  int PT = 16, pages_per_seq = 0, n_pages = 0;
  void *kv_t = nullptr, *kv_d = nullptr;
  std::vector<Tmap> kvmap_t, kvmap_d;  // bf16: TMA maps of each cache layer (attention)
  long long layer_stride = 0;
  int* d_pt = nullptr;
  std::vector<int> free_pages;
  std::vector<SeqHost> seqs;

  int *d_bonus = nullptr, *d_bonus_pos = nullptr;
  int *d_row_tok = nullptr, *d_row_pos = nullptr, *d_row_seq = nullptr, *d_inj_pos = nullptr, *d_ids = nullptr;
  int *d_slots = nullptr, *d_drafts = nullptr, *d_acc = nullptr, *d_n = nullptr, *d_gen = nullptr;
  unsigned long long* d_amax = nullptr;

  float* h = nullptr;
  void *xb = nullptr, *q = nullptr, *attn = nullptr, *act = nullptr, *taps = nullptr, *ctx = nullptr, *blk = nullptr;
  void* xraw = nullptr;          // GEMM input rows, not normalised (model dtype)
  float *ss = nullptr, *ss_ctx = nullptr;  // per-row, per-128-feature-tile sums of squares
  float* tmp = nullptr;
  float *dbg_logits = nullptr, *dbg_dlogits = nullptr, *dbg_dh = nullptr, *dbg_th = nullptr;
  float *dbg_tl = nullptr, *dbg_dl = nullptr;  // [layers + 1][rows][d] residual rows entering each layer, then the output
  float* ws = nullptr;
  int* counters = nullptr;
  float* part_acc = nullptr;
  float2* part_ml = nullptr;
  int n_chunk_slots = 0;
  float2* rope = nullptr;
  int* d_err = nullptr;
  int* h_pin = nullptr;  // pinned host staging for per-cycle results
  size_t h_pin_ints = 0;

  std::map<std::tuple<uintptr_t, int, int>, Tmap> xmaps;
  df_stats stats{};
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  cudaEvent_t cev[4 * KMAX_CYCLES] = {};  // draft/verify bracket events of each cycle of a graph
  int graph_cycles = 4;  // cycles df_generate captures into one graph (DF_GRAPH_CYCLES, 1..KMAX_CYCLES)
  std::string err;
  bool debug = false;
  bool failed = false;
  // graph replay of the decode cycle (df_generate)
  bool use_graphs = true;
  int graph_ready_cycles = 0;        // eager cycles run by this handle (the first sets kernel attributes)
  // in-situ timing (df_profile_enable mode 2): per stamped launch of the
  // cycles being recorded, its class, launch count and algorithmic bytes;
  // d_trace[2i], d_trace[2i + 1] are its stamps (see trace_entry)
  struct TraceSlot {
    int cls, n;
    double bytes, flops;
  };
  bool tracing = false;
  unsigned long long* d_trace = nullptr;
  std::vector<TraceSlot> trace_meta;
  struct GraphRec {
    cudaGraphExec_t exec = nullptr;
    int64_t launches = 0, h2d = 0, d2h = 0;  // counted again at each replay
    std::vector<TraceSlot> trace_meta;      // stamped launches of the graph (in-situ timing)
  };
  std::map<std::vector<int>, GraphRec> graphs;  // by slots, cycle count, block size (and sampling arguments)
  std::vector<int> glast;                       // key of the graph whose slots d_gslots holds
  // block size per cycle group (df_set_block_range): fixed at B unless blk_min < blk_max
  int blk_min = 0, blk_max = 0;
  // per sequence of the last df_generate call: histogram of k over the cycles
  // that emitted its tokens
  std::vector<std::array<int64_t, 33>> gen_khist;
  int* d_gslots = nullptr;
  cudaStream_t gstream = nullptr;    // capture/replay stream, joined to the caller's stream by events
  cudaEvent_t gjoin[2] = {nullptr, nullptr};
  // kernel-class profiling
  bool profiling = false;
  std::vector<cudaEvent_t> evpool;
  size_t ev_used = 0;
  struct Pending {
    int cls, e0, e1, n;
    double bytes, flops;
  };
  std::vector<Pending> pending;
  df_kernel_stat prof[8];
  int rows_last_target = 0, rows_last_draft = 0, rows_last_ctx = 0, rows_last_logits = 0;
  // speculative sampling (df_generate_sampled): the LM heads keep fp32 logits
  // and the cycle draws drafts, tests them and draws the final token
  bool sampling = false;
  float samp_inv_t = 0.f, samp_top_p = 1.f;
  unsigned long long samp_seed = 0;
  float *d_qlog = nullptr, *d_plog = nullptr;    // [max_batch * B][V] drafter / target logits
  SampleRow *d_qst = nullptr, *d_pst = nullptr;  // [max_batch * B] their sampling rows
  float* d_u = nullptr;                          // [max_batch][2B] uniforms of the current cycle
  uint32_t* d_ustream = nullptr;                 // [max_batch] generator stream of each slot
  unsigned long long* d_ucount = nullptr;        // [max_batch] uniforms each slot has used
};

namespace {

df_status fail(df_handle* h, df_status s, const std::string& msg) {
  if (h) h->err = msg;
  return s;
}

#define CK(expr)                                                                               \
  do {                                                                                         \
    cudaError_t e_ = (expr);                                                                   \
    if (e_ != cudaSuccess) {                                                                   \
      H->failed = true;                                                                        \
      return fail(H, DF_ECUDA, std::string(#expr) + ": " + cudaGetErrorString(e_));            \
    }                                                                                          \
  } while (0)

#define CKS(expr)                \
  do {                           \
    df_status s_ = (expr);       \
    if (s_ != DF_OK) return s_;  \
  } while (0)


// Kernel classes for profiling: the layer GEMMs, the LM-head GEMM (fused
// argmax), the fusion GEMM with its norm, the injection GEMM, attention, the
// layer norms, the embedding gather and the small control kernels.
enum { PC_GEMM = 0, PC_LMHEAD, PC_FUSE, PC_INJECT, PC_ATTN, PC_NORM, PC_EMBED, PC_CTRL, PC_N };
const char* const PC_NAMES[PC_N] = {"gemm", "lm_head", "fuse", "inject", "attention", "rmsnorm", "embed", "control"};
constexpr size_t EV_POOL = 4096;

// Read every pending event pair (the stream is synchronised first).
void prof_resolve(df_handle* H) {
  if (H->pending.empty()) {
    H->ev_used = 0;
    return;
  }
  cudaStreamSynchronize(H->st);
  for (const auto& p : H->pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, H->evpool[p.e0], H->evpool[p.e1]) == cudaSuccess) {
      df_kernel_stat& k = H->prof[p.cls];
      k.launches += p.n;
      k.total_us += 1000.0 * ms;
      k.bytes += p.bytes;
      k.flops += p.flops;
    }
  }
  H->pending.clear();
  H->ev_used = 0;
}

int ev_take(df_handle* H) {
  if (H->ev_used >= H->evpool.size()) prof_resolve(H);
  if (H->ev_used >= H->evpool.size()) return -1;
  return (int)H->ev_used++;
}

constexpr size_t TRACE_MAX = 8192;  // stamped launches per recorded run of cycles

// Counts this library's launches; with profiling on, brackets them with
// events; with in-situ timing on, gives GEMM and attention launches a stamp
// slot (tp, passed to the kernel).
struct ProfScope {
  df_handle* H;
  int cls, n, e0 = -1;
  double bytes, flops;
  unsigned long long* tp = nullptr;
  ProfScope(df_handle* h, int c, int nlaunch, double b = 0.0, double f = 0.0)
      : H(h), cls(c), n(nlaunch), bytes(b), flops(f) {
    H->stats.kernel_launches += n;
    if (H->profiling) {
      e0 = ev_take(H);
      if (e0 >= 0) cudaEventRecord(H->evpool[e0], H->st);
    }
    const bool stamped = c == PC_GEMM || c == PC_LMHEAD || c == PC_FUSE || c == PC_INJECT || c == PC_ATTN;
    if (H->tracing && stamped && H->trace_meta.size() < TRACE_MAX) {
      tp = H->d_trace + 2 * H->trace_meta.size();
      H->trace_meta.push_back({c, n, b, f});
    }
  }
  ~ProfScope() {
    if (!H->profiling || e0 < 0) return;
    const int e1 = ev_take(H);
    if (e1 < 0) return;
    cudaEventRecord(H->evpool[e1], H->st);
    H->pending.push_back({cls, e0, e1, n, bytes, flops});
  }
};

// In-situ timing: read the stamps of the launches in `meta` (the stream is
// synchronised) and charge each launch the time from the previous stamped
// exit (the first launch's entry for the first one) to its own exit.
cudaError_t trace_collect(df_handle* H, const std::vector<df_handle::TraceSlot>& meta) {
  if (meta.empty()) return cudaSuccess;
  std::vector<unsigned long long> t(2 * meta.size());
  cudaError_t e = cudaMemcpy(t.data(), H->d_trace, t.size() * 8, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  // DF_TRACE_FILE=<path>: also append every stamped launch (class, entry ns, exit ns) to that file
  static const char* dump_path = getenv("DF_TRACE_FILE");
  FILE* dump = dump_path ? fopen(dump_path, "a") : nullptr;
  unsigned long long prev = 0;
  for (size_t i = 0; i < meta.size(); ++i) {
    const unsigned long long entry = ~t[2 * i], exit = t[2 * i + 1];
    if (t[2 * i] == 0 || exit == 0) continue;  // not stamped (a path without stamps)
    if (dump) fprintf(dump, "%s %llu %llu\n", PC_NAMES[meta[i].cls], entry, exit);
    if (prev == 0) prev = entry;
    const unsigned long long dt = exit > prev ? exit - prev : 0ull;
    prev = exit > prev ? exit : prev;
    df_kernel_stat& k = H->prof[meta[i].cls];
    k.launches += meta[i].n;
    k.total_us += 1e-3 * (double)dt;
    k.bytes += meta[i].bytes;
    k.flops += meta[i].flops;
  }
  if (dump) fclose(dump);
  return cudaSuccess;
}

// Host<->device copies on the engine's stream, counted for the end-to-end byte totals.
cudaError_t h2d(df_handle* H, void* dst, const void* src, size_t bytes) {
  H->stats.h2d_bytes += (int64_t)bytes;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, H->st);
}
cudaError_t d2h(df_handle* H, void* dst, const void* src, size_t bytes) {
  H->stats.d2h_bytes += (int64_t)bytes;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, H->st);
}

df_status dalloc(df_handle* H, void** p, size_t bytes) {
  if (bytes == 0) bytes = 256;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    (void)cudaGetLastError();
    return fail(H, DF_ENOMEM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed");
  }
  H->allocs.push_back(*p);
  return DF_OK;
}
template <typename P>
df_status dalloc_t(df_handle* H, P** p, size_t bytes) {
  void* v = nullptr;
  df_status s = dalloc(H, &v, bytes);
  *p = reinterpret_cast<P*>(v);
  return s;
}

int feat_default(int L, int i) { return 2 + (i * (L - 4) + 2) / 4; }

// ---------------------------------------------------------------- weight list
struct WSpec {
  std::string name;
  int ndim;
  long long s0, s1;
};

std::vector<WSpec> weight_specs(const df_config& c) {
  std::vector<WSpec> w;
  const long long d = c.d_model, F = c.d_ffn, V = c.vocab, qd = (long long)c.n_q_heads * c.head_dim,
                  kd = (long long)c.n_kv_heads * c.head_dim;
  auto layer = [&](const std::string& p) {
    w.push_back({p + ".attn_norm", 1, d, 0});
    w.push_back({p + ".wq", 2, qd, d});
    w.push_back({p + ".wk", 2, kd, d});
    w.push_back({p + ".wv", 2, kd, d});
    w.push_back({p + ".wo", 2, d, qd});
    w.push_back({p + ".mlp_norm", 1, d, 0});
    w.push_back({p + ".w_gate", 2, F, d});
    w.push_back({p + ".w_up", 2, F, d});
    w.push_back({p + ".w_down", 2, d, F});
  };
  w.push_back({"embed", 2, V, d});
  for (int l = 0; l < c.n_layers; ++l) layer("t" + std::to_string(l));
  w.push_back({"final_norm", 1, d, 0});
  w.push_back({"lm_head", 2, V, d});
  w.push_back({"fc", 2, d, 5 * d});
  w.push_back({"fc_norm", 1, d, 0});
  for (int l = 0; l < c.draft_layers; ++l) layer("d" + std::to_string(l));
  w.push_back({"d_final_norm", 1, d, 0});
  return w;
}

df_status validate(const df_config* c, std::string& why) {
  auto bad = [&](const char* m) {
    why = m;
    return DF_EINVAL;
  };
  if (!c) return bad("null config");
  if (c->n_layers < 8 || c->n_layers > 1000) return bad("n_layers must be in [8, 1000]");
  if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads) return bad("bad head counts");
  if (c->n_q_heads / c->n_kv_heads > 8) return bad("query heads per KV head must be <= 8");
  if (c->d_model % 128 || c->d_model <= 0) return bad("d_model must be a multiple of 128");
  if ((c->n_q_heads * c->head_dim) % 128 || (c->n_kv_heads * c->head_dim) % 128)
    return bad("query and KV widths must be multiples of 128");
  if (c->d_ffn % 64 || c->d_ffn <= 0) return bad("d_ffn must be a multiple of 64");
  if (c->vocab % 128 || c->vocab <= 0) return bad("vocab must be a multiple of 128");
  if (c->draft_layers < 1) return bad("draft_layers must be >= 1");
  if (c->block_size < 2 || c->block_size > 32) return bad("block_size must be in [2, 32]");
  if (c->max_batch < 1 || c->max_ctx < c->block_size + 1) return bad("bad max_batch / max_ctx");
  if (c->page_tokens < 1) return bad("page_tokens must be >= 1");
  if (c->dtype != DF_FP32 && c->dtype != DF_BF16) return bad("dtype must be DF_FP32 or DF_BF16");
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab) return bad("mask_token_id out of range");
  for (int i = 0; i < 5; ++i) {
    if (c->feat_layers[i] < 1 || c->feat_layers[i] > c->n_layers - 1)
      return bad("feat_layers must be 1-based layers in [1, n_layers-1]");
    if (i && c->feat_layers[i] <= c->feat_layers[i - 1]) return bad("feat_layers must increase");
  }
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.f)) return bad("bad rms_eps / rope_theta");
  if (c->attn_kernel < DF_ATTN_AUTO || c->attn_kernel > DF_ATTN_PIPE) return bad("bad attn_kernel");
  return DF_OK;
}

// ---------------------------------------------------------------- GEMM dispatch
df_status xmap(df_handle* H, const void* ptr, int K, int nt, const void** out) {
  auto key = std::make_tuple(reinterpret_cast<uintptr_t>(ptr), K, nt);
  auto it = H->xmaps.find(key);
  if (it == H->xmaps.end()) {
    Tmap t;
    if (!make_tmap_bf16(t.b, ptr, H->Mmax, K, nt)) return fail(H, DF_ECUDA, "tensor map encode failed (activations)");
    it = H->xmaps.emplace(key, t).first;
  }
  *out = it->second.b;
  return DF_OK;
}

EpiParams epi(df_handle* H, int kind) {
  EpiParams e{};
  e.kind = kind;
  e.err = H->d_err;
  e.head_dim = H->hd;
  e.n_kv_heads = H->Hkv;
  e.kv_dim = H->kvdim;
  e.page_table = H->d_pt;
  e.pt_stride = H->pages_per_seq;
  e.page_tokens = H->PT;
  e.n_pages = H->n_pages;
  e.rope = H->rope;
  e.rope_rows = H->cfg.max_ctx;
  e.layer_stride = H->layer_stride;
  e.rows_cap = H->Mmax;
  return e;
}

// Algorithmic bytes of a GEMM launch: weights, inputs and outputs once each.
double gemm_bytes(const df_handle* H, const Linear& W, int M, const EpiParams& ep) {
  const double es = (double)H->esz;
  double out = 0.0;
  switch (ep.kind) {
    case EPI_STORE: case EPI_QKV: out = (double)M * W.N * es; break;
    case EPI_STORE_F32: out = (double)M * W.N * 4; break;
    case EPI_RESID: out = (double)M * W.N * 8; break;
    case EPI_SWIGLU: out = (double)M * (W.N / 2) * es; break;
    case EPI_ARGMAX: out = (double)M * 8; break;
  }
  return (double)W.N * W.K * es + (double)M * W.K * es + out;
}

df_status gemm(df_handle* H, const Linear& W, const void* X, int M, const EpiParams& ep, int cls = PC_GEMM) {
  if (M <= 0) return DF_OK;
  ProfScope ps(H, cls, H->bf16 ? 1 : 2, gemm_bytes(H, W, M, ep), 2.0 * M * W.N * W.K);
  if (H->bf16) {
    const int splits = tc_splits(W.N, W.K, H->split_target);
    const int wide = tc_wide_tile(M, W.N, W.K, splits);
    const int nt = wide ? wide : tc_token_tile(M);
    const void* tmX = nullptr;
    CKS(xmap(H, X, W.K, nt, &tmX));
    EpiParams e = ep;
    e.trace = ps.tp;
    e.l2_prefetch = H->l2_prefetch;
    if (wide) {
      CK(launch_gemm_tcw(W.tm.b, tmX, nt, M, W.N, W.K, splits, e, H->st));
    } else {
      CK(launch_gemm_tc(W.tm.b, tmX, nt, M, W.N, W.K, splits, H->ws, H->counters, e, H->st,
                        tc_cluster_reduce(nt, splits)));
    }
  } else {
    CK(launch_gemm_f32(reinterpret_cast<const float*>(X), reinterpret_cast<const float*>(W.ptr), H->tmp, M, W.N, W.K,
                       ep, H->st));
  }
  return DF_OK;
}

// ---------------------------------------------------------------- passes
// LM head with fused argmax over rows [row0, row0 + M) of xb -> d_ids[0..M).
df_status lm_head_argmax(df_handle* H, int M, float* dbg) {
  {
    ProfScope ps(H, PC_CTRL, 1);
    CK(launch_fill_u64(H->d_amax, 0ull, M, H->st));
  }
  EpiParams e = epi(H, EPI_ARGMAX);
  e.amax = H->d_amax;
  e.out = dbg;
  e.ldo = H->V;
  CKS(gemm(H, H->lm_head, H->xb, M, e, PC_LMHEAD));
  ProfScope ps(H, PC_CTRL, 1);
  CK(launch_argmax_finalize(H->d_amax, H->d_ids, M, H->st));
  return DF_OK;
}

// LM head over rows [0, M) of xb.  Greedy: fused argmax into d_ids.
// Sampling: fp32 logits into the drafter's (draft) or the target's buffer,
// then each row's sampling distribution.
df_status lm_head(df_handle* H, int M, float* dbg, bool draft) {
  if (!H->sampling) return lm_head_argmax(H, M, dbg);
  float* logits = draft ? H->d_qlog : H->d_plog;
  EpiParams e = epi(H, EPI_STORE_F32);
  e.out = logits;
  e.ldo = H->V;
  CKS(gemm(H, H->lm_head, H->xb, M, e, PC_LMHEAD));
  ProfScope ps(H, PC_CTRL, 1);
  CK(launch_sample_state(logits, H->V, M, H->V, H->samp_inv_t, H->samp_top_p, draft ? H->d_qst : H->d_pst, H->d_err,
                         H->st));
  return DF_OK;
}

df_status attention(df_handle* H, int M, int R, int nseq, bool causal, const void* cache_layer, const void* kv_map,
                    int max_len) {
  AttnParams p{};
  p.kv_map = kv_map;
  p.q = H->q;
  p.out = H->attn;
  p.M = M;
  p.rows_per_seq = R;
  p.n_seqs = nseq;
  p.Hq = H->Hq;
  p.Hkv = H->Hkv;
  p.hd = H->hd;
  p.row_pos = H->d_row_pos;
  p.row_seq = H->d_row_seq;
  p.causal = causal ? 1 : 0;
  p.cache = cache_layer;
  p.page_table = H->d_pt;
  p.pt_stride = H->pages_per_seq;
  p.page_tokens = H->PT;
  p.n_pages = H->n_pages;
  p.blk = H->blk;
  p.rows_cap = H->Mmax;
  p.chunk = ATTN_CHUNK;
  p.n_chunk_slots = H->n_chunk_slots;
  p.grid_chunks = std::max(1, (max_len + ATTN_CHUNK - 1) / ATTN_CHUNK);
  if (p.grid_chunks > H->n_chunk_slots - 1) return fail(H, DF_EINVAL, "context longer than max_ctx");
  p.part_acc = H->part_acc;
  p.part_ml = H->part_ml;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)H->hd));
  p.err = H->d_err;
  // algorithmic bytes: the visible keys/values of every sequence, queries and outputs
  const double kv_bytes = (double)nseq * (double)(max_len + (causal ? 0 : R)) * 2.0 * H->kvdim * H->esz;
  const double qo_bytes = 2.0 * M * H->qdim * H->esz;
  ProfScope ps(H, PC_ATTN, attention_launches(p, H->bf16), kv_bytes + qo_bytes,
               4.0 * M * H->qdim * (double)max_len);
  p.trace = ps.tp;
  p.pipelined = H->attn_pipe ? 1 : 0;
  p.cla = H->attn_cla;
  CK(launch_attention(p, H->bf16, H->st));
  return DF_OK;
}

void* kv_layer(df_handle* H, void* base, int l) {
  return reinterpret_cast<uint8_t*>(base) + (size_t)l * H->layer_stride * H->esz;
}

// One decoder layer over M rows.  causal: target (K/V into the paged target
// cache); otherwise drafter (K/V into the block row buffer, attention over the
// injected context + block).
// Fill in the folded-RMSNorm fields: the GEMM reads unnormalised rows and
// scales each output row by 1/rms from the per-tile sums of squares.
void fold_norm(df_handle* H, EpiParams& e, const float* ss) {
  e.ss_in = ss;
  e.ss_tiles = H->d / 128;
  e.inv_d = 1.0f / (float)H->d;
  e.eps = H->cfg.rms_eps;
}

// One decoder layer over M rows.  Its RMSNorms are folded into the QKV and
// gate/up GEMMs (gains in the weights, 1/rms in the epilogues); the residual
// epilogues of the O and down GEMMs write the next GEMM's input rows and their
// sums of squares.  causal: target (K/V into the paged target cache);
// otherwise drafter (K/V into the block row buffer, attention over the
// injected context + block).  next_tap: feature slot of the next layer's
// input (the output of this layer), or -1.
df_status layer_pass(df_handle* H, const Layer& Lw, int M, int R, int nseq, bool causal, int cache_layer, int max_len,
                     int next_tap) {
  EpiParams e = epi(H, EPI_QKV);
  e.out = H->q;
  e.ldo = H->qdim;
  e.q_dim = H->qdim;
  e.row_pos = H->d_row_pos;
  e.row_seq = H->d_row_seq;
  fold_norm(H, e, H->ss);
  if (causal) {
    e.kv_dest = KV_PAGED;
    e.kv_base = H->kv_t;
    e.layer0 = cache_layer;
  } else {
    e.kv_dest = KV_ROWS;
    e.kv_base = H->blk;
  }
  CKS(gemm(H, Lw.qkv, H->xraw, M, e));
  const std::vector<Tmap>& maps = causal ? H->kvmap_t : H->kvmap_d;
  const void* kvm = (size_t)cache_layer < maps.size() ? maps[cache_layer].b : nullptr;
  CKS(attention(H, M, R, nseq, causal, kv_layer(H, causal ? H->kv_t : H->kv_d, cache_layer), kvm, max_len));
  EpiParams r = epi(H, EPI_RESID);
  r.resid = H->h;
  r.ldr = H->d;
  r.xraw = H->xraw;
  r.ldx = H->d;
  r.ss_out = H->ss;
  r.ss_tiles = H->d / 128;
  CKS(gemm(H, Lw.wo, H->attn, M, r));
  EpiParams s = epi(H, EPI_SWIGLU);
  s.out = H->act;
  s.ldo = H->F;
  fold_norm(H, s, H->ss);
  CKS(gemm(H, Lw.gu, H->xraw, M, s));
  if (next_tap >= 0) {
    r.tap = H->taps;
    r.tap_index = next_tap;
  }
  CKS(gemm(H, Lw.down, H->act, M, r));
  return DF_OK;
}

// Debug capture: the fp32 residual rows [0, M) as they stand before layer
// `slot` (slot = layer count: after the last layer) into buf[slot][M][d].
df_status debug_layer_rows(df_handle* H, float* buf, int slot, int M) {
  CK(cudaMemcpyAsync(buf + (size_t)slot * M * H->d, H->h, (size_t)M * H->d * 4, cudaMemcpyDeviceToDevice, H->st));
  return DF_OK;
}

// Target over M rows (row_tok / row_pos / row_seq already set).  head_rows:
// 0 = no LM head; -1 = every row; else only the last row (prefill).
df_status target_pass(df_handle* H, int M, int R, int nseq, int max_len, bool want_taps, int head_mode) {
  { ProfScope ps_(H, PC_EMBED, 1); CK(launch_embed(H->embed, H->bf16, H->d_row_tok, H->h, H->xraw, H->ss, M, H->d, H->V, H->d_err, H->st)); }
  if (H->debug) CKS(debug_layer_rows(H, H->dbg_tl, 0, M));
  for (int l = 0; l < H->L; ++l) {
    // the output of layer l is the input of layer l+1: tap it if selected
    const int tap = (want_taps && l + 1 < H->L) ? H->tap_of_layer[l + 1] : -1;
    CKS(layer_pass(H, H->tl[l], M, R, nseq, true, l, max_len, tap));
    if (H->debug) CKS(debug_layer_rows(H, H->dbg_tl, l + 1, M));
  }
  H->rows_last_target = M;
  if (H->debug) CK(cudaMemcpyAsync(H->dbg_th, H->h, (size_t)M * H->d * 4, cudaMemcpyDeviceToDevice, H->st));
  if (head_mode == 0) return DF_OK;
  const int first = head_mode < 0 ? 0 : M - 1;
  const int rows = head_mode < 0 ? M : 1;
  H->rows_last_logits = rows;
  H->rows_last_logits = rows;
  { ProfScope ps_(H, PC_NORM, 1); CK(launch_rmsnorm(H->h + (size_t)first * H->d, H->d, H->final_norm, H->xb, H->d, H->bf16, rows, H->d,
                    H->cfg.rms_eps, nullptr, 0, nullptr, H->st)); }
  return lm_head(H, rows, H->debug ? H->dbg_logits : nullptr, false);
}

// Fuse the taps of rows [0, M) and inject K/V of every drafter layer at the
// rows' positions (row_pos < 0: inactive row).
// Fuse the taps of rows [0, M) and inject K/V of every drafter layer at the
// rows' positions (row_pos < 0: inactive row).  The fusion GEMM writes the FC
// output in the model dtype with its per-tile sums of squares; the RMSNorm
// after the FC is folded into the injection GEMM (fc_norm gain in its
// weights, 1/rms in its epilogue).
df_status fuse_inject(df_handle* H, int M, const int* row_pos) {
  EpiParams e = epi(H, EPI_STORE_SS);
  e.out = H->ctx;
  e.ldo = H->d;
  e.ss_out = H->ss_ctx;
  e.ss_tiles = H->d / 128;
  CKS(gemm(H, H->fc, H->taps, M, e, PC_FUSE));
  EpiParams k = epi(H, EPI_QKV);
  k.q_dim = 0;
  k.kv_dest = KV_PAGED;
  k.kv_base = H->kv_d;
  k.layer0 = 0;
  k.row_pos = row_pos;
  k.row_seq = H->d_row_seq;
  fold_norm(H, k, H->ss_ctx);
  CKS(gemm(H, H->inj, H->ctx, M, k, PC_INJECT));
  H->rows_last_ctx = M;
  return DF_OK;
}

// Drafter over blocks of b slots (b = 0: the configured block size B).
df_status drafter_pass(df_handle* H, int nseq, int max_ctx_len, int b = 0) {
  const int B = b > 0 ? b : H->B, M = nseq * B;
  { ProfScope ps_(H, PC_EMBED, 1); CK(launch_embed(H->embed, H->bf16, H->d_row_tok, H->h, H->xraw, H->ss, M, H->d, H->V, H->d_err, H->st)); }
  if (H->debug) CKS(debug_layer_rows(H, H->dbg_dl, 0, M));
  for (int l = 0; l < H->Ld; ++l) {
    CKS(layer_pass(H, H->dl[l], M, B, nseq, false, l, max_ctx_len, -1));
    if (H->debug) CKS(debug_layer_rows(H, H->dbg_dl, l + 1, M));
  }
  if (H->debug) CK(cudaMemcpyAsync(H->dbg_dh, H->h, (size_t)M * H->d * 4, cudaMemcpyDeviceToDevice, H->st));
  { ProfScope ps_(H, PC_NORM, 1); CK(launch_rmsnorm(H->h, H->d, H->d_final_norm, H->xb, H->d, H->bf16, M, H->d, H->cfg.rms_eps, nullptr, 0, nullptr,
                    H->st)); }
  CKS(lm_head(H, M, H->debug ? H->dbg_dlogits : nullptr, true));
  H->rows_last_draft = M;
  return DF_OK;
}

// ---------------------------------------------------------------- pages
df_status ensure_pages(df_handle* H, int slot, int npos) {
  SeqHost& s = H->seqs[slot];
  const int need = (npos + H->PT - 1) / H->PT;
  if (need > H->pages_per_seq) return fail(H, DF_EINVAL, "sequence would exceed max_ctx");
  bool changed = false;
  while ((int)s.pages.size() < need) {
    if (H->free_pages.empty()) return fail(H, DF_ENOMEM, "KV page pool exhausted");
    s.pages.push_back(H->free_pages.back());
    H->free_pages.pop_back();
    changed = true;
  }
  if (changed) {
    std::vector<int> row(H->pages_per_seq, -1);
    std::copy(s.pages.begin(), s.pages.end(), row.begin());
    CK(h2d(H, H->d_pt + (size_t)slot * H->pages_per_seq, row.data(), row.size() * 4));
  }
  return DF_OK;
}

// Return pages wholly past `keep` positions (rollback after acceptance).
df_status trim_pages(df_handle* H, int slot, int keep) {
  SeqHost& s = H->seqs[slot];
  const int need = (keep + H->PT - 1) / H->PT;
  bool changed = false;
  while ((int)s.pages.size() > need) {
    H->free_pages.push_back(s.pages.back());
    s.pages.pop_back();
    changed = true;
  }
  if (changed) {
    std::vector<int> row(H->pages_per_seq, -1);
    std::copy(s.pages.begin(), s.pages.end(), row.begin());
    CK(h2d(H, H->d_pt + (size_t)slot * H->pages_per_seq, row.data(), row.size() * 4));
  }
  return DF_OK;
}

df_status check_device_error(df_handle* H) {
  int e = 0;
  CK(d2h(H, &e, H->d_err, 4));
  CK(cudaStreamSynchronize(H->st));
  if (e) {
    H->failed = true;
    if (e & ERR_TIMEOUT) return fail(H, DF_ETIMEOUT, "a bounded device wait ran out (error word " + std::to_string(e) + ")");
    return fail(H, DF_ECUDA, "device error word " + std::to_string(e));
  }
  return DF_OK;
}

df_status sync(df_handle* H) {
  CK(cudaStreamSynchronize(H->st));
  if (H->profiling) prof_resolve(H);
  return check_device_error(H);
}

df_status check_slots(df_handle* H, const int32_t* slots, int nseq) {
  if (nseq < 1 || nseq > H->cfg.max_batch || !slots) return fail(H, DF_EINVAL, "bad sequence list");
  for (int i = 0; i < nseq; ++i) {
    if (slots[i] < 0 || slots[i] >= H->cfg.max_batch) return fail(H, DF_EINVAL, "sequence slot out of range");
    if (!H->seqs[slots[i]].active) return fail(H, DF_ESTATE, "sequence slot not prefilled");
    for (int j = 0; j < i; ++j)
      if (slots[j] == slots[i]) return fail(H, DF_EINVAL, "sequence listed twice");
  }
  return DF_OK;
}

df_status prefill_impl(df_handle* H, int seq, const int32_t* prompt, int len, bool inject, int* bonus_out) {
  if (seq < 0 || seq >= H->cfg.max_batch) return fail(H, DF_EINVAL, "sequence slot out of range");
  if (!prompt || len < 1) return fail(H, DF_EINVAL, "empty prompt");
  if (len + H->B > H->cfg.max_ctx) return fail(H, DF_EINVAL, "prompt too long for max_ctx");
  if (H->seqs[seq].active) return fail(H, DF_ESTATE, "sequence slot already in use");
  for (int i = 0; i < len; ++i)
    if (prompt[i] < 0 || prompt[i] >= H->V) return fail(H, DF_EINVAL, "prompt token out of range");
  SeqHost& s = H->seqs[seq];
  s.active = true;
  s.len = 0;
  s.pages.clear();
  CKS(ensure_pages(H, seq, len));
  const int chunk = std::min(PREFILL_CHUNK, H->Mmax);
  std::vector<int> tok(chunk), pos(chunk), sq(chunk, seq);
  for (int c0 = 0; c0 < len; c0 += chunk) {
    const int rows = std::min(chunk, len - c0);
    for (int i = 0; i < rows; ++i) {
      tok[i] = prompt[c0 + i];
      pos[i] = c0 + i;
    }
    CK(h2d(H, H->d_row_tok, tok.data(), rows * 4));
    CK(h2d(H, H->d_row_pos, pos.data(), rows * 4));
    CK(h2d(H, H->d_row_seq, sq.data(), rows * 4));
    const bool last = c0 + rows == len;
    CKS(target_pass(H, rows, rows, 1, c0 + rows, inject, last ? 1 : 0));
    if (inject) CKS(fuse_inject(H, rows, H->d_row_pos));
  }
  // bonus token = argmax at the last prompt position (sampling: a draw from
  // the target's distribution there, the sequence's first uniform); it sits
  // at position len
  if (H->sampling) {
    CK(h2d(H, H->d_slots, &seq, 4));
    ProfScope ps_(H, PC_CTRL, 2);
    CK(launch_cycle_uniforms(H->d_slots, 1, 1, H->samp_seed, H->d_ustream, H->d_ucount, H->d_u, 2 * H->B, H->st));
    CK(launch_sample_draw(H->d_plog, H->V, 1, H->V, H->d_pst, H->d_u, 1, 2 * H->B, 0, H->d_ids, H->d_err, H->st));
  }
  CK(cudaMemcpyAsync(H->d_bonus + seq, H->d_ids, 4, cudaMemcpyDeviceToDevice, H->st));
  CK(h2d(H, H->d_bonus_pos + seq, &len, 4));
  CK(d2h(H, H->h_pin, H->d_ids, 4));
  CKS(sync(H));
  s.len = len;
  s.bonus = H->h_pin[0];
  if (bonus_out) *bonus_out = s.bonus;
  return DF_OK;
}

df_status draft_impl(df_handle* H, const int32_t* slots, int nseq, int32_t* drafts_host) {
  CKS(check_slots(H, slots, nseq));
  const int B = H->B;
  CK(h2d(H, H->d_slots, slots, nseq * 4));
  int max_len = 0;
  for (int i = 0; i < nseq; ++i) max_len = std::max(max_len, H->seqs[slots[i]].len);
  CK(cudaEventRecord(H->ev[0], H->st));
  { ProfScope ps_(H, PC_CTRL, 1); CK(launch_prep_block(H->d_slots, nseq, B, H->d_bonus, H->d_bonus_pos, H->d_drafts, H->cfg.mask_token_id, 0,
                       H->d_row_tok, H->d_row_pos, H->d_row_seq, H->st)); }
  CKS(drafter_pass(H, nseq, max_len));
  { ProfScope ps_(H, PC_CTRL, 1); CK(launch_collect_drafts(H->d_ids, nseq, B, H->d_slots, H->d_drafts, H->st)); }
  CK(cudaEventRecord(H->ev[1], H->st));
  if (drafts_host) {
    CK(d2h(H, H->h_pin, H->d_drafts, (size_t)H->cfg.max_batch * (B - 1) * 4));
    CKS(sync(H));
    for (int i = 0; i < nseq; ++i)
      std::memcpy(drafts_host + (size_t)i * (B - 1), H->h_pin + (size_t)slots[i] * (B - 1), (B - 1) * 4);
  }
  return DF_OK;
}

df_status verify_impl(df_handle* H, const int32_t* slots, int nseq, const int32_t* drafts_host, int32_t* acc_host,
                      int32_t* n_host, bool timed) {
  CKS(check_slots(H, slots, nseq));
  const int B = H->B;
  int max_len = 0;
  for (int i = 0; i < nseq; ++i) {
    SeqHost& s = H->seqs[slots[i]];
    if (s.len + B > H->cfg.max_ctx) return fail(H, DF_EINVAL, "sequence would exceed max_ctx");
    CKS(ensure_pages(H, slots[i], s.len + B));
    max_len = std::max(max_len, s.len + B);
  }
  CK(h2d(H, H->d_slots, slots, nseq * 4));
  if (drafts_host) {
    for (int i = 0; i < nseq; ++i) {
      for (int j = 0; j < B - 1; ++j) {
        const int t = drafts_host[(size_t)i * (B - 1) + j];
        if (t < 0 || t >= H->V) return fail(H, DF_EINVAL, "draft token out of range");
      }
      CK(h2d(H, H->d_drafts + (size_t)slots[i] * (B - 1), drafts_host + (size_t)i * (B - 1), (B - 1) * 4));
    }
  }
  CK(cudaEventRecord(H->ev[2], H->st));
  { ProfScope ps_(H, PC_CTRL, 1); CK(launch_prep_block(H->d_slots, nseq, B, H->d_bonus, H->d_bonus_pos, H->d_drafts, H->cfg.mask_token_id, 1,
                       H->d_row_tok, H->d_row_pos, H->d_row_seq, H->st)); }
  const int M = nseq * B;
  CKS(target_pass(H, M, B, nseq, max_len, true, -1));
  { ProfScope ps_(H, PC_CTRL, 1); CK(launch_accept(H->d_slots, nseq, B, H->d_row_tok, H->d_ids, H->d_bonus, H->d_bonus_pos, H->d_acc, H->d_n,
                   H->d_inj_pos, H->st)); }
  CKS(fuse_inject(H, M, H->d_inj_pos));
  CK(cudaEventRecord(H->ev[3], H->st));
  CK(d2h(H, H->h_pin, H->d_acc, (size_t)nseq * B * 4));
  CK(d2h(H, H->h_pin + (size_t)nseq * B, H->d_n, (size_t)nseq * 4));
  CKS(sync(H));
  const int* acc = H->h_pin;
  const int* n = H->h_pin + (size_t)nseq * B;
  for (int i = 0; i < nseq; ++i) {
    SeqHost& s = H->seqs[slots[i]];
    const int k = n[i] - 1;
    if (k < 0 || k > B - 1) return fail(H, DF_ECUDA, "accept kernel produced an invalid count");
    s.len += k + 1;
    s.bonus = acc[(size_t)i * B + k];
    CKS(trim_pages(H, slots[i], s.len + B));
    H->stats.cycles += 1;
    H->stats.accepted_drafts += k;
    H->stats.accept_hist[std::min(k, 64)] += 1;
    H->stats.block_hist[B] += 1;
  }
  if (timed) {
    float a = 0.f, b = 0.f;
    if (cudaEventElapsedTime(&a, H->ev[0], H->ev[1]) == cudaSuccess) H->stats.draft_us += 1000.0 * a;
    if (cudaEventElapsedTime(&b, H->ev[2], H->ev[3]) == cudaSuccess) H->stats.verify_us += 1000.0 * b;
  }
  if (acc_host) std::memcpy(acc_host, acc, (size_t)nseq * B * 4);
  if (n_host) std::memcpy(n_host, n, (size_t)nseq * 4);
  return DF_OK;
}

// The device work of one draft + verify cycle for the sequences in d_slots_dev
// (stream-ordered, nothing read back): draft pass, verification, acceptance,
// fusion and injection, then the accepted tokens and counts copied to h_pin.
// ext_events: record the timing events as graph-visible event nodes.
// Cycle c of a run of cycles: its events are cev[4c..4c+3] and its accepted
// tokens ([nseq][b]) and counts ([nseq], at nseq * B) go to h_pin at
// cycle_pin(c).  b is the cycle's block size (<= B).
size_t cycle_pin(const df_handle* H, int nseq, int c) { return (size_t)c * nseq * (H->B + 1); }

df_status cycle_work(df_handle* H, const int* d_slots_dev, int nseq, int max_len_d, int max_len_t, bool ext_events,
                     int c, int b) {
  const int B = b;
  cudaEvent_t* ev = H->cev + 4 * c;
  auto rec = [&](cudaEvent_t e) {
    return ext_events ? cudaEventRecordWithFlags(e, H->st, cudaEventRecordExternal) : cudaEventRecord(e, H->st);
  };
  CK(rec(ev[0]));
  { ProfScope ps_(H, PC_CTRL, 1); CK(launch_prep_block(d_slots_dev, nseq, B, H->d_bonus, H->d_bonus_pos, H->d_drafts, H->cfg.mask_token_id, 0, H->d_row_tok, H->d_row_pos, H->d_row_seq, H->st)); }
  if (H->sampling) {
    // the cycle's 2B - 1 uniforms per sequence: B - 1 draft draws, B - 1 tests, the final draw
    ProfScope ps_(H, PC_CTRL, 1);
    CK(launch_cycle_uniforms(d_slots_dev, nseq, 2 * B - 1, H->samp_seed, H->d_ustream, H->d_ucount, H->d_u, 2 * B, H->st));
  }
  CKS(drafter_pass(H, nseq, max_len_d, B));
  if (H->sampling) {
    // draft i (slot i = 1..B-1) drawn from the drafter's distribution at slot i
    ProfScope ps_(H, PC_CTRL, 1);
    CK(launch_sample_draw(H->d_qlog, H->V, nseq * B, H->V, H->d_qst, H->d_u, B, 2 * B, 1, H->d_ids, H->d_err, H->st));
  }
  { ProfScope ps_(H, PC_CTRL, 1); CK(launch_collect_drafts(H->d_ids, nseq, B, d_slots_dev, H->d_drafts, H->st)); }
  CK(rec(ev[1]));
  CK(rec(ev[2]));
  { ProfScope ps_(H, PC_CTRL, 1); CK(launch_prep_block(d_slots_dev, nseq, B, H->d_bonus, H->d_bonus_pos, H->d_drafts, H->cfg.mask_token_id, 1, H->d_row_tok, H->d_row_pos, H->d_row_seq, H->st)); }
  const int M = nseq * B;
  CKS(target_pass(H, M, B, nseq, max_len_t, true, -1));
  if (H->sampling) {
    ProfScope ps_(H, PC_CTRL, 1);
    CK(launch_accept_sampled(d_slots_dev, nseq, B, H->d_row_tok + 1, B, H->d_qlog, H->V, H->d_qst, B, 1, H->d_plog, H->V,
                             H->d_pst, H->V, H->d_u, 2 * B, B - 1, H->d_bonus, H->d_bonus_pos, H->d_acc, H->d_n,
                             H->d_inj_pos, nullptr, nullptr, H->d_err, H->st));
  } else {
    ProfScope ps_(H, PC_CTRL, 1);
    CK(launch_accept(d_slots_dev, nseq, B, H->d_row_tok, H->d_ids, H->d_bonus, H->d_bonus_pos, H->d_acc, H->d_n, H->d_inj_pos, H->st));
  }
  CKS(fuse_inject(H, M, H->d_inj_pos));
  CK(rec(ev[3]));
  int* pin = H->h_pin + cycle_pin(H, nseq, c);
  CK(d2h(H, pin, H->d_acc, (size_t)nseq * B * 4));
  CK(d2h(H, pin + (size_t)nseq * H->B, H->d_n, (size_t)nseq * 4));
  return DF_OK;
}

// Host bookkeeping after cycle c (block size b) reached h_pin: lengths,
// bonus tokens, stats; acc_host ([nseq][B], first b of each row written) and
// n_host (optional) receive this cycle's rows.
df_status cycle_finish(df_handle* H, const int32_t* slots, int nseq, int c, int b, int32_t* acc_host,
                       int32_t* n_host) {
  const int B = b;
  const int* acc = H->h_pin + cycle_pin(H, nseq, c);
  const int* n = acc + (size_t)nseq * H->B;
  for (int i = 0; i < nseq; ++i) {
    SeqHost& s = H->seqs[slots[i]];
    const int k = n[i] - 1;
    if (k < 0 || k > B - 1) return fail(H, DF_ECUDA, "accept kernel produced an invalid count");
    s.len += k + 1;
    s.bonus = acc[(size_t)i * B + k];
    H->stats.cycles += 1;
    H->stats.accepted_drafts += k;
    H->stats.accept_hist[std::min(k, 64)] += 1;
    H->stats.block_hist[B] += 1;
  }
  const cudaEvent_t* ev = H->cev + 4 * c;
  float ta = 0.f, tb = 0.f;
  if (cudaEventElapsedTime(&ta, ev[0], ev[1]) == cudaSuccess) H->stats.draft_us += 1000.0 * ta;
  if (cudaEventElapsedTime(&tb, ev[2], ev[3]) == cudaSuccess) H->stats.verify_us += 1000.0 * tb;
  if (acc_host)
    for (int i = 0; i < nseq; ++i) std::memcpy(acc_host + (size_t)i * H->B, acc + (size_t)i * B, (size_t)B * 4);
  if (n_host) std::memcpy(n_host, n, (size_t)nseq * 4);
  return DF_OK;
}

// Pages past each sequence's kept length (+ one block) go back to the pool.
df_status trim_all(df_handle* H, const int32_t* slots, int nseq) {
  for (int i = 0; i < nseq; ++i) CKS(trim_pages(H, slots[i], H->seqs[slots[i]].len + H->B));
  return DF_OK;
}

// Block size for the next group of cycles: the smallest power of two that is
// at least twice the recent tokens per cycle, within [b_min, b_max] (b_max
// itself where the power of two would pass it).  A block twice the accepted
// length leaves room to grow: a group that keeps every draft doubles it.
int block_size_for(double tokens_per_cycle, int b_min, int b_max) {
  int b = 2;
  while (b < b_max && (double)b < 2.0 * tokens_per_cycle) b *= 2;
  return std::max(b_min, std::min(b, b_max));
}

void drop_graph(df_handle* H) {
  for (auto& g : H->graphs)
    if (g.second.exec) cudaGraphExecDestroy(g.second.exec);
  H->graphs.clear();
  H->glast.clear();
}

// K draft + verify cycles for df_generate (acc_host [K][nseq][B], n_host
// [K][nseq]).  Pages for K blocks of growth are reserved first.  After the
// first (eager) cycle of a handle, the K cycles' launches are captured once
// into a CUDA graph and replayed: the cycles chain on the device (positions,
// bonus tokens and rollback live in device memory) and the host reads all K
// results after one synchronisation.  The graph's attention launches are
// sized for max_ctx, so a new capture is made only for new slots, K or block
// size b; a few captured graphs are kept.
df_status cycle_impl(df_handle* H, const int32_t* slots, int nseq, int K, int b, int32_t* acc_host, int32_t* n_host) {
  CKS(check_slots(H, slots, nseq));
  const int B = H->B;
  if (K < 1 || K > KMAX_CYCLES) return fail(H, DF_EINVAL, "bad cycle count");
  if (b < 2 || b > B) return fail(H, DF_EINVAL, "bad block size");
  for (int i = 0; i < nseq; ++i) {
    SeqHost& s = H->seqs[slots[i]];
    if (s.len + K * B > H->cfg.max_ctx) return fail(H, DF_EINVAL, "sequence would exceed max_ctx");
    CKS(ensure_pages(H, slots[i], s.len + K * B));
  }
  auto out_acc = [&](int c) { return acc_host ? acc_host + (size_t)c * nseq * B : nullptr; };
  auto out_n = [&](int c) { return n_host ? n_host + (size_t)c * nseq : nullptr; };
  const bool graphs = H->use_graphs && !H->profiling && H->graph_ready_cycles > 0;
  if (!graphs) {
    for (int c = 0; c < K; ++c) {
      int max_t = 0, max_d = 0;
      for (int i = 0; i < nseq; ++i) {
        const SeqHost& s = H->seqs[slots[i]];
        max_t = std::max(max_t, s.len + b);
        max_d = std::max(max_d, s.len);
      }
      CK(h2d(H, H->d_slots, slots, nseq * 4));
      H->trace_meta.clear();
      if (H->tracing) CK(cudaMemsetAsync(H->d_trace, 0, TRACE_MAX * 16, H->st));
      CKS(cycle_work(H, H->d_slots, nseq, max_d, max_t, false, 0, b));
      CKS(sync(H));
      if (H->tracing) CK(trace_collect(H, H->trace_meta));
      H->graph_ready_cycles += 1;
      CKS(cycle_finish(H, slots, nseq, 0, b, out_acc(c), out_n(c)));
    }
    return trim_all(H, slots, nseq);
  }
  std::vector<int> key(slots, slots + nseq);
  key.push_back(K);
  key.push_back(b);
  key.push_back(H->tracing ? 1 : 0);  // stamp slots are launch arguments of the captured kernels
  if (H->sampling) {
    // the sampling parameters are launch arguments of the captured kernels
    int tb = 0, pb = 0;
    std::memcpy(&tb, &H->samp_inv_t, 4);
    std::memcpy(&pb, &H->samp_top_p, 4);
    key.insert(key.end(), {-1, tb, pb, (int)(uint32_t)H->samp_seed, (int)(uint32_t)(H->samp_seed >> 32)});
  }
  const int max_len = H->cfg.max_ctx;  // length-independent launches
  // the caller's stream may be the legacy default stream, which cannot be
  // captured: graphs run on the engine's own stream, ordered after the
  // caller's stream and joined back to it with events
  const cudaStream_t user = H->st;
  CK(cudaEventRecord(H->gjoin[0], user));
  CK(cudaStreamWaitEvent(H->gstream, H->gjoin[0], 0));
  auto it = H->graphs.find(key);
  if (it == H->graphs.end()) {
    if (H->graphs.size() >= MAX_GRAPHS) drop_graph(H);
    CK(h2d(H, H->d_gslots, slots, nseq * 4));
    H->glast = key;
    CK(cudaStreamSynchronize(user));
    const df_stats before = H->stats;
    H->trace_meta.clear();
    bool ok = cudaStreamBeginCapture(H->gstream, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
    df_status st = DF_OK;
    cudaGraph_t g = nullptr;
    if (ok) {
      H->st = H->gstream;
      for (int c = 0; c < K && st == DF_OK; ++c) st = cycle_work(H, H->d_gslots, nseq, max_len, max_len, true, c, b);
      H->st = user;
      ok = cudaStreamEndCapture(H->gstream, &g) == cudaSuccess && st == DF_OK;
    }
    H->st = user;
    df_handle::GraphRec rec;
    if (ok) ok = cudaGraphInstantiate(&rec.exec, g, 0) == cudaSuccess;
    if (g) cudaGraphDestroy(g);
    rec.launches = H->stats.kernel_launches - before.kernel_launches;
    rec.h2d = H->stats.h2d_bytes - before.h2d_bytes;
    rec.d2h = H->stats.d2h_bytes - before.d2h_bytes;
    rec.trace_meta = H->trace_meta;
    H->stats = before;  // counted again at each replay
    if (!ok) {
      // capture is not available here: run this handle's cycles eagerly
      (void)cudaGetLastError();
      drop_graph(H);
      H->use_graphs = false;
      return cycle_impl(H, slots, nseq, K, b, acc_host, n_host);
    }
    it = H->graphs.emplace(key, rec).first;
  } else if (H->glast != key) {
    // the graphs read their slots from d_gslots: put this graph's there
    CK(h2d(H, H->d_gslots, slots, nseq * 4));
    CK(cudaEventRecord(H->gjoin[0], user));
    CK(cudaStreamWaitEvent(H->gstream, H->gjoin[0], 0));
    H->glast = key;
  }
  if (!it->second.trace_meta.empty()) CK(cudaMemsetAsync(H->d_trace, 0, it->second.trace_meta.size() * 16, H->gstream));
  CK(cudaGraphLaunch(it->second.exec, H->gstream));
  CK(cudaEventRecord(H->gjoin[1], H->gstream));
  CK(cudaStreamWaitEvent(H->st, H->gjoin[1], 0));
  H->stats.kernel_launches += it->second.launches;
  H->stats.h2d_bytes += it->second.h2d;
  H->stats.d2h_bytes += it->second.d2h;
  CKS(sync(H));
  if (!it->second.trace_meta.empty()) CK(trace_collect(H, it->second.trace_meta));
  for (int c = 0; c < K; ++c) CKS(cycle_finish(H, slots, nseq, c, b, out_acc(c), out_n(c)));
  return trim_all(H, slots, nseq);
}

df_status release(df_handle* H, int slot) {
  SeqHost& s = H->seqs[slot];
  for (int p : s.pages) H->free_pages.push_back(p);
  s.pages.clear();
  s.active = false;
  s.len = 0;
  s.bonus = -1;
  std::vector<int> row(H->pages_per_seq, -1);
  CK(h2d(H, H->d_pt + (size_t)slot * H->pages_per_seq, row.data(), row.size() * 4));
  CK(cudaStreamSynchronize(H->st));
  return DF_OK;
}

df_status check_batch_args(df_handle* H, const int32_t* prompts, const int32_t* lens, int nseq, int n_new, void* out) {
  if (!prompts || !lens || !out || nseq < 1 || nseq > H->cfg.max_batch || n_new < 1)
    return fail(H, DF_EINVAL, "bad batch arguments");
  for (int i = 0; i < nseq; ++i) {
    if (H->seqs[i].active) return fail(H, DF_ESTATE, "slots 0..nseq-1 must be free");
    if (lens[i] < 1 || (long long)lens[i] + n_new + H->B > H->cfg.max_ctx)
      return fail(H, DF_EINVAL, "prompt length + n_new + block exceeds max_ctx");
  }
  return DF_OK;
}

// ---------------------------------------------------------------- init helpers
df_status pack_weights(df_handle* H, const void* const* w, int nw) {
  const df_config& c = H->cfg;
  const size_t es = H->esz;
  const int d = H->d;
  std::vector<WSpec> specs = weight_specs(c);
  if ((int)specs.size() != nw) return fail(H, DF_EINVAL, "wrong number of weights");
  for (int i = 0; i < nw; ++i)
    if (!w[i]) return fail(H, DF_EINVAL, "null weight pointer: " + specs[i].name);

  // Arena layout: every matrix 256-byte aligned; norm gains stored as fp32.
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~size_t(255);
    return o;
  };
  struct Slot {
    size_t off;
  };
  const long long V = H->V, F = H->F, qd = H->qdim, kd = H->kvdim;
  size_t o_embed = take(V * d * es), o_lm = take(V * d * es), o_fc = take((size_t)d * 5 * d * es);
  size_t o_inj = take((size_t)H->Ld * 2 * kd * d * es);
  size_t o_fn = take(d * 4), o_fcn = take(d * 4), o_dfn = take(d * 4);
  struct LOff {
    size_t an, qkv, wo, mn, gu, down;
  };
  std::vector<LOff> lo(H->L + H->Ld);
  for (auto& x : lo) {
    x.an = take(d * 4);
    x.qkv = take((size_t)H->qkv_n * d * es);
    x.wo = take((size_t)d * qd * es);
    x.mn = take(d * 4);
    x.gu = take((size_t)2 * F * d * es);
    x.down = take((size_t)d * F * es);
  }
  CKS(dalloc(H, &H->arena, off));
  uint8_t* A = reinterpret_cast<uint8_t*>(H->arena);
  cudaStream_t st = H->st;
  auto cp = [&](size_t dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(A + dst, src, bytes, cudaMemcpyDeviceToDevice, st);
  };
  // gains: device -> host -> fp32 -> device
  auto gain = [&](size_t dst, const void* src) -> df_status {
    std::vector<float> g(d);
    if (H->bf16) {
      std::vector<uint16_t> b(d);
      CK(cudaMemcpy(b.data(), src, d * 2, cudaMemcpyDeviceToHost));
      for (int i = 0; i < d; ++i) {
        uint32_t u = (uint32_t)b[i] << 16;
        std::memcpy(&g[i], &u, 4);
      }
    } else {
      CK(cudaMemcpy(g.data(), src, d * 4, cudaMemcpyDeviceToHost));
    }
    CK(cudaMemcpy(A + dst, g.data(), d * 4, cudaMemcpyHostToDevice));
    return DF_OK;
  };

  int i = 0;
  CK(cp(o_embed, w[i++], V * d * es));
  H->embed = A + o_embed;
  auto layer = [&](int li, Layer& Lw) -> df_status {
    const LOff& x = lo[li];
    CKS(gain(x.an, w[i++]));
    CK(cp(x.qkv, w[i++], qd * d * es));
    CK(cp(x.qkv + qd * d * es, w[i++], kd * d * es));
    CK(cp(x.qkv + (qd + kd) * d * es, w[i++], kd * d * es));
    CK(cp(x.wo, w[i++], (size_t)d * qd * es));
    CKS(gain(x.mn, w[i++]));
    const void* gate = w[i++];
    const void* up = w[i++];
    const size_t blk = (size_t)64 * d * es;
    CK(cudaMemcpy2DAsync(A + x.gu, 2 * blk, gate, blk, blk, F / 64, cudaMemcpyDeviceToDevice, st));
    CK(cudaMemcpy2DAsync(A + x.gu + blk, 2 * blk, up, blk, blk, F / 64, cudaMemcpyDeviceToDevice, st));
    CK(cp(x.down, w[i++], (size_t)d * F * es));
    Lw.attn_norm = reinterpret_cast<float*>(A + x.an);
    Lw.mlp_norm = reinterpret_cast<float*>(A + x.mn);
    Lw.qkv = Linear{A + x.qkv, H->qkv_n, d, {}};
    Lw.wo = Linear{A + x.wo, d, (int)qd, {}};
    Lw.gu = Linear{A + x.gu, (int)(2 * F), d, {}};
    Lw.down = Linear{A + x.down, d, (int)F, {}};
    return DF_OK;
  };
  H->tl.resize(H->L);
  H->dl.resize(H->Ld);
  for (int l = 0; l < H->L; ++l) CKS(layer(l, H->tl[l]));
  CKS(gain(o_fn, w[i++]));
  H->final_norm = reinterpret_cast<float*>(A + o_fn);
  CK(cp(o_lm, w[i++], V * d * es));
  H->lm_head = Linear{A + o_lm, (int)V, d, {}};
  CK(cp(o_fc, w[i++], (size_t)d * 5 * d * es));
  H->fc = Linear{A + o_fc, d, 5 * d, {}};
  CKS(gain(o_fcn, w[i++]));
  H->fc_norm = reinterpret_cast<float*>(A + o_fcn);
  // the drafter layers; their W_k/W_v also feed the injection matrix
  for (int l = 0; l < H->Ld; ++l) {
    const int base = i;
    CKS(layer(H->L + l, H->dl[l]));
    const size_t kv_bytes = (size_t)kd * d * es;
    CK(cp(o_inj + (size_t)l * 2 * kv_bytes, w[base + 2], kv_bytes));
    CK(cp(o_inj + (size_t)l * 2 * kv_bytes + kv_bytes, w[base + 3], kv_bytes));
  }
  H->inj = Linear{A + o_inj, (int)(H->Ld * 2 * kd), d, {}};
  CKS(gain(o_dfn, w[i++]));
  H->d_final_norm = reinterpret_cast<float*>(A + o_dfn);
  // Fold each RMSNorm's gain into the columns of the weight that consumes the
  // normalised rows (the norms themselves run in those GEMMs' epilogues).
  for (auto* layers : {&H->tl, &H->dl})
    for (Layer& Lw : *layers) {
      CK(launch_scale_cols(Lw.qkv.ptr, H->bf16, Lw.qkv.N, d, Lw.attn_norm, st));
      CK(launch_scale_cols(Lw.gu.ptr, H->bf16, Lw.gu.N, d, Lw.mlp_norm, st));
    }
  CK(launch_scale_cols(H->inj.ptr, H->bf16, H->inj.N, d, H->fc_norm, st));
  CK(cudaStreamSynchronize(st));

  if (H->bf16) {
    std::vector<Linear*> all = {&H->lm_head, &H->fc, &H->inj};
    for (auto& Lw : H->tl) all.insert(all.end(), {&Lw.qkv, &Lw.wo, &Lw.gu, &Lw.down});
    for (auto& Lw : H->dl) all.insert(all.end(), {&Lw.qkv, &Lw.wo, &Lw.gu, &Lw.down});
    for (Linear* Lp : all)
      if (!make_tmap_bf16(Lp->tm.b, Lp->ptr, Lp->N, Lp->K, 128))
        return fail(H, DF_ECUDA, "tensor map encode failed (weights)");
  }
  return DF_OK;
}

df_status alloc_state(df_handle* H) {
  const df_config& c = H->cfg;
  const size_t es = H->esz;
  const int d = H->d, M = H->Mmax;
  H->PT = c.page_tokens;
  H->pages_per_seq = (c.max_ctx + H->PT - 1) / H->PT;
  H->n_pages = H->pages_per_seq * c.max_batch;
  const size_t page_elems = (size_t)2 * H->Hkv * H->PT * H->hd;
  H->layer_stride = (long long)(page_elems * H->n_pages);
  CKS(dalloc(H, &H->kv_t, (size_t)H->layer_stride * H->L * es));
  CKS(dalloc(H, &H->kv_d, (size_t)H->layer_stride * H->Ld * es));
  if (H->bf16 && H->hd == 128) {
    H->kvmap_t.resize(H->L);
    H->kvmap_d.resize(H->Ld);
    for (int l = 0; l < H->L; ++l)
      if (!make_tmap_kvcache(H->kvmap_t[l].b, kv_layer(H, H->kv_t, l), H->n_pages, H->Hkv, H->PT))
        return fail(H, DF_ECUDA, "tensor map encode failed (target cache)");
    for (int l = 0; l < H->Ld; ++l)
      if (!make_tmap_kvcache(H->kvmap_d[l].b, kv_layer(H, H->kv_d, l), H->n_pages, H->Hkv, H->PT))
        return fail(H, DF_ECUDA, "tensor map encode failed (drafter cache)");
  }
  CKS(dalloc_t(H, &H->d_pt, (size_t)c.max_batch * H->pages_per_seq * 4));
  CK(cudaMemset(H->d_pt, 0xFF, (size_t)c.max_batch * H->pages_per_seq * 4));
  for (int p = H->n_pages - 1; p >= 0; --p) H->free_pages.push_back(p);
  H->seqs.assign(c.max_batch, SeqHost{});

  CKS(dalloc_t(H, &H->d_bonus, c.max_batch * 4));
  CKS(dalloc_t(H, &H->d_bonus_pos, c.max_batch * 4));
  CKS(dalloc_t(H, &H->d_row_tok, M * 4));
  CKS(dalloc_t(H, &H->d_row_pos, M * 4));
  CKS(dalloc_t(H, &H->d_row_seq, M * 4));
  CKS(dalloc_t(H, &H->d_inj_pos, M * 4));
  CKS(dalloc_t(H, &H->d_ids, M * 4));
  CKS(dalloc_t(H, &H->d_slots, c.max_batch * 4));
  CKS(dalloc_t(H, &H->d_gslots, c.max_batch * 4));
  CKS(dalloc_t(H, &H->d_drafts, (size_t)c.max_batch * H->B * 4));
  CKS(dalloc_t(H, &H->d_acc, (size_t)c.max_batch * H->B * 4));
  CKS(dalloc_t(H, &H->d_n, c.max_batch * 4));
  CKS(dalloc_t(H, &H->d_amax, M * 8));
  CKS(dalloc_t(H, &H->d_err, 4));
  CK(cudaMemset(H->d_err, 0, 4));
  CK(cudaMemset(H->d_drafts, 0, (size_t)c.max_batch * H->B * 4));

  CKS(dalloc_t(H, &H->h, (size_t)M * d * 4));
  CKS(dalloc(H, &H->xb, (size_t)M * d * es));
  CKS(dalloc(H, &H->q, (size_t)M * H->qdim * es));
  CKS(dalloc(H, &H->attn, (size_t)M * H->qdim * es));
  CKS(dalloc(H, &H->act, (size_t)M * H->F * es));
  CKS(dalloc(H, &H->taps, (size_t)M * 5 * d * es));
  CKS(dalloc(H, &H->ctx, (size_t)M * d * es));
  CKS(dalloc(H, &H->blk, (size_t)2 * H->Hkv * M * H->hd * es));
  CKS(dalloc(H, &H->xraw, (size_t)M * d * es));
  CKS(dalloc_t(H, &H->ss, (size_t)M * (d / 128) * 4));
  CKS(dalloc_t(H, &H->ss_ctx, (size_t)M * (d / 128) * 4));
  CK(cudaMemset(H->xraw, 0, (size_t)M * d * es));
  CK(cudaMemset(H->ss, 0, (size_t)M * (d / 128) * 4));
  CK(cudaMemset(H->ss_ctx, 0, (size_t)M * (d / 128) * 4));
  // zero the activation buffers once so rows a pass does not write are finite
  CK(cudaMemset(H->xb, 0, (size_t)M * d * es));
  CK(cudaMemset(H->attn, 0, (size_t)M * H->qdim * es));
  CK(cudaMemset(H->act, 0, (size_t)M * H->F * es));
  CK(cudaMemset(H->taps, 0, (size_t)M * 5 * d * es));
  CK(cudaMemset(H->ctx, 0, (size_t)M * d * es));

  // GEMM shapes: split-K workspace and tile tickets
  std::vector<std::pair<int, int>> shapes = {{H->qkv_n, d}, {d, H->qdim}, {2 * H->F, d}, {d, H->F},
                                             {H->V, d},     {d, 5 * d},   {H->inj.N, d}};
  size_t ws = 0, cnt = 0;
  if (H->bf16) {
    for (auto& s : shapes) {
      const int splits = tc_splits(s.first, s.second, H->split_target);
      for (int nt : {16, 32, 64, 128, 256}) {
        ws = std::max(ws, tc_workspace_floats(M, s.first, splits, nt));
        cnt = std::max(cnt, tc_counter_ints(M, s.first, nt));
      }
    }
  } else {
    size_t maxN = 0;
    for (auto& s : shapes) maxN = std::max(maxN, (size_t)s.first);
    CKS(dalloc_t(H, &H->tmp, (size_t)M * maxN * 4));
  }
  CKS(dalloc_t(H, &H->ws, std::max<size_t>(ws, 64) * 4));
  CKS(dalloc_t(H, &H->counters, std::max<size_t>(cnt, 64) * 4));
  CK(cudaMemset(H->counters, 0, std::max<size_t>(cnt, 64) * 4));

  H->n_chunk_slots = (c.max_ctx + ATTN_CHUNK - 1) / ATTN_CHUNK + 1;
  CKS(dalloc_t(H, &H->part_acc, (size_t)M * H->Hq * H->n_chunk_slots * H->hd * 4));
  CKS(dalloc_t(H, &H->part_ml, (size_t)M * H->Hq * H->n_chunk_slots * 8));

  // rotary table in double precision on the host: angle = pos * theta^(-2j/hd)
  const int half = H->hd / 2;
  std::vector<float2> rope((size_t)c.max_ctx * half);
  for (int pos = 0; pos < c.max_ctx; ++pos)
    for (int j = 0; j < half; ++j) {
      const double inv = std::pow((double)c.rope_theta, -2.0 * j / H->hd);
      const double a = (double)pos * inv;
      rope[(size_t)pos * half + j] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  CKS(dalloc_t(H, &H->rope, rope.size() * sizeof(float2)));
  CK(cudaMemcpy(H->rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice));

  H->h_pin_ints = std::max<size_t>((size_t)KMAX_CYCLES * c.max_batch * (H->B + 1) + (size_t)c.max_batch * (H->B + 2) * 2, 64);
  CK(cudaMallocHost(&H->h_pin, H->h_pin_ints * 4));
  for (auto& e : H->ev) CK(cudaEventCreate(&e));
  for (auto& e : H->cev) CK(cudaEventCreate(&e));
  CK(cudaStreamCreateWithFlags(&H->gstream, cudaStreamNonBlocking));
  for (auto& e : H->gjoin) CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  return DF_OK;
}

df_status ensure_debug_buffers(df_handle* H) {
  if (H->dbg_logits) return DF_OK;
  const size_t M = H->Mmax;
  CKS(dalloc_t(H, &H->dbg_logits, M * H->V * 4));
  CKS(dalloc_t(H, &H->dbg_dlogits, M * H->V * 4));
  CKS(dalloc_t(H, &H->dbg_dh, M * H->d * 4));
  CKS(dalloc_t(H, &H->dbg_th, M * H->d * 4));
  CKS(dalloc_t(H, &H->dbg_tl, (size_t)(H->L + 1) * M * H->d * 4));
  CKS(dalloc_t(H, &H->dbg_dl, (size_t)(H->Ld + 1) * M * H->d * 4));
  return DF_OK;
}

// Buffers of speculative sampling, allocated on first use.
df_status ensure_sampling_buffers(df_handle* H) {
  if (H->d_qlog) return DF_OK;
  if (H->V > SAMPLE_MAX_VOCAB) return fail(H, DF_EINVAL, "vocabulary too large for sampling");
  const size_t rows = (size_t)H->cfg.max_batch * H->B;
  CKS(dalloc_t(H, &H->d_qlog, rows * H->V * 4));
  CKS(dalloc_t(H, &H->d_plog, rows * H->V * 4));
  CKS(dalloc_t(H, &H->d_qst, rows * sizeof(SampleRow)));
  CKS(dalloc_t(H, &H->d_pst, rows * sizeof(SampleRow)));
  CKS(dalloc_t(H, &H->d_u, (size_t)H->cfg.max_batch * 2 * H->B * 4));
  CKS(dalloc_t(H, &H->d_ustream, (size_t)H->cfg.max_batch * 4));
  CKS(dalloc_t(H, &H->d_ucount, (size_t)H->cfg.max_batch * 8));
  return DF_OK;
}

}  // namespace

// =============================================================================
// C ABI
// =============================================================================
extern "C" {

df_status df_default_feat_layers(int32_t n_layers, int32_t out[5]) {
  if (!out || n_layers < 8) return DF_EINVAL;
  for (int i = 0; i < 5; ++i) out[i] = feat_default(n_layers, i);
  return DF_OK;
}

int32_t df_num_weights(const df_config* cfg) {
  if (!cfg || cfg->n_layers < 0 || cfg->draft_layers < 0) return -1;
  return (int32_t)weight_specs(*cfg).size();
}

df_status df_weight_info(const df_config* cfg, int32_t index, char name[32], int32_t* ndim, int64_t shape[2]) {
  if (!cfg) return DF_EINVAL;
  std::vector<WSpec> s = weight_specs(*cfg);
  if (index < 0 || index >= (int)s.size()) return DF_EINVAL;
  if (name) {
    std::memset(name, 0, 32);
    std::strncpy(name, s[index].name.c_str(), 31);
  }
  if (ndim) *ndim = s[index].ndim;
  if (shape) {
    shape[0] = s[index].s0;
    shape[1] = s[index].s1;
  }
  return DF_OK;
}

df_status df_init(const df_config* cfg, const void* const* weights, int32_t n_weights, void* stream,
                  df_handle** out) {
  if (!out) return DF_EINVAL;
  *out = nullptr;
  std::string why;
  if (validate(cfg, why) != DF_OK) return DF_EINVAL;
  if (!weights) return DF_EINVAL;
  df_handle* H = new df_handle();
  H->cfg = *cfg;
  H->st = reinterpret_cast<cudaStream_t>(stream);
  H->bf16 = cfg->dtype == DF_BF16;
  H->esz = H->bf16 ? 2 : 4;
  H->d = cfg->d_model;
  H->hd = cfg->head_dim;
  H->Hq = cfg->n_q_heads;
  H->Hkv = cfg->n_kv_heads;
  H->F = cfg->d_ffn;
  H->V = cfg->vocab;
  H->L = cfg->n_layers;
  H->Ld = cfg->draft_layers;
  H->B = cfg->block_size;
  H->blk_min = H->blk_max = H->B;
  H->qdim = H->Hq * H->hd;
  H->kvdim = H->Hkv * H->hd;
  H->qkv_n = H->qdim + 2 * H->kvdim;
  H->Mmax = std::max(std::min(PREFILL_CHUNK, cfg->max_ctx), cfg->max_batch * cfg->block_size);
  // attention kernel of the handle: the pipelined tcgen05 kernel for batches of 2 or more sequences or
  // one sequence beyond 8K positions, where it streams the cache fastest (clusters of 4, or of 8 for a
  // single sequence, which then has only 8 KV heads to spread); the mma.sync kernel (lowest latency)
  // for one sequence up to 8K positions.  Measured at batch 1 (one launch of the Qwen3-8B block
  // attention): 1K 16.4 vs 20.5 us, 8K 32.8 vs 32.8, 32K 86.0 vs 71.7 (mma.sync vs pipelined, 8 CTAs);
  // at batch 2: 1K 26.6 vs 22.5, 32K 157.7 vs 127.0 (clusters of 4).
  H->attn_pipe = H->bf16 && (cfg->attn_kernel == DF_ATTN_PIPE ||
                             (cfg->attn_kernel == DF_ATTN_AUTO && (cfg->max_batch >= DF_ATTN_PIPE_MIN_BATCH ||
                                                                   cfg->max_ctx > DF_ATTN_PIPE_MIN_CTX)));
  H->attn_cla = cfg->max_batch == 1 ? DF_ATTN_PIPE_CLUSTER_ONE : DF_ATTN_PIPE_CLUSTER;
  {
    const char* g = getenv("DF_NO_GRAPH");
    H->use_graphs = !(g && g[0] == '1');
    const char* gc = getenv("DF_GRAPH_CYCLES");  // cycles per captured graph in df_generate
    if (gc && atoi(gc) > 0) H->graph_cycles = std::min(KMAX_CYCLES, atoi(gc));
  }
  for (int l = 0; l < 1024; ++l) H->tap_of_layer[l] = -1;
  for (int i = 0; i < 5; ++i) H->tap_of_layer[cfg->feat_layers[i]] = i;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&H->sm_count, cudaDevAttrMultiProcessorCount, dev);
  H->split_target = tc_split_target(H->sm_count);
  {
    const char* sc = getenv("DF_SPLIT_CTAS");
    if (sc && atoi(sc) > 0) H->split_target = atoi(sc);
    const char* pf = getenv("DF_GEMM_L2PF");
    if (pf && atoi(pf) > 0) H->l2_prefetch = std::min(atoi(pf), 64);
  }
  if (e != cudaSuccess) {
    delete H;
    (void)cudaGetLastError();
    return DF_ECUDA;
  }
  if (H->bf16) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10) {
      delete H;
      return DF_ECUDA;
    }
  }
  if (tc_prepare() != cudaSuccess || attention_prepare() != cudaSuccess || sampling_prepare() != cudaSuccess) {
    delete H;
    (void)cudaGetLastError();
    return DF_ECUDA;
  }
  df_status s = pack_weights(H, weights, n_weights);
  if (s == DF_OK) s = alloc_state(H);
  if (s != DF_OK) {
    df_destroy(H);
    return s;
  }
  *out = H;
  return DF_OK;
}

#define GUARD(H)                                                              \
  do {                                                                        \
    if (!(H)) return DF_EINVAL;                                               \
    if ((H)->failed) return fail(H, DF_ECUDA, "handle is in a failed state"); \
  } while (0)

df_status df_prefill(df_handle* H, int32_t seq, const int32_t* prompt_host, int32_t len, int32_t* bonus_out) {
  GUARD(H);
  cudaEvent_t a = H->ev[0], b = H->ev[1];
  cudaEventRecord(a, H->st);
  df_status s = prefill_impl(H, seq, prompt_host, len, true, bonus_out);
  if (s != DF_OK) {
    if (seq >= 0 && seq < H->cfg.max_batch && H->seqs[seq].active && H->seqs[seq].len == 0) release(H, seq);
    return s;
  }
  cudaEventRecord(b, H->st);
  cudaEventSynchronize(b);
  float ms = 0.f;
  if (cudaEventElapsedTime(&ms, a, b) == cudaSuccess) H->stats.prefill_us += 1000.0 * ms;
  return DF_OK;
}

df_status df_draft_block(df_handle* H, const int32_t* seqs_host, int32_t nseq, int32_t* drafts_host) {
  GUARD(H);
  return draft_impl(H, seqs_host, nseq, drafts_host);
}

df_status df_verify_accept(df_handle* H, const int32_t* seqs_host, int32_t nseq, const int32_t* drafts_host,
                           int32_t* accepted_host, int32_t* n_host) {
  GUARD(H);
  return verify_impl(H, seqs_host, nseq, drafts_host, accepted_host, n_host, false);
}

static df_status generate_impl(df_handle* H, const int32_t* prompts_host, const int32_t* lens_host, int32_t nseq,
                               int32_t n_new, int32_t* out_host, df_stats* stats) {
  CKS(check_batch_args(H, prompts_host, lens_host, nseq, n_new, out_host));
  const df_stats before = H->stats;
  const int B = H->B;
  std::vector<int> count(nseq, 0);
  size_t off = 0;
  df_status s = DF_OK;
  for (int i = 0; i < nseq && s == DF_OK; ++i) {
    int bonus = 0;
    s = df_prefill(H, i, prompts_host + off, lens_host[i], &bonus);
    off += lens_host[i];
    if (s == DF_OK) out_host[(size_t)i * n_new] = bonus, count[i] = 1;
  }
  std::vector<int> active, acc((size_t)KMAX_CYCLES * nseq * B), n((size_t)KMAX_CYCLES * nseq);
  long long cyc = 0, emitted = 0;  // sequence-cycles run and tokens they emitted, for the choice of K
  // block size: fixed, or chosen per group from the recent tokens per cycle
  // (an average over groups, each weighted half as much as the next)
  const bool adaptive = H->blk_min < H->blk_max;
  int b = H->blk_max;
  H->gen_khist.assign(nseq, std::array<int64_t, 33>{});
  double tau = 0.0;
  bool have_tau = false;
  while (s == DF_OK) {
    active.clear();
    int remaining = n_new, room = KMAX_CYCLES;
    for (int i = 0; i < nseq; ++i)
      if (count[i] < n_new) {
        active.push_back(i);
        remaining = std::min(remaining, n_new - count[i]);
        room = std::min(room, (H->cfg.max_ctx - H->seqs[i].len) / B);
      }
    if (active.empty()) break;
    // Cycles per graph: as many as the sequence nearest to its end still
    // needs at the tokens per cycle seen so far (no wasted cycles at one token
    // per cycle), at most graph_cycles, and within max_ctx.
    const double per_cycle = cyc > 0 ? std::max(1.0, (double)emitted / (double)cyc) : 1.0;
    int K = (int)((double)remaining / per_cycle);
    K = std::max(1, std::min({K, H->graph_cycles, room}));
    const int na = (int)active.size();
    s = cycle_impl(H, active.data(), na, K, b, acc.data(), n.data());
    if (s != DF_OK) break;
    long long g_cyc = 0, g_emit = 0;
    for (int c = 0; c < K; ++c)
      for (int j = 0; j < na; ++j) {
        const int i = active[j];
        const int nj = n[(size_t)c * na + j];
        g_cyc += 1;
        g_emit += nj;
        if (count[i] < n_new) H->gen_khist[i][std::min(std::max(nj - 1, 0), 32)] += 1;
        for (int t = 0; t < nj && count[i] < n_new; ++t)
          out_host[(size_t)i * n_new + count[i]++] = acc[((size_t)c * na + j) * B + t];
      }
    cyc += g_cyc;
    emitted += g_emit;
    if (adaptive && g_cyc > 0) {
      const double t = (double)g_emit / (double)g_cyc;
      tau = have_tau ? 0.5 * tau + 0.5 * t : t;
      have_tau = true;
      b = block_size_for(tau, H->blk_min, H->blk_max);
    }
  }
  for (int i = 0; i < nseq; ++i)
    if (H->seqs[i].active) release(H, i);
  if (s != DF_OK) return s;
  for (int i = 0; i < nseq; ++i) H->stats.emitted_tokens += count[i];
  if (stats) {
    df_stats d{};
    d.cycles = H->stats.cycles - before.cycles;
    d.accepted_drafts = H->stats.accepted_drafts - before.accepted_drafts;
    d.emitted_tokens = H->stats.emitted_tokens - before.emitted_tokens;
    for (int k = 0; k < 65; ++k) d.accept_hist[k] = H->stats.accept_hist[k] - before.accept_hist[k];
    for (int k = 0; k < 33; ++k) d.block_hist[k] = H->stats.block_hist[k] - before.block_hist[k];
    d.draft_us = H->stats.draft_us - before.draft_us;
    d.verify_us = H->stats.verify_us - before.verify_us;
    d.prefill_us = H->stats.prefill_us - before.prefill_us;
    d.kernel_launches = H->stats.kernel_launches - before.kernel_launches;
    d.h2d_bytes = H->stats.h2d_bytes - before.h2d_bytes;
    d.d2h_bytes = H->stats.d2h_bytes - before.d2h_bytes;
    *stats = d;
  }
  return DF_OK;
}

df_status df_generate(df_handle* H, const int32_t* prompts_host, const int32_t* lens_host, int32_t nseq,
                      int32_t n_new, int32_t* out_host, df_stats* stats) {
  GUARD(H);
  return generate_impl(H, prompts_host, lens_host, nseq, n_new, out_host, stats);
}

df_status df_debug_wait_probe(df_handle* H) {
  GUARD(H);
  {
    ProfScope ps_(H, PC_CTRL, 1);
    CK(launch_wait_probe(H->d_err, H->st));
  }
  return sync(H);
}

df_status df_generate_accept_hist(const df_handle* H, int32_t seq, int64_t out[33]) {
  if (!H || !out) return DF_EINVAL;
  if (seq < 0 || seq >= (int32_t)H->gen_khist.size()) return DF_EINVAL;
  for (int k = 0; k < 33; ++k) out[k] = H->gen_khist[seq][k];
  return DF_OK;
}

df_status df_set_block_range(df_handle* H, int32_t b_min, int32_t b_max) {
  GUARD(H);
  if (b_min < 2 || b_min > b_max || b_max > H->B)
    return fail(H, DF_EINVAL, "block range must satisfy 2 <= b_min <= b_max <= block_size");
  H->blk_min = b_min;
  H->blk_max = b_max;
  return DF_OK;
}

int32_t df_block_size_for(double tokens_per_cycle, int32_t b_min, int32_t b_max) {
  if (b_min < 2 || b_min > b_max || b_max > 32 || !(tokens_per_cycle >= 0.0)) return -1;
  return block_size_for(tokens_per_cycle, b_min, b_max);
}

df_status df_generate_sampled(df_handle* H, const int32_t* prompts_host, const int32_t* lens_host, int32_t nseq,
                              int32_t n_new, float temperature, float top_p, uint64_t seed, int32_t* out_host,
                              df_stats* stats) {
  GUARD(H);
  if (!sampling_args_ok(temperature, top_p))
    return fail(H, DF_EINVAL, "temperature must be 0 or in [1e-3, 1e3] and top_p in [0, 1]");
  CKS(check_batch_args(H, prompts_host, lens_host, nseq, n_new, out_host));
  CKS(ensure_sampling_buffers(H));
  // sequence i of the call draws from generator stream i, from its first uniform
  std::vector<uint32_t> streams(nseq);
  for (int i = 0; i < nseq; ++i) streams[i] = (uint32_t)i;
  std::vector<unsigned long long> used(nseq, 0ull);
  CK(h2d(H, H->d_ustream, streams.data(), (size_t)nseq * 4));
  CK(h2d(H, H->d_ucount, used.data(), (size_t)nseq * 8));
  H->sampling = true;
  H->samp_inv_t = sampling_inv_t(temperature);
  H->samp_top_p = top_p;
  H->samp_seed = seed;
  const df_status s = generate_impl(H, prompts_host, lens_host, nseq, n_new, out_host, stats);
  H->sampling = false;
  return s;
}

df_status df_greedy_reference(df_handle* H, const int32_t* prompts_host, const int32_t* lens_host, int32_t nseq,
                              int32_t n_new, int32_t* out_host) {
  GUARD(H);
  CKS(check_batch_args(H, prompts_host, lens_host, nseq, n_new, out_host));
  std::vector<int> bonus(nseq), pos(nseq), sq(nseq);
  size_t off = 0;
  df_status s = DF_OK;
  for (int i = 0; i < nseq && s == DF_OK; ++i) {
    s = prefill_impl(H, i, prompts_host + off, lens_host[i], false, &bonus[i]);
    off += lens_host[i];
    pos[i] = lens_host[i];
    sq[i] = i;
  }
  int* d_gen = nullptr;
  if (s == DF_OK) {
    if (cudaMalloc(&d_gen, (size_t)nseq * n_new * 4) != cudaSuccess) s = fail(H, DF_ENOMEM, "output buffer");
  }
  auto body = [&]() -> df_status {
    CK(h2d(H, H->d_row_tok, bonus.data(), nseq * 4));
    CK(h2d(H, H->d_row_pos, pos.data(), nseq * 4));
    CK(h2d(H, H->d_row_seq, sq.data(), nseq * 4));
    CK(h2d(H, H->d_ids, bonus.data(), nseq * 4));
    { ProfScope ps_(H, PC_CTRL, 1); CK(launch_greedy_step(H->d_ids, nseq, 0, n_new, d_gen, H->d_row_tok, H->d_row_pos, H->st)); }
    // greedy_step advanced the positions; undo that for step 0's inputs
    CK(h2d(H, H->d_row_pos, pos.data(), nseq * 4));
    for (int t = 1; t < n_new; ++t) {
      int max_len = 0;
      for (int i = 0; i < nseq; ++i) {
        const int p = lens_host[i] + t - 1;  // position of this step's input token
        CKS(ensure_pages(H, i, p + 1));
        max_len = std::max(max_len, p + 1);
      }
      CKS(target_pass(H, nseq, 1, nseq, max_len, false, -1));
      { ProfScope ps_(H, PC_CTRL, 1); CK(launch_greedy_step(H->d_ids, nseq, t, n_new, d_gen, H->d_row_tok, H->d_row_pos, H->st)); }
    }
    CK(d2h(H, out_host, d_gen, (size_t)nseq * n_new * 4));
    return sync(H);
  };
  if (s == DF_OK) s = body();
  if (d_gen) cudaFree(d_gen);
  for (int i = 0; i < nseq; ++i)
    if (H->seqs[i].active) release(H, i);
  return s;
}

df_status df_reset_seq(df_handle* H, int32_t seq) {
  if (!H) return DF_EINVAL;
  if (seq < 0 || seq >= H->cfg.max_batch) return fail(H, DF_EINVAL, "sequence slot out of range");
  return release(H, seq);
}

df_status df_get_stats(const df_handle* H, df_stats* out) {
  if (!H || !out) return DF_EINVAL;
  *out = H->stats;
  return DF_OK;
}

df_status df_reset_stats(df_handle* H) {
  if (!H) return DF_EINVAL;
  H->stats = df_stats{};
  return DF_OK;
}

df_status df_seq_info(const df_handle* H, int32_t seq, int32_t* length, int32_t* bonus) {
  if (!H || seq < 0 || seq >= H->cfg.max_batch) return DF_EINVAL;
  if (length) *length = H->seqs[seq].len;
  if (bonus) *bonus = H->seqs[seq].bonus;
  return DF_OK;
}

void df_destroy(df_handle* H) {
  if (!H) return;
  if (H->st) cudaStreamSynchronize(H->st);
  else cudaDeviceSynchronize();
  for (void* p : H->allocs) cudaFree(p);
  if (H->h_pin) cudaFreeHost(H->h_pin);
  for (auto& e : H->ev)
    if (e) cudaEventDestroy(e);
  for (auto& e : H->evpool) cudaEventDestroy(e);
  drop_graph(H);
  if (H->gstream) {
    cudaStreamSynchronize(H->gstream);
    cudaStreamDestroy(H->gstream);
  }
  for (auto& e : H->gjoin)
    if (e) cudaEventDestroy(e);
  for (auto& e : H->cev)
    if (e) cudaEventDestroy(e);
  delete H;
}

const char* df_last_error(const df_handle* H) {
  if (!H) return "null handle";
  return H->err.c_str();
}

df_status df_debug_enable(df_handle* H, int32_t on) {
  if (!H) return DF_EINVAL;
  if (on) CKS(ensure_debug_buffers(H));
  H->debug = on != 0;
  return DF_OK;
}

df_status df_debug_read(df_handle* H, int32_t what, float* out_host, int64_t max_floats, int32_t* rows_out) {
  if (!H || !out_host) return DF_EINVAL;
  CK(cudaStreamSynchronize(H->st));
  const void* src = nullptr;
  bool typed = false;  // stored in the model dtype (else fp32)
  int rows = 0;
  size_t cols = 0;
  switch (what) {
    case DF_DBG_TAPS: src = H->taps; typed = true; rows = H->rows_last_target; cols = (size_t)5 * H->d; break;
    case DF_DBG_LOGITS: src = H->dbg_logits; rows = H->rows_last_logits; cols = H->V; break;
    case DF_DBG_DRAFT_LOGITS: src = H->dbg_dlogits; rows = H->rows_last_draft; cols = H->V; break;
    case DF_DBG_DRAFT_HIDDEN: src = H->dbg_dh; rows = H->rows_last_draft; cols = H->d; break;
    case DF_DBG_CTX: src = H->ctx; typed = true; rows = H->rows_last_ctx; cols = H->d; break;  // normalised below
    case DF_DBG_HIDDEN: src = H->dbg_th; rows = H->rows_last_target; cols = H->d; break;
    case DF_DBG_TARGET_LAYERS: src = H->dbg_tl; rows = (H->L + 1) * H->rows_last_target; cols = H->d; break;
    case DF_DBG_DRAFT_LAYERS: src = H->dbg_dl; rows = (H->Ld + 1) * H->rows_last_draft; cols = H->d; break;
    default: return fail(H, DF_EINVAL, "unknown debug buffer");
  }
  if (!src) return fail(H, DF_ESTATE, "debug buffers are off (df_debug_enable)");
  const size_t n = (size_t)rows * cols;
  if ((int64_t)n > max_floats) return fail(H, DF_EINVAL, "output buffer too small");
  if (typed && H->bf16) {
    std::vector<uint16_t> b(n);
    CK(cudaMemcpy(b.data(), src, n * 2, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < n; ++i) {
      uint32_t u = (uint32_t)b[i] << 16;
      std::memcpy(out_host + i, &u, 4);
    }
  } else {
    CK(cudaMemcpy(out_host, src, n * 4, cudaMemcpyDeviceToHost));
  }
  if (what == DF_DBG_CTX && rows > 0) {
    // the fused context rows are stored before their RMSNorm (which runs folded
    // into the injection GEMM): apply it here for inspection
    const int tiles = H->d / 128;
    std::vector<float> ss((size_t)rows * tiles), g(H->d);
    CK(cudaMemcpy(ss.data(), H->ss_ctx, ss.size() * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g.data(), H->fc_norm, g.size() * 4, cudaMemcpyDeviceToHost));
    for (int r = 0; r < rows; ++r) {
      double t = 0.0;
      for (int k = 0; k < tiles; ++k) t += ss[(size_t)r * tiles + k];
      const double inv = 1.0 / std::sqrt(t / H->d + (double)H->cfg.rms_eps);
      for (int i = 0; i < H->d; ++i) out_host[(size_t)r * H->d + i] = (float)(out_host[(size_t)r * H->d + i] * inv * g[i]);
    }
  }
  if (rows_out) *rows_out = rows;
  return DF_OK;
}

df_status df_debug_weight_ptr(const df_handle* H, int32_t which, uint64_t* addr) {
  if (!H || !addr) return DF_EINVAL;
  switch (which) {
    case 0:  // target embedding
    case 1:  // drafter embedding: the same table
      *addr = reinterpret_cast<uint64_t>(H->embed);
      return DF_OK;
    case 2:  // target LM head
    case 3:  // drafter LM head: the same matrix
      *addr = reinterpret_cast<uint64_t>(H->lm_head.ptr);
      return DF_OK;
    default: return DF_EINVAL;
  }
}

df_status df_profile_enable(df_handle* H, int32_t on) {
  if (!H || on < 0 || on > 2) return DF_EINVAL;
  if (on == 1 && H->evpool.empty()) {
    H->evpool.resize(EV_POOL, nullptr);
    for (auto& e : H->evpool) CK(cudaEventCreate(&e));
  }
  if (on == 2 && !H->d_trace) CKS(dalloc_t(H, &H->d_trace, TRACE_MAX * 16));
  if (on != 1) prof_resolve(H);
  H->profiling = on == 1;
  H->tracing = on == 2;
  H->trace_meta.clear();
  for (int c = 0; c < PC_N; ++c) {
    std::memset(H->prof[c].name, 0, 32);
    std::strncpy(H->prof[c].name, PC_NAMES[c], 31);
  }
  return DF_OK;
}

df_status df_profile_read(df_handle* H, df_kernel_stat* out, int32_t max, int32_t* n) {
  if (!H || !out || max < 0) return DF_EINVAL;
  prof_resolve(H);
  const int k = std::min<int>(max, PC_N);
  for (int c = 0; c < k; ++c) {
    out[c] = H->prof[c];
    std::memset(out[c].name, 0, 32);
    std::strncpy(out[c].name, PC_NAMES[c], 31);
  }
  for (int c = 0; c < PC_N; ++c) {
    H->prof[c].launches = 0;
    H->prof[c].total_us = H->prof[c].bytes = H->prof[c].flops = 0.0;
  }
  if (n) *n = k;
  return DF_OK;
}

df_status df_bench_drafter_step(df_handle* H, int32_t nseq, int32_t ctx_len, const float* taps_host,
                                 int32_t taps_rows, int32_t iters, double us_out[6]) {
  GUARD(H);
  const int B = H->B, d = H->d;
  if (nseq < 1 || nseq > H->cfg.max_batch || ctx_len < 1 || ctx_len + B > H->cfg.max_ctx || iters < 1 || !us_out ||
      !taps_host || taps_rows < nseq * B || taps_rows > H->Mmax)
    return fail(H, DF_EINVAL, "bad drafter-step benchmark arguments");
  for (int i = 0; i < nseq; ++i)
    if (H->seqs[i].active) return fail(H, DF_ESTATE, "slots 0..nseq-1 must be free");
  // taps rows in the model dtype
  {
    const size_t n = (size_t)taps_rows * 5 * d;
    if (H->bf16) {
      std::vector<uint16_t> b(n);
      for (size_t i = 0; i < n; ++i) {
        uint32_t u;
        std::memcpy(&u, taps_host + i, 4);
        u = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
        b[i] = (uint16_t)u;
      }
      CK(cudaMemcpy(H->taps, b.data(), n * 2, cudaMemcpyHostToDevice));
    } else {
      CK(cudaMemcpy(H->taps, taps_host, n * 4, cudaMemcpyHostToDevice));
    }
  }
  auto body = [&]() -> df_status {
    // context: every position of every sequence gets an injected feature row
    for (int sq = 0; sq < nseq; ++sq) {
      SeqHost& s = H->seqs[sq];
      s.active = true;
      s.len = ctx_len;
      s.bonus = 0;
      CKS(ensure_pages(H, sq, ctx_len + B));
      std::vector<int> pos(taps_rows), seqv(taps_rows, sq);
      for (int c0 = 0; c0 < ctx_len; c0 += taps_rows) {
        const int rows = std::min(taps_rows, ctx_len - c0);
        for (int i = 0; i < rows; ++i) pos[i] = c0 + i;
        CK(h2d(H, H->d_row_pos, pos.data(), rows * 4));
        CK(h2d(H, H->d_row_seq, seqv.data(), rows * 4));
        CKS(fuse_inject(H, rows, H->d_row_pos));
      }
      const int zero = 0;
      CK(h2d(H, H->d_bonus + sq, &zero, 4));
      CK(h2d(H, H->d_bonus_pos + sq, &ctx_len, 4));
    }
    std::vector<int> slots(nseq);
    for (int i = 0; i < nseq; ++i) slots[i] = i;
    CK(h2d(H, H->d_slots, slots.data(), nseq * 4));
    CKS(sync(H));
    const bool was = H->profiling;
    CKS(df_profile_enable(H, 1));
    df_kernel_stat junk[PC_N];
    int32_t nj = 0;
    CKS(df_profile_read(H, junk, PC_N, &nj));  // start from zero
    const int M = nseq * B;
    for (int it = 0; it < iters; ++it) {
      { ProfScope ps_(H, PC_CTRL, 1); CK(launch_prep_block(H->d_slots, nseq, B, H->d_bonus, H->d_bonus_pos, H->d_drafts, H->cfg.mask_token_id, 0, H->d_row_tok, H->d_row_pos, H->d_row_seq, H->st)); }
      // K1 fusion and K2 injection of one block of feature rows per sequence
      // (written at the block's positions, past the context the drafter reads)
      CKS(fuse_inject(H, M, H->d_row_pos));
      // K3 block attention (inside the drafter pass) and K5 LM-head argmax
      CKS(drafter_pass(H, nseq, ctx_len));
    }
    df_kernel_stat st[PC_N];
    CKS(df_profile_read(H, st, PC_N, &nj));
    CKS(df_profile_enable(H, 0));
    us_out[0] = st[PC_FUSE].total_us / iters;
    us_out[1] = st[PC_INJECT].total_us / iters;
    us_out[2] = st[PC_ATTN].total_us / iters;
    us_out[3] = st[PC_LMHEAD].total_us / iters;
    us_out[4] = st[PC_GEMM].total_us / iters;
    // the whole drafter pass without per-launch events (launch overlap intact)
    CK(cudaEventRecord(H->ev[0], H->st));
    for (int it = 0; it < iters; ++it) {
      { ProfScope ps_(H, PC_CTRL, 1); CK(launch_prep_block(H->d_slots, nseq, B, H->d_bonus, H->d_bonus_pos, H->d_drafts, H->cfg.mask_token_id, 0, H->d_row_tok, H->d_row_pos, H->d_row_seq, H->st)); }
      CKS(drafter_pass(H, nseq, ctx_len));
    }
    CK(cudaEventRecord(H->ev[1], H->st));
    CKS(sync(H));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, H->ev[0], H->ev[1]));
    us_out[5] = 1000.0 * ms / iters;
    if (was) CKS(df_profile_enable(H, 1));
    return DF_OK;
  };
  df_status s = body();
  for (int i = 0; i < nseq; ++i)
    if (H->seqs[i].active) release(H, i);
  return s;
}

// ---------------------------------------------------------------- single ops
df_status df_op_gemm_bf16(const void* x_dev, const void* w_dev, float* y_dev, int32_t M, int32_t N, int32_t K,
                          int32_t splits, int32_t token_tile, void* stream) {
  if (!x_dev || !w_dev || !y_dev || M < 1 || N % 128 || K % 64 || N <= 0 || K <= 0) return DF_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int sp = splits ? splits : tc_splits(N, K, tc_split_target(sms));
  if (sp < 1 || sp > K / 64) return DF_EINVAL;
  const int wide = token_tile < 0 ? -token_tile : (token_tile == 0 ? tc_wide_tile(M, N, K, sp) : 0);
  const int nt = wide ? wide : (token_tile ? token_tile : tc_token_tile(M));
  if (wide ? (nt != 64 && nt != 128) : (nt != 16 && nt != 32 && nt != 64 && nt != 128 && nt != 256)) return DF_EINVAL;
  Tmap tw, tx;
  if (!make_tmap_bf16(tw.b, w_dev, N, K, 128) || !make_tmap_bf16(tx.b, x_dev, M, K, nt)) return DF_EINVAL;
  EpiParams e{};
  e.kind = EPI_STORE_F32;
  e.out = y_dev;
  e.ldo = N;
  if (wide) return launch_gemm_tcw(tw.b, tx.b, nt, M, N, K, sp, e, st) == cudaSuccess ? DF_OK : DF_ECUDA;
  float* ws = nullptr;
  int* cnt = nullptr;
  const size_t wsf = tc_workspace_floats(M, N, sp, nt), cn = tc_counter_ints(M, N, nt);
  if (cudaMallocAsync(reinterpret_cast<void**>(&ws), std::max<size_t>(wsf, 1) * 4, st) != cudaSuccess) return DF_ENOMEM;
  if (cudaMallocAsync(reinterpret_cast<void**>(&cnt), cn * 4, st) != cudaSuccess) {
    cudaFreeAsync(ws, st);
    return DF_ENOMEM;
  }
  cudaMemsetAsync(cnt, 0, cn * 4, st);
  cudaError_t r = launch_gemm_tc(tw.b, tx.b, nt, M, N, K, sp, ws, cnt, e, st, tc_cluster_reduce(nt, sp));
  cudaFreeAsync(ws, st);
  cudaFreeAsync(cnt, st);
  return r == cudaSuccess ? DF_OK : DF_ECUDA;
}

df_status df_op_attention_bf16(const void* q_dev, void* out_dev, const void* cache_dev, int32_t n_pages,
                               const int32_t* page_table_dev, int32_t pt_stride, const int32_t* row_pos_dev,
                               const int32_t* row_seq_dev, const void* blk_dev, int32_t rows_cap, int32_t nseq,
                               int32_t rows_per_seq, int32_t n_q_heads, int32_t n_kv_heads, int32_t causal,
                               int32_t max_len, int32_t kernel, int32_t cluster_ctas, int32_t* err_dev,
                               void* stream) {
  if (!q_dev || !out_dev || !cache_dev || !page_table_dev || !row_pos_dev || !row_seq_dev || !err_dev) return DF_EINVAL;
  if (cluster_ctas != 0 && cluster_ctas != 2 && cluster_ctas != 4 && cluster_ctas != 8 && cluster_ctas != 16)
    return DF_EINVAL;
  if (n_pages < 1 || pt_stride < 1 || nseq < 1 || rows_per_seq < 1 || n_kv_heads < 1 || n_q_heads < n_kv_heads ||
      n_q_heads % n_kv_heads || n_q_heads / n_kv_heads > 8 || max_len < 1 || (causal != 0 && causal != 1) ||
      (kernel != DF_ATTN_MMA && kernel != DF_ATTN_PIPE))
    return DF_EINVAL;
  if ((long long)pt_stride * 16 < max_len) return DF_EINVAL;  // the page table cannot hold max_len positions
  if (!causal && (!blk_dev || rows_per_seq > 64 || rows_cap < nseq * rows_per_seq)) return DF_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Tmap map;
  if (!make_tmap_kvcache(map.b, cache_dev, n_pages, n_kv_heads, 16)) return DF_EINVAL;
  if (attention_prepare() != cudaSuccess) return DF_ECUDA;
  AttnParams p{};
  p.q = q_dev;
  p.out = out_dev;
  p.M = nseq * rows_per_seq;
  p.rows_per_seq = rows_per_seq;
  p.n_seqs = nseq;
  p.Hq = n_q_heads;
  p.Hkv = n_kv_heads;
  p.hd = 128;
  p.row_pos = row_pos_dev;
  p.row_seq = row_seq_dev;
  p.causal = causal;
  p.cache = cache_dev;
  p.page_table = page_table_dev;
  p.pt_stride = pt_stride;
  p.page_tokens = 16;
  p.n_pages = n_pages;
  p.blk = blk_dev;
  p.rows_cap = rows_cap;
  p.chunk = ATTN_CHUNK;
  p.grid_chunks = (max_len + ATTN_CHUNK - 1) / ATTN_CHUNK;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt(128.0));
  p.err = err_dev;
  p.kv_map = map.b;
  p.pipelined = kernel == DF_ATTN_PIPE ? 1 : 0;
  p.cla = cluster_ctas;
  if (!attention_cluster_fits(p)) return DF_EINVAL;
  // one of the two cluster kernels, never the partial + merge path (which needs workspaces)
  const cudaError_t e = p.pipelined ? launch_attention_tp(p, st) : launch_attention_cluster(p, st);
  if (e == cudaErrorInvalidValue) return DF_EINVAL;
  return e == cudaSuccess ? DF_OK : DF_ECUDA;
}

df_status df_op_lmhead_argmax_bf16(const void* x_dev, const void* wlm_dev, int32_t* ids_dev, int32_t M, int32_t V,
                                   int32_t K, void* stream) {
  if (!x_dev || !wlm_dev || !ids_dev || M < 1 || V % 128 || K % 64 || V <= 0 || K <= 0) return DF_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int sp = tc_splits(V, K, tc_split_target(sms));
  const int wide = tc_wide_tile(M, V, K, sp);  // the engine's choice of form
  const int nt = wide ? wide : tc_token_tile(M);
  Tmap tw, tx;
  if (!make_tmap_bf16(tw.b, wlm_dev, V, K, 128) || !make_tmap_bf16(tx.b, x_dev, M, K, nt)) return DF_EINVAL;
  float* ws = nullptr;
  int* cnt = nullptr;
  unsigned long long* amax = nullptr;
  const size_t wsf = tc_workspace_floats(M, V, sp, nt), cn = tc_counter_ints(M, V, nt);
  if (cudaMallocAsync(reinterpret_cast<void**>(&ws), std::max<size_t>(wsf, 1) * 4, st) != cudaSuccess) return DF_ENOMEM;
  if (cudaMallocAsync(reinterpret_cast<void**>(&cnt), cn * 4, st) != cudaSuccess ||
      cudaMallocAsync(reinterpret_cast<void**>(&amax), (size_t)M * 8, st) != cudaSuccess) {
    cudaFreeAsync(ws, st);
    if (cnt) cudaFreeAsync(cnt, st);
    return DF_ENOMEM;
  }
  cudaMemsetAsync(cnt, 0, cn * 4, st);
  cudaMemsetAsync(amax, 0, (size_t)M * 8, st);
  EpiParams e{};
  e.kind = EPI_ARGMAX;
  e.amax = amax;
  cudaError_t r = wide ? launch_gemm_tcw(tw.b, tx.b, nt, M, V, K, sp, e, st)
                       : launch_gemm_tc(tw.b, tx.b, nt, M, V, K, sp, ws, cnt, e, st, tc_cluster_reduce(nt, sp));
  if (r == cudaSuccess) r = launch_argmax_finalize(amax, ids_dev, M, st);
  cudaFreeAsync(ws, st);
  cudaFreeAsync(cnt, st);
  cudaFreeAsync(amax, st);
  return r == cudaSuccess ? DF_OK : DF_ECUDA;
}

df_status df_op_bench_gemm_bf16(const void* x_dev, const void* w_dev, float* y_dev, int32_t M, int32_t N, int32_t K,
                                int32_t splits, int32_t token_tile, int32_t iters, void* stream, float* us_per_launch) {
  if (!x_dev || !w_dev || !y_dev || !us_per_launch || M < 1 || N % 128 || K % 64 || N <= 0 || K <= 0 || iters < 1)
    return DF_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int sp = splits ? splits : tc_splits(N, K, tc_split_target(sms));
  if (sp < 1 || sp > K / 64) return DF_EINVAL;
  const int wide = token_tile < 0 ? -token_tile : (token_tile == 0 ? tc_wide_tile(M, N, K, sp) : 0);
  const int nt = wide ? wide : (token_tile ? token_tile : tc_token_tile(M));
  if (wide ? (nt != 64 && nt != 128) : (nt != 16 && nt != 32 && nt != 64 && nt != 128 && nt != 256)) return DF_EINVAL;
  Tmap tw, tx;
  if (!make_tmap_bf16(tw.b, w_dev, N, K, 128) || !make_tmap_bf16(tx.b, x_dev, M, K, nt)) return DF_EINVAL;
  float* ws = nullptr;
  int* cnt = nullptr;
  const size_t wsf = tc_workspace_floats(M, N, sp, nt), cn = tc_counter_ints(M, N, nt);
  if (cudaMalloc(reinterpret_cast<void**>(&ws), std::max<size_t>(wsf, 1) * 4) != cudaSuccess) return DF_ENOMEM;
  if (cudaMalloc(reinterpret_cast<void**>(&cnt), cn * 4) != cudaSuccess) {
    cudaFree(ws);
    return DF_ENOMEM;
  }
  cudaMemsetAsync(cnt, 0, cn * 4, st);
  EpiParams e{};
  e.kind = EPI_STORE_F32;
  e.out = y_dev;
  e.ldo = N;
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  const bool cr = tc_cluster_reduce(nt, sp);
  auto one = [&]() {
    return wide ? launch_gemm_tcw(tw.b, tx.b, nt, M, N, K, sp, e, st)
                : launch_gemm_tc(tw.b, tx.b, nt, M, N, K, sp, ws, cnt, e, st, cr);
  };
  cudaError_t r = one();  // warm-up
  cudaEventRecord(a, st);
  for (int i = 0; i < iters && r == cudaSuccess; ++i) r = one();
  cudaEventRecord(b, st);
  cudaStreamSynchronize(st);
  float ms = 0.f;
  cudaEventElapsedTime(&ms, a, b);
  *us_per_launch = 1000.f * ms / iters;
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaFree(ws);
  cudaFree(cnt);
  return r == cudaSuccess ? DF_OK : DF_ECUDA;
}

}  // extern "C"
