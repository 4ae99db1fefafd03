// df_op_gemm_bf16_noalloc: the tcgen05 GEMM of df_op_gemm_bf16 for callers
// that must not allocate device memory.
//
// df_op_gemm_bf16 adds split-K partials through a thread-block cluster, or
// else through a workspace and tile tickets from cudaMallocAsync on every
// call.  This variant always takes the workspace form, with scratch that is
// never allocated.  Some callers cannot allocate: a process whose
// device memory is reserved up front by its own pool (every byte accounted by
// that pool), or a latency-critical loop where an allocation and its release
// would add synchronisation.  This variant keeps that scratch in two
// file-scope device arrays of fixed size instead.  Each GPU that loads the
// library holds them (DF_NOALLOC_WS_FLOATS floats + DF_NOALLOC_TICKETS ints,
// a little over 4 MiB) until the process exits.
//
// In host code the arrays' names are host-side stand-ins, not device
// addresses, so the first call on each device looks their addresses up with
// cudaGetSymbolAddress while that device is current, and every later call on
// the device reuses them.  The addresses belong to the device's CUDA context:
// after a reset of that context (cudaDeviceReset, or a new primary context)
// the module is loaded again at other addresses, so the lookup is keyed on
// the current context as well and repeated when it changes.
#include <cuda.h>

#include <mutex>

#include "dflash.h"
#include "internal.h"

using namespace dfk;

static __device__ __align__(256) float g_noalloc_ws[DF_NOALLOC_WS_FLOATS];
static __device__ __align__(256) int g_noalloc_tickets[DF_NOALLOC_TICKETS];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceScratch {
  float* ws = nullptr;
  int* tickets = nullptr;
  CUcontext ctx = nullptr;  // the context the addresses were looked up in
  bool ready = false;
};

std::mutex g_scratch_mu;
DeviceScratch g_scratch[kMaxDevices];

typedef CUresult (*PFN_ctxGetCurrent_t)(CUcontext*);

// The current CUDA context (the runtime makes the device's primary context
// current on first use), through the driver entry point the runtime exposes.
cudaError_t current_context(CUcontext* ctx) {
  static PFN_ctxGetCurrent_t fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return cudaErrorNotSupported;
    fn = reinterpret_cast<PFN_ctxGetCurrent_t>(p);
  }
  *ctx = nullptr;
  return fn(ctx) == CUDA_SUCCESS && *ctx ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device addresses of the scratch arrays in the current device's context
// (looked up once per device and context).
cudaError_t scratch_on_current_device(float** ws, int** tickets) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  e = cudaSetDevice(dev);  // makes the device's primary context current if it is not yet
  if (e != cudaSuccess) return e;
  CUcontext ctx = nullptr;
  e = current_context(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  DeviceScratch& s = g_scratch[dev];
  if (!s.ready || s.ctx != ctx) {
    void* p = nullptr;
    void* q = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(&q, g_noalloc_tickets);
    if (e != cudaSuccess) return e;
    s.ws = static_cast<float*>(p);
    s.tickets = static_cast<int*>(q);
    s.ctx = ctx;
    s.ready = true;
  }
  *ws = s.ws;
  *tickets = s.tickets;
  return cudaSuccess;
}

}  // namespace

extern "C" df_status df_op_gemm_bf16_noalloc(const void* x_dev, const void* w_dev, float* y_dev, int32_t M, int32_t N,
                                             int32_t K, int32_t splits, int32_t token_tile, void* stream) {
  if (!x_dev || !w_dev || !y_dev || M < 1 || N <= 0 || K <= 0 || N % 128 || K % 64) return DF_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess) return DF_ECUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DF_ECUDA;
  const int nt = token_tile ? token_tile : tc_token_tile(M);
  if (nt != 16 && nt != 32 && nt != 64 && nt != 128 && nt != 256) return DF_EINVAL;
  const int sp = splits ? splits : tc_splits(N, K, tc_split_target(sms));
  if (sp < 1 || sp > K / 64) return DF_EINVAL;
  // The shape must fit the fixed scratch: reject it before touching the GPU.
  const size_t ws_floats = tc_workspace_floats(M, N, sp, nt);
  const size_t n_tickets = tc_counter_ints(M, N, nt);
  if (ws_floats > (size_t)DF_NOALLOC_WS_FLOATS || n_tickets > (size_t)DF_NOALLOC_TICKETS) return DF_EINVAL;
  alignas(64) uint8_t tw[TMAP_BYTES];
  alignas(64) uint8_t tx[TMAP_BYTES];
  if (!make_tmap_bf16(tw, w_dev, N, K, 128) || !make_tmap_bf16(tx, x_dev, M, K, nt)) return DF_EINVAL;
  float* ws = nullptr;
  int* tickets = nullptr;
  if (scratch_on_current_device(&ws, &tickets) != cudaSuccess) return DF_ECUDA;
  // Tickets must start at zero; a finished launch leaves them at zero, an
  // interrupted one may not, so clear the ones this shape uses.
  if (cudaMemsetAsync(tickets, 0, n_tickets * sizeof(int), st) != cudaSuccess) return DF_ECUDA;
  EpiParams e{};
  e.kind = EPI_STORE_F32;
  e.out = y_dev;
  e.ldo = N;
  return launch_gemm_tc(tw, tx, nt, M, N, K, sp, ws, tickets, e, st) == cudaSuccess ? DF_OK : DF_ECUDA;
}
