// noalloc.cu -- selection (scores -> max-pool -> per-head top-k) for callers that
// cannot allocate device memory.
//
// Some callers own every byte of device memory themselves: serving runtimes that
// carve all GPU memory into their own arena up front and keep exact accounting,
// or latency-critical loops where a cudaMalloc (which may synchronize the device
// and can fail under fragmentation) is not acceptable. kvc_select_noalloc gives
// them the prefill selection without any allocation: the caller passes inputs
// and outputs, and the intermediate buffers (partial row statistics, scores,
// pooled scores) live in one file-scope static device array
// of fixed size, KVC_NOALLOC_SCRATCH_BYTES.
//
// Properties of that array:
//   * every GPU that loads this library holds it until the process exits;
//   * all calls share it and it keeps the previous call's contents; every
//     element a call reads is first written by that same call, so nothing has
//     to be cleared;
//   * calls whose work overlaps on the GPU (different streams, or devices
//     sharing a context) race on it: serialize them.
// A second static array, zero at load, holds the scoring launch's counters (one
// per (sequence, kv head) plus one); each launch leaves them at zero again, and it
// bounds B*H at kMaxUnits. A third static word is the scoring launch's error
// word: a bounded wait that gives up sets it, the top-k launch then writes every
// kept index as -1 (never a stale selection), and kvc_select_noalloc_check
// reports and clears it.
// In host code the arrays' names are only host-side stand-ins, not device
// addresses, so their device addresses are looked up once per device
// (cudaGetSymbolAddress, with that device current) on the first call made on
// that device; make that first call before any stream capture. The runtime
// loads the module holding the arrays lazily, so that first lookup is also when
// the device commits the 32 MiB: make the first call before an arena reserves
// the rest of the device's memory (if it cannot be committed, the call returns
// KVC_E_OOM).
#include <mutex>

#include "kvc_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KVC_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_select_scratch[kScratchBytes];
constexpr int kMaxUnits = 8192;
static __device__ unsigned g_select_sync[1 + kMaxUnits] = {0u};
static __device__ unsigned g_select_err = 0u;

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
void* g_sync_addr[kMaxDevices] = {};
void* g_err_addr[kMaxDevices] = {};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

kvc_status scratch_for_current_device(void** out, unsigned** sync, unsigned** err) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_E_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    void* q = nullptr;
    void* r = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&q, g_select_sync);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&r, g_select_err);
    if (e != cudaSuccess || !p || !q || !r) {
      cudaGetLastError();
      return e == cudaErrorMemoryAllocation ? KVC_E_OOM : KVC_E_CUDA;
    }
    g_scratch_addr[dev] = p;
    g_sync_addr[dev] = q;
    g_err_addr[dev] = r;
  }
  *out = g_scratch_addr[dev];
  *sync = static_cast<unsigned*>(g_sync_addr[dev]);
  *err = static_cast<unsigned*>(g_err_addr[dev]);
  return KVC_OK;
}

}  // namespace

extern "C" kvc_status kvc_select_noalloc(const kvc_dims* dims, int32_t budget, const void* q_obs,
                                         const void* k, int32_t* kept, float* scores,
                                         void* stream) {
  if (!dims || !q_obs || !k || !kept || budget < 0) return KVC_E_ARG;
  const kvc_dims& d = *dims;
  if (d.batch < 1 || d.n_q_heads < 1 || d.n_kv_heads < 1 || d.n_q_heads % d.n_kv_heads)
    return KVC_E_SHAPE;
  const int g = d.n_q_heads / d.n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return KVC_E_SHAPE;
  if (d.head_dim != 64 && d.head_dim != 128) return KVC_E_SHAPE;
  if (d.prompt_len < 2 || d.obs_window < 1 || d.obs_window >= d.prompt_len) return KVC_E_SHAPE;
  if (g * d.obs_window > 256) return KVC_E_SHAPE;
  if (d.pool_kernel < 1 || d.pool_kernel % 2 == 0) return KVC_E_ARG;

  const size_t units = (size_t)d.batch * d.n_kv_heads;
  if (units > (size_t)kMaxUnits) return KVC_E_CAPACITY;
  const size_t M = (size_t)g * d.obs_window;
  const size_t ns = (size_t)d.prompt_len - d.obs_window;
  const size_t nch = kvc::score_stat_chunks(d.prompt_len);
  const size_t stats_b = align256(units * nch * M * sizeof(float2));
  const size_t score_b = align256(units * ns * sizeof(float));
  const size_t need = stats_b + (scores ? 0 : score_b) + score_b;
  if (need > kScratchBytes) return KVC_E_CAPACITY;   // larger than the static scratch

  void* base = nullptr;
  unsigned* gsync = nullptr;
  unsigned* err = nullptr;
  kvc_status st = scratch_for_current_device(&base, &gsync, &err);
  if (st != KVC_OK) return st;
  unsigned char* p = static_cast<unsigned char*>(base);
  float2* stats = reinterpret_cast<float2*>(p);
  float* pooled = reinterpret_cast<float*>(p + stats_b);
  float* sc = scores ? scores : reinterpret_cast<float*>(p + stats_b + score_b);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int k_sel = (size_t)budget < ns ? budget : (int)ns;
  cudaError_t e = kvc::launch_score_into(d, static_cast<const __nv_bfloat16*>(q_obs),
                                         static_cast<const __nv_bfloat16*>(k), stats, gsync, sc,
                                         err, s);
  if (e == cudaSuccess) e = kvc::launch_pool_topk_into(d, sc, pooled, kept, k_sel, err, s);
  if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? KVC_E_OOM : KVC_E_CUDA;
  return KVC_OK;
}

extern "C" kvc_status kvc_select_noalloc_check(void* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_E_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_addr[dev]) return KVC_OK;   // no call on this device yet
  }
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_E_CUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_select_err, sizeof(word)) != cudaSuccess) return KVC_E_CUDA;
  if (word == 0) return KVC_OK;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_select_err, &zero, sizeof(zero)) != cudaSuccess) return KVC_E_CUDA;
  return KVC_E_TIMEOUT;
}
