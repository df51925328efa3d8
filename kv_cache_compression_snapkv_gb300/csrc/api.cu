// api.cu -- the C ABI (include/kvc.h): argument validation, cache creation and
// sizing, host-side tracking of each layer's packed/window state, and the
// orchestration of the device kernels. No device arithmetic happens here.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <new>

#include <mutex>

#include "kvc_internal.cuh"

using kvc::LayerState;

namespace {

std::atomic<uint64_t> g_launches{0};

kvc_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return KVC_OK;
  if (e == cudaErrorMemoryAllocation) return KVC_E_OOM;
  return KVC_E_CUDA;
}

// Keeps the caller's current device and switches to the cache's device.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

kvc_status check_dims(const kvc_dims* d) {
  if (!d) return KVC_E_ARG;
  if (d->n_layers < 1 || d->n_layers > 256) return KVC_E_SHAPE;
  if (d->batch < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1) return KVC_E_SHAPE;
  if ((int64_t)d->batch * d->n_q_heads > KVC_MAX_QUERY_HEADS) return KVC_E_SHAPE;
  if (d->n_q_heads % d->n_kv_heads) return KVC_E_SHAPE;
  const int g = d->n_q_heads / d->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return KVC_E_SHAPE;
  if (d->head_dim != 64 && d->head_dim != 128) return KVC_E_SHAPE;
  if (d->prompt_len < 1 || d->prompt_len > KVC_MAX_PROMPT_LEN) return KVC_E_SHAPE;
  if (d->obs_window < 0 || d->obs_window >= d->prompt_len) return KVC_E_SHAPE;
  if (d->pool_kernel < 1 || d->pool_kernel % 2 == 0) return KVC_E_ARG;
  if (d->bits != 2 && d->bits != 4 && d->bits != 16) return KVC_E_ARG;
  if (d->group_size != KVC_GROUP) return KVC_E_ARG;
  // 16-bit storage keeps the whole cache in the bf16 window, which may then be long
  if (d->window_len < KVC_GROUP || d->window_len > (d->bits == 16 ? 65536 : 1024) ||
      d->window_len % KVC_GROUP)
    return KVC_E_SHAPE;
  if (d->max_new_tokens < 0) return KVC_E_ARG;
  if (d->max_new_tokens > KVC_MAX_NEW_TOKENS) return KVC_E_SHAPE;
  if (d->obs_window >= d->window_len) return KVC_E_SHAPE;
  if ((d->alloc == nullptr) != (d->free == nullptr)) return KVC_E_ARG;
  return KVC_OK;
}

bool same_dims(const kvc_dims& a, const kvc_dims& b) {
  return a.n_layers == b.n_layers && a.batch == b.batch && a.n_q_heads == b.n_q_heads &&
         a.n_kv_heads == b.n_kv_heads && a.head_dim == b.head_dim &&
         a.prompt_len == b.prompt_len && a.obs_window == b.obs_window &&
         a.pool_kernel == b.pool_kernel && a.bits == b.bits && a.group_size == b.group_size &&
         a.window_len == b.window_len && a.max_new_tokens == b.max_new_tokens;
}

void* dev_alloc(kvc_cache* c, size_t bytes) {
  if (bytes == 0) bytes = 16;
  void* p = nullptr;
  if (c->dims.alloc) {
    p = c->dims.alloc(bytes, nullptr, c->dims.alloc_ctx);
  } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    p = nullptr;
  }
  if (p) c->allocations.push_back(p);
  return p;
}

void release_all(kvc_cache* c) {
  for (void* p : c->allocations) {
    if (c->dims.free) c->dims.free(p, nullptr, c->dims.alloc_ctx);
    else cudaFree(p);
  }
  c->allocations.clear();
  if (c->err_pinned) cudaFreeHost(c->err_pinned);
  c->err_pinned = nullptr;
  c->err_host = nullptr;
}

// The cache's error word: in mapped pinned host memory when the device has native
// atomics on host memory (the kernels' atomicOr then lands where the host reads it
// without synchronising), else in device memory.
bool make_error_word(kvc_cache* c) {
  int native = 0, can_map = 0;
  if (cudaDeviceGetAttribute(&native, cudaDevAttrHostNativeAtomicSupported, c->device) ==
          cudaSuccess &&
      cudaDeviceGetAttribute(&can_map, cudaDevAttrCanMapHostMemory, c->device) == cudaSuccess &&
      native && can_map) {
    void* h = nullptr;
    void* d = nullptr;
    if (cudaHostAlloc(&h, 16, cudaHostAllocMapped | cudaHostAllocPortable) == cudaSuccess) {
      if (cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess) {
        std::memset(h, 0, 16);
        c->err_pinned = h;
        c->err_host = static_cast<volatile unsigned*>(h);
        c->err = static_cast<unsigned*>(d);
        return true;
      }
      cudaFreeHost(h);
    }
    cudaGetLastError();
  }
  c->err = static_cast<unsigned*>(dev_alloc(c, 16));
  return c->err != nullptr && cudaMemset(c->err, 0, 16) == cudaSuccess;
}

// A bounded device wait of earlier work on the cache gave up (seen without a
// synchronisation where the error word is host-visible): report it once.
kvc_status word_status(unsigned word) {
  if (word == 0u) return KVC_OK;
  return (word & kvc::kErrDeviceCheck) ? KVC_E_DEVICE_CHECK : KVC_E_TIMEOUT;
}

kvc_status pending_error(kvc_cache* c) {
  if (c->err_host && *c->err_host != 0u) {
    const unsigned word = *c->err_host;
    *c->err_host = 0u;
    return word_status(word);
  }
  return KVC_OK;
}

int kept_cap(const kvc_dims& d, int budget) {
  const int ns = d.prompt_len - d.obs_window;
  return budget < ns ? budget : ns;
}

// The initial window of a layer keeping n_kept tokens fits its ring of R slots: the
// tokens past the last whole group plus the observation tokens (2/4-bit), or, with
// 16-bit storage (no packed store, no flush), every kept, observation and appended
// token.
bool window_fits(const kvc_dims& d, int bits, int R, int n_kept) {
  if (bits == 16) return (int64_t)n_kept + d.obs_window + d.max_new_tokens <= R;
  return n_kept % KVC_GROUP + d.obs_window < R;
}

// Ring length of a layer stored at `bits`: the cache's window_len, except a 16-bit
// layer of a cache whose default precision is 2 or 4 bits, whose ring is sized to
// hold every token it will store.
int ring_len(const kvc_dims& d, int bits, int n_kept) {
  if (bits != 16 || d.bits == 16) return d.window_len;
  const int64_t need = (int64_t)n_kept + d.obs_window + d.max_new_tokens;
  const int64_t R = (need + KVC_GROUP - 1) / KVC_GROUP * KVC_GROUP;
  return (int)std::min<int64_t>(std::max<int64_t>(KVC_GROUP, R), INT32_MAX / 2);
}

kvc_status create(const kvc_dims* dims, const int32_t* budgets, const int32_t* layer_bits,
                  kvc_cache** out) {
  kvc_status st = check_dims(dims);
  if (st != KVC_OK) return st;
  if (!budgets || !out) return KVC_E_ARG;
  const kvc_dims& d = *dims;
  const int units = d.batch * d.n_kv_heads;
  const int g = d.n_q_heads / d.n_kv_heads;
  const int ns = d.prompt_len - d.obs_window;
  bool scoring = false;
  for (int l = 0; l < d.n_layers; ++l) {
    if (budgets[l] < 0) return KVC_E_ARG;
    const int bits = layer_bits ? layer_bits[l] : d.bits;
    if (bits != 2 && bits != 4 && bits != 16) return KVC_E_ARG;
    const int nk = kept_cap(d, budgets[l]);
    const int R = ring_len(d, bits, nk);
    if (R > 65536 || !window_fits(d, bits, R, nk)) return KVC_E_SHAPE;
    if (nk < ns) scoring = true;
  }
  if (scoring && (d.obs_window < 1 || g * d.obs_window > 256)) return KVC_E_SHAPE;

  kvc_cache* c = new (std::nothrow) kvc_cache();
  if (!c) return KVC_E_OOM;
  c->dims = d;
  c->g = g;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->n_sm, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return KVC_E_CUDA;
  }
  c->L.resize(d.n_layers);
  size_t packed = 0, win = 0;
  for (int l = 0; l < d.n_layers; ++l) {
    LayerState& ls = c->L[l];
    ls.bits = layer_bits ? layer_bits[l] : d.bits;
    ls.budget = kept_cap(d, budgets[l]);
    ls.R = ring_len(d, ls.bits, ls.budget);
    ls.block_bytes = ls.bits == 16 ? 0 : kvc::block_bytes(d.head_dim, ls.bits);
    ls.cap_groups = ls.bits == 16 ? 0 :   // 16-bit storage: everything stays in the window
                    ls.budget / KVC_GROUP +
                    (KVC_GROUP - 1 + d.obs_window + d.max_new_tokens + KVC_GROUP - 1) / KVC_GROUP + 1;
    ls.packed_off = packed;
    packed += (size_t)units * ls.cap_groups * ls.block_bytes;
    ls.win_off = win;
    win += (size_t)units * ls.R * d.head_dim;
  }
  c->packed_bytes = packed;
  c->win_elems = win;

  c->packed = static_cast<uint8_t*>(dev_alloc(c, packed));
  c->win_k = static_cast<__nv_bfloat16*>(dev_alloc(c, c->win_elems * 2));
  c->win_v = static_cast<__nv_bfloat16*>(dev_alloc(c, c->win_elems * 2));
  const bool err_ok = make_error_word(c);
  c->dec_ws_floats = kvc::decode_workspace_floats(c->n_sm, g, d.head_dim);
  c->dec_ws = static_cast<float*>(dev_alloc(c, c->dec_ws_floats * 4));
  c->dec_cnt = static_cast<unsigned*>(dev_alloc(c, (size_t)d.n_layers * units * 4));
  bool ok = c->packed && c->win_k && c->win_v && err_ok && c->dec_ws && c->dec_cnt;
  if (ok && scoring) {
    const int M = g * d.obs_window;
    c->stats_elems = (size_t)units * kvc::score_stat_chunks(d.prompt_len) * M;
    c->score_elems = (size_t)units * ns;
    c->stats = static_cast<float2*>(dev_alloc(c, c->stats_elems * 8));
    c->gsync = static_cast<unsigned*>(dev_alloc(c, (units + 1) * 4));
    c->scores = static_cast<float*>(dev_alloc(c, c->score_elems * 4));
    c->pooled = static_cast<float*>(dev_alloc(c, c->score_elems * 4));
    ok = c->stats && c->gsync && c->scores && c->pooled &&
         cudaMemset(c->gsync, 0, (units + 1) * 4) == cudaSuccess;
  }
  // kept positions are stored for selective layers (keep-all layers are the identity)
  if (ok) {
    size_t off = 0;
    for (int l = 0; l < d.n_layers; ++l) {
      c->L[l].kept_off = off;
      if (c->L[l].budget < ns) off += (size_t)units * c->L[l].budget;
    }
    c->kept_elems = off;
    c->kept = static_cast<int32_t*>(dev_alloc(c, off * 4));
    ok = c->kept != nullptr;
    for (int l = 0; ok && l < d.n_layers; ++l)
      if (c->L[l].budget < ns) c->L[l].kept_ptr = c->kept + c->L[l].kept_off;
  }
  if (ok) {
    // the window is zero-initialised: masked slots must hold finite values
    ok = cudaMemset(c->win_k, 0, c->win_elems * 2) == cudaSuccess &&
         cudaMemset(c->win_v, 0, c->win_elems * 2) == cudaSuccess &&
         cudaMemset(c->dec_cnt, 0, (size_t)d.n_layers * units * 4) == cudaSuccess &&
         cudaDeviceSynchronize() == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    release_all(c);
    delete c;
    return KVC_E_OOM;
  }
  *out = c;
  return KVC_OK;
}

kvc_status finish_prefill(kvc_cache* c, int layer, int n_kept, const int32_t* kept,
                          const void* k, const void* v, cudaStream_t stream, int sinks = -1,
                          int32_t* kept_out = nullptr) {
  const auto* K = static_cast<const __nv_bfloat16*>(k);
  const auto* V = static_cast<const __nv_bfloat16*>(v);
  // one launch: whole groups into the packed store plus the initial window
  cudaError_t e = kvc::launch_gather_quant(c, layer, kept, n_kept, K, V, stream, sinks, kept_out);
  if (e != cudaSuccess) return from_cuda(e);
  LayerState& ls = c->L[layer];
  const bool exact = ls.bits == 16;
  ls.n_kept = n_kept;
  ls.n_groups = exact ? 0 : n_kept / KVC_GROUP;
  ls.win_start = 0;
  ls.win_len = (exact ? n_kept : n_kept % KVC_GROUP) + c->dims.obs_window;
  ls.appended = 0;
  ls.prefilled = 1;
  return KVC_OK;
}

}  // namespace

void kvc::count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

cudaError_t kvc::ensure_smem(const void* kernel, size_t bytes) {
  struct Entry { const void* kernel; int device; size_t bytes; };
  static std::mutex mu;
  static std::vector<Entry> set;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (Entry& x : set)
    if (x.kernel == kernel && x.device == dev) {
      if (x.bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
      if (e == cudaSuccess) x.bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) set.push_back({kernel, dev, bytes});
  return e;
}

extern "C" {

uint64_t kvc_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

kvc_status kvc_cache_reset(kvc_cache* c) {
  if (!c) return KVC_E_ARG;
  for (LayerState& ls : c->L) {
    ls.prefilled = 0;
    ls.n_kept = 0;
    ls.n_groups = 0;
    ls.win_start = 0;
    ls.win_len = 0;
    ls.appended = 0;
    if (ls.budget >= c->dims.prompt_len - c->dims.obs_window) ls.scored = 0;
  }
  c->last_scored_layer = -1;
  return KVC_OK;
}

const char* kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "ok";
    case KVC_E_ARG: return "invalid argument";
    case KVC_E_SHAPE: return "unsupported or inconsistent dimensions";
    case KVC_E_OOM: return "device allocation failed";
    case KVC_E_CUDA: return "CUDA error";
    case KVC_E_STATE: return "call out of order";
    case KVC_E_CAPACITY: return "capacity exceeded";
    case KVC_E_TIMEOUT: return "device-side wait timed out";
    case KVC_E_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

kvc_status kvc_plan_budgets(const kvc_dims* dims, kvc_schedule schedule, int32_t avg_budget,
                            int32_t pyramid_depth, int32_t* budgets_out) {
  kvc_status st = check_dims(dims);
  if (st != KVC_OK) return st;
  if (!budgets_out) return KVC_E_ARG;
  const int L = dims->n_layers, G = dims->group_size;
  const int ns = dims->prompt_len - dims->obs_window;
  std::vector<long long> units(L);
  if (schedule == KVC_SCHED_NONE) {
    for (int l = 0; l < L; ++l) budgets_out[l] = dims->prompt_len;
  } else {
    if (avg_budget <= 0 || avg_budget % G) return KVC_E_ARG;
    const long long xu = avg_budget / G;
    if (schedule == KVC_SCHED_UNIFORM) {
      for (int l = 0; l < L; ++l) units[l] = xu;
    } else if (schedule == KVC_SCHED_PYRAMID) {
      if (pyramid_depth < 1) return KVC_E_ARG;
      const long long top = xu / pyramid_depth, bottom = 2 * xu - top;
      if (L == 1) {
        units[0] = xu;
      } else {
        // r_l = (bottom*(L-1) - (bottom-top)*l) / (L-1): floor, then the leftover
        // units to the largest remainders (ties to the lower layer)
        const long long den = L - 1;
        std::vector<long long> rem(L);
        long long used = 0;
        for (int l = 0; l < L; ++l) {
          const long long num = bottom * den - (bottom - top) * l;
          units[l] = num / den;
          rem[l] = num % den;
          used += units[l];
        }
        long long left = (long long)L * xu - used;
        std::vector<int> order(L);
        for (int l = 0; l < L; ++l) order[l] = l;
        std::stable_sort(order.begin(), order.end(),
                         [&](int a, int b) { return rem[a] > rem[b]; });
        for (int i = 0; i < left && i < L; ++i) units[order[i]] += 1;
      }
    } else {
      return KVC_E_ARG;
    }
    for (int l = 0; l < L; ++l) budgets_out[l] = (int32_t)(units[l] * G);
  }
  for (int l = 0; l < L; ++l) budgets_out[l] = std::min<int32_t>(budgets_out[l], ns);
  return KVC_OK;
}

kvc_status kvc_plan_budgets_weighted(const kvc_dims* dims, int32_t avg_budget,
                                     const double* weights, int32_t* budgets_out) {
  kvc_status st = check_dims(dims);
  if (st != KVC_OK) return st;
  if (!weights || !budgets_out) return KVC_E_ARG;
  const int L = dims->n_layers, G = dims->group_size;
  if (avg_budget <= 0 || avg_budget % G) return KVC_E_ARG;
  double wmax = 0.0;
  for (int l = 0; l < L; ++l) {
    if (!std::isfinite(weights[l]) || !(weights[l] > 0.0)) return KVC_E_ARG;
    wmax = std::max(wmax, weights[l]);
  }
  // integer weights q_l = max(1, rint(w_l / max(w) * 2^30)), round half to even
  std::vector<long long> q(L);
  unsigned __int128 qsum = 0;
  for (int l = 0; l < L; ++l) {
    q[l] = std::max(1LL, (long long)std::nearbyint((weights[l] / wmax) * 1073741824.0));
    qsum += (unsigned __int128)q[l];
  }
  // one group per layer, the spare groups shared by largest remainder (ties to
  // the lower layer)
  const long long total = (long long)L * (avg_budget / G), spare = total - L;
  std::vector<long long> units(L);
  std::vector<unsigned __int128> rem(L);
  long long used = 0;
  for (int l = 0; l < L; ++l) {
    const unsigned __int128 num = (unsigned __int128)spare * (unsigned __int128)q[l];
    units[l] = 1 + (long long)(num / qsum);
    rem[l] = num % qsum;
    used += units[l];
  }
  std::vector<int> order(L);
  for (int l = 0; l < L; ++l) order[l] = l;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return rem[a] > rem[b]; });
  for (long long i = 0; i < total - used && i < L; ++i) units[order[i]] += 1;
  const int ns = dims->prompt_len - dims->obs_window;
  for (int l = 0; l < L; ++l)
    budgets_out[l] = (int32_t)std::min<long long>(units[l] * G, (long long)ns);
  return KVC_OK;
}

kvc_status kvc_cache_create(const kvc_dims* dims, const int32_t* budgets, kvc_cache** cache) {
  if (!cache) return KVC_E_ARG;
  *cache = nullptr;
  return create(dims, budgets, nullptr, cache);
}

kvc_status kvc_cache_create_layers(const kvc_dims* dims, const int32_t* budgets,
                                   const int32_t* layer_bits, kvc_cache** cache) {
  if (!cache || !layer_bits) return KVC_E_ARG;
  *cache = nullptr;
  return create(dims, budgets, layer_bits, cache);
}

kvc_status kvc_prefill_compress(const kvc_dims* dims, const int32_t* budgets, int32_t layer,
                                const void* q_obs, const void* k, const void* v,
                                kvc_cache** cache, void* stream) {
  if (!cache || !dims) return KVC_E_ARG;
  if (*cache == nullptr) {
    // the call's own arguments first: a call that fails creates nothing
    kvc_status st = check_dims(dims);
    if (st != KVC_OK) return st;
    if (!budgets || !k || !v || layer < 0 || layer >= dims->n_layers) return KVC_E_ARG;
    if (budgets[layer] >= 0 && budgets[layer] < dims->prompt_len - dims->obs_window && !q_obs)
      return KVC_E_ARG;
    st = create(dims, budgets, nullptr, cache);
    if (st != KVC_OK) return st;
  } else if (!same_dims((*cache)->dims, *dims)) {
    return KVC_E_SHAPE;
  }
  kvc_cache* c = *cache;
  if (layer < 0 || layer >= c->dims.n_layers) return KVC_E_ARG;
  if (!k || !v) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  LayerState& ls = c->L[layer];
  if (ls.prefilled) return KVC_E_STATE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int ns = c->dims.prompt_len - c->dims.obs_window;
  const int n_kept = ls.budget;
  const int32_t* kept = nullptr;
  if (n_kept < ns) {
    if (!q_obs) return KVC_E_ARG;
    int32_t* kp = ls.kept_ptr;
    cudaError_t e = kvc::launch_score(c, layer, static_cast<const __nv_bfloat16*>(q_obs),
                                      static_cast<const __nv_bfloat16*>(k), s);
    if (e == cudaSuccess) e = kvc::launch_pool_topk(c, layer, kp, n_kept, s);
    if (e != cudaSuccess) return from_cuda(e);
    kept = kp;
    ls.scored = 1;
    c->last_scored_layer = layer;
  } else {
    ls.scored = 0;
  }
  return finish_prefill(c, layer, n_kept, kept, k, v, s);
}

kvc_status kvc_prefill_acumul(kvc_cache* c, int32_t layer, const void* q_full, const void* k,
                              const void* v, void* stream) {
  if (!c || !k || !v) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  if (layer < 0 || layer >= c->dims.n_layers) return KVC_E_ARG;
  LayerState& ls = c->L[layer];
  if (ls.prefilled) return KVC_E_STATE;
  const int ns = c->dims.prompt_len - c->dims.obs_window;
  const int n_kept = ls.budget < ns ? ls.budget : ns;
  if (!window_fits(c->dims, ls.bits, ls.R, n_kept)) return KVC_E_SHAPE;
  const int g = c->dims.n_q_heads / c->dims.n_kv_heads;
  if (g > 16 || 128 % g != 0) return KVC_E_SHAPE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_kept >= ns) {                 // the budget keeps every token
    ls.scored = 0;
    return finish_prefill(c, layer, n_kept, nullptr, k, v, s);
  }
  if (!q_full) return KVC_E_ARG;
  int32_t* kp = ls.kept_ptr;
  if (!c->score_fx) {
    c->score_fx = static_cast<unsigned long long*>(dev_alloc(c, c->score_elems * 8));
    if (!c->score_fx) return KVC_E_OOM;
  }
  cudaError_t e = kvc::launch_acumul(c->dims, static_cast<const __nv_bfloat16*>(q_full),
                                     static_cast<const __nv_bfloat16*>(k), c->scores,
                                     c->score_fx, c->err, s);
  if (e == cudaSuccess) e = kvc::launch_pool_topk(c, layer, kp, n_kept, s);
  if (e != cudaSuccess) return from_cuda(e);
  ls.scored = 1;
  c->last_scored_layer = layer;
  return finish_prefill(c, layer, n_kept, kp, k, v, s);
}

kvc_status kvc_prefill_attention(kvc_cache* c, int32_t layer, const void* q_full, const void* k,
                                 const void* v, void* x_out, void* stream) {
  if (!c || !k || !v || !q_full || !x_out) return KVC_E_ARG;
  if (reinterpret_cast<uintptr_t>(x_out) % 16) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  if (layer < 0 || layer >= c->dims.n_layers) return KVC_E_ARG;
  LayerState& ls = c->L[layer];
  if (ls.prefilled) return KVC_E_STATE;
  const int ns = c->dims.prompt_len - c->dims.obs_window;
  const int n_kept = ls.budget < ns ? ls.budget : ns;
  if (!window_fits(c->dims, ls.bits, ls.R, n_kept)) return KVC_E_SHAPE;
  const int g = c->dims.n_q_heads / c->dims.n_kv_heads;
  if (g > 16 || 128 % g != 0) return KVC_E_SHAPE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool scoring = n_kept < ns;
  if (scoring && !c->score_fx) {
    c->score_fx = static_cast<unsigned long long*>(dev_alloc(c, c->score_elems * 8));
    if (!c->score_fx) return KVC_E_OOM;
  }
  cudaError_t e = kvc::launch_acumul_xo(c->dims, static_cast<const __nv_bfloat16*>(q_full),
                                        static_cast<const __nv_bfloat16*>(k),
                                        static_cast<const __nv_bfloat16*>(v),
                                        scoring ? c->scores : nullptr, c->score_fx,
                                        static_cast<__nv_bfloat16*>(x_out), c->err, s);
  if (e != cudaSuccess) return from_cuda(e);
  if (!scoring) {                     // the budget keeps every token
    ls.scored = 0;
    return finish_prefill(c, layer, n_kept, nullptr, k, v, s);
  }
  int32_t* kp = ls.kept_ptr;
  e = kvc::launch_pool_topk(c, layer, kp, n_kept, s);
  if (e != cudaSuccess) return from_cuda(e);
  ls.scored = 1;
  c->last_scored_layer = layer;
  return finish_prefill(c, layer, n_kept, kp, k, v, s);
}

kvc_status kvc_prefill_sinks(kvc_cache* c, int32_t layer, int32_t n_sinks, const void* k,
                             const void* v, void* stream) {
  if (!c || !k || !v || n_sinks < 0) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  if (layer < 0 || layer >= c->dims.n_layers) return KVC_E_ARG;
  LayerState& ls = c->L[layer];
  if (ls.prefilled) return KVC_E_STATE;
  const int ns = c->dims.prompt_len - c->dims.obs_window;
  const int n_kept = ls.budget < ns ? ls.budget : ns;
  if (!window_fits(c->dims, ls.bits, ls.R, n_kept)) return KVC_E_SHAPE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_kept >= ns) {                 // the budget keeps every token
    ls.scored = 0;
    return finish_prefill(c, layer, n_kept, nullptr, k, v, s);
  }
  if (!ls.kept_ptr) {
    const int units = c->dims.batch * c->dims.n_kv_heads;
    ls.kept_ptr = static_cast<int32_t*>(dev_alloc(c, (size_t)units * n_kept * 4));
    if (!ls.kept_ptr) return KVC_E_OOM;
  }
  ls.scored = 1;                      // the positions are stored for export
  return finish_prefill(c, layer, n_kept, nullptr, k, v, s, n_sinks < n_kept ? n_sinks : n_kept,
                        ls.kept_ptr);
}

kvc_status kvc_prefill_selected(kvc_cache* c, int32_t layer, const int32_t* kept, int32_t n_kept,
                                const void* k, const void* v, void* stream) {
  if (!c || !k || !v || (!kept && n_kept > 0)) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  if (layer < 0 || layer >= c->dims.n_layers) return KVC_E_ARG;
  LayerState& ls = c->L[layer];
  if (ls.prefilled) return KVC_E_STATE;
  const int ns = c->dims.prompt_len - c->dims.obs_window;
  if (n_kept < 0 || n_kept > ns) return KVC_E_ARG;
  if (n_kept > ls.budget) return KVC_E_CAPACITY;
  if (!window_fits(c->dims, ls.bits, ls.R, n_kept)) return KVC_E_SHAPE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int units = c->dims.batch * c->dims.n_kv_heads;
  ls.scored = 0;
  if (n_kept > 0) {
    // keep a copy of the selection (row stride n_kept) for export; a keep-all layer
    // has no stored selection from creation: it gets one sized for the largest
    // selection the layer allows (its budget, clipped to prompt_len - obs_window),
    // so that a later call (after kvc_cache_reset) with more kept positions fits
    if (!ls.kept_ptr) {
      ls.kept_ptr = static_cast<int32_t*>(dev_alloc(c, (size_t)units * ls.budget * 4));
      if (!ls.kept_ptr) return KVC_E_OOM;
    }
    cudaError_t e = cudaMemcpyAsync(ls.kept_ptr, kept, (size_t)units * n_kept * 4,
                                    cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return from_cuda(e);
    ls.scored = 1;
  }
  return finish_prefill(c, layer, n_kept, ls.kept_ptr, k, v, s);
}

kvc_status kvc_append_layers(kvc_cache* c, int32_t layer_begin, int32_t layer_count,
                             const void* k_new, const void* v_new, void* stream) {
  if (!c || !k_new || !v_new) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  if (layer_count < 1 || layer_begin < 0 || layer_begin + layer_count > c->dims.n_layers)
    return KVC_E_ARG;
  for (int l = layer_begin; l < layer_begin + layer_count; ++l) {
    if (!c->L[l].prefilled) return KVC_E_STATE;
    if (c->L[l].appended >= c->dims.max_new_tokens) return KVC_E_CAPACITY;
  }
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  std::vector<int> flush(layer_count);
  for (int i = 0; i < layer_count; ++i) {   // 16-bit storage never flushes
    const LayerState& ls = c->L[layer_begin + i];
    flush[i] = ls.bits != 16 && ls.win_len + 1 == ls.R;
  }
  cudaError_t e = kvc::launch_append(c, layer_begin, layer_count,
                                     static_cast<const __nv_bfloat16*>(k_new),
                                     static_cast<const __nv_bfloat16*>(v_new), flush.data(),
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  for (int i = 0; i < layer_count; ++i) {
    LayerState& ls = c->L[layer_begin + i];
    ls.win_len += 1;
    ls.appended += 1;
    if (flush[i]) {
      ls.n_groups += 1;
      ls.win_start = (ls.win_start + KVC_GROUP) % ls.R;
      ls.win_len -= KVC_GROUP;
    }
  }
  return KVC_OK;
}

kvc_status kvc_append(kvc_cache* c, int32_t layer, const void* k_new, const void* v_new,
                      void* stream) {
  return kvc_append_layers(c, layer, 1, k_new, v_new, stream);
}

kvc_status kvc_decode_attn(kvc_cache* c, int32_t layer_begin, int32_t layer_count, const void* q,
                           float* out, void* stream) {
  if (!c || !q || !out) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  // q is staged by bulk copies and out written in 16-byte vectors
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16) return KVC_E_ARG;
  if (layer_count < 1 || layer_begin < 0 || layer_begin + layer_count > c->dims.n_layers)
    return KVC_E_ARG;
  for (int l = layer_begin; l < layer_begin + layer_count; ++l)
    if (!c->L[l].prefilled) return KVC_E_STATE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  return from_cuda(kvc::launch_decode(c, layer_begin, layer_count,
                                      static_cast<const __nv_bfloat16*>(q), out,
                                      static_cast<cudaStream_t>(stream)));
}

kvc_status kvc_decode_step(kvc_cache* c, int32_t layer_begin, int32_t layer_count, const void* q,
                           const void* k_new, const void* v_new, float* out, void* stream) {
  if (!c || !q || !out || !k_new || !v_new) return KVC_E_ARG;
  if (kvc_status pe = pending_error(c)) return pe;
  // q is staged by bulk copies and out written in 16-byte vectors
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16) return KVC_E_ARG;
  if (layer_count < 1 || layer_begin < 0 || layer_begin + layer_count > c->dims.n_layers)
    return KVC_E_ARG;
  for (int l = layer_begin; l < layer_begin + layer_count; ++l) {
    if (!c->L[l].prefilled) return KVC_E_STATE;
    if (c->L[l].appended >= c->dims.max_new_tokens) return KVC_E_CAPACITY;
  }
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  std::vector<int> flush(layer_count);
  for (int i = 0; i < layer_count; ++i) {   // 16-bit storage never flushes
    const LayerState& ls = c->L[layer_begin + i];
    flush[i] = ls.bits != 16 && ls.win_len + 1 == ls.R;
  }
  // one launch: append (+ flush of the oldest group) and attention for every layer
  cudaError_t e = kvc::launch_decode_step(c, layer_begin, layer_count,
                                          static_cast<const __nv_bfloat16*>(q),
                                          static_cast<const __nv_bfloat16*>(k_new),
                                          static_cast<const __nv_bfloat16*>(v_new), flush.data(),
                                          out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e);
  for (int i = 0; i < layer_count; ++i) {
    LayerState& ls = c->L[layer_begin + i];
    ls.win_len += 1;
    ls.appended += 1;
    if (flush[i]) {
      ls.n_groups += 1;
      ls.win_start = (ls.win_start + KVC_GROUP) % ls.R;
      ls.win_len -= KVC_GROUP;
    }
  }
  return KVC_OK;
}

kvc_status kvc_check_device(kvc_cache* c, void* stream) {
  if (!c) return KVC_E_ARG;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_E_CUDA;
  if (c->err_host) {
    word = *c->err_host;
    *c->err_host = 0u;
    return word_status(word);
  }
  if (cudaMemcpy(&word, c->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KVC_E_CUDA;
  if (word == 0) return KVC_OK;
  if (cudaMemset(c->err, 0, sizeof(word)) != cudaSuccess) return KVC_E_CUDA;
  return word_status(word);
}

int32_t kvc_build_checked(void) { return kvc::kChecked ? 1 : 0; }

kvc_status kvc_set_wait_limit(kvc_cache* c, int64_t polls) {
  if (!c) return KVC_E_ARG;
  c->wait_limit_set = polls >= 0;
  c->wait_limit = polls >= 0 ? (unsigned)std::min<int64_t>(polls, 0xffffffffLL) : 0u;
  return KVC_OK;
}

kvc_status kvc_free(kvc_cache* c) {
  if (!c) return KVC_OK;
  DeviceGuard dg(c->device);
  release_all(c);
  delete c;
  return KVC_OK;
}

kvc_status kvc_layer_info_get(const kvc_cache* c, int32_t layer, kvc_layer_info* out) {
  if (!c || !out || layer < 0 || layer >= c->dims.n_layers) return KVC_E_ARG;
  const LayerState& ls = c->L[layer];
  out->prefilled = ls.prefilled;
  out->budget = ls.budget;
  out->n_kept = ls.n_kept;
  out->packed_tokens = ls.n_groups * KVC_GROUP;
  out->capacity_tokens = ls.cap_groups * KVC_GROUP;
  out->window_tokens = ls.win_len;
  out->appended = ls.appended;
  out->packed_bytes = (int64_t)c->dims.batch * c->dims.n_kv_heads * ls.cap_groups * ls.block_bytes;
  out->bits = ls.bits;
  out->window_capacity = ls.R;
  return KVC_OK;
}

kvc_status kvc_export_layer(kvc_cache* c, int32_t layer, const kvc_export* dst, void* stream) {
  if (!c || !dst || layer < 0 || layer >= c->dims.n_layers) return KVC_E_ARG;
  if (!c->L[layer].prefilled) return KVC_E_STATE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  return from_cuda(kvc::launch_export(c, layer, dst, static_cast<cudaStream_t>(stream)));
}

kvc_status kvc_score_variance(kvc_cache* c, float* var_out, void* stream) {
  if (!c || !var_out) return KVC_E_ARG;
  if (c->last_scored_layer < 0 || !c->scores) return KVC_E_STATE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  const kvc_dims& d = c->dims;
  // the slices' partials go to the scoring launch's statistics scratch and the units'
  // tickets to its arrival counters (both idle between launches; the tickets return
  // to zero)
  return from_cuda(kvc::launch_score_variance(
      c->scores, d.batch * d.n_kv_heads, d.prompt_len - d.obs_window, var_out,
      reinterpret_cast<double*>(c->stats), c->stats_elems, c->gsync + 1,
      static_cast<cudaStream_t>(stream)));
}

kvc_status kvc_scores_layer(kvc_cache* c, float* scores, float* pooled, void* stream) {
  if (!c) return KVC_E_ARG;
  if (c->last_scored_layer < 0 || !c->scores) return KVC_E_STATE;
  DeviceGuard dg(c->device);
  if (!dg.ok) return KVC_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = c->score_elems * 4;
  cudaError_t e = cudaSuccess;
  if (scores) e = cudaMemcpyAsync(scores, c->scores, bytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && pooled)
    e = cudaMemcpyAsync(pooled, c->pooled, bytes, cudaMemcpyDeviceToDevice, s);
  return from_cuda(e);
}

}  // extern "C"
