// quant.cu -- group quantization into the packed store, the bf16 window, export.
//
// KIVI-style asymmetric groups (blog "Quantization: keep each token in fewer
// bits"; MiniKV §4.4): keys per channel over 32 consecutive stored tokens,
// values per token over 32 consecutive channels; zero-point = group min,
// scale = (max - min) / (2^b - 1); both stored as fp16 (round to nearest even).
// Codes use the stored fp16 values: code = rint((x - Z) / S) clamped to
// [0, 2^b - 1], the IEEE round-to-nearest fp32 subtract and divide (no
// contraction) and round-half-to-even conversion; S == 0 gives code 0 (the divide
// is taken through the reciprocal wherever that gives the same code). MiniKV Algorithm 1 (decoding): new tokens go to a 16-bit
// buffer that is quantized as it fills; here the oldest 32 tokens are quantized
// as one group whenever the window reaches R tokens.
#include "quant_device.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               :: "r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_one() {   // all but the latest group complete
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// --------------------------------------------------------------------- kernels
// Persistent: CTA b takes the contiguous range [G b / grid, G (b + 1) / grid) of
// the G = units * n_pack packed groups (unit-major; n_pack is the number of whole
// groups of kept tokens per unit, 0 with 16-bit storage where every kept token
// starts in the window), its rows staged by cp.async two groups ahead of the group
// being quantized (three stages), then, grid-strided, the units' initial windows (32
// rows per item). Kept position p of the unit is kept[p] when `kept` is given;
// else, with sinks >= 0, the sink + recent-window position (p < sinks: p; else n -
// alpha - (n_kept - sinks) + (p - sinks)), also stored to kept_out; else p.
template <int D, int BITS>
__global__ void __launch_bounds__(kThreads, 4)
gather_quant_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                    const int32_t* __restrict__ kept, int n_kept, int n, int alpha,
                    uint8_t* __restrict__ packed, int cap_groups, int block_bytes, int R,
                    __nv_bfloat16* __restrict__ win_k, __nv_bfloat16* __restrict__ win_v,
                    int sinks, int32_t* __restrict__ kept_out, int n_pack, int units,
                    int win_items, unsigned* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupStage<D>* stage = reinterpret_cast<GroupStage<D>*>(smem_raw);
  QuantScratch<D>& qs = *reinterpret_cast<QuantScratch<D>*>(smem_raw + 3 * sizeof(GroupStage<D>));
  pdl_wait();      // the selection is complete
  pdl_release();
  const int recent0 = n - alpha - (n_kept - sinks);
  auto index_of = [&](int unit, int p) -> int {
    if (kept) {
      int idx = __ldg(kept + (size_t)unit * n_kept + p);
      if (kChecked && (idx < 0 || idx >= n - alpha)) {   // outside the scored range
        if (err) atomicOr(err, kErrDeviceCheck);
        idx = 0;
      }
      return idx;
    }
    if (sinks >= 0) return p < sinks ? p : recent0 + (p - sinks);
    return p;
  };
  constexpr int CH = D / 8;                      // 16-byte chunks per row
  constexpr int TPR = kThreads / KVC_GROUP;      // threads per staged row
  static_assert(CH % TPR == 0, "row chunks");
  const int row = threadIdx.x / TPR, c0 = threadIdx.x % TPR;
  const int G = units * n_pack;
  const int g0 = (int)((long long)G * blockIdx.x / gridDim.x);
  const int g1 = (int)((long long)G * (blockIdx.x + 1) / gridDim.x);
  // cursors (unit, group) of the group being quantized and of the next one to stage
  int cu = 0, cj = 0;
  if (g0 < g1) { cu = g0 / n_pack; cj = g0 - cu * n_pack; }
  int nu = cu, nj = cj;
  auto advance = [&](int& u, int& j) { if (++j == n_pack) { j = 0; ++u; } };
  auto issue = [&](GroupStage<D>& st, int u, int j, int idx) {
    const __nv_bfloat16* ks = k + ((size_t)u * n + idx) * D;
    const __nv_bfloat16* vs = v + ((size_t)u * n + idx) * D;
#pragma unroll
    for (int ch = c0; ch < CH; ch += TPR) {
      cp_async16(&st.k[row][ch * 8], ks + ch * 8);
      cp_async16(&st.v[row][ch * 8], vs + ch * 8);
    }
    if (kept_out && c0 == 0) kept_out[(size_t)u * n_kept + j * KVC_GROUP + row] = idx;
  };
  // three stages: groups g + 1 and g + 2 are in flight while g is quantized
  int sidx = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (g0 + i < g1) {
      issue(stage[i], nu, nj, index_of(nu, nj * KVC_GROUP + row));
      advance(nu, nj);
    }
    cp_async_commit();
  }
  if (g0 + 2 < g1) sidx = index_of(nu, nj * KVC_GROUP + row);
  int st = 0;
  for (int g = g0; g < g1; ++g) {
    cp_async_wait_one();
    __syncthreads();   // stage st is complete; every thread is done with the group before
    const int s2 = st == 0 ? 2 : st - 1;   // (st + 2) % 3: the stage read one group ago
    if (g + 2 < g1) {
      issue(stage[s2], nu, nj, sidx);
      advance(nu, nj);
      if (g + 3 < g1) sidx = index_of(nu, nj * KVC_GROUP + row);
    }
    cp_async_commit();
    uint8_t* blk = packed + ((size_t)cu * cap_groups + cj) * block_bytes;
    quantize_block<D, BITS>(stage[st], qs, blk);
    advance(cu, cj);
    st = st == 2 ? 0 : st + 1;
  }
  cp_async_wait_all();
  if (win_items == 0) return;
  // initial windows: the kept tokens past the last whole group, then the alpha
  // observation tokens, in ring slots 0 .. W-1 (item = (unit, 32-row slice))
  const int n_full = n_pack * KVC_GROUP, tail = n_kept - n_full, W = tail + alpha;
  const int per_unit = win_items / units;
  for (int it = blockIdx.x; it < win_items; it += gridDim.x) {
    const int unit = it / per_unit, wj = it - unit * per_unit;
    const int w0 = wj * KVC_GROUP, w1 = min(W, w0 + KVC_GROUP);
    const __nv_bfloat16* K = k + (size_t)unit * n * D;
    const __nv_bfloat16* V = v + (size_t)unit * n * D;
    int32_t* ko = kept_out ? kept_out + (size_t)unit * n_kept : nullptr;
    __nv_bfloat16* wk = win_k + (size_t)unit * R * D;
    __nv_bfloat16* wv = win_v + (size_t)unit * R * D;
    for (int i = w0 * D + threadIdx.x; i < w1 * D; i += kThreads) {
      const int w = i / D, c = i % D;
      const int idx = w < tail ? index_of(unit, n_full + w) : n - alpha + (w - tail);
      if (ko && c == 0 && w < tail) ko[n_full + w] = idx;
      window_store(wk, wv, w, c, D, K[(size_t)idx * D + c], V[(size_t)idx * D + c]);
    }
  }
}

struct AppendParams {
  int slot[KVC_MAX_LAUNCH_LAYERS];        // ring slot of the new token
  int flush_start[KVC_MAX_LAUNCH_LAYERS]; // -1: no flush; else ring slot of the oldest token
  int flush_group[KVC_MAX_LAUNCH_LAYERS]; // packed group index to write
  long long packed_off[KVC_MAX_LAUNCH_LAYERS];
  long long win_off[KVC_MAX_LAUNCH_LAYERS];  // element offset of the layer's rings
  int cap_groups[KVC_MAX_LAUNCH_LAYERS];
  int R[KVC_MAX_LAUNCH_LAYERS];           // ring length
  int bits[KVC_MAX_LAUNCH_LAYERS];        // 2, 4 or 16 (16 never flushes)
};

// grid.x = layer_rel * units + unit
template <int D>
__global__ void __launch_bounds__(kThreads)
append_kernel(AppendParams P, int units, const __nv_bfloat16* __restrict__ k_new,
              const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* __restrict__ win_k,
              __nv_bfloat16* __restrict__ win_v, uint8_t* __restrict__ packed) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  pdl_wait();      // the previous step's reads of the window are complete
  pdl_release();
  const int lrel = blockIdx.x / units, unit = blockIdx.x % units;
  const int R = P.R[lrel];
  __nv_bfloat16* wk = win_k + P.win_off[lrel] + (size_t)unit * R * D;
  __nv_bfloat16* wv = win_v + P.win_off[lrel] + (size_t)unit * R * D;
  const __nv_bfloat16* kn = k_new + ((size_t)lrel * units + unit) * D;
  const __nv_bfloat16* vn = v_new + ((size_t)lrel * units + unit) * D;
  const int slot = P.slot[lrel];
  for (int c = threadIdx.x; c < D; c += kThreads) window_store(wk, wv, slot, c, D, kn[c], vn[c]);
  const int fs = P.flush_start[lrel];
  if (fs < 0) return;
  __syncthreads();   // the new token may belong to the flushed group (R == 32)
  GroupStage<D>& s = *reinterpret_cast<GroupStage<D>*>(smem_raw);
  QuantScratch<D>& qs = *reinterpret_cast<QuantScratch<D>*>(smem_raw + sizeof(GroupStage<D>));
  for (int i = threadIdx.x; i < KVC_GROUP * D; i += kThreads) {
    const int t = i / D, c = i % D;
    const int sl = fs + t;
    s.k[t][c] = window_load_k(wk, sl, c, D);
    s.v[t][c] = window_load_v(wv, sl, c, D);
  }
  __syncthreads();
  const int bits = P.bits[lrel];
  uint8_t* blk = packed + P.packed_off[lrel] +
                 ((size_t)unit * P.cap_groups[lrel] + P.flush_group[lrel]) * block_bytes(D, bits);
  if (bits == 2) quantize_block<D, 2>(s, qs, blk);
  else quantize_block<D, 4>(s, qs, blk);
}

// Export: grid.x = group j (or window when j == n_groups), grid.y = unit
template <int D, int BITS>
__global__ void __launch_bounds__(kThreads)
export_kernel(const uint8_t* __restrict__ packed, int cap_groups, int n_groups, int block_bytes,
              const __nv_bfloat16* __restrict__ win_k, const __nv_bfloat16* __restrict__ win_v,
              int R, int win_start, int win_len, kvc_export dst) {
  const int j = blockIdx.x, unit = blockIdx.y;
  if (j == n_groups) {
    const __nv_bfloat16* wk = win_k + (size_t)unit * R * D;
    const __nv_bfloat16* wv = win_v + (size_t)unit * R * D;
    __nv_bfloat16* ok = reinterpret_cast<__nv_bfloat16*>(dst.win_k);
    __nv_bfloat16* ov = reinterpret_cast<__nv_bfloat16*>(dst.win_v);
    for (int i = threadIdx.x; i < win_len * D; i += kThreads) {
      const int w = i / D, c = i % D;
      const int slot = (win_start + w) % R;
      const size_t o = ((size_t)unit * win_len + w) * D + c;
      if (ok) ok[o] = window_load_k(wk, slot, c, D);
      if (ov) ov[o] = window_load_v(wv, slot, c, D);
    }
    return;
  }
  const uint8_t* blk = packed + ((size_t)unit * cap_groups + j) * block_bytes;
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(blk + off_kcodes(D, BITS));
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(blk + off_vcodes(D, BITS));
  const __half* kS = reinterpret_cast<const __half*>(blk + off_kscale(D, BITS));
  const __half* kZ = reinterpret_cast<const __half*>(blk + off_kzero(D, BITS));
  const __half* vS = reinterpret_cast<const __half*>(blk + off_vscale(D, BITS));
  const __half* vZ = reinterpret_cast<const __half*>(blk + off_vzero(D, BITS));
  const int T = n_groups * KVC_GROUP;
  const uint32_t mask = (1u << BITS) - 1;
  for (int i = threadIdx.x; i < KVC_GROUP * D; i += kThreads) {
    const int t = i / D, c = i % D;
    const size_t o = ((size_t)unit * T + (size_t)j * KVC_GROUP + t) * D + c;
    const CodePos pk = kcode_pos(t, c, D, BITS);
    const CodePos pv = vcode_pos(t, c, D, BITS);
    if (dst.k_codes) dst.k_codes[o] = (uint8_t)((kw[pk.word] >> pk.bit) & mask);
    if (dst.v_codes) dst.v_codes[o] = (uint8_t)((vw[pv.word] >> pv.bit) & mask);
  }
  constexpr int NGC = D / KVC_GROUP;
  for (int c = threadIdx.x; c < D; c += kThreads) {
    const size_t o = ((size_t)unit * n_groups + j) * D + c;
    if (dst.k_scale) reinterpret_cast<__half*>(dst.k_scale)[o] = kS[kperm(c, D)];
    if (dst.k_zero) reinterpret_cast<__half*>(dst.k_zero)[o] = kZ[kperm(c, D)];
  }
  for (int i = threadIdx.x; i < KVC_GROUP * NGC; i += kThreads) {
    const int t = i / NGC, gc = i % NGC;
    const size_t o = ((size_t)unit * T + (size_t)j * KVC_GROUP) * NGC + i;
    if (dst.v_scale) reinterpret_cast<__half*>(dst.v_scale)[o] = vS[vs_index(t, gc, NGC)];
    if (dst.v_zero) reinterpret_cast<__half*>(dst.v_zero)[o] = vZ[vsz_index(t, gc, NGC)];
  }
}

__global__ void export_kept_kernel(const int32_t* __restrict__ kept, int n_kept, int units,
                                   int32_t* __restrict__ out) {
  const size_t total = (size_t)units * n_kept;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = kept ? kept[i] : (int32_t)(i % n_kept);
}

template <int D>
constexpr size_t group_smem() { return sizeof(GroupStage<D>) + sizeof(QuantScratch<D>); }
template <int D>
constexpr size_t gather_smem() { return 3 * sizeof(GroupStage<D>) + sizeof(QuantScratch<D>); }

}  // namespace

// ------------------------------------------------------------------ host side
#define KVC_DISPATCH_DB(D_, BITS_, ...)                                           \
  do {                                                                            \
    if ((D_) == 128 && (BITS_) == 2) { constexpr int D = 128, BITS = 2; __VA_ARGS__; } \
    else if ((D_) == 128 && (BITS_) == 4) { constexpr int D = 128, BITS = 4; __VA_ARGS__; } \
    else if ((D_) == 64 && (BITS_) == 2) { constexpr int D = 64, BITS = 2; __VA_ARGS__; } \
    else if ((D_) == 64 && (BITS_) == 4) { constexpr int D = 64, BITS = 4; __VA_ARGS__; } \
    else return cudaErrorInvalidValue;                                            \
  } while (0)

template <typename Kern>
static cudaError_t set_smem(Kern kernel, size_t bytes) {
  return ensure_smem(reinterpret_cast<const void*>(kernel), bytes);
}

// Packs the kept tokens' whole groups and writes the initial window (one launch).
cudaError_t launch_gather_quant(const kvc_cache* c, int layer, const int32_t* kept, int n_kept,
                                const __nv_bfloat16* k, const __nv_bfloat16* v,
                                cudaStream_t stream, int sinks, int32_t* kept_out) {
  const kvc_dims& d = c->dims;
  const LayerState& ls = c->L[layer];
  const bool exact = ls.bits == 16;   // 16-bit storage: no packed groups, all in the window
  const int groups = exact ? 0 : n_kept / KVC_GROUP;
  const int win_rows = n_kept - groups * KVC_GROUP + d.obs_window;
  const int win_ctas = (win_rows + KVC_GROUP - 1) / KVC_GROUP;
  const int units = d.batch * d.n_kv_heads;
  const size_t woff = ls.win_off;
  if ((long long)units * groups >= (1ll << 31)) return cudaErrorInvalidValue;
  const int win_items = units * win_ctas;
  KVC_DISPATCH_DB(d.head_dim, exact ? 2 : ls.bits, {
    const size_t sm = gather_smem<D>();
    cudaError_t e = set_smem(gather_quant_kernel<D, BITS>, sm);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_quant_kernel<D, BITS>,
                                                      kThreads, sm);
    if (e != cudaSuccess) return e;
    const long long want = (long long)units * groups > win_items ? (long long)units * groups
                                                                 : win_items;
    long long grid = (long long)c->n_sm * (per_sm > 0 ? per_sm : 1);
    if (grid > want) grid = want;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = stream;
    cudaLaunchAttribute at[1] = {pdl_attr()};
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gather_quant_kernel<D, BITS>, k, v, kept, n_kept, d.prompt_len,
                           d.obs_window, c->packed + ls.packed_off, ls.cap_groups,
                           ls.block_bytes, ls.R, c->win_k + woff, c->win_v + woff,
                           sinks, kept_out, groups, units, win_items, c->err);
    if (e != cudaSuccess) return e;
  });
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_append(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* k_new, const __nv_bfloat16* v_new,
                          const int* flush_flags, cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  const int units = d.batch * d.n_kv_heads;
  for (int base = 0; base < layer_count; base += KVC_MAX_LAUNCH_LAYERS) {
    const int cnt = layer_count - base < KVC_MAX_LAUNCH_LAYERS ? layer_count - base
                                                               : KVC_MAX_LAUNCH_LAYERS;
    AppendParams P;
    for (int i = 0; i < cnt; ++i) {
      const LayerState& ls = c->L[layer_begin + base + i];
      P.slot[i] = (ls.win_start + ls.win_len) % ls.R;
      P.flush_start[i] = flush_flags[base + i] ? ls.win_start : -1;
      P.flush_group[i] = ls.n_groups;
      P.packed_off[i] = (long long)ls.packed_off;
      P.win_off[i] = (long long)ls.win_off;
      P.cap_groups[i] = ls.cap_groups;
      P.R[i] = ls.R;
      P.bits[i] = ls.bits;
    }
    const __nv_bfloat16* kn = k_new + (size_t)base * units * d.head_dim;
    const __nv_bfloat16* vn = v_new + (size_t)base * units * d.head_dim;
    KVC_DISPATCH_DB(d.head_dim, 2, {
      const size_t sm = group_smem<D>();
      cudaError_t e = set_smem(append_kernel<D>, sm);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cnt * units);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = sm;
      cfg.stream = stream;
      cudaLaunchAttribute at[1] = {pdl_attr()};
      cfg.attrs = at;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, append_kernel<D>, P, units, kn, vn, c->win_k, c->win_v,
                             c->packed);
      if (e != cudaSuccess) return e;
    });
    count_launches(1);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_export(const kvc_cache* c, int layer, const kvc_export* dst,
                          cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  const LayerState& ls = c->L[layer];
  const int units = d.batch * d.n_kv_heads;
  const size_t woff = ls.win_off;
  KVC_DISPATCH_DB(d.head_dim, ls.bits == 16 ? 2 : ls.bits, {   // 16-bit: window only
    export_kernel<D, BITS><<<dim3(ls.n_groups + 1, units), kThreads, 0, stream>>>(
        c->packed + ls.packed_off, ls.cap_groups, ls.n_groups, ls.block_bytes, c->win_k + woff,
        c->win_v + woff, ls.R, ls.win_start, ls.win_len, *dst);
  });
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dst->kept && ls.n_kept > 0) {
    const int32_t* kp = ls.scored ? ls.kept_ptr : nullptr;
    export_kept_kernel<<<256, 256, 0, stream>>>(kp, ls.n_kept, units, dst->kept);
    count_launches(1);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace kvc
