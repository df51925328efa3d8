// quant.cu -- group quantization into the packed store, the bf16 window, export.
//
// KIVI-style asymmetric groups (blog "Quantization: keep each token in fewer
// bits"; MiniKV §4.4): keys per channel over 32 consecutive stored tokens,
// values per token over 32 consecutive channels; zero-point = group min,
// scale = (max - min) / (2^b - 1); both stored as fp16 (round to nearest even).
// Codes use the stored fp16 values: code = rint((x - Z) / S) clamped to
// [0, 2^b - 1], evaluated with explicit IEEE round-to-nearest fp32 subtract and
// divide (no contraction, no reciprocal), round-half-to-even conversion;
// S == 0 gives code 0. MiniKV Algorithm 1 (decoding): new tokens go to a 16-bit
// buffer that is quantized as it fills; here the oldest 32 tokens are quantized
// as one group whenever the window reaches R tokens.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ void group_params(float lo, float hi, int bits, __half& S, __half& Z,
                                             float& Sf, float& Zf) {
  float rng = __fsub_rn(hi, lo);
  float s32 = __fdiv_rn(rng, (float)((1 << bits) - 1));
  S = __float2half_rn(s32);
  Z = __float2half_rn(lo);
  Sf = __half2float(S);
  Zf = __half2float(Z);
}

__device__ __forceinline__ int quant_code(float x, float Zf, float Sf, int bits) {
  if (Sf == 0.f) return 0;
  float q = __fdiv_rn(__fsub_rn(x, Zf), Sf);
  int c = __float2int_rn(q);
  int top = (1 << bits) - 1;
  return c < 0 ? 0 : (c > top ? top : c);
}

// Shared-memory staging of one group: 32 key rows and 32 value rows (fp32,
// natural channel order) plus their codes.
template <int D>
struct GroupSmem {
  float k[KVC_GROUP][D + 1];
  float v[KVC_GROUP][D + 1];
  uint8_t kc[KVC_GROUP][D];
  uint8_t vc[KVC_GROUP][D];
};

// Quantize the staged group and write one block. All kThreads threads call it.
template <int D, int BITS>
__device__ void quantize_block(GroupSmem<D>& s, uint8_t* __restrict__ blk) {
  __half* kS = reinterpret_cast<__half*>(blk + off_kscale(D, BITS));
  __half* kZ = reinterpret_cast<__half*>(blk + off_kzero(D, BITS));
  __half* vS = reinterpret_cast<__half*>(blk + off_vscale(D, BITS));
  __half* vZ = reinterpret_cast<__half*>(blk + off_vzero(D, BITS));
  // keys: one group per channel over the 32 tokens
  for (int c = threadIdx.x; c < D; c += kThreads) {
    float lo = s.k[0][c], hi = lo;
#pragma unroll 8
    for (int t = 1; t < KVC_GROUP; ++t) { lo = fminf(lo, s.k[t][c]); hi = fmaxf(hi, s.k[t][c]); }
    __half S, Z; float Sf, Zf;
    group_params(lo, hi, BITS, S, Z, Sf, Zf);
    for (int t = 0; t < KVC_GROUP; ++t) s.kc[t][c] = (uint8_t)quant_code(s.k[t][c], Zf, Sf, BITS);
    kS[kperm(c, D)] = S;
    kZ[kperm(c, D)] = Z;
  }
  // values: one group per (token, 32 channels)
  constexpr int NGC = D / KVC_GROUP;
  for (int i = threadIdx.x; i < KVC_GROUP * NGC; i += kThreads) {
    int t = i / NGC, gc = i % NGC;
    const float* row = &s.v[t][gc * KVC_GROUP];
    float lo = row[0], hi = lo;
#pragma unroll 8
    for (int j = 1; j < KVC_GROUP; ++j) { lo = fminf(lo, row[j]); hi = fmaxf(hi, row[j]); }
    __half S, Z; float Sf, Zf;
    group_params(lo, hi, BITS, S, Z, Sf, Zf);
    for (int j = 0; j < KVC_GROUP; ++j)
      s.vc[t][gc * KVC_GROUP + j] = (uint8_t)quant_code(row[j], Zf, Sf, BITS);
    vS[vsz_index(t, gc, NGC)] = S;
    vZ[vsz_index(t, gc, NGC)] = Z;
  }
  __syncthreads();
  // pack code words in fragment order
  constexpr int WPL = D * BITS / 32;
  constexpr int PPW = 16 / BITS;
  constexpr int NW = 32 * WPL;
  uint32_t* kw = reinterpret_cast<uint32_t*>(blk + off_kcodes(D, BITS));
  uint32_t* vw = reinterpret_cast<uint32_t*>(blk + off_vcodes(D, BITS));
  for (int widx = threadIdx.x; widx < 2 * NW; widx += kThreads) {
    bool is_v = widx >= NW;
    int w = is_v ? widx - NW : widx;
    int lane = (w & 127) >> 2;
    int wi = (w >> 7) * 4 + (w & 3);
    int gid = lane >> 2, tid = lane & 3;
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < PPW; ++p) {
      int pi = wi * PPW + p;
      int half = pi & 1, q = pi >> 1;
      uint32_t ce, co;
      if (!is_v) {
        int nt = q / (D / 16), ks = q % (D / 16);
        int t = nt * 8 + gid, c = 16 * ks + 2 * tid + 8 * half;
        ce = s.kc[t][c]; co = s.kc[t][c + 1];
      } else {
        int ks = q / (D / 8), nt = q % (D / 8);
        int t = 16 * ks + 2 * tid + 8 * half, c = 8 * nt + gid;
        ce = s.vc[t][c]; co = s.vc[t + 1][c];
      }
      word |= ce << (BITS * p);
      word |= co << (16 + BITS * p);
    }
    (is_v ? vw : kw)[w] = word;
  }
}

__device__ __forceinline__ void load_row_bf16_to_smem(float* dst, const __nv_bfloat16* src, int D,
                                                      int lane16, int n16) {
  // one thread copies 8 channels (16 bytes)
  (void)n16;
  uint4 u = *reinterpret_cast<const uint4*>(src + lane16 * 8);
  const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
  for (int j = 0; j < 8; ++j) dst[lane16 * 8 + j] = __bfloat162float(h[j]);
  (void)D;
}

// --------------------------------------------------------------------- kernels
// grid.x = group index j within the unit, grid.y = unit (b * H + h)
template <int D, int BITS>
__global__ void __launch_bounds__(kThreads)
gather_quant_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                    const int32_t* __restrict__ kept, int n_kept, int n, uint8_t* __restrict__ packed,
                    int cap_groups, int block_bytes) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  GroupSmem<D>& s = *reinterpret_cast<GroupSmem<D>*>(smem_raw);
  const int j = blockIdx.x, unit = blockIdx.y;
  const __nv_bfloat16* K = k + (size_t)unit * n * D;
  const __nv_bfloat16* V = v + (size_t)unit * n * D;
  const int32_t* kp = kept ? kept + (size_t)unit * n_kept : nullptr;
  constexpr int CH = D / 8;   // 16-byte chunks per row
  for (int i = threadIdx.x; i < KVC_GROUP * CH; i += kThreads) {
    int t = i / CH, ch = i % CH;
    int idx = kp ? kp[j * KVC_GROUP + t] : j * KVC_GROUP + t;
    load_row_bf16_to_smem(s.k[t], K + (size_t)idx * D, D, ch, CH);
    load_row_bf16_to_smem(s.v[t], V + (size_t)idx * D, D, ch, CH);
  }
  __syncthreads();
  uint8_t* blk = packed + ((size_t)unit * cap_groups + j) * block_bytes;
  quantize_block<D, BITS>(s, blk);
}

// Window rows: keys permuted by kperm, values in token pairs permuted by vperm.
__device__ __forceinline__ void window_store(__nv_bfloat16* __restrict__ wk,
                                             __nv_bfloat16* __restrict__ wv, int slot, int c, int D,
                                             __nv_bfloat16 kval, __nv_bfloat16 vval) {
  wk[(size_t)slot * D + kperm(c, D)] = kval;
  wv[((size_t)(slot >> 1) * D + vperm(c, D)) * 2 + (slot & 1)] = vval;
}

__device__ __forceinline__ __nv_bfloat16 window_load_k(const __nv_bfloat16* wk, int slot, int c,
                                                       int D) {
  return wk[(size_t)slot * D + kperm(c, D)];
}
__device__ __forceinline__ __nv_bfloat16 window_load_v(const __nv_bfloat16* wv, int slot, int c,
                                                       int D) {
  return wv[((size_t)(slot >> 1) * D + vperm(c, D)) * 2 + (slot & 1)];
}

// grid.x = unit; copies the initial window (kept tail, then observation tokens)
__global__ void __launch_bounds__(kThreads)
window_init_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                   const int32_t* __restrict__ kept, int n_kept, int n_full, int n, int alpha,
                   int D, int R, __nv_bfloat16* __restrict__ win_k,
                   __nv_bfloat16* __restrict__ win_v) {
  const int unit = blockIdx.x;
  const int tail = n_kept - n_full;
  const int W = tail + alpha;
  const __nv_bfloat16* K = k + (size_t)unit * n * D;
  const __nv_bfloat16* V = v + (size_t)unit * n * D;
  __nv_bfloat16* wk = win_k + (size_t)unit * R * D;
  __nv_bfloat16* wv = win_v + (size_t)unit * R * D;
  const int32_t* kp = kept ? kept + (size_t)unit * n_kept : nullptr;
  for (int i = threadIdx.x; i < W * D; i += kThreads) {
    int w = i / D, c = i % D;
    int idx = w < tail ? (kp ? kp[n_full + w] : n_full + w) : n - alpha + (w - tail);
    window_store(wk, wv, w, c, D, K[(size_t)idx * D + c], V[(size_t)idx * D + c]);
  }
}

struct AppendParams {
  int slot[KVC_MAX_LAUNCH_LAYERS];        // ring slot of the new token
  int flush_start[KVC_MAX_LAUNCH_LAYERS]; // -1: no flush; else ring slot of the oldest token
  int flush_group[KVC_MAX_LAUNCH_LAYERS]; // packed group index to write
  long long packed_off[KVC_MAX_LAUNCH_LAYERS];
  int cap_groups[KVC_MAX_LAUNCH_LAYERS];
};

// grid.x = layer_rel * units + unit
template <int D, int BITS>
__global__ void __launch_bounds__(kThreads)
append_kernel(AppendParams P, int layer_begin, int units, int R, const __nv_bfloat16* __restrict__ k_new,
              const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* __restrict__ win_k,
              __nv_bfloat16* __restrict__ win_v, uint8_t* __restrict__ packed, int block_bytes) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int lrel = blockIdx.x / units, unit = blockIdx.x % units;
  const size_t wunit = (size_t)(layer_begin + lrel) * units + unit;
  __nv_bfloat16* wk = win_k + wunit * R * D;
  __nv_bfloat16* wv = win_v + wunit * R * D;
  const __nv_bfloat16* kn = k_new + ((size_t)lrel * units + unit) * D;
  const __nv_bfloat16* vn = v_new + ((size_t)lrel * units + unit) * D;
  const int slot = P.slot[lrel];
  for (int c = threadIdx.x; c < D; c += kThreads) window_store(wk, wv, slot, c, D, kn[c], vn[c]);
  const int fs = P.flush_start[lrel];
  if (fs < 0) return;
  __syncthreads();   // the new token may belong to the flushed group (R == 32)
  GroupSmem<D>& s = *reinterpret_cast<GroupSmem<D>*>(smem_raw);
  for (int i = threadIdx.x; i < KVC_GROUP * D; i += kThreads) {
    int t = i / D, c = i % D;
    int sl = fs + t;
    s.k[t][c] = __bfloat162float(window_load_k(wk, sl, c, D));
    s.v[t][c] = __bfloat162float(window_load_v(wv, sl, c, D));
  }
  __syncthreads();
  uint8_t* blk = packed + P.packed_off[lrel] +
                 ((size_t)unit * P.cap_groups[lrel] + P.flush_group[lrel]) * block_bytes;
  quantize_block<D, BITS>(s, blk);
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
      int w = i / D, c = i % D;
      int slot = (win_start + w) % R;
      size_t o = ((size_t)unit * win_len + w) * D + c;
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
    int t = i / D, c = i % D;
    size_t o = ((size_t)unit * T + (size_t)j * KVC_GROUP + t) * D + c;
    CodePos pk = kcode_pos(t, c, D, BITS);
    CodePos pv = vcode_pos(t, c, D, BITS);
    if (dst.k_codes) dst.k_codes[o] = (uint8_t)((kw[pk.word] >> pk.bit) & mask);
    if (dst.v_codes) dst.v_codes[o] = (uint8_t)((vw[pv.word] >> pv.bit) & mask);
  }
  constexpr int NGC = D / KVC_GROUP;
  for (int c = threadIdx.x; c < D; c += kThreads) {
    size_t o = ((size_t)unit * n_groups + j) * D + c;
    if (dst.k_scale) reinterpret_cast<__half*>(dst.k_scale)[o] = kS[kperm(c, D)];
    if (dst.k_zero) reinterpret_cast<__half*>(dst.k_zero)[o] = kZ[kperm(c, D)];
  }
  for (int i = threadIdx.x; i < KVC_GROUP * NGC; i += kThreads) {
    const int t = i / NGC, gc = i % NGC;
    size_t o = ((size_t)unit * T + (size_t)j * KVC_GROUP) * NGC + i;
    if (dst.v_scale) reinterpret_cast<__half*>(dst.v_scale)[o] = vS[vsz_index(t, gc, NGC)];
    if (dst.v_zero) reinterpret_cast<__half*>(dst.v_zero)[o] = vZ[vsz_index(t, gc, NGC)];
  }
}

__global__ void export_kept_kernel(const int32_t* __restrict__ kept, int n_kept, int units,
                                   int32_t* __restrict__ out) {
  size_t total = (size_t)units * n_kept;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = kept ? kept[i] : (int32_t)(i % n_kept);
}

template <int D>
constexpr size_t group_smem() { return sizeof(GroupSmem<D>); }

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

template <typename K>
static cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_gather_quant(const kvc_cache* c, int layer, const int32_t* kept, int n_kept,
                                const __nv_bfloat16* k, const __nv_bfloat16* v,
                                cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  const LayerState& ls = c->L[layer];
  int groups = n_kept / KVC_GROUP;
  int units = d.batch * d.n_kv_heads;
  if (groups == 0) return cudaSuccess;
  KVC_DISPATCH_DB(d.head_dim, d.bits, {
    size_t sm = group_smem<D>();
    cudaError_t e = set_smem(gather_quant_kernel<D, BITS>, sm);
    if (e != cudaSuccess) return e;
    gather_quant_kernel<D, BITS><<<dim3(groups, units), kThreads, sm, stream>>>(
        k, v, kept, n_kept, d.prompt_len, c->packed + ls.packed_off, ls.cap_groups,
        c->block_bytes);
  });
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_window_init(const kvc_cache* c, int layer, const int32_t* kept, int n_kept,
                               const __nv_bfloat16* k, const __nv_bfloat16* v,
                               cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  int units = d.batch * d.n_kv_heads;
  int n_full = (n_kept / KVC_GROUP) * KVC_GROUP;
  size_t off = (size_t)layer * units * d.window_len * d.head_dim;
  window_init_kernel<<<units, kThreads, 0, stream>>>(k, v, kept, n_kept, n_full, d.prompt_len,
                                                      d.obs_window, d.head_dim, d.window_len,
                                                      c->win_k + off, c->win_v + off);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_append(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* k_new, const __nv_bfloat16* v_new,
                          const int* flush_flags, cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  int units = d.batch * d.n_kv_heads;
  for (int base = 0; base < layer_count; base += KVC_MAX_LAUNCH_LAYERS) {
    int cnt = layer_count - base < KVC_MAX_LAUNCH_LAYERS ? layer_count - base
                                                         : KVC_MAX_LAUNCH_LAYERS;
    AppendParams P;
    for (int i = 0; i < cnt; ++i) {
      const LayerState& ls = c->L[layer_begin + base + i];
      P.slot[i] = (ls.win_start + ls.win_len) % d.window_len;
      P.flush_start[i] = flush_flags[base + i] ? ls.win_start : -1;
      P.flush_group[i] = ls.n_groups;
      P.packed_off[i] = (long long)ls.packed_off;
      P.cap_groups[i] = ls.cap_groups;
    }
    const __nv_bfloat16* kn = k_new + (size_t)base * units * d.head_dim;
    const __nv_bfloat16* vn = v_new + (size_t)base * units * d.head_dim;
    KVC_DISPATCH_DB(d.head_dim, d.bits, {
      size_t sm = group_smem<D>();
      cudaError_t e = set_smem(append_kernel<D, BITS>, sm);
      if (e != cudaSuccess) return e;
      append_kernel<D, BITS><<<cnt * units, kThreads, sm, stream>>>(
          P, layer_begin + base, units, d.window_len, kn, vn, c->win_k, c->win_v, c->packed,
          c->block_bytes);
    });
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_export(const kvc_cache* c, int layer, const kvc_export* dst,
                          cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  const LayerState& ls = c->L[layer];
  int units = d.batch * d.n_kv_heads;
  size_t woff = (size_t)layer * units * d.window_len * d.head_dim;
  KVC_DISPATCH_DB(d.head_dim, d.bits, {
    export_kernel<D, BITS><<<dim3(ls.n_groups + 1, units), kThreads, 0, stream>>>(
        c->packed + ls.packed_off, ls.cap_groups, ls.n_groups, c->block_bytes, c->win_k + woff,
        c->win_v + woff, d.window_len, ls.win_start, ls.win_len, *dst);
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
