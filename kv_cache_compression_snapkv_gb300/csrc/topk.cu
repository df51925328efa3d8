// topk.cu -- max-pool the scores and keep the per-head top-k.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2: a pooling layer smooths the scores so massive activations do
// not mislead the selection; in each layer and head the top k^l tokens are kept
// and all others discarded for good.
//
// One CTA of 1024 threads per (sequence, kv head):
//   1. pooled[i] = max of scores[i - (w-1)/2 .. i + (w-1)/2] clipped to the range;
//   2. radix select of the k-th largest pooled value tau on its fp32 bit pattern
//      (scores are >= 0, so unsigned order == float order), four 8-bit passes;
//   3. ordered compaction: every index with pooled > tau, plus the lowest-index
//      entries equal to tau until k are kept, written in ascending index order.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kWarps = kTopkThreads / 32;

struct TopkSmem {
  unsigned hist[256];
  unsigned warp_a[kWarps];
  unsigned warp_b[kWarps];
  unsigned sel_bin;
  unsigned krem;
};

// Block-wide exclusive scan of two counters (all threads participate).
__device__ __forceinline__ void block_scan2(TopkSmem& s, unsigned a, unsigned b, unsigned& ea,
                                            unsigned& eb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned ta = __shfl_up_sync(0xffffffffu, ia, o);
    unsigned tb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) { ia += ta; ib += tb; }
  }
  if (lane == 31) { s.warp_a[warp] = ia; s.warp_b[warp] = ib; }
  __syncthreads();
  if (warp == 0) {
    unsigned wa = s.warp_a[lane], wb = s.warp_b[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned ta = __shfl_up_sync(0xffffffffu, wa, o);
      unsigned tb = __shfl_up_sync(0xffffffffu, wb, o);
      if (lane >= o) { wa += ta; wb += tb; }
    }
    s.warp_a[lane] = wa;  // inclusive over warps
    s.warp_b[lane] = wb;
  }
  __syncthreads();
  const unsigned pa = warp ? s.warp_a[warp - 1] : 0u;
  const unsigned pb = warp ? s.warp_b[warp - 1] : 0u;
  ea = pa + ia - a;
  eb = pb + ib - b;
}

__global__ void __launch_bounds__(kTopkThreads)
pool_topk_kernel(const float* __restrict__ scores, float* __restrict__ pooled, int ns, int w,
                 int k_sel, int32_t* __restrict__ kept) {
  __shared__ TopkSmem s;
  const int unit = blockIdx.x;
  const float* sc = scores + (size_t)unit * ns;
  float* pl = pooled + (size_t)unit * ns;
  int32_t* out = kept + (size_t)unit * k_sel;
  const int r = (w - 1) / 2;
  for (int i = threadIdx.x; i < ns; i += kTopkThreads) {
    float m = sc[i];
    const int lo = i - r < 0 ? 0 : i - r, hi = i + r >= ns ? ns - 1 : i + r;
    for (int t = lo; t <= hi; ++t) m = fmaxf(m, sc[t]);
    pl[i] = m;
  }
  if (k_sel >= ns) {
    for (int i = threadIdx.x; i < ns; i += kTopkThreads) out[i] = i;
    return;
  }
  __syncthreads();
  if (k_sel <= 0) return;

  unsigned prefix = 0, mask = 0;
  if (threadIdx.x == 0) { s.krem = (unsigned)k_sel; s.sel_bin = 0; }
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = threadIdx.x; b < 256; b += kTopkThreads) s.hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < ns; i += kTopkThreads) {
      const unsigned u = __float_as_uint(pl[i]);
      if ((u & mask) == prefix) atomicAdd(&s.hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns bins [8l, 8l + 8); suffix sums from the top bin down
      const int lane = threadIdx.x;
      unsigned own = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) own += s.hist[8 * lane + j];
      unsigned suf = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      const unsigned above = suf - own;   // elements in bins of higher lanes
      const unsigned krem = s.krem;
      if (suf >= krem && above < krem) {
        unsigned cum = above;
        for (int b = 8 * lane + 7; b >= 8 * lane; --b) {
          const unsigned h = s.hist[b];
          if (cum + h >= krem) { s.sel_bin = (unsigned)b; s.krem = krem - cum; break; }
          cum += h;
        }
      }
    }
    __syncthreads();
    prefix |= s.sel_bin << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  const unsigned tau = prefix;
  const unsigned need_eq = s.krem;

  // ordered compaction over contiguous per-thread segments
  const int seg = (ns + kTopkThreads - 1) / kTopkThreads;
  const int i0 = threadIdx.x * seg;
  const int i1 = i0 + seg < ns ? i0 + seg : ns;
  unsigned gt = 0, eq = 0;
  for (int i = i0; i < i1; ++i) {
    const unsigned u = __float_as_uint(pl[i]);
    gt += u > tau;
    eq += u == tau;
  }
  unsigned egt, eeq;
  block_scan2(s, gt, eq, egt, eeq);
  unsigned pos = egt + (eeq < need_eq ? eeq : need_eq);
  unsigned eq_seen = eeq;
  for (int i = i0; i < i1; ++i) {
    const unsigned u = __float_as_uint(pl[i]);
    bool take = u > tau;
    if (u == tau) take = eq_seen++ < need_eq;
    if (take) {
      if (pos < (unsigned)k_sel) out[pos] = i;   // bounded even if the select were wrong
      ++pos;
    }
  }
}

}  // namespace

cudaError_t launch_pool_topk(const kvc_cache* c, int layer, int32_t* kept_out, int k_sel,
                             cudaStream_t stream) {
  (void)layer;
  const kvc_dims& d = c->dims;
  const int units = d.batch * d.n_kv_heads;
  const int ns = d.prompt_len - d.obs_window;
  pool_topk_kernel<<<units, kTopkThreads, 0, stream>>>(c->scores, c->pooled, ns, d.pool_kernel,
                                                        k_sel, kept_out);
  count_launches(1);
  return cudaGetLastError();
}

// The same launch with the score and pooled buffers given explicitly (used by
// the allocation-free selection entry point).
cudaError_t launch_pool_topk_into(const kvc_dims& d, const float* scores, float* pooled,
                                  int32_t* kept_out, int k_sel, cudaStream_t stream) {
  const int units = d.batch * d.n_kv_heads;
  const int ns = d.prompt_len - d.obs_window;
  pool_topk_kernel<<<units, kTopkThreads, 0, stream>>>(scores, pooled, ns, d.pool_kernel, k_sel,
                                                        kept_out);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace kvc
