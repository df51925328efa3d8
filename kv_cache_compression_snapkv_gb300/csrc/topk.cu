// topk.cu -- max-pool the scores and keep the per-head top-k.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2: a pooling layer smooths the scores so massive activations do
// not mislead the selection; in each layer and head the top k^l tokens are kept
// and all others discarded for good.
//
// One CTA of 1024 threads per (sequence, kv head):
//   1. pooled[i] = max of scores[i - (w-1)/2 .. i + (w-1)/2] clipped to the range;
//      the pooled row is staged in shared memory when it fits (n - alpha <=
//      kSmemMax), otherwise it is re-read from global memory (L2);
//   2. radix select of the k-th largest pooled value tau on its fp32 bit pattern
//      (scores are >= 0, so unsigned order == float order), four 8-bit passes;
//   3. ordered compaction: every index with pooled > tau, plus the lowest-index
//      entries equal to tau until k are kept, written in ascending index order.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kWarps = kTopkThreads / 32;
constexpr int kSmemMax = 32 * 1024;     // rows up to this length are staged in shared memory

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

// When the scoring launch before this one gave up a wait (*abort_flag != 0; the
// flag may be NULL), its scores are incomplete: every kept index is written as -1.
// Every thread of every CTA must read the same value (a CTA of a cluster that left
// early would strand its peers at a cluster barrier), so the flag is final when it
// is read: only the scoring launch writes it, the plain launch starts after that
// launch and the cluster launch reads it after griddepcontrol.wait, and the host
// clears it only after synchronising the stream. The cache's own selections pass
// no flag (their error word is host-visible and cleared by the next call).
__device__ __forceinline__ bool selection_aborted(const unsigned* abort_flag, int32_t* out,
                                                  int k_sel, bool writer) {
  if (!abort_flag || *reinterpret_cast<const volatile unsigned*>(abort_flag) == 0u) return false;
  if (writer)
    for (int i = threadIdx.x; i < k_sel; i += blockDim.x) out[i] = -1;
  return true;
}

// SMEM: the pooled row lives in dynamic shared memory; else in `pooled` (global).
template <bool SMEM>
__global__ void __launch_bounds__(kTopkThreads)
pool_topk_kernel(const float* __restrict__ scores, float* __restrict__ pooled, int ns, int w,
                 int k_sel, int32_t* __restrict__ kept, const unsigned* abort_flag) {
  __shared__ TopkSmem s;
  extern __shared__ __align__(16) float spool[];
  const int unit = blockIdx.x;
  const float* sc = scores + (size_t)unit * ns;
  float* pg = pooled + (size_t)unit * ns;
  float* pl = SMEM ? spool : pg;
  int32_t* out = kept + (size_t)unit * k_sel;
  if (selection_aborted(abort_flag, out, k_sel < ns ? k_sel : ns, true)) return;
  const int r = (w - 1) / 2;
  if constexpr (SMEM) {
    // stage the scores (coalesced), pool from shared memory into registers, write back
    constexpr int PER = kSmemMax / kTopkThreads;
    for (int i = threadIdx.x; i < ns; i += kTopkThreads) spool[i] = __ldg(sc + i);
    __syncthreads();
    float pv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = threadIdx.x + j * kTopkThreads;
      float m = 0.f;
      if (i < ns) {
        m = spool[i];
        const int lo = i - r < 0 ? 0 : i - r, hi = i + r >= ns ? ns - 1 : i + r;
        for (int t = lo; t <= hi; ++t) m = fmaxf(m, spool[t]);
      }
      pv[j] = m;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = threadIdx.x + j * kTopkThreads;
      if (i < ns) { spool[i] = pv[j]; pg[i] = pv[j]; }
    }
  } else {
    for (int i = threadIdx.x; i < ns; i += kTopkThreads) {
      float m = __ldg(sc + i);
      const int lo = i - r < 0 ? 0 : i - r, hi = i + r >= ns ? ns - 1 : i + r;
      for (int t = lo; t <= hi; ++t) m = fmaxf(m, __ldg(sc + t));
      pg[i] = m;
    }
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
    // scores cluster in a few bins: aggregate equal bins within a warp first so
    // the shared-memory atomics do not serialize on one address
    for (int base = 0; base < ns; base += kTopkThreads) {
      const int i = base + threadIdx.x;
      unsigned key = 256u;                              // "no bin"
      if (i < ns) {
        const unsigned u = __float_as_uint(pl[i]);
        if ((u & mask) == prefix) key = (u >> shift) & 255u;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      if (key < 256u && (threadIdx.x & 31) == __ffs(peers) - 1)
        atomicAdd(&s.hist[key], (unsigned)__popc(peers));
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

  // ordered compaction: warp w owns the contiguous span [w*span, (w+1)*span) and
  // walks it 32 consecutive indices at a time (lanes read consecutive elements, so
  // shared-memory reads are conflict-free); ballots give in-order ranks.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int span = (ns + kWarps - 1) / kWarps;
  const int w0 = warp * span, w1 = w0 + span < ns ? w0 + span : ns;
  unsigned gt = 0, eq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const unsigned u = i < w1 ? __float_as_uint(pl[i]) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, i < w1 && u > tau));
    eq += __popc(__ballot_sync(0xffffffffu, i < w1 && u == tau));
  }
  // exclusive scan over warps (lane 0 of each warp contributes its totals)
  unsigned egt, eeq;
  block_scan2(s, threadIdx.x == warp * 32 ? gt : 0u, threadIdx.x == warp * 32 ? eq : 0u, egt,
              eeq);
  egt = __shfl_sync(0xffffffffu, egt, 0);
  eeq = __shfl_sync(0xffffffffu, eeq, 0);
  unsigned pos = egt + (eeq < need_eq ? eeq : need_eq);
  unsigned eq_seen = eeq;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const unsigned u = i < w1 ? __float_as_uint(pl[i]) : 0u;
    const bool is_gt = i < w1 && u > tau, is_eq = i < w1 && u == tau;
    const unsigned beq = __ballot_sync(0xffffffffu, is_eq);
    const bool take = is_gt || (is_eq && eq_seen + __popc(beq & lt) < need_eq);
    const unsigned bt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const unsigned p = pos + __popc(bt & lt);
      if (p < (unsigned)k_sel) out[p] = i;   // bounded even if the select were wrong
    }
    pos += __popc(bt);
    eq_seen += __popc(beq);
  }
}

// ------------------------------------------------------------ cluster version
// One thread-block cluster of kCluster CTAs per (sequence, kv head). CTA r pools
// and selects over its segment [r * seg, (r + 1) * seg) of the scores (staged in
// shared memory with a halo of (w - 1) / 2 on each side). Each radix pass builds a
// 256-bin histogram per CTA (per-warp histograms, then summed); the CTAs read each other's histograms through distributed shared
// memory after one cluster barrier, so every CTA takes the same decision and also
// learns, per CTA, how many of its elements the pass already decided "kept" (bins
// above the selected one): the ordered compaction needs no further exchange. The
// passes stop early once the selected bin is kept whole.
constexpr int kCluster = 8;
constexpr int kCThreads = 1024;   // threads 0..255 also own one histogram bin each
constexpr int kCWarps = kCThreads / 32;
constexpr int kMaxSeg = 22 * 1024;   // elements per CTA (two fp32 copies in shared memory)
constexpr size_t kOnePerSm = 120 * 1024;   // dynamic shared memory that leaves room for one CTA

struct ClusterSmem {
  unsigned whist[kCWarps][256];   // per-warp histograms of the current pass
  unsigned hist[2][256];          // this CTA's histogram, by pass parity (read remotely)
  unsigned total[256];            // the cluster's histogram
  unsigned red[kCWarps][kCluster];
  unsigned gtc[kCluster];         // per CTA: elements decided kept by the bins above
  unsigned eqc[kCluster];         // per CTA: elements in the final selected bin
  unsigned warp_gt[kCWarps], warp_eq[kCWarps];
  unsigned sel_bin, krem, done;
};

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ unsigned ld_cluster_u32(const unsigned* p, unsigned rank) {
  const unsigned a = (unsigned)__cvta_generic_to_shared(p);
  unsigned ra, v;
  asm("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

// Dynamic shared memory of the selection for a segment of `seg` and pool radius hw.
__host__ __device__ inline size_t select_smem_floats(int seg, int hw) {
  return (size_t)((seg + 2 * hw + 4 + 3) / 4 * 4) + seg;
}

// Pool and select within the cluster; CTA `rank` writes the kept positions of its
// segment to out (ascending, ranks offset by the preceding CTAs). No remote
// shared-memory access remains when it returns; the caller ends with a cluster
// barrier before any CTA of the cluster exits.
__device__ void cluster_pool_select(ClusterSmem& s, float* dyn, const float* __restrict__ sc,
                                    float* __restrict__ pg, int32_t* __restrict__ out, int ns,
                                    int w, int k_sel) {
  const unsigned rank = cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = (ns + kCluster - 1) / kCluster;
  const int i0 = min(ns, (int)rank * seg), i1 = min(ns, i0 + seg);
  const int n_loc = i1 - i0;
  const int hw = (w - 1) / 2;
  float* sx = dyn;                                          // [i0 - hw, i1 + hw), -inf outside
  float* pl = dyn + (seg + 2 * hw + 4 + 3) / 4 * 4;          // pooled scores of [i0, i1)

  // 1. stage the segment with its halo: every element an independent 4-byte
  //    asynchronous copy (all in flight at once); -inf outside the row
  const int n_halo = n_loc + 2 * hw;
  for (int t = threadIdx.x; t < n_halo; t += kCThreads) {
    const int i = i0 - hw + t;
    if (i >= 0 && i < ns) {
      const unsigned d = (unsigned)__cvta_generic_to_shared(sx + t);
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" :: "r"(d), "l"(sc + i) : "memory");
    } else {
      sx[t] = -INFINITY;
    }
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();
  // 2. max-pool, four outputs per thread: the windows of outputs t0..t0+3 share
  //    their middle [t0 + 3, t0 + 2hw]; reads past the halo only feed outputs past
  //    the segment, which are not written
  for (int q = threadIdx.x; 4 * q < n_loc; q += kCThreads) {
    const int t0 = 4 * q;
    float m[4];
    if (hw == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) m[j] = sx[t0 + j];
    } else {
      float core = -INFINITY;
      for (int d = 3; d <= 2 * hw; ++d) core = fmaxf(core, sx[t0 + d]);
      const float a0 = sx[t0], a1 = sx[t0 + 1], a2 = sx[t0 + 2];
      const float b1 = sx[t0 + 2 * hw + 1], b2 = sx[t0 + 2 * hw + 2], b3 = sx[t0 + 2 * hw + 3];
      m[0] = fmaxf(core, fmaxf(a0, fmaxf(a1, a2)));
      m[1] = fmaxf(core, fmaxf(a1, fmaxf(a2, b1)));
      m[2] = fmaxf(core, fmaxf(a2, fmaxf(b1, b2)));
      m[3] = fmaxf(core, fmaxf(b1, fmaxf(b2, b3)));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (t0 + j < n_loc) { pl[t0 + j] = m[j]; pg[i0 + t0 + j] = m[j]; }
  }
  if (k_sel >= ns) {   // everything is kept
    for (int t = threadIdx.x; t < n_loc; t += kCThreads) out[i0 + t] = i0 + t;
    return;
  }
  if (k_sel <= 0) return;
  if (threadIdx.x == 0) { s.krem = (unsigned)k_sel; s.done = 0u; }

  // 3. radix select of the k-th largest pooled score (fp32 bits: scores are >= 0)
  unsigned prefix = 0, mask = 0;
  unsigned gacc[kCluster];         // this thread's bin: per CTA, counts of bins above the selection
  unsigned v[kCluster];
#pragma unroll
  for (int r = 0; r < kCluster; ++r) gacc[r] = 0u;
  int shift = 24;
  for (int pass = 0; pass < 4; ++pass, shift -= 8) {
    unsigned* h = s.hist[pass & 1];
    for (int t = threadIdx.x; t < kCWarps * 256; t += kCThreads) (&s.whist[0][0])[t] = 0u;
    __syncthreads();
    for (int t = threadIdx.x; t < n_loc; t += kCThreads) {
      const unsigned u = __float_as_uint(pl[t]);
      if ((u & mask) == prefix) atomicAdd(&s.whist[warp][(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 256) {
      unsigned hb = 0;
#pragma unroll
      for (int ww = 0; ww < kCWarps; ++ww) hb += s.whist[ww][threadIdx.x];
      h[threadIdx.x] = hb;
    }
    cluster_sync_all();   // every CTA's histogram of this pass is complete
    if (threadIdx.x < 256) {
      const int b = threadIdx.x;
#pragma unroll
      for (int r = 0; r < kCluster; ++r) v[r] = ld_cluster_u32(&h[b], (unsigned)r);
      unsigned tot = 0;
#pragma unroll
      for (int r = 0; r < kCluster; ++r) tot += v[r];
      s.total[b] = tot;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins [8l, 8l + 8); suffix sums from the top bin down
      unsigned own = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) own += s.total[8 * lane + j];
      unsigned suf = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      const unsigned above = suf - own;
      const unsigned krem = s.krem;
      __syncwarp();
      if (suf >= krem && above < krem) {
        unsigned cum = above;
        for (int b = 8 * lane + 7; b >= 8 * lane; --b) {
          const unsigned hb = s.total[b];
          if (cum + hb >= krem) {
            s.sel_bin = (unsigned)b;
            s.krem = krem - cum;
            s.done = (cum + hb == krem) ? 1u : 0u;   // the bin is kept whole
            break;
          }
          cum += hb;
        }
      }
    }
    __syncthreads();
    const unsigned sel = s.sel_bin;
    if (threadIdx.x < 256 && (unsigned)threadIdx.x > sel) {
#pragma unroll
      for (int r = 0; r < kCluster; ++r) gacc[r] += v[r];
    }
    prefix |= sel << shift;
    mask |= 255u << shift;
    if (s.done || pass == 3) {
      if ((unsigned)threadIdx.x == sel) {
#pragma unroll
        for (int r = 0; r < kCluster; ++r) s.eqc[r] = v[r];
      }
      break;
    }
  }
  // tau: the selected value (all 32 bits decided), or, when the passes stopped
  // early, the lowest value of the selected bin, every element >= tau being kept
  const unsigned tau = prefix;
  const bool ge = s.done != 0u;
  const unsigned need_eq = ge ? 0u : s.krem;
  // per-CTA counts of the bins above the selection, summed over the block
#pragma unroll
  for (int r = 0; r < kCluster; ++r) {
    unsigned x = gacc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) s.red[warp][r] = x;
  }
  __syncthreads();
  if (threadIdx.x < kCluster) {
    unsigned x = 0;
#pragma unroll
    for (int ww = 0; ww < kCWarps; ++ww) x += s.red[ww][threadIdx.x];
    s.gtc[threadIdx.x] = x;
  }
  __syncthreads();
  unsigned base_gt = 0, base_eq = 0;
  for (unsigned r = 0; r < rank; ++r) { base_gt += s.gtc[r]; base_eq += s.eqc[r]; }
  if (ge) { base_gt += base_eq; base_eq = 0; }

  // 4. ordered compaction: warp w owns the contiguous span [w*span, (w+1)*span) of
  //    the segment; the preceding CTAs' and warps' counts give the offsets
  const int span = (n_loc + kCWarps - 1) / kCWarps;
  const int w0 = min(n_loc, warp * span), w1 = min(n_loc, w0 + span);
  unsigned gt = 0, eq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int t = base + lane;
    const unsigned u = t < w1 ? __float_as_uint(pl[t]) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, t < w1 && (ge ? u >= tau : u > tau)));
    eq += __popc(__ballot_sync(0xffffffffu, t < w1 && !ge && u == tau));
  }
  if (lane == 0) { s.warp_gt[warp] = gt; s.warp_eq[warp] = eq; }
  __syncthreads();
  unsigned egt = base_gt, eeq = base_eq;
  for (int ww = 0; ww < warp; ++ww) { egt += s.warp_gt[ww]; eeq += s.warp_eq[ww]; }
  unsigned pos = egt + (eeq < need_eq ? eeq : need_eq);
  unsigned eq_seen = eeq;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int t = base + lane;
    const unsigned u = t < w1 ? __float_as_uint(pl[t]) : 0u;
    const bool is_gt = t < w1 && (ge ? u >= tau : u > tau);
    const bool is_eq = t < w1 && !ge && u == tau;
    const unsigned beq = __ballot_sync(0xffffffffu, is_eq);
    const bool take = is_gt || (is_eq && eq_seen + __popc(beq & lt) < need_eq);
    const unsigned bt = __ballot_sync(0xffffffffu, take);
    if (take) {
      const unsigned p = pos + __popc(bt & lt);
      if (p < (unsigned)k_sel) out[p] = i0 + t;   // bounded even if the select were wrong
    }
    pos += __popc(bt);
    eq_seen += __popc(beq);
  }
}

__global__ void __launch_bounds__(kCThreads)
pool_topk_cluster_kernel(const float* __restrict__ scores, float* __restrict__ pooled, int ns,
                         int w, int k_sel, int32_t* __restrict__ kept,
                         const unsigned* abort_flag) {
  __shared__ ClusterSmem s;
  extern __shared__ __align__(16) float dyn[];
  const int unit = blockIdx.x / kCluster;
  pdl_wait();      // the scores are complete
  // every CTA of the cluster reads the same flag (written before this launch) and
  // leaves before any cluster barrier
  if (selection_aborted(abort_flag, kept + (size_t)unit * k_sel, k_sel < ns ? k_sel : ns,
                        blockIdx.x % kCluster == 0)) {
    pdl_release();
    return;
  }
  cluster_pool_select(s, dyn, scores + (size_t)unit * ns, pooled + (size_t)unit * ns,
                      kept + (size_t)unit * k_sel, ns, w, k_sel);
  // only now: dependents scheduled earlier would wait on these SMs beside the selection
  pdl_release();
  cluster_sync_all();   // no CTA leaves while another may still read its shared memory
}

cudaError_t launch_topk_cluster(const float* scores, float* pooled, int units, int ns, int w,
                                int k_sel, int32_t* kept, const unsigned* abort_flag,
                                cudaStream_t stream) {
  const int seg = (ns + kCluster - 1) / kCluster;
  // a dependent launch (its set-up overlaps the scoring launch's end); the shared
  // memory is padded so that one CTA fits an SM: scheduled early, the CTAs would
  // otherwise pack several to an SM as the scoring CTAs leave, and run far slower
  size_t sm = select_smem_floats(seg, (w - 1) / 2) * sizeof(float);
  if (sm < kOnePerSm) sm = kOnePerSm;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(pool_topk_cluster_kernel), sm);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * kCluster);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attr();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, pool_topk_cluster_kernel, scores, pooled, ns, w, k_sel, kept,
                         abort_flag);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The cluster kernel spreads a long row over 8 SMs, for few units; with many units,
// or rows short enough that a cluster's barriers would outweigh its work, one CTA per
// unit (the row staged in shared memory) fills the GPU by itself.
static bool use_cluster(int units, int ns, int w) {
  if ((ns + kCluster - 1) / kCluster > kMaxSeg || w > 129) return false;
  if (ns > kSmemMax) return true;
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n_sm = 148;
  }
  return ns > 8192 && units * 2 <= n_sm;
}

cudaError_t launch_topk(const float* scores, float* pooled, int units, int ns, int w, int k_sel,
                        int32_t* kept, const unsigned* abort_flag, cudaStream_t stream) {
  if (use_cluster(units, ns, w))
    return launch_topk_cluster(scores, pooled, units, ns, w, k_sel, kept, abort_flag, stream);
  if (ns <= kSmemMax) {
    const size_t sm = (size_t)ns * sizeof(float);
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(pool_topk_kernel<true>), sm);
    if (e != cudaSuccess) return e;
    pool_topk_kernel<true><<<units, kTopkThreads, sm, stream>>>(scores, pooled, ns, w, k_sel,
                                                                 kept, abort_flag);
  } else {
    pool_topk_kernel<false><<<units, kTopkThreads, 0, stream>>>(scores, pooled, ns, w, k_sel,
                                                                 kept, abort_flag);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pool_topk(const kvc_cache* c, int layer, int32_t* kept_out, int k_sel,
                             cudaStream_t stream) {
  (void)layer;
  const kvc_dims& d = c->dims;
  return launch_topk(c->scores, c->pooled, d.batch * d.n_kv_heads, d.prompt_len - d.obs_window,
                     d.pool_kernel, k_sel, kept_out, nullptr, stream);
}

// The same launch with the score and pooled buffers given explicitly (used by
// the allocation-free selection entry point, whose scoring error word is
// abort_flag).
cudaError_t launch_pool_topk_into(const kvc_dims& d, const float* scores, float* pooled,
                                  int32_t* kept_out, int k_sel, const unsigned* abort_flag,
                                  cudaStream_t stream) {
  return launch_topk(scores, pooled, d.batch * d.n_kv_heads, d.prompt_len - d.obs_window,
                     d.pool_kernel, k_sel, kept_out, abort_flag, stream);
}

}  // namespace kvc
