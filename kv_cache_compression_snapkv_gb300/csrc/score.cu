// score.cu -- entry points of the scoring launch (score_tc.cu): the cache's own
// scratch, or scratch given explicitly; and the variance of a layer's scores.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2 "KV Cache Selection"; MiniKV §2 eq. (1).
#include "kvc_internal.cuh"

namespace kvc {

cudaError_t launch_score(const kvc_cache* c, int layer, const __nv_bfloat16* q_obs,
                         const __nv_bfloat16* k, cudaStream_t stream) {
  (void)layer;
  return launch_score_tc(c->dims, q_obs, k, c->stats, c->gsync, c->scores, c->err, stream);
}

// The same launch with the scratch buffers and the error word given explicitly
// (used by the allocation-free selection entry point).
cudaError_t launch_score_into(const kvc_dims& d, const __nv_bfloat16* q_obs,
                              const __nv_bfloat16* k, float2* stats, unsigned* gsync,
                              float* scores, unsigned* err, cudaStream_t stream) {
  return launch_score_tc(d, q_obs, k, stats, gsync, scores, err, stream);
}

namespace {

// Unevaluated sum hi + lo of two fp32 values (double-float), added with the
// error-free two-sum so that a block total keeps ~48 significant bits without fp64
// arithmetic per element or per thread (the part's fp64 rate is a small fraction of
// its fp32 rate).
struct FF { float hi, lo; };
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float err = (a.hi - (s - bb)) + (b.hi - bb);
  const float lo = a.lo + b.lo + err;
  const float hi = s + lo;
  return {hi, lo - (hi - s)};
}

// Sum of the threads' values over the block, identical in every thread: double-float
// within each warp (shuffles), the warps' totals added in fp64 by one thread in warp
// order. Callable repeatedly: the first barrier keeps a previous call's readers
// ahead of this call's writers.
__device__ double block_sum(FF v, FF* red, double* total) {
  for (int o = 16; o; o >>= 1) {
    FF t;
    t.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
    t.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
    v = ff_add(v, t);
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += (double)red[w].hi + (double)red[w].lo;
    *total = t;
  }
  __syncthreads();
  return *total;
}

// MiniKV §4.2 "Layer-Specific Selectivity" (the variance policy) and Figure 7:
// the variance score of cumulated attention: population variance of each (sequence,
// kv head) unit's m selection scores. Each unit is cut into S slices, one CTA each:
// the slice's mean (compensated fp32 sums of its strided elements, the block's
// partials added in fp64 in a fixed order) and its sum of squared deviations about
// the fp32-rounded slice mean (corrected for that rounding); the CTA arriving last
// at the unit's ticket merges the S (count, sum, M2) partials in slice order
// (pairwise update: M2 = sum over slices of M2_s + n_s (mean_s - mean)^2, fp64),
// writes the variance and returns the ticket to zero. (fp64 arithmetic per element
// would run at the part's small fp64 rate.)
constexpr int kVarThreads = 256;
constexpr int kVarSliceMin = 4096;   // elements per slice at least (a CTA's work)
constexpr int kVarSlicesMax = 32;

struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  __device__ __forceinline__ FF value() const { return {s, -c}; }
};

__global__ void __launch_bounds__(kVarThreads) score_variance_kernel(
    const float* __restrict__ scores, int m, int S, double* __restrict__ ws,
    unsigned* __restrict__ cnt, float* __restrict__ var) {
  __shared__ FF red[kVarThreads / 32];
  __shared__ double total;
  __shared__ bool last;
  const int unit = blockIdx.x / S, sl = blockIdx.x % S;
  const int i0 = (int)((long long)m * sl / S), i1 = (int)((long long)m * (sl + 1) / S);
  const int n = i1 - i0;
  const float* row = scores + (size_t)unit * m + i0;
  Kahan acc;
  for (int i = threadIdx.x; i < n; i += kVarThreads) acc.add(row[i]);
  __shared__ double s_mean;
  __shared__ float s_mean_f;
  const double sum = block_sum(acc.value(), red, &total);
  if (threadIdx.x == 0) {   // fp64 arithmetic in one thread only
    s_mean = n > 0 ? sum / n : 0.0;
    s_mean_f = (float)s_mean;
  }
  __syncthreads();
  const float mean_f = s_mean_f;
  Kahan acc2;
  for (int i = threadIdx.x; i < n; i += kVarThreads) {
    const float dv = row[i] - mean_f;
    acc2.add(dv * dv);
  }
  const double ss = block_sum(acc2.value(), red, &total);
  double* part = ws + ((size_t)unit * S + sl) * 3;
  if (threadIdx.x == 0) {
    // sum (x - mean_f)^2 = sum (x - mean)^2 + n (mean - mean_f)^2: remove the second term
    const double dm = s_mean - (double)mean_f;
    const double m2 = ss - n * dm * dm;
    part[0] = (double)n;
    part[1] = sum;
    part[2] = m2 > 0.0 ? m2 : 0.0;
    __threadfence();
    last = atomicAdd(&cnt[unit], 1u) == (unsigned)S - 1;
  }
  __syncthreads();
  if (!last || threadIdx.x >= 32) return;
  // the last CTA's first warp: lane k loads slice k's partial (all loads in flight at
  // once), lane 0 adds them in slice order
  __threadfence();
  const int lane = threadIdx.x;
  double nk = 0.0, sk = 0.0, mk = 0.0;
  if (lane < S) {
    const double* q = ws + ((size_t)unit * S + lane) * 3;
    nk = __ldcg(q);
    sk = __ldcg(q + 1);
    mk = __ldcg(q + 2);
  }
  double tot = 0.0;
  for (int k = 0; k < S; ++k) tot += __shfl_sync(0xffffffffu, sk, k);
  const double mu = tot / m;
  const double dk = nk > 0.0 ? sk / nk - mu : 0.0;
  const double term = mk + nk * dk * dk;
  double M2 = 0.0;
  for (int k = 0; k < S; ++k) M2 += __shfl_sync(0xffffffffu, term, k);
  if (lane != 0) return;
  const double v = M2 / m;
  var[unit] = (float)(v > 0.0 ? v : 0.0);
  cnt[unit] = 0u;   // the ticket returns to zero for the next launch
}

}  // namespace

cudaError_t launch_score_variance(const float* scores, int units, int m, float* var,
                                  double* ws, size_t ws_doubles, unsigned* cnt,
                                  cudaStream_t stream) {
  if (units <= 0 || m <= 0) return cudaSuccess;
  int S = (m + kVarSliceMin - 1) / kVarSliceMin;
  if (S > kVarSlicesMax) S = kVarSlicesMax;
  const size_t fit = ws_doubles / ((size_t)units * 3);
  if ((size_t)S > fit) S = (int)fit;
  if (S < 1) return cudaErrorInvalidValue;
  score_variance_kernel<<<units * S, kVarThreads, 0, stream>>>(scores, m, S, ws, cnt, var);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace kvc
