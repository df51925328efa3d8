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

// Sum of v over the block, identical in every thread (each thread adds the
// per-warp partial sums in the same order). Callable repeatedly: the first
// barrier keeps a previous call's readers ahead of this call's writers.
__device__ double block_sum(double v, double* red) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// MiniKV §4.2 "Layer-Specific Selectivity" (the variance policy) and Figure 7:
// the variance score of cumulated attention. One CTA per (sequence, kv head):
// population variance of its m selection scores, two passes (mean, then squared
// deviations). Each thread keeps a compensated fp32 sum (Kahan) of its strided
// elements; the block adds the 256 partial sums in fp64 in a fixed order. (fp64
// arithmetic per element would run at the part's small fp64 rate.)
constexpr int kVarThreads = 256;

struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  __device__ __forceinline__ double value() const { return (double)s - (double)c; }
};

__global__ void __launch_bounds__(kVarThreads) score_variance_kernel(
    const float* __restrict__ scores, int m, float* __restrict__ var) {
  __shared__ double red[kVarThreads / 32];
  const float* row = scores + (size_t)blockIdx.x * m;
  Kahan acc;
  for (int i = threadIdx.x; i < m; i += kVarThreads) acc.add(row[i]);
  const double mean = block_sum(acc.value(), red) / m;
  const float mean_f = (float)mean;
  Kahan acc2;
  for (int i = threadIdx.x; i < m; i += kVarThreads) {
    const float dv = row[i] - mean_f;
    acc2.add(dv * dv);
  }
  // sum (x - mean_f)^2 = n var + n (mean - mean_f)^2: remove the second term
  const double dm = mean - (double)mean_f;
  const double v = block_sum(acc2.value(), red) / m - dm * dm;
  if (threadIdx.x == 0) var[blockIdx.x] = (float)(v > 0.0 ? v : 0.0);
}

}  // namespace

cudaError_t launch_score_variance(const float* scores, int units, int m, float* var,
                                  cudaStream_t stream) {
  if (units <= 0 || m <= 0) return cudaSuccess;
  score_variance_kernel<<<units, kVarThreads, 0, stream>>>(scores, m, var);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace kvc
