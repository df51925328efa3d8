// score.cu -- merge of the per-(row, tile) softmax statistics into one normaliser
// per observation row, and the entry points of the scoring launches.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2 "KV Cache Selection"; MiniKV §2 eq. (1): every observation row
// is a softmax over the keys it sees. The row-statistics pass (score_tc.cu) leaves,
// per (row, key tile), the tile's largest scaled logit m_c and sum_c of exp2 of the
// logits minus m_c; this kernel forms b_r = M_r + log2(sum_c sum_c 2^(m_c - M_r))
// with M_r = max_c m_c, so that the column pass can weight each logit by
// exp2(l * log2(e)/sqrt(d) - b_r) = softmax row r at that key.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

// grid (units, ceil(M / 8)), block 256: one warp per row,
// b_r = M_r + log2(sum_c s_c 2^(m_c - M_r)) over the row's chunk statistics.
__global__ void score_combine_kernel(const float2* __restrict__ stats, int nch, int M,
                                     float* __restrict__ rowbias) {
  const int unit = blockIdx.x, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 8 + (threadIdx.x >> 5);
  if (r >= M) return;
  const float2* st = stats + ((size_t)unit * M + r) * nch;
  float mx = -INFINITY;
  for (int ch = lane; ch < nch; ch += 32) mx = fmaxf(mx, st[ch].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float z = 0.f;
  for (int ch = lane; ch < nch; ch += 32) {
    const float2 v = st[ch];
    if (v.y > 0.f) z += v.y * exp2f(v.x - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane == 0) rowbias[(size_t)unit * M + r] = mx + log2f(z);
}

}  // namespace

cudaError_t launch_score_combine(const float2* stats, int nch, int M, int units, float* rowbias,
                                 cudaStream_t stream) {
  score_combine_kernel<<<dim3(units, (M + 7) / 8), 256, 0, stream>>>(stats, nch, M, rowbias);
  count_launches(1);
  return cudaGetLastError();
}

namespace {

cudaError_t launch_all(const kvc_dims& d, const __nv_bfloat16* q_obs, const __nv_bfloat16* k,
                       float2* stats, float* rowbias, float* scores, unsigned* err,
                       cudaStream_t stream) {
  return launch_score_tc(d, q_obs, k, stats, rowbias, scores, err, stream);
}

}  // namespace

cudaError_t launch_score(const kvc_cache* c, int layer, const __nv_bfloat16* q_obs,
                         const __nv_bfloat16* k, cudaStream_t stream) {
  (void)layer;
  return launch_all(c->dims, q_obs, k, c->stats, reinterpret_cast<float*>(c->rowstat), c->scores,
                    c->err, stream);
}

// The same launches with the scratch buffers given explicitly (used by the
// allocation-free selection entry point, which has no error word).
cudaError_t launch_score_into(const kvc_dims& d, const __nv_bfloat16* q_obs,
                              const __nv_bfloat16* k, float2* stats, float* rowbias,
                              float* scores, cudaStream_t stream) {
  return launch_all(d, q_obs, k, stats, rowbias, scores, nullptr, stream);
}

}  // namespace kvc
