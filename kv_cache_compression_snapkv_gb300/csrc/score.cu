// score.cu -- observation-window scores of every prompt key.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2 "KV Cache Selection": each prompt key i < n - alpha is scored
// by the attention the last alpha ("instruction") tokens pay it; MiniKV §2
// eq. (1): A = softmax(Q K^T / sqrt(d)). Per (sequence, kv head) the rows are the
// alpha observation queries of each of the g query heads that share the kv head
// (M = g * alpha rows); a row at prompt position p sees keys 0..p (causal); each
// row is normalised over all the keys it sees, then rows are summed per key.
//
// Two passes over the keys, both tiled 128 keys per CTA, one 16-row slice per warp:
//   stats   per (chunk, row): max and sum of exp2 of the scaled logits
//   combine per row: global max M_r and log2 of the normaliser -> b_r
//   cols    per key: sum_r exp2(l_ri * log2(e)/sqrt(d) - b_r)
// Logit tiles are tensor-core products (mma m16n8k16 bf16 -> fp32) of the
// register-resident query rows with a shared-memory key tile.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kChunk = kScoreChunk;   // 128 keys per CTA

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int D>
struct ScoreSmem {
  __nv_bfloat16 k[kChunk][D + 8];   // +8 halves: conflict-free fragment loads
  float col[16][kChunk];
};

// Stage keys [k0, k0 + 128) of one unit (zero beyond `limit`).
template <int D>
__device__ __forceinline__ void load_key_tile(ScoreSmem<D>& s, const __nv_bfloat16* __restrict__ K,
                                              int k0, int limit) {
  constexpr int CH = D / 8;
  for (int i = threadIdx.x; i < kChunk * CH; i += blockDim.x) {
    int r = i / CH, ch = i % CH;
    int key = k0 + r;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (key < limit) u = *reinterpret_cast<const uint4*>(K + (size_t)key * D + ch * 8);
    *reinterpret_cast<uint4*>(&s.k[r][ch * 8]) = u;
  }
}

// Query fragments of this warp's 16 rows (rows >= M are zero).
template <int D>
__device__ __forceinline__ void load_query_frags(uint32_t (&a)[D / 16][4],
                                                 const __nv_bfloat16* __restrict__ Q, int row0, int M) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const int r0 = row0 + gid, r1 = r0 + 8;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c = 16 * ks + 2 * tid;
    a[ks][0] = r0 < M ? *reinterpret_cast<const uint32_t*>(Q + (size_t)r0 * D + c) : 0u;
    a[ks][1] = r1 < M ? *reinterpret_cast<const uint32_t*>(Q + (size_t)r1 * D + c) : 0u;
    a[ks][2] = r0 < M ? *reinterpret_cast<const uint32_t*>(Q + (size_t)r0 * D + c + 8) : 0u;
    a[ks][3] = r1 < M ? *reinterpret_cast<const uint32_t*>(Q + (size_t)r1 * D + c + 8) : 0u;
  }
}

// Logits of the warp's 16 rows against the 128 staged keys.
template <int D>
__device__ __forceinline__ void logit_tile(float (&c)[16][4], const uint32_t (&a)[D / 16][4],
                                           const ScoreSmem<D>& s) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
    const __nv_bfloat16* kr = &s.k[nt * 8 + gid][2 * tid];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + 16 * ks);
      uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 16 * ks + 8);
      mma_bf16(c[nt], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
    }
  }
}

// grid (n_chunks, units): per-chunk row max / sum of exp2.
template <int D>
__global__ void score_stats_kernel(const __nv_bfloat16* __restrict__ q_obs,
                                   const __nv_bfloat16* __restrict__ k, int n, int alpha, int M,
                                   float sl2, float2* __restrict__ stats) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ScoreSmem<D>& s = *reinterpret_cast<ScoreSmem<D>*>(smem_raw);
  const int chunk = blockIdx.x, unit = blockIdx.y, nch = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const __nv_bfloat16* K = k + (size_t)unit * n * D;
  const __nv_bfloat16* Q = q_obs + (size_t)unit * M * D;
  const int k0 = chunk * kChunk;
  load_key_tile<D>(s, K, k0, n);
  uint32_t a[D / 16][4];
  load_query_frags<D>(a, Q, warp * 16, M);
  __syncthreads();
  float c[16][4];
  logit_tile<D>(c, a, s);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = warp * 16 + gid + 8 * half;
    const int pos = n - alpha + (row % alpha);
    float m = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = k0 + nt * 8 + 2 * tid + e;
        float x = c[nt][2 * half + e] * sl2;
        x = (key <= pos && key < n) ? x : -INFINITY;
        c[nt][2 * half + e] = x;
        m = fmaxf(m, x);
      }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    float sum = 0.f;
    if (m != -INFINITY) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) sum += fast_exp2(c[nt][2 * half + e] - m);
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (tid == 0 && row < M) stats[((size_t)unit * nch + chunk) * M + row] = make_float2(m, sum);
  }
}

// grid (units), block 256: b_r = M_r + log2(sum_c s_c 2^(m_c - M_r))
__global__ void score_combine_kernel(const float2* __restrict__ stats, int nch, int M,
                                     float* __restrict__ rowbias) {
  const int unit = blockIdx.x;
  for (int r = threadIdx.x; r < M; r += blockDim.x) {
    const float2* st = stats + (size_t)unit * nch * M + r;
    float mx = -INFINITY;
    for (int ch = 0; ch < nch; ++ch) mx = fmaxf(mx, st[(size_t)ch * M].x);
    float z = 0.f;
    for (int ch = 0; ch < nch; ++ch) {
      float2 v = st[(size_t)ch * M];
      if (v.y > 0.f) z += v.y * exp2f(v.x - mx);
    }
    rowbias[(size_t)unit * M + r] = mx + log2f(z);
  }
}

// grid (chunks over [0, n - alpha), units): column sums of normalised rows.
template <int D>
__global__ void score_cols_kernel(const __nv_bfloat16* __restrict__ q_obs,
                                  const __nv_bfloat16* __restrict__ k, int n, int alpha, int M,
                                  float sl2, const float* __restrict__ rowbias,
                                  float* __restrict__ scores) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ScoreSmem<D>& s = *reinterpret_cast<ScoreSmem<D>*>(smem_raw);
  const int chunk = blockIdx.x, unit = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const int nwarps = blockDim.x >> 5;
  const int ns = n - alpha;
  const __nv_bfloat16* K = k + (size_t)unit * n * D;
  const __nv_bfloat16* Q = q_obs + (size_t)unit * M * D;
  const int k0 = chunk * kChunk;
  load_key_tile<D>(s, K, k0, ns);
  uint32_t a[D / 16][4];
  load_query_frags<D>(a, Q, warp * 16, M);
  const int r0 = warp * 16 + gid, r1 = r0 + 8;
  const float b0 = r0 < M ? rowbias[(size_t)unit * M + r0] : INFINITY;
  const float b1 = r1 < M ? rowbias[(size_t)unit * M + r1] : INFINITY;
  __syncthreads();
  float c[16][4];
  logit_tile<D>(c, a, s);
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = fast_exp2(c[nt][e] * sl2 - b0) + fast_exp2(c[nt][2 + e] * sl2 - b1);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      if (gid == 0) s.col[warp][nt * 8 + 2 * tid + e] = v;
    }
  }
  __syncthreads();
  for (int col = threadIdx.x; col < kChunk; col += blockDim.x) {
    float acc = 0.f;
    for (int w = 0; w < nwarps; ++w) acc += s.col[w][col];
    const int key = k0 + col;
    if (key < ns) scores[(size_t)unit * ns + key] = acc;
  }
}

}  // namespace

cudaError_t launch_score(const kvc_cache* c, int layer, const __nv_bfloat16* q_obs,
                         const __nv_bfloat16* k, cudaStream_t stream) {
  (void)layer;
  const kvc_dims& d = c->dims;
  const int units = d.batch * d.n_kv_heads;
  const int n = d.prompt_len, alpha = d.obs_window;
  const int M = c->g * alpha;
  const int warps = (M + 15) / 16;
  const int nch1 = (n + kChunk - 1) / kChunk;
  const int nch2 = (n - alpha + kChunk - 1) / kChunk;
  const float sl2 = 1.4426950408889634f / sqrtf((float)d.head_dim);
  float* rowbias = reinterpret_cast<float*>(c->rowstat);
  cudaError_t e;
  if (d.head_dim == 128) {
    size_t sm = sizeof(ScoreSmem<128>);
    if ((e = cudaFuncSetAttribute(score_stats_kernel<128>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    if ((e = cudaFuncSetAttribute(score_cols_kernel<128>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    score_stats_kernel<128><<<dim3(nch1, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                          sl2, c->stats);
    score_combine_kernel<<<units, 256, 0, stream>>>(c->stats, nch1, M, rowbias);
    score_cols_kernel<128><<<dim3(nch2, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                         sl2, rowbias, c->scores);
  } else if (d.head_dim == 64) {
    size_t sm = sizeof(ScoreSmem<64>);
    if ((e = cudaFuncSetAttribute(score_stats_kernel<64>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    if ((e = cudaFuncSetAttribute(score_cols_kernel<64>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    score_stats_kernel<64><<<dim3(nch1, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                         sl2, c->stats);
    score_combine_kernel<<<units, 256, 0, stream>>>(c->stats, nch1, M, rowbias);
    score_cols_kernel<64><<<dim3(nch2, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                        sl2, rowbias, c->scores);
  } else {
    return cudaErrorInvalidValue;
  }
  count_launches(3);
  return cudaGetLastError();
}

// The same three scoring launches with the scratch buffers given explicitly
// (used by the allocation-free selection entry point).
cudaError_t launch_score_into(const kvc_dims& d, const __nv_bfloat16* q_obs,
                              const __nv_bfloat16* k, float2* stats, float* rowbias,
                              float* scores, cudaStream_t stream) {
  const int units = d.batch * d.n_kv_heads;
  const int n = d.prompt_len, alpha = d.obs_window;
  const int M = (d.n_q_heads / d.n_kv_heads) * alpha;
  const int warps = (M + 15) / 16;
  const int nch1 = (n + kChunk - 1) / kChunk;
  const int nch2 = (n - alpha + kChunk - 1) / kChunk;
  const float sl2 = 1.4426950408889634f / sqrtf((float)d.head_dim);
  cudaError_t e;
  if (d.head_dim == 128) {
    size_t sm = sizeof(ScoreSmem<128>);
    if ((e = cudaFuncSetAttribute(score_stats_kernel<128>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    if ((e = cudaFuncSetAttribute(score_cols_kernel<128>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    score_stats_kernel<128><<<dim3(nch1, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                          sl2, stats);
    score_combine_kernel<<<units, 256, 0, stream>>>(stats, nch1, M, rowbias);
    score_cols_kernel<128><<<dim3(nch2, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                         sl2, rowbias, scores);
  } else if (d.head_dim == 64) {
    size_t sm = sizeof(ScoreSmem<64>);
    if ((e = cudaFuncSetAttribute(score_stats_kernel<64>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    if ((e = cudaFuncSetAttribute(score_cols_kernel<64>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
      return e;
    score_stats_kernel<64><<<dim3(nch1, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                         sl2, stats);
    score_combine_kernel<<<units, 256, 0, stream>>>(stats, nch1, M, rowbias);
    score_cols_kernel<64><<<dim3(nch2, units), warps * 32, sm, stream>>>(q_obs, k, n, alpha, M,
                                                                        sl2, rowbias, scores);
  } else {
    return cudaErrorInvalidValue;
  }
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace kvc
