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
// Two passes over the keys in chunks of 128, one 16-row slice per warp:
//   stats   per (row, chunk): max and sum of exp2 of the scaled logits
//   combine per row: global max M_r and log2 of the normaliser -> b_r
//   cols    per key: sum_r exp2(l_ri * log2(e)/sqrt(d) - b_r)
// Both passes run persistent CTAs over contiguous ranges of (unit, chunk) work
// with the next key tile copied asynchronously (cp.async, 16-byte pieces into a
// padded, bank-conflict-free tile) while the current one is multiplied. Logit
// tiles are tensor-core products (mma m16n8k16 bf16 -> fp32) of register-resident
// query rows with the shared-memory key tile.
#include <algorithm>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kChunk = kScoreChunk;   // 128 keys per tile

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

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int bytes = valid ? 16 : 0;   // 0: zero-fill, nothing read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
               :: "r"(s), "l"(gmem), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait1() {
  asm volatile("cp.async.wait_group 1;\n" ::: "memory");
}

template <int D>
struct ScoreSmem {
  __nv_bfloat16 k[2][kChunk][D + 8];   // double-buffered tile; +8 halves: conflict-free
  float col[16][kChunk];
};

// Issue the asynchronous copy of keys [k0, k0 + 128) of one unit (zero beyond limit).
template <int D>
__device__ __forceinline__ void prefetch_tile(__nv_bfloat16 (*dst)[D + 8],
                                              const __nv_bfloat16* __restrict__ K, int k0,
                                              int limit) {
  constexpr int CH = D / 8;
  for (int i = threadIdx.x; i < kChunk * CH; i += blockDim.x) {
    const int r = i / CH, ch = i % CH;
    const int key = k0 + r;
    const bool ok = key < limit;
    cp_async16(&dst[r][ch * 8], K + (size_t)(ok ? key : 0) * D + ch * 8, ok);
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
                                           const __nv_bfloat16 (*tile)[D + 8]) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
    const __nv_bfloat16* kr = &tile[nt * 8 + gid][2 * tid];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kr + 16 * ks);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kr + 16 * ks + 8);
      mma_bf16(c[nt], a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
    }
  }
}

// PASS 0: per (unit, row, chunk) max / sum of exp2 over keys [0, n) (causal).
// PASS 1: per key i < n - alpha, sum over rows of exp2(l * sl2 - b_r).
// Work item = (unit, chunk) with nch chunks per unit; CTA b takes items
// [b * total / G, (b + 1) * total / G).
template <int D, int PASS>
__global__ void __launch_bounds__(512, 1) score_pass_kernel(const __nv_bfloat16* __restrict__ q_obs,
                                  const __nv_bfloat16* __restrict__ k, int n, int alpha, int M,
                                  int nch, int total, float sl2, float2* __restrict__ stats,
                                  const float* __restrict__ rowbias, float* __restrict__ scores) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  ScoreSmem<D>& s = *reinterpret_cast<ScoreSmem<D>*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const int nwarps = blockDim.x >> 5;
  const int ns = n - alpha;
  const int limit = PASS == 0 ? n : ns;
  const int it0 = (int)((long long)blockIdx.x * total / gridDim.x);
  const int it1 = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
  if (it0 >= it1) return;

  prefetch_tile<D>(s.k[0], k + (size_t)(it0 / nch) * n * D, (it0 % nch) * kChunk, limit);
  cp_async_commit();
  int cur_unit = -1;
  uint32_t a[D / 16][4];
  float b0 = 0.f, b1 = 0.f;
  for (int it = it0; it < it1; ++it) {
    const int unit = it / nch, chunk = it % nch, buf = (it - it0) & 1;
    if (it + 1 < it1)
      prefetch_tile<D>(s.k[buf ^ 1], k + (size_t)((it + 1) / nch) * n * D,
                       ((it + 1) % nch) * kChunk, limit);
    cp_async_commit();
    if (unit != cur_unit) {
      cur_unit = unit;
      load_query_frags<D>(a, q_obs + (size_t)unit * M * D, warp * 16, M);
      if constexpr (PASS == 1) {
        const int r0 = warp * 16 + gid, r1 = r0 + 8;
        b0 = r0 < M ? rowbias[(size_t)unit * M + r0] : INFINITY;
        b1 = r1 < M ? rowbias[(size_t)unit * M + r1] : INFINITY;
      }
    }
    cp_async_wait1();
    __syncthreads();
    const int k0 = chunk * kChunk;
    float c[16][4];
    logit_tile<D>(c, a, s.k[buf]);
    if constexpr (PASS == 0) {
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
        if (tid == 0 && row < M) stats[((size_t)unit * M + row) * nch + chunk] = make_float2(m, sum);
      }
    } else {
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
    __syncthreads();   // the tile (and col) buffers are rewritten next iteration
  }
}

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

template <int D>
cudaError_t launch_passes(const kvc_dims& d, const __nv_bfloat16* q_obs, const __nv_bfloat16* k,
                          float2* stats, float* rowbias, float* scores, cudaStream_t stream) {
  const int units = d.batch * d.n_kv_heads;
  const int n = d.prompt_len, alpha = d.obs_window;
  const int M = (d.n_q_heads / d.n_kv_heads) * alpha;
  const int threads = ((M + 15) / 16) * 32;
  const int nch1 = (n + kChunk - 1) / kChunk;
  const int nch2 = (n - alpha + kChunk - 1) / kChunk;
  const float sl2 = 1.4426950408889634f / sqrtf((float)d.head_dim);
  const size_t sm = sizeof(ScoreSmem<D>);
  int dev = 0, n_sm = 0, per0 = 0, per1 = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)))
    return e;
  if ((e = cudaFuncSetAttribute(score_pass_kernel<D, 0>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) ||
      (e = cudaFuncSetAttribute(score_pass_kernel<D, 1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)) ||
      (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per0, score_pass_kernel<D, 0>, threads, sm)) ||
      (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per1, score_pass_kernel<D, 1>, threads, sm)))
    return e;
  const int total1 = units * nch1, total2 = units * nch2;
  const int g1 = std::max(1, std::min(total1, n_sm * std::max(per0, 1)));
  const int g2 = std::max(1, std::min(total2, n_sm * std::max(per1, 1)));
  score_pass_kernel<D, 0><<<g1, threads, sm, stream>>>(q_obs, k, n, alpha, M, nch1, total1, sl2,
                                                       stats, nullptr, nullptr);
  score_combine_kernel<<<dim3(units, (M + 7) / 8), 256, 0, stream>>>(stats, nch1, M, rowbias);
  score_pass_kernel<D, 1><<<g2, threads, sm, stream>>>(q_obs, k, n, alpha, M, nch2, total2, sl2,
                                                       nullptr, rowbias, scores);
  count_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_all(const kvc_dims& d, const __nv_bfloat16* q_obs, const __nv_bfloat16* k,
                       float2* stats, float* rowbias, float* scores, cudaStream_t stream) {
  if (d.head_dim == 128) return launch_passes<128>(d, q_obs, k, stats, rowbias, scores, stream);
  if (d.head_dim == 64) return launch_passes<64>(d, q_obs, k, stats, rowbias, scores, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_score(const kvc_cache* c, int layer, const __nv_bfloat16* q_obs,
                         const __nv_bfloat16* k, cudaStream_t stream) {
  (void)layer;
  return launch_all(c->dims, q_obs, k, c->stats, reinterpret_cast<float*>(c->rowstat), c->scores,
                    stream);
}

// The same launches with the scratch buffers given explicitly (used by the
// allocation-free selection entry point).
cudaError_t launch_score_into(const kvc_dims& d, const __nv_bfloat16* q_obs,
                              const __nv_bfloat16* k, float2* stats, float* rowbias,
                              float* scores, cudaStream_t stream) {
  return launch_all(d, q_obs, k, stats, rowbias, scores, stream);
}

}  // namespace kvc
