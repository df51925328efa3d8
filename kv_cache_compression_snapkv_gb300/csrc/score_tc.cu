// score_tc.cu -- observation-window scores on the 5th-generation tensor cores.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2 "KV Cache Selection": every prompt key i < n - alpha is scored
// by the attention the last alpha ("instruction") tokens pay it; MiniKV §2 eq. (1):
// A = softmax(Q K^T / sqrt(d)). Per (sequence, kv head) the rows are the alpha
// observation queries of each of the g query heads sharing the kv head (M = g *
// alpha rows, M <= 256); a row at prompt position p sees keys 0..p (causal); each
// row is normalised over all the keys it sees, then rows are summed per key.
//
// Two passes over the keys, each a persistent warp-specialised kernel:
//   warp 0      TMA producer: key tiles into a ring of shared-memory stages, the
//               unit's observation queries into their own buffer;
//   warp 1      allocates tensor memory and issues the tcgen05 MMAs (one thread);
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulators (one row or key per
//               thread) and the softmax arithmetic.
//   Row-stats pass:  D[row][key] = Q_obs . K_tile^T (M = 128 rows per MMA tile, N =
//               256 keys, or 128 keys when M = 256); each thread owns one row and
//               keeps an online (max, sum of exp2) over the tile's keys, written
//               per (row, tile); a small kernel merges them into b_r = max +
//               log2(sum) per row.
//   Column pass: D[key][row] = K_tile . Q_obs^T (M = 128 keys, N = M rows rounded
//               up to 16); each thread owns one key and sums exp2(l * log2(e)/sqrt(d)
//               - b_r) over the rows: the per-key score.
// Both reductions stay inside a thread. Accumulators are double-buffered in tensor
// memory so the epilogue of one tile overlaps the MMAs of the next.
#include <algorithm>
#include <cudaTypedefs.h>

#include "kvc_internal.cuh"
#include "tc_common.cuh"

namespace kvc {
namespace {

constexpr int kEpiWarps = 16;                      // four per tensor-memory lane quarter
constexpr int kSplit = kEpiWarps / 4;              // column splits of a tile
constexpr int kTcThreads = 64 + 32 * kEpiWarps;    // producer, MMA, epilogue warps
constexpr int kTmemCols = 512;

template <int D, int PASS, int QT>
struct TcCfg {
  static constexpr int KB = D / 64;                     // 64-element K blocks
  static constexpr int QROWS = QT * 128;                 // staged query rows
  static constexpr int KROWS = PASS == 0 ? (QT == 1 ? 256 : 128) : 128;   // keys per tile
  static constexpr int QBYTES = QROWS * D * 2;
  static constexpr int KBYTES = KROWS * D * 2;
  // as many key stages as shared memory holds: the bytes in flight per SM set the
  // DRAM throughput a pass reaches
  static constexpr int STAGES = PASS == 0 ? (QT == 1 ? 3 : 5) : (QT == 1 ? 5 : 4);
  // tensor-memory accumulator buffers: two of 256 columns for the row-stats pass,
  // four of 128 columns for the column pass (two of 256 when M > 128)
  static constexpr int NBUF = (PASS == 1 && QT == 1) ? 4 : 2;
  static constexpr int BUFCOLS = 512 / NBUF;
  static constexpr int oQ = 0;
  static constexpr int oK = QBYTES;
  static constexpr int oBar = oK + STAGES * KBYTES;
  // full[S], empty[S], qfull, qempty, tfull[NBUF], tempty[NBUF], drain
  static constexpr int NBAR = 2 * STAGES + 3 + 2 * NBUF;
  static constexpr int oTmem = oBar + NBAR * 8;
  static constexpr int oBias = (oTmem + 16 + 15) / 16 * 16;
  static constexpr int BIASB = PASS == 1 ? 4 * 256 * 4 : 0;   // column pass: 4 bias copies
  static constexpr int total = oBias + BIASB + 1024;            // + alignment slack
  static_assert(total <= 232448, "fits the shared memory of one CTA");
  static_assert(QBYTES % 1024 == 0 && KBYTES % 1024 == 0, "1024-byte aligned tiles");
};

struct TcArgs {
  int n;          // keys per unit (prompt length)
  int ns;         // scored keys (n - alpha)
  int alpha;
  int M;          // rows per unit (g * alpha)
  int units;
  int tiles;      // tiles per unit
  float sl2;      // log2(e) / sqrt(d)
  float2* stats;  // row-stats pass: [unit][row][tile]
  const float* rowbias;   // column pass: [unit][row]
  float* scores;          // column pass: [unit][ns]
  unsigned* err;
};

template <int D, int PASS, int QT>
__global__ void __launch_bounds__(kTcThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                const TcArgs a) {
  using C = TcCfg<D, PASS, QT>;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t* sQ = dsm + C::oQ;
  uint8_t* sK = dsm + C::oK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + C::oBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* qfull = bars + 2 * C::STAGES;
  uint64_t* qempty = qfull + 1;
  uint64_t* tfull = qfull + 2;
  uint64_t* tempty = tfull + C::NBUF;
  uint64_t* drain = tempty + C::NBUF;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(dsm + C::oTmem);
  float* sbias = reinterpret_cast<float*>(dsm + C::oBias);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const long long total = (long long)a.units * a.tiles;
  const int it0 = (int)(blockIdx.x * total / gridDim.x);
  const int it1 = (int)((blockIdx.x + 1) * total / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { tc::mbar_init(&full[s], 1); tc::mbar_init(&empty[s], 1); }
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qempty, 1);
    for (int b = 0; b < C::NBUF; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], PASS == 0 ? kEpiWarps : 4);
    }
    tc::mbar_init(drain, 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmQ);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_holder;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      int cur = -1, nq = 0, issued = 0;
      for (int it = it0, k = 0; it < it1 && ok; ++it, ++k) {
        const int unit = it / a.tiles, tile = it % a.tiles;
        if (unit != cur) {
          if (nq > 0) ok = tc::mbar_wait(qempty, (uint32_t)((nq - 1) & 1), a.err, 8u);
          if (!ok) break;
          tc::mbar_expect_tx(qfull, (uint32_t)C::QBYTES);
          for (int kb = 0; kb < C::KB; ++kb)
            for (int qt = 0; qt < QT; ++qt)
              tc::tma_load_2d(sQ + kb * C::QROWS * 128 + qt * 128 * 128, &tmQ, kb * 64,
                              unit * a.M + qt * 128, qfull);
          ++nq;
          cur = unit;
        }
        const int s = k % C::STAGES, round = k / C::STAGES;
        if (round > 0) ok = tc::mbar_wait(&empty[s], (uint32_t)((round - 1) & 1), a.err, 8u);
        if (!ok) break;
        tc::mbar_expect_tx(&full[s], (uint32_t)C::KBYTES);
        uint8_t* dst = sK + s * C::KBYTES;
        for (int kb = 0; kb < C::KB; ++kb)
          for (int r = 0; r < C::KROWS / 128; ++r)
            tc::tma_load_2d(dst + kb * C::KROWS * 128 + r * 128 * 128, &tmK, kb * 64,
                            unit * a.n + tile * C::KROWS + r * 128, &full[s]);
        issued = k + 1;
      }
      // every copy this thread issued has landed before the CTA can leave (in the
      // normal case the MMA thread already waited for all of them)
      for (int k = std::max(0, issued - C::STAGES); k < issued; ++k)
        tc::mbar_wait(&full[k % C::STAGES], (uint32_t)((k / C::STAGES) & 1), a.err, 8u);
      if (nq > 0) tc::mbar_wait(qfull, (uint32_t)((nq - 1) & 1), a.err, 8u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc = PASS == 0 ? tc::idesc_bf16_f32(128, C::KROWS) : 0u;
      const int MP = (a.M + 15) / 16 * 16;
      const uint32_t idesc1 = tc::idesc_bf16_f32(128, MP);
      int cur = -1, nq = 0;
      for (int it = it0, k = 0; it < it1 && ok; ++it, ++k) {
        const int unit = it / a.tiles;
        const int s = k % C::STAGES, round = k / C::STAGES;
        ok = tc::mbar_wait(&full[s], (uint32_t)(round & 1), a.err, 16u);
        if (!ok) break;
        if (unit != cur) {
          ok = tc::mbar_wait(qfull, (uint32_t)(nq & 1), a.err, 16u);
          if (!ok) break;
          ++nq;
          cur = unit;
        }
        const int b = k % C::NBUF, rb = k / C::NBUF;
        if (rb > 0) ok = tc::mbar_wait(&tempty[b], (uint32_t)((rb - 1) & 1), a.err, 16u);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t sQa = tc::saddr(sQ), sKa = tc::saddr(sK + s * C::KBYTES);
        const uint32_t dcol = tbase + (uint32_t)(b * C::BUFCOLS);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int kb = kk / 4, kin = (kk % 4) * 32;
          if (PASS == 0) {
#pragma unroll
            for (int mt = 0; mt < QT; ++mt) {
              const uint64_t ad = tc::sw128_desc(sQa + kb * C::QROWS * 128 + mt * 128 * 128 + kin);
              const uint64_t bd = tc::sw128_desc(sKa + kb * C::KROWS * 128 + kin);
              tc::mma_bf16(dcol + mt * C::KROWS, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
          } else {
            const uint64_t ad = tc::sw128_desc(sKa + kb * C::KROWS * 128 + kin);
            const uint64_t bd = tc::sw128_desc(sQa + kb * C::QROWS * 128 + kin);
            tc::mma_bf16(dcol, ad, bd, idesc1, kk > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&tfull[b]);
        const bool last_of_unit = (it + 1 >= it1) || ((it + 1) / a.tiles != unit);
        if (last_of_unit) tc::mma_commit(qempty);
      }
      // every MMA issued here has completed before tensor memory is released
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0u, a.err, 16u);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int e = warp - 2;
    const int sub = warp & 3;                    // tensor-memory lane quarter
    const int row_in = sub * 32 + lane;          // row (pass 0) or key (pass 1) in the tile
    const uint32_t lane_addr = (uint32_t)(sub * 32) << 16;
    if (PASS == 0) {
      // every tile: warp e reads lane quarter e % 4 and column split e / 4
      const int split = e >> 2;
      for (int it = it0, k = 0; it < it1; ++it, ++k) {
        const int unit = it / a.tiles, tile = it % a.tiles;
        const int b = k % C::NBUF, rb = k / C::NBUF;
        if (ok) ok = tc::mbar_wait(&tfull[b], (uint32_t)(rb & 1), a.err, 32u);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
        const uint32_t tcol = tbase + lane_addr + (uint32_t)(b * C::BUFCOLS);
        constexpr int HC = C::KROWS / kSplit;     // columns of this split
        static_assert(HC % 32 == 0, "whole 32-column loads");
        const int key0 = tile * C::KROWS + split * HC;
        // only the tiles reaching the observation window need the causal / range mask
        const bool masked = key0 + HC > a.n - a.alpha;
#pragma unroll
        for (int mt = 0; mt < QT; ++mt) {
          const int r = mt * 128 + row_in;
          const int pos = a.n - a.alpha + (r % a.alpha);
          const int lim = min(a.n - 1, pos) - key0;   // last visible column of this split
          float m = -INFINITY, ssum = 0.f;
#pragma unroll
          for (int c0 = 0; c0 < HC; c0 += 32) {
            float v[32];
            tc::tmem_ld32(tcol + (uint32_t)(mt * C::KROWS + split * HC + c0), v);
            if (masked) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = (c0 + j <= lim) ? v[j] : -INFINITY;
            }
            float mx[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) mx[j] = fmaxf(fmaxf(v[j], v[j + 8]), fmaxf(v[j + 16], v[j + 24]));
            const float cm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            if (cm != -INFINITY) {
              const float cms = cm * a.sl2;
              if (cms > m) {
                ssum = (m == -INFINITY) ? 0.f : ssum * exp2f(m - cms);
                m = cms;
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                float x = fmaf(v[j], a.sl2, -m);
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(v[j]) : "f"(x));
              }
#pragma unroll
              for (int w = 16; w > 0; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) v[j] += v[j + w];
              ssum += v[0];
            }
          }
          if (ok && r < a.M)
            a.stats[((size_t)unit * a.M + r) * (kSplit * a.tiles) + kSplit * tile + split] =
                make_float2(m, ssum);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty[b]);
      }
    } else {
      // group gi = e / 4 (four warps, one per lane quarter) takes the tiles k with
      // k % NBUF == gi, all MP columns: no data crosses warps
      const int gi = e >> 2;
      const int MP = (a.M + 15) / 16 * 16;
      float* gbias = sbias + gi * 256;           // this group's negated row normalisers
      int cur = -1;
      if (gi < C::NBUF) {
        for (int it = it0 + gi, k = gi; it < it1; it += C::NBUF, k += C::NBUF) {
          const int unit = it / a.tiles, tile = it % a.tiles;
          if (unit != cur) {
            asm volatile("bar.sync %0, 128;" :: "r"(1 + gi) : "memory");
            for (int j = sub * 32 + lane; j < 256; j += 128)
              gbias[j] = j < a.M ? -a.rowbias[(size_t)unit * a.M + j] : -INFINITY;
            asm volatile("bar.sync %0, 128;" :: "r"(1 + gi) : "memory");
            cur = unit;
          }
          const int b = gi, rb = k / C::NBUF;
          if (ok) ok = tc::mbar_wait(&tfull[b], (uint32_t)(rb & 1), a.err, 32u);
          ok = __all_sync(0xffffffffu, ok);
          tc::fence_after_sync();
          const uint32_t tcol = tbase + lane_addr + (uint32_t)(b * C::BUFCOLS);
          float acc = 0.f;
#pragma unroll 1
          for (int c0 = 0; c0 < MP; c0 += 32) {
            float v[32];
            tc::tmem_ld32(tcol + (uint32_t)c0, v);
            const float4* nb4 = reinterpret_cast<const float4*>(gbias + c0);
            if (c0 + 32 <= a.M) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                const float4 nb = nb4[j / 4];
                v[j] = fmaf(v[j], a.sl2, nb.x);
                v[j + 1] = fmaf(v[j + 1], a.sl2, nb.y);
                v[j + 2] = fmaf(v[j + 2], a.sl2, nb.z);
                v[j + 3] = fmaf(v[j + 3], a.sl2, nb.w);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = (c0 + j < a.M) ? fmaf(v[j], a.sl2, gbias[c0 + j]) : -INFINITY;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(v[j]) : "f"(v[j]));
#pragma unroll
            for (int w = 16; w > 0; w >>= 1)
#pragma unroll
              for (int j = 0; j < w; ++j) v[j] += v[j + w];
            acc += v[0];
          }
          const int key = tile * C::KROWS + row_in;
          if (ok && key < a.ns) a.scores[(size_t)unit * a.ns + key] = acc;
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&tempty[b]);
        }
      }
    }
  }

  // teardown: every MMA this CTA issued has completed once the epilogue consumed
  // its last tile; on an error path, drain before releasing tensor memory
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 map over [rows][d] with a 64 x 128 box and 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, long long rows, int d) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int PASS, int QT>
cudaError_t launch_pass(const CUtensorMap& mk, const CUtensorMap& mq, const TcArgs& a,
                        cudaStream_t stream) {
  using C = TcCfg<D, PASS, QT>;
  static int n_sm[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!n_sm[dev]) {
    e = cudaFuncSetAttribute(score_tc_kernel<D, PASS, QT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::total);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    n_sm[dev] = n;
  }
  const long long items = (long long)a.units * a.tiles;
  const int grid = (int)std::min<long long>(n_sm[dev], items);
  if (grid < 1) return cudaSuccess;
  score_tc_kernel<D, PASS, QT><<<grid, kTcThreads, C::total, stream>>>(mk, mq, a);
  count_launches(1);
  return cudaGetLastError();
}

template <int D>
cudaError_t run_passes(const kvc_dims& d, const __nv_bfloat16* q_obs, const __nv_bfloat16* k,
                       float2* stats, float* rowbias, float* scores, unsigned* err,
                       cudaStream_t stream) {
  const int units = d.batch * d.n_kv_heads;
  const int n = d.prompt_len, alpha = d.obs_window;
  const int M = (d.n_q_heads / d.n_kv_heads) * alpha;
  CUtensorMap mk, mq;
  cudaError_t e;
  if ((e = make_map(&mk, k, (long long)units * n, D)) != cudaSuccess) return e;
  if ((e = make_map(&mq, q_obs, (long long)units * M, D)) != cudaSuccess) return e;
  TcArgs a{};
  a.n = n;
  a.ns = n - alpha;
  a.alpha = alpha;
  a.M = M;
  a.units = units;
  a.sl2 = 1.4426950408889634f / sqrtf((float)D);
  a.stats = stats;
  a.rowbias = rowbias;
  a.scores = scores;
  a.err = err;
  // row statistics over all n keys
  const int qt = M > 128 ? 2 : 1;
  const int kr0 = qt == 1 ? 256 : 128;
  a.tiles = (n + kr0 - 1) / kr0;
  const int tiles0 = a.tiles;
  e = qt == 1 ? launch_pass<D, 0, 1>(mk, mq, a, stream) : launch_pass<D, 0, 2>(mk, mq, a, stream);
  if (e != cudaSuccess) return e;
  e = launch_score_combine(stats, kSplit * tiles0, M, units, rowbias, stream);
  if (e != cudaSuccess) return e;
  // per-key column sums over the scored keys
  a.tiles = (a.ns + 127) / 128;
  const int qt1 = (M + 15) / 16 * 16 > 128 ? 2 : 1;
  return qt1 == 1 ? launch_pass<D, 1, 1>(mk, mq, a, stream) : launch_pass<D, 1, 2>(mk, mq, a, stream);
}

}  // namespace

// Scores of one layer on the tensor cores: stats, row normalisers and the per-key
// column sums (the same contract as the warp-level path).
cudaError_t launch_score_tc(const kvc_dims& d, const __nv_bfloat16* q_obs, const __nv_bfloat16* k,
                            float2* stats, float* rowbias, float* scores, unsigned* err,
                            cudaStream_t stream) {
  if (d.head_dim == 128) return run_passes<128>(d, q_obs, k, stats, rowbias, scores, err, stream);
  if (d.head_dim == 64) return run_passes<64>(d, q_obs, k, stats, rowbias, scores, err, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvc
