// score_tc.cu -- observation-window scores on the 5th-generation tensor cores, one
// cooperative persistent launch per layer.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2 "KV Cache Selection": every prompt key i < n - alpha is scored
// by the attention the last alpha ("instruction") tokens pay it; MiniKV §2 eq. (1):
// A = softmax(Q K^T / sqrt(d)). Per unit (sequence, kv head) the rows are the alpha
// observation queries of each of the g query heads sharing the kv head (M = g *
// alpha rows, M <= 256); a row at prompt position p sees keys 0..p (causal); each
// row is normalised over all the keys it sees, then rows are summed per key.
//
// Keys are cut into tiles of 256 (one shared-memory stage each); all units form one
// batch (the kernel takes units in batches of a.ubatch), two phases over its tiles:
//   row-stats phase  D[row][key] = Q_obs . K_tile^T, one MMA chain (M = 128 rows,
//                    N = 256 keys) per 128-row block into one of two tensor-memory
//                    buffers; every epilogue thread owns one row and one quarter of
//                    the 256 columns and keeps an online (max, sum of exp2) of the
//                    scaled logits; at the end of a unit the quarters are merged in
//                    shared memory, one partial per (unit, CTA) is written and the
//                    unit's arrival counter is raised;
//   column phase     D[key][row] = K_tile . Q_obs^T, one chain (M = 128 keys, N = M
//                    rows rounded up to 16) per half tile; once every CTA owning
//                    row-stats tiles of the unit has arrived (epilogue warps only
//                    wait: the producer and MMA warps already run ahead), the row
//                    normaliser b_r = max + log2(sum) is merged from the row's
//                    partials; each thread owns one key and a quarter of the rows and
//                    sums exp2(l * log2(e)/sqrt(d) - b_r); the quarters meet in shared
//                    memory (fixed order) into the key's score.
// The staged queries serve both phases of a unit. Roles: warp 0 TMA producer (key
// tiles into a ring of shared-memory stages, the unit's observation queries into
// their own buffer), warp 1 tensor-memory owner and MMA issuer (one thread), warps
// 2..17 epilogue, all sixteen on each accumulator buffer in turn (warp w reads the
// tensor-memory lane quarter w % 4; the four warps of a quarter split the columns),
// so that the MMAs of one buffer run while the other is reduced.
// Every wait is bounded; a wait that gives up sets a bit of the error word.
#include <algorithm>
#include <cudaTypedefs.h>

#include "kvc_internal.cuh"
#include "tc_common.cuh"

namespace kvc {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kTcThreads = 64 + 32 * kEpiWarps;    // producer, MMA, epilogue warps
constexpr int kTmemCols = 512;
constexpr int kBufCols = 256;                      // two accumulator buffers
constexpr int kKeys = 256;                         // keys per tile (one stage)
constexpr int kSmemLimit = 232448;                 // opt-in shared memory per CTA

enum : unsigned { kErrProducer = 8u, kErrMma = 16u, kErrEpilogue = 32u, kErrUnit = 64u };

template <int D, int QT>
struct TcCfg {
  static constexpr int KB = D / 64;                // 64-element K blocks
  static constexpr int QROWS = QT * 128;           // staged query rows
  static constexpr int QBYTES = QROWS * D * 2;
  static constexpr int KBYTES = kKeys * D * 2;
  static constexpr int QBUF = QT == 1 ? 2 : 1;     // query buffers
  // bias [256], column partials [2][4][128], row partials [4][QROWS]
  static constexpr int TAILB = 256 * 4 + 2 * 4 * 128 * 4 + 4 * QROWS * 8;
  static constexpr int FIT = (kSmemLimit - QBUF * QBYTES - TAILB - 2048) / KBYTES;
  static constexpr int STAGES = FIT > 8 ? 8 : FIT;   // key stages: bytes in flight per SM
  static constexpr int oQ = 0;
  static constexpr int oK = QBUF * QBYTES;
  static constexpr int oBar = oK + STAGES * KBYTES;
  // full[S], empty[S], qfull[QBUF], qempty[QBUF], tfull[2], tempty[2], drain
  static constexpr int NBAR = 2 * STAGES + 2 * QBUF + 4 + 1;
  static constexpr int oTmem = oBar + NBAR * 8;
  static constexpr int oBias = (oTmem + 16 + 15) / 16 * 16;   // [256] negated b_r
  static constexpr int oPart = oBias + 256 * 4;               // [2][4][128] column quarters
  static constexpr int oRow = oPart + 2 * 4 * 128 * 4;        // [4][QROWS] row partials
  static constexpr int total = oRow + 4 * QROWS * 8 + 1024;   // + alignment slack
  static_assert(STAGES >= 2, "at least two key stages");
  static_assert(NBAR <= 64, "barrier area");
  static_assert(total <= kSmemLimit, "fits the shared memory of one CTA");
  static_assert(QBYTES % 1024 == 0 && KBYTES % 1024 == 0, "1024-byte aligned tiles");
};

struct TcArgs {
  int n;          // keys per unit (prompt length)
  int ns;         // scored keys (n - alpha)
  int alpha;
  int M;          // rows per unit (g * alpha)
  int MP;         // M rounded up to 16 (N of the column-phase MMA)
  int units;
  int ubatch;     // units per batch; every batch must give each CTA a row-stats tile
                  // (a unit's wait counts the CTAs over its tiles, and a CTA
                  // without a tile of the batch would never arrive)
  int tiles0;     // 256-key tiles per unit, row-stats phase (all n keys)
  int tiles1;     // 256-key tiles per unit, column phase (the ns scored keys)
  int smax;       // partial slots per (unit, row)
  float sl2;      // log2(e) / sqrt(d)
  float2* stats;  // [unit][slot][row] partial (max, sum), one slot per CTA
  float* scores;  // [unit][ns]
  unsigned* gsync;  // [0] CTAs done, [1 + unit] arrivals; all zero between launches
  unsigned* err;
};

// Items [b, e) of `total` that CTA c of G owns, and the owner of item i.
struct Slice { long long b, e; };
__device__ __forceinline__ Slice slice_of(long long total, int c, int G) {
  return {total * c / G, total * (c + 1) / G};
}
__device__ __forceinline__ int owner_of(long long i, long long total, int G) {
  return (int)(((i + 1) * G + total - 1) / total) - 1;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until `*cnt` reaches `target` (acquire). One thread per group.
__device__ bool wait_count(const unsigned* cnt, unsigned target, unsigned* err) {
  if (ld_acquire(cnt) >= target) return true;
  const unsigned long long t0 = tc::gtimer();
  while (ld_acquire(cnt) < target) {
    if (tc::gtimer() - t0 > tc::kWaitNs) {
      if (err) atomicOr(err, kErrUnit);
      return false;
    }
  }
  return true;
}
// Count one arrival; the writes this CTA made before (ordered by a barrier with
// this thread) are visible to a thread whose acquire load sees the count.
__device__ __forceinline__ void arrive_release(unsigned* cnt) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" :: "l"(cnt) : "memory");
}

// (max, sum) merge of two partials of exp2 sums: M = max, S = s_a 2^(m_a - M) + ...
__device__ __forceinline__ float2 merge_ms(float2 p, float2 q) {
  if (q.y <= 0.f) return p;
  if (p.y <= 0.f) return q;
  const float m = fmaxf(p.x, q.x);
  return make_float2(m, fmaf(p.y, exp2f(p.x - m), q.y * exp2f(q.x - m)));
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// Unit of the item that follows item i of phase ph of batch j in this CTA's walk
// (per batch: its row-stats items, then its column items), or -1 at the end.
__device__ int next_unit(const TcArgs& a, int G, int cta, int nbatch, int j, int ph, long long i) {
  for (;;) {
    const int u0 = j * a.ubatch, nu = min(a.ubatch, a.units - u0);
    const int tiles = ph ? a.tiles1 : a.tiles0;
    const Slice sl = slice_of((long long)nu * tiles, cta, G);
    if (i + 1 < sl.e) return u0 + (int)((i + 1) / tiles);
    if (ph == 0) {
      ph = 1;
    } else {
      ph = 0;
      if (++j >= nbatch) return -1;
    }
    const int v0 = j * a.ubatch, nv = min(a.ubatch, a.units - v0);
    i = slice_of((long long)nv * (ph ? a.tiles1 : a.tiles0), cta, G).b - 1;
  }
}

template <int D, int QT>
__global__ void __launch_bounds__(kTcThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                const TcArgs a) {
  using C = TcCfg<D, QT>;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t* sQ = dsm + C::oQ;
  uint8_t* sK = dsm + C::oK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + C::oBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* qfull = bars + 2 * C::STAGES;
  uint64_t* qempty = qfull + C::QBUF;
  uint64_t* tfull = qempty + C::QBUF;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(dsm + C::oTmem);
  float* sbias = reinterpret_cast<float*>(dsm + C::oBias);
  float* spart = reinterpret_cast<float*>(dsm + C::oPart);
  float2* srow = reinterpret_cast<float2*>(dsm + C::oRow);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int nbatch = (a.units + a.ubatch - 1) / a.ubatch;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { tc::mbar_init(&full[s], 1); tc::mbar_init(&empty[s], 1); }
    for (int q = 0; q < C::QBUF; ++q) { tc::mbar_init(&qfull[q], 1); tc::mbar_init(&qempty[q], 1); }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], kEpiWarps);
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
  pdl_wait();      // the previous kernels' writes (keys, queries, scratch) are visible
  pdl_release();

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      int k = 0, nq = 0, qunit = -1;
      for (int j = 0; j < nbatch && ok; ++j) {
        const int u0 = j * a.ubatch, nu = min(a.ubatch, a.units - u0);
        for (int ph = 0; ph < 2 && ok; ++ph) {
          const int tiles = ph ? a.tiles1 : a.tiles0;
          const Slice sl = slice_of((long long)nu * tiles, cta, G);
          for (long long i = sl.b; i < sl.e && ok; ++i, ++k) {
            const int unit = u0 + (int)(i / tiles), tile = (int)(i % tiles);
            if (unit != qunit) {
              const int qb = nq % C::QBUF;
              if (nq >= C::QBUF)
                ok = tc::mbar_wait(&qempty[qb], (uint32_t)((nq / C::QBUF - 1) & 1), a.err,
                                   kErrProducer);
              if (!ok) break;
              tc::mbar_expect_tx(&qfull[qb], (uint32_t)C::QBYTES);
              uint8_t* q = sQ + qb * C::QBYTES;
              for (int kb = 0; kb < C::KB; ++kb)
                for (int qt = 0; qt < QT; ++qt)
                  tc::tma_load_2d(q + kb * C::QROWS * 128 + qt * 128 * 128, &tmQ, kb * 64,
                                  unit * a.M + qt * 128, &qfull[qb]);
              ++nq;
              qunit = unit;
            }
            const int s = k % C::STAGES, round = k / C::STAGES;
            if (round > 0)
              ok = tc::mbar_wait(&empty[s], (uint32_t)((round - 1) & 1), a.err, kErrProducer);
            if (!ok) break;
            tc::mbar_expect_tx(&full[s], (uint32_t)C::KBYTES);
            uint8_t* dst = sK + s * C::KBYTES;
            for (int kb = 0; kb < C::KB; ++kb)
              tc::tma_load_2d(dst + kb * kKeys * 128, &tmK, kb * 64, unit * a.n + tile * kKeys,
                              &full[s]);
          }
        }
      }
      // every copy issued here has landed before the CTA can leave (normally the
      // MMA thread already waited for all of them)
      for (int kk = max(0, k - C::STAGES); kk < k; ++kk)
        tc::mbar_wait(&full[kk % C::STAGES], (uint32_t)((kk / C::STAGES) & 1), a.err,
                      kErrProducer);
      for (int q = max(0, nq - C::QBUF); q < nq; ++q)
        tc::mbar_wait(&qfull[q % C::QBUF], (uint32_t)((q / C::QBUF) & 1), a.err, kErrProducer);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc0 = tc::idesc_bf16_f32(128, kKeys);
      const uint32_t idesc1 = tc::idesc_bf16_f32(128, a.MP);
      int k = 0, job = 0, nq = 0, qunit = -1, qb = 0;
      for (int j = 0; j < nbatch && ok; ++j) {
        const int u0 = j * a.ubatch, nu = min(a.ubatch, a.units - u0);
        for (int ph = 0; ph < 2 && ok; ++ph) {
          const int tiles = ph ? a.tiles1 : a.tiles0;
          const Slice sl = slice_of((long long)nu * tiles, cta, G);
          for (long long i = sl.b; i < sl.e && ok; ++i, ++k) {
            const int unit = u0 + (int)(i / tiles);
            const int s = k % C::STAGES, round = k / C::STAGES;
            ok = tc::mbar_wait(&full[s], (uint32_t)(round & 1), a.err, kErrMma);
            if (!ok) break;
            if (unit != qunit) {
              qb = nq % C::QBUF;
              ok = tc::mbar_wait(&qfull[qb], (uint32_t)((nq / C::QBUF) & 1), a.err, kErrMma);
              if (!ok) break;
              ++nq;
              qunit = unit;
            }
            const uint32_t sQa = tc::saddr(sQ + qb * C::QBYTES);
            const uint32_t sKa = tc::saddr(sK + s * C::KBYTES);
            // row-stats: one chain per 128-row block; column: one per 128-key half
            const int njobs = ph ? 2 : QT;
            for (int jb = 0; jb < njobs && ok; ++jb, ++job) {
              const int b = job & 1, rb = job >> 1;
              if (rb > 0) ok = tc::mbar_wait(&tempty[b], (uint32_t)((rb - 1) & 1), a.err, kErrMma);
              if (!ok) break;
              tc::fence_after_sync();
              const uint32_t dcol = tbase + (uint32_t)(b * kBufCols);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const int kb = kk / 4, kin = (kk % 4) * 32;
                if (ph == 0) {
                  const uint64_t ad =
                      tc::sw128_desc(sQa + kb * C::QROWS * 128 + jb * 128 * 128 + kin);
                  const uint64_t bd = tc::sw128_desc(sKa + kb * kKeys * 128 + kin);
                  tc::mma_bf16(dcol, ad, bd, idesc0, kk > 0 ? 1u : 0u);
                } else {
                  const uint64_t ad =
                      tc::sw128_desc(sKa + kb * kKeys * 128 + jb * 128 * 128 + kin);
                  const uint64_t bd = tc::sw128_desc(sQa + kb * C::QROWS * 128 + kin);
                  tc::mma_bf16(dcol, ad, bd, idesc1, kk > 0 ? 1u : 0u);
                }
              }
              tc::mma_commit(&tfull[b]);
            }
            if (!ok) break;
            tc::mma_commit(&empty[s]);
            if (next_unit(a, G, cta, nbatch, j, ph, i) != unit) tc::mma_commit(&qempty[qb]);
          }
        }
      }
      // every MMA issued here has completed before tensor memory is released
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0u, a.err, kErrMma);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int e = warp - 2;                      // 0 .. 15
    const int q = warp & 3;                      // tensor-memory lane quarter
    const int cq = e >> 2;                       // column quarter
    const int te = e * 32 + lane;                // thread within the epilogue
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    __shared__ int s_bad;                        // the wait for a unit gave up
    if (te == 0) s_bad = 0;
    int job = 0;
    auto acquire = [&](int b) {
      if (ok) ok = tc::mbar_wait(&tfull[b], (uint32_t)((job >> 1) & 1), a.err, kErrEpilogue);
      ok = __all_sync(0xffffffffu, ok);
      tc::fence_after_sync();
    };
    auto release = [&](int b) {
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[b]);
      ++job;
    };
    for (int j = 0; j < nbatch; ++j) {
      const int u0 = j * a.ubatch, nu = min(a.ubatch, a.units - u0);
      const long long tot0 = (long long)nu * a.tiles0;
      // ---------------------------------------------------- row-stats phase
      {
        const Slice sl = slice_of(tot0, cta, G);
        long long i = sl.b;
        while (i < sl.e) {
          const int ul = (int)(i / a.tiles0);
          const long long iend = min(sl.e, (long long)(ul + 1) * a.tiles0);
          float m[QT], z[QT];
#pragma unroll
          for (int mt = 0; mt < QT; ++mt) { m[mt] = -INFINITY; z[mt] = 0.f; }
          for (; i < iend; ++i) {
            const int key0 = (int)(i % a.tiles0) * kKeys + cq * 64;   // this thread's columns
            // only tiles reaching the observation window need the causal / range mask
            const bool masked = (int)(i % a.tiles0) * kKeys + kKeys > a.n - a.alpha;
#pragma unroll
            for (int mt = 0; mt < QT; ++mt) {
              const int b = job & 1;
              acquire(b);
              const int r = mt * 128 + q * 32 + lane;               // the row this thread owns
              const int pos = a.n - a.alpha + (r % a.alpha);        // its prompt position
              const int lim = min(a.n - 1, pos) - key0;             // last visible column
              const uint32_t tcol = tbase + lane_addr + (uint32_t)(b * kBufCols + cq * 64);
              // two 32-column chunks; the buffer is released once the last one is in
              // registers, so that the MMAs of job + 2 overlap its exponentials
              auto chunk = [&](const uint32_t (&rr)[32], int c0) {
                float v[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) v[jj] = __uint_as_float(rr[jj]);
                if (masked) {
#pragma unroll
                  for (int jj = 0; jj < 32; ++jj) v[jj] = (c0 + jj <= lim) ? v[jj] : -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                  mx[jj] = fmaxf(fmaxf(v[jj], v[jj + 8]), fmaxf(v[jj + 16], v[jj + 24]));
                const float cm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                if (cm != -INFINITY) {
                  const float cms = cm * a.sl2;
                  if (cms > m[mt]) {
                    z[mt] = (m[mt] == -INFINITY) ? 0.f : z[mt] * exp2f(m[mt] - cms);
                    m[mt] = cms;
                  }
#pragma unroll
                  for (int jj = 0; jj < 32; ++jj) {
                    const float x = fmaf(v[jj], a.sl2, -m[mt]);
                    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(v[jj]) : "f"(x));
                  }
#pragma unroll
                  for (int w = 16; w > 0; w >>= 1)
#pragma unroll
                    for (int jj = 0; jj < w; ++jj) v[jj] += v[jj + w];
                  z[mt] += v[0];
                }
              };
              {
                uint32_t rr[32];
                tc::tmem_ld32_async(tcol, rr);
                tc::tmem_wait_ld32(rr);
                chunk(rr, 0);
              }
              {
                uint32_t rr[32];
                tc::tmem_ld32_async(tcol + 32u, rr);
                tc::tmem_wait_ld32(rr);
                release(b);
                chunk(rr, 32);
              }
            }
          }
          // the column quarters of the unit merge into this CTA's partial (a quarter
          // without a visible key holds the empty partial), then the unit's counter
          // counts the CTA in
#pragma unroll
          for (int mt = 0; mt < QT; ++mt)
            srow[cq * C::QROWS + mt * 128 + q * 32 + lane] = make_float2(m[mt], z[mt]);
          named_bar(5, 32 * kEpiWarps);
          if (te < a.M) {
            float2 p = srow[te];
#pragma unroll
            for (int cc = 1; cc < 4; ++cc) p = merge_ms(p, srow[cc * C::QROWS + te]);
            const int cf = owner_of((long long)ul * a.tiles0, tot0, G);
            a.stats[((size_t)(u0 + ul) * a.smax + (cta - cf)) * a.M + te] = p;
          }
          named_bar(5, 32 * kEpiWarps);
          if (te == 0) arrive_release(a.gsync + 1 + u0 + ul);
        }
      }
      // ------------------------------------------------------- column phase
      {
        const Slice sl = slice_of((long long)nu * a.tiles1, cta, G);
        int cur = -1;
        for (long long i = sl.b; i < sl.e; ++i) {
          const int ul = (int)(i / a.tiles1), tile = (int)(i % a.tiles1);
          if (ul != cur) {
            // b_r of the unit's rows, merged from the partials of every CTA owning
            // row-stats tiles of the unit, once all of them have arrived
            const int cf = owner_of((long long)ul * a.tiles0, tot0, G);
            const int cl = owner_of((long long)(ul + 1) * a.tiles0 - 1, tot0, G);
            const int nct = cl - cf + 1;
            named_bar(5, 32 * kEpiWarps);
            if (te == 0 && ok && !wait_count(a.gsync + 1 + u0 + ul, (unsigned)nct, a.err))
              s_bad = 1;
            named_bar(5, 32 * kEpiWarps);
            ok = ok && s_bad == 0;
            if (te < 256) {
              float nb = -INFINITY;
              if (te < a.M) {
                const float2* st = a.stats + (size_t)(u0 + ul) * a.smax * a.M + te;
                // all loads of a round in flight at once: one L2 round trip per 24 CTAs
                float2 p = make_float2(-INFINITY, 0.f);
                for (int s0 = 0; s0 < nct; s0 += 24) {
                  float2 v[24];
#pragma unroll
                  for (int c = 0; c < 24; ++c)
                    v[c] = s0 + c < nct ? __ldcg(st + (size_t)(s0 + c) * a.M)
                                        : make_float2(-INFINITY, 0.f);
#pragma unroll
                  for (int c = 0; c < 24; ++c) p = merge_ms(p, v[c]);
                }
                nb = -(p.x + log2f(p.y));
              }
              sbias[te] = nb;
            }
            named_bar(5, 32 * kEpiWarps);
            cur = ul;
          }
#pragma unroll 1
          for (int kt = 0; kt < 2; ++kt) {
            const int b = job & 1;
            float* part = spart + (b * 4) * 128;   // [4][128] by the buffer's parity
            acquire(b);
            const uint32_t tcol = tbase + lane_addr + (uint32_t)(b * kBufCols);
            // rows in chunks of 32: chunks cq and cq + 4 (rows >= M carry the bias
            // -inf; columns >= MP of a last partial chunk were not written and are
            // masked); the buffer is released once the last chunk is in registers
            float acc = 0.f;
            auto chunk = [&](const uint32_t (&rr)[32], int c0) {
              float v[32];
              const float4* nb4 = reinterpret_cast<const float4*>(sbias + c0);
              if (c0 + 32 <= a.MP) {
#pragma unroll
                for (int jj = 0; jj < 32; jj += 4) {
                  const float4 nb = nb4[jj / 4];
                  v[jj] = fmaf(__uint_as_float(rr[jj]), a.sl2, nb.x);
                  v[jj + 1] = fmaf(__uint_as_float(rr[jj + 1]), a.sl2, nb.y);
                  v[jj + 2] = fmaf(__uint_as_float(rr[jj + 2]), a.sl2, nb.z);
                  v[jj + 3] = fmaf(__uint_as_float(rr[jj + 3]), a.sl2, nb.w);
                }
              } else {
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                  v[jj] = (c0 + jj < a.MP) ? fmaf(__uint_as_float(rr[jj]), a.sl2, sbias[c0 + jj])
                                           : -INFINITY;
              }
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(v[jj]) : "f"(v[jj]));
#pragma unroll
              for (int w = 16; w > 0; w >>= 1)
#pragma unroll
                for (int jj = 0; jj < w; ++jj) v[jj] += v[jj + w];
              acc += v[0];
            };
            const int c0a = cq * 32, c0b = cq * 32 + 128;
            if (c0b < a.MP) {
              uint32_t rr[32];
              tc::tmem_ld32_async(tcol + (uint32_t)c0a, rr);
              tc::tmem_wait_ld32(rr);
              chunk(rr, c0a);
              tc::tmem_ld32_async(tcol + (uint32_t)c0b, rr);
              tc::tmem_wait_ld32(rr);
              release(b);
              chunk(rr, c0b);
            } else if (c0a < a.MP) {
              uint32_t rr[32];
              tc::tmem_ld32_async(tcol + (uint32_t)c0a, rr);
              tc::tmem_wait_ld32(rr);
              release(b);
              chunk(rr, c0a);
            } else {
              release(b);
            }
            // the four row quarters of the key meet in shared memory, added in a
            // fixed order (the buffer of job j is rewritten by job j + 2 only after
            // its reader passed the barrier of job j + 1)
            part[cq * 128 + q * 32 + lane] = acc;
            named_bar(1 + q, 128);
            if (cq == 0) {
              const int key = tile * kKeys + kt * 128 + q * 32 + lane;
              if (ok && key < a.ns)
                a.scores[(size_t)(u0 + ul) * a.ns + key] =
                    ((part[q * 32 + lane] + part[128 + q * 32 + lane]) +
                     part[256 + q * 32 + lane]) + part[384 + q * 32 + lane];
            }
          }
        }
      }
    }
  }

  // teardown: every MMA this CTA issued has completed once the epilogue consumed
  // its last tile; on an error path the MMA thread drained before this point
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, kTmemCols);
  }
  // the last CTA to finish returns the counters to zero for the next launch
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.gsync, 1u) == (unsigned)G - 1) {
      for (int u = 0; u < a.units; ++u) a.gsync[1 + u] = 0u;
      a.gsync[0] = 0u;
      __threadfence();
    }
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

// 2-D bf16 map over [rows][d] with a 64 x box_rows box and 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, long long rows, int d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int QT>
cudaError_t launch_fused(const CUtensorMap& mk, const CUtensorMap& mq, const TcArgs& a,
                         cudaStream_t stream) {
  using C = TcCfg<D, QT>;
  static int max_ctas[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!max_ctas[dev]) {
    e = cudaFuncSetAttribute(score_tc_kernel<D, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::total);
    if (e != cudaSuccess) return e;
    int n_sm = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, score_tc_kernel<D, QT>, kTcThreads,
                                                      C::total);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    max_ctas[dev] = n_sm * per_sm;
  }
  // every CTA owns row-stats tiles of the first (largest) batch
  const long long items0 = (long long)std::min(a.ubatch, a.units) * a.tiles0;
  const int grid = (int)std::min<long long>(max_ctas[dev], items0);
  if (grid < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = C::total;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: waits across CTAs are safe
  at[0].val.cooperative = 1;
  at[1] = pdl_attr();
  cfg.attrs = at;
  // a driver that does not take the dependent-launch attribute on a cooperative
  // launch gets the plain cooperative launch from then on
  static bool no_pdl = false;
  cfg.numAttrs = no_pdl ? 1 : 2;
  e = cudaLaunchKernelEx(&cfg, score_tc_kernel<D, QT>, mk, mq, a);
  if (e != cudaSuccess && !no_pdl) {
    cudaGetLastError();
    no_pdl = true;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, score_tc_kernel<D, QT>, mk, mq, a);
  }
  if (e != cudaSuccess) return e;
  count_launches(1);
  return cudaSuccess;
}

template <int D>
cudaError_t run_fused(const kvc_dims& d, const __nv_bfloat16* q_obs, const __nv_bfloat16* k,
                      float2* stats, unsigned* gsync, float* scores, unsigned* err,
                      cudaStream_t stream) {
  const int units = d.batch * d.n_kv_heads;
  const int n = d.prompt_len, alpha = d.obs_window;
  const int M = (d.n_q_heads / d.n_kv_heads) * alpha;
  CUtensorMap mk, mq;
  cudaError_t e;
  if ((e = make_map(&mk, k, (long long)units * n, D, kKeys)) != cudaSuccess) return e;
  if ((e = make_map(&mq, q_obs, (long long)units * M, D, 128)) != cudaSuccess) return e;
  TcArgs a{};
  a.n = n;
  a.ns = n - alpha;
  a.alpha = alpha;
  a.M = M;
  a.MP = (M + 15) / 16 * 16;
  a.units = units;
  // one batch: a CTA's key tiles stream in at the same pace from L2 or DRAM, so
  // batches sized for L2 would only add phase switches (each a pipeline drain and
  // a wait for the slowest CTA's row statistics)
  a.ubatch = units;
  a.tiles0 = (n + kKeys - 1) / kKeys;
  a.tiles1 = (a.ns + kKeys - 1) / kKeys;
  a.smax = (int)score_stat_chunks(n);
  a.sl2 = 1.4426950408889634f / sqrtf((float)D);
  a.stats = stats;
  a.scores = scores;
  a.gsync = gsync;
  a.err = err;
  return M > 128 ? launch_fused<D, 2>(mk, mq, a, stream) : launch_fused<D, 1>(mk, mq, a, stream);
}

}  // namespace

// Scores of one layer on the tensor cores: row statistics, their merge into row
// normalisers and the per-key column sums, in one launch.
cudaError_t launch_score_tc(const kvc_dims& d, const __nv_bfloat16* q_obs, const __nv_bfloat16* k,
                            float2* stats, unsigned* gsync, float* scores, unsigned* err,
                            cudaStream_t stream) {
  if (d.head_dim == 128) return run_fused<128>(d, q_obs, k, stats, gsync, scores, err, stream);
  if (d.head_dim == 64) return run_fused<64>(d, q_obs, k, stats, gsync, scores, err, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvc
