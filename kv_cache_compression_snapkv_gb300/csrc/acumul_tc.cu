// acumul_tc.cu -- full-prompt cumulated attention (MiniKV's A_cumul) on the
// 5th-generation tensor cores, one persistent launch per layer.
//
// MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
// Cache, §4.3 "selective flash-attention" and Figure 9; Algorithm 1 (prefill: the
// heavy hitters are chosen from A_cumul). Every prompt query attends causally to
// the prompt keys; the keys are visited in blocks of 128 from the first on, each
// visit raises every row's running maximum to the block's, and the tile
// P = exp(S - running maximum) is added column by column into A_cumul. Rows are
// never normalised. The g query heads sharing a kv head add into one score per
// kv head; only the columns [0, n - alpha) are kept (the observation window
// stays whole), so key blocks past them are not visited.
//
// Work: an item is (unit = (sequence, kv head), row block) with a row block of
// P = 128 / g consecutive prompt positions for each of the g query heads (128
// rows, head-major). Items are dealt to the CTAs longest first in snake order.
// Per item the query tile stays in shared memory while its key tiles 0..T-1
// stream through a ring of stages; for every key tile the MMA thread issues
//   D1[row][key] = Q . K^T   (the running row maxima), and
//   D2[key][row] = K . Q^T   (the column sums, one key per thread),
// each 128 x 128 in tensor memory. A CTA runs two items at once, one per
// epilogue group of eight warps: even items of its list go to group 0, odd ones
// to group 1, and the producer and MMA thread interleave the two items' tiles
// (group 0, group 1, group 0, ...; one group alone once the other has run out),
// so that one group's epilogue overlaps the other's MMAs. Group x owns tensor
// memory columns [256 x, 256 x + 256) and query buffer x. A group takes each tile
// in two column halves: the row maxima of D1 are merged in shared memory into the
// running maxima, then each thread sums exp2(D2 * log2(e)/sqrt(d) - m_row) over
// its half of the rows for its key; the halves meet in shared memory and one
// atomic add per key lands the item's contribution in the score row (zeroed
// before the launch).
//
// Roles: warp 0 TMA producer, warp 1 tensor-memory owner and MMA issuer, warps
// 2..17 epilogue (two groups). Every wait is bounded; a wait that gives up sets a
// bit of the error word and the CTA winds down without further waits.
#include <algorithm>
#include <cudaTypedefs.h>

#include "kvc_internal.cuh"
#include "tc_common.cuh"

namespace kvc {
namespace {

constexpr int kAcGroupWarps = 8;                    // epilogue warps per group
constexpr int kAcThreads = 64 + 2 * 32 * kAcGroupWarps;   // producer, MMA, two groups
constexpr int kAcTmemCols = 512;
constexpr int kAcSmemLimit = 232448;                // opt-in shared memory per CTA

enum : unsigned { kErrAcProducer = 128u, kErrAcMma = 256u, kErrAcEpilogue = 512u };

template <int D>
struct AcCfg {
  static constexpr int KB = D / 64;                 // 64-element K blocks
  static constexpr int TBYTES = 128 * D * 2;        // one 128-row bf16 tile
  static constexpr int QBUF = 2;                    // one query buffer per group
  static constexpr int FIT = (kAcSmemLimit - QBUF * TBYTES - 8192) / TBYTES;
  static constexpr int STAGES = FIT > 6 ? 6 : FIT;
  static constexpr int oQ = 0;
  static constexpr int oK = QBUF * TBYTES;
  static constexpr int oBar = oK + STAGES * TBYTES;
  // full[S], empty[S], qfull[QBUF], qempty[QBUF], tfull[2], tempty[2], drain
  static constexpr int NBAR = 2 * STAGES + 2 * QBUF + 2 * 2 + 1;
  static constexpr int oTmem = oBar + NBAR * 8;
  // per group: [2 halves][128] row maxima, [128] -m per row, [128] half sums
  static constexpr int oMax = (oTmem + 16 + 15) / 16 * 16;
  static constexpr int oNegM = oMax + 2 * 2 * 128 * 4;
  static constexpr int oPart = oNegM + 2 * 128 * 4;
  static constexpr int total = oPart + 2 * 128 * 4 + 1024;   // + alignment slack
  static_assert(STAGES >= 2, "at least two key stages");
  static_assert(total <= kAcSmemLimit, "fits the shared memory of one CTA");
  static_assert(TBYTES % 1024 == 0, "1024-byte aligned tiles");
};

struct AcArgs {
  int n;           // prompt length
  int ns;          // scored keys (n - alpha)
  int g;           // query heads per kv head
  int P;           // positions per row block (128 / g)
  int Hq, Hk;
  int units;       // batch * Hk
  int rblocks;     // row blocks per unit
  long long items; // units * rblocks
  float sl2;       // log2(e) / sqrt(d)
  unsigned long long* fx;   // [unit][ns] fixed-point column sums, zero before the launch
  unsigned* err;
};

// The j-th item of CTA c (of G): items are dealt in snake order, c, 2G-1-c,
// 2G+c, 4G-1-c, ...; the sequence is increasing, so the first index past the end
// ends the CTA's list.
__device__ __forceinline__ long long item_at(int c, int j, int G) {
  const long long base = (long long)(j >> 1) * 2 * G;
  return base + ((j & 1) ? (2 * G - 1 - c) : c);
}

struct Item {
  int unit, p0, T;
};
// Item i: longest first (the last row blocks), units interleaved. T = key tiles
// visited: through the row block's last position, at most through the last
// scored key.
__device__ __forceinline__ Item item_of(long long i, const AcArgs& a) {
  Item it;
  it.unit = (int)(i % a.units);
  const int rb = a.rblocks - 1 - (int)(i / a.units);
  it.p0 = rb * a.P;
  const int last = min(it.p0 + a.P, a.n) - 1;
  it.T = min(last, a.ns - 1) / 128 + 1;
  return it;
}

// The interleaved tile order of the producer and the MMA thread: group x works
// through items x, x + 2, x + 4, ... of the CTA's list; turns alternate between
// the groups while both have tiles left.
struct Cursor {
  Item it;
  int t;       // next tile of the current item
  int jn;      // next list position of this group
  bool live;
};
__device__ __forceinline__ void cursor_next_item(Cursor& c, int cta, int G, const AcArgs& a) {
  const long long i = item_at(cta, c.jn, G);
  c.live = i < a.items;
  if (c.live) c.it = item_of(i, a);
  c.t = 0;
  c.jn += 2;
}

// The items' contributions to a score are added as 64-bit fixed-point integers
// (units of 2^-40): integer addition does not depend on the order the items
// arrive in, so the scores (and the kept sets) are the same on every run. A
// score is at most g * n <= 16 * 2^19 (2^23), far inside the 2^63 / 2^40 range.
constexpr float kFixScale = 1099511627776.f;   // 2^40
__device__ __forceinline__ void add_fixed(unsigned long long* dst, float v) {
  atomicAdd(dst, __float2ull_rn(v * kFixScale));
}
__global__ void fixed_to_float_kernel(const unsigned long long* __restrict__ fx, float* __restrict__ out,
                                      long long count) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
       i += (long long)gridDim.x * blockDim.x)
    out[i] = __ull2float_rn(fx[i]) * (1.f / kFixScale);
}
cudaError_t fixed_to_float(const unsigned long long* fx, float* out, long long count,
                           cudaStream_t stream) {
  fixed_to_float_kernel<<<(int)std::min<long long>(1024, (count + 255) / 256), 256, 0, stream>>>(
      fx, out, count);
  count_launches(1);
  return cudaGetLastError();
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kAcThreads, 1)
acumul_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                 const AcArgs a) {
  using C = AcCfg<D>;
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
  float* smax = reinterpret_cast<float*>(dsm + C::oMax);
  float* snegm = reinterpret_cast<float*>(dsm + C::oNegM);
  float* spart = reinterpret_cast<float*>(dsm + C::oPart);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { tc::mbar_init(&full[s], 1); tc::mbar_init(&empty[s], 1); }
    for (int q = 0; q < C::QBUF; ++q) { tc::mbar_init(&qfull[q], 1); tc::mbar_init(&qempty[q], 1); }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], kAcGroupWarps);
    }
    tc::mbar_init(drain, 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmQ);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, kAcTmemCols);
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
      int k = 0, nq0 = 0, nq1 = 0, turn = 0;
      Cursor c0, c1;                // kept in registers: selected by value, written back
      c0.jn = 0; cursor_next_item(c0, cta, G, a);
      c1.jn = 1; cursor_next_item(c1, cta, G, a);
      while (ok && (c0.live || c1.live)) {
        const int x = (turn ? c1.live : c0.live) ? turn : turn ^ 1;
        Cursor c = x ? c1 : c0;
        const int nqx = x ? nq1 : nq0;
        if (c.t == 0) {
          // the row block: P positions of each of the g query heads, head-major
          if (nqx > 0)
            ok = tc::mbar_wait(&qempty[x], (uint32_t)((nqx - 1) & 1), a.err, kErrAcProducer);
          if (!ok) break;
          tc::mbar_expect_tx(&qfull[x], (uint32_t)C::TBYTES);
          uint8_t* q = sQ + x * C::TBYTES;
          const int b = c.it.unit / a.Hk, hk = c.it.unit % a.Hk;
          for (int hh = 0; hh < a.g; ++hh) {
            const int row = ((b * a.Hq + hk * a.g + hh) * a.n) + c.it.p0;
            for (int kb = 0; kb < C::KB; ++kb)
              tc::tma_load_2d(q + kb * 128 * 128 + hh * a.P * 128, &tmQ, kb * 64, row,
                              &qfull[x]);
          }
          if (x) ++nq1; else ++nq0;
        }
        const int s = k % C::STAGES, round = k / C::STAGES;
        if (round > 0)
          ok = tc::mbar_wait(&empty[s], (uint32_t)((round - 1) & 1), a.err, kErrAcProducer);
        if (!ok) break;
        tc::mbar_expect_tx(&full[s], (uint32_t)C::TBYTES);
        uint8_t* dst = sK + s * C::TBYTES;
        for (int kb = 0; kb < C::KB; ++kb)
          tc::tma_load_2d(dst + kb * 128 * 128, &tmK, kb * 64, c.it.unit * a.n + c.t * 128,
                          &full[s]);
        ++k;
        if (++c.t == c.it.T) cursor_next_item(c, cta, G, a);
        if (x) c1 = c; else c0 = c;
        turn = x ^ 1;
      }
      // every copy issued here has landed before the CTA can leave
      for (int kk = max(0, k - C::STAGES); kk < k; ++kk)
        tc::mbar_wait(&full[kk % C::STAGES], (uint32_t)((kk / C::STAGES) & 1), a.err,
                      kErrAcProducer);
      if (nq0 > 0) tc::mbar_wait(&qfull[0], (uint32_t)((nq0 - 1) & 1), a.err, kErrAcProducer);
      if (nq1 > 0) tc::mbar_wait(&qfull[1], (uint32_t)((nq1 - 1) & 1), a.err, kErrAcProducer);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 128);
      int k = 0, nq0 = 0, nq1 = 0, kx0 = 0, kx1 = 0, turn = 0;
      Cursor c0, c1;                // kept in registers: selected by value, written back
      c0.jn = 0; cursor_next_item(c0, cta, G, a);
      c1.jn = 1; cursor_next_item(c1, cta, G, a);
      while (ok && (c0.live || c1.live)) {
        const int x = (turn ? c1.live : c0.live) ? turn : turn ^ 1;
        Cursor c = x ? c1 : c0;
        const int kxx = x ? kx1 : kx0;
        if (c.t == 0) {
          ok = tc::mbar_wait(&qfull[x], (uint32_t)((x ? nq1 : nq0) & 1), a.err, kErrAcMma);
          if (!ok) break;
          if (x) ++nq1; else ++nq0;
        }
        const int s = k % C::STAGES;
        ok = tc::mbar_wait(&full[s], (uint32_t)((k / C::STAGES) & 1), a.err, kErrAcMma);
        if (!ok) break;
        if (kxx > 0) ok = tc::mbar_wait(&tempty[x], (uint32_t)((kxx - 1) & 1), a.err, kErrAcMma);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t sQa = tc::saddr(sQ + x * C::TBYTES);
        const uint32_t sKa = tc::saddr(sK + s * C::TBYTES);
        const uint32_t d1 = tbase + (uint32_t)(x * 256), d2 = d1 + 128u;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int kb = kk / 4, kin = (kk % 4) * 32;
          const uint64_t qd = tc::sw128_desc(sQa + kb * 128 * 128 + kin);
          const uint64_t kd = tc::sw128_desc(sKa + kb * 128 * 128 + kin);
          tc::mma_bf16(d1, qd, kd, idesc, kk > 0 ? 1u : 0u);   // [row][key]
          tc::mma_bf16(d2, kd, qd, idesc, kk > 0 ? 1u : 0u);   // [key][row]
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&tfull[x]);
        ++k;
        if (x) ++kx1; else ++kx0;
        if (++c.t == c.it.T) {
          tc::mma_commit(&qempty[x]);
          cursor_next_item(c, cta, G, a);
        }
        if (x) c1 = c; else c0 = c;
        turn = x ^ 1;
      }
      // every MMA issued here has completed before tensor memory is released
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0u, a.err, kErrAcMma);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int x = (warp - 2) / kAcGroupWarps;    // group
    const int quarter = warp & 3;                 // tensor-memory lane quarter
    const int half = ((warp - 2) % kAcGroupWarps) >> 2;   // column half of each tile
    const int r = quarter * 32 + lane;            // row of D1 / key of D2 this thread reads
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int ET = 32 * kAcGroupWarps;
    float* gmax = smax + x * 256;
    float* gnegm = snegm + x * 128;
    float* gpart = spart + x * 128;
    int k = 0;                                    // tiles of this group so far
    for (int j = x;; j += 2) {
      const long long i = item_at(cta, j, G);
      if (i >= a.items) break;
      const Item it = item_of(i, a);
      const int pos_r = it.p0 + r % a.P;          // prompt position of row r
      const bool row_ok = pos_r < a.n;
      float m = -INFINITY;                        // running maximum of row r (log2 units)
      for (int t = 0; t < it.T; ++t, ++k) {
        if (ok) ok = tc::mbar_wait(&tfull[x], (uint32_t)(k & 1), a.err, kErrAcEpilogue);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
        const int key0 = t * 128;
        // does some row miss some key of this tile (causal diagonal, or rows past n)?
        const bool masked = key0 + 127 > it.p0 || it.p0 + a.P > a.n;
        // --- row maxima: row r, columns [64 half, 64 half + 64) of D1
        const uint32_t c1 = tbase + lane_addr + (uint32_t)(x * 256 + half * 64);
        float pm = -INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          float v[32];
          tc::tmem_ld32(c1 + (uint32_t)c0, v);
          if (masked) {
            const int lim = row_ok ? pos_r - (key0 + half * 64 + c0) : -1;   // last visible column
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) v[jj] = jj <= lim ? v[jj] : -INFINITY;
          }
          float ma = v[0], mb = v[16];
#pragma unroll
          for (int jj = 1; jj < 15; jj += 2) {
            ma = max3(ma, v[jj], v[jj + 1]);
            mb = max3(mb, v[jj + 16], v[jj + 17]);
          }
          pm = max3(pm, max3(ma, v[15], v[31]), mb);
        }
        gmax[half * 128 + r] = pm;
        named_bar(1 + x, ET);
        const float mt = fmaxf(gmax[r], gmax[128 + r]);
        if (mt != -INFINITY) m = fmaxf(m, mt * a.sl2);
        if (half == 0) gnegm[r] = -m;
        named_bar(1 + x, ET);
        // --- column sums: key r, rows [64 half, 64 half + 64) of D2
        const uint32_t c2 = tbase + lane_addr + (uint32_t)(x * 256 + 128 + half * 64);
        const float* nm = gnegm + half * 64;
        const int key = key0 + r;
        float acc = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          float v[32];
          tc::tmem_ld32(c2 + (uint32_t)c0, v);
          if (!masked) {
            // paired fp32 arithmetic: two logits per instruction
            const float4* nm4 = reinterpret_cast<const float4*>(nm + c0);
            const float2 s2 = make_float2(a.sl2, a.sl2);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
              const float4 b4 = nm4[jj / 4];
              const float2 lo = __ffma2_rn(make_float2(v[jj], v[jj + 1]), s2,
                                           make_float2(b4.x, b4.y));
              const float2 hi = __ffma2_rn(make_float2(v[jj + 2], v[jj + 3]), s2,
                                           make_float2(b4.z, b4.w));
              v[jj] = lo.x; v[jj + 1] = lo.y; v[jj + 2] = hi.x; v[jj + 3] = hi.y;
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int row = half * 64 + c0 + jj;
              const int pos = it.p0 + row % a.P;
              v[jj] = (pos < a.n && key <= pos) ? fmaf(v[jj], a.sl2, nm[c0 + jj]) : -INFINITY;
            }
          }
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(v[jj]) : "f"(v[jj]));
          float2 sum[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            sum[q] = __fadd2_rn(make_float2(v[2 * q], v[2 * q + 1]),
                                make_float2(v[2 * q + 16], v[2 * q + 17]));
#pragma unroll
          for (int w = 4; w > 0; w >>= 1)
#pragma unroll
            for (int q = 0; q < w; ++q) sum[q] = __fadd2_rn(sum[q], sum[q + w]);
          acc += sum[0].x + sum[0].y;
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty[x]);
        // the halves meet in shared memory; one atomic add per key
        if (half == 1) gpart[r] = acc;
        named_bar(1 + x, ET);
        if (half == 0 && ok && key < a.ns) add_fixed(a.fx + (size_t)it.unit * a.ns + key,
                                                    acc + gpart[r]);
      }
    }
  }

  // teardown: every MMA this CTA issued has completed once the epilogue consumed
  // its last tile; on an error path the MMA thread drained before this point
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, kAcTmemCols);
  }
}

// ======================================================================
// Selective flash-attention with its attention output (MiniKV §4.3, Figure 9:
// the kernel returns X_O, the weighted sum of the values, beside A_cumul).
//
// Same items, key tiles and A_cumul arithmetic as above, one item at a time per
// CTA with one epilogue group of eight warps. Per key tile the MMA thread issues
//   S1[row][key] = Q . K^T and S2[key][row] = K . Q^T   (tensor memory), then,
// once the epilogue has written P, O[row][d] += P . V    (tensor memory),
// where P[row][key] = exp2(S1 * log2(e)/sqrt(d) - r_row) is stored as bf16 in
// shared memory (128-byte swizzled, K-major: the A operand) and V is read from
// its TMA tile in place (MN-major B operand: rows of the tile run along K). The
// reference r_row of P is the running row maximum, raised only when the maximum
// passes it by more than kXoSlack (log2 units): then O and the row sum l are
// rescaled in place by exp2(r_old - r_new). A_cumul keeps the exact running
// maximum, as above. At the end of an item X_O = O / l (l summed in fp32 over the
// unrounded P) is written as bf16. Key tiles run through each row block's last
// position (X_O needs every causal key; only keys < n - alpha add to A_cumul).
//
// Tensor memory: S1 at columns [0, 128), S2 at [128, 256), O at [256, 256 + d).
// Roles: warp 0 TMA producer (K and V tiles of a stage, the query tile), warp 1
// tensor-memory owner and MMA issuer, warps 2..9 epilogue (lane quarter = warp %
// 4, column half = (warp - 2) / 4). Every wait is bounded.
constexpr int kXoEpiWarps = 8;
constexpr int kXoThreads = 64 + 32 * kXoEpiWarps;
constexpr float kXoSlack = 8.f;

template <int D>
struct XoCfg {
  static constexpr int KB = D / 64;                 // 64-element K blocks of Q, K, V
  static constexpr int TBYTES = 128 * D * 2;        // one 128-row bf16 tile
  static constexpr int PBYTES = 128 * 128 * 2;      // P: 128 rows x 128 keys bf16
  static constexpr int STAGES = 2;                  // K + V tiles per stage
  static constexpr int oQ = 0;
  static constexpr int oP = oQ + TBYTES;
  static constexpr int oKV = oP + PBYTES;           // stage s: K at +2s TBYTES, V after it
  static constexpr int oBar = oKV + STAGES * 2 * TBYTES;
  // full[S], empty[S], qfull, qempty, sfull, sfree, pfull, pvdone, drain
  static constexpr int NBAR = 2 * STAGES + 7;
  static constexpr int oTmem = oBar + NBAR * 8;
  static constexpr int oMax = (oTmem + 16 + 15) / 16 * 16;   // [2][128] half-row maxima
  static constexpr int oNegM = oMax + 2 * 128 * 4;           // [128] -m per row
  static constexpr int oPart = oNegM + 128 * 4;              // [128] half column sums
  static constexpr int oL = oPart + 128 * 4;                 // [2][128] half-row sums of P
  static constexpr int total = oL + 2 * 128 * 4 + 1024;      // + alignment slack
  static_assert(total <= kAcSmemLimit, "fits the shared memory of one CTA");
  static_assert(TBYTES % 1024 == 0 && PBYTES % 1024 == 0, "1024-byte aligned tiles");
};

struct XoArgs {
  AcArgs a;
  __nv_bfloat16* x_out;   // [B][Hq][n][d]
  int d;
};

// Keys visited by an item for its attention output: through its last position.
__device__ __forceinline__ int xo_tiles(const Item& it, const AcArgs& a) {
  return (min(it.p0 + a.P, a.n) - 1) / 128 + 1;
}

template <int D>
__global__ void __launch_bounds__(kXoThreads, 1)
acumul_xo_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmQ, const XoArgs xa) {
  using C = XoCfg<D>;
  const AcArgs& a = xa.a;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~uintptr_t(1023));
  uint8_t* sQ = dsm + C::oQ;
  uint8_t* sP = dsm + C::oP;
  uint8_t* sKV = dsm + C::oKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + C::oBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* qfull = bars + 2 * C::STAGES;
  uint64_t* qempty = qfull + 1;
  uint64_t* sfull = qfull + 2;
  uint64_t* sfree = qfull + 3;
  uint64_t* pfull = qfull + 4;
  uint64_t* pvdone = qfull + 5;
  uint64_t* drain = qfull + 6;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(dsm + C::oTmem);
  float* gmax = reinterpret_cast<float*>(dsm + C::oMax);
  float* gnegm = reinterpret_cast<float*>(dsm + C::oNegM);
  float* gpart = reinterpret_cast<float*>(dsm + C::oPart);
  float* gl = reinterpret_cast<float*>(dsm + C::oL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { tc::mbar_init(&full[s], 1); tc::mbar_init(&empty[s], 1); }
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qempty, 1);
    tc::mbar_init(sfull, 1);
    tc::mbar_init(sfree, kXoEpiWarps);
    tc::mbar_init(pfull, kXoEpiWarps);
    tc::mbar_init(pvdone, 1);
    tc::mbar_init(drain, 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_desc(&tmK);
    tc::tma_prefetch_desc(&tmV);
    tc::tma_prefetch_desc(&tmQ);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, kAcTmemCols);
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
      int k = 0, nq = 0;
      for (int j = 0; ok; ++j) {
        const long long i = item_at(cta, j, G);
        if (i >= a.items) break;
        const Item it = item_of(i, a);
        const int T = xo_tiles(it, a);
        if (nq > 0) ok = tc::mbar_wait(qempty, (uint32_t)((nq - 1) & 1), a.err, kErrAcProducer);
        if (!ok) break;
        tc::mbar_expect_tx(qfull, (uint32_t)C::TBYTES);
        const int b = it.unit / a.Hk, hk = it.unit % a.Hk;
        for (int hh = 0; hh < a.g; ++hh) {
          const int row = ((b * a.Hq + hk * a.g + hh) * a.n) + it.p0;
          for (int kb = 0; kb < C::KB; ++kb)
            tc::tma_load_2d(sQ + kb * 128 * 128 + hh * a.P * 128, &tmQ, kb * 64, row, qfull);
        }
        ++nq;
        for (int t = 0; t < T && ok; ++t, ++k) {
          const int s = k % C::STAGES, round = k / C::STAGES;
          if (round > 0)
            ok = tc::mbar_wait(&empty[s], (uint32_t)((round - 1) & 1), a.err, kErrAcProducer);
          if (!ok) break;
          tc::mbar_expect_tx(&full[s], (uint32_t)(2 * C::TBYTES));
          uint8_t* dk = sKV + s * 2 * C::TBYTES;
          uint8_t* dv = dk + C::TBYTES;
          for (int kb = 0; kb < C::KB; ++kb) {
            tc::tma_load_2d(dk + kb * 128 * 128, &tmK, kb * 64, it.unit * a.n + t * 128, &full[s]);
            tc::tma_load_2d(dv + kb * 128 * 128, &tmV, kb * 64, it.unit * a.n + t * 128, &full[s]);
          }
        }
      }
      // every copy issued here has landed before the CTA can leave
      for (int kk = max(0, k - C::STAGES); kk < k; ++kk)
        tc::mbar_wait(&full[kk % C::STAGES], (uint32_t)((kk / C::STAGES) & 1), a.err,
                      kErrAcProducer);
      if (nq > 0) tc::mbar_wait(qfull, (uint32_t)((nq - 1) & 1), a.err, kErrAcProducer);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, 128);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32_bmn(128, D);
      const uint32_t s1 = tbase, s2 = tbase + 128u, od = tbase + 256u;
      const uint32_t sQa = tc::saddr(sQ), sPa = tc::saddr(sP);
      int k = 0, nq = 0;
      for (int j = 0; ok; ++j) {
        const long long i = item_at(cta, j, G);
        if (i >= a.items) break;
        const Item it = item_of(i, a);
        const int T = xo_tiles(it, a);
        ok = tc::mbar_wait(qfull, (uint32_t)(nq & 1), a.err, kErrAcMma);
        if (!ok) break;
        ++nq;
        for (int t = 0; t < T; ++t, ++k) {
          const int s = k % C::STAGES;
          ok = tc::mbar_wait(&full[s], (uint32_t)((k / C::STAGES) & 1), a.err, kErrAcMma);
          if (ok && k > 0) ok = tc::mbar_wait(sfree, (uint32_t)((k - 1) & 1), a.err, kErrAcMma);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t sKa = tc::saddr(sKV + s * 2 * C::TBYTES);
          const uint32_t sVa = sKa + (uint32_t)C::TBYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int kb = kk / 4, kin = (kk % 4) * 32;
            const uint64_t qd = tc::sw128_desc(sQa + kb * 128 * 128 + kin);
            const uint64_t kd = tc::sw128_desc(sKa + kb * 128 * 128 + kin);
            tc::mma_bf16(s1, qd, kd, idesc_s, kk > 0 ? 1u : 0u);   // [row][key]
            tc::mma_bf16(s2, kd, qd, idesc_s, kk > 0 ? 1u : 0u);   // [key][row]
          }
          tc::mma_commit(sfull);
          if (t == T - 1) tc::mma_commit(qempty);
          // P of this tile, written by the epilogue (which also rescaled O)
          ok = tc::mbar_wait(pfull, (uint32_t)(k & 1), a.err, kErrAcMma);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 128 / 16; ++kk) {
            // A = P (K-major: keys); B = V (MN-major: its rows are the keys)
            const uint64_t pd = tc::sw128_desc(sPa + (kk / 4) * 128 * 128 + (kk % 4) * 32);
            const uint64_t vd = tc::sw128_mn_desc(sVa + kk * 16 * 128, 128 * 128, 1024);
            tc::mma_bf16(od, pd, vd, idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit(&empty[s]);
          tc::mma_commit(pvdone);
        }
      }
      // every MMA issued here has completed before tensor memory is released
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0u, a.err, kErrAcMma);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quarter = warp & 3;                 // tensor-memory lane quarter
    const int half = (warp - 2) >> 2;             // column half of each tile
    const int r = quarter * 32 + lane;            // row of S1 and O / key of S2
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int ET = 32 * kXoEpiWarps;
    int k = 0;                                    // tiles so far
    for (int j = 0;; ++j) {
      const long long i = item_at(cta, j, G);
      if (i >= a.items) break;
      const Item it = item_of(i, a);
      const int T = xo_tiles(it, a);
      const int pos_r = it.p0 + r % a.P;          // prompt position of row r
      const bool row_ok = pos_r < a.n;
      float m = -INFINITY;                        // exact running maximum (log2 units)
      float ref = -INFINITY;                      // reference maximum of P
      float lsum = 0.f;                           // this half's sum of P over the tiles
      for (int t = 0; t < T; ++t, ++k) {
        if (ok) ok = tc::mbar_wait(sfull, (uint32_t)(k & 1), a.err, kErrAcEpilogue);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
        const int key0 = t * 128;
        const bool masked = key0 + 127 > it.p0 || it.p0 + a.P > a.n;
        // --- row maxima: row r, columns [64 half, 64 half + 64) of S1
        const uint32_t c1 = tbase + lane_addr + (uint32_t)(half * 64);
        float pm = -INFINITY;
        const int lim0 = row_ok ? pos_r - (key0 + half * 64) : -1;   // last visible column
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          float v[32];
          tc::tmem_ld32(c1 + (uint32_t)c0, v);
          if (masked) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) v[jj] = jj + c0 <= lim0 ? v[jj] : -INFINITY;
          }
          float ma = v[0], mb = v[16];
#pragma unroll
          for (int jj = 1; jj < 15; jj += 2) {
            ma = max3(ma, v[jj], v[jj + 1]);
            mb = max3(mb, v[jj + 16], v[jj + 17]);
          }
          pm = max3(pm, max3(ma, v[15], v[31]), mb);
        }
        gmax[half * 128 + r] = pm;
        named_bar(1, ET);
        const float mt = fmaxf(gmax[r], gmax[128 + r]);
        if (mt != -INFINITY) m = fmaxf(m, mt * a.sl2);
        if (half == 0) gnegm[r] = -m;
        // the reference of P: raised when the exact maximum passes it by kXoSlack
        const float ref_new = (ref == -INFINITY || m > ref + kXoSlack) ? m : ref;
        // P of the previous tile has been consumed (and O is at rest) before this
        // tile's P is written or O rescaled
        if (ok && k > 0) ok = tc::mbar_wait(pvdone, (uint32_t)((k - 1) & 1), a.err, kErrAcEpilogue);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
        // (the tensor-memory loads and stores are whole-warp instructions: every lane
        // takes part when any lane's row is rescaled, the others with factor 1)
        const bool resc = t > 0 && ref_new != ref && ref != -INFINITY;
        if (__any_sync(0xffffffffu, resc)) {
          const float alpha = resc ? exp2f(ref - ref_new) : 1.f;
          lsum *= alpha;
          const uint32_t oc = tbase + lane_addr + 256u + (uint32_t)(half * (D / 2));
#pragma unroll 1
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            float v[32];
            tc::tmem_ld32(oc + (uint32_t)c0, v);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) v[jj] *= alpha;
            tc::tmem_st32(oc + (uint32_t)c0, v);
          }
        }
        ref = ref_new;
        // --- P = exp2(S1 * sl2 - ref) of row r, keys [64 half, 64 half + 64), as bf16
        //     into the 128-byte swizzled K-major tile (k-block = half)
        {
          uint8_t* prow = sP + half * 128 * 128 + r * 128;
          const float nref = ref == -INFINITY ? 0.f : -ref;
#pragma unroll 1
          for (int c0 = 0; c0 < 64; c0 += 32) {
            float v[32];
            tc::tmem_ld32(c1 + (uint32_t)c0, v);
            // paired fp32 arithmetic; a hidden key's logit becomes -inf (weight 0)
            const float2 s2 = make_float2(a.sl2, a.sl2), n2 = make_float2(nref, nref);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 2) {
              const float2 e = __ffma2_rn(make_float2(v[jj], v[jj + 1]), s2, n2);
              v[jj] = e.x;
              v[jj + 1] = e.y;
            }
            if (masked) {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) v[jj] = jj + c0 <= lim0 ? v[jj] : -INFINITY;
            }
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(v[jj]) : "f"(v[jj]));
            uint32_t pk[16];
            float2 ls = make_float2(0.f, 0.f);
#pragma unroll
            for (int jj = 0; jj < 32; jj += 2) {
              ls = __fadd2_rn(ls, make_float2(v[jj], v[jj + 1]));
              const __nv_bfloat162 h = __floats2bfloat162_rn(v[jj], v[jj + 1]);
              pk[jj / 2] = *reinterpret_cast<const uint32_t*>(&h);
            }
            lsum += ls.x + ls.y;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int chunk = c0 / 8 + q4;      // 16-byte chunk of the 128-byte row
              *reinterpret_cast<uint4*>(prow + ((chunk ^ (r & 7)) * 16)) =
                  make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(pfull);
        named_bar(1, ET);                         // -m of every row is in shared memory
        // --- column sums: key r, rows [64 half, 64 half + 64) of S2
        const uint32_t c2 = tbase + lane_addr + 128u + (uint32_t)(half * 64);
        const float* nm = gnegm + half * 64;
        const int key = key0 + r;
        float acc = 0.f;
        if (key0 < a.ns && a.fx) {
#pragma unroll 1
          for (int c0 = 0; c0 < 64; c0 += 32) {
            float v[32];
            tc::tmem_ld32(c2 + (uint32_t)c0, v);
            if (!masked) {
              const float4* nm4 = reinterpret_cast<const float4*>(nm + c0);
              const float2 s2 = make_float2(a.sl2, a.sl2);
#pragma unroll
              for (int jj = 0; jj < 32; jj += 4) {
                const float4 b4 = nm4[jj / 4];
                const float2 lo = __ffma2_rn(make_float2(v[jj], v[jj + 1]), s2,
                                             make_float2(b4.x, b4.y));
                const float2 hi = __ffma2_rn(make_float2(v[jj + 2], v[jj + 3]), s2,
                                             make_float2(b4.z, b4.w));
                v[jj] = lo.x; v[jj + 1] = lo.y; v[jj + 2] = hi.x; v[jj + 3] = hi.y;
              }
            } else {
              // rows are head-major: row = head * P + (position - p0), P a power of two
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const int pos = it.p0 + ((half * 64 + c0 + jj) & (a.P - 1));
                v[jj] = (pos < a.n && key <= pos) ? fmaf(v[jj], a.sl2, nm[c0 + jj]) : -INFINITY;
              }
            }
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(v[jj]) : "f"(v[jj]));
            float2 sum[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              sum[q] = __fadd2_rn(make_float2(v[2 * q], v[2 * q + 1]),
                                  make_float2(v[2 * q + 16], v[2 * q + 17]));
#pragma unroll
            for (int w = 4; w > 0; w >>= 1)
#pragma unroll
              for (int q = 0; q < w; ++q) sum[q] = __fadd2_rn(sum[q], sum[q + w]);
            acc += sum[0].x + sum[0].y;
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(sfree);
        if (half == 1) gpart[r] = acc;
        named_bar(1, ET);
        if (half == 0 && ok && key < a.ns && a.fx)
          add_fixed(a.fx + (size_t)it.unit * a.ns + key, acc + gpart[r]);
      }
      // --- the item's attention output: O / l of row r, this half's d columns
      if (ok) ok = tc::mbar_wait(pvdone, (uint32_t)((k - 1) & 1), a.err, kErrAcEpilogue);
      ok = __all_sync(0xffffffffu, ok);
      tc::fence_after_sync();
      gl[half * 128 + r] = lsum;
      named_bar(1, ET);
      const float l = gl[r] + gl[128 + r];
      named_bar(1, ET);                           // gl is free for the next item
      {
        // whole-warp tensor-memory loads; only rows inside the prompt are stored
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int b = it.unit / a.Hk, hk = it.unit % a.Hk, hh = r / a.P;
        __nv_bfloat16* dst = xa.x_out +
            ((size_t)(b * a.Hq + hk * a.g + hh) * a.n + (row_ok ? pos_r : 0)) * D + half * (D / 2);
        const uint32_t oc = tbase + lane_addr + 256u + (uint32_t)(half * (D / 2));
#pragma unroll 1
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          float v[32];
          tc::tmem_ld32(oc + (uint32_t)c0, v);
          if (ok && row_ok) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h =
                    __floats2bfloat162_rn(v[8 * q8 + 2 * e] * inv, v[8 * q8 + 2 * e + 1] * inv);
                w[e] = *reinterpret_cast<const uint32_t*>(&h);
              }
              *reinterpret_cast<uint4*>(dst + c0 + 8 * q8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          __syncwarp();   // converged before the next whole-warp load
        }
      }
      // O is read before this CTA's next P is published (the next item's first
      // product overwrites it)
      tc::fence_before_sync();
    }
  }

  // teardown: every MMA this CTA issued has completed once the epilogue consumed
  // its last tile; on an error path the MMA thread drained before this point
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, kAcTmemCols);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 ac_encode_fn() {
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

// 2-D bf16 map over [rows][d]: boxes of 64 elements x box_rows rows, 128-byte swizzle.
cudaError_t ac_make_map(CUtensorMap* m, const void* base, long long rows, int d, int box_rows) {
  auto fn = ac_encode_fn();
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

template <int D>
cudaError_t run_acumul(const kvc_dims& d, const __nv_bfloat16* q_full, const __nv_bfloat16* k,
                       float* scores, unsigned long long* fx, unsigned* err, cudaStream_t stream) {
  using C = AcCfg<D>;
  const int g = d.n_q_heads / d.n_kv_heads;
  AcArgs a{};
  a.n = d.prompt_len;
  a.ns = d.prompt_len - d.obs_window;
  a.g = g;
  a.P = 128 / g;
  a.Hq = d.n_q_heads;
  a.Hk = d.n_kv_heads;
  a.units = d.batch * d.n_kv_heads;
  a.rblocks = (a.n + a.P - 1) / a.P;
  a.items = (long long)a.units * a.rblocks;
  a.sl2 = 1.4426950408889634f / sqrtf((float)D);
  a.fx = fx;
  a.err = err;
  cudaError_t e = cudaMemsetAsync(fx, 0, (size_t)a.units * a.ns * 8, stream);
  if (e != cudaSuccess) return e;
  CUtensorMap mk, mq;
  if ((e = ac_make_map(&mk, k, (long long)a.units * a.n, D, 128)) != cudaSuccess) return e;
  if ((e = ac_make_map(&mq, q_full, (long long)d.batch * a.Hq * a.n, D, a.P)) != cudaSuccess)
    return e;
  e = ensure_smem(reinterpret_cast<const void*>(acumul_tc_kernel<D>), C::total);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int grid = (int)std::min<long long>(n_sm, a.items);
  acumul_tc_kernel<D><<<grid, kAcThreads, C::total, stream>>>(mk, mq, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launches(1);
  return fixed_to_float(fx, scores, (long long)a.units * a.ns, stream);
}

template <int D>
cudaError_t run_acumul_xo(const kvc_dims& d, const __nv_bfloat16* q_full, const __nv_bfloat16* k,
                          const __nv_bfloat16* v, float* scores, unsigned long long* fx,
                          __nv_bfloat16* x_out, unsigned* err, cudaStream_t stream) {
  using C = XoCfg<D>;
  const int g = d.n_q_heads / d.n_kv_heads;
  XoArgs xa{};
  AcArgs& a = xa.a;
  a.n = d.prompt_len;
  a.ns = d.prompt_len - d.obs_window;
  a.g = g;
  a.P = 128 / g;
  a.Hq = d.n_q_heads;
  a.Hk = d.n_kv_heads;
  a.units = d.batch * d.n_kv_heads;
  a.rblocks = (a.n + a.P - 1) / a.P;
  a.items = (long long)a.units * a.rblocks;
  a.sl2 = 1.4426950408889634f / sqrtf((float)D);
  a.fx = scores ? fx : nullptr;
  a.err = err;
  xa.x_out = x_out;
  xa.d = D;
  cudaError_t e = scores ? cudaMemsetAsync(fx, 0, (size_t)a.units * a.ns * 8, stream)
                         : cudaSuccess;
  if (e != cudaSuccess) return e;
  CUtensorMap mk, mv, mq;
  if ((e = ac_make_map(&mk, k, (long long)a.units * a.n, D, 128)) != cudaSuccess) return e;
  if ((e = ac_make_map(&mv, v, (long long)a.units * a.n, D, 128)) != cudaSuccess) return e;
  if ((e = ac_make_map(&mq, q_full, (long long)d.batch * a.Hq * a.n, D, a.P)) != cudaSuccess)
    return e;
  e = ensure_smem(reinterpret_cast<const void*>(acumul_xo_kernel<D>), C::total);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int grid = (int)std::min<long long>(n_sm, a.items);
  acumul_xo_kernel<D><<<grid, kXoThreads, C::total, stream>>>(mk, mv, mq, xa);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  count_launches(1);
  return scores ? fixed_to_float(fx, scores, (long long)a.units * a.ns, stream) : cudaSuccess;
}

}  // namespace

cudaError_t launch_acumul_xo(const kvc_dims& d, const __nv_bfloat16* q_full,
                             const __nv_bfloat16* k, const __nv_bfloat16* v, float* scores,
                             unsigned long long* fx, __nv_bfloat16* x_out, unsigned* err,
                             cudaStream_t stream) {
  const int g = d.n_q_heads / d.n_kv_heads;
  if (g < 1 || g > 16 || 128 % g != 0) return cudaErrorInvalidValue;
  if (d.prompt_len - d.obs_window < 1) return cudaErrorInvalidValue;
  if (d.head_dim == 128) return run_acumul_xo<128>(d, q_full, k, v, scores, fx, x_out, err, stream);
  if (d.head_dim == 64) return run_acumul_xo<64>(d, q_full, k, v, scores, fx, x_out, err, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_acumul(const kvc_dims& d, const __nv_bfloat16* q_full, const __nv_bfloat16* k,
                          float* scores, unsigned long long* fx, unsigned* err,
                          cudaStream_t stream) {
  const int g = d.n_q_heads / d.n_kv_heads;
  if (g < 1 || g > 16 || 128 % g != 0) return cudaErrorInvalidValue;
  if (d.prompt_len - d.obs_window < 1) return cudaErrorInvalidValue;
  if (d.head_dim == 128) return run_acumul<128>(d, q_full, k, scores, fx, err, stream);
  if (d.head_dim == 64) return run_acumul<64>(d, q_full, k, scores, fx, err, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvc
