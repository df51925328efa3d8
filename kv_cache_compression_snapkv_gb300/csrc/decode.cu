// decode.cu -- split-K decode attention over the packed cache plus the bf16 window,
// optionally fused with the append (and group flush) of the step's new token.
//
// MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
// Cache, §2 eq. (1) and Algorithm 1 (decoding): append the new key/value to the
// 16-bit buffer, quantize when it fills, then one softmax over the dequantized
// packed keys and the buffer's keys; output = A_quant . dequant(Q_V) +
// A_unquant . R_V. Blog "KV Cache Compression: Eviction and Quantization",
// "Measured on a real model": exact recent window, rounded rest, one softmax.
//
// Work decomposition (one launch for a range of layers):
//   unit = (layer, sequence b, kv head h). "Packed" CTAs take 16 group blocks (2
//   per warp); "window" CTAs 128 ring slots (16 per warp). Every warp first
//   stages its whole chunk into shared memory with one or two bulk async copies
//   (cp.async.bulk on an mbarrier, bounded wait), then computes from shared
//   memory. Each warp keeps an online softmax for the g query heads of its kv
//   head; warps merge in shared memory, CTAs write (m, l, o) partials, and the
//   last CTA of the unit (atomic ticket, no waiting) merges them with a
//   log-sum-exp combine and writes the fp32 output.
//   In the fused step the window CTAs also store the new token into the ring and,
//   when the window reaches R, quantize its oldest group (written to the packed
//   store and attended from shared memory in the same launch).
//
// Arithmetic. Per 32-token group block the key logits are
//     q . k_t = sum_c (q_c S_c) code_tc + sum_c q_c Z_c
// and the value output is
//     o_c = sum_t (p_t S_t,gc) code_tc + sum_t p_t Z_t,gc.
// Both code sums run on the tensor cores (mma m16n8k16, fp16 operands, fp32
// accumulate): codes are unpacked in registers to exact fp16 integers, and the
// fp16 operand products (q_c S_c, p_t S_t) are split into hi + lo fp16 parts that
// occupy separate rows of the 16-row operand (rows 0..g-1 hi, g..2g-1 lo), so the
// rounding of the operand does not limit accuracy. The zero-point sums are small
// extra tensor-core products (q against the warp's groups' key zeros; p against
// the value zeros). The window runs the same flow on bf16 operands.
#include <algorithm>
#include <utility>

#include "quant_device.cuh"

namespace kvc {
namespace {

constexpr int kThreads = kDecWarps * 32;
constexpr int kGroupsPerWarp = kGroupsPerCta / kDecWarps;
constexpr int kSlotsPerWarp = kWinSlotsPerCta / kDecWarps;
static_assert(kSlotsPerWarp == 32, "window warps take 32 slots");
constexpr unsigned kWaitLimit = 1u << 20;   // bounded mbarrier polls (far above any copy)
static_assert(kGroupsPerWarp <= 8, "the key zero-point product covers at most 8 groups");

struct DecLayer {
  int n_groups;     // packed groups read from the store (a group flushed here excluded)
  int win_start;    // ring start slot after this launch's append
  int win_len;      // window tokens after this launch's append
  int n_ctas;       // CTAs per unit
  int cta_begin;    // first CTA of the layer in the grid
  int cap_groups;
  int new_slot;     // ring slot of the token appended in this launch, or -1
  int flush_start;  // ring slot of the oldest token when this launch flushes a group, or -1
  int wchunks;      // window chunks (32 slots) per unit; packed chunks (4 groups) follow
  int cpc;          // chunks per CTA
  long long packed_off;
};

struct DecParams {
  DecLayer L[KVC_MAX_LAUNCH_LAYERS];
  const __nv_bfloat16* k_new;   // [n_layers][units][D] (fused step only)
  const __nv_bfloat16* v_new;
  unsigned* err;                // device error word (bit 0: a staging wait gave up)
  int n_layers;                 // layers in this launch
  int layer_begin;              // absolute index of L[0]
  int units;                    // batch * n_kv_heads
  int R;                        // window ring length
  float sl2;                    // log2(e) / sqrt(head_dim)
};

template <int D, int BITS>
constexpr int warp_buf_bytes() {
  return kGroupsPerWarp * block_bytes(D, BITS) > kSlotsPerWarp * D * 4
             ? kGroupsPerWarp * block_bytes(D, BITS)
             : kSlotsPerWarp * D * 4;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------- bulk staging helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Stage up to two contiguous global ranges into shared memory (whole warp calls).
// The warp's barrier was initialised at kernel start; `phase` counts its uses.
// Returns false if the wait gave up (error word set; a second bounded wait lets
// copies still in flight land before the CTA can exit).
__device__ bool warp_stage(uint64_t* bar, unsigned phase, void* dst0, const void* src0,
                           uint32_t bytes0, void* dst1, const void* src1, uint32_t bytes1,
                           unsigned* err) {
  const int lane = threadIdx.x & 31;
  __syncwarp();   // every lane is done reading the buffer's previous contents
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                 :: "r"(smem_u32(bar)), "r"(bytes0 + bytes1) : "memory");
    bulk_g2s(dst0, src0, bytes0, bar);
    if (bytes1) bulk_g2s(dst1, src1, bytes1, bar);
  }
  const unsigned parity = phase & 1u;
  bool done = false;
  for (unsigned it = 0; it < kWaitLimit && !done; ++it) done = mbar_try_wait(bar, parity);
  if (!done) {
    if (lane == 0) atomicOr(err, 1u);
    for (unsigned it = 0; it < kWaitLimit && !done; ++it) done = mbar_try_wait(bar, parity);
    done = false;
  }
  __syncwarp();
  return __all_sync(0xffffffffu, done);
}

// ------------------------------------------------------------ fragment helpers
template <typename F, int... I>
__device__ __forceinline__ void static_for_impl(F&& f, std::integer_sequence<int, I...>) {
  (f(std::integral_constant<int, I>{}), ...);
}
// f(integral_constant<int, i>) for i = 0 .. N-1, indices known at compile time
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  static_for_impl(f, std::make_integer_sequence<int, N>{});
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Transpose of an 8x8 matrix of 16-bit elements held in the operand-fragment
// layout (lane = 4*row + col/2): afterwards lane 4*r + c/2 holds row r of the
// transpose.
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// v as an fp16 pair (hi, lo) with hi = fp16(v), lo = fp16(v - hi): hi in the low half.
__device__ __forceinline__ uint32_t split_f16(float v) {
  const float hi = __half2float(__float2half_rn(v));
  return h2u(__floats2half2_rn(v, v - hi));
}
__device__ __forceinline__ uint32_t split_bf16(float v) {
  const float hi = __bfloat162float(__float2bfloat16_rn(v));
  const __nv_bfloat162 p = __floats2bfloat162_rn(v, v - hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Exact fp16 pair of the two codes in pair slot P of word w. The field of slot P
// is masked in place under the fp16 exponent of 2^e, e = 10 - BITS*j (j = field
// index inside its byte), so each half reads 2^e + code; one subtraction leaves
// the code.
template <int BITS, int P>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w) {
  constexpr int CPB = 8 / BITS, SB = P / CPB, J = P % CPB;
  constexpr uint32_t mask = (((1u << BITS) - 1u) * 0x00010001u) << (BITS * J);
  constexpr uint32_t mag = ((uint32_t)(25 - BITS * J) << 10) * 0x00010001u;
  const uint32_t v = ((SB ? (w >> 8) : w) & mask) | mag;
  return h2u(__hsub2(u2h(v), u2h(mag)));
}

// A operand of key product (MT, KS) (rows = tokens, k = channels) from the lane's
// key code words.
template <int D, int BITS, int MT, int KS>
__device__ __forceinline__ void key_afrag(const uint32_t* kw, uint32_t (&a)[4]) {
  if constexpr (BITS == 2) {
    constexpr int wi = MT * (D / 32) + KS / 2, b = 2 * (KS & 1);
    a[0] = unpack_pair<2, b>(kw[wi]);
    a[1] = unpack_pair<2, 4 + b>(kw[wi]);
    a[2] = unpack_pair<2, b + 1>(kw[wi]);
    a[3] = unpack_pair<2, 5 + b>(kw[wi]);
  } else {
    constexpr int wi = MT * (D / 16) + KS;
    a[0] = unpack_pair<4, 0>(kw[wi]);
    a[1] = unpack_pair<4, 2>(kw[wi]);
    a[2] = unpack_pair<4, 1>(kw[wi]);
    a[3] = unpack_pair<4, 3>(kw[wi]);
  }
}
// A operand of value product (MT, KS) (rows = channels, k = tokens).
template <int BITS, int MT, int KS>
__device__ __forceinline__ void value_afrag(const uint32_t* vw, uint32_t (&a)[4]) {
  if constexpr (BITS == 2) {
    constexpr int b = 2 * KS;
    a[0] = unpack_pair<2, b>(vw[MT]);
    a[1] = unpack_pair<2, 4 + b>(vw[MT]);
    a[2] = unpack_pair<2, b + 1>(vw[MT]);
    a[3] = unpack_pair<2, 5 + b>(vw[MT]);
  } else {
    constexpr int wi = 2 * MT + KS;
    a[0] = unpack_pair<4, 0>(vw[wi]);
    a[1] = unpack_pair<4, 2>(vw[wi]);
    a[2] = unpack_pair<4, 1>(vw[wi]);
    a[3] = unpack_pair<4, 3>(vw[wi]);
  }
}

// Column layout of the B operands: column n of n-tile u belongs to query head
// 4u + n/2; even columns carry the leading ("hi") fp16/bf16 part of an operand
// product, odd columns the remainder ("lo"). A lane's C fragment (columns 2tid,
// 2tid+1) therefore holds both parts for head 4u + tid, and their sum is the
// full-precision product.
template <int GQ>
constexpr int n_tiles() { return (GQ + 3) / 4; }

template <int D, int GQ>
struct WarpState {
  static constexpr int NH = n_tiles<GQ>();
  float m[NH];                 // running max of the raw logits (head 4u + tid)
  float l[NH];                 // lane-partial sum of the weights
  float o[NH][D / 16][4];      // value accumulators: rows = channels, columns = (head, part)
  float cz[NH][4];             // value zero-point sums: rows = channel groups
};

template <int D, int GQ>
__device__ __forceinline__ void state_init(WarpState<D, GQ>& st) {
  constexpr int NH = n_tiles<GQ>();
#pragma unroll
  for (int u = 0; u < NH; ++u) {
    st.m[u] = -INFINITY;
    st.l[u] = 0.f;
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[u][i][e] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) st.cz[u][e] = 0.f;
  }
}

// Query operands of the packed path: qh = fp16 query pair of this lane's B column
// (zero beyond the group's heads); qn = -qh in "lo" columns, 0 in "hi" columns.
template <int D, int GQ>
struct QRegs {
  static constexpr int NH = n_tiles<GQ>();
  uint32_t qh[NH][D / 16][2];
  uint32_t qn[NH][D / 16][2];
};

template <int D, int GQ>
__device__ __forceinline__ void load_qregs(QRegs<D, GQ>& qr, const __nv_bfloat16* qs) {
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
#pragma unroll
  for (int u = 0; u < n_tiles<GQ>(); ++u) {
    const int h = 4 * u + (gid >> 1);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int c = 16 * ks + 2 * tid + 8 * e2;
        float a = 0.f, b = 0.f;
        if (h < GQ) {
          a = __bfloat162float(qs[h * D + c]);
          b = __bfloat162float(qs[h * D + c + 1]);
        }
        const __half2 q2 = __floats2half2_rn(a, b);
        qr.qh[u][ks][e2] = h2u(q2);
        qr.qn[u][ks][e2] = (gid & 1) ? h2u(__hneg2(q2)) : 0u;
      }
  }
}

// Online-softmax update with the logits of 32 tokens: x[u][mt][r] is token
// 16mt + gid + 8r for head 4u + tid. The weights replace the logits.
template <int D, int GQ>
__device__ __forceinline__ void softmax_update(WarpState<D, GQ>& st, float (&x)[n_tiles<GQ>()][2][2],
                                               float sl2) {
#pragma unroll
  for (int u = 0; u < n_tiles<GQ>(); ++u) {
    float gm = fmaxf(fmaxf(x[u][0][0], x[u][0][1]), fmaxf(x[u][1][0], x[u][1][1]));
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
    gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
    const float mnew = fmaxf(st.m[u], gm);
    if (__any_sync(0xffffffffu, mnew > st.m[u])) {
      const float corr = (st.m[u] == -INFINITY) ? 0.f : fast_exp2((st.m[u] - mnew) * sl2);
      st.l[u] *= corr;
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[u][i][e] *= corr;
#pragma unroll
      for (int e = 0; e < 4; ++e) st.cz[u][e] *= corr;
      st.m[u] = mnew;
    }
    const float msl = (st.m[u] == -INFINITY) ? 0.f : st.m[u] * sl2;
    float s = 0.f;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float p = fast_exp2(fmaf(x[u][mt][r], sl2, -msl));
        x[u][mt][r] = p;
        s += p;
      }
    st.l[u] += s;
  }
}

// ------------------------------------------------------------ packed groups
// `base` points at n_grp (<= kGroupsPerWarp) consecutive group blocks in shared
// memory. Per group: key logits (rows = tokens), one online-softmax update, the
// value products (rows = channels). The group loop stays rolled so that the hot
// code fits the instruction cache.
template <int D, int BITS, int GQ>
__device__ void packed_warp(WarpState<D, GQ>& st, const QRegs<D, GQ>& qr, const uint8_t* base,
                            int n_grp, float sl2) {
  constexpr int KS = D / 16, NGC = D / 32, BB = 8 * D * (BITS + 1), WPL = D * BITS / 32;
  constexpr int NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;

  // key zero-point sums of every group of the chunk: C[group][n] = Z_group . q_n
  // (A rows = groups, B = the queries in the "hi" columns)
  float zb[NH];
  {
    uint32_t za[KS][2];
    const int gz = gid < n_grp ? gid : 0;
    const uint4* zp = reinterpret_cast<const uint4*>(base + (size_t)gz * BB + off_kzero(D, BITS) +
                                                     tid * (D / 4) * 2);
#pragma unroll
    for (int i = 0; i < KS / 2; ++i) {
      const uint4 z = zp[i];
      const bool live = gid < n_grp;
      za[2 * i][0] = live ? z.x : 0u;
      za[2 * i][1] = live ? z.y : 0u;
      za[2 * i + 1][0] = live ? z.z : 0u;
      za[2 * i + 1][1] = live ? z.w : 0u;
    }
#pragma unroll
    for (int u = 0; u < NH; ++u) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t b0 = (gid & 1) ? 0u : qr.qh[u][ks][0];
        const uint32_t b1 = (gid & 1) ? 0u : qr.qh[u][ks][1];
        mma_f16(c, za[ks][0], 0u, za[ks][1], 0u, b0, b1);
      }
      zb[u] = c[0];   // group gid, head 4u + tid
    }
  }

#pragma unroll 1
  for (int j = 0; j < n_grp; ++j) {
    const uint8_t* blk = base + (size_t)j * BB;
    float x[NH][2][2];
    {
      // B = hi/lo(q * S_k): one fp16 product, or its rounding remainder
      uint32_t bq[NH][KS][2];
      const uint4* sp = reinterpret_cast<const uint4*>(blk + off_kscale(D, BITS) + tid * (D / 4) * 2);
#pragma unroll
      for (int i = 0; i < KS / 2; ++i) {
        const uint4 s4 = sp[i];
        const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int u = 0; u < NH; ++u)
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int ks = 2 * i + (h >> 1), e2 = h & 1;
            const __half2 S2 = u2h(sv[h]);
            bq[u][ks][e2] = h2u(__hfma2(u2h(qr.qh[u][ks][e2]), S2,
                                        __hmul2(u2h(qr.qn[u][ks][e2]), S2)));
          }
      }
      uint32_t kw[WPL];
      {
        const uint4* p = reinterpret_cast<const uint4*>(blk);
#pragma unroll
        for (int i = 0; i < WPL / 4; ++i) {
          const uint4 w4 = p[i * 32 + lane];
          kw[4 * i] = w4.x; kw[4 * i + 1] = w4.y; kw[4 * i + 2] = w4.z; kw[4 * i + 3] = w4.w;
        }
      }
      float acc[NH][2][2][4];   // [u][mt][chain][C]: even / odd k-steps
#pragma unroll
      for (int u = 0; u < NH; ++u) {
        const float bias = __shfl_sync(0xffffffffu, zb[u], j * 4 + tid);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[u][mt][0][e] = (e & 1) ? 0.f : bias;
            acc[u][mt][1][e] = 0.f;
          }
      }
      static_for<2>([&](auto MT_) {
        constexpr int MT = decltype(MT_)::value;
        static_for<KS>([&](auto KS_) {
          constexpr int K = decltype(KS_)::value;
          uint32_t a[4];
          key_afrag<D, BITS, MT, K>(kw, a);
#pragma unroll
          for (int u = 0; u < NH; ++u)
            mma_f16(acc[u][MT][K & 1], a[0], a[1], a[2], a[3], bq[u][K][0], bq[u][K][1]);
        });
      });
#pragma unroll
      for (int u = 0; u < NH; ++u)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          x[u][mt][0] = (acc[u][mt][0][0] + acc[u][mt][0][1]) + (acc[u][mt][1][0] + acc[u][mt][1][1]);
          x[u][mt][1] = (acc[u][mt][0][2] + acc[u][mt][0][3]) + (acc[u][mt][1][2] + acc[u][mt][1][3]);
        }
    }
    softmax_update<D, GQ>(st, x, sl2);

    // values: o[channel][n] += sum_t code[channel][t] * hi/lo(p_t S_t,gc)[t][n]
    uint32_t vw[WPL];
    {
      const uint4* p = reinterpret_cast<const uint4*>(blk + off_vcodes(D, BITS));
#pragma unroll
      for (int i = 0; i < WPL / 4; ++i) {
        const uint4 w4 = p[i * 32 + lane];
        vw[4 * i] = w4.x; vw[4 * i + 1] = w4.y; vw[4 * i + 2] = w4.z; vw[4 * i + 3] = w4.w;
      }
    }
    const __half* vs = reinterpret_cast<const __half*>(blk + off_vscale(D, BITS));
    const uint32_t* vz = reinterpret_cast<const uint32_t*>(blk + off_vzero(D, BITS));
    static_for<2>([&](auto KS_) {
      constexpr int K = decltype(KS_)::value;
      // scales of this lane's tokens 16K + gid and 16K + gid + 8, all channel groups
      float S[2][NGC];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int gc = 0; gc < NGC; ++gc)
          S[r][gc] = __half2float(vs[vs_index(16 * K + gid + 8 * r, gc, NGC)]);
      // zero-point sums: rows = channel groups (A = zeros, token pairs), B = hi/lo(p)
      const uint32_t az0 = gid < NGC ? vz[(8 * K + tid) * NGC + gid] : 0u;
      const uint32_t az2 = gid < NGC ? vz[(8 * K + 4 + tid) * NGC + gid] : 0u;
#pragma unroll
      for (int u = 0; u < NH; ++u) {
        const uint32_t bz0 = movm_t(split_f16(x[u][K][0]));
        const uint32_t bz1 = movm_t(split_f16(x[u][K][1]));
        mma_f16(st.cz[u], az0, 0u, az2, 0u, bz0, bz1);
      }
      static_for<NGC>([&](auto GC_) {
        constexpr int GC = decltype(GC_)::value;
#pragma unroll
        for (int u = 0; u < NH; ++u) {
          const uint32_t b0 = movm_t(split_f16(x[u][K][0] * S[0][GC]));
          const uint32_t b1 = movm_t(split_f16(x[u][K][1] * S[1][GC]));
          static_for<2>([&](auto H_) {
            constexpr int MV = 2 * GC + decltype(H_)::value;
            uint32_t a[4];
            value_afrag<BITS, MV, K>(vw, a);
            mma_f16(st.o[u][MV], a[0], a[1], a[2], a[3], b0, b1);
          });
        }
      });
    });
  }
}

// ------------------------------------------------------------- window slots
// wk: NS = 32 staged key rows (win_k_index layout); wv: 16 staged value pair rows
// (win_v_index layout); the first n_valid slots are live. bf16 products, exact
// queries, hi/lo weights.
template <int D, int GQ>
__device__ void window_warp(WarpState<D, GQ>& st, const __nv_bfloat16* qs, const __nv_bfloat16* wk,
                            const uint32_t* wv, int n_valid, float sl2) {
  constexpr int KS = D / 16, NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  float x[NH][2][2];
  {
    uint32_t bq[NH][KS][2];
#pragma unroll
    for (int u = 0; u < NH; ++u) {
      const int h = 4 * u + (gid >> 1);
      const bool live = h < GQ && !(gid & 1);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2)
          bq[u][ks][e2] = live ? *reinterpret_cast<const uint32_t*>(qs + h * D + 16 * ks + 2 * tid + 8 * e2)
                               : 0u;
    }
    float acc[NH][2][2][4];
#pragma unroll
    for (int u = 0; u < NH; ++u)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) { acc[u][mt][0][e] = 0.f; acc[u][mt][1][e] = 0.f; }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      // rows 16mt + gid (rl 0) and 16mt + gid + 8 (rl 1); 16-byte chunks swizzled by gid
      const uint4* r0 = reinterpret_cast<const uint4*>(wk + (size_t)(16 * mt + gid) * D);
      const uint4* r1 = reinterpret_cast<const uint4*>(wk + (size_t)(16 * mt + gid + 8) * D);
#pragma unroll
      for (int i = 0; i < KS / 2; ++i) {
        const int ch = (tid * (KS / 2) + i) ^ gid;
        const uint4 u0 = r0[ch], u1 = r1[ch];
#pragma unroll
        for (int u = 0; u < NH; ++u) {
          mma_bf16(acc[u][mt][0], u0.x, u1.x, u0.y, u1.y, bq[u][2 * i][0], bq[u][2 * i][1]);
          mma_bf16(acc[u][mt][1], u0.z, u1.z, u0.w, u1.w, bq[u][2 * i + 1][0], bq[u][2 * i + 1][1]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < NH; ++u)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float v = (acc[u][mt][0][2 * r] + acc[u][mt][0][2 * r + 1]) +
                          (acc[u][mt][1][2 * r] + acc[u][mt][1][2 * r + 1]);
          x[u][mt][r] = (16 * mt + gid + 8 * r) < n_valid ? v : -INFINITY;
        }
  }
  softmax_update<D, GQ>(st, x, sl2);
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    uint32_t b0[NH], b1[NH];
#pragma unroll
    for (int u = 0; u < NH; ++u) {
      b0[u] = movm_t(split_bf16(x[u][ks][0]));
      b1[u] = movm_t(split_bf16(x[u][ks][1]));
    }
    // pair rows 8ks + tid (tokens 16ks + 2tid, +1) and 8ks + 4 + tid; chunks swizzled by tid
    const uint4* p0 = reinterpret_cast<const uint4*>(wv + (size_t)(8 * ks + tid) * D);
    const uint4* p1 = reinterpret_cast<const uint4*>(wv + (size_t)(8 * ks + 4 + tid) * D);
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const int ch = (gid * (D / 32) + i) ^ tid;
      const uint4 v0 = p0[ch], v1 = p1[ch];
      // words: (mt = 2i, rl 0), (2i, rl 1), (2i + 1, rl 0), (2i + 1, rl 1)
#pragma unroll
      for (int u = 0; u < NH; ++u) {
        mma_bf16(st.o[u][2 * i], v0.x, v0.y, v1.x, v1.y, b0[u], b1[u]);
        mma_bf16(st.o[u][2 * i + 1], v0.z, v0.w, v1.z, v1.w, b0[u], b1[u]);
      }
    }
  }
}

// ----------------------------------------------------------- merge helpers
template <int D, int GQ>
struct DecSmem {
  float m[kDecWarps][GQ];      // log2-domain running max per warp and head
  float l[kDecWarps][GQ];
  float o[kDecWarps][GQ][D];
  float wt[kDecWarps][GQ];     // CTA merge weights
  float M[GQ], L[GQ];
  int last;
};

// Write the warp's per-head state (both column parts and the value zero-point
// sums folded in) into shared memory.
template <int D, int GQ>
__device__ void warp_to_smem(WarpState<D, GQ>& st, DecSmem<D, GQ>& sm, int warp, float sl2) {
  constexpr int NGC = D / 32, NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
#pragma unroll
  for (int u = 0; u < NH; ++u) {
    const int h = 4 * u + tid;
    float l = st.l[u];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    float z[NGC];
    const float zl = st.cz[u][0] + st.cz[u][1];   // channel group gid, head h
#pragma unroll
    for (int gc = 0; gc < NGC; ++gc) z[gc] = __shfl_sync(0xffffffffu, zl, gc * 4 + tid);
    if (h < GQ) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        sm.o[warp][h][16 * mt + gid] = st.o[u][mt][0] + st.o[u][mt][1] + z[mt / 2];
        sm.o[warp][h][16 * mt + gid + 8] = st.o[u][mt][2] + st.o[u][mt][3] + z[mt / 2];
      }
      if (gid == 0) {
        sm.m[warp][h] = st.m[u] == -INFINITY ? -INFINITY : st.m[u] * sl2;
        sm.l[warp][h] = l;
      }
    }
  }
}

// The staging area at the start of dynamic shared memory is shared, in turn, by
// the warps' staged chunks, the group being flushed (fp32 rows + codes) and the
// CTA's merge scratch: it is sized for the largest of the three.
template <int D, int BITS, int GQ>
constexpr int stage_bytes() {
  constexpr int a = kDecWarps * warp_buf_bytes<D, BITS>();
  constexpr int b = (int)sizeof(GroupSmem<D, kThreads>);
  constexpr int c = (int)sizeof(DecSmem<D, GQ>);
  constexpr int m = a > b ? (a > c ? a : c) : (b > c ? b : c);
  return (m + 127) / 128 * 128;
}
template <int D, int BITS, int GQ>
constexpr int dyn_smem_bytes() {
  return stage_bytes<D, BITS, GQ>() + block_bytes(D, BITS) + kDecWarps * 8 + GQ * D * 2;
}

template <int D, int BITS, int GQ>
__global__ void __launch_bounds__(kThreads, 3)
decode_kernel(const DecParams P, uint8_t* __restrict__ packed, __nv_bfloat16* __restrict__ win_k,
              __nv_bfloat16* __restrict__ win_v, const __nv_bfloat16* __restrict__ q,
              float* __restrict__ out, float* __restrict__ part, unsigned* __restrict__ tickets) {
  constexpr int BB = block_bytes(D, BITS), WB = warp_buf_bytes<D, BITS>();
  extern __shared__ __align__(128) uint8_t dsm[];
  // the merge scratch reuses the staging buffers once every warp is done with them
  DecSmem<D, GQ>& sm = *reinterpret_cast<DecSmem<D, GQ>*>(dsm);
  static_assert(sizeof(DecSmem<D, GQ>) <= stage_bytes<D, BITS, GQ>(), "merge scratch fits");
  static_assert(sizeof(GroupSmem<D, kThreads>) <= stage_bytes<D, BITS, GQ>(), "flush staging fits");
  static_assert(kDecWarps * WB <= stage_bytes<D, BITS, GQ>(), "warp buffers fit");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* wbuf = dsm + warp * WB;
  uint8_t* fblk = dsm + stage_bytes<D, BITS, GQ>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(fblk + BB);
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(bars + kDecWarps);

  // locate (layer, unit, cta index)
  int li = 0;
  while (li + 1 < P.n_layers && (int)blockIdx.x >= P.L[li + 1].cta_begin) ++li;
  const DecLayer& Ld = P.L[li];
  const int local = blockIdx.x - Ld.cta_begin;
  const int unit = local / Ld.n_ctas, cidx = local % Ld.n_ctas;
  const int layer = P.layer_begin + li;
  // the GQ query heads of kv head h of sequence b are rows unit*GQ .. unit*GQ+GQ-1
  const __nv_bfloat16* qrow = q + ((size_t)li * P.units + unit) * GQ * D;
  uint8_t* ubase = packed + Ld.packed_off + (size_t)unit * Ld.cap_groups * BB;

  // the unit's queries, staged once for every warp
  for (int i = threadIdx.x; i < GQ * D / 8; i += kThreads)
    reinterpret_cast<uint4*>(qs)[i] = reinterpret_cast<const uint4*>(qrow)[i];
  WarpState<D, GQ> st;
  state_init(st);
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" :: "r"(smem_u32(&bars[warp])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  unsigned phase = 0;
  const size_t wunit = (size_t)layer * P.units + unit;
  __nv_bfloat16* wk = win_k + wunit * P.R * D;
  __nv_bfloat16* wv = win_v + wunit * P.R * D;
  const bool flush = cidx == 0 && Ld.flush_start >= 0;
  const __nv_bfloat16* kn = P.k_new + ((size_t)li * P.units + unit) * D;
  const __nv_bfloat16* vn = P.v_new + ((size_t)li * P.units + unit) * D;
  // the new token: window chunk holding it (-1 if it left the window with a flush); the
  // CTA covering that chunk (CTA 0 after a flush) stores it into the ring
  int new_chunk = -1;
  if (Ld.new_slot >= 0) {
    new_chunk = Ld.win_len > 0 ? (Ld.win_len - 1) / kSlotsPerWarp : -1;
    const int owner = new_chunk >= 0 ? new_chunk / Ld.cpc : 0;
    if (cidx == owner)
      for (int c = threadIdx.x; c < D; c += kThreads)
        window_store(wk, wv, Ld.new_slot, c, D, kn[c], vn[c]);
  }
  __syncthreads();   // queries staged
  QRegs<D, GQ> qr;
  load_qregs<D, GQ>(qr, qs);
  if (flush) {
    // quantize the oldest group of the window into a new packed block (the new token
    // belongs to it only when R == 32, and then this CTA stored it above)
    __syncthreads();
    GroupSmem<D, kThreads>& gs = *reinterpret_cast<GroupSmem<D, kThreads>*>(dsm);
    for (int i = threadIdx.x; i < KVC_GROUP * D; i += kThreads) {
      const int t = i / D, c = i % D;
      gs.k[t][c] = __bfloat162float(window_load_k(wk, Ld.flush_start + t, c, D));
      gs.v[t][c] = __bfloat162float(window_load_v(wv, Ld.flush_start + t, c, D));
    }
    __syncthreads();
    quantize_block<D, BITS, kThreads>(gs, fblk);
    __syncthreads();
    uint4* dst = reinterpret_cast<uint4*>(ubase + (size_t)Ld.n_groups * BB);
    const uint4* src = reinterpret_cast<const uint4*>(fblk);
    for (int i = threadIdx.x; i < BB / 16; i += kThreads) dst[i] = src[i];
    __syncthreads();   // the staging area is reused by the copies below
    if (warp == 0) packed_warp<D, BITS, GQ>(st, qr, fblk, 1, P.sl2);
  }
  // this CTA's chunks of the unit, round robin over the warps
  const int total = Ld.wchunks + (Ld.n_groups + kGroupsPerWarp - 1) / kGroupsPerWarp;
  const int cb = cidx * Ld.cpc, ce = min(cb + Ld.cpc, total);
  const int wend = min(ce, Ld.wchunks);
  bool ok = true;
  for (int ch = cb + warp; ch < wend; ch += kDecWarps) {
    const int pos0 = ch * kSlotsPerWarp;
    const int n_valid = min(kSlotsPerWarp, Ld.win_len - pos0);
    const int slot0 = (Ld.win_start + pos0) % P.R;
    __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(wbuf);
    uint32_t* sv = reinterpret_cast<uint32_t*>(wbuf + kSlotsPerWarp * D * 2);
    ok = warp_stage(&bars[warp], phase++, sk, wk + (size_t)slot0 * D,
                    (uint32_t)(kSlotsPerWarp * D * 2), sv, wv + (size_t)(slot0 >> 1) * D * 2,
                    (uint32_t)(kSlotsPerWarp * D * 2), P.err);
    if (!ok) break;
    if (ch == new_chunk) {
      // the new token was stored through the generic path in this launch: take it
      // from the inputs rather than from the asynchronous copy
      const int r = Ld.new_slot - slot0;
      __nv_bfloat16* svh = reinterpret_cast<__nv_bfloat16*>(sv);
      for (int c = lane; c < D; c += 32) {
        sk[win_k_index(r, c, D)] = kn[c];
        svh[win_v_index(r, c, D)] = vn[c];
      }
      __syncwarp();
    }
    window_warp<D, GQ>(st, qs, sk, sv, n_valid, P.sl2);
  }
  // packed chunks continue the round robin where the window chunks left off
  if (ok) {
    const int first = max(cb, Ld.wchunks);
    int ch = first + ((warp - (first - cb)) % kDecWarps + kDecWarps) % kDecWarps;
    for (; ch < ce; ch += kDecWarps) {
      const int g0 = (ch - Ld.wchunks) * kGroupsPerWarp;
      const int ng = min(kGroupsPerWarp, Ld.n_groups - g0);
      if (!warp_stage(&bars[warp], phase++, wbuf, ubase + (size_t)g0 * BB,
                      (uint32_t)(ng * BB), nullptr, nullptr, 0u, P.err))
        break;
      packed_warp<D, BITS, GQ>(st, qr, wbuf, ng, P.sl2);
    }
  }
  __syncthreads();   // every warp is done with the staging area
  warp_to_smem<D, GQ>(st, sm, warp, P.sl2);
  __syncthreads();

  // merge the CTA's warps into one partial: part[cta][head][0..D+1] = (m, l, o[D]);
  // the per-(head, warp) weights are computed once
  if (threadIdx.x < GQ) {
    const int r = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm.m[w][r]);
    float L = 0.f;
    for (int w = 0; w < kDecWarps; ++w) {
      const float f = sm.l[w][r] > 0.f ? exp2f(sm.m[w][r] - M) : 0.f;
      sm.wt[w][r] = f;
      L += sm.l[w][r] * f;
    }
    sm.M[r] = M;
    sm.L[r] = L;
  }
  __syncthreads();
  if (Ld.n_ctas == 1) {
    // the whole unit ran in this CTA: no partials to merge
    float* o = out + ((size_t)li * P.units + unit) * GQ * D;
    for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
      const int r = i / D, cch = i % D;
      float O = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) O += sm.o[w][r][cch] * sm.wt[w][r];
      o[(size_t)r * D + cch] = O / sm.L[r];
    }
    return;
  }
  float* mypart = part + (size_t)blockIdx.x * GQ * (D + 2);
  for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
    const int r = i / D, cch = i % D;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) O += sm.o[w][r][cch] * sm.wt[w][r];
    mypart[r * (D + 2) + 2 + cch] = O;
    if (cch == 0) { mypart[r * (D + 2)] = sm.M[r]; mypart[r * (D + 2) + 1] = sm.L[r]; }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned t = atomicAdd(&tickets[(size_t)layer * P.units + unit], 1u);
    sm.last = (t == (unsigned)(Ld.n_ctas - 1));
    if (sm.last) tickets[(size_t)layer * P.units + unit] = 0u;
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  // the last CTA of the unit merges all partials: (m, l) of every split in one batch
  // of loads, the weights once per (head, split), then independent output loads
  const int nc = Ld.n_ctas;
  const float* up = part + (size_t)(Ld.cta_begin + unit * nc) * GQ * (D + 2);
  float* o = out + ((size_t)li * P.units + unit) * GQ * D;
  constexpr int kMlOff = ((int)sizeof(DecSmem<D, GQ>) + 15) / 16 * 16;
  float* ml = reinterpret_cast<float*>(dsm + kMlOff);
  if (kMlOff + nc * GQ * 2 * (int)sizeof(float) <= stage_bytes<D, BITS, GQ>()) {
    for (int idx = threadIdx.x; idx < nc * GQ; idx += kThreads) {
      const float* ps = up + (size_t)idx * (D + 2);   // idx = s * GQ + r
      ml[2 * idx] = __ldcg(ps);
      ml[2 * idx + 1] = __ldcg(ps + 1);
    }
    __syncthreads();
    if (threadIdx.x < GQ) {
      const int r = threadIdx.x;
      float M = -INFINITY;
      for (int s = 0; s < nc; ++s) M = fmaxf(M, ml[2 * (s * GQ + r)]);
      float L = 0.f;
      for (int s = 0; s < nc; ++s) {
        const float ls = ml[2 * (s * GQ + r) + 1];
        const float f = ls > 0.f ? exp2f(ml[2 * (s * GQ + r)] - M) : 0.f;
        ml[2 * (s * GQ + r)] = f;      // the weight replaces the max
        L += ls * f;
      }
      sm.L[r] = L;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
      const int r = i / D, cch = i % D;
      float O = 0.f;
#pragma unroll 4
      for (int s = 0; s < nc; ++s)
        O += ml[2 * (s * GQ + r)] * __ldcg(up + ((size_t)s * GQ + r) * (D + 2) + 2 + cch);
      o[(size_t)r * D + cch] = O / sm.L[r];
    }
  } else {
    for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
      const int r = i / D, cch = i % D;
      float M = -INFINITY;
      for (int s = 0; s < nc; ++s) M = fmaxf(M, __ldcg(up + ((size_t)s * GQ + r) * (D + 2)));
      float L = 0.f, O = 0.f;
      for (int s = 0; s < nc; ++s) {
        const float* ps = up + ((size_t)s * GQ + r) * (D + 2);
        const float ls = __ldcg(ps + 1);
        if (ls > 0.f) {
          const float f = exp2f(__ldcg(ps) - M);
          L += ls * f;
          O += __ldcg(ps + 2 + cch) * f;
        }
      }
      o[(size_t)r * D + cch] = O / L;
    }
  }
}

template <int D, int BITS, int GQ>
cudaError_t launch_one(const DecParams& P, int ctas, const kvc_cache* c,
                       const __nv_bfloat16* q, float* out, cudaStream_t stream) {
  constexpr int sm = dyn_smem_bytes<D, BITS, GQ>();
  // kernel attributes are set once per device for each instantiation
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(configured & (1ull << dev))) {
    e = cudaFuncSetAttribute(decode_kernel<D, BITS, GQ>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_kernel<D, BITS, GQ>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured |= 1ull << dev;
  }
  decode_kernel<D, BITS, GQ><<<ctas, kThreads, sm, stream>>>(P, c->packed, c->win_k, c->win_v, q,
                                                             out, c->dec_part, c->tickets);
  return cudaSuccess;
}

template <int D, int BITS>
cudaError_t launch_g(const DecParams& P, int ctas, const kvc_cache* c, const __nv_bfloat16* q,
                     float* out, cudaStream_t stream) {
  switch (c->g) {
    case 1: return launch_one<D, BITS, 1>(P, ctas, c, q, out, stream);
    case 2: return launch_one<D, BITS, 2>(P, ctas, c, q, out, stream);
    case 4: return launch_one<D, BITS, 4>(P, ctas, c, q, out, stream);
    case 8: return launch_one<D, BITS, 8>(P, ctas, c, q, out, stream);
    default: return cudaErrorInvalidValue;
  }
}

// CTAs of the decode kernel that fit on the device at once.
int resident_ctas(const kvc_cache* c) {
  static int cached[64][2][2][4] = {};
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 456;
  const int di = c->dims.head_dim == 128, bi = c->dims.bits == 4;
  const int gi = c->g == 1 ? 0 : c->g == 2 ? 1 : c->g == 4 ? 2 : 3;
  int& v = cached[dev][di][bi][gi];
  if (v) return v;
  int per = 0;
  cudaError_t e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
#define KVC_OCC(DD, BB2, GG)                                                                  \
  if (e == cudaSuccess) {                                                                     \
    e = cudaFuncSetAttribute(decode_kernel<DD, BB2, GG>,                                      \
                             cudaFuncAttributeMaxDynamicSharedMemorySize,                     \
                             dyn_smem_bytes<DD, BB2, GG>());                                  \
    if (e == cudaSuccess)                                                                     \
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, decode_kernel<DD, BB2, GG>,     \
                                                        kThreads, dyn_smem_bytes<DD, BB2, GG>()); \
  }
#define KVC_OCC_G(DD, BB2)                                                            \
  switch (c->g) {                                                                      \
    case 1: KVC_OCC(DD, BB2, 1) break; case 2: KVC_OCC(DD, BB2, 2) break;              \
    case 4: KVC_OCC(DD, BB2, 4) break; default: KVC_OCC(DD, BB2, 8) break;             \
  }
  if (c->dims.head_dim == 128) { if (c->dims.bits == 2) { KVC_OCC_G(128, 2) } else { KVC_OCC_G(128, 4) } }
  else { if (c->dims.bits == 2) { KVC_OCC_G(64, 2) } else { KVC_OCC_G(64, 4) } }
#undef KVC_OCC_G
#undef KVC_OCC
  if (e != cudaSuccess || per < 1) { cudaGetLastError(); per = 1; }
  v = n_sm * per;
  return v;
}

// Shared host path: a non-null k_new selects the fused append + flush + attention.
cudaError_t launch_common(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* q, const __nv_bfloat16* k_new,
                          const __nv_bfloat16* v_new, const int* flush_flags, float* out,
                          cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  const int units = d.batch * d.n_kv_heads;
  const int D = d.head_dim, R = d.window_len;
  const bool appending = k_new != nullptr;
  for (int base = 0; base < layer_count; base += KVC_MAX_LAUNCH_LAYERS) {
    const int cnt = layer_count - base < KVC_MAX_LAUNCH_LAYERS ? layer_count - base
                                                               : KVC_MAX_LAUNCH_LAYERS;
    DecParams P;
    P.n_layers = cnt;
    P.layer_begin = layer_begin + base;
    P.units = units;
    P.R = R;
    P.sl2 = 1.4426950408889634f / sqrtf((float)D);
    P.err = c->err;
    P.k_new = appending ? k_new + (size_t)base * units * D : nullptr;
    P.v_new = appending ? v_new + (size_t)base * units * D : nullptr;
    int ctas = 0;
    for (int i = 0; i < cnt; ++i) {
      const LayerState& ls = c->L[layer_begin + base + i];
      DecLayer& L = P.L[i];
      L.n_groups = ls.n_groups;
      L.cap_groups = ls.cap_groups;
      L.packed_off = (long long)ls.packed_off;
      bool flush = false;
      if (appending) {
        flush = flush_flags[base + i] != 0;
        L.new_slot = (ls.win_start + ls.win_len) % R;
        L.flush_start = flush ? ls.win_start : -1;
        L.win_start = flush ? (ls.win_start + KVC_GROUP) % R : ls.win_start;
        L.win_len = ls.win_len + 1 - (flush ? KVC_GROUP : 0);
      } else {
        L.new_slot = -1;
        L.flush_start = -1;
        L.win_start = ls.win_start;
        L.win_len = ls.win_len;
      }
      L.wchunks = (L.win_len + kSlotsPerWarp - 1) / kSlotsPerWarp;
      L.cta_begin = 0;
      L.n_ctas = 0;
      L.cpc = 0;
    }
    // chunks per CTA: the smallest multiple of the warp count that keeps the whole
    // grid resident in one wave
    const int capacity = resident_ctas(c);
    int cpc = kDecWarps;
    for (;;) {
      ctas = 0;
      for (int i = 0; i < cnt; ++i) {
        const DecLayer& L = P.L[i];
        const int chunks = L.wchunks + (L.n_groups + kGroupsPerWarp - 1) / kGroupsPerWarp;
        ctas += units * std::max(1, (chunks + cpc - 1) / cpc);
      }
      if (ctas <= capacity || cpc >= 1024) break;
      cpc += kDecWarps;
    }
    ctas = 0;
    for (int i = 0; i < cnt; ++i) {
      DecLayer& L = P.L[i];
      const int chunks = L.wchunks + (L.n_groups + kGroupsPerWarp - 1) / kGroupsPerWarp;
      L.cpc = cpc;
      L.n_ctas = std::max(1, (chunks + cpc - 1) / cpc);
      L.cta_begin = ctas;
      ctas += units * L.n_ctas;
    }
    if ((size_t)ctas * c->g * (D + 2) > c->dec_part_elems) return cudaErrorInvalidValue;
    const __nv_bfloat16* qb = q + (size_t)base * units * c->g * D;
    float* ob = out + (size_t)base * units * c->g * D;
    cudaError_t e;
    if (D == 128 && d.bits == 2) e = launch_g<128, 2>(P, ctas, c, qb, ob, stream);
    else if (D == 128 && d.bits == 4) e = launch_g<128, 4>(P, ctas, c, qb, ob, stream);
    else if (D == 64 && d.bits == 2) e = launch_g<64, 2>(P, ctas, c, qb, ob, stream);
    else if (D == 64 && d.bits == 4) e = launch_g<64, 4>(P, ctas, c, qb, ob, stream);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* q, float* out, cudaStream_t stream) {
  return launch_common(c, layer_begin, layer_count, q, nullptr, nullptr, nullptr, out, stream);
}

cudaError_t launch_decode_step(const kvc_cache* c, int layer_begin, int layer_count,
                               const __nv_bfloat16* q, const __nv_bfloat16* k_new,
                               const __nv_bfloat16* v_new, const int* flush_flags, float* out,
                               cudaStream_t stream) {
  return launch_common(c, layer_begin, layer_count, q, k_new, v_new, flush_flags, out, stream);
}

}  // namespace kvc
