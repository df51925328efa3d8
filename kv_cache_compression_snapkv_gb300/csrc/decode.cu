// decode.cu -- decode attention over the packed cache plus the bf16 window,
// optionally fused with the append of the step's new token.
//
// MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
// Cache, §2 eq. (1) and Algorithm 1 (decoding): append the new key/value to the
// 16-bit buffer, quantize when it fills, then one softmax over the dequantized
// packed keys and the buffer's keys; output = A_quant . dequant(Q_V) +
// A_unquant . R_V. Blog "KV Cache Compression: Eviction and Quantization",
// "Measured on a real model": exact recent window, rounded rest, one softmax.
//
// Work decomposition (one launch for a range of layers): a unit = (layer,
//   sequence b, kv head h); its work is cut into chunks of 16 window slots or
//   GPC packed group blocks (GPC = groups that fill one window chunk's bytes: 2 at
//   2 bits, 1 at 4 bits). The chunks of every unit of the launch are laid end to
//   end (layer by layer, unit by unit) and the list is cut into equal contiguous
//   ranges, one per warp of the grid (one CTA per SM): a split-K over the whole
//   launch, so a large unit is spread over many warps of many SMs and small units
//   share a warp, and every warp gets the same number of chunks. Each warp
//   double-buffers its chunks in shared memory with bulk asynchronous copies
//   (cp.async.bulk on per-slot mbarriers, bounded waits); the copy of a unit's
//   first chunk also brings the unit's g queries. A warp keeps an online softmax
//   of the g query heads over the part of a unit it holds. A unit held whole by
//   one warp is normalised and written by it; otherwise each holder writes its
//   partial state (m, l, o) to a workspace in global memory and takes a ticket
//   from the unit's arrival counter, and the holder that arrives last merges
//   the partial states with a log-sum-exp combine in a fixed order (the result
//   does not depend on arrival order), writes the fp32 output and resets the
//   counter. Nothing waits on another warp or CTA.
//   The new token of a fused step is stored into the ring by the warp whose
//   window chunk holds its slot (which also patches its staged copy). A step in
//   which some layer's window reaches R runs the append kernel first (it stores
//   the new tokens and quantizes the oldest group of each full window) and then
//   this kernel over the updated cache. Layers of one launch may differ in
//   precision (2 or 4 bits, or 16: window only) and in ring length.
//
// Arithmetic. Per 32-token group block the key logits are
//     q . k_t = sum_c (q_c S_c) code_tc + sum_c q_c Z_c
// and the value output is
//     o_c = sum_t (p_t S_t,gc) code_tc + sum_t p_t Z_t,gc.
// Both code sums run on the tensor cores (mma m16n8k16, fp16 operands, fp32
// accumulate): codes are unpacked in registers to exact fp16 integers, and the
// fp16 operand products (q_c S_c, p_t S_t) are split into hi + lo fp16 parts in
// adjacent columns of the 8-column operand (column 2h hi, 2h + 1 lo for head h),
// so the rounding of the operand does not limit accuracy. The key zero-point sums
// are one small extra product per chunk (q against the chunk's groups' key zeros).
// The value zero-point sums are products of the zero-points (every row of a channel
// group carrying Z_t) against hi/lo(p), accumulated into the same registers as the
// code sums of the same 16 tokens: the two terms nearly cancel (the code term is
// about +range/2 times the weight, the zero term about -range/2 times it), so
// keeping them apart would leave a small result as the difference of two large
// fp32 sums over all tokens. The window runs the same flow on bf16 operands.
#include <algorithm>
#include <utility>

#include "quant_device.cuh"

namespace kvc {
namespace {

constexpr int kSlotsPerWarp = kDecSlotsPerChunk;
static_assert(kSlotsPerWarp == 16, "window warps take 16 slots");
constexpr unsigned kWaitLimit = 1u << 20;   // bounded mbarrier polls (far above any copy)

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

// v as a bf16 pair (hi, lo) with hi = bf16(v), lo = bf16(v - hi): hi in the low half.
__device__ __forceinline__ uint32_t split_bf16(float v) {
  const float hi = __bfloat162float(__float2bfloat16_rn(v));
  const __nv_bfloat162 p = __floats2bfloat162_rn(v, v - hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// The masks of the code fields inside a byte of each 16-bit half, held in
// registers: with the mask a register operand, the field and the fp16 exponent
// bits are merged by one three-input logic instruction with the exponent as its
// immediate (a mask and an exponent both as immediates take two).
template <int BITS>
struct CodeMasks { uint32_t m[8 / BITS]; };

template <int BITS>
__device__ __forceinline__ CodeMasks<BITS> code_masks() {
  CodeMasks<BITS> cm;
  static_for<8 / BITS>([&](auto J_) {
    constexpr int J = decltype(J_)::value;
    constexpr uint32_t v = (((1u << BITS) - 1u) * 0x00010001u) << (BITS * J);
    asm volatile("mov.b32 %0, %1;" : "=r"(cm.m[J]) : "n"(v));
  });
  return cm;
}

// Exact fp16 pair of the two codes in pair slot P of word w (w8 = w >> 8). The
// field of slot P is masked in place under the fp16 exponent of 2^e, e = 10 -
// BITS*j (j = field index inside its byte), so each half reads 2^e + code; one
// subtraction leaves the code.
template <int BITS, int P>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, uint32_t w8, const CodeMasks<BITS>& cm) {
  constexpr int CPB = 8 / BITS, SB = P / CPB, J = P % CPB;
  constexpr uint32_t mag = ((uint32_t)(25 - BITS * J) << 10) * 0x00010001u;
  uint32_t v;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(SB ? w8 : w), "r"(cm.m[J]), "n"(mag));
  return h2u(__hsub2(u2h(v), u2h(mag)));
}

// A operand of key product (MT, KS) (rows = tokens, k = channels) from the lane's
// key code words.
template <int D, int BITS, int MT, int KS>
__device__ __forceinline__ void key_afrag(const uint32_t* kw, const CodeMasks<BITS>& cm,
                                          uint32_t (&a)[4]) {
  if constexpr (BITS == 2) {
    constexpr int wi = MT * (D / 32) + KS / 2, b = 2 * (KS & 1);
    const uint32_t w = kw[wi], w8 = w >> 8;
    a[0] = unpack_pair<2, b>(w, w8, cm);
    a[1] = unpack_pair<2, 4 + b>(w, w8, cm);
    a[2] = unpack_pair<2, b + 1>(w, w8, cm);
    a[3] = unpack_pair<2, 5 + b>(w, w8, cm);
  } else {
    constexpr int wi = MT * (D / 16) + KS;
    const uint32_t w = kw[wi], w8 = w >> 8;
    a[0] = unpack_pair<4, 0>(w, w8, cm);
    a[1] = unpack_pair<4, 2>(w, w8, cm);
    a[2] = unpack_pair<4, 1>(w, w8, cm);
    a[3] = unpack_pair<4, 3>(w, w8, cm);
  }
}
// A operand of value product (MT, KS) (rows = channels, k = tokens).
template <int BITS, int MT, int KS>
__device__ __forceinline__ void value_afrag(const uint32_t* vw, const CodeMasks<BITS>& cm,
                                            uint32_t (&a)[4]) {
  if constexpr (BITS == 2) {
    constexpr int b = 2 * KS;
    const uint32_t w = vw[MT], w8 = w >> 8;
    a[0] = unpack_pair<2, b>(w, w8, cm);
    a[1] = unpack_pair<2, 4 + b>(w, w8, cm);
    a[2] = unpack_pair<2, b + 1>(w, w8, cm);
    a[3] = unpack_pair<2, 5 + b>(w, w8, cm);
  } else {
    constexpr int wi = 2 * MT + KS;
    const uint32_t w = vw[wi], w8 = w >> 8;
    a[0] = unpack_pair<4, 0>(w, w8, cm);
    a[1] = unpack_pair<4, 2>(w, w8, cm);
    a[2] = unpack_pair<4, 1>(w, w8, cm);
    a[3] = unpack_pair<4, 3>(w, w8, cm);
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
        float2 f = make_float2(0.f, 0.f);
        if (h < GQ) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(qs + h * D + c));
        const __half2 q2 = __float22half2_rn(f);
        qr.qh[u][ks][e2] = h2u(q2);
        qr.qn[u][ks][e2] = (gid & 1) ? h2u(__hneg2(q2)) : 0u;
      }
  }
}

// Online-softmax update with the logits of 16 * NMT tokens: x[u][mt][r] is token
// 16mt + gid + 8r for head 4u + tid. The weights replace the logits.
template <int D, int GQ, int NMT>
__device__ __forceinline__ void softmax_update(WarpState<D, GQ>& st,
                                               float (&x)[n_tiles<GQ>()][NMT][2], float sl2) {
#pragma unroll
  for (int u = 0; u < n_tiles<GQ>(); ++u) {
    float gm = fmaxf(x[u][0][0], x[u][0][1]);
#pragma unroll
    for (int mt = 1; mt < NMT; ++mt) gm = fmaxf(gm, fmaxf(x[u][mt][0], x[u][mt][1]));
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
      st.m[u] = mnew;
    }
    const float msl = (st.m[u] == -INFINITY) ? 0.f : st.m[u] * sl2;
    float s = 0.f;
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
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
// `base` points at n_grp (<= 8) consecutive group blocks in shared
// memory. Per group: key logits (rows = tokens), one online-softmax update, the
// value products (rows = channels). The group loop stays rolled so that the hot
// code fits the instruction cache.
template <int D, int BITS, int GQ>
__device__ void packed_warp(WarpState<D, GQ>& st, const QRegs<D, GQ>& qr, const uint8_t* base,
                            int n_grp, float sl2) {
  constexpr int KS = D / 16, NGC = D / 32, BB = 8 * D * (BITS + 1), WPL = D * BITS / 32;
  constexpr int NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;

  const CodeMasks<BITS> cm = code_masks<BITS>();
  // key zero-point sums of every group of the chunk: C[group][n] = Z_group . q_n
  // (A rows = groups; rows past the chunk's groups repeat group 0 and are not
  // read; B = the queries, whose "hi" column is read)
  float zb[NH];
  {
    uint32_t za[KS][2];
    const int gz = gid < n_grp ? gid : 0;
    const uint4* zp = reinterpret_cast<const uint4*>(base + (size_t)gz * BB + off_kzero(D, BITS) +
                                                     tid * (D / 4) * 2);
#pragma unroll
    for (int i = 0; i < KS / 2; ++i) {
      const uint4 z = zp[i];
      za[2 * i][0] = z.x;
      za[2 * i][1] = z.y;
      za[2 * i + 1][0] = z.z;
      za[2 * i + 1][1] = z.w;
    }
#pragma unroll
    for (int u = 0; u < NH; ++u) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
        mma_f16(c, za[ks][0], 0u, za[ks][1], 0u, qr.qh[u][ks][0], qr.qh[u][ks][1]);
      zb[u] = c[0];   // group gid, head 4u + tid ("hi" column)
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
          key_afrag<D, BITS, MT, K>(kw, cm, a);
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
    softmax_update<D, GQ, 2>(st, x, sl2);

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
    const uint32_t* vs = reinterpret_cast<const uint32_t*>(blk + off_vscale(D, BITS));
    const uint32_t* vz = reinterpret_cast<const uint32_t*>(blk + off_vzero(D, BITS));
    static_for<2>([&](auto KS_) {
      constexpr int K = decltype(KS_)::value;
      // scales of this lane's tokens (16K + gid, 16K + gid + 8) for every channel group
      uint32_t S2[NGC];
      if constexpr (NGC == 4) {
        const uint4 v4 = *reinterpret_cast<const uint4*>(vs + (K * 8 + gid) * NGC);
        S2[0] = v4.x; S2[1] = v4.y; S2[2] = v4.z; S2[3] = v4.w;
      } else {
        const uint2 v2 = *reinterpret_cast<const uint2*>(vs + (K * 8 + gid) * NGC);
        S2[0] = v2.x; S2[1] = v2.y;
      }
#pragma unroll
      for (int u = 0; u < NH; ++u) {
        // p of the two tokens as fp16 pairs hi (ph) + lo (pl), p = ph + pl
        const float p0 = x[u][K][0], p1 = x[u][K][1];
        const __half2 ph = __floats2half2_rn(p0, p1);
        const float2 phf = __half22float2(ph);
        const __half2 pl = __floats2half2_rn(p0 - phf.x, p1 - phf.y);
        // zero-point term operand: (hi, lo) of p per token
        const uint32_t bz0 = movm_t(__byte_perm(h2u(ph), h2u(pl), 0x5410));
        const uint32_t bz1 = movm_t(__byte_perm(h2u(ph), h2u(pl), 0x7632));
        static_for<NGC>([&](auto GC_) {
          constexpr int GC = decltype(GC_)::value;
          const uint32_t z0 = vz[(8 * K + tid) * NGC + GC];
          const uint32_t z1 = vz[(8 * K + 4 + tid) * NGC + GC];
          // (hi, lo) of p * S: hi = fp16(ph S), lo = fp16(pl S + (ph S - hi)), the
          // remainder of the fp16 product exact through the fused multiply-add
          const __half2 s2 = u2h(S2[GC]);
          const __half2 hi = __hmul2(ph, s2);
          const __half2 lo = __hfma2(pl, s2, __hfma2(ph, s2, __hneg2(hi)));
          const uint32_t b0 = movm_t(__byte_perm(h2u(hi), h2u(lo), 0x5410));
          const uint32_t b1 = movm_t(__byte_perm(h2u(hi), h2u(lo), 0x7632));
          static_for<2>([&](auto H_) {
            constexpr int MV = 2 * GC + decltype(H_)::value;
            uint32_t a[4];
            value_afrag<BITS, MV, K>(vw, cm, a);
            mma_f16(st.o[u][MV], z0, z0, z1, z1, bz0, bz1);
            mma_f16(st.o[u][MV], a[0], a[1], a[2], a[3], b0, b1);
          });
        });
      }
    });
  }
}

// ------------------------------------------------------------- window slots
// wk: 16 staged key rows (win_k_index layout, first slot a multiple of 16); wv: 8
// staged value pair rows (win_v_index layout); the first n_valid slots are live.
// bf16 products, exact queries, hi/lo weights.
template <int D, int GQ>
__device__ void window_warp(WarpState<D, GQ>& st, const __nv_bfloat16* qs, const __nv_bfloat16* wk,
                            const uint32_t* wv, int n_valid, float sl2) {
  constexpr int KS = D / 16, NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  float x[NH][1][2];
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
    float acc[NH][2][4];
#pragma unroll
    for (int u = 0; u < NH; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) { acc[u][0][e] = 0.f; acc[u][1][e] = 0.f; }
    // rows gid (rl 0) and gid + 8 (rl 1); 16-byte chunks swizzled by gid
    const uint4* r0 = reinterpret_cast<const uint4*>(wk + (size_t)gid * D);
    const uint4* r1 = reinterpret_cast<const uint4*>(wk + (size_t)(gid + 8) * D);
#pragma unroll
    for (int i = 0; i < KS / 2; ++i) {
      const int ch = (tid * (KS / 2) + i) ^ gid;
      const uint4 u0 = r0[ch], u1 = r1[ch];
#pragma unroll
      for (int u = 0; u < NH; ++u) {
        mma_bf16(acc[u][0], u0.x, u1.x, u0.y, u1.y, bq[u][2 * i][0], bq[u][2 * i][1]);
        mma_bf16(acc[u][1], u0.z, u1.z, u0.w, u1.w, bq[u][2 * i + 1][0], bq[u][2 * i + 1][1]);
      }
    }
#pragma unroll
    for (int u = 0; u < NH; ++u)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float v = (acc[u][0][2 * r] + acc[u][0][2 * r + 1]) +
                        (acc[u][1][2 * r] + acc[u][1][2 * r + 1]);
        x[u][0][r] = (gid + 8 * r) < n_valid ? v : -INFINITY;
      }
  }
  softmax_update<D, GQ, 1>(st, x, sl2);
  uint32_t b0[NH], b1[NH];
#pragma unroll
  for (int u = 0; u < NH; ++u) {
    b0[u] = movm_t(split_bf16(x[u][0][0]));
    b1[u] = movm_t(split_bf16(x[u][0][1]));
  }
  // pair rows tid (tokens 2tid, 2tid + 1) and 4 + tid (tokens 8 + 2tid, +1); chunks
  // swizzled by tid
  const uint4* p0 = reinterpret_cast<const uint4*>(wv + (size_t)tid * D);
  const uint4* p1 = reinterpret_cast<const uint4*>(wv + (size_t)(4 + tid) * D);
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

// ------------------------------------------------------------ launch layout
struct DecLayer {
  long long chunk_begin;  // first chunk of the layer in the launch's chunk list
  long long packed_off;   // byte offset of the layer inside the packed store
  long long win_off;      // element offset of the layer's window rings
  int n_groups;           // packed groups read (a group flushed in this step included)
  int win_start;          // ring start slot after this launch's append
  int win_len;            // window tokens after this launch's append
  int cap_groups;
  int new_slot;           // ring slot of the token appended in this launch, or -1
  int wchunks;            // window chunks (16 slots) per unit; packed chunks follow
  int pchunks;            // packed chunks per unit
  int gpc;                // packed groups per chunk
  int R;                  // ring length
  int bits;               // 2, 4 or 16 (16: no packed chunks)
};

struct DecParams {
  DecLayer L[KVC_MAX_LAUNCH_LAYERS];
  const __nv_bfloat16* k_new;   // [n_layers][units][D] (fused append only)
  const __nv_bfloat16* v_new;
  unsigned* err;                // device error word (bit 0: a staging wait gave up)
  float* ws;                    // partial states, two per CTA: [2 * grid][dep_floats]
  unsigned* cnt;                // arrival tickets per (layer, unit) of the cache; zero between launches
  long long total;              // chunks in the launch
  int n_vwarps;                 // warps of the grid
  int n_layers;                 // layers in this launch
  int layer_begin;              // absolute index of L[0]
  int units;                    // batch * n_kv_heads
  unsigned wait_limit;          // polls of one staging wait before it gives up
  float sl2;                    // log2(e) / sqrt(head_dim)
};

// One partial state in the workspace: o[GQ][D] (unnormalised; both column parts
// and the value zero-point sums folded in), then m[GQ] (log2 units) and l[GQ],
// padded to a whole number of 16-byte vectors so that every o starts aligned.
__host__ __device__ constexpr int dep_floats(int D, int GQ) { return GQ * D + (2 * GQ + 3) / 4 * 4; }

// BMASK: bit 0 = the launch has 2-bit layers, bit 1 = 4-bit layers (the packed
// code of each present precision is instantiated; 16-bit layers need neither).
template <int D, int GQ, int BMASK>
struct DecCfg {
  static constexpr int WB = kSlotsPerWarp * D * 4;   // one window chunk (keys + values)
  static constexpr int PB2 = (BMASK & 1) ? dec_groups_per_chunk(D, 2) * block_bytes(D, 2) : 0;
  static constexpr int PB4 = (BMASK & 2) ? dec_groups_per_chunk(D, 4) * block_bytes(D, 4) : 0;
  static constexpr int SLOT = WB > PB2 ? (WB > PB4 ? WB : PB4) : (PB2 > PB4 ? PB2 : PB4);
  static constexpr int QB = GQ * D * 2;              // one unit's queries (bf16)
  static constexpr int DEPW = dep_floats(D, GQ);     // floats of one partial state
  static constexpr int per_warp = 2 * SLOT + 2 * QB + 2 * DEPW * 4 + 2 * 8 + 4;
  // warps per CTA: as many as shared memory holds, at most 12 (8 with four or more
  // query heads, whose state needs more registers per thread than 12 warps leave)
  static constexpr int pick(int nw) { return nw * per_warp <= 227 * 1024 ? nw : pick(nw - 1); }
  static constexpr int NW = pick(GQ > 2 ? 8 : 12);
  static constexpr int kThreads = NW * 32;
  static constexpr int oRing = 0;                    // [NW][2][SLOT]
  static constexpr int oDep = oRing + NW * 2 * SLOT; // [NW][2][DEPW] fp32 partial states
  static constexpr int oQ = oDep + NW * 2 * DEPW * 4;// [NW][2][GQ][D] bf16
  static constexpr int oBars = oQ + NW * 2 * QB;     // [NW][2] mbarriers
  static constexpr int oCnt = oBars + NW * 2 * 8;    // [NW] arrival tickets
  static constexpr int total = oCnt + NW * 4;
  static_assert(SLOT % 16 == 0 && QB % 16 == 0 && oDep % 16 == 0 && oBars % 8 == 0, "alignment");
  static_assert(NW >= 4, "at least four warps per CTA");
};

template <int D, int GQ>
__device__ void write_partial(WarpState<D, GQ>& st, float* dep, float sl2) {
  constexpr int NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
#pragma unroll
  for (int u = 0; u < NH; ++u) {
    const int h = 4 * u + tid;
    float l = st.l[u];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    if (h < GQ) {
      float* o = dep + h * D;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[16 * mt + gid] = st.o[u][mt][0] + st.o[u][mt][1];
        o[16 * mt + gid + 8] = st.o[u][mt][2] + st.o[u][mt][3];
      }
      if (gid == 0) {
        dep[GQ * D + h] = st.m[u] == -INFINITY ? -INFINITY : st.m[u] * sl2;
        dep[GQ * D + GQ + h] = l;
      }
    }
  }
}

// The warp's state normalised (o / l per head) into out[GQ][D].
template <int D, int GQ>
__device__ void write_final(WarpState<D, GQ>& st, float* __restrict__ out) {
  constexpr int NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
#pragma unroll
  for (int u = 0; u < NH; ++u) {
    const int h = 4 * u + tid;
    float l = st.l[u];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (h < GQ) {
      float* o = out + h * D;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[16 * mt + gid] = (st.o[u][mt][0] + st.o[u][mt][1]) * inv;
        o[16 * mt + gid + 8] = (st.o[u][mt][2] + st.o[u][mt][3]) * inv;
      }
    }
  }
}

template <bool GLOBAL>
__device__ __forceinline__ float ld_dep(const float* p) {
  if constexpr (GLOBAL) return __ldcg(p);
  else return *p;
}
template <bool GLOBAL>
__device__ __forceinline__ float4 ld_dep4(const float4* p) {
  if constexpr (GLOBAL) return __ldcg(p);
  else return *p;
}

// Log-sum-exp combine of the partial states dep_of(0 .. nc-1), in that order (the
// result does not depend on which holder arrived last). GLOBAL: the partials were
// written by other SMs and are read through L2; else they are in this CTA's
// shared memory. NORMALISE: out[GQ][D] = o / l; else out is written as one
// partial state (o, m, l) of the whole set. The maxima and weights are taken with
// the lanes spread over the contributors; the outputs then loop over the
// contributors with loads that do not depend on each other.
template <int D, int GQ, bool GLOBAL, bool NORMALISE, typename DepOf>
__device__ void merge_partials(int nc, DepOf dep_of, float* __restrict__ out) {
  constexpr int N4 = GQ * D / 4;            // float4 outputs
  constexpr int E4 = (N4 + 31) / 32;        // per lane
  const int lane = threadIdx.x & 31;
  float M[GQ];
#pragma unroll
  for (int h = 0; h < GQ; ++h) M[h] = -INFINITY;
  for (int w0 = 0; w0 < nc; w0 += 32) {
    if (w0 + lane < nc) {
      const float* d = dep_of(w0 + lane) + GQ * D;
#pragma unroll
      for (int h = 0; h < GQ; ++h)
        if (ld_dep<GLOBAL>(d + GQ + h) > 0.f) M[h] = fmaxf(M[h], ld_dep<GLOBAL>(d + h));
    }
  }
#pragma unroll
  for (int h = 0; h < GQ; ++h)
#pragma unroll
    for (int o = 16; o; o >>= 1) M[h] = fmaxf(M[h], __shfl_xor_sync(0xffffffffu, M[h], o));
  float4 acc[E4];
  float L[GQ];
#pragma unroll
  for (int i = 0; i < E4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int h = 0; h < GQ; ++h) L[h] = 0.f;
  // lane element i covers outputs 4 (lane + 32 i) .. + 3 (one head)
  for (int w0 = 0; w0 < nc; w0 += 32) {
    float f[GQ];
    if (w0 + lane < nc) {
      const float* d = dep_of(w0 + lane) + GQ * D;
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        const float l = ld_dep<GLOBAL>(d + GQ + h);
        f[h] = l > 0.f ? exp2f(ld_dep<GLOBAL>(d + h) - M[h]) : 0.f;
        L[h] += f[h] * l;
      }
    } else {
#pragma unroll
      for (int h = 0; h < GQ; ++h) f[h] = 0.f;
    }
    const int cnt = min(32, nc - w0);
#pragma unroll 4
    for (int k = 0; k < cnt; ++k) {
      const float4* o4 = reinterpret_cast<const float4*>(dep_of(w0 + k));
      float fk[GQ];
#pragma unroll
      for (int h = 0; h < GQ; ++h) fk[h] = __shfl_sync(0xffffffffu, f[h], k);
#pragma unroll
      for (int i = 0; i < E4; ++i) {
        const int idx = lane + 32 * i;
        if (idx < N4) {
          const float4 v = ld_dep4<GLOBAL>(o4 + idx);
          const float fh = fk[(4 * idx) / D];
          acc[i].x += fh * v.x; acc[i].y += fh * v.y; acc[i].z += fh * v.z; acc[i].w += fh * v.w;
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < GQ; ++h)
#pragma unroll
    for (int o = 16; o; o >>= 1) L[h] += __shfl_xor_sync(0xffffffffu, L[h], o);
  float4* out4 = reinterpret_cast<float4*>(out);
#pragma unroll
  for (int i = 0; i < E4; ++i) {
    const int idx = lane + 32 * i;
    if (idx < N4) {
      float inv = 1.f;
      if constexpr (NORMALISE) {
        const int h = (4 * idx) / D;
        inv = L[h] > 0.f ? 1.f / L[h] : 0.f;
      }
      out4[idx] = make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
    }
  }
  if constexpr (!NORMALISE) {
    if (lane < GQ) {
      float m = -INFINITY, l = 0.f;
#pragma unroll
      for (int h = 0; h < GQ; ++h)
        if (h == lane) { m = M[h]; l = L[h]; }
      out[GQ * D + lane] = m;
      out[GQ * D + GQ + lane] = l;
    }
  }
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// An even split of [base, base + T) into N contiguous ranges: range i is
// [first(i), first(i+1)), and owner(c) is the range holding c. When T * N < 2^32
// (every launch of ordinary size) all products fit 32 bits: 32-bit divisions.
struct Split {
  long long T, N, base;
  __device__ long long first(long long i) const {
    if (T * N < (1LL << 32)) return base + (long long)((unsigned)i * (unsigned)T / (unsigned)N);
    return base + i * T / N;
  }
  __device__ long long owner(long long c) const {
    const long long x = c - base;
    if (T * N < (1LL << 32))
      return (long long)((((unsigned)x + 1u) * (unsigned)N - 1u) / (unsigned)T);
    return ((x + 1) * N - 1) / T;
  }
};

template <int D, int GQ, int BMASK>
__global__ void __launch_bounds__(DecCfg<D, GQ, BMASK>::kThreads, 1)
decode_kernel(const DecParams P, uint8_t* __restrict__ packed, __nv_bfloat16* __restrict__ win_k,
              __nv_bfloat16* __restrict__ win_v, const __nv_bfloat16* __restrict__ q,
              float* __restrict__ out) {
  using C = DecCfg<D, GQ, BMASK>;
  constexpr int NW = C::NW;
  extern __shared__ __align__(128) uint8_t dsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(dsm + C::oBars) + warp * 2;
  uint8_t* ring = dsm + C::oRing + (size_t)warp * 2 * C::SLOT;
  float* sdep = reinterpret_cast<float*>(dsm + C::oDep);           // [NW][2][DEPW]
  unsigned* scnt = reinterpret_cast<unsigned*>(dsm + C::oCnt);     // [NW]
  __nv_bfloat16* qbuf = reinterpret_cast<__nv_bfloat16*>(dsm + C::oQ) + (size_t)warp * 2 * GQ * D;
  if (lane == 0) {
    mbar_init(&bar[0]);
    mbar_init(&bar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    scnt[warp] = 0u;
  }
  __syncthreads();
  pdl_wait();      // the previous kernels' writes (queries, cache) are visible
  pdl_release();
  // the launch's chunk list, cut into one contiguous range per CTA, each cut into one
  // contiguous range per warp
  const Split cs{P.total, (long long)gridDim.x, 0};
  const long long C0 = cs.first(blockIdx.x), C1 = cs.first(blockIdx.x + 1);
  const int nvw = (int)(C1 - C0 < NW ? C1 - C0 : NW);   // warps with chunks (>= 1: grid <= total)
  if (warp >= nvw) return;
  const Split ws{C1 - C0, (long long)nvw, C0};
  const long long c0 = ws.first(warp), c1 = ws.first(warp + 1);
  const int n = (int)(c1 - c0);   // >= 1

  // chunk cursor: layer, unit, chunk index j inside the unit, chunks per unit
  struct Cur { int li, unit, j, cpu; };
  auto cpu_of = [&](int li) { return P.L[li].wchunks + P.L[li].pchunks; };
  auto locate = [&](long long c) {
    Cur r;
    r.li = 0;
    while (r.li + 1 < P.n_layers && c >= P.L[r.li + 1].chunk_begin) ++r.li;
    r.cpu = cpu_of(r.li);
    const long long loc = c - P.L[r.li].chunk_begin;
    r.unit = (int)(loc / r.cpu);
    r.j = (int)(loc - (long long)r.unit * r.cpu);
    return r;
  };
  auto step = [&](Cur& r) {
    if (++r.j < r.cpu) return;
    r.j = 0;
    if (++r.unit < P.units) return;
    r.unit = 0;
    do { ++r.li; } while (r.li < P.n_layers && cpu_of(r.li) == 0);
    r.cpu = r.li < P.n_layers ? cpu_of(r.li) : 1;
  };
  // lane 0: stage chunk i (cursor r) into slot i & 1, with the unit's queries into
  // qbuf[qpar] when the chunk starts one of the warp's unit segments
  auto issue = [&](int i, const Cur& r, int qpar, bool with_q) {
    const DecLayer& L = P.L[r.li];
    uint64_t* b = &bar[i & 1];
    uint8_t* dst = ring + (i & 1) * C::SLOT;
    const uint32_t qb = with_q ? (uint32_t)C::QB : 0u;
    if (r.j < L.wchunks) {
      const size_t rb = (size_t)L.win_off + (size_t)r.unit * L.R * D;
      const int slot0 = (L.win_start + r.j * kSlotsPerWarp) % L.R;
      const uint32_t wb = (uint32_t)(kSlotsPerWarp * D * 2);
      mbar_expect(b, 2 * wb + qb);
      bulk_g2s(dst, win_k + rb + (size_t)slot0 * D, wb, b);
      bulk_g2s(dst + wb, win_v + rb + (size_t)(slot0 >> 1) * D * 2, wb, b);
    } else {
      const int bb = block_bytes(D, L.bits);
      const int g0 = (r.j - L.wchunks) * L.gpc;
      const int ng = min(L.gpc, L.n_groups - g0);
      const uint8_t* src = packed + L.packed_off + ((size_t)r.unit * L.cap_groups + g0) * bb;
      mbar_expect(b, (uint32_t)(ng * bb) + qb);
      bulk_g2s(dst, src, (uint32_t)(ng * bb), b);
    }
    if (with_q)
      bulk_g2s(qbuf + qpar * GQ * D, q + ((size_t)r.li * P.units + r.unit) * GQ * D, qb, b);
  };

  Cur cur = locate(c0), pre = cur;
  int pre_seg = 0;   // segment ordinal of the prefetch cursor's chunk
  auto produce = [&](int i) {   // all lanes: advance the prefetch cursor to chunk i; lane 0 issues
    if (i > 0) {
      step(pre);
      if (pre.j == 0) ++pre_seg;
    }
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      issue(i, pre, pre_seg & 1, i == 0 || pre.j == 0);
    }
  };
  produce(0);
  if (n > 1) produce(1);

  WarpState<D, GQ> st;
  QRegs<D, GQ> qr;
  int seg = -1;
  int fail = -1;   // chunk whose staging wait gave up
  // A segment = the chunks of one unit this warp holds. At its end the unit is
  // written whole; or its partial state goes to this CTA's shared memory, where the
  // last of the CTA's holders merges them; a unit that other CTAs also hold is
  // handed on as the CTA's partial state in global memory, where the last CTA
  // merges them. Tickets come from arrival counters (shared, then global); nothing
  // waits.
  auto finish = [&](const Cur& r, int seg_ord, bool failed) {
    const DecLayer& L = P.L[r.li];
    const long long ubeg = L.chunk_begin + (long long)r.unit * r.cpu, uend = ubeg + r.cpu;
    const size_t ul = (size_t)r.li * P.units + r.unit;
    float* o = out + ul * GQ * D;
    if (ubeg >= c0 && uend <= c1) {
      if (!failed) write_final<D, GQ>(st, o);
      return;
    }
    const long long lbeg = max(ubeg, C0), lend = min(uend, C1);   // the CTA's part
    const bool cta_whole = ubeg >= C0 && uend <= C1;
    const int wa = (int)ws.owner(lbeg), wb = (int)ws.owner(lend - 1);
    // this CTA's state of a unit that other CTAs also hold goes to global memory
    const int cslot = lbeg == C0 ? 0 : 1;
    float* gdep = P.ws + ((size_t)blockIdx.x * 2 + cslot) * C::DEPW;
    if (wb > wa) {
      // several holders in this CTA: partial state to shared memory, CTA ticket
      float* mine = sdep + ((size_t)warp * 2 + (seg_ord == 0 ? 0 : 1)) * C::DEPW;
      if (!failed) write_partial<D, GQ>(st, mine, P.sl2);
      __threadfence_block();
      __syncwarp();
      unsigned last = 0;
      if (lane == 0) last = atomicAdd(&scnt[wa], 1u) == (unsigned)(wb - wa);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) return;
      __threadfence_block();
      const bool wa_late = ws.first(wa) < lbeg;   // its segment is its last one
      auto sdep_of = [&](int k) -> const float* {
        return sdep + ((size_t)(wa + k) * 2 + ((k == 0 && wa_late) ? 1 : 0)) * C::DEPW;
      };
      if (lane == 0) scnt[wa] = 0u;
      if (cta_whole) {
        if (!failed) merge_partials<D, GQ, false, true>(wb - wa + 1, sdep_of, o);
        return;
      }
      if (!failed) merge_partials<D, GQ, false, false>(wb - wa + 1, sdep_of, gdep);
    } else if (!failed) {
      write_partial<D, GQ>(st, gdep, P.sl2);
    }
    __threadfence();
    __syncwarp();
    const long long ca = cs.owner(ubeg), cb = cs.owner(uend - 1);
    unsigned* cnt = P.cnt + (size_t)(P.layer_begin + r.li) * P.units + r.unit;
    unsigned last = 0;
    if (lane == 0) last = atomicAdd(cnt, 1u) == (unsigned)(cb - ca);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    const bool ca_late = cs.first(ca) < ubeg;   // the first CTA's segment is its last one
    if (!failed)
      merge_partials<D, GQ, true, true>((int)(cb - ca + 1), [&](int k) -> const float* {
        return P.ws + ((size_t)(ca + k) * 2 + ((k == 0 && ca_late) ? 1 : 0)) * C::DEPW;
      }, o);
    __syncwarp();
    if (lane == 0) *cnt = 0u;   // ready for the next launch
  };

  for (int i = 0; i < n; ++i) {
    if (i > 0) step(cur);
    const bool seg_start = i == 0 || cur.j == 0;
    if (seg_start) {
      ++seg;
      state_init(st);
    }
    // wait for the chunk (and, at a segment start, the unit's queries)
    const uint32_t par = (uint32_t)((i >> 1) & 1);
    bool done = false;
    for (unsigned it = 0; it < P.wait_limit && !done; ++it) done = mbar_try_wait(&bar[i & 1], par);
    if (!__all_sync(0xffffffffu, done)) {
      if (lane == 0) atomicOr(P.err, 1u);
      fail = i;
      break;
    }
    const DecLayer& L = P.L[cur.li];
    const __nv_bfloat16* qs = qbuf + (seg & 1) * GQ * D;
    if (seg_start) load_qregs<D, GQ>(qr, qs);
    uint8_t* sbuf = ring + (i & 1) * C::SLOT;
    if (cur.j < L.wchunks) {
      __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(sbuf);
      uint32_t* sv = reinterpret_cast<uint32_t*>(sbuf + kSlotsPerWarp * D * 2);
      const int pos0 = cur.j * kSlotsPerWarp;
      const int n_valid = min(kSlotsPerWarp, L.win_len - pos0);
      if (L.new_slot >= 0 && cur.j == (L.win_len - 1) / kSlotsPerWarp) {
        // the step's new token: store it into the ring (later steps read it) and
        // patch the staged copy (the bulk copy may predate the store)
        const size_t ul = (size_t)cur.li * P.units + cur.unit;
        const size_t rb = (size_t)L.win_off + (size_t)cur.unit * L.R * D;
        const __nv_bfloat16* kn = P.k_new + ul * D;
        const __nv_bfloat16* vn = P.v_new + ul * D;
        const int r = L.new_slot - (L.win_start + pos0) % L.R;
        __nv_bfloat16* svh = reinterpret_cast<__nv_bfloat16*>(sv);
        for (int c = lane; c < D; c += 32) {
          const __nv_bfloat16 kv = kn[c], vv = vn[c];
          window_store(win_k + rb, win_v + rb, L.new_slot, c, D, kv, vv);
          sk[win_k_index(r, c, D)] = kv;
          svh[win_v_index(r, c, D)] = vv;
        }
        __syncwarp();
      }
      window_warp<D, GQ>(st, qs, sk, sv, n_valid, P.sl2);
    } else {
      const int g0 = (cur.j - L.wchunks) * L.gpc;
      const int ng = min(L.gpc, L.n_groups - g0);
      if constexpr (BMASK == 1) {
        packed_warp<D, 2, GQ>(st, qr, sbuf, ng, P.sl2);
      } else if constexpr (BMASK == 2) {
        packed_warp<D, 4, GQ>(st, qr, sbuf, ng, P.sl2);
      } else {
        if (L.bits == 2) packed_warp<D, 2, GQ>(st, qr, sbuf, ng, P.sl2);
        else packed_warp<D, 4, GQ>(st, qr, sbuf, ng, P.sl2);
      }
    }
    __syncwarp();   // the slot is read: refill it with the chunk two ahead
    if (i + 2 < n) produce(i + 2);
    if (i == n - 1 || cur.j == cur.cpu - 1) finish(cur, seg, false);
  }
  if (fail >= 0) {
    // let the copies in flight land (chunk fail and the one after it), then hand
    // over the split units left open so every counter still returns to zero
    for (int i = fail; i < n && i <= fail + 1; ++i) {
      bool done = false;
      for (unsigned it = 0; it < kWaitLimit && !done; ++it)
        done = mbar_try_wait(&bar[i & 1], (uint32_t)((i >> 1) & 1));
    }
    __syncwarp();
    finish(cur, seg, true);
    const Cur last = locate(c1 - 1);
    if (last.li != cur.li || last.unit != cur.unit) finish(last, seg + 1, true);
  }
}

template <int D, int GQ, int BMASK>
cudaError_t launch_one(DecParams& P, const kvc_cache* c, const __nv_bfloat16* q, float* out,
                       cudaStream_t stream) {
  using C = DecCfg<D, GQ, BMASK>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(decode_kernel<D, GQ, BMASK>), C::total);
  if (e != cudaSuccess) return e;
  // one CTA per SM, each holding at least one chunk per warp where the launch has
  // that many (fewer, fuller CTAs merge less across SMs)
  const long long T = P.total;
  const int grid = (int)std::max<long long>(1, std::min<long long>(c->n_sm, T / C::NW));
  P.n_vwarps = grid * C::NW;
  if ((size_t)grid * 2 * C::DEPW > c->dec_ws_floats) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::total;
  cfg.stream = stream;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, GQ, BMASK>, P, c->packed, c->win_k, c->win_v,
                            q, out);
}

template <int D, int BMASK>
cudaError_t launch_g(DecParams& P, const kvc_cache* c, const __nv_bfloat16* q, float* out,
                     cudaStream_t stream) {
  switch (c->g) {
    case 1: return launch_one<D, 1, BMASK>(P, c, q, out, stream);
    case 2: return launch_one<D, 2, BMASK>(P, c, q, out, stream);
    case 4: return launch_one<D, 4, BMASK>(P, c, q, out, stream);
    case 8: return launch_one<D, 8, BMASK>(P, c, q, out, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Shared host path: a non-null k_new appends the step's token first. Without a
// group flush in the step the decode launch stores the new token itself; when
// some layer's window reaches R, the append kernel (which also quantizes the
// flushed groups) runs first and the decode launch reads the updated cache.
cudaError_t launch_common(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* q, const __nv_bfloat16* k_new,
                          const __nv_bfloat16* v_new, const int* flush_flags, float* out,
                          cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  const int units = d.batch * d.n_kv_heads;
  const int D = d.head_dim;
  bool appending = k_new != nullptr;
  bool any_flush = false;
  if (appending)
    for (int i = 0; i < layer_count; ++i) any_flush = any_flush || flush_flags[i] != 0;
  if (any_flush) {
    cudaError_t e = launch_append(c, layer_begin, layer_count, k_new, v_new, flush_flags, stream);
    if (e != cudaSuccess) return e;
  }
  for (int base = 0; base < layer_count; base += KVC_MAX_LAUNCH_LAYERS) {
    const int cnt = layer_count - base < KVC_MAX_LAUNCH_LAYERS ? layer_count - base
                                                               : KVC_MAX_LAUNCH_LAYERS;
    DecParams P;
    P.n_layers = cnt;
    P.layer_begin = layer_begin + base;
    P.units = units;
    P.sl2 = 1.4426950408889634f / sqrtf((float)D);
    P.err = c->err;
    P.ws = c->dec_ws;
    P.cnt = c->dec_cnt;
    P.wait_limit = c->wait_limit_set ? c->wait_limit : kWaitLimit;
    const bool fused = appending && !any_flush;
    P.k_new = fused ? k_new + (size_t)base * units * D : nullptr;
    P.v_new = fused ? v_new + (size_t)base * units * D : nullptr;
    long long total = 0;
    int bmask = 0;
    const size_t gq = (size_t)c->g * D;
    float* ob = out + (size_t)base * units * gq;
    for (int i = 0; i < cnt; ++i) {
      const LayerState& ls = c->L[layer_begin + base + i];
      DecLayer& L = P.L[i];
      const int R = ls.R;
      L.cap_groups = ls.cap_groups;
      L.packed_off = (long long)ls.packed_off;
      L.win_off = (long long)ls.win_off;
      L.R = R;
      L.bits = ls.bits;
      L.gpc = dec_groups_per_chunk(D, ls.bits == 16 ? 2 : ls.bits);
      if (appending) {
        const bool flush = flush_flags[base + i] != 0;
        L.new_slot = fused ? (ls.win_start + ls.win_len) % R : -1;
        L.n_groups = ls.n_groups + (flush ? 1 : 0);
        L.win_start = flush ? (ls.win_start + KVC_GROUP) % R : ls.win_start;
        L.win_len = ls.win_len + 1 - (flush ? KVC_GROUP : 0);
      } else {
        L.new_slot = -1;
        L.n_groups = ls.n_groups;
        L.win_start = ls.win_start;
        L.win_len = ls.win_len;
      }
      L.wchunks = (L.win_len + kSlotsPerWarp - 1) / kSlotsPerWarp;
      L.pchunks = (L.n_groups + L.gpc - 1) / L.gpc;
      L.chunk_begin = total;
      total += (long long)units * (L.wchunks + L.pchunks);
      if (L.pchunks > 0) bmask |= ls.bits == 2 ? 1 : (ls.bits == 4 ? 2 : 0);
      if (L.wchunks + L.pchunks == 0) {   // nothing stored: the output is zero
        cudaError_t e = cudaMemsetAsync(ob + (size_t)i * units * gq, 0, units * gq * 4, stream);
        if (e != cudaSuccess) return e;
      }
    }
    P.total = total;
    if (total == 0) continue;
    const __nv_bfloat16* qb = q + (size_t)base * units * gq;
    if (bmask == 0) bmask = 1;   // window only: any instantiation serves
    cudaError_t e;
    if (D == 128 && bmask == 1) e = launch_g<128, 1>(P, c, qb, ob, stream);
    else if (D == 128 && bmask == 2) e = launch_g<128, 2>(P, c, qb, ob, stream);
    else if (D == 128) e = launch_g<128, 3>(P, c, qb, ob, stream);
    else if (bmask == 1) e = launch_g<64, 1>(P, c, qb, ob, stream);
    else if (bmask == 2) e = launch_g<64, 2>(P, c, qb, ob, stream);
    else e = launch_g<64, 3>(P, c, qb, ob, stream);
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

size_t decode_workspace_floats(int n_sm, int g, int D) {
  return (size_t)2 * n_sm * 16 * dep_floats(D, g);
}

}  // namespace kvc
