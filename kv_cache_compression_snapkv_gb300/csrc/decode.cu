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
// Work decomposition (one persistent launch for a range of layers):
//   unit = (layer, sequence b, kv head h); its work is cut into chunks of 16
//   window slots or 1 packed group block. There is one CTA per SM; CTA i takes
//   the units i, 2P-1-i, 2P+i, ... (P CTAs, snake order over units that come
//   largest first) and lays their chunks end to end. When the CTA's units all fit
//   in the query ring, warp w takes the w-th of NW contiguous runs of that list
//   (a unit is split over as few warps as the balance allows, so few partial
//   states are merged); otherwise warp w takes chunks w, w + NW, w + 2 NW, ...,
//   which keeps the warps within a few units of each other (a unit's queries are
//   issued only when the unit QR places before it has been merged). Each warp
//   double-buffers its chunks in
//   shared memory with bulk asynchronous copies (cp.async.bulk on per-slot
//   mbarriers, bounded waits): the copy of its next-but-one chunk is issued as
//   soon as a slot is read. A warp keeps an online softmax for the g query heads
//   of its current unit and deposits it (m, l, o) in shared memory when it leaves
//   the unit; the last warp to deposit merges the deposits with a log-sum-exp
//   combine and writes the fp32 output. No state crosses CTAs and nothing waits
//   on another CTA.
//   The new token of a fused step is stored into the ring by the warp whose
//   window chunk holds its slot (which also patches its staged copy). A step in
//   which some layer's window reaches R runs the append kernel first (it stores
//   the new tokens and quantizes the oldest group of each full window) and then
//   this kernel over the updated cache.
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

constexpr int kGroupsPerWarp = kDecGroupsPerChunk;
constexpr int kSlotsPerWarp = kDecSlotsPerChunk;
static_assert(kSlotsPerWarp == 16, "window warps take 16 slots");
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
  int wchunks;      // window chunks (16 slots) per unit; packed chunks (1 group) follow
  int pchunks;      // packed chunks per unit
  long long packed_off;
};

struct DecParams {
  DecLayer L[KVC_MAX_LAUNCH_LAYERS];
  const __nv_bfloat16* k_new;   // [n_layers][units][D] (fused append only)
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
            value_afrag<BITS, MV, K>(vw, a);
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

// ----------------------------------------------------------- merge helpers
// ----------------------------------------------------------- persistent layout
// One CTA per SM. A CTA takes whole units (snake order over the launch's units,
// which come largest first: layer 0 of a pyramid schedule holds the most groups)
// and lays their chunks end to end; warp w takes chunks w, w + NW, w + 2 NW, ...
// of that list, each staged by a bulk copy into one of its two ring slots (the
// next one is in flight while the current one is computed). A warp deposits its
// softmax state when it leaves a unit; the last warp to deposit merges the unit's
// deposits in shared memory and writes the output. No state crosses CTAs.
template <int D, int BITS, int GQ>
struct DecCfg {
  static constexpr int SLOT = warp_buf_bytes<D, BITS>();   // one chunk
  static constexpr int DEPW = GQ * (D + 2);                // floats of one deposit: m, l, o
  static constexpr int QB = GQ * D * 2;                    // bytes of one unit's queries
  static constexpr int kQRing = 4;                         // query ring entries (<= 8)
  // Two deposit buffers (by unit parity): a warp leaving unit k waits, before it
  // deposits, for the merge of unit k - 2 (it may already compute unit k + 1).
  static constexpr int NDEP = 2;
  static constexpr int bytes(int nw) {
    return nw * 2 * SLOT + NDEP * nw * DEPW * 4 + 16 + kQRing * QB + (2 * nw + kQRing) * 8 + 64;
  }
  static constexpr int pick(int nw) { return (nw <= 4 || bytes(nw) <= 224 * 1024) ? nw : pick(nw - 1); }
  static constexpr int NW = pick(GQ > 4 ? 8 : 12);           // warps per CTA
  static constexpr int kThreadsC = NW * 32;
  // byte offsets inside dynamic shared memory
  static constexpr int oRing = 0;
  static constexpr int oDep = oRing + NW * 2 * SLOT;
  static constexpr int oQ = (oDep + NDEP * NW * DEPW * 4 + 15) / 16 * 16;
  static constexpr int oBars = oQ + kQRing * QB;
  static constexpr int oCtl = oBars + (2 * NW + kQRing) * 8;
  static constexpr int total = oCtl + 64;
  static_assert(SLOT % 16 == 0 && DEPW % 1 == 0 && QB % 16 == 0, "alignment");
  static_assert(oQ % 16 == 0 && oBars % 8 == 0, "alignment");
};

// Control words of a CTA (shared memory): per unit parity, the number of deposits,
// the mask of depositing warps and the number of merges done.
struct DecCtl {
  unsigned count[2];
  unsigned mask[2];
  unsigned gen[2];
  int qunit[8];      // unit whose queries the ring entry was last issued for
};
static_assert(sizeof(DecCtl) <= 64, "control words fit their shared-memory region");

// Unit k of CTA i (snake order): k even -> k*P + i, k odd -> (k+1)*P - 1 - i.
__device__ __forceinline__ int snake_unit(int k, int i, int P) {
  return (k & 1) ? (k + 1) * P - 1 - i : k * P + i;
}

// Write the warp's per-head state (both column parts and the value zero-point sums
// folded in) as one deposit: m[GQ], l[GQ], o[GQ][D].
template <int D, int GQ>
__device__ void warp_deposit(WarpState<D, GQ>& st, float* dep, float sl2) {
  constexpr int NH = n_tiles<GQ>();
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  float* dm = dep;
  float* dl = dep + GQ;
  float* dout = dep + 2 * GQ;
#pragma unroll
  for (int u = 0; u < NH; ++u) {
    const int h = 4 * u + tid;
    float l = st.l[u];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    if (h < GQ) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        dout[h * D + 16 * mt + gid] = st.o[u][mt][0] + st.o[u][mt][1];
        dout[h * D + 16 * mt + gid + 8] = st.o[u][mt][2] + st.o[u][mt][3];
      }
      if (gid == 0) {
        dm[h] = st.m[u] == -INFINITY ? -INFINITY : st.m[u] * sl2;
        dl[h] = l;
      }
    }
  }
}

// One warp merges the deposits of the warps in `mask` (log-sum-exp combine) and
// writes o[GQ][D] (fp32). The weight of each (warp, head) replaces its m slot.
template <int D, int GQ, int NW>
__device__ void merge_deposits(float* dep, unsigned mask, float* __restrict__ o) {
  constexpr int DEPW = GQ * (D + 2);
  constexpr int NWH = (NW * GQ + 31) / 32;
  const int lane = threadIdx.x & 31;
  float f[NWH];
#pragma unroll
  for (int i = 0; i < NWH; ++i) {
    const int idx = lane + 32 * i, w = idx / GQ, h = idx % GQ;
    f[i] = 0.f;
    if (idx < NW * GQ && (mask >> w & 1u) && dep[w * DEPW + GQ + h] > 0.f) {
      float M = -INFINITY;
      for (int v = 0; v < NW; ++v)
        if (mask >> v & 1u) M = fmaxf(M, dep[v * DEPW + h]);
      f[i] = exp2f(dep[w * DEPW + h] - M);
    }
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < NWH; ++i) {
    const int idx = lane + 32 * i, w = idx / GQ, h = idx % GQ;
    if (idx < NW * GQ) dep[w * DEPW + h] = f[i];   // unused warps get weight 0
  }
  __syncwarp();
  // lane h < GQ sums head h's weighted l over the deposits; the sums are shuffled out
  float Lh_lane = 0.f;
  if (lane < GQ)
    for (int w = 0; w < NW; ++w)
      if (mask >> w & 1u) Lh_lane += dep[w * DEPW + lane] * dep[w * DEPW + GQ + lane];
  float L[GQ];
#pragma unroll
  for (int h = 0; h < GQ; ++h) L[h] = __shfl_sync(0xffffffffu, Lh_lane, h);
  // each lane owns E outputs; the deposits are walked in the outer loop so the E
  // accumulations are independent (their shared-memory loads overlap)
  constexpr int E = GQ * D / 32;
  float acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = 0.f;
  for (int w = 0; w < NW; ++w) {
    if (!(mask >> w & 1u)) continue;
    const float* dw = dep + w * DEPW;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int e = lane + 32 * i;
      acc[i] += dw[e / D] * dw[2 * GQ + e];
    }
  }
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int e = lane + 32 * i, h = e / D;
    float Lh = 0.f;
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) Lh = hh == h ? L[hh] : Lh;
    o[e] = Lh > 0.f ? acc[i] / Lh : 0.f;
  }
}

template <int D, int BITS, int GQ>
__global__ void __launch_bounds__(DecCfg<D, BITS, GQ>::kThreadsC, 1)
decode_kernel(const DecParams P, uint8_t* __restrict__ packed, __nv_bfloat16* __restrict__ win_k,
              __nv_bfloat16* __restrict__ win_v, const __nv_bfloat16* __restrict__ q,
              float* __restrict__ out) {
  using C = DecCfg<D, BITS, GQ>;
  constexpr int NW = C::NW, BB = block_bytes(D, BITS), QR = C::kQRing;
  extern __shared__ __align__(128) uint8_t dsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* cbar = reinterpret_cast<uint64_t*>(dsm + C::oBars);   // [NW][2] chunk slots
  uint64_t* qbar = cbar + 2 * NW;                                 // [QR] query ring
  DecCtl& ctl = *reinterpret_cast<DecCtl*>(dsm + C::oCtl);
  // layer table read in place from the launch parameters, each read warp-uniform (a
  // per-thread copy into shared memory made the constant cache serialise)
  const DecLayer* lay = P.L;
  __nv_bfloat16* qring = reinterpret_cast<__nv_bfloat16*>(dsm + C::oQ);
  const int P_ = gridDim.x, cta = blockIdx.x;
  const int total_units = P.n_layers * P.units;

  // the CTA's units: k = 0, 1, ... while snake_unit(k) < total_units
  auto unit_of = [&](int k) { return snake_unit(k, cta, P_); };
  auto chunks_of = [&](int g) { const DecLayer& L = lay[g / P.units]; return L.wchunks + L.pchunks; };
  auto q_copy = [&](int k) {   // queries of the CTA's unit k into ring entry k % QR
    const int g = unit_of(k);
    if (g >= total_units) return;
    uint64_t* b = &qbar[k % QR];
    *reinterpret_cast<volatile int*>(&ctl.qunit[k % QR]) = k;
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                 :: "r"(smem_u32(b)), "r"((uint32_t)C::QB) : "memory");
    bulk_g2s(qring + (k % QR) * GQ * D, q + (size_t)g * GQ * D, (uint32_t)C::QB, b);
  };
  // barriers and control words, then the first units' queries
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * NW + QR; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" :: "r"(smem_u32(&cbar[i])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    for (int p = 0; p < 2; ++p) { ctl.count[p] = 0u; ctl.mask[p] = 0u; ctl.gen[p] = 0u; }
    for (int e = 0; e < 8; ++e) ctl.qunit[e] = -1;
  }
  pdl_wait();      // the previous kernels' writes (queries, cache) are visible
  pdl_release();
  if (threadIdx.x == 0)
    for (int k = 0; k < QR; ++k) q_copy(k);
  __syncthreads();

  // this warp's chunk stream: positions w, w + NW, ... of the CTA's chunk list
  struct Cursor { int k, base, g, n; };   // unit k of the CTA, first list position, unit, chunks
  auto advance = [&](Cursor& c, int pos) {   // move c to the unit holding list position pos
    while (c.g < total_units && pos >= c.base + c.n) {
      c.base += c.n;
      ++c.k;
      c.g = unit_of(c.k);
      c.n = c.g < total_units ? chunks_of(c.g) : 0;
    }
    return c.g < total_units;
  };
  auto issue = [&](int slot, const Cursor& c, int pos) {   // lane 0: stage chunk pos - base of unit c.g
    const DecLayer& L = lay[c.g / P.units];
    const int unit = c.g % P.units, j = pos - c.base;
    uint64_t* b = &cbar[warp * 2 + slot];
    uint8_t* dst = dsm + C::oRing + (warp * 2 + slot) * C::SLOT;
    if (j < L.wchunks) {
      const size_t wunit = (size_t)(P.layer_begin + c.g / P.units) * P.units + unit;
      const int slot0 = (L.win_start + j * kSlotsPerWarp) % P.R;
      const uint32_t wb = (uint32_t)(kSlotsPerWarp * D * 2);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                   :: "r"(smem_u32(b)), "r"(2 * wb) : "memory");
      bulk_g2s(dst, win_k + (wunit * P.R + slot0) * D, wb, b);
      bulk_g2s(dst + wb, win_v + wunit * P.R * D + (size_t)(slot0 >> 1) * D * 2, wb, b);
    } else {
      const int g0 = (j - L.wchunks) * kGroupsPerWarp;
      const int ng = min(kGroupsPerWarp, L.n_groups - g0);
      const uint8_t* src = packed + L.packed_off + ((size_t)unit * L.cap_groups + g0) * BB;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                   :: "r"(smem_u32(b)), "r"((uint32_t)(ng * BB)) : "memory");
      bulk_g2s(dst, src, (uint32_t)(ng * BB), b);
    }
  };

  // chunk list positions of this warp: a contiguous run when the CTA's units all
  // fit in the query ring, else every NW-th position (-1: none left)
  int n_units = 0, total = 0;
  for (int k = 0; unit_of(k) < total_units; ++k) { ++n_units; total += chunks_of(unit_of(k)); }
  const bool blocked = n_units <= QR;
  const int per = (total + NW - 1) / NW;
  const int w0 = min(total, warp * per), w1 = min(total, w0 + per);
  auto position = [&](int n) -> int {
    if (blocked) return w0 + n < w1 ? w0 + n : -1;
    return warp + n * NW;   // past the list: advance() fails
  };

  Cursor cur{0, 0, unit_of(0), 0};
  cur.n = cur.g < total_units ? chunks_of(cur.g) : 0;
  Cursor pre = cur;   // cursor of the prefetch stream (runs two chunks ahead)
  // prime the two slots
  for (int s = 0; s < 2; ++s) {
    const int pos = position(s);
    if (pos >= 0 && advance(pre, pos) && lane == 0) issue(s, pre, pos);
  }

  WarpState<D, GQ> st;
  QRegs<D, GQ> qr;
  int k_cur = -1, base_cur = 0;   // the warp's current unit and its first list position
  bool ok = true;
  const int units_per_layer = P.units;

  auto deposit = [&](int k, int base) {   // hand over unit k's state; the last depositor merges
    const int par = k % C::NDEP;
    const int g = unit_of(k);
    // depositors: the warps whose positions meet the unit's [base, base + chunks)
    const unsigned expect = blocked ? (unsigned)((base + chunks_of(g) - 1) / per - base / per + 1)
                                    : (unsigned)min(NW, chunks_of(g));
    // the deposit buffer of unit k is free once unit k - NDEP is merged
    if (lane == 0) {
      bool ready = false;
      for (unsigned it = 0; it < kWaitLimit && !ready; ++it)
        ready = *reinterpret_cast<volatile unsigned*>(&ctl.gen[par]) == (unsigned)(k / C::NDEP);
      if (!ready) { atomicOr(P.err, 2u); ok = false; }
    }
    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    if (!ok) return;
    float* dep = reinterpret_cast<float*>(dsm + C::oDep) + (par * NW) * C::DEPW;
    warp_deposit<D, GQ>(st, dep + warp * C::DEPW, P.sl2);
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) {
      __threadfence_block();
      atomicOr(&ctl.mask[par], 1u << warp);
      last = atomicAdd(&ctl.count[par], 1u) == expect - 1u;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence_block();
    const unsigned mask = *reinterpret_cast<volatile unsigned*>(&ctl.mask[par]);
    const int li = g / units_per_layer, unit = g % units_per_layer;
    merge_deposits<D, GQ, NW>(dep, mask, out + ((size_t)li * units_per_layer + unit) * GQ * D);
    __syncwarp();
    if (lane == 0) {
      ctl.count[par] = 0u;
      ctl.mask[par] = 0u;
      // the query entry of unit k is free: fetch unit k + QR
      q_copy(k + QR);
      __threadfence_block();
      atomicAdd(&ctl.gen[par], 1u);
    }
  };

  for (int n = 0;; ++n) {
    const int pos = position(n);
    if (pos < 0 || !advance(cur, pos)) break;
    const int slot = n & 1;
    if (cur.k != k_cur) {
      if (k_cur >= 0) deposit(k_cur, base_cur);
      if (!ok) break;
      k_cur = cur.k;
      base_cur = cur.base;
      state_init(st);
      // this unit's queries: the ring entry must hold this unit's copy (issued once
      // the unit QR places before it is merged, so the entry's mbarrier is at most
      // one phase behind), then a bounded wait for that copy
      bool done = false;
      for (unsigned it = 0; it < kWaitLimit && !done; ++it)
        done = *reinterpret_cast<volatile int*>(&ctl.qunit[k_cur % QR]) == k_cur;
      const uint32_t qpar = (uint32_t)((k_cur / QR) & 1);
      if (done) {
        done = false;
        for (unsigned it = 0; it < kWaitLimit && !done; ++it)
          done = mbar_try_wait(&qbar[k_cur % QR], qpar);
      }
      if (!__all_sync(0xffffffffu, done)) { if (lane == 0) atomicOr(P.err, 1u); ok = false; break; }
      load_qregs<D, GQ>(qr, qring + (k_cur % QR) * GQ * D);
    }
    // wait for the chunk
    bool done = false;
    uint64_t* b = &cbar[warp * 2 + slot];
    const uint32_t par = (uint32_t)((n >> 1) & 1);
    for (unsigned it = 0; it < kWaitLimit && !done; ++it) done = mbar_try_wait(b, par);
    if (!done) {
      if (lane == 0) atomicOr(P.err, 1u);
      for (unsigned it = 0; it < kWaitLimit && !done; ++it) done = mbar_try_wait(b, par);
      ok = false;
      break;
    }
    __syncwarp();
    const DecLayer& L = lay[cur.g / P.units];
    const int unit = cur.g % P.units, j = pos - cur.base;
    uint8_t* sbuf = dsm + C::oRing + (warp * 2 + slot) * C::SLOT;
    const __nv_bfloat16* qs = qring + (k_cur % QR) * GQ * D;
    if (j < L.wchunks) {
      __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(sbuf);
      uint32_t* sv = reinterpret_cast<uint32_t*>(sbuf + kSlotsPerWarp * D * 2);
      const int pos0 = j * kSlotsPerWarp;
      const int n_valid = min(kSlotsPerWarp, L.win_len - pos0);
      if (L.new_slot >= 0 && j == (L.win_len - 1) / kSlotsPerWarp) {
        // the step's new token: store it into the ring (later steps read it) and
        // patch the staged copy (the bulk copy may predate the store)
        const int li = cur.g / P.units;
        const size_t wunit = (size_t)(P.layer_begin + li) * P.units + unit;
        const __nv_bfloat16* kn = P.k_new + ((size_t)li * P.units + unit) * D;
        const __nv_bfloat16* vn = P.v_new + ((size_t)li * P.units + unit) * D;
        const int slot0 = (L.win_start + pos0) % P.R;
        const int r = L.new_slot - slot0;
        __nv_bfloat16* svh = reinterpret_cast<__nv_bfloat16*>(sv);
        for (int c = lane; c < D; c += 32) {
          const __nv_bfloat16 kv = kn[c], vv = vn[c];
          window_store(win_k + wunit * P.R * D, win_v + wunit * P.R * D, L.new_slot, c, D, kv, vv);
          sk[win_k_index(r, c, D)] = kv;
          svh[win_v_index(r, c, D)] = vv;
        }
        __syncwarp();
      }
      window_warp<D, GQ>(st, qs, sk, sv, n_valid, P.sl2);
    } else {
      const int g0 = (j - L.wchunks) * kGroupsPerWarp;
      packed_warp<D, BITS, GQ>(st, qr, sbuf, min(kGroupsPerWarp, L.n_groups - g0), P.sl2);
    }
    __syncwarp();   // the slot is read: refill it with the chunk two steps ahead
    const int npos = position(n + 2);
    if (npos >= 0 && advance(pre, npos) && lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      issue(slot, pre, npos);
    }
  }
  if (ok && k_cur >= 0) deposit(k_cur, base_cur);
}

template <int D, int BITS, int GQ>
cudaError_t launch_one(const DecParams& P, const kvc_cache* c, const __nv_bfloat16* q, float* out,
                       cudaStream_t stream) {
  using C = DecCfg<D, BITS, GQ>;
  // kernel attributes and the SM count are looked up once per device
  static int n_sm[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!n_sm[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<D, BITS, GQ>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::total);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    n_sm[dev] = n;
  }
  const int total_units = P.n_layers * P.units;
  const int grid = std::min(n_sm[dev], total_units);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreadsC);
  cfg.dynamicSmemBytes = C::total;
  cfg.stream = stream;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, BITS, GQ>, P, c->packed, c->win_k, c->win_v,
                            q, out);
}

template <int D, int BITS>
cudaError_t launch_g(const DecParams& P, const kvc_cache* c, const __nv_bfloat16* q, float* out,
                     cudaStream_t stream) {
  switch (c->g) {
    case 1: return launch_one<D, BITS, 1>(P, c, q, out, stream);
    case 2: return launch_one<D, BITS, 2>(P, c, q, out, stream);
    case 4: return launch_one<D, BITS, 4>(P, c, q, out, stream);
    case 8: return launch_one<D, BITS, 8>(P, c, q, out, stream);
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
  const int D = d.head_dim, R = d.window_len;
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
    P.R = R;
    P.sl2 = 1.4426950408889634f / sqrtf((float)D);
    P.err = c->err;
    const bool fused = appending && !any_flush;
    P.k_new = fused ? k_new + (size_t)base * units * D : nullptr;
    P.v_new = fused ? v_new + (size_t)base * units * D : nullptr;
    for (int i = 0; i < cnt; ++i) {
      const LayerState& ls = c->L[layer_begin + base + i];
      DecLayer& L = P.L[i];
      L.cap_groups = ls.cap_groups;
      L.packed_off = (long long)ls.packed_off;
      L.flush_start = -1;
      L.n_ctas = 0;
      L.cta_begin = 0;
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
      L.pchunks = (L.n_groups + kGroupsPerWarp - 1) / kGroupsPerWarp;
    }
    const __nv_bfloat16* qb = q + (size_t)base * units * c->g * D;
    float* ob = out + (size_t)base * units * c->g * D;
    cudaError_t e;
    // 16-bit storage has no packed groups (everything is in the window): any packed
    // instantiation serves it
    const int bits = d.bits == 16 ? 2 : d.bits;
    if (D == 128 && bits == 2) e = launch_g<128, 2>(P, c, qb, ob, stream);
    else if (D == 128 && bits == 4) e = launch_g<128, 4>(P, c, qb, ob, stream);
    else if (D == 64 && bits == 2) e = launch_g<64, 2>(P, c, qb, ob, stream);
    else if (D == 64 && bits == 4) e = launch_g<64, 4>(P, c, qb, ob, stream);
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
