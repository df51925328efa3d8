// decode.cu -- split-K decode attention over the packed cache plus the bf16 window.
//
// MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative KV
// Cache, §2 eq. (1) and Algorithm 1 (decoding): one softmax over the
// dequantized packed keys and the 16-bit buffer's keys; the output is
// A_quant . dequant(Q_V) + A_unquant . R_V. The blog "KV Cache Compression:
// Eviction and Quantization", "Measured on a real model": exact recent window,
// rounded rest, one softmax over both.
//
// Work decomposition (one launch for a range of layers):
//   unit = (layer, sequence b, kv head h); a unit's tokens are split over CTAs:
//   "packed" CTAs take 64 group blocks (16 per warp), "window" CTAs 128 ring
//   slots (32 per warp). Each warp keeps an online softmax for the g query heads
//   of the kv head; warps merge in shared memory, CTAs write (m, l, o) partials,
//   and the last CTA of the unit (atomic ticket, no waiting) merges them with a
//   log-sum-exp combine and writes the fp32 output.
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
// extra tensor-core products (q against 8 groups' key zeros; p against the value
// zeros). The window runs the same flow on bf16 operands.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = kDecWarps * 32;

struct DecLayer {
  int n_groups, win_start, win_len, n_pctas, n_ctas, cta_begin, cap_groups, pad;
  long long packed_off;
};

struct DecParams {
  DecLayer L[KVC_MAX_LAUNCH_LAYERS];
  int n_layers;        // layers in this launch
  int layer_begin;     // absolute index of L[0]
  int units;           // batch * n_kv_heads
  int R;               // window ring length
  float sl2;           // log2(e) / sqrt(head_dim)
};

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two codes of pair slot P of a word as an exact fp16 pair (even code low half).
// The masked field sits at bit BITS*j of a byte under the fp16 exponent of 1024,
// so the half is 1024 + code * 2^(BITS*j); one fused multiply-add rescales it.
template <int BITS, int P>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w) {
  constexpr int CPB = 8 / BITS;              // codes per byte
  constexpr int S = P / CPB, J = P % CPB;
  constexpr uint32_t mask = (((1u << BITS) - 1u) * 0x00010001u) << (BITS * J);
  uint32_t v = ((w >> (8 * S)) & mask) | 0x64006400u;
  constexpr float sc = 1.0f / (float)(1 << (BITS * J));
  const __half2 scale = __float2half2_rn(sc);
  const __half2 bias = __float2half2_rn(-1024.0f * sc);
  return h2u(__hfma2(u2h(v), scale, bias));
}

template <int BITS>
__device__ __forceinline__ uint32_t unpack_rt(uint32_t w, int p) {
  // p is a compile-time constant after unrolling; the switch folds away.
  if constexpr (BITS == 2) {
    switch (p) {
      case 0: return unpack_pair<2, 0>(w); case 1: return unpack_pair<2, 1>(w);
      case 2: return unpack_pair<2, 2>(w); case 3: return unpack_pair<2, 3>(w);
      case 4: return unpack_pair<2, 4>(w); case 5: return unpack_pair<2, 5>(w);
      case 6: return unpack_pair<2, 6>(w); default: return unpack_pair<2, 7>(w);
    }
  } else {
    switch (p) {
      case 0: return unpack_pair<4, 0>(w); case 1: return unpack_pair<4, 1>(w);
      case 2: return unpack_pair<4, 2>(w); default: return unpack_pair<4, 3>(w);
    }
  }
}

template <int D, int GQ>
struct WarpState {
  static constexpr int NTV = D / 8;
  float m;            // running max (log2 domain) of this lane's row
  float l;            // lane-partial sum of exp2
  float o[NTV][4];    // value accumulators (rows gid, gid+8)
  float cz[4];        // value zero-point accumulators (cols = value channel groups)
};

template <int D, int GQ>
__device__ __forceinline__ void state_init(WarpState<D, GQ>& st) {
  st.m = -INFINITY;
  st.l = 0.f;
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[i][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) st.cz[e] = 0.f;
}

// Row roles of this lane in the 16-row operands.
template <int GQ>
struct Roles {
  bool hi, lo;
  int head;
  __device__ Roles(int gid) {
    if constexpr (GQ == 8) { hi = true; lo = true; head = gid; }
    else { hi = gid < GQ; lo = gid >= GQ && gid < 2 * GQ; head = gid % GQ; }
  }
};

// Online-softmax update from the raw (unscaled, hi+lo-combined) logits x[NT][2].
// Returns exp2 weights in x.
template <int D, int GQ, int NT>
__device__ __forceinline__ void softmax_update(WarpState<D, GQ>& st, float (&x)[NT][2], float sl2) {
  float tmax = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) { x[nt][e] *= sl2; tmax = fmaxf(tmax, x[nt][e]); }
  tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
  tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
  const float mnew = fmaxf(st.m, tmax);
  if (__any_sync(0xffffffffu, mnew > st.m)) {
    const float corr = (mnew == -INFINITY) ? 1.f : exp2f(st.m - mnew);
    st.l *= corr;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.o[i][e] *= corr;
#pragma unroll
    for (int e = 0; e < 4; ++e) st.cz[e] *= corr;
    st.m = mnew;
  }
  float s = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float p = (x[nt][e] == -INFINITY) ? 0.f : exp2f(x[nt][e] - st.m);
      x[nt][e] = p;
      s += p;
    }
  st.l += s;
}

// Combine the hi and lo rows of a C fragment into the full per-head value.
template <int GQ>
__device__ __forceinline__ float combine_rows(float c_row, float c_row8) {
  if constexpr (GQ == 8) return c_row + c_row8;
  else return c_row + __shfl_xor_sync(0xffffffffu, c_row, 4 * GQ);
}

// ------------------------------------------------------------ packed groups
template <int D, int BITS, int GQ>
__device__ void packed_warp(WarpState<D, GQ>& st, const uint8_t* __restrict__ base, int g_begin,
                            int g_end, const __nv_bfloat16* __restrict__ qrow_base, float sl2) {
  constexpr int KS = D / 16, NTV = D / 8, WPL = D * BITS / 32, PPW = 16 / BITS;
  constexpr int NGC = D / 32, BB = 8 * D * (BITS + 1);
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const Roles<GQ> R(gid);
  const bool active = R.hi || R.lo;

  // query pairs for this lane's channels, fp16 (exact for bf16 queries in range)
  __half2 qh[KS][2];
  {
    const __nv_bfloat16* qr = qrow_base + (size_t)R.head * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        int c = 16 * ks + 2 * tid + 8 * e2;
        float a = active ? __bfloat162float(qr[c]) : 0.f;
        float b = active ? __bfloat162float(qr[c + 1]) : 0.f;
        qh[ks][e2] = __floats2half2_rn(a, b);
      }
  }
  float zb[2] = {0.f, 0.f};   // key zero-point sums of the current 8-group batch

  for (int gg = g_begin; gg < g_end; ++gg) {
    const int j = gg - g_begin;
    if ((j & 7) == 0) {
      // zero-point sums for groups gg .. gg+7: C[row][col] = q_row . Z_{gg+col}
      int gz = gg + gid < g_end ? gg + gid : gg;
      const uint8_t* bz = base + (size_t)gz * BB + off_kzero(D, BITS);
      const uint4* zp = reinterpret_cast<const uint4*>(bz + tid * (D / 4) * 2);
      float cz4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint4 z = __ldg(zp + ch);
        // each uint4 holds two k-steps: (e01, e23) of ks = 2ch, then of ks = 2ch + 1
        const int ks0 = 2 * ch;
        uint32_t a0 = R.hi ? h2u(qh[ks0][0]) : 0u, a2 = R.hi ? h2u(qh[ks0][1]) : 0u;
        mma_f16(cz4, a0, 0u, a2, 0u, z.x, z.y);
        uint32_t c0 = R.hi ? h2u(qh[ks0 + 1][0]) : 0u, c2 = R.hi ? h2u(qh[ks0 + 1][1]) : 0u;
        mma_f16(cz4, c0, 0u, c2, 0u, z.z, z.w);
      }
      zb[0] = cz4[0];
      zb[1] = cz4[1];
    }
    const int src = gid * 4 + ((j & 7) >> 1);
    const float z0 = __shfl_sync(0xffffffffu, zb[0], src);
    const float z1 = __shfl_sync(0xffffffffu, zb[1], src);
    const float bias = (j & 1) ? z1 : z0;

    const uint8_t* blk = base + (size_t)gg * BB;
    // ---- keys: codes, scales, operand A
    uint32_t kw[WPL];
    {
      const uint4* p = reinterpret_cast<const uint4*>(blk);
#pragma unroll
      for (int i = 0; i < WPL / 4; ++i) {
        uint4 u = __ldg(p + i * 32 + lane);
        kw[4 * i] = u.x; kw[4 * i + 1] = u.y; kw[4 * i + 2] = u.z; kw[4 * i + 3] = u.w;
      }
    }
    uint32_t ak[KS][4];
    {
      const uint4* sp = reinterpret_cast<const uint4*>(blk + off_kscale(D, BITS) + tid * (D / 4) * 2);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint4 s = __ldg(sp + ch);
        const uint32_t sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ks = 2 * ch + h;
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            __half2 S2 = u2h(sv[2 * h + e2]);
            __half2 hi = __hmul2(qh[ks][e2], S2);
            __half2 lo = __hfma2(qh[ks][e2], S2, __hneg2(hi));
            if constexpr (GQ == 8) {
              ak[ks][e2 * 2] = h2u(hi);
              ak[ks][e2 * 2 + 1] = h2u(lo);
            } else {
              ak[ks][e2 * 2] = R.hi ? h2u(hi) : (R.lo ? h2u(lo) : 0u);
              ak[ks][e2 * 2 + 1] = 0u;
            }
          }
        }
      }
    }
    float c[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      c[nt][0] = bias; c[nt][1] = bias; c[nt][2] = 0.f; c[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int pi = (nt * KS + ks) * 2;
        uint32_t b0 = unpack_rt<BITS>(kw[pi / PPW], pi % PPW);
        uint32_t b1 = unpack_rt<BITS>(kw[(pi + 1) / PPW], (pi + 1) % PPW);
        mma_f16(c[nt], ak[ks][0], ak[ks][1], ak[ks][2], ak[ks][3], b0, b1);
      }
    }
    float x[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      x[nt][0] = combine_rows<GQ>(c[nt][0], c[nt][2]);
      x[nt][1] = combine_rows<GQ>(c[nt][1], c[nt][3]);
    }
    softmax_update<D, GQ, 4>(st, x, sl2);

    // ---- values
    uint32_t vw[WPL];
    {
      const uint4* p = reinterpret_cast<const uint4*>(blk + off_vcodes(D, BITS));
#pragma unroll
      for (int i = 0; i < WPL / 4; ++i) {
        uint4 u = __ldg(p + i * 32 + lane);
        vw[4 * i] = u.x; vw[4 * i + 1] = u.y; vw[4 * i + 2] = u.z; vw[4 * i + 3] = u.w;
      }
    }
    const uint32_t* vs = reinterpret_cast<const uint32_t*>(blk + off_vscale(D, BITS));
    const uint32_t* vz = reinterpret_cast<const uint32_t*>(blk + off_vzero(D, BITS));
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      // p of tokens 16ks + 2tid + {0,1} and + 8 + {0,1}
      const float p0 = x[2 * ks][0], p1 = x[2 * ks][1], p2 = x[2 * ks + 1][0], p3 = x[2 * ks + 1][1];
      __half2 ph01 = __floats2half2_rn(p0, p1), ph23 = __floats2half2_rn(p2, p3);
      __half2 pl01 = __floats2half2_rn(p0 - __low2float(ph01), p1 - __high2float(ph01));
      __half2 pl23 = __floats2half2_rn(p2 - __low2float(ph23), p3 - __high2float(ph23));
      const int P0 = 8 * ks + tid, P1 = P0 + 4;     // token-pair indices
      // value zero-points: C[row][gc] += p_row,t * Z_t,gc  (B col = gc = gid)
      {
        uint32_t bz0 = gid < NGC ? __ldg(vz + P0 * NGC + gid) : 0u;
        uint32_t bz1 = gid < NGC ? __ldg(vz + P1 * NGC + gid) : 0u;
        uint32_t a0, a1, a2, a3;
        if constexpr (GQ == 8) { a0 = h2u(ph01); a1 = h2u(pl01); a2 = h2u(ph23); a3 = h2u(pl23); }
        else {
          a0 = R.hi ? h2u(ph01) : (R.lo ? h2u(pl01) : 0u); a1 = 0u;
          a2 = R.hi ? h2u(ph23) : (R.lo ? h2u(pl23) : 0u); a3 = 0u;
        }
        mma_f16(st.cz, a0, a1, a2, a3, bz0, bz1);
      }
#pragma unroll
      for (int gc = 0; gc < NGC; ++gc) {
        __half2 S01 = u2h(__ldg(vs + P0 * NGC + gc));
        __half2 S23 = u2h(__ldg(vs + P1 * NGC + gc));
        __half2 h01 = __hmul2(ph01, S01), h23 = __hmul2(ph23, S23);
        __half2 l01 = __hfma2(pl01, S01, __hfma2(ph01, S01, __hneg2(h01)));
        __half2 l23 = __hfma2(pl23, S23, __hfma2(ph23, S23, __hneg2(h23)));
        uint32_t a0, a1, a2, a3;
        if constexpr (GQ == 8) { a0 = h2u(h01); a1 = h2u(l01); a2 = h2u(h23); a3 = h2u(l23); }
        else {
          a0 = R.hi ? h2u(h01) : (R.lo ? h2u(l01) : 0u); a1 = 0u;
          a2 = R.hi ? h2u(h23) : (R.lo ? h2u(l23) : 0u); a3 = 0u;
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int nt = gc * 4 + q4;
          const int pi = (ks * NTV + nt) * 2;
          uint32_t b0 = unpack_rt<BITS>(vw[pi / PPW], pi % PPW);
          uint32_t b1 = unpack_rt<BITS>(vw[(pi + 1) / PPW], (pi + 1) % PPW);
          mma_f16(st.o[nt], a0, a1, a2, a3, b0, b1);
        }
      }
    }
  }
}

// ------------------------------------------------------------- window slots
template <int D, int GQ>
__device__ void window_warp(WarpState<D, GQ>& st, const __nv_bfloat16* __restrict__ wk,
                            const __nv_bfloat16* __restrict__ wv, int slot0, int n_valid,
                            const __nv_bfloat16* __restrict__ qrow_base, float sl2) {
  constexpr int KS = D / 16, NTV = D / 8;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const Roles<GQ> R(gid);
  // A = q (bf16, exact) in the hi rows only
  uint32_t aq[KS][2];
  {
    const __nv_bfloat16* qr = qrow_base + (size_t)R.head * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        int c = 16 * ks + 2 * tid + 8 * e2;
        uint32_t u = *reinterpret_cast<const uint32_t*>(qr + c);
        aq[ks][e2] = R.hi ? u : 0u;
      }
  }
  float c[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
    const int slot = slot0 + nt * 8 + gid;
    const uint4* kr = reinterpret_cast<const uint4*>(wk + (size_t)slot * D + tid * (D / 4));
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint4 u = __ldg(kr + ch);
      mma_bf16(c[nt], aq[2 * ch][0], 0u, aq[2 * ch][1], 0u, u.x, u.y);
      mma_bf16(c[nt], aq[2 * ch + 1][0], 0u, aq[2 * ch + 1][1], 0u, u.z, u.w);
    }
  }
  float x[4][2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = combine_rows<GQ>(c[nt][e], c[nt][e + 2]);
      int col = nt * 8 + 2 * tid + e;
      x[nt][e] = col < n_valid ? v : -INFINITY;
    }
  softmax_update<D, GQ, 4>(st, x, sl2);
  const uint32_t* wv32 = reinterpret_cast<const uint32_t*>(wv);
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const float p0 = x[2 * ks][0], p1 = x[2 * ks][1], p2 = x[2 * ks + 1][0], p3 = x[2 * ks + 1][1];
    __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1), h23 = __floats2bfloat162_rn(p2, p3);
    __nv_bfloat162 l01 = __floats2bfloat162_rn(p0 - __low2float(h01), p1 - __high2float(h01));
    __nv_bfloat162 l23 = __floats2bfloat162_rn(p2 - __low2float(h23), p3 - __high2float(h23));
    uint32_t H01 = *reinterpret_cast<uint32_t*>(&h01), H23 = *reinterpret_cast<uint32_t*>(&h23);
    uint32_t L01 = *reinterpret_cast<uint32_t*>(&l01), L23 = *reinterpret_cast<uint32_t*>(&l23);
    uint32_t a0, a1, a2, a3;
    if constexpr (GQ == 8) { a0 = H01; a1 = L01; a2 = H23; a3 = L23; }
    else {
      a0 = R.hi ? H01 : (R.lo ? L01 : 0u); a1 = 0u;
      a2 = R.hi ? H23 : (R.lo ? L23 : 0u); a3 = 0u;
    }
    const int P0 = (slot0 >> 1) + 8 * ks + tid, P1 = P0 + 4;
    const uint4* v0 = reinterpret_cast<const uint4*>(wv32 + (size_t)P0 * D + gid * (D / 8));
    const uint4* v1 = reinterpret_cast<const uint4*>(wv32 + (size_t)P1 * D + gid * (D / 8));
#pragma unroll
    for (int ch = 0; ch < NTV / 4; ++ch) {
      uint4 b0 = __ldg(v0 + ch), b1 = __ldg(v1 + ch);
      mma_bf16(st.o[4 * ch + 0], a0, a1, a2, a3, b0.x, b1.x);
      mma_bf16(st.o[4 * ch + 1], a0, a1, a2, a3, b0.y, b1.y);
      mma_bf16(st.o[4 * ch + 2], a0, a1, a2, a3, b0.z, b1.z);
      mma_bf16(st.o[4 * ch + 3], a0, a1, a2, a3, b0.w, b1.w);
    }
  }
}

// ----------------------------------------------------------- merge helpers
template <int D, int GQ>
struct DecSmem {
  float m[kDecWarps][GQ];
  float l[kDecWarps][GQ];
  float o[kDecWarps][GQ][D];
  float bias[kDecWarps][GQ][D / 32];
  int last;
};

// Write the warp's per-head state (hi + lo rows combined) into shared memory.
template <int D, int GQ>
__device__ void warp_to_smem(WarpState<D, GQ>& st, DecSmem<D, GQ>& sm, int warp) {
  constexpr int NTV = D / 8;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tid = lane & 3;
  const Roles<GQ> R(gid);
  float l = st.l;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
#pragma unroll
  for (int nt = 0; nt < NTV; ++nt) {
    float o0 = combine_rows<GQ>(st.o[nt][0], st.o[nt][2]);
    float o1 = combine_rows<GQ>(st.o[nt][1], st.o[nt][3]);
    if (R.hi) {
      sm.o[warp][R.head][nt * 8 + 2 * tid] = o0;
      sm.o[warp][R.head][nt * 8 + 2 * tid + 1] = o1;
    }
  }
  float z0 = combine_rows<GQ>(st.cz[0], st.cz[2]);
  float z1 = combine_rows<GQ>(st.cz[1], st.cz[3]);
  if (R.hi) {
    if (2 * tid < D / 32) sm.bias[warp][R.head][2 * tid] = z0;
    if (2 * tid + 1 < D / 32) sm.bias[warp][R.head][2 * tid + 1] = z1;
    if (tid == 0) { sm.m[warp][R.head] = st.m; sm.l[warp][R.head] = l; }
  }
}

template <int D, int BITS, int GQ>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const DecParams P, const uint8_t* __restrict__ packed,
              const __nv_bfloat16* __restrict__ win_k, const __nv_bfloat16* __restrict__ win_v,
              const __nv_bfloat16* __restrict__ q, float* __restrict__ out,
              float* __restrict__ part, unsigned* __restrict__ tickets) {
  __shared__ DecSmem<D, GQ> sm;
  const int warp = threadIdx.x >> 5;
  // locate (layer, unit, cta index)
  int li = 0;
  while (li + 1 < P.n_layers && (int)blockIdx.x >= P.L[li + 1].cta_begin) ++li;
  const DecLayer& Ld = P.L[li];
  const int local = blockIdx.x - Ld.cta_begin;
  const int unit = local / Ld.n_ctas, cidx = local % Ld.n_ctas;
  const int layer = P.layer_begin + li;
  // the GQ query heads of kv head h of sequence b are rows unit*GQ .. unit*GQ+GQ-1
  const __nv_bfloat16* qrow = q + ((size_t)li * P.units + unit) * GQ * D;

  WarpState<D, GQ> st;
  state_init(st);
  if (cidx < Ld.n_pctas) {
    const int g0 = cidx * kGroupsPerCta;
    const int g1 = min(g0 + kGroupsPerCta, Ld.n_groups);
    const int per = (g1 - g0 + kDecWarps - 1) / kDecWarps;
    const int wb = g0 + warp * per, we = min(wb + per, g1);
    const uint8_t* base = packed + Ld.packed_off +
                          (size_t)unit * Ld.cap_groups * (8 * D * (BITS + 1));
    if (wb < we) packed_warp<D, BITS, GQ>(st, base, wb, we, qrow, P.sl2);
  } else {
    const int wc = cidx - Ld.n_pctas;
    const int pos0 = wc * kWinSlotsPerCta + warp * 32;
    const int n_valid = min(32, Ld.win_len - pos0);
    if (n_valid > 0) {
      const size_t wunit = (size_t)layer * P.units + unit;
      const int slot0 = (Ld.win_start + pos0) % P.R;
      window_warp<D, GQ>(st, win_k + wunit * P.R * D, win_v + wunit * P.R * D, slot0, n_valid,
                         qrow, P.sl2);
    }
  }
  warp_to_smem<D, GQ>(st, sm, warp);
  __syncthreads();

  // merge the CTA's warps into one partial: part[cta][head][0..D+1] = (m, l, o[D])
  float* mypart = part + (size_t)blockIdx.x * GQ * (D + 2);
  for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
    const int r = i / D, cch = i % D;
    float M = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm.m[w][r]);
    float L = 0.f, O = 0.f;
    for (int w = 0; w < kDecWarps; ++w) {
      float lw = sm.l[w][r];
      if (lw > 0.f) {
        float f = exp2f(sm.m[w][r] - M);
        L += lw * f;
        O += (sm.o[w][r][cch] + sm.bias[w][r][cch / 32]) * f;
      }
    }
    mypart[r * (D + 2) + 2 + cch] = O;
    if (cch == 0) { mypart[r * (D + 2)] = M; mypart[r * (D + 2) + 1] = L; }
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
  const float* up = part + (size_t)(Ld.cta_begin + unit * Ld.n_ctas) * GQ * (D + 2);
  float* o = out + ((size_t)li * P.units + unit) * GQ * D;
  for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
    const int r = i / D, cch = i % D;
    float M = -INFINITY;
    for (int s = 0; s < Ld.n_ctas; ++s) M = fmaxf(M, __ldcg(up + ((size_t)s * GQ + r) * (D + 2)));
    float L = 0.f, O = 0.f;
    for (int s = 0; s < Ld.n_ctas; ++s) {
      const float* ps = up + ((size_t)s * GQ + r) * (D + 2);
      float ls = __ldcg(ps + 1);
      if (ls > 0.f) {
        float f = exp2f(__ldcg(ps) - M);
        L += ls * f;
        O += __ldcg(ps + 2 + cch) * f;
      }
    }
    o[(size_t)r * D + cch] = O / L;
  }
}

}  // namespace

cudaError_t launch_decode(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* q, float* out, cudaStream_t stream) {
  const kvc_dims& d = c->dims;
  const int units = d.batch * d.n_kv_heads;
  const int D = d.head_dim;
  for (int base = 0; base < layer_count; base += KVC_MAX_LAUNCH_LAYERS) {
    const int cnt = layer_count - base < KVC_MAX_LAUNCH_LAYERS ? layer_count - base
                                                               : KVC_MAX_LAUNCH_LAYERS;
    DecParams P;
    P.n_layers = cnt;
    P.layer_begin = layer_begin + base;
    P.units = units;
    P.R = d.window_len;
    P.sl2 = 1.4426950408889634f / sqrtf((float)D);
    int ctas = 0;
    for (int i = 0; i < cnt; ++i) {
      const LayerState& ls = c->L[layer_begin + base + i];
      DecLayer& L = P.L[i];
      L.n_groups = ls.n_groups;
      L.win_start = ls.win_start;
      L.win_len = ls.win_len;
      L.n_pctas = packed_ctas(ls.n_groups);
      L.n_ctas = L.n_pctas + window_ctas(ls.win_len);
      L.cta_begin = ctas;
      L.cap_groups = ls.cap_groups;
      L.pad = 0;
      L.packed_off = (long long)ls.packed_off;
      ctas += units * L.n_ctas;
    }
    if ((size_t)ctas * c->g * (D + 2) > c->dec_part_elems) return cudaErrorInvalidValue;
    const __nv_bfloat16* qb = q + (size_t)base * units * c->g * D;
    float* ob = out + (size_t)base * units * c->g * D;
#define KVC_DEC_LAUNCH(DD, BB, GG)                                                         \
  decode_kernel<DD, BB, GG><<<ctas, kThreads, 0, stream>>>(P, c->packed, c->win_k, c->win_v, \
                                                         qb, ob, c->dec_part, c->tickets)
#define KVC_DEC_G(DD, BB)                                      \
  switch (c->g) {                                              \
    case 1: KVC_DEC_LAUNCH(DD, BB, 1); break;                  \
    case 2: KVC_DEC_LAUNCH(DD, BB, 2); break;                  \
    case 4: KVC_DEC_LAUNCH(DD, BB, 4); break;                  \
    case 8: KVC_DEC_LAUNCH(DD, BB, 8); break;                  \
    default: return cudaErrorInvalidValue;                     \
  }
    if (D == 128 && d.bits == 2) { KVC_DEC_G(128, 2) }
    else if (D == 128 && d.bits == 4) { KVC_DEC_G(128, 4) }
    else if (D == 64 && d.bits == 2) { KVC_DEC_G(64, 2) }
    else if (D == 64 && d.bits == 4) { KVC_DEC_G(64, 4) }
    else return cudaErrorInvalidValue;
#undef KVC_DEC_G
#undef KVC_DEC_LAUNCH
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvc
