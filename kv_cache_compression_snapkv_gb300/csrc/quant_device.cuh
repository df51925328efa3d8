// quant_device.cuh -- the group quantizer and window-ring accessors, shared by
// the prefill/append kernels (quant.cu) and the fused decode step (decode.cu).
//
// KIVI-style asymmetric groups (blog "Quantization: keep each token in fewer
// bits"; MiniKV §4.4): keys per channel over 32 consecutive stored tokens,
// values per token over 32 consecutive channels; zero-point = group min,
// scale = (max - min) / (2^b - 1), both stored as fp16 (round to nearest even).
// Codes use the stored fp16 values: code = rint((x - Z) / S) clamped to
// [0, 2^b - 1], with explicit IEEE round-to-nearest fp32 subtract and divide (no
// contraction) and round-half-to-even conversion; S == 0 gives 0. The quotient is
// formed without a divide instruction where that provably gives the IEEE result
// (code_fragment), else by the divide itself.
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

// S = fp16(fl((hi - lo) / (2^b - 1))), Z = fp16(lo) and their fp32 values, with
// the reciprocal 1/S rounded to fp32 (0 when S == 0). The fp32 quotient by the
// constant 3 or 15 is formed by one FMA correction of the product with the
// rounded reciprocal (the step code_fragment describes; a divisor of at most 4
// bits keeps every quotient at least 2^-5 ulp away from a rounding midpoint, so
// the result is the IEEE quotient); a range that is not finite is divided as is.
__device__ __forceinline__ void group_params(float lo, float hi, int bits, __half& S, __half& Z,
                                             float& Sf, float& Zf, float& rS) {
  const float rng = __fsub_rn(hi, lo);
  const float top = bits == 2 ? 3.f : 15.f;
  const float rtop = __uint_as_float(bits == 2 ? 0x3eaaaaabu : 0x3d888889u);   // RN(1 / top)
  const float q0 = __fmul_rn(rng, rtop);
  float s32 = __fmaf_rn(__fmaf_rn(-q0, top, rng), rtop, q0);
  if (!(rng <= 3.40282347e38f)) s32 = rng;   // inf / top = inf; NaN stays NaN
  S = __float2half_rn(s32);
  Z = __float2half_rn(lo);
  Sf = __half2float(S);
  Zf = __half2float(Z);
  rS = Sf == 0.f ? 0.f : __frcp_rn(Sf);
}

// Exact code of one element (the definition itself, for the rare elements the
// paired path below cannot decide): IEEE fp32 subtract and divide, round half to
// even, clamp; S == 0 gives 0.
__device__ __forceinline__ uint32_t quant_code_exact(float x, float Zf, float Sf, int bits) {
  if (Sf == 0.f) return 0;
  const int c = __float2int_rn(__fdiv_rn(__fsub_rn(x, Zf), Sf));
  const int top = (1 << bits) - 1;
  return (uint32_t)(c < 0 ? 0 : (c > top ? top : c));
}

// ------------------------------------------------------------ paired fp32
// Two fp32 lanes in one 64-bit register (Blackwell's paired fp32 arithmetic).
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Staging of one 32-token group: key and value rows as stored (bf16, natural
// channel order), rows padded by 8 elements so that the 8 rows of each 8x8
// matrix load fall in distinct shared-memory banks.
template <int D>
struct GroupStage {
  __nv_bfloat16 k[KVC_GROUP][D + 8];
  __nv_bfloat16 v[KVC_GROUP][D + 8];
};

// Quantization parameters of one group, in the order the code words consume
// them: the 4 groups a thread's 16x16 tile fragment touches are adjacent
// (kq_pos / vq_pos), so one 16-byte load fetches them.
template <int D>
struct QuantScratch {
  float z[2][D];          // Z as fp32 ([0] key channels, [1] value groups)
  float rcp[2][D];        // 1/S rounded to fp32 (0 when S == 0)
  float nsc[2][D];        // -S as fp32
  __half s[2][D];         // S as stored
  uint8_t exact[2][D];    // 1: the group's codes are taken by the divide itself
  uint2 kred[2][D / 2];   // per channel pair: (min, max) as bf16x2 over 16 tokens
};

// Key channel c: fragment slot (c >> 4, (c & 7) >> 1), element (c & 1) + 2 ((c >> 3) & 1).
__host__ __device__ constexpr int kq_pos(int c) {
  return ((c >> 4) * 4 + ((c & 7) >> 1)) * 4 + (c & 1) + 2 * ((c >> 3) & 1);
}
// Value group (token t, channels 32 gc ..): slot (gc, t >> 4, (t & 7) >> 1).
__host__ __device__ constexpr int vq_pos(int t, int gc) {
  return (((gc * 2 + (t >> 4)) * 4 + ((t & 7) >> 1)) * 4 + (t & 1) + 2 * ((t >> 3) & 1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

// Parameters of one group from its minimum and maximum, at position `pos` of
// section `kind` of the scratch; the global copies of S and Z go to sdst / zdst.
// The divide-free path (code_fragment) is taken where S and Z are finite and
// every element's |x - Z| / S stays at most 2^14 (checked at the group's two
// ends: the rounded difference is monotone in x); else the divide itself.
template <int D, int BITS>
__device__ __forceinline__ bool set_params(float lo, float hi, QuantScratch<D>& q, int kind,
                                           int pos, __half* sdst, __half* zdst) {
  __half S, Z;
  float Sf, Zf, rS;
  group_params(lo, hi, BITS, S, Z, Sf, Zf, rS);
  const float qlo = __fsub_rn(lo, Zf) * rS, qhi = __fsub_rn(hi, Zf) * rS;
  const bool paired = fabsf(Sf) <= 65504.f && fabsf(Zf) <= 65504.f && fabsf(qlo) <= 16384.f &&
                      fabsf(qhi) <= 16384.f;   // false on NaN
  // every element's quotient inside (-1/2, 2^b - 1/2): its code needs no clamp
  const bool inside = qlo > -0.49f && qhi < (float)((1 << BITS) - 1) + 0.49f;
  q.z[kind][pos] = Zf;
  q.rcp[kind][pos] = rS;
  q.nsc[kind][pos] = -Sf;
  q.s[kind][pos] = S;
  q.exact[kind][pos] = paired ? 0 : 1;
  *sdst = S;
  *zdst = Z;
  return !paired || !inside;
}

// Codes of one 16x16 tile fragment pair-packed into `word` (BITS-bit fields at
// shift(k) and 16 + shift(k) for register k), two elements per fp32-pair
// instruction:
//   d  = x - Z                      (IEEE, as the definition)
//   q0 = d * (1/S)                  (rounded; within 1.5 ulp of d / S)
//   q1 = fma(fma(q0, -S, d), 1/S, q0)
// q1 is the IEEE quotient fl(d / S) (the FMA correction step of P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor",
// IBM J. Res. Dev. 34(1), 1990): before its final rounding q1 lies within 2^-22
// ulp of d / S, and d / S is never an fp32 rounding midpoint nor closer than
// 2^-12 ulp to one (a midpoint has 25 significant bits, S at most 11, so S times
// a midpoint is no fp32 value, and d - S m, when non-zero, is a multiple of
// ulp(S) ulp(m)). Adding M = 1.5 * 2^23 then rounds q1 to the nearest integer,
// ties to even, into the low bits of t, read as a 16-bit integer (|q1| <= 2^14)
// and clamped to [0, 2^b - 1] two at a time (CLAMP; without it every quotient of
// the fragment's groups lies in (-1/2, 2^b - 1/2)).
template <int BITS, bool CLAMP>
__device__ __forceinline__ void code_fragment(const uint32_t (&r)[4], float4 zq, float4 rq,
                                              float4 nq, int s_shift, uint32_t& word) {
  constexpr float kMagic = 12582912.f;           // 1.5 * 2^23
  constexpr uint32_t top2 = ((1u << BITS) - 1) * 0x10001u;
  const unsigned long long M2 = f2pack(kMagic, kMagic);
  const unsigned long long z01 = f2pack(zq.x, zq.y), z23 = f2pack(zq.z, zq.w);
  const unsigned long long r01 = f2pack(rq.x, rq.y), r23 = f2pack(rq.z, rq.w);
  const unsigned long long n01 = f2pack(nq.x, nq.y), n23 = f2pack(nq.z, nq.w);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rh = k & 1;
    const float xe = __uint_as_float(r[k] << 16), xo = __uint_as_float(r[k] & 0xffff0000u);
    const unsigned long long R2 = rh ? r23 : r01;
    const unsigned long long d = f2sub(f2pack(xe, xo), rh ? z23 : z01);
    const unsigned long long q0 = f2mul(d, R2);
    const unsigned long long q1 = f2fma(f2fma(q0, rh ? n23 : n01, d), R2, q0);
    float t0, t1;
    f2unpack(f2add(q1, M2), t0, t1);
    uint32_t v = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x5410);
    if (CLAMP) asm("min.relu.s16x2 %0, %1, %2;" : "=r"(v) : "r"(v), "r"(top2));
    const int sh = BITS == 4 ? 4 * k : 8 * (k >> 1) + 2 * rh + s_shift;
    word += v << sh;
  }
}

// The same fields by the definition (groups outside the divide-free path).
template <int BITS>
__device__ __noinline__ uint32_t code_fragment_exact(uint32_t r0, uint32_t r1, uint32_t r2,
                                                     uint32_t r3, const float* z,
                                                     const __half* s, int s_shift) {
  const uint32_t r[4] = {r0, r1, r2, r3};
  uint32_t word = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rh = k & 1;
    const int sh = BITS == 4 ? 4 * k : 8 * (k >> 1) + 2 * rh + s_shift;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float x = __uint_as_float(e ? (r[k] & 0xffff0000u) : (r[k] << 16));
      const uint32_t c = quant_code_exact(x, z[2 * rh + e], __half2float(s[2 * rh + e]), BITS);
      word |= c << (sh + 16 * e);
    }
  }
  return word;
}

// One warp's code words of one section (KIND 0: keys, 1: values): the warp covers
// D / 32 of the section's 16x16 tiles (4 for D = 128), one 8x8-matrix load per
// tile (transposed for values, whose fragment pairs run along tokens), and stores
// its lanes' words with one vector store per lane.
template <int D, int BITS, int KIND, bool PLAIN>
__device__ __forceinline__ void code_words(const GroupStage<D>& g, const QuantScratch<D>& q,
                                           uint32_t* __restrict__ out, int sub, int lane) {
  constexpr int KS = D / 16;
  constexpr int TPW = D / 32;                  // tiles per warp
  constexpr int TPWD = BITS == 4 ? 1 : 2;      // tiles per code word
  constexpr int WW = TPW / TPWD;               // words per lane
  const int wi0 = WW * sub;
  const int tid = lane & 3, m = lane >> 3, i8 = lane & 7;
  const __nv_bfloat16* base = KIND ? &g.v[0][0] : &g.k[0][0];
  uint32_t words[WW];
#pragma unroll
  for (int wj = 0; wj < WW; ++wj) {
    const int wi = wi0 + wj;
    uint32_t word = 0;
#pragma unroll
    for (int s = 0; s < TPWD; ++s) {
      int mt, ks;
      if (KIND == 0) {
        if (BITS == 4) { mt = wi / KS; ks = wi % KS; }
        else { mt = wi / (KS / 2); ks = 2 * (wi % (KS / 2)) + s; }
      } else {
        if (BITS == 4) { mt = wi >> 1; ks = wi & 1; }
        else { mt = wi; ks = s; }
      }
      int tok, ch, quad;
      if (KIND == 0) {   // rows = tokens 16 mt (+8 for matrices 2, 3), channels 16 ks (+8 for 1, 3)
        tok = 16 * mt + 8 * (m >> 1) + i8;
        ch = 16 * ks + 8 * (m & 1);
        quad = ks * 4 + tid;
      } else {           // rows = tokens 16 ks (+8 for 1, 3), channels 16 mt (+8 for 2, 3)
        tok = 16 * ks + 8 * (m & 1) + i8;
        ch = 16 * mt + 8 * (m >> 1);
        quad = ((mt >> 1) * 2 + ks) * 4 + tid;
      }
      uint32_t r[4];
      const uint32_t addr = (uint32_t)__cvta_generic_to_shared(base + tok * (D + 8) + ch);
      if (KIND == 0) ldsm_x4(addr, r);
      else ldsm_x4_t(addr, r);
      uint32_t bits = 0;
      if (PLAIN || *reinterpret_cast<const uint32_t*>(&q.exact[KIND][quad * 4]) == 0) {
        const float4 zq = *reinterpret_cast<const float4*>(&q.z[KIND][quad * 4]);
        const float4 rq = *reinterpret_cast<const float4*>(&q.rcp[KIND][quad * 4]);
        const float4 nq = *reinterpret_cast<const float4*>(&q.nsc[KIND][quad * 4]);
        code_fragment<BITS, !PLAIN>(r, zq, rq, nq, 4 * s, bits);
      } else {
        bits = code_fragment_exact<BITS>(r[0], r[1], r[2], r[3], &q.z[KIND][quad * 4],
                                         &q.s[KIND][quad * 4], 4 * s);
      }
      word |= bits;
    }
    words[wj] = word;
  }
  uint32_t* dst = out + (wi0 >> 2) * 128 + lane * 4 + (wi0 & 3);
  if constexpr (WW == 4) *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
  else if constexpr (WW == 2) *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
  else *dst = words[0];
}

// Quantize the staged group into one block at `blk` (global). Called by all 256
// threads once the staged rows are visible to every thread; the caller synchronizes
// again before it reuses `g` or `q`.
//   1. (min, max) of key channel pairs over each half of the tokens (threads < D)
//      and of the value groups (token, 32 channels) (threads 128 .. 128 + D - 1);
//   2. parameters: key channels (the halves combined) and value groups;
//   3. code words: warps 0-3 keys, 4-7 values.
template <int D, int BITS>
__device__ void quantize_block(const GroupStage<D>& g, QuantScratch<D>& q,
                               uint8_t* __restrict__ blk) {
  static_assert(D == 64 || D == 128, "head dim");
  constexpr int NGC = D / KVC_GROUP;
  __half* kS = reinterpret_cast<__half*>(blk + off_kscale(D, BITS));
  __half* kZ = reinterpret_cast<__half*>(blk + off_kzero(D, BITS));
  __half* vS = reinterpret_cast<__half*>(blk + off_vscale(D, BITS));
  __half* vZ = reinterpret_cast<__half*>(blk + off_vzero(D, BITS));
  const int th = threadIdx.x;
  const int vv = th - 128, gc = vv >> 5, t = vv & 31;   // value role
  float vl = 0.f, vh = 0.f;
  if (th < D) {
    const int cp = th % (D / 2), hf = th / (D / 2);
    const __nv_bfloat162* col = reinterpret_cast<const __nv_bfloat162*>(&g.k[16 * hf][2 * cp]);
    constexpr int RS = (D + 8) / 2;   // row stride in pairs
    __nv_bfloat162 lo = col[0], hi = lo;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      const __nv_bfloat162 x = col[i * RS];
      lo = __hmin2(lo, x);
      hi = __hmax2(hi, x);
    }
    q.kred[hf][cp] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  } else if (vv >= 0 && vv < D) {
    const uint4* row = reinterpret_cast<const uint4*>(&g.v[t][gc * KVC_GROUP]);
    uint4 a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = row[i];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(a);
    __nv_bfloat162 lo = p[0], hi = p[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      lo = __hmin2(lo, p[i]);
      hi = __hmax2(hi, p[i]);
    }
    vl = fminf(__low2float(lo), __high2float(lo));
    vh = fmaxf(__low2float(hi), __high2float(hi));
  }
  __syncthreads();
  bool exact = false;
  if (th < D) {
    const int c = th;
    const uint2 a = q.kred[0][c >> 1], b = q.kred[1][c >> 1];
    const int sh = (c & 1) * 16;
    const float lo = fminf(__uint_as_float((a.x >> sh) << 16), __uint_as_float((b.x >> sh) << 16));
    const float hi = fmaxf(__uint_as_float((a.y >> sh) << 16), __uint_as_float((b.y >> sh) << 16));
    exact = set_params<D, BITS>(lo, hi, q, 0, kq_pos(c), &kS[kperm(c, D)], &kZ[kperm(c, D)]);
  } else if (vv >= 0 && vv < D) {
    exact = set_params<D, BITS>(vl, vh, q, 1, vq_pos(t, gc), &vS[vs_index(t, gc, NGC)],
                                &vZ[vsz_index(t, gc, NGC)]);
  }
  // block-uniform: every group plain (divide-free, no clamp), or check each tile
  const bool plain = __syncthreads_or(exact) == 0;
  const int warp = th >> 5, lane = th & 31;
  uint32_t* kw = reinterpret_cast<uint32_t*>(blk + off_kcodes(D, BITS));
  uint32_t* vw = reinterpret_cast<uint32_t*>(blk + off_vcodes(D, BITS));
  if (plain) {
    if (warp < 4) code_words<D, BITS, 0, true>(g, q, kw, warp, lane);
    else code_words<D, BITS, 1, true>(g, q, vw, warp - 4, lane);
  } else {
    if (warp < 4) code_words<D, BITS, 0, false>(g, q, kw, warp, lane);
    else code_words<D, BITS, 1, false>(g, q, vw, warp - 4, lane);
  }
}

// Window ring rows (layout maps win_k_index / win_v_index).
__device__ __forceinline__ void window_store(__nv_bfloat16* __restrict__ wk,
                                             __nv_bfloat16* __restrict__ wv, int slot, int c, int D,
                                             __nv_bfloat16 kval, __nv_bfloat16 vval) {
  wk[win_k_index(slot, c, D)] = kval;
  wv[win_v_index(slot, c, D)] = vval;
}

__device__ __forceinline__ __nv_bfloat16 window_load_k(const __nv_bfloat16* wk, int slot, int c,
                                                       int D) {
  return wk[win_k_index(slot, c, D)];
}
__device__ __forceinline__ __nv_bfloat16 window_load_v(const __nv_bfloat16* wv, int slot, int c,
                                                       int D) {
  return wv[win_v_index(slot, c, D)];
}

}  // namespace kvc
