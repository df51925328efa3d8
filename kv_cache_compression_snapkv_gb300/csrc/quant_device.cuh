// quant_device.cuh -- the group quantizer and window-ring accessors, shared by
// the prefill/append kernels (quant.cu) and the fused decode step (decode.cu).
//
// KIVI-style asymmetric groups (blog "Quantization: keep each token in fewer
// bits"; MiniKV §4.4): keys per channel over 32 consecutive stored tokens,
// values per token over 32 consecutive channels; zero-point = group min,
// scale = (max - min) / (2^b - 1), both stored as fp16 (round to nearest even).
// Codes use the stored fp16 values: code = rint((x - Z) / S) clamped to
// [0, 2^b - 1], with explicit IEEE round-to-nearest fp32 subtract and divide (no
// contraction) and round-half-to-even conversion; S == 0 gives 0. The divide is
// taken through the reciprocal where that provably gives the same code.
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

__device__ __forceinline__ void group_params(float lo, float hi, int bits, __half& S, __half& Z,
                                             float& Sf, float& Zf, float& rS) {
  const float rng = __fsub_rn(hi, lo);
  const float s32 = __fdiv_rn(rng, (float)((1 << bits) - 1));
  S = __float2half_rn(s32);
  Z = __float2half_rn(lo);
  Sf = __half2float(S);
  Zf = __half2float(Z);
  rS = Sf == 0.f ? 0.f : __frcp_rn(Sf);
}

// code = rint((x - Z) / S) with the quotient first rounded to fp32 (IEEE
// division), clamped to [0, 2^b - 1]; S == 0 gives 0. Evaluated as (x - Z) * rS,
// rS the correctly rounded reciprocal of S: that product and the rounded quotient
// each lie within 2^-24 (relative) of the exact quotient plus one rounding, so they
// differ by less than 2^-22 |q|, and their nearest integers agree unless the
// product lies within that distance of a half-integer. There (margin 2^-18 |q|)
// the division itself is evaluated, so every code equals the division's.
__device__ __forceinline__ int quant_code(float x, float Zf, float Sf, float rS, int bits) {
  if (Sf == 0.f) return 0;
  const float d = __fsub_rn(x, Zf);
  float q = __fmul_rn(d, rS);
  const float fr = __fsub_rn(q, floorf(q));
  if (fabsf(__fsub_rn(fr, 0.5f)) <= 3.814697265625e-06f * fmaxf(1.f, fabsf(q)))
    q = __fdiv_rn(d, Sf);
  const int c = __float2int_rn(q);
  const int top = (1 << bits) - 1;
  return c < 0 ? 0 : (c > top ? top : c);
}

// Staging of one group: 32 key rows and 32 value rows (bf16 as stored, natural
// channel order, rows padded by 8 elements), their codes, and partial min/max
// when a group is split over threads.
template <int D, int NT>
struct GroupSmem {
  static constexpr int NP = NT / D;   // threads per quantization group
  static_assert(NP >= 1 && KVC_GROUP % NP == 0, "thread count must be a multiple of D");
  __nv_bfloat16 k[KVC_GROUP][D + 8];
  __nv_bfloat16 v[KVC_GROUP][D + 8];
  uint8_t kc[KVC_GROUP][D];
  uint8_t vc[KVC_GROUP][D];
  float klo[NP][D], khi[NP][D], vlo[NP][D], vhi[NP][D];
};

// Quantize the staged group into one block at `blk` (global or shared). All NT
// threads of the block call it. Each of the D key groups (channels) and D value
// groups (token, 32 channels) is handled by NP threads taking 32/NP elements.
template <int D, int BITS, int NT>
__device__ void quantize_block(GroupSmem<D, NT>& s, uint8_t* __restrict__ blk) {
  constexpr int NP = GroupSmem<D, NT>::NP, PER = KVC_GROUP / NP, NGC = D / KVC_GROUP;
  __half* kS = reinterpret_cast<__half*>(blk + off_kscale(D, BITS));
  __half* kZ = reinterpret_cast<__half*>(blk + off_kzero(D, BITS));
  __half* vS = reinterpret_cast<__half*>(blk + off_vscale(D, BITS));
  __half* vZ = reinterpret_cast<__half*>(blk + off_vzero(D, BITS));
  const int g = threadIdx.x % D, part = threadIdx.x / D;
  const bool act = threadIdx.x < NP * D;
  const int vt = g / NGC, vgc = g % NGC;       // value group g = (token vt, channels vgc*32..)
  const __nv_bfloat16* vrow = &s.v[vt][vgc * KVC_GROUP + part * PER];
  if (act) {
    float lo = __bfloat162float(s.k[part * PER][g]), hi = lo;
#pragma unroll
    for (int t = 1; t < PER; ++t) {
      const float x = __bfloat162float(s.k[part * PER + t][g]);
      lo = fminf(lo, x);
      hi = fmaxf(hi, x);
    }
    s.klo[part][g] = lo;
    s.khi[part][g] = hi;
    float vl = __bfloat162float(vrow[0]), vh = vl;
#pragma unroll
    for (int j = 1; j < PER; ++j) {
      const float x = __bfloat162float(vrow[j]);
      vl = fminf(vl, x);
      vh = fmaxf(vh, x);
    }
    s.vlo[part][g] = vl;
    s.vhi[part][g] = vh;
  }
  __syncthreads();
  if (act) {
    float lo = s.klo[0][g], hi = s.khi[0][g];
#pragma unroll
    for (int p = 1; p < NP; ++p) { lo = fminf(lo, s.klo[p][g]); hi = fmaxf(hi, s.khi[p][g]); }
    __half S, Z; float Sf, Zf, rS;
    group_params(lo, hi, BITS, S, Z, Sf, Zf, rS);
#pragma unroll
    for (int t = 0; t < PER; ++t)
      s.kc[part * PER + t][g] =
          (uint8_t)quant_code(__bfloat162float(s.k[part * PER + t][g]), Zf, Sf, rS, BITS);
    if (part == 0) { kS[kperm(g, D)] = S; kZ[kperm(g, D)] = Z; }
  }
  if (act) {
    float lo = s.vlo[0][g], hi = s.vhi[0][g];
#pragma unroll
    for (int p = 1; p < NP; ++p) { lo = fminf(lo, s.vlo[p][g]); hi = fmaxf(hi, s.vhi[p][g]); }
    __half S, Z; float Sf, Zf, rS;
    group_params(lo, hi, BITS, S, Z, Sf, Zf, rS);
#pragma unroll
    for (int j = 0; j < PER; ++j)
      s.vc[vt][vgc * KVC_GROUP + part * PER + j] =
          (uint8_t)quant_code(__bfloat162float(vrow[j]), Zf, Sf, rS, BITS);
    if (part == 0) { vS[vs_index(vt, vgc, NGC)] = S; vZ[vsz_index(vt, vgc, NGC)] = Z; }
  }
  __syncthreads();
  // pack code words in fragment order
  constexpr int WPL = D * BITS / 32;
  constexpr int PPW = 16 / BITS;
  constexpr int NW = 32 * WPL;
  uint32_t* kw = reinterpret_cast<uint32_t*>(blk + off_kcodes(D, BITS));
  uint32_t* vw = reinterpret_cast<uint32_t*>(blk + off_vcodes(D, BITS));
  for (int widx = threadIdx.x; widx < 2 * NW; widx += NT) {
    const bool is_v = widx >= NW;
    const int w = is_v ? widx - NW : widx;
    const int lane = (w & 127) >> 2;
    const int wi = (w >> 7) * 4 + (w & 3);
    const int gid = lane >> 2, tid = lane & 3;
    uint32_t word = 0;
#pragma unroll
    for (int P = 0; P < PPW; ++P) {
      uint32_t ce, co;
      if (!is_v) {
        const FragPos f = key_frag(wi, P, D, BITS);
        const int t = 16 * f.mt + gid + 8 * f.rl, c = 16 * f.ks + 2 * tid + 8 * f.rh;
        ce = s.kc[t][c]; co = s.kc[t][c + 1];
      } else {
        const FragPos f = value_frag(wi, P, BITS);
        const int t = 16 * f.ks + 2 * tid + 8 * f.rh, c = 16 * f.mt + gid + 8 * f.rl;
        ce = s.vc[t][c]; co = s.vc[t + 1][c];
      }
      word |= ce << pair_bit(P, BITS);
      word |= co << (16 + pair_bit(P, BITS));
    }
    (is_v ? vw : kw)[w] = word;
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
