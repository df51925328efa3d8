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
#include "quant_device.cuh"

namespace kvc {
namespace {

constexpr int kThreads = kDecWarps * 32;
constexpr int kGroupsPerWarp = kGroupsPerCta / kDecWarps;
constexpr int kSlotsPerWarp = kWinSlotsPerCta / kDecWarps;
static_assert(kSlotsPerWarp == 16 || kSlotsPerWarp == 32, "window warps take 16 or 32 slots");
constexpr unsigned kWaitLimit = 1u << 20;   // bounded mbarrier polls (far above any copy)
static_assert(kGroupsPerWarp <= 8, "the key zero-point product covers at most 8 groups");

struct DecLayer {
  int n_groups;     // packed groups read by the packed CTAs (a group flushed here excluded)
  int win_start;    // ring start slot after this launch's append
  int win_len;      // window tokens after this launch's append
  int n_pctas, n_ctas, cta_begin, cap_groups;
  int new_slot;     // ring slot of the token appended in this launch, or -1
  int flush_start;  // ring slot of the oldest token when this launch flushes a group, or -1
  int pad;
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
// Returns false if the wait gave up (error word set; a second bounded wait lets
// copies still in flight land before the CTA can exit).
__device__ bool warp_stage(uint64_t* bar, void* dst0, const void* src0, uint32_t bytes0,
                           void* dst1, const void* src1, uint32_t bytes1, unsigned* err) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" :: "r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  if (lane == 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                 :: "r"(smem_u32(bar)), "r"(bytes0 + bytes1) : "memory");
    bulk_g2s(dst0, src0, bytes0, bar);
    if (bytes1) bulk_g2s(dst1, src1, bytes1, bar);
  }
  bool done = false;
  for (unsigned it = 0; it < kWaitLimit && !done; ++it) done = mbar_try_wait(bar, 0);
  if (!done) {
    if (lane == 0) atomicOr(err, 1u);
    for (unsigned it = 0; it < kWaitLimit && !done; ++it) done = mbar_try_wait(bar, 0);
    done = false;
  }
  __syncwarp();
  return __all_sync(0xffffffffu, done);
}

// Two codes of pair slot P of a word as an exact fp16 pair (even code low half).
// The masked field sits at bit BITS*j of a byte under the fp16 exponent of 1024,
// so the half is 1024 + code * 2^(BITS*j); one fused multiply-add rescales it.
template <int BITS, int P>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w) {
  constexpr int CPB = 8 / BITS;              // codes per byte
  constexpr int S = P / CPB, J = P % CPB;
  constexpr uint32_t mask = (((1u << BITS) - 1u) * 0x00010001u) << (BITS * J);
  const uint32_t v = ((w >> (8 * S)) & mask) | 0x64006400u;
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

// Accumulator registers a lane keeps per C fragment: rows gid and gid+8 when both
// carry data (g = 8: hi rows 0-7, lo rows 8-15), else only row gid (rows 8-15 of
// the operands are zero for g <= 4, so their results are never kept).
template <int GQ>
constexpr int acc_regs() { return GQ == 8 ? 4 : 2; }

template <int D, int GQ>
struct WarpState {
  float m;                       // running max (log2 domain) of this lane's row
  float l;                       // lane-partial sum of exp2
  float o[D / 8][acc_regs<GQ>()];  // value accumulators
  float cz[acc_regs<GQ>()];      // value zero-point accumulators (cols = channel groups)
};

// c += A * B on a kept-rows accumulator (rows gid+8 discarded when g <= 4).
template <int GQ>
__device__ __forceinline__ void mma_acc(float (&c)[acc_regs<GQ>()], uint32_t a0, uint32_t a1,
                                        uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1,
                                        bool bf16 = false);

template <int GQ>
__device__ __forceinline__ void mma_acc(float (&c)[acc_regs<GQ>()], uint32_t a0, uint32_t a1,
                                        uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1,
                                        bool bf16) {
  if constexpr (GQ == 8) {
    if (bf16) mma_bf16(c, a0, a1, a2, a3, b0, b1);
    else mma_f16(c, a0, a1, a2, a3, b0, b1);
  } else {
    // rows gid+8 are zero operands: feed zero accumulators, drop their results
    float d2, d3;
    if (bf16)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%10,%11,%12,%12};\n"
          : "=f"(c[0]), "=f"(c[1]), "=f"(d2), "=f"(d3)
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
            "f"(0.f));
    else
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%10,%11,%12,%12};\n"
          : "=f"(c[0]), "=f"(c[1]), "=f"(d2), "=f"(d3)
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
            "f"(0.f));
  }
}

// Row gid+8 of an accumulator (zero when it is not kept).
template <int GQ>
__device__ __forceinline__ float row8(const float (&c)[acc_regs<GQ>()], int e) {
  if constexpr (GQ == 8) return c[2 + e];
  else return 0.f;
}

template <int D, int GQ>
__device__ __forceinline__ void state_init(WarpState<D, GQ>& st) {
  st.m = -INFINITY;
  st.l = 0.f;
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < acc_regs<GQ>(); ++e) st.o[i][e] = 0.f;
#pragma unroll
  for (int e = 0; e < acc_regs<GQ>(); ++e) st.cz[e] = 0.f;
}

// Row roles of this lane in the 16-row operands.
template <int GQ>
struct Roles {
  bool hi, lo;
  int head;
  __device__ explicit Roles(int gid) {
    if constexpr (GQ == 8) { hi = true; lo = true; head = gid; }
    else { hi = gid < GQ; lo = gid >= GQ && gid < 2 * GQ; head = gid % GQ; }
  }
};

// Online-softmax update from the combined logits x[NT][2] (exp2 weights returned in x).
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
      for (int e = 0; e < acc_regs<GQ>(); ++e) st.o[i][e] *= corr;
#pragma unroll
    for (int e = 0; e < acc_regs<GQ>(); ++e) st.cz[e] *= corr;
    st.m = mnew;
  }
  float s = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float p = (x[nt][e] == -INFINITY) ? 0.f : exp2f(x[nt][e] - st.m);
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
// `base` points at n_grp (<= kGroupsPerWarp) consecutive group blocks in shared
// memory. Two phases: the key logits of every group (independent tensor-core
// chains, each split over two accumulators), one online-softmax update over all
// the warp's tokens, then the value products.
template <int D, int BITS, int GQ>
__device__ void packed_warp(WarpState<D, GQ>& st, const uint8_t* base, int n_grp,
                            const __nv_bfloat16* __restrict__ qrow_base, float sl2) {
  constexpr int KS = D / 16, NTV = D / 8, WPL = D * BITS / 32, PPW = 16 / BITS;
  constexpr int NGC = D / 32, BB = 8 * D * (BITS + 1), R2 = acc_regs<GQ>();
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
        const int c = 16 * ks + 2 * tid + 8 * e2;
        const float a = active ? __bfloat162float(qr[c]) : 0.f;
        const float b = active ? __bfloat162float(qr[c + 1]) : 0.f;
        qh[ks][e2] = __floats2half2_rn(a, b);
      }
  }
  // key zero-point sums for all the warp's groups: C[row][col] = q_row . Z_{col}
  float zb0, zb1;
  {
    const int gz = gid < n_grp ? gid : 0;
    const uint4* zp = reinterpret_cast<const uint4*>(base + (size_t)gz * BB + off_kzero(D, BITS) +
                                                     tid * (D / 4) * 2);
    float cz4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      const uint4 z = zp[ch];
      const int ks0 = 2 * ch;
      mma_f16(cz4, R.hi ? h2u(qh[ks0][0]) : 0u, 0u, R.hi ? h2u(qh[ks0][1]) : 0u, 0u, z.x, z.y);
      mma_f16(cz4, R.hi ? h2u(qh[ks0 + 1][0]) : 0u, 0u, R.hi ? h2u(qh[ks0 + 1][1]) : 0u, 0u,
              z.z, z.w);
    }
    zb0 = cz4[0];
    zb1 = cz4[1];
  }

  // ---- phase 1: key logits of every group
  float x[kGroupsPerWarp * 4][2];
#pragma unroll
  for (int j = 0; j < kGroupsPerWarp; ++j) {
    if (j >= n_grp) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) x[j * 4 + nt][0] = x[j * 4 + nt][1] = -INFINITY;
      continue;
    }
    const int src = gid * 4 + (j >> 1);
    const float z0 = __shfl_sync(0xffffffffu, zb0, src);
    const float z1 = __shfl_sync(0xffffffffu, zb1, src);
    const float bias = (j & 1) ? z1 : z0;
    const uint8_t* blk = base + (size_t)j * BB;
    // operand A = hi/lo(q * S) per channel pair
    uint32_t ak[KS][4];
    {
      const uint4* sp = reinterpret_cast<const uint4*>(blk + off_kscale(D, BITS) + tid * (D / 4) * 2);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        const uint4 s = sp[ch];
        const uint32_t sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ks = 2 * ch + h;
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const __half2 S2 = u2h(sv[2 * h + e2]);
            const __half2 hi = __hmul2(qh[ks][e2], S2);
            const __half2 lo = __hfma2(qh[ks][e2], S2, __hneg2(hi));
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
    uint32_t kw[WPL];
    {
      const uint4* p = reinterpret_cast<const uint4*>(blk);
#pragma unroll
      for (int i = 0; i < WPL / 4; ++i) {
        const uint4 u = p[i * 32 + lane];
        kw[4 * i] = u.x; kw[4 * i + 1] = u.y; kw[4 * i + 2] = u.z; kw[4 * i + 3] = u.w;
      }
    }
    float ca[4][R2], cb[4][R2];   // even / odd k-steps: two independent chains
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < R2; ++e) { ca[nt][e] = (e < 2) ? bias : 0.f; cb[nt][e] = 0.f; }
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int pi = (nt * KS + ks) * 2;
        const uint32_t b0 = unpack_rt<BITS>(kw[pi / PPW], pi % PPW);
        const uint32_t b1 = unpack_rt<BITS>(kw[(pi + 1) / PPW], (pi + 1) % PPW);
        if (ks & 1) mma_acc<GQ>(cb[nt], ak[ks][0], ak[ks][1], ak[ks][2], ak[ks][3], b0, b1);
        else mma_acc<GQ>(ca[nt], ak[ks][0], ak[ks][1], ak[ks][2], ak[ks][3], b0, b1);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float c8 = 0.f;
        if constexpr (GQ == 8) c8 = ca[nt][2 + e] + cb[nt][2 + e];
        x[j * 4 + nt][e] = combine_rows<GQ>(ca[nt][e] + cb[nt][e], c8);
      }
  }
  softmax_update<D, GQ, kGroupsPerWarp * 4>(st, x, sl2);

  // ---- phase 2: values
#pragma unroll
  for (int j = 0; j < kGroupsPerWarp; ++j) {
    if (j >= n_grp) continue;
    const uint8_t* blk = base + (size_t)j * BB;
    uint32_t vw[WPL];
    {
      const uint4* p = reinterpret_cast<const uint4*>(blk + off_vcodes(D, BITS));
#pragma unroll
      for (int i = 0; i < WPL / 4; ++i) {
        const uint4 u = p[i * 32 + lane];
        vw[4 * i] = u.x; vw[4 * i + 1] = u.y; vw[4 * i + 2] = u.z; vw[4 * i + 3] = u.w;
      }
    }
    const uint32_t* vs = reinterpret_cast<const uint32_t*>(blk + off_vscale(D, BITS));
    const uint32_t* vz = reinterpret_cast<const uint32_t*>(blk + off_vzero(D, BITS));
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      // p of tokens 16ks + 2tid + {0,1} and + 8 + {0,1}
      const float p0 = x[j * 4 + 2 * ks][0], p1 = x[j * 4 + 2 * ks][1];
      const float p2 = x[j * 4 + 2 * ks + 1][0], p3 = x[j * 4 + 2 * ks + 1][1];
      const __half2 ph01 = __floats2half2_rn(p0, p1), ph23 = __floats2half2_rn(p2, p3);
      const __half2 pl01 = __floats2half2_rn(p0 - __low2float(ph01), p1 - __high2float(ph01));
      const __half2 pl23 = __floats2half2_rn(p2 - __low2float(ph23), p3 - __high2float(ph23));
      const int P0 = 8 * ks + tid, P1 = P0 + 4;     // token-pair indices
      {
        // value zero-points: C[row][gc] += p_row,t * Z_t,gc  (B column gc = gid)
        const uint32_t bz0 = gid < NGC ? vz[P0 * NGC + gid] : 0u;
        const uint32_t bz1 = gid < NGC ? vz[P1 * NGC + gid] : 0u;
        if constexpr (GQ == 8) {
          mma_acc<GQ>(st.cz, h2u(ph01), h2u(pl01), h2u(ph23), h2u(pl23), bz0, bz1);
        } else {
          const uint32_t a0 = R.hi ? h2u(ph01) : (R.lo ? h2u(pl01) : 0u);
          const uint32_t a2 = R.hi ? h2u(ph23) : (R.lo ? h2u(pl23) : 0u);
          mma_acc<GQ>(st.cz, a0, 0u, a2, 0u, bz0, bz1);
        }
      }
#pragma unroll
      for (int gc = 0; gc < NGC; ++gc) {
        const __half2 S01 = u2h(vs[P0 * NGC + gc]);
        const __half2 S23 = u2h(vs[P1 * NGC + gc]);
        const __half2 h01 = __hmul2(ph01, S01), h23 = __hmul2(ph23, S23);
        const __half2 l01 = __hfma2(pl01, S01, __hfma2(ph01, S01, __hneg2(h01)));
        const __half2 l23 = __hfma2(pl23, S23, __hfma2(ph23, S23, __hneg2(h23)));
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
          const uint32_t b0 = unpack_rt<BITS>(vw[pi / PPW], pi % PPW);
          const uint32_t b1 = unpack_rt<BITS>(vw[(pi + 1) / PPW], (pi + 1) % PPW);
          mma_acc<GQ>(st.o[nt], a0, a1, a2, a3, b0, b1);
        }
      }
    }
  }
}

// ------------------------------------------------------------- window slots
// wk: NS staged key rows [slot][D] (kperm order); wv: NS/2 staged value pair rows
// [pair][D] of 32-bit words (vperm order); the first n_valid slots are live.
template <int D, int GQ, int NS>
__device__ void window_warp(WarpState<D, GQ>& st, const __nv_bfloat16* wk, const uint32_t* wv,
                            int n_valid, const __nv_bfloat16* __restrict__ qrow_base, float sl2) {
  constexpr int KS = D / 16, NTV = D / 8, NT = NS / 8, KSV = NS / 16;
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
        const int c = 16 * ks + 2 * tid + 8 * e2;
        const uint32_t u = *reinterpret_cast<const uint32_t*>(qr + c);
        aq[ks][e2] = R.hi ? u : 0u;
      }
  }
  float x[NT][2];
  {
    float c[NT][acc_regs<GQ>()], cb[NT][acc_regs<GQ>()];   // even / odd k-steps
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < acc_regs<GQ>(); ++e) { c[nt][e] = 0.f; cb[nt][e] = 0.f; }
      const uint4* kr = reinterpret_cast<const uint4*>(wk + (size_t)(nt * 8 + gid) * D + tid * (D / 4));
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        const uint4 u = kr[ch];
        mma_acc<GQ>(c[nt], aq[2 * ch][0], 0u, aq[2 * ch][1], 0u, u.x, u.y, true);
        mma_acc<GQ>(cb[nt], aq[2 * ch + 1][0], 0u, aq[2 * ch + 1][1], 0u, u.z, u.w, true);
      }
#pragma unroll
      for (int e = 0; e < acc_regs<GQ>(); ++e) c[nt][e] += cb[nt][e];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = combine_rows<GQ>(c[nt][e], row8<GQ>(c[nt], e));
        const int col = nt * 8 + 2 * tid + e;
        x[nt][e] = col < n_valid ? v : -INFINITY;
      }
  }
  softmax_update<D, GQ, NT>(st, x, sl2);
#pragma unroll
  for (int ks = 0; ks < KSV; ++ks) {
    const float p0 = x[2 * ks][0], p1 = x[2 * ks][1], p2 = x[2 * ks + 1][0], p3 = x[2 * ks + 1][1];
    __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1), h23 = __floats2bfloat162_rn(p2, p3);
    __nv_bfloat162 l01 = __floats2bfloat162_rn(p0 - __low2float(h01), p1 - __high2float(h01));
    __nv_bfloat162 l23 = __floats2bfloat162_rn(p2 - __low2float(h23), p3 - __high2float(h23));
    const uint32_t H01 = *reinterpret_cast<uint32_t*>(&h01), H23 = *reinterpret_cast<uint32_t*>(&h23);
    const uint32_t L01 = *reinterpret_cast<uint32_t*>(&l01), L23 = *reinterpret_cast<uint32_t*>(&l23);
    uint32_t a0, a1, a2, a3;
    if constexpr (GQ == 8) { a0 = H01; a1 = L01; a2 = H23; a3 = L23; }
    else {
      a0 = R.hi ? H01 : (R.lo ? L01 : 0u); a1 = 0u;
      a2 = R.hi ? H23 : (R.lo ? L23 : 0u); a3 = 0u;
    }
    const int P0 = 8 * ks + tid, P1 = P0 + 4;
    const uint4* v0 = reinterpret_cast<const uint4*>(wv + (size_t)P0 * D + gid * (D / 8));
    const uint4* v1 = reinterpret_cast<const uint4*>(wv + (size_t)P1 * D + gid * (D / 8));
#pragma unroll
    for (int ch = 0; ch < NTV / 4; ++ch) {
      const uint4 b0 = v0[ch], b1 = v1[ch];
      mma_acc<GQ>(st.o[4 * ch + 0], a0, a1, a2, a3, b0.x, b1.x, true);
      mma_acc<GQ>(st.o[4 * ch + 1], a0, a1, a2, a3, b0.y, b1.y, true);
      mma_acc<GQ>(st.o[4 * ch + 2], a0, a1, a2, a3, b0.z, b1.z, true);
      mma_acc<GQ>(st.o[4 * ch + 3], a0, a1, a2, a3, b0.w, b1.w, true);
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
  float wt[kDecWarps][GQ];   // CTA merge weights
  float M[GQ], L[GQ];
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
    const float o0 = combine_rows<GQ>(st.o[nt][0], row8<GQ>(st.o[nt], 0));
    const float o1 = combine_rows<GQ>(st.o[nt][1], row8<GQ>(st.o[nt], 1));
    if (R.hi) {
      sm.o[warp][R.head][nt * 8 + 2 * tid] = o0;
      sm.o[warp][R.head][nt * 8 + 2 * tid + 1] = o1;
    }
  }
  const float z0 = combine_rows<GQ>(st.cz[0], row8<GQ>(st.cz, 0));
  const float z1 = combine_rows<GQ>(st.cz[1], row8<GQ>(st.cz, 1));
  if (R.hi) {
    if (2 * tid < D / 32) sm.bias[warp][R.head][2 * tid] = z0;
    if (2 * tid + 1 < D / 32) sm.bias[warp][R.head][2 * tid + 1] = z1;
    if (tid == 0) { sm.m[warp][R.head] = st.m; sm.l[warp][R.head] = l; }
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
  return stage_bytes<D, BITS, GQ>() + block_bytes(D, BITS) + kDecWarps * 8;
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

  WarpState<D, GQ> st;
  state_init(st);
  if (cidx < Ld.n_pctas) {
    const int g0 = cidx * kGroupsPerCta + warp * kGroupsPerWarp;
    const int ng = min(kGroupsPerWarp, Ld.n_groups - g0);
    if (ng > 0 &&
        warp_stage(&bars[warp], wbuf, ubase + (size_t)g0 * BB, (uint32_t)(ng * BB), nullptr,
                   nullptr, 0u, P.err))
      packed_warp<D, BITS, GQ>(st, wbuf, ng, qrow, P.sl2);
  } else {
    const int wc = cidx - Ld.n_pctas;
    const size_t wunit = (size_t)layer * P.units + unit;
    __nv_bfloat16* wk = win_k + wunit * P.R * D;
    __nv_bfloat16* wv = win_v + wunit * P.R * D;
    const bool flush = wc == 0 && Ld.flush_start >= 0;
    int owner = -1;
    if (Ld.new_slot >= 0) owner = Ld.win_len == 0 ? 0 : (Ld.win_len - 1) / kWinSlotsPerCta;
    const __nv_bfloat16* kn = P.k_new + ((size_t)li * P.units + unit) * D;
    const __nv_bfloat16* vn = P.v_new + ((size_t)li * P.units + unit) * D;
    if (wc == owner)
      for (int c = threadIdx.x; c < D; c += kThreads)
        window_store(wk, wv, Ld.new_slot, c, D, kn[c], vn[c]);
    if (flush) {
      // quantize the oldest group of the window into a new packed block
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
      __syncthreads();   // the staging area is reused by the window copies below
    }
    const int pos0 = wc * kWinSlotsPerCta + warp * kSlotsPerWarp;
    const int n_valid = min(kSlotsPerWarp, Ld.win_len - pos0);
    if (n_valid > 0) {
      const int slot0 = (Ld.win_start + pos0) % P.R;
      __nv_bfloat16* sk = reinterpret_cast<__nv_bfloat16*>(wbuf);
      uint32_t* sv = reinterpret_cast<uint32_t*>(wbuf + kSlotsPerWarp * D * 2);
      if (warp_stage(&bars[warp], sk, wk + (size_t)slot0 * D, (uint32_t)(kSlotsPerWarp * D * 2),
                     sv, wv + (size_t)(slot0 >> 1) * D * 2, (uint32_t)(kSlotsPerWarp * D * 2),
                     P.err)) {
        if (wc == owner && Ld.new_slot >= slot0 && Ld.new_slot < slot0 + kSlotsPerWarp) {
          // the new token was stored through the generic path in this launch: take it
          // from the inputs rather than from the asynchronous copy
          const int r = Ld.new_slot - slot0;
          __nv_bfloat16* svh = reinterpret_cast<__nv_bfloat16*>(sv);
          for (int c = lane; c < D; c += 32) {
            sk[(size_t)r * D + kperm(c, D)] = kn[c];
            svh[((size_t)(r >> 1) * D + vperm(c, D)) * 2 + (r & 1)] = vn[c];
          }
          __syncwarp();
        }
        window_warp<D, GQ, kSlotsPerWarp>(st, sk, sv, n_valid, qrow, P.sl2);
      }
    }
    if (flush && warp == 0) packed_warp<D, BITS, GQ>(st, fblk, 1, qrow, P.sl2);
  }
  __syncthreads();   // every warp is done with the staging area
  warp_to_smem<D, GQ>(st, sm, warp);
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
  float* mypart = part + (size_t)blockIdx.x * GQ * (D + 2);
  for (int i = threadIdx.x; i < GQ * D; i += kThreads) {
    const int r = i / D, cch = i % D;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) O += (sm.o[w][r][cch] + sm.bias[w][r][cch / 32]) * sm.wt[w][r];
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
      L.pad = 0;
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
      L.n_pctas = packed_ctas(ls.n_groups);
      int wctas = window_ctas(L.win_len);
      if (flush && wctas == 0) wctas = 1;
      L.n_ctas = L.n_pctas + wctas;
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
