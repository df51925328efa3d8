// kvc_internal.cuh -- shared definitions of the compressed-KV-cache library.
//
// Storage layout (all of it device memory owned by the cache):
//
//   packed store  one 32-token "group block" after another, per (layer, b, kv head):
//     [K codes  D*4*BITS bytes][V codes  D*4*BITS bytes]
//     [K scale  D fp16][K zero  D fp16]          per-channel key groups
//     [V scale  32*(D/32) fp16][V zero  ...]     per-token value groups: scales
//                                                [t][gc], zeros [pair][gc][2]
//   The code words are laid out so that lane l of a warp reading words
//   (wi/4)*128 + l*4 + wi%4 holds exactly the A-operand fragments of the
//   m16n8k16 tensor-core products the decode kernel issues (keys: rows = tokens,
//   k = channels; values: rows = channels, k = tokens), two codes per 16-bit half
//   pair. Pair slots are arranged so that the bit position of a code depends only
//   on the operand's k index (see key_pair / value_pair).
//   Key scales/zeros are stored in the order the operand lanes consume them.
//
//   window        bf16 ring of R slots per (layer, b, kv head):
//     keys   [R][D]     channels permuted (kperm) into fragment order, 16-byte
//                       chunks of a row XOR-swizzled by (slot & 7)
//     values [R/2][D][2] token pairs interleaved, channels permuted (vperm),
//                       16-byte chunks of a pair row XOR-swizzled by (pair & 3)
//
// Every layout map below is used by the writer (quantize / append), the reader
// (decode) and the exporter, so they cannot drift apart.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <vector>

#include "kvc.h"

#define KVC_GROUP 32
#define KVC_MAX_LAUNCH_LAYERS 64

namespace kvc {

// ----------------------------------------------------------------- layout maps
// Position of key channel c inside a permuted 16-bit row (window keys, key
// scales/zeros): the 4 values a lane needs per k-step (channels 16ks + 2tid +
// {0, 1, 8, 9}) are adjacent, and a lane's k-steps are contiguous.
__host__ __device__ constexpr int kperm(int c, int D) {
  int ks = c >> 4, r = c & 15;
  int tid = (r & 7) >> 1;
  int e = (r & 1) + 2 * (r >> 3);
  return (tid * (D >> 4) + ks) * 4 + e;
}
// Position of value channel c inside a permuted window value pair-row.
__host__ __device__ constexpr int vperm(int c, int D) {
  return (c & 7) * (D >> 3) + (c >> 3);
}

// Index (in fp16 units) of the value zero of (token t, channel group gc) inside
// its section: token pairs interleaved, so (t, t+1) of one gc form a half2.
__host__ __device__ constexpr int vsz_index(int t, int gc, int ngc) {
  return ((t >> 1) * ngc + gc) * 2 + (t & 1);
}
// Index of the value scale of (token t, channel group gc): tokens t and t + 8 of
// a 16-token half (same gc) form one half2, and the half2 of all channel groups of
// one (half, t % 8) are adjacent.
__host__ __device__ constexpr int vs_index(int t, int gc, int ngc) {
  return (((t >> 4) * 8 + (t & 7)) * ngc + gc) * 2 + ((t >> 3) & 1);
}

// Bytes of one 32-token group block.
__host__ __device__ constexpr int block_bytes(int D, int bits) { return 8 * D * (bits + 1); }
__host__ __device__ constexpr int code_bytes(int D, int bits) { return 4 * D * bits; }

struct CodePos {
  int word;   // 32-bit word index inside the K-code (or V-code) section
  int bit;    // bit offset of the code inside the word
};

// Bit of pair slot P inside each 16-bit half of a word: slot P sits in byte
// P / (8/bits) at field P % (8/bits).
__host__ __device__ constexpr int pair_bit(int P, int bits) {
  return 8 * (P / (8 / bits)) + bits * (P % (8 / bits));
}

// Fragment coordinates of a pair slot. For product (mt, ks) and A register
// r = 2*rh + rl: keys cover token 16mt + gid + 8rl and channels 16ks + 2tid + 8rh
// + {0,1}; values cover channel 16mt + gid + 8rl and tokens 16ks + 2tid + 8rh +
// {0,1}. Word and slot of register (mt, ks, rl, rh):
//   keys   2-bit: word mt*(D/32) + ks/2, slot 4rl + 2(ks&1) + rh
//          4-bit: word mt*(D/16) + ks,   slot 2rl + rh
//   values 2-bit: word mt,               slot 4rl + 2ks + rh
//          4-bit: word 2mt + ks,         slot 2rl + rh
// so the field of a code (slot % (8/bits)) depends only on its k index.
// kcode_pos / vcode_pos below give the word and bit of each (token, channel).

__host__ __device__ inline int word_addr(int lane, int wi) { return (wi >> 2) * 128 + lane * 4 + (wi & 3); }

// Key code of (token t in the group, channel c).
__host__ __device__ inline CodePos kcode_pos(int t, int c, int D, int bits) {
  const int mt = t >> 4, rl = (t >> 3) & 1, gid = t & 7;
  const int ks = c >> 4, rh = (c >> 3) & 1, tid = (c & 7) >> 1, odd = c & 1;
  const int KS = D >> 4;
  int wi, P;
  if (bits == 2) { wi = mt * (KS >> 1) + (ks >> 1); P = 4 * rl + 2 * (ks & 1) + rh; }
  else { wi = mt * KS + ks; P = 2 * rl + rh; }
  CodePos cp;
  cp.word = word_addr(gid * 4 + tid, wi);
  cp.bit = pair_bit(P, bits) + (odd ? 16 : 0);
  return cp;
}

// Value code of (token t in the group, channel c).
__host__ __device__ inline CodePos vcode_pos(int t, int c, int D, int bits) {
  (void)D;
  const int ks = t >> 4, rh = (t >> 3) & 1, tid = (t & 7) >> 1, odd = t & 1;
  const int mt = c >> 4, rl = (c >> 3) & 1, gid = c & 7;
  int wi, P;
  if (bits == 2) { wi = mt; P = 4 * rl + 2 * ks + rh; }
  else { wi = 2 * mt + ks; P = 2 * rl + rh; }
  CodePos cp;
  cp.word = word_addr(gid * 4 + tid, wi);
  cp.bit = pair_bit(P, bits) + (odd ? 16 : 0);
  return cp;
}

// Window ring positions (bf16 element index inside one unit's ring).
__host__ __device__ inline int win_k_index(int slot, int c, int D) {
  const int pos = kperm(c, D);
  return slot * D + ((((pos >> 3) ^ (slot & 7)) << 3) | (pos & 7));
}
__host__ __device__ inline int win_v_index(int slot, int c, int D) {
  const int w = vperm(c, D);
  const int ws = (((w >> 2) ^ ((slot >> 1) & 3)) << 2) | (w & 3);
  return ((slot >> 1) * D + ws) * 2 + (slot & 1);
}

// Section offsets inside a block (bytes).
__host__ __device__ constexpr int off_kcodes(int, int) { return 0; }
__host__ __device__ constexpr int off_vcodes(int D, int bits) { return code_bytes(D, bits); }
__host__ __device__ constexpr int off_kscale(int D, int bits) { return 2 * code_bytes(D, bits); }
__host__ __device__ constexpr int off_kzero(int D, int bits) { return 2 * code_bytes(D, bits) + 2 * D; }
__host__ __device__ constexpr int off_vscale(int D, int bits) { return 2 * code_bytes(D, bits) + 4 * D; }
__host__ __device__ constexpr int off_vzero(int D, int bits) { return 2 * code_bytes(D, bits) + 6 * D; }

// A device-side check of the checked build (compiled with -DKVC_CHECKED=1) that
// found a caller-supplied index out of range sets this bit of the cache's error word
// (the access is skipped); the next call on the cache returns KVC_E_DEVICE_CHECK.
// Waits that give up set other bits (KVC_E_TIMEOUT).
constexpr unsigned kErrDeviceCheck = 1u << 31;
#if defined(KVC_CHECKED) && KVC_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// ------------------------------------------------------------------ cache state
struct LayerState {
  int prefilled = 0;
  int bits = 2;          // 2 or 4 (packed groups), or 16 (every token exact in the window)
  int R = 0;             // window ring length (slots)
  int block_bytes = 0;   // bytes of one packed group block (0 at 16 bits)
  int budget = 0;        // clipped budget (tokens per head)
  int n_kept = 0;        // selected prompt tokens per head
  int scored = 0;        // 1 if the selection is stored in kept_ptr (else identity)
  int32_t* kept_ptr = nullptr;  // stored selection [units][n_kept]
  int cap_groups = 0;    // packed capacity per (b, h) in groups
  int n_groups = 0;      // packed groups per (b, h)
  int win_start = 0;     // ring start slot
  int win_len = 0;       // tokens in the window
  int appended = 0;
  size_t packed_off = 0; // byte offset of the layer inside the packed store
  size_t win_off = 0;    // element offset of the layer's rings inside win_k / win_v
  size_t kept_off = 0;   // element offset of the layer inside kept[]
};

}  // namespace kvc

struct kvc_cache {
  kvc_dims dims{};
  int device = 0;
  int n_sm = 0;                 // SMs of the device (decode grid)
  int g = 1;                    // GQA group
  std::vector<kvc::LayerState> L;
  // storage
  uint8_t* packed = nullptr;  size_t packed_bytes = 0;
  __nv_bfloat16* win_k = nullptr;
  __nv_bfloat16* win_v = nullptr; size_t win_elems = 0;
  int32_t* kept = nullptr;    size_t kept_elems = 0;
  // scratch
  float2* stats = nullptr;    size_t stats_elems = 0;  // scoring partial row stats
  unsigned* gsync = nullptr;  // scoring counters, 1 + B*H words (zero between launches)
  float* scores = nullptr;
  float* pooled = nullptr;    size_t score_elems = 0;
  unsigned long long* score_fx = nullptr;  // fixed-point sums of the cumulated attention
  float* dec_ws = nullptr;    size_t dec_ws_floats = 0;  // decode partial states
  unsigned* dec_cnt = nullptr; // decode arrival tickets, n_layers * B*H words (zero between launches)
  // error word set by bounded device waits that gave up: mapped pinned host memory
  // where the device has native host atomics (err_host then reads it without a
  // synchronisation, so the next call on the cache reports it), else device memory
  unsigned* err = nullptr;
  volatile unsigned* err_host = nullptr;
  void* err_pinned = nullptr;
  bool wait_limit_set = false; // polls per decode staging wait set by kvc_set_wait_limit
  unsigned wait_limit = 0;
  int last_scored_layer = -1;
  std::vector<void*> allocations;
};

namespace kvc {

// Process-wide count of kernels launched by this library (kvc_launch_count).
void count_launches(int n);

// Raise `kernel`'s dynamic shared-memory limit to at least `bytes` on the current
// device; the driver call is made only when the limit has to grow.
cudaError_t ensure_smem(const void* kernel, size_t bytes);

// Programmatic dependent launch. Kernels of this library are launched with the
// programmatic-stream-serialization attribute: a kernel may be scheduled while the
// previous kernel of the stream drains, runs its shared-memory set-up, and waits
// in pdl_wait() (until the previous grids have completed and their writes are
// visible) before it reads or writes global memory; pdl_release() then lets the
// next kernel be scheduled early in turn. Without the attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Launch attribute for the above (fills attr, returns it for chaining).
inline cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// --------------------------------------------------------------- launch helpers
// (defined in the .cu files; all enqueue on `stream` and return a CUDA error)
cudaError_t launch_score(const kvc_cache* c, int layer, const __nv_bfloat16* q_obs,
                         const __nv_bfloat16* k, cudaStream_t stream);
cudaError_t launch_pool_topk(const kvc_cache* c, int layer, int32_t* kept_out, int k_sel,
                             cudaStream_t stream);
// Gather + quantize + pack of the kept tokens: kept[] positions, or (kept == NULL,
// sinks >= 0) the sink + recent-window positions, stored to kept_out; else all.
cudaError_t launch_gather_quant(const kvc_cache* c, int layer, const int32_t* kept, int n_kept,
                                const __nv_bfloat16* k, const __nv_bfloat16* v,
                                cudaStream_t stream, int sinks = -1,
                                int32_t* kept_out = nullptr);
cudaError_t launch_append(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* k_new, const __nv_bfloat16* v_new,
                          const int* flush_flags, cudaStream_t stream);
cudaError_t launch_decode_step(const kvc_cache* c, int layer_begin, int layer_count,
                               const __nv_bfloat16* q, const __nv_bfloat16* k_new,
                               const __nv_bfloat16* v_new, const int* flush_flags, float* out,
                               cudaStream_t stream);
cudaError_t launch_decode(const kvc_cache* c, int layer_begin, int layer_count,
                          const __nv_bfloat16* q, float* out, cudaStream_t stream);
cudaError_t launch_export(const kvc_cache* c, int layer, const kvc_export* dst,
                          cudaStream_t stream);
// Scoring on the tensor cores (row statistics, their merge into row normalisers,
// per-key column sums) in one cooperative launch. gsync: 1 + B*H words of device
// memory that are zero before the launch and are zero again after it; err may be
// NULL.
cudaError_t launch_score_tc(const kvc_dims& d, const __nv_bfloat16* q_obs,
                            const __nv_bfloat16* k, float2* stats, unsigned* gsync, float* scores,
                            unsigned* err, cudaStream_t stream);
// Selection launches with explicit scratch (allocation-free entry point); err is
// the scoring launch's error word.
cudaError_t launch_score_into(const kvc_dims& d, const __nv_bfloat16* q_obs,
                              const __nv_bfloat16* k, float2* stats, unsigned* gsync,
                              float* scores, unsigned* err, cudaStream_t stream);
// Full-prompt cumulated attention (un-normalised column sums, key blocks of 128 with
// running row maxima) of every unit into scores [unit][n - alpha]; q_full is
// [B][Hq][n][d]. The sums are accumulated in fx (64-bit fixed point, [unit][n -
// alpha], zeroed first) and then converted: the same scores on every run. err may
// be NULL.
cudaError_t launch_acumul(const kvc_dims& d, const __nv_bfloat16* q_full, const __nv_bfloat16* k,
                          float* scores, unsigned long long* fx, unsigned* err,
                          cudaStream_t stream);
// The same scores (skipped when scores is NULL) and, from the same tiles, the
// causal attention output of every prompt query x_out [B][Hq][n][d] (bf16); v is
// [B][Hkv][n][d].
cudaError_t launch_acumul_xo(const kvc_dims& d, const __nv_bfloat16* q_full,
                             const __nv_bfloat16* k, const __nv_bfloat16* v, float* scores,
                             unsigned long long* fx, __nv_bfloat16* x_out, unsigned* err,
                             cudaStream_t stream);
// Population variance of each of `units` rows of m scores (fp32 out, one per row).
cudaError_t launch_score_variance(const float* scores, int units, int m, float* var,
                                  double* ws, size_t ws_doubles, unsigned* cnt,
                                  cudaStream_t stream);
// abort_flag (may be NULL): when it is non-zero at launch time every kept index is
// written as -1.
cudaError_t launch_pool_topk_into(const kvc_dims& d, const float* scores, float* pooled,
                                  int32_t* kept_out, int k_sel, const unsigned* abort_flag,
                                  cudaStream_t stream);

// Decode work decomposition: a unit's work is cut into chunks of 16 window slots
// or of the packed groups that fill the same bytes (at least one).
constexpr int kDecSlotsPerChunk = 16;
__host__ __device__ constexpr int dec_groups_per_chunk(int D, int bits) {
  return kDecSlotsPerChunk * D * 4 / block_bytes(D, bits) > 1
             ? kDecSlotsPerChunk * D * 4 / block_bytes(D, bits) : 1;
}
// Floats of the decode workspace of a cache: two partial states per warp, at
// most 16 warps per SM.
size_t decode_workspace_floats(int n_sm, int g, int D);

// Scoring: partial row statistics kept per (unit, row) for a prompt of n keys
// (at most four epilogue groups in each CTA that owns one of the ceil(n/128) key
// tiles).
inline size_t score_stat_chunks(int n) { return 4 * (size_t)((n + 127) / 128) + 4; }

}  // namespace kvc
