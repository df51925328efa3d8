// score.cu -- entry points of the scoring launch (score_tc.cu): the cache's own
// scratch, or scratch given explicitly.
//
// PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
// Funneling, §4.2.2 "KV Cache Selection"; MiniKV §2 eq. (1).
#include "kvc_internal.cuh"

namespace kvc {

cudaError_t launch_score(const kvc_cache* c, int layer, const __nv_bfloat16* q_obs,
                         const __nv_bfloat16* k, cudaStream_t stream) {
  (void)layer;
  return launch_score_tc(c->dims, q_obs, k, c->stats, c->gsync, c->scores, c->err, stream);
}

// The same launch with the scratch buffers given explicitly (used by the
// allocation-free selection entry point, which has no error word).
cudaError_t launch_score_into(const kvc_dims& d, const __nv_bfloat16* q_obs,
                              const __nv_bfloat16* k, float2* stats, unsigned* gsync,
                              float* scores, cudaStream_t stream) {
  return launch_score_tc(d, q_obs, k, stats, gsync, scores, nullptr, stream);
}

}  // namespace kvc
