// tcgen05 tensor-core path of the tree attention prefix pass (bf16 caches).
#include "common.cuh"
#include "kernels.h"

namespace medusa {

bool attn_tc_supported(const medusa_tree_t& t, int Hq, const medusa_kv_t& c) {
  (void)t; (void)Hq; (void)c;
  return false;
}

void attn_tc_plan(AttnPlan& p) { (void)p; }

cudaError_t launch_attn_tc(const AttnPlan& p, const medusa_tree_t& t, const void* q,
                           const void* k_new, const void* v_new, const medusa_kv_t& c,
                           const int32_t* L, const float* th_hi, const float* th_lo,
                           float scale_log2, float* out, float* lse, int32_t* status, void* ws,
                           cudaStream_t st) {
  (void)p; (void)t; (void)q; (void)k_new; (void)v_new; (void)c; (void)L; (void)th_hi;
  (void)th_lo; (void)scale_log2; (void)out; (void)lse; (void)status; (void)ws; (void)st;
  return cudaErrorNotSupported;
}

}  // namespace medusa
