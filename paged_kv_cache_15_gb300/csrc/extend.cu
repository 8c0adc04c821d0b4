// forward_extend on the tensor cores (placeholder until the tcgen05 kernel lands).
#include "pkv_internal.cuh"

namespace pkv {

int launch_extend(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, void* out,
                  float* lse, cudaStream_t st) {
  (void)c; (void)q; (void)k_pool; (void)v_pool; (void)sm_scale; (void)out; (void)lse; (void)st;
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
