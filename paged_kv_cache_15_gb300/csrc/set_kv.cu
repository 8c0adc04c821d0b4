// save_kv_cache / set_kv_buffer ("[SGLang] Hybrid Attention", section "forward:
// 선형 어텐션까지 지원하는 범용 위임": forward(..., save_kv_cache=True) stores the
// step's K/V into the pool before attention).
//
//   pool[loc[i], h, :] = new[i, h, :]        bf16 pool: same bits
//   pool[loc[i], h, :] = e4m3(new * inv)     E4M3 pool: fp32 multiply, then
//                                            cvt.rn.satfinite to E4M3FN
//
// HBM-bound copy: every thread moves one 16-byte vector (8 elements) of K and
// the matching vector of V; consecutive threads cover consecutive bytes of a
// [token][kv_head][width] row, so loads and stores are fully coalesced. When
// the V heads are narrower than the K heads, the threads past a V row's end
// move only their K vector.
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint2 quant8(uint4 x, float inv) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint16_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = f32x2_to_e4m3x2(bf16_lo(w[i]) * inv, bf16_hi(w[i]) * inv);
  return make_uint2((uint32_t)c[0] | ((uint32_t)c[1] << 16), (uint32_t)c[2] | ((uint32_t)c[3] << 16));
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads) set_kv_kernel(void* __restrict__ k_pool, void* __restrict__ v_pool,
                                                          const int* __restrict__ loc,
                                                          const uint4* __restrict__ k_new,
                                                          const uint4* __restrict__ v_new, long long n_vec,
                                                          int vec_per_token, int vec_per_token_v,
                                                          long long num_slots, float k_inv, float v_inv, int* plan) {
  // launched with programmatic serialization: the next kernel may start
  // launching now, and this one touches memory only after the previous grid
  // (which may have produced the new K/V or the slots) has finished
  pdl_launch_dependents();
  pdl_wait();
  for (long long u = (long long)blockIdx.x * kThreads + threadIdx.x; u < n_vec;
       u += (long long)gridDim.x * kThreads) {
    long long tok = u / vec_per_token;
    int within = (int)(u - tok * vec_per_token);
    long long slot = loc[tok];
    if (slot < 0 || slot >= num_slots) {
      if (within == 0) record_error(plan, PKV_DEV_BAD_SLOT, (int)tok);
      continue;
    }
    // K row: vec_per_token vectors; V row: vec_per_token_v (at most as many)
    const uint4 kx = __ldcs(k_new + u);
    const long long dst = slot * vec_per_token + within;
    const bool has_v = within < vec_per_token_v;
    const long long vsrc = tok * vec_per_token_v + within;
    const long long vdst = slot * vec_per_token_v + within;
    if constexpr (kFp8) {
      reinterpret_cast<uint2*>(k_pool)[dst] = quant8(kx, k_inv);
      if (has_v) reinterpret_cast<uint2*>(v_pool)[vdst] = quant8(__ldcs(v_new + vsrc), v_inv);
    } else {
      reinterpret_cast<uint4*>(k_pool)[dst] = kx;
      if (has_v) reinterpret_cast<uint4*>(v_pool)[vdst] = __ldcs(v_new + vsrc);
    }
  }
}

}  // namespace

int launch_set_kv_buffer(Ctx& c, void* k_pool, void* v_pool, const int32_t* loc, const void* k, const void* v,
                         int n, float k_inv, float v_inv, cudaStream_t st) {
  if (n == 0) return PKV_OK;
  // the K heads are at least as wide as the V heads (check_config)
  int vec_per_token = c.cfg.num_kv_heads * c.cfg.head_dim / 8;
  int vec_per_token_v = c.cfg.num_kv_heads * head_dim_v(c.cfg) / 8;
  long long n_vec = (long long)n * vec_per_token;
  long long blocks = (n_vec + kThreads - 1) / kThreads;
  long long cap = (long long)c.num_sms * 16;
  int grid = (int)(blocks < cap ? blocks : cap);
  long long num_slots = (long long)c.cfg.num_pages * c.cfg.page_size;
  int* plan = make_meta(c).plan;
  cudaError_t e;
  if (c.cfg.kv_dtype == PKV_KV_FP8_E4M3)
    e = launch_pdl(set_kv_kernel<true>, dim3(grid), dim3(kThreads), 0, st, k_pool, v_pool, loc, (const uint4*)k,
                   (const uint4*)v, n_vec, vec_per_token, vec_per_token_v, num_slots, k_inv, v_inv, plan);
  else
    e = launch_pdl(set_kv_kernel<false>, dim3(grid), dim3(kThreads), 0, st, k_pool, v_pool, loc, (const uint4*)k,
                   (const uint4*)v, n_vec, vec_per_token, vec_per_token_v, num_slots, k_inv, v_inv, plan);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
