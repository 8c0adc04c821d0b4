// A decode entry point for callers that cannot allocate device memory.
//
// pkv_forward_decode needs a context over a caller-provided workspace, which
// someone has to cudaMalloc. Some callers cannot do that: code that runs inside
// another framework whose caching allocator owns the device's memory (a raw
// cudaMalloc there can fail or fragment the pool), and latency-sensitive loops
// that must not call cudaMalloc/cudaFree because those calls can synchronise
// the device and stall every other stream. This file gives them one call that
// allocates nothing: the metadata and split-KV scratch live in a fixed-size
// array in the library's own device memory, reserved when the library is
// loaded and kept by every GPU that loads it until the process exits.
//
// The kernels are the same ones pkv_forward_decode launches; only the place
// their scratch lives differs.
#include <mutex>

#include <cmath>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

// Scratch for one call: plan words, per-request metadata, the split-KV work
// list and the partial outputs. Shared by every call on a device.
static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per
// device. The host-side name of the array is not a device address, so it is
// never handed to a kernel directly.
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

int static_config_ok(const pkv_config* cfg);
size_t static_layout_bytes(const pkv_config& cfg, int num_sms, Layout* lay);
void static_grid_sizes(const pkv_config& cfg, int num_sms, int* decode_ctas, int* extend_ctas);

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_forward_decode_static(const pkv_config* cfg, int32_t batch, const int32_t* d_seq_lens,
                                         const int32_t* d_page_table, int32_t page_table_stride, const void* d_q,
                                         const void* d_k_pool, const void* d_v_pool, float sm_scale, float k_scale,
                                         float v_scale, void* d_out, float* d_lse, int32_t* d_error, void* stream) {
  int st = static_config_ok(cfg);
  if (st != PKV_OK) return st;
  if (batch < 0) return PKV_ERR_INVALID_ARG;
  if (batch > cfg->max_batch) return PKV_ERR_CAPACITY;
  if (batch > 0 && (!d_seq_lens || !d_page_table || page_table_stride <= 0)) return PKV_ERR_INVALID_ARG;
  if (!d_q || !d_k_pool || !d_v_pool || !d_out) return PKV_ERR_INVALID_ARG;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!a16(d_q) || !a16(d_k_pool) || !a16(d_v_pool) || !a16(d_out)) return PKV_ERR_INVALID_ARG;
  if (d_lse && (reinterpret_cast<uintptr_t>(d_lse) & 3)) return PKV_ERR_INVALID_ARG;
  if (d_error && (reinterpret_cast<uintptr_t>(d_error) & 3)) return PKV_ERR_INVALID_ARG;
  // masked scores become -inf before the scale multiplies them: it must be positive
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return PKV_ERR_INVALID_ARG;
  if (cfg->kv_dtype == PKV_KV_FP8_E4M3 &&
      (!(k_scale > 0.f) || !std::isfinite(k_scale) || !(v_scale > 0.f) || !std::isfinite(v_scale)))
    return PKV_ERR_INVALID_ARG;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
  Ctx c;
  c.cfg = *cfg;
  if (static_layout_bytes(*cfg, sms, &c.lay) > PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_CAPACITY;
  void* scratch = nullptr;
  st = scratch_address(dev, &scratch);
  if (st != PKV_OK) return st;
  c.ws = static_cast<char*>(scratch);
  c.num_sms = sms;
  static_grid_sizes(*cfg, sms, &c.decode_ctas, &c.extend_ctas);
  c.batch = batch;
  c.mode = PKV_MODE_DECODE;
  c.qo_given = false;
  c.device = dev;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the previous call's error word must not leak into this one
  if (cudaMemsetAsync(c.ws + c.lay.plan, 0, sizeof(int) * kPlanWords, s) != cudaSuccess) return PKV_ERR_CUDA;
  if (batch > 0) {
    st = launch_build_metadata(c, batch, d_seq_lens, nullptr, d_page_table, page_table_stride, s);
    if (st != PKV_OK) return st;
    st = launch_decode(c, d_q, d_k_pool, d_v_pool, sm_scale, k_scale, v_scale, d_out, d_lse, s);
    if (st != PKV_OK) return st;
  }
  if (d_error &&
      cudaMemcpyAsync(d_error, c.ws + c.lay.plan, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}
