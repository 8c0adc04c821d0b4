// Host side of the C ABI declared in include/pkv.h: argument checks, the
// workspace layout, context lifetime, ForwardMode dispatch and launches.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cmath>
#include <new>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_config(const pkv_config* cfg) {
  if (!cfg) return PKV_ERR_INVALID_ARG;
  if (cfg->num_q_heads <= 0 || cfg->num_kv_heads <= 0 || cfg->head_dim <= 0 || cfg->page_size <= 0 ||
      cfg->num_pages <= 0 || cfg->max_batch <= 0 || cfg->max_pages_total <= 0 || cfg->max_q_tokens <= 0 ||
      cfg->max_qo_len <= 0)
    return PKV_ERR_INVALID_ARG;
  if (cfg->kv_dtype != PKV_KV_BF16 && cfg->kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
  if (cfg->num_q_heads % cfg->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int group = cfg->num_q_heads / cfg->num_kv_heads;
  if (group > 16) return PKV_ERR_UNSUPPORTED;
  if (cfg->page_size != kPageSizeSmall && cfg->page_size != kPageSizeLarge) return PKV_ERR_UNSUPPORTED;
  if (cfg->head_dim_v < 0) return PKV_ERR_INVALID_ARG;
  // head widths: 64/64, 128/128, and 192/128 (K and V heads of different widths)
  const int dk = cfg->head_dim, dv = head_dim_v(*cfg);
  if (!((dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 192 && dv == 128))) return PKV_ERR_UNSUPPORTED;
  // E4M3 pools: 128-wide heads (an E4M3 row of 128 codes is one 128-byte span)
  if (cfg->kv_dtype == PKV_KV_FP8_E4M3 && dk != 128) return PKV_ERR_UNSUPPORTED;
  if (decode_row_warps(*cfg) == 0) return PKV_ERR_UNSUPPORTED;  // max_qo_len * group > 128
  // slot indices and pool element offsets must fit the kernels' index types
  const long long slots = (long long)cfg->num_pages * cfg->page_size;
  if (slots > (1ll << 31) - 1) return PKV_ERR_UNSUPPORTED;
  if ((long long)cfg->max_q_tokens * cfg->num_q_heads * dk > (1ll << 40)) return PKV_ERR_UNSUPPORTED;
  // segment counts (pages times segments per page) must fit an int
  if ((long long)cfg->max_pages_total * (cfg->page_size / kSegSlots) > (1ll << 30)) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

// 16-slot segments the batch's pages can hold at most
long long max_segments(const pkv_config& cfg) {
  return (long long)cfg.max_pages_total * (cfg.page_size / kSegSlots);
}

// Persistent-grid sizes: two decode CTAs and one extend CTA per SM, never
// more than the configuration can ever give them work. Decode items per batch
// are at most (segments) / (minimum chunk) + max_batch (every request adds at
// most one partial chunk); extend units at most
// ceil(max_q_tokens * group / 256) + max_batch, plus as many KV splits as
// decode items.
void grid_sizes(const pkv_config& cfg, int num_sms, int* decode_ctas, int* extend_ctas) {
  const long long group = cfg.num_q_heads / cfg.num_kv_heads;
  const long long dec_units =
      (long long)cfg.num_kv_heads * (max_segments(cfg) / kDecodeMinChunkPages + cfg.max_batch + 1);
  const long long ext_units =
      (long long)cfg.num_kv_heads * (((long long)cfg.max_q_tokens * group + kExtendUnitRows - 1) / kExtendUnitRows +
                                     cfg.max_batch) +
      dec_units;  // KV splits of requests whose rows fit one unit
  // two per SM: the decode shapes fit twice; the verify shapes fit once, and
  // the second wave then picks up units as CTAs of the first one finish
  *decode_ctas = (int)(dec_units < num_sms * 2ll ? dec_units : num_sms * 2ll);
  *extend_ctas = (int)(ext_units < num_sms ? ext_units : num_sms);
  if (*decode_ctas < 1) *decode_ctas = 1;
  if (*extend_ctas < 1) *extend_ctas = 1;
}

Layout make_layout(const pkv_config& cfg, int num_sms) {
  Layout L;
  int dctas, ectas;
  grid_sizes(cfg, num_sms, &dctas, &ectas);
  const int group = cfg.num_q_heads / cfg.num_kv_heads;
  const long long target = (long long)dctas * kDecodeTargetWaves;
  L.max_decode_items = (int)(target + cfg.max_batch + 1);
  // unsplit units, plus the splits of requests whose rows fit one unit
  L.max_extend_tiles = (int)(((long long)cfg.max_q_tokens * group + kExtendUnitRows - 1) / kExtendUnitRows +
                             cfg.max_batch + L.max_decode_items);
  long long cap = 2ll * cfg.max_q_tokens;
  if (cap < cfg.max_q_tokens + target) cap = cfg.max_q_tokens + target;
  L.partial_rows_cap = (int)cap;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.plan = take(sizeof(int) * kPlanWords);
  L.kv_indptr = take(sizeof(int) * (cfg.max_batch + 1));
  L.kv_indices = take(sizeof(int) * (size_t)cfg.max_pages_total);
  L.kv_last_page_len = take(sizeof(int) * cfg.max_batch);
  L.qo_indptr = take(sizeof(int) * (cfg.max_batch + 1));
  L.kv_len = take(sizeof(int) * cfg.max_batch);
  L.n_splits = take(sizeof(int) * cfg.max_batch);
  L.ext_splits = take(sizeof(int) * cfg.max_batch);
  L.partial_indptr = take(sizeof(int) * (cfg.max_batch + 1));
  L.token_req = take(sizeof(int) * (size_t)cfg.max_q_tokens);
  L.seg_per_page = cfg.page_size / kSegSlots;
  L.seg_indptr = L.seg_per_page > 1 ? take(sizeof(int) * (cfg.max_batch + 1)) : L.kv_indptr;
  L.seg_indices = L.seg_per_page > 1 ? take(sizeof(int) * (size_t)max_segments(cfg)) : L.kv_indices;
  L.decode_items = take(sizeof(DecodeItem) * (size_t)L.max_decode_items);
  L.extend_tiles = take(sizeof(ExtendTile) * (size_t)L.max_extend_tiles);
  L.partial_o = take(sizeof(uint16_t) * (size_t)cap * cfg.num_q_heads * head_dim_v(cfg));
  L.partial_lse = take(sizeof(float) * (size_t)cap * cfg.num_q_heads);
  L.total = off;
  return L;
}

int device_sms(int* dev_out, int* sms_out) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
  *dev_out = dev;
  *sms_out = sms;
  return PKV_OK;
}

// cuTensorMapEncodeTiled, fetched from the driver at run time
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int get_encoder() {
  if (g_encode) return PKV_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return PKV_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return PKV_OK;
}

// Masked scores become -inf before the scale multiplies them: the scales
// must be positive (k_scale and v_scale matter only for E4M3 pools).
int check_scales(const Ctx& c, float sm_scale, float k_scale, float v_scale) {
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return PKV_ERR_INVALID_ARG;
  if (c.cfg.kv_dtype == PKV_KV_FP8_E4M3 &&
      (!(k_scale > 0.f) || !std::isfinite(k_scale) || !(v_scale > 0.f) || !std::isfinite(v_scale)))
    return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

int check_forward_args(pkv_ctx* ctx, const void* q, const void* kp, const void* vp, const void* out,
                       const float* lse) {
  if (!ctx || !q || !kp || !vp || !out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kp) || !aligned16(vp) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3)) return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

}  // namespace

Meta make_meta(const Ctx& c) {
  Meta m;
  char* w = c.ws;
  m.plan = reinterpret_cast<int*>(w + c.lay.plan);
  m.kv_indptr = reinterpret_cast<const int*>(w + c.lay.kv_indptr);
  m.kv_indices = reinterpret_cast<const int*>(w + c.lay.kv_indices);
  m.seg_indptr = reinterpret_cast<const int*>(w + c.lay.seg_indptr);
  m.seg_indices = reinterpret_cast<const int*>(w + c.lay.seg_indices);
  m.kv_last_page_len = reinterpret_cast<const int*>(w + c.lay.kv_last_page_len);
  m.qo_indptr = reinterpret_cast<const int*>(w + c.lay.qo_indptr);
  m.kv_len = reinterpret_cast<const int*>(w + c.lay.kv_len);
  m.n_splits = reinterpret_cast<const int*>(w + c.lay.n_splits);
  m.ext_splits = reinterpret_cast<const int*>(w + c.lay.ext_splits);
  m.partial_indptr = reinterpret_cast<const int*>(w + c.lay.partial_indptr);
  m.token_req = reinterpret_cast<const int*>(w + c.lay.token_req);
  m.decode_items = reinterpret_cast<const DecodeItem*>(w + c.lay.decode_items);
  m.extend_tiles = reinterpret_cast<const ExtendTile*>(w + c.lay.extend_tiles);
  m.partial_o = reinterpret_cast<uint16_t*>(w + c.lay.partial_o);
  m.partial_lse = reinterpret_cast<float*>(w + c.lay.partial_lse);
  return m;
}

int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz,
                   CUtensorMapL2promotion promo) {
  if (get_encoder() != PKV_OK) return PKV_ERR_CUDA;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

int encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                   CUtensorMapSwizzle swz) {
  if (get_encoder() != PKV_OK) return PKV_ERR_CUDA;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// Accessors for the allocation-free decode entry point (its own translation unit).
int static_config_ok(const pkv_config* cfg) { return check_config(cfg); }

size_t static_layout_bytes(const pkv_config& cfg, int num_sms, Layout* lay) {
  *lay = make_layout(cfg, num_sms);
  return lay->total;
}

void static_grid_sizes(const pkv_config& cfg, int num_sms, int* decode_ctas, int* extend_ctas) {
  grid_sizes(cfg, num_sms, decode_ctas, extend_ctas);
}

}  // namespace pkv

using namespace pkv;

struct pkv_ctx : public Ctx {};

extern "C" {

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK:
      return "ok";
    case PKV_ERR_INVALID_ARG:
      return "invalid argument";
    case PKV_ERR_UNSUPPORTED:
      return "unsupported shape or feature";
    case PKV_ERR_CAPACITY:
      return "capacity exceeded";
    case PKV_ERR_CUDA:
      return "CUDA error";
    case PKV_ERR_DEVICE:
      return "device recorded a data error";
    default:
      return "unknown status";
  }
}

int pkv_workspace_bytes(const pkv_config* cfg, size_t* bytes_out) {
  int st = check_config(cfg);
  if (st != PKV_OK) return st;
  if (!bytes_out) return PKV_ERR_INVALID_ARG;
  int dev, sms;
  if (device_sms(&dev, &sms) != PKV_OK) return PKV_ERR_CUDA;
  *bytes_out = make_layout(*cfg, sms).total;
  return PKV_OK;
}

int pkv_pool_bytes(const pkv_config* cfg, size_t* bytes_out) {
  if (!cfg || !bytes_out || cfg->num_pages < 0 || cfg->page_size <= 0 || cfg->num_kv_heads <= 0 ||
      cfg->head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (cfg->kv_dtype != PKV_KV_BF16 && cfg->kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
  const size_t elem = cfg->kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2;
  *bytes_out = (size_t)cfg->num_pages * cfg->page_size * cfg->num_kv_heads * cfg->head_dim * elem;
  return PKV_OK;
}

int pkv_create(const pkv_config* cfg, void* d_workspace, size_t workspace_bytes, pkv_ctx** ctx_out) {
  int st = check_config(cfg);
  if (st != PKV_OK) return st;
  if (!d_workspace || !ctx_out) return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_workspace) & 255) return PKV_ERR_INVALID_ARG;
  int dev, sms;
  if (device_sms(&dev, &sms) != PKV_OK) return PKV_ERR_CUDA;
  Layout lay = make_layout(*cfg, sms);
  if (workspace_bytes < lay.total) return PKV_ERR_CAPACITY;
  if (get_encoder() != PKV_OK) return PKV_ERR_CUDA;
  pkv_ctx* c = new (std::nothrow) pkv_ctx();
  if (!c) return PKV_ERR_CAPACITY;
  c->cfg = *cfg;
  c->lay = lay;
  c->ws = static_cast<char*>(d_workspace);
  c->num_sms = sms;
  grid_sizes(*cfg, sms, &c->decode_ctas, &c->extend_ctas);
  c->batch = 0;
  c->mode = PKV_MODE_IDLE;
  c->qo_given = false;
  c->device = dev;
  // a clean plan: no batch built yet
  if (cudaMemset(c->ws + lay.plan, 0, sizeof(int) * kPlanWords) != cudaSuccess) {
    delete c;
    return PKV_ERR_CUDA;
  }
  *ctx_out = c;
  return PKV_OK;
}

int pkv_destroy(pkv_ctx* ctx) {
  delete ctx;
  return PKV_OK;
}

int pkv_select_backend(int forward_mode, int spec_mode) {
  if (spec_mode != PKV_SPEC_PREFILL && spec_mode != PKV_SPEC_DECODE) return PKV_PATH_INVALID;
  switch (forward_mode) {
    case PKV_MODE_DECODE:
    case PKV_MODE_IDLE:
      return PKV_PATH_DECODE;
    case PKV_MODE_TARGET_VERIFY:
    case PKV_MODE_DRAFT_EXTEND:
      return spec_mode == PKV_SPEC_DECODE ? PKV_PATH_DECODE : PKV_PATH_EXTEND;
    case PKV_MODE_EXTEND:
      return PKV_PATH_EXTEND;
    default:
      return PKV_PATH_INVALID;
  }
}

int pkv_build_metadata(pkv_ctx* ctx, int forward_mode, int32_t batch, const int32_t* d_seq_lens,
                       const int32_t* d_qo_lens, const int32_t* d_page_table, int32_t page_table_stride,
                       void* stream) {
  if (!ctx) return PKV_ERR_INVALID_ARG;
  if (pkv_select_backend(forward_mode, PKV_SPEC_PREFILL) == PKV_PATH_INVALID) return PKV_ERR_INVALID_ARG;
  if (batch < 0) return PKV_ERR_INVALID_ARG;
  if (batch > ctx->cfg.max_batch) return PKV_ERR_CAPACITY;
  if (forward_mode == PKV_MODE_IDLE) batch = 0;
  if (batch > 0 && (!d_seq_lens || !d_page_table || page_table_stride <= 0)) return PKV_ERR_INVALID_ARG;
  if (forward_mode == PKV_MODE_DECODE && d_qo_lens) return PKV_ERR_INVALID_ARG;
  int st = launch_build_metadata(*ctx, batch, d_seq_lens, d_qo_lens, d_page_table, page_table_stride,
                                 static_cast<cudaStream_t>(stream));
  if (st != PKV_OK) return st;
  ctx->batch = batch;
  ctx->mode = forward_mode;
  ctx->qo_given = d_qo_lens != nullptr;
  return PKV_OK;
}

int pkv_get_metadata(pkv_ctx* ctx, const int32_t** kv_indptr, const int32_t** kv_indices,
                     const int32_t** kv_last_page_len, const int32_t** qo_indptr) {
  if (!ctx) return PKV_ERR_INVALID_ARG;
  Meta m = make_meta(*ctx);
  if (kv_indptr) *kv_indptr = m.kv_indptr;
  if (kv_indices) *kv_indices = m.kv_indices;
  if (kv_last_page_len) *kv_last_page_len = m.kv_last_page_len;
  if (qo_indptr) *qo_indptr = m.qo_indptr;
  return PKV_OK;
}

int pkv_set_kv_buffer(pkv_ctx* ctx, void* d_k_pool, void* d_v_pool, const int32_t* d_loc, const void* d_k,
                      const void* d_v, int32_t n_tokens, float k_inv_scale, float v_inv_scale, void* stream) {
  if (!ctx || n_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!d_k_pool || !d_v_pool || !d_loc || !d_k || !d_v) return PKV_ERR_INVALID_ARG;
  if (!aligned16(d_k_pool) || !aligned16(d_v_pool) || !aligned16(d_k) || !aligned16(d_v)) return PKV_ERR_INVALID_ARG;
  return launch_set_kv_buffer(*ctx, d_k_pool, d_v_pool, d_loc, d_k, d_v, n_tokens, k_inv_scale, v_inv_scale,
                              static_cast<cudaStream_t>(stream));
}

int pkv_forward_decode(pkv_ctx* ctx, const void* d_q, const void* d_k_pool, const void* d_v_pool, float sm_scale,
                       float k_scale, float v_scale, void* d_out, float* d_lse, void* stream) {
  int st = check_forward_args(ctx, d_q, d_k_pool, d_v_pool, d_out, d_lse);
  if (st != PKV_OK) return st;
  st = check_scales(*ctx, sm_scale, k_scale, v_scale);
  if (st != PKV_OK) return st;
  if (ctx->batch == 0) return PKV_OK;
  return launch_decode(*ctx, d_q, d_k_pool, d_v_pool, sm_scale, k_scale, v_scale, d_out, d_lse,
                       static_cast<cudaStream_t>(stream));
}

int pkv_forward_extend(pkv_ctx* ctx, const void* d_q, const void* d_k_pool, const void* d_v_pool, float sm_scale,
                       float k_scale, float v_scale, void* d_out, float* d_lse, void* stream) {
  int st = check_forward_args(ctx, d_q, d_k_pool, d_v_pool, d_out, d_lse);
  if (st != PKV_OK) return st;
  st = check_scales(*ctx, sm_scale, k_scale, v_scale);
  if (st != PKV_OK) return st;
  if (ctx->batch == 0) return PKV_OK;
  return launch_extend(*ctx, d_q, d_k_pool, d_v_pool, sm_scale, k_scale, v_scale, d_out, d_lse,
                       static_cast<cudaStream_t>(stream));
}

int pkv_forward(pkv_ctx* ctx, int forward_mode, int spec_mode, const void* d_q, const void* d_k_pool,
                const void* d_v_pool, float sm_scale, float k_scale, float v_scale, void* d_out, float* d_lse,
                void* stream) {
  if (!ctx) return PKV_ERR_INVALID_ARG;
  const int path = pkv_select_backend(forward_mode, spec_mode);
  if (path == PKV_PATH_INVALID) return PKV_ERR_INVALID_ARG;
  if (forward_mode == PKV_MODE_IDLE) return PKV_OK;
  if (forward_mode == PKV_MODE_DECODE && ctx->qo_given) return PKV_ERR_INVALID_ARG;
  if (path == PKV_PATH_DECODE)
    return pkv_forward_decode(ctx, d_q, d_k_pool, d_v_pool, sm_scale, k_scale, v_scale, d_out, d_lse, stream);
  return pkv_forward_extend(ctx, d_q, d_k_pool, d_v_pool, sm_scale, k_scale, v_scale, d_out, d_lse, stream);
}

int pkv_set_tree_mask(pkv_ctx* ctx, const uint64_t* d_tree_mask) {
  if (!ctx) return PKV_ERR_INVALID_ARG;
  if (d_tree_mask && (reinterpret_cast<uintptr_t>(d_tree_mask) & 7u) != 0) return PKV_ERR_INVALID_ARG;
  ctx->tree = d_tree_mask;
  return PKV_OK;
}

int pkv_set_attention_sinks(pkv_ctx* ctx, const float* d_sinks) {
  if (!ctx) return PKV_ERR_INVALID_ARG;
  if (d_sinks && (reinterpret_cast<uintptr_t>(d_sinks) & 3u) != 0) return PKV_ERR_INVALID_ARG;
  ctx->sinks = d_sinks;
  return PKV_OK;
}

// One int32 plan word of the context, written from the host; synchronises the stream.
static int write_plan_word(pkv_ctx* ctx, int word, int32_t value, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(ctx->ws + ctx->lay.plan + sizeof(int32_t) * word, &value, sizeof(value),
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return PKV_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_set_wait_limit(pkv_ctx* ctx, uint32_t limit_ns, void* stream) {
  if (!ctx) return PKV_ERR_INVALID_ARG;
  return write_plan_word(ctx, kWaitLimitNs, (int32_t)limit_ns, stream);
}

int pkv_test_hold_first_load(pkv_ctx* ctx, int enable, void* stream) {
  if (!ctx) return PKV_ERR_INVALID_ARG;
  return write_plan_word(ctx, kHoldLoad, enable ? 1 : 0, stream);
}

int pkv_get_device_error(pkv_ctx* ctx, int32_t* code, void* stream) {
  if (!ctx || !code) return PKV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t words[2] = {0, 0};
  if (cudaMemcpyAsync(words, ctx->ws + ctx->lay.plan, sizeof(words), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_ERR_CUDA;
  *code = words[0];
  if (words[0] != 0) {
    if (cudaMemsetAsync(ctx->ws + ctx->lay.plan, 0, sizeof(words), st) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_ERR_DEVICE;
  }
  return PKV_OK;
}

int pkv_describe(pkv_ctx* ctx, char* buf, size_t n) {
  if (!ctx || !buf || n == 0) return PKV_ERR_INVALID_ARG;
  const pkv_config& c = ctx->cfg;
  const int group = c.num_q_heads / c.num_kv_heads;
  const int rows = c.max_qo_len * group;
  char dec[160];
  if (decode_row_warps(c) > 1)
    snprintf(dec, sizeof dec, "split-KV on tcgen05 %dx%d tiles (verify shapes, up to %d rows/unit), grid %d",
             kExtendRows, kExtendKeys, rows, ctx->extend_ctas);
  else
    snprintf(dec, sizeof dec, "split-KV TMA+mma.sync key-major, up to %d rows/unit, %d pages/stage, grid %d",
             rows <= 8 ? 8 : 16, decode_stage_pages(c), ctx->decode_ctas);
  snprintf(buf, n,
           "pkv sm_103a: heads %d/%d (group %d) head_dim %d/%d page_size %d kv %s pool_pages %d | decode: %s | "
           "extend: tcgen05 %dx%d tiles, grid %d | SMs %d",
           c.num_q_heads, c.num_kv_heads, group, c.head_dim, head_dim_v(c), c.page_size,
           c.kv_dtype == PKV_KV_FP8_E4M3 ? "fp8_e4m3" : "bf16", c.num_pages, dec, kExtendRows, kExtendKeys,
           ctx->extend_ctas, ctx->num_sms);
  return PKV_OK;
}

}  // extern "C"
