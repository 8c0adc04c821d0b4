// Internal declarations shared by the library's translation units: workspace
// layout, launch parameter blocks, and small inline-PTX helpers for sm_103a
// (mbarrier with bounded waits, TMA tensor loads, ldmatrix, warp-level MMA).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pkv.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Fixed tiling constants
// ---------------------------------------------------------------------------
// The kernels gather the KV cache in segments of 16 consecutive slots of one
// page (one 16-row TMA box per segment and 128-byte column block): a page of
// 16 tokens is one segment, a page of 128 tokens eight. The metadata build
// lists every request's segments (seg_indptr / seg_indices, the slot of
// segment s being seg_indices[s] * 16); with 16-token pages the segment lists
// are the page lists themselves.
constexpr int kSegSlots = 16;
// page sizes the library accepts (tokens per page)
constexpr int kPageSizeSmall = 16;
constexpr int kPageSizeLarge = 128;
// split-KV aims at this many work units per CTA slot: 16-row decode units
// are light and balance best when fine; the verify shapes' units carry up to
// 128 rows each and pay more per unit
constexpr int kDecodeTargetWaves = 8;
constexpr int kVerifyTargetWaves = 4;
// decode splits of one request at most: the merge reads two per lane (so at
// most 64); a lone long request then still spreads over the whole grid
constexpr int kMaxSplitsPerRequest = 64;
constexpr int kDecodeMinChunkPages = 8; // never cut a (request, head) range finer than 128 keys
constexpr int kExtendRows = 128;        // query rows (token x head-in-group) per extend tile
constexpr int kExtendUnitRows = 256;    // an extend work unit holds two tiles (A, B) sharing K/V
constexpr int kExtendKeys = 128;        // keys per extend KV tile
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s bound on any mbarrier wait

// A bounded wait ran out (the public PKV_DEV_TIMEOUT)
constexpr int kDevTimeout = PKV_DEV_TIMEOUT;

// ---------------------------------------------------------------------------
// Plan header (int32 words at the start of the workspace)
// ---------------------------------------------------------------------------
enum PlanWord : int {
  kErr = 0,            // first device error (PKV_DEV_*), 0 when clean
  kErrIndex = 1,       // index that raised it
  kBatch = 2,          // batch size of the last build
  kTotalSegs = 3,      // seg_indptr[bs]: 16-slot segments of the batch
  kTotalQ = 4,         // qo_indptr[bs]
  kDecodeItems = 5,    // number of (request, split) items on the decode path
  kChunkPages = 6,     // pages per split on the decode path
  kExtendTiles = 7,    // number of (request, q-tile) items on the extend path
  kPartialRows = 8,    // rows of the partial-output buffer in use
  kMaxQo = 9,          // max qo_len in the batch
  kSplitDecode = 10,   // requests with more than one split on the decode path
  kSplitExtend = 11,   // requests split along their KV range on the extend path
  kDecodeNext = 12,    // decode units claimed past the first wave (zeroed after every decode)
  kWaitLimitNs = 14,   // bound on every mbarrier wait in ns (0: kWaitTimeoutNs), pkv_set_wait_limit
  kHoldLoad = 15,      // test support: CTA 0 never issues its first K/V load (pkv_test_hold_first_load)
  kPlanWords = 32
};

// Work item of the decode path: request, split index, segment range [p0, p1)
// of the request's 16-slot segments.
struct DecodeItem {
  int b, split, p0, p1;
};
// Work item of the extend path: request, first query row (token * group +
// head-in-group) of a 256-row unit, the number of 128-key KV tiles its first
// and second 128-row tile reach (0 when the tile has no rows), and the KV tile
// range [kv0, kv1) it covers. A request whose rows fit one unit is split along
// its KV range like the decode path (split >= 0: the unit writes fp32
// partials merged afterwards); otherwise split = -1 and the range is whole.
// dual = 1: the rows fit one 128-row tile; both tiles hold them, tile A takes
// the first half of the unit's KV tiles and tile B the rest, and the two
// halves are merged by LSE inside the CTA before anything is written.
struct ExtendTile {
  int b, row0, kv_a, kv_b, split, kv0, kv1, dual;
};

// Byte offsets of every buffer inside the caller's workspace.
struct Layout {
  size_t plan, kv_indptr, kv_indices, kv_last_page_len, qo_indptr, kv_len, n_splits, ext_splits, partial_indptr,
      token_req, decode_items, extend_tiles, partial_o, partial_lse, total;
  // segment lists of pages larger than one segment (seg_per_page > 1);
  // with one segment per page they alias kv_indptr / kv_indices
  size_t seg_indptr, seg_indices;
  int seg_per_page;
  int max_decode_items, max_extend_tiles, partial_rows_cap;
};

struct Ctx {
  pkv_config cfg;
  Layout lay;
  char* ws;  // device workspace base
  int num_sms;
  int decode_ctas;  // persistent grid of the decode kernel
  int extend_ctas;
  int batch;  // batch size of the last pkv_build_metadata
  int mode;
  bool qo_given;  // last build had explicit qo_lens
  int device;
  const uint64_t* tree = nullptr;  // draft-tree mask words (pkv_set_tree_mask), or null
  const float* sinks = nullptr;    // per-query-head sink logits (pkv_set_attention_sinks), or null
};

// Width of the V heads and of the output rows (head_dim_v, 0 meaning head_dim).
inline int head_dim_v(const pkv_config& c) { return c.head_dim_v > 0 ? c.head_dim_v : c.head_dim; }

// The tree mask the next forward applies: only after a build in a verify mode.
inline const uint64_t* active_tree(const Ctx& c) {
  return (c.mode == PKV_MODE_TARGET_VERIFY || c.mode == PKV_MODE_DRAFT_EXTEND) ? c.tree : nullptr;
}

// Device-side view of the metadata in the workspace.
struct Meta {
  int* plan;
  const int* kv_indptr;    // pages (the public metadata)
  const int* kv_indices;
  const int* seg_indptr;   // 16-slot segments: what the kernels gather
  const int* seg_indices;  // segment s of the batch covers slots seg_indices[s] * 16 .. + 15
  const int* kv_last_page_len;
  const int* qo_indptr;
  const int* kv_len;
  const int* n_splits;    // decode-path splits per request
  const int* ext_splits;  // extend-path KV splits per request (1 when not split); never above n_splits
  const int* partial_indptr;
  const int* token_req;
  const DecodeItem* decode_items;
  const ExtendTile* extend_tiles;
  uint16_t* partial_o;  // bf16 [rows][Hq][Dv]: normalised partial outputs of split units
  float* partial_lse;
};

Meta make_meta(const Ctx& c);

// Entry points of the kernels' host launchers (one per translation unit).
int launch_build_metadata(Ctx& c, int batch, const int32_t* seq_lens, const int32_t* qo_lens,
                          const int32_t* page_table, int stride, cudaStream_t st);
int launch_set_kv_buffer(Ctx& c, void* k_pool, void* v_pool, const int32_t* loc, const void* k, const void* v,
                         int n, float k_inv, float v_inv, cudaStream_t st);
int launch_decode(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
                  float v_scale, void* out, float* lse, cudaStream_t st);
int launch_extend(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
                  float v_scale, void* out, float* lse, cudaStream_t st);
// The decode path's verify shapes (more than 16 query rows per KV head): the
// tcgen05 tile kernel of the extend path, run over the decode plan's split-KV
// items and merged by the decode path's merge.
int launch_decode_tc(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
                     float v_scale, void* out, float* lse, cudaStream_t st);
// LSE merge of split partials for requests whose rows per KV head are at most
// max_rows_per_head (the decode path: its largest tile; the extend path: 256,
// the requests it split).
int launch_split_merge(Ctx& c, void* out, float* lse, int max_rows_per_head, bool extend_path, cudaStream_t st);
// decode-path tile shape of a configuration: warps of 16 rows per unit (0 if
// max_qo_len * group exceeds 128) and K/V pages per pipeline stage
int decode_row_warps(const pkv_config& cfg);
int decode_stage_pages(const pkv_config& cfg);

// Tensor-map encoding through the driver entry point (no link-time libcuda dependency).
// promo: the L2 fill granularity of a copy. Pool rows of one head are 256
// bytes wide for bf16 (128 elements) and 128 for E4M3, the neighbouring head
// following; a fill wider than the row brings in the next head's bytes too.
int encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz,
                   CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
int encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                   CUtensorMapSwizzle swz);

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes, so it must execute pdl_wait()
// before touching any global memory that earlier work writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
// Wait until the preceding grid in the stream has finished and its memory
// operations are visible (no-op when launched without programmatic serialization).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel in the stream start launching its CTAs.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void record_error(int* plan, int code, int index) {
  if (atomicCAS(&plan[kErr], 0, code) == 0) plan[kErrIndex] = index;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The wait bound of the context (read once a wait has not succeeded at once).
__device__ __forceinline__ unsigned long long wait_limit_ns(const int* plan) {
  const unsigned v = (unsigned)__ldcg(plan + kWaitLimitNs);
  return v ? (unsigned long long)v : kWaitTimeoutNs;
}

// Wait for the phase with the given parity to complete. Bounded: gives up
// after the context's wait limit, records kDevTimeout and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* plan) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns(), limit = wait_limit_ns(plan);
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit) {
      record_error(plan, kDevTimeout, 0);
      return false;
    }
  }
}

// Same wait, but it also gives up as soon as the CTA's abort flag is set
// (another role timed out), so one failure stops every waiter quickly.
__device__ __forceinline__ bool mbar_wait_ab(uint64_t* bar, uint32_t parity, int* plan, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns(), limit = wait_limit_ns(plan);
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit) {
      record_error(plan, kDevTimeout, 0);
      return false;
    }
  }
}

// The same wait for a whole warp: every lane waits, and the warp gets one
// answer (false if any lane gave up).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* plan, volatile int* abort_flag) {
  const bool ok = mbar_wait_ab(bar, parity, plan, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA: 2-D tiled load into shared memory, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit elements held the way ldmatrix
// leaves it (lane l: row l/4, columns 2(l%4) and 2(l%4)+1, low half first):
// returns the same layout of the transposed matrix.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Two E4M3 codes (low byte first) -> two f16 in one register (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Attention sink: the head's sink logit joins the softmax as a key with a zero
// value vector. Given a finished row's natural-log LSE over its keys, returns
// the factor that scales its output and moves lse to include the sink (a row
// with no keys gets factor 0 and lse = sink).
__device__ __forceinline__ float sink_factor(float& lse, float sink) {
  const float mx = fmaxf(lse, sink);
  if (mx == -INFINITY) return 1.f;  // no key and a -inf sink
  const float a = expf(lse - mx), c = expf(sink - mx);
  lse = mx + logf(a + c);
  return a / (a + c);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so
// every one of them takes the same branch afterwards.
__device__ __forceinline__ int named_bar_or(int id, int threads, int pred) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred), "r"(id), "r"(threads)
      : "memory");
  return r;
}

}  // namespace pkv

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) helpers, cta_group::1
// ---------------------------------------------------------------------------
namespace pkv {

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)
         | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// The same with A and B in f16 (kind::f16, A/B format 0).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                       // D format: f32
         | ((a_mn_major ? 1u : 0u) << 15)
         | ((b_mn_major ? 1u : 0u) << 16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M rows x 16 K) sits in TMEM, row m in
// lane m, two bf16 per 32-bit column, lower K index in the low half.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05 operation issued so far by
// this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Warp-wide forms: every lane of a converged warp computes the operands (so
// they stay warp-uniform) and one elected lane issues the instruction. A
// tcgen05.mma issued this way costs the warp fewer cycles than one issued from
// a single-lane branch.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n" : "=r"(e));
  return e != 0;
}

__device__ __forceinline__ void umma_bf16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               bool accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.u32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                  bool accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n elect.sync _|e, 0xffffffff;\n setp.ne.u32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar))
      : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace pkv
