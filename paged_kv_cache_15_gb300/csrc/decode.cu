// forward_decode over the paged KV cache ("--attention-backend", section "What an
// attention backend is": forward_decode runs one query token per request against
// its cached keys; section "Two backends in one server": decode reads one query
// against a long cache, so it is bound by memory traffic).
//
// Split-KV flash decoding:
//   * The metadata build cut every (request, KV head) key range into chunks of
//     chunk_pages pages; one work unit = (request, split, KV head). CTA j of the
//     persistent grid starts on unit j and claims further units from a
//     batch-wide counter as it frees up.
//   * GQA packing: the group's query heads (times the request's query tokens on
//     the verify path) are the query rows of one MMA tile, so every K/V byte
//     fetched from HBM is used by all heads of its group.
//   * A producer warp gathers pages with TMA (one 2-D box of 16 token rows x 128
//     bytes per page, 128-byte swizzle) into a ring of shared-memory stages; the
//     consumer warps wait on the stage's mbarrier, compute scores and outputs
//     with m16n8k16 tensor-core MMAs, and keep an online softmax per row
//     (running max m, running sum l) in registers, in the log2 domain.
//   * Decode shapes (at most 16 query rows per unit) use key-major tiles:
//     S^T = K Q^T with 16 keys along the MMA's M and the rows along N in one or
//     two 8-row tiles, then O^T += V^T P^T, P^T reaching the B operand through
//     an in-register 8x8 transpose (movmatrix). Four key warps split each
//     stage's keys and combine through shared memory.
//   * Verify shapes (target verify on the decode path: more than 16 and up to
//     128 query rows per KV head) are a dense contraction of a full 128-row
//     tile against every key, so they run on the 5th-generation tensor cores:
//     the tcgen05 tile kernel of extend.cu walks this path's plan (the same
//     split items, the same merge below).
//   * Each unit ends with its normalised output and LSE. A request with one split
//     writes the final bf16 output directly; otherwise the unit writes a bf16
//     partial row and an fp32 LSE, and the merge kernel (one warp per
//     (token, query head) row) combines them:
//        lse = ln sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s.
//   * FP8 E4M3 pools: codes are widened to f16 in registers (cvt e4m3x2 -> f16x2,
//     exact), the MMAs run in f16 (Q and P rounded to f16), and the per-pool
//     scales are folded into the score scale and the output.
// Keys past the request's length inside its last page are zeroed in shared
// memory before use, and every other key outside the visible range is masked
// to -inf, so unused pool slots never reach the result.
#include <math.h>

#include <algorithm>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// DK: width of the Q and K heads; DV: of the V heads and output rows (equal
// except for models whose K and V heads differ, 192 / 128).
template <int DK_, int DV_, bool FP8_, int WK_, int KPW_, int STAGES_, int RT_>
struct DecodeCfg {
  static constexpr int DK = DK_;
  static constexpr int DV = DV_;
  static constexpr bool FP8 = FP8_;
  // key-major tile: keys along the MMA's M, RT tiles of 8 query rows along N
  static constexpr int RT = RT_;
  static constexpr int WR = 1;    // one row position (the rows are the MMA's N)
  static constexpr int WK = WK_;  // key warps (split each stage's keys)
  static constexpr int KPW = KPW_;  // keys per key-warp per stage (multiple of 16)
  static constexpr int STAGES = STAGES_;
  static constexpr int kConsumerWarps = WR * WK;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kMinBlocks = kThreads <= 160 ? 2 : 1;  // two CTAs per SM hide latency for the decode shapes
  static constexpr int kRows = 8 * RT;
  static constexpr int kStageKeys = WK * KPW;
  static constexpr int kStagePages = kStageKeys / kSegSlots;
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kRowBytesK = DK * kElem;
  static constexpr int kRowBytesV = DV * kElem;
  static constexpr int kColBlocksK = kRowBytesK / 128;
  static constexpr int kColBlocksV = kRowBytesV / 128;
  static constexpr int kTileBytesK = kStageKeys * kRowBytesK;  // a stage: K tile, then V tile
  static constexpr int kTileBytesV = kStageKeys * kRowBytesV;
  static constexpr int kStageBytes = kTileBytesK + kTileBytesV;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kMlOffset = kBarOffset + 2 * STAGES * 8;
  static constexpr int kAbortOffset = kMlOffset + WK * 16 * 2 * 4;
  static constexpr int kUnitQOffset = kAbortOffset + 16;  // unit queue: 2 full + 2 empty barriers, 2 ids
  static constexpr int kSmemBytes = kUnitQOffset + 40 + 1024;  // + alignment slack
  static_assert(kRowBytesK % 128 == 0 && kRowBytesV % 128 == 0, "rows must be whole 128-byte swizzle spans");
  static_assert(KPW % 16 == 0 && kStageKeys % kSegSlots == 0, "stage must hold whole pages");
  static_assert(!(WK > 1) || (WK * 16 * DV * 4 <= kStageBytes), "merge scratch must fit in one stage");
  static_assert(WK > 1 && RT >= 1 && RT <= 2, "key-major tiles: one or two 8-row tiles, key warps combined");
};

struct DecodeArgs {
  Meta m;
  const uint16_t* q;  // bf16 [T][Hq][DK]
  uint16_t* out;      // bf16 [T][Hq][DV]
  float* lse;         // fp32 [T][Hq] or null
  int num_q_heads, num_kv_heads, group;
  float scale_log2;  // sm_scale * k_scale * log2(e)
  float v_scale;     // multiplies the output (E4M3 pools), 1 for bf16
  const uint64_t* tree;  // draft-tree mask word per query token, or null (chain drafts)
  const float* sinks;    // sink logit per query head, or null
};

// Byte offset of (row, 16-byte chunk) inside a swizzled [rows][128 B] column block.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Combine the nsplit partial rows of one (token, query head) row:
//   lse = ln sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s.
// One warp per row, lanes across head_dim. Lane s reads the LSEs of splits s
// and s + 32 in the same round trip as the first kMergeBatch partial rows
// (their addresses do not depend on the weights); the weights then come from a
// warp max and sum.
// Partials were written by other CTAs, so they are read through L2
// (ld.global.cg), never from a stale L1 line.
constexpr int kMergeBatch = 8;

template <int D>
struct MergeVec;
// partial rows are bf16: 4 (D = 128) or 2 (D = 64) elements per lane
template <>
struct MergeVec<128> {
  using T = uint2;
  __device__ static T load(const uint16_t* p) { return __ldcg(reinterpret_cast<const uint2*>(p)); }
  __device__ static void fma(float* acc, float w, const T& x) {
    acc[0] += w * bf16lo(x.x);
    acc[1] += w * bf16hi(x.x);
    acc[2] += w * bf16lo(x.y);
    acc[3] += w * bf16hi(x.y);
  }
};
template <>
struct MergeVec<64> {
  using T = uint32_t;
  __device__ static T load(const uint16_t* p) { return __ldcg(reinterpret_cast<const unsigned int*>(p)); }
  __device__ static void fma(float* acc, float w, const T& x) {
    acc[0] += w * bf16lo(x);
    acc[1] += w * bf16hi(x);
  }
};

template <int D>
__device__ __forceinline__ void merge_row(const DecodeArgs& a, long long pbase, int qo, int i, int h, int nsplit,
                                          long long orow, int lane) {
  constexpr int PER = D / 32;
  using V = MergeVec<D>;
  auto prow = [&](int sp) { return (pbase + (long long)sp * qo + i) * a.num_q_heads + h; };
  auto lse_of = [&](int sp) { return __ldcg(a.m.partial_lse + prow(sp)); };
  auto part = [&](int sp) { return V::load(a.m.partial_o + prow(sp) * D + lane * PER); };
  typename V::T x[kMergeBatch];
#pragma unroll
  for (int sp = 0; sp < kMergeBatch; ++sp)
    if (sp < nsplit) x[sp] = part(sp);
  static_assert(kMaxSplitsPerRequest <= 64, "two splits per lane");
  const float l0 = lane < nsplit ? lse_of(lane) : -INFINITY;
  const float l1 = lane + 32 < nsplit ? lse_of(lane + 32) : -INFINITY;
  float M = fmaxf(l0, l1);
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float w0 = M != -INFINITY && lane < nsplit ? fast_exp2((l0 - M) * kLog2e) : 0.f;
  float w1 = M != -INFINITY && lane + 32 < nsplit ? fast_exp2((l1 - M) * kLog2e) : 0.f;
  float Z = w0 + w1;
  for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
  const float invZ = Z > 0.f ? 1.f / Z : 0.f;
  w0 *= invZ;
  w1 *= invZ;
  // split sp's weight: lane sp % 32 holds it, in w0 below 32 and w1 above
  auto weight = [&](int sp) { return __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31); };
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
#pragma unroll
  for (int sp = 0; sp < kMergeBatch; ++sp)
    if (sp < nsplit) V::fma(acc, weight(sp), x[sp]);
  for (int s0 = kMergeBatch; s0 < nsplit; s0 += kMergeBatch) {
#pragma unroll
    for (int sp = 0; sp < kMergeBatch; ++sp)
      if (s0 + sp < nsplit) x[sp] = part(s0 + sp);
#pragma unroll
    for (int sp = 0; sp < kMergeBatch; ++sp) {
      if (s0 + sp >= nsplit) break;
      V::fma(acc, weight(s0 + sp), x[sp]);
    }
  }
  float lse = Z > 0.f ? M + __logf(Z) : -INFINITY;
  if (a.sinks) {
    const float f = sink_factor(lse, a.sinks[h]);
#pragma unroll
    for (int j = 0; j < PER; ++j) acc[j] *= f;
  }
  uint16_t* dst = a.out + orow * D + lane * PER;
  if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1]);
  }
  if (a.lse && lane == 0) a.lse[orow] = lse;
}

// EXTRAS: draft-tree mask words or attention sinks are in use (a separate
// instantiation, so plain batches run without that code).
template <class C, bool EXTRAS>
__global__ void __launch_bounds__(C::kThreads, C::kMinBlocks) decode_splitkv_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                     const __grid_constant__ CUtensorMap tmap_v,
                                                                     DecodeArgs a) {
  constexpr int DK = C::DK, DV = C::DV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty = full + C::STAGES;
  float* s_ml = reinterpret_cast<float*>(smem + C::kMlOffset);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kAbortOffset);
  // queue of the units this CTA runs, filled by the producer: ids in s_uq,
  // uq_full[q] (producer arrives), uq_empty[q] (one arrival per consumer warp)
  uint64_t* uq_full = reinterpret_cast<uint64_t*>(smem + C::kUnitQOffset);
  uint64_t* uq_empty = uq_full + 2;
  volatile int* s_uq = reinterpret_cast<volatile int*>(uq_empty + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t* const tree_words = EXTRAS ? a.tree : nullptr;
  const float* const sinks = EXTRAS ? a.sinks : nullptr;
  int* plan = a.m.plan;
  pdl_launch_dependents();

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&uq_full[q], 1);
      mbar_init(&uq_empty[q], C::kConsumerWarps);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  // Stage buffers start as zeros: rows of a partly filled stage are then always
  // finite (zeros or earlier valid keys) and their zero weights stay zero.
  for (int i = tid; i < C::STAGES * C::kStageBytes / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();
  // launched with programmatic serialization: the metadata (and the K/V this
  // step stored) are only read after the preceding grid has finished
  pdl_wait();

  const int n_units = plan[kDecodeItems] * a.num_kv_heads;

  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer (one lane)
    if (lane == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
      const uint64_t pol = policy_evict_first();
      int slot = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_phase = 0;
      // Units: blockIdx.x first, then whatever the batch-wide counter hands
      // out as CTAs free up (units differ in length: the last split of a
      // request is short). The next claim is made when a unit starts, and
      // each id is published to the consumer warps through the queue.
      int w = (int)blockIdx.x < n_units ? (int)blockIdx.x : -1;
      bool stop = false;
      // test support: CTA 0 arms its first stage but never loads it
      const bool hold_first = blockIdx.x == 0 && __ldcg(plan + kHoldLoad) != 0;
      for (int iu = 0; !stop; ++iu) {
        const int q = iu & 1;
        if (!mbar_wait_ab(&uq_empty[q], ((iu >> 1) & 1) ^ 1, plan, s_abort)) {
          *s_abort = 1;
          break;
        }
        s_uq[q] = w;
        mbar_arrive(&uq_full[q]);
        if (w < 0) break;
        // (no claim when the first wave already covers every unit)
        const int claimed = n_units > (int)gridDim.x ? (int)gridDim.x + atomicAdd(&plan[kDecodeNext], 1) : n_units;
        const DecodeItem it = a.m.decode_items[w / a.num_kv_heads];
        const int g = w % a.num_kv_heads;
        const int base = a.m.seg_indptr[it.b] + it.p0;
        const int npages = it.p1 - it.p0;
        const int nst = (npages + C::kStagePages - 1) / C::kStagePages;
        for (int st = 0; st < nst; ++st) {
          if (!mbar_wait_ab(&empty[slot], phase ^ 1, plan, s_abort)) {
            *s_abort = 1;
            stop = true;
            break;
          }
          const int np = min(C::kStagePages, npages - st * C::kStagePages);
          mbar_arrive_expect_tx(&full[slot], (uint32_t)(np * kSegSlots * (C::kRowBytesK + C::kRowBytesV)));
          uint8_t* kdst = smem + slot * C::kStageBytes;
          uint8_t* vdst = kdst + C::kTileBytesK;
          for (int p = 0; p < np && !(hold_first && iu == 0 && st == 0); ++p) {
            const int page = a.m.seg_indices[base + st * C::kStagePages + p];
#pragma unroll
            for (int cb = 0; cb < C::kColBlocksK; ++cb)
              tma_load_2d_hint(kdst + cb * C::kStageKeys * 128 + p * kSegSlots * 128, &tmap_k,
                               g * DK + cb * (128 / C::kElem), page * kSegSlots, &full[slot], pol);
#pragma unroll
            for (int cb = 0; cb < C::kColBlocksV; ++cb)
              tma_load_2d_hint(vdst + cb * C::kStageKeys * 128 + p * kSegSlots * 128, &tmap_v,
                               g * DV + cb * (128 / C::kElem), page * kSegSlots, &full[slot], pol);
          }
          armed |= 1u << slot;
          armed_phase = (armed_phase & ~(1u << slot)) | (phase << slot);
          if (++slot == C::STAGES) {
            slot = 0;
            phase ^= 1;
          }
        }
        w = claimed < n_units ? claimed : -1;
      }
      for (int s = 0; s < C::STAGES; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (armed_phase >> s) & 1, plan);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp;  // consumer warp
  const int wk = cw % C::WK;  // key warp
  const int G = a.group;
  int slot = 0;
  uint32_t phase = 0;
  bool aborted = false;

  for (int iu = 0;; ++iu) {
    // next unit from the producer's queue; all consumer warps read the same id
    // and leave together (the vote also ends the loop after an abort)
    const int q = iu & 1;
    int w = -1;
    if (!aborted && !mbar_wait_ab(&uq_full[q], (iu >> 1) & 1, plan, s_abort)) {
      *s_abort = 1;
      aborted = true;
    }
    if (!aborted) w = s_uq[q];
    __syncwarp();
    if (lane == 0) mbar_arrive(&uq_empty[q]);
    if (named_bar_or(1, C::kConsumerWarps * 32, *s_abort || w < 0)) break;
    const DecodeItem it = a.m.decode_items[w / a.num_kv_heads];
    const int g = w % a.num_kv_heads;
    const int b = it.b;
    const int L = a.m.kv_len[b];
    const int q0 = a.m.qo_indptr[b];
    const int qo = a.m.qo_indptr[b + 1] - q0;
    const int nsplit = a.m.n_splits[b];
    const int np_req = a.m.seg_indptr[b + 1] - a.m.seg_indptr[b];
    const int rows_valid = qo * G;
    const bool skip = rows_valid > C::kRows;  // tile too small: recorded, pipeline still drained
    if (skip && lane == 0 && wk == 0) record_error(plan, PKV_DEV_QO_TOO_LONG, b);
    const int key_begin = it.p0 * kSegSlots;
    const int key_end = min(it.p1 * kSegSlots, L);
    const int npages = it.p1 - it.p0;
    const int nst = (npages + C::kStagePages - 1) / C::kStagePages;

    {
      // ---------------------------------------------- key-major tile (decode)
      // S^T = K Q^T with the stage's keys along the MMA's M (16 per block) and
      // the unit's query rows along N (RT tiles of 8), then O^T += V^T P^T with
      // head-dim columns along M. With GQA groups of 8 or fewer rows no MMA
      // row is padding on the key side, so the MMAs and exponentials per key
      // are half those of a 16-row query tile. Lane (g8 = lane/4, t4 = lane%4)
      // holds rows 8j + 2*t4 + {0,1} of every row tile j.
      constexpr int RT = C::RT;
      constexpr int MT = DV / 16;  // 16-column m-tiles of O^T
      const int t4 = lane & 3, g8 = lane >> 2;
      const int prefix = L - qo;
      int lim[RT][2];
#pragma unroll
      for (int j = 0; j < RT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) lim[j][e] = prefix + min((8 * j + 2 * t4 + e) / G, qo - 1);
      // draft trees: a row's mask word clears the drafts outside its tree (the
      // causal limit above still bounds it); the words are read only in the
      // blocks that reach the drafts
      const bool tree = tree_words != nullptr;
      if (tree && qo > 64 && lane == 0 && wk == 0) record_error(plan, PKV_DEV_TREE_TOO_LONG, b);

      // Q^T fragments (B operand): column g8 of row tile j is query row 8j + g8
      uint32_t qf[DK / 16][RT][2];
#pragma unroll
      for (int j = 0; j < RT; ++j) {
        const int rn = 8 * j + g8;
        const bool vn = rn < rows_valid;
        const long long qrow = ((long long)(q0 + rn / G) * a.num_q_heads + g * G + rn % G) * DK;
        if constexpr (!C::FP8) {
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const int c0 = kk * 16 + 2 * t4;
            qf[kk][j][0] = vn ? *reinterpret_cast<const uint32_t*>(a.q + qrow + c0) : 0u;
            qf[kk][j][1] = vn ? *reinterpret_cast<const uint32_t*>(a.q + qrow + c0 + 8) : 0u;
          }
        } else {
          // contraction order permuted to match the 8-byte K loads below:
          // k-step 2p  : slots {2t,2t+1} <- D 32p+8t+{0,1}, {2t+8,2t+9} <- D 32p+8t+{2,3}
          // k-step 2p+1: slots {2t,2t+1} <- D 32p+8t+{4,5}, {2t+8,2t+9} <- D 32p+8t+{6,7}
#pragma unroll
          for (int p = 0; p < DK / 32; ++p) {
            const uint4 x = vn ? *reinterpret_cast<const uint4*>(a.q + qrow + p * 32 + 8 * t4) : make_uint4(0, 0, 0, 0);
            qf[2 * p][j][0] = pack_f16(bf16lo(x.x), bf16hi(x.x));
            qf[2 * p][j][1] = pack_f16(bf16lo(x.y), bf16hi(x.y));
            qf[2 * p + 1][j][0] = pack_f16(bf16lo(x.z), bf16hi(x.z));
            qf[2 * p + 1][j][1] = pack_f16(bf16lo(x.w), bf16hi(x.w));
          }
        }
      }

      // O^T accumulators: o[mt][j] = {(c, 8j+2t4), (c, 8j+2t4+1), (c', 8j+2t4), (c', 8j+2t4+1)}
      // with columns c = kcol(mt, 0), c' = kcol(mt, 1)
      float o[MT][RT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < RT; ++j) o[mt][j][0] = o[mt][j][1] = o[mt][j][2] = o[mt][j][3] = 0.f;
      float m[RT][2], l[RT][2];
#pragma unroll
      for (int j = 0; j < RT; ++j) m[j][0] = m[j][1] = -INFINITY, l[j][0] = l[j][1] = 0.f;
      auto kcol = [&](int mt, int hi) { return C::FP8 ? 16 * mt + 2 * g8 + hi : 16 * mt + 8 * hi + g8; };

      for (int st = 0; st < nst; ++st) {
        // a failed wait keeps this warp on the common control flow (so every
        // named barrier still sees all consumer warps); the loop-top vote ends it
        if (!aborted && !mbar_wait_ab(&full[slot], phase, plan, s_abort)) {
          *s_abort = 1;
          aborted = true;
        }
        const uint32_t kbase = smem_u32(smem + slot * C::kStageBytes);
        const uint32_t vbase = kbase + C::kTileBytesK;
        const int stage_key0 = key_begin + st * C::kStageKeys;
        // last page of the request with a partial fill: zero the V rows past L
        const bool tail = (it.p1 == np_req) && (st == nst - 1) && (L % kSegSlots) != 0;
        if (tail) {
          const int r0 = L - stage_key0;
          const int r1 = min(C::kStagePages, npages - st * C::kStagePages) * kSegSlots;
          uint8_t* vb8 = smem + slot * C::kStageBytes + C::kTileBytesK;
          const int n16 = (r1 - r0) * C::kColBlocksV * 8;
          for (int i = cw * 32 + lane; i < n16; i += C::kConsumerWarps * 32) {
            const int row = r0 + i / (C::kColBlocksV * 8);
            const int rest = i % (C::kColBlocksV * 8);
            const int cb = rest / 8, ch = rest % 8;
            *reinterpret_cast<uint4*>(vb8 + cb * C::kStageKeys * 128 + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          named_bar_sync(1, C::kConsumerWarps * 32);
        }

        if (!skip) {
#pragma unroll
          for (int kb = 0; kb < C::KPW / 16; ++kb) {
            const int kr0 = wk * C::KPW + kb * 16;  // first stage row of this 16-key block
            const int abs0 = stage_key0 + kr0;
            if (abs0 >= key_end) break;
            // ---- S^T = K Q^T: s[j] = {(key g8, row 2t4), (g8, 2t4+1), (g8+8, 2t4), (g8+8, 2t4+1)}
            float s[RT][4];
#pragma unroll
            for (int j = 0; j < RT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
            if constexpr (!C::FP8) {
              const int key = kr0 + (lane & 15);
#pragma unroll
              for (int kk = 0; kk < DK / 16; ++kk) {
                const int chunk = 2 * kk + (lane >> 4);
                const uint32_t addr = kbase + (chunk >> 3) * (C::kStageKeys * 128) + swz(key, chunk & 7);
                uint32_t ka[4];
                ldsm_x4(addr, ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
                for (int j = 0; j < RT; ++j) mma_bf16(s[j], ka, qf[kk][j][0], qf[kk][j][1]);
              }
            } else {
#pragma unroll
              for (int p = 0; p < DK / 32; ++p) {
                const int byte = p * 32 + 8 * t4;
                uint32_t x0[2], x1[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint32_t addr = kbase + swz(kr0 + g8 + 8 * h, byte >> 4) + (byte & 15);
                  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(x0[h]), "=r"(x1[h]) : "r"(addr));
                }
                const uint32_t ka0[4] = {e4m3x2_to_f16x2((uint16_t)(x0[0] & 0xffff)),
                                         e4m3x2_to_f16x2((uint16_t)(x0[1] & 0xffff)),
                                         e4m3x2_to_f16x2((uint16_t)(x0[0] >> 16)),
                                         e4m3x2_to_f16x2((uint16_t)(x0[1] >> 16))};
                const uint32_t ka1[4] = {e4m3x2_to_f16x2((uint16_t)(x1[0] & 0xffff)),
                                         e4m3x2_to_f16x2((uint16_t)(x1[1] & 0xffff)),
                                         e4m3x2_to_f16x2((uint16_t)(x1[0] >> 16)),
                                         e4m3x2_to_f16x2((uint16_t)(x1[1] >> 16))};
#pragma unroll
                for (int j = 0; j < RT; ++j) {
                  mma_f16(s[j], ka0, qf[2 * p][j][0], qf[2 * p][j][1]);
                  mma_f16(s[j], ka1, qf[2 * p + 1][j][0], qf[2 * p + 1][j][1]);
                }
              }
            }
            // ---- mask, online softmax over the 16 keys (log2 domain) ----
            if (tree && abs0 + 15 >= prefix) {
              // the block reaches the drafts: raw scores of drafts outside a
              // row's tree to -inf (the scale below is positive)
#pragma unroll
              for (int j = 0; j < RT; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int r = 8 * j + 2 * t4 + e;
                  const uint64_t tw = r < rows_valid ? tree_words[q0 + r / G] : ~0ull;
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    const int dj = abs0 + g8 + 8 * h - prefix;
                    if (dj >= 0 && !(dj < 64 && ((tw >> dj) & 1ull))) s[j][2 * h + e] = -INFINITY;
                  }
                }
            }
            float al[RT][2];
            bool rescale = false;
#pragma unroll
            for (int j = 0; j < RT; ++j) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int kp = abs0 + g8 + 8 * h;
                const bool ok = kp < key_end;
#pragma unroll
                for (int e = 0; e < 2; ++e)
                  s[j][2 * h + e] = (ok && kp <= lim[j][e]) ? s[j][2 * h + e] * a.scale_log2 : -INFINITY;
              }
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float mx = fmaxf(s[j][e], s[j][2 + e]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(m[j][e], mx);
                const float ref = mn == -INFINITY ? 0.f : mn;
                al[j][e] = fast_exp2(m[j][e] - ref);
                m[j][e] = mn;
                s[j][e] = fast_exp2(s[j][e] - ref);
                s[j][2 + e] = fast_exp2(s[j][2 + e] - ref);
                l[j][e] = l[j][e] * al[j][e] + s[j][e] + s[j][2 + e];
                rescale |= al[j][e] != 1.f;
              }
            }
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int j = 0; j < RT; ++j) {
                  o[mt][j][0] *= al[j][0];
                  o[mt][j][1] *= al[j][1];
                  o[mt][j][2] *= al[j][0];
                  o[mt][j][3] *= al[j][1];
                }
            }
            // ---- P^T as the B operand: the accumulator layout of keys 0-7 and
            // 8-15 is that of an ldmatrix fragment, and its transpose is B's
            uint32_t pb[RT][2];
#pragma unroll
            for (int j = 0; j < RT; ++j) {
              pb[j][0] = movmatrix_trans(C::FP8 ? pack_f16(s[j][0], s[j][1]) : pack_bf16(s[j][0], s[j][1]));
              pb[j][1] = movmatrix_trans(C::FP8 ? pack_f16(s[j][2], s[j][3]) : pack_bf16(s[j][2], s[j][3]));
            }
            // ---- O^T += V^T P^T ----
            if constexpr (!C::FP8) {
              const int key = kr0 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const int chunk = 2 * mt + ((lane >> 3) & 1);
                const uint32_t addr = vbase + (chunk >> 3) * (C::kStageKeys * 128) + swz(key, chunk & 7);
                uint32_t va[4];
                ldsm_x4_t(addr, va[0], va[1], va[2], va[3]);
#pragma unroll
                for (int j = 0; j < RT; ++j) mma_bf16(o[mt][j], va, pb[j][0], pb[j][1]);
              }
            } else {
              const int key = kr0 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
              for (int mp = 0; mp < DV / 32; ++mp) {
                // 16-byte chunks 2mp (D 32mp..+15) and 2mp+1 (D 32mp+16..+31);
                // r0: keys 0-7 / chunk 2mp, r1: keys 8-15 / chunk 2mp, r2, r3: chunk 2mp+1.
                // bytes of r: V[2t][2g], V[2t][2g+1], V[2t+1][2g], V[2t+1][2g+1], so
                // m-row g of a tile is column 2g and m-row g+8 is column 2g+1
                const int chunk = 2 * mp + (lane >> 4);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(vbase + swz(key, chunk), r0, r1, r2, r3);
                const uint32_t va0[4] = {e4m3x2_to_f16x2((uint16_t)__byte_perm(r0, 0, 0x0020)),
                                         e4m3x2_to_f16x2((uint16_t)__byte_perm(r0, 0, 0x0031)),
                                         e4m3x2_to_f16x2((uint16_t)__byte_perm(r1, 0, 0x0020)),
                                         e4m3x2_to_f16x2((uint16_t)__byte_perm(r1, 0, 0x0031))};
                const uint32_t va1[4] = {e4m3x2_to_f16x2((uint16_t)__byte_perm(r2, 0, 0x0020)),
                                         e4m3x2_to_f16x2((uint16_t)__byte_perm(r2, 0, 0x0031)),
                                         e4m3x2_to_f16x2((uint16_t)__byte_perm(r3, 0, 0x0020)),
                                         e4m3x2_to_f16x2((uint16_t)__byte_perm(r3, 0, 0x0031))};
#pragma unroll
                for (int j = 0; j < RT; ++j) {
                  mma_f16(o[2 * mp][j], va0, pb[j][0], pb[j][1]);
                  mma_f16(o[2 * mp + 1][j], va1, pb[j][0], pb[j][1]);
                }
              }
            }
          }
        }
        const bool hold = st == nst - 1;  // last stage doubles as merge scratch
        if (!hold) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
          if (++slot == C::STAGES) {
            slot = 0;
            phase ^= 1;
          }
        }
      }
      // ------------------------------------------------ epilogue (key-major)
      // each lane summed its own keys: add over the eight lanes of a row
#pragma unroll
      for (int j = 0; j < RT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          l[j][e] += __shfl_xor_sync(0xffffffffu, l[j][e], 4);
          l[j][e] += __shfl_xor_sync(0xffffffffu, l[j][e], 8);
          l[j][e] += __shfl_xor_sync(0xffffffffu, l[j][e], 16);
        }
      const bool direct = nsplit == 1;
      const int split = it.split;
      auto out_row = [&](int r, uint16_t*& orow, float*& lrow) {
        const int i = r / G, h = g * G + r % G;
        const long long t = q0 + i;
        if (direct) {
          orow = a.out + (t * a.num_q_heads + h) * DV;
          lrow = a.lse ? a.lse + t * a.num_q_heads + h : nullptr;
        } else {
          const long long pr = (long long)a.m.partial_indptr[b] + (long long)split * qo + i;
          orow = a.m.partial_o + (pr * a.num_q_heads + h) * DV;
          lrow = a.m.partial_lse + pr * a.num_q_heads + h;
        }
      };
      // scratch columns XOR-swizzled by row so a store's 32 lanes hit 32 banks
      auto kswz = [](int r) { return ((r >> 1) & 3) << (C::FP8 ? 4 : 3); };
      if (nst == 0) {
        // empty key range (padding request): zero output, -inf LSE
        if (wk == 0 && !skip) {
          for (int idx = lane; idx < rows_valid * (DV / 2); idx += 32) {
            const int r = idx / (DV / 2), c2 = idx % (DV / 2);
            uint16_t* orow;
            float* lrow;
            out_row(r, orow, lrow);
            *reinterpret_cast<uint32_t*>(orow + 2 * c2) = 0u;
            // no key: the LSE is the sink's alone (final rows only)
            if (c2 == 0 && lrow) *lrow = (direct && sinks) ? sinks[g * G + r % G] : -INFINITY;
          }
        }
      } else {
        named_bar_sync(1, C::kConsumerWarps * 32);  // everyone done reading the held stage
        float* scr = reinterpret_cast<float*>(smem + slot * C::kStageBytes);  // [WK][16][DV]
        float* my = scr + wk * 16 * DV;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < RT; ++j)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int r = 8 * j + 2 * t4 + e;
                my[r * DV + (kcol(mt, hi) ^ kswz(r))] = o[mt][j][2 * hi + e];
              }
        if (g8 == 0) {
#pragma unroll
          for (int j = 0; j < RT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = 8 * j + 2 * t4 + e;
              s_ml[(wk * 16 + r) * 2 + 0] = m[j][e];
              s_ml[(wk * 16 + r) * 2 + 1] = l[j][e];
            }
        }
        named_bar_sync(1, C::kConsumerWarps * 32);
        // each consumer thread finishes float4 pieces of the rows x DV tile
        const int nthr = C::kConsumerWarps * 32;
        const int ctid = cw * 32 + lane;
        const int nrows = skip ? 0 : min(rows_valid, C::kRows);
        for (int idx = ctid; idx < nrows * (DV / 4); idx += nthr) {
          const int r = idx / (DV / 4), c4 = idx % (DV / 4);
          float mw[C::WK], lw[C::WK];
          float M = -INFINITY;
#pragma unroll
          for (int k = 0; k < C::WK; ++k) {
            mw[k] = s_ml[(k * 16 + r) * 2 + 0];
            lw[k] = s_ml[(k * 16 + r) * 2 + 1];
            M = fmaxf(M, mw[k]);
          }
          float Lsum = 0.f, wgt[C::WK];
#pragma unroll
          for (int k = 0; k < C::WK; ++k) {
            wgt[k] = (M == -INFINITY) ? 0.f : fast_exp2(mw[k] - M);
            Lsum += lw[k] * wgt[k];
          }
          const float inv = Lsum > 0.f ? a.v_scale / Lsum : 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k = 0; k < C::WK; ++k) {
            const float4 x = *reinterpret_cast<const float4*>(scr + (k * 16 + r) * DV + ((c4 * 4) ^ kswz(r)));
            acc.x += x.x * wgt[k];
            acc.y += x.y * wgt[k];
            acc.z += x.z * wgt[k];
            acc.w += x.w * wgt[k];
          }
          float lse_r = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
          const float fs = (direct && sinks) ? sink_factor(lse_r, sinks[g * G + r % G]) : 1.f;
          uint16_t* orow;
          float* lrow;
          out_row(r, orow, lrow);
          *reinterpret_cast<uint2*>(orow + c4 * 4) = make_uint2(pack_bf16(acc.x * inv * fs, acc.y * inv * fs),
                                                                pack_bf16(acc.z * inv * fs, acc.w * inv * fs));
          if (c4 == 0 && lrow) *lrow = lse_r;
        }
        fence_proxy_async_smem();
        named_bar_sync(1, C::kConsumerWarps * 32);  // scratch reads done before the stage is refilled
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == C::STAGES) {
          slot = 0;
          phase ^= 1;
        }
      }
    }

  }

}


// Split merge: every (request, KV head) group's rows (query tokens x heads of
// the group) get one warp each; blocks of 4 warps walk (group, row block)
// items with a grid stride. Groups of requests with one split, or with more
// rows per head than max_rows_per_head (those were not split on the calling
// path), are skipped. The extend path merges its own (tile-aligned) split
// counts, the decode path the decode plan's.
// One warp per (token, query head) row of the batch; rows of requests that
// were not split on this path are skipped.
template <int D>
__global__ void __launch_bounds__(256, 3) split_merge_kernel(DecodeArgs a, int max_rows_per_head, int count_word,
                                                          int extend_path) {
  pdl_wait();  // the partial rows come from the preceding attention grid
  // the decode grid has finished: its unit counter starts from zero next time
  if (blockIdx.x == 0 && threadIdx.x == 0) a.m.plan[kDecodeNext] = 0;
  if (a.m.plan[count_word] == 0) return;  // nothing was split on this path
  const int rows = a.m.plan[kTotalQ] * a.num_q_heads;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  // each warp takes a contiguous run of rows (consecutive heads of a token),
  // so a token's request and split count are looked up once for its heads
  // rather than once per row through a chain of dependent loads
  const int per = (rows + nwarps - 1) / nwarps;
  const int row0 = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * per;
  const int row1 = min(rows, row0 + per);
  int cur_t = -1, b = 0, nsplit = 0, q0 = 0, qo = 0, pbase = 0;
  for (int row = row0; row < row1; ++row) {
    const int t = row / a.num_q_heads, h = row - t * a.num_q_heads;
    if (t != cur_t) {
      cur_t = t;
      b = a.m.token_req[t];
      nsplit = extend_path ? a.m.ext_splits[b] : a.m.n_splits[b];
      q0 = a.m.qo_indptr[b];
      qo = a.m.qo_indptr[b + 1] - q0;
      pbase = a.m.partial_indptr[b];
    }
    if (nsplit <= 1 || qo * a.group > max_rows_per_head) continue;
    merge_row<D>(a, pbase, qo, t - q0, h, nsplit, (long long)row, lane);
  }
}

template <class C>
int run_decode(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
               float v_scale, void* out, float* lse, cudaStream_t st) {
  CUtensorMap tk, tv;
  const CUtensorMapDataType dt = C::FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t inner_k = (uint64_t)c.cfg.num_kv_heads * C::DK;
  const uint64_t inner_v = (uint64_t)c.cfg.num_kv_heads * C::DV;
  const uint64_t slots = (uint64_t)c.cfg.num_pages * c.cfg.page_size;
  const uint32_t box_inner = 128 / C::kElem;
  // L2 fills no wider than one head's row of an E4M3 pool (128 bytes)
  const CUtensorMapL2promotion promo = C::FP8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  if (encode_tmap_2d(&tk, dt, const_cast<void*>(k_pool), inner_k, slots, inner_k * C::kElem, box_inner, kSegSlots,
                     CU_TENSOR_MAP_SWIZZLE_128B, promo) != PKV_OK)
    return PKV_ERR_CUDA;
  if (encode_tmap_2d(&tv, dt, const_cast<void*>(v_pool), inner_v, slots, inner_v * C::kElem, box_inner, kSegSlots,
                     CU_TENSOR_MAP_SWIZZLE_128B, promo) != PKV_OK)
    return PKV_ERR_CUDA;
  DecodeArgs a;
  a.m = make_meta(c);
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.num_q_heads = c.cfg.num_q_heads;
  a.num_kv_heads = c.cfg.num_kv_heads;
  a.group = c.cfg.num_q_heads / c.cfg.num_kv_heads;
  const bool fp8 = c.cfg.kv_dtype == PKV_KV_FP8_E4M3;
  a.scale_log2 = sm_scale * (fp8 ? k_scale : 1.f) * kLog2e;
  a.v_scale = fp8 ? v_scale : 1.f;
  a.tree = active_tree(c);
  a.sinks = c.sinks;
  auto kernel = (a.tree || a.sinks) ? decode_splitkv_kernel<C, true> : decode_splitkv_kernel<C, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (launch_pdl(kernel, dim3(c.decode_ctas), dim3(C::kThreads), C::kSmemBytes, st, tk, tv, a) != cudaSuccess)
    return PKV_ERR_CUDA;
  return launch_split_merge(c, out, lse, c.cfg.max_qo_len * a.group, false, st);
}

// Tile shapes: one or two 8-row key-major tiles per unit; four key warps
// split each stage's keys. With 192-wide K heads (bf16) a stage is 40 KB, so
// two stages keep two CTAs on an SM.
using DecBf16D128_1 = DecodeCfg<128, 128, false, 4, 16, 3, 1>;
using DecBf16D128_2 = DecodeCfg<128, 128, false, 4, 16, 3, 2>;
using DecBf16D64_1 = DecodeCfg<64, 64, false, 4, 16, 4, 1>;
using DecBf16D64_2 = DecodeCfg<64, 64, false, 4, 16, 4, 2>;
using DecFp8D128_1 = DecodeCfg<128, 128, true, 4, 32, 3, 1>;
using DecFp8D128_2 = DecodeCfg<128, 128, true, 4, 32, 3, 2>;
using DecBf16D192_1 = DecodeCfg<192, 128, false, 4, 16, 2, 1>;
using DecBf16D192_2 = DecodeCfg<192, 128, false, 4, 16, 2, 2>;


}  // namespace

// Rows a decode-path unit must hold: every query row of one request's group.
int decode_row_warps(const pkv_config& cfg) {
  const int rows = cfg.max_qo_len * (cfg.num_q_heads / cfg.num_kv_heads);
  if (rows <= 16) return 1;
  if (rows <= 32) return 2;
  if (rows <= 64) return 4;
  if (rows <= 128) return 8;
  return 0;
}

// Pages per pipeline stage of the decode kernel; the metadata rounds the
// decode plan's chunks to whole stages. The verify shapes run on the tcgen05
// tile kernel, whose KV tiles are 128 keys (8 pages): their chunks are whole
// tiles.
int decode_stage_pages(const pkv_config& cfg) {
  if (decode_row_warps(cfg) > 1) return kExtendKeys / kSegSlots;
  return cfg.kv_dtype == PKV_KV_FP8_E4M3 ? 8 : 4;
}

int launch_decode(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
                  float v_scale, void* out, float* lse, cudaStream_t st) {
  const bool fp8 = c.cfg.kv_dtype == PKV_KV_FP8_E4M3;
  const int D = c.cfg.head_dim;
  // verify shapes (more than 16 rows per KV head): the tcgen05 tile kernel
  // over this path's plan
  if (decode_row_warps(c.cfg) > 1)
    return launch_decode_tc(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out, lse, st);
  // decode shapes (at most 16 rows): key-major tiles of one or two 8-row tiles
  const bool rt1 = c.cfg.max_qo_len * (c.cfg.num_q_heads / c.cfg.num_kv_heads) <= 8;
#define PKV_RUN(CFG) return run_decode<CFG>(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out, lse, st)
  if (!fp8 && D == 128) {
    if (rt1) PKV_RUN(DecBf16D128_1);
    PKV_RUN(DecBf16D128_2);
  } else if (!fp8 && D == 64) {
    if (rt1) PKV_RUN(DecBf16D64_1);
    PKV_RUN(DecBf16D64_2);
  } else if (fp8 && D == 128) {
    if (rt1) PKV_RUN(DecFp8D128_1);
    PKV_RUN(DecFp8D128_2);
  } else if (!fp8 && D == 192) {
    if (rt1) PKV_RUN(DecBf16D192_1);
    PKV_RUN(DecBf16D192_2);
  }
#undef PKV_RUN
  return PKV_ERR_UNSUPPORTED;
}

int launch_split_merge(Ctx& c, void* out, float* lse, int max_rows_per_head, bool extend_path, cudaStream_t st) {
  DecodeArgs a;
  a.m = make_meta(c);
  a.q = nullptr;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.num_q_heads = c.cfg.num_q_heads;
  a.num_kv_heads = c.cfg.num_kv_heads;
  a.group = c.cfg.num_q_heads / c.cfg.num_kv_heads;
  a.scale_log2 = 0.f;
  a.v_scale = 1.f;
  a.tree = nullptr;
  a.sinks = c.sinks;
  // one warp per (token, head) row, 8 warps per CTA, 3 CTAs per SM
  const long long rows = (long long)c.cfg.max_q_tokens * c.cfg.num_q_heads;
  const long long grid = std::min<long long>((rows + 7) / 8, (long long)c.num_sms * 3);
  if (rows <= 0) return PKV_OK;
  const int word = extend_path ? kSplitExtend : kSplitDecode;
  cudaError_t e;
  // partial and output rows have the V heads' width
  if (head_dim_v(c.cfg) == 128)
    e = launch_pdl(split_merge_kernel<128>, dim3((unsigned)grid), dim3(256), 0, st, a, max_rows_per_head, word,
                   extend_path ? 1 : 0);
  else
    e = launch_pdl(split_merge_kernel<64>, dim3((unsigned)grid), dim3(256), 0, st, a, max_rows_per_head, word,
                   extend_path ? 1 : 0);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
