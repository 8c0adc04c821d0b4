// forward_extend on the 5th-generation tensor cores ("--attention-backend",
// section "What an attention backend is": forward_extend runs prefill; section
// "Two backends in one server": prefill reads long query blocks and is bound by
// compute). The same kernel runs target-verify on the prefill path ("[SGLang]
// Hybrid Attention", section "_select_backend: ForwardMode 기반 동적 전환").
//
// A work unit is (request, 256 query rows, KV head): two 128-row tiles A and
// B that share every K/V tile. A row is a (query token, head-in-group) pair,
// so the GQA group shares K/V as well. Row of token i sees keys 0 .. P + i
// (P = cached prefix of the request).
//
// Warp roles (352 threads, one CTA per SM, persistent over units):
//   warps 0-3  softmax A, warps 4-7 softmax B: thread r of a warpgroup owns
//              row r of its tile (TMEM lane r). It reads S from TMEM, masks,
//              keeps the running sum against a reference in the log2 domain,
//              writes P (bf16) back into the first half of its S columns,
//              moves the reference and rescales O in TMEM only when the tile
//              sum leaves a fixed range (the factor cancels in O / l), and
//              writes the output rows.
//   warps 8, 10 producers: gather K (warp 8) and V (warp 10) pages with TMA
//              (one 16-token box per page and 128-byte column block, 128-byte
//              swizzle) into separate K and V rings; lane p reads the tile's
//              p-th page index and an elected lane issues the copies. Warp 8
//              also fills the Q tiles of the next unit as soon as the last QK
//              on them has finished: one TMA box of 128/G tokens x the G heads
//              of the group per column block when G divides 128 and the box
//              lies inside the batch, else the softmax warps copy their rows.
//   warp 9     MMA: owns 512 TMEM columns and issues tcgen05.mma
//              (kind::f16, bf16 in, fp32 accumulate) from an elected lane of
//              the converged warp:
//                S_X = Q_X K^T      (M=128, N=128 keys, K=head_dim; A, B from smem)
//                O_X += P_X V       (M=128, N=head_dim, K=128 keys; P from TMEM)
//              in the order PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1), so one
//              tile's softmax runs while the tensor core works on the other.
// TMEM columns: S_A 0-127, S_B 128-255, O_A 256-383, O_B 384-511.
#include <math.h>
#include <string.h>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Bounds on one tile's row sum of p = 2^(s * scale - m_ref) between which the
// reference m_ref stays put (see the softmax role). With bf16 P any p up to
// 2^16 is representable; with f16 P (E4M3 pools) p stays at most 2^15, below
// the f16 maximum, and a row's first mass at least 2^-8, so its largest p
// is a normal f16 number.
constexpr float kSumHigh = 65536.0f;               // 2^16
constexpr float kSumLow = 5.421010862427522e-20f;  // 2^-64
constexpr float kSumHighF16 = 32768.0f;            // 2^15
constexpr float kSumLowF16 = 0.00390625f;          // 2^-8

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

constexpr uint32_t kNegInfBits = 0xff800000u;

// 32-byte global store (sm_100+): a whole sector per lane, half the store
// instructions of 16-byte vectors. The address must be 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Visibility of the 32 keys key_base .. key_base + 31 for one row, one bit
// each: keys up to the row's limit, less the drafts (keys from draft0 on)
// whose bit is clear in the row's tree word (draft0 lies past every key when
// no tree is set).
__device__ __forceinline__ uint32_t visible32(int key_base, int limit, int draft0, uint64_t word) {
  const int n = limit - key_base + 1;  // keys within the limit
  const uint32_t v = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
  const int off = key_base - draft0;  // draft index of the first key
  uint32_t t;
  if (off >= 64)
    t = 0u;
  else if (off >= 0)
    t = (uint32_t)(word >> off);
  else if (off > -32)
    t = (uint32_t)(word << (-off)) | ((1u << (-off)) - 1u);
  else
    t = 0xffffffffu;
  return v & t;
}

// Raw scores of the keys whose bit is clear in vis to -inf.
__device__ __forceinline__ void mask32_bits(uint32_t* sr, uint32_t vis) {
#pragma unroll
  for (int c = 0; c < 32; ++c) sr[c] = (vis >> c) & 1u ? sr[c] : kNegInfBits;
}

// Masks raw scores of keys past the row's limit (sets them to -inf).
__device__ __forceinline__ void mask32(uint32_t* sr, int key_base, int limit) {
#pragma unroll
  for (int c = 0; c < 32; ++c) sr[c] = key_base + c > limit ? kNegInfBits : sr[c];
}

// Max of 32 raw scores with four independent 3-input chains.
__device__ __forceinline__ float max32(const uint32_t* sr, float m) {
  float a0 = m, a1 = m, a2 = m, a3 = m;
#pragma unroll
  for (int c = 0; c < 32; c += 8) {
    a0 = max3f(a0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
    a1 = max3f(a1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
    a2 = max3f(a2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
    a3 = max3f(a3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
  }
  return max3f(fmaxf(a0, a1), a2, a3);
}

// p = exp2(s * scale - ref) for 32 raw scores: packed bf16 (F16: f16) pairs
// into pk, running sums in four packed accumulators.
template <bool F16>
__device__ __forceinline__ void exp32(const uint32_t* sr, uint64_t sc2, uint64_t nref2, uint32_t* pk, uint64_t* acc) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nref2);
    const float p0 = fast_exp2(f2_lo(x)), p1 = fast_exp2(f2_hi(x));
    acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(p0, p1));
    pk[c >> 1] = F16 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// 8 bf16 -> 8 f16 (round to nearest even; exact for the normal range)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& v) {
  auto cv = [](uint32_t w) { return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); };
  return make_uint4(cv(v.x), cv(v.y), cv(v.z), cv(v.w));
}

// The two tiles' KV ranges inside a unit, and the order in which the unit's
// KV tiles pass through the K and V rings. A shared unit streams KV tile
// kv0 + j once, for both tiles; a dual unit (both tiles hold the same rows,
// tile A the first half of the KV range, tile B the rest) streams, for each
// step j, tile A's tile and then tile B's. Producers, MMA warp and softmax
// warps all walk this same sequence.
struct UnitKV {
  int s0, s1, n0, n1;  // tile A's and tile B's KV tiles: [s0, s0 + n0), [s1, s1 + n1)
  bool dual;
  __device__ __forceinline__ int start(int x) const { return x == 0 ? s0 : s1; }
  __device__ __forceinline__ int n(int x) const { return x == 0 ? n0 : n1; }
  __device__ __forceinline__ int steps() const { return max(n0, n1); }
  __device__ __forceinline__ int len() const { return dual ? n0 + n1 : max(n0, n1); }
  // position in the unit's ring sequence of tile X's j-th KV tile
  __device__ __forceinline__ int pos(int x, int j) const {
    if (!dual) return j;
    return x == 0 ? j + min(j, n1) : j + min(j + 1, n0);
  }
  // tile X's QKs read Q tile X (a dual unit's tiles both read Q tile A)
  __device__ __forceinline__ bool uses_q(int x) const { return dual ? x == 0 : n(x) > 0; }
};

__device__ __forceinline__ UnitKV unit_kv(const ExtendTile& u) {
  UnitKV k;
  k.dual = u.dual != 0;
  if (k.dual) {
    const int n = max(0, min(u.kv1, u.kv_a) - u.kv0);
    k.s0 = u.kv0;
    k.n0 = (n + 1) >> 1;
    k.s1 = u.kv0 + k.n0;
    k.n1 = n - k.n0;
  } else {
    k.s0 = k.s1 = u.kv0;
    k.n0 = max(0, min(u.kv1, u.kv_a) - u.kv0);
    k.n1 = max(0, min(u.kv1, u.kv_b) - u.kv0);
  }
  return k;
}

// DK: width of the Q and K heads; DV: of the V heads and the output rows
// (equal except for models whose K and V heads differ, 192 / 128).
// FP8: E4M3 pools. TMA brings the codes into raw rings (RK / RV tiles of one
// byte per code), the K and V producer warps widen them to f16 (exactly) into
// the operand rings, and the MMAs run in f16 with Q and P rounded to f16.
template <int DK_, int DV_, int NK_, int NV_, bool FP8_ = false, int RK_ = 0, int RV_ = 0>
struct ExtCfg {
  static constexpr int DK = DK_;
  static constexpr int DV = DV_;
  static constexpr int NK = NK_;  // K ring depth
  static constexpr int NV = NV_;  // V ring depth
  static constexpr bool FP8 = FP8_;
  static constexpr int RK = RK_;  // raw E4M3 K tiles in flight
  static constexpr int RV = RV_;
  static constexpr int kThreads = 352;
  static constexpr int kProducerWarp = 8;   // K tiles
  static constexpr int kMmaWarp = 9;
  static constexpr int kVProducerWarp = 10;  // V tiles
  static constexpr int kColBlocksK = DK / 64;                // 128-byte swizzle spans per Q or K row
  static constexpr int kColBlocksV = DV / 64;                // per V row
  static constexpr int kQBytes = kExtendRows * DK * 2;       // one Q tile: [cb][128 rows][128 B]
  static constexpr int kTileBytesK = kExtendKeys * DK * 2;   // one K tile
  static constexpr int kTileBytesV = kExtendKeys * DV * 2;   // one V tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kQBytes;
  static constexpr int kVOff = kKOff + NK * kTileBytesK;
  static constexpr int kRawTileBytes = kExtendKeys * 128;  // 128 E4M3 codes per row
  static constexpr int kRawKOff = kVOff + NV * kTileBytesV;
  static constexpr int kRawVOff = kRawKOff + RK * kRawTileBytes;
  static constexpr int kBarOff = kRawVOff + RV * kRawTileBytes;
  static constexpr int kNumBars = 2 + 2 * NK + 2 * NV + 6 + 4 + 2 + RK + RV + 1;
  static constexpr int kMergeOff = kBarOff + kNumBars * 8;           // dual units: tile B's (m, l) per row
  static constexpr int kTmemSlotOff = kMergeOff + 2 * kExtendRows * 4;
  static constexpr int kAbortOff = kTmemSlotOff + 8;
  static constexpr int kSmemBytes = kAbortOff + 8 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(DV <= 128, "O needs at most 128 TMEM columns per tile");
  static_assert(!FP8 || (DK == 128 && DV == 128 && RK >= 1 && RV >= 1), "E4M3 rows are one 128-byte span");
  static_assert(FP8 || (RK == 0 && RV == 0), "raw rings only for E4M3 pools");
};

struct ExtendArgs {
  Meta m;
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  int num_q_heads, num_kv_heads, group;
  float scale_log2;
  float v_scale;     // multiplies the output rows (the V pool's scale of an E4M3 pool; 1 for bf16)
  int q_tma;         // 1 when the group divides 128: a Q tile is one TMA box of 128/G tokens x G heads
  int q_box_tokens;  // 128 / group
  int out_32B;       // out is 32-byte aligned: output rows are written with 32-byte stores
  const uint64_t* tree;  // draft-tree mask word per query token, or null (chain drafts)
  const float* sinks;    // sink logit per query head, or null
  // 1: the units are the decode plan's (request, split) items, the decode
  // path's verify shapes (at most 128 rows per KV head); 0: the extend plan
  int dplan;
};

// Work unit idx of the plan the kernel runs. A decode-plan item (request b,
// split s, pages [p0, p1)) becomes a dual unit: its rows (every query token
// of the request times the group's heads) fit one 128-row tile, both tiles
// hold them and take half of the item's KV tiles each. The decode plan's
// chunks are whole 128-key tiles on these shapes, so [p0, p1) maps onto KV
// tiles exactly; a request cut into several items writes partial rows that
// the decode path's merge combines.
__device__ __forceinline__ ExtendTile load_unit(const ExtendArgs& a, int idx) {
  if (!a.dplan) return a.m.extend_tiles[idx];
  constexpr int kPagesPerTile = kExtendKeys / kSegSlots;
  const DecodeItem it = a.m.decode_items[idx];
  ExtendTile u;
  u.b = it.b;
  u.row0 = 0;
  u.kv_a = (a.m.kv_len[it.b] + kExtendKeys - 1) / kExtendKeys;  // the last row sees every key
  u.kv_b = 0;
  u.split = a.m.n_splits[it.b] > 1 ? it.split : -1;
  u.kv0 = it.p0 / kPagesPerTile;
  u.kv1 = (it.p1 + kPagesPerTile - 1) / kPagesPerTile;
  u.dual = 1;
  return u;
}

// EXTRAS: draft-tree mask words or attention sinks are in use (a separate
// instantiation, so plain batches run the causal kernel without that code).
template <class C, bool EXTRAS>
__global__ void __launch_bounds__(C::kThreads, 1) extend_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                   const __grid_constant__ CUtensorMap tmap_v,
                                                                   const __grid_constant__ CUtensorMap tmap_q,
                                                                   ExtendArgs a) {
  constexpr int DK = C::DK, DV = C::DV;
  constexpr int NK = C::NK, NV = C::NV;
  constexpr int kPagesPerTile = kExtendKeys / kSegSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;              // [2] tile A, B: Q rows written
  uint64_t* k_full = bars + 2;          // [NK]
  uint64_t* k_empty = k_full + NK;      // [NK]
  uint64_t* v_full = k_empty + NK;      // [NV]
  uint64_t* v_empty = v_full + NV;      // [NV]
  uint64_t* s_full = v_empty + NV;      // [2] S_X computed
  uint64_t* p_full = s_full + 2;        // [2] P_X written
  uint64_t* pv_done = p_full + 2;       // [2] last PV_X of a unit finished
  uint64_t* q_empty = pv_done + 2;      // [2] last QK_X of a unit finished: Q_X may be refilled
  uint64_t* q_written = q_empty + 2;    // [2] softmax warps wrote Q_X (tiles not loaded by TMA)
  uint64_t* b_done = q_written + 2;     // dual unit: tile B's O is final and its (m, l) are in smem
  uint64_t* a_read = b_done + 1;        // dual unit: tile A has read tile B's O and (m, l)
  uint64_t* raw_full = a_read + 1;      // E4M3: [RK] raw K tiles, then [RV] raw V tiles, landed
  uint64_t* mma_drain = raw_full + C::RK + C::RV;  // after an abort: the MMAs issued so far have finished
  float* s_merge = reinterpret_cast<float*>(smem + C::kMergeOff);  // [2][128]: m, l of tile B's rows
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kTmemSlotOff);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* plan = a.m.plan;
  pdl_launch_dependents();

  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);  // the K producer (plus the TMA bytes when Q comes by TMA)
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);  // one arrival per softmax warp
      mbar_init(&pv_done[x], 1);
      mbar_init(&q_empty[x], 1);
      mbar_init(&q_written[x], 4);
    }
    mbar_init(b_done, 4);  // one arrival per softmax warp
    mbar_init(a_read, 4);
    // K / V operand tiles: the producer's arrival (with the TMA bytes, or
    // after widening E4M3 codes)
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < C::RK + C::RV; ++s) mbar_init(&raw_full[s], 1);
    mbar_init(mma_drain, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  // K/V stages start as zeros so rows of a partly loaded tile are finite
  for (int i = tid; i < (NK * C::kTileBytesK + NV * C::kTileBytesV) / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(smem + C::kKOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // launched with programmatic serialization: metadata, Q and the K/V this
  // step stored are only read after the preceding grid has finished
  pdl_wait();

  const int n_units = plan[a.dplan ? kDecodeItems : kExtendTiles] * a.num_kv_heads;
  const int G = a.group;
  const uint32_t smem_base = smem_u32(smem);
  const int total_q = plan[kTotalQ];
  // Tile X of unit u takes its Q by TMA when the box of 128/G tokens lies
  // inside the batch's tokens (never past the end of the caller's q buffer);
  // otherwise the softmax warps write it.
  auto q_by_tma = [&](const ExtendTile& u, int x) {
    return a.q_tma != 0 && a.m.qo_indptr[u.b] + (u.row0 + x * kExtendRows) / G + a.q_box_tokens <= total_q;
  };

  if (C::FP8 && (warp == C::kProducerWarp || warp == C::kVProducerWarp)) {
    // ------------------------------------------------------------ E4M3 producers
    // Warp 8 streams K, warp 10 V. TMA lands each tile's codes in the raw ring
    // (one 16-row x 128-byte box per page, 128-byte swizzle); the warp widens
    // the rows of the loaded pages to f16 (exact) into the operand ring, in
    // the operand layout (two 64-column blocks, 128-byte swizzle), and marks
    // the operand tile full. A raw slot is requested again as soon as the warp
    // has read it, R tiles ahead of the widening. Warp 8 also hands Q over.
    const bool is_v = warp == C::kVProducerWarp;
    const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
    if (elect_one()) prefetch_tmap(tmap);
    const int R = is_v ? C::RV : C::RK;
    const int depth = is_v ? NV : NK;
    uint64_t* rfull = is_v ? raw_full + C::RK : raw_full;
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* empty = is_v ? v_empty : k_empty;
    uint8_t* raw_ring = smem + (is_v ? C::kRawVOff : C::kRawKOff);
    const uint32_t raw_base = smem_u32(raw_ring);
    const uint32_t op_base = smem_u32(smem + (is_v ? C::kVOff : C::kKOff));
    constexpr int kOpTile = kExtendKeys * 128 * 2;  // one f16 tile of 128-wide rows
    const uint64_t pol_stream = policy_evict_first();  // the bf16 producers' choice, below
    const uint64_t pol_reuse = policy_evict_normal();
    uint32_t jt = 0;  // operand tiles so far
    uint32_t rt = 0, ct = 0;  // raw tiles requested / widened so far
    uint32_t qcount[2] = {0, 0}, qtcount[2] = {0, 0};
    bool stop = false;
    const int c = lane & 7, r0 = lane >> 3;  // 16-code chunk and first row of this lane
    // test support: CTA 0 arms its first raw K tile but never loads it
    const bool hold_first = !is_v && blockIdx.x == 0 && __ldcg(plan + kHoldLoad) != 0;
    for (int w = blockIdx.x; w < n_units && !stop; w += gridDim.x) {
      const ExtendTile u = load_unit(a, w / a.num_kv_heads);
      const int g = w % a.num_kv_heads;
      const UnitKV ukv = unit_kv(u);
      const int np = a.m.seg_indptr[u.b + 1] - a.m.seg_indptr[u.b];
      const int page_base = a.m.seg_indptr[u.b];
      const bool reused = !a.dplan && (a.m.qo_indptr[u.b + 1] - a.m.qo_indptr[u.b]) * G > kExtendUnitRows;
      const uint64_t pol = reused ? pol_reuse : pol_stream;
      auto seq_tile = [&](int e) {
        if (!ukv.dual) return ukv.s0 + e;
        const int m = min(ukv.n0, ukv.n1);
        const int step = e < 2 * m ? e >> 1 : e - m;
        const int x = e < 2 * m ? (e & 1) : (ukv.n0 > ukv.n1 ? 0 : 1);
        return ukv.start(x) + step;
      };
      const int len = ukv.len();
      // page indices of 4 consecutive tiles: lane 8k + p holds page p of tile e0 + k
      auto load_group = [&](int e0) {
        const int e = e0 + (lane >> 3), p = lane & 7;
        if (e >= len) return 0;
        const int jj = seq_tile(e);
        return p < np - jj * kPagesPerTile ? __ldg(a.m.seg_indices + page_base + jj * kPagesPerTile + p) : 0;
      };
      int grp = load_group(0);
      int grp_next = load_group(4);
      int issued = 0;
      // request raw tile `issued` of the unit into raw slot rt % R (read already)
      auto issue = [&]() {
        const int e = issued;
        if (e > 0 && (e & 3) == 0) {
          grp = grp_next;
          grp_next = load_group(e + 4);
        }
        const int j = seq_tile(e);
        const int npg = min(kPagesPerTile, np - j * kPagesPerTile);
        const int rs = (int)(rt % R);
        const bool leader = elect_one();
        if (leader) mbar_arrive_expect_tx(&rfull[rs], (uint32_t)(npg * kSegSlots * 128));
        uint8_t* dst = raw_ring + rs * C::kRawTileBytes;
#pragma unroll
        for (int p = 0; p < kPagesPerTile; ++p) {
          const int pg = __shfl_sync(0xffffffffu, grp, ((e & 3) << 3) + p);
          if (p < npg && leader && !(hold_first && rt == 0))
            tma_load_2d_hint(dst + p * (kSegSlots * 128), tmap, g * 128, pg * kSegSlots, &rfull[rs], pol);
        }
        ++rt;
        ++issued;
      };
      for (int k = 0; k < R && issued < len; ++k) issue();
      if (!is_v) {
        // Q of the unit: written (f16) by the softmax warps once the previous
        // unit's last QK on the tile has finished, then handed to the MMA warp
        // (the first raw tiles are in flight meanwhile)
        for (int x = 0; x < 2 && !stop; ++x) {
          if (!ukv.uses_q(x)) continue;
          if (!mbar_wait_warp(&q_empty[x], (qcount[x] & 1) ^ 1, plan, s_abort) ||
              !mbar_wait_warp(&q_written[x], qtcount[x] & 1, plan, s_abort)) {
            stop = true;
            break;
          }
          ++qtcount[x];
          ++qcount[x];
          if (elect_one()) mbar_arrive(&q_full[x]);
        }
        if (stop) break;
      }
      for (int e = 0; e < len; ++e, ++jt) {
        const int rs = (int)(ct % R);
        if (!mbar_wait_warp(&rfull[rs], (ct / R) & 1, plan, s_abort)) {
          stop = true;
          break;
        }
        ++ct;
        const int j = seq_tile(e);
        const int npg = min(kPagesPerTile, np - j * kPagesPerTile);
        const int st = jt % depth;
        if (!mbar_wait_warp(&empty[st], ((jt / depth) & 1) ^ 1, plan, s_abort)) {
          stop = true;
          break;
        }
        const uint32_t src = raw_base + rs * C::kRawTileBytes;
        const uint32_t out_blk = op_base + st * kOpTile + (c >> 2) * (kExtendKeys * 128);
        // lane: chunk c (codes 16c .. 16c + 15) of rows r0 + 4k; one 16-byte
        // chunk in, f16 chunks 2c and 2c + 1 of column block c / 4 out. Four
        // rows a group, the next group's chunks loaded before this one is widened.
        auto ld = [&](int k) {
          const int r = r0 + 4 * k;
          return lds128(src + r * 128 + ((c ^ (r & 7)) << 4));
        };
        auto widen = [&](int k, const uint4& x) {
          const int r = r0 + 4 * k;
          const uint4 lo = make_uint4(e4m3x2_to_f16x2((uint16_t)(x.x & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x.x >> 16)),
                                      e4m3x2_to_f16x2((uint16_t)(x.y & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x.y >> 16)));
          const uint4 hi = make_uint4(e4m3x2_to_f16x2((uint16_t)(x.z & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x.z >> 16)),
                                      e4m3x2_to_f16x2((uint16_t)(x.w & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x.w >> 16)));
          const uint32_t row = out_blk + r * 128;
          sts128(row + ((((2 * c) & 7) ^ (r & 7)) << 4), lo);
          sts128(row + ((((2 * c + 1) & 7) ^ (r & 7)) << 4), hi);
        };
        const int nk = npg * 4;  // groups of four rows (a multiple of 4)
        uint4 x[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) x[v] = ld(v);
        for (int k0 = 0; k0 < nk; k0 += 4) {
          uint4 y[4];
          const bool more = k0 + 4 < nk;
#pragma unroll
          for (int v = 0; v < 4; ++v) y[v] = more ? ld(k0 + 4 + v) : x[v];
#pragma unroll
          for (int v = 0; v < 4; ++v) widen(k0 + v, x[v]);
#pragma unroll
          for (int v = 0; v < 4; ++v) x[v] = y[v];
        }
        // the f16 tile is read by the tensor core (async proxy), and the raw
        // slot is refilled by TMA next
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
        if (issued < len) issue();
      }
    }
    if (stop && lane == 0) *s_abort = 1;
    // never leave the CTA with a TMA still writing into shared memory: raw
    // tiles requested and not yet waited for (these waits ignore the abort
    // flag on purpose)
    for (uint32_t t = ct; t < rt; ++t) mbar_wait(&rfull[t % R], (t / R) & 1, plan);
    __syncwarp();
  } else if (warp == C::kProducerWarp || warp == C::kVProducerWarp) {
    // ------------------------------------------------------------ producers
    // one warp streams K tiles, the other V tiles, each through its own ring,
    // so a full V ring never holds back the next K tile
    const bool is_v = warp == C::kVProducerWarp;
    const int depth = is_v ? NV : NK;
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* empty = is_v ? v_empty : k_empty;
    const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
    const int ring_off = is_v ? C::kVOff : C::kKOff;
    const int width = is_v ? DV : DK;  // elements of a K or V row of one head
    const int tile_bytes = is_v ? C::kTileBytesV : C::kTileBytesK;
    // the whole warp runs the loop; lane p loads the tile's p-th page index and
    // one elected lane issues the copies
    if (elect_one()) {
      prefetch_tmap(tmap);
      if (!is_v && a.q_tma) prefetch_tmap(&tmap_q);
    }
    // L2 priority of the K/V tiles: a request whose rows span several units
    // has every one of them read its K/V tiles, so those lines stay at normal
    // priority for the other units (on the prefix-cached extend batch DRAM
    // traffic fell from 3.4x to 0.96x the algorithmic bytes); K/V that only
    // one unit reads streams through at evict-first priority (verify batches
    // ran 10 % slower at normal priority)
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_reuse = policy_evict_normal();
    uint32_t jt = 0;
    uint32_t armed = 0, armed_ph = 0;
    uint32_t qcount[2] = {0, 0};   // Q tiles issued per X (phase of q_full / q_empty)
    uint32_t qtcount[2] = {0, 0};  // of those, written by the softmax warps (phase of q_written)
    bool stop = false;
    // test support: CTA 0 arms its first K tile but never loads it
    const bool hold_first = !is_v && blockIdx.x == 0 && __ldcg(plan + kHoldLoad) != 0;
    for (int w = blockIdx.x; w < n_units && !stop; w += gridDim.x) {
      const ExtendTile u = load_unit(a, w / a.num_kv_heads);
      const int g = w % a.num_kv_heads;
      const UnitKV ukv = unit_kv(u);
      const int np = a.m.seg_indptr[u.b + 1] - a.m.seg_indptr[u.b];
      const int page_base = a.m.seg_indptr[u.b];
      const bool reused = !a.dplan && (a.m.qo_indptr[u.b + 1] - a.m.qo_indptr[u.b]) * G > kExtendUnitRows;
      const uint64_t pol = reused ? pol_reuse : pol_stream;
      // the unit's Q tiles (K producer), each once the previous unit's last QK
      // on it has finished: by TMA (a box of 128/G tokens x the group's G
      // heads), or forwarded from the softmax warps that wrote it
      auto fill_q = [&]() {
        for (int x = 0; x < 2; ++x) {
          if (!ukv.uses_q(x)) continue;
          if (!mbar_wait_warp(&q_empty[x], (qcount[x] & 1) ^ 1, plan, s_abort)) {
            stop = true;
            break;
          }
          if (q_by_tma(u, x)) {
            if (elect_one()) {
              mbar_arrive_expect_tx(&q_full[x], (uint32_t)C::kQBytes);
              const int tok = a.m.qo_indptr[u.b] + (u.row0 + x * kExtendRows) / G;
#pragma unroll
              for (int cb = 0; cb < C::kColBlocksK; ++cb)
                tma_load_3d(smem + C::kQOff + x * C::kQBytes + cb * (kExtendRows * 128), &tmap_q, cb * 64, g * G,
                            tok, &q_full[x]);
            }
          } else {
            if (!mbar_wait_warp(&q_written[x], qtcount[x] & 1, plan, s_abort)) {
              stop = true;
              break;
            }
            ++qtcount[x];
            if (elect_one()) mbar_arrive(&q_full[x]);
          }
          ++qcount[x];
        }
      };
      if (!is_v) {
        fill_q();
        if (stop) break;
      }
      // e-th KV tile of the unit's sequence
      auto seq_tile = [&](int e) {
        if (!ukv.dual) return ukv.s0 + e;
        const int m = min(ukv.n0, ukv.n1);
        const int step = e < 2 * m ? e >> 1 : e - m;
        const int x = e < 2 * m ? (e & 1) : (ukv.n0 > ukv.n1 ? 0 : 1);
        return ukv.start(x) + step;
      };
      // page indices of 4 consecutive tiles of the sequence: lane 8k + p holds
      // page p of tile e0 + k; the next group is loaded while this one is used
      const int len = ukv.len();
      auto load_group = [&](int e0) {
        const int e = e0 + (lane >> 3), p = lane & 7;
        if (e >= len) return 0;
        const int jj = seq_tile(e);
        return p < np - jj * kPagesPerTile ? __ldg(a.m.seg_indices + page_base + jj * kPagesPerTile + p) : 0;
      };
      int grp = load_group(0);
      int grp_next = load_group(4);
      for (int e = 0; e < len; ++e, ++jt) {
        if (e > 0 && (e & 3) == 0) {
          grp = grp_next;
          grp_next = load_group(e + 4);
        }
        const int j = seq_tile(e);
        const int npg = min(kPagesPerTile, np - j * kPagesPerTile);
        const int st = jt % depth;
        const uint32_t ph = (jt / depth) & 1;
        if (!mbar_wait_warp(&empty[st], ph ^ 1, plan, s_abort)) {
          stop = true;
          break;
        }
        const bool leader = elect_one();
        if (leader) mbar_arrive_expect_tx(&full[st], (uint32_t)(npg * kSegSlots * width * 2));
        uint8_t* dst = smem + ring_off + st * tile_bytes;
#pragma unroll
        for (int p = 0; p < kPagesPerTile; ++p) {
          const int pg = __shfl_sync(0xffffffffu, grp, ((e & 3) << 3) + p);
          if (p < npg && leader && !(hold_first && jt == 0)) {
            for (int cb = 0; cb < width / 64; ++cb)
              tma_load_2d_hint(dst + cb * (kExtendKeys * 128) + p * (kSegSlots * 128), tmap, g * width + cb * 64,
                               pg * kSegSlots, &full[st], pol);
          }
        }
        armed |= 1u << st;
        armed_ph = (armed_ph & ~(1u << st)) | (ph << st);
      }
    }
    if (stop && lane == 0) *s_abort = 1;
    // never leave the CTA with a TMA still writing into shared memory (these
    // waits ignore the abort flag on purpose). The last phase of each Q
    // barrier completes only after every earlier one.
    for (int s2 = 0; s2 < depth; ++s2)
      if (armed & (1u << s2)) mbar_wait(&full[s2], (armed_ph >> s2) & 1, plan);
    for (int x = 0; x < 2; ++x)
      if (qcount[x] > 0) mbar_wait(&q_full[x], (qcount[x] - 1) & 1, plan);
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and one elected lane issues each tcgen05
    // instruction. Descriptors: the start-address field is the low bits, so a
    // byte offset b inside the tile adds b >> 4.
    constexpr uint32_t idesc_qk = C::FP8 ? umma_idesc_f16(kExtendRows, kExtendKeys, false, false)
                                         : umma_idesc_bf16(kExtendRows, kExtendKeys, false, false);
    constexpr uint32_t idesc_pv = C::FP8 ? umma_idesc_f16(kExtendRows, DV, false, true)
                                         : umma_idesc_bf16(kExtendRows, DV, false, true);
    const uint64_t q_desc0 = umma_desc_sw128(smem_base + C::kQOff, 16, 1024);
    const uint64_t k_desc0 = umma_desc_sw128(smem_base + C::kKOff, 16, 1024);
    const uint64_t v_desc0 = umma_desc_sw128(smem_base + C::kVOff, kExtendKeys * 128, 1024);
    uint32_t kt = 0, vt = 0;      // K and V ring tiles consumed so far
    uint32_t tcount[2] = {0, 0};  // tiles processed per X (phase of s_full / p_full)
    uint32_t ucount[2] = {0, 0};  // units that used Q tile X (phase of q_full)
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok && !mbar_wait_warp(bar, parity, plan, s_abort)) ok = false;
      return ok;
    };
    // S_X = Q_qx K^T for the K tile in ring slot ks
    auto issue_qk = [&](int x, int qx, int ks) {
      const uint64_t qd = q_desc0 + (uint32_t)((qx * C::kQBytes) >> 4);
      const uint64_t kd = k_desc0 + (uint32_t)((ks * C::kTileBytesK) >> 4);
#pragma unroll
      for (int kk = 0; kk < DK / 16; ++kk) {
        const uint32_t qo = ((kk >> 2) * (kExtendRows * 128) + (kk & 3) * 32) >> 4;
        const uint32_t ko = ((kk >> 2) * (kExtendKeys * 128) + (kk & 3) * 32) >> 4;
        umma_bf16_warp(tmem + x * 128, qd + qo, kd + ko, idesc_qk, kk > 0);
      }
      umma_commit_warp(&s_full[x]);
    };
    // pv_done is committed only after the last PV of the unit for tile X (the
    // epilogue waits for it); an earlier PV_X is known complete once the
    // s_full commit that follows it has fired
    auto issue_pv = [&](int x, int vs, bool first, bool last) {
      const uint64_t vd = v_desc0 + (uint32_t)((vs * C::kTileBytesV) >> 4);
#pragma unroll
      for (int kk = 0; kk < kExtendKeys / 16; ++kk)
        umma_bf16_ts_warp(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, vd + ((kk * 16 * 128) >> 4), idesc_pv,
                          !(first && kk == 0));
      if (last) umma_commit_warp(&pv_done[x]);
    };
    for (int w = blockIdx.x; w < n_units && ok; w += gridDim.x) {
      const ExtendTile u = load_unit(a, w / a.num_kv_heads);
      const UnitKV ukv = unit_kv(u);
      const int n[2] = {ukv.n0, ukv.n1};
      const int nT = ukv.steps();
      if (nT == 0) continue;
      for (int x = 0; x < 2; ++x)
        if (ukv.uses_q(x) && !wait(&q_full[x], ucount[x] & 1)) break;
      if (!ok) break;
      tc_fence_after();
      if (!ukv.dual) {
        // ---- shared unit: both tiles consume KV tile kv0 + j
        // prologue: S_X of the first tile for both tiles
        if (!wait(&k_full[kt % NK], (kt / NK) & 1)) break;
        tc_fence_after();
        for (int x = 0; x < 2; ++x) {
          if (n[x] == 0) continue;
          issue_qk(x, x, kt % NK);
          if (n[x] == 1) umma_commit_warp(&q_empty[x]);  // the unit's last QK_X: Q_X may be refilled
        }
        umma_commit_warp(&k_empty[kt % NK]);
        ++kt;
        for (int j = 0; j < nT && ok; ++j) {
          const int vs = vt % NV;
          bool v_ready = false, k_ready = false;
          for (int x = 0; x < 2; ++x) {
            if (j >= n[x]) continue;
            if (!wait(&p_full[x], tcount[x] & 1)) break;
            if (!v_ready) {
              if (!wait(&v_full[vs], (vt / NV) & 1)) break;
              v_ready = true;
            }
            // The unit's first PV_X overwrites O_X. The previous unit's epilogue
            // has read it: the softmax warps release p_full of this tile only
            // after finishing that epilogue.
            tc_fence_after();
            issue_pv(x, vs, j == 0, j + 1 == n[x]);
            ++tcount[x];
            if (j + 1 < n[x]) {
              if (!k_ready) {
                if (!wait(&k_full[kt % NK], (kt / NK) & 1)) break;
                tc_fence_after();
                k_ready = true;
              }
              issue_qk(x, x, kt % NK);
              if (j + 2 == n[x]) umma_commit_warp(&q_empty[x]);  // the unit's last QK_X
            }
          }
          if (!ok) break;
          umma_commit_warp(&v_empty[vs]);
          ++vt;
          if (k_ready) {
            umma_commit_warp(&k_empty[kt % NK]);
            ++kt;
          }
        }
      } else {
        // ---- dual unit: each tile its own KV tiles, in ring order A(j), B(j);
        // both tiles read Q tile A, refilled after the unit's last QK
        const int qk_total = n[0] + n[1];
        int qk_issued = 0;
        auto qk_next = [&](int x) {
          if (!wait(&k_full[kt % NK], (kt / NK) & 1)) return false;
          tc_fence_after();
          issue_qk(x, 0, kt % NK);
          umma_commit_warp(&k_empty[kt % NK]);
          ++kt;
          if (++qk_issued == qk_total) umma_commit_warp(&q_empty[0]);
          return true;
        };
        for (int x = 0; x < 2 && ok; ++x)
          if (n[x] > 0) qk_next(x);
        for (int j = 0; j < nT && ok; ++j) {
          for (int x = 0; x < 2; ++x) {
            if (j >= n[x]) continue;
            if (!wait(&p_full[x], tcount[x] & 1)) break;
            if (!wait(&v_full[vt % NV], (vt / NV) & 1)) break;
            tc_fence_after();
            issue_pv(x, vt % NV, j == 0, j + 1 == n[x]);
            umma_commit_warp(&v_empty[vt % NV]);
            ++vt;
            ++tcount[x];
            if (j + 1 < n[x] && !qk_next(x)) break;
          }
        }
        if (!ok) break;
      }
      for (int x = 0; x < 2; ++x)
        if (ukv.uses_q(x)) ++ucount[x];
    }
    if (!ok) {
      if (lane == 0) *s_abort = 1;
      // MMAs issued before the abort finish before the tensor memory they
      // write is freed (this wait ignores the abort flag on purpose)
      umma_commit_warp(mma_drain);
      mbar_wait(mma_drain, 0, plan);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int x = warp >> 2;          // tile of this warpgroup
    const int r = tid & 127;          // row within the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = x * 128, o_col = 256 + x * 128;
    uint8_t* qtile = smem + C::kQOff + x * C::kQBytes;
    uint32_t jt = 0, tcount = 0;
    uint32_t ucount = 0;  // units with work for this tile (phase of pv_done)
    uint32_t du = 0;      // dual units with work (phase of b_done / a_read)
    for (int w = blockIdx.x; w < n_units && !*s_abort; w += gridDim.x) {
      const ExtendTile u = load_unit(a, w / a.num_kv_heads);
      const int g = w % a.num_kv_heads;
      const UnitKV ukv = unit_kv(u);
      const int kb = ukv.start(x);  // this tile's KV tiles: [kb, kb + nX)
      const int nX = ukv.n(x);
      const int nA = ukv.n0;
      const bool split = u.split >= 0;
      const int b = u.b;
      const int q0 = a.m.qo_indptr[b];
      const int qo = a.m.qo_indptr[b + 1] - q0;
      const int L = a.m.kv_len[b];
      const int np = a.m.seg_indptr[b + 1] - a.m.seg_indptr[b];
      const int R = u.row0 + (ukv.dual ? 0 : x * kExtendRows) + r;  // a dual unit's tiles hold the same rows
      const bool valid = R < qo * G;
      // a decode-plan unit holds one 128-row tile of rows (the configuration
      // bounds max_qo_len * group); the rows of a longer request past the
      // tile are recorded and left unwritten
      if (a.dplan && qo * G > kExtendRows && r == 0 && x == 0) record_error(plan, PKV_DEV_QO_TOO_LONG, b);
      const int tok = min(R / G, qo - 1);
      const int limit = L - qo + tok;
      // draft trees: the row's mask word clears the drafts outside its tree
      uint64_t tword = ~0ull;
      int draft0 = 0x3fffffff;  // first draft key (none without a tree)
      if constexpr (EXTRAS) {
        if (a.tree) {
          tword = valid ? a.tree[q0 + R / G] : ~0ull;
          draft0 = L - qo;
          if (qo > 64 && r == 0 && x == 0) record_error(plan, PKV_DEV_TREE_TOO_LONG, b);
        }
      }
      const long long orow = (long long)(q0 + R / G) * a.num_q_heads + g * G + R % G;
      // split units write bf16 partial rows (normalised output) and fp32 LSE that
      // the merge kernel combines across the request's splits
      const long long prow =
          split ? ((long long)a.m.partial_indptr[b] + (long long)u.split * qo + R / G) * a.num_q_heads + g * G + R % G
                : 0;
      if (nX == 0) {
        if (ukv.dual && x == 1) {
          // a dual unit's tile B without KV tiles hands an empty half to tile A
          if (ukv.n0 > 0) {
            s_merge[r] = 0.f;
            s_merge[kExtendRows + r] = 0.f;
            __syncwarp();
            if (lane == 0) mbar_arrive(b_done);
            if (!mbar_wait_warp(a_read, du & 1, plan, s_abort)) {
              *s_abort = 1;
              break;
            }
            ++du;
          }
        } else if (valid) {
          if (split) {
            for (int c = 0; c < DV; c += 8)
              *reinterpret_cast<uint4*>(a.m.partial_o + prow * DV + c) = make_uint4(0, 0, 0, 0);
            a.m.partial_lse[prow] = -INFINITY;
          } else {
            for (int c = 0; c < DV; c += 8)
              *reinterpret_cast<uint4*>(a.out + orow * DV + c) = make_uint4(0, 0, 0, 0);
            // no key: the LSE is the sink's alone
            if (a.lse) a.lse[orow] = (EXTRAS && a.sinks) ? a.sinks[g * G + R % G] : -INFINITY;
          }
        }
        jt += ukv.len();
        continue;
      }
      // Q tiles the producer does not load by TMA: this row of Q -> shared
      // memory (swizzled, K-major); the tile's previous QKs finished before the
      // previous epilogue saw its last PV complete
      if (ukv.uses_q(x) && !q_by_tma(u, x)) {
#pragma unroll
        for (int h = 0; h < DK / 64; ++h) {  // 128 bytes of the row at a time
          uint4 v[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            v[c] = valid ? __ldg(reinterpret_cast<const uint4*>(a.q + orow * DK) + h * 8 + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(qtile + h * (kExtendRows * 128) + r * 128 + ((c ^ (r & 7)) << 4)) =
                C::FP8 ? bf16x8_to_f16x8(v[c]) : v[c];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_written[x]);
      }
      // m_ref: the row's reference in the log2 domain (p = 2^(s * scale - m_ref));
      // l: the row's running sum of p
      float m_ref = 0.f, l = 0.f;
      bool aborted = false;
      for (int jr = 0; jr < nX; ++jr) {
        const int j = kb + jr;                      // absolute KV tile
        const uint32_t jj = jt + ukv.pos(x, jr);    // its place in the V ring sequence
        // warp-uniform waits: every lane of the warp leaves the loop together
        if (!mbar_wait_warp(&s_full[x], tcount & 1, plan, s_abort)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const int key0 = j * kExtendKeys;
        // some keys of this tile are masked for this row: past its limit, or
        // drafts that its tree may hide
        const bool diag = key0 + kExtendKeys - 1 > limit || (EXTRAS && key0 + kExtendKeys > draft0);
        // the request's last page inside this KV tile: zero the V rows past L
        // (done by the first tile that reads this V tile, before its PV)
        if ((ukv.dual || x == 0 || jr >= nA) && np <= (j + 1) * kPagesPerTile && (L % kSegSlots) != 0) {
          const int vs = jj % NV;
          if (!mbar_wait_warp(&v_full[vs], (jj / NV) & 1, plan, s_abort)) {
            aborted = true;
            break;
          }
          const int r0 = L - j * kExtendKeys;
          const int r1 = (np - j * kPagesPerTile) * kSegSlots;
          uint8_t* vt = smem + C::kVOff + vs * C::kTileBytesV;
          const int n16 = (r1 - r0) * C::kColBlocksV * 8;
          for (int i = r; i < n16; i += 128) {
            const int row = r0 + i / (C::kColBlocksV * 8);
            const int rest = i % (C::kColBlocksV * 8);
            *reinterpret_cast<uint4*>(vt + (rest >> 3) * (kExtendKeys * 128) + row * 128 + (rest & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
        uint32_t pk[kExtendKeys / 2];  // P as bf16 pairs, written to TMEM once final
        // S read 64 columns per TMEM wait; masked keys become -inf
        auto load_s = [&](int cc, uint32_t* sr) {
          tmem_ld32(lane_base + s_col + cc * 32, sr);
          tmem_ld32(lane_base + s_col + cc * 32 + 32, sr + 32);
          tmem_wait_ld();
          if (diag) {
            if constexpr (EXTRAS) {
              mask32_bits(sr, visible32(key0 + cc * 32, limit, draft0, tword));
              mask32_bits(sr + 32, visible32(key0 + cc * 32 + 32, limit, draft0, tword));
            } else {
              mask32(sr, key0 + cc * 32, limit);
              mask32(sr + 32, key0 + cc * 32 + 32, limit);
            }
          }
        };
        // P of the tile against the reference; returns the tile's row sum
        auto exp_pass = [&]() {
          const uint64_t nref2 = f2_pack(-m_ref, -m_ref);
          uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
          for (int cc = 0; cc < kExtendKeys / 32; cc += 2) {
            uint32_t sr[64];
            load_s(cc, sr);
            exp32<C::FP8>(sr, sc2, nref2, pk + cc * 16, acc);
            exp32<C::FP8>(sr + 32, sc2, nref2, pk + cc * 16 + 16, acc);
          }
          const uint64_t accs = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
          return f2_lo(accs) + f2_hi(accs);
        };
        float tsum = exp_pass();
        // The tile sum bounds every p of the row: while it is at most 2^16 no p
        // can overflow bf16 P or the fp32 O and l, and the reference (which
        // cancels in O / l) stays put, so the common path needs no row max.
        // Otherwise (a score far above the reference, or a row with no mass
        // yet whose visible scores sit far below it) take the tile's exact
        // max, move the reference, rescale O and l, and run the pass again: S
        // is still intact in TMEM. TMEM loads and stores are warp-collective,
        // so the whole warp takes this branch when any of its rows needs it;
        // the other rows keep their reference and get the same P again. A row
        // that sees no key of this tile (limit < key0) never needs it.
        constexpr float kHigh = C::FP8 ? kSumHighF16 : kSumHigh, kLow = C::FP8 ? kSumLowF16 : kSumLow;
        const bool need = (!(tsum <= kHigh) || (l == 0.f && tsum < kLow)) && limit >= key0;
        if (__any_sync(0xffffffffu, need)) {
          float mx = -INFINITY;
#pragma unroll
          for (int cc = 0; cc < kExtendKeys / 32; cc += 2) {
            uint32_t sr[64];
            load_s(cc, sr);
            mx = max32(sr + 32, max32(sr, mx));
          }
          const float mt = mx * a.scale_log2;
          const bool move = need && mt != -INFINITY && (mt > m_ref || l == 0.f);
          // O_X holds every earlier PV: the s_full commit waited on above was
          // issued after PV_X of the previous tile
          const float alpha = move && l > 0.f ? fast_exp2(m_ref - mt) : 1.f;
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < DV / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(lane_base + o_col + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(lane_base + o_col + c * 32, o);
            }
            tmem_wait_st();
          }
          if (move) {
            l *= alpha;
            m_ref = mt;
          }
          tsum = exp_pass();
        }
        // P overwrites the first half of this tile's S columns
        tmem_st32(lane_base + s_col, pk);
        tmem_st32(lane_base + s_col + 32, pk + 32);
        l += tsum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
        ++tcount;
      }
      if (aborted) {
        *s_abort = 1;
        break;
      }
      // epilogue: O / l once the last PV of this tile has finished
      if (!mbar_wait_warp(&pv_done[x], ucount & 1, plan, s_abort)) {
        *s_abort = 1;
        break;
      }
      ++ucount;
      tc_fence_after();
      if (ukv.dual && x == 1) {
        // dual unit, tile B: hand this half (O in TMEM, m and l in shared
        // memory) to tile A, which merges and writes the row; O_B stays
        // untouched until tile A has read it
        s_merge[r] = m_ref;
        s_merge[kExtendRows + r] = l;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_done);
        if (!mbar_wait_warp(a_read, du & 1, plan, s_abort)) {
          *s_abort = 1;
          break;
        }
        ++du;
        jt += ukv.len();
        continue;
      }
      // weights of this tile's O (and, in a dual unit, of tile B's O), with 1/l folded in
      float wa = 1.f, wb = 0.f;
      if (ukv.dual) {
        if (!mbar_wait_warp(b_done, du & 1, plan, s_abort)) {
          *s_abort = 1;
          break;
        }
        tc_fence_after();
        const float mb = s_merge[r], lb = s_merge[kExtendRows + r];
        const float m = lb > 0.f && (l == 0.f || mb > m_ref) ? mb : m_ref;
        wa = l > 0.f ? fast_exp2(m_ref - m) : 0.f;
        wb = lb > 0.f ? fast_exp2(mb - m) : 0.f;
        l = l * wa + lb * wb;
        m_ref = m;
      }
      float inv = l > 0.f ? 1.f / l : 0.f;
      if constexpr (C::FP8) inv *= a.v_scale;  // V codes times the pool's scale
      if constexpr (EXTRAS) {
        // final rows of a model with sinks: the head's sink joins the normaliser
        if (!split && valid && a.sinks) {
          float lse_s = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
          inv *= sink_factor(lse_s, a.sinks[g * G + R % G]);
        }
      }
      wa *= inv;
      wb *= inv;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + o_col + c * 32, o);
        if (ukv.dual) {
          uint32_t ob[32];
          tmem_ld32(lane_base + 256 + kExtendRows + c * 32, ob);  // tile B's O, same rows
          tmem_wait_ld();
          // tile B's O counts only with a nonzero weight: without KV tiles its
          // TMEM columns may hold anything (even NaN patterns)
          const bool use_b = wb != 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float fb = use_b ? __uint_as_float(ob[i]) * wb : 0.f;
            o[i] = __float_as_uint(__uint_as_float(o[i]) * wa + fb);
          }
        } else {
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * wa);
        }
        // the rows of a warp are scattered (one 256- or 128-byte row per lane),
        // so each store instruction costs one transaction per lane: 32-byte
        // stores halve their number (partial rows live in the 256-byte aligned
        // workspace; out only when the caller's buffer is 32-byte aligned)
        if (valid) {
          // the output row, or (split units) a bf16 partial row of the same layout
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = pack_bf16(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
          {
            uint16_t* dst = split ? a.m.partial_o + prow * DV + c * 32 : a.out + orow * DV + c * 32;
            if (split || a.out_32B) {
              st_global_32B(dst, v);
              st_global_32B(dst + 16, v + 8);
            } else {
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<uint4*>(dst + 2 * i) = make_uint4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
          }
        }
      }
      tc_fence_before();
      if (ukv.dual) {
        // tile B's O and (m, l) have been read
        __syncwarp();
        if (lane == 0) mbar_arrive(a_read);
        ++du;
      }
      if (valid) {
        float lse_v = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        if constexpr (EXTRAS) {
          if (!split && a.sinks) (void)sink_factor(lse_v, a.sinks[g * G + R % G]);
        }
        if (split)
          a.m.partial_lse[prow] = lse_v;
        else if (a.lse)
          a.lse[orow] = lse_v;
      }
      jt += ukv.len();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <class C>
int run_extend(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
               float v_scale, void* out, float* lse, cudaStream_t st, bool dplan) {
  CUtensorMap tk, tv;
  const uint64_t inner_k = (uint64_t)c.cfg.num_kv_heads * C::DK;
  const uint64_t inner_v = (uint64_t)c.cfg.num_kv_heads * C::DV;
  const uint64_t slots = (uint64_t)c.cfg.num_pages * c.cfg.page_size;
  // boxes of 16 slots x 128 bytes: 64 bf16 elements, or 128 E4M3 codes (the
  // whole row of a 128-wide head)
  const CUtensorMapDataType dt = C::FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t esz = C::FP8 ? 1 : 2;
  // L2 fills no wider than one head's row of an E4M3 pool (128 bytes)
  const CUtensorMapL2promotion promo = C::FP8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  if (encode_tmap_2d(&tk, dt, const_cast<void*>(k_pool), inner_k, slots, inner_k * esz, 128 / esz, kSegSlots,
                     CU_TENSOR_MAP_SWIZZLE_128B, promo) != PKV_OK)
    return PKV_ERR_CUDA;
  if (encode_tmap_2d(&tv, dt, const_cast<void*>(v_pool), inner_v, slots, inner_v * esz, 128 / esz, kSegSlots,
                     CU_TENSOR_MAP_SWIZZLE_128B, promo) != PKV_OK)
    return PKV_ERR_CUDA;
  ExtendArgs a;
  a.m = make_meta(c);
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.num_q_heads = c.cfg.num_q_heads;
  a.num_kv_heads = c.cfg.num_kv_heads;
  a.group = c.cfg.num_q_heads / c.cfg.num_kv_heads;
  // E4M3 codes are widened exactly: the K pool's scale joins the score scale
  // and the V pool's scale multiplies the output
  a.scale_log2 = sm_scale * (C::FP8 ? k_scale : 1.f) * kLog2e;
  a.v_scale = C::FP8 ? v_scale : 1.f;
  a.out_32B = (reinterpret_cast<uintptr_t>(out) & 31) == 0 ? 1 : 0;
  a.tree = active_tree(c);
  a.sinks = c.sinks;
  a.dplan = dplan ? 1 : 0;
  // Q as [tokens][heads][head_dim]: a box of 64 elements x G heads x 128/G
  // tokens is one 128-row tile column block, rows ordered (token, head) like
  // the tile's rows. The token extent only bounds the map; the kernel loads a
  // box only when all its tokens are inside the batch.
  CUtensorMap tq;
  memset(&tq, 0, sizeof(tq));
  a.q_tma = 0;
  a.q_box_tokens = 0;
  // (E4M3 pools: the softmax warps copy Q, converting it to f16 on the way)
  if (!C::FP8 && kExtendRows % a.group == 0) {
    const uint32_t box_tok = kExtendRows / a.group;
    const uint64_t tokens = (uint64_t)(c.cfg.max_q_tokens > (int)box_tok ? c.cfg.max_q_tokens : (int)box_tok);
    if (encode_tmap_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(q), C::DK,
                       (uint64_t)c.cfg.num_q_heads, tokens, (uint64_t)C::DK * 2,
                       (uint64_t)c.cfg.num_q_heads * C::DK * 2, 64, (uint32_t)a.group, box_tok,
                       CU_TENSOR_MAP_SWIZZLE_128B) != PKV_OK)
      return PKV_ERR_CUDA;
    a.q_tma = 1;
    a.q_box_tokens = (int)box_tok;
  }
  auto kernel = (a.tree || a.sinks) ? extend_tc_kernel<C, true> : extend_tc_kernel<C, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (launch_pdl(kernel, dim3(c.extend_ctas), dim3(C::kThreads), C::kSmemBytes, st, tk, tv, tq, a) != cudaSuccess)
    return PKV_ERR_CUDA;
  // the decode plan's split requests are merged by the decode path's merge
  // (its split counts); on the extend path, the requests whose rows fit one
  // unit were split along their KV range
  if (dplan) return launch_split_merge(c, out, lse, c.cfg.max_qo_len * a.group, false, st);
  return launch_split_merge(c, out, lse, kExtendUnitRows, true, st);
}

int run_tc(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
           float v_scale, void* out, float* lse, cudaStream_t st, bool dplan) {
  if (c.cfg.kv_dtype == PKV_KV_FP8_E4M3) {
    // E4M3 pools (128-wide heads): f16 operand rings of two K and two V tiles,
    // one raw tile of codes in flight for each
    if (c.cfg.head_dim != 128) return PKV_ERR_UNSUPPORTED;
    return run_extend<ExtCfg<128, 128, 2, 2, true, 1, 1>>(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out,
                                                          lse, st, dplan);
  }
  if (c.cfg.head_dim == 128)
    return run_extend<ExtCfg<128, 128, 3, 2>>(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out, lse, st, dplan);
  if (c.cfg.head_dim == 64)
    return run_extend<ExtCfg<64, 64, 4, 4>>(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out, lse, st, dplan);
  // 192-wide Q/K heads with 128-wide V heads: two 48 KB Q tiles, so the rings
  // hold two 48 KB K tiles and one 32 KB V tile
  if (c.cfg.head_dim == 192)
    return run_extend<ExtCfg<192, 128, 1, 2>>(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out, lse, st, dplan);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace

int launch_extend(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
                  float v_scale, void* out, float* lse, cudaStream_t st) {
  return run_tc(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out, lse, st, false);
}

int launch_decode_tc(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, float k_scale,
                     float v_scale, void* out, float* lse, cudaStream_t st) {
  return run_tc(c, q, k_pool, v_pool, sm_scale, k_scale, v_scale, out, lse, st, true);
}

}  // namespace pkv
