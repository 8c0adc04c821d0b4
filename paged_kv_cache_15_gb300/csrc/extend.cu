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
// reference m_ref stays put (see the softmax role).
constexpr float kSumHigh = 65536.0f;               // 2^16
constexpr float kSumLow = 5.421010862427522e-20f;  // 2^-64

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

// p = exp2(s * scale - ref) for 32 raw scores: packed bf16 pairs into pk,
// running sums in four packed accumulators.
__device__ __forceinline__ void exp32(const uint32_t* sr, uint64_t sc2, uint64_t nref2, uint32_t* pk, uint64_t* acc) {
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const uint64_t x = f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, nref2);
    const float p0 = fast_exp2(f2_lo(x)), p1 = fast_exp2(f2_hi(x));
    acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(p0, p1));
    pk[c >> 1] = pack_bf16(p0, p1);
  }
}

template <int D_, int NK_, int NV_>
struct ExtCfg {
  static constexpr int D = D_;
  static constexpr int NK = NK_;  // K ring depth
  static constexpr int NV = NV_;  // V ring depth
  static constexpr int kThreads = 352;
  static constexpr int kProducerWarp = 8;   // K tiles
  static constexpr int kMmaWarp = 9;
  static constexpr int kVProducerWarp = 10;  // V tiles
  static constexpr int kColBlocks = D / 64;               // 128-byte swizzle spans per row
  static constexpr int kQBytes = kExtendRows * D * 2;     // one Q tile: [cb][128 rows][128 B]
  static constexpr int kTileBytes = kExtendKeys * D * 2;  // one K or V tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kQBytes;
  static constexpr int kVOff = kKOff + NK * kTileBytes;
  static constexpr int kBarOff = kVOff + NV * kTileBytes;
  static constexpr int kNumBars = 2 + 2 * NK + 2 * NV + 6 + 4;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kAbortOff = kTmemSlotOff + 8;
  static constexpr int kSmemBytes = kAbortOff + 8 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(D <= 128, "O needs at most 128 TMEM columns per tile");
};

struct ExtendArgs {
  Meta m;
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  int num_q_heads, num_kv_heads, group;
  float scale_log2;
  int q_tma;         // 1 when the group divides 128: a Q tile is one TMA box of 128/G tokens x G heads
  int q_box_tokens;  // 128 / group
};

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1) extend_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                   const __grid_constant__ CUtensorMap tmap_v,
                                                                   const __grid_constant__ CUtensorMap tmap_q,
                                                                   ExtendArgs a) {
  constexpr int D = C::D;
  constexpr int NK = C::NK, NV = C::NV;
  constexpr int kPagesPerTile = kExtendKeys / kPageSize;
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
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  // K/V stages start as zeros so rows of a partly loaded tile are finite
  for (int i = tid; i < (NK + NV) * C::kTileBytes / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(smem + C::kKOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // launched with programmatic serialization: metadata, Q and the K/V this
  // step stored are only read after the preceding grid has finished
  pdl_wait();

  const int n_units = plan[kExtendTiles] * a.num_kv_heads;
  const int G = a.group;
  const uint32_t smem_base = smem_u32(smem);
  const int total_q = plan[kTotalQ];
  // Tile X of unit u takes its Q by TMA when the box of 128/G tokens lies
  // inside the batch's tokens (never past the end of the caller's q buffer);
  // otherwise the softmax warps write it.
  auto q_by_tma = [&](const ExtendTile& u, int x) {
    return a.q_tma != 0 && a.m.qo_indptr[u.b] + (u.row0 + x * kExtendRows) / G + a.q_box_tokens <= total_q;
  };

  if (warp == C::kProducerWarp || warp == C::kVProducerWarp) {
    // ------------------------------------------------------------ producers
    // one warp streams K tiles, the other V tiles, each through its own ring,
    // so a full V ring never holds back the next K tile
    const bool is_v = warp == C::kVProducerWarp;
    const int depth = is_v ? NV : NK;
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* empty = is_v ? v_empty : k_empty;
    const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
    const int ring_off = is_v ? C::kVOff : C::kKOff;
    // the whole warp runs the loop; lane p loads the tile's p-th page index and
    // one elected lane issues the copies
    if (elect_one()) {
      prefetch_tmap(tmap);
      if (!is_v && a.q_tma) prefetch_tmap(&tmap_q);
    }
    const uint64_t pol = policy_evict_first();
    uint32_t jt = 0;
    uint32_t armed = 0, armed_ph = 0;
    uint32_t qcount[2] = {0, 0};   // Q tiles issued per X (phase of q_full / q_empty)
    uint32_t qtcount[2] = {0, 0};  // of those, written by the softmax warps (phase of q_written)
    bool stop = false;
    for (int w = blockIdx.x; w < n_units && !stop; w += gridDim.x) {
      const ExtendTile u = a.m.extend_tiles[w / a.num_kv_heads];
      const int g = w % a.num_kv_heads;
      const int kend = min(u.kv1, max(u.kv_a, u.kv_b));
      const int np = a.m.kv_indptr[u.b + 1] - a.m.kv_indptr[u.b];
      const int page_base = a.m.kv_indptr[u.b];
      if (!is_v) {
        // the unit's Q tiles, each once the previous unit's last QK on it has
        // finished: by TMA (a box of 128/G tokens x the group's G heads), or
        // forwarded from the softmax warps that wrote it
        for (int x = 0; x < 2; ++x) {
          if (min(u.kv1, x == 0 ? u.kv_a : u.kv_b) <= u.kv0) continue;  // no KV tile for X
          if (!mbar_wait_warp(&q_empty[x], (qcount[x] & 1) ^ 1, plan, s_abort)) {
            stop = true;
            break;
          }
          if (q_by_tma(u, x)) {
            if (elect_one()) {
              mbar_arrive_expect_tx(&q_full[x], (uint32_t)C::kQBytes);
              const int tok = a.m.qo_indptr[u.b] + (u.row0 + x * kExtendRows) / G;
#pragma unroll
              for (int cb = 0; cb < C::kColBlocks; ++cb)
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
        if (stop) break;
      }
      for (int j = u.kv0; j < kend; ++j, ++jt) {
        const int npg = min(kPagesPerTile, np - j * kPagesPerTile);
        const int my_pg = lane < npg ? __ldg(a.m.kv_indices + page_base + j * kPagesPerTile + lane) : 0;
        const int st = jt % depth;
        const uint32_t ph = (jt / depth) & 1;
        if (!mbar_wait_warp(&empty[st], ph ^ 1, plan, s_abort)) {
          stop = true;
          break;
        }
        const bool leader = elect_one();
        if (leader) mbar_arrive_expect_tx(&full[st], (uint32_t)(npg * kPageSize * D * 2));
        uint8_t* dst = smem + ring_off + st * C::kTileBytes;
#pragma unroll
        for (int p = 0; p < kPagesPerTile; ++p) {
          const int pg = __shfl_sync(0xffffffffu, my_pg, p);
          if (p < npg && leader) {
#pragma unroll
            for (int cb = 0; cb < C::kColBlocks; ++cb)
              tma_load_2d_hint(dst + cb * (kExtendKeys * 128) + p * (kPageSize * 128), tmap, g * D + cb * 64,
                               pg * kPageSize, &full[st], pol);
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
    constexpr uint32_t idesc_qk = umma_idesc_bf16(kExtendRows, kExtendKeys, false, false);
    constexpr uint32_t idesc_pv = umma_idesc_bf16(kExtendRows, D, false, true);
    const uint64_t q_desc0 = umma_desc_sw128(smem_base + C::kQOff, 16, 1024);
    const uint64_t k_desc0 = umma_desc_sw128(smem_base + C::kKOff, 16, 1024);
    const uint64_t v_desc0 = umma_desc_sw128(smem_base + C::kVOff, kExtendKeys * 128, 1024);
    uint32_t jt = 0;
    uint32_t tcount[2] = {0, 0};  // tiles processed per X (phase of s_full / p_full)
    uint32_t ucount[2] = {0, 0};  // units processed per X (phase of q_full)
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      if (ok && !mbar_wait_warp(bar, parity, plan, s_abort)) ok = false;
      return ok;
    };
    auto issue_qk = [&](int x, int ks) {
      const uint64_t qd = q_desc0 + (uint32_t)((x * C::kQBytes) >> 4);
      const uint64_t kd = k_desc0 + (uint32_t)((ks * C::kTileBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
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
      const uint64_t vd = v_desc0 + (uint32_t)((vs * C::kTileBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < kExtendKeys / 16; ++kk)
        umma_bf16_ts_warp(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, vd + ((kk * 16 * 128) >> 4), idesc_pv,
                          !(first && kk == 0));
      if (last) umma_commit_warp(&pv_done[x]);
    };
    for (int w = blockIdx.x; w < n_units && ok; w += gridDim.x) {
      const ExtendTile u = a.m.extend_tiles[w / a.num_kv_heads];
      // tiles [kb, kb + n[x]) of this unit's KV range for tile X
      const int kb = u.kv0;
      const int n[2] = {max(0, min(u.kv1, u.kv_a) - kb), max(0, min(u.kv1, u.kv_b) - kb)};
      const int nT = max(n[0], n[1]);
      if (nT == 0) continue;
      for (int x = 0; x < 2; ++x)
        if (n[x] > 0 && !wait(&q_full[x], ucount[x] & 1)) break;
      if (!ok) break;
      tc_fence_after();
      // prologue: S_X of the first tile for both tiles
      if (!wait(&k_full[jt % NK], (jt / NK) & 1)) break;
      tc_fence_after();
      for (int x = 0; x < 2; ++x) {
        if (n[x] == 0) continue;
        issue_qk(x, jt % NK);
        if (n[x] == 1) umma_commit_warp(&q_empty[x]);  // the unit's last QK_X: Q_X may be refilled
      }
      umma_commit_warp(&k_empty[jt % NK]);
      for (int j = 0; j < nT && ok; ++j) {
        const uint32_t jj = jt + j;
        const int vs = jj % NV;
        bool v_ready = false, k_ready = false;
        for (int x = 0; x < 2; ++x) {
          if (j >= n[x]) continue;
          if (!wait(&p_full[x], tcount[x] & 1)) break;
          if (!v_ready) {
            if (!wait(&v_full[vs], (jj / NV) & 1)) break;
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
              if (!wait(&k_full[(jj + 1) % NK], ((jj + 1) / NK) & 1)) break;
              tc_fence_after();
              k_ready = true;
            }
            issue_qk(x, (jj + 1) % NK);
            if (j + 2 == n[x]) umma_commit_warp(&q_empty[x]);  // the unit's last QK_X
          }
        }
        if (!ok) break;
        umma_commit_warp(&v_empty[vs]);
        if (k_ready) umma_commit_warp(&k_empty[(jj + 1) % NK]);
      }
      jt += nT;
      for (int x = 0; x < 2; ++x)
        if (n[x] > 0) ++ucount[x];
    }
    if (!ok && lane == 0) *s_abort = 1;
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int x = warp >> 2;          // tile of this warpgroup
    const int r = tid & 127;          // row within the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = x * 128, o_col = 256 + x * 128;
    uint8_t* qtile = smem + C::kQOff + x * C::kQBytes;
    uint32_t jt = 0, tcount = 0;
    uint32_t ucount = 0;  // units with work for this tile (phase of pv_done)
    for (int w = blockIdx.x; w < n_units && !*s_abort; w += gridDim.x) {
      const ExtendTile u = a.m.extend_tiles[w / a.num_kv_heads];
      const int g = w % a.num_kv_heads;
      const int kb = u.kv0;
      const int endA = min(u.kv1, u.kv_a);                        // tile A: KV tiles [kb, endA)
      const int endX = min(u.kv1, x == 0 ? u.kv_a : u.kv_b);      // this warpgroup's tile
      const int nX = max(0, endX - kb);
      const int nT = max(0, min(u.kv1, max(u.kv_a, u.kv_b)) - kb);
      const bool split = u.split >= 0;
      const int b = u.b;
      const int q0 = a.m.qo_indptr[b];
      const int qo = a.m.qo_indptr[b + 1] - q0;
      const int L = a.m.kv_len[b];
      const int np = a.m.kv_indptr[b + 1] - a.m.kv_indptr[b];
      const int R = u.row0 + x * kExtendRows + r;
      const bool valid = R < qo * G;
      const int tok = min(R / G, qo - 1);
      const int limit = L - qo + tok;
      const long long orow = (long long)(q0 + R / G) * a.num_q_heads + g * G + R % G;
      // split units write fp32 partial rows (normalised output and LSE) that
      // the merge kernel combines across the request's splits
      const long long prow =
          split ? ((long long)a.m.partial_indptr[b] + (long long)u.split * qo + R / G) * a.num_q_heads + g * G + R % G
                : 0;
      if (nX == 0) {
        if (valid) {
          if (split) {
            for (int c = 0; c < D; c += 4)
              *reinterpret_cast<float4*>(a.m.partial_o + prow * D + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            a.m.partial_lse[prow] = -INFINITY;
          } else {
            for (int c = 0; c < D; c += 8)
              *reinterpret_cast<uint4*>(a.out + orow * D + c) = make_uint4(0, 0, 0, 0);
            if (a.lse) a.lse[orow] = -INFINITY;
          }
        }
        jt += nT;
        continue;
      }
      // Q tiles the producer does not load by TMA: this row of Q -> shared
      // memory (swizzled, K-major); the tile's previous QKs finished before the
      // previous epilogue saw its last PV complete
      if (!q_by_tma(u, x)) {
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {  // 128 bytes of the row at a time
          uint4 v[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            v[c] = valid ? __ldg(reinterpret_cast<const uint4*>(a.q + orow * D) + h * 8 + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(qtile + h * (kExtendRows * 128) + r * 128 + ((c ^ (r & 7)) << 4)) = v[c];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_written[x]);
      }
      // m_ref: the row's reference in the log2 domain (p = 2^(s * scale - m_ref));
      // l: the row's running sum of p
      float m_ref = 0.f, l = 0.f;
      bool aborted = false;
      for (int j = kb; j < endX; ++j) {
        const uint32_t jj = jt + (j - kb);
        // warp-uniform waits: every lane of the warp leaves the loop together
        if (!mbar_wait_warp(&s_full[x], tcount & 1, plan, s_abort)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const int key0 = j * kExtendKeys;
        const bool diag = key0 + kExtendKeys - 1 > limit;  // some keys of this tile are masked for this row
        // the request's last page inside this KV tile: zero the V rows past L
        // (done by the first tile that reads this V tile, before its PV)
        if ((x == 0 || j >= endA) && np <= (j + 1) * kPagesPerTile && (L % kPageSize) != 0) {
          const int vs = jj % NV;
          if (!mbar_wait_warp(&v_full[vs], (jj / NV) & 1, plan, s_abort)) {
            aborted = true;
            break;
          }
          const int r0 = L - j * kExtendKeys;
          const int r1 = (np - j * kPagesPerTile) * kPageSize;
          uint8_t* vt = smem + C::kVOff + vs * C::kTileBytes;
          const int n16 = (r1 - r0) * C::kColBlocks * 8;
          for (int i = r; i < n16; i += 128) {
            const int row = r0 + i / (C::kColBlocks * 8);
            const int rest = i % (C::kColBlocks * 8);
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
            mask32(sr, key0 + cc * 32, limit);
            mask32(sr + 32, key0 + cc * 32 + 32, limit);
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
            exp32(sr, sc2, nref2, pk + cc * 16, acc);
            exp32(sr + 32, sc2, nref2, pk + cc * 16 + 16, acc);
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
        const bool need = (!(tsum <= kSumHigh) || (l == 0.f && tsum < kSumLow)) && limit >= key0;
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
            for (int c = 0; c < D / 32; ++c) {
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
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + o_col + c * 32, o);
        tmem_wait_ld();
        if (valid) {
          if (split) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(a.m.partial_o + prow * D + c * 32 + i) =
                  make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                              __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
          } else {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[i + 0]) * inv, __uint_as_float(o[i + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
              *reinterpret_cast<uint4*>(a.out + orow * D + c * 32 + i) = v;
            }
          }
        }
      }
      tc_fence_before();
      if (valid) {
        const float lse_v = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        if (split)
          a.m.partial_lse[prow] = lse_v;
        else if (a.lse)
          a.lse[orow] = lse_v;
      }
      jt += nT;
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
int run_extend(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, void* out, float* lse,
               cudaStream_t st) {
  CUtensorMap tk, tv;
  const uint64_t inner = (uint64_t)c.cfg.num_kv_heads * C::D;
  const uint64_t slots = (uint64_t)c.cfg.num_pages * c.cfg.page_size;
  if (encode_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(k_pool), inner, slots, inner * 2, 64,
                     kPageSize, CU_TENSOR_MAP_SWIZZLE_128B) != PKV_OK)
    return PKV_ERR_CUDA;
  if (encode_tmap_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(v_pool), inner, slots, inner * 2, 64,
                     kPageSize, CU_TENSOR_MAP_SWIZZLE_128B) != PKV_OK)
    return PKV_ERR_CUDA;
  ExtendArgs a;
  a.m = make_meta(c);
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.num_q_heads = c.cfg.num_q_heads;
  a.num_kv_heads = c.cfg.num_kv_heads;
  a.group = c.cfg.num_q_heads / c.cfg.num_kv_heads;
  a.scale_log2 = sm_scale * kLog2e;
  // Q as [tokens][heads][head_dim]: a box of 64 elements x G heads x 128/G
  // tokens is one 128-row tile column block, rows ordered (token, head) like
  // the tile's rows. The token extent only bounds the map; the kernel loads a
  // box only when all its tokens are inside the batch.
  CUtensorMap tq;
  memset(&tq, 0, sizeof(tq));
  a.q_tma = 0;
  a.q_box_tokens = 0;
  if (kExtendRows % a.group == 0) {
    const uint32_t box_tok = kExtendRows / a.group;
    const uint64_t tokens = (uint64_t)(c.cfg.max_q_tokens > (int)box_tok ? c.cfg.max_q_tokens : (int)box_tok);
    if (encode_tmap_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(q), C::D,
                       (uint64_t)c.cfg.num_q_heads, tokens, (uint64_t)C::D * 2,
                       (uint64_t)c.cfg.num_q_heads * C::D * 2, 64, (uint32_t)a.group, box_tok,
                       CU_TENSOR_MAP_SWIZZLE_128B) != PKV_OK)
      return PKV_ERR_CUDA;
    a.q_tma = 1;
    a.q_box_tokens = (int)box_tok;
  }
  if (cudaFuncSetAttribute(extend_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  if (launch_pdl(extend_tc_kernel<C>, dim3(c.extend_ctas), dim3(C::kThreads), C::kSmemBytes, st, tk, tv, tq, a) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  // requests whose rows fit one unit were split along their KV range
  return launch_split_merge(c, out, lse, kExtendUnitRows, true, st);
}

}  // namespace

int launch_extend(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, void* out,
                  float* lse, cudaStream_t st) {
  if (c.cfg.head_dim == 128) return run_extend<ExtCfg<128, 3, 2>>(c, q, k_pool, v_pool, sm_scale, out, lse, st);
  if (c.cfg.head_dim == 64) return run_extend<ExtCfg<64, 4, 4>>(c, q, k_pool, v_pool, sm_scale, out, lse, st);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
