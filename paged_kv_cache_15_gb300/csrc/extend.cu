// forward_extend on the 5th-generation tensor cores ("--attention-backend",
// section "What an attention backend is": forward_extend runs prefill; section
// "Two backends in one server": prefill reads long query blocks and is bound by
// compute). The same kernel runs target-verify on the prefill path ("[SGLang]
// Hybrid Attention", section "_select_backend: ForwardMode 기반 동적 전환").
//
// One work unit = (request, 128-row query tile, KV head). A row is a
// (query token, head-in-group) pair, so the GQA group shares every K/V tile.
// The query block attends to the cached prefix plus the new tokens with the
// causal rule "row of token i sees keys 0 .. P + i" (P = cached prefix).
//
// Warp roles (192 threads, one CTA per SM, persistent over units):
//   warps 0-3  softmax: thread r owns row r (TMEM lane r). Reads S from TMEM,
//              masks, keeps the running max / sum in the log2 domain, writes
//              P (bf16) to shared memory, rescales O in TMEM when the max grows
//              by more than 2^8 (otherwise the stale max is kept: the result is
//              the same, the factor cancels in O / l), and writes the output.
//   warp 4     producer: copies the unit's Q rows into shared memory, then
//              gathers K/V pages with TMA (16-token boxes, 128-byte swizzle)
//              into a 2-stage ring.
//   warp 5     MMA: allocates 512 TMEM columns and issues tcgen05.mma
//              (kind::f16, bf16 in, fp32 accumulate):
//                S[slot] = Q K^T   (M=128 rows, N=128 keys, K=head_dim)
//                O      += P V     (M=128 rows, N=head_dim, K=128 keys)
//              QK of tile j is issued before PV of tile j-1, so the tensor
//              core computes the next scores while the softmax warps work.
// TMEM: S double buffer (columns 0-127, 128-255), O (columns 256-).
#include <math.h>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay below 2^8

template <int D_>
struct ExtCfg {
  static constexpr int D = D_;
  static constexpr int kThreads = 192;
  static constexpr int kColBlocks = D / 64;                 // 128-byte swizzle spans per row
  static constexpr int kQBytes = kExtendRows * D * 2;       // [cb][128 rows][128 B]
  static constexpr int kTileBytes = kExtendKeys * D * 2;    // K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kPBytes = kExtendRows * kExtendKeys * 2;  // [2][128 rows][128 B]
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQBytes;
  static constexpr int kPOff = kKVOff + 2 * kStageBytes;
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  static constexpr int kNumBars = 15;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kAbortOff = kTmemSlotOff + 8;
  static constexpr int kSmemBytes = kAbortOff + 8 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct ExtendArgs {
  Meta m;
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  int num_q_heads, num_kv_heads, group;
  float scale_log2;
};

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1) extend_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                   const __grid_constant__ CUtensorMap tmap_v,
                                                                   ExtendArgs a) {
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;   // [2]
  uint64_t* kv_empty = bars + 4;  // [2]
  uint64_t* s_full = bars + 6;    // [2]
  uint64_t* s_free = bars + 8;    // [2]
  uint64_t* p_full = bars + 10;   // [2]
  uint64_t* p_free = bars + 12;   // [2]
  uint64_t* o_free = bars + 14;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kTmemSlotOff);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* plan = a.m.plan;

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 128);
      mbar_init(&p_full[s], 128);
      mbar_init(&p_free[s], 1);
    }
    mbar_init(o_free, 128);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  // K/V stages start as zeros so rows of a partly loaded tile are finite
  for (int i = tid; i < 2 * C::kStageBytes / 16; i += C::kThreads)
    reinterpret_cast<uint4*>(smem + C::kKVOff)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  const int n_units = a.m.plan[kExtendTiles] * a.num_kv_heads;
  const int G = a.group;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
    }
    uint32_t jt = 0, uq = 0;
    uint32_t armed = 0, armed_ph = 0;
    for (int w = blockIdx.x; w < n_units && !*s_abort; w += gridDim.x) {
      const ExtendTile tile = a.m.extend_tiles[w / a.num_kv_heads];
      const int g = w % a.num_kv_heads;
      const int nkv = tile.kv_tiles;
      if (nkv == 0) continue;
      const int b = tile.b;
      const int q0 = a.m.qo_indptr[b];
      const int rows_valid = (a.m.qo_indptr[b + 1] - q0) * G;
      const int np = a.m.kv_indptr[b + 1] - a.m.kv_indptr[b];
      const int page_base = a.m.kv_indptr[b];
      if (!mbar_wait(q_empty, (uq & 1) ^ 1, plan)) {
        *s_abort = 1;
        break;
      }
      // Q rows -> shared memory (swizzled K-major), 16-byte chunks, two rows per warp pass
      constexpr int kChunksPerRow = D / 8;
      for (int it = 0; it < kExtendRows * kChunksPerRow / 32; it += 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ci = (it + u) * 32 + lane;
          const int row = ci / kChunksPerRow, c = ci % kChunksPerRow;
          const int R = tile.row0 + row;
          v[u] = make_uint4(0, 0, 0, 0);
          if (R < rows_valid) {
            const long long src = ((long long)(q0 + R / G) * a.num_q_heads + g * G + R % G) * D + c * 8;
            v[u] = __ldg(reinterpret_cast<const uint4*>(a.q + src));
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ci = (it + u) * 32 + lane;
          const int row = ci / kChunksPerRow, c = ci % kChunksPerRow;
          *reinterpret_cast<uint4*>(smem + C::kQOff + (c >> 3) * (kExtendRows * 128) + row * 128 +
                                    (((c & 7) ^ (row & 7)) << 4)) = v[u];
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(q_full);
        for (int j = 0; j < nkv; ++j, ++jt) {
          const int slot = jt & 1;
          if (!mbar_wait(&kv_empty[slot], ((jt >> 1) & 1) ^ 1, plan)) {
            *s_abort = 1;
            break;
          }
          const int npg = min(kExtendKeys / kPageSize, np - j * (kExtendKeys / kPageSize));
          mbar_arrive_expect_tx(&kv_full[slot], (uint32_t)(npg * kPageSize * D * 2 * 2));
          uint8_t* kd = smem + C::kKVOff + slot * C::kStageBytes;
          uint8_t* vd = kd + C::kTileBytes;
          for (int p = 0; p < npg; ++p) {
            const int page = a.m.kv_indices[page_base + j * (kExtendKeys / kPageSize) + p];
#pragma unroll
            for (int cb = 0; cb < C::kColBlocks; ++cb) {
              const int off = cb * (kExtendKeys * 128) + p * (kPageSize * 128);
              tma_load_2d_hint(kd + off, &tmap_k, g * D + cb * 64, page * kPageSize, &kv_full[slot], pol);
              tma_load_2d_hint(vd + off, &tmap_v, g * D + cb * 64, page * kPageSize, &kv_full[slot], pol);
            }
          }
          armed |= 1u << slot;
          armed_ph = (armed_ph & ~(1u << slot)) | (((jt >> 1) & 1) << slot);
        }
      } else {
        jt += nkv;
      }
      jt = __shfl_sync(0xffffffffu, jt, 0);
      ++uq;
    }
    if (lane == 0)
      for (int s = 0; s < 2; ++s)
        if (armed & (1u << s)) mbar_wait(&kv_full[s], (armed_ph >> s) & 1, plan);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kExtendRows, kExtendKeys, false, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kExtendRows, D, false, true);
      const uint32_t q_addr = smem_base + C::kQOff;
      uint32_t jt = 0, uq = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t jtp, bool first) -> bool {
        const int slot = jtp & 1;
        if (!mbar_wait(&p_full[slot], (jtp >> 1) & 1, plan)) return false;
        if (first && !mbar_wait(o_free, (uq & 1) ^ 1, plan)) return false;
        tc_fence_after();
        const uint32_t p_addr = smem_base + C::kPOff + slot * C::kPBytes;
        const uint32_t v_addr = smem_base + C::kKVOff + slot * C::kStageBytes + C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kExtendKeys / 16; ++kk) {
          const uint64_t pd = umma_desc_sw128(p_addr + (kk >> 2) * (kExtendRows * 128) + (kk & 3) * 32, 16, 1024);
          const uint64_t vd = umma_desc_sw128(v_addr + kk * 16 * 128, kExtendKeys * 128, 1024);
          umma_bf16(tmem + C::kOCol, pd, vd, idesc_pv, !(first && kk == 0));
        }
        umma_commit(&p_free[slot]);
        umma_commit(&kv_empty[slot]);
        return true;
      };
      for (int w = blockIdx.x; w < n_units && ok && !*s_abort; w += gridDim.x) {
        const ExtendTile tile = a.m.extend_tiles[w / a.num_kv_heads];
        const int nkv = tile.kv_tiles;
        if (nkv == 0) continue;
        if (!mbar_wait(q_full, uq & 1, plan)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int j = 0; j < nkv; ++j, ++jt) {
          const int slot = jt & 1;
          const uint32_t ph = (jt >> 1) & 1;
          if (!mbar_wait(&kv_full[slot], ph, plan) || !mbar_wait(&s_free[slot], ph ^ 1, plan)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_addr = smem_base + C::kKVOff + slot * C::kStageBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (kExtendRows * 128) + (kk & 3) * 32;
            const uint64_t qd = umma_desc_sw128(q_addr + off, 16, 1024);
            const uint64_t kd = umma_desc_sw128(k_addr + (kk >> 2) * (kExtendKeys * 128) + (kk & 3) * 32, 16, 1024);
            umma_bf16(tmem + slot * kExtendKeys, qd, kd, idesc_qk, kk > 0);
          }
          umma_commit(&s_full[slot]);
          if (j == nkv - 1) umma_commit(q_empty);
          if (j >= 1 && !issue_pv(jt - 1, j - 1 == 0)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (!issue_pv(jt - 1, nkv == 1)) {
          ok = false;
          break;
        }
        ++uq;
      }
      if (!ok) *s_abort = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int r = tid;  // row of the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t jt = 0, uq = 0;
    for (int w = blockIdx.x; w < n_units && !*s_abort; w += gridDim.x) {
      const ExtendTile tile = a.m.extend_tiles[w / a.num_kv_heads];
      const int g = w % a.num_kv_heads;
      const int nkv = tile.kv_tiles;
      const int b = tile.b;
      const int q0 = a.m.qo_indptr[b];
      const int qo = a.m.qo_indptr[b + 1] - q0;
      const int L = a.m.kv_len[b];
      const int np = a.m.kv_indptr[b + 1] - a.m.kv_indptr[b];
      const int R = tile.row0 + r;
      const bool valid = R < qo * G;
      const int tok = min(R / G, qo - 1);
      const int limit = L - qo + tok;
      const long long orow = ((long long)(q0 + R / G) * a.num_q_heads + g * G + R % G);
      if (nkv == 0) {
        if (valid) {
          for (int c = 0; c < D; c += 8)
            *reinterpret_cast<uint4*>(a.out + orow * D + c) = make_uint4(0, 0, 0, 0);
          if (a.lse) a.lse[orow] = -INFINITY;
        }
        continue;
      }
      float m_ref = -INFINITY, l = 0.f;
      bool aborted = false;
      for (int j = 0; j < nkv; ++j, ++jt) {
        const int slot = jt & 1;
        const uint32_t ph = (jt >> 1) & 1;
        if (!mbar_wait(&s_full[slot], ph, plan)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        float s[kExtendKeys];
        {
          uint32_t sr[kExtendKeys];
#pragma unroll
          for (int c = 0; c < kExtendKeys / 32; ++c) tmem_ld32(lane_base + slot * kExtendKeys + c * 32, sr + c * 32);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < kExtendKeys; ++c) s[c] = __uint_as_float(sr[c]);
        }
        tc_fence_before();
        mbar_arrive(&s_free[slot]);

        // the request's last page inside this tile: zero the V rows past L
        if (j == nkv - 1 && np <= (j + 1) * (kExtendKeys / kPageSize) && (L % kPageSize) != 0) {
          const int r0 = L - j * kExtendKeys;
          const int r1 = (np - j * (kExtendKeys / kPageSize)) * kPageSize;
          uint8_t* vt = smem + C::kKVOff + slot * C::kStageBytes + C::kTileBytes;
          const int n16 = (r1 - r0) * C::kColBlocks * 8;
          for (int i = r; i < n16; i += 128) {
            const int row = r0 + i / (C::kColBlocks * 8);
            const int rest = i % (C::kColBlocks * 8);
            *reinterpret_cast<uint4*>(vt + (rest >> 3) * (kExtendKeys * 128) + row * 128 + (rest & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }

        const int key0 = j * kExtendKeys;
        float mt = -INFINITY;
        if (key0 + kExtendKeys - 1 <= limit) {
#pragma unroll
          for (int c = 0; c < kExtendKeys; ++c) {
            s[c] *= a.scale_log2;
            mt = fmaxf(mt, s[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kExtendKeys; ++c) {
            s[c] = (key0 + c <= limit) ? s[c] * a.scale_log2 : -INFINITY;
            mt = fmaxf(mt, s[c]);
          }
        }
        if (j == 0) {
          m_ref = mt;
        } else if (mt > m_ref + kRescaleThreshold) {
          // O must hold every earlier PV before it is rescaled
          const uint32_t jp = jt - 1;
          if (!mbar_wait(&p_free[jp & 1], (jp >> 1) & 1, plan)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const float alpha = fast_exp2(m_ref - mt);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + C::kOCol + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + C::kOCol + c * 32, o);
          }
          tmem_wait_st();
          l *= alpha;
          m_ref = mt;
        }
        const float ref = m_ref == -INFINITY ? 0.f : m_ref;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < kExtendKeys; ++c) {
          s[c] = fast_exp2(s[c] - ref);
          rs += s[c];
        }
        l += rs;
        // P slot is free once the PV of two tiles ago has completed
        if (!mbar_wait(&p_free[slot], ph ^ 1, plan)) {
          aborted = true;
          break;
        }
        uint8_t* pt = smem + C::kPOff + slot * C::kPBytes;
#pragma unroll
        for (int c = 0; c < kExtendKeys / 8; ++c) {
          uint4 v;
          v.x = pack_bf16(s[8 * c + 0], s[8 * c + 1]);
          v.y = pack_bf16(s[8 * c + 2], s[8 * c + 3]);
          v.z = pack_bf16(s[8 * c + 4], s[8 * c + 5]);
          v.w = pack_bf16(s[8 * c + 6], s[8 * c + 7]);
          *reinterpret_cast<uint4*>(pt + (c >> 3) * (kExtendRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[slot]);
      }
      if (aborted) {
        *s_abort = 1;
        break;
      }
      // epilogue: O / l
      const uint32_t jl = jt - 1;
      if (!mbar_wait(&p_free[jl & 1], (jl >> 1) & 1, plan)) {
        *s_abort = 1;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + C::kOCol + c * 32, o);
        tmem_wait_ld();
        if (valid) {
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
      tc_fence_before();
      mbar_arrive(o_free);
      if (valid && a.lse) a.lse[orow] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      ++uq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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
  if (cudaFuncSetAttribute(extend_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  extend_tc_kernel<C><<<c.extend_ctas, C::kThreads, C::kSmemBytes, st>>>(tk, tv, a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int launch_extend(Ctx& c, const void* q, const void* k_pool, const void* v_pool, float sm_scale, void* out,
                  float* lse, cudaStream_t st) {
  if (c.cfg.head_dim == 128) return run_extend<ExtCfg<128>>(c, q, k_pool, v_pool, sm_scale, out, lse, st);
  if (c.cfg.head_dim == 64) return run_extend<ExtCfg<64>>(c, q, k_pool, v_pool, sm_scale, out, lse, st);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
