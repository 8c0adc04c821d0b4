// Per-batch metadata build ("--attention-backend", section "What an attention
// backend is": a backend builds per-batch metadata such as page tables and
// index buffers; CUDA-graph replay needs them in fixed-size buffers).
//
// One launch, every input read on the device, so it can sit in a captured
// graph. Outputs, for request b with KV length L_b and qo_len_b query rows:
//   kv_indptr[b+1]      = kv_indptr[b] + ceil(L_b / page_size)
//   kv_indices          = page_table[b, 0 : pages_b] concatenated over b
//   kv_last_page_len[b] = L_b - (pages_b - 1) * page_size   (0 when L_b == 0)
//   qo_indptr[b+1]      = qo_indptr[b] + qo_len_b
// the same lists over 16-slot segments when a page holds several (128-token
// pages: segment k of a request is segment k % 8 of its page k / 8, id
// page * 8 + k % 8), which is what the attention kernels gather; and two work
// lists, counted in segments:
//   decode path: (request, split, page range) items; every request's pages are
//     cut into chunks of chunk_pages, with chunk_pages chosen so the number of
//     (item, KV head) units fills the persistent grid a few times over and the
//     partial-output buffer cannot overflow;
//   extend path: (request, first query row) units of 256 rows (two 128-row
//     tiles), where a row is (token, head-in-group), with the number of
//     128-key KV tiles each tile reaches; a request whose rows fit one unit
//     and whose decode plan splits it is cut along its KV range into equal
//     splits instead, the split size priced against the extend grid.
//
// Work split: CTA j owns a contiguous range of requests. Every CTA first
// reduces the batch totals (they fix chunk_pages and the capacity checks) and
// the prefix of each scanned quantity before its range, then scans its range.
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxCtas = 64;
constexpr int kPagesPerKvTile = kExtendKeys / kSegSlots;

struct ReqInfo {
  int L;       // KV length used (0 if the request's lengths were invalid)
  int qo;      // query rows
  int np;      // 16-slot segments
  int npg;     // pages
  int nsplit;  // decode splits
  int esplit;  // extend KV splits (1 unless the rows fit one unit and the range is cut)
  int prow;    // partial-output rows (0 when the request has a single split)
  int qtiles;  // extend query tiles
  bool bad;
};

struct Sums {
  long long np, qo, ns, pr, qt, npqo;  // np: segments
  long long npg;                       // pages
  long long et;  // KV tiles of the requests whose rows fit one extend unit
  int maxqo, splitd, splite;
  int maxnp;  // pages of the longest request
};

struct MetaArgs {
  int* plan;
  int* kv_indptr;
  int* kv_indices;
  int* kv_last_page_len;
  int* seg_indptr;   // aliases kv_indptr when a page is one segment
  int* seg_indices;  // aliases kv_indices when a page is one segment
  int* qo_indptr;
  int* kv_len;
  int* n_splits;
  int* ext_splits;
  int* partial_indptr;
  int* token_req;
  DecodeItem* items;
  ExtendTile* tiles;
  const int* seq_lens;
  const int* qo_lens;  // may be null: one row per request
  const int* page_table;
  int stride;
  int bs;
  int num_pages;
  int page_size;     // tokens per page: 16 or 128
  int seg_per_page;  // page_size / 16
  int group;  // num_q_heads / num_kv_heads
  int num_kv_heads;
  int stage_pages;  // the decode kernel's segments per pipeline stage
  // the decode path runs on the tcgen05 tile kernel (verify shapes): its
  // splits are equal shares of whole 128-key tiles, sized like the extend
  // path's KV splits
  int dec_tc;
  int units_target;      // decode work units to aim for
  int dec_ctas;          // CTAs of the persistent decode grid
  int fp8;               // E4M3 pools
  int ext_grid;          // CTAs of the extend kernel (units are dealt to them by a fixed stride)
  int partial_cap;
  int max_pages_total;
  int max_q_tokens;
  int max_items;
  int max_tiles;
};

// A request's lengths as given, validated: negative lengths, more query rows
// than keys, and a KV length whose pages do not fit one page-table row (the
// gather would read past the row, into the next request's or past the table)
// mark it bad, and a bad request is treated as empty.
__device__ __forceinline__ void raw_lengths(const MetaArgs& a, int b, int& L, int& qo, bool& bad) {
  L = a.seq_lens[b];
  qo = a.qo_lens ? a.qo_lens[b] : 1;
  bad = (L < 0) || (qo < 0) || (L > 0 && qo > L) || (L > 0 && (L - 1) / a.page_size >= a.stride);
  if (bad) {
    L = 0;
    qo = qo < 0 ? 0 : qo;
  }
}

// Requests whose validated lengths the first pass keeps in shared memory;
// every later pass reads them from there (the rest from global memory).
constexpr int kLenCache = 2048;
__shared__ int2 s_len_cache[kLenCache];  // {L, qo | bad << 31}

__device__ __forceinline__ void lengths(const MetaArgs& a, int b, int& L, int& qo, bool& bad) {
  if (b < kLenCache) {
    const int2 v = s_len_cache[b];
    L = v.x;
    qo = v.y & 0x7fffffff;
    bad = v.y < 0;
  } else {
    raw_lengths(a, b, L, qo, bad);
  }
}

// segments and pages of a validated length (no overflow near INT_MAX)
__device__ __forceinline__ int segs_of(int L) { return L > 0 ? (L - 1) / kSegSlots + 1 : 0; }
__device__ __forceinline__ int pages_of(const MetaArgs& a, int L) { return L > 0 ? (L - 1) / a.page_size + 1 : 0; }

__device__ __forceinline__ int kv_tiles_of(int np) { return (np + kPagesPerKvTile - 1) / kPagesPerKvTile; }

__device__ __forceinline__ ReqInfo req_info(const MetaArgs& a, int b, int chunk, int ext_ct) {
  ReqInfo r;
  lengths(a, b, r.L, r.qo, r.bad);
  r.np = segs_of(r.L);
  r.npg = pages_of(a, r.L);
  if (a.dec_tc) {
    const int tiles = kv_tiles_of(r.np);
    r.nsplit = tiles > ext_ct ? (tiles + ext_ct - 1) / ext_ct : 1;
  } else {
    r.nsplit = r.np > 0 ? (r.np + chunk - 1) / chunk : 1;
  }
  r.prow = r.nsplit > 1 ? r.nsplit * r.qo : 0;
  r.qtiles = (r.qo * a.group + kExtendUnitRows - 1) / kExtendUnitRows;
  // rows that fit one extend unit: cut the KV range into equal splits of at
  // most ext_ct 128-key tiles; ext_ct spans at least one decode chunk, so the
  // split count never exceeds the decode plan's and its partial rows fit
  r.esplit = (r.qtiles == 1 && r.nsplit > 1) ? (kv_tiles_of(r.np) + ext_ct - 1) / ext_ct : 1;
  if (r.esplit > 1) r.qtiles = r.esplit;
  return r;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_max(int v) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum of a Sums record (result valid in every thread).
__device__ Sums block_sum(Sums s) {
  __shared__ long long red[8][kThreads / 32];
  __shared__ int redm[kThreads / 32], redd[kThreads / 32], rede[kThreads / 32], redp[kThreads / 32];
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  s.np = warp_sum(s.np);
  s.qo = warp_sum(s.qo);
  s.ns = warp_sum(s.ns);
  s.pr = warp_sum(s.pr);
  s.qt = warp_sum(s.qt);
  s.npqo = warp_sum(s.npqo);
  s.et = warp_sum(s.et);
  s.npg = warp_sum(s.npg);
  s.maxqo = warp_max(s.maxqo);
  s.maxnp = warp_max(s.maxnp);
  s.splitd = warp_sum(s.splitd);
  s.splite = warp_sum(s.splite);
  __syncthreads();
  if (l == 0) {
    red[0][w] = s.np;
    red[1][w] = s.qo;
    red[2][w] = s.ns;
    red[3][w] = s.pr;
    red[4][w] = s.qt;
    red[5][w] = s.npqo;
    red[6][w] = s.et;
    red[7][w] = s.npg;
    redm[w] = s.maxqo;
    redp[w] = s.maxnp;
    redd[w] = s.splitd;
    rede[w] = s.splite;
  }
  __syncthreads();
  Sums t{};
  for (int i = 0; i < kThreads / 32; ++i) {
    t.splitd += redd[i];
    t.splite += rede[i];
    t.np += red[0][i];
    t.qo += red[1][i];
    t.ns += red[2][i];
    t.pr += red[3][i];
    t.qt += red[4][i];
    t.npqo += red[5][i];
    t.et += red[6][i];
    t.npg += red[7][i];
    t.maxqo = max(t.maxqo, redm[i]);
    t.maxnp = max(t.maxnp, redp[i]);
  }
  return t;
}

// Tiles per extend KV split. The extend kernel deals its units to CTAs by a
// fixed stride, so a step lasts about as long as its busiest CTA:
// ceil(units / grid) units of up to ct tiles, each with a fixed cost (Q load,
// the in-CTA merge, output stores) of about two tiles. Candidates start where
// about eight units fall to each CTA (finer splits only add fixed costs),
// never below one decode chunk; the cheapest wins, ties going to the larger
// split. Thread t prices candidate t % 64 over every fourth request. A batch
// of single-row requests (decode) keeps the smallest candidate without
// pricing: the decode path does not read these splits. Called by every thread
// of the block; identical in every CTA.
constexpr int kExtCandidates = 64;
constexpr int kExtUnitCostTiles = 2;
constexpr int kExtMaxUnitsPerCta = 8;
constexpr int kExtGroups = kThreads / kExtCandidates;
static_assert(kThreads % kExtCandidates == 0 && kExtCandidates == 64, "two warps of candidates");

__device__ int extend_split_tiles(const MetaArgs& a, int chunk, const Sums& tot) {
  __shared__ int s_units[kExtGroups][kExtCandidates];
  __shared__ unsigned long long s_key[2];
  const int ct_min = kv_tiles_of(chunk);
  const long long grid = a.ext_grid > 0 ? a.ext_grid : 1;
  // tot.et counts the tiles of every request whose rows fit one unit, a bound
  // on those that get split
  const long long per = (long long)kExtMaxUnitsPerCta * grid;
  long long lo = (tot.et * a.num_kv_heads + per - 1) / per;
  if (lo < ct_min) lo = ct_min;
  if (lo > (1 << 24)) lo = 1 << 24;
  const int ct_lo = (int)lo;
  if (tot.maxqo <= 1 || tot.et == 0) return ct_lo;
  const int c = threadIdx.x % kExtCandidates, grp = threadIdx.x / kExtCandidates;
  const int ct = ct_lo + c;
  int split_units = 0, fixed_units = 0;
  for (int b = grp; b < a.bs; b += kExtGroups) {
    int L, qo;
    bool bad;
    lengths(a, b, L, qo, bad);
    const int np = segs_of(L);
    const int qt = (qo * a.group + kExtendUnitRows - 1) / kExtendUnitRows;
    if (qt == 1 && np > chunk)
      split_units += (kv_tiles_of(np) + ct - 1) / ct;
    else
      fixed_units += qt;
  }
  s_units[grp][c] = split_units + fixed_units;
  __syncthreads();
  if (threadIdx.x < kExtCandidates) {
    int u = 0;
#pragma unroll
    for (int g = 0; g < kExtGroups; ++g) u += s_units[g][c];
    const long long units = (long long)u * a.num_kv_heads;
    const unsigned long long cost = (unsigned long long)((units + grid - 1) / grid) * (ct + kExtUnitCostTiles);
    // cheapest, ties to the larger split: minimum of cost * 64 + (63 - c)
    unsigned long long key = cost * kExtCandidates + (kExtCandidates - 1 - c);
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, key, o);
      if (y < key) key = y;
    }
    if ((threadIdx.x & 31) == 0) s_key[threadIdx.x >> 5] = key;
  }
  __syncthreads();
  const unsigned long long best = s_key[0] < s_key[1] ? s_key[0] : s_key[1];
  return ct_lo + (kExtCandidates - 1 - (int)(best % kExtCandidates));
}

// Decode chunk size. The persistent decode grid takes (item, KV head) units
// in order as its CTAs free up, and in a batch of a few long requests nearly
// every unit is one whole chunk long: the step then lasts about
// ceil(units / CTAs) chunks, and a chunk that leaves the last round of units
// nearly empty idles most of the grid for one chunk's time. The candidates run
// up from the smallest admissible chunk in whole pipeline stages; each costs
// the larger of ceil(units / CTAs) chunks and an even share of all the pages,
// both with a fixed cost per unit; the cheapest wins, ties going to the
// smaller chunk. Thread t prices candidate t % 64 over every fourth request.
// Which batches are priced: a bf16 unit is bound by memory, and when CTAs
// fall idle at the end the ones still running take over most of their share
// of the bandwidth, so there the smallest chunk stands unless its units do
// not fill the grid kDecPriceRounds times; an E4M3 unit is bound by its
// widening and MMA work, the running CTAs cannot speed up, and every such
// batch is priced. Verify shapes on the tile kernel split by their own rule,
// and batches of many requests (whose short last splits fill any round) are
// not priced. Called by every thread of the block; identical in every CTA.
constexpr int kDecCandidates = 64;
constexpr int kDecUnitCostPages = 2;
constexpr int kDecPriceMaxBatch = 256;
constexpr int kDecPriceRounds = 4;
static_assert(kThreads % kDecCandidates == 0 && kDecCandidates == 64, "two warps of candidates");

__device__ int decode_chunk_pages(const MetaArgs& a, int chunk0, const Sums& tot) {
  if (a.dec_tc || a.bs > kDecPriceMaxBatch || tot.np == 0) return chunk0;
  if (!a.fp8) {
    // units of the smallest chunk: a request takes ceil(np / chunk0) splits,
    // at most np / chunk0 + 1, so a bound on the sum needs no pass
    const long long ctas = a.dec_ctas > 0 ? a.dec_ctas : 1;
    const long long units_lo = tot.np / chunk0 * a.num_kv_heads;
    if (units_lo >= kDecPriceRounds * ctas) return chunk0;
  }
  __shared__ int s_items[kExtGroups][kDecCandidates];
  __shared__ unsigned long long s_key[2];
  const int ci = threadIdx.x % kDecCandidates, grp = threadIdx.x / kDecCandidates;
  const long long cp = (long long)chunk0 + (long long)ci * a.stage_pages;
  int items = 0;
  for (int b = grp; b < a.bs; b += kExtGroups) {
    int L, qo;
    bool bad;
    lengths(a, b, L, qo, bad);
    const int np = segs_of(L);
    items += np > 0 ? (int)((np + cp - 1) / cp) : 1;
  }
  s_items[grp][ci] = items;
  __syncthreads();
  if (threadIdx.x < kDecCandidates) {
    long long units = 0;
#pragma unroll
    for (int g = 0; g < kExtGroups; ++g) units += s_items[g][ci];
    units *= a.num_kv_heads;
    const long long ctas = a.dec_ctas > 0 ? a.dec_ctas : 1;
    const long long rounds = (units + ctas - 1) / ctas;
    const long long share = (tot.np * a.num_kv_heads + units * kDecUnitCostPages + ctas - 1) / ctas;
    long long cost = rounds * (cp + kDecUnitCostPages);
    if (cost < share) cost = share;
    unsigned long long key = (unsigned long long)cost * kDecCandidates + ci;
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, key, o);
      if (y < key) key = y;
    }
    if ((threadIdx.x & 31) == 0) s_key[threadIdx.x >> 5] = key;
  }
  __syncthreads();
  const unsigned long long best = s_key[0] < s_key[1] ? s_key[0] : s_key[1];
  return chunk0 + (int)(best % kDecCandidates) * a.stage_pages;
}

// Exclusive block scan of six ints; returns this thread's prefix and the tile total.
constexpr int kScanN = 6;
struct ScanV {
  int v[kScanN];
};
__device__ ScanV block_exclusive_scan(const ScanV& x, ScanV& total) {
  __shared__ int part[kScanN][kThreads / 32];
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  ScanV inc = x;
  for (int k = 0; k < kScanN; ++k) {
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, inc.v[k], o);
      if (l >= o) inc.v[k] += y;
    }
  }
  __syncthreads();
  if (l == 31)
    for (int k = 0; k < kScanN; ++k) part[k][w] = inc.v[k];
  __syncthreads();
  ScanV ex;
  for (int k = 0; k < kScanN; ++k) {
    int before = 0, all = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
      if (i < w) before += part[k][i];
      all += part[k][i];
    }
    ex.v[k] = before + inc.v[k] - x.v[k];
    total.v[k] = all;
  }
  return ex;
}

__global__ void __launch_bounds__(kThreads) build_metadata_kernel(MetaArgs a) {
  // the attention kernel launched next may start its prologue now; it waits
  // for this grid before reading any metadata
  pdl_launch_dependents();
  // launched with programmatic serialization too: the lengths and page table
  // (and the workspace the previous kernels read) only after the previous
  // grid has finished
  pdl_wait();
  // ---- 1. batch totals (identical in every CTA) ----
  Sums s{};
  for (int b = threadIdx.x; b < a.bs; b += kThreads) {
    int L, qo;
    bool bad;
    raw_lengths(a, b, L, qo, bad);
    if (b < kLenCache) s_len_cache[b] = make_int2(L, bad ? (int)((unsigned)qo | 0x80000000u) : qo);
    long long np = segs_of(L);
    s.np += np;
    s.npg += pages_of(a, L);
    s.qo += qo;
    s.npqo += np * qo;
    s.maxqo = max(s.maxqo, qo);
    s.maxnp = max(s.maxnp, (int)np);
    if (qo > 0 && (long long)qo * a.group <= kExtendUnitRows) s.et += kv_tiles_of((int)np);
  }
  Sums tot = block_sum(s);
  bool over = tot.npg > a.max_pages_total || tot.qo > a.max_q_tokens || tot.qo >= a.partial_cap;

  // decode split size: fill the grid, never finer than the minimum chunk, and
  // keep sum over split requests of nsplit*qo below the partial buffer
  long long chunk = (tot.np * a.num_kv_heads + a.units_target - 1) / a.units_target;
  if (chunk < kDecodeMinChunkPages) chunk = kDecodeMinChunkPages;
  // at most kMaxSplitsPerRequest splits of any request (the merge reads two per lane)
  const long long cmax = (tot.maxnp + kMaxSplitsPerRequest - 1) / kMaxSplitsPerRequest;
  if (chunk < cmax) chunk = cmax;
  long long room = (long long)a.partial_cap - tot.qo;
  if (room > 0) {
    long long c2 = (tot.npqo + room - 1) / room;
    if (c2 > chunk) chunk = c2;
  }
  chunk = (chunk + a.stage_pages - 1) / a.stage_pages * a.stage_pages;
  if (chunk > (1 << 30)) chunk = 1 << 30;
  // the pricing only moves the chunk up, which keeps every bound above
  const int ichunk = decode_chunk_pages(a, (int)chunk, tot);
  const int ext_ct = extend_split_tiles(a, ichunk, tot);

  if (over) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      record_error(a.plan, PKV_DEV_CAPACITY, (int)tot.npg);
      a.plan[kBatch] = 0;
      a.plan[kTotalSegs] = 0;
      a.plan[kTotalQ] = 0;
      a.plan[kDecodeItems] = 0;
      a.plan[kExtendTiles] = 0;
      a.plan[kPartialRows] = 0;
      a.plan[kChunkPages] = ichunk;
      a.plan[kMaxQo] = 0;
      a.plan[kSplitDecode] = 0;
      a.plan[kSplitExtend] = 0;
      a.plan[kDecodeNext] = 0;
    }
    return;
  }

  // ---- 2. this CTA's request range and the prefix before it ----
  int per = (a.bs + gridDim.x - 1) / gridDim.x;
  int b0 = min(a.bs, (int)blockIdx.x * per), b1 = min(a.bs, b0 + per);
  Sums pre{};
  for (int b = threadIdx.x; b < b0; b += kThreads) {
    ReqInfo r = req_info(a, b, ichunk, ext_ct);
    pre.np += r.np;
    pre.npg += r.npg;
    pre.qo += r.qo;
    pre.ns += r.nsplit;
    pre.pr += r.prow;
    pre.qt += r.qtiles;
  }
  Sums base = block_sum(pre);
  // totals of the scanned quantities over the whole batch (for the plan words)
  Sums all{};
  if (blockIdx.x == 0) {
    for (int b = threadIdx.x; b < a.bs; b += kThreads) {
      ReqInfo r = req_info(a, b, ichunk, ext_ct);
      all.ns += r.nsplit;
      all.pr += r.prow;
      all.qt += r.qtiles;
      all.splitd += r.nsplit > 1 ? 1 : 0;
      all.splite += r.esplit > 1 ? 1 : 0;
    }
    all = block_sum(all);
  }

  // ---- 3. scan the range tile by tile; per-element writes spread over the CTA ----
  ScanV carry{{(int)base.np, (int)base.qo, (int)base.ns, (int)base.pr, (int)base.qt, (int)base.npg}};
  enum { kNp, kPBase, kQo, kQBase, kNs, kSBase, kQt, kTBase, kL, kEs, kGBase, kInfo };
  __shared__ int s_info[kThreads][kInfo];
  const bool segs = a.seg_per_page > 1;  // segment lists of their own (else they are the page lists)
  for (int t0 = b0; t0 < b1; t0 += kThreads) {
    const int b = t0 + threadIdx.x;
    ReqInfo r{0, 0, 0, 0, 0, 1, 0, 0, false};
    const bool live = b < b1;
    if (live) r = req_info(a, b, ichunk, ext_ct);
    ScanV x{{r.np, r.qo, r.nsplit, r.prow, r.qtiles, r.npg}};
    if (!live) x = ScanV{};
    ScanV tile_tot;
    ScanV ex = block_exclusive_scan(x, tile_tot);
    const int p_np = carry.v[0] + ex.v[0], p_qo = carry.v[1] + ex.v[1], p_ns = carry.v[2] + ex.v[2];
    const int p_pr = carry.v[3] + ex.v[3], p_qt = carry.v[4] + ex.v[4], p_pg = carry.v[5] + ex.v[5];
    if (live) {
      if (r.bad) record_error(a.plan, PKV_DEV_BAD_LENGTH, b);
      a.kv_indptr[b] = p_pg;
      if (segs) a.seg_indptr[b] = p_np;
      a.qo_indptr[b] = p_qo;
      a.partial_indptr[b] = p_pr;
      a.kv_len[b] = r.L;
      a.n_splits[b] = r.nsplit;
      a.ext_splits[b] = r.esplit;
      a.kv_last_page_len[b] = r.npg > 0 ? r.L - (r.npg - 1) * a.page_size : 0;
      if (b == a.bs - 1) {
        a.kv_indptr[a.bs] = p_pg + r.npg;
        if (segs) a.seg_indptr[a.bs] = p_np + r.np;
        a.qo_indptr[a.bs] = p_qo + r.qo;
        a.partial_indptr[a.bs] = p_pr + r.prow;
      }
      int* inf = s_info[threadIdx.x];
      inf[kNp] = r.np;
      inf[kPBase] = p_np;
      inf[kGBase] = p_pg;
      inf[kQo] = r.qo;
      inf[kQBase] = p_qo;
      inf[kNs] = r.nsplit;
      inf[kSBase] = p_ns;
      inf[kQt] = r.qtiles;
      inf[kTBase] = p_qt;
      inf[kL] = r.L;
      inf[kEs] = r.esplit;
    }
    __syncthreads();
    const int nreq = min(kThreads, b1 - t0);
    for (int j = 0; j < nreq; ++j) {
      const int bb = t0 + j;
      const int* inf = s_info[j];
      const int np = inf[kNp], pbase = inf[kPBase], qo = inf[kQo], qbase = inf[kQBase];
      const int ns = inf[kNs], sbase = inf[kSBase], qt = inf[kQt], tbase = inf[kTBase], L = inf[kL];
      const int* __restrict__ row = a.page_table + (long long)bb * a.stride;
      // segment k is segment k % R of page k / R (R = segments per page); the
      // page list takes each page once
      const int R = a.seg_per_page, gbase = inf[kGBase];
      for (int k = threadIdx.x; k < np; k += kThreads) {
        const int p = k / R, sub = k - p * R;
        int page = row[p];
        if (page < 0 || page >= a.num_pages) {
          record_error(a.plan, PKV_DEV_BAD_PAGE, bb);
          page = 0;
        }
        if (sub == 0) a.kv_indices[gbase + p] = page;
        if (segs) a.seg_indices[pbase + k] = page * R + sub;
      }
      for (int sp = threadIdx.x; sp < ns; sp += kThreads) {
        if (sbase + sp < a.max_items) {
          DecodeItem it;
          it.b = bb;
          it.split = sp;
          if (a.dec_tc) {
            // equal shares of the request's 128-key tiles
            const int tiles = kv_tiles_of(np);
            it.p0 = (int)((long long)sp * tiles / ns) * kPagesPerKvTile;
            it.p1 = min(np, (int)((long long)(sp + 1) * tiles / ns) * kPagesPerKvTile);
          } else {
            it.p0 = sp * ichunk;
            it.p1 = min(np, (sp + 1) * ichunk);
          }
          a.items[sbase + sp] = it;
        }
      }
      const int rows = qo * a.group;
      auto kv_tiles_to = [&](int row_end) {  // KV tiles reached by rows [.., row_end)
        const int last_tok = (row_end - 1) / a.group;
        return L > 0 ? (L - qo + last_tok + 1 + kExtendKeys - 1) / kExtendKeys : 0;
      };
      const bool split = inf[kEs] > 1;
      const int es = inf[kEs], ntiles = kv_tiles_of(np);
      for (int t = threadIdx.x; t < qt; t += kThreads) {
        if (tbase + t < a.max_tiles) {
          const int row0 = split ? 0 : t * kExtendUnitRows;
          ExtendTile et;
          et.b = bb;
          et.row0 = row0;
          et.kv_a = kv_tiles_to(min(row0 + kExtendRows, rows));
          et.kv_b = row0 + kExtendRows < rows ? kv_tiles_to(min(row0 + kExtendUnitRows, rows)) : 0;
          et.split = split ? t : -1;
          // split t takes an equal share of the request's KV tiles
          et.kv0 = split ? (int)((long long)t * ntiles / es) : 0;
          et.kv1 = split ? (int)((long long)(t + 1) * ntiles / es) : 0x7fffffff;
          // rows that fit one 128-row tile: both tiles hold them, each takes
          // half of the unit's KV range, and the halves are merged in the CTA
          et.dual = rows <= kExtendRows ? 1 : 0;
          a.tiles[tbase + t] = et;
        }
      }
      for (int i = threadIdx.x; i < qo; i += kThreads) a.token_req[qbase + i] = bb;
    }
    for (int k = 0; k < kScanN; ++k) carry.v[k] += tile_tot.v[k];
    __syncthreads();
  }

  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (a.bs == 0) {
      a.kv_indptr[0] = 0;
      if (segs) a.seg_indptr[0] = 0;
      a.qo_indptr[0] = 0;
      a.partial_indptr[0] = 0;
    }
    bool items_over = all.ns > a.max_items || all.qt > a.max_tiles;
    if (items_over) record_error(a.plan, PKV_DEV_CAPACITY, -1);
    a.plan[kBatch] = a.bs;
    a.plan[kTotalSegs] = (int)tot.np;
    a.plan[kTotalQ] = (int)tot.qo;
    a.plan[kDecodeItems] = items_over ? 0 : (int)all.ns;
    a.plan[kChunkPages] = ichunk;
    a.plan[kExtendTiles] = items_over ? 0 : (int)all.qt;
    a.plan[kPartialRows] = (int)all.pr;
    a.plan[kMaxQo] = tot.maxqo;
    a.plan[kSplitDecode] = items_over ? 0 : all.splitd;
    a.plan[kSplitExtend] = items_over ? 0 : all.splite;
    a.plan[kDecodeNext] = 0;
  }
}

}  // namespace

int launch_build_metadata(Ctx& c, int batch, const int32_t* seq_lens, const int32_t* qo_lens,
                          const int32_t* page_table, int stride, cudaStream_t st) {
  Meta m = make_meta(c);
  MetaArgs a;
  a.plan = m.plan;
  a.kv_indptr = const_cast<int*>(m.kv_indptr);
  a.kv_indices = const_cast<int*>(m.kv_indices);
  a.kv_last_page_len = const_cast<int*>(m.kv_last_page_len);
  a.seg_indptr = const_cast<int*>(m.seg_indptr);
  a.seg_indices = const_cast<int*>(m.seg_indices);
  a.qo_indptr = const_cast<int*>(m.qo_indptr);
  a.kv_len = const_cast<int*>(m.kv_len);
  a.n_splits = const_cast<int*>(m.n_splits);
  a.ext_splits = const_cast<int*>(m.ext_splits);
  a.partial_indptr = const_cast<int*>(m.partial_indptr);
  a.token_req = const_cast<int*>(m.token_req);
  a.items = const_cast<DecodeItem*>(m.decode_items);
  a.tiles = const_cast<ExtendTile*>(m.extend_tiles);
  a.seq_lens = seq_lens;
  a.qo_lens = qo_lens;
  a.page_table = page_table;
  a.stride = stride;
  a.bs = batch;
  a.num_pages = c.cfg.num_pages;
  a.page_size = c.cfg.page_size;
  a.seg_per_page = c.cfg.page_size / kSegSlots;
  a.group = c.cfg.num_q_heads / c.cfg.num_kv_heads;
  a.num_kv_heads = c.cfg.num_kv_heads;
  a.stage_pages = decode_stage_pages(c.cfg);
  a.dec_tc = decode_row_warps(c.cfg) > 1 ? 1 : 0;
  a.units_target = c.decode_ctas * (decode_row_warps(c.cfg) == 1 ? kDecodeTargetWaves : kVerifyTargetWaves);
  a.dec_ctas = c.decode_ctas;
  a.fp8 = c.cfg.kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 0;
  a.ext_grid = c.extend_ctas;
  a.partial_cap = c.lay.partial_rows_cap;
  a.max_pages_total = c.cfg.max_pages_total;
  a.max_q_tokens = c.cfg.max_q_tokens;
  a.max_items = c.lay.max_decode_items;
  a.max_tiles = c.lay.max_extend_tiles;
  int grid = batch < 1 ? 1 : (batch < kMaxCtas ? batch : kMaxCtas);
  return launch_pdl(build_metadata_kernel, dim3(grid), dim3(kThreads), 0, st, a) == cudaSuccess ? PKV_OK
                                                                                      : PKV_ERR_CUDA;
}

}  // namespace pkv
