/*
 * pkv.h — C ABI of a paged-KV attention library for one NVIDIA GB300 (sm_103a).
 *
 * The calls follow the attention-backend interface described in
 * "--attention-backend" (SGLang manual), section "What an attention backend is":
 * a backend computes attention over the paged KV cache for one batch; it builds
 * per-batch metadata (page tables, index buffers), keeps state that CUDA-graph
 * capture and replay can reuse, and runs forward_extend (prefill) and
 * forward_decode (decode). The ForwardMode dispatch follows "[SGLang] Hybrid
 * Attention: Dense-Sparse 동적 전환 전략", section "_select_backend: ForwardMode 기반
 * 동적 전환", and the save_kv_cache step its section "forward: 선형 어텐션까지
 * 지원하는 범용 위임".
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every function returns an int status (PKV_OK == 0, or a PKV_ERR_* code).
 *   Nothing throws, aborts or prints. Arguments are checked on the host before
 *   anything is launched; a failed check launches nothing.
 * - Pointers named d_* are DEVICE pointers into memory the caller owns (for
 *   example PyTorch tensors). The library never allocates or frees device
 *   memory: its device state lives in the workspace the caller passes to
 *   pkv_create, plus the one fixed scratch array that loading the library
 *   reserves for pkv_forward_decode_static. Host-side, pkv_create allocates
 *   one small context object.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). Work is enqueued asynchronously on it; no call below synchronises
 *   except pkv_get_device_error. pkv_build_metadata, pkv_set_kv_buffer and the
 *   forward calls read lengths only on the device, so a sequence of them can be
 *   captured into a CUDA graph and replayed with new lengths of the same batch
 *   size.
 * - KV pool layout ("NHD"): one pool for K and one for V per layer,
 *   [num_pages * page_size slots][num_kv_heads][width], row-major, with
 *   slot = page * page_size + offset; the width is head_dim for K and
 *   head_dim_v for V (pkv_config). Elements are bf16, or FP8 E4M3FN bytes
 *   with one fp32 scale per pool (value = code * scale).
 * - Queries are bf16 [tokens][num_q_heads][head_dim], outputs bf16
 *   [tokens][num_q_heads][head_dim_v]; LSE is fp32 [tokens][num_q_heads], the
 *   natural log of sum_j exp(sm_scale * q . k_j).
 *   Query head h reads KV head h / (num_q_heads / num_kv_heads).
 * - Request b has seq_lens[b] = L_b KV tokens (prefix plus this step's new
 *   tokens, whose K/V pkv_set_kv_buffer has already stored) and qo_len_b query
 *   rows; its i-th query row sees keys 0 .. L_b - qo_len_b + i (causal,
 *   aligned to the end). Decode is qo_len_b == 1. A request with L_b == 0 is
 *   padding: its rows get output 0 and LSE -inf.
 * - Device-side faults in the data (a page id outside the pool, a slot outside
 *   the pool, lengths beyond the configured capacities) are never turned into
 *   out-of-bounds accesses: the kernel skips the offending work and records the
 *   first error in a word of the workspace, read by pkv_get_device_error.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG 1 /* null pointer, negative size, bad enum, misaligned pointer */
#define PKV_ERR_UNSUPPORTED 2 /* shape or feature the library does not implement */
#define PKV_ERR_CAPACITY 3    /* batch or workspace larger than the configured capacity */
#define PKV_ERR_CUDA 4        /* a CUDA runtime / driver call failed */
#define PKV_ERR_DEVICE 5      /* the device recorded a data error (see pkv_get_device_error) */

/* Device error word values (pkv_get_device_error). */
#define PKV_DEV_OK 0
#define PKV_DEV_BAD_LENGTH 1   /* seq_len < 0, qo_len < 0, qo_len > seq_len, or ceil(seq_len / page_size) > page_table_stride */
#define PKV_DEV_BAD_PAGE 2     /* page id outside [0, num_pages) */
#define PKV_DEV_CAPACITY 3     /* total pages / query rows beyond the configured capacity */
#define PKV_DEV_BAD_SLOT 4     /* set_kv_buffer loc outside [0, num_pages * page_size) */
#define PKV_DEV_QO_TOO_LONG 5  /* decode path: qo_len beyond config.max_qo_len */
#define PKV_DEV_TREE_TOO_LONG 6 /* draft-tree mask set and a request has more than 64 new tokens */
#define PKV_DEV_TIMEOUT 16     /* a wait inside a kernel ran past the wait limit (pkv_set_wait_limit); the
                                  CTA that waited gave up its remaining work, so the outputs are incomplete */

/* ---- enumerations -------------------------------------------------------- */
/* ForwardMode of the batch ("[SGLang] Hybrid Attention", section
 * "_select_backend: ForwardMode 기반 동적 전환"). */
typedef enum {
  PKV_MODE_EXTEND = 0,        /* prefill / extend */
  PKV_MODE_DECODE = 1,
  PKV_MODE_IDLE = 2,          /* empty batch on this rank */
  PKV_MODE_TARGET_VERIFY = 3, /* speculative verify of draft tokens */
  PKV_MODE_DRAFT_EXTEND = 4
} pkv_forward_mode;

/* --speculative-attention-mode ("--attention-backend", section "Two backends in
 * one server"): which path runs the verify pass; the default is prefill. */
typedef enum { PKV_SPEC_PREFILL = 0, PKV_SPEC_DECODE = 1 } pkv_spec_mode;

typedef enum { PKV_PATH_INVALID = -1, PKV_PATH_DECODE = 0, PKV_PATH_EXTEND = 1 } pkv_path;

typedef enum { PKV_KV_BF16 = 0, PKV_KV_FP8_E4M3 = 1 } pkv_kv_dtype;

/* ---- configuration --------------------------------------------------------
 * Fixed for the life of a context; every capacity bounds a fixed-size
 * metadata buffer in the workspace, so captured graphs can be replayed.
 * Supported: head_dim 64 or 128 with V heads of the same width, or Q/K heads
 * of 192 with V heads of 128 (head_dim 192, head_dim_v 128: models whose K and
 * V heads differ in width, which "--attention-backend", section "How SGLang
 * picks a default", routes to fa4 on SM100/SM103); page_size 16 or 128 (the
 * 16-token page of the configs the library is tuned on, and the 128-token page
 * that the same page, section "The obvious fix, and why it fails", names as
 * fa4's native page size); num_q_heads a multiple of num_kv_heads with a group
 * size num_q_heads / num_kv_heads of at most 16; E4M3 (FP8) pools with head_dim
 * 128 (and V heads of 128) on both paths (other widths with an E4M3 pool
 * return PKV_ERR_UNSUPPORTED). */
typedef struct {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t kv_dtype;        /* pkv_kv_dtype */
  int32_t num_pages;       /* pool capacity in pages (pool = num_pages * page_size slots) */
  int32_t max_batch;       /* max requests in one batch */
  int32_t max_pages_total; /* max sum over requests of ceil(seq_len / page_size) */
  int32_t max_q_tokens;    /* max sum over requests of qo_len */
  int32_t max_qo_len;      /* max qo_len of one request on the decode path (verify drafts); 1 for plain decode */
  int32_t head_dim_v;      /* width of the V heads and of the output rows; 0 means head_dim */
} pkv_config;

typedef struct pkv_ctx pkv_ctx;

/* Human-readable name of a status code (static string, never NULL). */
const char* pkv_status_string(int status);

/* Bytes of device workspace a context with this configuration needs.
 * Errors: INVALID_ARG (null), UNSUPPORTED (shape outside the supported set). */
int pkv_workspace_bytes(const pkv_config* cfg, size_t* bytes_out);

/* Bytes of the K pool of one layer: num_pages * page_size * num_kv_heads *
 * head_dim * element size. The V pool takes the same with head_dim_v in place
 * of head_dim (the same bytes when the widths are equal). */
int pkv_pool_bytes(const pkv_config* cfg, size_t* bytes_out);

/* Create a context over caller-owned device workspace (256-byte aligned, at
 * least pkv_workspace_bytes). The context keeps the pointer; the caller keeps
 * the memory alive until pkv_destroy and must not use it for anything else.
 * Reads the current CUDA device's SM count. Errors: INVALID_ARG, UNSUPPORTED,
 * CAPACITY (workspace too small), CUDA. */
int pkv_create(const pkv_config* cfg, void* d_workspace, size_t workspace_bytes, pkv_ctx** ctx_out);

/* Free the host-side context (never the workspace). NULL is accepted. */
int pkv_destroy(pkv_ctx* ctx);

/* HybridAttnBackend._select_backend as a pure host function:
 * DECODE, IDLE -> PKV_PATH_DECODE; TARGET_VERIFY, DRAFT_EXTEND -> PKV_PATH_DECODE
 * when spec_mode == PKV_SPEC_DECODE, else PKV_PATH_EXTEND; EXTEND ->
 * PKV_PATH_EXTEND. Out-of-range arguments -> PKV_PATH_INVALID. */
int pkv_select_backend(int forward_mode, int spec_mode);

/* Per-batch metadata ("--attention-backend", section "What an attention backend
 * is"), built on the device into the workspace:
 *   kv_indptr[b+1]   = kv_indptr[b] + ceil(seq_lens[b] / page_size)
 *   kv_indices       = page_table rows b, entries 0 .. ceil(seq_lens[b]/page_size)-1, concatenated
 *   kv_last_page_len = seq_lens[b] - (pages_b - 1) * page_size (0 for an empty request)
 *   qo_indptr[b+1]   = qo_indptr[b] + qo_lens[b]
 * plus the split-KV work list of the decode path and the query-tile list of
 * the extend path. d_seq_lens, d_qo_lens: int32[batch] (d_qo_lens NULL means
 * one query row per request, as in decode). d_page_table: int32 rows of
 * page_table_stride entries. forward_mode selects nothing here (both paths'
 * plans are built); it is checked for validity, and IDLE (or batch == 0)
 * builds an empty plan. Errors: INVALID_ARG, CAPACITY (batch > max_batch),
 * CUDA. Data errors are recorded on the device: a request with negative
 * lengths, more query rows than keys, or more pages than one page-table row
 * holds (ceil(seq_len / page_size) > page_table_stride) records
 * PKV_DEV_BAD_LENGTH and is treated as empty (output 0, LSE -inf); its row of
 * the page table is not read. */
int pkv_build_metadata(pkv_ctx* ctx, int forward_mode, int32_t batch, const int32_t* d_seq_lens,
                       const int32_t* d_qo_lens, const int32_t* d_page_table, int32_t page_table_stride,
                       void* stream);

/* Device pointers to the metadata of the last pkv_build_metadata (valid once
 * that call's work has run on its stream). Any out pointer may be NULL. */
int pkv_get_metadata(pkv_ctx* ctx, const int32_t** kv_indptr, const int32_t** kv_indices,
                     const int32_t** kv_last_page_len, const int32_t** qo_indptr);

/* save_kv_cache: store this step's new K/V rows into the pools,
 *   pool[d_loc[i], h, :] = new[i, h, :]   for i < n_tokens, every KV head h.
 * d_k: bf16 [n_tokens][num_kv_heads][head_dim], d_v: bf16
 * [n_tokens][num_kv_heads][head_dim_v]; d_loc: int32 slots.
 * bf16 pools receive the same bits; E4M3 pools receive
 * e4m3_rn_satfinite(float(x) * inv_scale) (one fp32 multiply, round to nearest
 * even, finite values beyond +-448 saturate). Slots outside the pool are
 * skipped and recorded as PKV_DEV_BAD_SLOT. Duplicate slots: unspecified
 * winner. Pointers must be 16-byte aligned. */
int pkv_set_kv_buffer(pkv_ctx* ctx, void* d_k_pool, void* d_v_pool, const int32_t* d_loc, const void* d_k,
                      const void* d_v, int32_t n_tokens, float k_inv_scale, float v_inv_scale, void* stream);

/* forward_decode: attention of every query row against its request's paged
 * keys, using the metadata of the last pkv_build_metadata. Split-KV: each
 * (request, KV head) range is cut into chunks processed in parallel and merged
 * by their log-sum-exp. Handles qo_len up to config.max_qo_len per request
 * (target-verify on the decode path) with the causal rule above.
 * d_q: bf16 [T][num_q_heads][head_dim] (T = sum of qo_len), d_out: bf16
 * [T][num_q_heads][head_dim_v] (scores contract head_dim columns, the output
 * has the V heads' width), d_lse: fp32 [T][num_q_heads] or NULL. k_scale / v_scale multiply
 * E4M3 codes (ignored for bf16 pools). Pointers must be 16-byte aligned.
 * sm_scale must be positive and finite, and so must k_scale and v_scale with
 * an E4M3 pool (INVALID_ARG otherwise). Verify batches follow the draft-tree
 * mask when one is set (pkv_set_tree_mask).
 * Errors: INVALID_ARG, UNSUPPORTED (group size with max_qo_len beyond one
 * 128-row tile), CUDA. */
int pkv_forward_decode(pkv_ctx* ctx, const void* d_q, const void* d_k_pool, const void* d_v_pool, float sm_scale,
                       float k_scale, float v_scale, void* d_out, float* d_lse, void* stream);

/* forward_extend: causal attention of each request's query block (its
 * qo_len new tokens) against its cached prefix plus the new tokens, on the
 * tensor cores. Same arguments and layouts as pkv_forward_decode. With an
 * E4M3 pool the kernel widens each tile's codes to f16 in shared memory
 * (exact) and runs its MMAs in f16, Q and P rounded to f16, k_scale folded
 * into the score scale and v_scale into the output, as the decode path does;
 * the workspace holds no copy of the pool. */
int pkv_forward_extend(pkv_ctx* ctx, const void* d_q, const void* d_k_pool, const void* d_v_pool, float sm_scale,
                       float k_scale, float v_scale, void* d_out, float* d_lse, void* stream);

/* The hybrid backend's forward: pkv_select_backend(forward_mode, spec_mode)
 * picks pkv_forward_decode or pkv_forward_extend; IDLE returns PKV_OK and
 * launches nothing. forward_mode must be compatible with the metadata built
 * (DECODE needs one query row per request). */
int pkv_forward(pkv_ctx* ctx, int forward_mode, int spec_mode, const void* d_q, const void* d_k_pool,
                const void* d_v_pool, float sm_scale, float k_scale, float v_scale, void* d_out, float* d_lse,
                void* stream);

/* Draft trees for target verify (speculative decoding with top-k above 1;
 * "--attention-backend", sections "The obvious fix, and why it fails" and
 * "Our position" name it as a feature that limits which backends can run).
 * The pages give no mask format; this library's reading:
 *   d_tree_mask: device uint64 [total query tokens], in qo_indptr order. Bit j
 *   of token t's word lets t attend the j-th new (draft) token of its own
 *   request, at KV position seq_len - qo_len + j; every earlier (cached) key
 *   stays visible. Drafts are ordered with every ancestor before its
 *   descendants, so bits above the token's own index are ignored (a draft
 *   never sees a later one). A request may have at most 64 new tokens while a mask is
 *   set; a longer one records PKV_DEV_TREE_TOO_LONG and its rows see no draft
 *   past the 64th. NULL (the default) means chain drafts: token i sees new
 *   tokens 0..i, the bottom-right causal rule.
 * The mask applies to the forwards that follow a metadata build in
 * TARGET_VERIFY or DRAFT_EXTEND mode, on both paths; EXTEND and DECODE batches
 * ignore it. The caller owns the buffer and keeps it alive (with its contents
 * for the step) until those forwards have run; the context keeps the pointer,
 * so a captured graph replays with whatever the buffer holds then. */
int pkv_set_tree_mask(pkv_ctx* ctx, const uint64_t* d_tree_mask);

/* Attention sinks ("--attention-backend", section "The obvious fix, and why
 * it fails": a model that uses them rules some backends out). The pages give
 * no formula; this library's reading: d_sinks is a device fp32
 * [num_q_heads] array, and head h's sink logit joins every softmax of that
 * head as one more score whose value vector is zero:
 *   o = sum_j exp(s_j) v_j / (sum_j exp(s_j) + exp(sink_h)),
 *   lse = ln(sum_j exp(s_j) + exp(sink_h)),
 * with s_j = sm_scale * q . k_j as above; a row with no visible key gives
 * o = 0 and lse = sink_h. A -inf entry leaves its head unchanged. Applies to
 * every forward of the context (both paths, all modes) until set again; NULL
 * (the default) turns sinks off. The caller owns the buffer and keeps it
 * alive while forwards that use it run; a captured graph replays with
 * whatever it then holds. */
int pkv_set_attention_sinks(pkv_ctx* ctx, const float* d_sinks);

/* Bound on every wait inside the kernels (a warp waiting for a tile, a
 * result or a free buffer), in nanoseconds; 0 restores the default of 2 s.
 * A wait that runs past it records PKV_DEV_TIMEOUT: the CTA then stops
 * issuing work, waits (again bounded) for its copies in flight, releases its
 * tensor memory and exits, so the context stays usable; the outputs of that
 * launch are incomplete. The limit is kept in the context's workspace and
 * applies to every launch after this call. Synchronises `stream`. */
int pkv_set_wait_limit(pkv_ctx* ctx, uint32_t limit_ns, void* stream);

/* Test support for the bounded waits: with enable != 0, CTA 0 of every later
 * forward arms the barrier of its first K/V tile load but never issues the
 * copy, so the waits on that tile run out after the wait limit and the
 * timeout path runs (nothing faults; the other CTAs work normally). enable
 * = 0 turns it off. Synchronises `stream`. */
int pkv_test_hold_first_load(pkv_ctx* ctx, int enable, void* stream);

/* Synchronise `stream`, read the device error word into *code (PKV_DEV_*) and
 * clear it. Returns PKV_ERR_DEVICE when *code != PKV_DEV_OK. */
int pkv_get_device_error(pkv_ctx* ctx, int32_t* code, void* stream);

/* Write a one-line description of the context (paths, tile shapes, split
 * policy, SM count) into buf (always NUL-terminated when n > 0). */
int pkv_describe(pkv_ctx* ctx, char* buf, size_t n);

/* ---- decode without any device allocation -------------------------------
 * The source pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory. pkv_create needs a workspace that
 * somebody has to cudaMalloc; code running under another framework's caching
 * allocator (which owns the device memory, so a raw cudaMalloc can fail or
 * fragment its pool) and latency-critical loops (cudaMalloc / cudaFree can
 * synchronise the whole device) cannot. This call allocates nothing: its
 * metadata and split-KV scratch live in one fixed array of
 * PKV_STATIC_SCRATCH_BYTES in the library's device memory, which every GPU that
 * loads the library keeps until the process exits.
 *
 * It computes exactly what pkv_build_metadata (decode mode, d_qo_lens NULL)
 * followed by pkv_forward_decode computes, with the same kernels: one query
 * row per request, d_q / d_out bf16 [batch][num_q_heads][head_dim], d_lse
 * fp32 [batch][num_q_heads] or NULL, pools as in pkv_forward_decode. The K/V
 * of this step's tokens must already be in the pools (pkv_set_kv_buffer, or
 * the caller's own scatter).
 *   - cfg is checked as by pkv_workspace_bytes; a configuration whose scratch
 *     needs more than PKV_STATIC_SCRATCH_BYTES on this device (the split-KV
 *     partial buffer grows with max_q_tokens * num_q_heads * head_dim) returns
 *     PKV_ERR_CAPACITY and launches nothing.
 *   - d_error (device int32, nullable) receives the device error word of this
 *     call (PKV_DEV_*), written on `stream` after the kernels.
 *   - The array used is the one of the CURRENT device (cudaGetDevice), so
 *     `stream` must belong to the current device.
 *   - The first call on each device looks up the array's device address; make
 *     that first call before any stream capture on that device.
 *   - Every call on a device shares the one array, and it keeps the previous
 *     call's contents (the call clears the words that must start at zero).
 *     Calls whose work overlaps on the GPU (other streams, other host threads)
 *     race on it: serialise them. */
#define PKV_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

int pkv_forward_decode_static(const pkv_config* cfg, int32_t batch, const int32_t* d_seq_lens,
                              const int32_t* d_page_table, int32_t page_table_stride, const void* d_q,
                              const void* d_k_pool, const void* d_v_pool, float sm_scale, float k_scale,
                              float v_scale, void* d_out, float* d_lse, int32_t* d_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
