/*
 * okc_attn.h — C ABI of the GB300 (sm_103a) paged-FP8 gated attention block.
 *
 * The block is the part of a MuseSpark-style decoder layer that sits between
 * the QKV projection and the output projection ("012-attention-local-splits.py",
 * the docstring of the problem file: FusedQKNorm, set_kv_buffer/store_cache,
 * q.to(float8_e4m3fn), flash_attn_with_kvcache, rms_norm_gate). One step of it:
 *
 *   okc_attn_plan              host, once per decode step, shared by all layers
 *                              (okc_attn_plan_create: the same with default options)
 *   okc_prepare_qkv            steps 1-3: q/k RMSNorm (+RoPE), K/V E4M3 scatter, q E4M3
 *   okc_attn_decode            step 4: split-KV paged causal GQA attention
 *   okc_attn_combine_normgate  split merge fused with step 5, RMSNorm x sigmoid(gate)
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers unless the name ends in _host. Every buffer is
 *    owned by the caller; the library never frees or retains one past the call,
 *    except that a plan remembers the workspace it was uploaded into.
 *  - The kernel launches are asynchronous on `stream`. Entry points that launch
 *    kernels allocate nothing (no cudaMalloc, no host allocation).
 *  - Argument errors are detected on the host before any launch and return
 *    OKC_ERR_INVALID / OKC_ERR_UNSUPPORTED without touching the GPU. A failed
 *    launch returns OKC_ERR_CUDA. Nothing throws and nothing exits.
 *  - Alignment: qkv, out, q_fp8, the caches, o_partial and the norm weight
 *    16 bytes (vector loads and stores); positions and cache_loc 8 bytes; the
 *    int32 arrays, lse_partial and the scale scalars 4 bytes. A pointer that is
 *    not is an argument error (OKC_ERR_INVALID), never a misaligned access.
 *  - Errors that only the device can see (a cache row, page id or position out
 *    of range) never fault: the kernel skips the access, reads zeros where a
 *    key was expected, and ORs an OKC_DEVERR_* bit into the plan's device error
 *    word, which okc_attn_plan_read_errors returns.
 *  - Layouts (the problem file's `class Inputs`):
 *      qkv        bf16  [T, (2*Hq + 2*Hkv)*64]  per token: q | k | v | gate logits
 *      k_cache    e4m3  [num_pages, page_size, Hkv, 64]  flat row = page*page_size + offset
 *      v_cache    e4m3  same as k_cache
 *      page_table int32 [B, max_pages]  physical page of each logical page (-1 unused)
 *      out        bf16  [T, Hq*64]
 *    with T tokens: the step's new tokens, request b's tokens at rows
 *    cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and positions seq_lens[b] + i. A
 *    decode or verify step has T = B*L (cu_seqlens_q = 0, L, 2L, ...); a
 *    prefill/extend step (okc_attn_plan_varlen) q_lens[b] tokens per request.
 */
#ifndef OKC_ATTN_H
#define OKC_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that C callers need no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st* okc_stream;

typedef enum okc_status {
  OKC_OK = 0,
  OKC_ERR_INVALID = 1,      /* a bad argument: null pointer, size, shape or range */
  OKC_ERR_UNSUPPORTED = 2,  /* valid for the problem, but not a shape this library runs */
  OKC_ERR_CUDA = 3,         /* a CUDA runtime call or a kernel launch failed */
  OKC_ERR_WORKSPACE = 4     /* the workspace or a scratch buffer is too small or misaligned */
} okc_status;

/* Bits of the device error word (okc_attn_plan_read_errors). */
#define OKC_DEVERR_CACHE_LOC 0x1u  /* a cache_loc row outside the pool: that K/V row was not written */
#define OKC_DEVERR_POSITION 0x2u   /* a position outside the RoPE table: that token's q/k were written unrotated */
#define OKC_DEVERR_PAGE 0x4u       /* a page_table entry outside [0, num_pages) for a visible key: key read as zeros */
#define OKC_DEVERR_LENGTHS 0x8u    /* device lengths disagree with the plan (cache_seqlens, cu_seqlens_q, seq_lens) */
#define OKC_DEVERR_TIMEOUT 0x10u   /* a bounded in-kernel wait gave up (a copy never completed); the step's output is void */

/*
 * Mirrors the problem file's `class Config`. The library runs the per-GPU shape
 * of Muse Spark under TP8: num_q_heads = 16, num_kv_heads = 2, head_dim = 64
 * (anything else returns OKC_ERR_UNSUPPORTED), q_len in [1, 65536], page_size
 * a power of two in [1, 256], max_pages * page_size <= 2^30 and batch * q_len
 * <= 2^26 (larger: OKC_ERR_UNSUPPORTED).
 */
typedef struct okc_attn_config {
  int32_t batch;           /* B: requests in the step */
  int32_t q_len;           /* L: 1 for decode, 8 for a speculative verify block (causal inside it),
                              more for prefill/extend; with per-request q lengths the largest of them
                              (the problem file's max_seqlen_q) */
  int32_t num_q_heads;     /* Hq */
  int32_t num_kv_heads;    /* Hkv; each serves Hq/Hkv query heads */
  int32_t head_dim;        /* 64 */
  int32_t page_size;       /* cache rows per page */
  int32_t window;          /* 0 = all keys; else a token sees itself and the window-1 keys before it */
  int32_t max_pages;       /* columns of page_table */
  int32_t num_pages;       /* pages in each of k_cache and v_cache (bounds every device access) */
  float rope_theta;        /* 0 = no RoPE (full-attention layers) */
  float qk_scale_factor;   /* folded into the softmax scale */
  float sm_scale;          /* softmax scale before the factor, 1/8 */
  float kv_scale;          /* != 1 selects the scaled cache path (K/V divided by k/v_scale on write) */
  int32_t q_norm;          /* OKC_QNORM_BF16 (0) or OKC_QNORM_FOLDED_SCALE (1), below */
} okc_attn_config;
/*
 * q_norm selects the arithmetic of the q heads' RMSNorm (step 1):
 *  OKC_QNORM_BF16         the problem file's `_prepare_qkv`: q = bf16(x * rstd),
 *                         and qk_scale_factor is folded into the softmax scale
 *                         (softmax_scale = f32(sm_scale * qk_scale_factor));
 *  OKC_QNORM_FOLDED_SCALE the vLLM CuTeDSL `qk_norm` with an output scale
 *                         (`QKNormDirectKernel.kernel`, `qk_norm(x, head_dim,
 *                         eps, scale)`): q = bf16(f32(f32(x * rstd) * qk_scale_factor)),
 *                         the float32 products rounded as float32 and the bf16
 *                         store the only rounding to bf16; the factor is then
 *                         inside q and softmax_scale = sm_scale.
 * k heads are normed with scale 1 in both (the same arithmetic); RoPE, the E4M3
 * casts and the cache layout do not change.
 */
#define OKC_QNORM_BF16 0
#define OKC_QNORM_FOLDED_SCALE 1

/* Optional plan knobs. Pass NULL for the defaults (all zero). */
typedef struct okc_plan_options {
  int32_t chunk_keys;      /* keys per split work item; 0 = the built-in heuristic, else >= 16 */
  int32_t flags;           /* OKC_PLAN_NO_PDL: launch the kernels without programmatic dependent launch;
                              OKC_PLAN_NO_TCGEN05: q_len >= 2 decodes with the warp-level MMA kernel
                              (blocks of up to 16 tokens) instead of the tcgen05 one;
                              OKC_PLAN_STEP_ONE_LAUNCH / OKC_PLAN_STEP_THREE_LAUNCHES: force the form
                              of okc_attn_step at q_len 1 (default: chosen by the plan); the one-
                              kernel form also exists for blocks of 2..8 tokens on the tcgen05
                              kernel (q_len <= 8) and is used only when this flag asks for it;
                              OKC_PLAN_EARLY_GATHER: the caller promises that the kernels launched
                              before okc_attn_step on its stream write neither page_table, the
                              length arrays, nor any K/V cache row the step reads (the QKV
                              projection that precedes the block writes only qkv). The one-kernel
                              step then loads the lengths and page ids and streams the cached keys
                              while its predecessor still runs (programmatic dependent launch);
                              q, the new K/V rows and every write wait for the predecessor as
                              before. Results are unchanged. A step of the same layer that runs
                              right after another one on the same caches breaks the promise (it
                              reads the row the previous step writes): order them with a plain
                              kernel boundary or leave the flag off. */
  int32_t ctas_per_sm;     /* occupancy the split heuristic assumes; 0 = derived from the kernel */
  int32_t sm_count;        /* SMs the split heuristic assumes; 0 = the current device's. With
                              ctas_per_sm also set, planning (okc_attn_plan_sizes,
                              okc_attn_plan_items) makes no CUDA call */
  int32_t max_context;     /* 0: the work list is laid out for the plan's own step. > 0: a
                              fixed-capacity plan for every step whose requests hold at most
                              max_context tokens after it (uniform q_len only): the work list
                              is laid out at the capacity okc_attn_plan_max_sizes gives for
                              max_context, the decode launches cover that capacity and read
                              the live item count from the workspace (CTAs past it return at
                              once), and okc_attn_step keeps the form it was planned with. Every
                              okc_attn_plan_update within max_context then keeps the launches a
                              CUDA graph captured, so graphs replay correctly after any such
                              update (scratch sized by okc_attn_plan_max_sizes). */
} okc_plan_options;
#define OKC_PLAN_NO_PDL 0x1
#define OKC_PLAN_NO_TCGEN05 0x2
#define OKC_PLAN_STEP_ONE_LAUNCH 0x4
#define OKC_PLAN_STEP_THREE_LAUNCHES 0x8
#define OKC_PLAN_EARLY_GATHER 0x10

/* Sizes of the buffers a plan needs. All byte counts are multiples of 256. */
typedef struct okc_attn_sizes {
  size_t workspace_bytes;    /* device workspace the plan is uploaded into (okc_attn_plan) */
  size_t q_fp8_bytes;        /* scratch: E4M3 q [T, Hq, 64], written by prepare, read by decode */
  size_t o_partial_bytes;    /* scratch: f32 per-split outputs [num_work, S*Hq, 64], S the tokens
                                of a query block: min(q_len, 8) on the tcgen05 kernel (q_len >= 2),
                                min(q_len, 16) on the warp-level one */
  size_t lse_partial_bytes;  /* scratch: f32 per-split base-2 log-sum-exp [num_work, S*Hq] */
  int32_t num_work;          /* split work items of this step */
  int32_t num_tokens;        /* T: B*L, or the sum of the q lengths of a varlen plan */
  int32_t max_chunks;        /* largest number of splits of one query block */
  int32_t step_kernels;      /* kernels okc_attn_step launches: 1 (one fused kernel, q_len 1 only)
                                or 3 (prepare, decode, combine) */
} okc_attn_sizes;

typedef struct okc_attn_plan_s* okc_attn_plan_t;

/*
 * Sizes for a step (host only, no GPU work). seq_lens_host: int32 [B], cached
 * tokens per request before this step (the problem file's `Inputs.seq_lens`).
 */
okc_status okc_attn_plan_sizes(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                               const okc_plan_options* opts, okc_attn_sizes* sizes);

/*
 * The split work list a plan made with the same arguments would launch, for
 * inspection (load balance, tests): item i covers keys [first, end) of request
 * `request`, items in launch order, written as items[3*i + 0..2] = request,
 * first key, end key. Keys are counted from the request's first cached token;
 * the ranges assume the device lengths equal seq_lens_host + q_len.
 * `capacity` is the number of items `items` can hold; *count receives the
 * number of items (with items == NULL and capacity 0, only the count).
 * Returns OKC_ERR_WORKSPACE, with *count set, when capacity is too small.
 */
okc_status okc_attn_plan_items(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                               const okc_plan_options* opts, int32_t* items, int32_t capacity,
                               int32_t* count);

/*
 * Prefill / extend: per-request q lengths (the problem file's `Inputs.cu_seqlens_q`
 * with its `max_seqlen_q`). q_lens_host: int32 [B], the new tokens of each
 * request in this step, each in [0, cfg->q_len] (cfg->q_len is their largest
 * value; 0: the request takes no part); NULL = q_len each, which makes every
 * call below the same as its form without q lengths. The step's T is the sum of
 * the q lengths; request b's new tokens sit at positions seq_lens_host[b] + i,
 * i < q_lens_host[b], each attending causally to every earlier key and to the
 * block's earlier tokens (window: the window - 1 keys before it). A request's
 * new tokens are cut into query blocks of S consecutive tokens (okc_attn_sizes)
 * and every block's keys into split work items. The device inputs must agree:
 * cu_seqlens_q = 0 then the running sums of q_lens_host, cache_seqlens[b] =
 * seq_lens_host[b] + q_lens_host[b]; kernels that find other q lengths flag
 * OKC_DEVERR_LENGTHS. okc_attn_plan_items_varlen writes 4 ints per item:
 * request, first token of its block (within the request), first key, end key.
 * okc_attn_plan_update_varlen re-plans in place with new q lengths (a
 * fixed-capacity plan takes none: OKC_ERR_UNSUPPORTED); okc_attn_plan_update
 * keeps the plan's q lengths.
 */
okc_status okc_attn_plan_sizes_varlen(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                                      const int32_t* q_lens_host, const okc_plan_options* opts,
                                      okc_attn_sizes* sizes);
okc_status okc_attn_plan_items_varlen(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                                      const int32_t* q_lens_host, const okc_plan_options* opts, int32_t* items,
                                      int32_t capacity, int32_t* count);
okc_status okc_attn_plan_varlen(const okc_attn_config* cfg, const int32_t* seq_lens_host, const int32_t* q_lens_host,
                                const okc_plan_options* opts, void* workspace, size_t workspace_bytes,
                                okc_stream stream, okc_attn_plan_t* plan_out);

/*
 * Upper bounds of okc_attn_plan_sizes over every step of this config whose
 * requests each hold at most max_context tokens after the step
 * (seq_lens_host[b] + q_len <= max_context), under the same options and on
 * the same device: buffers of these sizes serve all such steps, so a plan
 * made in a workspace of workspace_bytes never fails okc_attn_plan_update
 * with OKC_ERR_WORKSPACE on them, and scratch of these sizes never needs to
 * grow. num_work and max_chunks are bounds as well; num_tokens is exact;
 * step_kernels is 0 (it depends on the lengths). Host only (no GPU work; the
 * device is queried for its SM count and occupancy unless opts give both).
 * Returns OKC_ERR_INVALID when max_context < q_len or max_context exceeds
 * max_pages * page_size.
 */
okc_status okc_attn_plan_max_sizes(const okc_attn_config* cfg, int32_t max_context, const okc_plan_options* opts,
                                   okc_attn_sizes* sizes);
/* The workspace bound of okc_attn_plan_max_sizes with the default options. */
okc_status okc_attn_plan_workspace_size(const okc_attn_config* cfg, int32_t max_total_ctx, size_t* bytes);

/*
 * okc_attn_plan — the per-step plan ("Differs from SGLang" note of the problem
 * file: positions, cache rows, lengths and the attention schedule are built once
 * per step for all layers). Validates cfg, splits every request's visible keys
 * into work items (the split count grows with the parallelism B*Hkv leaves idle
 * on the GPU and shrinks with the window, as the problem file's local-splits
 * bound does for H200), and copies the work list into `workspace` with an
 * asynchronous host-to-device copy on `stream`; it also zeroes the device error
 * word. Run it outside CUDA-graph capture. The workspace must stay allocated and
 * unmodified while kernels of this plan may run. Kernels read every per-request
 * length from device memory; a captured graph stays valid for any later step
 * whose lengths still fit this plan's splits (otherwise OKC_DEVERR_LENGTHS).
 * workspace: device, >= okc_attn_sizes.workspace_bytes, 256-byte aligned.
 * On success *plan_out owns host memory released by okc_attn_plan_destroy.
 */
okc_status okc_attn_plan(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                         const okc_plan_options* opts, void* workspace, size_t workspace_bytes,
                         okc_stream stream, okc_attn_plan_t* plan_out);
/* okc_attn_plan with the default options. */
okc_status okc_attn_plan_create(const okc_attn_config* cfg, const int32_t* seq_lens_host, void* workspace,
                                size_t workspace_bytes, okc_stream stream, okc_attn_plan_t* plan_out);
/*
 * Re-plans an existing plan in place for the next step's host lengths (same
 * config, options and workspace): the split list is recomputed and uploaded
 * asynchronously on `stream`, like okc_attn_plan, without creating a plan. The
 * first call allocates a page-locked staging buffer for the upload (freed by
 * okc_attn_plan_destroy); later calls allocate nothing while the head fits it,
 * and wait for the staging buffer's previous copy before reusing it. The
 * scratch sizes may change with the lengths: read them with
 * okc_attn_plan_get_sizes. Returns OKC_ERR_WORKSPACE, leaving the plan as it
 * was, when the new plan needs a larger workspace than the plan was made with
 * (okc_attn_plan_max_sizes gives a workspace that never does). After
 * OKC_ERR_CUDA the plan may no longer match its workspace: destroy it.
 * The workspace is overwritten in stream order: kernels of the previous step
 * issued on other streams must be ordered before the call. The device error
 * word is not part of the upload: bits set by earlier steps stay until
 * okc_attn_plan_clear_errors (or a new okc_attn_plan) clears them.
 * CUDA graphs: a launch captured in a graph keeps the grid size and the
 * workspace offsets of the plan as it was at capture. On a fixed-capacity plan
 * (okc_plan_options.max_context) neither ever changes, so a graph captured
 * once replays correctly after every update within max_context. On other
 * plans, replaying after an update is valid only while num_work is unchanged
 * (the work list and block table then keep their offsets); after an update
 * that changed num_work, capture again before replaying.
 */
okc_status okc_attn_plan_update(okc_attn_plan_t plan, const int32_t* seq_lens_host, okc_stream stream);
okc_status okc_attn_plan_update_varlen(okc_attn_plan_t plan, const int32_t* seq_lens_host,
                                       const int32_t* q_lens_host, okc_stream stream);

okc_status okc_attn_plan_destroy(okc_attn_plan_t plan);
/* The plan's sizes: the workspace it needs and the caller's scratch (q_fp8 and
   the split partials) for its step. okc_attn_plan_scratch_sizes is the same call. */
okc_status okc_attn_plan_get_sizes(okc_attn_plan_t plan, okc_attn_sizes* sizes);
okc_status okc_attn_plan_scratch_sizes(okc_attn_plan_t plan, okc_attn_sizes* sizes);
/* Synchronizes `stream`, then reads and returns the OKC_DEVERR_* bits seen so
   far: every bit the plan's kernels set since okc_attn_plan made the plan or
   okc_attn_plan_clear_errors last cleared them (okc_attn_plan_update keeps them). */
okc_status okc_attn_plan_read_errors(okc_attn_plan_t plan, okc_stream stream, uint32_t* flags_host);
/* Zeroes the plan's device error word, asynchronously on `stream` (ordered after
   the kernels issued before it on that stream). */
okc_status okc_attn_plan_clear_errors(okc_attn_plan_t plan, okc_stream stream);

/*
 * RoPE cos|sin table, built once per theta like the problem file's `_cos_sin`:
 * table[pos][0:32] = cos(pos * inv_freq), table[pos][32:64] = sin(pos * inv_freq),
 * inv_freq[i] = 1 / theta^(2i/64), all as float32 with the products and the
 * power rounded to float32 and cos/sin the float32 rounding of the exact value.
 * table: device float32 [num_positions, 64]; num_positions in [1, 2^21].
 */
okc_status okc_rope_table_init(float rope_theta, int32_t num_positions, float* table,
                               okc_stream stream);

/*
 * Steps 1-3 (the problem file's `_prepare_qkv` kernel). For every token and
 * every q and k head: float32 RMSNorm of the bf16 head (eps 1e-5), rounded to
 * bf16; if rope_theta != 0, interleaved RoPE on pairs (2i, 2i+1) at the token's
 * position, rounded to bf16. q is stored as E4M3 (no scale). k, and the raw v
 * heads, are divided by k_scale / v_scale and rounded to bf16 when the config is
 * scaled, then stored as E4M3 (round to nearest even, saturating to +-448) in
 * the cache row cache_loc[t].
 *  qkv        bf16 [T, (2Hq+2Hkv)*64], row stride (2Hq+2Hkv)*64, 16-byte aligned
 *  positions  int64 [T]; cache_loc int64 [T] (flat cache row)
 *  k_cache/v_cache  e4m3 pool, written in place at the cache_loc rows only
 *  k_scale/v_scale  device float32 scalars; read only when the config is scaled
 *  rope_table float32 [rope_positions, 64] from okc_rope_table_init, or NULL
 *             when rope_theta == 0
 *  q_fp8      scratch, >= okc_attn_sizes.q_fp8_bytes
 * T == 0 returns OKC_OK without a launch.
 */
okc_status okc_prepare_qkv(okc_attn_plan_t plan, const void* qkv, const int64_t* positions,
                           const int64_t* cache_loc, uint8_t* k_cache, uint8_t* v_cache,
                           const float* k_scale, const float* v_scale, const float* rope_table,
                           int32_t rope_positions, uint8_t* q_fp8, okc_stream stream);

/*
 * Step 4 (the problem file's flash_attn_with_kvcache call: paged, causal,
 * window_size (window-1, 0) or (-1,-1), softmax_scale = sm_scale*qk_scale_factor,
 * k/v descale when scaled). Query i of request b sits at position
 * cache_seqlens[b] - q_len_b + i and sees keys j with max(0, p-window+1) <= j <= p
 * (window 0: 0 <= j <= p); query head h reads KV head h / (Hq/Hkv). Each work item
 * of the plan covers a key range of one query block (the whole request for
 * decode and verify steps; S consecutive tokens of a longer one) for all its
 * query rows and both KV heads, and writes a normalized f32 partial output
 * (already times v_scale) and its base-2 log-sum-exp. q_len >= 2 runs on the
 * tcgen05 kernel (blocks of up to 8 tokens as M = 128 query rows, or past q_len 8
 * blocks of up to 16 tokens with M = 128 rows per KV head; accumulators in
 * tensor memory; on pages of 8 or more rows its K/V tiles arrive by TMA through
 * tensor maps the call encodes for k_cache and v_cache, so page_size *
 * num_pages rows must be addressable from both base pointers) unless the plan
 * was made with OKC_PLAN_NO_TCGEN05 (then blocks of up to 16 tokens on the
 * warp-level MMA kernel, which also runs q_len 1).
 *  q_fp8          from okc_prepare_qkv
 *  page_table     int32 [B, max_pages]
 *  cache_seqlens  int32 [B] = seq_lens + L; cu_seqlens_q int32 [B+1] = 0, L, 2L, ...
 *                 (varlen plans: seq_lens + q_lens and the running sums of q_lens)
 *  seq_lens       int32 [B] (checked against cache_seqlens; may be NULL)
 *  o_partial/lse_partial  scratch, >= the plan's sizes
 */
okc_status okc_attn_decode(okc_attn_plan_t plan, const uint8_t* q_fp8, const uint8_t* k_cache,
                           const uint8_t* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* page_table, const int32_t* cache_seqlens,
                           const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                           float* o_partial, float* lse_partial, okc_stream stream);

/*
 * Split merge fused with step 5 (the problem file's rms_norm_gate call, weight
 * None, has_norm, eps 1e-5). Per token and q head: o = log-sum-exp merge of the
 * request's splits, ob = bf16(o), out = bf16(ob * rsqrt(mean(ob^2) + eps) * w *
 * sigmoid(gate)) with gate = qkv[t, (Hq+2Hkv)*64 + h*64 + c] read in place.
 *  norm_weight  bf16 [64] or NULL (NULL = the problem file's weight None)
 *  out          bf16 [T, Hq*64]
 */
okc_status okc_attn_combine_normgate(okc_attn_plan_t plan, const float* o_partial,
                                     const float* lse_partial, const void* qkv,
                                     const void* norm_weight, float eps, void* out,
                                     okc_stream stream);

/*
 * okc_attn_step — the whole block in ONE launch: steps 1-3 (the
 * `_prepare_qkv` arithmetic, bit-identical to okc_prepare_qkv), step 4 and the
 * split merge with step 5 (bit-identical to okc_attn_combine_normgate). Each
 * decode CTA derives its q heads from qkv; the CTA whose key range holds a new
 * token's key computes that K/V row, uses it in place and writes it to the
 * cache at cache_loc; the last CTA of each request to finish (an atomic ticket
 * in the plan workspace, reset after use; no CTA waits on another) merges the
 * request's splits and writes `out`. The plan chooses this one-kernel form for
 * q_len 1 when its work list fills at least half of the GPU's resident CTA
 * slots with chunks of at most 2048 keys or takes more than one wave of them
 * (sizes.step_kernels == 1, or forced by OKC_PLAN_STEP_ONE_LAUNCH). For
 * q_len 2..8 on the tcgen05 kernel (one query block per request) the same form
 * runs only under OKC_PLAN_STEP_ONE_LAUNCH (measured slower on the verify
 * block than the three kernels). Otherwise, and always for q_len > 8 or the
 * warp-level kernel, the call runs the three kernels, keeping q in the plan
 * workspace. Either way the results equal the three calls' bit for bit.
 * Arguments: those of the three calls, minus q_fp8. cache_loc[t] must be the
 * page-table row of token t's position (the kernel uses the computed row
 * directly instead of reading it back).
 */
okc_status okc_attn_step(okc_attn_plan_t plan, const void* qkv, const int64_t* positions,
                         const int64_t* cache_loc, uint8_t* k_cache, uint8_t* v_cache, const float* k_scale,
                         const float* v_scale, const float* rope_table, int32_t rope_positions,
                         const int32_t* page_table, const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                         const int32_t* seq_lens, const void* norm_weight, float eps, float* o_partial,
                         float* lse_partial, void* out, okc_stream stream);

/*
 * One step from host buffers: the per-step inputs live in host memory, the
 * caches, scales, RoPE table, norm weight and scratch stay resident on the
 * device. The call runs okc_attn_step on the inputs and synchronizes `stream`:
 * on OKC_OK the output is in out_host. A host buffer in page-locked memory
 * that the device can address (cudaHostAlloc / cudaMallocHost, or
 * cudaHostRegister'ed with mapping; unified addressing maps them by default)
 * is read by the kernels in place, over the host link, and out_host is then
 * written in place: no copy. Any other host buffer (pageable memory, or qkv /
 * out_host not 16-byte aligned) is copied with cudaMemcpyAsync to its device
 * buffer first (out: from its device buffer afterwards); device buffers of
 * mapped host buffers are left untouched. Device buffers are caller-owned and
 * sized as the host ones: qkv bf16 [T, (2Hq+2Hkv)*64]; positions / cache_loc
 * int64 [T]; cache_seqlens, seq_lens int32 [B]; cu_seqlens_q int32 [B+1];
 * page_table int32 [B, max_pages]; out bf16 [T, Hq*64]. positions (and its
 * host copy) may be NULL when rope_theta == 0, seq_lens when unchecked; each
 * pair is NULL together or not at all. The host buffers must not change until
 * the call returns.
 */
typedef struct okc_host_step {
  const void* qkv_host;
  const int64_t* positions_host;
  const int64_t* cache_loc_host;
  const int32_t* cache_seqlens_host;
  const int32_t* cu_seqlens_q_host;
  const int32_t* seq_lens_host;
  const int32_t* page_table_host;
  void* out_host;
  void* qkv;
  int64_t* positions;
  int64_t* cache_loc;
  int32_t* cache_seqlens;
  int32_t* cu_seqlens_q;
  int32_t* seq_lens;
  int32_t* page_table;
  void* out;
} okc_host_step;
okc_status okc_attn_step_host(okc_attn_plan_t plan, const okc_host_step* io, uint8_t* k_cache, uint8_t* v_cache,
                              const float* k_scale, const float* v_scale, const float* rope_table,
                              int32_t rope_positions, const void* norm_weight, float eps, float* o_partial,
                              float* lse_partial, okc_stream stream);

const char* okc_status_string(okc_status status);

/*
 * Diagnostic of the kernels' bounded waits on the current device: one warp
 * waits on a shared-memory mbarrier that nothing arrives on, with the same
 * bounded wait every kernel uses but a limit of limit_us microseconds (at
 * least 4096 polls), ORs OKC_DEVERR_TIMEOUT into *err when the wait gives up,
 * and returns: the launch completes and the context stays usable. Nothing
 * faults and nothing hangs. err: device, one uint32, not cleared by the call.
 * Asynchronous on `stream`. Returns OKC_ERR_INVALID for a null err or a limit
 * outside [1, 1000000] us (checked before any GPU work).
 */
okc_status okc_selftest_bounded_wait(uint32_t* err, int32_t limit_us, okc_stream stream);

/*
 * okc_attn_decode_combine_noalloc — okc_attn_decode followed by
 * okc_attn_combine_normgate, for callers that cannot allocate device memory.
 * "012-attention-local-splits.py" has no counterpart of this entry point.
 *
 * Who needs it: an op hosted inside a framework that owns every device
 * allocation and hands the op only its input and output buffers (a plugin or
 * custom-op interface with no workspace), or code that must not trigger the
 * device-wide synchronisation that cudaMalloc/cudaFree can cause. This call
 * takes no plan, workspace or scratch buffer: the work list, the per-request
 * table and the split partials live in one static device array of 8 MiB inside
 * the library, which every GPU that loads the library holds until the process
 * exits. It calls no allocating routine (no cudaMalloc, cudaFree or other CUDA
 * allocating routine); its host-side work list is ordinary heap memory. The
 * array takes its device memory when the CUDA runtime loads the library's
 * device code on a device: at the first call on that device under lazy module
 * loading (the CUDA default), or when the library loads with
 * CUDA_MODULE_LOADING=EAGER; later calls leave the device's free memory as it is.
 *
 * Arguments are those of okc_attn_plan (cfg, seq_lens_host), okc_attn_decode and
 * okc_attn_combine_normgate; q_fp8 must already hold okc_prepare_qkv's output.
 * The result equals the three-call path's `out` for the same inputs.
 * Limits: at most 2048 requests and 4096 split work items, and the partials
 * (work items x S*16 rows x 260 bytes, S the plan's block tokens, plus the
 * tables) must fit in 8 MiB;
 * larger steps return OKC_ERR_WORKSPACE before any GPU work. Device-side range
 * errors are skipped as in okc_attn_decode but not reported (there is no plan
 * error word).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any stream
 * capture. All calls share the one array, which keeps the last call's contents:
 * calls that may overlap on the GPU (different streams without ordering, or
 * several host threads) race on it, so serialise them on one stream.
 */
okc_status okc_attn_decode_combine_noalloc(
    const okc_attn_config* cfg, const int32_t* seq_lens_host, const uint8_t* q_fp8,
    const uint8_t* k_cache, const uint8_t* v_cache, const float* k_scale, const float* v_scale,
    const int32_t* page_table, const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
    const int32_t* seq_lens, const void* qkv, const void* norm_weight, float eps, void* out,
    okc_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* OKC_ATTN_H */
