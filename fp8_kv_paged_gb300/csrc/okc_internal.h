// okc_internal.h — what the library's translation units share: the plan
// object, the kernel argument blocks and the launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "okc_attn.h"

namespace okc {

// Workspace layout (device, caller-owned):
//   [header | work list | block table | arrival counters | q (three-kernel step)]
// The header holds the device error word at byte 0 and the live work-item count
// at byte kWsCount; plans upload everything from kWsCount on, so the error word
// keeps what the kernels set.
constexpr size_t kWsHeader = 256;
constexpr size_t kWsCount = 64;

// A query block: up to S consecutive new tokens of one request, the unit whose
// q rows one decode CTA holds (S = 1 for q_len 1; 8 on the tcgen05 kernel, the
// 128 rows of its M = 128 operand; up to 16 on the warp-level MMA kernel). A
// request of ql new tokens has ceil(ql / S) blocks; decode and verify steps have
// one block per request.
//
// One split work item: keys [j0, j1) (under the plan's lengths; the kernel
// starts loading page ids with them) for query block tokens [i0, i0 + ntok) of
// request b, token t0 of the step its first (under the plan's q lengths). The
// kernel derives its keys from the device lengths: [lo + koff, min(hi, lo +
// koff + cap)) for the block's visible range [lo, hi), and checks that the
// block's items still cover it; cap is the item's key count, or more for a
// block's last item (the room the plan's chunking leaves for longer device
// lengths). Its output slot is wbase + chunk; nchunks and wbase repeat the
// block's split; `last` marks the request's last block.
struct WorkItem {
  int32_t b, koff, i0, ntok;
  int32_t chunk, j0, j1, cap;
  int32_t nchunks, wbase, t0, last;
};
// Per query block: first output slot, number of splits, first token of the
// step and tokens in the block (the merge's view).
struct BlockInfo {
  int32_t wbase, nchunks, t0, ntok;
};

struct PrepareArgs {
  const uint16_t* qkv;  // bf16 bits [T, width]
  const int64_t* positions;
  const int64_t* cache_loc;
  uint8_t* kc;
  uint8_t* vc;
  const float* k_scale;
  const float* v_scale;
  const float* rope_table;  // [rope_positions, 64] or null
  uint8_t* q8;              // [T, Hq, 64]
  unsigned* err;
  int64_t num_rows;  // num_pages * page_size
  int32_t T;
  int32_t rope_positions;
  int32_t rope;
  int32_t scaled;
  int32_t q_fold;  // OKC_QNORM_FOLDED_SCALE: q heads are x * rstd * q_scale in float32, then bf16
  float q_scale;   // qk_scale_factor under q_fold
};

struct DecodeArgs {
  const uint8_t* q8;
  const uint8_t* kc;
  const uint8_t* vc;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  const int32_t* cache_seqlens;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const WorkItem* work;
  const int32_t* live_work;  // fixed-capacity plans: the live item count (CTAs past it return); else null
  float* o_part;
  float* lse_part;
  unsigned* err;
  int32_t batch, L, window, max_pages, num_pages, page_shift, scaled, T;
  int32_t S;         // tokens per query block (rows per output slot: S * Hq)
  float scale_log2;  // softmax scale in base 2 (softmax_scale_log2)
  // ---- the fused step only (okc_attn_step): steps 1-3 and 5 inside the kernel
  const uint16_t* qkv;      // bf16 bits [T, width]
  const int64_t* positions;
  const int64_t* cache_loc;
  uint8_t* kc_w;            // the caches again, written at the new tokens' rows
  uint8_t* vc_w;
  const float* rope_table;  // [rope_positions, 64] or null
  int32_t rope_positions;
  int32_t rope;
  int64_t num_rows;         // num_pages * page_size
  int32_t* tickets;         // [B] arrival counters (per request), zero between launches
  const uint16_t* weight;   // norm-gate weight bf16 [64] or null
  uint16_t* out;            // bf16 [T, Hq*64]
  float eps;
  int32_t tc;               // 1: blocks of 2..16 tokens run on the tcgen05 kernel (decode_tc.cu)
  int32_t tc_groups;        // its form (tc_groups: 2, or 3 for one softmax warpgroup per KV head)
  int32_t q_fold;           // as PrepareArgs (the fused step derives q itself)
  float q_scale;
  int32_t early;            // OKC_PLAN_EARLY_GATHER: the fused step loads lengths, page ids and
                            // cached keys before the programmatic-dependency wait
  int32_t one_wave;         // the fused q_len-1 step: at most one wave of work items
};

struct CombineArgs {
  const float* o_part;
  const float* lse_part;
  const uint16_t* qkv;
  const uint16_t* weight;  // bf16 [64] or null
  uint16_t* out;
  const BlockInfo* blk;
  unsigned* err;
  int32_t nblocks, S, T;
  float eps;
};

}  // namespace okc

struct okc_attn_plan_s {
  okc_attn_config cfg;
  okc_plan_options opts;
  okc_attn_sizes sizes;
  std::vector<okc::WorkItem> work;
  std::vector<okc::BlockInfo> blocks;
  std::vector<okc::WorkItem> spare_work;    // okc_attn_plan_update: the lists replaced by the
  std::vector<okc::BlockInfo> spare_blocks; // last update, reused for the next one's capacity
  std::vector<int32_t> q_lens;  // the step's q lengths when given per request (else empty: q_len each)
  std::vector<uint8_t> upload;  // the workspace head as uploaded (one host-to-device copy)
  void* workspace;
  size_t workspace_bytes;
  int slots;                    // resident CTA slots the splits were made for
  int S;                        // tokens per query block
  int64_t work_cap;             // fixed-capacity plans: items the work list is laid out for (else 0)
  // okc_attn_plan_update: a page-locked staging buffer for the upload (grown on
  // demand) and the event of its last copy (the buffer is reused after it)
  void* pinned = nullptr;
  size_t pinned_bytes = 0;
  cudaEvent_t pinned_done = nullptr;
  unsigned* d_err;
  int32_t* d_live;     // the live work-item count in the header
  okc::WorkItem* d_work;
  okc::BlockInfo* d_blk;
  int32_t* d_tickets;  // the fused step's per-request arrival counters
  uint8_t* d_q8;       // q of okc_attn_step when it runs the three kernels
  bool tc;             // decode on the tcgen05 kernel (q_len >= 2: blocks of 2..16 tokens)
  int device;
  int sm_count;
  bool pdl;
  float scale_log2;
};

namespace okc {

// The softmax scale in base 2: f32(sm_scale * qk_scale_factor) * log2(e) under
// OKC_QNORM_BF16 (the factor folded into the scale, as the problem file does),
// f32(sm_scale) * log2(e) under OKC_QNORM_FOLDED_SCALE (the factor is inside q).
inline float softmax_scale_log2(const okc_attn_config& c) {
  const float scale = c.q_norm == OKC_QNORM_FOLDED_SCALE ? c.sm_scale
                                                          : (float)((double)c.sm_scale * (double)c.qk_scale_factor);
  return (float)((double)scale * 1.4426950408889634);
}

// The step's q_len >= 2 blocks decode on the tcgen05 kernel unless the options say not to.
inline bool uses_tc(const okc_attn_config& c, const okc_plan_options* o) {
  return c.q_len >= 2 && !(o && (o->flags & OKC_PLAN_NO_TCGEN05));
}
// The form of the tcgen05 kernel (decode_tc.cu): 2 (two softmax warpgroups on
// alternate tiles, one CTA per SM, blocks of up to 8 tokens x 16 heads as the
// M = 128 rows) for steps of at most 8 tokens per request (decode, verify: few
// blocks, many splits, where fewer, longer splits merge faster), 3 (one
// warpgroup per KV head, blocks of 16 tokens: each group's M = 128 rows are 16
// tokens x its 8 heads, half the tensor work per row) for longer extends.
inline int tc_groups(const okc_attn_config& c) { return c.q_len > 8 ? 3 : 2; }
// Tokens per query block: 1 for q_len 1, 8 on the tcgen05 kernel's form 2,
// 16 on its form 3 and on the warp-level kernel; q_len itself when smaller.
inline int block_tokens(const okc_attn_config& c, const okc_plan_options* o) {
  const int smax = uses_tc(c, o) && c.q_len <= 8 ? 8 : 16;
  return c.q_len < smax ? c.q_len : smax;
}

// Keys per split work item for a block of `nvis` visible keys split `k` ways:
// nvis / k rounded up so that the item's 64-key tiles are whole ones, counting
// the up to `pad` keys before the item that a tile start rounded down to a
// multiple of 8 adds (7 for the TMA-fed tcgen05 decode, else 0). No item gets
// more tiles than unrounded, and the last item of a block is shorter, so a
// block takes no more tiles in all.
inline int64_t split_chunk_keys(int64_t nvis, int64_t k, int64_t pad) {
  const int64_t x = (nvis + k - 1) / k;
  const int64_t r = (x + pad + 63) / 64 * 64 - pad;
  return r > 64 - pad ? r : 64 - pad;
}

// A step's split: the work items in launch order, the per-block table, the
// largest number of items of one block and of keys of one item, the step's
// tokens and the tokens per block.
struct SplitResult {
  std::vector<WorkItem> work;
  std::vector<BlockInfo> blocks;
  int max_chunks = 0;
  int64_t max_chunk_keys = 0;
  int64_t tokens = 0;
  int S = 1;
};
// The plan's split rule (okc_api.cu): every query block's visible keys into work
// items for `slots` resident CTA slots, under the plan options (may be null).
// q_lens: new tokens per request (null: cfg->q_len each).
okc_status make_splits(const okc_attn_config* c, const int32_t* seq, const int32_t* q_lens, const okc_plan_options* o,
                       int slots, SplitResult* r);

// Kernel launchers (each returns the cudaError_t of its launch).
cudaError_t launch_prepare(const PrepareArgs& a, bool pdl, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s);
// The whole step in one launch for q_len 1 (q from qkv, new K/V rows,
// attention, last-CTA merge).
cudaError_t launch_step_fused(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs& a, bool pdl, cudaStream_t s);
cudaError_t launch_rope_table(float theta, const float* inv_freq, int32_t n, float* table,
                              cudaStream_t s);
// Resident CTAs per SM of the decode kernels for blocks of S tokens (tc: the
// tcgen05 kernel for blocks of 2..8), the lower of the three-call and the fused
// variant (0 on error).
int decode_ctas_per_sm(int S, bool tc, int tc_groups);
// decode_ctas_per_sm for device `dev`, queried once per (device, S, tc,
// tc_groups) and cached (the query also raises the kernels' shared-memory limit
// on the device).
int cached_ctas_per_sm(int dev, int S, bool tc, int tc_groups);
// The tcgen05 decode kernel for blocks of 2..16 tokens (decode_tc.cu) in form
// a.tc_groups.
cudaError_t launch_decode_tc(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s);
// The whole step in one launch for blocks of 2..8 tokens on the tcgen05 kernel
// (q and the new K/V rows from qkv, attention, last-CTA merge and norm-gate);
// requires L == S (one block per request) and two softmax groups.
cudaError_t launch_step_fused_tc(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s);
int decode_tc_ctas_per_sm(int tc_groups);

}  // namespace okc
