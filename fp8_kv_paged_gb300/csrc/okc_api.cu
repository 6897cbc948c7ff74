// okc_api.cu — the C ABI declared in okc_attn.h: argument validation, the
// per-step plan (split work list, workspace layout), and the launches.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>
#include <vector>

#include "okc_common.cuh"
#include "okc_internal.h"

using okc::make_splits;
using okc::BlockInfo;
using okc::SplitResult;
using okc::WorkItem;

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

okc_status check_config(const okc_attn_config* c) {
  if (!c) return OKC_ERR_INVALID;
  if (c->batch < 0 || c->q_len < 1 || c->q_len > okc::kMaxQLen) return OKC_ERR_INVALID;
  if (c->num_q_heads <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0) return OKC_ERR_INVALID;
  if (c->num_q_heads % c->num_kv_heads != 0) return OKC_ERR_INVALID;
  if (c->window < 0 || c->max_pages < 1 || c->num_pages < 1 || c->page_size < 1) return OKC_ERR_INVALID;
  if (!(c->rope_theta >= 0.f) || !std::isfinite(c->rope_theta)) return OKC_ERR_INVALID;
  if (!(c->sm_scale > 0.f) || !(c->qk_scale_factor > 0.f) || !(c->kv_scale > 0.f)) return OKC_ERR_INVALID;
  if (!std::isfinite(c->sm_scale) || !std::isfinite(c->qk_scale_factor) || !std::isfinite(c->kv_scale))
    return OKC_ERR_INVALID;
  if (c->q_norm != OKC_QNORM_BF16 && c->q_norm != OKC_QNORM_FOLDED_SCALE) return OKC_ERR_INVALID;
  if (c->head_dim != okc::kHeadDim || c->num_q_heads != okc::kNumQHeads ||
      c->num_kv_heads != okc::kNumKvHeads)
    return OKC_ERR_UNSUPPORTED;
  if (!is_pow2(c->page_size) || c->page_size > 256) return OKC_ERR_UNSUPPORTED;
  // every flat cache row and page-table index must fit the kernels' int32 key math
  if ((int64_t)c->max_pages * c->page_size > (int64_t)1 << 30) return OKC_ERR_UNSUPPORTED;
  // token counts (grids of one CTA per token, int32 sizes) stay far below 2^31
  if ((int64_t)c->batch * c->q_len > (int64_t)1 << 26) return OKC_ERR_UNSUPPORTED;
  return OKC_OK;
}

int page_shift(int P) {
  int s = 0;
  while ((1 << s) < P) s++;
  return s;
}

}  // namespace

// Split every query block's visible keys into work items. Request b's ql new
// tokens sit at positions seq[b] .. seq[b] + ql - 1 and form ceil(ql / S)
// blocks of S consecutive tokens (S from block_tokens). Block [i0, i0 + ntok)
// sees keys [lo, hi): hi = seq + i0 + ntok, lo = max(0, seq + i0 - window + 1)
// on window layers (the union of its queries' windows), else 0. The split count
// follows the parallelism the batch leaves idle: as many items as the GPU has
// resident CTA slots (SMs x CTAs per SM, both read at run time), never below
// 128 keys per item unless the block is shorter, so short or windowed blocks
// get few splits and long ones many (the H200 bound cdiv(132, B*Hkv) of
// "012-attention-local-splits.py" plays the same role with a fixed SM count).
// The tail of a work list of more than one wave in finer items. Items start
// in launch order as resident CTA slots free up, and equal items do not run at
// equal speed (the CTAs on an SM share its bandwidth), so the items that
// start last decide the step's end: the items that would start in the last
// kTailPct percent of the work (each item counted with `item_cost` keys on top
// of its own) are cut into up to kTailParts items of at least kTailMinKeys
// keys each, at whole 64-key tiles from the item's start, within the list's
// capacity `wcap`, and the tail is put back in largest-first order. A block's
// items stay contiguous in slot order: slots, chunk numbers and counts are
// renumbered by one prefix sum over the pieces per original slot, and a
// block's last piece keeps the room its last item had for longer device
// lengths.
#ifndef OKC_TAIL_PCT
#define OKC_TAIL_PCT 30
#endif
#ifndef OKC_TAIL_PARTS
#define OKC_TAIL_PARTS 3
#endif
namespace {
constexpr int kTailPct = OKC_TAIL_PCT, kTailParts = OKC_TAIL_PARTS;
constexpr int64_t kTailMinKeys = 256;

void split_tail(okc::SplitResult* r, int64_t wcap, int slots, int64_t item_cost) {
  std::vector<WorkItem>& work = r->work;
  const int64_t W = (int64_t)work.size();
  if (kTailPct <= 0 || kTailParts < 2 || W <= slots || W >= wcap) return;
  int64_t total = 0;
  for (const WorkItem& w : work) total += (int64_t)(w.j1 - w.j0) + item_cost;
  // pieces per original slot (the list holds slots 0 .. W-1 once each)
  std::vector<int32_t> parts((size_t)W + 1, 1);
  const int64_t start_tail = total - total * kTailPct / 100;
  int64_t before = 0, added = 0;
  for (const WorkItem& w : work) {
    const int64_t n = (int64_t)(w.j1 - w.j0);
    if (before >= start_tail) {
      const int64_t p = std::min<int64_t>(kTailParts, n / std::max<int64_t>(kTailMinKeys, 64));
      if (p >= 2 && W + added + p - 1 <= wcap) {
        parts[(size_t)(w.wbase + w.chunk)] = (int32_t)p;
        added += p - 1;
      }
    }
    before += n + item_cost;
  }
  if (added == 0) return;
  // first new slot of each original slot (exclusive prefix sum)
  std::vector<int32_t> first((size_t)W + 1);
  int32_t acc = 0;
  for (int64_t s = 0; s < W; s++) {
    first[(size_t)s] = acc;
    acc += parts[(size_t)s];
  }
  first[(size_t)W] = acc;
  for (okc::BlockInfo& q : r->blocks) {
    const int32_t w0 = first[(size_t)q.wbase], w1 = first[(size_t)(q.wbase + q.nchunks)];
    q.wbase = w0;
    q.nchunks = w1 - w0;
    r->max_chunks = std::max(r->max_chunks, (int)q.nchunks);
  }
  std::vector<WorkItem> out;
  out.reserve((size_t)acc);
  size_t tail_from = 0;  // the first piece of a split item (the tail starts there)
  bool in_tail = false;
  for (const WorkItem& w : work) {
    const int32_t old_slot = w.wbase + w.chunk, p = parts[(size_t)old_slot];
    const int32_t wbase = first[(size_t)w.wbase];
    const int32_t nchunks = first[(size_t)(w.wbase + w.nchunks)] - wbase;
    const int64_t n = (int64_t)(w.j1 - w.j0);
    if (p > 1 && !in_tail) {
      in_tail = true;
      tail_from = out.size();
    }
    for (int32_t q = 0; q < p; q++) {
      WorkItem x = w;
      const int64_t a = n * q / p / 64 * 64, b = q + 1 < p ? n * (q + 1) / p / 64 * 64 : n;
      x.j0 = w.j0 + (int32_t)a;
      x.j1 = w.j0 + (int32_t)b;
      x.koff = w.koff + (int32_t)a;
      x.cap = q + 1 < p ? (int32_t)(b - a) : w.cap - (int32_t)a;  // the last piece keeps the item's end room
      x.chunk = first[(size_t)old_slot] - wbase + q;
      x.wbase = wbase;
      x.nchunks = nchunks;
      out.push_back(x);
    }
  }
  // the tail largest first (ties: launch order)
  std::stable_sort(out.begin() + (std::ptrdiff_t)tail_from, out.end(),
                   [](const WorkItem& x, const WorkItem& y) { return x.j1 - x.j0 > y.j1 - y.j0; });
  work.swap(out);
}
}  // namespace

okc_status okc::make_splits(const okc_attn_config* c, const int32_t* seq, const int32_t* q_lens,
                            const okc_plan_options* o, int slots, SplitResult* r) {
  const int B = c->batch, Lmax = c->q_len;
  if (o && o->chunk_keys != 0 && o->chunk_keys < 16) return OKC_ERR_INVALID;
  const int S = okc::block_tokens(*c, o);
  r->S = S;
  r->max_chunks = 0;
  r->max_chunk_keys = 0;
  // ---- the query blocks (units of the split): request, first token, tokens,
  // first token of the step, key range end and visible keys
  struct Unit {
    int32_t b, i0, ntok, t0, last;
    int64_t hi, nvis;
  };
  std::vector<Unit> units;
  units.reserve((size_t)B * (size_t)((Lmax + S - 1) / S));
  int64_t t0 = 0, total = 0;
  for (int b = 0; b < B; b++) {
    const int ql = q_lens ? q_lens[b] : Lmax;
    if (seq[b] < 0 || ql < 0 || ql > Lmax) return OKC_ERR_INVALID;
    if ((int64_t)seq[b] + ql > (int64_t)c->max_pages * c->page_size) return OKC_ERR_INVALID;
    for (int i0 = 0; i0 < ql; i0 += S) {
      const int ntok = std::min(S, ql - i0);
      const int64_t hi = (int64_t)seq[b] + i0 + ntok;
      const int64_t lo = c->window > 0 ? std::max<int64_t>(0, (int64_t)seq[b] + i0 - c->window + 1) : 0;
      units.push_back(Unit{b, i0, ntok, (int32_t)(t0 + i0), i0 + S >= ql ? 1 : 0, hi, hi - lo});
      total += hi - lo;
    }
    t0 += ql;
  }
  r->tokens = t0;
  const int U = (int)units.size();
  if ((int64_t)units.size() > ((int64_t)1 << 30)) return OKC_ERR_UNSUPPORTED;
  // Choose one key budget C for every block (a block's keys are then split
  // into ceil(n_u / C) equal chunks). For m = 1..4 waves of the `slots` resident
  // CTA slots, take the smallest C whose items fit m waves and score it as
  //   max(largest item, ceil(items / slots) * mean item),
  // each item costing kItemCost keys on top of its own (start-up, the split's
  // partial output and its merge). The lowest score wins (ties: fewer waves).
  // Skewed batches pick more waves of smaller items; uniform ones one wave.
  const int64_t min_chunk = 128, kItemCost = 128;
  int64_t nmax = 1;
  for (const Unit& u : units) nmax = std::max(nmax, u.nvis);
  // (key counts and budgets are below 2^31: 32-bit divisions)
  auto cdiv = [](int64_t a, int64_t b) { return (int64_t)(((uint32_t)a + (uint32_t)b - 1u) / (uint32_t)b); };
  // The search evaluates items(C) only at budgets C >= c_floor (the least any
  // wave count below can pick), where a block of at most c_floor keys is one
  // item: those are counted once. Blocks of the largest size (on window
  // layers every block whose context fills the window, on full layers a batch
  // of equal contexts) are counted once times their number.
  const int64_t c_floor =
      slots > 0 ? std::max<int64_t>(min_chunk, (total + 4 * (int64_t)slots - 1) / (4 * (int64_t)slots)) : min_chunk;
  int64_t n_top = 0, n_small = 0, max_small = 0;
  std::vector<int64_t> rest;
  rest.reserve(units.size());
  for (const Unit& u : units) {
    const int64_t v = u.nvis;
    if (v == nmax) {
      n_top++;
    } else if (v <= c_floor) {
      n_small++;
      max_small = std::max(max_small, v);
    } else {
      rest.push_back(v);
    }
  }
  // items(C) = sum over blocks of ceil(n_u / C) (every n_u >= 1): the
  // quotient from one reciprocal per C, corrected to the exact integer (the
  // double estimate of a quotient below 2^31 is off by at most one), instead
  // of a division per block
  auto items = [&](int64_t C) {
    const double rc = 1.0 / (double)C;
    auto nch = [&](int64_t v) {
      int64_t q = (int64_t)((double)(v - 1) * rc);  // floor((v - 1) / C), +-1
      q -= (int64_t)(q * C > v - 1);
      q += (int64_t)((q + 1) * C <= v - 1);
      return q + 1;
    };
    int64_t w = n_small + (n_top ? n_top * nch(nmax) : 0);
    for (const int64_t v : rest) w += nch(v);
    return w;
  };
  int64_t Cbud = std::max<int64_t>(min_chunk, nmax);
  if (slots > 0 && U > 0) {
    double best = -1.0, excess = 0.5 * U;
    const int64_t cmax = std::max<int64_t>(min_chunk, nmax);  // items(cmax) = U
    for (int m = 1; m <= 4; m++) {
      // smallest C in [min_chunk, cmax] with items(C) <= cap (cmax when none).
      // Since total / C <= items(C) <= total / C + U, that C is at least
      // ceil(total / cap) and at most ceil(total / (cap - U)) when cap > U.
      const int64_t cap = (int64_t)m * slots;
      int64_t lo_c = cmax, hi_c = cmax;
      if (cap > U) {
        lo_c = std::min(cmax, std::max(min_chunk, (total + cap - 1) / cap));
        hi_c = std::min(cmax, std::max(lo_c, (total + cap - U - 1) / (cap - U)));
      }
      // Safeguarded search: probe where the model items(C) = total / C + e
      // puts items at cap (e: the excess over total / C seen at the last
      // probe, between 0 and U), clamped into the bracket, and bisect after a
      // probe that did not halve it. Every probe keeps the answer inside
      // [lo_c, hi_c] with items(hi_c) <= cap, so the result is the bisection's,
      // in a few probes instead of log2 of the bracket.
      int64_t w_hi = -1;  // items(hi_c), once probed
      bool model = true;
      while (lo_c < hi_c) {
        const int64_t width = hi_c - lo_c;
        int64_t probe = (lo_c + hi_c) / 2;
        if (model && (double)cap > excess) {
          const double g = std::ceil((double)total / ((double)cap - excess));
          probe = g <= (double)lo_c ? lo_c : g >= (double)(hi_c - 1) ? hi_c - 1 : (int64_t)g;
        }
        const int64_t w = items(probe);
        excess = (double)w - (double)total / (double)probe;
        if (w <= cap) {
          hi_c = probe;
          w_hi = w;
        } else {
          lo_c = probe + 1;
        }
        model = 2 * (hi_c - lo_c) <= width;
      }
      const int64_t C = lo_c, W = w_hi >= 0 && hi_c == C ? w_hi : items(C);
      auto item_keys = [&](int64_t v) { return cdiv(v, std::max<int64_t>(1, cdiv(v, C))); };
      int64_t biggest = std::max(max_small, n_top ? item_keys(nmax) : 0);  // a block of v <= C keys: v
      for (const int64_t v : rest) biggest = std::max(biggest, item_keys(v));
      const double mean = (double)(total + W * kItemCost) / (double)W;
      const double waves = (double)((W + slots - 1) / slots);
      const double score = std::max((double)(biggest + kItemCost), waves * mean);
      if (best < 0.0 || score < best) {
        best = score;
        Cbud = C;
      }
      if (C == min_chunk) break;  // smaller items are not allowed
    }
  }
  // blocks of 2..16 tokens decode on the tcgen05 kernel, fed by TMA on pages of 8+ rows
  const bool tc_tma = okc::uses_tc(*c, o) && c->page_size >= 8;
  const int64_t tma_pad = tc_tma ? 7 : 0;
  r->blocks.assign((size_t)U, BlockInfo{0, 0, 0, 0});
  std::vector<int32_t> chunk_of((size_t)U);
  int64_t wbase = 0;
  int64_t prev_n = -1, chunk = 0, nch = 0;  // blocks of equal size share their split
  for (int u = 0; u < U; u++) {
    const int64_t nv = units[(size_t)u].nvis;
    if (nv != prev_n) {
      prev_n = nv;
      if (o && o->chunk_keys > 0) {
        chunk = o->chunk_keys;
      } else {
        const int64_t k = std::max<int64_t>(1, cdiv(nv, Cbud));
        chunk = okc::split_chunk_keys(nv, k, tma_pad);
      }
      nch = std::max<int64_t>(1, cdiv(nv, chunk));
    }
    if (nch > (1 << 20) || wbase + nch > ((int64_t)1 << 30)) return OKC_ERR_UNSUPPORTED;
    r->blocks[(size_t)u] = BlockInfo{(int32_t)wbase, (int32_t)nch, units[(size_t)u].t0, units[(size_t)u].ntok};
    chunk_of[(size_t)u] = (int32_t)chunk;
    r->max_chunks = std::max<int>(r->max_chunks, (int)nch);
    r->max_chunk_keys = std::max<int64_t>(r->max_chunk_keys, chunk);
    wbase += nch;
  }
  // Launch order: the largest items first (the last chunk of a block may be
  // short), ties in slot order. A block's items before its last all hold
  // chunk_keys keys, so the order is a merge of two sorted runs: those items,
  // block by block in (chunk_keys desc, block) order, and the last items in
  // (keys desc, block) order. Sort words pack (2^31-1 - keys, u).
  auto last_keys = [&](int u) {
    const BlockInfo& q = r->blocks[(size_t)u];
    return units[(size_t)u].nvis - (int64_t)(q.nchunks - 1) * chunk_of[(size_t)u];
  };
  auto pack = [](int64_t keys, int u) { return ((uint64_t)(0x7FFFFFFF - keys) << 32) | (uint32_t)u; };
  std::vector<uint64_t> run_full, run_last((size_t)U);
  run_full.reserve((size_t)U);
  for (int u = 0; u < U; u++) {
    if (r->blocks[(size_t)u].nchunks > 1) run_full.push_back(pack(chunk_of[(size_t)u], u));
    run_last[(size_t)u] = pack(last_keys(u), u);
  }
  std::sort(run_full.begin(), run_full.end());
  std::sort(run_last.begin(), run_last.end());
  r->work.resize((size_t)wbase);
  WorkItem* out = r->work.data();
  auto item = [&](int u, int k, int64_t j0, int64_t j1) {
    const Unit& x = units[(size_t)u];
    const BlockInfo& q = r->blocks[(size_t)u];
    return WorkItem{x.b, (int32_t)(j0 - (x.hi - x.nvis)), x.i0, x.ntok, k, (int32_t)j0, (int32_t)j1,
                    chunk_of[(size_t)u], q.nchunks, q.wbase, x.t0, x.last};
  };
  size_t il = 0;
  auto emit_last_before = [&](uint64_t key_word, int32_t slot) {  // last items ahead of (key, slot)
    while (il < run_last.size()) {
      const uint64_t w = run_last[il];
      const int u = (int)(w & 0xFFFFFFFFu);
      const BlockInfo& q = r->blocks[(size_t)u];
      const int32_t ls = q.wbase + q.nchunks - 1;
      if ((w >> 32) > (key_word >> 32) || ((w >> 32) == (key_word >> 32) && ls > slot)) break;
      const Unit& x = units[(size_t)u];
      *out++ = item(u, q.nchunks - 1, x.hi - x.nvis + (int64_t)(q.nchunks - 1) * chunk_of[(size_t)u], x.hi);
      il++;
    }
  };
  // A block's items before its last take slots wbase .. wbase + nchunks - 2,
  // a range no other block's slot falls into, so the last items that go
  // before any of them go before the first: one merge step per block.
  for (const uint64_t w : run_full) {
    const int u = (int)(w & 0xFFFFFFFFu);
    const BlockInfo& q = r->blocks[(size_t)u];
    emit_last_before(w, q.wbase);
    const int64_t ck = chunk_of[(size_t)u];
    int64_t j0 = units[(size_t)u].hi - units[(size_t)u].nvis;  // these items hold chunk_keys keys each
    for (int k = 0; k + 1 < q.nchunks; k++, j0 += ck) *out++ = item(u, k, j0, j0 + ck);
  }
  emit_last_before(~0ull, 0);
  if (!(o && o->chunk_keys > 0) && S == 1 && slots > 0)
    split_tail(r, (int64_t)std::max<int64_t>(U, 4 * (int64_t)slots), slots, kItemCost);
  return OKC_OK;
}

namespace {

// Kernels okc_attn_step launches: 1 (the fused step kernel, q_len 1) when the
// work list fills at least half of the resident CTA slots with chunks of at
// most 2048 keys, or takes more than one wave (measured faster there: the
// merge tail is short against the step, or the first wave's merges overlap
// the second wave), else 3 (prepare, decode, combine: faster for very small
// batches, where the kernels' latencies overlap under programmatic launch, and
// for one wave of long chunks, where the separate merge overlaps the decode's
// tail).
int step_kernels(const okc_attn_config* c, const SplitResult& s, const okc_plan_options* o, int slots) {
  const int flags = o ? o->flags : 0;
  if (c->q_len != 1) {
    // blocks of 2..8 tokens on the tcgen05 kernel (one block per request): the
    // one-kernel form when the options ask for it
    const bool one = c->q_len <= 8 && okc::uses_tc(*c, o) && okc::tc_groups(*c) == 2 && s.S == c->q_len;
    return one && (flags & OKC_PLAN_STEP_ONE_LAUNCH) && !(flags & OKC_PLAN_STEP_THREE_LAUNCHES) ? 1 : 3;
  }
  if (flags & OKC_PLAN_STEP_THREE_LAUNCHES) return 3;
  if (flags & OKC_PLAN_STEP_ONE_LAUNCH) return 1;
  const int64_t W = (int64_t)s.work.size();
  return (2 * W >= slots && (s.max_chunk_keys <= 2048 || W > slots)) ? 1 : 3;
}

// Buffer sizes of a step of W work items laid out in a work list of cap >= W
// entries, NB query blocks of S tokens and T tokens (the workspace, q and the
// split partials).
void sizes_for(const okc_attn_config* c, int64_t W, int64_t cap, int64_t NB, int64_t T, int S, int max_chunks,
               okc_attn_sizes* z) {
  const int64_t rows = (int64_t)S * c->num_q_heads;
  std::memset(z, 0, sizeof *z);
  z->workspace_bytes = okc::kWsHeader + round_up(cap * sizeof(WorkItem)) + round_up(NB * sizeof(BlockInfo)) +
                       round_up(c->batch * sizeof(int32_t)) +         // + the one-launch step's arrival counters
                       round_up(T * c->num_q_heads * c->head_dim);  // + q for the three-launch step
  z->q_fp8_bytes = round_up(T * c->num_q_heads * c->head_dim);
  z->o_partial_bytes = round_up(W * rows * c->head_dim * sizeof(float));
  z->lse_partial_bytes = round_up(W * rows * sizeof(float));
  z->num_work = (int32_t)W;
  z->num_tokens = (int32_t)T;
  z->max_chunks = max_chunks;
  z->step_kernels = 3;
}

// Upper bounds of the split counts over every step whose requests each hold at
// most max_context keys after the step. A request has at most ceil(q_len / S)
// query blocks, and a block sees at most min(max_context, window + S - 1)
// keys (window layers) or max_context. A block of n visible keys gets
// ceil(n / chunk_keys) items under a forced chunk size; under the heuristic
// k = ceil(n / C) items for the budget C >= 128 (its chunk holds at least
// ceil(n / k) keys), and the budget's work list either fits the m waves it was
// chosen for (m <= 4: at most 4 x slots items) or is one item per block.
void split_bounds(const okc_attn_config* c, int64_t max_context, const okc_plan_options* o, int slots,
                  int64_t* max_work, int64_t* max_chunks, int64_t* max_blocks) {
  const int S = okc::block_tokens(*c, o);
  const int64_t NB = (int64_t)c->batch * ((c->q_len + S - 1) / S);
  const int64_t nvis = c->window > 0 ? std::min<int64_t>(max_context, (int64_t)c->window + S - 1) : max_context;
  const int64_t per = (o && o->chunk_keys > 0) ? o->chunk_keys : 128;
  const int64_t k = std::max<int64_t>(1, (nvis + per - 1) / per);
  *max_chunks = k;
  *max_blocks = NB;
  *max_work = NB * k;
  if (!(o && o->chunk_keys > 0)) *max_work = std::min(*max_work, std::max<int64_t>(NB, 4 * (int64_t)slots));
}

// A plan with a fixed-capacity work list: okc_plan_options.max_context > 0.
bool fixed_capacity(const okc_plan_options* o) { return o && o->max_context > 0; }

// The sizes of a step under the options (the live split `s`; on a
// fixed-capacity plan the work list laid out at the capacity for max_context,
// returned in *cap_out), and its okc_attn_step form.
okc_status plan_sizes_of(const okc_attn_config* c, const SplitResult& s, const okc_plan_options* o, int slots,
                         okc_attn_sizes* z, int64_t* cap_out) {
  const int64_t W = (int64_t)s.work.size();
  int64_t cap = W;
  if (fixed_capacity(o)) {
    int64_t wb = 0, kb = 0, nb = 0;
    split_bounds(c, o->max_context, o, slots, &wb, &kb, &nb);
    if (W > wb) return OKC_ERR_WORKSPACE;  // (the bound holds for every step within max_context)
    cap = wb;
  }
  sizes_for(c, W, cap, (int64_t)s.blocks.size(), s.tokens, s.S, s.max_chunks, z);
  z->step_kernels = step_kernels(c, s, o, slots);
  if (cap_out) *cap_out = fixed_capacity(o) ? cap : 0;
  return OKC_OK;
}

// Steps a fixed-capacity plan serves: uniform q lengths, every request within max_context.
okc_status check_fixed(const okc_attn_config* c, const int32_t* seq, const int32_t* q_lens,
                       const okc_plan_options* o) {
  if (!fixed_capacity(o)) return OKC_OK;
  if (o->max_context < c->q_len || (int64_t)o->max_context > (int64_t)c->max_pages * c->page_size)
    return OKC_ERR_INVALID;
  if (q_lens) return OKC_ERR_UNSUPPORTED;
  for (int b = 0; b < c->batch; b++)
    if (seq[b] < 0 || (int64_t)seq[b] + c->q_len > o->max_context) return OKC_ERR_INVALID;
  return OKC_OK;
}

}  // namespace

// Resident decode CTAs per SM for (device, block tokens, kernel family), queried
// once per key: the query also raises the kernels' shared-memory limit on the device.
int okc::cached_ctas_per_sm(int dev, int S, bool tc, int tc_groups) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, bool, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, S, tc, tc ? tc_groups : 0);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const int occ = okc::decode_ctas_per_sm(S, tc, tc_groups);
  if (occ > 0) cache[key] = occ;
  return occ;
}

namespace {

int slots_for(const okc_attn_config* c, const okc_plan_options* o, int* sm_count_out) {
  int sms = (o && o->sm_count > 0) ? o->sm_count : 0;
  int per_sm = (o && o->ctas_per_sm > 0) ? o->ctas_per_sm : 0;
  if (sms == 0 || per_sm == 0) {  // read from the current device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (sms == 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (per_sm == 0)
      per_sm = okc::cached_ctas_per_sm(dev, okc::block_tokens(*c, o), okc::uses_tc(*c, o), okc::tc_groups(*c));
    if (per_sm <= 0) return -1;
  }
  if (sm_count_out) *sm_count_out = sms;
  return sms * per_sm;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// Natural alignment of the element type the kernels load through p (null passes:
// the null checks are separate).
bool aligned(const void* p, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0; }

// The plan takes a split result: sizes, work list, block table, and the
// workspace layout (header | work list | block table | arrival counters | q).
// A fixed-capacity plan lays the work list out at its capacity, so the offsets
// after it never move.
void set_splits(okc_attn_plan_s* p, SplitResult& s, const okc_attn_sizes& z) {
  p->sizes = z;
  p->work.swap(s.work);
  p->blocks.swap(s.blocks);
  p->S = s.S;
  const size_t cap = p->work_cap > 0 ? (size_t)p->work_cap : p->work.size();
  uint8_t* ws = static_cast<uint8_t*>(p->workspace);
  p->d_err = reinterpret_cast<unsigned*>(ws);
  p->d_live = reinterpret_cast<int32_t*>(ws + okc::kWsCount);
  p->d_work = reinterpret_cast<WorkItem*>(ws + okc::kWsHeader);
  p->d_blk = reinterpret_cast<BlockInfo*>(ws + okc::kWsHeader + round_up(cap * sizeof(WorkItem)));
  p->d_tickets = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(p->d_blk) +
                                            round_up(p->blocks.size() * sizeof(BlockInfo)));
  // (one arrival counter per request: the one-kernel step runs at most one
  // block per request)
  p->d_q8 = reinterpret_cast<uint8_t*>(p->d_tickets) + round_up((size_t)p->cfg.batch * sizeof(int32_t));
}

// Bytes of the workspace head the plan uploads (everything before q).
size_t upload_bytes(const okc_attn_plan_s* p) {
  return static_cast<size_t>(p->d_q8 - static_cast<uint8_t*>(p->workspace));
}

// The live item count, the work list and the block table at their workspace
// offsets in a zeroed host image of the head (the error word and the arrival
// counters stay zero).
void write_head(const okc_attn_plan_s* p, uint8_t* head) {
  const uint8_t* ws = static_cast<const uint8_t*>(p->workspace);
  const int32_t live = (int32_t)p->work.size();
  std::memcpy(head + okc::kWsCount, &live, sizeof live);
  if (!p->work.empty())
    std::memcpy(head + (reinterpret_cast<const uint8_t*>(p->d_work) - ws), p->work.data(),
                p->work.size() * sizeof(WorkItem));
  if (!p->blocks.empty())
    std::memcpy(head + (reinterpret_cast<const uint8_t*>(p->d_blk) - ws), p->blocks.data(),
                p->blocks.size() * sizeof(BlockInfo));
}

// Work items the decode launches cover: the capacity on a fixed-capacity plan
// (CTAs past the live count return at once), else the step's own count.
int launch_items(const okc_attn_plan_s* p) {
  return p->work_cap > 0 ? (int)p->work_cap : p->sizes.num_work;
}

// The device address of a page-locked, device-mapped host buffer, else NULL
// (pageable or unknown memory).
const void* mapped_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

// One warp waits on a shared-memory mbarrier that nothing arrives on, with the
// bounded wait every kernel uses (here limited to limit_ns), and flags the
// timeout the way the kernels do; the kernel then returns.
__global__ void bounded_wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = okc::smem_u32(&bar);
  if (threadIdx.x == 0) {
    okc::mbar_init(b, 1);
    okc::fence_mbar_init();
  }
  __syncthreads();
  const bool ok = okc::mbar_wait(b, 0, limit_ns);
  if (!__any_sync(0xffffffffu, ok) && threadIdx.x == 0) okc::set_error(err, OKC_DEVERR_TIMEOUT);
}

}  // namespace

extern "C" {

const char* okc_status_string(okc_status s) {
  switch (s) {
    case OKC_OK: return "ok";
    case OKC_ERR_INVALID: return "invalid argument";
    case OKC_ERR_UNSUPPORTED: return "unsupported shape";
    case OKC_ERR_CUDA: return "CUDA error";
    case OKC_ERR_WORKSPACE: return "workspace or scratch too small or misaligned";
  }
  return "unknown status";
}

okc_status okc_attn_plan_sizes_varlen(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                                      const int32_t* q_lens_host, const okc_plan_options* opts,
                                      okc_attn_sizes* sizes) {
  okc_status st = check_config(cfg);
  if (st != OKC_OK) return st;
  if (!sizes || (cfg->batch > 0 && !seq_lens_host)) return OKC_ERR_INVALID;
  st = check_fixed(cfg, seq_lens_host, q_lens_host, opts);
  if (st != OKC_OK) return st;
  const int slots = cfg->batch > 0 ? slots_for(cfg, opts, nullptr) : 1;
  if (slots < 0) return OKC_ERR_CUDA;
  SplitResult s;
  st = make_splits(cfg, seq_lens_host, q_lens_host, opts, slots, &s);
  if (st != OKC_OK) return st;
  return plan_sizes_of(cfg, s, opts, slots, sizes, nullptr);
}

okc_status okc_attn_plan_sizes(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                               const okc_plan_options* opts, okc_attn_sizes* sizes) {
  return okc_attn_plan_sizes_varlen(cfg, seq_lens_host, nullptr, opts, sizes);
}

okc_status okc_attn_plan_max_sizes(const okc_attn_config* cfg, int32_t max_context, const okc_plan_options* opts,
                                   okc_attn_sizes* sizes) {
  okc_status st = check_config(cfg);
  if (st != OKC_OK) return st;
  if (!sizes || max_context < cfg->q_len || (int64_t)max_context > (int64_t)cfg->max_pages * cfg->page_size)
    return OKC_ERR_INVALID;
  if (opts && opts->chunk_keys != 0 && opts->chunk_keys < 16) return OKC_ERR_INVALID;
  const int slots = cfg->batch > 0 ? slots_for(cfg, opts, nullptr) : 1;
  if (slots < 0) return OKC_ERR_CUDA;
  int64_t W = 0, kmax = 0, NB = 0;
  split_bounds(cfg, max_context, opts, slots, &W, &kmax, &NB);
  if (cfg->batch == 0) W = kmax = NB = 0;
  if (kmax > (1 << 20) || W > ((int64_t)1 << 30)) return OKC_ERR_UNSUPPORTED;
  int64_t cap = W;
  if (fixed_capacity(opts)) {  // the work list of a fixed-capacity plan is laid out for its own max_context
    int64_t wc = 0, kc = 0, nc = 0;
    split_bounds(cfg, std::max<int64_t>(opts->max_context, cfg->q_len), opts, slots, &wc, &kc, &nc);
    cap = cfg->batch > 0 ? std::max(W, wc) : 0;
  }
  sizes_for(cfg, W, cap, NB, (int64_t)cfg->batch * cfg->q_len, okc::block_tokens(*cfg, opts), (int)kmax, sizes);
  sizes->step_kernels = 0;  // depends on the lengths
  return OKC_OK;
}

okc_status okc_attn_plan_workspace_size(const okc_attn_config* cfg, int32_t max_total_ctx, size_t* bytes) {
  if (!bytes) return OKC_ERR_INVALID;
  okc_attn_sizes z;
  const okc_status st = okc_attn_plan_max_sizes(cfg, max_total_ctx, nullptr, &z);
  if (st == OKC_OK) *bytes = z.workspace_bytes;
  return st;
}

okc_status okc_attn_plan_items_varlen(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                                      const int32_t* q_lens_host, const okc_plan_options* opts, int32_t* items,
                                      int32_t capacity, int32_t* count) {
  okc_status st = check_config(cfg);
  if (st != OKC_OK) return st;
  if (!count || capacity < 0 || (capacity > 0 && !items) || (cfg->batch > 0 && !seq_lens_host))
    return OKC_ERR_INVALID;
  const int slots = cfg->batch > 0 ? slots_for(cfg, opts, nullptr) : 1;
  if (slots < 0) return OKC_ERR_CUDA;
  SplitResult s;
  st = make_splits(cfg, seq_lens_host, q_lens_host, opts, slots, &s);
  if (st != OKC_OK) return st;
  *count = (int32_t)s.work.size();
  if ((int64_t)s.work.size() > capacity) return capacity == 0 && !items ? OKC_OK : OKC_ERR_WORKSPACE;
  for (size_t i = 0; i < s.work.size(); i++) {
    items[4 * i] = s.work[i].b;
    items[4 * i + 1] = s.work[i].i0;
    items[4 * i + 2] = s.work[i].j0;
    items[4 * i + 3] = s.work[i].j1;
  }
  return OKC_OK;
}

okc_status okc_attn_plan_items(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                               const okc_plan_options* opts, int32_t* items, int32_t capacity,
                               int32_t* count) {
  okc_status st = check_config(cfg);
  if (st != OKC_OK) return st;
  if (!count || capacity < 0 || (capacity > 0 && !items) || (cfg->batch > 0 && !seq_lens_host))
    return OKC_ERR_INVALID;
  const int slots = cfg->batch > 0 ? slots_for(cfg, opts, nullptr) : 1;
  if (slots < 0) return OKC_ERR_CUDA;
  SplitResult s;
  st = make_splits(cfg, seq_lens_host, nullptr, opts, slots, &s);
  if (st != OKC_OK) return st;
  *count = (int32_t)s.work.size();
  if ((int64_t)s.work.size() > capacity) return capacity == 0 && !items ? OKC_OK : OKC_ERR_WORKSPACE;
  for (size_t i = 0; i < s.work.size(); i++) {
    items[3 * i] = s.work[i].b;
    items[3 * i + 1] = s.work[i].j0;
    items[3 * i + 2] = s.work[i].j1;
  }
  return OKC_OK;
}

okc_status okc_attn_plan_varlen(const okc_attn_config* cfg, const int32_t* seq_lens_host, const int32_t* q_lens_host,
                                const okc_plan_options* opts, void* workspace, size_t workspace_bytes,
                                okc_stream stream, okc_attn_plan_t* plan_out) {
  okc_status st = check_config(cfg);
  if (st != OKC_OK) return st;
  if (!plan_out || (cfg->batch > 0 && !seq_lens_host) || !workspace) return OKC_ERR_INVALID;
  *plan_out = nullptr;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return OKC_ERR_WORKSPACE;
  st = check_fixed(cfg, seq_lens_host, q_lens_host, opts);
  if (st != OKC_OK) return st;
  int sms = 0;
  const int slots = slots_for(cfg, opts, &sms);
  if (slots < 0) return OKC_ERR_CUDA;
  // the decode kernels' shared-memory limits are raised on the device by the
  // (cached) occupancy query, which forced options skip: run it here for every plan
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      okc::cached_ctas_per_sm(dev, okc::block_tokens(*cfg, opts), okc::uses_tc(*cfg, opts), okc::tc_groups(*cfg)) <= 0)
    return OKC_ERR_CUDA;
  SplitResult s;
  st = make_splits(cfg, seq_lens_host, q_lens_host, opts, slots, &s);
  if (st != OKC_OK) return st;
  okc_attn_sizes z;
  int64_t cap = 0;
  st = plan_sizes_of(cfg, s, opts, slots, &z, &cap);
  if (st != OKC_OK) return st;
  if (workspace_bytes < z.workspace_bytes) return OKC_ERR_WORKSPACE;

  okc_attn_plan_s* p = new (std::nothrow) okc_attn_plan_s();
  if (!p) return OKC_ERR_INVALID;
  p->cfg = *cfg;
  if (opts) p->opts = *opts; else std::memset(&p->opts, 0, sizeof p->opts);
  if (q_lens_host) p->q_lens.assign(q_lens_host, q_lens_host + cfg->batch);
  p->workspace = workspace;
  p->workspace_bytes = workspace_bytes;
  p->slots = slots;
  p->work_cap = cap;
  cudaGetDevice(&p->device);
  p->sm_count = sms;
  p->pdl = !(p->opts.flags & OKC_PLAN_NO_PDL);
  p->tc = okc::uses_tc(*cfg, opts);
  p->scale_log2 = okc::softmax_scale_log2(*cfg);
  set_splits(p, s, z);
  // One upload of the workspace's head: the zeroed error word, the live item
  // count, the work list, the block table and the zeroed arrival counters, as
  // laid out on the device.
  const size_t up_bytes = upload_bytes(p);
  p->upload.assign(up_bytes, 0);
  write_head(p, p->upload.data());
  cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(workspace, p->upload.data(), up_bytes, cudaMemcpyHostToDevice, str);
  if (e != cudaSuccess) {
    delete p;
    return OKC_ERR_CUDA;
  }
  *plan_out = p;
  return OKC_OK;
}

okc_status okc_attn_plan(const okc_attn_config* cfg, const int32_t* seq_lens_host,
                         const okc_plan_options* opts, void* workspace, size_t workspace_bytes,
                         okc_stream stream, okc_attn_plan_t* plan_out) {
  return okc_attn_plan_varlen(cfg, seq_lens_host, nullptr, opts, workspace, workspace_bytes, stream, plan_out);
}

okc_status okc_attn_plan_create(const okc_attn_config* cfg, const int32_t* seq_lens_host, void* workspace,
                                size_t workspace_bytes, okc_stream stream, okc_attn_plan_t* plan_out) {
  return okc_attn_plan(cfg, seq_lens_host, nullptr, workspace, workspace_bytes, stream, plan_out);
}

okc_status okc_attn_plan_update_varlen(okc_attn_plan_t plan, const int32_t* seq_lens_host,
                                       const int32_t* q_lens_host, okc_stream stream) {
  if (!plan || (plan->cfg.batch > 0 && !seq_lens_host)) return OKC_ERR_INVALID;
  okc_status st = check_fixed(&plan->cfg, seq_lens_host, q_lens_host, &plan->opts);
  if (st != OKC_OK) return st;
  // The new split is built in the spare lists (the ones the previous update
  // replaced: their capacity is reused); the plan's current lists, sizes and
  // workspace stay as they are until every step that can fail has passed.
  SplitResult s;
  s.work.swap(plan->spare_work);
  s.blocks.swap(plan->spare_blocks);
  auto restore = [&](okc_status e) {
    s.work.swap(plan->spare_work);
    s.blocks.swap(plan->spare_blocks);
    return e;
  };
  st = make_splits(&plan->cfg, seq_lens_host, q_lens_host, &plan->opts, plan->slots, &s);
  if (st != OKC_OK) return restore(st);
  okc_attn_sizes z;
  st = plan_sizes_of(&plan->cfg, s, &plan->opts, plan->slots, &z, nullptr);
  if (st != OKC_OK) return restore(st);
  // a fixed-capacity plan keeps the okc_attn_step form it was made with (a
  // graph captured from it keeps its launches)
  if (plan->work_cap > 0) z.step_kernels = plan->sizes.step_kernels;
  // the staging buffer for the head (up to q: header, work list, block table,
  // arrival counters) is made ready before the plan changes
  if (plan->workspace_bytes < z.workspace_bytes) return restore(OKC_ERR_WORKSPACE);
  const size_t cap = plan->work_cap > 0 ? (size_t)plan->work_cap : s.work.size();
  const size_t up_bytes = okc::kWsHeader + round_up(cap * sizeof(WorkItem)) + round_up(s.blocks.size() * sizeof(BlockInfo)) +
                          round_up((size_t)plan->cfg.batch * sizeof(int32_t));
  // the staging buffer may still feed the previous update's copy
  if (plan->pinned_done && cudaEventSynchronize(plan->pinned_done) != cudaSuccess) return restore(OKC_ERR_CUDA);
  if (plan->pinned_bytes < up_bytes) {
    if (plan->pinned) cudaFreeHost(plan->pinned);
    plan->pinned = nullptr;
    plan->pinned_bytes = 0;
    const size_t want = std::max<size_t>(up_bytes, 64 * 1024);
    if (cudaMallocHost(&plan->pinned, want) != cudaSuccess) {
      plan->pinned = nullptr;
      return restore(OKC_ERR_CUDA);
    }
    plan->pinned_bytes = want;
  }
  if (!plan->pinned_done && cudaEventCreateWithFlags(&plan->pinned_done, cudaEventDisableTiming) != cudaSuccess) {
    plan->pinned_done = nullptr;
    return restore(OKC_ERR_CUDA);
  }
  set_splits(plan, s, z);  // s now holds the replaced lists: they become the spares
  s.work.swap(plan->spare_work);
  s.blocks.swap(plan->spare_blocks);
  if (!q_lens_host)
    plan->q_lens.clear();
  else if (q_lens_host != plan->q_lens.data())
    plan->q_lens.assign(q_lens_host, q_lens_host + plan->cfg.batch);
  uint8_t* head = static_cast<uint8_t*>(plan->pinned);
  std::memset(head, 0, up_bytes);
  write_head(plan, head);
  // The upload starts past the error word: the device error word keeps the
  // bits earlier steps set until the caller reads or clears them.
  cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(static_cast<uint8_t*>(plan->workspace) + okc::kWsCount, head + okc::kWsCount,
                      up_bytes - okc::kWsCount, cudaMemcpyHostToDevice, str) != cudaSuccess ||
      cudaEventRecord(plan->pinned_done, str) != cudaSuccess)
    return OKC_ERR_CUDA;
  return OKC_OK;
}

okc_status okc_attn_plan_update(okc_attn_plan_t plan, const int32_t* seq_lens_host, okc_stream stream) {
  if (!plan) return OKC_ERR_INVALID;
  return okc_attn_plan_update_varlen(plan, seq_lens_host, plan->q_lens.empty() ? nullptr : plan->q_lens.data(),
                                     stream);
}

okc_status okc_attn_plan_destroy(okc_attn_plan_t plan) {
  if (!plan) return OKC_OK;
  if (plan->pinned_done) {
    cudaEventSynchronize(plan->pinned_done);  // the staging buffer's last copy
    cudaEventDestroy(plan->pinned_done);
  }
  if (plan->pinned) cudaFreeHost(plan->pinned);
  delete plan;
  return OKC_OK;
}

okc_status okc_attn_plan_get_sizes(okc_attn_plan_t plan, okc_attn_sizes* sizes) {
  if (!plan || !sizes) return OKC_ERR_INVALID;
  *sizes = plan->sizes;
  return OKC_OK;
}

okc_status okc_attn_plan_scratch_sizes(okc_attn_plan_t plan, okc_attn_sizes* sizes) {
  return okc_attn_plan_get_sizes(plan, sizes);
}

okc_status okc_attn_plan_read_errors(okc_attn_plan_t plan, okc_stream stream, uint32_t* flags_host) {
  if (!plan || !flags_host) return OKC_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, plan->d_err, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return OKC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return OKC_ERR_CUDA;
  *flags_host = v;
  return OKC_OK;
}

okc_status okc_attn_plan_clear_errors(okc_attn_plan_t plan, okc_stream stream) {
  if (!plan) return OKC_ERR_INVALID;
  return cudaMemsetAsync(plan->d_err, 0, sizeof(unsigned), reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? OKC_OK
             : OKC_ERR_CUDA;
}

okc_status okc_selftest_bounded_wait(uint32_t* err, int32_t limit_us, okc_stream stream) {
  if (!err || limit_us < 1 || limit_us > 1000000) return OKC_ERR_INVALID;
  bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<unsigned*>(err), (uint64_t)limit_us * 1000u);
  return cudaGetLastError() == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
}

okc_status okc_rope_table_init(float rope_theta, int32_t num_positions, float* table, okc_stream stream) {
  if (!(rope_theta > 0.f) || !std::isfinite(rope_theta) || !table) return OKC_ERR_INVALID;
  if (num_positions < 1 || num_positions > okc::kRopePositionsMax) return OKC_ERR_INVALID;
  if (!aligned16(table)) return OKC_ERR_INVALID;
  // inv_freq = 1 / theta^(arange(0, 64, 2)/64): the power rounded once to float32
  // (computed in double), then a float32 division.
  float inv[okc::kHeadDim / 2];
  for (int i = 0; i < okc::kHeadDim / 2; i++) {
    const float e = (float)(2 * i) / (float)okc::kHeadDim;
    const float pw = (float)std::pow((double)rope_theta, (double)e);
    volatile float one = 1.0f;  // keep the division in float32
    inv[i] = one / pw;
  }
  cudaError_t err = okc::launch_rope_table(rope_theta, inv, num_positions, table,
                                           reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
}

okc_status okc_prepare_qkv(okc_attn_plan_t plan, const void* qkv, const int64_t* positions,
                           const int64_t* cache_loc, uint8_t* k_cache, uint8_t* v_cache,
                           const float* k_scale, const float* v_scale, const float* rope_table,
                           int32_t rope_positions, uint8_t* q_fp8, okc_stream stream) {
  if (!plan) return OKC_ERR_INVALID;
  const okc_attn_config& c = plan->cfg;
  const int T = plan->sizes.num_tokens;
  if (T == 0) return OKC_OK;
  if (!qkv || !cache_loc || !k_cache || !v_cache || !q_fp8) return OKC_ERR_INVALID;
  if (!aligned16(qkv) || !aligned16(q_fp8) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned(positions, 8) || !aligned(cache_loc, 8) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return OKC_ERR_INVALID;
  const bool rope = c.rope_theta != 0.f;
  const bool scaled = c.kv_scale != 1.f;
  if (rope && (!positions || !rope_table || !aligned16(rope_table) || rope_positions < 1 ||
               rope_positions > okc::kRopePositionsMax))
    return OKC_ERR_INVALID;
  if (scaled && (!k_scale || !v_scale)) return OKC_ERR_INVALID;
  okc::PrepareArgs a;
  a.qkv = static_cast<const uint16_t*>(qkv);
  a.positions = positions;
  a.cache_loc = cache_loc;
  a.kc = k_cache;
  a.vc = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.rope_table = rope ? rope_table : nullptr;
  a.q8 = q_fp8;
  a.err = plan->d_err;
  a.num_rows = (int64_t)c.num_pages * c.page_size;
  a.T = T;
  a.rope_positions = rope ? rope_positions : 0;
  a.rope = rope;
  a.scaled = scaled;
  a.q_fold = c.q_norm == OKC_QNORM_FOLDED_SCALE;
  a.q_scale = c.qk_scale_factor;
  cudaError_t e = okc::launch_prepare(a, plan->pdl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
}

okc_status okc_attn_decode(okc_attn_plan_t plan, const uint8_t* q_fp8, const uint8_t* k_cache,
                           const uint8_t* v_cache, const float* k_scale, const float* v_scale,
                           const int32_t* page_table, const int32_t* cache_seqlens,
                           const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                           float* o_partial, float* lse_partial, okc_stream stream) {
  if (!plan) return OKC_ERR_INVALID;
  const okc_attn_config& c = plan->cfg;
  if (launch_items(plan) == 0) return OKC_OK;
  if (!q_fp8 || !k_cache || !v_cache || !page_table || !cache_seqlens || !cu_seqlens_q ||
      !o_partial || !lse_partial)
    return OKC_ERR_INVALID;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_partial) || !aligned16(q_fp8) ||
      !aligned(lse_partial, 4) || !aligned(page_table, 4) || !aligned(cache_seqlens, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(seq_lens, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return OKC_ERR_INVALID;
  const bool scaled = c.kv_scale != 1.f;
  if (scaled && (!k_scale || !v_scale)) return OKC_ERR_INVALID;
  okc::DecodeArgs a = {};
  a.tc = plan->tc ? 1 : 0;
  a.tc_groups = okc::tc_groups(c);
  a.q8 = q_fp8;
  a.kc = k_cache;
  a.vc = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.page_table = page_table;
  a.cache_seqlens = cache_seqlens;
  a.cu_seqlens_q = cu_seqlens_q;
  a.seq_lens = seq_lens;
  a.work = plan->d_work;
  a.live_work = plan->work_cap > 0 ? plan->d_live : nullptr;
  a.o_part = o_partial;
  a.lse_part = lse_partial;
  a.err = plan->d_err;
  a.batch = c.batch;
  a.L = c.q_len;
  a.S = plan->S;
  a.window = c.window;
  a.max_pages = c.max_pages;
  a.num_pages = c.num_pages;
  a.page_shift = page_shift(c.page_size);
  a.scaled = scaled;
  a.T = plan->sizes.num_tokens;
  a.scale_log2 = plan->scale_log2;  // the kernel multiplies in *k_scale when scaled
  cudaError_t e = okc::launch_decode(a, launch_items(plan), plan->pdl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
}

okc_status okc_attn_combine_normgate(okc_attn_plan_t plan, const float* o_partial,
                                     const float* lse_partial, const void* qkv,
                                     const void* norm_weight, float eps, void* out,
                                     okc_stream stream) {
  if (!plan) return OKC_ERR_INVALID;
  const int T = plan->sizes.num_tokens;
  if (T == 0) return OKC_OK;
  if (!o_partial || !lse_partial || !qkv || !out) return OKC_ERR_INVALID;
  if (!aligned16(qkv) || !aligned16(out) || !aligned16(o_partial) || !aligned(lse_partial, 4) ||
      (norm_weight && !aligned16(norm_weight)))
    return OKC_ERR_INVALID;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return OKC_ERR_INVALID;
  okc::CombineArgs a;
  a.o_part = o_partial;
  a.lse_part = lse_partial;
  a.qkv = static_cast<const uint16_t*>(qkv);
  a.weight = static_cast<const uint16_t*>(norm_weight);
  a.out = static_cast<uint16_t*>(out);
  a.blk = plan->d_blk;
  a.err = plan->d_err;
  a.nblocks = (int32_t)plan->blocks.size();
  a.S = plan->S;
  a.T = T;
  a.eps = eps;
  cudaError_t e = okc::launch_combine(a, plan->pdl, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
}

okc_status okc_attn_step(okc_attn_plan_t plan, const void* qkv, const int64_t* positions,
                         const int64_t* cache_loc, uint8_t* k_cache, uint8_t* v_cache, const float* k_scale,
                         const float* v_scale, const float* rope_table, int32_t rope_positions,
                         const int32_t* page_table, const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
                         const int32_t* seq_lens, const void* norm_weight, float eps, float* o_partial,
                         float* lse_partial, void* out, okc_stream stream) {
  if (!plan) return OKC_ERR_INVALID;
  const okc_attn_config& c = plan->cfg;
  if (launch_items(plan) == 0) return OKC_OK;
  if (!qkv || !cache_loc || !k_cache || !v_cache || !page_table || !cache_seqlens || !cu_seqlens_q ||
      !o_partial || !lse_partial || !out)
    return OKC_ERR_INVALID;
  if (!aligned16(qkv) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o_partial) ||
      !aligned16(out) || (norm_weight && !aligned16(norm_weight)) || !aligned(lse_partial, 4) ||
      !aligned(positions, 8) || !aligned(cache_loc, 8) || !aligned(page_table, 4) ||
      !aligned(cache_seqlens, 4) || !aligned(cu_seqlens_q, 4) || !aligned(seq_lens, 4) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4))
    return OKC_ERR_INVALID;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return OKC_ERR_INVALID;
  const bool rope = c.rope_theta != 0.f;
  const bool scaled = c.kv_scale != 1.f;
  if (rope && (!positions || !rope_table || !aligned16(rope_table) || rope_positions < 1 ||
               rope_positions > okc::kRopePositionsMax))
    return OKC_ERR_INVALID;
  if (scaled && (!k_scale || !v_scale)) return OKC_ERR_INVALID;
  okc::DecodeArgs a = {};
  std::memset(&a, 0, sizeof a);
  a.kc = k_cache;
  a.vc = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.page_table = page_table;
  a.cache_seqlens = cache_seqlens;
  a.cu_seqlens_q = cu_seqlens_q;
  a.seq_lens = seq_lens;
  a.work = plan->d_work;
  a.live_work = plan->work_cap > 0 ? plan->d_live : nullptr;
  a.o_part = o_partial;
  a.lse_part = lse_partial;
  a.err = plan->d_err;
  a.batch = c.batch;
  a.L = c.q_len;
  a.S = plan->S;
  a.window = c.window;
  a.max_pages = c.max_pages;
  a.num_pages = c.num_pages;
  a.page_shift = page_shift(c.page_size);
  a.scaled = scaled;
  a.T = plan->sizes.num_tokens;
  a.scale_log2 = plan->scale_log2;
  a.qkv = static_cast<const uint16_t*>(qkv);
  a.positions = positions;
  a.cache_loc = cache_loc;
  a.kc_w = k_cache;
  a.vc_w = v_cache;
  a.rope_table = rope ? rope_table : nullptr;
  a.rope_positions = rope ? rope_positions : 0;
  a.rope = rope;
  a.num_rows = (int64_t)c.num_pages * c.page_size;
  a.tickets = plan->d_tickets;
  a.weight = static_cast<const uint16_t*>(norm_weight);
  a.out = static_cast<uint16_t*>(out);
  a.eps = eps;
  a.q_fold = c.q_norm == OKC_QNORM_FOLDED_SCALE;
  a.q_scale = c.qk_scale_factor;
  a.early = (plan->opts.flags & OKC_PLAN_EARLY_GATHER) && plan->pdl ? 1 : 0;
  a.one_wave = launch_items(plan) <= plan->slots ? 1 : 0;
  cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
  if (plan->sizes.step_kernels == 1) {
    cudaError_t e;
    if (plan->tc) {
      a.tc = 1;
      a.tc_groups = okc::tc_groups(c);
      e = okc::launch_step_fused_tc(a, launch_items(plan), plan->pdl, str);
    } else {
      e = okc::launch_step_fused(a, launch_items(plan), plan->pdl, str);
    }
    return e == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
  }
  // the three kernels, with q in the plan workspace
  okc_status st = okc_prepare_qkv(plan, qkv, positions, cache_loc, k_cache, v_cache, k_scale, v_scale, rope_table,
                                  rope_positions, plan->d_q8, stream);
  if (st != OKC_OK) return st;
  st = okc_attn_decode(plan, plan->d_q8, k_cache, v_cache, k_scale, v_scale, page_table, cache_seqlens,
                       cu_seqlens_q, seq_lens, o_partial, lse_partial, stream);
  if (st != OKC_OK) return st;
  return okc_attn_combine_normgate(plan, o_partial, lse_partial, qkv, norm_weight, eps, out, stream);
}

okc_status okc_attn_step_host(okc_attn_plan_t plan, const okc_host_step* io, uint8_t* k_cache, uint8_t* v_cache,
                              const float* k_scale, const float* v_scale, const float* rope_table,
                              int32_t rope_positions, const void* norm_weight, float eps, float* o_partial,
                              float* lse_partial, okc_stream stream) {
  if (!plan || !io) return OKC_ERR_INVALID;
  const okc_attn_config& c = plan->cfg;
  const size_t T = (size_t)plan->sizes.num_tokens, B = (size_t)c.batch;
  if (B > 0 && (!io->qkv_host || !io->cache_loc_host || !io->cache_seqlens_host || !io->cu_seqlens_q_host ||
                !io->page_table_host || !io->out_host || !io->qkv || !io->cache_loc || !io->cache_seqlens ||
                !io->cu_seqlens_q || !io->page_table || !io->out))
    return OKC_ERR_INVALID;
  if ((io->positions_host == nullptr) != (io->positions == nullptr) ||
      (io->seq_lens_host == nullptr) != (io->seq_lens == nullptr))
    return OKC_ERR_INVALID;
  cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0) return cudaStreamSynchronize(str) == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
  const size_t width = (size_t)(2 * c.num_q_heads + 2 * c.num_kv_heads) * c.head_dim;
  // Each input is read where the device can read it: straight from the host
  // buffer when that is page-locked and mapped and aligned as the kernels load
  // it (16-byte vectors of qkv, naturally aligned indices), else from its
  // device buffer after a copy.
  bool fail = false;
  auto source = [&](const void* host, void* dev, size_t bytes, uintptr_t align) -> const void* {
    if (!host) return nullptr;
    const void* mapped = mapped_host(host);
    if (mapped && (reinterpret_cast<uintptr_t>(mapped) & (align - 1)) == 0) return mapped;
    if (bytes && cudaMemcpyAsync(dev, host, bytes, cudaMemcpyHostToDevice, str) != cudaSuccess) fail = true;
    return dev;
  };
  const void* qkv = source(io->qkv_host, io->qkv, T * width * 2, 16);
  const void* positions = source(io->positions_host, io->positions, T * sizeof(int64_t), 8);
  const void* cache_loc = source(io->cache_loc_host, io->cache_loc, T * sizeof(int64_t), 8);
  const void* cache_seqlens = source(io->cache_seqlens_host, io->cache_seqlens, B * sizeof(int32_t), 4);
  const void* cu_seqlens_q = source(io->cu_seqlens_q_host, io->cu_seqlens_q, (B + 1) * sizeof(int32_t), 4);
  const void* seq_lens = source(io->seq_lens_host, io->seq_lens, B * sizeof(int32_t), 4);
  const void* page_table = source(io->page_table_host, io->page_table, B * (size_t)c.max_pages * sizeof(int32_t), 4);
  if (fail) return OKC_ERR_CUDA;
  // the output: written straight into the host buffer when mapped and aligned
  const void* out_mapped = mapped_host(io->out_host);
  void* out = (out_mapped && aligned16(out_mapped)) ? const_cast<void*>(out_mapped) : io->out;
  okc_status st = okc_attn_step(plan, qkv, static_cast<const int64_t*>(positions),
                                static_cast<const int64_t*>(cache_loc), k_cache, v_cache, k_scale, v_scale, rope_table,
                                rope_positions, static_cast<const int32_t*>(page_table),
                                static_cast<const int32_t*>(cache_seqlens), static_cast<const int32_t*>(cu_seqlens_q),
                                static_cast<const int32_t*>(seq_lens), norm_weight, eps, o_partial, lse_partial, out,
                                stream);
  if (st != OKC_OK) return st;
  const size_t out_bytes = T * (size_t)c.num_q_heads * c.head_dim * 2;
  if (out == io->out && out_bytes &&
      cudaMemcpyAsync(io->out_host, io->out, out_bytes, cudaMemcpyDeviceToHost, str) != cudaSuccess)
    return OKC_ERR_CUDA;
  return cudaStreamSynchronize(str) == cudaSuccess ? OKC_OK : OKC_ERR_CUDA;
}

}  // extern "C"
