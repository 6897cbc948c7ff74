// decode.cu — step 4 of the block: split-KV paged causal GQA attention over the
// E4M3 cache (the flash_attn_with_kvcache call of "012-attention-local-splits.py":
// paged, causal, window_size (window-1, 0), softmax_scale sm_scale*qk_scale_factor,
// k/v descale on the scaled path).
//
// Work item = (query block of a request, chunk of its visible keys), covering
// BOTH KV heads and all the block's query tokens (the whole request for q_len 1
// and 2..16; blocks of 16 consecutive tokens for longer ones), so that at
// page_size 1 every key is one contiguous 128-byte cache row per tensor (K and V).
//
// Warp-specialised pipeline. Four producer warps (16 keys of every tile each)
// turn page-table entries into cache rows and gather them with 16-byte
// cp.async (eight lanes per 128-byte row, so one warp instruction fetches four
// rows) into a ring of kStages tiles of 64 keys (the first page ids are loaded
// from the plan's key range while the device lengths load, and reloaded only
// if they differ); each tile's K and V rows land at a 144-byte pitch so that the
// consumers' ldmatrix reads are bank-conflict free. Each producer lane signals
// a stage's "full" mbarrier when its copies have landed
// (cp.async.mbarrier.arrive); consumer warps release a stage through its
// "empty" mbarrier. Keys that are masked, or whose page id is invalid, are
// zero-filled without a read (an invalid page reads as zeros). Every mbarrier
// wait is bounded in time (mbar_wait): a wait that gives up flags
// OKC_DEVERR_TIMEOUT, and the producer still waits for its own copies before
// it returns.
// (One TMA bulk copy per 128-byte row was measured slower: the copy engine's
// per-request cost caps a small-row gather well below HBM bandwidth.)
//
// With programmatic dependent launch the producer starts fetching the rows of
// keys that were already cached before the prepare kernel has finished; only a
// tile holding one of the step's new keys (written by prepare) waits for it.
//
// Math per consumer warp (one KV head g x a set of query tokens x a share of
// the keys of each tile):
//  QK^T  "swap-AB": D[16 keys x 8 heads] = K_tile[16 x 64] * q^T, two
//        mma.m16n8k32 E4M3 x E4M3 -> f32 (K fragment by ldmatrix.x4 straight
//        from the E4M3 tile, q fragment from registers).
//  softmax: online (m, l) per query row in f32, base 2 with the scale folded in;
//        window/causal/chunk masks only on tiles that need them.
//  PV    D[16 d x 8 heads] += V^T[16 d x 16 keys] * P^T[16 keys x 8 heads] in
//        mma.m16n8k16 f16 -> f32. V^T fragments come from ldmatrix.x4.trans on
//        the E4M3 tile (pairs of bytes moved as b16, then split with a byte
//        permute and converted E4M3->f16 exactly; this permutes the d rows of
//        the output, which the epilogue undoes). P stays in 16-bit precision:
//        the S accumulator fragment becomes the PV B fragment with one
//        movmatrix transpose per 8x8 block.
// Epilogue: warps that split the keys of a tile merge (m, l, O) through shared
// memory; the item writes O/l (times v_scale) and its base-2 log-sum-exp.
//
// The FUSED variant (q_len 1, okc_attn_step in its one-kernel form) also runs
// steps 1-3 (q from qkv in the consumers' fragment layout; the new token's K/V
// row computed by the warp that owns its tile row and written to the cache)
// and step 5 (the last CTA of each request merges the splits).
#include <algorithm>

#include "fused_rows.cuh"
#include "normgate.cuh"
#include "okc_common.cuh"
#include "okc_internal.h"

namespace okc {

namespace {

constexpr int kTileKeys = 64;
constexpr int kRowPitch = kRowBytes + 16;          // 144: conflict-free ldmatrix rows
constexpr int kTileSmem = kTileKeys * kRowPitch;   // one tensor's tile
constexpr int kStageSmem = 2 * kTileSmem;          // K + V
// Build-time tuning knobs (the defaults are the measured best on GB300).
#ifndef OKC_DECODE_STAGES
#define OKC_DECODE_STAGES 4
#endif
#ifndef OKC_DECODE_PRODUCERS
#define OKC_DECODE_PRODUCERS 4  // producer warps per CTA (1, 2 or 4)
#endif
#ifndef OKC_DECODE_KS_L1
#define OKC_DECODE_KS_L1 2  // q_len 1: key shares per KV head (consumer warps = 2 x this)
#endif
#ifndef OKC_DECODE_MINBLOCKS_L1
#define OKC_DECODE_MINBLOCKS_L1 3  // residency hint for the q_len 1 variant
#endif
constexpr int kStages = OKC_DECODE_STAGES;
constexpr int kProducers = OKC_DECODE_PRODUCERS;
static_assert(kProducers == 1 || kProducers == 2 || kProducers == 4, "1, 2 or 4 producer warps");
constexpr int kBarOffset = kStages * kStageSmem;             // full[kStages], empty[kStages]
constexpr int kFlagOffset = kBarOffset + 2 * kStages * 8;    // one int: "this CTA merges"
constexpr int kSmemBytes = kFlagOffset + 16;

// ---- the fused step: steps 1-3 inside the decode CTA (the arithmetic of the
// prepare kernel: correctly rounded RMS inverse (rms_inverse), each float32
// product and sum of the rotation rounded separately, bf16 roundings, E4M3 RNE
// satfinite).

// This lane's q fragment of token t, q head `head`: dims kk*32 + jj*16 + 4*tq + e
// (e = 0..3) land in byte e of q[kk][jj]. The four lanes tq = 0..3 that share the
// head reduce its sum of squares; `live` false makes this lane contribute zeros.
__device__ __forceinline__ void fused_q_frag(const DecodeArgs& a, int64_t t, int head, int tq, bool live,
                                             uint32_t (&q)[2][2], bool& pos_err) {
  float x[16];
  const uint16_t* row = a.qkv + t * kQkvWidth + head * kHeadDim;
#pragma unroll
  for (int grp = 0; grp < 4; grp++) {  // grp = kk*2 + jj
    const uint2 raw = live ? *reinterpret_cast<const uint2*>(row + (grp >> 1) * 32 + (grp & 1) * 16 + 4 * tq)
                           : make_uint2(0u, 0u);
    x[grp * 4 + 0] = bf16_bits_to_f32(raw.x & 0xFFFFu);
    x[grp * 4 + 1] = bf16_bits_to_f32(raw.x >> 16);
    x[grp * 4 + 2] = bf16_bits_to_f32(raw.y & 0xFFFFu);
    x[grp * 4 + 3] = bf16_bits_to_f32(raw.y >> 16);
  }
  const float inv = rms_inverse<4, 16>(x, kRmsEps);
  float y[16];
#pragma unroll
  for (int i = 0; i < 16; i++)  // OKC_QNORM_FOLDED_SCALE: the factor before the one bf16 rounding
    y[i] = bf16_round(a.q_fold ? __fmul_rn(__fmul_rn(x[i], inv), a.q_scale) : __fmul_rn(x[i], inv));
  if (a.rope && live) {
    const int64_t pos = a.positions[t];
    if (pos >= 0 && pos < a.rope_positions) {
      const float* tab = a.rope_table + pos * kHeadDim;
#pragma unroll
      for (int grp = 0; grp < 4; grp++) {
        const int p0 = (grp >> 1) * 16 + (grp & 1) * 8 + 2 * tq;  // pair index of dims 4*... and +1
        const float2 c = *reinterpret_cast<const float2*>(tab + p0);
        const float2 sn = *reinterpret_cast<const float2*>(tab + kHeadDim / 2 + p0);
        const float cc[2] = {c.x, c.y}, sv[2] = {sn.x, sn.y};
#pragma unroll
        for (int u = 0; u < 2; u++) {
          const float e = y[grp * 4 + 2 * u], o = y[grp * 4 + 2 * u + 1];
          y[grp * 4 + 2 * u] = bf16_round(__fsub_rn(__fmul_rn(e, cc[u]), __fmul_rn(o, sv[u])));
          y[grp * 4 + 2 * u + 1] = bf16_round(__fadd_rn(__fmul_rn(o, cc[u]), __fmul_rn(e, sv[u])));
        }
      }
    } else {
      pos_err = true;
    }
  }
#pragma unroll
  for (int grp = 0; grp < 4; grp++)
    q[grp >> 1][grp & 1] = (uint32_t)f32x2_to_e4m3x2(y[grp * 4], y[grp * 4 + 1]) |
                           ((uint32_t)f32x2_to_e4m3x2(y[grp * 4 + 2], y[grp * 4 + 3]) << 16);
}

template <int KS, int NTW, int NCW>
struct DecodeCfg {
  static constexpr int kMTiles = 4 / KS;  // 16-key m-tiles per consumer warp per tile
};

// FUSED false: the decode kernel of the three-call path (q from q_fp8, partials
// out); true: the whole step (okc_attn_step), last-CTA merge through tickets.
// QCVT: the V conversion's form, four E4M3 codes per pair of cvt instructions
// straight from the register halves, or the per-pair form (the same exact
// values; which runs faster depends on the step, see launch_step_fused).
template <int KS, int NTW, int NCW, bool FUSED, bool QCVT = !FUSED>
__global__ void __launch_bounds__((NCW + kProducers) * 32, KS > 1 ? OKC_DECODE_MINBLOCKS_L1 : 1)
    decode_kernel(DecodeArgs a) {
  using C = DecodeCfg<KS, NTW, NCW>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sbase = smem_u32(smem);
  auto full_bar = [&](int s) { return sbase + kBarOffset + 8 * s; };
  auto empty_bar = [&](int s) { return sbase + kBarOffset + 8 * (kStages + s); };

  // The work item is plan data (written when the plan was made): it is read
  // before the programmatic-dependency wait, overlapping the previous kernel.
  // A fixed-capacity plan launches its capacity: CTAs past the live count return.
  if (a.live_work && (int)blockIdx.x >= *a.live_work) return;
  const WorkItem wk = a.work[blockIdx.x];
  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(full_bar(s), 32 * kProducers);  // one cp.async-tracked arrival per producer lane
      mbar_init(empty_bar(s), NCW);
    }
    fence_mbar_init();
  }
  const int b = wk.b;

  if constexpr (FUSED) {
    // The first kernel of the step: its predecessor may write any input, so by
    // default everything waits for it. Under OKC_PLAN_EARLY_GATHER the caller
    // promises that the preceding kernels write neither the page table, the
    // lengths, nor any cache row this step reads: then the lengths, the page ids
    // and the already-cached keys are loaded before the wait, and only the
    // consumers wait (q, the new K/V rows and every global write come after it).
    if (!a.early) {
      pdl_wait();
      pdl_launch_dependents();
    }
    // the gate logits and norm weight the merge reads at the end: into L2 now
    // (the block's first token under the plan's q lengths)
    if (tid < 16) prefetch_l2(a.qkv + (int64_t)wk.t0 * kQkvWidth + kGateCol + tid * 64);
    if (tid == 16 && a.weight) prefetch_l2(a.weight);
  }

  // ---- producer set-up: page ids of the first kStages tiles, loaded with the
  // item's key range under the plan's lengths while the request's lengths
  // (caller inputs) are still in flight; checked against them below.
  // Producer warp pw owns keys [pw*kKeysPW, (pw+1)*kKeysPW) of every tile.
  // Lane (rr, ch) = (lane >> 3, lane & 7) copies 16-byte chunk ch of the owned
  // rows rr, rr+4, ...; eight lanes cover one 128-byte row, so each warp
  // instruction fetches four whole rows. Page ids: lane l loads the ids of owned
  // keys l, l+32, ... and the row owners read them by shuffle.
  constexpr int kKeysPW = kTileKeys / kProducers;  // keys per producer warp per tile
  constexpr int kIds = kKeysPW >= 32 ? kKeysPW / 32 : 1;  // page ids per lane per tile
  const int pw = warp - NCW, kbase = pw * kKeysPW;
  const int32_t* pt = a.page_table + (int64_t)b * a.max_pages;
  // ids of tile `tile` of key range [jb, je)
  auto load_ids = [&](int (&dst)[kIds], int tile, int jb, int je) {
#pragma unroll
    for (int q = 0; q < kIds; q++) {
      const int j = jb + tile * kTileKeys + kbase + 32 * q + lane;
      dst[q] = (32 * q + lane < kKeysPW && j < je) ? __ldg(pt + (j >> a.page_shift)) : -1;
    }
  };
  // Page ids live in a register ring one slot per stage: the ids of tile k are
  // loaded when tile k - kStages is issued, so their latency hides behind a
  // whole ring of copies.
  int ids[kStages][kIds];
  if (warp >= NCW) {
#pragma unroll
    for (int t = 0; t < kStages; t++) load_ids(ids[t], t, wk.j0, wk.j1);
  }

  // ---- the request's lengths (caller inputs)
  int n = a.cache_seqlens[b];
  const int qb = a.cu_seqlens_q[b];
  int ql = a.cu_seqlens_q[b + 1] - qb;
  const int P = 1 << a.page_shift;
  bool bad_len = ql < 0 || ql > a.L || qb < 0 || qb + ql > a.T || n < ql ||
                 (a.seq_lens && a.seq_lens[b] != n - ql) || (int64_t)n > (int64_t)a.max_pages * P;
  if (bad_len) {  // keep every access in range; the result of this request is void
    ql = max(0, min(ql, a.L));
    if (qb < 0 || qb + ql > a.T) ql = 0;
    n = max(ql, min(n, a.max_pages * P));
  }
  // this block's tokens i0 .. i0 + ntk - 1 of the request, at positions pbase + tok
  // (blocks of one token start at the request's first: i0 = 0)
  const int i0 = (KS > 1) ? 0 : wk.i0;
  const int ntk = max(0, min(a.S, ql - i0));
  if (ntk != wk.ntok || (wk.last && i0 + ntk < ql)) bad_len = true;  // q lengths differ from the plan's
  const int pbase = n - ql + i0;
  const int hi = pbase + ntk;                                           // keys < hi
  const int lo = a.window > 0 ? max(0, pbase - a.window + 1) : 0;     // first key any query sees
  const int j0 = lo + wk.koff;
  const int j1 = min(hi, j0 + wk.cap);
  if (wk.chunk == wk.nchunks - 1 && j1 < hi) bad_len = true;  // plan does not cover the keys
  if (bad_len && tid == 0) set_error(a.err, OKC_DEVERR_LENGTHS);
  const int ntiles = j1 > j0 ? (j1 - j0 + kTileKeys - 1) / kTileKeys : 0;
  __syncthreads();  // barriers initialised

  if (warp >= NCW) {
    // ================================================================ producer
    if (j0 != wk.j0 || j1 != wk.j1) {  // the lengths differ from the plan's: reload
#pragma unroll
      for (int t = 0; t < kStages; t++) load_ids(ids[t], t, j0, j1);
    }
    const int pmask = P - 1;
    const int newk = n - ql;  // keys >= newk are written by the prepare kernel (three-call path)
    const int rr = lane >> 3, ch = lane & 7;
    // no wait before a tile: the three-call decode waits for the prepare kernel
    // before a tile holding one of the step's new keys; the fused step computes
    // those keys itself (the gathered row is replaced), having waited already or
    // needing no wait (OKC_PLAN_EARLY_GATHER)
    bool dep = FUSED, bad_page = false;
    auto issue = [&](int k, const int (&id)[kIds]) {
      const int s = k % kStages;
      const uint32_t sK = sbase + s * kStageSmem, sV = sK + kTileSmem;
      const int tj = j0 + k * kTileKeys;
      if (!dep && min(j1, tj + kTileKeys) > newk) {  // this tile holds a key prepare writes
        pdl_wait();
        dep = true;
      }
#pragma unroll
      for (int i = 0; i < kKeysPW / 4; i++) {
        const int rl = rr + 4 * i;  // row within this warp's keys
        const int r = kbase + rl;
        const int pg = __shfl_sync(0xffffffffu, id[rl >> 5], rl & 31);
        const int j = tj + r;
        int64_t row = 0;
        int bytes = 0;  // 0: zero-fill, read nothing (masked key or invalid page)
        if (j < j1) {
          if (pg >= 0 && pg < a.num_pages) {
            row = ((int64_t)pg << a.page_shift) | (j & pmask);
            bytes = 16;
          } else {
            bad_page = true;
          }
        }
        const uint32_t off = r * kRowPitch + ch * 16;
        cp_async_16(sK + off, a.kc + row * kRowBytes + ch * 16, bytes);
        cp_async_16(sV + off, a.vc + row * kRowBytes + ch * 16, bytes);
      }
      cp_async_mbar_arrive(full_bar(s));
    };

#pragma unroll
    for (int t = 0; t < kStages; t++) {
      if (t < ntiles) issue(t, ids[t]);
      load_ids(ids[t], t + kStages, j0, j1);
    }
    bool ok = true;
    for (int k0 = kStages; k0 < ntiles && ok; k0 += kStages) {
#pragma unroll
      for (int u = 0; u < kStages; u++) {  // tile k = k0 + u uses ring slot u
        const int k = k0 + u;
        if (k >= ntiles) break;
        if (!mbar_wait(empty_bar(u), ((k / kStages) & 1) ^ 1)) { ok = false; break; }
        issue(k, ids[u]);
        load_ids(ids[u], k + kStages, j0, j1);
      }
    }
    if (bad_page && ch == 0) set_error(a.err, OKC_DEVERR_PAGE);
    if (!ok && lane == 0) set_error(a.err, OKC_DEVERR_TIMEOUT);
    cp_async_wait_all();  // this warp's copies have landed before it leaves
    return;
  }

  // ================================================================ consumers
  const int g = warp & 1;                       // KV head of this warp
  const int sub = warp >> 1;
  const int ks = (KS > 1) ? sub : 0;            // key share (L = 1 mode)
  const int tok0 = (KS > 1) ? 0 : sub * NTW;    // first query token of this warp
  const int gq = lane >> 2, tq = lane & 3;      // mma fragment coordinates
  // logit scale in base 2; on the scaled path every key is its E4M3 value times k_scale
  const float scale_log2 = a.scaled ? a.scale_log2 * __ldg(a.k_scale) : a.scale_log2;

  bool pos_err = false;
  uint32_t qf[NTW][2][2];
  if constexpr (FUSED) {
    if (a.early) {  // qkv and the outputs: after the predecessor has finished
      pdl_wait();
      pdl_launch_dependents();
    }
#pragma unroll
    for (int nt = 0; nt < NTW; nt++) {
      const int tok = tok0 + nt;
      fused_q_frag(a, (int64_t)qb + i0 + (tok < ntk ? tok : 0), g * kGroup + gq, tq, tok < ntk, qf[nt], pos_err);
    }
  } else {
    pdl_wait();  // q_fp8 is the prepare kernel's output
    pdl_launch_dependents();
#pragma unroll
    for (int nt = 0; nt < NTW; nt++) {
      const int tok = tok0 + nt;
      const uint8_t* qrow = a.q8 + ((int64_t)(qb + i0 + tok) * kNumQHeads + g * kGroup + gq) * kHeadDim;
#pragma unroll
      for (int kk = 0; kk < 2; kk++) {
        qf[nt][kk][0] = tok < ntk ? *reinterpret_cast<const uint32_t*>(qrow + kk * 32 + tq * 4) : 0u;
        qf[nt][kk][1] = tok < ntk ? *reinterpret_cast<const uint32_t*>(qrow + kk * 32 + 16 + tq * 4) : 0u;
      }
    }
  }

  float o[4][NTW][4];
  float m[NTW][2], l[NTW][2];
#pragma unroll
  for (int nt = 0; nt < NTW; nt++) {
#pragma unroll
    for (int c = 0; c < 2; c++) { m[nt][c] = -INFINITY; l[nt][c] = 0.f; }
#pragma unroll
    for (int dt = 0; dt < 4; dt++)
#pragma unroll
      for (int e = 0; e < 4; e++) o[dt][nt][e] = 0.f;
  }
  const int tok_last = min(tok0 + NTW, ntk) - 1;
  // lane-dependent parts of the ldmatrix addresses
  const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8, k_ch = g * 4 + (lane >> 4);
  const int v_row = (lane & 7) + (lane >> 4) * 8, v_ch = g * 4 + ((lane >> 3) & 1);

  for (int k = 0; k < ntiles; k++) {
    const int s = k % kStages;
    if (!mbar_wait(full_bar(s), (k / kStages) & 1)) {
      if (lane == 0) set_error(a.err, OKC_DEVERR_TIMEOUT);
      break;
    }
    const uint32_t ks_base = sbase + s * kStageSmem;
    const uint32_t vs_base = ks_base + kTileSmem;
    const int tile_j = j0 + k * kTileKeys;
    if constexpr (FUSED) {
      // The step's new keys in this warp's rows of the tile: computed here from
      // qkv, put in place of the gathered row, and written to the cache (once,
      // by the warp that owns the row in its key share / the first token group).
      const int wlo = tile_j + ks * C::kMTiles * 16;
      const int whi = min(j1, wlo + C::kMTiles * 16);
      const bool writer = (KS > 1) || sub == 0;
      for (int j = max(wlo, pbase); j < whi; j++) {
        const int64_t t = (int64_t)qb + i0 + (j - pbase);
        uint16_t k8, v8;
        fused_new_kv(a, t, g, lane, k8, v8, pos_err);
        const int r = j - tile_j;
        uint8_t* srow = smem + s * kStageSmem + r * kRowPitch + g * kHeadDim + 2 * lane;
        *reinterpret_cast<uint16_t*>(srow) = k8;
        *reinterpret_cast<uint16_t*>(srow + kTileSmem) = v8;
        if (writer) {
          const int64_t slot = a.cache_loc[t];
          if (slot >= 0 && slot < a.num_rows) {
            *reinterpret_cast<uint16_t*>(a.kc_w + slot * kRowBytes + g * kHeadDim + 2 * lane) = k8;
            *reinterpret_cast<uint16_t*>(a.vc_w + slot * kRowBytes + g * kHeadDim + 2 * lane) = v8;
          } else if (lane == 0) {
            set_error(a.err, OKC_DEVERR_CACHE_LOC);
          }
        }
      }
      __syncwarp();
    }
    if (tok_last >= tok0) {
      const int key_hi = tile_j + kTileKeys - 1;
      const int p_lo = pbase + tok0, p_hi = pbase + tok_last;
      const bool full = key_hi < j1 && key_hi <= p_lo &&
                        (a.window == 0 || tile_j >= p_hi - a.window + 1) && (tok0 + NTW - 1 < ntk);

      float sc[C::kMTiles][NTW][4];
#pragma unroll
      for (int mi = 0; mi < C::kMTiles; mi++) {
        const int mt = ks * C::kMTiles + mi;
        uint32_t a0[4], a1[4];
        const uint32_t ra = ks_base + (mt * 16 + k_row) * kRowPitch;
        ldsm_x4(a0, ra + k_ch * 16);
        ldsm_x4(a1, ra + (k_ch + 2) * 16);
#pragma unroll
        for (int nt = 0; nt < NTW; nt++) {
          sc[mi][nt][0] = sc[mi][nt][1] = sc[mi][nt][2] = sc[mi][nt][3] = 0.f;
          mma_e4m3_16832(sc[mi][nt], a0, qf[nt][0][0], qf[nt][0][1]);
          mma_e4m3_16832(sc[mi][nt], a1, qf[nt][1][0], qf[nt][1][1]);
        }
      }
#pragma unroll
      for (int mi = 0; mi < C::kMTiles; mi++) {
        const int mt = ks * C::kMTiles + mi;
#pragma unroll
        for (int nt = 0; nt < NTW; nt++) {
#pragma unroll
          for (int e = 0; e < 4; e++) {
            float v = sc[mi][nt][e] * scale_log2;
            if (!full) {
              const int j = tile_j + mt * 16 + gq + (e >> 1) * 8;
              const int tok = tok0 + nt;
              const int p = pbase + tok;
              const bool okm = j < j1 && tok < ntk && j <= p && (a.window == 0 || j >= p - a.window + 1);
              v = okm ? v : -INFINITY;
            }
            sc[mi][nt][e] = v;
          }
        }
      }
      uint32_t pb[C::kMTiles][NTW][2];
#pragma unroll
      for (int nt = 0; nt < NTW; nt++) {
#pragma unroll
        for (int c = 0; c < 2; c++) {
          float mx = -INFINITY;
#pragma unroll
          for (int mi = 0; mi < C::kMTiles; mi++) mx = fmaxf(mx, fmaxf(sc[mi][nt][c], sc[mi][nt][c + 2]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m[nt][c], mx);
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          const float alpha = fast_exp2(m[nt][c] - m_use);
          m[nt][c] = m_new;
          float sum = 0.f;
#pragma unroll
          for (int mi = 0; mi < C::kMTiles; mi++) {
            sc[mi][nt][c] = fast_exp2(sc[mi][nt][c] - m_use);
            sc[mi][nt][c + 2] = fast_exp2(sc[mi][nt][c + 2] - m_use);
            sum += sc[mi][nt][c] + sc[mi][nt][c + 2];
          }
          l[nt][c] = l[nt][c] * alpha + sum;
#pragma unroll
          for (int dt = 0; dt < 4; dt++) {
            o[dt][nt][c] *= alpha;
            o[dt][nt][c + 2] *= alpha;
          }
        }
#pragma unroll
        for (int mi = 0; mi < C::kMTiles; mi++) {
          pb[mi][nt][0] = movmatrix_trans(pack_half2(sc[mi][nt][0], sc[mi][nt][1]));
          pb[mi][nt][1] = movmatrix_trans(pack_half2(sc[mi][nt][2], sc[mi][nt][3]));
        }
      }
#pragma unroll
      for (int mi = 0; mi < C::kMTiles; mi++) {
        const int mt = ks * C::kMTiles + mi;
        const uint32_t rv = vs_base + (mt * 16 + v_row) * kRowPitch;
#pragma unroll
        for (int half = 0; half < 2; half++) {  // d in [32*half, 32*half+32)
          uint32_t r[4];
          ldsm_x4_trans(r, rv + (v_ch + half * 2) * 16);
          uint32_t ax[4], ay[4];
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const uint32_t pr = __byte_perm(r[i], 0u, 0x3120);
            if constexpr (QCVT) {
              e4m3x4_to_f16x2x2(pr, ax[i], ay[i]);
            } else {
              ax[i] = e4m3x2_to_f16x2((uint16_t)(pr & 0xFFFFu));
              ay[i] = e4m3x2_to_f16x2((uint16_t)(pr >> 16));
            }
          }
#pragma unroll
          for (int nt = 0; nt < NTW; nt++) {
            mma_f16_16816(o[half * 2 + 0][nt], ax, pb[mi][nt][0], pb[mi][nt][1]);
            mma_f16_16816(o[half * 2 + 1][nt], ay, pb[mi][nt][0], pb[mi][nt][1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(s));  // this warp is done reading stage s
  }

  // ---- epilogue: full row sums, merge key shares, write the partials
#pragma unroll
  for (int nt = 0; nt < NTW; nt++)
#pragma unroll
    for (int c = 0; c < 2; c++) {
      l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 4);
      l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 8);
      l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 16);
    }
  if constexpr (KS > 1) {
    // warps with ks > 0 park (o, m, l) in shared memory; ks == 0 merges them
    named_bar_sync(1, NCW * 32);  // every consumer is past its last tile: reuse the ring
    float* xs = reinterpret_cast<float*>(smem);
    constexpr int kPer = 4 * NTW * 4 + NTW * 4;  // o + (m, l) per lane
    if (ks > 0) {
      float* dst = xs + (((ks - 1) * 2 + g) * 32 + lane) * kPer;
      int q = 0;
#pragma unroll
      for (int dt = 0; dt < 4; dt++)
#pragma unroll
        for (int nt = 0; nt < NTW; nt++)
#pragma unroll
          for (int e = 0; e < 4; e++) dst[q++] = o[dt][nt][e];
#pragma unroll
      for (int nt = 0; nt < NTW; nt++)
#pragma unroll
        for (int c = 0; c < 2; c++) { dst[q++] = m[nt][c]; dst[q++] = l[nt][c]; }
    }
    named_bar_sync(1, NCW * 32);
    if (ks == 0) {
#pragma unroll 1
    for (int other = 1; other < KS; other++) {
      const float* src = xs + (((other - 1) * 2 + g) * 32 + lane) * kPer;
      float o2[4][NTW][4];
      int q = 0;
#pragma unroll
      for (int dt = 0; dt < 4; dt++)
#pragma unroll
        for (int nt = 0; nt < NTW; nt++)
#pragma unroll
          for (int e = 0; e < 4; e++) o2[dt][nt][e] = src[q++];
#pragma unroll
      for (int nt = 0; nt < NTW; nt++)
#pragma unroll
        for (int c = 0; c < 2; c++) {
          const float m2 = src[q++], l2 = src[q++];
          const float mm = fmaxf(m[nt][c], m2);
          const float mu = mm == -INFINITY ? 0.f : mm;
          const float f1 = fast_exp2(m[nt][c] - mu), f2 = fast_exp2(m2 - mu);
          m[nt][c] = mm;
          l[nt][c] = l[nt][c] * f1 + l2 * f2;
#pragma unroll
          for (int dt = 0; dt < 4; dt++) {
            o[dt][nt][c] = o[dt][nt][c] * f1 + o2[dt][nt][c] * f2;
            o[dt][nt][c + 2] = o[dt][nt][c + 2] * f1 + o2[dt][nt][c + 2] * f2;
          }
        }
    }
    }  // ks == 0
  }

  const float vscale = a.scaled ? *a.v_scale : 1.0f;
  const int rows = a.S * kNumQHeads;  // rows of an output slot: the block's tokens x heads
  const int64_t slot = (int64_t)wk.wbase + wk.chunk;
  float* obase = a.o_part + slot * rows * kHeadDim;
  float* lbase = a.lse_part + slot * rows;
#pragma unroll
  for (int nt = 0; nt < NTW; nt++) {
    if (ks > 0) break;  // key shares were merged into ks == 0
    const int tok = tok0 + nt;
    if (tok >= ntk) continue;
#pragma unroll
    for (int c = 0; c < 2; c++) {
      const int head = g * kGroup + 2 * tq + c;
      const int row = tok * kNumQHeads + head;
      const float lv = l[nt][c];
      const float inv = lv > 0.f ? vscale / lv : 0.f;
      float* orow = obase + (int64_t)row * kHeadDim;
      // output row of o[dt][nt][c + 2*hi]: d = 32*(dt>>1) + 16*hi + 2*gq + (dt&1)
#pragma unroll
      for (int half = 0; half < 2; half++)
#pragma unroll
        for (int hi = 0; hi < 2; hi++) {
          const int d = 32 * half + 16 * hi + 2 * gq;
          *reinterpret_cast<float2*>(orow + d) =
              make_float2(o[half * 2][nt][c + 2 * hi] * inv, o[half * 2 + 1][nt][c + 2 * hi] * inv);
        }
      if (gq == 0) lbase[row] = lv > 0.f ? m[nt][c] + log2f(lv) : -INFINITY;
    }
  }

  if constexpr (FUSED) {
    // Last CTA of the request merges every split and applies the norm-gate: once
    // the CTA's partials are written (barrier), one thread takes a ticket with
    // an acquire-release atomic (publishing them; measured 0.5 us faster on the
    // sliding step than a fence on each side of a relaxed atomic); the CTA that
    // draws the last ticket reads all partials (L2 loads) and resets the counter
    // for the next launch. Nothing waits on another CTA.
    volatile int& s_last = *reinterpret_cast<int*>(smem + kFlagOffset);
    if (pos_err && lane == 0) set_error(a.err, OKC_DEVERR_POSITION);
    named_bar_sync(1, NCW * 32);
    if (tid == 0) {
      // the release publishes the partials the CTA wrote (they precede it
      // through the barrier); for the last CTA the acquire orders the other
      // splits' partials before the merge's reads (the barrier below)
      int prev;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(prev) : "l"(a.tickets + b) : "memory");
      s_last = prev == wk.nchunks - 1;
    }
    named_bar_sync(1, NCW * 32);
    if (s_last) {
      const int64_t base_lse = (int64_t)wk.wbase * rows;
      for (int rowi = tid >> 3; rowi < ntk * kNumQHeads; rowi += NCW * 4) {  // 8 lanes per row
        const int tok = rowi / kNumQHeads, h = rowi % kNumQHeads;
        const int64_t t = (int64_t)qb + i0 + tok;
        const int c0 = (tid & 7) * 8;
        float gg[8], ww[8];
        load_gate_weight(a.qkv, a.weight, (int)t, h, c0, gg, ww);
        merge_normgate(a.lse_part + base_lse + rowi, rows,
                       a.o_part + (base_lse + rowi) * kHeadDim + c0, (int64_t)rows * kHeadDim, wk.nchunks, gg,
                       ww, a.eps, a.out + t * (kNumQHeads * kHeadDim) + h * kHeadDim + c0);
      }
      if (tid == 0) a.tickets[b] = 0;
    }
  }
}

template <int KS, int NTW, int NCW, bool FUSED, bool QCVT = !FUSED>
cudaError_t launch_variant(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  // the dynamic shared-memory limit was raised when the plan was made (occupancy query)
  auto kern = decode_kernel<KS, NTW, NCW, FUSED, QCVT>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_work);
  cfg.blockDim = dim3((NCW + kProducers) * 32);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int KS, int NTW, int NCW, bool FUSED, bool QCVT = !FUSED>
int occupancy_variant() {
  int nb = 0;
  auto kern = decode_kernel<KS, NTW, NCW, FUSED, QCVT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, (NCW + kProducers) * 32, kSmemBytes) != cudaSuccess)
    return 0;
  return nb;
}

// The variant for query blocks of S tokens (S <= 16).
cudaError_t launch_any(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  if (num_work == 0) return cudaSuccess;
  if (a.S < 1 || a.S > 16) return cudaErrorInvalidValue;
  if (a.S == 1) return launch_variant<OKC_DECODE_KS_L1, 1, 2 * OKC_DECODE_KS_L1, false>(a, num_work, pdl, s);
  if (a.S <= 2) return launch_variant<1, 2, 2, false>(a, num_work, pdl, s);
  if (a.S <= 4) return launch_variant<1, 2, 4, false>(a, num_work, pdl, s);
  if (a.S <= 8) return launch_variant<1, 2, 8, false>(a, num_work, pdl, s);
  return launch_variant<1, 2, 16, false>(a, num_work, pdl, s);
}

int occupancy_any(int S) {
  if (S == 1) return occupancy_variant<OKC_DECODE_KS_L1, 1, 2 * OKC_DECODE_KS_L1, false>();
  if (S <= 2) return occupancy_variant<1, 2, 2, false>();
  if (S <= 4) return occupancy_variant<1, 2, 4, false>();
  if (S <= 8) return occupancy_variant<1, 2, 8, false>();
  return occupancy_variant<1, 2, 16, false>();
}

}  // namespace

// Blocks of 1 token: 2*KS consumer warps (2 KV heads x KS key shares), one
// n-tile of 8 heads each; blocks of 2..16 tokens: one consumer warp per KV head
// per pair of tokens; on the tcgen05 kernel when the plan chose it.
cudaError_t launch_decode(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  if (a.tc) return launch_decode_tc(a, num_work, pdl, s);
  return launch_any(a, num_work, pdl, s);
}

// The single-launch step is built for q_len 1 only: for a verify block the
// three kernels are faster (one CTA per SM at the fused variant's registers,
// and every split recomputing the block's new K/V rows).
//
// Its V conversion: the four-code form for steps of at most one wave of items
// (the sliding batch: 15.6 -> 14.5 us per step), the per-pair form for longer
// ones (the mixed batch: 162.9 us with the four-code form, 159.9 us without).
cudaError_t launch_step_fused(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  if (a.L != 1 || a.S != 1) return cudaErrorInvalidValue;
  if (num_work == 0) return cudaSuccess;
  if (a.one_wave) return launch_variant<OKC_DECODE_KS_L1, 1, 2 * OKC_DECODE_KS_L1, true, true>(a, num_work, pdl, s);
  return launch_variant<OKC_DECODE_KS_L1, 1, 2 * OKC_DECODE_KS_L1, true, false>(a, num_work, pdl, s);
}

int decode_ctas_per_sm(int S, bool tc, int tc_groups) {
  if (tc) return decode_tc_ctas_per_sm(tc_groups);
  const int a = occupancy_any(S);
  if (S != 1) return a;
  const int b = occupancy_variant<OKC_DECODE_KS_L1, 1, 2 * OKC_DECODE_KS_L1, true, false>();
  const int c = occupancy_variant<OKC_DECODE_KS_L1, 1, 2 * OKC_DECODE_KS_L1, true, true>();
  return std::min(a, std::min(b, c));
}

}  // namespace okc
