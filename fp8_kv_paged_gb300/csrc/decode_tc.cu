// decode_tc.cu — step 4 for query blocks of 2..16 tokens on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory): the
// flash_attn_with_kvcache call of "012-attention-local-splits.py" with a
// block's queries, paged, causal within the block, window (window-1, 0). It
// serves the speculative verify block (q_len <= 8: one block per request) and
// prefill/extend (requests cut into blocks of 16 consecutive tokens).
//
// One CTA per work item (query block of a request, chunk of its visible keys),
// as in decode.cu, in one of two forms (TcCfg<NG>, chosen by the plan; one CTA
// per SM, 512 TMEM columns):
//  - form 2 (blocks of up to 8 tokens): the CTA holds all 128 q rows of the
//    block (up to 8 tokens x 16 heads, rows g*64 + i*8 + hh for KV head g,
//    token i of the block, head g*8 + hh; rows of tokens past the block are
//    zero and ignored) as ONE M = 128 operand, and two softmax warpgroups take
//    alternate tiles:
//      S [128 x 64 keys] = Q [128 x 128] . K_tile^T   (kind::f8f6f4, E4M3 x E4M3)
//      O [128 x 144]    += P [128 x 64] . [V_tile | 1] (kind::f16, P and V in
//                          f16, P read from tensor memory)
//    GQA without splitting the MMA by KV head: a q row of KV head g carries its
//    64 dims at K positions [64g, 64g+64) and zeros elsewhere, against K rows
//    that hold both heads' 64 dims (the cache row as stored), so S = q . k_g
//    exactly; for PV every row gets both heads' 64 output dims and keeps its
//    own half;
//  - form 3 (blocks of up to 16 tokens): one softmax warpgroup per KV head j,
//    both on every tile, group j's 128 rows the block's 16 tokens x the 8 q
//    heads of KV head j (row 8 i + hh):
//      S_j [128 x 64 keys] = Q_j [128 x 64] . K_tile,j^T  (head j's 64 K bytes)
//      O_j [128 x 80]     += P_j [128 x 64] . [V_tile,j | 1]
//    half the tensor work per q row of form 2, and each tile's V conversion
//    split between the groups.
// Column 64 (form 3) or 128 (form 2) of the PV's B operand is all ones, so
// O's column there is the row sum of P as the tensor core saw it (f16 P, f32
// sums): the softmax denominator, consistent with the numerator and kept by
// the same rescales.
//
// Q is the QK's A operand in TMEM, so the QK reads only K from shared memory.
// Warps: the softmax groups (thread r of a group owns q row r), then one warp
// that issues the QK and PV MMAs (one thread, a ready PV before the next QK)
// and owns the TMEM allocation, then two gather warps: on pages of 8 or more
// rows each issues the TMA loads of four of a tile's eight 8-row groups (8-row
// boxes, 128-byte swizzle, read by the MMA through a swizzled descriptor; one
// warp's TMA issues are serialised, so two issuing warps gather faster than
// one), else both run the cp.async producer of decode.cu (K rows in the MMA's
// no-swizzle canonical layout, V rows in a staging tile). Each group j has its
// own S, P and O in TMEM and its own V^T tile in shared memory, so one group's
// softmax overlaps the other group's MMAs. Per tile k of group j:
//   MMA:     wait tile k -> S_j = Q K^T -> commit(s_ready_j)
//   group j: wait s_ready_j -> S row from TMEM -> arrive(s_free_j) -> mask; row
//            max; P = 2^(s - m) (f16 pairs) in registers -> wait pv_done_j of
//            its previous tile -> P into TMEM (tcgen05.st); V tile E4M3 -> f16
//            transposed (ldmatrix, exact conversion, stmatrix.trans; V^T rows
//            permuted within 16-dim blocks, vt_pos, so the stores hit no bank
//            conflicts) -> arrive(p_ready_j)
//   MMA:     wait p_ready_j -> free the stage (form 3: once both groups have
//            consumed the tile) -> O_j += P V -> commit(pv_done_j)
// O accumulates in TMEM against a reference max m per row that moves when the
// row's max grows past m + kTcRescale (log2 units; 0 by default: the exact
// running max, P <= 1): then the row's O is rescaled in TMEM (tcgen05.ld / st)
// before the next PV. At the end (form 2: the groups merge their (m, l, O))
// the CTA writes O/l (times v_scale) through shared memory (whole 128-byte
// lines) and the base-2 LSE per row, as decode.cu does; the combine kernel
// merges the splits. The one-kernel step (FUSED, form 2) also derives q and the
// step's new K/V rows from qkv and merges the splits in the block's last CTA.
//
// Shared-memory operands (V^T, K on the cp.async path) use the no-swizzle
// K-major layout (8-row x 16-byte core matrices; core matrices 128 bytes apart
// along K, 8-row groups 1024 bytes apart for 128-byte rows); K on the TMA path
// the 128-byte-swizzle K-major layout. Every wait is bounded (mbar_wait); on a
// timeout the kernel flags OKC_DEVERR_TIMEOUT, waits for the copies and MMAs
// it issued and frees its TMEM before it returns.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "fused_rows.cuh"
#include "normgate.cuh"
#include "okc_common.cuh"
#include "okc_internal.h"

namespace okc {

namespace {

constexpr int kTcTileKeys = 64;
constexpr int kTcRows = 128;      // q rows per CTA (M)
constexpr int kTcVPitch = 144;    // V staging row pitch: conflict-free ldmatrix
constexpr uint32_t kTcLbo = 128;  // next core matrix along K
constexpr uint32_t kTcSbo = 1024; // next 8-row group (rows of 128 bytes)
#ifndef OKC_TC_RESCALE
#define OKC_TC_RESCALE 0
#endif
constexpr float kTcRescale = OKC_TC_RESCALE;  // log2 headroom of the reference max (0: exact max)
constexpr int kTcPvN = 144;                   // PV's N: 128 dims + the ones column
// The form of the kernel (chosen by the plan, tc_groups), NG; either runs one
// CTA per SM (512 TMEM columns, 6 stages):
//  2: two softmax warpgroups taking alternate tiles (tile k goes to group k & 1, its
//     phase is bit 0 of k >> 1), blocks of up to 8 tokens x 16 heads;
//  3: two warpgroups, one per KV head, both on every tile: blocks of up to 16
//     tokens, group j's 128 rows the block's 16 tokens x the 8 q
//     heads of KV head j (row 8 i + hh: token i, head 8 j + hh), so the QK reads
//     only head j's 64 K bytes (K = 64) and the PV only head j's 64 V dims
//     (N = 64 + 16): half the tensor work per q row of form 2, whose rows mix
//     both heads, and one V conversion per tile for the block's 256 rows. (A
//     one-group form at two CTAs per SM on blocks of 8 tokens ran extends 11 %
//     slower.)

// The layout of a CTA of form NG. Warps 0 .. 4 kGroups - 1 run the softmax,
// warp 4 kGroups issues the MMAs, the next kProducers gather.
template <int NG>
struct TcCfg {
  static_assert(NG == 2 || NG == 3, "forms 2 and 3");
  static constexpr bool kPH = NG == 3;              // one group per KV head
  static constexpr int kGroups = kPH ? 2 : NG;      // softmax warpgroups
  static constexpr int kStep = kPH ? 1 : NG;        // group j's tiles: j (0 for kPH), + kStep, ...
  static constexpr int kShift = kPH ? 0 : NG - 1;   // the phase of tile k: bit 0 of k >> kShift
  static constexpr int kPvN = kPH ? 64 + 16 : kTcPvN;  // PV's N: the dims + the ones column (and zeros)
  static constexpr int kVTBytes = kPvN * 128;       // [V | 1]^T f16 [kPvN x 64 keys]
  static constexpr int kStages = 6;
  static constexpr int kMmaWarp = 4 * kGroups;
  // gather warps: TMA issues from one warp are serialised, so each producer
  // warp issues its share of a tile's boxes (a third or fourth warp gathered
  // no faster, and a fourth held back the CTAs of the neighbouring kernels)
  static constexpr int kProducers = 2;
  static constexpr int kThreads = (kMmaWarp + 1 + kProducers) * 32;
  // shared memory (Q, the QK's A operand, is in TMEM: the QK reads only K
  // from shared memory)
  static constexpr int kK = 0;                                            // K E4M3 [stage][64 x 128 B]
  static constexpr int kV = kK + kStages * kTcTileKeys * 128;             // V E4M3 [stage][64 x 144 B]
  static constexpr int kVT = kV + kStages * kTcTileKeys * kTcVPitch;      // [V | 1]^T f16 [group][kPvN x 64 keys]
  static constexpr int kX = kVT + kGroups * kVTBytes;                     // each group's reference max per row
  // the one-kernel step: the step's new K and V rows for this CTA's keys (at
  // most 8 keys x K | V x 128 bytes), computed once and put into the tiles
  static constexpr int kNew = kX + kGroups * kTcRows * 4;
  static constexpr int kNewBytes = NG == 2 ? 8 * 2 * 128 : 0;
  static constexpr int kBar = kNew + kNewBytes;
  // barriers: full[S], empty[S], s_ready[NG], p_ready[NG], pv_done[NG], s_free[NG], mma_done, new_ready
  static constexpr int kTmemSlot = kBar + (2 * kStages + 4 * kGroups + 2) * 8;
  static constexpr int kSmem = kTmemSlot + 16 + 2048;  // + slack past the last operand
  // TMEM columns. NG = 2: S_j at 64 j (64), O_j at 128 + 160 j (144), P_j (f16,
  // two per 32-bit column: the PV's A operand read from TMEM) at 432 + 32 j.
  // NG = 3: S_j at 64 j, O_j at 128 + 80 j (80), P_j at 288 + 32 j.
  static constexpr uint32_t kCols = 512;
  __host__ __device__ static constexpr uint32_t col_s(int j) { return 64u * j; }
  __host__ __device__ static constexpr uint32_t col_o(int j) { return NG == 2 ? 128u + 160u * j : 128u + 80u * j; }
  __host__ __device__ static constexpr uint32_t col_p(int j) { return NG == 2 ? 432u + 32u * j : 288u + 32u * j; }
  // Q's K bytes [32 kk, 32 kk + 32) (4 per column) at col_q(kk). NG = 2:
  // the columns between O_0 and O_1 and after P_1; NG = 3: after P_1, group j's
  // 64 bytes (its KV head's dims) as kk = 2 j, 2 j + 1
  __host__ __device__ static constexpr uint32_t col_q(int kk) {
    return NG == 3 ? 352u + 8u * kk : kk < 2 ? 272u + 8u * kk : 496u + 8u * (kk - 2);
  }
  static_assert(kK % 1024 == 0 && kV % 1024 == 0 && kVT % 1024 == 0, "operand alignment");
};
static_assert(TcCfg<2>::col_o(1) + kTcPvN <= TcCfg<2>::col_p(0) && TcCfg<2>::col_p(1) + 32 <= TcCfg<2>::col_q(2) &&
                  TcCfg<2>::col_o(0) + kTcPvN <= TcCfg<2>::col_q(0) && TcCfg<2>::col_q(1) + 8 <= TcCfg<2>::col_o(1) &&
                  TcCfg<2>::col_q(3) + 8 <= 512,
              "TMEM columns");
static_assert(TcCfg<3>::col_s(1) + 64 <= TcCfg<3>::col_o(0) && TcCfg<3>::col_o(1) + TcCfg<3>::kPvN <= TcCfg<3>::col_p(0) &&
                  TcCfg<3>::col_p(1) + 32 <= TcCfg<3>::col_q(0) && TcCfg<3>::col_q(3) + 8 <= 512,
              "TMEM columns");

// Byte offset of (row r, byte kb) in a canonical tile of 128-byte rows.
__device__ __forceinline__ uint32_t canon(int r, int kb) {
  return (uint32_t)((r >> 3) * kTcSbo + (kb >> 4) * kTcLbo + (r & 7) * 16 + (kb & 15));
}

// Row of [V | 1]^T (= column of O) that holds output dim d (d < 128): within
// each block of 16 dims, dims 4a + 2b + c sit at 8b + 2a + c, so that each
// 8-row matrix the V conversion stores with stmatrix.trans lies in one core
// matrix (conflict-free; in dim order it straddled two, 2-way conflicts). The
// epilogue reads O's columns through the same map.
__host__ __device__ constexpr int vt_pos(int d) {
  return (d & ~15) | (((d >> 1) & 1) << 3) | (((d >> 2) & 3) << 1) | (d & 1);
}

// The K and V caches as 2-D byte tensors [num_rows, 128] for TMA tile loads of
// 8 rows (one swizzle atom), used when a page holds a multiple of 8 rows.
struct TcMaps {
  CUtensorMap k, v;
};

// kTma: K and V tiles arrive by TMA, eight 8-row boxes per tile (one page id
// each), into the 128-byte-swizzle layout; tiles start at the chunk's first key
// rounded down to a multiple of 8 (those rows share the page of the first key
// and hold earlier keys of the request; they are masked). The 8-row group that
// holds the chunk's last key comes by cp.async, up to that key only: past the
// request's last key a page may hold any bytes, and a NaN there would reach
// the PV product through P = 0. Rows never loaded keep what the stage held
// before (zeros at the start, else keys of earlier tiles). Otherwise tiles
// arrive by 16-byte cp.async per row chunk (any page size).
template <bool kTma, int NG, bool FUSED>
__global__ void __launch_bounds__(TcCfg<NG>::kThreads)
    decode_tc_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ TcMaps maps) {
  using C = TcCfg<NG>;
  static_assert(!FUSED || NG == 2, "the one-kernel step runs blocks of at most 8 tokens with two softmax groups");
  constexpr int kTcStages = C::kStages, kTcGroups = C::kGroups, kTcMmaWarp = C::kMmaWarp, kTcThreads = C::kThreads;
  constexpr bool kPH = C::kPH;
  constexpr int kStep = C::kStep, kShift = C::kShift;
  constexpr int kTcProducers = C::kProducers;
  constexpr int kGroupsPW = 8 / kTcProducers;  // TMA: 8-row groups of a tile per producer warp
  constexpr int kTcK = C::kK, kTcV = C::kV, kTcVT = C::kVT, kTcX = C::kX, kTcBar = C::kBar;
  constexpr int kTcTmemSlot = C::kTmemSlot;
  constexpr uint32_t kTcCols = C::kCols;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sb = smem_u32(smem);
  auto full_bar = [&](int s) { return sb + kTcBar + 8 * s; };
  auto empty_bar = [&](int s) { return sb + kTcBar + 8 * (kTcStages + s); };
  auto s_ready = [&](int j) { return sb + kTcBar + 8 * (2 * kTcStages + j); };
  auto p_ready = [&](int j) { return sb + kTcBar + 8 * (2 * kTcStages + kTcGroups + j); };
  auto pv_done = [&](int j) { return sb + kTcBar + 8 * (2 * kTcStages + 2 * kTcGroups + j); };
  auto s_free = [&](int j) { return sb + kTcBar + 8 * (2 * kTcStages + 3 * kTcGroups + j); };
  const uint32_t mma_done = sb + kTcBar + 8 * (2 * kTcStages + 4 * kTcGroups);
  const uint32_t new_ready = mma_done + 8;  // the one-kernel step: the new K/V rows are in kNew

  // a fixed-capacity plan launches its capacity: CTAs past the live count return
  if (a.live_work && (int)blockIdx.x >= *a.live_work) return;
  const WorkItem wk = a.work[blockIdx.x];  // plan data
  if (tid == 0) {
    for (int s = 0; s < kTcStages; s++) {
      // TMA: per producer warp one arrival with its boxes' bytes and one
      // cp.async-tracked arrival per lane; cp.async: one per producer lane
      mbar_init(full_bar(s), kTma ? kTcProducers * (1 + 32) : 32 * kTcProducers);
      mbar_init(empty_bar(s), 1);                  // the MMA thread frees a stage
    }
    for (int j = 0; j < kTcGroups; j++) {
      mbar_init(s_ready(j), 1);
      mbar_init(p_ready(j), kTcRows);
      mbar_init(pv_done(j), 1);
      mbar_init(s_free(j), kTcRows);
    }
    mbar_init(mma_done, 1);
    mbar_init(new_ready, 32 * kTcProducers);
    fence_mbar_init();
  }
  if (warp == kTcMmaWarp) tmem_alloc(sb + kTcTmemSlot, kTcCols);
  if constexpr (kTma) {  // the tensor maps' descriptors: fetched now, while the lengths load
    if (warp == kTcMmaWarp + 1 && lane == 0) {
      prefetch_tensormap(&maps.k);
      prefetch_tensormap(&maps.v);
    }
  }
  const int b = wk.b;
  // The one-kernel step reads only caller inputs that the preceding kernels may
  // write: it waits for them first, unless the plan's OKC_PLAN_EARLY_GATHER
  // promise lets it load lengths, page ids and cached keys before the wait
  // (q, the new rows and every write still wait).
  if constexpr (FUSED) {
    if (!a.early) pdl_wait();
  }

  // ---- producer set-up (as decode.cu): page ids of the first tiles with the
  // plan's key range while the device lengths load. Producer warp pw owns keys
  // [pw kKeysPW, (pw + 1) kKeysPW) of every tile; lane l < kKeysPW loads the id
  // of its key l.
  constexpr int kKeysPW = kTcTileKeys / kTcProducers;
  static_assert(kKeysPW == 16 || kKeysPW == 32, "at most one page id per producer lane per tile");
  const int pw = warp - (kTcMmaWarp + 1), kbase = pw * kKeysPW;
  const int32_t* pt = a.page_table + (int64_t)b * a.max_pages;
  // (TMA: lane l < kGroupsPW of producer warp pw loads the id of the tile's
  // 8-row group pw kGroupsPW + l, tiles starting at the key range's start
  // rounded down to 8)
  auto load_ids = [&](int& dst, int tile, int jb, int je) {
    if constexpr (kTma) {
      const int j = (jb & ~7) + tile * kTcTileKeys + 8 * (pw * kGroupsPW + lane);
      dst = (lane < kGroupsPW && j < je) ? __ldg(pt + (j >> a.page_shift)) : -1;
    } else {
      const int j = jb + tile * kTcTileKeys + kbase + lane;
      dst = (lane < kKeysPW && j < je) ? __ldg(pt + (j >> a.page_shift)) : -1;
    }
  };
  int ids[kTcStages];
  if (warp > kTcMmaWarp) {
#pragma unroll
    for (int t = 0; t < kTcStages; t++) load_ids(ids[t], t, wk.j0, wk.j1);
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
  // this block's tokens i0 .. i0 + ntk - 1 of the request, at positions pbase + i
  const int ntk = max(0, min(a.S, ql - wk.i0));
  if (ntk != wk.ntok || (wk.last && wk.i0 + ntk < ql)) bad_len = true;  // q lengths differ from the plan's
  const int pbase = n - ql + wk.i0;
  const int hi = pbase + ntk;  // keys < hi
  const int lo = a.window > 0 ? max(0, pbase - a.window + 1) : 0;
  const int j0 = lo + wk.koff;
  const int j1 = min(hi, j0 + wk.cap);
  if (wk.chunk == wk.nchunks - 1 && j1 < hi) bad_len = true;  // plan does not cover the keys
  if (bad_len && tid == 0) set_error(a.err, OKC_DEVERR_LENGTHS);
  const int jt = kTma ? (j0 & ~7) : j0;  // first key of tile 0 (keys below j0 are masked)
  const int ntiles = j1 > j0 ? (j1 - jt + kTcTileKeys - 1) / kTcTileKeys : 0;
  if constexpr (kTma) {
    // V rows a tile leaves unloaded must hold finite values: zero the stages
    for (int i = tid; i < kTcStages * kTcTileKeys * kTcVPitch / 16; i += kTcThreads)
      *reinterpret_cast<uint4*>(smem + kTcV + i * 16) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();  // before the TMA loads write the same bytes
  }
  tc_fence_before();
  __syncthreads();  // barriers initialised, TMEM address in shared memory
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTcTmemSlot);

  if (warp > kTcMmaWarp) {
    // ================================================================ producer
    if (j0 != wk.j0 || j1 != wk.j1) {  // the lengths differ from the plan's: reload
#pragma unroll
      for (int t = 0; t < kTcStages; t++) load_ids(ids[t], t, j0, j1);
    }
    const int pmask = P - 1;
    const int newk = n - ql;  // keys >= newk are the step's new keys (written by the prepare kernel)
    const int rr = lane >> 3, ch = lane & 7;
    bool dep = false, bad_page = false, pos_err = false, new_ok = true;
    // The one-kernel step: the new keys of this CTA's tiles, [max(jt, newk), j1),
    // computed here (producer warp pw: KV head pw) into kNew; the keys of its
    // own range [j0, j1) also written to the cache (keys below j0 belong to the
    // previous chunk's CTA, which writes them; its tiles would read them from
    // the cache while they are written). The block is the request's only one
    // (q_len <= 8), so key newk + i is token i of the request.
    static_assert(!FUSED || kTcProducers == kNumKvHeads, "one producer warp per KV head");
    auto new_rows = [&]() {
      pdl_wait();  // qkv, positions and cache_loc: caller inputs
      const int jb = max(jt, newk), cnt = max(0, min(8, j1 - jb));
      uint16_t k8[8], v8[8];
      int64_t slot[8];
#pragma unroll
      for (int i = 0; i < 8; i++) slot[i] = (i < cnt && jb + i >= j0) ? a.cache_loc[qb + (jb + i - newk)] : -1;
      fused_new_kv8(a, (int64_t)qb + (jb - newk), cnt, pw, lane, k8, v8, pos_err);
#pragma unroll
      for (int i = 0; i < 8; i++) {
        if (i >= cnt) break;
        const int j = jb + i;
        uint8_t* dst = smem + C::kNew + (j - newk) * 256 + pw * kHeadDim + 2 * lane;
        *reinterpret_cast<uint16_t*>(dst) = k8[i];
        *reinterpret_cast<uint16_t*>(dst + 128) = v8[i];
        if (j >= j0) {
          if (slot[i] >= 0 && slot[i] < a.num_rows) {
            *reinterpret_cast<uint16_t*>(a.kc_w + slot[i] * kRowBytes + pw * kHeadDim + 2 * lane) = k8[i];
            *reinterpret_cast<uint16_t*>(a.vc_w + slot[i] * kRowBytes + pw * kHeadDim + 2 * lane) = v8[i];
          } else if (lane == 0) {
            set_error(a.err, OKC_DEVERR_CACHE_LOC);
          }
        }
      }
      mbar_arrive(new_ready);                         // this warp's rows are in kNew
      if (!mbar_wait(new_ready, 0)) new_ok = false;   // and the other warp's (bounded)
    };
    auto issue = [&](int k, int id) {
      const int s = k % kTcStages;
      const uint32_t sK = sb + kTcK + s * (kTcTileKeys * 128), sV = sb + kTcV + s * (kTcTileKeys * kTcVPitch);
      const int tj = jt + k * kTcTileKeys;
      if (!dep && min(j1, tj + kTcTileKeys) > newk) {  // this tile holds a new key
        if constexpr (FUSED)
          new_rows();
        else
          pdl_wait();  // written by the prepare kernel
        dep = true;
      }
      if constexpr (kTma) {
        // lane l < kGroupsPW: the 8 rows of group gi, keys tj + 8 gi .. +7, lie in one page
        const int gi = pw * kGroupsPW + lane;
        const int key = tj + 8 * gi;
        int nrows = 0;  // rows of group gi to load: 8, or up to the chunk's last key
        int row = 0;
        if (lane < kGroupsPW && key < j1) {
          if (id >= 0 && id < a.num_pages) {
            row = (id << a.page_shift) | (key & pmask);
            nrows = min(8, j1 - key);
          } else {
            bad_page = true;
          }
        }
        // (the one-kernel step: a group holding a new key is not loaded whole)
        const bool plain = nrows == 8 && (!FUSED || key + 8 <= newk);
        const unsigned whole = __ballot_sync(0xffffffffu, plain);
        if (lane == 0) mbar_arrive_expect_tx(full_bar(s), (uint32_t)__popc(whole) * 2u * 1024u);
        __syncwarp();
        if (plain) {
          tma_load_2d(sK + gi * 1024, &maps.k, 0, row, full_bar(s));
          tma_load_2d(sV + gi * 1024, &maps.v, 0, row, full_bar(s));
        }
        // the group cut by the chunk's end (at most one) and, in the one-kernel
        // step, the groups holding new keys: their rows by 16-byte chunks into
        // the same swizzled positions, all lanes; cached rows by cp.async, new
        // rows from kNew
        unsigned rest = __ballot_sync(0xffffffffu, nrows > 0 && !plain);
        while (rest) {
          const int lc = __ffs(rest) - 1, gc = pw * kGroupsPW + lc;
          rest &= rest - 1;
          const int crow = __shfl_sync(0xffffffffu, row, lc), cn = __shfl_sync(0xffffffffu, nrows, lc);
          const int ckey = tj + 8 * gc;
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const int cid = lane + 32 * h, r = cid >> 3, c = cid & 7;  // row r, chunk c of the group
            if (r < cn) {
              const uint32_t off = gc * 1024 + r * 128 + ((c ^ r) * 16);
              if (!FUSED || ckey + r < newk) {
                cp_async_16(sK + off, a.kc + (int64_t)(crow + r) * kRowBytes + c * 16, 16);
                cp_async_16(sV + off, a.vc + (int64_t)(crow + r) * kRowBytes + c * 16, 16);
              } else {
                const uint8_t* src = smem + C::kNew + (ckey + r - newk) * 256 + c * 16;
                *reinterpret_cast<uint4*>(smem + (sK - sb) + off) = *reinterpret_cast<const uint4*>(src);
                *reinterpret_cast<uint4*>(smem + (sV - sb) + off) = *reinterpret_cast<const uint4*>(src + 128);
              }
            }
          }
        }
        if constexpr (FUSED) {  // the stored rows: before the arrival, for the MMA (async proxy) too
          __threadfence_block();
          fence_proxy_async();
        }
        cp_async_mbar_arrive(full_bar(s));
      } else {
#pragma unroll
        for (int i = 0; i < kKeysPW / 4; i++) {
          const int rl = rr + 4 * i;
          const int r = kbase + rl;
          const int pg = __shfl_sync(0xffffffffu, id, rl);
          const int j = tj + r;
          if (FUSED && j < j1 && j >= newk) {  // a new key: from kNew (no copy, whose zero fill would race)
            const uint8_t* src = smem + C::kNew + (j - newk) * 256 + ch * 16;
            *reinterpret_cast<uint4*>(smem + (sK - sb) + canon(r, ch * 16)) = *reinterpret_cast<const uint4*>(src);
            *reinterpret_cast<uint4*>(smem + (sV - sb) + r * kTcVPitch + ch * 16) =
                *reinterpret_cast<const uint4*>(src + 128);
            continue;
          }
          int64_t row = 0;
          int bytes = 0;
          if (j < j1) {
            if (pg >= 0 && pg < a.num_pages) {
              row = ((int64_t)pg << a.page_shift) | (j & pmask);
              bytes = 16;
            } else {
              bad_page = true;
            }
          }
          cp_async_16(sK + canon(r, ch * 16), a.kc + row * kRowBytes + ch * 16, bytes);
          cp_async_16(sV + r * kTcVPitch + ch * 16, a.vc + row * kRowBytes + ch * 16, bytes);
        }
        if constexpr (FUSED) {
          __threadfence_block();
          fence_proxy_async();
        }
        cp_async_mbar_arrive(full_bar(s));
      }
    };
#pragma unroll
    for (int t = 0; t < kTcStages; t++) {
      if (t < ntiles) issue(t, ids[t]);
      load_ids(ids[t], t + kTcStages, j0, j1);
    }
    // the one-kernel step: the new rows of a later tile now, while the first
    // tiles are consumed, not when that tile is issued
    if constexpr (FUSED) {
      if (!dep && ntiles > 0 && j1 > newk) {
        new_rows();
        dep = true;
      }
    }
    bool ok = true;
    int issued = min(ntiles, kTcStages);  // tiles whose copies were issued
    for (int k0 = kTcStages; k0 < ntiles && ok; k0 += kTcStages) {
#pragma unroll
      for (int u = 0; u < kTcStages; u++) {
        const int k = k0 + u;
        if (k >= ntiles) break;
        if (!mbar_wait(empty_bar(u), ((k / kTcStages) & 1) ^ 1)) { ok = false; break; }
        issue(k, ids[u]);
        issued = k + 1;
        load_ids(ids[u], k + kTcStages, j0, j1);
      }
    }
    if (bad_page && (kTma || ch == 0)) set_error(a.err, OKC_DEVERR_PAGE);
    if (pos_err && lane == 0) set_error(a.err, OKC_DEVERR_POSITION);
    if (!new_ok) ok = false;
    if constexpr (kTma) {
      // the CTA's shared memory must outlive the copies in flight: wait (bounded,
      // also after a timeout) until the last issued tile of every stage landed
      for (int k = max(0, issued - kTcStages); k < issued; k++)
        if (!mbar_wait(full_bar(k % kTcStages), (k / kTcStages) & 1)) ok = false;
    }
    if (!ok && lane == 0) set_error(a.err, OKC_DEVERR_TIMEOUT);
    cp_async_wait_all();
    return;
  }

  if (warp == kTcMmaWarp) {
    // ================================================================ MMA issue
    named_bar_sync(1, (kTcMmaWarp + 1) * 32);  // Q is in TMEM or shared memory
    tc_fence_after();
    if (kPH && lane == 0) {
      // form 3, every tile k for both groups: S_j = Q_j K_k^T over KV head j's
      // 64 K bytes, O_j (+)= P_j [V_k,j | 1]. Each is issued once its inputs
      // are ready (polled, a ready PV first, as below); a stage is freed once
      // both groups have consumed its tile (P written, their V dims converted).
      constexpr uint32_t id_qk = umma_idesc(0, kTcRows, kTcTileKeys);  // E4M3 x E4M3 -> f32, 128 x 64
      constexpr uint32_t id_pv = umma_idesc(0, kTcRows, C::kPvN);      // f16 x f16 -> f32, 128 x 80
      auto qk = [&](int k, int j) {
        const uint32_t kt = sb + kTcK + (k % kTcStages) * (kTcTileKeys * 128);
#pragma unroll
        for (int kk = 0; kk < 2; kk++) {  // head j's 64 bytes of K: 32 per instruction
          const int kb = 2 * j + kk;
          const uint64_t kdesc =
              kTma ? umma_desc_sw128(kt + kb * 32, kTcSbo) : umma_desc(kt + kb * 2 * kTcLbo, kTcLbo, kTcSbo);
          umma_f8_ta(tmem + C::col_s(j), tmem + C::col_q(kb), kdesc, id_qk, kk > 0);
        }
        umma_commit(s_ready(j));
      };
      auto pv = [&](int k, int j) {
        const uint32_t va = sb + kTcVT + j * C::kVTBytes;
#pragma unroll
        for (int kk = 0; kk < 4; kk++)  // 64 keys: 16 per instruction
          umma_f16_ta(tmem + C::col_o(j), tmem + C::col_p(j) + kk * 8,
                      umma_desc(va + kk * 2 * kTcLbo, kTcLbo, kTcSbo), id_pv, (k > 0 || kk > 0) ? 1u : 0u);
        umma_commit(pv_done(j));
      };
      bool ok = true;
      int nq[2] = {0, 0}, np[2] = {0, 0}, freed = 0;  // next QK / PV per group, stages freed
      uint64_t t_idle = 0;
      while (np[0] < ntiles || np[1] < ntiles) {
        bool did = false;
#pragma unroll
        for (int j = 0; j < 2; j++) {
          if (np[j] < nq[j] && mbar_test_wait(p_ready(j), np[j] & 1)) {
            fence_proxy_async();  // V^T_j, written through the generic proxy
            tc_fence_after();
            pv(np[j], j);
            np[j]++;
            did = true;
          }
        }
        for (; freed < min(np[0], np[1]); freed++) mbar_arrive(empty_bar(freed % kTcStages));
#pragma unroll
        for (int j = 0; j < 2; j++) {
          const int k = nq[j];
          if (k < ntiles && (k == 0 || mbar_test_wait(s_free(j), (k - 1) & 1)) &&
              mbar_test_wait(full_bar(k % kTcStages), (k / kTcStages) & 1)) {
            fence_proxy_async();  // the gathered tile, written through the generic proxy
            tc_fence_after();
            qk(k, j);
            nq[j]++;
            did = true;
          }
        }
        if (did) {
          t_idle = 0;
        } else if (t_idle == 0) {
          t_idle = global_ns();
        } else if (global_ns() - t_idle > kWaitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) set_error(a.err, OKC_DEVERR_TIMEOUT);
      umma_commit(mma_done);  // arrives once every MMA issued above has completed
      if (!mbar_wait(mma_done, 0)) set_error(a.err, OKC_DEVERR_TIMEOUT);
    }
    if (!kPH && lane == 0) {
      constexpr uint32_t id_qk = umma_idesc(0, kTcRows, kTcTileKeys);  // E4M3 x E4M3 -> f32, 128 x 64
      constexpr uint32_t id_pv = umma_idesc(0, kTcRows, kTcPvN);       // f16 x f16 -> f32, 128 x 144
      // S_j = Q K_k^T for tile k (group j = k & 1)
      auto qk = [&](int k) -> bool {
        const int s = k % kTcStages, j = k & (NG - 1);
        if (!mbar_wait(full_bar(s), (k / kTcStages) & 1)) return false;
        fence_proxy_async();  // the gathered tile, written through the generic proxy
        tc_fence_after();
        const uint32_t kt = sb + kTcK + s * (kTcTileKeys * 128);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {  // 128 bytes of K: 32 per instruction (two core matrices)
          const uint64_t kdesc =
              kTma ? umma_desc_sw128(kt + kk * 32, kTcSbo) : umma_desc(kt + kk * 2 * kTcLbo, kTcLbo, kTcSbo);
          umma_f8_ta(tmem + C::col_s(j), tmem + C::col_q(kk), kdesc, id_qk, kk > 0);
        }
        umma_commit(s_ready(j));
        return true;
      };
      // O_j (+)= P_j V_k once group j has written P and V^T of tile k
      auto pv = [&](int k) -> bool {
        const int j = k & (NG - 1);
        if (!mbar_wait(p_ready(j), (k >> (NG - 1)) & 1)) return false;
        fence_proxy_async();
        tc_fence_after();
        mbar_arrive(empty_bar(k % kTcStages));  // K read (S_k consumed), V converted: the stage is free
        const uint32_t va = sb + kTcVT + j * C::kVTBytes;
#pragma unroll
        for (int kk = 0; kk < 4; kk++)  // 64 keys: 16 per instruction
          umma_f16_ta(tmem + C::col_o(j), tmem + C::col_p(j) + kk * 8,
                      umma_desc(va + kk * 2 * kTcLbo, kTcLbo, kTcSbo), id_pv, (k >= kTcGroups || kk > 0) ? 1u : 0u);
        umma_commit(pv_done(j));
        return true;
      };
      // Issue order follows readiness: PV of tile t (P_j written) and QK of
      // tile t (S_j free: group j has read S of tile t-2; tile t landed) are
      // polled without blocking and issued as soon as their inputs are ready,
      // a ready PV first (its group waits on it to write the next P; the QKs
      // run ahead), so a late tile never holds back a PV. Bounded: gives up
      // after kWaitNs without progress.
      bool ok = true;
      int nq = 0, np = 0;  // next QK / PV to issue
      uint64_t t_idle = 0;
      while (np < ntiles) {
        bool did = false;
        if (np < nq && mbar_test_wait(p_ready(np & (NG - 1)), (np >> (NG - 1)) & 1)) {
          ok = pv(np);  // its wait succeeds at once
          np++;
          did = true;
        }
        if (ok && nq < ntiles && (nq < NG || mbar_test_wait(s_free(nq & (NG - 1)), ((nq - NG) >> (NG - 1)) & 1)) &&
            mbar_test_wait(full_bar(nq % kTcStages), (nq / kTcStages) & 1)) {
          tc_fence_after();
          ok = qk(nq);  // its waits succeed at once
          nq++;
          did = true;
        }
        if (!ok) break;
        if (did) {
          t_idle = 0;
        } else if (t_idle == 0) {
          t_idle = global_ns();
        } else if (global_ns() - t_idle > kWaitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) set_error(a.err, OKC_DEVERR_TIMEOUT);
      umma_commit(mma_done);  // arrives once every MMA issued above has completed
      if (!mbar_wait(mma_done, 0)) set_error(a.err, OKC_DEVERR_TIMEOUT);
    }
    __syncwarp();
    tc_fence_before();
    named_bar_sync(2, (kTcMmaWarp + 1) * 32);  // the softmax warps are done with TMEM
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
    return;
  }

  // ================================================================== softmax
  const int jw = warp >> 2;  // this thread's group: tiles jw, jw + 2, ...
  const int r = tid & (kTcRows - 1);  // q row
  // KV head, token and head of row r (form 3: the group's KV head, 16 tokens)
  const int g = kPH ? jw : r >> 6, ti = kPH ? r >> 3 : (r >> 3) & 7, hh = r & 7;
  const int head = g * kGroup + hh;
  const bool live = ti < ntk;
  pdl_wait();  // q_fp8 is the prepare kernel's output (the one-kernel step: qkv, a caller input)
  pdl_launch_dependents();
  bool q_pos_err = false;
  {
    // Q row r: the 64 E4M3 dims of (token ti, head). Form 2: at K bytes
    // [64g, 64g+64), zeros elsewhere; group jw writes K bytes [64 jw, 64 jw +
    // 64), 16 TMEM columns from col_q(2 jw). Form 3: the group's 64 K bytes.
    const uint4* src = reinterpret_cast<const uint4*>(
        a.q8 + ((int64_t)(qb + wk.i0 + (live ? ti : 0)) * kNumQHeads + head) * kHeadDim);
    {
      float qv[16];
      if constexpr (FUSED) {  // the row from qkv (steps 1-3 of the block), by the group of its KV head
        uint32_t qw[16];
        fused_q_row(a, (int64_t)qb + wk.i0 + (live ? ti : 0), head, live && g == jw, qw, q_pos_err);
#pragma unroll
        for (int i = 0; i < 16; i++) qv[i] = __uint_as_float(qw[i]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; c++) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (live && g == jw) v = src[c];
          qv[4 * c] = __uint_as_float(v.x);
          qv[4 * c + 1] = __uint_as_float(v.y);
          qv[4 * c + 2] = __uint_as_float(v.z);
          qv[4 * c + 3] = __uint_as_float(v.w);
        }
      }
      tmem_st16(tmem + ((uint32_t)((warp & 3) * 32) << 16) + C::col_q(2 * jw), qv);
    }
  }
  {
    // the last 16 rows of each group's [V | 1]^T (from row kPvN - 16, the
    // first after the dims): that row ones, the rest zeros (never rewritten;
    // the V conversion writes the dims' rows)
    constexpr int kOnes = C::kPvN - 16;
    const int gj = tid >> 7, rr2 = kOnes + ((tid >> 3) & 15), c = tid & 7;
    const uint32_t one2 = rr2 == kOnes ? 0x3C003C00u : 0u;  // f16 1.0 pairs
    *reinterpret_cast<uint4*>(smem + kTcVT + gj * C::kVTBytes + canon(rr2, c * 16)) = make_uint4(one2, one2, one2, one2);
  }
  if (__any_sync(0xffffffffu, q_pos_err) && lane == 0) set_error(a.err, OKC_DEVERR_POSITION);
  fence_proxy_async();  // shared-memory operands, for the MMAs
  tc_fence_before();    // Q's TMEM stores, before the MMA thread reads them
  named_bar_sync(1, (kTcMmaWarp + 1) * 32);

  const float scale_log2 = a.scaled ? a.scale_log2 * __ldg(a.k_scale) : a.scale_log2;
  const int pos = pbase + ti;  // this row's query position
  const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t tS = t_lane + C::col_s(jw);              // this row's S
  const uint32_t tO = t_lane + C::col_o(jw) + (kPH ? 0 : 64 * g);  // this row's O dims
  const uint32_t tL = t_lane + C::col_o(jw) + C::kPvN - 16;       // this row's P sum
  const uint32_t tP = t_lane + C::col_p(jw);               // this row's P (f16 pairs)
  const uint32_t sVT = kTcVT + jw * C::kVTBytes;
  float m = -INFINITY;  // reference max (log2 units)
  bool ok = true;
  int last = -1;  // this group's last tile
  // this row's valid keys [row_lo, row_hi): the chunk's range, the window and
  // causality (empty for a dead row)
  const int row_lo = live ? max(j0, a.window > 0 ? pos - a.window + 1 : 0) : 0;
  const int row_hi = live ? min(j1, pos + 1) : 0;
  // The V conversion's shared-memory addresses, the same for every tile but
  // the stage's base: warp w of the group converts key groups 2w, 2w+1 (8 keys
  // each) x 8 groups of 16 dims (form 3: the 4 groups of its KV head's dims),
  // kIts ldmatrix.x4 loads and 2 kIts stmatrix.trans stores.
  constexpr int kIts = kPH ? 2 : 4;
  uint32_t v_ld[kIts], v_st[kIts][2];
#pragma unroll
  for (int it = 0; it < kIts; it++) {
    const int a8 = 2 * (warp & 3) + (kPH ? it : it >> 1);  // key group
    const int cbase = kPH ? 4 * jw : (it & 1) * 4;          // first 16-dim group of this x4
    // matrix mi = lane >> 3: keys a8*8 + (lane & 7), bytes 16 (cbase + mi) .. +15
    // (TMA: 8-row groups 1024 bytes apart, chunks XORed with the row mod 8)
    v_ld[it] = kTma ? a8 * 1024 + (lane & 7) * 128 + (((cbase + (lane >> 3)) ^ (lane & 7)) * 16)
                    : (a8 * 8 + (lane & 7)) * kTcVPitch + (cbase + (lane >> 3)) * 16;
    // stored matrix jm (lanes 8jm..8jm+7 give its rows): {lo, hi} of block 2*half + (jm >> 1);
    // its row cc holds dim 16 c16 + 4 (cc >> 1) + 2 (jm & 1) + (cc & 1) for the 8 keys,
    // stored at row vt_pos(dim) = 16 c16 + 8 (jm & 1) + cc
    const int jm = lane >> 3, cc = lane & 7;
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int c16 = cbase + half * 2 + (jm >> 1) - (kPH ? 4 * jw : 0);  // (of the group's dims)
      v_st[it][half] = sb + sVT + canon(16 * c16 + 8 * (jm & 1) + cc, a8 * 16);
    }
  }
  int s = kPH ? 0 : jw, sph = 0;  // tile k's stage and the phase bit of its fill
  for (int k = kPH ? 0 : jw; k < ntiles; k += kStep) {
    const bool w = mbar_wait(s_ready(jw), (k >> kShift) & 1) && mbar_wait(full_bar(s), sph);
    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
    tc_fence_after();
    const int tile_j = jt + k * kTcTileKeys;
    float s0[32], s1[32];
    tmem_ld32(tS, s0);
    tmem_ld32(tS + 32, s1);
    tc_fence_before();
    mbar_arrive(s_free(jw));  // S of this tile is in registers: the next QK may overwrite it
    // ---- mask: this row's valid keys of the tile are [klo, khi) (window,
    // causal, chunk end; none for a dead row); row max on the raw scores
    const int klo = max(0, row_lo - tile_j), khi = min(kTcTileKeys, row_hi - tile_j);
    const uint32_t kn = khi > klo ? (uint32_t)(khi - klo) : 0u;
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (__all_sync(0xffffffffu, klo == 0 && khi == kTcTileKeys)) {  // every key valid for the warp's rows
#pragma unroll
      for (int c = 0; c < 32; c++) mx4[c & 3] = fmax3(mx4[c & 3], s0[c], s1[c]);
    } else {
#pragma unroll
      for (int c = 0; c < 32; c++) {
        s0[c] = (uint32_t)(c - klo) < kn ? s0[c] : -INFINITY;
        s1[c] = (uint32_t)(32 + c - klo) < kn ? s1[c] : -INFINITY;
        mx4[c & 3] = fmax3(mx4[c & 3], s0[c], s1[c]);
      }
    }
    // in log2 units (the scale is positive)
    const float mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]) * scale_log2;
    // ---- reference max: moves when the row max passes it by more than 2^8
    const float m_new = (m == -INFINITY || mx > m + kTcRescale) ? fmaxf(m, mx) : m;
    const float alpha = m_new == m ? 1.f : (m == -INFINITY ? 0.f : fast_exp2(m - m_new));
    m = m_new;
    const float m_use = m == -INFINITY ? 0.f : m;
    // ---- P row (f16), two keys per 32-bit word: p = 2^(s * scale - m) in f32,
    // rounded to f16; computed before the wait below, which it does not need
    uint32_t pw[32];
#pragma unroll
    for (int c = 0; c < 32; c++) {
      const float x0 = c < 16 ? s0[2 * c] : s1[2 * c - 32], x1 = c < 16 ? s0[2 * c + 1] : s1[2 * c - 31];
      float e0, e1;
      ffma2(x0, x1, scale_log2, -m_use, e0, e1);  // (two keys' s * scale - m per instruction)
      pw[c] = pack_half2(fast_exp2(e0), fast_exp2(e1));
    }
    // ---- P, V^T and O of this group are free once its previous PV completed
    if (k >= kStep) {
      const bool w2 = mbar_wait(pv_done(jw), ((k - kStep) >> kShift) & 1);
      if (!__all_sync(0xffffffffu, w2)) { ok = false; break; }
      tc_fence_after();
    }
    if (k >= kStep && __any_sync(0xffffffffu, alpha != 1.f)) {  // rescale O rows (and sums) in TMEM
      float ov[16];
#pragma unroll
      for (int h4 = 0; h4 < 4; h4++) {  // (the stores complete at the sum's store below)
        tmem_ld16(tO + 16 * h4, ov);
#pragma unroll
        for (int d = 0; d < 16; d += 2) fmul2(ov[d], ov[d + 1], alpha, ov[d], ov[d + 1]);
        tmem_st16_async(tO + 16 * h4, ov);
      }
      tmem_st1(tL, tmem_ld1(tL) * alpha);
    }
    // ---- P into this group's TMEM P columns (the PV's A operand)
    tmem_st32u(tP, pw);
    // ---- V tile E4M3 -> f16, transposed into this group's canonical B tile
    // (dims x keys; the addresses above)
    {
      const uint32_t vs = sb + kTcV + s * (kTcTileKeys * kTcVPitch);
#pragma unroll
      for (int it = 0; it < kIts; it++) {
        uint32_t rg[4];
        ldsm_x4(rg, vs + v_ld[it]);
        // rg[mi]: key a8*8 + lane/4, dims 16 (cbase+mi) + 4 (lane%4) + {0,1,2,3}
        uint32_t lo4[4], hi4[4];
#pragma unroll
        for (int mi = 0; mi < 4; mi++) {
          e4m3x4_to_f16x2x2(rg[mi], lo4[mi], hi4[mi]);  // dims +0, +1 and +2, +3
        }
#pragma unroll
        for (int half = 0; half < 2; half++)
          stsm_x4_trans(v_st[it][half], lo4[half * 2], hi4[half * 2], lo4[half * 2 + 1], hi4[half * 2 + 1]);
      }
    }
    fence_proxy_async();  // V^T, written through the generic proxy, for the MMA
    tc_fence_before();
    mbar_arrive(p_ready(jw));
    last = k;
    s += kStep;  // the next tile's stage
    if (s >= kTcStages) {
      s -= kTcStages;
      sph ^= 1;
    }
  }
  // this group's O is complete once its last PV has
  if (ok && last >= 0) {
    const bool w3 = mbar_wait(pv_done(jw), (last >> kShift) & 1);
    if (!__all_sync(0xffffffffu, w3)) ok = false;
    tc_fence_after();
  }
  if (!ok && lane == 0) set_error(a.err, OKC_DEVERR_TIMEOUT);

  // ---- merge the two groups and write the split: the groups swap their
  // reference maxima through shared memory, then group j writes dims
  // [32 j, 32 j + 32) of each row's 64 (group 0 also the row's LSE)
  float* xml = reinterpret_cast<float*>(smem + kTcX);
  xml[jw * kTcRows + r] = m;
  tc_fence_before();
  named_bar_sync(3, kTcGroups * kTcRows);
  tc_fence_after();
  {
    // groups that ran a PV for this row (form 3: this group alone holds it)
    const bool has0 = ok && ntiles >= 1, has1 = NG == 2 && ok && ntiles >= 2;
    const float m0 = kPH ? m : xml[r], m1 = NG == 2 ? xml[kTcRows + r] : -INFINITY;
    const float l = has0 ? tmem_ld1(kPH ? tL : t_lane + C::col_o(0) + 128) : 0.f;
    const float l1 = has1 ? tmem_ld1(t_lane + C::col_o(1) + 128) : 0.f;
    const float M = fmaxf(m0, m1);
    const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M), f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
    const float L = l * f0 + l1 * f1;
    const float vscale = a.scaled ? *a.v_scale : 1.0f;
    const float inv = L > 0.f ? vscale / L : 0.f;
    const int rows = a.S * kNumQHeads;  // rows of an output slot: the block's tokens x heads
    const int row = ti * kNumQHeads + head;
    // (the slot is read from the work item again here: kept live through the
    // tile loop it cost the kernel about 30 registers)
    const int64_t slot = (int64_t)__ldg(&a.work[blockIdx.x].wbase) + __ldg(&a.work[blockIdx.x].chunk);
    float* opart = a.o_part + slot * rows * kHeadDim;
    // The split's partials leave through shared memory: each warp stages its
    // 32 rows' half rows (32 floats at a 144-byte pitch: conflict-free float4
    // writes and reads) in the K stages, idle now (every tile landed and was
    // consumed, every MMA completed), then stores 4 half rows (four whole
    // 128-byte lines) per instruction instead of one 16-byte piece of 32 rows.
    constexpr int kStgPitch = 36;  // floats
    static_assert(4 * kTcGroups * 32 * kStgPitch * 4 <= kTcStages * kTcTileKeys * 128, "staging fits the K stages");
    float* stg = reinterpret_cast<float*>(smem + kTcK) + warp * 32 * kStgPitch;
#pragma unroll
    for (int hh2 = 0; hh2 < (NG == 2 ? 1 : 2); hh2++) {  // this group's halves of the row
      const int h2 = NG == 2 ? jw : hh2;
      float o0[32], o1[32];
      if (has0) tmem_ld32(t_lane + (kPH ? C::col_o(jw) : C::col_o(0) + 64 * g) + 32 * h2, o0);
      if (has1) tmem_ld32(t_lane + C::col_o(1) + 64 * g + 32 * h2, o1);
#pragma unroll
      for (int d = 0; d < 32; d += 4) {  // dims 32 h2 + d + e, O columns through vt_pos
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; e++)
          v[e] = ((has0 ? o0[vt_pos(d + e)] * f0 : 0.f) + (has1 ? o1[vt_pos(d + e)] * f1 : 0.f)) * inv;
        *reinterpret_cast<float4*>(stg + lane * kStgPitch + d) = make_float4(v[0], v[1], v[2], v[3]);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const int lr = 4 * i + (lane >> 3);             // the warp's row lr: q row rq
        const int rq = (warp & 3) * 32 + lr;
        const int ti2 = kPH ? rq >> 3 : (rq >> 3) & 7;
        if (ti2 < ntk) {
          const int row2 = ti2 * kNumQHeads + (kPH ? jw : rq >> 6) * kGroup + (rq & 7);
          *reinterpret_cast<float4*>(opart + row2 * kHeadDim + 32 * h2 + 4 * (lane & 7)) =
              *reinterpret_cast<const float4*>(stg + lr * kStgPitch + 4 * (lane & 7));
        }
      }
      __syncwarp();  // the staging is rewritten by the next half
    }
    if (live && (kPH || jw == 0)) a.lse_part[slot * rows + row] = L > 0.f ? M + log2f(L) : -INFINITY;
  }
  tc_fence_before();
  named_bar_sync(2, (kTcMmaWarp + 1) * 32);  // TMEM reads done: the MMA warp may free it
  if constexpr (FUSED) {
    // The block's last CTA merges every split and applies the norm-gate: once
    // both groups' partials are written (barrier), one thread takes a ticket
    // with an acquire-release atomic (publishing them); the CTA that draws the
    // last ticket reads all partials (L2 loads) and resets the counter for the
    // next launch. Nothing waits on another CTA.
    volatile int& s_last = *reinterpret_cast<volatile int*>(smem + kTcX);  // (the maxima are read)
    named_bar_sync(3, kTcGroups * kTcRows);
    if (tid == 0) {
      int prev;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(prev) : "l"(a.tickets + b) : "memory");
      s_last = prev == wk.nchunks - 1;
    }
    named_bar_sync(3, kTcGroups * kTcRows);
    if (s_last) {
      const int rows = a.S * kNumQHeads;
      const int64_t base = (int64_t)wk.wbase * rows;
      for (int rowi = tid >> 3; rowi < ntk * kNumQHeads; rowi += kTcGroups * kTcRows / 8) {  // 8 lanes per row
        const int tok = rowi / kNumQHeads, h = rowi % kNumQHeads;
        const int64_t t = (int64_t)qb + wk.i0 + tok;
        const int c0 = (tid & 7) * 8;
        float gg[8], ww[8];
        load_gate_weight(a.qkv, a.weight, (int)t, h, c0, gg, ww);
        merge_normgate<4>(a.lse_part + base + rowi, rows, a.o_part + (base + rowi) * kHeadDim + c0,
                          (int64_t)rows * kHeadDim, wk.nchunks, gg, ww, a.eps,
                          a.out + t * (kNumQHeads * kHeadDim) + h * kHeadDim + c0);
      }
      if (tid == 0) a.tickets[b] = 0;
    }
  }
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null when unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<EncodeTiledFn>(nullptr);
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A cache viewed as [rows, 128] bytes, loaded as boxes of 8 rows with 128-byte
// swizzle.
bool encode_cache_map(CUtensorMap* m, const uint8_t* base, int64_t rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn || rows < 8) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kRowBytes};
  const cuuint32_t box[2] = {(cuuint32_t)kRowBytes, 8};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NG, bool FUSED>
cudaError_t launch_tc(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  using C = TcCfg<NG>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_work);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  // pages of 8 or more rows: TMA boxes of 8 rows never cross a page
  TcMaps maps;
  std::memset(&maps, 0, sizeof maps);
  const int64_t rows = (int64_t)a.num_pages << a.page_shift;
  if (a.page_shift >= 3 && encode_cache_map(&maps.k, a.kc, rows) && encode_cache_map(&maps.v, a.vc, rows))
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<true, NG, FUSED>, a, maps);
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<false, NG, FUSED>, a, maps);
}

cudaError_t launch_decode_tc(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  if (num_work == 0) return cudaSuccess;
  if (a.S < 1 || a.S > (a.tc_groups == 3 ? 16 : 8)) return cudaErrorInvalidValue;
  if (a.tc_groups == 2) return launch_tc<2, false>(a, num_work, pdl, s);
  if (a.tc_groups == 3) return launch_tc<3, false>(a, num_work, pdl, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_step_fused_tc(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  if (num_work == 0) return cudaSuccess;
  if (a.L < 2 || a.L > 8 || a.S != a.L || a.tc_groups != 2) return cudaErrorInvalidValue;
  return launch_tc<2, true>(a, num_work, pdl, s);
}

template <int NG>
int tc_ctas_per_sm() {
  using C = TcCfg<NG>;
  int lowest = 0;
  // (every variant's shared-memory limit is raised here, the one-kernel step's too)
  for (int v = 0; v < 4; v++) {
    if (v >= 2 && NG != 2) break;
    auto kern = v == 0 ? decode_tc_kernel<false, NG, false> : v == 1 ? decode_tc_kernel<true, NG, false>
              : v == 2 ? decode_tc_kernel<false, NG, NG == 2> : decode_tc_kernel<true, NG, NG == 2>;
    int nb = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, C::kThreads, C::kSmem) != cudaSuccess)
      return 0;
    lowest = v ? std::min(lowest, nb) : nb;
  }
  return lowest;
}

int decode_tc_ctas_per_sm(int tc_groups) {
  return tc_groups == 2 ? tc_ctas_per_sm<2>() : tc_groups == 3 ? tc_ctas_per_sm<3>() : 0;
}

}  // namespace okc
