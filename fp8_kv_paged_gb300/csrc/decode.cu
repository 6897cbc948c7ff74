// decode.cu — step 4 of the block: split-KV paged causal GQA attention over the
// E4M3 cache (the flash_attn_with_kvcache call of "012-attention-local-splits.py":
// paged, causal, window_size (window-1, 0), softmax_scale sm_scale*qk_scale_factor,
// k/v descale on the scaled path).
//
// Work item = (request b, chunk of its visible keys), covering BOTH KV heads and
// all L query tokens, so that at page_size 1 every key is one contiguous 128-byte
// cache row per tensor (K and V), fetched as 8 x 16-byte cp.async per row.
//
// Pipeline: a ring of kStages tiles of 64 keys (8 KB of K + 8 KB of V each) in
// shared memory, filled with cp.async (zero-fill for masked or invalid rows);
// the 16-byte chunks of each row are XOR-swizzled by the row index so that the
// ldmatrix reads below are bank-conflict free. Page-table entries for tile
// k+kStages are loaded into registers one iteration before their copies issue.
//
// Math per warp (warp = one KV head g x a set of query tokens x a share of keys):
//  QK^T  "swap-AB": D[16 keys x 8 heads] = K_tile[16 x 64] * q^T, two
//        mma.m16n8k32 E4M3 x E4M3 -> f32 (K fragment by ldmatrix.x4 straight
//        from the E4M3 tile, q fragment from registers). Products of E4M3 values
//        are exact; the sum is the tensor core's f32 accumulation.
//  softmax: online (m, l) per query row in f32, base-2 with the scale folded in;
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
#include "okc_common.cuh"
#include "okc_internal.h"

namespace okc {

namespace {

constexpr int kTileKeys = 64;
constexpr int kTileBytes = kTileKeys * kRowBytes;  // 8 KB per tensor
constexpr int kStages = 4;
constexpr int kStageBytes = 2 * kTileBytes;        // K + V
constexpr int kSmemBytes = kStages * kStageBytes;  // 64 KB

// Shared-memory offset of 16-byte chunk `ch` (0..7) of tile row `r`.
__device__ __forceinline__ uint32_t swz(int r, int ch) {
  return (uint32_t)(r * kRowBytes + ((ch ^ (r & 7)) << 4));
}

template <int KS, int NTW, int NWARPS>
struct DecodeCfg {
  static constexpr int kThreads = NWARPS * 32;
  static constexpr int kRowsPerPass = kThreads / 8;               // 8 threads per 128-byte row
  static constexpr int kRowsPerThread = kTileKeys / kRowsPerPass;  // rows each thread copies per tile
  static constexpr int kMTiles = 4 / KS;                           // 16-key m-tiles per warp per tile
  static_assert(kRowsPerThread >= 1 && kTileKeys % kRowsPerPass == 0, "bad thread count");
};

template <int KS, int NTW, int NWARPS>
__global__ void __launch_bounds__(NWARPS * 32) decode_kernel(DecodeArgs a) {
  using C = DecodeCfg<KS, NTW, NWARPS>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = warp & 1;                          // KV head of this warp
  const int sub = warp >> 1;
  const int ks = (KS == 2) ? sub : 0;              // key share (L = 1 mode)
  const int tok0 = (KS == 2) ? 0 : sub * NTW;      // first query token of this warp
  const int gq = lane >> 2, tq = lane & 3;         // mma fragment coordinates

  // ---- the work item and the request's lengths (caller inputs: read before the
  //      dependency wait so that this overlaps the prepare kernel's tail)
  const WorkItem wk = a.work[blockIdx.x];
  const int b = wk.b;
  const ReqInfo rq = a.req[b];
  int n = a.cache_seqlens[b];
  const int qb = a.cu_seqlens_q[b];
  int ql = a.cu_seqlens_q[b + 1] - qb;
  const int P = 1 << a.page_shift;
  bool bad_len = ql < 0 || ql > a.L || qb < 0 || qb + ql > a.T || n < ql ||
                 (a.seq_lens && a.seq_lens[b] != n - ql) ||
                 (int64_t)n > (int64_t)a.max_pages * P;
  if (bad_len) {  // keep every access in range; the result of this request is void
    ql = max(0, min(ql, a.L));
    if (qb < 0 || qb + ql > a.T) ql = 0;
    n = max(ql, min(n, a.max_pages * P));
  }
  const int lo = a.window > 0 ? max(0, n - ql - a.window + 1) : 0;  // first key any query sees
  const int j0 = lo + wk.chunk * rq.chunk_keys;
  const int j1 = min(n, j0 + rq.chunk_keys);
  if (wk.chunk == rq.nchunks - 1 && j1 < n) bad_len = true;  // plan does not cover the keys
  if (bad_len && tid == 0) set_error(a.err, OKC_DEVERR_LENGTHS);
  const int ntiles = j1 > j0 ? (j1 - j0 + kTileKeys - 1) / kTileKeys : 0;
  const int32_t* pt = a.page_table + (int64_t)b * a.max_pages;
  const int pmask = P - 1;
  // logit scale in base 2; on the scaled path every key is its E4M3 value times k_scale
  const float scale_log2 = a.scaled ? a.scale_log2 * __ldg(a.k_scale) : a.scale_log2;

  // Page ids of this thread's rows of tile `tile` (raw; checked when used).
  auto load_pages = [&](int (&pf)[C::kRowsPerThread], int tile) {
#pragma unroll
    for (int i = 0; i < C::kRowsPerThread; i++) {
      const int r = (tid >> 3) + i * C::kRowsPerPass;
      const int j = j0 + tile * kTileKeys + r;
      pf[i] = (tile < ntiles && j < j1) ? __ldg(pt + (j >> a.page_shift)) : -1;
    }
  };
  auto issue_tile = [&](const int (&pf)[C::kRowsPerThread], int tile) {
    const uint32_t kbase = smem_u32(smem) + (uint32_t)((tile % kStages) * kStageBytes);
    const int ch = tid & 7;
#pragma unroll
    for (int i = 0; i < C::kRowsPerThread; i++) {
      const int r = (tid >> 3) + i * C::kRowsPerPass;
      const int j = j0 + tile * kTileKeys + r;
      int64_t row = 0;
      int bytes = 0;
      if (j < j1) {
        if (pf[i] >= 0 && pf[i] < a.num_pages) {
          row = ((int64_t)pf[i] << a.page_shift) | (j & pmask);
          bytes = 16;
        } else if (ch == 0) {
          set_error(a.err, OKC_DEVERR_PAGE);
        }
      }
      cp_async_16(kbase + swz(r, ch), a.kc + row * kRowBytes + ch * 16, bytes);
      cp_async_16(kbase + kTileBytes + swz(r, ch), a.vc + row * kRowBytes + ch * 16, bytes);
    }
  };

  // page ids of the first kStages tiles, all in flight together
  int pg[kStages][C::kRowsPerThread];
#pragma unroll
  for (int st = 0; st < kStages; st++) load_pages(pg[st], st);

  // ---- everything below may read what the prepare kernel wrote
  pdl_wait();
  pdl_launch_dependents();

  // q fragments (B operand of QK^T): column = head gq of KV head g, token tok0+n
  uint32_t qf[NTW][2][2];
#pragma unroll
  for (int nt = 0; nt < NTW; nt++) {
    const int tok = tok0 + nt;
    const uint8_t* qrow = a.q8 + ((int64_t)(qb + tok) * kNumQHeads + g * kGroup + gq) * kHeadDim;
#pragma unroll
    for (int kk = 0; kk < 2; kk++) {
      qf[nt][kk][0] = tok < ql ? *reinterpret_cast<const uint32_t*>(qrow + kk * 32 + tq * 4) : 0u;
      qf[nt][kk][1] = tok < ql ? *reinterpret_cast<const uint32_t*>(qrow + kk * 32 + 16 + tq * 4) : 0u;
    }
  }

  // prologue: tiles 0 .. kStages-2 in flight
#pragma unroll
  for (int st = 0; st < kStages - 1; st++) {
    if (st < ntiles) issue_tile(pg[st], st);
    cp_async_commit();
  }
  int pf[C::kRowsPerThread];
#pragma unroll
  for (int i = 0; i < C::kRowsPerThread; i++) pf[i] = pg[kStages - 1][i];

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
  // query positions of this warp's tokens
  const int pbase = n - ql;  // position of token 0
  const int tok_last = min(tok0 + NTW, ql) - 1;

  for (int k = 0; k < ntiles; k++) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    if (k + kStages - 1 < ntiles) issue_tile(pf, k + kStages - 1);
    cp_async_commit();
    load_pages(pf, k + kStages);

    const uint32_t ks_base = smem_u32(smem) + (uint32_t)((k % kStages) * kStageBytes);
    const uint32_t vs_base = ks_base + kTileBytes;
    const int tile_j = j0 + k * kTileKeys;
    if (tok_last < tok0) continue;  // warp has no live query token

    // masks needed? (warp-uniform)
    const int key_hi = tile_j + kTileKeys - 1;
    const int p_lo = pbase + tok0, p_hi = pbase + tok_last;
    const bool full = key_hi < j1 && key_hi <= p_lo && (a.window == 0 || tile_j >= p_hi - a.window + 1) &&
                      (tok0 + NTW - 1 < ql);

    float s[C::kMTiles][NTW][4];
#pragma unroll
    for (int mi = 0; mi < C::kMTiles; mi++) {
      const int mt = (KS == 2) ? ks * 2 + mi : mi;
      uint32_t a0[4], a1[4];
      {
        const int r = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chb = g * 4 + (lane >> 4);
        ldsm_x4(a0, ks_base + swz(r, chb));
        ldsm_x4(a1, ks_base + swz(r, chb + 2));
      }
#pragma unroll
      for (int nt = 0; nt < NTW; nt++) {
        s[mi][nt][0] = s[mi][nt][1] = s[mi][nt][2] = s[mi][nt][3] = 0.f;
        mma_e4m3_16832(s[mi][nt], a0, qf[nt][0][0], qf[nt][0][1]);
        mma_e4m3_16832(s[mi][nt], a1, qf[nt][1][0], qf[nt][1][1]);
      }
    }
    // scale (log2 domain) and mask
#pragma unroll
    for (int mi = 0; mi < C::kMTiles; mi++) {
      const int mt = (KS == 2) ? ks * 2 + mi : mi;
#pragma unroll
      for (int nt = 0; nt < NTW; nt++) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
          float v = s[mi][nt][e] * scale_log2;
          if (!full) {
            const int j = tile_j + mt * 16 + gq + (e >> 1) * 8;
            const int tok = tok0 + nt;
            const int p = pbase + tok;
            const bool ok = j < j1 && tok < ql && j <= p && (a.window == 0 || j >= p - a.window + 1);
            v = ok ? v : -INFINITY;
          }
          s[mi][nt][e] = v;
        }
      }
    }
    // online softmax per query column (2 per thread per n-tile)
    uint32_t pb[C::kMTiles][NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; nt++) {
#pragma unroll
      for (int c = 0; c < 2; c++) {
        float mx = -INFINITY;
#pragma unroll
        for (int mi = 0; mi < C::kMTiles; mi++) mx = fmaxf(mx, fmaxf(s[mi][nt][c], s[mi][nt][c + 2]));
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
          s[mi][nt][c] = fast_exp2(s[mi][nt][c] - m_use);
          s[mi][nt][c + 2] = fast_exp2(s[mi][nt][c + 2] - m_use);
          sum += s[mi][nt][c] + s[mi][nt][c + 2];
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
        pb[mi][nt][0] = movmatrix_trans(pack_half2(s[mi][nt][0], s[mi][nt][1]));
        pb[mi][nt][1] = movmatrix_trans(pack_half2(s[mi][nt][2], s[mi][nt][3]));
      }
    }
    // PV
#pragma unroll
    for (int mi = 0; mi < C::kMTiles; mi++) {
      const int mt = (KS == 2) ? ks * 2 + mi : mi;
#pragma unroll
      for (int half = 0; half < 2; half++) {  // d in [32*half, 32*half+32)
        uint32_t r[4];
        const int key = mt * 16 + (lane & 7) + (lane >> 4) * 8;
        const int ch = g * 4 + half * 2 + ((lane >> 3) & 1);
        ldsm_x4_trans(r, vs_base + swz(key, ch));
        uint32_t ax[4], ay[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const uint32_t pr = __byte_perm(r[i], 0u, 0x3120);
          ax[i] = e4m3x2_to_f16x2((uint16_t)(pr & 0xFFFFu));
          ay[i] = e4m3x2_to_f16x2((uint16_t)(pr >> 16));
        }
#pragma unroll
        for (int nt = 0; nt < NTW; nt++) {
          mma_f16_16816(o[half * 2 + 0][nt], ax, pb[mi][nt][0], pb[mi][nt][1]);
          mma_f16_16816(o[half * 2 + 1][nt], ay, pb[mi][nt][0], pb[mi][nt][1]);
        }
      }
    }
  }
  cp_async_wait<0>();

  // ---- epilogue: full row sums, merge key shares, write the partials
#pragma unroll
  for (int nt = 0; nt < NTW; nt++)
#pragma unroll
    for (int c = 0; c < 2; c++) {
      l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 4);
      l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 8);
      l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 16);
    }
  if constexpr (KS == 2) {
    __syncthreads();  // tiles are dead: reuse the ring
    float* xs = reinterpret_cast<float*>(smem);
    constexpr int kPer = 4 * NTW * 4 + NTW * 4;  // o + (m, l) per lane
    if (ks == 1) {
      float* dst = xs + (g * 32 + lane) * kPer;
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
    __syncthreads();
    if (ks == 1) return;
    const float* src = xs + (g * 32 + lane) * kPer;
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

  const float vscale = a.scaled ? *a.v_scale : 1.0f;
  const int rows = a.L * kNumQHeads;
  float* obase = a.o_part + (int64_t)wk.slot * rows * kHeadDim;
  float* lbase = a.lse_part + (int64_t)wk.slot * rows;
#pragma unroll
  for (int nt = 0; nt < NTW; nt++) {
    const int tok = tok0 + nt;
    if (tok >= ql) continue;
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
}

template <int KS, int NTW, int NWARPS>
cudaError_t launch_variant(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  // the dynamic shared-memory limit was raised when the plan was made (occupancy query)
  auto kern = decode_kernel<KS, NTW, NWARPS>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_work);
  cfg.blockDim = dim3(NWARPS * 32);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int KS, int NTW, int NWARPS>
int occupancy_variant() {
  int nb = 0;
  auto kern = decode_kernel<KS, NTW, NWARPS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NWARPS * 32, kSmemBytes) != cudaSuccess)
    return 0;
  return nb;
}

}  // namespace

// q_len 1: 4 warps (2 KV heads x 2 key shares), one n-tile of 8 heads each.
// q_len 2..16: one warp per KV head per pair of tokens (n-tiles of 8 heads).
cudaError_t launch_decode(const DecodeArgs& a, int num_work, bool pdl, cudaStream_t s) {
  if (num_work == 0) return cudaSuccess;
  if (a.L == 1) return launch_variant<2, 1, 4>(a, num_work, pdl, s);
  if (a.L <= 2) return launch_variant<1, 2, 2>(a, num_work, pdl, s);
  if (a.L <= 4) return launch_variant<1, 2, 4>(a, num_work, pdl, s);
  if (a.L <= 8) return launch_variant<1, 2, 8>(a, num_work, pdl, s);
  return launch_variant<1, 2, 16>(a, num_work, pdl, s);
}

int decode_ctas_per_sm(int L) {
  if (L == 1) return occupancy_variant<2, 1, 4>();
  if (L <= 2) return occupancy_variant<1, 2, 2>();
  if (L <= 4) return occupancy_variant<1, 2, 4>();
  if (L <= 8) return occupancy_variant<1, 2, 8>();
  return occupancy_variant<1, 2, 16>();
}

}  // namespace okc
