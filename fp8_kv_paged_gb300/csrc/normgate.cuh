// normgate.cuh — merge of split-KV partials and step 5 of the block (the
// rms_norm_gate call of "012-attention-local-splits.py": per-head RMSNorm of the
// bf16 attention output times sigmoid of the gate logits, weight None or a
// bf16 [64] weight), for one (token, q head) row with 8 lanes of a warp (lanes
// 8k..8k+7), each owning 8 consecutive columns.
//
// Merge: M = max_s lse_s, o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M)
// (lse in base 2). Then ob = bf16(o) (the attention output is bf16, as FA3
// returns it), r = 1/sqrt(mean(ob^2) + eps) over the head's 8 lanes, and
// out = bf16(ob * r * w * sigmoid(gate)) in float32.
#pragma once

#include "okc_common.cuh"

namespace okc {

// Gate logits and weight of this lane's 8 columns (caller inputs).
__device__ __forceinline__ void load_gate_weight(const uint16_t* qkv, const uint16_t* weight, int t, int h,
                                                 int c0, float (&g)[8], float (&w)[8]) {
  const uint4 graw = *reinterpret_cast<const uint4*>(qkv + (size_t)t * kQkvWidth + kGateCol + h * kHeadDim + c0);
  const uint32_t gw[4] = {graw.x, graw.y, graw.z, graw.w};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    g[2 * k] = bf16_bits_to_f32(gw[k] & 0xFFFFu);
    g[2 * k + 1] = bf16_bits_to_f32(gw[k] >> 16);
  }
  if (weight) {
    const uint4 wraw = *reinterpret_cast<const uint4*>(weight + c0);
    const uint32_t ww[4] = {wraw.x, wraw.y, wraw.z, wraw.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      w[2 * k] = bf16_bits_to_f32(ww[k] & 0xFFFFu);
      w[2 * k + 1] = bf16_bits_to_f32(ww[k] >> 16);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; k++) w[k] = 1.f;
  }
}

// Splits are visited in batches of kB (8 by default) with every load of a
// batch in flight (one round trip per batch; each split holds 9 registers).
// Online over batches: the running sums are rescaled by 2^(M_old - M_new) when
// a batch raises the maximum; with at most kB splits this is the plain
// two-pass merge (M = max of all lse).
constexpr int kMergeBatch = 8;

template <int kB>
__device__ __forceinline__ void merge_accumulate(const float (&ls)[kB], const float4 (&x0)[kB],
                                                 const float4 (&x1)[kB], float& M, float (&acc)[8],
                                                 float& wsum) {
  float bm = M;
#pragma unroll
  for (int u = 0; u < kB; u++) bm = fmaxf(bm, ls[u]);
  const float bmu = bm == -INFINITY ? 0.f : bm;
  if (M != -INFINITY && bm != M) {  // an earlier batch: rescale its sums to the new maximum
    const float sc = exp2f(M - bmu);
    wsum *= sc;
#pragma unroll
    for (int k = 0; k < 8; k++) acc[k] *= sc;
  }
  M = bm;
#pragma unroll
  for (int u = 0; u < kB; u++) {
    const float wt = ls[u] == -INFINITY ? 0.f : exp2f(ls[u] - bmu);
    wsum += wt;
    acc[0] += wt * x0[u].x; acc[1] += wt * x0[u].y; acc[2] += wt * x0[u].z; acc[3] += wt * x0[u].w;
    acc[4] += wt * x1[u].x; acc[5] += wt * x1[u].y; acc[6] += wt * x1[u].z; acc[7] += wt * x1[u].w;
  }
}

// o = acc / wsum rounded to bf16, then the row's RMS over its 8 lanes and the
// gated, weighted bf16 output (8 columns, one 16-byte store).
__device__ __forceinline__ void normgate_store(const float (&acc)[8], float wsum, const float (&g)[8],
                                               const float (&w)[8], float eps, uint16_t* dst) {
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  float ob[8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < 8; k++) {
    ob[k] = bf16_round(acc[k] * inv);
    ss += ob[k] * ob[k];
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  const float r = 1.f / sqrtf(ss / (float)kHeadDim + eps);
  uint32_t outw[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; e++) {
      const float sig = 1.f / (1.f + expf(-g[2 * k + e]));
      v[e] = ob[2 * k + e] * r * w[2 * k + e] * sig;
    }
    const __nv_bfloat162 p = __floats2bfloat162_rn(v[0], v[1]);
    outw[k] = *reinterpret_cast<const uint32_t*>(&p);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
}

// Splits in global memory. lse: the row's base-2 LSE of split 0, consecutive
// splits `lse_stride` floats apart; op: this lane's 8 columns of split 0, splits
// `o_stride` floats apart. Loads bypass L1 (partials written by other CTAs of
// the same grid). kB: splits per batch.
template <int kB = kMergeBatch>
__device__ __forceinline__ void merge_normgate(const float* lse, int64_t lse_stride, const float* op,
                                               int64_t o_stride, int nchunks, const float (&g)[8],
                                               const float (&w)[8], float eps, uint16_t* dst) {
  float M = -INFINITY;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  for (int s0 = 0; s0 < nchunks; s0 += kB) {
    float ls[kB];
    float4 x0[kB], x1[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const bool live = s0 + u < nchunks;
      ls[u] = live ? __ldcg(lse + (int64_t)(s0 + u) * lse_stride) : -INFINITY;
      const float4* src = reinterpret_cast<const float4*>(op + (int64_t)(live ? s0 + u : 0) * o_stride);
      x0[u] = live ? __ldcg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      x1[u] = live ? __ldcg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    merge_accumulate(ls, x0, x1, M, acc, wsum);
  }
  normgate_store(acc, wsum, g, w, eps, dst);
}

}  // namespace okc
