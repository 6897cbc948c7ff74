// fused_rows.cuh — steps 1-3 of the block ("012-attention-local-splits.py",
// _prepare_qkv) computed inside a one-kernel step instead of by the prepare
// kernel: a q head's E4M3 row and a new key's E4M3 K and V rows, with the
// prepare kernel's arithmetic (correctly rounded RMS inverse, each float32
// product and sum of the rotation rounded separately, bf16 roundings, E4M3 RNE
// satfinite).
#pragma once

#include "okc_common.cuh"
#include "okc_internal.h"

namespace okc {

// The new key row of token t for KV head g: this lane's dims 2*lane, 2*lane+1 of
// K (RMSNorm + RoPE, / k_scale on the scaled path) and of V (raw, / v_scale),
// as two E4M3 pairs. All 32 lanes take part (the head's reduction).
__device__ __forceinline__ void fused_new_kv(const DecodeArgs& a, int64_t t, int g, int lane, uint16_t& k8,
                                             uint16_t& v8, bool& pos_err) {
  const uint16_t* row = a.qkv + t * kQkvWidth;
  const uint32_t kr = *reinterpret_cast<const uint32_t*>(row + (kNumQHeads + g) * kHeadDim + 2 * lane);
  const uint32_t vr = *reinterpret_cast<const uint32_t*>(row + (kNumQHeads + kNumKvHeads + g) * kHeadDim + 2 * lane);
  const float x0 = bf16_bits_to_f32(kr & 0xFFFFu), x1 = bf16_bits_to_f32(kr >> 16);
  const float xs[2] = {x0, x1};
  const float inv = rms_inverse<32, 2>(xs, kRmsEps);
  float y0 = bf16_round(__fmul_rn(x0, inv)), y1 = bf16_round(__fmul_rn(x1, inv));
  if (a.rope) {
    const int64_t pos = a.positions[t];
    if (pos >= 0 && pos < a.rope_positions) {
      const float c = a.rope_table[pos * kHeadDim + lane], sn = a.rope_table[pos * kHeadDim + kHeadDim / 2 + lane];
      const float e = y0, o = y1;
      y0 = bf16_round(__fsub_rn(__fmul_rn(e, c), __fmul_rn(o, sn)));
      y1 = bf16_round(__fadd_rn(__fmul_rn(o, c), __fmul_rn(e, sn)));
    } else {
      pos_err = true;
    }
  }
  float v0 = bf16_bits_to_f32(vr & 0xFFFFu), v1 = bf16_bits_to_f32(vr >> 16);
  if (a.scaled) {
    const float ks = *a.k_scale, vs = *a.v_scale;
    y0 = bf16_round(__fdiv_rn(y0, ks));
    y1 = bf16_round(__fdiv_rn(y1, ks));
    v0 = bf16_round(__fdiv_rn(v0, vs));
    v1 = bf16_round(__fdiv_rn(v1, vs));
  }
  k8 = f32x2_to_e4m3x2(y0, y1);
  v8 = f32x2_to_e4m3x2(v0, v1);
}

// Up to 8 new key rows for KV head g at once (this lane's dims 2*lane, 2*lane+1
// of each, as fused_new_kv): the rows' inputs are loaded for all keys first
// (qkv pairs, positions, then the RoPE entries), so the loads of different
// keys overlap instead of forming one chain per key. Key i < count is token
// t0 + i.
__device__ __forceinline__ void fused_new_kv8(const DecodeArgs& a, int64_t t0, int count, int g, int lane,
                                              uint16_t (&k8)[8], uint16_t (&v8)[8], bool& pos_err) {
  uint32_t kr[8], vr[8];
  int64_t pos[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    kr[i] = vr[i] = 0u;
    pos[i] = 0;
    if (i < count) {
      const uint16_t* row = a.qkv + (t0 + i) * kQkvWidth;
      kr[i] = *reinterpret_cast<const uint32_t*>(row + (kNumQHeads + g) * kHeadDim + 2 * lane);
      vr[i] = *reinterpret_cast<const uint32_t*>(row + (kNumQHeads + kNumKvHeads + g) * kHeadDim + 2 * lane);
      if (a.rope) pos[i] = a.positions[t0 + i];
    }
  }
  float cs[8], sn[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    cs[i] = 1.f;
    sn[i] = 0.f;
    if (a.rope && i < count) {
      if (pos[i] >= 0 && pos[i] < a.rope_positions) {
        cs[i] = a.rope_table[pos[i] * kHeadDim + lane];
        sn[i] = a.rope_table[pos[i] * kHeadDim + kHeadDim / 2 + lane];
      } else {
        pos_err = true;
      }
    }
  }
  const float ks = a.scaled ? *a.k_scale : 1.f, vs = a.scaled ? *a.v_scale : 1.f;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    if (i >= count) break;  // (count is uniform across the warp)
    const float x0 = bf16_bits_to_f32(kr[i] & 0xFFFFu), x1 = bf16_bits_to_f32(kr[i] >> 16);
    const float xs[2] = {x0, x1};
    const float inv = rms_inverse<32, 2>(xs, kRmsEps);
    float y0 = bf16_round(__fmul_rn(x0, inv)), y1 = bf16_round(__fmul_rn(x1, inv));
    if (a.rope && pos[i] >= 0 && pos[i] < a.rope_positions) {
      const float e = y0, o = y1;
      y0 = bf16_round(__fsub_rn(__fmul_rn(e, cs[i]), __fmul_rn(o, sn[i])));
      y1 = bf16_round(__fadd_rn(__fmul_rn(o, cs[i]), __fmul_rn(e, sn[i])));
    }
    float v0 = bf16_bits_to_f32(vr[i] & 0xFFFFu), v1 = bf16_bits_to_f32(vr[i] >> 16);
    if (a.scaled) {
      y0 = bf16_round(__fdiv_rn(y0, ks));
      y1 = bf16_round(__fdiv_rn(y1, ks));
      v0 = bf16_round(__fdiv_rn(v0, vs));
      v1 = bf16_round(__fdiv_rn(v1, vs));
    }
    k8[i] = f32x2_to_e4m3x2(y0, y1);
    v8[i] = f32x2_to_e4m3x2(v0, v1);
  }
}

// The E4M3 q row of token t, q head `head`, held by one thread: word i holds
// dims 4i .. 4i+3, dim 4i in the low byte (the byte order of the prepare
// kernel's q output). RoPE rotates the pairs (2i, 2i+1) by the table's entry
// i (cos) and 32 + i (sin). `live` false gives zeros; every lane of the warp
// calls it (the RMS inverse's rare double-precision path is warp-wide).
__device__ __forceinline__ void fused_q_row(const DecodeArgs& a, int64_t t, int head, bool live, uint32_t (&w)[16],
                                            bool& pos_err) {
  float y[64];
  const uint4* row = reinterpret_cast<const uint4*>(a.qkv + t * kQkvWidth + head * kHeadDim);
#pragma unroll
  for (int c = 0; c < 8; c++) {
    const uint4 raw = live ? row[c] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      y[8 * c + 2 * k] = bf16_bits_to_f32(u[k] & 0xFFFFu);
      y[8 * c + 2 * k + 1] = bf16_bits_to_f32(u[k] >> 16);
    }
  }
  const float inv = rms_inverse<1, 64>(y, kRmsEps);
#pragma unroll
  for (int i = 0; i < 64; i++)  // OKC_QNORM_FOLDED_SCALE: the factor before the one bf16 rounding
    y[i] = bf16_round(a.q_fold ? __fmul_rn(__fmul_rn(y[i], inv), a.q_scale) : __fmul_rn(y[i], inv));
  if (a.rope && live) {
    const int64_t pos = a.positions[t];
    if (pos >= 0 && pos < a.rope_positions) {
      const float* tab = a.rope_table + pos * kHeadDim;
#pragma unroll
      for (int i = 0; i < 32; i++) {
        const float c = tab[i], sn = tab[kHeadDim / 2 + i];
        const float e = y[2 * i], o = y[2 * i + 1];
        y[2 * i] = bf16_round(__fsub_rn(__fmul_rn(e, c), __fmul_rn(o, sn)));
        y[2 * i + 1] = bf16_round(__fadd_rn(__fmul_rn(o, c), __fmul_rn(e, sn)));
      }
    } else {
      pos_err = true;
    }
  }
#pragma unroll
  for (int i = 0; i < 16; i++)
    w[i] = (uint32_t)f32x2_to_e4m3x2(y[4 * i], y[4 * i + 1]) | ((uint32_t)f32x2_to_e4m3x2(y[4 * i + 2], y[4 * i + 3]) << 16);
}

}  // namespace okc
