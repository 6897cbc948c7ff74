// prepare.cu — steps 1-3 of the block (the `_prepare_qkv` kernel of
// "012-attention-local-splits.py"): per-head RMSNorm of q and k from the fused
// bf16 qkv row, interleaved RoPE on rope layers, E4M3 q, and the E4M3 K/V
// scatter into the paged cache at the token's cache row.
//
// Mapping: one CTA per token, 8 lanes per head (20 heads -> 160 threads). Each
// lane owns 8 consecutive columns, loaded as one 16-byte vector; the RMS sum
// is reduced over the head's 8 lanes with __shfl_xor_sync. A RoPE pair (2i,
// 2i+1) always lies inside one lane's vector, so the partner exchange is a
// register swap. Each lane stores its 8 E4M3 bytes with one 8-byte store; the
// 8 lanes of a head cover the head's 64-byte segment of the row.
//
// Under OKC_QNORM_FOLDED_SCALE (the vLLM CuTeDSL qk_norm with an output scale)
// a q head is bf16(f32(f32(x * rstd) * qk_scale_factor)): both products in
// float32, the bf16 store its only rounding to bf16.
//
// Numerics (the reading the oracle also takes): the RMS inverse is the float32
// rounding of 1/sqrt(sum(x^2)/64 + eps) (rms_inverse: float32 arithmetic with a
// double-precision fallback near rounding boundaries, so the rounding does not
// depend on summation order); every
// float32 product and sum of the rotation is rounded separately (explicit
// __fmul_rn / __fadd_rn, no contraction); the scaled path divides with
// IEEE division (__fdiv_rn).
#include "okc_common.cuh"
#include "okc_internal.h"

namespace okc {

namespace {

constexpr int kPrepThreads = 8 * (kNumQHeads + 2 * kNumKvHeads);  // 160

__device__ __forceinline__ uint2 pack_e4m3x8(const float (&v)[8]) {
  uint2 r;
  r.x = static_cast<uint32_t>(f32x2_to_e4m3x2(v[0], v[1])) |
        (static_cast<uint32_t>(f32x2_to_e4m3x2(v[2], v[3])) << 16);
  r.y = static_cast<uint32_t>(f32x2_to_e4m3x2(v[4], v[5])) |
        (static_cast<uint32_t>(f32x2_to_e4m3x2(v[6], v[7])) << 16);
  return r;
}

__global__ void __launch_bounds__(kPrepThreads) prepare_kernel(PrepareArgs a) {
  const int t = blockIdx.x;
  const int h = threadIdx.x >> 3;       // head: [0,Hq) q, [Hq,Hq+Hkv) k, then v
  const int c0 = (threadIdx.x & 7) * 8;  // first of this lane's 8 columns
  // This kernel reads only caller inputs and writes rows nobody in flight reads:
  // let the dependent launch begin right away.
  pdl_wait();
  pdl_launch_dependents();

  const uint4 raw = *reinterpret_cast<const uint4*>(a.qkv + (size_t)t * kQkvWidth + h * kHeadDim + c0);
  float x[8];
  {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
      x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
  }
  // RMS inverse of the head (all lanes take part so the 8-lane shuffles see
  // full groups; the v heads ignore the result)
  const float inv = rms_inverse<8, 8>(x, kRmsEps);

  const int64_t slot = a.cache_loc[t];
  const bool slot_ok = slot >= 0 && slot < a.num_rows;
  if (!slot_ok && threadIdx.x == 0) set_error(a.err, OKC_DEVERR_CACHE_LOC);

  if (h < kNumQHeads + kNumKvHeads) {
    float y[8];
    if (a.q_fold && h < kNumQHeads) {  // q under OKC_QNORM_FOLDED_SCALE: the factor before the one bf16 rounding
#pragma unroll
      for (int i = 0; i < 8; i++) y[i] = bf16_round(__fmul_rn(__fmul_rn(x[i], inv), a.q_scale));
    } else {
#pragma unroll
      for (int i = 0; i < 8; i++) y[i] = bf16_round(__fmul_rn(x[i], inv));
    }
    if (a.rope) {
      const int64_t pos = a.positions[t];
      if (pos >= 0 && pos < a.rope_positions) {
        const float* row = a.rope_table + pos * kHeadDim;
        const float4 cs = *reinterpret_cast<const float4*>(row + c0 / 2);
        const float4 sn = *reinterpret_cast<const float4*>(row + kHeadDim / 2 + c0 / 2);
        const float cc[4] = {cs.x, cs.y, cs.z, cs.w};
        const float ssn[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const float e = y[2 * k], o = y[2 * k + 1];
          y[2 * k] = bf16_round(__fsub_rn(__fmul_rn(e, cc[k]), __fmul_rn(o, ssn[k])));
          y[2 * k + 1] = bf16_round(__fadd_rn(__fmul_rn(o, cc[k]), __fmul_rn(e, ssn[k])));
        }
      } else if ((threadIdx.x & 7) == 0) {
        set_error(a.err, OKC_DEVERR_POSITION);
      }
    }
    if (h < kNumQHeads) {
      *reinterpret_cast<uint2*>(a.q8 + ((size_t)t * kNumQHeads + h) * kHeadDim + c0) = pack_e4m3x8(y);
    } else if (slot_ok) {
      if (a.scaled) {
        const float ks = *a.k_scale;
#pragma unroll
        for (int i = 0; i < 8; i++) y[i] = bf16_round(__fdiv_rn(y[i], ks));
      }
      *reinterpret_cast<uint2*>(a.kc + slot * kRowBytes + (h - kNumQHeads) * kHeadDim + c0) =
          pack_e4m3x8(y);
    }
  } else if (slot_ok) {
    if (a.scaled) {
      const float vs = *a.v_scale;
#pragma unroll
      for (int i = 0; i < 8; i++) x[i] = bf16_round(__fdiv_rn(x[i], vs));
    }
    *reinterpret_cast<uint2*>(a.vc + slot * kRowBytes + (h - kNumQHeads - kNumKvHeads) * kHeadDim + c0) =
        pack_e4m3x8(x);
  }
}

struct InvFreq {
  float v[kHeadDim / 2];
};

// table[pos][0:32] = cos(f32(pos * inv_freq)), [32:64] = sin(...), each the
// float32 rounding of the double-precision value.
__global__ void rope_table_kernel(InvFreq inv, int32_t n, float* table) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (pos, pair)
  if (idx >= (int64_t)n * (kHeadDim / 2)) return;
  const int64_t pos = idx / (kHeadDim / 2);
  const int i = (int)(idx % (kHeadDim / 2));
  const float ang = __fmul_rn((float)pos, inv.v[i]);
  double s, c;
  sincos((double)ang, &s, &c);
  table[pos * kHeadDim + i] = (float)c;
  table[pos * kHeadDim + kHeadDim / 2 + i] = (float)s;
}

}  // namespace

cudaError_t launch_prepare(const PrepareArgs& a, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.T);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prepare_kernel, a);
}

cudaError_t launch_rope_table(float theta, const float* inv_freq, int32_t n, float* table,
                              cudaStream_t s) {
  (void)theta;
  InvFreq inv;
  for (int i = 0; i < kHeadDim / 2; i++) inv.v[i] = inv_freq[i];
  const int64_t total = (int64_t)n * (kHeadDim / 2);
  const int threads = 256;
  const unsigned blocks = (unsigned)((total + threads - 1) / threads);
  rope_table_kernel<<<blocks, threads, 0, s>>>(inv, n, table);
  return cudaGetLastError();
}

}  // namespace okc
