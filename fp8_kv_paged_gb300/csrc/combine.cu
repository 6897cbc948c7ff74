// combine.cu — merge of the split-KV partials fused with step 5 of the block
// (the rms_norm_gate call of "012-attention-local-splits.py": per-head RMSNorm
// of the bf16 attention output times sigmoid of the gate logits, weight None
// or a bf16 [64] weight, eps 1e-5).
//
// One CTA per token, 8 lanes per q head (16 heads -> 128 threads); a lane owns
// 8 consecutive columns (two float4 loads per split, one 16-byte gate load,
// one 16-byte output store). Merge: M = max_s lse_s, o = sum_s 2^(lse_s - M) o_s
// / sum_s 2^(lse_s - M) (lse in base 2). Then ob = bf16(o) (the attention
// output is bf16, as FA3 returns it), r = 1/sqrt(mean(ob^2) + eps) over the
// head's 8 lanes, out = bf16(ob * r * w * sigmoid(gate)) in float32.
#include "okc_common.cuh"
#include "okc_internal.h"

namespace okc {

namespace {

constexpr int kCombThreads = 8 * kNumQHeads;  // 128

__global__ void __launch_bounds__(kCombThreads) combine_kernel(CombineArgs a) {
  const int t = blockIdx.x;
  const int h = threadIdx.x >> 3;
  const int c0 = (threadIdx.x & 7) * 8;
  const int b = t / a.L, i = t - b * a.L;

  // caller inputs first (overlaps the decode kernel's tail)
  const uint4 graw = *reinterpret_cast<const uint4*>(a.qkv + (size_t)t * kQkvWidth + kGateCol + h * kHeadDim + c0);
  float w[8];
  if (a.weight) {
    const uint4 wraw = *reinterpret_cast<const uint4*>(a.weight + c0);
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
  pdl_wait();
  pdl_launch_dependents();

  const ReqInfo rq = a.req[b];
  const int rows = a.L * kNumQHeads;
  const int row = i * kNumQHeads + h;
  const float* lse = a.lse_part + (int64_t)rq.wbase * rows + row;
  const float* op = a.o_part + ((int64_t)rq.wbase * rows + row) * kHeadDim + c0;
  const int64_t ostride = (int64_t)rows * kHeadDim;
  // splits are visited in batches of kB with every load of a batch in flight at once
  constexpr int kB = 8;
  float M = -INFINITY;
  for (int s0 = 0; s0 < rq.nchunks; s0 += kB) {
    float ls[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) ls[u] = s0 + u < rq.nchunks ? lse[(int64_t)(s0 + u) * rows] : -INFINITY;
#pragma unroll
    for (int u = 0; u < kB; u++) M = fmaxf(M, ls[u]);
  }
  const float Mu = M == -INFINITY ? 0.f : M;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  for (int s0 = 0; s0 < rq.nchunks; s0 += kB) {
    float ls[kB];
    float4 x0[kB], x1[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const bool live = s0 + u < rq.nchunks;
      ls[u] = live ? lse[(int64_t)(s0 + u) * rows] : -INFINITY;
      const float4* src = reinterpret_cast<const float4*>(op + (int64_t)(live ? s0 + u : 0) * ostride);
      x0[u] = live ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
      x1[u] = live ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const float wt = ls[u] == -INFINITY ? 0.f : exp2f(ls[u] - Mu);
      wsum += wt;
      acc[0] += wt * x0[u].x; acc[1] += wt * x0[u].y; acc[2] += wt * x0[u].z; acc[3] += wt * x0[u].w;
      acc[4] += wt * x1[u].x; acc[5] += wt * x1[u].y; acc[6] += wt * x1[u].z; acc[7] += wt * x1[u].w;
    }
  }
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
  const float r = 1.f / sqrtf(ss / (float)kHeadDim + a.eps);

  const uint32_t gw[4] = {graw.x, graw.y, graw.z, graw.w};
  uint32_t outw[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; e++) {
      const float gt = bf16_bits_to_f32(e ? (gw[k] >> 16) : (gw[k] & 0xFFFFu));
      const float sig = 1.f / (1.f + expf(-gt));
      v[e] = ob[2 * k + e] * r * w[2 * k + e] * sig;
    }
    const __nv_bfloat162 p = __floats2bfloat162_rn(v[0], v[1]);
    outw[k] = *reinterpret_cast<const uint32_t*>(&p);
  }
  *reinterpret_cast<uint4*>(a.out + (size_t)t * (kNumQHeads * kHeadDim) + h * kHeadDim + c0) =
      make_uint4(outw[0], outw[1], outw[2], outw[3]);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, bool pdl, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.T);
  cfg.blockDim = dim3(kCombThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace okc
