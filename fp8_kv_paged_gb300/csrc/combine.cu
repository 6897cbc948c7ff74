// combine.cu — merge of the split-KV partials fused with step 5 of the block
// (the rms_norm_gate call of "012-attention-local-splits.py"). The arithmetic
// is normgate.cuh's, shared with the fused step kernel's last-CTA epilogue.
//
// One CTA per token: blockIdx.x the query block, blockIdx.y its token; 8 lanes
// per q head (16 heads -> 128 threads); a lane owns 8 consecutive columns (two
// float4 loads per split, one 16-byte gate load, one 16-byte output store).
#include "normgate.cuh"
#include "okc_internal.h"

namespace okc {

namespace {

constexpr int kCombThreads = 8 * kNumQHeads;  // 128
// Splits merged per round trip: 8 for blocks of one token (steps whose
// requests have many splits); 4 for longer blocks (verify and extend steps: few
// splits per block, many blocks), which keeps the kernel under 64 registers a
// thread so that two of its CTAs fit beside a tcgen05 decode CTA on one SM (the
// combine is launched under programmatic dependent launch while the decode runs).

template <int kB>
__global__ void __launch_bounds__(kCombThreads) combine_kernel(CombineArgs a) {
  const int i = blockIdx.y;  // token of the block
  const int h = threadIdx.x >> 3;
  const int c0 = (threadIdx.x & 7) * 8;
  const BlockInfo bl = a.blk[blockIdx.x];  // plan data
  if (i >= bl.ntok) return;
  const int t = bl.t0 + i;

  // caller inputs first (overlaps the decode kernel's tail)
  float g[8], w[8];
  load_gate_weight(a.qkv, a.weight, t, h, c0, g, w);
  pdl_wait();
  pdl_launch_dependents();

  const int rows = a.S * kNumQHeads;
  const int row = i * kNumQHeads + h;
  merge_normgate<kB>(a.lse_part + (int64_t)bl.wbase * rows + row, rows,
                 a.o_part + ((int64_t)bl.wbase * rows + row) * kHeadDim + c0, (int64_t)rows * kHeadDim,
                 bl.nchunks, g, w, a.eps, a.out + (size_t)t * (kNumQHeads * kHeadDim) + h * kHeadDim + c0);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, bool pdl, cudaStream_t s) {
  if (a.T == 0 || a.nblocks == 0) return cudaSuccess;
  if (a.S < 1 || a.S > 16) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nblocks, a.S);
  cfg.blockDim = dim3(kCombThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return a.S == 1 ? cudaLaunchKernelEx(&cfg, combine_kernel<8>, a) : cudaLaunchKernelEx(&cfg, combine_kernel<4>, a);
}

}  // namespace okc
