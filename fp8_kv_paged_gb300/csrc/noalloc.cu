// noalloc.cu — okc_attn_decode_combine_noalloc: split-KV decode plus the merge
// and norm-gate for callers that cannot allocate device memory.
//
// Some callers can't call cudaMalloc: an op hosted inside a framework that owns
// every device allocation and hands the op only its input and output buffers
// (a plugin or custom-op interface with no workspace), or code that must not
// trigger the device synchronisation cudaMalloc/cudaFree may cause. For them the
// split partials, the work list and the per-request table live in one
// file-scope device array instead of caller buffers. The array is fixed at
// kNoAllocScratchBytes (8 MiB); every GPU that loads this library holds it until
// the process exits.
//
// The decode and combine kernels are the library's own, launched with pointers
// into the array. The array's device address is looked up once per device with
// cudaGetSymbolAddress (host code may not use the symbol's name as an address).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "okc_common.cuh"
#include "okc_internal.h"

namespace okc {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kMaxWork = 4096;     // work items per call
constexpr int kMaxBatch = 2048;    // requests per call
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Device address of g_noalloc_scratch on the current device (set up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace okc

extern "C" okc_status okc_attn_decode_combine_noalloc(
    const okc_attn_config* cfg, const int32_t* seq_lens_host, const uint8_t* q_fp8,
    const uint8_t* k_cache, const uint8_t* v_cache, const float* k_scale, const float* v_scale,
    const int32_t* page_table, const int32_t* cache_seqlens, const int32_t* cu_seqlens_q,
    const int32_t* seq_lens, const void* qkv, const void* norm_weight, float eps, void* out,
    okc_stream stream) {
  using namespace okc;
  if (!cfg || !seq_lens_host) return OKC_ERR_INVALID;
  const okc_attn_config& c = *cfg;
  if (c.batch < 1 || c.q_len < 1 || c.q_len > kMaxQLen || c.window < 0 || c.max_pages < 1 ||
      c.num_pages < 1 || !(c.sm_scale > 0.f) || !(c.qk_scale_factor > 0.f) || !(c.kv_scale > 0.f) ||
      !std::isfinite(c.sm_scale) || !std::isfinite(c.qk_scale_factor) || !std::isfinite(c.kv_scale) ||
      !(eps >= 0.f) || !std::isfinite(eps) || (c.q_norm != OKC_QNORM_BF16 && c.q_norm != OKC_QNORM_FOLDED_SCALE))
    return OKC_ERR_INVALID;
  if (c.head_dim != kHeadDim || c.num_q_heads != kNumQHeads || c.num_kv_heads != kNumKvHeads ||
      c.page_size < 1 || c.page_size > 256 || (c.page_size & (c.page_size - 1)) ||
      (int64_t)c.max_pages * c.page_size > (int64_t)1 << 30)
    return OKC_ERR_UNSUPPORTED;
  if (!q_fp8 || !k_cache || !v_cache || !page_table || !cache_seqlens || !cu_seqlens_q || !qkv || !out)
    return OKC_ERR_INVALID;
  const bool scaled = c.kv_scale != 1.f;
  if (scaled && (!k_scale || !v_scale)) return OKC_ERR_INVALID;
  auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
  if (!al(q_fp8, 16) || !al(k_cache, 16) || !al(v_cache, 16) || !al(qkv, 16) || !al(out, 16) ||
      (norm_weight && !al(norm_weight, 16)) || !al(page_table, 4) || !al(cache_seqlens, 4) ||
      !al(cu_seqlens_q, 4) || !al(seq_lens, 4) || !al(k_scale, 4) || !al(v_scale, 4))
    return OKC_ERR_INVALID;
  if (c.batch > kMaxBatch) return OKC_ERR_WORKSPACE;

  // The work list of okc_attn_plan with the default options (the same split
  // rule, launch order and kernel choice), for this device's resident CTA slots.
  const int B = c.batch, L = c.q_len;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return OKC_ERR_CUDA;
  const bool use_tc = uses_tc(c, nullptr);  // the default plan's kernel choice
  const int S = block_tokens(c, nullptr);
  const int per_sm = cached_ctas_per_sm(dev, S, use_tc, tc_groups(c));
  if (per_sm <= 0) return OKC_ERR_CUDA;
  SplitResult split;
  const okc_status st = make_splits(cfg, seq_lens_host, nullptr, nullptr, sms * per_sm, &split);
  if (st != OKC_OK) return st;
  const int64_t W = (int64_t)split.work.size();
  const int64_t NB = (int64_t)split.blocks.size();
  if (W > kMaxWork) return OKC_ERR_WORKSPACE;
  // Scratch layout in the static array: work list | block table | LSE | partial outputs.
  const int64_t rows = (int64_t)S * kNumQHeads;
  const size_t off_req = up256((size_t)W * sizeof(WorkItem));
  const size_t off_lse = off_req + up256((size_t)NB * sizeof(BlockInfo));
  const size_t off_o = off_lse + up256((size_t)W * rows * sizeof(float));
  const size_t need = off_o + (size_t)W * rows * kHeadDim * sizeof(float);
  if (need > kNoAllocScratchBytes) return OKC_ERR_WORKSPACE;

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return OKC_ERR_CUDA;
  uint8_t* s8 = static_cast<uint8_t*>(base);
  cudaStream_t str = reinterpret_cast<cudaStream_t>(stream);
  // pageable sources are staged before cudaMemcpyAsync returns
  if (cudaMemcpyAsync(s8, split.work.data(), (size_t)W * sizeof(WorkItem), cudaMemcpyHostToDevice, str) !=
          cudaSuccess ||
      cudaMemcpyAsync(s8 + off_req, split.blocks.data(), (size_t)NB * sizeof(BlockInfo), cudaMemcpyHostToDevice,
                      str) != cudaSuccess)
    return OKC_ERR_CUDA;

  int shift = 0;
  while ((1 << shift) < c.page_size) shift++;
  DecodeArgs d = {};
  d.tc = use_tc ? 1 : 0;
  d.tc_groups = tc_groups(c);
  d.q8 = q_fp8;
  d.kc = k_cache;
  d.vc = v_cache;
  d.k_scale = k_scale;
  d.v_scale = v_scale;
  d.page_table = page_table;
  d.cache_seqlens = cache_seqlens;
  d.cu_seqlens_q = cu_seqlens_q;
  d.seq_lens = seq_lens;
  d.work = reinterpret_cast<const WorkItem*>(s8);
  d.o_part = reinterpret_cast<float*>(s8 + off_o);
  d.lse_part = reinterpret_cast<float*>(s8 + off_lse);
  d.err = nullptr;  // out-of-range accesses are still skipped, just not reported
  d.batch = B;
  d.L = L;
  d.S = S;
  d.window = c.window;
  d.max_pages = c.max_pages;
  d.num_pages = c.num_pages;
  d.page_shift = shift;
  d.scaled = scaled;
  d.T = (int32_t)split.tokens;
  d.scale_log2 = softmax_scale_log2(c);
  if (launch_decode(d, (int)W, false, str) != cudaSuccess) return OKC_ERR_CUDA;

  CombineArgs m;
  m.o_part = d.o_part;
  m.lse_part = d.lse_part;
  m.qkv = static_cast<const uint16_t*>(qkv);
  m.weight = static_cast<const uint16_t*>(norm_weight);
  m.out = static_cast<uint16_t*>(out);
  m.blk = reinterpret_cast<const BlockInfo*>(s8 + off_req);
  m.err = nullptr;
  m.nblocks = (int32_t)NB;
  m.S = S;
  m.T = (int32_t)split.tokens;
  m.eps = eps;
  if (launch_combine(m, false, str) != cudaSuccess) return OKC_ERR_CUDA;
  return OKC_OK;
}
