// step_host_routing.cu — okc_attn_step_host's routing of host buffers without a
// GPU: the CUDA runtime calls are host fakes (a set of "mapped" host buffers,
// each with a distinct device alias; copies recorded, not performed) and the
// kernel launchers stubs that record their arguments. For every combination of
// mapped and pageable inputs, and of aligned and misaligned qkv / out, checks:
// a mapped input whose alias is aligned as its kernel loads it is read in place
// (the kernel gets the alias, no copy); any other input is copied host-to-device
// once, with its exact byte count, into its device buffer, which the kernel
// gets; the output is written in place when mapped and aligned, else copied
// back from the device buffer with its exact byte count; the stream is then
// synchronized; a missing buffer is an argument error before any copy.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <random>
#include <vector>
struct CopyRec { void* dst; const void* src; size_t n; int kind; };
static std::vector<CopyRec> g_copies;
static std::map<const void*, const void*> g_alias;  // mapped host buffer -> device alias
static int g_syncs = 0;
static cudaError_t fake_memcpy(void* d, const void* s, size_t n, cudaMemcpyKind k, cudaStream_t) {
  g_copies.push_back({d, s, n, (int)k});
  return cudaSuccess;
}
static cudaError_t fake_ptr_attr(cudaPointerAttributes* a, const void* p) {
  memset(a, 0, sizeof *a);
  auto it = g_alias.find(p);
  if (it == g_alias.end()) { a->type = cudaMemoryTypeUnregistered; return cudaSuccess; }
  a->type = cudaMemoryTypeHost;
  a->devicePointer = const_cast<void*>(it->second);
  return cudaSuccess;
}
static cudaError_t fake_sync(cudaStream_t) { g_syncs++; return cudaSuccess; }
static cudaError_t fake_get_device(int* d) { *d = 0; return cudaSuccess; }
static cudaError_t fake_attr(int* v, cudaDeviceAttr, int) { *v = 152; return cudaSuccess; }
static cudaError_t fake_get_last_error() { return cudaSuccess; }
#define cudaMemcpyAsync fake_memcpy
#define cudaPointerGetAttributes fake_ptr_attr
#define cudaStreamSynchronize fake_sync
#define cudaGetDevice fake_get_device
#define cudaDeviceGetAttribute fake_attr
#define cudaGetLastError fake_get_last_error
#include "okc_api.cu"
static okc::DecodeArgs g_dec;
static okc::PrepareArgs g_prep;
static okc::CombineArgs g_comb;
static int g_fused = 0, g_three = 0;
namespace okc {
cudaError_t launch_prepare(const PrepareArgs& a, bool, cudaStream_t) { g_prep = a; g_three++; return cudaSuccess; }
cudaError_t launch_decode(const DecodeArgs& a, int, bool, cudaStream_t) { g_dec = a; g_three++; return cudaSuccess; }
cudaError_t launch_step_fused(const DecodeArgs& a, int, bool, cudaStream_t) { g_dec = a; g_fused++; return cudaSuccess; }
cudaError_t launch_step_fused_tc(const DecodeArgs& a, int, bool, cudaStream_t) { g_dec = a; g_fused++; return cudaSuccess; }
cudaError_t launch_combine(const CombineArgs& a, bool, cudaStream_t) { g_comb = a; g_three++; return cudaSuccess; }
cudaError_t launch_rope_table(float, const float*, int32_t, float*, cudaStream_t) { return cudaSuccess; }
int decode_ctas_per_sm(int, bool tc, int) { return tc ? 1 : 3; }
cudaError_t launch_decode_tc(const DecodeArgs& a, int, bool, cudaStream_t) { g_dec = a; g_three++; return cudaSuccess; }
int decode_tc_ctas_per_sm(int) { return 1; }
}
#define CHECK(c) do { if (!(c)) { printf("FAIL case %d line %d: %s\n", cs, __LINE__, #c); return 1; } } while (0)

int main() {
  // two configs: q_len 1 in the one-kernel form, a verify block in three kernels
  const int B = 3, P = 16, maxp = 8;
  std::vector<int32_t> seq = {10, 50, 100};
  int cs = 0, checked = 0;
  for (int form = 0; form < 2; form++) {
    const int L = form == 0 ? 1 : 8;
    okc_attn_config c = {B, L, 16, 2, 64, P, 2048, maxp, B * maxp, 5e5f, 5.473f, 0.125f, 1.f};
    okc_plan_options o = {0, form == 0 ? OKC_PLAN_STEP_ONE_LAUNCH : 0, 0, 0};
    okc_attn_sizes z;
    CHECK(okc_attn_plan_sizes(&c, seq.data(), &o, &z) == OKC_OK);
    std::vector<uint8_t> ws(z.workspace_bytes + 256);
    uint8_t* w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws.data()) + 255) / 256 * 256);
    okc_attn_plan_t plan = nullptr;
    CHECK(okc_attn_plan(&c, seq.data(), &o, w, z.workspace_bytes, nullptr, &plan) == OKC_OK);
    const size_t T = (size_t)B * L, width = 2304;
    const size_t bytes[8] = {T * width * 2, T * 8, T * 8, B * 4, (B + 1) * 4, B * 4, (size_t)B * maxp * 4,
                             T * 1024 * 2};  // qkv, positions, cache_loc, cache_seqlens, cu_seqlens_q, seq_lens, page_table, out
    const size_t align[8] = {16, 8, 8, 4, 4, 4, 4, 16};
    // host buffers, device buffers and device aliases: distinct fake addresses
    alignas(64) static uint8_t arena[1 << 22];
    for (int mask = 0; mask < 256; mask++) {        // which of the 8 buffers are mapped
      for (int mis = 0; mis < 4; mis++, cs++) {     // misaligned alias of qkv (bit 0) / out (bit 1)
        g_alias.clear();
        g_copies.clear();
        g_syncs = g_fused = g_three = 0;
        const void* hostp[8];
        void* devp[8];
        const void* alias[8];
        size_t off = 0;
        for (int i = 0; i < 8; i++) {
          hostp[i] = arena + off; off += (bytes[i] + 64) / 64 * 64;
          devp[i] = arena + off; off += (bytes[i] + 64) / 64 * 64;
          const size_t shift = ((i == 0 && (mis & 1)) || (i == 7 && (mis & 2))) ? 8 : 0;
          alias[i] = arena + off + shift; off += (bytes[i] + 128) / 64 * 64;
          if (mask & (1 << i)) g_alias[hostp[i]] = alias[i];
        }
        okc_host_step io;
        io.qkv_host = hostp[0]; io.positions_host = (const int64_t*)hostp[1]; io.cache_loc_host = (const int64_t*)hostp[2];
        io.cache_seqlens_host = (const int32_t*)hostp[3]; io.cu_seqlens_q_host = (const int32_t*)hostp[4];
        io.seq_lens_host = (const int32_t*)hostp[5]; io.page_table_host = (const int32_t*)hostp[6];
        io.out_host = const_cast<void*>(hostp[7]);
        io.qkv = devp[0]; io.positions = (int64_t*)devp[1]; io.cache_loc = (int64_t*)devp[2];
        io.cache_seqlens = (int32_t*)devp[3]; io.cu_seqlens_q = (int32_t*)devp[4]; io.seq_lens = (int32_t*)devp[5];
        io.page_table = (int32_t*)devp[6]; io.out = devp[7];
        alignas(16) static uint8_t kc[64], vc[64], opart[64], lpart[64], rt[64], wgt[64];
        alignas(16) static float ks[4], vs[4];
        const okc_status st = okc_attn_step_host(plan, &io, kc, vc, ks, vs, (const float*)rt, 1 << 20, wgt, 1e-5f,
                                                 (float*)opart, (float*)lpart, nullptr);
        CHECK(st == OKC_OK);
        // inputs: which pointer reached the kernels, and which were copied
        const void* got[7];
        if (form == 0) {
          CHECK(g_fused == 1 && g_three == 0);
          got[0] = g_dec.qkv; got[1] = g_dec.positions; got[2] = g_dec.cache_loc; got[3] = g_dec.cache_seqlens;
          got[4] = g_dec.cu_seqlens_q; got[5] = g_dec.seq_lens; got[6] = g_dec.page_table;
        } else {
          CHECK(g_fused == 0 && g_three == 3);
          CHECK(g_prep.qkv == g_comb.qkv);
          got[0] = g_prep.qkv; got[1] = g_prep.positions; got[2] = g_prep.cache_loc; got[3] = g_dec.cache_seqlens;
          got[4] = g_dec.cu_seqlens_q; got[5] = g_dec.seq_lens; got[6] = g_dec.page_table;
        }
        size_t h2d = 0;
        for (int i = 0; i < 7; i++) {
          const bool inplace = (mask & (1 << i)) && (reinterpret_cast<uintptr_t>(alias[i]) % align[i] == 0);
          CHECK(got[i] == (inplace ? alias[i] : devp[i]));
          int n = 0;
          for (const auto& r : g_copies)
            if (r.src == hostp[i]) { n++; CHECK(r.dst == devp[i] && r.n == bytes[i] && r.kind == cudaMemcpyHostToDevice); }
          CHECK(n == (inplace ? 0 : 1));
          h2d += inplace ? 0 : 1;
        }
        // output: in place when mapped and aligned, else copied back once after the launch
        const bool out_inplace = (mask & 0x80) && (reinterpret_cast<uintptr_t>(alias[7]) % 16 == 0);
        const void* out_got = form == 0 ? (const void*)g_dec.out : (const void*)g_comb.out;
        CHECK(out_got == (out_inplace ? alias[7] : devp[7]));
        int nout = 0;
        for (const auto& r : g_copies)
          if (r.dst == hostp[7]) { nout++; CHECK(r.src == devp[7] && r.n == bytes[7] && r.kind == cudaMemcpyDeviceToHost); }
        CHECK(nout == (out_inplace ? 0 : 1));
        CHECK(g_copies.size() == h2d + (out_inplace ? 0 : 1));
        CHECK(g_syncs == 1);
        checked++;
      }
    }
    // a missing device buffer is refused before any copy
    {
      okc_host_step io;
      memset(&io, 0, sizeof io);
      g_copies.clear();
      CHECK(okc_attn_step_host(plan, &io, nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, 1e-5f, nullptr,
                               nullptr, nullptr) == OKC_ERR_INVALID);
      CHECK(g_copies.empty());
    }
    okc_attn_plan_destroy(plan);
  }
  printf("ok: %d routings checked\n", checked);
  return 0;
}
