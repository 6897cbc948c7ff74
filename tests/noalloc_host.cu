// noalloc_host.cu — okc_attn_decode_combine_noalloc's host side without a GPU:
// its CUDA runtime calls are replaced by host fakes (the static device array is
// host memory, uploads are memcpys, the device has 152 SMs) and the launchers by
// stubs that record their arguments. Checks, over random configs and lengths:
// the uploaded work list and request table are the plan's split (the same
// function, in the same launch order), the decode launch covers every item
// with pointers into the array, the scratch layout stays inside the array, and
// the documented limits (2048 requests, 4096 items, 8 MiB) give
// OKC_ERR_WORKSPACE exactly when they are exceeded.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <random>
#include <vector>
static std::vector<unsigned char> g_array(8u << 20);
struct Copy { size_t off, n; };
static std::vector<Copy> g_copies;
static cudaError_t fake_memcpy(void* d, const void* s, size_t n, cudaMemcpyKind, cudaStream_t) {
  memcpy(d, s, n);
  g_copies.push_back({(size_t)((unsigned char*)d - g_array.data()), n});
  return cudaSuccess;
}
static cudaError_t fake_get_device(int* d) { *d = 0; return cudaSuccess; }
static cudaError_t fake_attr(int* v, cudaDeviceAttr, int) { *v = 152; return cudaSuccess; }
static cudaError_t fake_symaddr(void** p) { *p = g_array.data(); return cudaSuccess; }
#define cudaMemcpyAsync fake_memcpy
#define cudaGetDevice fake_get_device
#define cudaDeviceGetAttribute fake_attr
#define cudaGetSymbolAddress(p, sym) fake_symaddr(p)
#include "okc_api.cu"
#include "noalloc.cu"
static okc::DecodeArgs g_dec;
static okc::CombineArgs g_comb;
static int g_W = -1, g_launches = 0;
namespace okc {
cudaError_t launch_prepare(const PrepareArgs&, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_decode(const DecodeArgs& a, int nw, bool, cudaStream_t) { g_dec = a; g_W = nw; g_launches++; return cudaSuccess; }
cudaError_t launch_step_fused(const DecodeArgs&, int, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_step_fused_tc(const DecodeArgs&, int, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_combine(const CombineArgs& a, bool, cudaStream_t) { g_comb = a; g_launches++; return cudaSuccess; }
cudaError_t launch_rope_table(float, const float*, int32_t, float*, cudaStream_t) { return cudaSuccess; }
int decode_ctas_per_sm(int, bool tc, int) { return tc ? 1 : 3; }
cudaError_t launch_decode_tc(const DecodeArgs&, int, bool, cudaStream_t) { return cudaSuccess; }
int decode_tc_ctas_per_sm(int) { return 1; }
}
#define CHECK(c) do { if (!(c)) { printf("FAIL case %d line %d: %s\n", it, __LINE__, #c); return 1; } } while (0)

int main(int argc, char** argv) {
  std::mt19937 g(11);
  alignas(16) static unsigned char dummy[64];
  const unsigned char* base = g_array.data();
  int ok = 0, refused = 0;
  const int iters = argc > 1 ? atoi(argv[1]) : 2000;
  for (int it = 0; it < iters; it++) {
    const int L = std::vector<int>{1, 2, 8, 12, 16}[g() % 5];
    const int P = std::vector<int>{1, 8, 64}[g() % 3];
    const int window = std::vector<int>{0, 64, 2048}[g() % 3];
    const int B = std::vector<int>{1, 3, 64, 300, 2048, 2049}[g() % 6];
    const int maxctx = 1 + g() % (g() % 2 ? 3000 : 140000);
    const int max_pages = (maxctx + L + P - 1) / P + 1;
    okc_attn_config c = {B, L, 16, 2, 64, P, window, max_pages, B * max_pages, 5e5f, 5.473f, 0.125f, 1.f};
    std::vector<int32_t> seq(B);
    for (auto& x : seq) x = g() % (maxctx + 1);
    g_copies.clear();
    g_W = -1;
    g_launches = 0;
    const okc_status st = okc_attn_decode_combine_noalloc(
        &c, seq.data(), dummy, dummy, dummy, nullptr, nullptr, (const int32_t*)dummy, (const int32_t*)dummy,
        (const int32_t*)dummy, nullptr, dummy, nullptr, 1e-5f, dummy, nullptr);
    // the plan's split for the same device
    okc::SplitResult want;
    const bool tc = L >= 2;
    CHECK(okc::make_splits(&c, seq.data(), nullptr, nullptr, 152 * (tc ? 1 : 3), &want) == OKC_OK);
    const int S = tc ? std::min(L, 16) : 1;  // (q_len past 8: the per-KV-head form, blocks of up to 16)
    CHECK(want.S == S);
    const size_t W = want.work.size(), NB = want.blocks.size(), rows = (size_t)S * 16;
    CHECK(NB == (size_t)B * ((L + S - 1) / S));
    const size_t off_req = (W * sizeof(okc::WorkItem) + 255) / 256 * 256;
    const size_t off_lse = off_req + (NB * sizeof(okc::BlockInfo) + 255) / 256 * 256;
    const size_t off_o = off_lse + (W * rows * 4 + 255) / 256 * 256;
    const size_t need = off_o + W * rows * 64 * 4;
    const bool over = B > 2048 || W > 4096 || need > (8u << 20);
    if (over) {
      CHECK(st == OKC_ERR_WORKSPACE && g_launches == 0);
      refused++;
      continue;
    }
    CHECK(st == OKC_OK);
    CHECK(g_copies.size() == 2 && g_copies[0].off == 0 && g_copies[0].n == W * sizeof(okc::WorkItem));
    CHECK(g_copies[1].off == off_req && g_copies[1].n == NB * sizeof(okc::BlockInfo));
    CHECK(memcmp(base, want.work.data(), g_copies[0].n) == 0);
    CHECK(memcmp(base + off_req, want.blocks.data(), g_copies[1].n) == 0);
    CHECK(g_launches == 2 && g_W == (int)W && g_dec.tc == (tc ? 1 : 0) && g_dec.S == S && g_comb.S == S);
    CHECK((const unsigned char*)g_dec.work == base && (const unsigned char*)g_comb.blk == base + off_req);
    CHECK((const unsigned char*)g_dec.lse_part == base + off_lse && (const unsigned char*)g_dec.o_part == base + off_o);
    CHECK(g_comb.o_part == g_dec.o_part && g_comb.lse_part == g_dec.lse_part && g_comb.nblocks == (int)NB);
    CHECK(g_comb.T == B * L && g_dec.T == B * L && g_dec.live_work == nullptr);
    ok++;
  }
  if (ok == 0 || refused == 0) { printf("FAIL: %d run, %d refused\n", ok, refused); return 1; }
  printf("ok: %d calls checked against the plan's split, %d refused over the limits\n", ok, refused);
  return 0;
}
