// plan_update_host.cu — the planner's host logic without a GPU: the CUDA runtime
// calls that okc_attn_plan and okc_attn_plan_update make are replaced by host
// fakes (the "device" workspace is host memory, the upload a memcpy, and the
// page-locked staging allocation can be made to fail), and the library's own
// source is compiled in, so the real planner code runs on the host.
//
// Checks, over random configs, options and lengths: every in-place update
// uploads the same workspace head (work list, request table, arrival
// counters) and reports the same sizes as a fresh plan of the same lengths,
// within okc_attn_plan_max_sizes, and leaves the device error word (the
// header) as the kernels left it; a failed staging allocation, a length past
// the page table and a too-small workspace each leave the plan's sizes and
// workspace head unchanged, and the plan keeps working afterwards; a failed
// upload returns OKC_ERR_CUDA, and a later update makes the plan whole again;
// the default-option entry points (okc_attn_plan_create, _scratch_sizes,
// _workspace_size) agree with the general ones.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>
#include <vector>
static int g_fail_mallochost = 0, g_copies = 0, g_alloc_failures = 0, g_fail_memcpy = 0, g_upload_failures = 0;
static cudaError_t fake_memcpy_async(void* d, const void* s, size_t n, cudaMemcpyKind, cudaStream_t) {
  if (g_fail_memcpy) { g_fail_memcpy--; return cudaErrorLaunchFailure; }
  memcpy(d, s, n); g_copies++; return cudaSuccess;
}
static cudaError_t fake_malloc_host(void** p, size_t n) {
  if (g_fail_mallochost) { g_fail_mallochost--; *p = nullptr; return cudaErrorMemoryAllocation; }
  *p = malloc(n); return cudaSuccess;
}
static cudaError_t fake_free_host(void* p) { free(p); return cudaSuccess; }
static cudaError_t fake_event_sync(cudaEvent_t) { return cudaSuccess; }
static cudaError_t fake_event_create(cudaEvent_t* e, unsigned) { *e = (cudaEvent_t)0x1234; return cudaSuccess; }
static cudaError_t fake_event_record(cudaEvent_t, cudaStream_t) { return cudaSuccess; }
static cudaError_t fake_event_destroy(cudaEvent_t) { return cudaSuccess; }
static cudaError_t fake_get_device(int* d) { *d = 0; return cudaSuccess; }
static cudaError_t fake_attr(int* v, cudaDeviceAttr, int) { *v = 152; return cudaSuccess; }
#define cudaMemcpyAsync fake_memcpy_async
#define cudaMallocHost fake_malloc_host
#define cudaFreeHost fake_free_host
#define cudaEventSynchronize fake_event_sync
#define cudaEventCreateWithFlags fake_event_create
#define cudaEventRecord fake_event_record
#define cudaEventDestroy fake_event_destroy
#define cudaGetDevice fake_get_device
#define cudaDeviceGetAttribute fake_attr
#include "okc_api.cu"
namespace okc {
cudaError_t launch_prepare(const PrepareArgs&, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_decode(const DecodeArgs&, int, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_step_fused(const DecodeArgs&, int, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_step_fused_tc(const DecodeArgs&, int, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_combine(const CombineArgs&, bool, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_rope_table(float, const float*, int32_t, float*, cudaStream_t) { return cudaSuccess; }
int decode_ctas_per_sm(int, bool, int) { return 3; }
cudaError_t launch_decode_tc(const DecodeArgs&, int, bool, cudaStream_t) { return cudaSuccess; }
int decode_tc_ctas_per_sm(int) { return 1; }
}
#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); exit(1); } } while (0)

static size_t head_bytes(okc_attn_plan_t p) { return upload_bytes(p); }

int main(int argc, char** argv) {
  std::mt19937 g(7);
  int cases = 0;
  const int iters = argc > 1 ? atoi(argv[1]) : 1000;
  for (int it = 0; it < iters; it++) {
    const int L = std::vector<int>{1, 2, 8, 16, 100}[g() % 5];
    const int P = std::vector<int>{1, 8, 64}[g() % 3];
    const int window = std::vector<int>{0, 64, 2048}[g() % 3];
    const int B = std::vector<int>{1, 3, 64, 300}[g() % 4];
    const int maxctx = 1 + g() % 60000;
    const int max_pages = (maxctx + L + P - 1) / P + 1;
    okc_attn_config c = {B, L, 16, 2, 64, P, window, max_pages, B * max_pages, 5e5f, 5.473f, 0.125f, 1.f};
    okc_plan_options o = {0, 0, (int)(1 + g() % 3), 152, 0};
    if (g() % 4 == 0) o.chunk_keys = 16 + g() % 3000;
    // kind 0: a plan for its own step; 1: a fixed-capacity plan (max_context);
    // 2: per-request q lengths (varlen), new ones at every update
    const int kind = g() % 3;
    if (kind == 1) o.max_context = maxctx + L;
    auto lengths = [&](int hi) { std::vector<int32_t> v(B); for (auto& x : v) x = g() % (hi + 1); return v; };
    auto qlens = [&]() { std::vector<int32_t> v(B); for (auto& x : v) x = g() % (L + 1); return v; };
    std::vector<int32_t> ql = qlens();
    auto qp = [&]() -> const int32_t* { return kind == 2 ? ql.data() : nullptr; };
    auto update = [&](okc_attn_plan_t pl, const int32_t* sq) {
      return kind == 2 ? okc_attn_plan_update_varlen(pl, sq, qp(), nullptr) : okc_attn_plan_update(pl, sq, nullptr);
    };
    okc_attn_sizes bound;
    CHECK(okc_attn_plan_max_sizes(&c, maxctx + L, &o, &bound) == OKC_OK);
    // a plan in a workspace of the bound, and a fresh plan per step to compare with
    std::vector<uint8_t> ws(bound.workspace_bytes + 4096, 0xAB), ws2(bound.workspace_bytes + 4096, 0xCD);
    uint8_t* w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws.data()) + 255) / 256 * 256);
    uint8_t* w2 = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws2.data()) + 255) / 256 * 256);
    auto s0 = lengths(std::min(maxctx, 50));
    okc_attn_plan_t p = nullptr;
    CHECK(okc_attn_plan_varlen(&c, s0.data(), qp(), &o, w, bound.workspace_bytes, nullptr, &p) == OKC_OK);
    const size_t fixed_head = head_bytes(p);  // a fixed-capacity plan's offsets never move
    for (int step = 0; step < 6; step++) {
      auto s1 = lengths(maxctx);
      if (kind == 2) ql = qlens();
      okc_attn_sizes before;
      okc_attn_plan_get_sizes(p, &before);
      std::vector<uint8_t> head_before(w, w + head_bytes(p));
      const int mode = g() % 5;
      if (mode == 0) {  // a failed staging allocation leaves everything as it was
        g_fail_mallochost = 1;
        // force a (re)allocation: only the first update allocates, or a larger one
        okc_status st = update(p, s1.data());
        if (st == OKC_ERR_CUDA) {
          g_alloc_failures++;
          okc_attn_sizes after;
          okc_attn_plan_get_sizes(p, &after);
          CHECK(memcmp(&before, &after, sizeof before) == 0);
          CHECK(memcmp(head_before.data(), w, head_before.size()) == 0);
          CHECK(head_bytes(p) == head_before.size());
        }
        g_fail_mallochost = 0;
      } else if (mode == 2) {  // the upload itself fails: reported, and the next update repairs the plan
        g_fail_memcpy = 1;
        CHECK(update(p, s1.data()) == OKC_ERR_CUDA);
        g_fail_memcpy = 0;
        g_upload_failures++;
      } else if (mode == 1) {  // a length past the page table: refused, plan unchanged
        auto bad = s1;
        const int i = (int)(g() % B);
        bad[i] = max_pages * P;  // + its q length > max_pages * P
        if (kind == 2 && ql[i] == 0) ql[i] = 1;
        CHECK(update(p, bad.data()) == OKC_ERR_INVALID);
        okc_attn_sizes after;
        okc_attn_plan_get_sizes(p, &after);
        CHECK(memcmp(&before, &after, sizeof before) == 0);
        CHECK(memcmp(head_before.data(), w, head_before.size()) == 0);
      }
      // bits the kernels set in the error word survive the update
      const uint32_t err_word = (uint32_t)g() | 1u;
      memcpy(w, &err_word, sizeof err_word);
      CHECK(update(p, s1.data()) == OKC_OK);
      CHECK(memcmp(w, &err_word, sizeof err_word) == 0);
      if (kind == 1) CHECK(head_bytes(p) == fixed_head);
      okc_attn_plan_t q = nullptr;
      CHECK(okc_attn_plan_varlen(&c, s1.data(), qp(), &o, w2, bound.workspace_bytes, nullptr, &q) == OKC_OK);
      okc_attn_sizes zp, zq;
      okc_attn_plan_get_sizes(p, &zp);
      okc_attn_plan_get_sizes(q, &zq);
      if (kind == 1) zq.step_kernels = zp.step_kernels;  // a fixed-capacity plan keeps its form
      CHECK(memcmp(&zp, &zq, sizeof zp) == 0);
      int32_t live = -1;
      memcpy(&live, w + okc::kWsCount, sizeof live);
      CHECK(live == zp.num_work);
      CHECK(head_bytes(p) == head_bytes(q));
      // the uploaded heads are identical past the error word (the fresh plan zeroed its own)
      CHECK(memcmp(w + okc::kWsCount, w2 + okc::kWsCount, head_bytes(p) - okc::kWsCount) == 0);
      memset(w, 0, sizeof err_word);
      CHECK(zp.workspace_bytes <= bound.workspace_bytes && zp.o_partial_bytes <= bound.o_partial_bytes &&
            zp.num_work <= bound.num_work);
      okc_attn_plan_destroy(q);
      cases++;
    }
    // a workspace too small for the next step: refused, plan unchanged
    {
      if (kind != 0) {  // (the refusal below is for plans sized to their own step)
        okc_attn_plan_destroy(p);
        continue;
      }
      auto big = std::vector<int32_t>(B, maxctx);
      okc_attn_sizes zb;
      CHECK(okc_attn_plan_sizes(&c, big.data(), &o, &zb) == OKC_OK);
      okc_attn_sizes cur;
      okc_attn_plan_get_sizes(p, &cur);
      okc_attn_plan_t small = nullptr;
      std::vector<int32_t> tiny(B, 0);
      okc_attn_sizes zt;
      CHECK(okc_attn_plan_sizes(&c, tiny.data(), &o, &zt) == OKC_OK);
      std::vector<uint8_t> ws3(zt.workspace_bytes + 512);
      uint8_t* w3 = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws3.data()) + 255) / 256 * 256);
      CHECK(okc_attn_plan(&c, tiny.data(), &o, w3, zt.workspace_bytes, nullptr, &small) == OKC_OK);
      std::vector<uint8_t> h(w3, w3 + head_bytes(small));
      if (zb.workspace_bytes > zt.workspace_bytes) {
        CHECK(okc_attn_plan_update(small, big.data(), nullptr) == OKC_ERR_WORKSPACE);
        okc_attn_sizes a;
        okc_attn_plan_get_sizes(small, &a);
        CHECK(memcmp(&a, &zt, sizeof a) == 0);
        CHECK(memcmp(h.data(), w3, h.size()) == 0);
        CHECK(okc_attn_plan_update(small, tiny.data(), nullptr) == OKC_OK);
        CHECK(memcmp(h.data(), w3, h.size()) == 0);
      }
      okc_attn_plan_destroy(small);
    }
    okc_attn_plan_destroy(p);
  }
  CHECK(g_alloc_failures > 0 && g_upload_failures > 0);
  // the default-option forms: okc_attn_plan_create is okc_attn_plan with no
  // options, okc_attn_plan_scratch_sizes its sizes, okc_attn_plan_workspace_size
  // the workspace bound of okc_attn_plan_max_sizes (152 SMs, the stubs' occupancy)
  for (int it = 0; it < 200; it++) {
    const int L = std::vector<int>{1, 8}[g() % 2];
    const int B = 1 + g() % 300, maxctx = 1 + g() % 40000, max_pages = maxctx + L + 1;
    okc_attn_config c = {B, L, 16, 2, 64, 1, (g() % 2) ? 2048 : 0, max_pages, B * max_pages, 5e5f, 5.473f, 0.125f,
                         1.f};
    std::vector<int32_t> s(B);
    for (auto& x : s) x = g() % (maxctx + 1);
    size_t wsb = 0;
    okc_attn_sizes bound, z1, z2;
    CHECK(okc_attn_plan_workspace_size(&c, maxctx + L, &wsb) == OKC_OK);
    CHECK(okc_attn_plan_max_sizes(&c, maxctx + L, nullptr, &bound) == OKC_OK && bound.workspace_bytes == wsb);
    std::vector<uint8_t> a(wsb + 256), b2(wsb + 256);
    uint8_t* wa = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(a.data()) + 255) / 256 * 256);
    uint8_t* wb = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(b2.data()) + 255) / 256 * 256);
    okc_attn_plan_t p1 = nullptr, p2 = nullptr;
    CHECK(okc_attn_plan_create(&c, s.data(), wa, wsb, nullptr, &p1) == OKC_OK);
    CHECK(okc_attn_plan(&c, s.data(), nullptr, wb, wsb, nullptr, &p2) == OKC_OK);
    CHECK(okc_attn_plan_scratch_sizes(p1, &z1) == OKC_OK && okc_attn_plan_get_sizes(p2, &z2) == OKC_OK);
    CHECK(memcmp(&z1, &z2, sizeof z1) == 0 && z1.workspace_bytes <= wsb && z1.num_work <= bound.num_work);
    CHECK(memcmp(wa, wb, head_bytes(p1)) == 0);
    okc_attn_plan_destroy(p1);
    okc_attn_plan_destroy(p2);
  }
  printf("ok: %d updates compared with fresh plans, %d failed staging allocations, %d failed uploads\n", cases,
         g_alloc_failures, g_upload_failures);
}
