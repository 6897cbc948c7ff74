// arg_validation_host.cu — the launching entry points reject bad arguments on
// the host, before any launch, without a GPU: the plan is made with host fakes
// of its CUDA calls and the launchers are stubs that count launches. For each
// of okc_prepare_qkv, okc_attn_decode, okc_attn_combine_normgate and
// okc_attn_step: a valid call launches; every missing buffer, every pointer
// not aligned as its kernel loads it (16 bytes for vector loads, 8 for int64,
// 4 for int32 and float), a RoPE layer without positions or a usable table, a
// scaled cache without scales, and a bad eps return OKC_ERR_INVALID with no
// launch.
#include <cuda_runtime.h>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <vector>
static cudaError_t fake_memcpy(void* d, const void* s, size_t n, cudaMemcpyKind, cudaStream_t) {
  memcpy(d, s, n);
  return cudaSuccess;
}
static cudaError_t fake_get_device(int* d) { *d = 0; return cudaSuccess; }
static cudaError_t fake_attr(int* v, cudaDeviceAttr, int) { *v = 152; return cudaSuccess; }
#define cudaMemcpyAsync fake_memcpy
#define cudaGetDevice fake_get_device
#define cudaDeviceGetAttribute fake_attr
#include "okc_api.cu"
static int g_launches = 0;
namespace okc {
cudaError_t launch_prepare(const PrepareArgs&, bool, cudaStream_t) { g_launches++; return cudaSuccess; }
cudaError_t launch_decode(const DecodeArgs&, int, bool, cudaStream_t) { g_launches++; return cudaSuccess; }
cudaError_t launch_step_fused(const DecodeArgs&, int, bool, cudaStream_t) { g_launches++; return cudaSuccess; }
cudaError_t launch_step_fused_tc(const DecodeArgs&, int, bool, cudaStream_t) { g_launches++; return cudaSuccess; }
cudaError_t launch_combine(const CombineArgs&, bool, cudaStream_t) { g_launches++; return cudaSuccess; }
cudaError_t launch_rope_table(float, const float*, int32_t, float*, cudaStream_t) { return cudaSuccess; }
int decode_ctas_per_sm(int, bool tc, int) { return tc ? 1 : 3; }
cudaError_t launch_decode_tc(const DecodeArgs&, int, bool, cudaStream_t) { g_launches++; return cudaSuccess; }
int decode_tc_ctas_per_sm(int) { return 1; }
}

alignas(256) static uint8_t arena[1 << 16];
static uint8_t* buf(int i) { return arena + 1024 * i; }  // distinct 1 KB slots, 256-byte aligned

struct Args {  // every argument of okc_attn_step (the other calls take subsets)
  const void* qkv; const int64_t* positions; const int64_t* cache_loc; uint8_t* kc; uint8_t* vc;
  const float* ks; const float* vs; const float* rope; int32_t npos; const int32_t* pt; const int32_t* csl;
  const int32_t* cuq; const int32_t* sl; const void* w; float eps; float* op; float* lp; void* out; uint8_t* q8;
};
static Args valid() {
  return Args{buf(0), (const int64_t*)buf(1), (const int64_t*)buf(2), buf(3), buf(4), (const float*)buf(5),
              (const float*)buf(6), (const float*)buf(7), 4096, (const int32_t*)buf(8), (const int32_t*)buf(9),
              (const int32_t*)buf(10), (const int32_t*)buf(11), buf(12), 1e-5f, (float*)buf(13), (float*)buf(14),
              buf(15), buf(16)};
}
template <class T> static T off(T p, int bytes) { return (T)((const uint8_t*)p + bytes); }

int main() {
  int bad = 0, checked = 0;
  for (int L : {1, 8}) {
    okc_attn_config c = {3, L, 16, 2, 64, 16, 2048, 8, 24, 5e5f, 5.473f, 0.125f, 0.5f};  // RoPE, scaled
    okc_plan_options o = {0, L == 1 ? OKC_PLAN_STEP_ONE_LAUNCH : 0, 0, 0};
    int32_t seq[3] = {10, 50, 100};
    okc_attn_sizes z;
    if (okc_attn_plan_sizes(&c, seq, &o, &z) != OKC_OK) return 1;
    std::vector<uint8_t> ws(z.workspace_bytes + 256);
    uint8_t* w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws.data()) + 255) / 256 * 256);
    okc_attn_plan_t p = nullptr;
    if (okc_attn_plan(&c, seq, &o, w, z.workspace_bytes, nullptr, &p) != OKC_OK) return 1;
    auto prepare = [&](const Args& a) {
      return okc_prepare_qkv(p, a.qkv, a.positions, a.cache_loc, a.kc, a.vc, a.ks, a.vs, a.rope, a.npos, a.q8, nullptr);
    };
    auto decode = [&](const Args& a) {
      return okc_attn_decode(p, a.q8, a.kc, a.vc, a.ks, a.vs, a.pt, a.csl, a.cuq, a.sl, a.op, a.lp, nullptr);
    };
    auto combine = [&](const Args& a) {
      return okc_attn_combine_normgate(p, a.op, a.lp, a.qkv, a.w, a.eps, a.out, nullptr);
    };
    auto step = [&](const Args& a) {
      return okc_attn_step(p, a.qkv, a.positions, a.cache_loc, a.kc, a.vc, a.ks, a.vs, a.rope, a.npos, a.pt, a.csl,
                           a.cuq, a.sl, a.w, a.eps, a.op, a.lp, a.out, nullptr);
    };
    struct Call { const char* name; std::function<okc_status(const Args&)> f; };
    const Call calls[4] = {{"prepare", prepare}, {"decode", decode}, {"combine", combine}, {"step", step}};
    // the argument changes each call must refuse (by the arguments it takes)
    struct Bad { const char* what; std::function<void(Args&)> change; unsigned calls; };  // bit per call
    const unsigned P_ = 1, D_ = 2, C_ = 4, S_ = 8;
    const std::vector<Bad> bads = {
        {"qkv null", [](Args& a) { a.qkv = nullptr; }, P_ | C_ | S_},
        {"qkv +2", [](Args& a) { a.qkv = off(a.qkv, 2); }, P_ | C_ | S_},
        {"positions null", [](Args& a) { a.positions = nullptr; }, P_ | S_},
        {"positions +4", [](Args& a) { a.positions = off(a.positions, 4); }, P_ | S_},
        {"cache_loc null", [](Args& a) { a.cache_loc = nullptr; }, P_ | S_},
        {"cache_loc +4", [](Args& a) { a.cache_loc = off(a.cache_loc, 4); }, P_ | S_},
        {"k_cache null", [](Args& a) { a.kc = nullptr; }, P_ | D_ | S_},
        {"k_cache +8", [](Args& a) { a.kc = off(a.kc, 8); }, P_ | D_ | S_},
        {"v_cache +8", [](Args& a) { a.vc = off(a.vc, 8); }, P_ | D_ | S_},
        {"k_scale null", [](Args& a) { a.ks = nullptr; }, P_ | D_ | S_},
        {"v_scale +2", [](Args& a) { a.vs = off(a.vs, 2); }, P_ | D_ | S_},
        {"rope table null", [](Args& a) { a.rope = nullptr; }, P_ | S_},
        {"rope table +4", [](Args& a) { a.rope = off(a.rope, 4); }, P_ | S_},
        {"rope positions 0", [](Args& a) { a.npos = 0; }, P_ | S_},
        {"rope positions 2^21 + 1", [](Args& a) { a.npos = (1 << 21) + 1; }, P_ | S_},
        {"q_fp8 null", [](Args& a) { a.q8 = nullptr; }, P_ | D_},
        {"q_fp8 +8", [](Args& a) { a.q8 = off(a.q8, 8); }, P_ | D_},
        {"page_table null", [](Args& a) { a.pt = nullptr; }, D_ | S_},
        {"page_table +2", [](Args& a) { a.pt = off(a.pt, 2); }, D_ | S_},
        {"cache_seqlens +2", [](Args& a) { a.csl = off(a.csl, 2); }, D_ | S_},
        {"cu_seqlens_q null", [](Args& a) { a.cuq = nullptr; }, D_ | S_},
        {"cu_seqlens_q +2", [](Args& a) { a.cuq = off(a.cuq, 2); }, D_ | S_},
        {"seq_lens +2", [](Args& a) { a.sl = off(a.sl, 2); }, D_ | S_},
        {"o_partial null", [](Args& a) { a.op = nullptr; }, D_ | C_ | S_},
        {"o_partial +8", [](Args& a) { a.op = off(a.op, 8); }, D_ | C_ | S_},
        {"lse_partial null", [](Args& a) { a.lp = nullptr; }, D_ | C_ | S_},
        {"lse_partial +2", [](Args& a) { a.lp = off(a.lp, 2); }, D_ | C_ | S_},
        {"norm weight +8", [](Args& a) { a.w = off(a.w, 8); }, C_ | S_},
        {"out null", [](Args& a) { a.out = nullptr; }, C_ | S_},
        {"out +8", [](Args& a) { a.out = off(a.out, 8); }, C_ | S_},
        {"eps -1", [](Args& a) { a.eps = -1.f; }, C_ | S_},
        {"eps nan", [](Args& a) { a.eps = NAN; }, C_ | S_},
        {"eps inf", [](Args& a) { a.eps = INFINITY; }, C_ | S_},
    };
    for (int ci = 0; ci < 4; ci++) {
      g_launches = 0;
      if (calls[ci].f(valid()) != OKC_OK || g_launches == 0) {
        printf("FAIL L=%d %s: a valid call did not launch\n", L, calls[ci].name);
        bad++;
      }
      for (const Bad& b : bads) {
        if (!(b.calls & (1u << ci))) continue;
        Args a = valid();
        b.change(a);
        g_launches = 0;
        const okc_status st = calls[ci].f(a);
        checked++;
        if (st != OKC_ERR_INVALID || g_launches != 0) {
          printf("FAIL L=%d %s with %s: status %d, %d launches\n", L, calls[ci].name, b.what, (int)st, g_launches);
          bad++;
        }
      }
    }
    okc_attn_plan_destroy(p);
  }
  if (bad) return 1;
  printf("ok: %d refused argument sets, no launch\n", checked);
  return 0;
}
