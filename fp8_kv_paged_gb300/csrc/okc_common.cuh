// okc_common.cuh — device helpers shared by the sm_103a kernels of the paged-FP8
// gated attention block: inline-PTX wrappers for cp.async, ldmatrix, movmatrix,
// the warp-level FP8/FP16 tensor-core mma, programmatic dependent launch, and
// the bf16 / E4M3 conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "okc_attn.h"

namespace okc {

constexpr int kHeadDim = 64;
constexpr int kNumQHeads = 16;
constexpr int kNumKvHeads = 2;
constexpr int kGroup = kNumQHeads / kNumKvHeads;  // q heads served by one KV head
constexpr int kRowBytes = kNumKvHeads * kHeadDim;  // one cache row (both KV heads), E4M3
constexpr int kQkvWidth = (2 * kNumQHeads + 2 * kNumKvHeads) * kHeadDim;
constexpr int kGateCol = (kNumQHeads + 2 * kNumKvHeads) * kHeadDim;
constexpr int kRopePositionsMax = 1 << 21;
constexpr int kMaxQLen = 1 << 16;  // new tokens of one request in one step
constexpr float kRmsEps = 1.0e-5f;

// ------------------------------------------------------------ launch control
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor still runs;
// griddepcontrol.wait blocks until the predecessor grid has completed and its
// memory is visible. Both are no-ops when the launch carried no attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Fetch the 128-byte line holding `p` into L2 (a hint; nothing is returned).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// --------------------------------------------------------------- async copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy through L2 only; src_bytes 0 fills zeros and
// reads nothing (used for masked or invalid rows).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Wait until every cp.async this thread issued has completed (wait_all also
// covers copies never committed to a group, as the mbarrier-tracked ones here).
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
// Phase-tracked shared-memory barriers. Every wait is bounded by the caller
// (mbar_wait returns false after `limit` polls) so that a lost completion can
// never hang the GPU.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase of parity `parity` (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of parity `parity` to complete. Bounded in time: a poll of
// try_wait may suspend the thread for a hardware-defined while, so a poll count
// alone does not bound the wait; it gives up (returns false) once it has polled
// kWaitMinPolls times and kWaitNs have passed since its first failed poll (the
// poll count keeps a kernel that was preempted mid-wait from giving up early).
constexpr uint32_t kWaitMinPolls = 1u << 12;
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s; a tile lands within microseconds
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; i++) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= kWaitMinPolls && global_ns() - t0 > limit_ns) return false;
  }
}
// Fetch a TMA tensor map (a __grid_constant__ kernel parameter) into the
// descriptor cache ahead of its first use.
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// Arrive on mbarrier `bar` and add `bytes` to the transaction count its
// current phase waits for (the bytes of the bulk copies that complete on it).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
// TMA: the box at (x, y) of the 2-D tensor map `tmap` (a kernel parameter)
// into shared memory at `dst`; completes `bytes` of transactions on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Arrive on mbarrier `bar` once every cp.async this thread has issued so far has
// completed (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
// Named barrier over the first `threads` threads of the CTA (id != 0).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// ----------------------------------------------------------- shared loads
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// Transpose an 8x8 b16 matrix held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

// Store four 8x8 b16 matrices transposed: register j of lane l holds elements
// (l/4, 2(l%4)) and (l/4, 2(l%4)+1) of matrix j; lane 8j+c gives the address of
// row c of the stored (transposed) matrix j, i.e. column c of the register
// matrix, 16 contiguous bytes.
__device__ __forceinline__ void stsm_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(r0),
               "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

// ---------------------------------------------- 5th-generation tensor cores
// tcgen05: the MMA reads A and B from shared memory through matrix
// descriptors, accumulates in tensor memory (TMEM: 128 lanes x 512 columns of
// 32 bits per SM), and signals completion on an mbarrier (tcgen05.commit).
// Shared-memory operands here use the no-swizzle K-major layout: 8-row x
// 16-byte core matrices (128 contiguous bytes, rows 16 bytes apart); core
// matrices adjacent along K are LBO bytes apart, 8-row groups SBO bytes apart.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);  // descriptor version 1, no swizzle
}
// The same for the 128-byte-swizzle K-major layout that a TMA tile load with
// 128-byte swizzling writes: rows of 128 bytes whose 16-byte chunks are XORed
// with the row index mod 8, 8-row groups `sbo` bytes apart, the tile
// 1024-byte aligned; the leading offset is unused. A step along K inside the
// 128-byte row adds its byte offset to saddr (the swizzle applies to the
// resulting address).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
         (1ull << 46) | (2ull << 61);  // descriptor version 1, layout 2 = 128-byte swizzle
}
// Instruction descriptor: f32 accumulator, A/B format code `ab` (kind::f16: 0 =
// f16; kind::f8f6f4: 0 = E4M3), both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc(uint32_t ab, int M, int N) {
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// kind::f16 MMA (f16 x f16 -> f32 in TMEM) with A read from tensor memory (lane
// = row, 32-bit columns holding two f16 values each, lower K index in the low
// half) and B from shared memory.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// kind::f8f6f4 MMA (E4M3 x E4M3 -> f32 in TMEM) with A read from tensor memory
// (lane = row, 32-bit columns holding four 8-bit values each, lower K index in
// the low byte: K = 32 per instruction spans 8 columns) and B from shared memory.
__device__ __forceinline__ void umma_f8_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive once on mbarrier `bar` when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes of this thread become visible to the async
// proxy (the tensor core's operand reads).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Warp-wide TMEM allocation of `ncols` columns; the address lands in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_saddr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_saddr), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// 32 columns of this warp's 32 TMEM lanes (one lane per thread) into registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"  // in the same statement: the outputs are valid after it
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// One column of this warp's 32 TMEM lanes (one value per thread).
// 16 columns of this warp's 32 TMEM lanes (one per thread), waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
// The same store without waiting for it (a later tcgen05.wait::st, as in
// tmem_st1 or tmem_st32u, covers it).
__device__ __forceinline__ void tmem_st16_async(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
// 32 words into 32 columns of this warp's 32 TMEM lanes; returns once stored.
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v))
      : "memory");
}

// ------------------------------------------------------------ tensor cores
// D(16x8,f32) += A(16x32,e4m3,row) * B(32x8,e4m3,col)
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D(16x8,f32) += A(16x16,f16,row) * B(16x8,f16,col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------- conversions
// Two E4M3 codes (low byte = first element) -> f16x2 (low half = first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}
// Four E4M3 codes (v, code i in byte i) -> two f16 pairs: lo holds codes 0, 1,
// hi codes 2, 3 (the lower code in the lower half), exact; one cvt per pair
// straight from the halves of v.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(v));
}
// Two floats -> two E4M3 codes, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later):
// exact, so a tree of them gives the same maximum as one of fmaxf.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Two float32 FMAs or products in one instruction (the f32x2 forms, sm_100
// and later): (a0, a1) * b + c and (a0, a1) * b, each lane rounded once to
// nearest, as __fmaf_rn and __fmul_rn.
__device__ __forceinline__ void ffma2(float a0, float a1, float b, float c, float& y0, float& y1) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n"
      " mov.b64 rc, {%5, %5};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(y0), "=f"(y1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void fmul2(float a0, float a1, float b, float& y0, float& y1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(y0), "=f"(y1)
      : "f"(a0), "f"(a1), "f"(b));
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ RMS inverse
// inv = float32 rounding of 1 / sqrt(sum(x^2) / 64 + eps) for one head of 64
// bf16 values spread over LPH lanes (N values each; the LPH lanes of a head are
// consecutive and LPH-aligned). Float32 arithmetic, exact in the result:
//  - squares of bf16 values are exact in float32; the sum is accumulated
//    error-free into a float pair (hi, lo) (TwoSum), relative error <= ~2^-42;
//  - inv = rsqrtf seed + one float-float Newton correction, rounded once;
//  - if the correction leaves the value within 2^-40 (relative) of a float32
//    rounding midpoint, or anything overflowed, the whole warp recomputes in
//    double precision (sum of squares exact in double, IEEE sqrt and divide),
//    so the result is the correctly rounded value in every case. The double
//    path runs for about one head in 2^15.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

template <int LPH, int N>
__device__ __forceinline__ float rms_inverse(const float (&x)[N], float eps) {
  float h = 0.f, l = 0.f;
#pragma unroll
  for (int i = 0; i < N; i++) {
    float s, e;
    two_sum(h, __fmul_rn(x[i], x[i]), s, e);
    h = s;
    l = __fadd_rn(l, e);
  }
#pragma unroll
  for (int o = 1; o < LPH; o <<= 1) {
    const float ho = __shfl_xor_sync(0xffffffffu, h, o), lo = __shfl_xor_sync(0xffffffffu, l, o);
    float s, e;
    two_sum(h, ho, s, e);
    h = s;
    l = __fadd_rn(__fadd_rn(l, lo), e);
  }
  // m = S/64 + eps as a float pair (the scalings by 1/64 are exact)
  float mh, ml;
  {
    float s, e;
    two_sum(__fmul_rn(h, 1.f / 64.f), eps, s, e);
    mh = s;
    ml = __fadd_rn(__fmul_rn(l, 1.f / 64.f), e);
    const float t = __fadd_rn(mh, ml);  // renormalise
    ml = __fsub_rn(ml, __fsub_rn(t, mh));
    mh = t;
  }
  const float y0 = rsqrtf(mh);
  // e = 1 - m*y0^2 with products split exactly (fma), corrections in float
  const float a = __fmul_rn(y0, y0), b = __fmaf_rn(y0, y0, -a);
  const float c = __fmul_rn(mh, a), d = __fmaf_rn(mh, a, -c);
  const float e = __fsub_rn(__fsub_rn(__fsub_rn(__fsub_rn(1.f, c), d), __fmul_rn(mh, b)), __fmul_rn(ml, a));
  // 1/sqrt(m) = y0 * (1 - e)^(-1/2) = y0 * (1 + e/2 + 3e^2/8 + ...)
  const float corr = __fmul_rn(y0, __fmaf_rn(__fmul_rn(0.375f, e), e, __fmul_rn(0.5f, e)));
  const float r = __fadd_rn(y0, corr);
  const float z = __fsub_rn(corr, __fsub_rn(r, y0));  // what the rounding dropped
  const float nb = z >= 0.f ? __int_as_float(__float_as_int(r) + 1) : __int_as_float(__float_as_int(r) - 1);
  const float half = 0.5f * fabsf(__fsub_rn(nb, r));
  const bool amb = !(mh > 0x1p-100f) || !isfinite(mh) || !isfinite(r) ||
                   fabsf(__fsub_rn(fabsf(z), half)) <= __fmul_rn(r, 0x1p-40f);
  if (!__any_sync(0xffffffffu, amb)) return r;
  double ss = 0.0;
#pragma unroll
  for (int i = 0; i < N; i++) ss = fma((double)x[i], (double)x[i], ss);
#pragma unroll
  for (int o = 1; o < LPH; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return (float)(1.0 / sqrt(ss / 64.0 + (double)eps));
}

__device__ __forceinline__ void set_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

}  // namespace okc
