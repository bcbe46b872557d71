// pa_common.cuh -- sm_103a building blocks shared by the paged-attention kernels:
// mbarrier + TMA (cp.async.bulk.tensor) staging, warp-level tensor-core mma,
// ldmatrix / movmatrix fragment moves, and the device error flag.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

constexpr int kTile = 16;                     // tokens per pipeline stage (one mma M/K tile)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kWaitSpins = 1u << 24;     // bound on every mbarrier wait loop

// unit info bits (low byte: valid tokens in the tile, 1..16)
constexpr int kFirstOfPair = 1 << 8;
constexpr int kLastOfPair = 1 << 9;
constexpr int kPieceStart = 1 << 10;
constexpr int kPieceEnd = 1 << 11;
constexpr int kHintShared = 1 << 12;   // tile lies in a prefix other sequences share
constexpr int kHintPrivate = 1 << 13;  // tile is private (hints given, not shared)
constexpr int kCascade = 1 << 14;      // the sequence's shared prefix is done by the cascade
constexpr int kInvalidPhys = -1;
// Quantised caches: P enters the PV mma as f16 times the ratio of the tile's V scale to
// the accumulator's.  The ratio stays <= 2^7, so that a weight <= 2^8 times it is well
// inside f16, and >= 2^-12, so that a tile's largest weights keep f16's normal range;
// outside that the accumulator is re-expressed in the tile's scale.
constexpr float kRatMax = 128.f;
constexpr float kRatMin = 1.f / 4096.f;

__device__ __forceinline__ void set_err(int32_t *flag, int bits) {
  if (flag) atomicOr(flag, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for the phase with the given parity; false if it never completed
// (after kSpins polls).
template <uint32_t kSpins = kWaitSpins>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kSpins; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ------------------------------------------------------------------ bulk copies

// 2D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The same with an L2 eviction-priority policy (from make_l2_policy) for the box.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int x,
                                                 int y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policies: keep a line as long as possible (data many readers will reuse) or
// evict it first (data read once).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Plain bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 4-byte asynchronous copy global -> shared, tracked by cp_async_arrive.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Both addresses 8-byte aligned.
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

// Make `bar` wait for this thread's outstanding cp.async copies (no count increment:
// the barrier's expected arrival count must include this arrival).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ------------------------------------------------------------------ programmatic dependent launch

// Wait until the grid this one depends on (the previous kernel in the stream) has
// completed and its writes are visible.  Returns at once when there is none.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next kernel in the stream be scheduled before this grid finishes.  The
// next kernel still runs pdl_wait() before it touches anything this grid touches.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ fragments

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ scalar helpers

__device__ __forceinline__ float ex2(float x) {  // 2^x on the SFU; ex2(-inf) = +0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// two E4M3 codes (low 16 bits) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
  uint32_t r;
  asm("{\n .reg .b16 c;\n cvt.u16.u32 c, %1;\n cvt.rn.f16x2.e4m3x2 %0, c;\n}\n"
      : "=r"(r)
      : "r"(codes));
  return r;
}

// two E4M3 codes (high 16 bits) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t codes) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, hi;\n}\n"
      : "=r"(r)
      : "r"(codes));
  return r;
}

// two E4M3 codes (low 16 bits) -> two floats, exact
// Four signed 4-bit codes stored as offset-binary nibbles at bits 4i.. and 4i+16..
// of w: returns {nibble i, nibble i + 4} as f16x2.  Even i: the nibbles masked into
// the low mantissa bits of 0x6400 (f16 1024 + u), minus 1032.  Odd i: masked in place
// at bits 4..7 (1024 + 16u), times 1/16 minus 72.  Both are exact, and i >= 2 reads
// w >> 8, so one shift serves four pairs.
__device__ __forceinline__ uint32_t int4_pair_f16(uint32_t w, int i) {
  uint32_t h;
  const uint32_t x = i >= 2 ? w >> 8 : w;
  const uint32_t mask = (i & 1) ? 0x00F000F0u : 0x000F000Fu;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(h) : "r"(x), "r"(mask), "r"(0x64006400u));
  const __half2 hv = *reinterpret_cast<const __half2 *>(&h);
  const __half2 v = (i & 1) ? __hfma2(hv, __floats2half2_rn(0.0625f, 0.0625f), __floats2half2_rn(-72.f, -72.f))
                            : __hsub2(hv, __floats2half2_rn(1032.f, 1032.f));
  return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t codes) {
  const uint32_t h = e4m3x2_to_f16x2(codes);
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// two floats -> two E4M3 codes (lo -> byte 0, hi -> byte 1), RNE, saturating
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b16 c;\n cvt.rn.satfinite.e4m3x2.f32 c, %1, %2;\n cvt.u32.u16 %0, c;\n}\n"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ int4 shfl_int4(int4 v, int src) {
  v.x = __shfl_sync(0xffffffffu, v.x, src);
  v.y = __shfl_sync(0xffffffffu, v.y, src);
  v.z = __shfl_sync(0xffffffffu, v.z, src);
  v.w = __shfl_sync(0xffffffffu, v.w, src);
  return v;
}

}  // namespace pa
