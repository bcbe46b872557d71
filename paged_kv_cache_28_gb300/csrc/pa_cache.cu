// pa_cache.cu -- the slot-mapped cache write (reshape_and_cache).
//
// "Taming the Token Torrent", "How Paging Works in the LLM Context" / "The Block
// Table Logic": each step's new K/V vectors go to slot s = block * bs + offset,
// i.e. row (s / bs, s % bs) of the block pool [nblocks, bs, Hkv, D].
// FP8 pools follow "KV Cache Engineering for LLM Serving", section 8 (absmax
// scale, divide, round, clip), with one fp32 scale per (block, KV head) that
// tracks the block's absmax and re-encodes earlier rows when it grows.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// BF16: one CTA per token, 16-byte vector copies of the token's Hkv*D row.
__global__ void __launch_bounds__(128) cache_write_bf16_kernel(
    const uint4 *k_new, const uint4 *v_new, uint4 *k_pool, uint4 *v_pool,
    const int64_t *slot_mapping, int bs, int nblocks, int row16, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(nblocks) * bs) {
    if (threadIdx.x == 0) set_err(err, PA_DEVERR_SLOT);
    return;
  }
  const size_t dst = static_cast<size_t>(slot) * row16;
  const size_t src = static_cast<size_t>(t) * row16;
  for (int i = threadIdx.x; i < row16; i += blockDim.x) {
    k_pool[dst + i] = k_new[src + i];
    v_pool[dst + i] = v_new[src + i];
  }
}

// FP8 (D = 128): one CTA per token, one warp per (KV head, K or V); each lane owns
// four consecutive elements of the head vector.
__global__ void __launch_bounds__(256) cache_write_fp8_kernel(
    const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_pool, uint8_t *v_pool,
    float *k_scale, float *v_scale, const int64_t *slot_mapping, int T, int Hkv, int bs,
    int nblocks, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  constexpr int D = 128;
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(nblocks) * bs) {
    if (threadIdx.x == 0) set_err(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / bs;
  const int off = static_cast<int>(slot - blk * bs);
  // two tokens of this call in one block would race on its scale: skip both
  int clash = 0;
  for (int u = threadIdx.x; u < T; u += blockDim.x) {
    const int64_t o = slot_mapping[u];
    if (u != t && o >= 0 && o / bs == blk) clash = 1;
  }
  if (__syncthreads_or(clash)) {
    if (threadIdx.x == 0) set_err(err, PA_DEVERR_FP8_CONFLICT);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int job = warp; job < 2 * Hkv; job += blockDim.x >> 5) {
    const int h = job >> 1;
    const bool is_v = job & 1;
    const uint16_t *x = (is_v ? v_new : k_new) + (static_cast<size_t>(t) * Hkv + h) * D;
    uint8_t *pool = is_v ? v_pool : k_pool;
    float *scale = (is_v ? v_scale : k_scale) + blk * Hkv + h;
    const uint2 raw = *reinterpret_cast<const uint2 *>(x + lane * 4);
    const float v0 = bf16_lo(raw.x), v1 = bf16_hi(raw.x), v2 = bf16_lo(raw.y), v3 = bf16_hi(raw.y);
    float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float cand = __fdiv_rn(amax, 448.0f);
    const float old = *scale;
    const float s_new = (off == 0 || cand > old) ? cand : old;
    if (off > 0 && s_new > old) {
      for (int r = 0; r < off; ++r) {
        uint32_t *row = reinterpret_cast<uint32_t *>(
            pool + ((blk * bs + r) * Hkv + h) * static_cast<int64_t>(D) + lane * 4);
        const uint32_t c = *row;
        uint32_t nc = 0;
        if (s_new != 0.f) {
          const float2 lo = e4m3x2_to_float2(c), hi = e4m3x2_to_float2(c >> 16);
          nc = f32x2_to_e4m3x2(__fdiv_rn(__fmul_rn(lo.x, old), s_new),
                               __fdiv_rn(__fmul_rn(lo.y, old), s_new)) |
               (f32x2_to_e4m3x2(__fdiv_rn(__fmul_rn(hi.x, old), s_new),
                                __fdiv_rn(__fmul_rn(hi.y, old), s_new))
                << 16);
        }
        *row = nc;
      }
    }
    uint32_t code = 0;
    if (s_new != 0.f)
      code = f32x2_to_e4m3x2(__fdiv_rn(v0, s_new), __fdiv_rn(v1, s_new)) |
             (f32x2_to_e4m3x2(__fdiv_rn(v2, s_new), __fdiv_rn(v3, s_new)) << 16);
    *reinterpret_cast<uint32_t *>(pool + ((blk * bs + off) * Hkv + h) * static_cast<int64_t>(D) +
                                  lane * 4) = code;
    __syncwarp();
    if (lane == 0) *scale = s_new;
  }
}

// 4-bit (D = 128): the FP8 kernel's structure with codes clip(rint(x / scale), -7, 7)
// stored as offset-binary nibbles; each lane owns four consecutive elements (two bytes).
__device__ __forceinline__ uint32_t int4_code(float x, float scale) {
  if (scale == 0.f) return 8u;
  const float c = fminf(fmaxf(rintf(__fdiv_rn(x, scale)), -7.f), 7.f);
  return static_cast<uint32_t>(static_cast<int>(c) + 8);
}

__global__ void __launch_bounds__(256) cache_write_int4_kernel(
    const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_pool, uint8_t *v_pool,
    float *k_scale, float *v_scale, const int64_t *slot_mapping, int T, int Hkv, int bs,
    int nblocks, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  constexpr int D = 128, ROWB = D / 2;
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(nblocks) * bs) {
    if (threadIdx.x == 0) set_err(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / bs;
  const int off = static_cast<int>(slot - blk * bs);
  int clash = 0;
  for (int u = threadIdx.x; u < T; u += blockDim.x) {
    const int64_t o = slot_mapping[u];
    if (u != t && o >= 0 && o / bs == blk) clash = 1;
  }
  if (__syncthreads_or(clash)) {
    if (threadIdx.x == 0) set_err(err, PA_DEVERR_FP8_CONFLICT);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int job = warp; job < 2 * Hkv; job += blockDim.x >> 5) {
    const int h = job >> 1;
    const bool is_v = job & 1;
    const uint16_t *x = (is_v ? v_new : k_new) + (static_cast<size_t>(t) * Hkv + h) * D;
    uint8_t *pool = is_v ? v_pool : k_pool;
    float *scale = (is_v ? v_scale : k_scale) + blk * Hkv + h;
    const uint2 raw = *reinterpret_cast<const uint2 *>(x + lane * 4);
    const float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float cand = __fdiv_rn(amax, 7.0f);
    const float old = *scale;
    const float s_new = (off == 0 || cand > old) ? cand : old;
    if (off > 0 && s_new > old) {
      for (int r = 0; r < off; ++r) {
        uint16_t *row = reinterpret_cast<uint16_t *>(
            pool + ((blk * bs + r) * Hkv + h) * static_cast<int64_t>(ROWB) + lane * 2);
        const uint32_t c = *row;
        uint32_t nc = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float restored =
              __fmul_rn(static_cast<float>(static_cast<int>((c >> (4 * e)) & 0xF) - 8), old);
          nc |= int4_code(restored, s_new) << (4 * e);
        }
        *row = static_cast<uint16_t>(nc);
      }
    }
    uint32_t code = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) code |= int4_code(v[e], s_new) << (4 * e);
    *reinterpret_cast<uint16_t *>(pool + ((blk * bs + off) * Hkv + h) * static_cast<int64_t>(ROWB) +
                                  lane * 2) = static_cast<uint16_t>(code);
    __syncwarp();
    if (lane == 0) *scale = s_new;
  }
}

pa_status run_reshape_and_cache(const pa_shape &s, const void *k_new, const void *v_new,
                                void *k_pool, void *v_pool, float *k_scale, float *v_scale,
                                const int64_t *slot_mapping, int32_t *err, cudaStream_t stream) {
  cudaError_t e;
  if (s.kv_dtype == PA_KV_INT4) {
    e = launch_pdl(cache_write_int4_kernel, dim3(s.B), dim3(256), 0, stream,
                   static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                   static_cast<uint8_t *>(k_pool), static_cast<uint8_t *>(v_pool), k_scale,
                   v_scale, slot_mapping, s.B, s.Hkv, s.block_size, s.nblocks, err);
  } else if (s.kv_dtype == PA_KV_FP8_E4M3) {
    e = launch_pdl(cache_write_fp8_kernel, dim3(s.B), dim3(256), 0, stream,
                   static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                   static_cast<uint8_t *>(k_pool), static_cast<uint8_t *>(v_pool), k_scale,
                   v_scale, slot_mapping, s.B, s.Hkv, s.block_size, s.nblocks, err);
  } else {
    const int row16 = s.Hkv * s.D * 2 / 16;
    e = launch_pdl(cache_write_bf16_kernel, dim3(s.B), dim3(128), 0, stream,
                   static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
                   static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool), slot_mapping,
                   s.block_size, s.nblocks, row16, err);
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
