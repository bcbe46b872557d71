// pa_cache.cu -- the slot-mapped cache write (reshape_and_cache).
//
// "Taming the Token Torrent", "How Paging Works in the LLM Context" / "The Block
// Table Logic": each step's new K/V vectors go to slot s = block * bs + offset,
// i.e. row (s / bs, s % bs) of the block pool [nblocks, bs, Hkv, D].
// FP8 and 4-bit pools follow "KV Cache Engineering for LLM Serving", section 8
// (absmax scale, divide, round, clip), with one fp32 scale per (block, KV head) that
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

// Quantised pools (D = 128).  Per (block, KV head), separately for K and V, a token
// written at offset off updates the block's absmax scale and re-encodes the codes at
// offsets below off when the scale grows ("KV Cache Engineering for LLM Serving",
// section 8), so the tokens of one call that land in one block are applied one after
// the other, in token order.  One CTA per token: the block's first token of the call
// (its leader) applies every token of the call in that block; the others leave.  Warps
// take (KV head, K or V) jobs; each lane owns four consecutive elements of a head
// vector, so a lane only ever re-encodes the codes it wrote itself.

// E4M3 codes, one byte per element; a lane's four codes are one 32-bit word.
struct Fp8Codec {
  static constexpr int kRowBytes = 128;
  static constexpr float kMaxCode = 448.f;
  using Word = uint32_t;
  static __device__ __forceinline__ Word encode(const float (&v)[4], float s) {
    if (s == 0.f) return 0u;
    return f32x2_to_e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s)) |
           (f32x2_to_e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s)) << 16);
  }
  // codes restored with the old scale (one fp32 product each), encoded with the new
  static __device__ __forceinline__ Word reencode(Word c, float old, float s) {
    const float2 lo = e4m3x2_to_float2(c), hi = e4m3x2_to_float2(c >> 16);
    const float v[4] = {__fmul_rn(lo.x, old), __fmul_rn(lo.y, old), __fmul_rn(hi.x, old),
                        __fmul_rn(hi.y, old)};
    return encode(v, s);
  }
};

// 4-bit codes clip(rint(x / scale), -7, 7) stored as offset-binary nibbles, element 2j in
// the low nibble of byte j; a lane's four codes are one 16-bit word.
__device__ __forceinline__ uint32_t int4_code(float x, float scale) {
  if (scale == 0.f) return 8u;
  const float c = fminf(fmaxf(rintf(__fdiv_rn(x, scale)), -7.f), 7.f);
  return static_cast<uint32_t>(static_cast<int>(c) + 8);
}

struct Int4Codec {
  static constexpr int kRowBytes = 64;
  static constexpr float kMaxCode = 7.f;
  using Word = uint16_t;
  static __device__ __forceinline__ Word encode(const float (&v)[4], float s) {
    uint32_t code = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) code |= int4_code(v[e], s) << (4 * e);
    return static_cast<Word>(code);
  }
  static __device__ __forceinline__ Word reencode(Word c, float old, float s) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[e] = __fmul_rn(static_cast<float>(static_cast<int>((c >> (4 * e)) & 0xF) - 8), old);
    return encode(v, s);
  }
};

template <class Codec>
__global__ void __launch_bounds__(256) cache_write_quant_kernel(
    const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_pool, uint8_t *v_pool,
    float *k_scale, float *v_scale, const int64_t *slot_mapping, int T, int Hkv, int bs,
    int nblocks, int32_t *err) {
  using Word = typename Codec::Word;
  constexpr int D = 128, kWarps = 8;
  __shared__ int members[256];      // this chunk's tokens of the block, in token order
  __shared__ int member_off[256];
  __shared__ int warp_count[kWarps];
  __shared__ uint32_t offsets_seen;
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  const int64_t nslots = static_cast<int64_t>(nblocks) * bs;
  if (slot >= nslots) {
    if (tid == 0) set_err(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / bs;
  auto in_block = [&](int64_t o) { return o >= 0 && o < nslots && o / bs == blk; };
  // only the block's first token of the call goes on.  A token right after another of
  // its block (a prompt's tokens fill their blocks in order) leaves at once; the others
  // look through every earlier token.
  if (t > 0 && in_block(slot_mapping[t - 1])) return;
  int earlier = 0;
  for (int u = tid; u < t - 1; u += blockDim.x) earlier |= in_block(slot_mapping[u]);
  if (__syncthreads_or(earlier)) return;
  if (tid == 0) offsets_seen = 0u;
  for (int c0 = t; c0 < T; c0 += blockDim.x) {
    // the chunk's tokens of this block, in token order (ballot compaction)
    const int u = c0 + tid;
    const int64_t o = u < T ? slot_mapping[u] : -1;
    const bool mine = in_block(o);
    const uint32_t ballot = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) warp_count[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, n = 0;
    for (int w = 0; w < kWarps; ++w) {
      before += w < warp ? warp_count[w] : 0;
      n += warp_count[w];
    }
    if (mine) {
      const int i = before + __popc(ballot & ((1u << lane) - 1u));
      const int off = static_cast<int>(o - blk * bs);
      members[i] = u;
      member_off[i] = off;
      // a second token for one slot: applied after the first, and reported
      if (atomicOr(&offsets_seen, 1u << off) & (1u << off)) set_err(err, PA_DEVERR_FP8_CONFLICT);
    }
    __syncthreads();
    for (int job = warp; job < 2 * Hkv; job += kWarps) {
      const int h = job >> 1;
      const bool is_v = job & 1;
      uint8_t *pool = is_v ? v_pool : k_pool;
      float *scale = (is_v ? v_scale : k_scale) + blk * Hkv + h;
      float s = *scale;
      for (int i = 0; i < n; ++i) {
        const int tok = members[i], off = member_off[i];
        const uint16_t *x = (is_v ? v_new : k_new) + (static_cast<size_t>(tok) * Hkv + h) * D;
        const uint2 raw = *reinterpret_cast<const uint2 *>(x + lane * 4);
        const float v[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
        const float cand = __fdiv_rn(amax, Codec::kMaxCode);
        const float s_new = (off == 0 || cand > s) ? cand : s;
        auto word = [&](int r) {
          return reinterpret_cast<Word *>(
              pool + ((blk * bs + r) * Hkv + h) * static_cast<int64_t>(Codec::kRowBytes) +
              lane * sizeof(Word));
        };
        if (off > 0 && s_new > s)
          for (int r = 0; r < off; ++r) *word(r) = Codec::reencode(*word(r), s, s_new);
        *word(off) = Codec::encode(v, s_new);
        s = s_new;
      }
      if (lane == 0) *scale = s;
    }
    __syncthreads();   // the member lists and the scales are reused by the next chunk
  }
}

pa_status run_reshape_and_cache(const pa_shape &s, const void *k_new, const void *v_new,
                                void *k_pool, void *v_pool, float *k_scale, float *v_scale,
                                const int64_t *slot_mapping, int32_t *err, cudaStream_t stream) {
  cudaError_t e;
  if (s.kv_dtype == PA_KV_INT4) {
    e = launch_pdl(cache_write_quant_kernel<Int4Codec>, dim3(s.B), dim3(256), 0, stream,
                   static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                   static_cast<uint8_t *>(k_pool), static_cast<uint8_t *>(v_pool), k_scale,
                   v_scale, slot_mapping, s.B, s.Hkv, s.block_size, s.nblocks, err);
  } else if (s.kv_dtype == PA_KV_FP8_E4M3) {
    e = launch_pdl(cache_write_quant_kernel<Fp8Codec>, dim3(s.B), dim3(256), 0, stream,
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
