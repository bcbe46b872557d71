// pa_quest.cu -- query-aware page selection ("KV Cache Engineering for LLM Serving",
// section 7, Quest): per-page key summaries, page scoring and top-k selection.
//
// A page is a 16-token tile of the pool (a block of 16 or 32 tokens holds one or two
// pages), so page g covers pool rows [16 g, 16 g + 16) and, in a sequence's block
// table, logical page j of sequence b is page block_tables[b][16 j / bs] * bs / 16
// + (16 j % bs) / 16.  Its summary is the per-channel minimum and maximum of the keys
// it holds; a query scores it by sum_d max(q_d min_d, q_d max_d), an upper bound of
// q . k over the page.  A GQA group shares one selection: each page keeps its best
// score over the group's query heads.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// Summaries [pages, Hkv, 2 (min, max), D] bf16, for the pages the listed slots were
// written to: min/max over the page's rows 0 .. slot % 16.  When several listed
// slots fall in one page only the last of them (largest slot, then largest index)
// writes.  One CTA per listed token.
__global__ void __launch_bounds__(128) quest_summarize_kernel(
    const uint16_t *k_pool, uint16_t *summ, const int64_t *slot_mapping, int T, int Hkv, int D,
    int64_t nrows, int32_t *err) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= nrows) {
    if (threadIdx.x == 0) set_err(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t page = slot / kTile;
  int later = 0;
  for (int u = threadIdx.x; u < T; u += blockDim.x) {
    const int64_t o = slot_mapping[u];
    if (u != t && o >= 0 && o / kTile == page && (o > slot || (o == slot && u > t))) later = 1;
  }
  if (__syncthreads_or(later)) return;
  const int rows = static_cast<int>(slot - page * kTile) + 1;
  const int row_elems = Hkv * D;
  for (int e = threadIdx.x; e < row_elems; e += blockDim.x) {
    const int h = e / D, d = e - h * D;
    float mn = INFINITY, mx = -INFINITY;
    for (int r = 0; r < rows; ++r) {
      const float v = __uint_as_float(
          static_cast<uint32_t>(k_pool[(page * kTile + r) * row_elems + e]) << 16);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    uint16_t *dst = summ + ((page * Hkv + h) * 2) * D;
    dst[d] = static_cast<uint16_t>(__float_as_uint(mn) >> 16);   // exact: bf16 inputs
    dst[D + d] = static_cast<uint16_t>(__float_as_uint(mx) >> 16);
  }
}

// Larger-is-better order of a float as an unsigned key.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One CTA per (sequence, KV head): score every page of the sequence, pick the topk
// best (ties to the lower page index) and write them in increasing page order to
// sel[b][kvh][0..topk), -1 past the number of pages.
__global__ void __launch_bounds__(256) quest_select_kernel(
    const uint16_t *q, const uint16_t *summ, const int32_t *block_tables,
    const int32_t *seq_lens, int B, int Hq, int Hkv, int D, int bs, int nblocks, int max_blocks,
    int topk, int32_t *sel, int32_t *err) {
  extern __shared__ uint32_t qs_raw[];
  __shared__ int hist[256];
  __shared__ int s_prefix, s_kleft, s_count;
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int b = pair / Hkv, kvh = pair - b * Hkv;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x;
  const int L = min(max(seq_lens[b], 0), max_blocks * bs);
  const int npg = (L + kTile - 1) / kTile;
  int32_t *out = sel + static_cast<size_t>(pair) * topk;
  float *qs = reinterpret_cast<float *>(qs_raw);                 // [G][D]
  uint32_t *key = qs_raw + G * D;                                 // [npg] order keys
  for (int e = tid; e < G * D; e += blockDim.x)
    qs[e] = __uint_as_float(
        static_cast<uint32_t>(q[(static_cast<size_t>(b) * Hq + kvh * G) * D + e]) << 16);
  __syncthreads();

  // ---- scores: one thread per page
  const int32_t *row = block_tables + static_cast<size_t>(b) * max_blocks;
  for (int j = tid; j < npg; j += blockDim.x) {
    const int phys = row[(j * kTile) / bs];
    float best = -INFINITY;
    if (phys < 0 || phys >= nblocks) {
      set_err(err, PA_DEVERR_BLOCK_ID);
    } else {
      const int64_t page = static_cast<int64_t>(phys) * (bs / kTile) + (j * kTile % bs) / kTile;
      const uint16_t *sm = summ + ((page * Hkv + kvh) * 2) * D;
      float acc[16];
#pragma unroll
      for (int g = 0; g < 16; ++g) acc[g] = 0.f;
      for (int d = 0; d < D; d += 2) {
        const uint32_t mn2 = *reinterpret_cast<const uint32_t *>(sm + d);
        const uint32_t mx2 = *reinterpret_cast<const uint32_t *>(sm + D + d);
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          if (g < G) {   // max(q mn, q mx) picks mx for q >= 0 and mn otherwise
            const float q0 = qs[g * D + d], q1 = qs[g * D + d + 1];
            acc[g] = fmaf(q0, q0 >= 0.f ? bf16_lo(mx2) : bf16_lo(mn2), acc[g]);
            acc[g] = fmaf(q1, q1 >= 0.f ? bf16_hi(mx2) : bf16_hi(mn2), acc[g]);
          }
        }
      }
#pragma unroll
      for (int g = 0; g < 16; ++g)
        if (g < G) best = fmaxf(best, acc[g]);
    }
    key[j] = order_key(best);
  }
  __syncthreads();

  if (npg <= topk) {          // every page is chosen
    for (int c = tid; c < topk; c += blockDim.x) out[c] = c < npg ? c : -1;
    return;
  }
  // ---- radix select of the topk-th largest key, 8 bits at a time from the top
  if (tid == 0) {
    s_prefix = 0;
    s_kleft = topk;
  }
  uint32_t mask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = static_cast<uint32_t>(s_prefix);
    for (int j = tid; j < npg; j += blockDim.x)
      if ((key[j] & mask) == prefix) atomicAdd(&hist[(key[j] >> shift) & 0xFF], 1);
    __syncthreads();
    if (tid == 0) {
      int k = s_kleft, bin = 255;
      while (bin > 0 && hist[bin] < k) k -= hist[bin--];
      s_prefix = static_cast<int>(prefix | (static_cast<uint32_t>(bin) << shift));
      s_kleft = k;
    }
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  // threshold T: take every key > T and the first s_kleft keys == T (lowest pages)
  const uint32_t T = static_cast<uint32_t>(s_prefix);
  const int take_equal = s_kleft;
  if (tid == 0) s_count = 0;
  __syncthreads();
  // ordered compaction in page order, one 256-page chunk at a time
  __shared__ int flags[256];
  __shared__ int eq_seen;
  if (tid == 0) eq_seen = 0;
  __syncthreads();
  for (int base = 0; base < npg; base += blockDim.x) {
    const int j = base + tid;
    int f = 0, eq = 0;
    if (j < npg) {
      f = key[j] > T;
      eq = key[j] == T;
    }
    // rank of this page among the chunk's equal keys
    flags[tid] = eq;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {         // inclusive scan of flags
      const int v = tid >= o ? flags[tid - o] : 0;
      __syncthreads();
      flags[tid] += v;
      __syncthreads();
    }
    const int eq_rank = eq_seen + flags[tid] - eq;   // equal keys before this page
    if (eq && eq_rank < take_equal) f = 1;
    __syncthreads();
    if (tid == blockDim.x - 1) eq_seen += flags[tid];
    flags[tid] = f;
    __syncthreads();
    for (int o = 1; o < 256; o <<= 1) {
      const int v = tid >= o ? flags[tid - o] : 0;
      __syncthreads();
      flags[tid] += v;
      __syncthreads();
    }
    if (f) out[s_count + flags[tid] - 1] = j;
    __syncthreads();
    if (tid == blockDim.x - 1) s_count += flags[tid];
    __syncthreads();
  }
}

pa_status run_quest_summarize(const pa_shape &s, const void *k_pool, void *summaries,
                              const int64_t *slot_mapping, int32_t *err, cudaStream_t stream) {
  return launch_pdl(quest_summarize_kernel, dim3(s.B), dim3(128), 0, stream,
                    static_cast<const uint16_t *>(k_pool), static_cast<uint16_t *>(summaries),
                    slot_mapping, s.B, s.Hkv, s.D,
                    static_cast<int64_t>(s.nblocks) * s.block_size, err) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

size_t quest_select_smem(const pa_shape &s) {
  const size_t max_pages = (static_cast<size_t>(s.max_blocks) * s.block_size + kTile - 1) / kTile;
  return static_cast<size_t>(s.Hq / s.Hkv) * s.D * 4 + max_pages * 4;
}

pa_status run_quest_select(const pa_shape &s, const void *q, const void *summaries,
                           const int32_t *block_tables, const int32_t *seq_lens, int topk,
                           int32_t *selected, int32_t *err, cudaStream_t stream) {
  const size_t smem = quest_select_smem(s);
  if (cudaFuncSetAttribute(quest_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return PA_ERR_CUDA;
  return launch_pdl(quest_select_kernel, dim3(s.B * s.Hkv), dim3(256), smem, stream,
                    static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(summaries),
                    block_tables, seq_lens, s.B, s.Hq, s.Hkv, s.D, s.block_size, s.nblocks,
                    s.max_blocks, topk, selected, err) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace pa
