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
#pragma unroll
    for (int r = 0; r < kTile; ++r) {            // loads issued together, rows < `rows` used
      if (r < rows) {
        const float v = __uint_as_float(
            static_cast<uint32_t>(k_pool[(page * kTile + r) * row_elems + e]) << 16);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
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

// Sum eight per-lane values v[0..8) over the warp: the lanes halve the set at each of
// xor 16, 8, 4 (exchanging half of their values), then finish with xor 2, 1.  On
// return lane l holds the total of value 4*bit4 + 2*bit3 + bit2 of l (9 shuffles).
__device__ __forceinline__ float warp_sum8(float (&v)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float a[4], c[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? v[i] : v[i + 4], keep = b4 ? v[i + 4] : v[i];
    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? a[i] : a[i + 2], keep = b3 ? a[i + 2] : a[i];
    c[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float r = (b2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, b2 ? c[0] : c[1], 4);
  r += __shfl_xor_sync(0xffffffffu, r, 2);
  r += __shfl_xor_sync(0xffffffffu, r, 1);
  return r;
}

// One CTA per (sequence, KV head): score every page of the sequence, pick the topk
// best (ties to the lower page index) and write them in increasing page order to
// sel[b][kvh][0..topk), -1 past the number of pages.
template <int NG>   // groups of 8 query heads (G <= 8 * NG)
__global__ void __launch_bounds__(512) quest_select_kernel(
    const uint16_t *q, const uint16_t *summ, const int32_t *block_tables,
    const int32_t *seq_lens, int B, int Hq, int Hkv, int D, int bs, int nblocks, int max_blocks,
    int topk, int32_t *sel, int32_t *err) {
  extern __shared__ uint32_t key[];              // [npg] order keys of the page scores
  __shared__ int hist[256];
  __shared__ int s_prefix, s_kleft, s_count;
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int b = pair / Hkv, kvh = pair - b * Hkv;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = min(max(seq_lens[b], 0), max_blocks * bs);
  const int npg = (L + kTile - 1) / kTile;
  int32_t *out = sel + static_cast<size_t>(pair) * topk;

  // ---- scores: one warp per page; lane l covers channels [l * E, l * E + E), E = D / 32,
  // and keeps the group's queries for those channels in registers
  constexpr int E_MAX = 4;                       // D <= 128
  const int E = D / 32;
  float qv[8 * NG][E_MAX];
#pragma unroll
  for (int g = 0; g < 8 * NG; ++g)
#pragma unroll
    for (int e = 0; e < E_MAX; ++e)
      qv[g][e] = (g < G && e < E)
                     ? __uint_as_float(static_cast<uint32_t>(
                           q[(static_cast<size_t>(b) * Hq + kvh * G + g) * D + lane * E + e]) << 16)
                     : 0.f;
  const int32_t *row = block_tables + static_cast<size_t>(b) * max_blocks;
  const int nwarps = blockDim.x >> 5;
  constexpr int P = 8;                           // pages in flight per warp
  for (int j0 = warp; j0 < npg; j0 += nwarps * P) {
    int phys[P];
#pragma unroll
    for (int k = 0; k < P; ++k) {
      const int j = j0 + k * nwarps;
      phys[k] = j < npg ? row[(j * kTile) / bs] : -1;
    }
    uint2 lo[P], hi[P];
#pragma unroll
    for (int k = 0; k < P; ++k) {
      const int j = j0 + k * nwarps;
      lo[k] = hi[k] = make_uint2(0u, 0u);
      if (j < npg && phys[k] >= 0 && phys[k] < nblocks) {
        const int64_t page =
            static_cast<int64_t>(phys[k]) * (bs / kTile) + (j * kTile % bs) / kTile;
        const uint16_t *sm = summ + ((page * Hkv + kvh) * 2) * D + lane * E;
        if (E == 4) {
          lo[k] = *reinterpret_cast<const uint2 *>(sm);
          hi[k] = *reinterpret_cast<const uint2 *>(sm + D);
        } else {                                 // D = 64: two channels per lane
          lo[k].x = *reinterpret_cast<const uint32_t *>(sm);
          hi[k].x = *reinterpret_cast<const uint32_t *>(sm + D);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < P; ++k) {
      const int j = j0 + k * nwarps;
      if (j >= npg) break;
      float best = -INFINITY;
      if (phys[k] < 0 || phys[k] >= nblocks) {
        if (lane == 0) set_err(err, PA_DEVERR_BLOCK_ID);
      } else {
        const float mn[E_MAX] = {bf16_lo(lo[k].x), bf16_hi(lo[k].x), bf16_lo(lo[k].y),
                                 bf16_hi(lo[k].y)};
        const float mx[E_MAX] = {bf16_lo(hi[k].x), bf16_hi(hi[k].x), bf16_lo(hi[k].y),
                                 bf16_hi(hi[k].y)};
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          float acc[8];        // max(q mn, q mx) picks mx for q >= 0 and mn otherwise
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            acc[g] = 0.f;
#pragma unroll
            for (int e = 0; e < E_MAX; ++e) {
              const float qq = qv[ng * 8 + g][e];
              acc[g] = fmaf(qq, qq >= 0.f ? mx[e] : mn[e], acc[g]);
            }
          }
          const int head = ng * 8 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
          float tot = warp_sum8(acc, lane);
          if (head >= G) tot = -INFINITY;
          tot = fmaxf(tot, __shfl_xor_sync(0xffffffffu, tot, 4));
          tot = fmaxf(tot, __shfl_xor_sync(0xffffffffu, tot, 8));
          tot = fmaxf(tot, __shfl_xor_sync(0xffffffffu, tot, 16));
          best = fmaxf(best, tot);
        }
      }
      if (lane == 0) key[j] = order_key(best);
    }
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
  // ordered compaction in page order, one blockDim-page chunk at a time
  __shared__ int flags[512];
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
    for (int o = 1; o < static_cast<int>(blockDim.x); o <<= 1) {   // inclusive scan
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
    for (int o = 1; o < static_cast<int>(blockDim.x); o <<= 1) {
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
  return max_pages * 4;
}

pa_status run_quest_select(const pa_shape &s, const void *q, const void *summaries,
                           const int32_t *block_tables, const int32_t *seq_lens, int topk,
                           int32_t *selected, int32_t *err, cudaStream_t stream) {
  const size_t smem = quest_select_smem(s);
  auto kernel = (s.Hq / s.Hkv <= 8) ? quest_select_kernel<1> : quest_select_kernel<2>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return PA_ERR_CUDA;
  return launch_pdl(kernel, dim3(s.B * s.Hkv), dim3(512), smem, stream,
                    static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(summaries),
                    block_tables, seq_lens, s.B, s.Hq, s.Hkv, s.D, s.block_size, s.nblocks,
                    s.max_blocks, topk, selected, err) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace pa
