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

// Pages of a sequence of length L (clamped to the block table's reach).
__device__ __forceinline__ int quest_pages(int L, int cap) {
  return (min(max(L, 0), cap) + kTile - 1) / kTile;
}

// prefix[b] = number of (KV head, page) units of the sequences before b, for b <= B
// (units of sequence b: Hkv * its pages).  Block-wide; ends with a barrier.
template <int THREADS>
__device__ void scan_units(const int32_t *seq_lens, int B, int Hkv, int cap, int32_t *prefix) {
  __shared__ int32_t warp_total[THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (B + THREADS - 1) / THREADS;
  const int lo = min(B, tid * per), hi = min(B, lo + per);
  int mine = 0;
  for (int b = lo; b < hi; ++b) mine += Hkv * quest_pages(__ldg(seq_lens + b), cap);
  int inc = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_total[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int t = lane < THREADS / 32 ? warp_total[lane] : 0;
    const int own = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += v;
    }
    if (lane < THREADS / 32) warp_total[lane] = t - own;
  }
  __syncthreads();
  int run = warp_total[warp] + inc - mine;
  for (int b = lo; b < hi; ++b) {
    prefix[b] = run;
    run += Hkv * quest_pages(__ldg(seq_lens + b), cap);
  }
  if (tid == THREADS - 1) prefix[B] = run;       // the last thread's range ends at B
  __syncthreads();
}

constexpr int kScoreThreads = 256;
constexpr int kScorePages = 8;                   // pages in flight per warp

// Page scores.  The (sequence, KV head, page) units, pages fastest, are cut into
// `nseg` equal contiguous segments, one per warp, so a long sequence spreads over
// many warps.  Lane l covers channels [l E, l E + E), E = D / 32, and keeps the
// group's queries for them in registers while its segment stays in one (sequence,
// KV head); score[b][kvh][j] = max over the group of sum_d max(q_d min_d, q_d max_d).
template <int NG>   // groups of 8 query heads (G <= 8 * NG)
__global__ void __launch_bounds__(kScoreThreads, 2) quest_score_kernel(
    const uint16_t *q, const uint16_t *summ, const int32_t *block_tables,
    const int32_t *seq_lens, int B, int Hq, int Hkv, int D, int bs, int nblocks, int max_blocks,
    int max_pages, int nseg, float *scores, int32_t *err) {
  extern __shared__ int32_t prefix[];            // [B + 1]
  pdl_trigger();
  const int cap = max_blocks * bs;
  scan_units<kScoreThreads>(seq_lens, B, Hkv, cap, prefix);
  pdl_wait();                                    // summaries come from the launch before
  const int lane = threadIdx.x & 31;
  const int seg = blockIdx.x * (kScoreThreads / 32) + (threadIdx.x >> 5);
  const int total = prefix[B];
  const int W = (total + nseg - 1) / nseg;
  int f = min(seg * W, total);
  const int end = min(f + W, total);
  const int G = Hq / Hkv;
  constexpr int E_MAX = 4;                       // D <= 128
  const int E = D / 32;
  while (f < end) {                              // warp-uniform
    int lo = 0, hi = B - 1;                      // last sequence starting at or before f
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= f) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int npg = (prefix[b + 1] - prefix[b]) / Hkv;
    const int r = f - prefix[b];
    const int kvh = r / npg, j0 = r - kvh * npg;
    const int run = min(end - f, npg - j0);
    float qv[8 * NG][E_MAX];
#pragma unroll
    for (int g = 0; g < 8 * NG; ++g)
#pragma unroll
      for (int e = 0; e < E_MAX; ++e)
        qv[g][e] = (g < G && e < E)
                       ? __uint_as_float(static_cast<uint32_t>(__ldg(
                             q + (static_cast<size_t>(b) * Hq + kvh * G + g) * D + lane * E + e))
                                         << 16)
                       : 0.f;
    const int32_t *row = block_tables + static_cast<size_t>(b) * max_blocks;
    float *out = scores + (static_cast<size_t>(b) * Hkv + kvh) * max_pages;
    for (int jb = j0; jb < j0 + run; jb += kScorePages) {
      const int n = min(kScorePages, j0 + run - jb);
      // lane k < n fetches the block-table entry of page jb + k
      const int my_phys = lane < n ? __ldg(row + ((jb + lane) * kTile) / bs) : 0;
      int phys[kScorePages];
      uint2 mnv[kScorePages], mxv[kScorePages];
#pragma unroll
      for (int k = 0; k < kScorePages; ++k) {
        phys[k] = __shfl_sync(0xffffffffu, my_phys, k);
        mnv[k] = mxv[k] = make_uint2(0u, 0u);
        if (k < n && phys[k] >= 0 && phys[k] < nblocks) {
          const int j = jb + k;
          const int64_t page =
              static_cast<int64_t>(phys[k]) * (bs / kTile) + (j * kTile % bs) / kTile;
          const uint16_t *sm = summ + ((page * Hkv + kvh) * 2) * D + lane * E;
          if (E == 4) {
            mnv[k] = __ldg(reinterpret_cast<const uint2 *>(sm));
            mxv[k] = __ldg(reinterpret_cast<const uint2 *>(sm + D));
          } else {                               // D = 64: two channels per lane
            mnv[k].x = __ldg(reinterpret_cast<const uint32_t *>(sm));
            mxv[k].x = __ldg(reinterpret_cast<const uint32_t *>(sm + D));
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kScorePages; ++k) {
        if (k >= n) break;
        float best = -INFINITY;
        if (phys[k] < 0 || phys[k] >= nblocks) {
          if (lane == 0) set_err(err, PA_DEVERR_BLOCK_ID);
        } else {
          const float mn[E_MAX] = {bf16_lo(mnv[k].x), bf16_hi(mnv[k].x), bf16_lo(mnv[k].y),
                                   bf16_hi(mnv[k].y)};
          const float mx[E_MAX] = {bf16_lo(mxv[k].x), bf16_hi(mxv[k].x), bf16_lo(mxv[k].y),
                                   bf16_hi(mxv[k].y)};
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            float acc[8];      // max(q mn, q mx) picks mx for q >= 0 and mn otherwise
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              acc[g] = 0.f;
#pragma unroll
              for (int e = 0; e < E_MAX; ++e) {
                const float qq = qv[ng * 8 + g][e];
                acc[g] = fmaf(qq, qq >= 0.f ? mx[e] : mn[e], acc[g]);
              }
            }
            const int head =
                ng * 8 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
            float tot = warp_sum8(acc, lane);
            if (head >= G) tot = -INFINITY;
            tot = fmaxf(tot, __shfl_xor_sync(0xffffffffu, tot, 4));
            tot = fmaxf(tot, __shfl_xor_sync(0xffffffffu, tot, 8));
            tot = fmaxf(tot, __shfl_xor_sync(0xffffffffu, tot, 16));
            best = fmaxf(best, tot);
          }
        }
        if (lane == k) out[jb + k] = best;       // spread the stores over the lanes
      }
    }
    f += run;
  }
}

constexpr int kTopkThreads = 512;

// Top-k of one (sequence, KV head) per CTA: the topk best pages by score (ties to
// the lower page index), written in increasing page order to sel[b][kvh][0..topk),
// -1 past the number of pages.  Radix select of the topk-th largest order key, eight
// bits a pass from the top, then an ordered compaction by warp ballots.
__global__ void __launch_bounds__(kTopkThreads) quest_topk_kernel(
    const float *scores, const int32_t *seq_lens, int Hkv, int cap, int max_pages, int topk,
    int32_t *sel) {
  extern __shared__ uint32_t key[];              // [npg] order keys of the page scores
  __shared__ int hist[256];
  __shared__ int warp_cnt[2][kTopkThreads / 32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_kleft;
  pdl_trigger();
  const int pair = blockIdx.x;
  const int b = pair / Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int npg = quest_pages(__ldg(seq_lens + b), cap);
  int32_t *out = sel + static_cast<size_t>(pair) * topk;
  if (npg <= topk) {                             // every page is chosen
    pdl_wait();                                  // `sel` may still be read by the launch before
    for (int c = tid; c < topk; c += kTopkThreads) out[c] = c < npg ? c : -1;
    return;
  }
  pdl_wait();
  const float *sc = scores + static_cast<size_t>(pair) * max_pages;
  for (int j = tid; j < npg; j += kTopkThreads) key[j] = order_key(sc[j]);
  if (tid == 0) {
    s_prefix = 0u;
    s_kleft = topk;
  }
  uint32_t mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int j = tid; j < npg; j += kTopkThreads)
      if ((key[j] & mask) == prefix) atomicAdd(&hist[(key[j] >> shift) & 0xFF], 1);
    __syncthreads();
    if (warp == 0) {
      // the highest bin whose count from the top reaches kleft: lane l holds bins
      // [8 l, 8 l + 8); suffix sums over the lanes find its lane, then its bin
      const int kleft = s_kleft;
      int c[8], mine = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[lane * 8 + i];
        mine += c[i];
      }
      int suf = mine;                            // sum over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += v;
      }
      const unsigned reach = __ballot_sync(0xffffffffu, suf >= kleft);
      const int t = 31 - __clz(static_cast<int>(reach | 1u));   // lane 0 reaches: kleft <= npg
      if (lane == t) {
        int k = kleft - (suf - mine);            // still needed within this lane's bins
        int bin = 7;
        while (bin > 0 && c[bin] < k) k -= c[bin--];
        s_prefix = prefix | (static_cast<uint32_t>(lane * 8 + bin) << shift);
        s_kleft = k;
      }
    }
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  // threshold T: every key > T and the first s_kleft keys == T (lowest pages)
  const uint32_t T = s_prefix;
  const int take_equal = s_kleft;
  int count = 0, eq_seen = 0;                    // identical in every thread
  for (int base = 0; base < npg; base += kTopkThreads) {
    const int j = base + tid;
    const bool gt = j < npg && key[j] > T, eq = j < npg && key[j] == T;
    const unsigned eq_bal = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_cnt[0][warp] = __popc(eq_bal);
    __syncthreads();
    int eq_before = eq_seen, eq_chunk = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
      const int v = warp_cnt[0][w];
      eq_before += w < warp ? v : 0;
      eq_chunk += v;
    }
    eq_before += __popc(eq_bal & ((1u << lane) - 1u));
    const bool take = gt || (eq && eq_before < take_equal);
    const unsigned tk_bal = __ballot_sync(0xffffffffu, take);
    if (lane == 0) warp_cnt[1][warp] = __popc(tk_bal);
    __syncthreads();
    int pos = count, chunk = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
      const int v = warp_cnt[1][w];
      pos += w < warp ? v : 0;
      chunk += v;
    }
    if (take) out[pos + __popc(tk_bal & ((1u << lane) - 1u))] = j;
    count += chunk;
    eq_seen += eq_chunk;
    __syncthreads();                             // warp_cnt is rewritten next chunk
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

int quest_max_pages(const pa_shape &s) {
  return static_cast<int>((static_cast<int64_t>(s.max_blocks) * s.block_size + kTile - 1) / kTile);
}

size_t quest_topk_smem(const pa_shape &s) { return static_cast<size_t>(quest_max_pages(s)) * 4; }

size_t quest_score_smem(const pa_shape &s) { return (static_cast<size_t>(s.B) + 1) * 4; }

pa_status run_quest_select(const pa_shape &s, const void *q, const void *summaries,
                           const int32_t *block_tables, const int32_t *seq_lens, int topk,
                           float *page_scores, int32_t *selected, int32_t *err,
                           cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  const int max_pages = quest_max_pages(s);
  const size_t score_smem = quest_score_smem(s);
  auto score = (s.Hq / s.Hkv <= 8) ? quest_score_kernel<1> : quest_score_kernel<2>;
  if (cudaFuncSetAttribute(score, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(score_smem)) != cudaSuccess)
    return PA_ERR_CUDA;
  const int grid = 2 * sms;                      // two 8-warp CTAs per SM
  const int nseg = grid * (kScoreThreads / 32);
  if (launch_pdl(score, dim3(grid), dim3(kScoreThreads), score_smem, stream,
                 static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(summaries),
                 block_tables, seq_lens, s.B, s.Hq, s.Hkv, s.D, s.block_size, s.nblocks,
                 s.max_blocks, max_pages, nseg, page_scores, err) != cudaSuccess)
    return PA_ERR_CUDA;
  const size_t topk_smem = quest_topk_smem(s);
  if (cudaFuncSetAttribute(quest_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(topk_smem)) != cudaSuccess)
    return PA_ERR_CUDA;
  return launch_pdl(quest_topk_kernel, dim3(s.B * s.Hkv), dim3(kTopkThreads), topk_smem, stream,
                    static_cast<const float *>(page_scores), seq_lens, s.Hkv,
                    s.max_blocks * s.block_size, max_pages, topk, selected) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace pa
