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
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// Pull the 128-byte line holding `p` into L2 (a hint: no data comes back).
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// A finite float rounded to bf16 toward +inf (UP) or -inf, as bits; -0 comes out as +0.
template <bool UP>
__device__ __forceinline__ uint32_t bf16_directed(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  const uint32_t t = u >> 16;
  if ((u & 0xFFFFu) == 0u) return t;              // a bf16 value already
  const bool neg = (u >> 31) != 0u;
  return neg != UP ? t + 1u : t;                  // away from zero, or toward it
}

// Quantised pools (KIND 1: E4M3 codes, one byte each; 2: 4-bit offset-binary codes,
// element 2j in the low nibble of byte j): eight consecutive channels of one KV head
// per thread and pass.  The restored keys code * scale are not bf16 values, so each
// product is taken rounded down for the minimum and up for the maximum, and the
// stored bf16 bounds are rounded the same way: the minimum never exceeds a key and
// the maximum is never below one, so the page score stays an upper bound.  (Directed
// rounding to fp32 and then to bf16 equals directed rounding to bf16.)
template <int KIND>
__device__ __forceinline__ void summarize_quant(const uint8_t *k_pool, const float *k_scale,
                                                uint16_t *summ, int64_t page, int rows, int Hkv,
                                                int D, int bs) {
  constexpr int kCodeBytes = KIND == 1 ? 8 : 4;   // bytes of eight codes
  const int row_vecs = Hkv * D / 8;
  const int64_t blk = page * kTile / bs;          // a page lies inside one block
  for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
    const int e = v * 8, h = e / D, d = e - h * D;
    const float sc = __ldg(k_scale + blk * Hkv + h);
    float mn[8], mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mn[i] = INFINITY;
      mx[i] = -INFINITY;
    }
#pragma unroll
    for (int r = 0; r < kTile; ++r) {
      if (r < rows) {
        const uint8_t *src = k_pool + ((page * kTile + r) * row_vecs + v) * kCodeBytes;
        float c[8];
        if constexpr (KIND == 1) {
          const uint2 w = __ldg(reinterpret_cast<const uint2 *>(src));
          const float2 a = e4m3x2_to_float2(w.x), b = e4m3x2_to_float2(w.x >> 16);
          const float2 x = e4m3x2_to_float2(w.y), y = e4m3x2_to_float2(w.y >> 16);
          c[0] = a.x; c[1] = a.y; c[2] = b.x; c[3] = b.y;
          c[4] = x.x; c[5] = x.y; c[6] = y.x; c[7] = y.y;
        } else {
          const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(src));
#pragma unroll
          for (int i = 0; i < 8; ++i) c[i] = static_cast<float>(static_cast<int>((w >> (4 * i)) & 0xFu) - 8);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          mn[i] = fminf(mn[i], __fmul_rd(c[i], sc));
          mx[i] = fmaxf(mx[i], __fmul_ru(c[i], sc));
        }
      }
    }
    uint32_t pmn[4], pmx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pmn[i] = bf16_directed<false>(mn[2 * i]) | (bf16_directed<false>(mn[2 * i + 1]) << 16);
      pmx[i] = bf16_directed<true>(mx[2 * i]) | (bf16_directed<true>(mx[2 * i + 1]) << 16);
    }
    uint16_t *dst = summ + ((page * Hkv + h) * 2) * D + d;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(pmn[0], pmn[1], pmn[2], pmn[3]);
    *reinterpret_cast<uint4 *>(dst + D) = make_uint4(pmx[0], pmx[1], pmx[2], pmx[3]);
  }
}

// Summaries [pages, Hkv, 2 (min, max), D] bf16, for the pages the listed slots were
// written to: min/max over the page's rows 0 .. slot % 16.  When several listed
// slots fall in one page only the last of them (largest slot, then largest index)
// writes.  One CTA per listed token.  KIND 0: bf16 keys (exact min/max); 1, 2:
// quantised keys restored with their (block, head) scale (summarize_quant).
template <int KIND>
__global__ void __launch_bounds__(128) quest_summarize_kernel(
    const void *k_pool_raw, const float *k_scale, uint16_t *summ, const int64_t *slot_mapping,
    int T, int Hkv, int D, int bs, int64_t nrows, int32_t *err) {
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
  if constexpr (KIND != 0) {
    summarize_quant<KIND>(static_cast<const uint8_t *>(k_pool_raw), k_scale, summ, page, rows,
                          Hkv, D, bs);
    return;
  }
  const uint16_t *k_pool = static_cast<const uint16_t *>(k_pool_raw);
  // eight consecutive channels of one KV head per thread and pass (16-byte loads of
  // all 16 rows in flight; rows >= `rows` are not used)
  const int row_vecs = Hkv * D / 8;
  const uint4 *src = reinterpret_cast<const uint4 *>(k_pool + page * kTile * Hkv * D);
  for (int v = threadIdx.x; v < row_vecs; v += blockDim.x) {
    uint4 x[kTile];
#pragma unroll
    for (int r = 0; r < kTile; ++r)
      x[r] = r < rows ? __ldg(src + r * row_vecs + v) : make_uint4(0u, 0u, 0u, 0u);
    float mn[8], mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mn[i] = INFINITY;
      mx[i] = -INFINITY;
    }
#pragma unroll
    for (int r = 0; r < kTile; ++r) {
      if (r < rows) {
        const uint32_t w[4] = {x[r].x, x[r].y, x[r].z, x[r].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
          mn[2 * i] = fminf(mn[2 * i], lo);
          mx[2 * i] = fmaxf(mx[2 * i], lo);
          mn[2 * i + 1] = fminf(mn[2 * i + 1], hi);
          mx[2 * i + 1] = fmaxf(mx[2 * i + 1], hi);
        }
      }
    }
    uint32_t pmn[4], pmx[4];                      // exact: the inputs are bf16
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pmn[i] = (__float_as_uint(mn[2 * i]) >> 16) | (__float_as_uint(mn[2 * i + 1]) & 0xFFFF0000u);
      pmx[i] = (__float_as_uint(mx[2 * i]) >> 16) | (__float_as_uint(mx[2 * i + 1]) & 0xFFFF0000u);
    }
    const int e = v * 8, h = e / D, d = e - h * D;
    uint16_t *dst = summ + ((page * Hkv + h) * 2) * D + d;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(pmn[0], pmn[1], pmn[2], pmn[3]);
    *reinterpret_cast<uint4 *>(dst + D) = make_uint4(pmx[0], pmx[1], pmx[2], pmx[3]);
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

// Page scoring as a tensor-core contraction.  Because min_d <= max_d,
//     sum_d max(q_d min_d, q_d max_d) = sum_d q-_d min_d + sum_d q+_d max_d
// with q+ = max(q, 0) and q- = min(q, 0): the product of a page's summary row
// [min_0 .. min_{D-1}, max_0 .. max_{D-1}] (bf16, exactly as stored) with the
// column [q-; q+] (bf16, exact).  A warp scores 16 pages of one (sequence, KV head)
// against the group's 8 (or 16) query heads with m16n8k16 mma, fp32 accumulation.
template <int D_, int NG_>
struct ScoreCfg {
  static constexpr int D = D_;
  static constexpr int NG = NG_;                   // 8-head n-tiles (G <= 8 NG)
  static constexpr int ROWB = 4 * D;               // one summary row: 2 D bf16
  static constexpr int ROWP = ROWB + 16;           // padded row in shared memory: the 8 rows
                                                   // an ldmatrix reads fall in distinct banks
  static constexpr int CH = 16;                    // pages per chunk (the mma's m)
  static constexpr int KSQ = D / 16;               // k-steps over one half of the row
  static constexpr int BUF = CH * ROWP;            // one stage: a chunk's summary rows
  static constexpr int STAGES = 2;                 // one chunk in flight while one is scored
  static constexpr int WARPS = 4;
  static constexpr int THREADS = 32 * WARPS;
  // per warp: stages, then chunk descriptors (int4), mbarriers and valid-row masks, each
  // array after the stages at a multiple of its own alignment
  static constexpr int FIXED = WARPS * STAGES * (BUF + 16 + 8 + 4);
  static_assert(BUF % 16 == 0, "bulk copies need 16-byte aligned stages");
};

// The warp's share of the score workspace: a contiguous run of units cut into
// chunks of at most 16 pages of one (sequence, KV head).
struct ScoreChunk {
  int b, kvh, j0, n;
};

template <class S>
__global__ void __launch_bounds__(S::THREADS) quest_score_kernel(
    const uint16_t *q, const uint16_t *summ, const int32_t *block_tables,
    const int32_t *seq_lens, int B, int Hq, int Hkv, int bs, int nblocks, int max_blocks,
    int max_pages, int nseg, float *scores, int32_t *err) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int D = S::D, ST = S::STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *stage = smem + warp * ST * S::BUF;
  uint8_t *tail = smem + S::WARPS * ST * S::BUF;
  int4 *desc = reinterpret_cast<int4 *>(tail) + warp * ST;
  uint64_t *bar = reinterpret_cast<uint64_t *>(tail + S::WARPS * ST * 16) + warp * ST;
  unsigned *okms = reinterpret_cast<unsigned *>(tail + S::WARPS * ST * 24) + warp * ST;
  int32_t *prefix = reinterpret_cast<int32_t *>(smem + S::FIXED);
  const int G = Hq / Hkv;
  pdl_trigger();
  if (lane == 0) {
    for (int st = 0; st < ST; ++st) mbar_init(smem_u32(&bar[st]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int cap = max_blocks * bs;
  scan_units<S::THREADS>(seq_lens, B, Hkv, cap, prefix);
  pdl_wait();                                      // summaries come from the launch before

  const int seg = blockIdx.x * S::WARPS + warp;
  const int total = prefix[B];
  const int W = (total + nseg - 1) / nseg;
  int f = min(seg * W, total);
  const int end = min(f + W, total);
  // the unit (sequence b, KV head kvh) holding position f: [ustart, uend) of npg pages;
  // the next unit is the next KV head of the same sequence unless that was the last
  int ub = -1, ukvh = 0, unpg = 0, ustart = 0, uend = 0;
  auto take = [&](ScoreChunk &c) -> bool {         // next chunk of the segment
    if (f >= end) return false;
    if (f >= uend) {
      if (ub >= 0 && ukvh + 1 < Hkv) {
        ++ukvh;
        ustart = uend;
        uend += unpg;
      } else {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (prefix[mid] <= f) lo = mid; else hi = mid - 1;
        }
        ub = lo;
        unpg = (prefix[lo + 1] - prefix[lo]) / Hkv;
        ukvh = (f - prefix[lo]) / unpg;
        ustart = prefix[lo] + ukvh * unpg;
        uend = ustart + unpg;
      }
    }
    c.b = ub;
    c.kvh = ukvh;
    c.j0 = f - ustart;
    c.n = min(min(S::CH, end - f), uend - f);
    f += c.n;
    return true;
  };
  const int pshift = bs == 32 ? 1 : 0;             // 16-token pages per block: 1 or 2
  auto qrows = [&](int b, int kvh) { return q + (static_cast<size_t>(b) * Hq + kvh * G) * D; };
  // copy chunk c's summary rows into stage st and record its descriptor and the mask of
  // rows whose block-table entry is valid; a chunk that starts its unit also pulls the
  // group's query rows into L2 for the fragments built when it is scored
  int last_pair = -1;
  auto issue = [&](const ScoreChunk &c, int st) {
    uint8_t *buf = stage + st * S::BUF;
    const uint32_t bb = smem_u32(&bar[st]);
    int page = 0;
    bool ok = false;
    if (lane < c.n) {
      const int j = c.j0 + lane;
      const int phys = __ldg(block_tables + static_cast<size_t>(c.b) * max_blocks + (j >> pshift));
      ok = phys >= 0 && phys < nblocks;
      page = ok ? (phys << pshift) + (j & pshift) : 0;
    }
    const unsigned okm = __ballot_sync(0xffffffffu, ok);
    const int pair = c.b * Hkv + c.kvh;
    if (pair != last_pair && lane * 128 < G * D * 2)
      prefetch_l2(reinterpret_cast<const uint8_t *>(qrows(c.b, c.kvh)) + lane * 128);
    last_pair = pair;
    fence_proxy_async();                           // the stage was last read by ldmatrix
    __syncwarp();
    if (lane == 0) {
      desc[st] = make_int4(c.b, c.kvh, c.j0, c.n);
      okms[st] = okm;
      mbar_arrive_expect_tx(bb, __popc(okm) * S::ROWB);
    }
    __syncwarp();
    if (ok)
      bulk_load(smem_u32(buf + lane * S::ROWP),
                summ + (static_cast<size_t>(page) * Hkv + c.kvh) * 2 * D, S::ROWB, bb);
  };

  uint32_t bneg[S::NG][S::KSQ][2], bpos[S::NG][S::KSQ][2];   // B fragments of q-, q+
  int issued = 0;
  {
    ScoreChunk c;
    while (issued < ST && take(c)) issue(c, issued++);
  }
  int frag_pair = -1;
  for (int k = 0; k < issued; ++k) {
    const int st = k % ST;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar[st]), (k / ST) & 1))) {
      if (lane == 0) set_err(err, PA_DEVERR_TIMEOUT);
      for (int j = k; j < issued && j < k + ST; ++j)   // copies still in flight
        mbar_wait(smem_u32(&bar[j % ST]), (j / ST) & 1);
      return;
    }
    const int4 cd = desc[st];
    const unsigned okm_cur = okms[st];
    const uint8_t *buf = stage + st * S::BUF;
    if (cd.x * Hkv + cd.y != frag_pair) {          // a new unit: B fragments from q rows,
      frag_pair = cd.x * Hkv + cd.y;               // k pairs of the channels split by sign
      const uint16_t *qr = qrows(cd.x, cd.y);
#pragma unroll
      for (int nt = 0; nt < S::NG; ++nt) {
        const int g = nt * 8 + (lane >> 2);
#pragma unroll
        for (int kk = 0; kk < S::KSQ; ++kk)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t v =
                g < G ? __ldg(reinterpret_cast<const uint32_t *>(qr + g * D + 16 * kk + 8 * j +
                                                                 2 * (lane & 3)))
                      : 0u;
            const uint32_t neg = ((v >> 15) & 0x00010001u) * 0xFFFFu;   // halves with q < 0
            bneg[nt][kk][j] = v & neg;
            bpos[nt][kk][j] = v & ~neg;
          }
      }
    }
    float acc[S::NG][2][4];
#pragma unroll
    for (int nt = 0; nt < S::NG; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][h][i] = 0.f;
    const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int ks = 0; ks < 2 * S::KSQ; ++ks) {      // ks < KSQ: the min half, else the max half
      uint32_t a[4];
      ldsm_x4(a, smem_u32(buf + row * S::ROWP + (2 * ks + (lane >> 4)) * 16));
      const int kq = ks % S::KSQ;
#pragma unroll
      for (int nt = 0; nt < S::NG; ++nt) {
        if (ks < S::KSQ)
          mma_bf16(acc[nt][0], a, bneg[nt][kq][0], bneg[nt][kq][1]);
        else
          mma_bf16(acc[nt][1], a, bpos[nt][kq][0], bpos[nt][kq][1]);
      }
    }
    // element i of the accumulator: page (lane >> 2) + 8 (i >> 1), head 2 (lane & 3) + (i & 1)
    float best[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < S::NG; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int head = nt * 8 + 2 * (lane & 3) + (i & 1);
        if (head < G) best[i >> 1] = fmaxf(best[i >> 1], acc[nt][0][i] + acc[nt][1][i]);
      }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      best[h] = fmaxf(best[h], __shfl_xor_sync(0xffffffffu, best[h], 1));
      best[h] = fmaxf(best[h], __shfl_xor_sync(0xffffffffu, best[h], 2));
    }
    if ((lane & 3) == 0) {
      float *out = scores + (static_cast<size_t>(cd.x) * Hkv + cd.y) * max_pages + cd.z;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = (lane >> 2) + 8 * h;
        if (r < cd.w) {
          const bool ok = (okm_cur >> r) & 1u;
          if (!ok) set_err(err, PA_DEVERR_BLOCK_ID);
          out[r] = ok ? best[h] : -INFINITY;
        }
      }
    }
    __syncwarp();                                  // the stage and its record are consumed
    ScoreChunk c;
    if (issued < k + 1 + ST && take(c)) issue(c, issued++ % ST);
  }
}

constexpr int kTopkThreads = 512;

// Top-k of one (sequence, KV head) per CTA: the topk best pages by score (ties to
// the lower page index), written in increasing page order to sel[b][kvh][0..topk),
// -1 past the number of pages.  Radix select of the topk-th largest order key, eight
// bits a pass from the top (two histograms, so that clearing the next one costs no
// barrier), then one ordered compaction: each thread owns a contiguous run of pages,
// and a block-wide scan of its (above, equal) counts places its chosen pages.
__global__ void __launch_bounds__(kTopkThreads) quest_topk_kernel(
    const float *scores, const int32_t *seq_lens, int Hkv, int cap, int max_pages, int topk,
    int32_t *sel) {
  extern __shared__ uint32_t key[];              // [npg] order keys of the page scores
  __shared__ int hist[2][256];
  __shared__ unsigned long long warp_tot[kTopkThreads / 32];
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
  for (int i = tid; i < 256; i += kTopkThreads) hist[0][i] = 0;
  if (tid == 0) {
    s_prefix = 0u;
    s_kleft = topk;
  }
  __syncthreads();
  uint32_t mask = 0u;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int *h = hist[pass & 1];
    const uint32_t prefix = s_prefix;
    for (int j = tid; j < npg; j += kTopkThreads)
      if ((key[j] & mask) == prefix) atomicAdd(&h[(key[j] >> shift) & 0xFF], 1);
    // the other histogram was last read by warp 0 in the pass before: clear it for the next
    for (int i = tid; i < 256; i += kTopkThreads) hist[(pass + 1) & 1][i] = 0;
    __syncthreads();
    if (warp == 0) {
      // the highest bin whose count from the top reaches kleft: lane l holds bins
      // [8 l, 8 l + 8); suffix sums over the lanes find its lane, then its bin
      const int kleft = s_kleft;
      int c[8], mine = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = h[lane * 8 + i];
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
  const int per = (npg + kTopkThreads - 1) / kTopkThreads;
  const int j0 = min(npg, tid * per), j1 = min(npg, j0 + per);
  int gt = 0, eq = 0;
  for (int j = j0; j < j1; ++j) {
    gt += key[j] > T;
    eq += key[j] == T;
  }
  // exclusive block scan of (eq, gt) packed as the high and low halves of 64 bits
  const unsigned long long mineq = (static_cast<unsigned long long>(eq) << 32) | static_cast<unsigned>(gt);
  unsigned long long inc = mineq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = lane < kTopkThreads / 32 ? warp_tot[lane] : 0ull;
    const unsigned long long own = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long v = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += v;
    }
    if (lane < kTopkThreads / 32) warp_tot[lane] = t - own;
  }
  __syncthreads();
  const unsigned long long before = warp_tot[warp] + inc - mineq;
  const int gt_before = static_cast<int>(before & 0xFFFFFFFFull);
  int eq_seen = static_cast<int>(before >> 32);
  // equal keys are taken in page order until take_equal of them are in
  int pos = gt_before + min(eq_seen, take_equal);
  for (int j = j0; j < j1; ++j) {
    const uint32_t k = key[j];
    if (k > T || (k == T && eq_seen++ < take_equal)) out[pos++] = j;
  }
}

pa_status run_quest_summarize(const pa_shape &s, const void *k_pool, const float *k_scale,
                              void *summaries, const int64_t *slot_mapping, int32_t *err,
                              cudaStream_t stream) {
  auto launch = [&](auto kernel) {
    return launch_pdl(kernel, dim3(s.B), dim3(128), 0, stream, k_pool, k_scale,
                      static_cast<uint16_t *>(summaries), slot_mapping, s.B, s.Hkv, s.D,
                      s.block_size, static_cast<int64_t>(s.nblocks) * s.block_size, err);
  };
  const cudaError_t e = s.kv_dtype == PA_KV_FP8_E4M3 ? launch(quest_summarize_kernel<1>)
                        : s.kv_dtype == PA_KV_INT4   ? launch(quest_summarize_kernel<2>)
                                                     : launch(quest_summarize_kernel<0>);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int quest_max_pages(const pa_shape &s) {
  return static_cast<int>((static_cast<int64_t>(s.max_blocks) * s.block_size + kTile - 1) / kTile);
}

size_t quest_topk_smem(const pa_shape &s) { return static_cast<size_t>(quest_max_pages(s)) * 4; }

template <int D, int NG>
static size_t score_smem(int B) {
  return ScoreCfg<D, NG>::FIXED + (static_cast<size_t>(B) + 1) * 4;
}

size_t quest_score_smem(const pa_shape &s) {
  const bool two = s.Hq / s.Hkv > 8;
  if (s.D == 64) return two ? score_smem<64, 2>(s.B) : score_smem<64, 1>(s.B);
  return two ? score_smem<128, 2>(s.B) : score_smem<128, 1>(s.B);
}

template <class S>
static cudaError_t launch_score(const pa_shape &s, int sms, const void *q, const void *summaries,
                                const int32_t *block_tables, const int32_t *seq_lens,
                                float *page_scores, int32_t *err, cudaStream_t stream) {
  const size_t smem = S::FIXED + (static_cast<size_t>(s.B) + 1) * 4;
  cudaError_t e = cudaFuncSetAttribute(quest_score_kernel<S>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // as many CTAs per SM as shared memory holds (227 KB usable, 1 KB reserved per CTA)
  const int per_sm = std::max(1, std::min(4, static_cast<int>((227 * 1024) / (smem + 1024))));
  const int grid = per_sm * sms;
  return launch_pdl(quest_score_kernel<S>, dim3(grid), dim3(S::THREADS), smem, stream,
                    static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(summaries),
                    block_tables, seq_lens, s.B, s.Hq, s.Hkv, s.block_size, s.nblocks,
                    s.max_blocks, quest_max_pages(s), grid * S::WARPS, page_scores, err);
}

pa_status run_quest_select(const pa_shape &s, const void *q, const void *summaries,
                           const int32_t *block_tables, const int32_t *seq_lens, int topk,
                           float *page_scores, int32_t *selected, int32_t *err,
                           cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  const int max_pages = quest_max_pages(s);
  const bool two = s.Hq / s.Hkv > 8;
  cudaError_t e;
  if (s.D == 64)
    e = two ? launch_score<ScoreCfg<64, 2>>(s, sms, q, summaries, block_tables, seq_lens,
                                             page_scores, err, stream)
            : launch_score<ScoreCfg<64, 1>>(s, sms, q, summaries, block_tables, seq_lens,
                                             page_scores, err, stream);
  else
    e = two ? launch_score<ScoreCfg<128, 2>>(s, sms, q, summaries, block_tables, seq_lens,
                                              page_scores, err, stream)
            : launch_score<ScoreCfg<128, 1>>(s, sms, q, summaries, block_tables, seq_lens,
                                              page_scores, err, stream);
  if (e != cudaSuccess) return PA_ERR_CUDA;
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
