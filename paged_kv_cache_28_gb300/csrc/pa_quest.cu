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
  static constexpr int QB = 8 * NG * D * 2;        // the group's query rows, zero-padded
  static constexpr int BUF = CH * ROWP + QB;       // one stage
  static constexpr int WARPS = 4;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int FIXED = WARPS * 2 * BUF + WARPS * 2 * 8;   // stages + mbarriers
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
  constexpr int D = S::D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *stage = smem + warp * 2 * S::BUF;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::WARPS * 2 * S::BUF) + warp * 2;
  int32_t *prefix = reinterpret_cast<int32_t *>(smem + S::FIXED);
  const int G = Hq / Hkv;
  pdl_trigger();
  if (lane == 0) {
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    fence_mbar_init();
  }
  for (int st = 0; st < 2; ++st) {                 // query rows G .. 8 NG - 1 stay zero
    uint8_t *pad = stage + st * S::BUF + S::CH * S::ROWP + G * D * 2;
    for (int o = lane * 16; o < (8 * S::NG - G) * D * 2; o += 32 * 16)
      *reinterpret_cast<uint4 *>(pad + o) = make_uint4(0u, 0u, 0u, 0u);
  }
  const int cap = max_blocks * bs;
  scan_units<S::THREADS>(seq_lens, B, Hkv, cap, prefix);
  pdl_wait();                                      // summaries come from the launch before

  const int seg = blockIdx.x * S::WARPS + warp;
  const int total = prefix[B];
  const int W = (total + nseg - 1) / nseg;
  int f = min(seg * W, total);
  const int end = min(f + W, total);
  auto take = [&](ScoreChunk &c) -> bool {         // next chunk of the segment
    if (f >= end) return false;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= f) lo = mid; else hi = mid - 1;
    }
    const int npg = (prefix[lo + 1] - prefix[lo]) / Hkv;
    const int r = f - prefix[lo];
    c.b = lo;
    c.kvh = r / npg;
    c.j0 = r - c.kvh * npg;
    c.n = min(min(S::CH, end - f), npg - c.j0);
    f += c.n;
    return true;
  };
  // copy chunk c's summary rows (and the group's query rows when with_q) into stage
  // st; returns the mask of rows whose block-table entry is valid
  auto issue = [&](const ScoreChunk &c, int st, bool with_q) -> unsigned {
    uint8_t *buf = stage + st * S::BUF;
    const uint32_t b = smem_u32(&bar[st]);
    int page = 0;
    bool ok = false;
    if (lane < c.n) {
      const int j = c.j0 + lane;
      const int phys = __ldg(block_tables + static_cast<size_t>(c.b) * max_blocks + (j * kTile) / bs);
      ok = phys >= 0 && phys < nblocks;
      page = ok ? phys * (bs / kTile) + (j * kTile % bs) / kTile : 0;
    }
    const unsigned okm = __ballot_sync(0xffffffffu, ok);
    const uint32_t bytes = __popc(okm) * S::ROWB + (with_q ? G * D * 2 : 0);
    fence_proxy_async();                           // the stage was last read by ldmatrix
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(b, bytes);
    __syncwarp();
    if (ok)
      bulk_load(smem_u32(buf + lane * S::ROWP),
                summ + (static_cast<size_t>(page) * Hkv + c.kvh) * 2 * D, S::ROWB, b);
    if (with_q && lane == 0)
      bulk_load(smem_u32(buf + S::CH * S::ROWP),
                q + (static_cast<size_t>(c.b) * Hq + c.kvh * G) * D, G * D * 2, b);
    return okm;
  };

  uint32_t bneg[S::NG][S::KSQ][2], bpos[S::NG][S::KSQ][2];   // B fragments of q-, q+
  ScoreChunk cur, nxt;
  bool have = take(cur);
  // per stage (held in scalars so that nothing is indexed by the runtime stage):
  // valid-row masks, and bits 0/1 phase, 2/3 copies pending, 4/5 new query rows
  unsigned okm0 = 0u, okm1 = 0u;
  uint32_t flags = 0u;
  int last_pair = -1;
  if (have) {
    okm0 = issue(cur, 0, true);
    flags |= (1u << 2) | (1u << 4);
    last_pair = cur.b * Hkv + cur.kvh;
  }
  int st = 0;
  while (have) {
    const int ot = st ^ 1;
    const bool have_n = take(nxt);
    if (have_n) {                                  // prefetch the next chunk
      const int pr = nxt.b * Hkv + nxt.kvh;
      const bool nq = pr != last_pair;
      const unsigned m = issue(nxt, ot, nq);
      if (ot) okm1 = m; else okm0 = m;
      flags = (flags & ~(1u << (4 + ot))) | (1u << (2 + ot)) | (nq ? 1u << (4 + ot) : 0u);
      last_pair = pr;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar[st]), (flags >> st) & 1u))) {
      if (lane == 0) set_err(err, PA_DEVERR_TIMEOUT);
      if (flags & (1u << (2 + ot))) mbar_wait(smem_u32(&bar[ot]), (flags >> ot) & 1u);
      return;
    }
    flags ^= 1u << st;                             // phase
    flags &= ~(1u << (2 + st));                    // nothing pending
    const unsigned okm_cur = st ? okm1 : okm0;
    const uint8_t *buf = stage + st * S::BUF;
    if (flags & (1u << (4 + st))) {                                // B fragments: q rows n, k pairs of the
#pragma unroll                                     // chunk's channels, split by sign
      for (int nt = 0; nt < S::NG; ++nt)
#pragma unroll
        for (int kq = 0; kq < S::KSQ; kq += 2) {
          uint32_t r[4];
          ldsm_x4(r, smem_u32(buf + S::CH * S::ROWP + (nt * 8 + (lane & 7)) * D * 2 +
                              (2 * kq + (lane >> 3)) * 16));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t neg = ((r[i] >> 15) & 0x00010001u) * 0xFFFFu;   // halves with q < 0
            bneg[nt][kq + (i >> 1)][i & 1] = r[i] & neg;
            bpos[nt][kq + (i >> 1)][i & 1] = r[i] & ~neg;
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
      float *out = scores + (static_cast<size_t>(cur.b) * Hkv + cur.kvh) * max_pages + cur.j0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = (lane >> 2) + 8 * h;
        if (r < cur.n) {
          const bool ok = (okm_cur >> r) & 1u;
          if (!ok) set_err(err, PA_DEVERR_BLOCK_ID);
          out[r] = ok ? best[h] : -INFINITY;
        }
      }
    }
    __syncwarp();
    cur = nxt;
    have = have_n;
    st ^= 1;
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
  const int grid = 2 * sms;                       // two CTAs per SM
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
