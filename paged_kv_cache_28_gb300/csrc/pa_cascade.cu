// pa_cascade.cu -- prefix-aware (cascade) decode: attention over the tokens a group
// of sequences shares, computed once for all its members.
//
// "appendonly", "Prefix sharing is where the real win lives": most requests start
// with the same system prompt, so many block tables point at the same physical
// blocks.  The split decode would stream those blocks once per sequence (from L2
// after the first reader).  Here the query rows of all members of a group, for one
// KV head, are stacked into one matrix Q_g (members x G rows) and attended over the
// group's shared tiles in one pass:
//     S = Q_g K^T, online softmax per row, O = P V,
// a dense contraction that runs on the tensor cores with Q as the A operand.  Each
// row leaves a partial (o, lse) over the shared tiles; the split kernel covers the
// rest of each sequence and the merge joins them (exact up to rounding order: the
// same log-sum-exp merge as for split pieces).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kCasRows = 64;        // query rows per work item: 4 warps x 16 rows
constexpr int kCasWarps = 4;
constexpr int kCasThreads = 32 * kCasWarps;
constexpr int kCasStages = 4;

template <int D_>
struct CasCfg {
  static constexpr int D = D_;
  static constexpr int ROW = 2 * D;             // bytes of one token's head row (bf16)
  static constexpr int BOXES = ROW / 128;       // 128-byte TMA boxes per row
  static constexpr int KV_BYTES = kTile * ROW;  // one 16-token tile of K (or V)
  static constexpr int STAGE = 2 * KV_BYTES;
  static constexpr int KS = D / 16;             // QK k-steps
  static constexpr int DT = D / 8;              // PV n-tiles (8 output channels each)
  static constexpr int FIXED = 1024 + kCasStages * STAGE + 2 * kCasStages * 8;
  static_assert(ROW % 128 == 0, "rows are whole 128-byte boxes");
};

struct CascadeParams {
  const uint16_t *q;
  const int32_t *block_tables;
  const int32_t *group_offsets;
  const int32_t *group_seqs;
  const int32_t *group_prefix_len;
  int32_t *member;          // cascade workspace regions (see CascadeLayout)
  int32_t *tiles;
  int32_t *pieces;
  float *lse;
  float *o;
  int32_t *next;            // work-item counter
  int32_t *err;
  int num_groups, B, Hq, Hkv, G, bs, nblocks, max_blocks;
  float sl2;                // sm_scale * log2(e)
};

constexpr int kCasPieceTiles = 64;  // a shared prefix longer than this is cut into pieces

// Work of group g: rows = members x G, chunks of 64 rows, shared tiles (at most the
// block table's reach) cut into `pieces` non-empty runs of `tp` tiles (the last
// may be shorter); one item per (KV head, chunk, piece).
struct GroupWork {
  int members, tiles, pieces, tp, chunks;
  __device__ __forceinline__ int items(int Hkv) const { return Hkv * chunks * pieces; }
};

__device__ __forceinline__ GroupWork group_work(const CascadeParams &p, int g) {
  GroupWork w;
  w.members = max(0, p.group_offsets[g + 1] - p.group_offsets[g]);
  w.tiles = min(max(0, p.group_prefix_len[g]), p.max_blocks * p.bs) / kTile;
  if (w.members == 0 || w.tiles == 0) {
    w.tiles = w.pieces = w.tp = w.chunks = 0;
    return w;
  }
  const int want = min(kCascadePieces, (w.tiles + kCasPieceTiles - 1) / kCasPieceTiles);
  w.tp = (w.tiles + want - 1) / want;
  w.pieces = (w.tiles + w.tp - 1) / w.tp;       // every piece holds at least one tile
  w.chunks = (w.members * p.G + kCasRows - 1) / kCasRows;
  return w;
}

// Per-sequence cascade info for the split kernel and the merge: member slot, shared
// tiles, pieces (one CTA).
__global__ void __launch_bounds__(256) cascade_plan_kernel(const CascadeParams p) {
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();                                    // the previous step's merge reads these
  if (tid == 0) *p.next = 0;
  for (int b = tid; b < p.B; b += blockDim.x) {
    p.member[b] = -1;
    p.tiles[b] = 0;
    p.pieces[b] = 0;
  }
  __syncthreads();
  const int nm = p.group_offsets[p.num_groups];
  for (int i = tid; i < nm; i += blockDim.x) {
    int lo = 0, hi = p.num_groups - 1;           // group of member i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.group_offsets[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int b = p.group_seqs[i];
    if (i >= p.B || b < 0 || b >= p.B || atomicCAS(&p.member[b], -1, i) != -1) {
      set_err(p.err, PA_DEVERR_SEQ_LEN);         // not a sequence, in two groups, too many
      continue;
    }
    const GroupWork w = group_work(p, lo);
    p.tiles[b] = w.tiles;
    p.pieces[b] = w.pieces;
  }
}

template <int D>
__global__ void __launch_bounds__(kCasThreads, 3)
    cascade_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const CascadeParams p) {
  using C = CasCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(stages + kCasStages * C::STAGE);
  uint64_t *empty = full + kCasStages;            // all four warps are done with the stage
  int32_t *gprefix = reinterpret_cast<int32_t *>(empty + kCasStages);  // [num_groups + 1]
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, tig = lane & 3;
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kCasStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kCasWarps);
    }
    fence_mbar_init();
    s_abort = 0;
  }
  // items per group (caller inputs only): block-wide exclusive scan into shared memory
  {
    __shared__ int warp_total[kCasWarps];
    const int per = (p.num_groups + kCasThreads - 1) / kCasThreads;
    const int lo = min(p.num_groups, tid * per), hi = min(p.num_groups, lo + per);
    int mine = 0;
    for (int g = lo; g < hi; ++g) mine += group_work(p, g).items(p.Hkv);
    int inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) warp_total[warp] = inc;
    __syncthreads();
    int run = inc - mine;
    for (int w2 = 0; w2 < warp; ++w2) run += warp_total[w2];
    for (int g = lo; g < hi; ++g) {
      gprefix[g] = run;
      run += group_work(p, g).items(p.Hkv);
    }
    if (tid == kCasThreads - 1) gprefix[p.num_groups] = run;   // its range ends the list
    __syncthreads();
  }
  // launched after the plan kernel (and so after the cache write) has finished

  const int total = gprefix[p.num_groups];
  uint32_t it = 0;                               // tiles consumed by this CTA so far
  __shared__ int s_item;
  for (;;) {                                     // items from the shared counter
    if (tid == 0) s_item = atomicAdd(p.next, 1);
    __syncthreads();
    const int item = s_item;
    __syncthreads();
    if (item >= total) break;
    int g = 0;
    {
      int lo = 0, hi = p.num_groups - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (gprefix[mid] <= item) lo = mid; else hi = mid - 1;
      }
      g = lo;
    }
    const GroupWork w = group_work(p, g);
    const int off = p.group_offsets[g];
    int r = item - gprefix[g];
    const int kvh = r / (w.chunks * w.pieces);
    r -= kvh * w.chunks * w.pieces;
    const int chunk = r / w.pieces, piece = r - chunk * w.pieces;
    const int t0 = piece * w.tp, n = min(w.tiles, t0 + w.tp) - t0;   // n >= 1
    const int32_t *row = p.block_tables + static_cast<size_t>(max(p.group_seqs[off], 0)) * p.max_blocks;

    // tile t0 + j of the item is the CTA's (it + j)-th tile, into stage (it + j) % S once
    // every warp has released that stage's previous tile; false: a wait gave up
    auto issue = [&](int j) -> bool {
      const uint32_t u = it + j;
      const int s = u % kCasStages;
      if (u >= kCasStages &&
          !mbar_wait(smem_u32(&empty[s]), ((u - kCasStages) / kCasStages) & 1u))
        return false;
      const int t = t0 + j;
      int phys = __ldg(row + (t * kTile) / p.bs);
      if (phys < 0 || phys >= p.nblocks) {
        set_err(p.err, PA_DEVERR_BLOCK_ID);
        phys = kInvalidPhys;                     // box below the tensor: zero fill
      }
      const int y = (phys == kInvalidPhys) ? p.nblocks * p.bs : phys * p.bs + (t * kTile) % p.bs;
      const uint32_t bar = smem_u32(&full[s]);
      const uint32_t dst = smem_u32(stages + s * C::STAGE);
      fence_proxy_async();
      mbar_arrive_expect_tx(bar, 2 * C::KV_BYTES);
#pragma unroll
      for (int h = 0; h < C::BOXES; ++h) {
        const int x = kvh * D + h * 64;
        tma_load_2d(dst + h * (kTile * 128), &tmK, x, y, bar);
        tma_load_2d(dst + C::KV_BYTES + h * (kTile * 128), &tmV, x, y, bar);
      }
      return true;
    };
    int issued = 0;                              // tiles of this item given to TMA (thread 0)
    if (tid == 0)
      for (; issued < kCasStages && issued < n; ++issued)
        if (!issue(issued)) {
          set_err(p.err, PA_DEVERR_TIMEOUT);
          s_abort = 1;
          break;
        }

    // the warp's 16 query rows: row R = chunk * 64 + warp * 16 + (g4 | g4 + 8) is
    // query head R % G of member R / G; A fragments over k-steps of 16 channels
    uint32_t qa[C::KS][4];
    int rmember[2], rhead[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int R = chunk * kCasRows + warp * 16 + g4 + 8 * h;
      rmember[h] = R / p.G;
      rhead[h] = R - rmember[h] * p.G;
      // rows past the members pad the last chunk; member slots are bounded by B
      if (rmember[h] >= w.members || off + rmember[h] >= p.B) rmember[h] = -1;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t *qr = nullptr;
      if (rmember[h] >= 0) {
        const int b = p.group_seqs[off + rmember[h]];
        if (b >= 0 && b < p.B)
          qr = reinterpret_cast<const uint32_t *>(
              p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.G + rhead[h]) * D);
      }
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        qa[ks][h] = qr ? __ldg(qr + ks * 8 + tig) : 0u;         // channels 16ks + 2tig..
        qa[ks][h + 2] = qr ? __ldg(qr + ks * 8 + 4 + tig) : 0u; // 16ks + 8 + 2tig..
      }
    }
    float acc[C::DT][4];
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[dt][i] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    __syncthreads();                             // s_abort from the first issues
    int j = 0;
    for (; j < n && !*reinterpret_cast<volatile int *>(&s_abort); ++j) {
      const int s = (it + j) % kCasStages;
      const uint32_t parity = ((it + j) / kCasStages) & 1u;
      if (!mbar_wait(smem_u32(&full[s]), parity)) {   // bounded wait gave up
        set_err(p.err, PA_DEVERR_TIMEOUT);
        s_abort = 1;
        break;
      }
      const uint32_t kt = smem_u32(stages + s * C::STAGE), vt = kt + C::KV_BYTES;

      // ---- S = Q K^T for 16 rows x 16 tokens (two n-tiles of 8 tokens)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          const int c16 = 2 * ks + ((lane >> 3) & 1);
          uint32_t b[4];
          ldsm_x4(b, kt + (c16 >> 3) * (kTile * 128) + tok * 128 + (((c16 & 7) ^ (tok & 7)) << 4));
          mma_bf16(sc[0], qa[ks], b[0], b[1]);
          mma_bf16(sc[1], qa[ks], b[2], b[3]);
        }
      }
      // ---- online softmax per row (log2 domain); element i: row g4 + 8 (i >> 1).  A
      // row's reference maximum moves only when a score exceeds it by more than 8, so
      // p <= 2^8 (o and l share the reference); a tile that moves none skips the
      // reduction across lanes and the accumulator rescale.
      float pr[2][4];
      bool over = false;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sc[nt][i] *= p.sl2;
          over |= sc[nt][i] > m[i >> 1] + 8.f;
        }
      if (__any_sync(0xffffffffu, over)) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float mx = fmaxf(fmaxf(sc[0][2 * h], sc[0][2 * h + 1]), fmaxf(sc[1][2 * h], sc[1][2 * h + 1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float mnew = fmaxf(m[h], mx);
          const float alpha = ex2(m[h] - mnew);
          m[h] = mnew;
          l[h] *= alpha;
#pragma unroll
          for (int dt = 0; dt < C::DT; ++dt) {
            acc[dt][2 * h] *= alpha;
            acc[dt][2 * h + 1] *= alpha;
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v = ex2(sc[nt][2 * h + e] - m[h]);
            pr[nt][2 * h + e] = v;
            l[h] += v;
          }
      // ---- P as the A operand (the accumulator layout is the A layout): bf16 hi + lo
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int nt = i >> 1, h = i & 1;        // a0: row g4, tokens 0-7; a1: row g4 + 8; ...
        const float p0 = pr[nt][2 * h], p1 = pr[nt][2 * h + 1];
        ph[i] = pack_bf16(p0, p1);
        pl[i] = pack_bf16(p0 - bf16_lo(ph[i]), p1 - bf16_hi(ph[i]));
      }
      // ---- O += P V: V^T fragments by ldmatrix.trans on the token rows
      {
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int jd = 0; jd < C::DT / 2; ++jd) {
          const int c16 = 2 * jd + (lane >> 4);
          uint32_t b[4];
          ldsm_x4_trans(b, vt + (c16 >> 3) * (kTile * 128) + tok * 128 +
                               (((c16 & 7) ^ (tok & 7)) << 4));
          mma_bf16(acc[2 * jd], ph, b[0], b[1]);
          mma_bf16(acc[2 * jd], pl, b[0], b[1]);
          mma_bf16(acc[2 * jd + 1], ph, b[2], b[3]);
          mma_bf16(acc[2 * jd + 1], pl, b[2], b[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));   // this warp is done with stage s
      // refill the stage of tile j - 1 (released by the slower warps by now)
      if (tid == 0 && j >= 1 && issued < n && issued == j - 1 + kCasStages) {
        if (!issue(issued)) {
          set_err(p.err, PA_DEVERR_TIMEOUT);
          s_abort = 1;
        } else {
          ++issued;
        }
      }
    }
    if (__syncthreads_or(*reinterpret_cast<volatile int *>(&s_abort))) {
      if (tid == 0)                              // let the copies in flight land first
        for (int k = j; k < issued; ++k)
          mbar_wait(smem_u32(&full[(it + k) % kCasStages]), ((it + k) / kCasStages) & 1u);
      return;
    }
    it += n;

    // ---- partial of each valid row: o = acc / l, lse = (m + log2 l) ln 2
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float lt = l[h];
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      if (rmember[h] < 0) continue;
      const size_t slot =
          ((static_cast<size_t>(off + rmember[h]) * p.Hkv + kvh) * kCascadePieces + piece) * p.G +
          rhead[h];
      const float inv = 1.f / lt;
      float *orow = p.o + slot * D;
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt)
        *reinterpret_cast<float2 *>(orow + dt * 8 + 2 * tig) =
            make_float2(acc[dt][2 * h] * inv, acc[dt][2 * h + 1] * inv);
      if (tig == 0) p.lse[slot] = (m[h] + __log2f(lt)) * kLn2;
    }
  }
}

static CascadeParams cascade_params(const pa_shape &s, const void *q, const int32_t *bt,
                                    const pa_decode_opts &opts, float sm_scale, int32_t *err);

pa_status run_cascade_plan(const pa_shape &s, const pa_decode_opts &opts, int32_t *err,
                           cudaStream_t stream) {
  const CascadeParams p = cascade_params(s, nullptr, nullptr, opts, 1.f, err);
  return launch_pdl(cascade_plan_kernel, dim3(1), dim3(256), 0, stream, p) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

static CascadeParams cascade_params(const pa_shape &s, const void *q, const int32_t *bt,
                                    const pa_decode_opts &opts, float sm_scale, int32_t *err) {
  const CascadeLayout cl = cascade_layout(s.B, s.Hq, s.D);
  uint8_t *ws = static_cast<uint8_t *>(opts.cascade_workspace);
  CascadeParams p{};
  p.q = static_cast<const uint16_t *>(q);
  p.block_tables = bt;
  p.group_offsets = opts.group_offsets;
  p.group_seqs = opts.group_seqs;
  p.group_prefix_len = opts.group_prefix_len;
  p.member = reinterpret_cast<int32_t *>(ws + cl.member);
  p.tiles = reinterpret_cast<int32_t *>(ws + cl.tiles);
  p.pieces = reinterpret_cast<int32_t *>(ws + cl.pieces);
  p.lse = reinterpret_cast<float *>(ws + cl.lse);
  p.o = reinterpret_cast<float *>(ws + cl.o);
  p.next = reinterpret_cast<int32_t *>(ws + cl.next);
  p.err = err;
  p.num_groups = opts.num_prefix_groups;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = s.Hq / s.Hkv;
  p.bs = s.block_size;
  p.nblocks = s.nblocks;
  p.max_blocks = s.max_blocks;
  p.sl2 = sm_scale * kLog2e;
  return p;
}

pa_status run_cascade(const pa_shape &s, const CUtensorMap &mk, const CUtensorMap &mv,
                      const void *q, const int32_t *bt, const pa_decode_opts &opts,
                      float sm_scale, int32_t *err, int ctas, cudaStream_t stream) {
  const CascadeParams p = cascade_params(s, q, bt, opts, sm_scale, err);
  const int grid = ctas;
  cudaError_t e;
  if (s.D == 128) {
    const size_t smem = CasCfg<128>::FIXED + (static_cast<size_t>(p.num_groups) + 1) * 4;
    e = cudaFuncSetAttribute(cascade_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) {
      cascade_kernel<128><<<grid, kCasThreads, smem, stream>>>(mk, mv, p);
      e = cudaGetLastError();
    }
  } else {
    const size_t smem = CasCfg<64>::FIXED + (static_cast<size_t>(p.num_groups) + 1) * 4;
    e = cudaFuncSetAttribute(cascade_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) {
      cascade_kernel<64><<<grid, kCasThreads, smem, stream>>>(mk, mv, p);
      e = cudaGetLastError();
    }
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
