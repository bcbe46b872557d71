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

// KIND 0: bf16 pools.  1: E4M3 code pools, 2: 4-bit code pools (offset-binary nibbles,
// element 2j in the low nibble of byte j), each with one fp32 scale per (block, KV
// head) for K and for V ("KV Cache Engineering for LLM Serving", section 8), D = 128.
template <int D_, int KIND_>
struct CasCfg {
  static constexpr int D = D_;
  static constexpr int KIND = KIND_;
  static constexpr bool FP8 = KIND == 1, INT4 = KIND == 2, QUANT = KIND != 0;
  static constexpr int ROW = INT4 ? D / 2 : (FP8 ? D : 2 * D);   // bytes of a head row
  static constexpr int BOX = ROW < 128 ? ROW : 128;   // TMA box width (= swizzle span)
  static constexpr int BOXES = ROW / BOX;
  static constexpr int KV_BYTES = kTile * ROW;  // one 16-token tile of K (or V)
  static constexpr int STAGE = 2 * KV_BYTES;
  static constexpr int KS = D / 16;             // QK k-steps
  static constexpr int DT = D / 8;              // PV n-tiles (8 output channels each)
  // stages, full and empty barriers, each stage's (k scale, v scale)
  static constexpr int FIXED = 1024 + kCasStages * STAGE + 2 * kCasStages * 8 + kCasStages * 8;
  static_assert(ROW % BOX == 0 && (BOX == 128 || (INT4 && BOX == 64)), "whole boxes");
  static_assert(STAGE % 1024 == 0, "swizzled tiles must be 1024-byte aligned");
  static_assert(!QUANT || D == 128, "quantised pools have D = 128");
};

struct CascadeParams {
  const uint16_t *q;
  const float *k_scale;     // E4M3 pools: [nblocks, Hkv] scales, else null
  const float *v_scale;
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

// E4M3 tiles: the mma's k order within a 16-channel step is permuted so that a lane's
// four consecutive codes (one ldmatrix byte-pair word) give both of its K^T fragment
// registers: k slots 2t, 2t+1 <- channels 4t, 4t+1 and 2t+8, 2t+9 <- 4t+2, 4t+3.  The
// query rows (A operand) take the same order.  P V reads V codes by ldmatrix.trans on
// the byte-pair view: lane (r, t) receives tokens 2t, 2t+1 of channels 2r, 2r+1; one
// byte permute splits them into channel 2r (even n-tile) and 2r+1 (odd n-tile).
__device__ __forceinline__ uint32_t f16x2_of_bf16x2(uint32_t w, float up) {
  return pack_f16(bf16_lo(w) * up, bf16_hi(w) * up);
}

// 4-bit tiles (64-byte rows, 64-byte swizzle): a lane's ldmatrix byte-pair word holds
// eight consecutive channels 8t..8t+7 of one token; int4_pair_f16 gives the pairs
// (i, i+4), which fill k-step 2c with (0,4), (1,5) and k-step 2c+1 with (2,6), (3,7)
// (chunk c: channels 32c..32c+31); the query rows take the same order.  For P V the
// transposed word holds channels 4r..4r+3 of tokens 2t and 2t+1, so int4_pair_f16(., j)
// is the fragment of channel 4r + j: n-tile 4c + j covers channels 32c + 4r + j.
__device__ __forceinline__ uint32_t swz64(uint32_t tile, int row, int c) {
  return tile + row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
}

template <int D, int KIND>
__global__ void __launch_bounds__(kCasThreads, 3)
    cascade_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const CascadeParams p) {
  using C = CasCfg<D, KIND>;
  constexpr bool FP8 = C::FP8, INT4 = C::INT4, QUANT = C::QUANT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(stages + kCasStages * C::STAGE);
  uint64_t *empty = full + kCasStages;            // all four warps are done with the stage
  float *scl = reinterpret_cast<float *>(empty + kCasStages);   // [stage][k scale, v scale]
  int32_t *gprefix = reinterpret_cast<int32_t *>(scl + 2 * kCasStages);  // [num_groups + 1]
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, tig = lane & 3;
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kCasStages; ++s) {
      mbar_init(smem_u32(&full[s]), QUANT ? 2 : 1);  // codes: plus the scales' cp.async
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
      if constexpr (QUANT) {                     // the tile's block scales, with the tile
        float *sc = scl + 2 * s;
        if (phys != kInvalidPhys) {
          cp_async_4(smem_u32(sc), p.k_scale + static_cast<size_t>(phys) * p.Hkv + kvh);
          cp_async_4(smem_u32(sc + 1), p.v_scale + static_cast<size_t>(phys) * p.Hkv + kvh);
        } else {
          sc[0] = sc[1] = 0.f;
        }
        cp_async_arrive(bar);
      }
      fence_proxy_async();
      mbar_arrive_expect_tx(bar, 2 * C::KV_BYTES);
      constexpr int kEB = QUANT ? 1 : 2;          // bytes per tensor-map element
#pragma unroll
      for (int h = 0; h < C::BOXES; ++h) {
        const int x = (kvh * C::ROW + h * C::BOX) / kEB;
        tma_load_2d(dst + h * (kTile * C::BOX), &tmK, x, y, bar);
        tma_load_2d(dst + C::KV_BYTES + h * (kTile * C::BOX), &tmV, x, y, bar);
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
    float qshift[2] = {1.f, 1.f};                // codes: 2^-k undoing each row's scaling
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t *qr = nullptr;
      if (rmember[h] >= 0) {
        const int b = p.group_seqs[off + rmember[h]];
        if (b >= 0 && b < p.B)
          qr = reinterpret_cast<const uint32_t *>(
              p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.G + rhead[h]) * D);
      }
      if constexpr (!QUANT) {
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          qa[ks][h] = qr ? __ldg(qr + ks * 8 + tig) : 0u;         // channels 16ks + 2tig..
          qa[ks][h + 2] = qr ? __ldg(qr + ks * 8 + 4 + tig) : 0u; // 16ks + 8 + 2tig..
        }
      } else {
        // the permuted k order, scaled by 2^k so that the row's largest magnitude sits
        // just below 2^15: exact in f16.  E4M3: raw[ks] = channels 16ks + 4tig + {0,1},
        // {2,3}.  4-bit: raw[2c], raw[2c + 1] = channels 32c + 8tig + {0,1}, {2,3} and
        // {4,5}, {6,7}.
        uint32_t raw[C::KS][2];
        float amax = 0.f;
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          const int w = INT4 ? (ks >> 1) * 16 + 4 * tig + (ks & 1) * 2 : ks * 8 + 2 * tig;
          raw[ks][0] = qr ? __ldg(qr + w) : 0u;
          raw[ks][1] = qr ? __ldg(qr + w + 1) : 0u;
#pragma unroll
          for (int e = 0; e < 2; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(raw[ks][e])), fabsf(bf16_hi(raw[ks][e]))));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));   // the row's quad
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int k = 0;
        if (amax > 0.f) {
          const int e = ((__float_as_uint(amax) >> 23) & 0xFF) - 126;   // amax < 2^e
          k = min(max(15 - e, -100), 100);
        }
        const float up = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
        qshift[h] = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          if constexpr (INT4) {
            // k-step 2c: (0,4), (1,5); 2c + 1: (2,6), (3,7) of the lane's eight channels
            const uint32_t lo4 = raw[ks & ~1][0], lo6 = raw[ks & ~1][1];   // 0,1 / 2,3
            const uint32_t hi4 = raw[ks | 1][0], hi6 = raw[ks | 1][1];     // 4,5 / 6,7
            const uint32_t e = (ks & 1) ? lo6 : lo4, f = (ks & 1) ? hi6 : hi4;
            qa[ks][h] = pack_f16(bf16_lo(e) * up, bf16_lo(f) * up);
            qa[ks][h + 2] = pack_f16(bf16_hi(e) * up, bf16_hi(f) * up);
          } else {
            qa[ks][h] = f16x2_of_bf16x2(raw[ks][0], up);
            qa[ks][h + 2] = f16x2_of_bf16x2(raw[ks][1], up);
          }
        }
      }
    }
    float acc[C::DT][4];
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[dt][i] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    // codes: the accumulator is in units of vref (the item's first nonzero V scale, or
    // a later one when the ratio leaves [kRatMin, kRatMax]); vinv = 0 before it
    float vref = 1.f, vinv = 0.f;

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
      if constexpr (!QUANT) {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          const int c16 = 2 * ks + ((lane >> 3) & 1);
          uint32_t b[4];
          ldsm_x4(b, kt + (c16 >> 3) * (kTile * 128) + tok * 128 + (((c16 & 7) ^ (tok & 7)) << 4));
          mma_bf16(sc[0], qa[ks], b[0], b[1]);
          mma_bf16(sc[1], qa[ks], b[2], b[3]);
        }
      } else if constexpr (INT4) {
        // matrices: tokens 0-7 / 8-15 of 32-code chunks c and c + 1
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int c0 = 0; c0 < D / 32; c0 += 2) {
          uint32_t b[4];
          ldsm_x4(b, swz64(kt, tok, c0 + (lane >> 4)));
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              const uint32_t w = b[2 * u + nt];
              const int ks = 2 * (c0 + u);
              mma_f16(sc[nt], qa[ks], int4_pair_f16(w, 0), int4_pair_f16(w, 1));
              mma_f16(sc[nt], qa[ks + 1], int4_pair_f16(w, 2), int4_pair_f16(w, 3));
            }
        }
      } else {
        // matrices: tokens 0-7 / 8-15 of 16-code chunks ks and ks + 1
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int ks = 0; ks < C::KS; ks += 2) {
          const int c = ks + (lane >> 4);
          uint32_t b[4];
          ldsm_x4(b, kt + tok * 128 + ((c ^ (tok & 7)) << 4));
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              mma_f16(sc[nt], qa[ks + u], e4m3x2_to_f16x2(b[2 * u + nt]),
                      e4m3x2_hi_to_f16x2(b[2 * u + nt]));
        }
      }
      // ---- online softmax per row (log2 domain); element i: row g4 + 8 (i >> 1).  A
      // row's reference maximum moves only when a score exceeds it by more than 8, so
      // p <= 2^8 (o and l share the reference); a tile that moves none skips the
      // reduction across lanes and the accumulator rescale.
      float pr[2][4];
      bool over = false;
      float ssc[2] = {p.sl2, p.sl2};             // raw mma score -> log2-domain score
      float rat = 1.f;                           // codes: tile V scale / accumulator's
      if constexpr (QUANT) {
        const float2 tsc = *reinterpret_cast<const float2 *>(scl + 2 * s);   // k, v scale
        ssc[0] = p.sl2 * tsc.x * qshift[0];
        ssc[1] = p.sl2 * tsc.x * qshift[1];
        rat = tsc.y * vinv;                      // warp-uniform; 0 for a zero V scale
        if (tsc.y > 0.f && !(rat <= kRatMax && rat >= kRatMin)) {
          const float f = vref / tsc.y;          // re-express in the tile's scale
#pragma unroll
          for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[dt][i] *= f;
          vref = tsc.y;
          vinv = 1.f / tsc.y;
          rat = 1.f;
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sc[nt][i] *= ssc[i >> 1];
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
      // ---- P as the A operand (the accumulator layout is the A layout), hi + lo terms:
      // bf16 against bf16 V; f16 times the V-scale ratio against code V
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int nt = i >> 1, h = i & 1;        // a0: row g4, tokens 0-7; a1: row g4 + 8; ...
        const float p0 = pr[nt][2 * h], p1 = pr[nt][2 * h + 1];
        if constexpr (!QUANT) {
          ph[i] = pack_bf16(p0, p1);
          pl[i] = pack_bf16(p0 - bf16_lo(ph[i]), p1 - bf16_hi(ph[i]));
        } else {
          const float a0 = p0 * rat, a1 = p1 * rat;
          ph[i] = pack_f16(a0, a1);
          const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&ph[i]));
          pl[i] = pack_f16(a0 - hf.x, a1 - hf.y);
        }
      }
      // ---- O += P V: V^T fragments by ldmatrix.trans on the token rows
      if constexpr (INT4) {
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int c0 = 0; c0 < D / 32; c0 += 2) {
          uint32_t b[4];
          ldsm_x4_trans(b, swz64(vt, tok, c0 + (lane >> 4)));
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int n = 4 * (c0 + u) + j;
              const uint32_t v0 = int4_pair_f16(b[2 * u], j), v1 = int4_pair_f16(b[2 * u + 1], j);
              mma_f16(acc[n], ph, v0, v1);
              mma_f16(acc[n], pl, v0, v1);
            }
        }
      } else if constexpr (FP8) {
        // n-tile 2c + e: channels 16c + 2r + e (r = lane / 4) of 16-code chunk c
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int jc = 0; jc < D / 16; jc += 2) {
          const int c = jc + (lane >> 4);
          uint32_t b[4];
          ldsm_x4_trans(b, vt + tok * 128 + ((c ^ (tok & 7)) << 4));
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t x0 = __byte_perm(b[2 * u], 0u, 0x3120);       // tokens 2t, 2t+1
            const uint32_t x1 = __byte_perm(b[2 * u + 1], 0u, 0x3120);   // tokens 2t+8, 2t+9
            const int n0 = 2 * (jc + u);
            const uint32_t e0 = e4m3x2_to_f16x2(x0), e1 = e4m3x2_to_f16x2(x1);
            const uint32_t o0 = e4m3x2_hi_to_f16x2(x0), o1 = e4m3x2_hi_to_f16x2(x1);
            mma_f16(acc[n0], ph, e0, e1);
            mma_f16(acc[n0], pl, e0, e1);
            mma_f16(acc[n0 + 1], ph, o0, o1);
            mma_f16(acc[n0 + 1], pl, o0, o1);
          }
        }
      } else {
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
      const float inv = (QUANT ? vref : 1.f) / lt;
      float *orow = p.o + slot * D;
      if constexpr (INT4) {  // n-tile 4c + j holds channels 32c + 8tig + j and + 4 + j
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float *o8 = orow + 32 * c + 8 * tig;
          *reinterpret_cast<float4 *>(o8) =
              make_float4(acc[4 * c][2 * h] * inv, acc[4 * c + 1][2 * h] * inv,
                          acc[4 * c + 2][2 * h] * inv, acc[4 * c + 3][2 * h] * inv);
          *reinterpret_cast<float4 *>(o8 + 4) =
              make_float4(acc[4 * c][2 * h + 1] * inv, acc[4 * c + 1][2 * h + 1] * inv,
                          acc[4 * c + 2][2 * h + 1] * inv, acc[4 * c + 3][2 * h + 1] * inv);
        }
      } else if constexpr (FP8) {   // n-tiles 2c, 2c + 1 hold channels 16c + 4tig + {0, 2} and {1, 3}
#pragma unroll
        for (int c = 0; c < D / 16; ++c)
          *reinterpret_cast<float4 *>(orow + 16 * c + 4 * tig) =
              make_float4(acc[2 * c][2 * h] * inv, acc[2 * c + 1][2 * h] * inv,
                          acc[2 * c][2 * h + 1] * inv, acc[2 * c + 1][2 * h + 1] * inv);
      } else {
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt)
          *reinterpret_cast<float2 *>(orow + dt * 8 + 2 * tig) =
              make_float2(acc[dt][2 * h] * inv, acc[dt][2 * h + 1] * inv);
      }
      if (tig == 0) p.lse[slot] = (m[h] + __log2f(lt)) * kLn2;
    }
  }
}

static CascadeParams cascade_params(const pa_shape &s, const void *q, const int32_t *bt,
                                    const float *k_scale, const float *v_scale,
                                    const pa_decode_opts &opts, float sm_scale, int32_t *err);

pa_status run_cascade_plan(const pa_shape &s, const pa_decode_opts &opts, int32_t *err,
                           cudaStream_t stream) {
  const CascadeParams p = cascade_params(s, nullptr, nullptr, nullptr, nullptr, opts, 1.f, err);
  return launch_pdl(cascade_plan_kernel, dim3(1), dim3(256), 0, stream, p) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

static CascadeParams cascade_params(const pa_shape &s, const void *q, const int32_t *bt,
                                    const float *k_scale, const float *v_scale,
                                    const pa_decode_opts &opts, float sm_scale, int32_t *err) {
  const CascadeLayout cl = cascade_layout(s.B, s.Hq, s.D);
  uint8_t *ws = static_cast<uint8_t *>(opts.cascade_workspace);
  CascadeParams p{};
  p.q = static_cast<const uint16_t *>(q);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
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

template <int D, int KIND>
static cudaError_t launch_cascade(const CUtensorMap &mk, const CUtensorMap &mv,
                                  const CascadeParams &p, int grid, cudaStream_t stream) {
  const size_t smem = CasCfg<D, KIND>::FIXED + (static_cast<size_t>(p.num_groups) + 1) * 4;
  cudaError_t e = cudaFuncSetAttribute(cascade_kernel<D, KIND>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cascade_kernel<D, KIND><<<grid, kCasThreads, smem, stream>>>(mk, mv, p);
  return cudaGetLastError();
}

pa_status run_cascade(const pa_shape &s, const CUtensorMap &mk, const CUtensorMap &mv,
                      const void *q, const int32_t *bt, const float *k_scale,
                      const float *v_scale, const pa_decode_opts &opts, float sm_scale,
                      int32_t *err, int ctas, cudaStream_t stream) {
  const CascadeParams p = cascade_params(s, q, bt, k_scale, v_scale, opts, sm_scale, err);
  cudaError_t e;
  if (s.kv_dtype == PA_KV_FP8_E4M3)
    e = launch_cascade<128, 1>(mk, mv, p, ctas, stream);
  else if (s.kv_dtype == PA_KV_INT4)
    e = launch_cascade<128, 2>(mk, mv, p, ctas, stream);
  else if (s.D == 128)
    e = launch_cascade<128, 0>(mk, mv, p, ctas, stream);
  else
    e = launch_cascade<64, 0>(mk, mv, p, ctas, stream);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
