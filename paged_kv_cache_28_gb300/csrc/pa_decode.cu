// pa_decode.cu -- paged decode attention for sm_103a.
//
// What is computed ("Taming the Token Torrent", section "Custom PagedAttention
// Kernels"; "KV Cache Engineering for LLM Serving", section 1): for every
// sequence b and query head h,
//     out[b][h] = softmax_t(sm_scale * <q[b][h], K_b[t]>) V_b[t],  t < seq_lens[b],
// where K_b / V_b are gathered through the block table and query head h reads KV
// head h / G.
//
// How (GB300 design):
//  * The unit of work is a 16-token tile of one (sequence, KV head) pair.  A
//    warp streams its tiles through a private ring of shared-memory stages.
//    Each stage is filled by TMA (two or one 128-byte-swizzled boxes for K, the
//    same for V) plus, when a new pair starts, a bulk copy of the pair's G query
//    rows; completion is tracked by one mbarrier per stage.
//  * The whole query group of a KV head is served at once with warp-level
//    tensor-core mma (m16n8k16): S^T = K Q^T (tokens x heads, the group is the
//    n = 8 side), online softmax in fp32 registers with warp shuffles, then
//    O^T += V^T P^T with P split into a high and a low 16-bit part so that the
//    weights keep ~16 significant bits.
//  * FP8 (E4M3) pools are converted to f16 in registers (exact); the per-block
//    K scale folds into the score scale and the V scale into the running
//    rescale factor, so dequantisation costs no per-element multiply.
//  * pa_decode: one CTA per (sequence, KV head); its warps take interleaved
//    tiles and merge their softmax states in shared memory at the end.
//  * pa_decode_splitkv: the tiles of all pairs, laid end to end, are cut into
//    equal segments, one per warp (flash-decoding with exact load balance).
//    Pairs inside a segment are finished in place; cut pairs leave (o, lse)
//    partials that pa_merge_lse combines.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// ----------------------------------------------------------------------------
// configuration
// ----------------------------------------------------------------------------

// Cached element kinds.
constexpr int kKindBf16 = 0;
constexpr int kKindFp8 = 1;   // E4M3 codes, one per byte
constexpr int kKindInt4 = 2;  // 4-bit codes, two per byte (offset binary)
// 4-bit codes with two adjacent KV heads per unit: their 64-byte rows sit side by
// side in the pool, so one 128-byte box per token feeds both and every fetched
// byte is used (a lone 64-byte row costs a 128-byte DRAM fetch); n-tile h serves
// the group of KV head 2 u + h.
constexpr int kKindInt4x2 = 3;
// E4M3 units of two adjacent KV heads, in the split decode: a token row holds both heads'
// 128-byte rows (two TMA boxes); n-tile h serves the group of KV head 2 u + h.  Per byte
// of codes, the tile bookkeeping (records, barrier waits, copy issue) is shared by two
// heads and each warp keeps twice the bytes in flight.  pa_decode without a workspace
// keeps one E4M3 head per unit: there the paired form's three CTAs per SM (against
// four) measured slower.
constexpr int kKindFp8x2 = 4;

template <int D_, int NT_, int KIND_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int NT = NT_;            // 8-head n-tiles (G <= 8 * NT)
  static constexpr int KIND = KIND_;
  static constexpr bool FP8 = KIND == kKindFp8 || KIND == kKindFp8x2;
  static constexpr bool INT4 = KIND == kKindInt4 || KIND == kKindInt4x2;
  static constexpr bool PAIRED = KIND == kKindInt4x2 || KIND == kKindFp8x2;
  static constexpr int HEADS = PAIRED ? 2 : 1;      // KV heads per unit
  static constexpr bool QUANT = KIND != kKindBf16;   // codes x per-(block, head) scale
  static constexpr int KS = D / 16;         // QK k-steps of 16 elements
  static constexpr int DT = D / 16;         // PV 16-row output tiles
  static constexpr int ROW = HEADS * (INT4 ? D / 2 : (FP8 ? D : 2 * D));  // bytes of a unit's row
  static constexpr int BOX_BYTES = ROW < 128 ? ROW : 128;        // TMA box width (swizzle span)
  static constexpr int BOXES = ROW / BOX_BYTES;                  // boxes per tile row
  static constexpr int BOX_X = BOX_BYTES / (KIND == kKindBf16 ? 2 : 1);  // box width in elements
  static constexpr int KV_BYTES = kTile * ROW;
  // Paired 4-bit units read a piece's query rows straight from global memory and keep
  // the Q^T fragments in a per-warp shared-memory area: no Q slot in the stages (a
  // quarter less shared memory) and 32 registers freed for the tile loop, which made
  // pa_decode on these pools 8 % faster.  Other kinds carry the query rows in the
  // stage that starts a piece and hold the fragments in registers.
  static constexpr bool QSMEM = PAIRED;
  static constexpr int Q_BYTES = QSMEM ? 0 : 8 * NT * D * 2;
  static constexpr int QF_BYTES = QSMEM ? NT * KS * 32 * 8 : 0;   // per warp: uint2 per lane
  static constexpr int STAGE_BYTES = 2 * KV_BYTES + Q_BYTES;
  static constexpr int STAGES = PAIRED ? 2 : (INT4 ? 4 : 2);
  static constexpr int WARPS = 4;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int META_BYTES = 32;     // int4 unit + k/v scale
  static constexpr int SMEM = 1024 + WARPS * (STAGES * (STAGE_BYTES + 8 + META_BYTES) + QF_BYTES);
  // CTAs per SM that shared memory allows (227 KB usable, 1 KB reserved per CTA, 4 KB
  // left for the split kernel's length scan); the register budget is held to it.
  // Paired 4-bit units stop at three: four would fit in shared memory, but their
  // 128-register budget spills and measured slower than three CTAs at up to 168.
  static constexpr int MIN_BLOCKS_RAW = (227 * 1024) / (SMEM + 1024 + 4096);
  static constexpr int MIN_BLOCKS =
      QSMEM ? 3 : (MIN_BLOCKS_RAW < 1 ? 1 : (MIN_BLOCKS_RAW > 4 ? 4 : MIN_BLOCKS_RAW));
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(!PAIRED || (NT == 2 && D == 128), "paired heads: one n-tile per KV head");
  static_assert(KV_BYTES % 1024 == 0, "swizzled tiles must be 1024-byte aligned");
  static_assert(!QSMEM || PAIRED, "query rows from global memory: paired units only");
  // pa_decode's CTA merges its warps' accumulators in the stage area; their m and l go
  // after every per-warp area (mbarrier memory is never reused)
  static_assert(WARPS * 8 * NT * D * 4 <= WARPS * STAGES * STAGE_BYTES, "pair merge must fit");
  // after them: the CTA's folded m and l (cluster launches) and one cluster mbarrier
  static constexpr int PAIR_SMEM = SMEM + (2 * WARPS + 2) * 8 * NT * 4 + 16;
};

struct Params {
  float *out;
  const uint16_t *q;
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_tables;
  const int32_t *seq_lens;
  const int32_t *shared_prefix_lens;   // optional L2 hint per sequence
  int window;                          // > 0: attend over the last `window` positions only
  int topk;                            // > 0: attend over the pages listed in sel only
  const int32_t *sel;                  // [B, Hkv, topk] chosen 16-token pages (ascending)
  const int32_t *casc_tiles;           // [B] shared tiles done by the cascade kernel, or null
  uint64_t casc_ws;                    // the cascade workspace address (0: none), for the merge
  int32_t *err;
  int B, Hq, Hkv, G, bs, nblocks, max_blocks;
  float sl2;  // sm_scale * log2(e)
  // split-KV
  int32_t *prefix_out;   // workspace copy of the tile prefix, read by the merge
  float *o_part;
  float *lse_part;
  int num_splits;        // segments (split workers)
  // pa_decode_splitkv: every piece goes to caller arrays parts_o [B, Hq, S, D] and
  // parts_lse [B, Hq, S] (S = parts_S slots per query head, unused slots -inf);
  // parts_S = 0: workspace mode (units finished in one segment go straight to out)
  int parts_S;
  float *parts_o;
  float *parts_lse;
};

// ----------------------------------------------------------------------------
// per-warp softmax state
// ----------------------------------------------------------------------------

template <class C>
struct State {
  float acc[C::NT][C::DT][4];   // O^T fragments (d x heads)
  float m[C::NT][2];            // running max, log2 domain, heads 2q, 2q+1 of each n-tile
  float l[C::NT][2];            // this thread's share of the running sum
  uint32_t qf[C::QSMEM ? 1 : C::NT][C::QSMEM ? 1 : C::KS][2]; // Q^T B-fragments (else in smem)
  float qshift;                 // quantised: 2^-k undoing the power-of-two scaling of q
  float vref[C::NT];            // quantised: V scale each n-tile's accumulator is expressed in
  float vinv[C::NT];            // 1 / vref, or 0 before the piece's first nonzero V scale

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][dt][i] = 0.f;
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
      vref[nt] = 1.f;
      vinv[nt] = 0.f;
    }
    qshift = 1.f;
  }
};

// Output row (d) of accumulator element i of d-tile dt for this lane.
template <class C>
__device__ __forceinline__ int acc_d(int dt, int i, int lane) {
  if constexpr (C::INT4)   // d-tile (chunk c = dt/2, half dt%2): rows 4r + 2 half + {0, 1}
    return (dt >> 1) * 32 + 4 * (lane >> 2) + 2 * (dt & 1) + (i >> 1);
  else if constexpr (C::FP8)
    return dt * 16 + 2 * (lane >> 2) + (i >> 1);
  else
    return dt * 16 + (lane >> 2) + (i >> 1) * 8;
}

// Load the group's Q^T fragments from the stage's Q slot ([8*NT rows][D] bf16), or,
// with C::QSMEM, from the query rows in global memory into the warp's fragment area
// qfs (lane-private: each lane reads back only what it wrote).
template <class C>
__device__ __forceinline__ void load_q(State<C> &st, uint32_t qslot, const uint16_t *qslot_ptr,
                                       uint4 *qfs, int G, int lane) {
  if constexpr (!C::QUANT) {
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int ks = 0; ks < C::KS; ks += 2) {
        uint32_t r[4];
        const int g = nt * 8 + (lane & 7);
        const int chunk = ks * 2 + (lane >> 3);
        ldsm_x4(r, qslot + g * (C::D * 2) + chunk * 16);
        st.qf[nt][ks][0] = r[0];
        st.qf[nt][ks][1] = r[1];
        st.qf[nt][ks + 1][0] = r[2];
        st.qf[nt][ks + 1][1] = r[3];
      }
  } else {
    // K codes arrive in a permuted order (see process_tile).  FP8: k-step ks, lane
    // (r, q) pairs Q[g=r][16ks + 4q + {0,1}] and Q[g=r][16ks + 4q + {2,3}].  4-bit:
    // k-step ks = 2c + u pairs Q[r][b + 2u + {0,4}] and Q[r][b + 2u + {1,5}] with
    // b = 32c + 8q.  q is scaled by 2^k so that its largest magnitude sits just
    // below 2^15 (exact in f16).
    const int r = lane >> 2, qd = lane & 3;
    uint2 raw[C::NT][C::KS];
    float amax = 0.f;
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        // 4-bit: the eight values b..b+7 of chunk c arrive as two uint2 (u = 0, 1)
        const int off = C::INT4 ? (ks >> 1) * 32 + qd * 8 + (ks & 1) * 4 : ks * 16 + qd * 4;
        const uint2 *src = reinterpret_cast<const uint2 *>(qslot_ptr + (nt * 8 + r) * C::D + off);
        if constexpr (C::QSMEM)   // global memory: rows past the group read as zeros
          raw[nt][ks] = nt * 8 + r < G ? __ldg(src) : make_uint2(0u, 0u);
        else
          raw[nt][ks] = *src;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(raw[nt][ks].x)), fabsf(bf16_hi(raw[nt][ks].x))),
                                 fmaxf(fabsf(bf16_lo(raw[nt][ks].y)), fabsf(bf16_hi(raw[nt][ks].y)))));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int k = 0;
    if (amax > 0.f) {
      const int e = ((__float_as_uint(amax) >> 23) & 0xFF) - 126;   // amax < 2^e
      k = min(max(15 - e, -100), 100);
    }
    const float up = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
    st.qshift = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        if constexpr (C::INT4) {
          // ks = 2c + u: values b + 2u + {0,1,2,3} sit in raw[.][2c] (u = 0: 0..3 of b)
          // and raw[.][2c + 1] (4..7 of b); pair (2u, 2u + 4) and (2u + 1, 2u + 5)
          const uint2 lo4 = raw[nt][ks & ~1], hi4 = raw[nt][ks | 1];
          const uint32_t e = (ks & 1) ? lo4.y : lo4.x;   // values b+2u, b+2u+1
          const uint32_t f = (ks & 1) ? hi4.y : hi4.x;   // values b+2u+4, b+2u+5
          const uint32_t f0 = pack_f16(bf16_lo(e) * up, bf16_lo(f) * up);
          const uint32_t f1 = pack_f16(bf16_hi(e) * up, bf16_hi(f) * up);
          if constexpr (C::QSMEM) {   // k-steps 2j and 2j + 1 share one 16-byte entry
            uint4 &q4 = qfs[(nt * (C::KS / 2) + (ks >> 1)) * 32 + lane];
            if (ks & 1) {
              q4.z = f0;
              q4.w = f1;
            } else {
              q4.x = f0;
              q4.y = f1;
            }
          } else {
            st.qf[nt][ks][0] = f0;
            st.qf[nt][ks][1] = f1;
          }
        } else {
          const uint2 v = raw[nt][ks];
          const uint32_t f0 = pack_f16(bf16_lo(v.x) * up, bf16_hi(v.x) * up);
          const uint32_t f1 = pack_f16(bf16_lo(v.y) * up, bf16_hi(v.y) * up);
          if constexpr (C::QSMEM) {   // k-steps 2j and 2j + 1 share one 16-byte entry
            uint4 &q4 = qfs[(nt * (C::KS / 2) + (ks >> 1)) * 32 + lane];
            if (ks & 1) {
              q4.z = f0;
              q4.w = f1;
            } else {
              q4.x = f0;
              q4.y = f1;
            }
          } else {
            st.qf[nt][ks][0] = f0;
            st.qf[nt][ks][1] = f1;
          }
        }
      }
  }
}

// The 16-token tiles a sequence of L cached tokens is attended over: with a window
// ("KV Cache Engineering for LLM Serving", section 3) only positions
// [max(0, L - window), L) count, so whole tiles before that are skipped and the
// first kept tile may start part-way.
struct SeqTiles {
  int first;       // absolute index of the first tile
  int count;       // tiles attended
  int last_valid;  // valid tokens in the last tile (1..16)
  int first_skip;  // tokens before the window in the first tile (0..15)
};

__device__ __forceinline__ SeqTiles seq_tiles(int L, int window, int cascade_tiles = 0) {
  int start = (window > 0 && L > window) ? L - window : 0;
  // tiles of a shared prefix that the cascade kernel attends over are skipped here
  start = max(start, min(cascade_tiles * kTile, L));
  const int end_tiles = (L + kTile - 1) / kTile;
  SeqTiles t;
  t.first = start / kTile;
  t.count = end_tiles - t.first;
  t.last_valid = L - (end_tiles - 1) * kTile;
  t.first_skip = start - t.first * kTile;
  return t;
}

constexpr int kLoShift = 16;   // unit info bits 16..19: first valid token of the tile
constexpr int kKvhShift = 20;  // unit info bits 20..30: the unit's KV head (of the unit view)
constexpr int kKvhMask = 0x7FF;

// A head's reference maximum (log2 domain) moves only when a score exceeds it by more
// than this, so every p stays <= 2^8.
constexpr float kMaxSlack = 8.f;
// Quantised caches: largest restored |V| of a tile (V scale x largest code) for which P
// enters the PV product as one f16 term; the term's rounding then adds at most
// 2^-12 * 16 < 4e-3 to an output, a fifth of the quantised tolerance 2e-2.
constexpr float kOneTermV = 16.f;

// Tiles attended per (sequence, KV head): the window's tiles, the chosen pages, or
// the tiles after a cascaded shared prefix.
__device__ __forceinline__ int pair_tile_count(int L, int window, int topk,
                                               int cascade_tiles = 0) {
  if (topk > 0) return min(topk, (L + kTile - 1) / kTile);
  return seq_tiles(L, window, cascade_tiles).count;
}

// One 16-token tile: scores, online-softmax update, P V accumulation.
// sscale[nt]: factor from raw mma scores to log2-domain scores; vs[nt]: V scale of a
// quantised tile; vzero[h]: the tile's V scale of the unit's KV head h is zero, so
// its V rows count as zeros.  The accumulator stays in units of the piece's first
// nonzero V scale: a tile with another scale enters through P scaled by the ratio.
template <class C, bool LO>
__device__ __forceinline__ void process_tile(State<C> &st, const uint4 *qfs, uint32_t ktile,
                                             uint32_t vtile, int lo, int nvalid,
                                             const float (&sscale)[C::NT],
                                             const float (&vs)[C::NT],
                                             const bool (&vzero)[C::HEADS], int lane) {
  // tokens lo <= t < nvalid of the tile are attended
  const int r = lane >> 2, qd = lane & 3;
  float s[C::NT][4];
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;

  // ---- S^T = K Q^T
  if constexpr (!C::QUANT) {
    const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const int c = ((ks & 3) << 1) + (lane >> 4);
      uint32_t a[4];
      ldsm_x4(a, ktile + (ks >> 2) * (kTile * 128) + row * 128 + ((c ^ (row & 7)) << 4));
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) mma_bf16(s[nt], a, st.qf[nt][ks][0], st.qf[nt][ks][1]);
    }
  } else if constexpr (C::INT4) {
    // 64-byte head rows: lane (r, q) receives nibbles b..b+7 (b = 32c + 8q) of row r;
    // int4_pair_f16 yields the pairs (b+i, b+i+4) that load_q mirrors.  One head: a
    // 64-byte-swizzled box; paired heads: head h is chunks 4h..4h+3 of a 128-byte-
    // swizzled row and feeds n-tile h only.
    const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int h = 0; h < C::HEADS; ++h)
#pragma unroll
      for (int cc = 0; cc < C::D / 64; ++cc) {
        const int c = 2 * cc + (lane >> 4);
        uint32_t R[4];
        if constexpr (C::PAIRED)
          ldsm_x4(R, ktile + row * 128 + (((4 * h + c) ^ (row & 7)) << 4));
        else
          ldsm_x4(R, ktile + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // chunk 2cc + half: R[2 half] rows r, R[2 half + 1] rows r + 8
          uint4 q4 = make_uint4(0u, 0u, 0u, 0u);
          if constexpr (C::QSMEM) q4 = qfs[(h * (C::KS / 2) + 2 * cc + half) * 32 + lane];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t a[4] = {int4_pair_f16(R[2 * half], 2 * u),
                                   int4_pair_f16(R[2 * half + 1], 2 * u),
                                   int4_pair_f16(R[2 * half], 2 * u + 1),
                                   int4_pair_f16(R[2 * half + 1], 2 * u + 1)};
            const int ks = (2 * cc + half) * 2 + u;
            if constexpr (C::QSMEM) {
              mma_f16(s[h], a, u ? q4.z : q4.x, u ? q4.w : q4.y);
            } else if constexpr (C::PAIRED) {
              mma_f16(s[h], a, st.qf[h][ks][0], st.qf[h][ks][1]);
            } else {
#pragma unroll
              for (int nt = 0; nt < C::NT; ++nt)
                mma_f16(s[nt], a, st.qf[nt][ks][0], st.qf[nt][ks][1]);
            }
          }
        }
      }
  } else {
    // ldmatrix on byte pairs: lane (r, q) receives codes 4q..4q+3 of a 16-code chunk;
    // the mma's k order is permuted accordingly (load_q applies the same order to q).
    // Paired heads: head h is box h of the tile and feeds n-tile h only.
    const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
    for (int h = 0; h < C::HEADS; ++h)
#pragma unroll
      for (int kk = 0; kk < C::D / 32; ++kk) {
        const int c = 2 * kk + (lane >> 4);
        uint32_t R[4];
        ldsm_x4(R, ktile + h * (kTile * 128) + row * 128 + ((c ^ (row & 7)) << 4));
        const uint32_t a0[4] = {e4m3x2_to_f16x2(R[0]), e4m3x2_to_f16x2(R[1]),
                                e4m3x2_hi_to_f16x2(R[0]), e4m3x2_hi_to_f16x2(R[1])};
        const uint32_t a1[4] = {e4m3x2_to_f16x2(R[2]), e4m3x2_to_f16x2(R[3]),
                                e4m3x2_hi_to_f16x2(R[2]), e4m3x2_hi_to_f16x2(R[3])};
        if constexpr (C::PAIRED) {
          const uint4 q4 = qfs[(h * (C::KS / 2) + kk) * 32 + lane];
          mma_f16(s[h], a0, q4.x, q4.y);
          mma_f16(s[h], a1, q4.z, q4.w);
        } else {
#pragma unroll
          for (int nt = 0; nt < C::NT; ++nt) {
            mma_f16(s[nt], a0, st.qf[nt][2 * kk][0], st.qf[nt][2 * kk][1]);
            mma_f16(s[nt], a1, st.qf[nt][2 * kk + 1][0], st.qf[nt][2 * kk + 1][1]);
          }
        }
      }
  }

  // ---- V scale of a quantised tile relative to the accumulator's unit (warp-uniform).
  // The piece starts with vinv = 0, so its first nonzero scale takes the rare branch
  // that (re)expresses the accumulator in the tile's own scale.
  float rat[C::NT];
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt) {
    rat[nt] = 1.f;
    if constexpr (C::QUANT) {
      rat[nt] = vs[nt] * st.vinv[nt];
      if (!vzero[C::PAIRED ? nt : 0] && !(rat[nt] <= kRatMax && rat[nt] >= kRatMin)) {
        const float f = st.vref[nt] / vs[nt];
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
          for (int i = 0; i < 4; ++i) st.acc[nt][dt][i] *= f;
        st.vref[nt] = vs[nt];
        st.vinv[nt] = 1.f / vs[nt];
        rat[nt] = 1.f;
      }
    }
  }

  // ---- online softmax (log2 domain); element i: token r + 8*(i>>1), head 2q + (i&1).
  // Each head's reference maximum st.m moves only when a score exceeds it by more than
  // kMaxSlack, so p <= 2^kMaxSlack; the result is the same (o and l share the
  // reference).  A tile that moves no reference needs no reduction across lanes and
  // no rescaling of the accumulator: one compare per score and a warp vote.
  const bool ragged = nvalid < kTile || lo > 0;   // warp-uniform
  float x[C::NT][4];
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) x[nt][i] = s[nt][i] * sscale[nt];
  if (ragged) {
    const bool in0 = r >= lo && r < nvalid, in1 = r + 8 >= lo && r + 8 < nvalid;
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (!((i >> 1) ? in1 : in0)) x[nt][i] = -INFINITY;
  }
  bool over = false;
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) over |= x[nt][i] > st.m[nt][i & 1] + kMaxSlack;
  if (__any_sync(0xffffffffu, over)) {
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      float alpha[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float mx = fmaxf(x[nt][j], x[nt][j + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(st.m[nt][j], mx);
        alpha[j] = ex2(st.m[nt][j] - mnew);
        st.l[nt][j] *= alpha[j];
        st.m[nt][j] = mnew;
      }
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
        for (int i = 0; i < 4; ++i) st.acc[nt][dt][i] *= alpha[i & 1];
    }
  }
  float p[C::NT][4];
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      p[nt][j] = ex2(x[nt][j] - st.m[nt][j]);
      p[nt][j + 2] = ex2(x[nt][j + 2] - st.m[nt][j]);
      st.l[nt][j] += p[nt][j] + p[nt][j + 2];
    }

  // ---- P^T fragments, transposed in registers.  bf16 caches split p into two bf16
  // terms, hi + lo (16 significant bits).  Quantised caches feed p times the tile's
  // V-scale ratio as one f16 term (relative rounding <= 2^-12).  With LO (tiles whose
  // restored V values exceed kOneTermV, chosen by the caller) the f16 remainder follows
  // as a second term, 22 significant bits in all: its fragments are parked in the tile's
  // K area (free once S is computed) and the same PV code runs a second time with them,
  // so this rare instantiation needs no more registers than the common one.
  uint32_t bh[C::NT][2], bl[C::NT][2];
  if constexpr (C::QUANT && LO) __syncwarp();   // every lane is done reading the K tile
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if constexpr (!C::QUANT) {
        const float p0 = p[nt][2 * h], p1 = p[nt][2 * h + 1];
        const uint32_t hi = pack_bf16(p0, p1);
        bh[nt][h] = movmatrix_trans(hi);
        bl[nt][h] = movmatrix_trans(pack_bf16(p0 - bf16_lo(hi), p1 - bf16_hi(hi)));
      } else {
        const float p0 = p[nt][2 * h] * rat[nt], p1 = p[nt][2 * h + 1] * rat[nt];
        const uint32_t hi = pack_f16(p0, p1);
        bh[nt][h] = movmatrix_trans(hi);
        if constexpr (LO) {
          const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
          sts_u32(ktile + ((nt * 2 + h) * 32 + lane) * 4,
                  movmatrix_trans(pack_f16(p0 - hf.x, p1 - hf.y)));
        }
      }
    }
  // the second pass of a quantised LO tile: the parked remainders become the P fragments
  auto take_lo = [&]() {
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) bh[nt][h] = lds_u32(ktile + ((nt * 2 + h) * 32 + lane) * 4);
  };

  // ---- O^T += V^T P^T.  A masked token has p = 0 exactly, but stale bf16 or E4M3 rows
  // may hold non-finite values (0 * NaN = NaN), so for those caches the V rows of a
  // ragged tile (and of a tile whose V scale is zero) are zeroed in registers under
  // one warp-uniform branch; full tiles skip it.  Every 4-bit code converts to a finite
  // value and a zero V scale already makes P zero (rat = 0), so 4-bit tiles need no
  // mask.
  if constexpr (!C::QUANT) {
    auto pv = [&](auto masked) {
      constexpr bool MASK = decltype(masked)::value;
      uint32_t m01 = 0xFFFFFFFFu, m23 = 0xFFFFFFFFu;
      if constexpr (MASK) {
        auto in = [&](int t) { return t >= lo && t < nvalid; };
        m01 = (in(2 * qd) ? 0x0000FFFFu : 0u) | (in(2 * qd + 1) ? 0xFFFF0000u : 0u);
        m23 = (in(2 * qd + 8) ? 0x0000FFFFu : 0u) | (in(2 * qd + 9) ? 0xFFFF0000u : 0u);
      }
      const int t = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt) {
        const int c = ((dt & 3) << 1) + ((lane >> 3) & 1);
        uint32_t a[4];
        ldsm_x4_trans(a, vtile + (dt >> 2) * (kTile * 128) + t * 128 + ((c ^ (t & 7)) << 4));
        if constexpr (MASK) {
          a[0] &= m01;
          a[1] &= m01;
          a[2] &= m23;
          a[3] &= m23;
        }
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          mma_bf16(st.acc[nt][dt], a, bh[nt][0], bh[nt][1]);
          mma_bf16(st.acc[nt][dt], a, bl[nt][0], bl[nt][1]);
        }
      }
    };
    if (ragged) pv(std::true_type{}); else pv(std::false_type{});
  } else if constexpr (C::INT4) {
    // ldmatrix.trans on the byte-pair view gives lane (r, q) the nibbles d = 32c + 4r
    // .. +3 of tokens 2q (low half) and 2q + 1 (high half): int4_pair_f16(., i) is
    // V^T row d = 32c + 4r + i over tokens (2q, 2q + 1).  Paired heads as for K.
    const int t = (lane & 7) + (((lane >> 3) & 1) << 3);
    auto pv = [&]() {
#pragma unroll
      for (int h = 0; h < C::HEADS; ++h) {
#pragma unroll
        for (int cc = 0; cc < C::D / 64; ++cc) {
          const int c = 2 * cc + (lane >> 4);
          uint32_t R[4];
          if constexpr (C::PAIRED)
            ldsm_x4_trans(R, vtile + t * 128 + (((4 * h + c) ^ (t & 7)) << 4));
          else
            ldsm_x4_trans(R, vtile + t * 64 + ((c ^ ((t >> 1) & 3)) << 4));
#pragma unroll
          for (int half = 0; half < 2; ++half)    // chunk 2cc + half
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {      // rows 4r + 2mt + {0, 1}
              const uint32_t a[4] = {int4_pair_f16(R[2 * half], 2 * mt),
                                     int4_pair_f16(R[2 * half], 2 * mt + 1),
                                     int4_pair_f16(R[2 * half + 1], 2 * mt),
                                     int4_pair_f16(R[2 * half + 1], 2 * mt + 1)};
              const int dt = (2 * cc + half) * 2 + mt;
              if constexpr (C::PAIRED) {
                mma_f16(st.acc[h][dt], a, bh[h][0], bh[h][1]);
              } else {
#pragma unroll
                for (int nt = 0; nt < C::NT; ++nt) mma_f16(st.acc[nt][dt], a, bh[nt][0], bh[nt][1]);
              }
            }
        }
      }
    };
    pv();
    if constexpr (LO) {
      take_lo();
      pv();
    }
  } else {
    // ldmatrix.trans on byte pairs gives lane (r, q): bytes (t=2q: d=2r, 2r+1) and
    // (t=2q+1: d=2r, 2r+1); regrouping by d yields V^T rows d = 2r (even) and 2r+1
    // (odd) -- the tile's 16 output rows in the order (2r, 2r+1).
    // Paired heads: head h is box h of the tile and feeds n-tile h only.
    auto pv = [&](auto masked) {
      constexpr bool MASK = decltype(masked)::value;
      uint32_t m01[C::HEADS], m23[C::HEADS];
#pragma unroll
      for (int h = 0; h < C::HEADS; ++h) {
        m01[h] = m23[h] = 0xFFFFFFFFu;
        if constexpr (MASK) {
          if (vzero[h]) {
            m01[h] = m23[h] = 0u;
          } else {
            auto in = [&](int t) { return t >= lo && t < nvalid; };
            m01[h] = (in(2 * qd) ? 0x0000FFFFu : 0u) | (in(2 * qd + 1) ? 0xFFFF0000u : 0u);
            m23[h] = (in(2 * qd + 8) ? 0x0000FFFFu : 0u) | (in(2 * qd + 9) ? 0xFFFF0000u : 0u);
          }
        }
      }
      const int t = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int h = 0; h < C::HEADS; ++h)
#pragma unroll
        for (int cc = 0; cc < C::D / 32; ++cc) {
          const int c = 2 * cc + (lane >> 4);
          uint32_t R[4];
          ldsm_x4_trans(R, vtile + h * (kTile * 128) + t * 128 + ((c ^ (t & 7)) << 4));
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // one permute per register: (t0 d0, t0 d1, t1 d0, t1 d1) -> (t0 d0, t1 d0,
            // t0 d1, t1 d1); its low half is row 2r, its high half row 2r + 1
            const uint32_t lo8 = __byte_perm(R[2 * hh], 0, 0x3120);
            const uint32_t hi8 = __byte_perm(R[2 * hh + 1], 0, 0x3120);
            uint32_t a[4] = {e4m3x2_to_f16x2(lo8), e4m3x2_hi_to_f16x2(lo8),
                             e4m3x2_to_f16x2(hi8), e4m3x2_hi_to_f16x2(hi8)};
            if constexpr (MASK) {
              a[0] &= m01[h];
              a[1] &= m01[h];
              a[2] &= m23[h];
              a[3] &= m23[h];
            }
            if constexpr (C::PAIRED) {
              mma_f16(st.acc[h][2 * cc + hh], a, bh[h][0], bh[h][1]);
            } else {
#pragma unroll
              for (int nt = 0; nt < C::NT; ++nt)
                mma_f16(st.acc[nt][2 * cc + hh], a, bh[nt][0], bh[nt][1]);
            }
          }
        }
    };
    bool zmask = false;
#pragma unroll
    for (int h = 0; h < C::HEADS; ++h) zmask |= vzero[h];
    if (ragged || zmask) pv(std::true_type{}); else pv(std::false_type{});
    if constexpr (LO) {
      take_lo();
      if (ragged || zmask) pv(std::true_type{}); else pv(std::false_type{});
    }
  }
}

// Sum l over the 8 lanes that share a head pair; returns the per-head total.
template <class C>
__device__ __forceinline__ void reduce_l(const State<C> &st, float (&ltot)[C::NT][2]) {
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = st.l[nt][j];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      ltot[nt][j] = v;
    }
}

// Write o = acc / l (normalised) for heads g < G to dst[g * hstride + d]; and, if
// requested, lse to lse_dst[g * lstride].
template <class C>
__device__ __forceinline__ void write_normalised(const State<C> &st, float *dst, float *lse_dst,
                                                 int G, int lane, size_t hstride = C::D,
                                                 size_t lstride = 1) {
  float ltot[C::NT][2];
  reduce_l<C>(st, ltot);
  const int qd = lane & 3;
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int g = nt * 8 + 2 * qd + j;
      if (g >= G) continue;
      const float f = (C::QUANT ? st.vref[nt] : 1.f) / ltot[nt][j];
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt) {
        dst[g * hstride + acc_d<C>(dt, j, lane)] = st.acc[nt][dt][j] * f;
        dst[g * hstride + acc_d<C>(dt, j + 2, lane)] = st.acc[nt][dt][j + 2] * f;
      }
      if (lse_dst && (lane >> 2) == 0)
        lse_dst[g * lstride] = (st.m[nt][j] + __log2f(ltot[nt][j])) * kLn2;
    }
}

// The cascade partials of sequence b, KV head kvh: lse [pieces][G] and o
// [pieces][G][D] in the cascade workspace at `cws` (0: none).  Returns the pieces.
__device__ __forceinline__ int cascade_partials(uint64_t cws, int B, int Hq, int Hkv, int G,
                                                int D, int b, int kvh, const float *&clse,
                                                const float *&co) {
  if (!cws) return 0;
  const CascadeLayout cl = cascade_layout(B, Hq, D);
  const uint8_t *cw = reinterpret_cast<const uint8_t *>(cws);
  const int m = reinterpret_cast<const int32_t *>(cw + cl.member)[b];
  if (m < 0) return 0;
  const size_t c0 = (static_cast<size_t>(m) * Hkv + kvh) * kCascadePieces * G;
  clse = reinterpret_cast<const float *>(cw + cl.lse) + c0;
  co = reinterpret_cast<const float *>(cw + cl.o) + c0 * D;
  return reinterpret_cast<const int32_t *>(cw + cl.pieces)[b];
}

// ----------------------------------------------------------------------------
// unit sources: which tiles a warp processes, in order
// ----------------------------------------------------------------------------

// Tiles w, w + NW, ... of one (b, kvh) pair's attended tiles, read straight from
// the block table.
// The copy record of one tile, built lane-parallel when a source loads 32 tiles:
// (row of the tile's first token in the pools' 2-D view, unit, scale index
// phys * Hkv + kvh of the unit view or -1 for a bad block, info bits).  A bad block
// reads the rows past the pool, which the copy fills with zeros.
__device__ __forceinline__ int4 tile_record(int phys, int tile, int unit, int kvh, int hkv,
                                            int bs, int nblocks, int info) {
  if (phys == kInvalidPhys) return make_int4(nblocks * bs, unit, -1, info);
  // block_size is 16 or 32: the tile's first row in its block is a mask away
  return make_int4(phys * bs + ((tile * kTile) & (bs - 1)), unit, phys * hkv + kvh, info);
}

struct PairSource {
  const int32_t *row;
  const int32_t *sel;   // this pair's chosen pages, or null
  int32_t *err;
  int pair, kvh, hkv, w, nw, bs, nblocks;
  SeqTiles geo;         // with a selection: count = pages chosen, first = 0
  int npages;           // 16-token pages of the sequence
  int shared_len;       // L2 hint: leading tokens in shared blocks, or -1 (no hint)
  int base;
  int4 cur, nxt;

  __device__ __forceinline__ int count() const {
    return geo.count > w ? (geo.count - w + nw - 1) / nw : 0;
  }
  __device__ __forceinline__ int4 load(int i) const {
    const int j = w + i * nw;
    if (j >= geo.count) return make_int4(0, 0, -1, 0);   // never issued
    int tile = geo.first + j, last_tile = geo.first + geo.count - 1;
    if (sel) {
      tile = __ldg(sel + j);
      last_tile = npages - 1;
    }
    const bool bad_page = sel && (tile < 0 || tile >= npages);
    if (bad_page) {
      set_err(err, PA_DEVERR_BLOCK_ID);
      tile = 0;
    }
    int phys = bad_page ? kInvalidPhys : __ldg(row + (tile * kTile) / bs);
    if (phys < 0 || phys >= nblocks) {
      set_err(err, PA_DEVERR_BLOCK_ID);
      phys = kInvalidPhys;
    }
    int info = (tile == last_tile) ? geo.last_valid : kTile;
    if (j == 0) info |= kFirstOfPair | (sel ? 0 : geo.first_skip << kLoShift);
    if (j == geo.count - 1) info |= kLastOfPair;
    if (i == 0) info |= kPieceStart;
    if (j + nw >= geo.count) info |= kPieceEnd;
    if (shared_len >= 0) info |= ((tile + 1) * kTile <= shared_len) ? kHintShared : kHintPrivate;
    return tile_record(phys, tile, pair, kvh, hkv, bs, nblocks, info | (kvh << kKvhShift));
  }
  __device__ __forceinline__ void init(int lane) {
    base = 0;
    cur = load(lane);
    nxt = load(32 + lane);
  }
  __device__ __forceinline__ int4 get(int i, int lane) {
    while (i >= base + 32) {
      cur = nxt;
      base += 32;
      nxt = load(base + 32 + lane);
    }
    return shfl_int4(cur, i - base);
  }
};

// A contiguous segment [begin, end) of the tile stream: position f belongs to the
// sequence b with prefix[b] <= f < prefix[b + 1] (binary search in shared memory),
// then to KV head (f - prefix[b]) / count(b) and attended tile (f - prefix[b]) % count(b).
struct SegmentSource {
  const int32_t *prefix;     // shared: [B + 1]
  const int32_t *seq_lens;
  const int32_t *block_tables;
  const int32_t *shared_prefix_lens;   // may be null
  const int32_t *sel;                  // [B, Hkv, topk] chosen pages, or null
  const int32_t *casc_tiles;           // [B] cascaded shared tiles, or null
  int32_t *err;
  int B, Hkv, bs, nblocks, max_blocks, window, topk;
  int begin, end;
  int base;
  int4 cur, nxt;

  __device__ __forceinline__ int count() const { return end - begin; }
  __device__ __forceinline__ int4 load(int i) const {
    const int f = begin + i;
    if (f >= end) return make_int4(0, 0, -1, 0);   // never issued
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= f) lo = mid; else hi = mid - 1;
    }
    const int b = lo, start = prefix[b];
    const int nt = (prefix[b + 1] - start) / Hkv;
    const int r = f - start;
    const int kvh = r / nt, j = r - kvh * nt;
    const int L = min(max(__ldg(seq_lens + b), 0), max_blocks * bs);
    const int ct = casc_tiles ? casc_tiles[b] : 0;
    const SeqTiles geo = seq_tiles(L, window, ct);
    int tile = geo.first + j, last_tile = geo.first + geo.count - 1;
    bool bad_page = false;
    if (sel) {
      const int npages = (L + kTile - 1) / kTile;
      tile = __ldg(sel + (static_cast<size_t>(b) * Hkv + kvh) * topk + j);
      last_tile = npages - 1;
      bad_page = tile < 0 || tile >= npages;
      if (bad_page) {
        set_err(err, PA_DEVERR_BLOCK_ID);
        tile = 0;
      }
    }
    int phys = bad_page ? kInvalidPhys
                        : __ldg(block_tables + static_cast<size_t>(b) * max_blocks + (tile * kTile) / bs);
    if (phys < 0 || phys >= nblocks) {
      set_err(err, PA_DEVERR_BLOCK_ID);
      phys = kInvalidPhys;
    }
    int info = (tile == last_tile) ? geo.last_valid : kTile;
    if (j == 0) info |= kFirstOfPair | kPieceStart | (sel ? 0 : geo.first_skip << kLoShift);
    if (j == nt - 1) info |= kLastOfPair | kPieceEnd;
    if (i == 0) info |= kPieceStart;
    if (f == end - 1) info |= kPieceEnd;
    if (shared_prefix_lens)
      info |= ((tile + 1) * kTile <= __ldg(shared_prefix_lens + b)) ? kHintShared : kHintPrivate;
    if (ct > 0) info |= kCascade;
    return tile_record(phys, tile, b * Hkv + kvh, kvh, Hkv, bs, nblocks,
                       info | (kvh << kKvhShift));
  }
  __device__ __forceinline__ void init(int lane) {
    base = 0;
    cur = load(lane);
    nxt = load(32 + lane);
  }
  __device__ __forceinline__ int4 get(int i, int lane) {
    while (i >= base + 32) {
      cur = nxt;
      base += 32;
      nxt = load(base + 32 + lane);
    }
    return shfl_int4(cur, i - base);
  }
};

// ----------------------------------------------------------------------------
// the per-warp pipeline
// ----------------------------------------------------------------------------

struct WarpSmem {
  uint8_t *stage;     // STAGES * STAGE_BYTES, 1024-aligned
  uint64_t *bar;      // STAGES mbarriers
  int4 *meta;         // STAGES * 2 int4: unit, then the unit's k scales and v scales
  uint4 *qf;          // Q^T fragments when they live in shared memory, else null
};

template <class C>
__device__ __forceinline__ void issue(const WarpSmem &ws, int s, int4 u, const Params &p,
                                      const CUtensorMap *tmK, const CUtensorMap *tmV, int lane) {
  if (lane != 0) return;
  uint8_t *stage = ws.stage + s * C::STAGE_BYTES;
  const uint32_t bar = smem_u32(&ws.bar[s]);
  const int y = u.x, sidx = u.z;
  const int kvh = (u.w >> kKvhShift) & kKvhMask;
  ws.meta[2 * s] = u;
  if constexpr (C::QUANT) {
    // the k scales of the unit's KV heads (kvh, or 2 kvh and 2 kvh + 1), then their
    // v scales
    float *sc = reinterpret_cast<float *>(&ws.meta[2 * s + 1]);
    if (sidx >= 0) {
      const size_t i = static_cast<size_t>(sidx) * C::HEADS;
      if constexpr (C::PAIRED) {
        cp_async_8(smem_u32(sc), p.k_scale + i);
        cp_async_8(smem_u32(sc + 2), p.v_scale + i);
      } else {
        cp_async_4(smem_u32(sc), p.k_scale + i);
        cp_async_4(smem_u32(sc + 2), p.v_scale + i);
      }
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) sc[h] = 0.f;
    }
    cp_async_arrive(bar);
  }
  const bool with_q = !C::QSMEM && (u.w & kPieceStart) != 0;
  const uint32_t bytes = 2 * C::KV_BYTES + (with_q ? p.G * C::D * 2 : 0);
  const uint32_t dst = smem_u32(stage);
  fence_proxy_async();
  mbar_arrive_expect_tx(bar, bytes);
  // the row of KV head kvh starts at element kvh * (ROW / element bytes)
  const int x0 = kvh * C::BOXES * C::BOX_X;
  if (u.w & (kHintShared | kHintPrivate)) {
    const uint64_t pol = (u.w & kHintShared) ? l2_policy_evict_last() : l2_policy_evict_first();
#pragma unroll
    for (int h = 0; h < C::BOXES; ++h) {
      const int x = x0 + h * C::BOX_X;
      tma_load_2d_hint(dst + h * (kTile * C::BOX_BYTES), tmK, x, y, bar, pol);
      tma_load_2d_hint(dst + C::KV_BYTES + h * (kTile * C::BOX_BYTES), tmV, x, y, bar, pol);
    }
  } else {
#pragma unroll
    for (int h = 0; h < C::BOXES; ++h) {
      const int x = x0 + h * C::BOX_X;
      tma_load_2d(dst + h * (kTile * C::BOX_BYTES), tmK, x, y, bar);
      tma_load_2d(dst + C::KV_BYTES + h * (kTile * C::BOX_BYTES), tmV, x, y, bar);
    }
  }
  if (with_q) {                                  // a piece starts: the group's query rows
    const int b = u.y / p.Hkv;
    bulk_load(dst + 2 * C::KV_BYTES, p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.G) * C::D,
              p.G * C::D * 2, bar);
  }
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Runs all units of `src` (already init()ed) through the warp's ring.
// on_piece_end(u, piece_has_pair_start, st) is called after the last tile of every
// piece.  Returns false after a wait timeout.
template <class C, class Src, class OnEnd>
__device__ __forceinline__ bool run_warp(Src &src, const WarpSmem &ws, State<C> &st,
                                         const Params &p, const CUtensorMap *tmK,
                                         const CUtensorMap *tmV, OnEnd &&on_piece_end,
                                         int lane) {
  const int n = src.count();
#pragma unroll
  for (int s = 0; s < C::STAGES; ++s)
    if (s < n) issue<C>(ws, s, src.get(s, lane), p, tmK, tmV, lane);
  bool piece_first = false;
  for (int i = 0; i < n; ++i) {
    const int s = i % C::STAGES;
    const uint32_t bar = smem_u32(&ws.bar[s]);
    if (!warp_wait(bar, (i / C::STAGES) & 1)) {
      set_err(lane == 0 ? p.err : nullptr, PA_DEVERR_TIMEOUT);
      for (int j = i; j < n && j < i + C::STAGES; ++j)
        mbar_wait(smem_u32(&ws.bar[j % C::STAGES]), (j / C::STAGES) & 1);
      return false;
    }
    const int4 u = ws.meta[2 * s];
    uint8_t *stage = ws.stage + s * C::STAGE_BYTES;
    const uint32_t ktile = smem_u32(stage);
    float sscale[C::NT], vs[C::NT];
    bool vzero[C::HEADS];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      sscale[nt] = p.sl2;
      vs[nt] = 1.f;
    }
#pragma unroll
    for (int h = 0; h < C::HEADS; ++h) vzero[h] = false;
    if (u.w & kPieceStart) {
      st.reset();
      if constexpr (C::QSMEM) {   // the group's query rows, straight from global memory
        const int b = u.y / p.Hkv, kvh = (u.w >> kKvhShift) & kKvhMask;
        load_q<C>(st, 0u, p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.G) * C::D, ws.qf,
                  p.G, lane);
      } else {
        load_q<C>(st, ktile + 2 * C::KV_BYTES,
                  reinterpret_cast<const uint16_t *>(stage + 2 * C::KV_BYTES), nullptr, p.G,
                  lane);
      }
      piece_first = (u.w & kFirstOfPair) != 0;
    }
    if constexpr (C::QUANT) {
      // n-tile nt reads KV head nt of the unit (paired) or the unit's one head; a zero
      // V scale zeroes the tile's V rows
      const float4 sc = *reinterpret_cast<const float4 *>(&ws.meta[2 * s + 1]);
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) {
        const int h = C::PAIRED ? nt : 0;
        const float ks = h ? sc.y : sc.x, v = h ? sc.w : sc.z;
        sscale[nt] = p.sl2 * ks * st.qshift;
        vzero[h] = !(v > 0.f);
        vs[nt] = v;
      }
    }
    // quantised tiles whose restored V values exceed kOneTermV take the two-term weights
    bool lo = false;
    if constexpr (C::QUANT) {
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) lo |= vs[nt] * (C::FP8 ? 448.f : 7.f) > kOneTermV;
    }
    if (lo)
      process_tile<C, true>(st, ws.qf, ktile, ktile + C::KV_BYTES, (u.w >> kLoShift) & 0xF,
                            u.w & 0xFF, sscale, vs, vzero, lane);
    else
      process_tile<C, false>(st, ws.qf, ktile, ktile + C::KV_BYTES, (u.w >> kLoShift) & 0xF,
                             u.w & 0xFF, sscale, vs, vzero, lane);
    if (u.w & kPieceEnd) on_piece_end(u, piece_first, st);
    __syncwarp();
    if (i + C::STAGES < n) issue<C>(ws, s, src.get(i + C::STAGES, lane), p, tmK, tmV, lane);
  }
  return true;
}

template <class C>
__device__ __forceinline__ WarpSmem setup_smem(uint8_t *raw, int warp, int G, int lane) {
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  WarpSmem ws;
  ws.stage = base + warp * C::STAGES * C::STAGE_BYTES;
  uint8_t *tail = base + C::WARPS * C::STAGES * C::STAGE_BYTES;
  ws.bar = reinterpret_cast<uint64_t *>(tail) + warp * C::STAGES;
  ws.meta = reinterpret_cast<int4 *>(tail + C::WARPS * C::STAGES * 8) + warp * C::STAGES * 2;
  ws.qf = nullptr;
  if constexpr (C::QSMEM)
    ws.qf = reinterpret_cast<uint4 *>(tail + C::WARPS * C::STAGES * (8 + C::META_BYTES) +
                                      warp * C::QF_BYTES);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) mbar_init(smem_u32(&ws.bar[s]), C::QUANT ? 2 : 1);
    fence_mbar_init();
  }
  // query rows G..8*NT-1 of every Q slot stay zero (the bulk copy writes G rows)
  if constexpr (!C::QSMEM) {
    const int pad = (8 * C::NT - G) * C::D * 2;
    for (int s = 0; s < C::STAGES; ++s) {
      uint8_t *qs = ws.stage + s * C::STAGE_BYTES + 2 * C::KV_BYTES + G * C::D * 2;
      for (int o = lane * 16; o < pad; o += 32 * 16)
        *reinterpret_cast<uint4 *>(qs + o) = make_uint4(0, 0, 0, 0);
    }
  }
  __syncwarp();
  return ws;
}

// First byte after the per-warp stages, barriers, metadata and Q^T fragment areas
// (16-byte aligned).
template <class C>
__device__ __forceinline__ uint8_t *split_tail(uint8_t *raw) {
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  return base + C::WARPS * (C::STAGES * (C::STAGE_BYTES + 8 + C::META_BYTES) + C::QF_BYTES);
}

// Dynamic shared memory of the split kernel: stages plus the length scan.
template <class C>
__host__ __device__ constexpr int split_smem(int B) {
  return C::SMEM + ((B + 1) * 4 + 15) / 16 * 16;
}

// ----------------------------------------------------------------------------
// pa_decode: one CTA per (sequence, KV head), or a cluster of CTAs per unit
// ----------------------------------------------------------------------------

// Thread-block clusters.  When a batch has few (sequence, KV head) units, pa_decode
// launches clusters of CTAs, one cluster per unit: the cluster's CTAs share the unit's
// tiles and CTA 0 merges their states through distributed shared memory.
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int cluster_ctas() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return static_cast<int>(r);
}
// Every thread of every CTA of the cluster arrives, then waits for all the others.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// The shared::cluster address of `addr` (this CTA's shared memory) in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// Arrive on an mbarrier in another CTA of the cluster, releasing this thread's prior
// writes (and those ordered before them by a CTA barrier) at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Bounded wait with acquire at cluster scope; false if the phase never completed.
template <uint32_t kSpins = kWaitSpins>
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kSpins; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Fewest tiles a warp takes when a cluster shares a unit: a unit of n tiles keeps
// ceil(n / (kClusterWarpTiles * WARPS)) of the cluster's CTAs (at least one, at most
// all); the others leave at once.
constexpr int kClusterWarpTiles = 16;
// Batches up to this many sequences are served longest first: up to kExactRankMaxB by an
// exact ranking (B^2 / threads key comparisons per CTA), above it by quarter-octave
// buckets of the tile count (linear in B; one byte per sequence in the stage area).
constexpr int kLongestFirstMaxB = 16384;
constexpr int kExactRankMaxB = 128;
constexpr int kRankBuckets = 256;
// Shared scratch of longest_first: bucket counts, the count above each bucket, the
// search's results and per-warp counts, then one bucket byte per sequence.
constexpr int kRankScratch = (2 * kRankBuckets + 8) * 4 + kLongestFirstMaxB;

// Small batches: unit slot c serves the sequence of rank c / Hkv when the sequences
// are ordered by attended tiles, most first (ties by index).  Each sequence gets one
// 32-bit key, tiles above its index (larger = earlier, all distinct), and its rank
// is the number of larger keys: every thread ranks two candidates in one pass over
// the keys, four at a time.  keys: shared scratch of 4 * (round4(B) + 1) bytes,
// 16-byte aligned, free again on return.
__device__ int longest_first_exact(const Params &p, int pair, uint32_t *keys) {
  static_assert(kExactRankMaxB <= 512, "keys hold the sequence index in 9 bits");
  const int cap = p.max_blocks * p.bs;
  const int nb4 = (p.B + 3) >> 2;
  for (int b = threadIdx.x; b < 4 * nb4; b += blockDim.x) {
    uint32_t key = 0u;   // padding: counted by no rank
    if (b < p.B) {
      const int c = pair_tile_count(min(max(__ldg(p.seq_lens + b), 0), cap), p.window, p.topk);
      key = (static_cast<uint32_t>(min(c, (1 << 23) - 1)) << 9) | static_cast<uint32_t>(511 - b);
    }
    keys[b] = key;
  }
  __syncthreads();
  const int want = pair / p.Hkv;
  int *chosen = reinterpret_cast<int *>(keys + 4 * nb4);
  const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
  for (int b0 = threadIdx.x; b0 < p.B; b0 += 2 * blockDim.x) {
    const int b1 = b0 + blockDim.x;
    const uint32_t c0 = keys[b0], c1 = b1 < p.B ? keys[b1] : 0xFFFFFFFFu;
    int r0 = 0, r1 = 0;
    for (int j = 0; j < nb4; ++j) {
      const uint4 k = k4[j];
      r0 += (k.x > c0) + (k.y > c0) + (k.z > c0) + (k.w > c0);
      r1 += (k.x > c1) + (k.y > c1) + (k.z > c1) + (k.w > c1);
    }
    // ranks are a permutation of 0..B-1: exactly one thread writes
    if (r0 == want) *chosen = b0;
    if (b1 < p.B && r1 == want) *chosen = b1;
  }
  __syncthreads();
  const int seq = *chosen;
  __syncthreads();   // every thread has read it before the stages are filled
  return seq * p.Hkv + (pair - want * p.Hkv);
}

// Unit slot c (a CTA, or a cluster) serves the sequence of rank c / Hkv when the
// sequences are ordered by their bucket of attended tiles, fullest first, then by index:
// the longest units start first and do not end the launch alone.  Buckets are quarter
// octaves (n tiles: 4 floor(log2 n) + the next two bits of n, plus one), so a wave of
// CTAs mixes lengths within about a fifth of each other: on batches of near-equal
// lengths an exact order makes whole waves start and finish in step, with the DRAM idle
// at each boundary.  A histogram of the buckets and a scan from the top give the bucket
// holding the rank; a scan over runs of consecutive sequences finds its member.  The
// cost is linear in B.  scratch: kRankScratch bytes of shared memory, 16-byte
// aligned, free again on return.
__device__ __forceinline__ int tile_bucket(int n) {
  if (n <= 0) return 0;
  const int e = 31 - __clz(n);                                 // n in [2^e, 2^(e+1))
  const int frac = e >= 2 ? (n >> (e - 2)) & 3 : (n << (2 - e)) & 3;
  return 4 * e + frac + 1;                                     // <= 4 * 30 + 3 + 1
}

__device__ int longest_first_bucketed(const Params &p, int pair, uint8_t *scratch) {
  constexpr int NB = kRankBuckets;
  static_assert(NB == 2 * 128, "two buckets per thread of a 128-thread CTA");
  int *hist = reinterpret_cast<int *>(scratch);
  int *above = hist + NB;                        // sequences in higher buckets
  int *sel = above + NB;                         // bucket, rank within it, the sequence
  int *wcnt = sel + 4;                           // per-warp counts
  uint8_t *bucket = reinterpret_cast<uint8_t *>(wcnt + 4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cap = p.max_blocks * p.bs;
  static_assert(4 * 30 + 3 + 1 < NB, "every tile count has a bucket");
  for (int k = tid; k < NB; k += blockDim.x) hist[k] = 0;
  __syncthreads();
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int c = pair_tile_count(min(max(__ldg(p.seq_lens + b), 0), cap), p.window, p.topk);
    const int k = tile_bucket(c);
    bucket[b] = static_cast<uint8_t>(k);
    atomicAdd(&hist[k], 1);
  }
  __syncthreads();
  // above[k] = sum of hist[k'] over k' > k: thread t holds buckets NB-1-2t and NB-2-2t
  {
    const int k0 = NB - 1 - 2 * tid, k1 = k0 - 1;
    const int v = hist[k0] + hist[k1];
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) wcnt[warp] = inc;
    __syncthreads();
    int ex = inc - v;
    for (int w = 0; w < warp; ++w) ex += wcnt[w];
    above[k0] = ex;
    above[k1] = ex + hist[k0];
  }
  __syncthreads();
  const int want = pair / p.Hkv;                 // < B: exactly one bucket holds it
  for (int k = tid; k < NB; k += blockDim.x)
    if (above[k] <= want && want < above[k] + hist[k]) {
      sel[0] = k;
      sel[1] = want - above[k];
    }
  __syncthreads();
  // the j-th member of bucket kb in index order: each thread counts the members in its
  // own run of consecutive sequences, a scan over the threads finds the run holding it
  {
    const int kb = sel[0], j = sel[1];
    const int per = (p.B + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
    const int lo = min(p.B, tid * per), hi = min(p.B, lo + per);
    int mine = 0;
    for (int b = lo; b < hi; ++b) mine += bucket[b] == kb;
    int inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) wcnt[warp] = inc;
    __syncthreads();
    int ex = inc - mine;
    for (int w = 0; w < warp; ++w) ex += wcnt[w];
    if (j >= ex && j < ex + mine) {
      int r = j - ex;
      for (int b = lo; b < hi; ++b)
        if (bucket[b] == kb && r-- == 0) {
          sel[2] = b;
          break;
        }
    }
    __syncthreads();
  }
  const int seq = sel[2];
  __syncthreads();   // every thread has read it before the stages are filled
  return seq * p.Hkv + (pair - want * p.Hkv);
}

__device__ __forceinline__ int longest_first(const Params &p, int pair, uint8_t *scratch) {
  return p.B <= kExactRankMaxB ? longest_first_exact(p, pair, reinterpret_cast<uint32_t *>(scratch))
                               : longest_first_bucketed(p, pair, scratch);
}

// CLUSTER: launched in clusters, one per unit (else one CTA per unit).
template <class C, bool CLUSTER>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS)
    decode_pair_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params p) {
  static_assert(kRankScratch <= C::WARPS * C::STAGES * C::STAGE_BYTES && C::THREADS == 128,
                "the ordering's scratch lives in the stage area");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int ncl = CLUSTER ? cluster_ctas() : 1, crank = CLUSTER ? cluster_rank() : 0;
  int pair = blockIdx.x / ncl;
  // a window or a Quest selection bounds every unit's tiles: near-uniform units gain
  // nothing from an order that costs more than the exact ranking of a small batch
  const bool bounded = p.window > 0 || p.topk > 0;
  if (p.B <= (bounded ? kExactRankMaxB : kLongestFirstMaxB))
    pair = longest_first(p, pair, base);
  const int b = pair / p.Hkv, kvh = pair - b * p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int L = p.seq_lens[b];
  const int cap = p.max_blocks * p.bs;
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0 && kvh == 0) set_err(p.err, PA_DEVERR_SEQ_LEN);
    L = min(max(L, 0), cap);
  }
  WarpSmem ws = setup_smem<C>(smem_raw, warp, p.G, lane);
  State<C> st;
  st.reset();
  PairSource src;
  src.row = p.block_tables + static_cast<size_t>(b) * p.max_blocks;
  src.err = p.err;
  src.pair = pair;
  src.kvh = kvh;
  src.hkv = p.Hkv;
  src.geo = seq_tiles(L, p.window);
  src.npages = (L + kTile - 1) / kTile;
  src.shared_len = p.shared_prefix_lens ? __ldg(p.shared_prefix_lens + b) : -1;
  src.sel = nullptr;
  if (p.sel) {
    src.sel = p.sel + static_cast<size_t>(pair) * p.topk;
    src.geo.first = 0;
    src.geo.count = pair_tile_count(L, 0, p.topk);
  }
  constexpr int GP = 8 * C::NT;
  float *sm_acc = reinterpret_cast<float *>(base);               // [WARPS][GP][D], stage area
  float *sm_m = reinterpret_cast<float *>(split_tail<C>(smem_raw));   // [WARPS][GP]
  float *sm_l = sm_m + C::WARPS * GP;                            // [WARPS][GP]
  float *cta_m = sm_l + C::WARPS * GP;                           // [GP] folded over warps
  float *cta_l = cta_m + GP;                                     // [GP]
  const uint32_t cl_bar = smem_u32(cta_l + GP);                  // cluster mbarrier
  // A cluster shares the unit's tiles among its first `active` CTAs; the others leave.
  int active = 1;
  if (ncl > 1) {
    const int per_cta = kClusterWarpTiles * C::WARPS;
    active = min(ncl, max(1, (src.geo.count + per_cta - 1) / per_cta));
    if (threadIdx.x == 0) {   // CTA 0 hears from the other active CTAs, each of them from CTA 0
      mbar_init(cl_bar, crank == 0 ? max(active - 1, 1) : 1);
      fence_mbar_init();
    }
    cluster_barrier();   // every CTA's cluster mbarrier is initialised
    if (crank >= active) return;
  }
  src.w = crank * C::WARPS + warp;
  src.nw = active * C::WARPS;
  src.bs = p.bs;
  src.nblocks = p.nblocks;
  src.init(lane);
  run_warp<C>(src, ws, st, p, &tmK, &tmV, [](int4, bool, State<C> &) {}, lane);

  // ---- merge the warps' states: warp w leaves m, l, acc (in absolute units)
  __syncthreads();
  {
    float ltot[C::NT][2];
    reduce_l<C>(st, ltot);
    const int qd = lane & 3;
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int g = nt * 8 + 2 * qd + j;
        if ((lane >> 2) == 0) {
          sm_m[warp * GP + g] = st.m[nt][j];
          sm_l[warp * GP + g] = ltot[nt][j];
        }
        const float f = C::QUANT ? st.vref[nt] : 1.f;
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) {
          sm_acc[(warp * GP + g) * C::D + acc_d<C>(dt, j, lane)] = st.acc[nt][dt][j] * f;
          sm_acc[(warp * GP + g) * C::D + acc_d<C>(dt, j + 2, lane)] = st.acc[nt][dt][j + 2] * f;
        }
      }
  }
  __syncthreads();
  float *out = p.out + (static_cast<size_t>(b) * p.Hq + kvh * p.G) * C::D;
  for (int e = threadIdx.x; e < p.G * C::D; e += C::THREADS) {
    const int g = e / C::D, d = e - g * C::D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::WARPS; ++w) M = fmaxf(M, sm_m[w * GP + g]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < C::WARPS; ++w) {
        const float mw = sm_m[w * GP + g];
        if (mw == -INFINITY) continue;
        const float f = ex2(mw - M);
        num += f * sm_acc[(w * GP + g) * C::D + d];
        den += f * sm_l[w * GP + g];
      }
    }
    if (ncl == 1) {
      out[e] = den > 0.f ? num / den : 0.f;
    } else {   // this CTA's state, relative to its own maximum M, for CTA 0 to merge
      sm_acc[g * C::D + d] = num;   // warp 0's entry (g, d): no other thread touches it
      if (d == 0) {
        cta_m[g] = M;
        cta_l[g] = den;
      }
    }
  }
  if (ncl == 1) return;

  // ---- cluster: CTA 0 merges the active CTAs' states through distributed shared memory
  __syncthreads();
  if (crank > 0) {
    if (threadIdx.x == 0) mbar_arrive_cluster(cluster_map(cl_bar, 0));
    // stay until CTA 0 has read this CTA's shared memory; this wait is bounded four times
    // longer than CTA 0's, so a CTA 0 that gave up (and reads nothing) is the only way
    // it runs out
    if (!mbar_wait_cluster<4 * kWaitSpins>(cl_bar, 0) && threadIdx.x == 0)
      set_err(p.err, PA_DEVERR_TIMEOUT);
    return;
  }
  // the other CTAs' states are complete once the phase completed for any thread
  const bool merged = __syncthreads_or(active <= 1 || mbar_wait_cluster(cl_bar, 0));
  if (!merged) {                     // no remote read: report, write zeros, release nobody
    if (threadIdx.x == 0) set_err(p.err, PA_DEVERR_TIMEOUT);
    for (int e = threadIdx.x; e < p.G * C::D; e += C::THREADS) out[e] = 0.f;
    return;
  }
  constexpr int kMaxCluster = 8;
  for (int e = threadIdx.x; e < p.G * C::D; e += C::THREADS) {
    const int g = e / C::D, d = e - g * C::D;
    const uint32_t am = smem_u32(&cta_m[g]), al = smem_u32(&cta_l[g]);
    const uint32_t aa = smem_u32(&sm_acc[g * C::D + d]);
    float mc[kMaxCluster];
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      mc[c] = c < active ? ld_cluster_f32(cluster_map(am, c)) : -INFINITY;
      M = fmaxf(M, mc[c]);
    }
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) {
        if (mc[c] == -INFINITY) continue;
        const float f = ex2(mc[c] - M);
        num += f * ld_cluster_f32(cluster_map(aa, c));
        den += f * ld_cluster_f32(cluster_map(al, c));
      }
    }
    out[e] = den > 0.f ? num / den : 0.f;
  }
  __syncthreads();   // every read of the other CTAs' shared memory is done: release them
  if (threadIdx.x > 0 && threadIdx.x < active) mbar_arrive_cluster(cluster_map(cl_bar, threadIdx.x));
}

// ----------------------------------------------------------------------------
// pa_decode without a workspace on many units: persistent CTAs
// ----------------------------------------------------------------------------

// A bf16 batch with more (sequence, KV head) units than two per resident CTA, and no
// window or page selection, runs one CTA of eight warps per SM instead of one CTA per
// unit.  Every CTA computes the same static schedule from the lengths ("water
// filling"): the units, longest first, are dealt out in rounds; each round's units
// fill the least loaded CTAs up to a common level, a unit going to the CTA in whose
// share the midpoint of its tiles falls.  Each CTA so gets about the mean number of
// tiles, and no unit is split across CTAs (there is no memory to merge them in).  A
// CTA's units form one stream of tiles, cut into eight equal contiguous segments, one
// per warp: each warp's ring runs on from one unit into the next, a long unit is read
// by several warps, and a unit inside one segment is finished by its warp alone.  A
// unit that crosses segments is joined in shared memory: each warp before the last
// that holds part of it leaves its state in its mailbox (a warp's only part that ends
// before the unit does), and the warp holding the unit's last tile folds those parts,
// in warp order, into its own and writes the output.  The schedule, the segments and
// the fold order are fixed by the inputs, so results repeat bit for bit.
constexpr int kPersistWarps = 8;
constexpr int kPersistMaxUnits = 4096;   // the unit list's capacity: any batch's units fit
constexpr int kPersistMaxBins = 256;     // CTAs of the launch (one per SM)
constexpr int kPersistMaxRounds = 24;    // rounds of the water filling (at least U / 16 units each)

template <class B>
struct PersistCfg : B {
  static constexpr int WARPS = kPersistWarps;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int GP = 8 * B::NT;
  static constexpr int RING = 1024 + WARPS * (B::STAGES * (B::STAGE_BYTES + 8 + B::META_BYTES) +
                                              B::QF_BYTES);
  static constexpr int MAILBOX_BYTES = WARPS * GP * (B::D + 2) * 4;   // acc, m, l per warp
  static constexpr int LIST_BYTES = kPersistMaxUnits * 2 + (kPersistMaxUnits + 1 + WARPS + 4) * 4;
  static constexpr int SMEM = RING + MAILBOX_BYTES + LIST_BYTES;
  static_assert(!B::QUANT && B::NT == 1, "persistent CTAs serve bf16 units of up to 8 heads");
  static_assert(SMEM <= 227 * 1024, "one persistent CTA per SM");
};

// Shared scratch of the schedule (in the stage area, before any copy is issued).
template <int NW>
struct PersistScratch {
  static constexpr int NB = kRankBuckets;
  int32_t gp[kPersistMaxUnits + 1];         // tiles of the units before position k
  int32_t lo[kPersistMaxBins];              // a round's first unit of each CTA
  int32_t tiles[kPersistMaxUnits];          // attended tiles per sequence
  int32_t order[kPersistMaxUnits];          // longest-first position -> sequence
  int32_t uid[kPersistMaxUnits];            // longest-first position -> unit
  int32_t hist[NW][NB];                     // per-warp bucket counts, then sort bases
  int32_t wsum[NW];                         // block scans: per-warp totals
  long long wsum64[NW];
  long long red[2][NW];                     // the fill level's reductions (two in turn)
  int32_t mine[kPersistMaxRounds][2];       // this CTA's unit range of each round
  uint8_t bucket[kPersistMaxUnits];
};

// Block-wide exclusive scan of one value per thread (every thread gets the total).
template <int THREADS, class T>
__device__ __forceinline__ T block_scan_excl(T v, T *wsum, T &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  T off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) {
    off += w < warp ? wsum[w] : 0;
    tot += wsum[w];
  }
  __syncthreads();   // wsum is free again
  total = tot;
  return off + inc - v;
}

// The schedule: this CTA's units (ids sequence * Hkv + KV head) in stream order, with
// starts[k] = tiles of the units before unit k (starts[n] = the CTA's tiles).  Returns n.
// The launch keeps every sum of tiles below 2^30.
template <int THREADS>
__device__ int persist_schedule(const Params &p, PersistScratch<THREADS / 32> &s,
                                uint16_t *units, int32_t *starts) {
  constexpr int NW = THREADS / 32, NB = PersistScratch<NW>::NB;
  static_assert(THREADS >= NB && THREADS >= kPersistMaxBins, "a bucket and a CTA per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B, H = p.Hkv, U = B * H, bins = gridDim.x;
  const int cap = p.max_blocks * p.bs;
  for (int b = tid; b < B; b += THREADS) {
    const int L = __ldg(p.seq_lens + b);
    if ((L < 0 || L > cap) && blockIdx.x == 0) set_err(p.err, PA_DEVERR_SEQ_LEN);
    const int n = seq_tiles(min(max(L, 0), cap), 0).count;
    s.tiles[b] = n;
    s.bucket[b] = static_cast<uint8_t>(tile_bucket(n));
  }
  for (int i = tid; i < NW * NB; i += THREADS) (&s.hist[0][0])[i] = 0;
  __syncthreads();
  // ---- stable order of the sequences: bucket descending, then index.  Warp w counts
  // and places the sequences of its own contiguous range.
  const int per = (B + NW - 1) / NW;
  const int lo = min(B, warp * per), hi = min(B, lo + per);
  for (int b = lo + lane; b < hi; b += 32) atomicAdd(&s.hist[warp][s.bucket[b]], 1);
  __syncthreads();
  {
    // first position of bucket k: the sequences in higher buckets (thread t: bucket NB-1-t)
    const int k = NB - 1 - tid;
    int cnt = 0;
    if (tid < NB)
#pragma unroll
      for (int w = 0; w < NW; ++w) cnt += s.hist[w][k];
    int total;
    int first = block_scan_excl<THREADS>(cnt, s.wsum, total);
    if (tid < NB)
#pragma unroll
      for (int w = 0; w < NW; ++w) {   // warp w's first position in bucket k
        const int c = s.hist[w][k];
        s.hist[w][k] = first;
        first += c;
      }
  }
  __syncthreads();
  for (int b0 = lo; b0 < hi; b0 += 32) {
    const int b = b0 + lane;
    const int key = b < hi ? s.bucket[b] : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const uint32_t below = peers & ((1u << lane) - 1u);
    if (b < hi) s.order[s.hist[warp][key] + __popc(below)] = b;
    __syncwarp();
    if (b < hi && below == 0) s.hist[warp][key] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // ---- the units in that order (KV heads in turn) and the prefix of their tiles
  {
    const int run = (U + THREADS - 1) / THREADS;
    const int k0 = min(U, tid * run), k1 = min(U, k0 + run);
    int mine = 0;
    for (int k = k0; k < k1; ++k) {
      const int q = k / H, b = s.order[q];
      s.uid[k] = b * H + (k - q * H);
      mine += s.tiles[b];
    }
    int total;
    int at = block_scan_excl<THREADS>(mine, s.wsum, total);
    for (int k = k0; k < k1; ++k) {
      s.gp[k] = at;
      at += s.tiles[s.uid[k] / H];
    }
    if (tid == 0) s.gp[U] = total;
  }
  __syncthreads();
  // ---- water filling.  Round r deals the next max(bins * (r + 1), U / 16) units of the
  // order; thread b < bins keeps CTA b's load.
  const bool has_bin = tid < bins;
  int lb = 0;
  int rounds = 0;
  for (int next = 0, r = 0; next < U; ++r) {
    const int c = min(U - next, max(bins * (r + 1), (U + 15) / 16));
    const int base = s.gp[next], tot = s.gp[next + c] - base;
    // The fill level: the CTAs S below it take the round's tiles, h = (tot + their
    // loads) / |S|.  From S = every CTA, dropping those at or above the level lowers
    // it; S is final when none drops (a round of no tiles keeps the least loaded).
    bool in = has_bin;
    long long A = 0;
    int m = 0;
    for (int it = 0;; ++it) {
      long long v = in ? ((1ll << 40) | lb) : 0ll;   // members in bits 40.., loads below
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s.red[it & 1][warp] = v;
      __syncthreads();
      long long t = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) t += s.red[it & 1][w];
      m = static_cast<int>(t >> 40);
      A = tot + (t & ((1ll << 40) - 1));
      const bool stay = in && static_cast<long long>(lb) * m < A;
      const int nm = __syncthreads_count(stay);
      if (nm == m || nm == 0) break;
      in = stay;
    }
    // shares in CTA order: h - load for each member, one tile more for its first rem
    // members, so that they add up to tot; CTA b's share is [cum, cum + share)
    const long long h = A / m, rem = A - h * m;
    long long shares;
    const long long px = block_scan_excl<THREADS>(in ? ((1ll << 40) | (h - lb)) : 0ll, s.wsum64,
                                                  shares);
    // CTA b takes the units whose tile midpoints fall in its share: from the first unit
    // whose midpoint reaches cum up to the next CTA's first (CTAs without a share take none)
    if (has_bin) {
      const long long cum2 = 2 * ((px & ((1ll << 40) - 1)) + min(px >> 40, rem));
      int a = next, z = next + c;   // first k in [next, next + c) with 2 mid(k) >= cum2
      while (a < z) {
        const int md = (a + z) >> 1;
        if (static_cast<long long>(s.gp[md]) + s.gp[md + 1] - 2ll * base >= cum2) z = md;
        else a = md + 1;
      }
      s.lo[tid] = a;
    }
    __syncthreads();
    if (has_bin) {
      const int k0 = tid == 0 ? next : s.lo[tid], k1 = tid + 1 < bins ? s.lo[tid + 1] : next + c;
      lb += s.gp[k1] - s.gp[k0];
      if (tid == static_cast<int>(blockIdx.x)) {
        s.mine[r][0] = k0;
        s.mine[r][1] = k1;
      }
    }
    __syncthreads();   // lo is read before the next round writes it
    next += c;
    rounds = r + 1;
  }
  // ---- this CTA's list: its ranges of the order, round by round
  int n = 0;
  for (int r = 0; r < rounds; ++r) {
    const int k0 = s.mine[r][0], k1 = s.mine[r][1];
    for (int k = k0 + tid; k < k1; k += THREADS) {
      units[n + k - k0] = static_cast<uint16_t>(s.uid[k]);
      starts[n + k - k0] = s.gp[k] - s.gp[k0];   // within the range, made absolute below
    }
    n += k1 - k0;
  }
  __syncthreads();
  for (int r = 0, at = 0, off = 0; r < rounds; ++r) {   // ranges' tile offsets
    const int k0 = s.mine[r][0], k1 = s.mine[r][1];
    for (int k = k0 + tid; k < k1; k += THREADS) starts[at + k - k0] += off;
    at += k1 - k0;
    off += s.gp[k1] - s.gp[k0];
    if (r == rounds - 1 && tid == 0) starts[n] = off;
  }
  __syncthreads();
  return n;
}

// Warp w's segment [begin, end) of its CTA's tile stream.
struct PersistSource {
  const uint16_t *units;           // shared: the CTA's list
  const int32_t *starts;
  const int32_t *seq_lens, *block_tables, *shared_prefix_lens;
  int32_t *err;
  int n, begin, end, Hkv, bs, nblocks, max_blocks;
  int base;
  int4 cur, nxt;

  __device__ __forceinline__ int count() const { return end - begin; }
  __device__ __forceinline__ int4 load(int i) const {
    const int g = begin + i;
    if (g >= end) return make_int4(0, 0, -1, 0);   // never issued
    int a = 0, z = n - 1;   // the unit holding position g: largest k with starts[k] <= g
    while (a < z) {
      const int md = (a + z + 1) >> 1;
      if (starts[md] <= g) a = md; else z = md - 1;
    }
    const int unit = units[a], b = unit / Hkv, kvh = unit - b * Hkv;
    const int nk = starts[a + 1] - starts[a], j = g - starts[a];
    const int L = min(max(__ldg(seq_lens + b), 0), max_blocks * bs);
    const SeqTiles geo = seq_tiles(L, 0);
    int phys = __ldg(block_tables + static_cast<size_t>(b) * max_blocks + (j * kTile) / bs);
    if (phys < 0 || phys >= nblocks) {
      set_err(err, PA_DEVERR_BLOCK_ID);
      phys = kInvalidPhys;
    }
    int info = (j == nk - 1) ? geo.last_valid : kTile;
    if (j == 0) info |= kFirstOfPair | kPieceStart;
    if (j == nk - 1) info |= kLastOfPair | kPieceEnd;
    if (i == 0) info |= kPieceStart;
    if (g == end - 1) info |= kPieceEnd;
    if (shared_prefix_lens)
      info |= ((j + 1) * kTile <= __ldg(shared_prefix_lens + b)) ? kHintShared : kHintPrivate;
    return tile_record(phys, j, unit, kvh, Hkv, bs, nblocks, info | (kvh << kKvhShift));
  }
  __device__ __forceinline__ void init(int lane) {
    base = 0;
    cur = load(lane);
    nxt = load(32 + lane);
  }
  __device__ __forceinline__ int4 get(int i, int lane) {
    while (i >= base + 32) {
      cur = nxt;
      base += 32;
      nxt = load(base + 32 + lane);
    }
    return shfl_int4(cur, i - base);
  }
};

// Lane 0 polls a shared flag until it reads nonzero (bounded: a wait that runs out sets
// the error flag and returns false).  Returns for the whole warp.
__device__ __forceinline__ bool persist_wait(const volatile int32_t *flag, int32_t *err, int lane) {
  int ok = 1;
  if (lane == 0) {
    uint32_t i = 0;
    while (*flag == 0) {
      if (++i == kWaitSpins) {
        ok = 0;
        set_err(err, PA_DEVERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __threadfence_block();
  return ok != 0;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    decode_persist_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const Params p) {
  constexpr int GP = C::GP, W = C::WARPS;
  using Scratch = PersistScratch<C::THREADS / 32>;
  static_assert(sizeof(Scratch) <= W * C::STAGES * C::STAGE_BYTES,
                "the schedule's scratch lives in the stage area");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  float *box_acc = reinterpret_cast<float *>(split_tail<C>(smem_raw));   // [W][GP][D]
  float *box_m = box_acc + W * GP * C::D;                                 // [W][GP]
  float *box_l = box_m + W * GP;                                          // [W][GP]
  uint16_t *units = reinterpret_cast<uint16_t *>(box_l + W * GP);        // [max units]
  int32_t *starts = reinterpret_cast<int32_t *>(units + kPersistMaxUnits); // [max units + 1]
  int32_t *filled = starts + kPersistMaxUnits + 1;                        // [W] mailbox flags
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  // the schedule reads only caller inputs (lengths); the output and the pools (written
  // by the cache write) are touched only after the previous grid has finished
  const int n = persist_schedule<C::THREADS>(p, *reinterpret_cast<Scratch *>(base), units, starts);
  pdl_wait();
  if (threadIdx.x < W) filled[threadIdx.x] = 0;
  // units without tiles (empty sequences) have no warp to write them
  for (int k = warp; k < n; k += W) {
    if (starts[k + 1] > starts[k]) continue;
    const int unit = units[k], b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    float *out = p.out + (static_cast<size_t>(b) * p.Hq + kvh * p.G) * C::D;
    for (int e = lane; e < p.G * C::D; e += 32) out[e] = 0.f;
  }
  __syncthreads();   // the scratch is read: the stages may be filled

  const int T = starts[n];
  auto seg = [&](int w) { return static_cast<int>(static_cast<long long>(w) * T / W); };
  WarpSmem ws = setup_smem<C>(smem_raw, warp, p.G, lane);
  State<C> st, held;
  st.reset();
  held.reset();
  PersistSource src;
  src.units = units;
  src.starts = starts;
  src.seq_lens = p.seq_lens;
  src.block_tables = p.block_tables;
  src.shared_prefix_lens = p.shared_prefix_lens;
  src.err = p.err;
  src.n = n;
  src.begin = seg(warp);
  src.end = seg(warp + 1);
  src.Hkv = p.Hkv;
  src.bs = p.bs;
  src.nblocks = p.nblocks;
  src.max_blocks = p.max_blocks;
  src.init(lane);
  auto out_of = [&](int unit) {
    const int b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    return p.out + (static_cast<size_t>(b) * p.Hq + kvh * p.G) * C::D;
  };
  const int qd = lane & 3;
  // this warp's mailbox: m, l (totals over the warp) and acc of a state
  auto deposit = [&](const float (&m)[2], const float (&l)[2], auto &&acc_of) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int g = 2 * qd + j;
      if ((lane >> 2) == 0) {
        box_m[warp * GP + g] = m[j];
        box_l[warp * GP + g] = l[j];
      }
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          box_acc[(warp * GP + g) * C::D + acc_d<C>(dt, j + 2 * h, lane)] = acc_of(dt, j + 2 * h);
    }
    __threadfence_block();
    __syncwarp();
    if (lane == 0) *reinterpret_cast<volatile int32_t *>(&filled[warp]) = 1;
  };
  int held_unit = -1;
  bool held_last = false;
  auto on_end = [&](int4 u, bool piece_first, State<C> &s) {
    const bool last = (u.w & kLastOfPair) != 0;
    if (piece_first && last) {              // a whole unit: finished here
      write_normalised<C>(s, out_of(u.y), nullptr, p.G, lane);
    } else if (!piece_first) {              // the unit came from the warps before
      held = s;
      held_unit = u.y;
      held_last = last;
    } else {                                // the unit goes on into the next warp
      float lt[1][2];
      reduce_l<C>(s, lt);
      const float mm[2] = {s.m[0][0], s.m[0][1]}, ll[2] = {lt[0][0], lt[0][1]};
      deposit(mm, ll, [&](int dt, int i) { return s.acc[0][dt][i]; });
    }
  };
  const bool ok = run_warp<C>(src, ws, st, p, &tmK, &tmV, on_end, lane);
  if (held_unit < 0 || !ok) return;
  float lt[1][2];
  reduce_l<C>(held, lt);
  if (!held_last) {   // the unit goes on past this segment: its last warp folds this part
    const float mm[2] = {held.m[0][0], held.m[0][1]}, ll[2] = {lt[0][0], lt[0][1]};
    deposit(mm, ll, [&](int dt, int i) { return held.acc[0][dt][i]; });
    return;
  }
  // ---- the unit's last warp: fold the parts the warps before left in their mailboxes,
  // in warp order, then its own, and write the output
  int k = 0;   // the unit: the one holding this segment's first tile
  for (int z = n - 1; k < z;) {
    const int md = (k + z + 1) >> 1;
    if (starts[md] <= src.begin) k = md; else z = md - 1;
  }
  float M[2] = {-INFINITY, -INFINITY}, L[2] = {0.f, 0.f}, acc[C::DT][4];
#pragma unroll
  for (int dt = 0; dt < C::DT; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
  auto fold = [&](const float (&mo)[2], const float (&lo)[2], auto &&acc_of) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float Mn = fmaxf(M[j], mo[j]);
      const float fa = M[j] == -INFINITY ? 0.f : ex2(M[j] - Mn);
      const float fb = mo[j] == -INFINITY ? 0.f : ex2(mo[j] - Mn);
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
        for (int h = 0; h < 2; ++h) acc[dt][j + 2 * h] = acc[dt][j + 2 * h] * fa + acc_of(dt, j + 2 * h) * fb;
      L[j] = L[j] * fa + lo[j] * fb;
      M[j] = Mn;
    }
  };
  for (int w = 0; w < warp; ++w) {
    if (seg(w + 1) <= starts[k] || seg(w) == seg(w + 1)) continue;   // holds none of the unit
    if (!persist_wait(&filled[w], p.err, lane)) return;
    float mo[2], lo[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mo[j] = box_m[w * GP + 2 * qd + j];
      lo[j] = box_l[w * GP + 2 * qd + j];
    }
    fold(mo, lo, [&](int dt, int i) {
      return box_acc[(w * GP + 2 * qd + (i & 1)) * C::D + acc_d<C>(dt, i, lane)];
    });
  }
  {
    const float mo[2] = {held.m[0][0], held.m[0][1]}, lo[2] = {lt[0][0], lt[0][1]};
    fold(mo, lo, [&](int dt, int i) { return held.acc[0][dt][i]; });
  }
  float *out = out_of(held_unit);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int g = 2 * qd + j;
    if (g >= p.G) continue;
    const float inv = L[j] > 0.f ? 1.f / L[j] : 0.f;
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
      for (int h = 0; h < 2; ++h) out[g * C::D + acc_d<C>(dt, j + 2 * h, lane)] = acc[dt][j + 2 * h] * inv;
  }
}

// ----------------------------------------------------------------------------
// pa_decode_splitkv: plan (scan + unit list), segmented decode, merge
// ----------------------------------------------------------------------------

__device__ __forceinline__ int clamp_len(int L, int cap) { return min(max(L, 0), cap); }

// Block-wide scan of the sequence lengths into shared memory:
//   prefix[b] = Hkv * sum_{b' < b} count(b'),  prefix[B] = total tiles,
// where count(b) is the number of 16-token tiles sequence b attends over.
// Out-of-range lengths are clamped (and reported once, by CTA 0).  Returns the
// largest count (the longest unit).
template <int THREADS>
__device__ int scan_lengths(const Params &p, int32_t *prefix) {
  __shared__ int warp_sums[THREADS / 32];
  __shared__ int carry_s, nmax_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cap = p.max_blocks * p.bs;
  if (tid == 0) carry_s = nmax_s = 0;
  __syncthreads();
  for (int base = 0; base < p.B; base += THREADS) {
    const int i = base + tid;
    int v = 0;
    if (i < p.B) {
      const int L0 = p.seq_lens[i];
      const int ct = p.casc_tiles ? p.casc_tiles[i] : 0;
      if ((L0 < 0 || L0 > cap || L0 < ct * kTile) && blockIdx.x == 0)
        set_err(p.err, PA_DEVERR_SEQ_LEN);
      const int c = pair_tile_count(clamp_len(L0, cap), p.window, p.topk, ct);
      if (c > 0) atomicMax(&nmax_s, c);
      v = p.Hkv * c;
    }
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    int before = carry_s;
    for (int w = 0; w < warp; ++w) before += warp_sums[w];
    if (i < p.B) prefix[i] = before + x - v;
    __syncthreads();
    if (tid == THREADS - 1) carry_s = before + x;
    __syncthreads();
  }
  if (tid == 0) prefix[p.B] = carry_s;
  __syncthreads();
  return nmax_s;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS)
    decode_segment_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  WarpSmem ws = setup_smem<C>(smem_raw, warp, p.G, lane);
  int32_t *prefix = reinterpret_cast<int32_t *>(split_tail<C>(smem_raw));
  if (p.casc_tiles) pdl_wait();   // the cascaded tiles are written by the cascade kernel
  const int nmax = scan_lengths<C::THREADS>(p, prefix);
  const int seg = blockIdx.x * C::WARPS + warp;
  const int total = prefix[p.B];
  int W = max(1, (total + p.num_splits - 1) / p.num_splits);
  // pa_decode_splitkv: a unit of n tiles is cut into at most ceil((n - 1) / W) + 1
  // pieces, so W >= (nmax - 1) / (S - 1) keeps every unit within its S slots; with
  // S = 1 the segment bounds move to the next unit start, so no unit is cut
  const int S = p.parts_S;
  if (S >= 2) W = max(W, (nmax - 1 + S - 2) / (S - 1));
  SegmentSource src;
  src.prefix = prefix;
  src.seq_lens = p.seq_lens;
  src.block_tables = p.block_tables;
  src.shared_prefix_lens = p.shared_prefix_lens;
  src.err = p.err;
  src.B = p.B;
  src.Hkv = p.Hkv;
  src.bs = p.bs;
  src.nblocks = p.nblocks;
  src.max_blocks = p.max_blocks;
  src.window = p.window;
  src.sel = p.sel;
  src.topk = p.topk;
  src.casc_tiles = p.casc_tiles;
  src.begin = min(seg * W, total);
  src.end = (seg < p.num_splits) ? min(src.begin + W, total) : src.begin;
  if (S == 1) {
    auto unit_start_at_or_after = [&](int f) {   // f <= total
      if (f >= total) return total;
      int lo = 0, hi = p.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= f) lo = mid; else hi = mid - 1;
      }
      const int nt = (prefix[lo + 1] - prefix[lo]) / p.Hkv;
      const int us = prefix[lo] + (f - prefix[lo]) / nt * nt;
      return us < f ? us + nt : us;
    };
    src.begin = unit_start_at_or_after(src.begin);
    src.end = unit_start_at_or_after(src.end);
  }
  // the chosen pages are written by the selection launched just before
  if (p.sel) pdl_wait();
  src.init(lane);
  // without a selection everything above reads only caller inputs (lengths, block
  // tables); the pools (written by the cache write) and the workspace (read by the
  // previous merge) are touched only after the previous grid has finished
  pdl_wait();
  if (S > 0) {
    // sequences with no tile to attend have no piece: all their slots are empty
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
      if (prefix[b + 1] != prefix[b]) continue;
      float *l = p.parts_lse + static_cast<size_t>(b) * p.Hq * S;
      const size_t n = static_cast<size_t>(p.Hq) * S;
      for (size_t i = threadIdx.x; i < n; i += C::THREADS) l[i] = -INFINITY;
    }
  } else if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= p.B; i += C::THREADS) p.prefix_out[i] = prefix[i];
    if (threadIdx.x == 0) {                 // for the merge: KV heads per unit, cascade
      p.prefix_out[p.B + 1] = C::HEADS;
      p.prefix_out[p.B + 2] = static_cast<int32_t>(static_cast<uint32_t>(p.casc_ws));
      p.prefix_out[p.B + 3] = static_cast<int32_t>(static_cast<uint32_t>(p.casc_ws >> 32));
    }
  }
  State<C> st;
  st.reset();
  run_warp<C>(
      src, ws, st, p, &tmK, &tmV,
      [&](int4 u, bool piece_first, State<C> &s) {
        const int b = u.y / p.Hkv, kvh = u.y - b * p.Hkv;
        const size_t row = static_cast<size_t>(b) * p.Hq + kvh * p.G;
        if (S > 0) {
          // piece k of the unit: the segments before this one that hold its tiles
          const int nt = (prefix[b + 1] - prefix[b]) / p.Hkv;
          const int k = S == 1 ? 0 : seg - (prefix[b] + kvh * nt) / W;
          write_normalised<C>(s, p.parts_o + (row * S + k) * C::D, p.parts_lse + row * S + k,
                              p.G, lane, static_cast<size_t>(S) * C::D, S);
          if (u.w & kLastOfPair) {              // the unit's last piece: later slots are empty
            const int rest = S - 1 - k;
            for (int i = lane; i < p.G * rest; i += 32) {
              const int g = i / rest;
              p.parts_lse[(row + g) * S + k + 1 + (i - g * rest)] = -INFINITY;
            }
          }
        } else if (piece_first && (u.w & kLastOfPair)) {   // the whole unit is in this segment
          if (u.w & kCascade) {                     // joined with its shared prefix by the merge
            const CascadeLayout cl = cascade_layout(p.B, p.Hq, C::D);
            uint8_t *cw = reinterpret_cast<uint8_t *>(p.casc_ws);
            write_normalised<C>(s, reinterpret_cast<float *>(cw + cl.uo) + row * C::D,
                                reinterpret_cast<float *>(cw + cl.ulse) + row, p.G, lane);
          } else {
            write_normalised<C>(s, p.out + row * C::D, nullptr, p.G, lane);
          }
        } else {
          const size_t slot = static_cast<size_t>(seg) * 2 + (piece_first ? 1 : 0);
          write_normalised<C>(s, p.o_part + slot * p.G * C::D, p.lse_part + slot * p.G, p.G,
                              lane);
        }
      },
      lane);
}

// One CTA per (b, kvh) pair; threads over (head, 4 consecutive d).  The pieces of a
// pair are visited eight at a time with their loads issued together.  The decode
// leaves the number of KV heads per unit (1, or 2 for paired 4-bit heads) after
// the tile prefix: head kvh's partials are then rows (kvh % 2) G .. of unit kvh / 2.
__global__ void __launch_bounds__(256) merge_kernel(float *out, const int32_t *prefix,
                                                    const float *o_part, const float *lse_part,
                                                    int B, int Hq, int Hkv, int G, int D,
                                                    int num_splits) {
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int b = pair / Hkv, kvh = pair - b * Hkv;
  const int heads = prefix[B + 1] == 2 ? 2 : 1;
  const int unit = kvh / heads, row0 = (kvh - unit * heads) * G;
  const int Hu = Hkv / heads, Gu = G * heads;      // units per sequence, rows per unit
  const int start_b = prefix[b];
  const int nt = (prefix[b + 1] - start_b) / Hu;
  const int total = prefix[B];
  const int W = max(1, (total + num_splits - 1) / num_splits);
  float *o = out + (static_cast<size_t>(b) * Hq + kvh * G) * D;
  const int D4 = D / 4;
  // a cascaded sequence adds the partials of its shared prefix (cascade workspace);
  // a unit finished inside one segment was joined with them there
  const uint64_t cws = (static_cast<uint64_t>(static_cast<uint32_t>(prefix[B + 3])) << 32) |
                       static_cast<uint32_t>(prefix[B + 2]);
  const float *clse = nullptr, *co = nullptr;
  const int cpieces = cascade_partials(cws, B, Hq, Hkv, G, D, b, kvh, clse, co);
  if (nt == 0 && cpieces == 0) {
    for (int e = threadIdx.x; e < G * D4; e += blockDim.x)
      reinterpret_cast<float4 *>(o)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int start = start_b + unit * nt, end = start + nt;
  // split pieces p0..p1 (none when the cascade covers the whole sequence)
  int p0 = nt > 0 ? start / W : 0, p1 = nt > 0 ? (end - 1) / W : -1;
  const bool inplace = nt > 0 && p0 == p1;         // finished inside one segment
  if (inplace && cpieces == 0) return;
  // a cascaded unit finished in place left its (o, lse) in the unit slots
  const float *ulse = nullptr, *uo = nullptr;
  if (inplace) {
    const CascadeLayout cl = cascade_layout(B, Hq, D);
    const uint8_t *cw = reinterpret_cast<const uint8_t *>(cws);
    const size_t row = static_cast<size_t>(b) * Hq + kvh * G;
    ulse = reinterpret_cast<const float *>(cw + cl.ulse) + row;
    uo = reinterpret_cast<const float *>(cw + cl.uo) + row * D;
    p1 = p0 - 1;                                   // no split pieces
  }
  // one pass: each batch of up to U pieces' (lse, o) is loaded together, then folded into
  // a running maximum M with num and den rescaled when it rises
  constexpr int U = 8;
  for (int e = threadIdx.x; e < G * D4; e += blockDim.x) {
    const int g = e / D4, d4 = e - g * D4, gu = row0 + g;
    auto slot = [&](int s) { return static_cast<size_t>(s) * 2 + (s == p0 ? 1 : 0); };
    float M = -INFINITY, den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fold = [&](float l, float4 x) {           // one piece; l = -inf adds nothing
      if (l > M) {
        const float r = expf(M - l);               // 0 while M is -inf
        num = make_float4(num.x * r, num.y * r, num.z * r, num.w * r);
        den *= r;
        M = l;
      }
      const float w = l == -INFINITY ? 0.f : expf(l - M);
      num.x += w * x.x;
      num.y += w * x.y;
      num.z += w * x.z;
      num.w += w * x.w;
      den += w;
    };
    if (ulse) fold(ulse[g], reinterpret_cast<const float4 *>(uo + g * D)[d4]);
    for (int c = 0; c < cpieces; ++c)              // the cascade's pieces of the prefix
      fold(clse[c * G + g], reinterpret_cast<const float4 *>(co + (c * G + g) * D)[d4]);
    for (int s0 = p0; s0 <= p1; s0 += U) {
      float l[U];
      float4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool ok = s0 + u <= p1;
        l[u] = ok ? __ldg(lse_part + slot(s0 + u) * Gu + gu) : -INFINITY;
        x[u] = ok ? __ldg(reinterpret_cast<const float4 *>(o_part + (slot(s0 + u) * Gu + gu) * D) + d4)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float bm = l[0];
#pragma unroll
      for (int u = 1; u < U; ++u) bm = fmaxf(bm, l[u]);
      if (bm > M) {                                // raise M once per batch
        const float r = expf(M - bm);
        num = make_float4(num.x * r, num.y * r, num.z * r, num.w * r);
        den *= r;
        M = bm;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float w = l[u] == -INFINITY ? 0.f : expf(l[u] - M);
        num.x += w * x[u].x;
        num.y += w * x[u].y;
        num.z += w * x[u].z;
        num.w += w * x[u].w;
        den += w;
      }
    }
    const float inv = 1.f / den;
    reinterpret_cast<float4 *>(o)[e] = make_float4(num.x * inv, num.y * inv, num.z * inv,
                                                   num.w * inv);
  }
}

// pa_merge_lse: one warp per query head (b, h), a CTA per (sequence, KV head) group.
// Partials of the head are o_part[b][h][i][:], lse[b][h][i] for i < S; an lse of -inf
// (or a weight that underflows to 0) marks an empty slot, whose o row is not read.
// Lane i reads slot i of each 32-slot chunk: the running maximum and the normaliser take
// warp reductions, and only the non-empty slots' o rows are read (each row coalesced
// over the warp, D / 32 elements per lane).  A head with no partial gets zeros.
template <int D>
__global__ void __launch_bounds__(512) merge_parts_kernel(float *out, const float *o_part,
                                                          const float *lse, int G, int S) {
  pdl_trigger();
  pdl_wait();
  constexpr int E = D / 32;   // elements per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t r = static_cast<size_t>(blockIdx.x) * G + warp;   // head row b * Hq + h
  const float *lr = lse + r * S;
  const float *orow = o_part + r * S * D;
  float M = -INFINITY;
  for (int s0 = 0; s0 < S; s0 += 32)
    M = fmaxf(M, s0 + lane < S ? __ldg(lr + s0 + lane) : -INFINITY);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float den = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < S; s0 += 32) {
      const float l = s0 + lane < S ? __ldg(lr + s0 + lane) : -INFINITY;
      const float w = l == -INFINITY ? 0.f : expf(l - M);
      den += w;
      // the live slots' rows in increasing slot order, four rows' loads in flight at
      // once (a head of a long sequence has tens of live slots)
      for (uint32_t live = __ballot_sync(0xffffffffu, w > 0.f); live;) {
        constexpr int U = 4;
        float wj[U], x[U][E];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = live ? __ffs(live) - 1 : -1;   // warp-uniform
          live &= live - 1;
          wj[u] = __shfl_sync(0xffffffffu, w, j < 0 ? 0 : j);
          const float *row = orow + static_cast<size_t>(s0 + (j < 0 ? 0 : j)) * D;
#pragma unroll
          for (int e = 0; e < E; ++e) x[u][e] = j < 0 ? 0.f : __ldg(row + e * 32 + lane);
          if (j < 0) wj[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] += wj[u] * x[u][e];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) out[r * D + e * 32 + lane] = acc[e] * inv;
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2D view of a pool: rows = nblocks * bs tokens, columns = one token's Hkv head rows
// (bf16 elements, or bytes for the code pools); box = 16 rows x one head row of up to
// 128 bytes, swizzled by the box width (128 or 64 bytes).
// s: the decode's view of the shape (Hkv counts units of `heads` adjacent KV heads).
bool make_pool_map(CUtensorMap *map, const void *pool, const pa_shape &s, int heads) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool bf16 = s.kv_dtype == PA_KV_BF16;
  const int row_bytes = heads * (s.kv_dtype == PA_KV_INT4 ? s.D / 2 : (bf16 ? 2 * s.D : s.D));
  const int box_bytes = row_bytes < 128 ? row_bytes : 128;
  const int eb = bf16 ? 2 : 1;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.Hkv) * row_bytes / eb,
                        static_cast<cuuint64_t>(s.nblocks) * s.block_size};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(s.Hkv) * row_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / eb), static_cast<cuuint32_t>(kTile)};
  cuuint32_t estr[2] = {1, 1};
  // promote L2 fills to one head row: 256 B for bf16 D = 128, 128 B for 128-byte
  // rows, none for 64-byte rows (a wider fill would pull in the next head's row)
  const CUtensorMapL2promotion promo =
      row_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                       : (row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                           : CU_TENSOR_MAP_L2_PROMOTION_NONE);
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void *>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, promo,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Opt the kernel in to the dynamic shared memory it needs (per call: cheap, and
// correct whichever device is current).
template <class K>
static cudaError_t prep_kernel(K kernel, int smem) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

static Params make_params(const pa_shape &s, float *out, const void *q, const float *k_scale,
                          const float *v_scale, const int32_t *bt, const int32_t *sl,
                          const pa_decode_opts *opts, float sm_scale, int32_t *err) {
  Params p{};
  p.window = opts ? opts->window : 0;
  p.topk = (opts && opts->selected_pages) ? opts->topk : 0;
  p.sel = p.topk > 0 ? opts->selected_pages : nullptr;
  p.out = out;
  p.q = static_cast<const uint16_t *>(q);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = bt;
  p.seq_lens = sl;
  p.err = err;
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

// CTAs per (sequence, KV head) unit in pa_decode.  With at most two units per resident
// CTA, one long sequence would be left to a single CTA at the end of the launch: such
// batches get a cluster of four CTAs per unit (of which a short unit keeps only as
// many as it has tiles for).  Larger batches keep one CTA per unit.  So do launches
// whose window or page selection bounds every unit's tiles when the units fill the GPU
// (bounded units are near-uniform: a cluster would only add CTAs), and launches whose
// bound is one CTA's share (the cluster's other CTAs would all sit idle).
template <class C>
static int pair_cluster_ctas(int units, int resident_ctas, int window, int topk) {
  if (units > 2 * resident_ctas) return 1;
  const bool bounded = topk > 0 || window > 0;
  if (bounded && units >= resident_ctas) return 1;
  const int share = kClusterWarpTiles * C::WARPS;   // tiles one CTA takes before another joins
  const int max_tiles = topk > 0 ? topk : (window > 0 ? (window + kTile - 2) / kTile + 1 : 1 << 30);
  return max_tiles <= share ? 1 : 4;
}

// pa_decode without a workspace on a bf16 batch of more units than two per resident
// CTA (and at most kPersistMaxUnits), with no window or page selection: one persistent
// CTA of eight warps per SM on a static water-filled schedule.
template <class C>
static pa_status launch_persist(const Params &p, const CUtensorMap &mk, const CUtensorMap &mv,
                                cudaStream_t stream, int sms) {
  using P = PersistCfg<C>;
  if (prep_kernel(decode_persist_kernel<P>, P::SMEM) != cudaSuccess) return PA_ERR_CUDA;
  return launch_pdl(decode_persist_kernel<P>, dim3(sms), dim3(P::THREADS), P::SMEM, stream, mk, mv,
                    p) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

template <class C>
static pa_status launch_pair_units(const Params &p, const CUtensorMap &mk, const CUtensorMap &mv,
                                   cudaStream_t stream) {
  const int units = p.B * p.Hkv;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  if constexpr (C::KIND == kKindBf16 && C::NT == 1) {
    // (every sum of tiles the schedule forms stays below 2^31)
    const long long max_tiles = (static_cast<long long>(p.max_blocks) * p.bs + kTile - 1) / kTile;
    if (units > 2 * sms * C::MIN_BLOCKS && units <= kPersistMaxUnits && sms <= kPersistMaxBins &&
        p.window == 0 && p.topk == 0 && units * max_tiles < (1ll << 30))
      return launch_persist<C>(p, mk, mv, stream, sms);
  }
  const int ncl = pair_cluster_ctas<C>(units, sms * C::MIN_BLOCKS, p.window, p.topk);
  auto one_cta_per_unit = [&]() {
    if (prep_kernel(decode_pair_kernel<C, false>, C::PAIR_SMEM) != cudaSuccess) return PA_ERR_CUDA;
    decode_pair_kernel<C, false><<<units, C::THREADS, C::PAIR_SMEM, stream>>>(mk, mv, p);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  };
  if (ncl == 1) return one_cta_per_unit();
  if (prep_kernel(decode_pair_kernel<C, true>, C::PAIR_SMEM) != cudaSuccess) return PA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units * ncl);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::PAIR_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_pair_kernel<C, true>, mk, mv, p) == cudaSuccess) return PA_OK;
  // a device (or a partition of one) that cannot place the cluster: the same
  // decode with one CTA per unit (the failed launch left no sticky error)
  (void)cudaGetLastError();
  return one_cta_per_unit();
}

// pa_decode without a workspace reads E4M3 heads singly (heads_per_unit), so the paired
// E4M3 kind has no instantiation of its kernel.
template <class C>
static pa_status launch_pair(const Params &p, const CUtensorMap &mk, const CUtensorMap &mv,
                             cudaStream_t stream) {
  if constexpr (C::KIND == kKindFp8x2)
    return PA_ERR_UNSUPPORTED;
  else
    return launch_pair_units<C>(p, mk, mv, stream);
}

template <class C>
static pa_status launch_segments(const Params &p, const CUtensorMap &mk, const CUtensorMap &mv,
                                 cudaStream_t stream) {
  const int smem = split_smem<C>(p.B);
  if (prep_kernel(decode_segment_kernel<C>, smem) != cudaSuccess) return PA_ERR_CUDA;
  const int grid = (p.num_splits + C::WARPS - 1) / C::WARPS;
  return launch_pdl(decode_segment_kernel<C>, dim3(grid), dim3(C::THREADS), smem, stream, mk, mv,
                    p) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// Dispatch on (D, n-tiles, dtype).
#define PA_DISPATCH(D_, NT_, KIND_, FN, ...)                                  \
  if (s.D == D_ && nt == NT_ && kind == KIND_) return FN<Cfg<D_, NT_, KIND_>>(__VA_ARGS__);

// 4-bit pools whose KV heads can be served two at a time: an even number of heads,
// groups of 8 query heads (one n-tile each), D = 128.  A Quest selection is per KV
// head, and the cascade stacks one KV head's query rows, so a decode with either
// serves the heads singly.
static bool int4_pairable(const pa_shape &s) {
  return s.kv_dtype == PA_KV_INT4 && s.D == 128 && s.Hkv % 2 == 0 && s.Hq == 8 * s.Hkv;
}
// E4M3 pools on the same rule.
static bool fp8_pairable(const pa_shape &s) {
  return s.kv_dtype == PA_KV_FP8_E4M3 && s.D == 128 && s.Hkv % 2 == 0 && s.Hq == 8 * s.Hkv;
}
static bool pairable(const pa_shape &s) { return int4_pairable(s) || fp8_pairable(s); }

// cascade: the decode runs the cascade (only pa_decode given a workspace does);
// cta_per_unit: pa_decode without a workspace (it pairs 4-bit heads, not E4M3 ones).
static int heads_per_unit(const pa_shape &s, const pa_decode_opts *opts, bool cascade = false,
                          bool cta_per_unit = false) {
  const bool per_head = (opts && opts->topk > 0 && opts->selected_pages) || cascade;
  const bool pair = int4_pairable(s) || (fp8_pairable(s) && !cta_per_unit);
  return (pair && !per_head) ? 2 : 1;
}

// The decode's view of the shape: units of `heads` adjacent KV heads.
static pa_shape unit_view(const pa_shape &s, int heads) {
  pa_shape v = s;
  v.Hkv = s.Hkv / heads;
  return v;
}

static int kind_of(const pa_shape &s, int heads) {
  if (s.kv_dtype == PA_KV_INT4) return heads == 2 ? kKindInt4x2 : kKindInt4;
  if (s.kv_dtype == PA_KV_FP8_E4M3) return heads == 2 ? kKindFp8x2 : kKindFp8;
  return kKindBf16;
}

#define PA_DISPATCH_ALL(FN, ...)                      \
  PA_DISPATCH(128, 1, kKindBf16, FN, __VA_ARGS__)     \
  PA_DISPATCH(128, 2, kKindBf16, FN, __VA_ARGS__)     \
  PA_DISPATCH(64, 1, kKindBf16, FN, __VA_ARGS__)      \
  PA_DISPATCH(64, 2, kKindBf16, FN, __VA_ARGS__)      \
  PA_DISPATCH(128, 1, kKindFp8, FN, __VA_ARGS__)      \
  PA_DISPATCH(128, 2, kKindFp8, FN, __VA_ARGS__)      \
  PA_DISPATCH(128, 1, kKindInt4, FN, __VA_ARGS__)     \
  PA_DISPATCH(128, 2, kKindInt4, FN, __VA_ARGS__)     \
  PA_DISPATCH(128, 2, kKindInt4x2, FN, __VA_ARGS__)   \
  PA_DISPATCH(128, 2, kKindFp8x2, FN, __VA_ARGS__)

// s: the unit view; p.G query heads per unit
static pa_status dispatch_pair(const pa_shape &s, int heads, const Params &p,
                               const CUtensorMap &mk, const CUtensorMap &mv, cudaStream_t st) {
  const int nt = (p.G + 7) / 8;
  const int kind = kind_of(s, heads);
  PA_DISPATCH_ALL(launch_pair, p, mk, mv, st)
  return PA_ERR_UNSUPPORTED;
}

static pa_status dispatch_segments(const pa_shape &s, int heads, const Params &p,
                                   const CUtensorMap &mk, const CUtensorMap &mv,
                                   cudaStream_t st) {
  const int nt = (p.G + 7) / 8;
  const int kind = kind_of(s, heads);
  PA_DISPATCH_ALL(launch_segments, p, mk, mv, st)
  return PA_ERR_UNSUPPORTED;
}

template <class C>
static int cfg_split_smem(int B) { return split_smem<C>(B); }
template <class C>
static int cfg_min_blocks(int) { return C::MIN_BLOCKS; }

// Sizing of the split kernel a decode with these options (NULL: none) launches.
int splitkv_smem_bytes(const pa_shape &shape, const pa_decode_opts *opts) {
  const int heads = heads_per_unit(shape, opts, opts && opts->num_prefix_groups > 0);
  const pa_shape s = unit_view(shape, heads);
  const int nt = (s.Hq / s.Hkv + 7) / 8;
  const int kind = kind_of(s, heads);
  PA_DISPATCH_ALL(cfg_split_smem, s.B)
  return 0;
}

int decode_warps_per_cta() { return Cfg<128, 1, false>::WARPS; }

int splitkv_min_blocks(const pa_shape &shape, const pa_decode_opts *opts) {
  const int heads = heads_per_unit(shape, opts, opts && opts->num_prefix_groups > 0);
  const pa_shape s = unit_view(shape, heads);
  const int nt = (s.Hq / s.Hkv + 7) / 8;
  const int kind = kind_of(s, heads);
  PA_DISPATCH_ALL(cfg_min_blocks, 0)
  return 1;
}

// prefix int32[B + 4] (tile prefix, KV heads per unit, cascade workspace address),
// lse f32[splits][2][Gu],
// o_part f32[splits][2][Gu][D]; Gu = query heads of the largest unit the shape allows.
WorkspaceLayout splitkv_layout(const pa_shape &s, int num_splits) {
  WorkspaceLayout w{};
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t G = static_cast<size_t>(s.Hq / s.Hkv) * (pairable(s) ? 2 : 1);
  w.prefix = 0;
  w.lse = up(w.prefix + (static_cast<size_t>(s.B) + 4) * 4);
  w.o_part = up(w.lse + static_cast<size_t>(num_splits) * 2 * G * 4);
  w.total = up(w.o_part + static_cast<size_t>(num_splits) * 2 * G * s.D * 4);
  return w;
}

pa_status run_decode(const pa_shape &s, float *out, const void *q, const void *k_pool,
                     const void *v_pool, const float *k_scale, const float *v_scale,
                     const int32_t *bt, const int32_t *sl, const pa_decode_opts *opts,
                     float sm_scale, int32_t *err, cudaStream_t stream) {
  const int heads = heads_per_unit(s, opts, false, true);
  const pa_shape v = unit_view(s, heads);
  CUtensorMap mk, mv;
  if (!make_pool_map(&mk, k_pool, v, heads) || !make_pool_map(&mv, v_pool, v, heads))
    return PA_ERR_CUDA;
  Params p = make_params(v, out, q, k_scale, v_scale, bt, sl, opts, sm_scale, err);
  p.shared_prefix_lens = opts ? opts->shared_prefix_lens : nullptr;
  return dispatch_pair(v, heads, p, mk, mv, stream);
}

pa_status run_decode_splitkv(const pa_shape &s, float *out, void *workspace, int num_splits,
                             const void *q, const void *k_pool, const void *v_pool,
                             const float *k_scale, const float *v_scale, const int32_t *bt,
                             const int32_t *sl, const pa_decode_opts *opts, float sm_scale,
                             int32_t *err, cudaStream_t stream) {
  const WorkspaceLayout w = splitkv_layout(s, num_splits);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const int heads = heads_per_unit(s, opts, opts && opts->num_prefix_groups > 0);
  const pa_shape v = unit_view(s, heads);
  CUtensorMap mk, mv;
  if (!make_pool_map(&mk, k_pool, v, heads) || !make_pool_map(&mv, v_pool, v, heads))
    return PA_ERR_CUDA;
  Params p = make_params(v, out, q, k_scale, v_scale, bt, sl, opts, sm_scale, err);
  p.shared_prefix_lens = opts ? opts->shared_prefix_lens : nullptr;
  p.prefix_out = reinterpret_cast<int32_t *>(ws + w.prefix);
  p.lse_part = reinterpret_cast<float *>(ws + w.lse);
  p.o_part = reinterpret_cast<float *>(ws + w.o_part);
  p.num_splits = num_splits;
  if (!opts || opts->num_prefix_groups <= 0) return dispatch_segments(v, heads, p, mk, mv, stream);

  // Cascade: plan on the caller's stream.  Given a side stream, fork: the cascade
  // kernel (tensor work on the shared prefixes) runs there with one CTA per SM, next
  // to the split kernel (HBM streaming of the rest, two CTAs per SM); a second cascade
  // launch after the split kernel takes the items still left at full occupancy; the
  // caller's stream waits for both before anything it runs next (the merge).  Without
  // one, the cascade runs after the split kernel on the caller's stream.
  pa_status st = run_cascade_plan(v, *opts, err, stream);
  if (st != PA_OK) return st;
  const CascadeLayout cl = cascade_layout(s.B, s.Hq, s.D);
  p.casc_tiles =
      reinterpret_cast<const int32_t *>(static_cast<const uint8_t *>(opts->cascade_workspace) + cl.tiles);
  p.casc_ws = reinterpret_cast<uint64_t>(opts->cascade_workspace);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  cudaStream_t side = reinterpret_cast<cudaStream_t>(opts->cascade_stream);
  cudaEvent_t fork = reinterpret_cast<cudaEvent_t>(opts->cascade_events[0]);
  cudaEvent_t join = reinterpret_cast<cudaEvent_t>(opts->cascade_events[1]);
  if (side) {
    if (cudaEventRecord(fork, stream) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess)
      return PA_ERR_CUDA;
    st = run_cascade(v, mk, mv, q, bt, k_scale, v_scale, *opts, sm_scale, err, sms, side);
    if (st != PA_OK) return st;
    if (cudaEventRecord(join, side) != cudaSuccess) return PA_ERR_CUDA;
  }
  st = dispatch_segments(v, heads, p, mk, mv, stream);
  if (st != PA_OK) return st;
  st = run_cascade(v, mk, mv, q, bt, k_scale, v_scale, *opts, sm_scale, err, 3 * sms, stream);
  if (st != PA_OK) return st;
  if (side && cudaStreamWaitEvent(stream, join, 0) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status run_decode_parts(const pa_shape &s, float *o_part, float *lse, int S, int workers,
                           const void *q, const void *k_pool, const void *v_pool,
                           const float *k_scale, const float *v_scale, const int32_t *bt,
                           const int32_t *sl, const pa_decode_opts *opts, float sm_scale,
                           int32_t *err, cudaStream_t stream) {
  const int heads = heads_per_unit(s, opts);
  const pa_shape v = unit_view(s, heads);
  CUtensorMap mk, mv;
  if (!make_pool_map(&mk, k_pool, v, heads) || !make_pool_map(&mv, v_pool, v, heads))
    return PA_ERR_CUDA;
  Params p = make_params(v, nullptr, q, k_scale, v_scale, bt, sl, opts, sm_scale, err);
  p.shared_prefix_lens = opts ? opts->shared_prefix_lens : nullptr;
  p.num_splits = workers;
  p.parts_S = S;
  p.parts_o = o_part;
  p.parts_lse = lse;
  return dispatch_segments(v, heads, p, mk, mv, stream);
}

pa_status run_merge_parts(const pa_shape &s, float *out, const float *o_part, const float *lse,
                          int S, cudaStream_t stream) {
  const int G = s.Hq / s.Hkv;   // <= 16: a CTA of at most 512 threads
  const dim3 grid(s.B * s.Hkv), block(32 * G);
  const cudaError_t e =
      s.D == 128 ? launch_pdl(merge_parts_kernel<128>, grid, block, 0, stream, out, o_part, lse, G, S)
                 : launch_pdl(merge_parts_kernel<64>, grid, block, 0, stream, out, o_part, lse, G, S);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status run_merge(const pa_shape &s, float *out, const void *workspace, int num_splits,
                    cudaStream_t stream) {
  const WorkspaceLayout w = splitkv_layout(s, num_splits);
  const uint8_t *ws = static_cast<const uint8_t *>(workspace);
  const int G = s.Hq / s.Hkv;
  // a CTA per (sequence, KV head); with thousands of them (large batches, where most
  // units finished inside one segment and exit at once) smaller CTAs keep more resident
  const int cap = s.B * s.Hkv >= 2048 ? 128 : 256;
  const int threads = min(cap, max(32, ((G * s.D / 4) + 31) / 32 * 32));
  return launch_pdl(merge_kernel, dim3(s.B * s.Hkv), dim3(threads), 0, stream, out,
                    reinterpret_cast<const int32_t *>(ws + w.prefix),
                    reinterpret_cast<const float *>(ws + w.o_part),
                    reinterpret_cast<const float *>(ws + w.lse), s.B, s.Hq, s.Hkv, G, s.D,
                    num_splits) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace pa
