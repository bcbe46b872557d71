// pa_internal.h -- host-side interfaces between the C ABI (pa_api.cu) and the
// kernel files.  Arguments reaching these functions are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "pa.h"

namespace pa {

// Launch `kernel` on `stream` so that it may start before the previous kernel in the
// stream has finished (programmatic dependent launch); every kernel launched this
// way calls pdl_wait() before it reads or writes memory an earlier kernel may use.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Byte offsets of the split-KV workspace regions (each 256-byte aligned):
//   prefix  int32 [B + 4]        tile-count prefix over sequences (x units), then KV
//                                heads per unit, then the cascade workspace address
//                                (two halves, 0 without a cascade)
//   lse     fp32  [num_splits][2][Gu]
//   o_part  fp32  [num_splits][2][Gu][D]
struct WorkspaceLayout {
  size_t prefix, lse, o_part, total;
};

// Shared-prefix pieces per cascade member: a group's shared tiles are cut into at
// most this many pieces so that long prefixes spread over several CTAs.
constexpr int kCascadePieces = 4;

// Byte offsets of the cascade workspace regions (each 256-byte aligned); m is the
// position of a sequence in the groups' member list (at most B members):
//   member int32 [B]   position of sequence b in the member list, or -1
//   tiles  int32 [B]   shared 16-token tiles of sequence b served by the cascade
//   pieces int32 [B]   cascade pieces of sequence b
//   lse    fp32  [B][Hkv][kCascadePieces][G]       indexed by m
//   o      fp32  [B][Hkv][kCascadePieces][G][D]
//   ulse   fp32  [B][Hq]      (o, lse) of a cascaded (sequence, KV head) whose rest
//   uo     fp32  [B][Hq][D]   lies inside one split segment (the split kernel's part)
//   next   int32              next cascade work item to take (reset by the plan)
struct CascadeLayout {
  size_t member, tiles, pieces, lse, o, ulse, uo, next, total;
};

__host__ __device__ inline CascadeLayout cascade_layout(int B, int Hq, int D) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  CascadeLayout c{};
  const size_t b = static_cast<size_t>(B);
  c.member = 0;
  c.tiles = up(b * 4);
  c.pieces = c.tiles + up(b * 4);
  c.lse = c.pieces + up(b * 4);
  c.o = c.lse + up(b * Hq * kCascadePieces * 4);
  c.ulse = c.o + up(b * Hq * kCascadePieces * static_cast<size_t>(D) * 4);
  c.uo = c.ulse + up(b * Hq * 4);
  c.next = c.uo + up(b * Hq * static_cast<size_t>(D) * 4);
  c.total = c.next + 256;
  return c;
}

// 2D TMA map of a pool for the decode's view of the shape (Hkv counts units of
// `heads` adjacent KV heads): 16-token boxes of up to 128 bytes per unit row.
bool make_pool_map(CUtensorMap *map, const void *pool, const pa_shape &s, int heads);

// Cascade (shared-prefix) part of a split decode; arguments validated.  The plan
// kernel writes the per-sequence cascade info and resets the work counter
// (programmatic dependent launch on the caller's stream); each cascade launch (`ctas`
// CTAs, a plain launch after the plan) takes work items from the counter until
// none are left, so several launches share the work.
pa_status run_cascade_plan(const pa_shape &s, const pa_decode_opts &opts, int32_t *err,
                           cudaStream_t stream);
pa_status run_cascade(const pa_shape &s, const CUtensorMap &mk, const CUtensorMap &mv,
                      const void *q, const int32_t *bt, const float *k_scale,
                      const float *v_scale, const pa_decode_opts &opts, float sm_scale,
                      int32_t *err, int ctas, cudaStream_t stream);

// Largest batch the split-KV kernel accepts (its length scan lives in shared memory).
constexpr int kMaxSplitBatch = 16384;

WorkspaceLayout splitkv_layout(const pa_shape &s, int num_splits);
int splitkv_smem_bytes(const pa_shape &s, const pa_decode_opts *opts = nullptr);
int decode_warps_per_cta();
// CTAs per SM the split kernel is compiled for (registers capped accordingly).
int splitkv_min_blocks(const pa_shape &s, const pa_decode_opts *opts = nullptr);

pa_status run_reshape_and_cache(const pa_shape &s, const void *k_new, const void *v_new,
                                void *k_pool, void *v_pool, float *k_scale, float *v_scale,
                                const int64_t *slot_mapping, int32_t *err, cudaStream_t stream);

pa_status run_decode(const pa_shape &s, float *out, const void *q, const void *k_pool,
                     const void *v_pool, const float *k_scale, const float *v_scale,
                     const int32_t *bt, const int32_t *sl, const pa_decode_opts *opts,
                     float sm_scale, int32_t *err, cudaStream_t stream);

pa_status run_decode_splitkv(const pa_shape &s, float *out, void *workspace, int num_splits,
                             const void *q, const void *k_pool, const void *v_pool,
                             const float *k_scale, const float *v_scale, const int32_t *bt,
                             const int32_t *sl, const pa_decode_opts *opts, float sm_scale,
                             int32_t *err, cudaStream_t stream);

pa_status run_merge(const pa_shape &s, float *out, const void *workspace, int num_splits,
                    cudaStream_t stream);

// pa_decode_splitkv / pa_merge_lse: the split kernel over `workers` segments with every
// piece written to caller arrays o_part [B, Hq, S, D] / lse [B, Hq, S], and their merge.
pa_status run_decode_parts(const pa_shape &s, float *o_part, float *lse, int S, int workers,
                           const void *q, const void *k_pool, const void *v_pool,
                           const float *k_scale, const float *v_scale, const int32_t *bt,
                           const int32_t *sl, const pa_decode_opts *opts, float sm_scale,
                           int32_t *err, cudaStream_t stream);
pa_status run_merge_parts(const pa_shape &s, float *out, const float *o_part, const float *lse,
                          int S, cudaStream_t stream);

pa_status run_quest_summarize(const pa_shape &s, const void *k_pool, const float *k_scale,
                              void *summaries,
                              const int64_t *slot_mapping, int32_t *err, cudaStream_t stream);
int quest_max_pages(const pa_shape &s);
size_t quest_score_smem(const pa_shape &s);
size_t quest_topk_smem(const pa_shape &s);
pa_status run_quest_select(const pa_shape &s, const void *q, const void *summaries,
                           const int32_t *block_tables, const int32_t *seq_lens, int topk,
                           float *page_scores, int32_t *selected, int32_t *err,
                           cudaStream_t stream);

}  // namespace pa
