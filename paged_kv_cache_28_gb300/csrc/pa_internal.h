// pa_internal.h -- host-side interfaces between the C ABI (pa_api.cu) and the
// kernel files.  Arguments reaching these functions are already validated.
#pragma once

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
//   prefix  int32 [B + 1]        tile-count prefix over sequences (x Hkv)
//   lse     fp32  [num_splits][2][G]
//   o_part  fp32  [num_splits][2][G][D]
struct WorkspaceLayout {
  size_t prefix, lse, o_part, total;
};

// Largest batch the split-KV kernel accepts (its length scan lives in shared memory).
constexpr int kMaxSplitBatch = 16384;

WorkspaceLayout splitkv_layout(const pa_shape &s, int num_splits);
int splitkv_smem_bytes(const pa_shape &s);
int decode_warps_per_cta();
// CTAs per SM the split kernel is compiled for (registers capped accordingly).
int splitkv_min_blocks(const pa_shape &s);

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

pa_status run_quest_summarize(const pa_shape &s, const void *k_pool, void *summaries,
                              const int64_t *slot_mapping, int32_t *err, cudaStream_t stream);
int quest_max_pages(const pa_shape &s);
size_t quest_score_smem(const pa_shape &s);
size_t quest_topk_smem(const pa_shape &s);
pa_status run_quest_select(const pa_shape &s, const void *q, const void *summaries,
                           const int32_t *block_tables, const int32_t *seq_lens, int topk,
                           float *page_scores, int32_t *selected, int32_t *err,
                           cudaStream_t stream);

}  // namespace pa
