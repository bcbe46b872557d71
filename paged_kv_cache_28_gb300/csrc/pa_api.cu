// pa_api.cu -- the extern "C" entry points declared in include/pa.h: host-side
// argument checks, then the launches in pa_cache.cu / pa_decode.cu.
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>

#include "pa.h"
#include "pa_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks common to every call.  need_q: Hq matters (decode).
pa_status check_shape(const pa_shape *s, bool need_q) {
  if (!s) return PA_ERR_INVALID_ARG;
  if (s->B < 0 || s->Hkv <= 0 || s->D <= 0 || s->block_size <= 0 || s->nblocks <= 0 ||
      s->max_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (s->Hkv > 2048) return PA_ERR_UNSUPPORTED;        // the decode packs the KV head in 11 bits
  if (s->kv_dtype != PA_KV_BF16 && s->kv_dtype != PA_KV_FP8_E4M3 && s->kv_dtype != PA_KV_INT4)
    return PA_ERR_INVALID_ARG;
  if (need_q) {
    if (s->Hq <= 0 || s->Hq % s->Hkv != 0) return PA_ERR_INVALID_ARG;
    if (s->Hq / s->Hkv > 16) return PA_ERR_UNSUPPORTED;
  }
  if (s->D != 64 && s->D != 128) return PA_ERR_UNSUPPORTED;
  if (s->block_size != 16 && s->block_size != 32) return PA_ERR_UNSUPPORTED;
  if (s->kv_dtype != PA_KV_BF16 && s->D != 128) return PA_ERR_UNSUPPORTED;
  // every row index and tile count below must fit in int32
  if (static_cast<int64_t>(s->nblocks) * s->block_size >= (int64_t(1) << 31))
    return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s->B) * s->max_blocks >= (int64_t(1) << 31)) return PA_ERR_INVALID_ARG;
  if (s->kv_dtype != PA_KV_BF16 && static_cast<int64_t>(s->nblocks) * s->Hkv >= (int64_t(1) << 31))
    return PA_ERR_INVALID_ARG;                          // scale indices
  const int64_t max_tiles = (static_cast<int64_t>(s->max_blocks) * s->block_size + 15) / 16;
  if (static_cast<int64_t>(s->B) * s->Hkv * max_tiles >= (int64_t(1) << 31))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

pa_status check_ptrs(std::initializer_list<const void *> ptrs) {
  for (const void *p : ptrs)
    if (!p || !aligned16(p)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

pa_status check_decode_args(const pa_shape *shape, const float *out, const void *q,
                            const void *k_pool, const void *v_pool, const float *k_scale,
                            const float *v_scale, const int32_t *bt, const int32_t *sl,
                            const pa_decode_opts *opts) {
  pa_status st = check_shape(shape, true);
  if (st != PA_OK) return st;
  st = check_ptrs({out, q, k_pool, v_pool, bt, sl});
  if (st != PA_OK) return st;
  if (shape->kv_dtype != PA_KV_BF16 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  if (opts) {
    if (opts->window < 0 || opts->topk < 0) return PA_ERR_INVALID_ARG;
    if (opts->shared_prefix_lens && !aligned16(opts->shared_prefix_lens)) return PA_ERR_INVALID_ARG;
    if ((opts->topk > 0) != (opts->selected_pages != nullptr)) return PA_ERR_INVALID_ARG;
    if (opts->selected_pages && !aligned16(opts->selected_pages)) return PA_ERR_INVALID_ARG;
    if (opts->topk > 0 && opts->window > 0) return PA_ERR_INVALID_ARG;
    if (opts->num_prefix_groups < 0) return PA_ERR_INVALID_ARG;
    if (opts->num_prefix_groups > 0) {              // cascade decode
      auto aligned4 = [](const void *q) { return q && (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
      if (!aligned4(opts->group_offsets) || !aligned4(opts->group_seqs) ||
          !aligned4(opts->group_prefix_len) || !opts->cascade_workspace ||
          (reinterpret_cast<uintptr_t>(opts->cascade_workspace) & 255u))
        return PA_ERR_INVALID_ARG;
      if (opts->window > 0 || opts->topk > 0) return PA_ERR_INVALID_ARG;
      if (opts->cascade_stream && (!opts->cascade_events[0] || !opts->cascade_events[1]))
        return PA_ERR_INVALID_ARG;
      if (opts->num_prefix_groups > pa::kMaxSplitBatch) return PA_ERR_UNSUPPORTED;
    }
  }
  return PA_OK;
}

constexpr int kMaxSplits = 65536;

// Split workers resident at once: CTAs per SM by shared memory (227 KB usable per SM,
// 1 KB reserved per CTA), capped by what the kernel's register budget was compiled
// for, times warps per CTA.
// Split workers resident at once for the split kernel a decode with these options
// (NULL: none) launches: a Quest selection or a cascade reads quantised heads singly.
int resident_segments(const pa_shape *shape, int sm_count, const pa_decode_opts *opts = nullptr) {
  const int per_cta = pa::splitkv_smem_bytes(*shape, opts) + 1024;
  const int warps = pa::decode_warps_per_cta();
  int ctas = (227 * 1024) / per_cta;
  if (ctas > pa::splitkv_min_blocks(*shape, opts)) ctas = pa::splitkv_min_blocks(*shape, opts);
  if (ctas < 1) ctas = 1;
  const int64_t n = static_cast<int64_t>(sm_count) * ctas * warps;
  return static_cast<int>(n > kMaxSplits ? kMaxSplits : n);
}

pa_status current_sm_count(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_reshape_and_cache(const pa_shape *shape, const void *k_new, const void *v_new,
                               void *k_pool, void *v_pool, float *k_scale, float *v_scale,
                               const int64_t *slot_mapping, int32_t *err_flag,
                               pa_stream_t stream) {
  pa_status st = check_shape(shape, false);
  if (st != PA_OK) return st;
  if (shape->B == 0) return PA_OK;
  st = check_ptrs({k_new, v_new, k_pool, v_pool, slot_mapping});
  if (st != PA_OK) return st;
  if (shape->kv_dtype != PA_KV_BF16 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  return pa::run_reshape_and_cache(*shape, k_new, v_new, k_pool, v_pool, k_scale, v_scale,
                                   slot_mapping, err_flag, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_decode(const pa_shape *shape, float *out, const void *q, const void *k_pool,
                    const void *v_pool, const float *k_scale, const float *v_scale,
                    const int32_t *block_tables, const int32_t *seq_lens,
                    const pa_decode_opts *opts, float sm_scale, int32_t *err_flag,
                    pa_stream_t stream) {
  if (!shape) return PA_ERR_INVALID_ARG;
  if (shape->B == 0) return check_shape(shape, true);
  pa_status st = check_decode_args(shape, out, q, k_pool, v_pool, k_scale, v_scale,
                                   block_tables, seq_lens, opts);
  if (st != PA_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (opts && opts->workspace) {                   // split decode + merge in one call
    int ns = opts->num_segments;
    if (ns <= 0) {
      int sms = 0;
      if (current_sm_count(&sms) != PA_OK) return PA_ERR_CUDA;
      ns = resident_segments(shape, sms);   // pa_default_num_segments: the caller sized for it
    }
    if (ns > kMaxSplits) return PA_ERR_INVALID_ARG;
    if (shape->B > pa::kMaxSplitBatch) return PA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(opts->workspace) & 255u) ||
        opts->workspace_bytes < pa::splitkv_layout(*shape, ns).total)
      return PA_ERR_INVALID_ARG;
    st = pa::run_decode_splitkv(*shape, out, opts->workspace, ns, q, k_pool, v_pool, k_scale,
                                v_scale, block_tables, seq_lens, opts, sm_scale, err_flag, cs);
    if (st != PA_OK) return st;
    return pa::run_merge(*shape, out, opts->workspace, ns, cs);
  }
  return pa::run_decode(*shape, out, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                        opts, sm_scale, err_flag, cs);
}

size_t pa_decode_workspace_bytes(const pa_shape *shape, int32_t num_segments) {
  if (check_shape(shape, true) != PA_OK || num_segments < 1 || num_segments > kMaxSplits)
    return 0;
  return pa::splitkv_layout(*shape, num_segments).total;
}

int32_t pa_default_num_segments(const pa_shape *shape, int32_t sm_count) {
  if (check_shape(shape, true) != PA_OK || sm_count <= 0) return 1;
  return resident_segments(shape, sm_count);
}

size_t pa_splitkv_workspace_bytes(const pa_shape *shape, int32_t num_splits) {
  if (check_shape(shape, true) != PA_OK || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return static_cast<size_t>(shape->B) * shape->Hq * num_splits * (shape->D + 1) * sizeof(float);
}

size_t pa_cascade_workspace_bytes(const pa_shape *shape) {
  if (check_shape(shape, true) != PA_OK) return 0;
  return pa::cascade_layout(shape->B, shape->Hq, shape->D).total;
}

int32_t pa_default_num_splits(const pa_shape *shape, int32_t sm_count) {
  if (check_shape(shape, true) != PA_OK || sm_count <= 0) return 1;
  // partial slots per query head: as many as 64 MiB of o_part holds, between 2 and 64,
  // and no more than a sequence has 16-token tiles
  const int64_t per_slot = static_cast<int64_t>(shape->B) * shape->Hq * shape->D * 4;
  const int64_t max_tiles = (static_cast<int64_t>(shape->max_blocks) * shape->block_size + 15) / 16;
  int64_t n = per_slot > 0 ? (int64_t(64) << 20) / per_slot : 64;
  if (n > 64) n = 64;
  if (n < 2) n = 2;
  if (n > max_tiles) n = max_tiles;
  return static_cast<int32_t>(n < 1 ? 1 : n);
}

pa_status pa_decode_splitkv(const pa_shape *shape, float *o_part, float *lse, int32_t num_splits,
                            const void *q, const void *k_pool, const void *v_pool,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_tables, const int32_t *seq_lens,
                            const pa_decode_opts *opts, float sm_scale, int32_t *err_flag,
                            pa_stream_t stream) {
  if (!shape) return PA_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > kMaxSplits) return PA_ERR_INVALID_ARG;
  if (shape->B == 0) return check_shape(shape, true);
  pa_status st = check_decode_args(shape, o_part, q, k_pool, v_pool, k_scale, v_scale,
                                   block_tables, seq_lens, opts);
  if (st != PA_OK) return st;
  st = check_ptrs({lse});
  if (st != PA_OK) return st;
  if (opts && opts->num_prefix_groups > 0) return PA_ERR_UNSUPPORTED;
  if (shape->B > pa::kMaxSplitBatch) return PA_ERR_UNSUPPORTED;
  int sms = 0;
  if (current_sm_count(&sms) != PA_OK) return PA_ERR_CUDA;
  return pa::run_decode_parts(*shape, o_part, lse, num_splits, resident_segments(shape, sms, opts), q,
                              k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens, opts,
                              sm_scale, err_flag, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_merge_lse(const pa_shape *shape, float *out, const float *o_part, const float *lse,
                       int32_t num_splits, pa_stream_t stream) {
  pa_status st = check_shape(shape, true);
  if (st != PA_OK) return st;
  if (num_splits < 1 || num_splits > kMaxSplits) return PA_ERR_INVALID_ARG;
  if (shape->B == 0) return PA_OK;
  st = check_ptrs({out, o_part, lse});
  if (st != PA_OK) return st;
  return pa::run_merge_parts(*shape, out, o_part, lse, num_splits,
                             reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_quest_summarize(const pa_shape *shape, const void *k_pool, const float *k_scale,
                             void *key_summaries, const int64_t *slot_mapping, int32_t *err_flag,
                             pa_stream_t stream) {
  pa_status st = check_shape(shape, false);
  if (st != PA_OK) return st;
  if (shape->B == 0) return PA_OK;
  st = check_ptrs({k_pool, key_summaries, slot_mapping});
  if (st != PA_OK) return st;
  if (shape->kv_dtype != PA_KV_BF16 && !k_scale) return PA_ERR_INVALID_ARG;
  return pa::run_quest_summarize(*shape, k_pool, k_scale, key_summaries, slot_mapping, err_flag,
                                 reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_quest_select(const pa_shape *shape, const void *q, const void *key_summaries,
                          const int32_t *block_tables, const int32_t *seq_lens, int32_t topk,
                          float *page_scores, int32_t *selected_pages, int32_t *err_flag,
                          pa_stream_t stream) {
  pa_status st = check_shape(shape, true);
  if (st != PA_OK) return st;
  if (topk < 1) return PA_ERR_INVALID_ARG;
  if (shape->B == 0) return PA_OK;
  st = check_ptrs({q, key_summaries, block_tables, seq_lens, page_scores, selected_pages});
  if (st != PA_OK) return st;
  if (pa::quest_topk_smem(*shape) > 200 * 1024 || pa::quest_score_smem(*shape) > 200 * 1024)
    return PA_ERR_UNSUPPORTED;
  // (sequence, KV head, page) units are counted in int32
  if (static_cast<int64_t>(shape->B) * shape->Hkv * pa::quest_max_pages(*shape) > INT32_MAX)
    return PA_ERR_UNSUPPORTED;
  return pa::run_quest_select(*shape, q, key_summaries, block_tables, seq_lens, topk,
                              page_scores, selected_pages, err_flag,
                              reinterpret_cast<cudaStream_t>(stream));
}

const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
  }
  return "PA_ERR_UNKNOWN";
}

pa_status pa_read_error_flag(const int32_t *err_flag, int32_t *host_value, pa_stream_t stream) {
  if (!err_flag || !host_value) return PA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(host_value, err_flag, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  return *host_value ? PA_ERR_DEVICE : PA_OK;
}

}  // extern "C"
