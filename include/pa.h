/*
 * pa.h -- C ABI of the paged-KV decode attention library (libpa.so, sm_103a).
 *
 * The library implements the data-parallel hot path of paged KV-cache LLM
 * decoding: the slot-mapped write of each step's new K/V into a block pool,
 * and single-token grouped-query attention over that pool through per-sequence
 * block tables.
 *
 * Sources of the operations (web pages the method is described on):
 *   [P1] "appendonly" (rajatmohan.com): "What is actually being cached"
 *        (K and V per token, 8 KV heads x 128 dims), "Paging, because contiguous
 *        allocation is a disaster" (fixed 16/32-token blocks, per-sequence block
 *        table, lazy allocation), "Prefix sharing is where the real win lives"
 *        (sequences point at the same physical blocks).
 *   [P3] "KV Cache Engineering for LLM Serving" (dailydoseofds): section 1
 *        (GQA: query head h reads KV head h / (Hq/Hkv)), section 8
 *        (absmax-scaled low-bit cache, restored = code * scale; FP8 cache),
 *        section 10 (PagedAttention block pool).
 *   [P4] "Taming the Token Torrent" (architects-blueprint): "How Paging Works in
 *        the LLM Context" (new tokens go to a block taken from a free pool),
 *        "The Block Table Logic" (logical index -> physical block + offset),
 *        "Custom PagedAttention Kernels" (grid over (sequence, head), walk the
 *        block table, stage each block in shared memory, attend, move on),
 *        "The Metadata Bottleneck" (block tables live on the GPU).
 * Split-KV with a log-sum-exp merge is not on the pages; it is the standard
 * flash-decoding extension, defined below by what it computes.
 *
 * ---------------------------------------------------------------------------
 * Conventions common to every entry point
 * ---------------------------------------------------------------------------
 *  - All array arguments are caller-owned DEVICE memory of the current CUDA
 *    device, row-major, 16-byte aligned.  The library allocates nothing, frees
 *    nothing and keeps no state between calls (pa_decode_splitkv_noalloc, at
 *    the end, is the one call with a library-owned scratch array).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and is asynchronous: no call synchronises.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and launches
 *    nothing.  A failed launch returns PA_ERR_CUDA.
 *  - Errors that depend on device data (a block id outside the pool, a
 *    sequence longer than its block table, a slot outside the pool, two
 *    quantised writes into one slot) are reported through `err_flag`: a device int32
 *    that the kernels OR a PA_DEVERR_* bit into.  The affected unit is skipped
 *    (or reads zeros), nothing traps.  The flag is sticky; the caller zeroes it
 *    and reads it after synchronising (see pa_read_error_flag).  err_flag may
 *    be NULL only if the caller vouches that the data is valid.
 *  - Cached values must be finite in the rows a decode attends.  A NaN or Inf there
 *    gives an undefined output (NaN, or a value that leaves those tokens out).  Rows
 *    it does not attend -- past a sequence's length, before a window -- may hold
 *    anything.
 *  - Shapes: B sequences (or tokens, for the cache write), Hq query heads,
 *    Hkv <= 2048 KV heads (Hq % Hkv == 0, G = Hq / Hkv <= 16), head dim D in {64, 128},
 *    block_size in {16, 32}.  FP8 and 4-bit pools need D = 128.  Indices stay in
 *    int32: nblocks * block_size, B * max_blocks, B * Hkv * ceil(max_blocks *
 *    block_size / 16) and, for code pools, nblocks * Hkv must be below 2^31
 *    (else PA_ERR_INVALID_ARG).
 *  - Layouts:
 *      q            [B, Hq, D]                  bf16
 *      out          [B, Hq, D]                  fp32
 *      k/v pool     [nblocks, block_size, Hkv, D] bf16, or E4M3 codes (uint8),
 *                   or [nblocks, block_size, Hkv, D/2] packed 4-bit codes
 *      k/v scale    [nblocks, Hkv]              fp32 (code pools only, else NULL)
 *      block_tables [B, max_blocks]             int32 physical block ids
 *      seq_lens     [B]                         int32 tokens in the cache,
 *                                               including this step's token
 *      slot_mapping [B]                         int64 slot = block * block_size
 *                                               + offset; negative = skip
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pa_stream_t;   /* same type as cudaStream_t */
typedef struct CUevent_st *pa_event_t;     /* same type as cudaEvent_t */

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or workspace */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not built: D, block_size, G, dtype */
    PA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or launch failed */
    PA_ERR_DEVICE = 4         /* pa_read_error_flag found a PA_DEVERR_* bit */
} pa_status;

/* Cached element formats.  PA_KV_INT4: signed 4-bit codes in [-7, 7] stored as
 * offset-binary nibbles (code + 8), two per byte -- element 2j in the low nibble of
 * byte j -- so a pool row is D / 2 bytes. */
typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1, PA_KV_INT4 = 2 } pa_kv_dtype;

/* Device error bits ORed into *err_flag (PA_DEVERR_FP8_CONFLICT also covers 4-bit
 * pools: two tokens of one write call with the same slot). */
#define PA_DEVERR_BLOCK_ID     1   /* block table entry outside [0, nblocks)        */
#define PA_DEVERR_SEQ_LEN      2   /* seq_len < 0 or > max_blocks * block_size      */
#define PA_DEVERR_SLOT         4   /* slot_mapping entry >= nblocks * block_size    */
#define PA_DEVERR_FP8_CONFLICT 8   /* two tokens of one FP8/4-bit write, one slot    */
#define PA_DEVERR_TIMEOUT      16  /* an internal pipeline wait gave up             */

typedef struct {
    int32_t B;            /* sequences (decode) or tokens to write (cache write) */
    int32_t Hq;           /* query heads */
    int32_t Hkv;          /* KV heads */
    int32_t D;            /* head dimension */
    int32_t block_size;   /* tokens per physical block */
    int32_t nblocks;      /* physical blocks in each pool */
    int32_t max_blocks;   /* columns of block_tables */
    int32_t kv_dtype;     /* pa_kv_dtype */
} pa_shape;

/*
 * Optional settings of a decode call (pass NULL for the defaults).
 *   window: > 0 attends over the last `window` positions of each sequence only,
 *     [max(0, L - window), L) -- a sliding-window layer ("KV Cache Engineering
 *     for LLM Serving", section 3).  Block-table entries of blocks wholly before
 *     the window are never read (they may be freed and hold any value).  0 = all.
 *   topk, selected_pages: query-aware sparse decode (section 7, Quest): with
 *     topk > 0, (sequence b, KV head h) attends only over the 16-token pages
 *     selected_pages[b][h][0 .. min(topk, pages of b)) -- logical page indices in
 *     increasing order, as pa_quest_select writes them (page j = tokens
 *     [16 j, min(16 j + 16, L))).  An index outside the sequence sets
 *     PA_DEVERR_BLOCK_ID and reads zeros.  Not combined with window.
 *   shared_prefix_lens: pa_decode (with or without a workspace).  Optional [B]
 *     int32 device array, a speed hint for batches with prefix sharing
 *     ("appendonly", "Prefix sharing is where the real win lives"): the number
 *     of leading tokens of sequence b that lie in blocks other sequences of the
 *     batch also reference.  Whole 16-token tiles inside that prefix are
 *     fetched with an L2 evict-last policy, all other tiles evict-first, so a
 *     shared block stays in L2 for its other readers.  Any value gives the same
 *     result, bit for bit.
 *   num_prefix_groups, group_offsets, group_seqs, group_prefix_len,
 *     cascade_workspace: prefix-aware (cascade) decode, in pa_decode given a
 *     workspace (pa_decode without one ignores them and attends over every
 *     token itself) ("appendonly", "Prefix sharing is where the real win lives":
 *     many sequences point at the same physical blocks).  Group g's members are
 *     group_seqs[group_offsets[g] .. group_offsets[g + 1]) (device int32
 *     arrays; group_offsets rises from 0, at most B members in all); their first
 *     group_prefix_len[g] tokens (device int32, a multiple of 16) hold the same
 *     keys and values, as when their block tables share those blocks.  A
 *     separate kernel attends over each group's shared tokens once for all
 *     members and KV heads at a time (the members' query rows stacked into one
 *     tensor-core contraction, reading the blocks through the first member's
 *     table); the split kernel covers the rest of each sequence and the merge
 *     joins the two.  Each sequence belongs to at most one group and every
 *     member holds at least group_prefix_len[g] tokens (a member with fewer sets
 *     PA_DEVERR_SEQ_LEN and its output is undefined).  cascade_workspace:
 *     device memory of at least pa_cascade_workspace_bytes bytes, 256-byte
 *     aligned.  Every pool kind: FP8-E4M3 and 4-bit codes are restored with
 *     their block scales as in the decode (a cascade decode on 4-bit pools reads
 *     the KV heads one at a time, not in pairs).  Not combined with window or
 *     topk.  The result equals the plain decode's up to rounding order.
 *   cascade_stream, cascade_events: where the cascade kernel runs.  NULL: on
 *     `stream`, after the split kernel.  Otherwise a caller-owned stream of the
 *     same device, on which the cascade kernel runs beside the split kernel (it
 *     does tensor work while the split kernel streams HBM), joined back before
 *     the merge: the call records cascade_events[0] on `stream`, makes
 *     cascade_stream wait for it, launches there, records cascade_events[1] on
 *     cascade_stream and makes `stream` wait for it.  The two events are
 *     caller-created (cudaEventDisableTiming is enough) and may be reused by the
 *     next call on the same streams.  The results are the same either way.
 *   workspace, workspace_bytes, num_segments: pa_decode only.  With a workspace
 *     (device memory of at least pa_decode_workspace_bytes(shape, n) bytes,
 *     256-byte aligned; n = num_segments, or pa_default_num_segments for this
 *     GPU when num_segments is 0) pa_decode runs the load-balanced split decode
 *     and the merge itself: the 16-token tiles of all (sequence, KV head) units,
 *     laid end to end, are cut into n equal segments, one per split worker; a
 *     unit inside one segment is finished there, a unit cut by segment bounds
 *     leaves one partial per piece in the workspace for the merge.  Without a
 *     workspace it needs no memory: one CTA per (sequence, KV head) unit, or,
 *     when the batch has at most two units per CTA the GPU holds at once, a
 *     cluster of four CTAs per unit that share its tiles (at least 16 per warp;
 *     a short unit leaves the extra CTAs idle) and merge through distributed
 *     shared memory; a window or topk that bounds every unit keeps one CTA per
 *     unit when the units fill the GPU or fit one CTA.  Batches of up to 16384
 *     sequences start their longest sequences first.  A bf16 batch of up to 8
 *     query heads per KV head with more units than two per CTA the GPU holds at
 *     once (and at most 4096), and no window or topk, runs one persistent CTA per
 *     SM instead: every CTA computes the same static schedule from seq_lens
 *     (whole units dealt out longest first so that each CTA gets about the mean
 *     number of tiles), cuts its tiles into one contiguous segment per warp, and
 *     joins units that cross segments in shared memory.  A batch whose longest
 *     sequence outweighs the rest is still held back by it; the split decode is
 *     not.  Every form gives the same result on every call, bit for bit.
 */
typedef struct {
    int32_t window;
    int32_t topk;
    const int32_t *shared_prefix_lens;
    const int32_t *selected_pages;      /* [B, Hkv, topk] int32, with topk > 0 */
    int32_t num_prefix_groups;          /* 0: no cascade */
    const int32_t *group_offsets;       /* [num_prefix_groups + 1] */
    const int32_t *group_seqs;          /* [group_offsets[num_prefix_groups]] */
    const int32_t *group_prefix_len;    /* [num_prefix_groups] */
    void *cascade_workspace;
    void *workspace;                    /* pa_decode: split workspace, or NULL */
    size_t workspace_bytes;
    int32_t num_segments;               /* pa_decode with a workspace; 0: default */
    pa_stream_t cascade_stream;         /* NULL: the cascade runs after the split kernel */
    pa_event_t cascade_events[2];       /* fork, join (with cascade_stream) */
} pa_decode_opts;

/*
 * pa_reshape_and_cache -- write this step's K/V into the block pools.
 * [P4] "How Paging Works in the LLM Context" and "The Block Table Logic";
 * [P1] "Paging".  For every token t < shape->B with s = slot_mapping[t] >= 0
 * and every KV head h:
 *     pool[s / block_size][s % block_size][h][:] = new[t][h][:]
 * k_new, v_new: [B, Hkv, D] bf16.  shape->Hq is ignored.
 *
 * BF16 pools: a bit-exact copy.  Two tokens with the same slot race (one wins).
 *
 * FP8 pools (kv_dtype = PA_KV_FP8_E4M3, k_scale/v_scale required), after
 * [P3] section 8, per (block, kv head) and separately for K and V:
 *   - scale = absmax of every value written into the (block, head) since its
 *     offset 0 was written, / 448 (fp32 IEEE division); writing offset 0
 *     starts a new scale;
 *   - code = E4M3(x / scale): fp32 IEEE division, round to nearest even,
 *     saturating to +-448; a zero scale stores +0 codes;
 *   - a write that raises the scale re-encodes the codes at offsets below it:
 *     code' = E4M3((E4M3 value of code * old scale) / new scale), fp32 product
 *     and division.
 *   Tokens of one call that land in the same block (a prompt, several appended
 *   tokens) are applied one after the other in token order, exactly as separate
 *   calls would apply them.  Two tokens of one call with the same slot are both
 *   applied, the later one last, and set PA_DEVERR_FP8_CONFLICT.
 * A slot beyond the pool sets PA_DEVERR_SLOT and is skipped.
 */
pa_status pa_reshape_and_cache(const pa_shape *shape, const void *k_new, const void *v_new,
                               void *k_pool, void *v_pool, float *k_scale, float *v_scale,
                               const int64_t *slot_mapping, int32_t *err_flag,
                               pa_stream_t stream);

/*
 * 4-bit pools (kv_dtype = PA_KV_INT4, D = 128) are written the same way with
 * largest code 7 ("KV Cache Engineering for LLM Serving", section 8, bits = 4):
 *   scale = absmax since offset 0 / 7 (fp32 division); code = clip(rint(x /
 *   scale), -7, 7) (fp32 division, ties to even); a growing scale re-encodes the
 *   earlier rows from code * old scale (fp32 product); a zero scale stores 0.
 */

/*
 * pa_decode -- single-token decode attention over the paged cache: one CTA (or,
 * for batches of few units, a cluster of CTAs) per (sequence, KV head) serving
 * the whole query group, persistent CTAs for bf16 batches of many units, or,
 * with a workspace in opts, the split decode and the merge in one call.
 * [P4] "Custom PagedAttention Kernels" (grid over sequence and head, block-table
 * walk, block staged in shared memory); [P3] section 1 (GQA grouping).
 *     out[b][h][:] = sum_t softmax_t(sm_scale * <q[b][h], K_b[t]>) V_b[t]
 * over t < seq_lens[b], where K_b[t] = k_pool[block_tables[b][t / bs]][t % bs]
 * [h / G] (same for V) and FP8 / 4-bit codes are restored as value *
 * scale[block][kvh].
 * seq_lens[b] = 0 gives zeros.  out is fp32 [B, Hq, D].  opts: see pa_decode_opts.
 */
pa_status pa_decode(const pa_shape *shape, float *out, const void *q, const void *k_pool,
                    const void *v_pool, const float *k_scale, const float *v_scale,
                    const int32_t *block_tables, const int32_t *seq_lens,
                    const pa_decode_opts *opts, float sm_scale, int32_t *err_flag,
                    pa_stream_t stream);

/*
 * Bytes of the optional split workspace of pa_decode (pa_decode_opts.workspace)
 * for this shape and num_segments; 0 if the arguments are invalid.  Host only.
 */
size_t pa_decode_workspace_bytes(const pa_shape *shape, int32_t num_segments);

/*
 * The number of segments pa_decode's split decode uses when num_segments is 0: the
 * split workers a GPU with sm_count SMs keeps resident at once.  Host only, no CUDA
 * call.
 */
int32_t pa_default_num_segments(const pa_shape *shape, int32_t sm_count);

/*
 * Bytes of device workspace a cascade decode (pa_decode_opts.num_prefix_groups
 * > 0) needs for this shape, besides the split workspace; 0 if the shape is
 * invalid.  Host only.
 */
size_t pa_cascade_workspace_bytes(const pa_shape *shape);

/*
 * Split-KV decode with caller-visible partials (flash-decoding), and the
 * log-sum-exp merge of such partials.  Not on the pages: the standard extension
 * of their per-(sequence, head) attention ("Taming the Token Torrent", "Custom
 * PagedAttention Kernels") to several workers per sequence.
 *
 * Partials of query head h of sequence b, S = num_splits slots:
 *     o_part [B, Hq, S, D] fp32   o_part[b][h][i][:] = sum_t e^(s_t - m_i) V_t / l_i
 *     lse    [B, Hq, S]    fp32   lse[b][h][i]       = m_i + ln l_i (natural log)
 * over the tokens t of piece i (s_t = sm_scale <q[b][h], K_b[t]>, m_i their
 * largest score, l_i = sum_t e^(s_t - m_i)).  An empty slot has lse = -inf and
 * its o_part row is not read (it may hold anything).  Merging every slot gives
 * the attention of pa_decode.
 */

/*
 * Bytes of o_part and lse together for num_splits slots, B * Hq * num_splits *
 * (D + 1) * 4 (o_part first, then lse, when both come from one allocation);
 * 0 if the arguments are invalid.  Host only.
 */
size_t pa_splitkv_workspace_bytes(const pa_shape *shape, int32_t num_splits);

/*
 * A num_splits for pa_decode_splitkv: the most slots (2 to 64) whose o_part fits
 * in 64 MiB, and no more than a sequence of max_blocks blocks has 16-token
 * tiles.  Host only, no CUDA call; sm_count is checked (> 0) but a GPU's size does
 * not change the slots a sequence needs.
 */
int32_t pa_default_num_splits(const pa_shape *shape, int32_t sm_count);

/*
 * pa_decode_splitkv -- write the partials of every query head (layout above),
 * 1 <= num_splits <= 65536.  How the tokens are cut: the 16-token tiles of all
 * (sequence, KV head) units, in (b, kvh, position) order, are laid end to end
 * and cut into equal segments of W tiles, one per split worker (the workers this
 * GPU keeps resident), W = max(ceil(total / workers), ceil((n_max - 1) /
 * (S - 1))) with n_max the tiles of the longest unit: the second bound keeps
 * every unit within S pieces (a unit of n tiles spans at most ceil((n - 1) / W)
 * + 1 segments).  Piece i of a unit is its part in the i-th segment that holds
 * it; slots after its last piece, and all slots of a sequence with seq_len 0,
 * get lse = -inf.  With S = 1 a segment's bounds move up to the next unit start,
 * so every unit is one piece.  4-bit and FP8-E4M3 pools with an even number of KV
 * heads and 8 query heads per KV head are read two adjacent KV heads at a time (a unit
 * is then (b, KV heads 2u, 2u + 1)) unless opts selects Quest pages; the result does
 * not depend on it.  opts (may be NULL): window, topk + selected_pages and
 * shared_prefix_lens as for pa_decode, the cut then running over the attended tiles
 * only; the workspace fields are ignored, and a cascade (num_prefix_groups > 0)
 * returns PA_ERR_UNSUPPORTED (its shared-prefix partials are merged by pa_decode's
 * own merge).
 * All arrays are caller-owned device memory; o_part and lse are outputs,
 * nothing in them needs initialising.  Batches of more than 16384 sequences
 * return PA_ERR_UNSUPPORTED (each CTA scans the lengths in shared memory).
 */
pa_status pa_decode_splitkv(const pa_shape *shape, float *o_part, float *lse, int32_t num_splits,
                            const void *q, const void *k_pool, const void *v_pool,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_tables, const int32_t *seq_lens,
                            const pa_decode_opts *opts, float sm_scale, int32_t *err_flag,
                            pa_stream_t stream);

/*
 * pa_merge_lse -- per query head (b, h), over the slots i < num_splits of
 * o_part [B, Hq, S, D] and lse [B, Hq, S] (fp32, caller-owned, from
 * pa_decode_splitkv or from anywhere else, e.g. partials of a prefix attended
 * elsewhere; lse = -inf marks an empty slot):
 *     M = max_i lse_i,  w_i = e^(lse_i - M),  out = sum_i w_i o_i / sum_i w_i
 * A head with every slot empty gets zeros.  out [B, Hq, D] fp32.
 */
pa_status pa_merge_lse(const pa_shape *shape, float *out, const float *o_part, const float *lse,
                       int32_t num_splits, pa_stream_t stream);

/*
 * pa_decode_splitkv_noalloc -- pa_decode's load-balanced split decode and merge
 * (pa_decode with opts.workspace and opts.num_segments = num_segments, no other
 * option), for callers that cannot allocate device memory.  The pages describe no
 * such call; it exists for users of this library who may not call cudaMalloc: a
 * plugin inside a host framework that owns all device memory through its own
 * pool, a latency-critical path where cudaMalloc's implicit device-wide
 * synchronisation is not acceptable, or a deployment whose memory budget is
 * fixed at start-up.
 *
 * Instead of a caller workspace it uses a scratch array of
 * PA_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library: every GPU that
 * loads libpa.so holds that array until the process exits.  The call allocates
 * nothing and frees nothing.  out [B, Hq, D] is complete when the work enqueued
 * on `stream` has finished.
 *
 * Limits and sharing:
 *   - returns PA_ERR_INVALID_ARG (launching nothing) when
 *     pa_decode_workspace_bytes(shape, num_segments) exceeds
 *     PA_NOALLOC_SCRATCH_BYTES, or for any argument pa_decode rejects;
 *   - num_segments = 0 takes pa_default_num_segments for the current GPU;
 *   - the array's device address is looked up (cudaGetSymbolAddress, on the
 *     current device) by every call made while `stream` is not being captured,
 *     so it stays right after cudaDeviceReset; a call made during stream capture
 *     reuses the address the last call on that device found, so make one call on
 *     each device before capturing;
 *   - all calls share the one array per device and it keeps the last call's
 *     contents (nothing in it needs to start at zero); calls whose work
 *     overlaps on the GPU -- on different streams, or from different threads --
 *     race on it and must be serialised by the caller.
 */
#define PA_NOALLOC_SCRATCH_BYTES (64u << 20)

pa_status pa_decode_splitkv_noalloc(const pa_shape *shape, float *out, int32_t num_segments,
                                    const void *q, const void *k_pool, const void *v_pool,
                                    const float *k_scale, const float *v_scale,
                                    const int32_t *block_tables, const int32_t *seq_lens,
                                    float sm_scale, int32_t *err_flag, pa_stream_t stream);

/*
 * Quest page summaries ("KV Cache Engineering for LLM Serving", section 7).  A page
 * is a 16-token tile of the pool: page g holds pool rows [16 g, 16 g + 16), i.e.
 * slots 16 g .. 16 g + 15 (a 32-token block is two pages).
 *
 * pa_quest_summarize -- for every token t < shape->B with slot s = slot_mapping[t]
 * >= 0, set the summary of page s / 16 to the per-channel minimum and maximum of its
 * keys in rows 0 .. s % 16:
 *     key_summaries[s / 16][h][0][d] = min_r K[r][h][d],  [1][d] = max_r K[r][h][d]
 * key_summaries: [nblocks * block_size / 16, Hkv, 2, D] bf16.  bf16 pools: exact.
 * FP8-E4M3 and 4-bit pools (section 8): K is the restored key code * k_scale[block]
 * [h] (k_scale [nblocks, Hkv] fp32, required), which bf16 may not hold, so the
 * minimum is stored rounded toward -inf and the maximum toward +inf: the page score
 * stays an upper bound of q . k (k_scale is ignored for bf16 pools).
 * Call it after pa_reshape_and_cache with the same slots; to build every summary
 * of a sequence, pass the slot of each page's last token.  When several listed
 * slots share a page the one with the largest slot writes.
 */
pa_status pa_quest_summarize(const pa_shape *shape, const void *k_pool, const float *k_scale,
                             void *key_summaries, const int64_t *slot_mapping, int32_t *err_flag,
                             pa_stream_t stream);

/*
 * pa_quest_select -- Quest's two steps for every (sequence b, KV head h): score
 * each 16-token page j of b (pages 0 .. ceil(L/16) - 1, reached through
 * block_tables) with every query head g of the group as
 *     sum_d max(q[b][g][d] * min_d, q[b][g][d] * max_d)      (fp32)
 * keep the page's largest score over the group in
 *     page_scores[b][h][j],  page_scores: [B, Hkv, P] fp32, P = ceil(max_blocks *
 *     block_size / 16), entries j >= pages of b left untouched,
 * then write the topk best pages (ties to the lower page index; all pages if
 * there are at most topk) in increasing order to selected_pages[b][h][0 .. topk),
 * -1 past the number of pages.  A page whose block-table entry is outside
 * [0, nblocks) sets PA_DEVERR_BLOCK_ID and scores -inf.  Any pool dtype (the
 * summaries are bf16); q [B, Hq, D] bf16; page_scores and selected_pages are
 * caller-owned device memory (outputs).  Pass selected_pages to pa_decode /
 * pa_decode_splitkv through pa_decode_opts.  Scores are fp32 sums, so pages whose
 * scores agree to rounding may be ordered differently from an exact computation.
 */
pa_status pa_quest_select(const pa_shape *shape, const void *q, const void *key_summaries,
                          const int32_t *block_tables, const int32_t *seq_lens, int32_t topk,
                          float *page_scores, int32_t *selected_pages, int32_t *err_flag,
                          pa_stream_t stream);

/* Human-readable name of a status. */
const char *pa_status_string(pa_status status);

/*
 * Synchronise `stream`, copy the device int32 *err_flag to *host_value and
 * return PA_ERR_DEVICE if it is nonzero, PA_OK otherwise.
 */
pa_status pa_read_error_flag(const int32_t *err_flag, int32_t *host_value, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
