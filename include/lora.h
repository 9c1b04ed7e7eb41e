/*
 * rank_adapter_gb300 -- C ABI of the batched multi-LoRA delta on sm_103a.
 *
 * What the library computes (row-vector orientation of the handbook page
 * "多 LoRA 服务：分段矩阵乘与适配器调度", section "不合并权重，批量计算"):
 *
 *     y[t] += scale[a] * (x[t] . A[a]) . B[a]      a = token_slot[t] != 0
 *
 * over a stacked GPU slot table of adapters; slot 0 means "no LoRA" and its
 * rows of y are never touched. The delta is split into a shrink (x -> rank r,
 * fp32 buffer) and an expand (buffer -> packed output slices, added into the
 * caller's base-layer output), as in section "两个低秩 GEMM:shrink、expand 与
 * fp32 中转缓冲" of the page "vLLM 源码完全拆解(十八): 多 LoRA 服务".
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Ownership: the caller owns every buffer (allocated with torch or
 *   cudaMalloc). The library allocates no device memory, keeps no pointer
 *   after a call returns, and holds no state between calls.
 * - Pointers named "device" must be device-accessible; all buffers must be
 *   16-byte aligned, and leading dimensions (ldx, ldy) times the element size
 *   must be multiples of 16 bytes.
 * - Every call is asynchronous on `stream` (NULL = the legacy default
 *   stream) and returns a lora_status. Argument errors are found on the host,
 *   before anything is launched. LORA_ECUDA means a launch failed;
 *   lora_last_cuda_error() returns the CUDA error code.
 * - Device-side conditions never trap or hang: a token slot id outside
 *   [0, num_slots) is treated as slot 0 and counted in meta->status
 *   (read it with lora_query_status).
 * - Kernels are launched with programmatic dependent launch: a kernel may
 *   start while the previous kernel on the stream drains, and reads the slot
 *   table (A, B, slot_rank, slot_scale) before waiting for it. Write the
 *   table through lora_set_slot / lora_reset_slot (they end with a launch
 *   that waits for the write to be visible); a table written any other way
 *   needs one more kernel, an event wait or a copy between the write and the
 *   next call of this library. lora_prepare_meta likewise reads
 *   meta->token_slot before waiting (it sorts while the previous kernel
 *   drains and writes its outputs after the wait): write token_slot with a
 *   copy, or with a kernel that has written it before it triggers its
 *   dependents (any kernel launched without programmatic dependent launch).
 * - Grid sizes depend only on host-known bounds (num_tokens, num_slots,
 *   shapes), never on device data, so a sequence of calls can be captured in
 *   a CUDA graph once it has run eagerly once.
 */
#ifndef RANK_ADAPTER_GB300_LORA_H
#define RANK_ADAPTER_GB300_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *lora_stream_t;

typedef enum {
  LORA_OK = 0,
  LORA_EINVAL = 1,        /* bad argument: null pointer, bad shape, mismatched sizes */
  LORA_ERANGE = 2,        /* a value outside its range: slot, rank, num_slots, num_tokens */
  LORA_EALIGN = 3,        /* a pointer or leading dimension is not 16-byte aligned */
  LORA_EUNSUPPORTED = 4,  /* valid but not implemented (e.g. SGMV on fp32 tables) */
  LORA_ECUDA = 5,         /* a CUDA launch or copy failed; see lora_last_cuda_error() */
  LORA_EBADSLOT = 6,      /* lora_query_status: some token slot ids were out of range */
  LORA_EDEVICE = 7,       /* lora_query_status: a kernel gave up waiting on its own pipeline
                             (a fault it avoided); outputs since lora_prepare_meta are invalid */
  LORA_EBADTOKEN = 8      /* lora_query_status: lora_embed_shrink met token ids outside the
                             vocabulary; those rows got no delta, the rest are valid */
} lora_status;

typedef enum { LORA_F32 = 0, LORA_BF16 = 1 } lora_dtype;

/* Which kernel family runs a shrink / expand.
 * BGMV: per-segment streaming of each adapter's A/B on CUDA cores (decode).
 * SGMV: tensor-core (tcgen05) tiles of 128 rows over same-adapter segments
 *       (prefill); bf16 tables with r_max >= 16 only (else LORA_EUNSUPPORTED).
 * AUTO: in a batch of at least LORA_AUTO_SGMV_MIN_TOKENS tokens that averages
 *       at least LORA_AUTO_SGMV_MIN_AVG tokens per adapter slot (num_tokens >=
 *       LORA_AUTO_SGMV_MIN_AVG * (num_slots - 1)) and has a segment of at
 *       least LORA_AUTO_LONG_ROWS tokens, segments with at least
 *       LORA_SGMV_MIN_ROWS tokens go to SGMV and the others to BGMV; other
 *       batches, and tables SGMV does not take, run all on BGMV (a batch that
 *       averages a few tokens per slot is decode-shaped, and its SGMV kernels
 *       would most likely find no segment to take). The choice depends only on
 *       num_tokens, the table and the metadata, so lora_shrink and lora_expand
 *       of one batch agree on it.
 * MIXED: AUTO's split for a batch of any size: segments with at least
 *       LORA_SGMV_MIN_ROWS tokens go to SGMV when the batch has a segment of
 *       at least LORA_AUTO_LONG_ROWS tokens, the others to BGMV (all BGMV for
 *       tables SGMV does not take). For a caller that knows its batch may hold
 *       a prefill chunk below AUTO's token thresholds (one new prompt beside a
 *       few hundred decode tokens runs several times faster this way); a
 *       batch without a long segment pays for SGMV launches that find
 *       nothing. */
typedef enum { LORA_AUTO = 0, LORA_BGMV = 1, LORA_SGMV = 2, LORA_MIXED = 3 } lora_kind;

#define LORA_MAX_SLICES 4
#define LORA_MAX_NUM_SLOTS 1024
#define LORA_MAX_RANK 128
#define LORA_MAX_TOKENS (1 << 24)
#define LORA_SGMV_MIN_ROWS 32      /* AUTO threshold: segment rows routed to SGMV */
#define LORA_SGMV_TILE_M 128       /* rows per SGMV tile (work-list granularity) */
#define LORA_AUTO_SGMV_MIN_TOKENS 1024  /* AUTO: smaller batches run all on BGMV */
#define LORA_AUTO_SGMV_MIN_AVG 20  /* AUTO: batches averaging fewer tokens per slot run all on BGMV */
#define LORA_AUTO_LONG_ROWS 64     /* AUTO: batches without a segment this long run all on BGMV */

/*
 * One LoRA-wrapped layer: the stacked slot table of one (packed) projection.
 * Layout follows the stacked per-slice buffers of the vLLM page, section
 * "包装层的形态" (lora_a_stacked / lora_b_stacked, one pair per packed slice),
 * stored in row-vector orientation:
 *   A[s]: device, [num_slots, d_in, r_max] row-major, dtype elements
 *   B[s]: device, [num_slots, r_max, out_sizes[s]] row-major
 *   slot_rank: device int32 [num_slots], rank of each slot (0 = empty)
 *   slot_scale: device fp32 [num_slots], scale applied to the shrink result
 * Slot 0 is reserved (kept zero, rank 0). Constraints: dtype in lora_dtype;
 * 1 <= n_slices <= LORA_MAX_SLICES; d_in and every out_sizes[s] positive
 * multiples of 8; r_max a power of two in [8, LORA_MAX_RANK];
 * 1 <= num_slots <= LORA_MAX_NUM_SLOTS; x_row_div >= 0. The library only
 * reads this struct.
 */
typedef struct {
  int32_t dtype;
  int32_t d_in;
  int32_t n_slices;
  int32_t out_sizes[LORA_MAX_SLICES];
  int32_t num_slots;
  int32_t r_max;
  void *A[LORA_MAX_SLICES];
  void *B[LORA_MAX_SLICES];
  int32_t *slot_rank;
  float *slot_scale;
  int32_t x_row_div;  /* LoRA row i of a call reads x row i / x_row_div (0 or 1: row i).
                         A mixture-of-experts w13 layer, whose LoRA rows are the
                         (token, choice) pairs of lora_moe_pair_slots, sets topk:
                         a token's hidden state serves its top-k pairs. */
} lora_layer_desc;

/*
 * Per-step token metadata (LoRAKernelMeta of the vLLM page, section
 * "LoRAKernelMeta:先按槽位排序"), relabelled so that slot 0 is no-LoRA.
 * All pointers are device pointers owned by the caller:
 *   token_slot  [num_tokens]     input: slot id of every token, batch order
 *   sorted_rows [num_tokens]     token indices, stably sorted by slot
 *   seg_slot    [num_slots]      slots present, ascending; then -1
 *   seg_count   [num_slots]      tokens per segment; then 0
 *   seg_start   [num_slots + 1]  first sorted row of each segment (leading 0),
 *                                then num_tokens
 *   num_segs, no_lora, status    [1] each: segments present; 1 if no token
 *                                uses a real adapter; count of token ids that
 *                                were outside [0, num_slots)
 *   tiles       work lists the kernels read (segment lists per kernel family
 *               and SGMV tile offsets); at least lora_meta_tiles_bytes(num_slots)
 *               bytes, 16-byte aligned. Its layout is private to the library.
 */
typedef struct {
  const int32_t *token_slot;
  int32_t num_tokens;
  int32_t num_slots;
  int32_t *sorted_rows;
  int32_t *seg_slot;
  int32_t *seg_count;
  int32_t *seg_start;
  int32_t *num_segs;
  int32_t *no_lora;
  int32_t *status;
  void *tiles;
  size_t tiles_bytes;
} lora_meta;

/*
 * Write an adapter into slot `slot` of every packed slice (set_lora of the
 * vLLM page, section "activate_adapter:把 CPU 上的低秩矩阵搬进 GPU 槽位").
 *   A_src[s]: device, [d_in, rank] row-major; B_src[s]: device,
 *   [rank, out_sizes[s]] row-major, desc->dtype elements; both arrays hold
 *   desc->n_slices pointers. A slice whose A_src and B_src are both NULL is
 *   zeroed (the adapter did not train it); exactly one NULL is LORA_EINVAL.
 * The rank tail [rank, r_max) is zero-filled so the math stays exact, and
 * slot_rank[slot] = rank, slot_scale[slot] = scale.
 * Errors: slot outside [1, num_slots) or rank outside [1, r_max] -> LORA_ERANGE.
 * The sources are only read during the call's kernels on `stream`.
 */
int lora_set_slot(const lora_layer_desc *desc, int32_t slot, int32_t rank, float scale,
                  const void *const *A_src, const void *const *B_src, lora_stream_t stream);

/*
 * Zero slot `slot` of every slice and set its rank and scale to 0 (reset_lora
 * of the same section). slot outside [1, num_slots) -> LORA_ERANGE.
 */
int lora_reset_slot(const lora_layer_desc *desc, int32_t slot, lora_stream_t stream);

/*
 * Build the per-step token metadata from meta->token_slot: a stable counting
 * sort of token indices by slot, the segments, no_lora, status and the work
 * lists, bit-exactly (LoRAKernelMeta.prepare_tensors of the vLLM page,
 * section "LoRAKernelMeta:先按槽位排序"). One call per step serves every
 * layer. num_tokens == 0 is valid (num_segs = 0, no_lora = 1).
 * Errors: num_slots outside [1, LORA_MAX_NUM_SLOTS], num_tokens outside
 * [0, LORA_MAX_TOKENS], a null output, tiles_bytes too small.
 */
int lora_prepare_meta(const lora_meta *meta, lora_stream_t stream);

/*
 * lora_prepare_meta for a metadata buffer that no kernel of the previous call
 * of this library on `stream` reads: the usual case is a serving loop that
 * alternates two lora_meta between steps, so the previous step's applies
 * read the other one. The outputs are the same, bit for bit, but they are
 * written as soon as they are computed instead of after the previous kernel
 * has finished, so the next shrink passes its wait as soon as the previous
 * step ends. When this call's kernel starts, everything before the previous
 * call's kernels is complete (this library's kernels release their successor
 * only after their own wait; a kernel launched without programmatic
 * dependent launch releases it when it ends), so only those kernels can
 * still be running. If one of them does read `meta`, the results of both
 * calls are undefined. Errors: as for lora_prepare_meta.
 */
int lora_prepare_meta_unshared(const lora_meta *meta, lora_stream_t stream);

/*
 * Shrink: for every token t whose slot a != 0 and every slice s,
 *   buf[s, t, k] = slot_scale[a] * sum_j x[t, j] * A[s][a, j, k]   (k < rank a)
 *   buf[s, t, k] = 0                                               (rank a <= k < r_max)
 * (lora_shrink / add_shrink of the vLLM page, section "shrink 核"; the scale
 * enters here as in section "PEFTHelper:认清 adapter 文件").
 *   x:   device, [num_tokens, d_in] with row stride ldx elements, desc->dtype
 *        (a row-parallel shard's d_in columns of a wider x: x advanced by the
 *        shard's first column, ldx the full width); with desc->x_row_div > 1,
 *        [ceil(num_tokens / x_row_div), d_in] and row i of the batch reads x
 *        row i / x_row_div (lora_apply reads x the same way)
 *   buf: device fp32, [n_slices, num_tokens, r_max] contiguous; rows of
 *        slot-0 tokens are not written
 *   ws:  device scratch of at least lora_workspace_bytes(desc, num_tokens,
 *        kind) bytes, 16-byte aligned, caller-owned. Both families split d_in
 *        and keep the partial rows of each split there (BGMV: chunks of
 *        32 KB of A; SGMV: as many splits as keep every SM busy, at most
 *        16); its contents need no initialisation and are meaningless
 *        between calls. Calls that share a workspace must not overlap in
 *        time (order them on one stream).
 * bf16 inputs are multiplied exactly and accumulated in fp32 in a fixed
 * order, and the splits are summed in split order (results do not depend
 * on the batch's other tokens, and repeat bitwise).
 */
int lora_shrink(const lora_layer_desc *desc, const lora_meta *meta, const void *x, int64_t ldx,
                float *buf, int32_t kind, void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * Expand: for every token t whose slot a != 0 and every slice s,
 *   y[t, off_s + n] = y[t, off_s + n] + sum_{k < rank a} buf[s, t, k] * B[s][a, k, n]
 * with off_s = out_sizes[0] + ... + out_sizes[s-1] (packed qkv / gate_up
 * outputs; lora_expand of the vLLM page, section "expand 核"). The sum is
 * formed in fp32 and added to y once; a bf16 y is rounded to nearest even.
 * Rows of slot-0 tokens are not read or written. Columns k >= rank a of buf
 * are ignored. The SGMV family multiplies buf as two bf16 parts (hi + lo,
 * relative error about 2^-17) on the tensor cores, with fp32 accumulation.
 *   buf: device fp32 [n_slices, num_tokens, r_max] as written by lora_shrink
 *   y:   device, [num_tokens, sum(out_sizes)] with row stride ldy elements,
 *        y_dtype (LORA_BF16 production; LORA_F32 for accuracy runs; an fp32
 *        table requires LORA_F32)
 * To add into a column range of a wider output -- the offset_start of the
 * fully-sharded variant (section "S-LoRA 式:把秩也切开"), where a shard's B
 * holds only its output columns -- pass y advanced by the range's first
 * column and ldy the full row width (16-byte alignment still applies).
 */
int lora_expand(const lora_layer_desc *desc, const lora_meta *meta, const float *buf, void *y,
                int64_t ldy, int32_t y_dtype, int32_t kind, lora_stream_t stream);

/*
 * Fused shrink + expand: the whole delta for every LoRA token in one call,
 *   y[t, off_s + n] += sum_k (scale[a] * x[t] . A[s][a])[k] * B[s][a, k, n]
 * with the same arithmetic, rounding and slot-0 rule as lora_shrink followed
 * by lora_expand (results are bitwise equal). The expand forms the rank-r
 * rows directly from the shrink's split partials in the workspace, so the
 * u buffer is optional (the "batched gather" form of the handbook page,
 * section "不合并权重，批量计算").
 *   buf: device fp32 [n_slices, num_tokens, r_max] or NULL. When non-NULL it
 *        also receives the shrink result.
 *   ws, ws_bytes: scratch as for lora_shrink.
 * Other arguments and errors as lora_shrink / lora_expand.
 */
int lora_apply(const lora_layer_desc *desc, const lora_meta *meta, const void *x, int64_t ldx, float *buf,
               void *y, int64_t ldy, int32_t y_dtype, int32_t kind, void *ws, size_t ws_bytes,
               lora_stream_t stream);

/* Scratch bytes lora_shrink / lora_apply need for this layer, kind and up to
 * max_tokens tokens on the current device (the SGMV part scales with its SM
 * count); 0 for an invalid desc or a kind the table does not support. */
size_t lora_workspace_bytes(const lora_layer_desc *desc, int32_t max_tokens, int32_t kind);

/* Bytes the meta->tiles work-list buffer needs for a table of num_slots slots. */
size_t lora_meta_tiles_bytes(int32_t num_slots);

/*
 * Mixture-of-experts LoRA (page "vLLM 源码完全拆解(十八): 多 LoRA 服务", section
 * "MoE 的 LoRA:按专家挂载、融合 kernel 与 EP 切片"): every expert has its own
 * low-rank pair per adapter, applied after w13 (before the activation) and
 * after w2 (before the top-k sum). This call gives each (token, choice) pair,
 * token-major (pair p = t * topk + k), the composite slot of its (adapter,
 * local expert):
 *   pair_slot[p] = 1 + (a - 1) * local_experts + expert_map[e]
 * with a = token_slot[t], e = topk_ids[t * topk + k]; 0 (no delta) when a is 0
 * or expert_map[e] < 0 (an expert another expert-parallel rank holds); -1
 * (counted as a bad id by lora_prepare_meta) when a is outside [0, num_loras],
 * e outside [0, num_experts) or expert_map[e] >= local_experts. expert_map
 * NULL means every expert is local (e itself). The composite table then has
 * 1 + num_loras * local_experts slots: slot 1 + (a - 1) * local_experts + j
 * holds adapter a's pair for local expert j. lora_prepare_meta over pair_slot
 * groups the pairs by (adapter, expert), which is what the pages'
 * moe_lora_align_block_size does; the w13 application is then lora_apply
 * (or shrink / expand) on the w13 table with x_row_div = topk and the token
 * rows as x, the w2 application the same on the w2 table with the pairs'
 * rows, both with the pairs' metadata.
 *   token_slot [num_tokens], topk_ids [num_tokens * topk], expert_map
 *   [num_experts] (or NULL), pair_slot [num_tokens * topk]: device int32,
 *   4-byte aligned, caller-owned. It waits for the previous kernel before it
 *   reads and releases its successor only when done (lora_prepare_meta reads
 *   pair_slot before waiting).
 * Errors: a null array (other than expert_map) -> LORA_EINVAL; num_tokens
 * outside [0, LORA_MAX_TOKENS / topk], topk outside [1, 64], num_loras < 0,
 * num_experts < 1, local_experts outside [1, num_experts], or a composite
 * table above LORA_MAX_NUM_SLOTS slots -> LORA_ERANGE; misaligned arrays ->
 * LORA_EALIGN. num_tokens == 0 is a no-op.
 */
int lora_moe_pair_slots(const int32_t *token_slot, const int32_t *topk_ids, int32_t num_tokens, int32_t topk,
                        int32_t num_loras, int32_t num_experts, int32_t local_experts, const int32_t *expert_map,
                        int32_t *pair_slot, lora_stream_t stream);

/*
 * Synchronise `stream`, copy meta->status to *out (host) and return
 * LORA_EDEVICE if a kernel since the last lora_prepare_meta gave up waiting
 * on its own pipeline, else LORA_EBADTOKEN if lora_embed_shrink met token ids
 * outside the vocabulary, else LORA_OK if *out is 0 and LORA_EBADSLOT if some
 * token slot ids were out of range.
 */
int lora_query_status(const lora_meta *meta, int32_t *out, lora_stream_t stream);

/*
 * Diagnostic of the device-side failure path. The tensor-core (SGMV)
 * kernels wait on their own pipeline barriers with a time limit (200 ms):
 * a wait that runs out records a bit in the metadata's device error word and
 * the kernel winds down instead of hanging, and lora_query_status then
 * returns LORA_EDEVICE. The multi-LoRA pages have no counterpart; this call
 * lets a caller (or a test) see that path work without any fault: it launches
 * one thread that runs the same bounded wait, with a limit of limit_us
 * microseconds, on a barrier nothing will ever arm. After it, until the next
 * lora_prepare_meta on `meta` (which clears the error word),
 * lora_query_status(meta) returns LORA_EDEVICE; the stream and the context
 * stay usable. The kernel issues no memory copy or MMA.
 *   limit_us: 1 .. 1,000,000, else LORA_ERANGE; meta as for lora_prepare_meta.
 */
int lora_probe_bounded_wait(const lora_meta *meta, uint32_t limit_us, lora_stream_t stream);

/*
 * Embedding lookup: the shrink of an embedding layer's LoRA (page "vLLM 源码完全
 * 拆解(十八): 多 LoRA 服务", section "embedding 的 LoRA 是一个查表增量"). With
 * desc->d_in the vocabulary size and one slice, A[0] = [num_slots, vocab, r_max]
 * holds slot a's r-vector for token id v at A[0][a, v, :] (the page's
 * lora_a_stacked; it indexes the flattened table at v + a * vocab). For every
 * token t whose slot a = meta->token_slot[t] != 0,
 *   buf[0, t, k] = scale[a] * A[0][a, token_id[t], k]     (k < rank a)
 *   buf[0, t, k] = 0                                       (rank a <= k < r_max)
 * -- lora_shrink's result for the one-hot row of token_id[t] -- and rows of
 * slot-0 tokens are not written. lora_expand with the layer's B then adds the
 * delta into the embedding output. A token id outside [0, d_in) gives a zero
 * row (no delta) and makes lora_query_status report LORA_EBADTOKEN; it never
 * traps.
 *   token_id: device int32 [num_tokens], batch order (the rows of meta)
 *   buf:      device fp32 [1, num_tokens, r_max], 16-byte aligned
 * Needs no metadata output (only meta->token_slot) and no workspace.
 * Errors: LORA_EINVAL for null pointers, n_slices != 1 or a table / meta
 * mismatch; LORA_EALIGN for a misaligned buf.
 */
int lora_embed_shrink(const lora_layer_desc *desc, const lora_meta *meta, const int32_t *token_id, float *buf,
                      lora_stream_t stream);

/*
 * Allocation-free shrink. The multi-LoRA pages have no counterpart to this
 * call; it exists for callers that cannot allocate device memory where they
 * run the shrink (inside another framework's memory pool, under an allocator
 * that forbids new device allocations, or on a serving path that must not
 * call an allocator at all).
 * Computes exactly what lora_shrink computes with kind LORA_BGMV (same
 * arguments, same results), but keeps the per-chunk partial rows in a fixed
 * 8 MiB array inside the library's device image instead of a caller
 * workspace; the caller still owns x and buf. Every GPU that loads the
 * library holds that array until the process exits.
 * - The first call on a device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture. The cached address belongs to that device's context:
 *   after cudaDeviceReset (or anything else that destroys and recreates
 *   the device's primary context) it is stale, so do not call this entry
 *   point again in that process.
 * - All calls share the one array and it keeps the last call's contents.
 *   Nothing in it needs to start at zero. Calls whose kernels overlap on the
 *   GPU (on different streams, or from different threads without ordering)
 *   race on it: order them.
 * - A layer and token count whose partial rows exceed
 *   lora_noalloc_scratch_bytes() return LORA_ERANGE and launch nothing.
 * - It never calls cudaMalloc, cudaFree or any allocating routine.
 */
int lora_shrink_noalloc(const lora_layer_desc *desc, const lora_meta *meta, const void *x, int64_t ldx,
                        float *buf, lora_stream_t stream);

/* Size in bytes of the fixed scratch array lora_shrink_noalloc uses. */
size_t lora_noalloc_scratch_bytes(void);

/* Static description of a lora_status value. */
const char *lora_strerror(int status);

/* CUDA error code of the last LORA_ECUDA returned on this host thread (0 if none). */
int lora_last_cuda_error(void);

/* Kernels this library has launched in this process, on every device and
 * thread, counting launches captured into CUDA graphs once (at capture). */
uint64_t lora_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* RANK_ADAPTER_GB300_LORA_H */
