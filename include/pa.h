/*
 * pa.h: C ABI of libpa, decode-time attention over a paged KV cache on one
 * NVIDIA GB300 (sm_103a).
 *
 * Operations, all asynchronous on the caller's CUDA stream:
 *
 *   pa_cache_write    slot-mapping scatter of new K/V rows into the block pool;
 *   pa_decode         grouped-query attention of one query token per sequence
 *                     over that sequence's cached context, read in place
 *                     through its block table;
 *   pa_verify         the k+1-token speculative-verify variant: writes the new
 *                     tokens' K/V and attends with a causal mask among them;
 *   pa_verify_ragged  the same with a different number of new tokens per
 *                     sequence (query_start), decode rows included;
 *   pa_prefill        causal attention of prompt chunks already in the cache;
 *   pa_validate       a device-side check of tables, lengths and slots;
 *   pa_decode_noalloc pa_decode with library-owned scratch.
 *
 * Where each operation is defined:
 *  - The cache is head-major, [kv_heads, num_blocks, block_size, head_dim], so
 *    one index over a sequence's slots returns its context in order ("From
 *    183 ms to 19 ms per decode step", section "2. Head-major KV cache").
 *  - Decode walks each sequence's block table and reads K and V straight from
 *    the cache, one (sequence, KV head) with its whole query-head group at a
 *    time, with an online softmax in fp32 (same page, section "3. A Triton
 *    paged-decode kernel"). Query head hq reads KV head hq / (q_heads /
 *    kv_heads) (same page, section "1. Grouped attention").
 *  - Each step's per-token inputs are cache slots, block tables and context
 *    lengths, copied into fixed buffers so the calls can be captured in a CUDA
 *    graph (same page, section "4. CUDA graphs per batch bucket").
 *  - Verify carries k+1 query tokens per sequence with a causal mask among
 *    them (same page, section "Then speculative decoding got slower").
 *  - A zero key is not neutral, so every key beyond a sequence's length is
 *    masked, scores and values both ("A Rust inference server for Qwen2 on
 *    Apple Silicon", Day 3 "Known gaps").
 *
 * Conventions shared by every call:
 *  - Pointers named d_* or documented as "device" point to device memory of
 *    the current device; all arrays are C-contiguous. Element pointers (cache,
 *    q, out, k_new, v_new) must be 16-byte aligned.
 *  - The caller owns every buffer, including the workspace. The library
 *    allocates nothing, frees nothing and keeps no pointer after a call
 *    returns. Buffers must stay alive until the stream reaches the call (a
 *    captured graph keeps reading the same addresses on every replay).
 *  - Calls never synchronise the host and never read device memory on the
 *    host; the launch grid depends on host arguments only, so every call can
 *    be captured in a CUDA graph.
 *  - Arguments the host can check are checked before anything is launched; a
 *    failing check returns an error status and nothing is written.
 *  - Device-resident indices (block ids, context lengths, slots) are the
 *    caller's contract. Kernels never read or write outside the cache for a
 *    bad index: a block id outside [0, num_blocks) reads zeros, a slot outside
 *    the pool is skipped, a length above the limits is clamped; each such
 *    event raises a bit in the workspace status word (pa_workspace_status)
 *    where a workspace is passed. pa_validate reports them without attending.
 *  - Kernels contain no trap and no unbounded wait. A wait that exceeds its
 *    limit raises PA_FLAG_TIMEOUT and the kernel returns.
 *
 * Supported shapes: head_dim 128, block_size 16, dtype bf16, fp32 or int8,
 * q_heads a multiple of kv_heads.
 *
 * The int8 pool ("A Rust inference server for Qwen2 on Apple Silicon", Day 4
 * "int8 KV", "Grouping is the whole question", "Partial blocks"):
 *  - k and v hold bytes q + 128 of symmetric codes q in [-127, 127], in the
 *    same head-major layout. k_scale holds one fp32 scale per (kv head,
 *    block, channel), [kv_heads, num_blocks, head_dim]. v_scale holds one per
 *    (kv head, block, row), [kv_heads, num_blocks, block_size].
 *  - A stored value is (byte - 128) * scale.
 *  - Quantising a group with m = max|x| > 0 stores the scale s = m / 127
 *    and the codes q = RN(x * (127 / m)), clamped to [-127, 127]: one IEEE
 *    fp32 division per group (127 / m), then one fp32 multiply per element,
 *    rounded to nearest with ties to even. An all-zero group has s = 0 and
 *    bytes 128.
 *  - Queries, new rows and outputs are bf16. Attention dequantises inside
 *    the kernel: the K scales multiply the query in fp32 and each product
 *    enters the score products as two f16 parts (about 22 bits); V bytes
 *    enter exactly, with the row scales folded into the softmax weights (one
 *    f16 rounding of each weight). Each product q * (K scale) must stay below
 *    65504 in magnitude.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the caches. For F32 and BF16, queries, new rows and
 * outputs have the same type; for INT8 they are bf16. */
typedef enum pa_dtype {
    PA_DTYPE_F32 = 0,
    PA_DTYPE_BF16 = 1,
    PA_DTYPE_INT8 = 2
} pa_dtype;

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null or misaligned pointer, negative size, inconsistent shapes */
    PA_ERR_UNSUPPORTED = 2, /* head_dim != 128, block_size != 16, unknown dtype, option out of range */
    PA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than pa_workspace_size() */
    PA_ERR_CUDA = 4         /* a CUDA runtime/driver call failed; see pa_last_cuda_error() */
} pa_status;

/* Bits of the device status word in the workspace (pa_workspace_status). */
#define PA_FLAG_BAD_BLOCK 0x1u   /* a block id outside [0, num_blocks) was met (zeros were read) */
#define PA_FLAG_BAD_LENGTH 0x2u  /* a context length < 0, > max_context_len or > table capacity (clamped) */
#define PA_FLAG_BAD_SLOT 0x4u    /* a slot >= num_blocks * block_size (the write was skipped) */
#define PA_FLAG_TIMEOUT 0x8u     /* a bounded wait gave up; results of that call are not valid */

/* The block pool: two head-major tensors [kv_heads, num_blocks, block_size,
 * head_dim] of `dtype`, device memory, 16-byte aligned. */
typedef struct pa_cache {
    void *k;
    void *v;
    int32_t kv_heads;
    int32_t num_blocks;
    int32_t block_size; /* must be 16 */
    int32_t head_dim;   /* must be 128 */
    int32_t dtype;      /* pa_dtype */
    /* PA_DTYPE_INT8 only (ignored otherwise): fp32 scales, device, 16-byte
     * aligned. k_scale [kv_heads, num_blocks, head_dim]; v_scale [kv_heads,
     * num_blocks, block_size]. */
    void *k_scale;
    void *v_scale;
} pa_cache;

/* Kernel choice for pa_decode / pa_verify / pa_prefill. */
typedef enum pa_kernel {
    PA_KERNEL_AUTO = 0,    /* bf16: PA_KERNEL_MMA; fp32: PA_KERNEL_SIMT */
    PA_KERNEL_MMA = 1,     /* bf16 only: a producer warp stages 16-token K/V tiles with TMA
                              tensor loads; bf16 tensor-core products, fp32 softmax */
    PA_KERNEL_SIMT = 2,    /* CUDA-core fp32 arithmetic, any dtype (the fp32 caches' kernel) */
    PA_KERNEL_TC = 4       /* pa_prefill only (its default): tcgen05 products with the S and O
                              accumulators and the Q and P operands in tensor memory */
} pa_kernel;

/* Optional settings for pa_decode / pa_verify / pa_verify_ragged /
 * pa_prefill; pass NULL for the defaults. */
typedef struct pa_options {
    /* Tokens per context split (flash-decoding split-K). A positive multiple
     * of block_size: every sequence uses this split. 0 = the default rule:
     * for a sequence of up to PA_LONG_CONTEXT_TOKENS tokens,
     * PA_DEFAULT_SPLIT_TOKENS (bf16, fp32) or PA_DEFAULT_SPLIT_TOKENS_INT8
     * (int8 pool); for a longer one, PA_DEFAULT_SPLIT_LONG (bf16, fp32) or
     * PA_DEFAULT_SPLIT_LONG_INT8. Either way a sequence's split depends only
     * on its own length and the pool's format, never on its batch-mates, so
     * its result is bit-identical across batch compositions. A call whose
     * longest sequence would need more than 65535 splits returns
     * PA_ERR_UNSUPPORTED. */
    int32_t split_tokens;
    int32_t kernel;   /* pa_kernel */
    /* Bound, in nanoseconds, on each wait of the tensor-core attention
     * kernels for a shared-memory stage or a peer warp; 0 = the default,
     * PA_DEFAULT_WAIT_LIMIT_NS (one second). A wait that runs past it raises
     * PA_FLAG_TIMEOUT, and the CTA lets its own copies in flight land (under
     * the default bound) and returns without writing its rows. The default
     * is far above any wait of a healthy call; a small value exists to
     * exercise the timeout path, whose results are then not valid. */
    uint32_t wait_limit_ns;
} pa_options;

#define PA_DEFAULT_WAIT_LIMIT_NS 1000000000u

#define PA_DEFAULT_SPLIT_TOKENS 768
#define PA_DEFAULT_SPLIT_TOKENS_INT8 1536
#define PA_LONG_CONTEXT_TOKENS 4096
#define PA_DEFAULT_SPLIT_LONG 1152
#define PA_DEFAULT_SPLIT_LONG_INT8 704

/*
 * pa_cache_write: cache[h, s / 16, s % 16, :] = new[i, h, :] for every token
 * i with slot s = slot_mapping[i] >= 0, for both K and V, copied bit for bit.
 * Defined by the per-step "cache slots" input ("From 183 ms to 19 ms per
 * decode step", section "4. CUDA graphs per batch bucket") and the
 * write-before-attend order of a decode step ("Anatomy of a Decode-Step
 * Stall", the engine's Model._layer).
 *
 *   cache         the pool (device tensors written in place).
 *   d_k_new, d_v_new  [num_tokens, kv_heads, head_dim] of cache->dtype (bf16
 *                     for an int8 pool), device.
 *   d_slot_mapping    [num_tokens] int32, device. s < 0: token skipped.
 *                     s >= num_blocks*16: skipped (no status word here; use
 *                     pa_validate to find it). Duplicate slots: unspecified
 *                     which write lands (int8: the later token).
 *
 * int8 pool: the write quantises ("Partial blocks" of the int8 page). For
 * every block that receives rows in this call, its K rows are dequantised,
 * the incoming rows overwrite theirs, each channel's scale is recomputed over
 * the block and every row is requantised. Each incoming V row is quantised
 * on its own scale. Bytes and scales are deterministic (exact fp32 steps).
 *   num_tokens    >= 0; 0 launches nothing.
 *   stream        cudaStream_t (NULL = legacy default stream).
 * Returns PA_OK or an error status (nothing launched on error).
 */
pa_status pa_cache_write(const pa_cache *cache, const void *d_k_new, const void *d_v_new,
                         const int32_t *d_slot_mapping, int32_t num_tokens, void *stream);

/*
 * Bytes of workspace pa_decode / pa_verify need for these sizes. The workspace
 * holds a status word, one arrival counter per (sequence, KV head, row group)
 * and the fp32 split partials. It must be zero-filled once before first use
 * (pa_workspace_init); every call leaves it ready for the next, except one
 * that raised PA_FLAG_TIMEOUT, which may leave arrival counters set: zero-fill
 * the workspace again before its next use.
 * num_queries is 1 for decode. Under the default split rule the size covers
 * either pool format (it counts the finer of their splits). Returns 0 if an
 * argument is invalid.
 */
size_t pa_workspace_size(int32_t batch, int32_t num_queries, int32_t q_heads, int32_t kv_heads,
                         int32_t head_dim, int32_t max_context_len, const pa_options *opts);

/* Zero-fill a workspace on `stream` (asynchronous). */
pa_status pa_workspace_init(void *d_workspace, size_t workspace_bytes, void *stream);

/*
 * Read and clear the workspace status word (PA_FLAG_* bits). Synchronises
 * `stream` and copies 4 bytes to the host: a diagnostic, not for the hot path.
 */
pa_status pa_workspace_status(void *d_workspace, uint32_t *host_flags, void *stream);

/*
 * pa_decode: for every sequence b and query head hq (KV head h = hq / G,
 * G = q_heads / kv_heads), with L = context_lens[b],
 *     s_t = scale * <q[b, hq, :], K[h, t, :]>            for t < L,
 *     out[b, hq, :] = sum_t softmax(s)_t * V[h, t, :],
 * where K[h, t, :] = cache.k[h, block_tables[b][t / 16], t % 16, :]
 * ("From 183 ms to 19 ms per decode step", sections "1. Grouped attention",
 * "2. Head-major KV cache", "3. A Triton paged-decode kernel"). L = 0 gives
 * zeros. The softmax runs in fp32 with a running max and sum; products of bf16
 * inputs accumulate in fp32; out is rounded to the cache dtype.
 *
 *   cache          the pool (read only).
 *   d_q            [batch, q_heads, head_dim], device.
 *   d_out          [batch, q_heads, head_dim], device; must not overlap inputs.
 *   d_block_tables [batch, max_blocks_per_seq] int32, device. Entries at or
 *                  beyond ceil(L/16) are never read.
 *   d_context_lens [batch] int32, device; each in [0, max_context_len] and
 *                  <= max_blocks_per_seq * 16 (else clamped and flagged).
 *   max_context_len host-side upper bound of context_lens; sizes the grid.
 *   scale          softmax scale (1/sqrt(head_dim) for the standard form).
 *   d_workspace    >= pa_workspace_size(batch, 1, ...) bytes, zeroed once.
 *   opts           NULL or pa_options.
 */
pa_status pa_decode(const pa_cache *cache, const void *d_q, void *d_out,
                    const int32_t *d_block_tables, int32_t max_blocks_per_seq,
                    const int32_t *d_context_lens, int32_t batch, int32_t q_heads,
                    int32_t max_context_len, float scale, void *d_workspace,
                    size_t workspace_bytes, const pa_options *opts, void *stream);

/*
 * pa_verify: one fused call of the speculative-verify step. The num_queries
 * new tokens of sequence b sit at positions L - num_queries + i (L =
 * context_lens[b] counts them). Their K/V rows are written to the cache at
 * slot_mapping[b * num_queries + i], and query i attends to positions
 * t <= L - num_queries + i (causal among the new tokens; "From 183 ms to 19 ms
 * per decode step", section "Then speculative decoding got slower"). The
 * result equals pa_cache_write followed by attention over the updated cache,
 * provided each slot is the table slot of its position (pa_validate checks
 * this); the attention reads the new rows from d_k_new / d_v_new directly.
 * A row whose position is negative returns zeros. Padded query rows are
 * computed like any other and may be discarded by the caller.
 *
 * int8 pool: the call runs the quantised pa_cache_write, then the attention
 * kernel as its programmatic dependent. That kernel streams the blocks
 * before the new tokens at once, and waits for the write only before the
 * blocks that hold them. The result equals pa_cache_write followed by
 * pa_decode-style attention over the requantised pool, for any slots.
 *
 *   d_q, d_out     [batch, num_queries, q_heads, head_dim], device.
 *   d_k_new, d_v_new [batch * num_queries, kv_heads, head_dim], device.
 *   d_slot_mapping [batch * num_queries] int32, device.
 *   Other arguments as in pa_decode; the cache is written in place.
 */
pa_status pa_verify(const pa_cache *cache, const void *d_q, void *d_out, const void *d_k_new,
                    const void *d_v_new, const int32_t *d_slot_mapping, int32_t num_queries,
                    const int32_t *d_block_tables, int32_t max_blocks_per_seq,
                    const int32_t *d_context_lens, int32_t batch, int32_t q_heads,
                    int32_t max_context_len, float scale, void *d_workspace,
                    size_t workspace_bytes, const pa_options *opts, void *stream);

/*
 * pa_verify_ragged: pa_verify for sequences with different numbers of new
 * tokens in one launch: decode sequences (one token) and verify sequences
 * (k+1 tokens) side by side, none padded ("From 183 ms to 19 ms per decode
 * step", section "Then speculative decoding got slower": padded guesses cost
 * a second set of graphs). Sequence b has n_b = query_start[b+1] -
 * query_start[b] new tokens, at positions L - n_b + i (L = context_lens[b]
 * counts them); its query, output, new-row and slot entries are the flat
 * rows query_start[b] .. query_start[b+1] - 1. Query i attends to positions
 * t <= L - n_b + i. The result equals pa_verify run on each sequence alone.
 *
 *   d_q, d_out     [total_queries, q_heads, head_dim], device.
 *   d_k_new, d_v_new [total_queries, kv_heads, head_dim], device.
 *   d_slot_mapping [total_queries] int32, device.
 *   d_query_start  [batch + 1] int32, device: 0 = query_start[0] <= ... <=
 *                  query_start[batch] = total_queries. An entry outside that
 *                  order, or an n_b above max_queries, is clamped and raises
 *                  PA_FLAG_BAD_LENGTH.
 *   max_queries    host bound on every n_b (>= 1); the workspace is sized with
 *                  it as num_queries (pa_workspace_size).
 *   Other arguments as in pa_verify.
 */
pa_status pa_verify_ragged(const pa_cache *cache, const void *d_q, void *d_out, const void *d_k_new,
                           const void *d_v_new, const int32_t *d_slot_mapping,
                           const int32_t *d_query_start, int32_t total_queries, int32_t max_queries,
                           const int32_t *d_block_tables, int32_t max_blocks_per_seq,
                           const int32_t *d_context_lens, int32_t batch, int32_t q_heads,
                           int32_t max_context_len, float scale, void *d_workspace,
                           size_t workspace_bytes, const pa_options *opts, void *stream);

/*
 * pa_prefill: causal attention of prompt chunks over the paged cache (prefill
 * or chunked prefill; "From 183 ms to 19 ms per decode step", section "What's
 * next"). Sequence b's chunk is its last n_b = query_start[b+1] -
 * query_start[b] positions, L - n_b .. L - 1 (L = context_lens[b] counts
 * them); their K/V must already be in the cache (pa_cache_write). Query token
 * i of the chunk attends to positions t <= L - n_b + i; a token at a negative
 * position gets zeros. Each K/V block is read once per 128 query rows (token x
 * query head of one KV head).
 *
 *   cache          bf16 only (PA_ERR_UNSUPPORTED otherwise).
 *   d_q, d_out     [total_queries, q_heads, head_dim] bf16, device.
 *   d_query_start  [batch + 1] int32, device, as in pa_verify_ragged;
 *                  max_queries bounds every n_b (it sizes the grid).
 *   d_workspace    optional (NULL: no status word): a 256-byte-aligned buffer of
 *                  >= 256 bytes whose first word receives PA_FLAG_* bits.
 *   opts           optional; opts->kernel and opts->wait_limit_ns are read
 *                  (split_tokens is not: a prefill has no split). kernel is
 *                  PA_KERNEL_AUTO, PA_KERNEL_TC (tcgen05 kernel, two CTAs per
 *                  SM; needs q_heads / kv_heads <= 128, else
 *                  PA_ERR_UNSUPPORTED) or PA_KERNEL_MMA (warp-level mma.sync
 *                  kernel: the one AUTO takes for groups above 128, where a
 *                  tcgen05 row tile cannot hold whole tokens); anything else
 *                  returns PA_ERR_UNSUPPORTED.
 *   Other arguments as in pa_decode. No split-K: one CTA reads the whole
 *   visible context of its 128 rows.
 */
pa_status pa_prefill(const pa_cache *cache, const void *d_q, void *d_out, const int32_t *d_query_start,
                     int32_t total_queries, int32_t max_queries, const int32_t *d_block_tables,
                     int32_t max_blocks_per_seq, const int32_t *d_context_lens, int32_t batch, int32_t q_heads,
                     int32_t max_context_len, float scale, void *d_workspace, size_t workspace_bytes,
                     const pa_options *opts, void *stream);

/*
 * pa_validate: check the device-resident per-step inputs without attending.
 * Writes a report of PA_VALIDATE_WORDS uint32 words to d_report (device):
 *   [0] PA_FLAG_* bits found;
 *   [1] count of sequences with a bad length (< 0, > max_context_len,
 *       > max_blocks_per_seq * 16, or < num_queries when num_queries > 1);
 *   [2] count of block-table entries in use outside [0, num_blocks);
 *   [3] count of slots outside [-1, num_blocks * 16) or not equal to the
 *       table slot of their position (only when d_slot_mapping is non-NULL).
 * d_slot_mapping may be NULL; it then holds batch * num_queries entries
 * otherwise. Never traps; graph-capturable.
 */
#define PA_VALIDATE_WORDS 4
pa_status pa_validate(const pa_cache *cache, const int32_t *d_block_tables,
                      int32_t max_blocks_per_seq, const int32_t *d_context_lens, int32_t batch,
                      int32_t max_context_len, const int32_t *d_slot_mapping,
                      int32_t num_queries, uint32_t *d_report, void *stream);

/*
 * pa_decode_noalloc: pa_decode for callers that cannot allocate device memory
 * at the point of the call, for example a plugin running inside a host program
 * that owns every device allocation itself, or code that must not grow the
 * device's memory footprint once it is running. The pages have no counterpart
 * to this call; it exists for those callers only.
 *
 * Arguments and results are those of pa_decode without the workspace: the
 * split partials, arrival counters and status word live instead in one
 * library-owned device array of PA_NOALLOC_SCRATCH_BYTES.
 *  - The first call on a device sets the array up there: it looks up the
 *    array's address with that device current, and that lookup loads the
 *    library's code module holding the array, so the CUDA runtime places the
 *    array (PA_NOALLOC_SCRATCH_BYTES of device memory) on the device at that
 *    moment (under the runtime's default lazy module loading; with
 *    CUDA_MODULE_LOADING=EAGER it is placed when the device's context is
 *    created). The device then holds it until the process exits. Make that
 *    first call at start-up: before the footprint must stay fixed and before
 *    any stream capture on the device. Every later call allocates and frees
 *    nothing.
 *  - Arguments are checked as pa_decode checks them, before anything else; a
 *    rejected call returns pa_decode's status and touches nothing. Sizes
 *    whose pa_workspace_size() exceeds PA_NOALLOC_SCRATCH_BYTES then return
 *    PA_ERR_WORKSPACE before anything is launched.
 *  - Every call reuses the same array and clears the parts that must start at
 *    zero. Calls whose work overlaps on the GPU (different streams, or
 *    different host threads on one device) race on it: serialise them.
 *  - The status word is not readable through this call; use pa_validate to
 *    check device-resident indices.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
pa_status pa_decode_noalloc(const pa_cache *cache, const void *d_q, void *d_out,
                            const int32_t *d_block_tables, int32_t max_blocks_per_seq,
                            const int32_t *d_context_lens, int32_t batch, int32_t q_heads,
                            int32_t max_context_len, float scale, const pa_options *opts,
                            void *stream);

/* Human-readable name of a status. */
const char *pa_status_string(pa_status status);

/* The last CUDA error code seen by a call that returned PA_ERR_CUDA (0 if none). */
int pa_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
