/*
 * mla.h -- C ABI of libmla_gb300: single-token Multi-Head Latent Attention
 * (MLA) decode over a paged, compressed KV cache, for one GB300 (sm_103a).
 *
 * Sources of the operations (page title, then section):
 *   "Beyond the Attention Bottleneck" (micrologics.org), sections
 *      "Down-Projection and Up-Projection Mechanics" (the latent c_t and the
 *      up-projections K_t = W^UK c_t, V_t = W^UV c_t) and "The RoPE
 *      Compatibility Problem" (decoupled positional key);
 *   "Seven Ways LLMs Handle Attention" (sotaaz.com), section 5 "Multi-head
 *      latent attention" (512-wide latent + 64-wide RoPE key = 576 numbers per
 *      token per layer; absorbing the expansions into the query and output
 *      projections);
 *   "The Architecture of Memory" (ashimsharma10.github.io), sections "The
 *      Weight Absorption Trick", "Decoupled Rotary Positional Encoding",
 *      "PagedAttention: Virtual Memory for LLMs", "The 2-Bit Quantization
 *      Barrier and KIVI", "Flash-Decoding and FlashInfer";
 *   "KV Cache Optimization" (managen.ai), sections 3 "KV Cache Quantization"
 *      and 7 "Paged Attention (vLLM)".
 *
 * Conventions for every entry point:
 *   - Every tensor argument is a DEVICE pointer to caller-owned, contiguous,
 *     row-major memory; the library allocates no device memory.  Scratch for
 *     mla_decode lives in a caller-provided workspace.
 *   - Work is enqueued asynchronously on the caller's stream; calls are
 *     stateless (apart from the profiling hook mla_set_timing_events) and
 *     may be issued from several host threads on different streams.
 *   - Errors that the host can see (null or misaligned pointers, bad sizes,
 *     unsupported dimensions, small workspace) are returned before anything is
 *     launched.  Errors found on the device (out-of-range page-table entries
 *     or sequence lengths, a bounded wait that ran out) are written as a
 *     status code to device memory and read back with mla_read_device_status;
 *     the offending work is skipped, never trapped.
 *   - Row layout of the cache: each token of each sequence occupies one row of
 *     576 numbers, [latent c_t (512) | RoPE key k_pe_t (64)].
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t / CUstream and cudaEvent_t / CUevent;
 * a NULL stream means the legacy default stream. */
typedef struct CUstream_st* mla_stream_t;
typedef struct CUevent_st* mla_event_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,     /* null/misaligned pointer, negative or inconsistent size   */
  MLA_ERR_UNSUPPORTED = -2,     /* dimensions this library does not implement              */
  MLA_ERR_WORKSPACE = -3,       /* workspace missing, misaligned or smaller than required  */
  MLA_ERR_CUDA = -4,            /* a CUDA runtime/driver call failed (launch, tensor map)  */
  MLA_ERR_DEVICE_TIMEOUT = -5,  /* device: a bounded wait inside a kernel ran out          */
  MLA_ERR_DEVICE_BOUNDS = -6    /* device: a page-table entry, position or length was out
                                   of range; that token / sequence was skipped             */
} mla_status;

typedef enum {
  MLA_CACHE_BF16 = 0,  /* cache rows are 576 bf16 values                                   */
  MLA_CACHE_INT8 = 1,  /* cache rows are 576 int8 codes plus fp32 (scale, zero point) per
                          row; value = scale * (code - zero_point)                          */
  MLA_CACHE_FP8 = 2    /* cache rows are 576 FP8 E4M3 codes (1 sign, 4 exponent bits with
                          bias 7, 3 mantissa bits; no infinities; 0x7F/0xFF are NaN) plus
                          one fp32 scale per row; value = scale * e4m3(code)                */
} mla_cache_dtype;

/* Model dimensions.  This library implements kv_lora_rank = 512, rope_dim = 64,
 * qk_nope_dim = 128, v_head_dim = 128 (the DeepSeek-V2/V3 shapes of "Seven
 * Ways LLMs Handle Attention", section 5), page_size in {16, 32, 64, 128},
 * and num_heads = 16 or any positive multiple of 32. */
typedef struct {
  int32_t num_heads;     /* H: query heads                                   */
  int32_t kv_lora_rank;  /* d_c: latent width                                */
  int32_t rope_dim;      /* d_rope: decoupled RoPE key width, shared by heads */
  int32_t qk_nope_dim;   /* per-head content query/key width                 */
  int32_t v_head_dim;    /* per-head value width                             */
  int32_t page_size;     /* P: tokens per cache page                         */
  int32_t cache_dtype;   /* mla_cache_dtype                                  */
} mla_dims;

/* Returns MLA_OK if this library implements `dims`, else MLA_ERR_INVALID_ARG
 * (null, non-positive sizes) or MLA_ERR_UNSUPPORTED. */
int mla_check_dims(const mla_dims* dims);

/*
 * mla_cache_append -- write new tokens into the paged latent cache.
 * "The Architecture of Memory", decode phase ("the new Key and Value are
 * appended") and "PagedAttention" (fixed-size pages mapped through a page
 * table); "Beyond the Attention Bottleneck", "The RoPE Compatibility
 * Problem" (the positional key carries RoPE); "KV Cache Optimization" section
 * 3 and "The Architecture of Memory", KIVI section (per-token min/max
 * quantisation) for MLA_CACHE_INT8 and MLA_CACHE_FP8.
 *
 * For token i (0 <= i < n_tokens): b = seq_ids[i], pos = positions[i],
 * physical page = block_table[b * max_pages_per_seq + pos / P], slot = pos % P.
 * The row written there is [c_kv[i] (512) | RoPE(pos, k_pe[i]) (64)], where
 * RoPE rotates each pair (x[2j], x[2j+1]) by the angle pos * theta^(-2j/64),
 * computed in fp64 and rounded once to bf16 (rope_theta <= 0: k_pe is stored
 * unrotated).  INT8 caches then quantise the 576 bf16 values of the row:
 * lo = min(min x, 0), hi = max(max x, 0), s = (hi - lo)/255 (1 if 0),
 * zp = clamp(rint(-128 - lo/s)), code = clamp(rint(x/s) + zp, -128, 127),
 * all in IEEE fp32 round-to-nearest-even, and store (s, zp).  FP8 caches
 * take a = max |x|, s = a/448 (1 if 0) and code = the E4M3 value nearest
 * to x/s (ties to the even mantissa, magnitudes past 448 saturate, the sign
 * of zero kept), in IEEE fp32 round-to-nearest-even, and store s.
 *
 *   cache            bf16, int8 or E4M3 (uint8) [num_pages, P, 576]
 *   cache_scale_zero fp32 [num_pages, P, 2] (INT8), fp32 [num_pages, P] (FP8),
 *                    NULL for bf16
 *   block_table      int32 [num_seqs, max_pages_per_seq]
 *   seq_ids, positions  int32 [n_tokens]
 *   c_kv             bf16 [n_tokens, 512];  k_pe bf16 [n_tokens, 64]
 *   device_status    optional int32 (device); if a token's seq id, position
 *                    or page-table entry is out of range the token is
 *                    skipped and MLA_ERR_DEVICE_BOUNDS is stored here.
 * Two tokens mapping to one slot in the same call race (last writer wins).
 * n_tokens = 0 is a no-op.
 */
int mla_cache_append(const mla_dims* dims, void* cache, float* cache_scale_zero, int32_t num_pages,
                     const int32_t* block_table, int32_t num_seqs, int32_t max_pages_per_seq,
                     const int32_t* seq_ids, const int32_t* positions, int32_t n_tokens,
                     const void* c_kv, const void* k_pe, double rope_theta,
                     int32_t* device_status, mla_stream_t stream);

/* Number of KV partitions mla_decode uses when num_splits = 0 on the current
 * device: one per attention unit that can be resident at once (a CTA pair,
 * or a CTA where pairs are not used) and row group.  < 0 on error. */
int mla_auto_num_splits(const mla_dims* dims, int32_t batch);

/* Bytes of workspace mla_decode needs for (dims, batch, num_splits); 0 if the
 * arguments are invalid.  num_splits = 0 means the automatic choice on the
 * current device. */
size_t mla_decode_workspace_size(const mla_dims* dims, int32_t batch, int32_t num_splits);

/*
 * mla_decode -- one decode step of MLA attention for every head of every
 * sequence, in the absorbed form.
 * "Beyond the Attention Bottleneck", "Down-Projection and Up-Projection
 * Mechanics" and "The RoPE Compatibility Problem" define the attention:
 * score_t = scale * (q_nope . W^UK c_t + q_pe . k_pe_t), o = sum_t p_t W^UV c_t.
 * "The Weight Absorption Trick" and "Seven Ways LLMs Handle Attention"
 * section 5 give the absorbed evaluation used here: q_lat = W^UK^T q_nope is
 * formed once per head, scores are taken against the 576-wide cached rows
 * directly, the probability-weighted latent sum is formed, and W^UV is
 * applied last.  "Flash-Decoding and FlashInfer" gives the split of the KV
 * length into chunks merged by log-sum-exp.
 *
 *   q_nope      bf16 [batch, H, 128]
 *   q_pe        bf16 [batch, H, 64], already rotated for the new position
 *   cache, cache_scale_zero   as for mla_cache_append (both 16-byte aligned)
 *   block_table int32 [batch, max_pages_per_seq]
 *   seq_lens    int32 [batch] (device): tokens attended by each sequence,
 *               including the one being decoded; 0 gives out = 0, lse = -inf.
 *               Lengths above max_pages_per_seq * P, and page-table entries
 *               outside [0, num_pages), raise MLA_ERR_DEVICE_BOUNDS on the
 *               device and the sequence (or page) is skipped.
 *   W_UK, W_UV  bf16 [H, 128, 512] (head h's W^UK_h, W^UV_h in R^{128x512})
 *   softmax_scale  multiplies the raw dot product (e.g. 1/sqrt(128+64))
 *   num_splits  KV partitions over the batch's total work (0 = automatic).
 *               The work of every row group is cut into num_splits equal
 *               pieces, so a sequence holding a fraction f of all tokens is
 *               split into about f * num_splits chunks.  The attention units
 *               take contiguous blocks of partitions: above the automatic
 *               count, a multiple of it gives every unit the same work.
 *   workspace   device scratch, 256-byte aligned, at least
 *               mla_decode_workspace_size(dims, batch, num_splits) bytes.
 *               Its first 4 bytes hold the device status of this call.
 *   out         bf16 [batch, H, 128]
 *   lse_out     optional fp32 [batch, H]: natural-log log-sum-exp of the
 *               scaled scores.
 * Results are bit-identical between runs with the same inputs and the same
 * num_splits; calls sharing one workspace must not overlap on the device.
 */
int mla_decode(const mla_dims* dims, const void* q_nope, const void* q_pe, const void* cache,
               const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
               int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
               const void* W_UK, const void* W_UV, float softmax_scale, int32_t num_splits,
               void* workspace, size_t workspace_bytes, void* out, float* lse_out,
               mla_stream_t stream);

/* Largest number of query tokens per sequence mla_decode_multi accepts. */
#define MLA_MAX_Q_LEN 8

/* Bytes of workspace mla_decode_multi needs for (dims, batch, q_len,
 * num_splits); 0 if the arguments are invalid.  q_len = 1 gives
 * mla_decode_workspace_size. */
size_t mla_decode_multi_workspace_size(const mla_dims* dims, int32_t batch, int32_t q_len, int32_t num_splits);

/*
 * mla_decode_multi -- decode q_len query tokens per sequence against the
 * paged cache in one pass: the verification read of speculative decoding
 * ("The Architecture of Memory", "Speculative Decoding: Amortizing the Memory
 * Fetch": the target model checks all drafted tokens in one forward pass that
 * reads its cache once) with a causal mask among the new tokens (same page,
 * "Tree Attention Verification": dense attention over the history, masked
 * among the new tokens; this entry point takes a chain, not a tree).
 *
 * The q_len new tokens of sequence b are the last q_len tokens of its cache
 * (append them first): query token t sits at position seq_lens[b] - q_len + t
 * and attends to cache positions [0, seq_lens[b] - q_len + t], itself
 * included.  A query whose position is below 0 (seq_lens[b] < q_len) attends
 * to nothing: out = 0, lse = -inf.  Everything else is as for mla_decode:
 *
 *   q_nope      bf16 [batch, q_len, H, 128]
 *   q_pe        bf16 [batch, q_len, H, 64], each rotated for its own position
 *   out         bf16 [batch, q_len, H, 128]
 *   lse_out     optional fp32 [batch, q_len, H]
 *   q_len       1 .. MLA_MAX_Q_LEN; q_len = 1 is exactly mla_decode
 *   workspace   at least mla_decode_multi_workspace_size(dims, batch, q_len,
 *               num_splits) bytes.
 * The work of the batch is that of a single-token decode with q_len * H
 * heads, so num_splits = 0 picks the automatic count for q_len * H heads.
 * Returns MLA_ERR_INVALID_ARG for q_len outside [1, MLA_MAX_Q_LEN].
 */
int mla_decode_multi(const mla_dims* dims, const void* q_nope, const void* q_pe, const void* cache,
                     const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                     int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                     const void* W_UK, const void* W_UV, float softmax_scale, int32_t num_splits,
                     void* workspace, size_t workspace_bytes, void* out, float* lse_out,
                     mla_stream_t stream);

/* Largest prefill chunk (new tokens per sequence) mla_prefill accepts. */
#define MLA_MAX_PREFILL_CHUNK 2048

/* Largest number of query rows (batch * tokens per sequence * H) of one
 * decode or prefill call; larger calls return MLA_ERR_INVALID_ARG (and their
 * workspace size is 0). */
#define MLA_MAX_QUERY_ROWS (1 << 26)

/* Bytes of workspace mla_prefill needs for (dims, batch, chunk, num_splits);
 * 0 if the arguments are invalid.  It holds the chunk's absorbed queries and
 * the partial latent outputs, batch * chunk * H * (1,152 + 2,048 per
 * partition) bytes and up. */
size_t mla_prefill_workspace_size(const mla_dims* dims, int32_t batch, int32_t chunk, int32_t num_splits);

/*
 * mla_prefill -- one chunk of chunked prefill: write the chunk's rows into
 * the paged cache, then attend each of its tokens to the cache up to and
 * including itself.
 * "The Architecture of Memory", "The Prefill Phase: Compute-Bound
 * Parallelism" (the prompt's tokens are processed together and their
 * key/value state goes into the cache that decode reads; a long prompt goes
 * in chunks, each attending to what the chunks before it wrote).
 *
 * Sequence b's chunk is the `chunk` tokens at positions seq_lens[b] - chunk
 * .. seq_lens[b] - 1 (seq_lens counts the cache after the chunk).  The call
 *   1. writes token t's row [c_kv[b][t] | RoPE(pos, k_pe[b][t])] at position
 *      pos = seq_lens[b] - chunk + t, exactly as mla_cache_append (1-byte
 *      caches quantise it); a token whose position is below 0 or past the
 *      page table is skipped and MLA_ERR_DEVICE_BOUNDS is recorded;
 *   2. computes, for every head of query token t, attention over positions
 *      0 .. pos, exactly as mla_decode_multi with q_len = chunk (a query
 *      below position 0 gets out = 0, lse = -inf).
 *
 *   cache, cache_scale_zero, block_table  as for mla_cache_append /
 *               mla_decode (the cache is written, then read)
 *   seq_lens    int32 [batch] (device)
 *   c_kv        bf16 [batch, chunk, 512];  k_pe bf16 [batch, chunk, 64]
 *               (unrotated; the append rotates it by rope_theta)
 *   q_nope      bf16 [batch, chunk, H, 128]
 *   q_pe        bf16 [batch, chunk, H, 64], rotated for each token's position
 *   out         bf16 [batch, chunk, H, 128]
 *   lse_out     optional fp32 [batch, chunk, H]
 *   chunk       1 .. MLA_MAX_PREFILL_CHUNK
 *   workspace   at least mla_prefill_workspace_size(dims, batch, chunk,
 *               num_splits) bytes; its first 4 bytes are the call's device
 *               status (mla_read_device_status), covering the append too.
 * The attention is query-tiled: the chunk's chunk * H (token, head) rows of
 * a sequence run in groups of 128 rows, each group on the MMA's M extent
 * against 64-token sub-tiles of the sequence's pages (a group of fewer rows
 * is padded; chunk * H of 32 or 64 rows on bf16 caches runs as 32-row
 * groups).  Each group streams its sequence's pages, from L2 after the
 * first.
 */
int mla_prefill(const mla_dims* dims, void* cache, float* cache_scale_zero, int32_t num_pages,
                const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                int32_t chunk, const void* c_kv, const void* k_pe, double rope_theta, const void* q_nope,
                const void* q_pe, const void* W_UK, const void* W_UV, float softmax_scale, int32_t num_splits,
                void* workspace, size_t workspace_bytes, void* out, float* lse_out, mla_stream_t stream);

/* Largest index-list length mla_decode_sparse accepts. */
#define MLA_MAX_TOP_K (1 << 20)

/* Bytes of workspace mla_decode_sparse needs for (dims, batch, top_k,
 * num_splits); 0 if the arguments are invalid. */
size_t mla_decode_sparse_workspace_size(const mla_dims* dims, int32_t batch, int32_t top_k, int32_t num_splits);

/*
 * mla_decode_sparse -- decode against a selection of each sequence's cached
 * tokens: the attention of DeepSeek Sparse Attention on MLA ("Seven Ways LLMs
 * Handle Attention", section 6, "Sparse attention: keep every token, read
 * only some": the whole cache stays, and each new token attends only to the
 * top-k tokens an indexer picked).  The indexer is not part of this library:
 * the caller passes its choice.
 *
 *   token_indices  int32 [batch, top_k] (device): positions in sequence b's
 *                  cache, each in [0, seq_lens[b]); -1 entries are padding.
 *                  The attention of (b, h) runs over the rows at the listed
 *                  positions, each listed entry once (a position listed
 *                  twice counts twice).  Other values raise
 *                  MLA_ERR_DEVICE_BOUNDS and the entry is skipped.
 *   top_k          1 .. MLA_MAX_TOP_K
 *   workspace      at least mla_decode_sparse_workspace_size(dims, batch,
 *                  top_k, num_splits) bytes; its first 4 bytes hold the
 *                  device status of this call.
 * Everything else is as for mla_decode (q_len = 1).  A sequence with no
 * valid entry gets out = 0, lse = -inf.  Listing every position 0 ..
 * seq_lens[b] - 1 in order gives exactly mla_decode's result.  The selected
 * rows are first copied, in list order, into pages inside the workspace
 * (about top_k * 1,152 bytes per sequence for bf16 caches), which the decode
 * then reads.
 */
int mla_decode_sparse(const mla_dims* dims, const void* q_nope, const void* q_pe, const void* cache,
                      const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                      int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                      const int32_t* token_indices, int32_t top_k, const void* W_UK, const void* W_UV,
                      float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                      void* out, float* lse_out, mla_stream_t stream);

/* Size of the fixed scratch array used by mla_decode_no_alloc. */
#define MLA_NO_ALLOC_WORKSPACE_BYTES (16u << 20)

/*
 * mla_decode_no_alloc -- mla_decode without a caller workspace.  The pages
 * have no counterpart to this entry point; it serves callers that cannot
 * allocate device memory: for example, a serving loop that must not call
 * cudaMalloc on its decode path (the call can synchronise the device and
 * stall every stream), or a plain C host that embeds this library inside a
 * process whose device memory is budgeted up front and owned by someone else.
 *
 * Arguments and results are those of mla_decode, minus the workspace.  The
 * scratch is one device array of MLA_NO_ALLOC_WORKSPACE_BYTES (16 MiB) that
 * lives in the library for as long as the process has it loaded, on every
 * GPU it runs on.  A call whose mla_decode_workspace_size(dims, batch,
 * num_splits) exceeds that size returns MLA_ERR_WORKSPACE without launching
 * anything; use mla_decode with a caller workspace for such shapes.  The
 * call allocates nothing.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current, so make a
 * first call on each device before any stream capture.  All calls on a
 * device share the one array: calls that may overlap on the GPU (different
 * streams, or different host threads) race on it and must be serialised by
 * the caller.  device_status (optional, int32 on the device) receives a
 * copy of the call's device status word, as mla_read_device_status would
 * report it for mla_decode.
 */
int mla_decode_no_alloc(const mla_dims* dims, const void* q_nope, const void* q_pe, const void* cache,
                        const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                        int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                        const void* W_UK, const void* W_UV, float softmax_scale, int32_t num_splits,
                        void* out, float* lse_out, int32_t* device_status, mla_stream_t stream);

/*
 * mla_combine -- merge per-chunk partial results by log-sum-exp ("The
 * Architecture of Memory", "Flash-Decoding and FlashInfer").
 *   partial_o    fp32 [batch, num_splits, H, kv_lora_rank], each normalised
 *                within its chunk
 *   partial_lse  fp32 [batch, num_splits, H], natural log; -inf marks an
 *                empty chunk (weight 0)
 *   o_lat_out    fp32 [batch, H, kv_lora_rank]:
 *                sum_s exp(lse_s - lse) * partial_o[s]
 *   lse_out      optional fp32 [batch, H]: lse = ln sum_s exp(lse_s)
 * A (b, h) whose chunks are all empty gives zeros and -inf.
 */
int mla_combine(const mla_dims* dims, const float* partial_o, const float* partial_lse,
                int32_t batch, int32_t num_splits, float* o_lat_out, float* lse_out,
                mla_stream_t stream);

/* Synchronises `stream`, then copies the device status word at the start of
 * `workspace` (as written by the last mla_decode that used it) to *status_out. */
int mla_read_device_status(const void* workspace, int32_t* status_out, mla_stream_t stream);

/* Synchronises `stream` and reads an append status word (see mla_cache_append). */
int mla_read_status_word(const int32_t* device_status, int32_t* status_out, mla_stream_t stream);

/* Human-readable text of a status code (static storage). */
const char* mla_status_string(int status);

/* Profiling hook: while set (both non-NULL), every mla_decode records
 * `start` just before and `stop` just after its attention kernel, on the
 * call's stream, so the caller can time that kernel with cudaEventElapsedTime.
 * Pass NULLs to clear.  Process-wide; not for concurrent profiling. */
int mla_set_timing_events(mla_event_t start, mla_event_t stop);

/* Test hook for the device-side failure detection (no counterpart on the
 * pages).  While enabled (non-zero), every mla_decode launches its attention
 * kernel with the first cache-page barrier of each CTA expecting 16 bytes more
 * than its copies deliver: that wait cannot complete, runs into its time
 * limit (about 2 s), and the kernel records MLA_ERR_DEVICE_TIMEOUT in the
 * workspace status word, releases its resources and returns; the device and
 * the context stay usable.  Nothing faults, traps or hangs.  Process-wide; 0
 * (the default) disables it.  Returns MLA_OK. */
int mla_test_inject_wait_timeout(int32_t enable);

/* Test hook (no counterpart on the pages): while enabled (non-zero), bf16
 * decodes use the single-CTA attention kernel that serves devices on which
 * the CTA-pair kernel cannot be placed (the pair kernel runs otherwise), so
 * that this fallback stays tested on devices that never need it.
 * Process-wide; 0 (the default) disables it.  Returns MLA_OK. */
int mla_test_force_single_cta(int32_t enable);

/* Library version: major * 10000 + minor * 100 + patch. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
