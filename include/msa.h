/*
 * msa.h -- C ABI of the GB300 (sm_103a) block-sparse attention (MSA) hot path.
 *
 * The method (MiniMax-M3 sparse attention, as the pages describe it):
 *   "MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120)", section "What this
 *   fixes": for each GQA group the model keeps the 16 key blocks with the
 *   largest block maxima of the index scores, always including the block
 *   that holds the current position.
 *   "minimax_m3: a CUDA backend for MiniMax-M3.1-Flash at TP over GB10s"
 *   (PR #1388), native Metal family commit: the lightning indexer scores
 *   keys and 16 blocks are chosen for each row and key head; a decode row
 *   attends to its chosen blocks in partial results merged afterwards, and
 *   prompt chunks run their attention on the matrix units, each tile over
 *   its chosen blocks.  Same PR, prompt-tile commit: the 16 query heads of a
 *   key head use the same chosen blocks, so one read of a key or value block
 *   serves them all.  Same PR, cache commit: the key, value and index-key
 *   caches hold bf16.
 *
 * For every query row r (absolute position p) and KV head h:
 *   s_t  = iq[r,h,:] . ik[t,h,:]                     t = 0..p        (indexer)
 *   m_j  = max { s_t : t in block j, t <= p }        j = 0..J, J = p / S
 *   K    = {J} + the (top_k-1) best j < J by (m_j desc, j asc); all j <= J
 *          when J < top_k; listed ascending
 *   out[r, h*G+g] = softmax_t(scale * q[r,h*G+g] . k[t,h]) . v[t,h]
 *          over t in the blocks of K with t <= p
 *
 * Conventions for every entry point
 *   - All tensors are device pointers (cudaMalloc'd or equivalent) owned by
 *     the caller.  The library allocates no device or pinned memory; scratch
 *     space comes from the caller's workspace (msa_workspace_size).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and launch only the library's own kernels.  No call
 *     synchronises the device or reads device memory on the host, so every
 *     call can be enqueued back to back.
 *   - bf16 is bfloat16: the upper 16 bits of an IEEE-754 binary32 (uint16_t); fp32 is float.
 *   - Layouts are contiguous, row-major:
 *       q    [total_rows, H*G, D]   bf16   q head g of KV head h is h*G+g
 *       iq   [total_rows, H, Di]    bf16
 *       k, v [cache_tokens, H, D]   bf16   token t of sequence b is row
 *                                   (int8 + fp32 scales [cache_tokens, H]
 *                                   with kv_dtype = MSA_KV_INT8)
 *       ik   [cache_tokens, H, Di]  bf16   cache_starts[b] + t  (H -> 1: shared key)
 *       out  [total_rows, H*G, D]   fp32 or bf16 (msa_problem.out_dtype)
 *       sel  [total_rows, H, top_k] int32, kept blocks ascending, -1 padded
 *       nsel [total_rows, H]        int32, number of kept blocks
 *     Every pointer must be 16-byte aligned.
 *   - Rows of sequence b are cu_rows[b] .. cu_rows[b+1]-1.  With n rows and
 *     cache length L (the rows' own tokens included), row i is at p = L-n+i.
 *   - Errors: invalid or unsupported arguments are rejected on the host
 *     before anything is enqueued (MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED,
 *     MSA_ERR_WORKSPACE).  A failed launch returns MSA_ERR_CUDA.  Device
 *     metadata (cu_rows, cache_lens, cache_starts, block_table) is read only by kernels:
 *     values inconsistent with the host-side bounds in msa_problem are the
 *     caller's error; kernels clamp them so that they never read or write
 *     out of the stated extents, and the affected outputs are unspecified.
 *     msa_last_error() returns a message for the calling thread's last
 *     failure.  Nothing traps on the device.
 *   - Supported set: D = 128, Di = 64, S = 64, 1 <= top_k <= 16,
 *     1 <= G <= 16, H in {1, 2, 4, 8}, max_cache_len <= 2^21,
 *     num_seqs <= 4096; other values return MSA_ERR_UNSUPPORTED.
 *   - Thread safety: calls from several host threads are safe; the only
 *     library state is per-device set-up (kernel shared-memory limits, the
 *     SM count), the thread-local error message and, for
 *     msa_attend_decode_noalloc alone, its scratch array and the per-context
 *     cache of that array's address.  Two calls sharing one workspace must
 *     be ordered on the GPU.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum msa_status {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad alignment        */
    MSA_ERR_UNSUPPORTED = 2, /* valid, but outside the supported set         */
    MSA_ERR_WORKSPACE = 3,   /* workspace null or smaller than required      */
    MSA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed  */
    MSA_ERR_INTERNAL = 5     /* a library invariant failed                   */
} msa_status;

enum { MSA_OUT_F32 = 0, MSA_OUT_BF16 = 1 };

/* Element type of the key and value caches (msa_problem.kv_dtype). */
enum { MSA_KV_BF16 = 0, MSA_KV_INT8 = 1 };

/* One batch: B sequences, each with n_b >= 1 query rows and a cache of L_b
 * tokens (n_b <= L_b).  Host fields size grids and workspaces; device
 * fields are read by the kernels. */
typedef struct msa_problem {
    int32_t num_seqs;         /* B >= 1                                        */
    int32_t num_kv_heads;     /* H                                             */
    int32_t group_size;       /* G, query heads per KV head                    */
    int32_t head_dim;         /* D = 128                                       */
    int32_t index_dim;        /* Di = 64                                       */
    int32_t block_size;       /* S = 64                                        */
    int32_t top_k;            /* kept blocks per row and KV head, local incl.  */
    float softmax_scale;      /* finite, >= 0; typically 1/sqrt(D)             */
    int32_t out_dtype;        /* MSA_OUT_F32 or MSA_OUT_BF16                   */
    int32_t total_rows;       /* R = cu_rows[B] (host copy)                    */
    int32_t max_rows_per_seq; /* >= every n_b (host bound); <= 8 = decode family only */
    int32_t max_cache_len;    /* >= every L_b (host bound)                     */
    int64_t cache_tokens;     /* rows in each of k, v, ik (host), < 2^31       */
    int32_t num_decode_seqs;  /* host count of decode-family sequences (1 to 8
                                 rows), or -1 if unknown (then both kernel
                                 families run and each skips the other's
                                 sequences)                                   */
    const int32_t* cu_rows;      /* device [B+1], cu_rows[0] = 0, ascending    */
    const int32_t* cache_lens;   /* device [B], 1 <= L_b <= max_cache_len      */
    const int64_t* cache_starts; /* device [B], start + L_b <= cache_tokens;
                                    NULL (not read) with a block table         */
    /* Paged caches (optional).  With block_table set, position t of sequence
     * b is row  block_table[b * block_table_stride + t / page_size] *
     * page_size + t % page_size  of k, v and ik (each a pool of cache_tokens
     * rows = num_pages * page_size); cache_starts is not read.  NULL: the
     * contiguous layout through cache_starts.  Page numbers outside
     * [0, cache_tokens / page_size) set the device error word (bad metadata)
     * and are not read. */
    const int32_t* block_table;  /* device [B, block_table_stride] int32 page numbers, or NULL */
    int32_t block_table_stride;  /* >= ceil(max_cache_len / page_size)           */
    int32_t page_size;           /* tokens per page: a power of two >= 64 (=S x 2^k) */
    /* Index keys per position: 0 or num_kv_heads = one per KV head (ik is
     * [cache_tokens, H, Di]); 1 = one key shared by every KV head (ik is
     * [cache_tokens, 1, Di]) and s_t = iq[r,h,:] . ik[t,0,:]. */
    int32_t index_key_heads;
    /* Key/value cache element type.  PR #1388, native Metal family commit:
     * keys and values cached as int8 with one scale per position and head
     * (a later commit of that PR returns to bf16).  MSA_KV_BF16 (0): k, v are
     * bf16 [cache_tokens, H, D].  MSA_KV_INT8 (1): k, v are int8
     * [cache_tokens, H, D] and the attention reads
     *     k[t, h, d] = k_scale[row * H + h] * k8[row, h, d]   (v likewise)
     * for the cache row `row` of position t; the index keys stay bf16.  The
     * scales are device fp32 [cache_tokens, H], read only with MSA_KV_INT8
     * (NULL otherwise).  Supported by msa_forward, msa_attend_decode and
     * msa_attend_prefill; msa_attend_decode_noalloc takes bf16 caches only. */
    int32_t kv_dtype;
    const float* k_scale;
    const float* v_scale;
    /* Host count of the rows of decode-family sequences (1 to 8 rows each),
     * or <= 0 if unknown.  msa_forward sizes the decode attention's grid by
     * it instead of num_seqs x min(max_rows_per_seq, 8) row slots, which in a
     * batch that mixes decode rows with prompt chunks launches mostly empty
     * work; a count below the device metadata's sets the bad-metadata bit of
     * the error word (the rows past it get no output), one above it only
     * launches work that exits at once.  Library mechanics: the pages have
     * no counterpart. */
    int32_t num_decode_rows;
} msa_problem;

/* Human-readable name of a status code (static string).  Library mechanics:
 * the pages define no interface for the method. */
const char* msa_status_string(msa_status status);

/* Message describing the calling thread's most recent failure ("" if none).
 * Library mechanics (no counterpart in the pages). */
const char* msa_last_error(void);

/* Bytes of scratch that msa_forward, msa_attend_decode and msa_attend_prefill
 * need for problem p (host only; enqueues nothing).  Library mechanics (no
 * counterpart in the pages).  The workspace must be
 * 256-byte aligned; its contents need no initialisation and are clobbered.
 * Its first 4 bytes are the device error word of the last call that used
 * it: 0, or a bitwise OR of 1 (a bounded wait gave up), 2 (device metadata
 * outside the host-side bounds, e.g. a sequence with more rows than
 * max_rows_per_seq; such a sequence is skipped, nothing is written outside
 * the buffers), 4 (tensor memory could not be allocated); valid once that
 * call has completed on the stream.
 * With an int8 key/value cache (kv_dtype MSA_KV_INT8) and prompt chunks whose
 * rows keep at least four times as many key rows (rows x top_k x 64) as the
 * attended sequences have positions (their count x max_cache_len, rounded up
 * to 64), the workspace also holds a bf16 copy of those sequences' keys and
 * values with their scales (520 x H bytes a position, at most 8 GiB): each
 * position is widened once per call (exactly: int8 values are bf16 integers)
 * instead of once per kept block of every row, and msa_forward launches one
 * more kernel (msa_forward_launches counts it). */
msa_status msa_workspace_size(const msa_problem* p, size_t* bytes);

/* Stage 1 alone: the lightning-indexer scores.  PR #1388, native Metal family
 * commit: the indexer scores the cached keys for each row and key head;
 * "MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120)", section "Alternative:
 * NVFP4 (SGLang)": the model's sparse layers carry this lightning indexer.
 * The pages give no formula; the score taken here is the plain dot product
 * of the row's index query with the position's index key:
 *   scores[r, h, t] = iq[r,h,:] . ik[t,h,:]   (fp32)   for t <= p,
 *   scores[r, h, t] = -inf                             for p < t < ld.
 * scores is [total_rows, H, ld] fp32 with ld >= max_cache_len.  fp32
 * accumulation: exact when the products and partial sums are integers below
 * 2^24 in magnitude (index values in [-8, 8] give |s| <= 4096).  This staged
 * path materialises every score and exists for stage-by-stage checking; the
 * fused path (msa_forward) never writes them. */
msa_status msa_index_scores(const msa_problem* p, const void* iq, const void* ik_cache,
                            float* scores, int64_t ld, void* stream);

/* Stage 2 alone.  "MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120)", section
 * "What this fixes": blocks are scored by the maximum of their index scores,
 * 16 blocks are kept per GQA group and the block holding the current
 * position is always among them; PR #1388, native Metal family commit: the
 * selection is made per row and key head.  Block max-pool of `scores` (as
 * written by msa_index_scores, entries past p ignored), then the local block
 * J plus the top_k-1 best blocks j < J, ties to the lower block index (every
 * block 0..J when J < top_k), listed ascending.  Writes sel and nsel. */
msa_status msa_select_blocks(const msa_problem* p, const float* scores, int64_t ld,
                             int32_t* sel, int32_t* nsel, void* stream);

/* Stage 3, decode form.  PR #1388, native Metal family commit: a decode row
 * attends to its kept blocks in partial results (32 keys each there) that
 * are merged afterwards.  Every sequence has 1 to 8 rows
 * (max_rows_per_seq <= 8), e.g. one decode row or a drafted window.  The
 * kept blocks of one (row, KV head) are
 * split over a cluster of 8 CTAs (two blocks each); their partial softmax
 * states (running max, sum, unnormalised output) are combined by
 * log-sum-exp on chip, through distributed shared memory.  sel/nsel as msa_select_blocks
 * writes them (entries must be causal blocks <= J, ascending, distinct;
 * 1 <= nsel <= top_k).  A count nsel < 1 or > top_k sets the bad-metadata
 * bit of the error word; with nsel < 1 (no kept block, an empty softmax)
 * the G outputs of that (row, KV head) are written as zeros.
 * Needs msa_workspace_size bytes of workspace. */
msa_status msa_attend_decode(const msa_problem* p, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* sel, const int32_t* nsel,
                             void* out, void* workspace, size_t workspace_bytes, void* stream);

/* Stage 3, decode form, for callers that cannot allocate device memory.
 * The pages describe no counterpart: this is a deployment variant of
 * msa_attend_decode for one decode row per sequence.  Some callers cannot call cudaMalloc at all -- code
 * enqueued while a framework captures a CUDA graph and forbids allocation
 * inside the capture, hosts whose device memory is carved out once at
 * start-up, plug-ins that do not own the process's allocator -- so this
 * entry point takes no workspace and allocates nothing: its scratch (split
 * partials, tickets, error word) is a fixed device array inside the library,
 * about 4 MiB, which every GPU that loads the library holds until the
 * process exits.  Limits: num_seqs * num_kv_heads <= 32 (larger problems
 * are rejected with MSA_ERR_UNSUPPORTED) and exactly one row per sequence
 * (max_rows_per_seq == 1, else MSA_ERR_INVALID_ARG; msa_attend_decode takes
 * up to 8).  Within those limits the arguments and results are those of
 * msa_attend_decode, including the zero output for nsel < 1.  The first call
 * in each CUDA context (normally once per device) looks up the array's
 * device address (a host-side query, made with that device current); make
 * that first call before any stream capture.  After cudaDeviceReset the
 * device has a new context and the next call looks the address up again.  Every call shares the one
 * array: calls that overlap on the GPU (several streams or host threads)
 * race and give wrong results, so order them on one stream.  Device-side
 * errors are recorded only in the library's own scratch and are not
 * reported by this entry point. */
msa_status msa_attend_decode_noalloc(const msa_problem* p, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* sel, const int32_t* nsel,
                                     void* out, void* stream);

/* Stage 3, prompt-chunk form (any rows per sequence).  PR #1388, native
 * Metal family commit: prompt chunks run their attention on the matrix units,
 * each tile over its kept blocks; same PR, prompt-tile commit: the 16 query
 * heads of a key head share the rows' selection, so one read of a key or
 * value block serves them all.  Here: tcgen05 tensor-core tiles of one
 * (row, KV head) whose G query heads share each key/value block read;
 * accumulators live in tensor memory.  Same arguments as the decode form. */
msa_status msa_attend_prefill(const msa_problem* p, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* sel, const int32_t* nsel,
                              void* out, void* workspace, size_t workspace_bytes, void* stream);

/* The fused hot path: all three stages for every row of the batch (the
 * passages cited at msa_index_scores, msa_select_blocks, msa_attend_decode
 * and msa_attend_prefill; the key, value and index-key caches hold bf16 as in
 * PR #1388, bf16-cache commit).
 * Sequences with 1 to 8 rows (the decode family: decode rows, drafted
 * windows) take the decode kernels (index-key scan with the block max-pool
 * fused in, one pass over the index keys for all of a sequence's rows, then
 * selection + split attention + combine per row); sequences with more rows
 * take the prompt-chunk kernels (tcgen05 indexer
 * with the pool and a running top-k in its epilogue, then tcgen05
 * attention).  No scores are materialised.  sel_out/nsel_out (nullable)
 * receive the selection. */
msa_status msa_forward(const msa_problem* p, const void* q, const void* iq, const void* k_cache,
                       const void* v_cache, const void* ik_cache, void* out, int32_t* sel_out,
                       int32_t* nsel_out, void* workspace, size_t workspace_bytes, void* stream);

/* msa_forward with timing marks (library mechanics, no counterpart in the
 * pages): events[i] (cudaEvent_t, created by the caller, may be NULL) is
 * recorded on `stream` at mark i:
 *   0 before the first kernel, 1 after the decode index scan, 2 after decode
 *   attention, 3 after the prompt-chunk indexer, 4 after prompt-chunk
 *   attention.  Marks of a path with no rows are recorded back to back.
 * n_events <= 5. */
msa_status msa_forward_marked(const msa_problem* p, const void* q, const void* iq,
                              const void* k_cache, const void* v_cache, const void* ik_cache,
                              void* out, int32_t* sel_out, int32_t* nsel_out, void* workspace,
                              size_t workspace_bytes, void* stream, void* const* events,
                              int32_t n_events);

/* Number of kernels msa_forward launches for p (host only; library
 * mechanics, no counterpart in the pages). */
int32_t msa_forward_launches(const msa_problem* p);

/* Diagnostics of the failure path (library mechanics, no counterpart in the
 * pages).  Every barrier wait in the library's
 * kernels gives up after a time limit, sets bit 1 of the device error word
 * and lets the kernel finish (after waiting, again with a limit, for its own
 * copies in flight), so a lost arrival ends a call with an error instead of
 * a hung GPU.  This call makes one such wait run out on purpose: one thread
 * waits on a barrier that nothing arrives on, gives up after limit_us
 * microseconds (1 .. 2,000,000) and ORs 1 into the 32-bit word at the start
 * of `workspace` (device memory, >= 4 bytes, owned by the caller; the word
 * is not cleared first).  Asynchronous on `stream`; argument errors return
 * MSA_ERR_INVALID_ARG or MSA_ERR_WORKSPACE without launching. */
msa_status msa_check_wait_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
