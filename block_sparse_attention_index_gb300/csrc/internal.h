// Host-side interface between the C ABI layer (msa_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

// Where the cache rows of a sequence live in k, v and ik: contiguous
// (position t of sequence b at row starts[b] + t) or paged (row
// table[b * stride + t / page] * page + t % page, page = 2^page_shift >= 64,
// so a 64-position block never straddles two pages).
struct CacheRows {
    const int64_t* starts;  // contiguous layout (table == nullptr)
    const int32_t* table;   // paged layout: [num_seqs, stride] page numbers
    int32_t stride;
    int32_t page_shift;
    int64_t num_pages;
};

#ifdef __CUDACC__
// Row of the first position of the 64-position block holding position t
// (t a multiple of 64, t < L_b) of sequence b, or -1 when its page number is
// outside the pool: the caller flags bad metadata and reads nothing there.
// (The contiguous layout is checked per sequence by seq_rows_ok.)
__device__ __forceinline__ int64_t block_row(const CacheRows& c, int b, int64_t t) {
    if (c.table == nullptr) return c.starts[b] + t;
    const int32_t pg = c.table[static_cast<int64_t>(b) * c.stride + (t >> c.page_shift)];
    if (pg < 0 || pg >= c.num_pages) return -1;
    return (static_cast<int64_t>(pg) << c.page_shift) + (t & ((int64_t{1} << c.page_shift) - 1));
}

// Whole-sequence check of the contiguous layout (paged layouts are checked
// block by block in block_row).
__device__ __forceinline__ bool seq_rows_ok(const CacheRows& c, int b, int L, int64_t cache_tokens) {
    if (c.table != nullptr) return true;
    const int64_t start = c.starts[b];
    return start >= 0 && start + L <= cache_tokens;
}
#endif

// Per-(sequence, KV head, split) partial softmax state of decode attention:
// unnormalised output O[16][128], running max m[16] (log2 domain), sum l[16].
constexpr int kPartialFloats = 16 * 128 + 16 + 16;

struct ScanArgs {
    const CUtensorMap* ik_map;  // ik as (Di, KH, tokens), box 64 x 1 x 64, host copy
    int H;
    int ik_shared;              // 1: one index key per position for all heads (KH = 1), else KH = H
    const uint16_t* iq;
    const uint16_t* ik;
    const int32_t* cu_rows;
    const int32_t* cache_lens;
    CacheRows cache;
    int num_seqs;
    int total_rows;
    int max_cache_len;
    int64_t cache_tokens;
    int max_blocks;
    int rows_per_seq;     // RS = min(max_rows_per_seq, kDecodeMaxRows): pooled row slots per sequence
    int64_t unit_bound;   // upper bound of the number of work units
    float* pooled;        // [B * RS, H, max_blocks]: slot b * RS + i = row i of sequence b
    int32_t* clear_words; // zeroed by the scan (tickets of the attention kernel)
    int n_clear;
    int32_t* drow_prefix; // nullable: [B + 1] prefix of decode-family rows per sequence, written by CTA 0
    uint32_t* err;
};

struct DecodeAttendArgs {
    const CUtensorMap* k_map;  // host copies, passed by value to the kernel
    const CUtensorMap* v_map;
    const uint16_t* q;
    const float* pooled;       // fused path: pooled scores [B * RS, H, max_blocks] (nullptr when sel is given)
    int max_blocks;
    int rows_per_seq;          // RS: pooled slot of row i of sequence b = b * RS + i; grid z = B * RS slots
    const int32_t* drow_prefix;  // fused path, nullable: grid z = decode-family row z, its sequence found in
                                 // this prefix of rows per sequence (written by the scan)
    int decode_rows;             // with drow_prefix: the grid's z extent (host count of decode-family rows)
    const int32_t* sel_in;     // staged path: given selection
    const int32_t* nsel_in;
    const int32_t* cu_rows;
    const int32_t* cache_lens;
    CacheRows cache;
    int num_seqs, H, G, top_k, total_rows, max_cache_len;
    int64_t cache_tokens;
    float scale_log2;          // softmax scale * log2(e)
    int kv_int8;               // 1: k, v are int8 [T, H, D] with fp32 scales [T, H]; 2: k, v are the
                               // int8 values widened to bf16 [T, H, D] (run_widen_kv), scales [H, T]
    const float* k_scale;
    const float* v_scale;
    void* out;
    int out_bf16;
    float* partials;           // [B, H, top_k, kPartialFloats]
    int32_t* tickets;          // [B, H], zero on entry
    int32_t* sel_out;          // nullable
    int32_t* nsel_out;         // nullable
    uint32_t* err;
};

struct StagedArgs {
    int H, G, top_k, num_seqs, total_rows, max_cache_len;
    int ik_shared;  // index keys per position: 1 (shared) or H
    int64_t cache_tokens;
    const int32_t* cu_rows;
    const int32_t* cache_lens;
    CacheRows cache;
};

struct PrefillIndexArgs {
    const CUtensorMap* iq_map;  // iq as (Di, H, rows)
    const CUtensorMap* ik_map;  // ik as (Di, KH, tokens), box 64 x 1 x 256 (64 x 1 x 64 when paged)
    int ik_shared;              // KH = 1: every head reads key head 0
    const int32_t* cu_rows;
    const int32_t* cache_lens;
    CacheRows cache;
    int num_seqs, H, top_k, total_rows, max_rows_per_seq, max_cache_len;
    int64_t cache_tokens;
    int32_t* sel;   // [R, H, top_k]
    int32_t* nsel;  // [R, H]
    int nsplit;         // position-range splits per (row tile, head); 1 = no merge
    uint64_t* cand;     // nsplit > 1: [R, H, nsplit, 15] best (pooled score, block) keys of each split
    int32_t* tickets;   // nsplit > 1: [tile bound, H] arrivals, zero on entry
    uint32_t* err;
};

constexpr int kIdxMaxSplit = 8;  // most position-range splits of the prompt-chunk indexer

struct PrefillAttendArgs {
    const CUtensorMap* q_map;  // q as (D, H*G, rows)
    const CUtensorMap* k_map;  // k as (D, H, tokens)
    const CUtensorMap* v_map;
    const int32_t* sel;
    const int32_t* nsel;
    const int32_t* cu_rows;
    const int32_t* cache_lens;
    CacheRows cache;
    int num_seqs, H, G, top_k, total_rows, max_rows_per_seq, max_cache_len;
    int64_t cache_tokens;
    float scale_log2;
    int kv_int8;               // 1: k, v are int8 [T, H, D] with fp32 scales [T, H]
    const float* k_scale;
    const float* v_scale;
    void* out;
    int out_bf16;
    int only_multi_row;  // 1: skip decode-family sequences (<= kDecodeMaxRows rows; fused path)
    uint32_t* err;
};

// int8 caches, prompt chunks: the positions of every sequence the prompt-chunk
// attention reads, widened once into a contiguous bf16 copy with the scales
// beside it (sequence b at row wide_starts[b] = slot_b * slot_rows).
constexpr int kWidenMaxSeqs = 8192;  // the slot prefix is kept in shared memory (4 bytes a sequence)
struct WidenArgs {
    const uint8_t* k8;  // int8 caches [T, H, D]
    const uint8_t* v8;
    const float* k_scale;  // [T, H]
    const float* v_scale;
    const int32_t* cu_rows;
    const int32_t* cache_lens;
    CacheRows cache;
    int num_seqs, H, max_cache_len;
    int64_t cache_tokens;
    int only_multi_row;  // 1: sequences with more than kDecodeMaxRows rows only (fused path); 0: all
    int max_slots;       // sequences the copy has room for
    int slot_rows;       // rows per slot: max_cache_len rounded up to a multiple of kBlock
    uint16_t* kw;        // bf16 [max_slots * slot_rows, H, D]
    uint16_t* vw;
    float* ksw;          // [H, max_slots * slot_rows] (head-major)
    float* vsw;
    int64_t* wide_starts;  // [num_seqs]
    uint32_t* err;
};
cudaError_t run_widen_kv(const WidenArgs& a, cudaStream_t stream);

// Allocation-free decode attention: scratch in a file-scope device array
// sized for at most kNoAllocMaxPairs (sequence, KV head) pairs per call.
constexpr int kNoAllocMaxPairs = 32;
cudaError_t run_decode_attend_noalloc(DecodeAttendArgs a, cudaStream_t stream);

cudaError_t run_decode_scan(const ScanArgs& a, cudaStream_t stream);
cudaError_t run_decode_attend(const DecodeAttendArgs& a, cudaStream_t stream);  // ticket combine through global memory
// Cluster form (combine through distributed shared memory); after_scan: launch
// as a programmatic dependent of the index scan that precedes it.
cudaError_t run_decode_cluster(const DecodeAttendArgs& a, bool after_scan, cudaStream_t stream);
cudaError_t run_index_scores(const StagedArgs& a, const uint16_t* iq, const uint16_t* ik, float* scores,
                             int64_t ld, cudaStream_t stream);
cudaError_t run_select_blocks(const StagedArgs& a, const float* scores, int64_t ld, int32_t* sel, int32_t* nsel,
                              cudaStream_t stream);
cudaError_t run_prefill_index(const PrefillIndexArgs& a, bool after_decode, cudaStream_t stream);
cudaError_t run_prefill_attend(const PrefillAttendArgs& a, cudaStream_t stream);
cudaError_t run_wait_timeout_check(uint32_t* err, uint64_t limit_ns, cudaStream_t stream);

int device_sm_count();

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the driver call is made only when the limit grows.
cudaError_t ensure_smem_limit(const void* kernel, size_t bytes);

}  // namespace msa
