// C ABI of the MSA hot path: argument checks, workspace layout, TMA tensor
// maps and the launch sequence.  See include/msa.h for the contract.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/msa.h"
#include "common.cuh"
#include "internal.h"

namespace {

thread_local std::string g_last_error;

msa_status fail(msa_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

msa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kMaxCacheLen = int64_t(1) << 21;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side validation shared by every entry point.
msa_status check_problem(const msa_problem* p) {
    if (p == nullptr) return fail(MSA_ERR_INVALID_ARG, "problem is null");
    if (p->num_seqs < 1) return fail(MSA_ERR_INVALID_ARG, "num_seqs must be >= 1 (got %d)", p->num_seqs);
    if (p->num_seqs > 4096) return fail(MSA_ERR_UNSUPPORTED, "num_seqs > 4096");
    if (p->head_dim != msa::kHeadDim) return fail(MSA_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", p->head_dim);
    if (p->index_dim != msa::kIndexDim)
        return fail(MSA_ERR_UNSUPPORTED, "index_dim must be 64 (got %d)", p->index_dim);
    if (p->block_size != msa::kBlock) return fail(MSA_ERR_UNSUPPORTED, "block_size must be 64 (got %d)", p->block_size);
    if (p->top_k < 1) return fail(MSA_ERR_INVALID_ARG, "top_k must be >= 1 (got %d)", p->top_k);
    if (p->top_k > msa::kMaxTopK) return fail(MSA_ERR_UNSUPPORTED, "top_k must be <= 16 (got %d)", p->top_k);
    if (p->group_size < 1) return fail(MSA_ERR_INVALID_ARG, "group_size must be >= 1");
    if (p->group_size > msa::kMaxGroup) return fail(MSA_ERR_UNSUPPORTED, "group_size must be <= 16");
    const int H = p->num_kv_heads;
    if (H < 1) return fail(MSA_ERR_INVALID_ARG, "num_kv_heads must be >= 1");
    if (!(H == 1 || H == 2 || H == 4 || H == 8)) return fail(MSA_ERR_UNSUPPORTED, "num_kv_heads must be 1, 2, 4 or 8");
    if (!std::isfinite(p->softmax_scale) || p->softmax_scale < 0.f)
        return fail(MSA_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
    if (p->out_dtype != MSA_OUT_F32 && p->out_dtype != MSA_OUT_BF16) return fail(MSA_ERR_INVALID_ARG, "bad out_dtype");
    if (p->total_rows < p->num_seqs) return fail(MSA_ERR_INVALID_ARG, "total_rows < num_seqs");
    if (p->max_rows_per_seq < 1 || p->max_rows_per_seq > p->total_rows)
        return fail(MSA_ERR_INVALID_ARG, "max_rows_per_seq out of range");
    if (p->max_cache_len < p->max_rows_per_seq) return fail(MSA_ERR_INVALID_ARG, "max_cache_len < max_rows_per_seq");
    if (p->max_cache_len > kMaxCacheLen) return fail(MSA_ERR_UNSUPPORTED, "max_cache_len > 2^21");
    if (p->cache_tokens < 1 || p->cache_tokens > INT32_MAX) return fail(MSA_ERR_INVALID_ARG, "cache_tokens out of range");
    if (p->num_decode_seqs < -1 || p->num_decode_seqs > p->num_seqs)
        return fail(MSA_ERR_INVALID_ARG, "num_decode_seqs out of range");
    if (p->max_rows_per_seq <= msa::kDecodeMaxRows && p->num_decode_seqs != -1 && p->num_decode_seqs != p->num_seqs)
        return fail(MSA_ERR_INVALID_ARG, "max_rows_per_seq <= 8 implies num_decode_seqs == num_seqs");
    if (!p->cu_rows || !p->cache_lens) return fail(MSA_ERR_INVALID_ARG, "device metadata is null");
    if ((reinterpret_cast<uintptr_t>(p->cu_rows) & 3u) || (reinterpret_cast<uintptr_t>(p->cache_lens) & 3u))
        return fail(MSA_ERR_INVALID_ARG, "cu_rows or cache_lens is not 4-byte aligned");
    if (p->kv_dtype != MSA_KV_BF16 && p->kv_dtype != MSA_KV_INT8)
        return fail(MSA_ERR_INVALID_ARG, "kv_dtype must be MSA_KV_BF16 or MSA_KV_INT8 (got %d)", p->kv_dtype);
    if (p->kv_dtype == MSA_KV_INT8) {
        if (!p->k_scale || !p->v_scale) return fail(MSA_ERR_INVALID_ARG, "an int8 cache needs k_scale and v_scale");
        if ((reinterpret_cast<uintptr_t>(p->k_scale) & 3u) || (reinterpret_cast<uintptr_t>(p->v_scale) & 3u))
            return fail(MSA_ERR_INVALID_ARG, "k_scale or v_scale is not 4-byte aligned");
    }
    if (p->num_decode_rows > p->total_rows)
        return fail(MSA_ERR_INVALID_ARG, "num_decode_rows > total_rows");
    if (p->num_decode_rows > 0 && p->num_decode_seqs >= 0 &&
        (p->num_decode_rows < p->num_decode_seqs ||
         static_cast<int64_t>(p->num_decode_rows) > static_cast<int64_t>(p->num_decode_seqs) * msa::kDecodeMaxRows))
        return fail(MSA_ERR_INVALID_ARG, "num_decode_rows must lie in [num_decode_seqs, 8 x num_decode_seqs]");
    if (p->index_key_heads != 0 && p->index_key_heads != 1 && p->index_key_heads != H)
        return fail(MSA_ERR_INVALID_ARG, "index_key_heads must be 0, 1 or num_kv_heads (got %d)", p->index_key_heads);
    if (p->block_table == nullptr) {
        if (!p->cache_starts) return fail(MSA_ERR_INVALID_ARG, "cache_starts is null (and no block table)");
        if (reinterpret_cast<uintptr_t>(p->cache_starts) & 7u) return fail(MSA_ERR_INVALID_ARG, "cache_starts misaligned");
    } else {
        const int32_t ps = p->page_size;
        if (ps < msa::kBlock || ps > (1 << 20) || (ps & (ps - 1)) != 0)
            return fail(MSA_ERR_UNSUPPORTED, "page_size must be a power of two in [64, 2^20] (got %d)", ps);
        if (p->cache_tokens % ps != 0) return fail(MSA_ERR_INVALID_ARG, "cache_tokens must be a multiple of page_size");
        if (static_cast<int64_t>(p->block_table_stride) * ps < p->max_cache_len)
            return fail(MSA_ERR_INVALID_ARG, "block_table_stride * page_size < max_cache_len");
        if (reinterpret_cast<uintptr_t>(p->block_table) & 3u) return fail(MSA_ERR_INVALID_ARG, "block_table misaligned");
    }
    return MSA_OK;
}

msa_status check_ptr(const void* ptr, const char* name) {
    if (ptr == nullptr) return fail(MSA_ERR_INVALID_ARG, "%s is null", name);
    if (!aligned16(ptr)) return fail(MSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return MSA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// 1 when one index key per position serves every KV head.
int ik_shared(const msa_problem* p) { return p->index_key_heads == 1 && p->num_kv_heads > 1 ? 1 : 0; }

msa::CacheRows cache_rows_of(const msa_problem* p) {
    msa::CacheRows c{};
    c.starts = p->cache_starts;
    c.table = p->block_table;
    if (c.table != nullptr) {
        c.stride = p->block_table_stride;
        int shift = 0;
        while ((1 << shift) < p->page_size) ++shift;
        c.page_shift = shift;
        c.num_pages = p->cache_tokens / p->page_size;
    }
    return c;
}

struct Layout {
    size_t err = 0, tickets = 0, idx_tickets = 0, pooled = 0, partials = 0, sel = 0, nsel = 0, idx_cand = 0,
           drow_prefix = 0, wide_starts = 0, wide_k = 0, wide_v = 0, wide_ks = 0, wide_vs = 0, total = 0;
    size_t header_bytes = 0;  // error word + tickets, cleared at the start of a call
};

// int8 caches, prompt-chunk attention: the sequences' keys and values are widened once per call
// into the workspace (run_widen_kv) when each widened position serves at least four kept key rows
// on average (every row may keep top_k blocks); otherwise the attention widens the int8 tiles it
// loads.  The sequences read are those with more than 8 rows (msa_forward: at most R / 9 of them,
// and num_seqs - num_decode_seqs when that count is given) or all of them (msa_attend_prefill).
constexpr int64_t kWidenMaxBytes = int64_t{8} << 30;
struct WidenPlan {
    bool on = false;
    int64_t slots = 0, slot_rows = 0;
};
int64_t widen_bytes_per_row(const msa_problem* p) {  // K and V bf16, two fp32 scales, per cache row
    return static_cast<int64_t>(p->num_kv_heads) * (2 * msa::kHeadDim * 2 + 2 * 4);
}
WidenPlan widen_plan(const msa_problem* p, bool only_multi_row) {
    WidenPlan w;
    if (p->kv_dtype != MSA_KV_INT8 || p->num_seqs > msa::kWidenMaxSeqs) return w;
    int64_t n = p->num_seqs;
    if (only_multi_row) {
        if (p->num_decode_seqs >= 0) n = std::min<int64_t>(n, p->num_seqs - p->num_decode_seqs);
        n = std::min<int64_t>(n, p->total_rows / (msa::kDecodeMaxRows + 1));
    } else {
        n = std::min<int64_t>(n, p->total_rows);
    }
    w.slots = n;
    w.slot_rows = (static_cast<int64_t>(p->max_cache_len) + msa::kBlock - 1) / msa::kBlock * msa::kBlock;
    if (n < 1) return w;
    const int64_t kept_rows = static_cast<int64_t>(p->total_rows) * p->top_k * msa::kBlock;
    w.on = kept_rows >= 4 * n * w.slot_rows && n * w.slot_rows * widen_bytes_per_row(p) <= kWidenMaxBytes;
    return w;
}

// Upper bound of the prompt-chunk indexer's row tiles (128 rows each).
int64_t index_tile_bound(const msa_problem* p) { return (p->total_rows + 127) / 128 + p->num_seqs; }

// Pooled-score row slots per sequence of the decode family.
size_t decode_rows_per_seq(const msa_problem* p) {
    return static_cast<size_t>(p->max_rows_per_seq < msa::kDecodeMaxRows ? p->max_rows_per_seq : msa::kDecodeMaxRows);
}

Layout layout_of(const msa_problem* p) {
    Layout l;
    const size_t B = p->num_seqs, H = p->num_kv_heads, R = p->total_rows, K = p->top_k;
    const size_t RS = decode_rows_per_seq(p);
    const size_t MB = (static_cast<size_t>(p->max_cache_len) + msa::kBlock - 1) / msa::kBlock;
    size_t off = 0;
    l.err = off;
    off += 16;
    l.tickets = off;
    off += B * H * sizeof(int32_t);
    l.idx_tickets = off;  // prompt-chunk indexer: arrivals per (row tile, head)
    off += (static_cast<size_t>(index_tile_bound(p)) * H) * sizeof(int32_t);
    l.header_bytes = off;
    off = align256(off);
    l.pooled = off;
    off = align256(off + B * RS * H * MB * sizeof(float));
    l.partials = off;  // none: decode partials are combined on chip (thread-block clusters)
    l.sel = off;
    off = align256(off + R * H * K * sizeof(int32_t));
    l.nsel = off;
    off = align256(off + R * H * sizeof(int32_t));
    l.idx_cand = off;  // prompt-chunk indexer: per-split top-15 lists
    if (p->max_rows_per_seq > msa::kDecodeMaxRows && p->num_decode_seqs != p->num_seqs)
        off = align256(off + R * H * msa::kIdxMaxSplit * 15 * sizeof(uint64_t));
    l.drow_prefix = off;  // decode-family rows per sequence, prefix (compact decode attention grid)
    off = align256(off + (B + 1) * sizeof(int32_t));
    // int8 caches, prompt chunks widened once per call: room for the larger of the two entry points' plans
    const WidenPlan wf = widen_plan(p, true), wa = widen_plan(p, false);
    const size_t wrows = static_cast<size_t>(std::max(wf.on ? wf.slots * wf.slot_rows : 0, wa.on ? wa.slots * wa.slot_rows : 0));
    l.wide_starts = off;
    if (wrows > 0) {
        off = align256(off + B * sizeof(int64_t));
        l.wide_k = off;
        off = align256(off + wrows * H * msa::kHeadDim * 2);
        l.wide_v = off;
        off = align256(off + wrows * H * msa::kHeadDim * 2);
        l.wide_ks = off;
        off = align256(off + wrows * H * sizeof(float));
        l.wide_vs = off;
        off = align256(off + wrows * H * sizeof(float));
    }
    l.total = off;
    return l;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 3-D tensor (d0 innermost, contiguous) of bf16 (elem_bytes 2) or one-byte
// elements with a box of b0 x b1 x b2 and 128-byte swizzle (b0 * elem_bytes
// must be 128).
msa_status make_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
                    uint32_t b1, uint32_t b2, const char* name, int elem_bytes = 2) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * elem_bytes, d0 * d1 * elem_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MSA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, int(r));
    return MSA_OK;
}

msa::StagedArgs staged_args(const msa_problem* p) {
    msa::StagedArgs a;
    a.H = p->num_kv_heads;
    a.G = p->group_size;
    a.top_k = p->top_k;
    a.num_seqs = p->num_seqs;
    a.total_rows = p->total_rows;
    a.max_cache_len = p->max_cache_len;
    a.cache_tokens = p->cache_tokens;
    a.ik_shared = ik_shared(p);
    a.cu_rows = p->cu_rows;
    a.cache_lens = p->cache_lens;
    a.cache = cache_rows_of(p);
    return a;
}

float scale_log2(const msa_problem* p) { return p->softmax_scale * 1.4426950408889634f; }

struct Marks {
    void* const* events;
    int n;
    cudaStream_t stream;
    msa_status mark(int i) {
        if (events && i < n && events[i]) {
            // inside a stream capture, record an event node of the graph so the
            // mark is taken at every replay
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            cudaError_t e = cudaStreamIsCapturing(stream, &cs);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
            e = cudaEventRecordWithFlags(static_cast<cudaEvent_t>(events[i]), stream,
                                         cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                             : cudaEventRecordDefault);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        }
        return MSA_OK;
    }
};

// Key or value cache map for the attention kernels: bf16 boxes of 64 dims x
// 64 tokens (two per block), or int8 boxes of all 128 dims x 64 tokens.
msa_status kv_map(CUtensorMap* map, const msa_problem* p, const void* base, const char* name) {
    const uint64_t T = p->cache_tokens, H = p->num_kv_heads;
    if (p->kv_dtype == MSA_KV_INT8) return make_map(map, base, 128, H, T, 128, 1, 64, name, 1);
    return make_map(map, base, 128, H, T, 64, 1, 64, name);
}

bool decode_family(const msa_problem* p) { return p->num_decode_seqs != 0; }

// The decode attention's grid covers the host's count of decode-family rows
// (when given and smaller than the row slots) instead of every row slot.
bool compact_decode_grid(const msa_problem* p) {
    return p->num_decode_rows > 0 &&
           static_cast<int64_t>(p->num_decode_rows) < static_cast<int64_t>(p->num_seqs) * decode_rows_per_seq(p);
}
bool prefill_family(const msa_problem* p) {
    return p->max_rows_per_seq > msa::kDecodeMaxRows && p->num_decode_seqs != p->num_seqs;
}

}  // namespace

int msa::device_sm_count() {
    static int counts[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& c = counts[dev & 63];
    if (c == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        c = v > 0 ? v : 1;
    }
    return c;
}

cudaError_t msa::ensure_smem_limit(const void* kernel, size_t bytes) {
    struct Entry {
        const void* kernel;
        int device;
        size_t bytes;
    };
    static std::mutex mu;
    static Entry table[256];
    static int used = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (table[i].kernel == kernel && table[i].device == dev) {
            if (table[i].bytes >= bytes) return cudaSuccess;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
            if (e == cudaSuccess) table[i].bytes = bytes;
            return e;
        }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && used < 256) table[used++] = Entry{kernel, dev, bytes};
    return e;
}

extern "C" {

const char* msa_status_string(msa_status s) {
    switch (s) {
        case MSA_OK: return "MSA_OK";
        case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
        case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
        case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
        case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
        case MSA_ERR_INTERNAL: return "MSA_ERR_INTERNAL";
    }
    return "MSA_ERR_UNKNOWN";
}

const char* msa_last_error(void) { return g_last_error.c_str(); }

msa_status msa_workspace_size(const msa_problem* p, size_t* bytes) {
    g_last_error.clear();
    msa_status s = check_problem(p);
    if (s != MSA_OK) return s;
    if (!bytes) return fail(MSA_ERR_INVALID_ARG, "bytes is null");
    *bytes = layout_of(p).total;
    return MSA_OK;
}

msa_status msa_index_scores(const msa_problem* p, const void* iq, const void* ik_cache, float* scores, int64_t ld,
                            void* stream) {
    g_last_error.clear();
    msa_status s;
    if ((s = check_problem(p)) != MSA_OK) return s;
    if ((s = check_ptr(iq, "iq")) != MSA_OK || (s = check_ptr(ik_cache, "ik_cache")) != MSA_OK ||
        (s = check_ptr(scores, "scores")) != MSA_OK)
        return s;
    if (ld < p->max_cache_len) return fail(MSA_ERR_INVALID_ARG, "ld < max_cache_len");
    cudaError_t e = msa::run_index_scores(staged_args(p), static_cast<const uint16_t*>(iq),
                                          static_cast<const uint16_t*>(ik_cache), scores, ld,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "index scores launch");
}

msa_status msa_select_blocks(const msa_problem* p, const float* scores, int64_t ld, int32_t* sel, int32_t* nsel,
                             void* stream) {
    g_last_error.clear();
    msa_status s;
    if ((s = check_problem(p)) != MSA_OK) return s;
    if ((s = check_ptr(scores, "scores")) != MSA_OK || (s = check_ptr(sel, "sel")) != MSA_OK ||
        (s = check_ptr(nsel, "nsel")) != MSA_OK)
        return s;
    if (ld < p->max_cache_len) return fail(MSA_ERR_INVALID_ARG, "ld < max_cache_len");
    cudaError_t e = msa::run_select_blocks(staged_args(p), scores, ld, sel, nsel, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "select blocks launch");
}

static msa_status check_workspace(const msa_problem* p, const void* ws, size_t ws_bytes, Layout* l) {
    *l = layout_of(p);
    if (ws == nullptr) return fail(MSA_ERR_WORKSPACE, "workspace is null");
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(MSA_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    if (ws_bytes < l->total) return fail(MSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, l->total);
    return MSA_OK;
}

static msa_status attend_common(const msa_problem* p, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* sel, const int32_t* nsel, void* out, void* ws, size_t ws_bytes,
                                Layout* l) {
    msa_status s;
    if ((s = check_problem(p)) != MSA_OK) return s;
    if ((s = check_ptr(q, "q")) != MSA_OK || (s = check_ptr(k_cache, "k_cache")) != MSA_OK ||
        (s = check_ptr(v_cache, "v_cache")) != MSA_OK || (s = check_ptr(sel, "sel")) != MSA_OK ||
        (s = check_ptr(nsel, "nsel")) != MSA_OK || (s = check_ptr(out, "out")) != MSA_OK)
        return s;
    return check_workspace(p, ws, ws_bytes, l);
}

static msa::DecodeAttendArgs decode_args(const msa_problem* p, const CUtensorMap* km, const CUtensorMap* vm,
                                         const void* q, void* out, uint8_t* ws, const Layout& l) {
    msa::DecodeAttendArgs a{};
    a.k_map = km;
    a.v_map = vm;
    a.q = static_cast<const uint16_t*>(q);
    a.max_blocks = static_cast<int>((p->max_cache_len + msa::kBlock - 1) / msa::kBlock);
    a.rows_per_seq = static_cast<int>(decode_rows_per_seq(p));
    a.cu_rows = p->cu_rows;
    a.cache_lens = p->cache_lens;
    a.cache = cache_rows_of(p);
    a.num_seqs = p->num_seqs;
    a.H = p->num_kv_heads;
    a.G = p->group_size;
    a.top_k = p->top_k;
    a.total_rows = p->total_rows;
    a.max_cache_len = p->max_cache_len;
    a.cache_tokens = p->cache_tokens;
    a.scale_log2 = scale_log2(p);
    a.kv_int8 = p->kv_dtype == MSA_KV_INT8;
    a.k_scale = a.kv_int8 ? p->k_scale : nullptr;
    a.v_scale = a.kv_int8 ? p->v_scale : nullptr;
    a.out = out;
    a.out_bf16 = p->out_dtype == MSA_OUT_BF16;
    a.partials = nullptr;  // the cluster kernel keeps its partials in distributed shared memory
    a.tickets = reinterpret_cast<int32_t*>(ws + l.tickets);
    a.err = reinterpret_cast<uint32_t*>(ws + l.err);
    return a;
}

msa_status msa_attend_decode(const msa_problem* p, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* sel, const int32_t* nsel, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    g_last_error.clear();
    Layout l;
    msa_status s = attend_common(p, q, k_cache, v_cache, sel, nsel, out, workspace, workspace_bytes, &l);
    if (s != MSA_OK) return s;
    if (p->max_rows_per_seq > msa::kDecodeMaxRows)
        return fail(MSA_ERR_INVALID_ARG, "msa_attend_decode needs at most 8 rows per sequence (max_rows_per_seq <= 8)");
    CUtensorMap km, vm;
    if ((s = kv_map(&km, p, k_cache, "k_cache")) != MSA_OK) return s;
    if ((s = kv_map(&vm, p, v_cache, "v_cache")) != MSA_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, l.header_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    msa::DecodeAttendArgs a = decode_args(p, &km, &vm, q, out, ws, l);
    a.pooled = nullptr;
    a.sel_in = sel;
    a.nsel_in = nsel;
    e = msa::run_decode_cluster(a, false, st);
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "decode attention launch");
}

static msa::PrefillAttendArgs prefill_attend_args(const msa_problem* p, const CUtensorMap* qm, const CUtensorMap* km,
                                                  const CUtensorMap* vm, const int32_t* sel, const int32_t* nsel,
                                                  void* out, uint8_t* ws, const Layout& l) {
    msa::PrefillAttendArgs a{};
    a.q_map = qm;
    a.k_map = km;
    a.v_map = vm;
    a.sel = sel;
    a.nsel = nsel;
    a.cu_rows = p->cu_rows;
    a.cache_lens = p->cache_lens;
    a.cache = cache_rows_of(p);
    a.num_seqs = p->num_seqs;
    a.H = p->num_kv_heads;
    a.G = p->group_size;
    a.top_k = p->top_k;
    a.total_rows = p->total_rows;
    a.max_rows_per_seq = p->max_rows_per_seq;
    a.max_cache_len = p->max_cache_len;
    a.cache_tokens = p->cache_tokens;
    a.scale_log2 = scale_log2(p);
    a.kv_int8 = p->kv_dtype == MSA_KV_INT8;
    a.k_scale = a.kv_int8 ? p->k_scale : nullptr;
    a.v_scale = a.kv_int8 ? p->v_scale : nullptr;
    a.out = out;
    a.out_bf16 = p->out_dtype == MSA_OUT_BF16;
    a.err = reinterpret_cast<uint32_t*>(ws + l.err);
    return a;
}

static msa_status attention_maps(const msa_problem* p, const void* q, const void* k, const void* v, CUtensorMap* qm,
                                 CUtensorMap* km, CUtensorMap* vm) {
    const uint64_t R = p->total_rows;
    const uint64_t HQ = static_cast<uint64_t>(p->num_kv_heads) * p->group_size;
    msa_status s;
    if (qm && (s = make_map(qm, q, 128, HQ, R, 64, 16, 1, "q")) != MSA_OK) return s;
    if ((s = kv_map(km, p, k, "k_cache")) != MSA_OK) return s;
    return kv_map(vm, p, v, "v_cache");
}

// Widens the int8 keys and values of the sequences the prompt-chunk attention reads into the
// workspace (enqueued on `st`) and points the attention's arguments at the copy: bf16 maps
// (*km, *vm), its rows, its scales.
static msa_status widen_for_attention(const msa_problem* p, const WidenPlan& w, bool only_multi_row,
                                      const void* k_cache, const void* v_cache, uint8_t* ws, const Layout& l,
                                      CUtensorMap* km, CUtensorMap* vm, msa::PrefillAttendArgs* a, cudaStream_t st) {
    msa::WidenArgs wa{};
    wa.k8 = static_cast<const uint8_t*>(k_cache);
    wa.v8 = static_cast<const uint8_t*>(v_cache);
    wa.k_scale = p->k_scale;
    wa.v_scale = p->v_scale;
    wa.cu_rows = p->cu_rows;
    wa.cache_lens = p->cache_lens;
    wa.cache = cache_rows_of(p);
    wa.num_seqs = p->num_seqs;
    wa.H = p->num_kv_heads;
    wa.max_cache_len = p->max_cache_len;
    wa.cache_tokens = p->cache_tokens;
    wa.only_multi_row = only_multi_row ? 1 : 0;
    wa.max_slots = static_cast<int>(w.slots);
    wa.slot_rows = static_cast<int>(w.slot_rows);
    wa.kw = reinterpret_cast<uint16_t*>(ws + l.wide_k);
    wa.vw = reinterpret_cast<uint16_t*>(ws + l.wide_v);
    wa.ksw = reinterpret_cast<float*>(ws + l.wide_ks);
    wa.vsw = reinterpret_cast<float*>(ws + l.wide_vs);
    wa.wide_starts = reinterpret_cast<int64_t*>(ws + l.wide_starts);
    wa.err = reinterpret_cast<uint32_t*>(ws + l.err);
    const uint64_t T = static_cast<uint64_t>(w.slots * w.slot_rows), H = p->num_kv_heads;
    msa_status s;
    if ((s = make_map(km, wa.kw, 128, H, T, 64, 1, 64, "widened k")) != MSA_OK) return s;
    if ((s = make_map(vm, wa.vw, 128, H, T, 64, 1, 64, "widened v")) != MSA_OK) return s;
    cudaError_t e = msa::run_widen_kv(wa, st);
    if (e != cudaSuccess) return cuda_fail(e, "key/value widening launch");
    a->k_map = km;
    a->v_map = vm;
    a->cache = msa::CacheRows{};
    a->cache.starts = wa.wide_starts;
    a->cache_tokens = static_cast<int64_t>(T);
    a->kv_int8 = 2;
    a->k_scale = wa.ksw;
    a->v_scale = wa.vsw;
    return MSA_OK;
}

msa_status msa_attend_prefill(const msa_problem* p, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* sel, const int32_t* nsel, void* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
    g_last_error.clear();
    Layout l;
    msa_status s = attend_common(p, q, k_cache, v_cache, sel, nsel, out, workspace, workspace_bytes, &l);
    if (s != MSA_OK) return s;
    CUtensorMap qm, km, vm;
    if ((s = attention_maps(p, q, k_cache, v_cache, &qm, &km, &vm)) != MSA_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, l.header_bytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    msa::PrefillAttendArgs a = prefill_attend_args(p, &qm, &km, &vm, sel, nsel, out, ws, l);
    a.only_multi_row = 0;
    const WidenPlan w = widen_plan(p, false);
    CUtensorMap kwm, vwm;
    if (w.on && (s = widen_for_attention(p, w, false, k_cache, v_cache, ws, l, &kwm, &vwm, &a, st)) != MSA_OK) return s;
    e = msa::run_prefill_attend(a, st);
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "prefill attention launch");
}

msa_status msa_attend_decode_noalloc(const msa_problem* p, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* sel, const int32_t* nsel, void* out, void* stream) {
    g_last_error.clear();
    msa_status s;
    if ((s = check_problem(p)) != MSA_OK) return s;
    if ((s = check_ptr(q, "q")) != MSA_OK || (s = check_ptr(k_cache, "k_cache")) != MSA_OK ||
        (s = check_ptr(v_cache, "v_cache")) != MSA_OK || (s = check_ptr(sel, "sel")) != MSA_OK ||
        (s = check_ptr(nsel, "nsel")) != MSA_OK || (s = check_ptr(out, "out")) != MSA_OK)
        return s;
    if (p->max_rows_per_seq != 1)
        return fail(MSA_ERR_INVALID_ARG, "msa_attend_decode_noalloc needs one row per sequence (max_rows_per_seq == 1)");
    if (p->kv_dtype != MSA_KV_BF16)
        return fail(MSA_ERR_UNSUPPORTED, "msa_attend_decode_noalloc takes bf16 key/value caches only");
    const int64_t pairs = static_cast<int64_t>(p->num_seqs) * p->num_kv_heads;
    if (pairs > msa::kNoAllocMaxPairs)
        return fail(MSA_ERR_UNSUPPORTED,
                    "msa_attend_decode_noalloc: num_seqs * num_kv_heads = %lld exceeds its fixed scratch of %d "
                    "(sequence, KV head) pairs; use msa_attend_decode with a workspace",
                    static_cast<long long>(pairs), msa::kNoAllocMaxPairs);
    const uint64_t T = p->cache_tokens, H = p->num_kv_heads;
    CUtensorMap km, vm;
    if ((s = make_map(&km, k_cache, 128, H, T, 64, 1, 64, "k_cache")) != MSA_OK) return s;
    if ((s = make_map(&vm, v_cache, 128, H, T, 64, 1, 64, "v_cache")) != MSA_OK) return s;
    Layout unused;
    msa::DecodeAttendArgs a = decode_args(p, &km, &vm, q, out, nullptr, unused);
    a.pooled = nullptr;
    a.sel_in = sel;
    a.nsel_in = nsel;
    cudaError_t e = msa::run_decode_attend_noalloc(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "allocation-free decode attention");
}

int32_t msa_forward_launches(const msa_problem* p) {
    if (check_problem(p) != MSA_OK) return -1;
    return (decode_family(p) ? 2 : 0) + (prefill_family(p) ? (widen_plan(p, true).on ? 3 : 2) : 0);
}

msa_status msa_forward_marked(const msa_problem* p, const void* q, const void* iq, const void* k_cache,
                              const void* v_cache, const void* ik_cache, void* out, int32_t* sel_out,
                              int32_t* nsel_out, void* workspace, size_t workspace_bytes, void* stream,
                              void* const* events, int32_t n_events) {
    g_last_error.clear();
    msa_status s;
    if ((s = check_problem(p)) != MSA_OK) return s;
    if ((s = check_ptr(q, "q")) != MSA_OK || (s = check_ptr(iq, "iq")) != MSA_OK ||
        (s = check_ptr(k_cache, "k_cache")) != MSA_OK || (s = check_ptr(v_cache, "v_cache")) != MSA_OK ||
        (s = check_ptr(ik_cache, "ik_cache")) != MSA_OK || (s = check_ptr(out, "out")) != MSA_OK)
        return s;
    if ((sel_out == nullptr) != (nsel_out == nullptr))
        return fail(MSA_ERR_INVALID_ARG, "sel_out and nsel_out must both be given or both be null");
    if (sel_out && ((s = check_ptr(sel_out, "sel_out")) != MSA_OK || (s = check_ptr(nsel_out, "nsel_out")) != MSA_OK))
        return s;
    if (n_events < 0 || n_events > 5) return fail(MSA_ERR_INVALID_ARG, "n_events must be in [0, 5]");
    Layout l;
    if ((s = check_workspace(p, workspace, workspace_bytes, &l)) != MSA_OK) return s;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    Marks marks{events, n_events, st};
    const bool dec = decode_family(p), pre = prefill_family(p);
    int32_t* sel = sel_out ? sel_out : reinterpret_cast<int32_t*>(ws + l.sel);
    int32_t* nsel = nsel_out ? nsel_out : reinterpret_cast<int32_t*>(ws + l.nsel);
    const uint64_t T = p->cache_tokens, H = p->num_kv_heads;
    const uint64_t KH = ik_shared(p) ? 1 : H;  // index-key heads per position
    const int max_blocks = static_cast<int>((p->max_cache_len + msa::kBlock - 1) / msa::kBlock);

    CUtensorMap km, vm, qm, iqm, ikm;
    if ((s = attention_maps(p, q, k_cache, v_cache, pre ? &qm : nullptr, &km, &vm)) != MSA_OK) return s;
    if (pre) {
        if ((s = make_map(&iqm, iq, 64, H, p->total_rows, 64, 1, 128, "iq")) != MSA_OK) return s;
        // a whole 256-position tile per box, or one box per 64-position block when paged
        const uint32_t box = p->block_table == nullptr ? 256 : 64;
        if ((s = make_map(&ikm, ik_cache, 64, KH, T, 64, 1, box, "ik_cache")) != MSA_OK) return s;
    }
    CUtensorMap ik_scan;
    if (dec && (s = make_map(&ik_scan, ik_cache, 64, KH, T, 64, 1, 64, "ik_cache")) != MSA_OK) return s;
    if ((s = marks.mark(0)) != MSA_OK) return s;
    cudaError_t e;
    if (dec) {
        msa::ScanArgs sa{};
        sa.ik_map = &ik_scan;
        sa.H = p->num_kv_heads;
        sa.ik_shared = ik_shared(p);
        sa.iq = static_cast<const uint16_t*>(iq);
        sa.ik = static_cast<const uint16_t*>(ik_cache);
        sa.cu_rows = p->cu_rows;
        sa.cache_lens = p->cache_lens;
        sa.cache = cache_rows_of(p);
        sa.num_seqs = p->num_seqs;
        sa.total_rows = p->total_rows;
        sa.max_cache_len = p->max_cache_len;
        sa.cache_tokens = p->cache_tokens;
        sa.max_blocks = max_blocks;
        sa.rows_per_seq = static_cast<int>(decode_rows_per_seq(p));
        const int64_t nd = p->num_decode_seqs >= 0 ? p->num_decode_seqs : p->num_seqs;
        sa.unit_bound = nd * max_blocks;
        sa.pooled = reinterpret_cast<float*>(ws + l.pooled);
        sa.clear_words = reinterpret_cast<int32_t*>(ws + l.err);
        sa.n_clear = static_cast<int>(l.header_bytes / sizeof(int32_t));
        sa.drow_prefix = compact_decode_grid(p) ? reinterpret_cast<int32_t*>(ws + l.drow_prefix) : nullptr;
        sa.err = reinterpret_cast<uint32_t*>(ws + l.err);
        if ((e = msa::run_decode_scan(sa, st)) != cudaSuccess) return cuda_fail(e, "decode scan launch");
        if ((s = marks.mark(1)) != MSA_OK) return s;
        msa::DecodeAttendArgs da = decode_args(p, &km, &vm, q, out, ws, l);
        da.pooled = sa.pooled;
        da.max_blocks = max_blocks;
        da.sel_out = sel;
        da.nsel_out = nsel;
        da.drow_prefix = sa.drow_prefix;
        da.decode_rows = p->num_decode_rows;
        const bool pdl = events == nullptr || n_events < 2 || events[1] == nullptr;  // a mark in between breaks it
        if ((e = msa::run_decode_cluster(da, pdl, st)) != cudaSuccess) return cuda_fail(e, "decode attention launch");
        if ((s = marks.mark(2)) != MSA_OK) return s;
    } else {
        if ((e = cudaMemsetAsync(ws, 0, l.header_bytes, st)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
        if ((s = marks.mark(1)) != MSA_OK || (s = marks.mark(2)) != MSA_OK) return s;
    }
    if (pre) {
        msa::PrefillIndexArgs ia{};
        ia.iq_map = &iqm;
        ia.ik_map = &ikm;
        ia.cu_rows = p->cu_rows;
        ia.cache_lens = p->cache_lens;
        ia.cache = cache_rows_of(p);
        ia.num_seqs = p->num_seqs;
        ia.H = p->num_kv_heads;
        ia.ik_shared = ik_shared(p);
        ia.top_k = p->top_k;
        ia.total_rows = p->total_rows;
        ia.max_rows_per_seq = p->max_rows_per_seq;
        ia.max_cache_len = p->max_cache_len;
        ia.cache_tokens = p->cache_tokens;
        ia.sel = sel;
        ia.nsel = nsel;
        {  // position-range splits so that the indexer's CTAs fill the GPU
            const int64_t pre_seqs = p->num_decode_seqs >= 0 ? p->num_seqs - p->num_decode_seqs : p->num_seqs;
            const int64_t ctas = ((p->total_rows + 127) / 128 + pre_seqs) * p->num_kv_heads;
            const int64_t col_tiles = (p->max_cache_len + 255) / 256;
            int64_t ns = msa::device_sm_count() / (ctas > 0 ? ctas : 1);
            if (ns > col_tiles / 2) ns = col_tiles / 2;  // at least two 256-position tiles a split
            ia.nsplit = static_cast<int>(ns < 1 ? 1 : (ns > msa::kIdxMaxSplit ? msa::kIdxMaxSplit : ns));
        }
        ia.cand = reinterpret_cast<uint64_t*>(ws + l.idx_cand);
        ia.tickets = reinterpret_cast<int32_t*>(ws + l.idx_tickets);
        ia.err = reinterpret_cast<uint32_t*>(ws + l.err);
        // behind the decode attention (no mark in between) the indexer overlaps its tail
        const bool pdl = dec && (events == nullptr || n_events < 3 || events[2] == nullptr);
        if ((e = msa::run_prefill_index(ia, pdl, st)) != cudaSuccess) return cuda_fail(e, "prefill indexer launch");
        if ((s = marks.mark(3)) != MSA_OK) return s;
        msa::PrefillAttendArgs pa = prefill_attend_args(p, &qm, &km, &vm, sel, nsel, out, ws, l);
        pa.only_multi_row = 1;
        const WidenPlan w = widen_plan(p, true);
        CUtensorMap kwm, vwm;
        if (w.on && (s = widen_for_attention(p, w, true, k_cache, v_cache, ws, l, &kwm, &vwm, &pa, st)) != MSA_OK)
            return s;
        if ((e = msa::run_prefill_attend(pa, st)) != cudaSuccess) return cuda_fail(e, "prefill attention launch");
        if ((s = marks.mark(4)) != MSA_OK) return s;
    } else {
        if ((s = marks.mark(3)) != MSA_OK || (s = marks.mark(4)) != MSA_OK) return s;
    }
    return MSA_OK;
}

msa_status msa_check_wait_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_us, void* stream) {
    g_last_error.clear();
    msa_status s;
    if ((s = check_ptr(workspace, "workspace")) != MSA_OK) return s;
    if (workspace_bytes < sizeof(uint32_t)) return fail(MSA_ERR_WORKSPACE, "workspace smaller than the error word");
    if (limit_us < 1 || limit_us > 2000000) return fail(MSA_ERR_INVALID_ARG, "limit_us outside [1, 2000000]");
    cudaError_t e = msa::run_wait_timeout_check(static_cast<uint32_t*>(workspace), 1000ull * limit_us,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MSA_OK : cuda_fail(e, "wait check launch");
}

msa_status msa_forward(const msa_problem* p, const void* q, const void* iq, const void* k_cache,
                       const void* v_cache, const void* ik_cache, void* out, int32_t* sel_out, int32_t* nsel_out,
                       void* workspace, size_t workspace_bytes, void* stream) {
    return msa_forward_marked(p, q, iq, k_cache, v_cache, ik_cache, out, sel_out, nsel_out, workspace,
                              workspace_bytes, stream, nullptr, 0);
}

}  // extern "C"
