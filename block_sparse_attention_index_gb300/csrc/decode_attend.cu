// Decode stage 2b+3: block selection, attention over the kept blocks as split
// partials, and the log-sum-exp combine.
//
// PR #1388 "minimax_m3: a CUDA backend for MiniMax-M3.1-Flash ...", native
// Metal family commit: a decode row attends to its chosen blocks in partial
// results that are merged afterwards.  Here one CTA = one (sequence, KV head,
// kept block):
//   - it selects the kept blocks from the pooled index scores (every split
//     of a (sequence, head) computes the same selection; the pooled scores
//     are a few KB in L2), or reads a given selection;
//   - TMA stages its 64-key K and V block (2 x 16 KB, 128-byte swizzle) into
//     shared memory while the 16 query heads of the group are loaded;
//   - S = Q K^T and O = P V on mma.sync tensor cores (a decode block is 16 x
//     64 x 128: far too small for tcgen05 tiles, and HBM-bound anyway).  P
//     enters the bf16 MMA as P_hi + P_lo, both bf16 (P_lo = P - P_hi), so
//     the weights keep ~16 significant bits instead of bf16's 8;
//   - it writes (m, l, O) for its block; the last split to finish (atomic
//     ticket) combines the partials:  M = max_s m_s,  L = sum_s l_s 2^(m_s-M),
//     out = sum_s O_s 2^(m_s-M) / L.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace msa {

constexpr int kAttThreads = 128;

struct __align__(1024) DecodeSmem {
    uint16_t k[2][64 * 64];  // [dim half][key][64 dims], 128B-swizzled by TMA
    uint16_t v[2][64 * 64];
    uint16_t q[16 * 128];    // [head][dim], 16-byte chunks XOR-swizzled by row
    uint16_t p[2][16 * 64];  // [hi/lo][head][key], same swizzle
    float wmax[4][16];
    float wsum[4][16];
    float weight[kMaxTopK][16];
    float ml[kMaxTopK][32];  // per split: m[16] then l[16]
    uint64_t bar;
    int32_t sel[kMaxTopK];
    int32_t nsel;
    int32_t last;
    SelectSmem<kAttThreads> select;
};

// byte offset of 16-byte chunk c of row `row` in a tile whose rows are
// `row_bytes` long, chunks XOR-swizzled with the row's low 3 bits
__device__ __forceinline__ uint32_t swz(int row, int chunk, int row_bytes) {
    return row * row_bytes + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool kSelGiven>
__global__ void __launch_bounds__(kAttThreads) decode_attend_kernel(const __grid_constant__ CUtensorMap k_map,
                                                                    const __grid_constant__ CUtensorMap v_map,
                                                                    const DecodeAttendArgs a) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, G = a.G;

    const int r = a.cu_rows[b];
    if (a.cu_rows[b + 1] - r != 1) {  // not a one-row sequence: the host bound said every one is
        if (tid == 0 && split == 0) atomicOr(a.err, kErrBadMetadata);
        return;
    }
    const int L = a.cache_lens[b];
    if (r < 0 || r >= a.total_rows || L < 1 || L > a.max_cache_len || !seq_rows_ok(a.cache, b, L, a.cache_tokens)) {
        if (tid == 0 && split == 0) atomicOr(a.err, kErrBadMetadata);
        return;
    }
    const int p = L - 1;
    const int J = p / kBlock;

    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    // ---- selection
    if constexpr (kSelGiven) {
        const int nraw = a.nsel_in[static_cast<int64_t>(r) * H + h];  // the same in every thread
        if (nraw < 1 || nraw > a.top_k) {
            if (tid == 0 && split == 0) atomicOr(a.err, kErrBadMetadata);
            if (nraw < 1) {  // no kept block: the softmax is empty; split 0 writes zeros
                if (split == 0) {
                    const int64_t o0 = (static_cast<int64_t>(r) * H * G + static_cast<int64_t>(h) * G) * kHeadDim;
                    for (int i = tid; i < G * kHeadDim; i += kAttThreads) {
                        if (a.out_bf16)
                            reinterpret_cast<__nv_bfloat16*>(a.out)[o0 + i] = __float2bfloat16_rn(0.f);
                        else
                            reinterpret_cast<float*>(a.out)[o0 + i] = 0.f;
                    }
                }
                return;
            }
        }
        if (tid < kMaxTopK) sm.sel[tid] = tid < a.top_k ? a.sel_in[(static_cast<int64_t>(r) * H + h) * a.top_k + tid] : -1;
        if (tid == 0) sm.nsel = min(nraw, a.top_k);
        __syncthreads();
    } else {
        const float* pooled = a.pooled + (static_cast<int64_t>(b) * H + h) * a.max_blocks;
        const int n = cta_select<kAttThreads>(pooled, J, a.top_k, sm.sel, sm.select);
        if (tid == 0) sm.nsel = n;
        __syncthreads();
        if (split == 0 && a.sel_out != nullptr && tid < a.top_k) {
            a.sel_out[(static_cast<int64_t>(r) * H + h) * a.top_k + tid] = sm.sel[tid];
            if (tid == 0) a.nsel_out[static_cast<int64_t>(r) * H + h] = n;
        }
    }
    const int nsel = sm.nsel;
    if (split >= nsel) return;
    int blk = sm.sel[split];
    if (blk < 0 || blk > J) {  // a given selection outside the causal range
        if (tid == 0) atomicOr(a.err, kErrBadMetadata);
        blk = J;
    }

    // ---- stage K/V of the block (TMA) and the group's queries
    int64_t row0 = block_row(a.cache, b, static_cast<int64_t>(blk) * kBlock);
    if (row0 < 0) {  // page outside the pool
        if (tid == 0) atomicOr(a.err, kErrBadMetadata);
        row0 = 0;
    }
    const int tok0 = static_cast<int>(row0);
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.bar, 4 * 64 * 64 * 2);
        tma_load_3d(sm.k[0], &k_map, &sm.bar, 0, h, tok0);
        tma_load_3d(sm.k[1], &k_map, &sm.bar, 64, h, tok0);
        tma_load_3d(sm.v[0], &v_map, &sm.bar, 0, h, tok0);
        tma_load_3d(sm.v[1], &v_map, &sm.bar, 64, h, tok0);
    }
    {
        const uint16_t* qrow = a.q + (static_cast<int64_t>(r) * H * G + static_cast<int64_t>(h) * G) * kHeadDim;
        for (int c = tid; c < 16 * 16; c += kAttThreads) {  // 16 heads x 16 chunks of 8 dims
            const int g = c >> 4, ch = c & 15;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (g < G) val = *reinterpret_cast<const uint4*>(qrow + g * kHeadDim + ch * 8);
            *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sm.q) + swz(g, ch, 256)) = val;
        }
    }
    __syncthreads();
    const bool ok = mbar_wait(&sm.bar, 0, a.err);
    if (!ok) {  // the copy never landed (the error word says so): wait once more, bounded, so
        mbar_wait(&sm.bar, 0, nullptr);  // that no copy is left in flight when the CTA ends
        return;
    }

    // ---- S = Q K^T for keys [16*warp, 16*warp + 16)
    const int grp = lane >> 2, tig = lane & 3;
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t q_base = smem_u32(sm.q);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {  // 16 dims per step
        uint32_t a0, a1, a2, a3;
        {
            const int mi = lane >> 3;
            const int row = (mi & 1) * 8 + (lane & 7);
            const int chunk = kk * 2 + (mi >> 1);
            ldsm_x4(q_base + swz(row, chunk, 256), a0, a1, a2, a3);
        }
        uint32_t b0, b1, b2, b3;
        {
            const int mi = lane >> 3;
            const int key = warp * 16 + (mi >> 1) * 8 + (lane & 7);
            const int dim = kk * 16 + (mi & 1) * 8;
            const uint32_t base = smem_u32(sm.k[dim >> 6]);
            ldsm_x4(base + swz(key, (dim & 63) >> 3, 128), b0, b1, b2, b3);
        }
        mma_bf16(s[0], a0, a1, a2, a3, b0, b1);
        mma_bf16(s[1], a0, a1, a2, a3, b2, b3);
    }
    // scale (log2 domain) and causal mask inside the block
    float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int key = warp * 16 + nt * 8 + tig * 2 + (e & 1);
            const bool valid = blk * kBlock + key <= p;
            s[nt][e] = valid ? s[nt][e] * a.scale_log2 : -INFINITY;
            rmax[e >> 1] = fmaxf(rmax[e >> 1], s[nt][e]);
        }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        rmax[i] = fmaxf(rmax[i], __shfl_xor_sync(0xffffffffu, rmax[i], 1));
        rmax[i] = fmaxf(rmax[i], __shfl_xor_sync(0xffffffffu, rmax[i], 2));
    }
    if (tig == 0) {
        sm.wmax[warp][grp] = rmax[0];
        sm.wmax[warp][grp + 8] = rmax[1];
    }
    __syncthreads();
    float m[2], lsum[2] = {0.f, 0.f};
    m[0] = fmaxf(fmaxf(sm.wmax[0][grp], sm.wmax[1][grp]), fmaxf(sm.wmax[2][grp], sm.wmax[3][grp]));
    m[1] = fmaxf(fmaxf(sm.wmax[0][grp + 8], sm.wmax[1][grp + 8]), fmaxf(sm.wmax[2][grp + 8], sm.wmax[3][grp + 8]));
    uint8_t* phi = reinterpret_cast<uint8_t*>(sm.p[0]);
    uint8_t* plo = reinterpret_cast<uint8_t*>(sm.p[1]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const float p0 = exp2f(s[nt][0] - m[0]), p1 = exp2f(s[nt][1] - m[0]);
        const float p2 = exp2f(s[nt][2] - m[1]), p3 = exp2f(s[nt][3] - m[1]);
        lsum[0] += p0 + p1;
        lsum[1] += p2 + p3;
        const int key = warp * 16 + nt * 8 + tig * 2;
        const int chunk = key >> 3, within = (key & 7) * 2;
        const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
        *reinterpret_cast<uint32_t*>(phi + swz(grp, chunk, 128) + within) = h01;
        *reinterpret_cast<uint32_t*>(phi + swz(grp + 8, chunk, 128) + within) = h23;
        *reinterpret_cast<uint32_t*>(plo + swz(grp, chunk, 128) + within) =
            pack_bf16x2(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
        *reinterpret_cast<uint32_t*>(plo + swz(grp + 8, chunk, 128) + within) =
            pack_bf16x2(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], 1);
        lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], 2);
    }
    if (tig == 0) {
        sm.wsum[warp][grp] = lsum[0];
        sm.wsum[warp][grp + 8] = lsum[1];
    }
    __syncthreads();

    // ---- O[:, 32*warp .. +32) = P V
    float o[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {  // 16 keys per step
        uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
        {
            const int mi = lane >> 3;
            const int row = (mi & 1) * 8 + (lane & 7);
            ldsm_x4(smem_u32(sm.p[0]) + swz(row, kk * 2 + (mi >> 1), 128), a0, a1, a2, a3);
            ldsm_x4(smem_u32(sm.p[1]) + swz(row, kk * 2 + (mi >> 1), 128), l0, l1, l2, l3);
        }
#pragma unroll
        for (int np = 0; np < 2; ++np) {  // pairs of 8-dim tiles
            uint32_t b0, b1, b2, b3;
            const int mi = lane >> 3;
            const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
            const int dim = warp * 32 + np * 16 + (mi >> 1) * 8;
            const uint32_t base = smem_u32(sm.v[dim >> 6]);
            ldsm_x4_t(base + swz(key, (dim & 63) >> 3, 128), b0, b1, b2, b3);
            mma_bf16(o[np * 2 + 0], a0, a1, a2, a3, b0, b1);
            mma_bf16(o[np * 2 + 1], a0, a1, a2, a3, b2, b3);
            mma_bf16(o[np * 2 + 0], l0, l1, l2, l3, b0, b1);
            mma_bf16(o[np * 2 + 1], l0, l1, l2, l3, b2, b3);
        }
    }
    // ---- partial (m, l, O) of this block
    float* part = a.partials + ((static_cast<int64_t>(b) * H + h) * a.top_k + split) * kPartialFloats;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int dim = warp * 32 + nt * 8 + tig * 2;
        *reinterpret_cast<float2*>(part + grp * 128 + dim) = make_float2(o[nt][0], o[nt][1]);
        *reinterpret_cast<float2*>(part + (grp + 8) * 128 + dim) = make_float2(o[nt][2], o[nt][3]);
    }
    if (tid < 16) {
        part[16 * 128 + tid] = fmaxf(fmaxf(sm.wmax[0][tid], sm.wmax[1][tid]), fmaxf(sm.wmax[2][tid], sm.wmax[3][tid]));
        part[16 * 128 + 16 + tid] = sm.wsum[0][tid] + sm.wsum[1][tid] + sm.wsum[2][tid] + sm.wsum[3][tid];
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(a.tickets + static_cast<int64_t>(b) * H + h, 1);
        sm.last = (prev == nsel - 1);
    }
    __syncthreads();
    if (!sm.last) return;

    // ---- last split: log-sum-exp combine of the nsel partials
    __threadfence();
    const float* parts = a.partials + (static_cast<int64_t>(b) * H + h) * a.top_k * kPartialFloats;
    // every split's (m, l) for the 16 head rows, fetched in one round of loads
    for (int t = tid; t < nsel * 32; t += kAttThreads)
        sm.ml[t >> 5][t & 31] = __ldcg(parts + (t >> 5) * kPartialFloats + 16 * 128 + (t & 31));
    __syncthreads();
    if (tid < 16) {
        float M = -INFINITY;
        for (int sp = 0; sp < nsel; ++sp) M = fmaxf(M, sm.ml[sp][tid]);
        float Ls = 0.f;
        for (int sp = 0; sp < nsel; ++sp) {
            const float w = exp2f(sm.ml[sp][tid] - M);
            sm.weight[sp][tid] = w;
            Ls += w * sm.ml[sp][16 + tid];
        }
        const float inv = 1.f / Ls;
        for (int sp = 0; sp < nsel; ++sp) sm.weight[sp][tid] *= inv;
    }
    __syncthreads();
    // thread = 4 consecutive dims of heads g0, g0+4, g0+8, g0+12; all splits'
    // loads of one head are issued together
    const int d4 = (tid & 31) * 4, g0 = tid >> 5;
    for (int g = g0; g < G; g += 4) {
        float4 v[kMaxTopK];
#pragma unroll
        for (int sp = 0; sp < kMaxTopK; ++sp)
            if (sp < nsel) v[sp] = __ldcg(reinterpret_cast<const float4*>(parts + sp * kPartialFloats + g * 128 + d4));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sp = 0; sp < kMaxTopK; ++sp)
            if (sp < nsel) {
                const float w = sm.weight[sp][g];
                acc.x = fmaf(w, v[sp].x, acc.x);
                acc.y = fmaf(w, v[sp].y, acc.y);
                acc.z = fmaf(w, v[sp].z, acc.z);
                acc.w = fmaf(w, v[sp].w, acc.w);
            }
        const int64_t oi = (static_cast<int64_t>(r) * H * G + static_cast<int64_t>(h) * G + g) * kHeadDim + d4;
        if (a.out_bf16) {
            uint2 pk;
            pk.x = pack_bf16x2(acc.x, acc.y);
            pk.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + oi) = pk;
        } else {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + oi) = acc;
        }
    }
    if (tid == 0) a.tickets[static_cast<int64_t>(b) * H + h] = 0;  // ready for the next call
}

cudaError_t run_decode_attend(const DecodeAttendArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(DecodeSmem) + 1024;
    dim3 grid(a.top_k, a.H, a.num_seqs);
    if (a.pooled != nullptr) {
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(decode_attend_kernel<false>), smem);
        if (e != cudaSuccess) return e;
        decode_attend_kernel<false><<<grid, kAttThreads, smem, stream>>>(*a.k_map, *a.v_map, a);
    } else {
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(decode_attend_kernel<true>), smem);
        if (e != cudaSuccess) return e;
        decode_attend_kernel<true><<<grid, kAttThreads, smem, stream>>>(*a.k_map, *a.v_map, a);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free launch of decode attention (msa_attend_decode_noalloc).
//
// Some callers cannot allocate device memory at all: code enqueued while a
// framework captures a CUDA graph and forbids allocation inside the capture,
// hosts whose device memory is carved out once at start-up (real-time or
// embedded serving), and plug-ins loaded into a process whose allocator they
// do not own.  For them the split partials, the per-(sequence, head) tickets
// and the error word live in the file-scope device array below instead of a
// caller workspace.  Every GPU that loads the library keeps this array
// (about 4 MiB) until the process exits.  All calls share it: calls that
// overlap on the GPU (other streams, other host threads) race and give
// wrong results; order them on one stream.
namespace {

constexpr size_t kNoAllocHeader = 256;  // error word + tickets
constexpr size_t kNoAllocBytes =
    kNoAllocHeader + static_cast<size_t>(kNoAllocMaxPairs) * kMaxTopK * kPartialFloats * sizeof(float);
static_assert(kNoAllocMaxPairs * sizeof(int32_t) + 16 <= kNoAllocHeader, "tickets must fit the header");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// The array's device address, cached per CUDA context.  A context has its own
// copy of the module and so its own address; after cudaDeviceReset (or a
// release and re-creation of the primary context) the device gets a new
// context whose ID differs, so a stale address is never reused.
struct NoAllocEntry {
    unsigned long long ctx_id;
    void* base;
};
std::mutex g_noalloc_mutex;
NoAllocEntry g_noalloc_cache[64];
int g_noalloc_used = 0;
int g_noalloc_next = 0;  // slot replaced when the cache is full (round robin)

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// ID of the calling thread's current context (0 if there is none yet).
cudaError_t current_context_id(unsigned long long* id) {
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (g_ctx_current == nullptr || g_ctx_id == nullptr) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
    *id = 0;
    if (ctx == nullptr) return cudaSuccess;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// Device address of the array in the current context (host code may not use
// the symbol itself as a device pointer).  The first call in a context looks
// it up with cudaGetSymbolAddress (which also makes the runtime set up the
// device's primary context if nothing has yet); later calls reuse it.
cudaError_t noalloc_base(void** out) {
    unsigned long long id = 0;
    cudaError_t e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (id != 0)
        for (int i = 0; i < g_noalloc_used; ++i)
            if (g_noalloc_cache[i].ctx_id == id) {
                *out = g_noalloc_cache[i].base;
                return cudaSuccess;
            }
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (id == 0 && (e = current_context_id(&id)) != cudaSuccess) return e;  // the lookup created the context
    if (id != 0) {
        const int slot = g_noalloc_used < 64 ? g_noalloc_used++ : (g_noalloc_next++ & 63);
        g_noalloc_cache[slot] = NoAllocEntry{id, ptr};
    }
    *out = ptr;
    return cudaSuccess;
}

}  // namespace

cudaError_t run_decode_attend_noalloc(DecodeAttendArgs a, cudaStream_t stream) {
    if (static_cast<int64_t>(a.num_seqs) * a.H > kNoAllocMaxPairs) return cudaErrorInvalidValue;
    void* base = nullptr;
    cudaError_t e = noalloc_base(&base);
    if (e != cudaSuccess) return e;
    uint8_t* s = static_cast<uint8_t*>(base);
    a.err = reinterpret_cast<uint32_t*>(s);
    a.tickets = reinterpret_cast<int32_t*>(s + 16);
    a.partials = reinterpret_cast<float*>(s + kNoAllocHeader);
    // the error word and the tickets must start at zero; the partials are
    // fully written before they are read
    e = cudaMemsetAsync(s, 0, 16 + static_cast<size_t>(a.num_seqs) * a.H * sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    return run_decode_attend(a, stream);
}

}  // namespace msa
