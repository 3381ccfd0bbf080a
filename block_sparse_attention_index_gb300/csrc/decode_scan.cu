// Decode stage 1+2a: lightning-indexer scan with the block max-pool fused in.
//
// For every sequence with exactly one query row (a decode row at p = L-1)
// and every KV head h, computes the pooled index score of every block j:
//     m_j = max_{t in block j, t <= p}  iq[r,h,:] . ik[t,h,:]
// ("MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120)", "What this fixes":
// max-pool scoring; PR #1388 "minimax_m3: a CUDA backend ...": the index
// scores per row and key head).  Only the pooled scores (4 bytes per block
// and head) leave the kernel; the per-position scores live in registers.
//
// The scan is HBM-bound: each cached position carries H x 64 bf16 index-key
// values (128 B per head) that are read exactly once.  Work unit = one
// 64-position block of one sequence with all H heads, which is H x 8 KB of
// contiguous memory.  The grid is a multiple of the SM count; CTA c takes an
// even share of all units of all decode sequences (the split is computed on
// the device from the per-sequence lengths, so ragged batches balance).
// Every thread owns one 16-byte slice (8 dims) of one head and issues all of
// its 16-byte loads of a unit before using them; eight lanes complete a dot
// product with three shuffles.
#include "common.cuh"
#include "internal.h"

namespace msa {

constexpr int kScanThreads = 256;

template <int H>
__global__ void __launch_bounds__(kScanThreads) decode_scan_kernel(
    const uint16_t* __restrict__ iq, const uint16_t* __restrict__ ik, const int32_t* __restrict__ cu_rows,
    const int32_t* __restrict__ cache_lens, const int64_t* __restrict__ cache_starts, int num_seqs,
    int total_rows, int max_cache_len, int64_t cache_tokens, int max_blocks, float* __restrict__ pooled,
    int32_t* __restrict__ clear_words, int n_clear) {
    static_assert(32 % H == 0, "H must divide 32");
    constexpr int kLoads = 2 * H;              // 16-byte loads per thread per unit
    constexpr int kPosPerIter = 32 / H;        // positions covered by one load round
    extern __shared__ int32_t prefix[];        // [num_seqs + 1] units before sequence b
    __shared__ float red[kScanThreads / 8];    // one slot per 8-lane group
    __shared__ int warp_tot[kScanThreads / 32];

    const int tid = threadIdx.x;
    // The attention kernel that follows uses these counters; clear them here.
    if (blockIdx.x == 0)
        for (int i = tid; i < n_clear; i += kScanThreads) clear_words[i] = 0;

    // Units per sequence: ceil(L/64) for decode sequences, 0 otherwise.
    // Block-wide exclusive scan in chunks of kScanThreads.
    int carry = 0;
    for (int base = 0; base < num_seqs; base += kScanThreads) {
        const int b = base + tid;
        int units = 0;
        if (b < num_seqs && cu_rows[b + 1] - cu_rows[b] == 1) {
            const int L = min(max(cache_lens[b], 0), max_cache_len);
            units = (L + kBlock - 1) / kBlock;
        }
        int incl = units;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, o);
            if ((tid & 31) >= o) incl += v;
        }
        if ((tid & 31) == 31) warp_tot[tid >> 5] = incl;
        __syncthreads();
        int before = 0;
        for (int w = 0; w < (tid >> 5); ++w) before += warp_tot[w];
        if (b < num_seqs) prefix[b] = carry + before + incl - units;
        int chunk_total = 0;
        for (int w = 0; w < kScanThreads / 32; ++w) chunk_total += warp_tot[w];
        __syncthreads();
        carry += chunk_total;
    }
    if (tid == 0) prefix[num_seqs] = carry;
    __syncthreads();

    const int64_t total = carry;
    const int64_t u0 = total * blockIdx.x / gridDim.x;
    const int64_t u1 = total * (blockIdx.x + 1) / gridDim.x;
    if (u0 >= u1) return;

    const int part = tid & 7;                  // which 8 dims of the head
    const int h = (tid >> 3) % H;              // head of this thread
    const int pos_off = tid / (8 * H);         // position offset within a round

    // first sequence of this CTA's range
    int b = 0;
    {
        int lo = 0, hi = num_seqs;  // largest b with prefix[b] <= u0
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (prefix[mid] <= u0) lo = mid; else hi = mid;
        }
        b = lo;
    }
    int cur_b = -1;
    float qv[8];
    int L = 0;
    int64_t start = 0;

    for (int64_t u = u0; u < u1; ++u) {
        while (u >= prefix[b + 1]) ++b;
        if (b != cur_b) {
            cur_b = b;
            const int r = min(max(cu_rows[b], 0), total_rows - 1);
            const uint4 w = *reinterpret_cast<const uint4*>(iq + (static_cast<int64_t>(r) * H + h) * kIndexDim + part * 8);
            qv[0] = bf16_lo(w.x); qv[1] = bf16_hi(w.x); qv[2] = bf16_lo(w.y); qv[3] = bf16_hi(w.y);
            qv[4] = bf16_lo(w.z); qv[5] = bf16_hi(w.z); qv[6] = bf16_lo(w.w); qv[7] = bf16_hi(w.w);
            L = min(max(cache_lens[b], 0), max_cache_len);
            start = cache_starts[b];
            if (start < 0 || start + L > cache_tokens || cu_rows[b] != r) L = 0;  // inconsistent metadata: pool nothing
        }
        const int j = static_cast<int>(u - prefix[b]);
        const int npos = min(kBlock, L - j * kBlock);
        const uint16_t* blk = ik + (start + static_cast<int64_t>(j) * kBlock) * (H * kIndexDim);

        uint4 v[kLoads];
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const int pos = i * kPosPerIter + pos_off;
            if (pos < npos)
                v[i] = ld_stream_v4(blk + (static_cast<int64_t>(pos) * H + h) * kIndexDim + part * 8);
            else
                v[i] = make_uint4(0, 0, 0, 0);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            float s = qv[0] * bf16_lo(v[i].x);
            s = fmaf(qv[1], bf16_hi(v[i].x), s);
            s = fmaf(qv[2], bf16_lo(v[i].y), s);
            s = fmaf(qv[3], bf16_hi(v[i].y), s);
            s = fmaf(qv[4], bf16_lo(v[i].z), s);
            s = fmaf(qv[5], bf16_hi(v[i].z), s);
            s = fmaf(qv[6], bf16_lo(v[i].w), s);
            s = fmaf(qv[7], bf16_hi(v[i].w), s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            const int pos = i * kPosPerIter + pos_off;
            if (pos < npos) mx = fmaxf(mx, s);
        }
        if (part == 0) red[tid >> 3] = mx;
        __syncthreads();
        if (tid < H) {
            float m = -INFINITY;
            for (int g = tid; g < kScanThreads / 8; g += H) m = fmaxf(m, red[g]);
            if (npos > 0) pooled[(static_cast<int64_t>(b) * H + tid) * max_blocks + j] = m;
        }
        __syncthreads();
    }
}

template <int H>
static cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(a.num_seqs + 1) * sizeof(int32_t);
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_scan_kernel<H>, kScanThreads, smem);
    if (e != cudaSuccess) return e;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(decode_scan_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    int64_t grid = static_cast<int64_t>(device_sm_count()) * (occ > 0 ? occ : 1);
    if (a.unit_bound < grid) grid = a.unit_bound > 0 ? a.unit_bound : 1;
    decode_scan_kernel<H><<<static_cast<unsigned>(grid), kScanThreads, smem, stream>>>(
        a.iq, a.ik, a.cu_rows, a.cache_lens, a.cache_starts, a.num_seqs, a.total_rows, a.max_cache_len, a.cache_tokens,
        a.max_blocks, a.pooled, a.clear_words, a.n_clear);
    return cudaGetLastError();
}

cudaError_t run_decode_scan(const ScanArgs& a, cudaStream_t stream) {
    switch (a.H) {
        case 1: return launch_scan<1>(a, stream);
        case 2: return launch_scan<2>(a, stream);
        case 4: return launch_scan<4>(a, stream);
        case 8: return launch_scan<8>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace msa
