// Staged (unfused) forms of stages 1 and 2, for stage-by-stage checking:
//   msa_index_scores  -> every score s[r, h, t] (fp32), -inf past the row
//   msa_select_blocks -> block max-pool of given scores + top-k selection
// The fused path never materialises scores; these kernels favour plainness.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace msa {

constexpr int kStagedThreads = 128;

__device__ __forceinline__ bool row_position(const StagedArgs& a, int r, int& b, int& p) {
    int lo = 0, hi = a.num_seqs;  // largest b with cu_rows[b] <= r
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.cu_rows[mid] <= r) lo = mid; else hi = mid;
    }
    b = lo;
    const int n = a.cu_rows[b + 1] - a.cu_rows[b];
    const int L = a.cache_lens[b];
    p = L - n + (r - a.cu_rows[b]);
    return r >= a.cu_rows[b] && r < a.cu_rows[b + 1] && L >= 1 && L <= a.max_cache_len && p >= 0 &&
           seq_rows_ok(a.cache, b, L, a.cache_tokens);
}

// grid (rows, H): one CTA per (row, head)
__global__ void __launch_bounds__(kStagedThreads) index_scores_kernel(StagedArgs a, const uint16_t* __restrict__ iq,
                                                                      const uint16_t* __restrict__ ik,
                                                                      float* __restrict__ scores, int64_t ld) {
    const int h = blockIdx.y, r = blockIdx.x;
    int b, p;
    const bool ok = row_position(a, r, b, p);
    float q[kIndexDim];
    const uint16_t* qp = iq + (static_cast<int64_t>(r) * a.H + h) * kIndexDim;
#pragma unroll
    for (int c = 0; c < kIndexDim / 8; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(qp + c * 8);
        q[c * 8 + 0] = bf16_lo(w.x); q[c * 8 + 1] = bf16_hi(w.x);
        q[c * 8 + 2] = bf16_lo(w.y); q[c * 8 + 3] = bf16_hi(w.y);
        q[c * 8 + 4] = bf16_lo(w.z); q[c * 8 + 5] = bf16_hi(w.z);
        q[c * 8 + 6] = bf16_lo(w.w); q[c * 8 + 7] = bf16_hi(w.w);
    }
    float* out = scores + (static_cast<int64_t>(r) * a.H + h) * ld;
    for (int64_t t = threadIdx.x; t < ld; t += kStagedThreads) {
        float s = -INFINITY;
        const int64_t row0 = ok && t <= p ? block_row(a.cache, b, t & ~int64_t{kBlock - 1}) : -1;
        if (row0 >= 0) {  // (a page outside the pool leaves -inf)
            const int kh = a.ik_shared ? 1 : a.H;  // index-key heads per position
            const uint16_t* kp = ik + ((row0 + (t & (kBlock - 1))) * kh + (a.ik_shared ? 0 : h)) * kIndexDim;
            s = 0.f;
#pragma unroll
            for (int c = 0; c < kIndexDim / 8; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(kp + c * 8);
                s = fmaf(q[c * 8 + 0], bf16_lo(w.x), s); s = fmaf(q[c * 8 + 1], bf16_hi(w.x), s);
                s = fmaf(q[c * 8 + 2], bf16_lo(w.y), s); s = fmaf(q[c * 8 + 3], bf16_hi(w.y), s);
                s = fmaf(q[c * 8 + 4], bf16_lo(w.z), s); s = fmaf(q[c * 8 + 5], bf16_hi(w.z), s);
                s = fmaf(q[c * 8 + 6], bf16_lo(w.w), s); s = fmaf(q[c * 8 + 7], bf16_hi(w.w), s);
            }
        }
        out[t] = s;
    }
}

// grid (rows, H): pool the row's scores into shared memory, then select.
__global__ void __launch_bounds__(kStagedThreads) select_blocks_kernel(StagedArgs a, const float* __restrict__ scores,
                                                                       int64_t ld, int32_t* __restrict__ sel,
                                                                       int32_t* __restrict__ nsel) {
    extern __shared__ float pooled[];  // [max_blocks]
    __shared__ SelectSmem<kStagedThreads> sm;
    const int h = blockIdx.y, r = blockIdx.x;
    int b, p;
    int32_t* out = sel + (static_cast<int64_t>(r) * a.H + h) * a.top_k;
    if (!row_position(a, r, b, p)) {
        for (int i = threadIdx.x; i < a.top_k; i += kStagedThreads) out[i] = -1;
        if (threadIdx.x == 0) nsel[static_cast<int64_t>(r) * a.H + h] = 0;
        return;
    }
    const int J = p / kBlock;
    const float* s = scores + (static_cast<int64_t>(r) * a.H + h) * ld;
    // one warp per block: lanes take two positions each
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < J; j += kStagedThreads / 32) {
        const float v0 = s[j * kBlock + lane], v1 = s[j * kBlock + 32 + lane];
        float m = fmaxf(v0, v1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) pooled[j] = m;
    }
    __syncthreads();
    const int n = cta_select<kStagedThreads>(pooled, J, a.top_k, out, sm);
    if (threadIdx.x == 0) nsel[static_cast<int64_t>(r) * a.H + h] = n;
}

cudaError_t run_index_scores(const StagedArgs& a, const uint16_t* iq, const uint16_t* ik, float* scores, int64_t ld,
                             cudaStream_t stream) {
    dim3 grid(a.total_rows, a.H);
    index_scores_kernel<<<grid, kStagedThreads, 0, stream>>>(a, iq, ik, scores, ld);
    return cudaGetLastError();
}

cudaError_t run_select_blocks(const StagedArgs& a, const float* scores, int64_t ld, int32_t* sel, int32_t* nsel,
                              cudaStream_t stream) {
    const int max_blocks = (a.max_cache_len + kBlock - 1) / kBlock;
    const size_t smem = static_cast<size_t>(max_blocks) * sizeof(float);
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(select_blocks_kernel), smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.total_rows, a.H);
    select_blocks_kernel<<<grid, kStagedThreads, smem, stream>>>(a, scores, ld, sel, nsel);
    return cudaGetLastError();
}

}  // namespace msa
