// int8 key/value cache (PR #1388, native Metal family commit: keys and values
// cached as int8 with one scale per position and head), prompt chunks.
//
// In a long prompt chunk every 64-position block is kept by hundreds of
// (row, head) items, so widening the int8 tiles inside the attention repeats
// the same work that many times.  This pass widens the positions of every
// sequence the prompt-chunk attention reads once per call, into a contiguous
// bf16 copy in the workspace: the integers exactly (an int8 value has at most
// 8 significant bits, so bf16 holds it), the scales copied beside them in
// fp32.  The attention then loads bf16 tiles and multiplies the scores by the
// key scales and the weights by the value scales exactly as it does for the
// tiles it widens itself, so its results are those of the int8 cache.
//
// Layout: sequence b's copy starts at row  slot_b * slot_rows  (slot_b counts
// the widened sequences before b; slot_rows = max_cache_len rounded up to a
// whole block), rows [T', H, 128] bf16 for K and V and [H, T'] fp32 for the
// scales (head-major, so that a warp staging one head's scales for 32
// consecutive keys reads one 128-byte line).  Positions from L_b to the end of their 64-position block are
// written as zeros: keys past a row's position are masked, and a zero value
// keeps 0 x value out of the P V products.  Row starts per sequence go to
// `wide_starts` (0 for a sequence that is not widened, -1 for one past the
// slots the workspace holds, which the attention then rejects).
#include "common.cuh"
#include "internal.h"

namespace msa {

constexpr int kWidenThreads = 256;
constexpr int kWidenPos = 16;    // positions per work unit (a quarter block)
constexpr int kWidenBatch = 4;   // 16-byte chunks of K and of V a thread loads before it stores

// Byte i of w as a signed integer, then 4 bytes as 4 bf16 (two words; exact: at most 8 significant bits)
__device__ __forceinline__ float i8_at(uint32_t w, int i) {
    const int v = static_cast<int>((w >> (8 * i)) & 0xffu);
    return static_cast<float>(v - ((v & 0x80) << 1));
}
__device__ __forceinline__ uint2 widen_i8x4(uint32_t w) {
    return make_uint2(pack_bf16x2(i8_at(w, 0), i8_at(w, 1)), pack_bf16x2(i8_at(w, 2), i8_at(w, 3)));
}

__global__ void __launch_bounds__(kWidenThreads) widen_kv_kernel(const WidenArgs a) {
    extern __shared__ int32_t slot_of[];  // [num_seqs]: slot of sequence b, or -1 (not widened)
    __shared__ int32_t warp_tot[kWidenThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.num_seqs;

    // ---- slots: thread t takes sequences [t per, (t + 1) per), then an exclusive block scan
    const int per = (B + kWidenThreads - 1) / kWidenThreads;
    const int b_lo = min(tid * per, B), b_hi = min(b_lo + per, B);
    int cnt = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int n = a.cu_rows[b + 1] - a.cu_rows[b];
        const int w = n >= 1 && !(a.only_multi_row && n <= kDecodeMaxRows);
        slot_of[b] = w;
        cnt += w;
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int excl = x - cnt;
    for (int i = 0; i < warp; ++i) excl += warp_tot[i];
    for (int b = b_lo; b < b_hi; ++b) slot_of[b] = slot_of[b] ? excl++ : -1;
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int b = tid; b < B; b += kWidenThreads) {
            const int s = slot_of[b];
            a.wide_starts[b] = s < 0 ? 0 : (s < a.max_slots ? static_cast<int64_t>(s) * a.slot_rows : -1);
            if (s >= a.max_slots) atomicOr(a.err, kErrBadMetadata);  // more such sequences than the host counted
        }
    }

    // ---- units: (sequence, 16 positions), all heads, K and V; a block's positions past L_b are
    // written as zeros, so the units run to the end of the last block
    const int H = a.H;
    const int64_t wide_rows = static_cast<int64_t>(a.max_slots) * a.slot_rows;
    const int groups = a.slot_rows / kWidenPos;
    const int64_t units = static_cast<int64_t>(B) * groups;
    const int row_chunks = H * (kHeadDim / 16);  // 16-byte int8 chunks per position
    const int unit_chunks = kWidenPos * row_chunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int b = static_cast<int>(u / groups), grp = static_cast<int>(u - static_cast<int64_t>(b) * groups);
        const int slot = slot_of[b];
        if (slot < 0 || slot >= a.max_slots) continue;
        const int L = a.cache_lens[b];
        const int t0 = grp * kWidenPos, tb = t0 & ~(kBlock - 1);  // first position, its block's
        if (L < 1 || L > a.max_cache_len || tb >= L) continue;  // the attention rejects such a sequence
        const int64_t brow = seq_rows_ok(a.cache, b, L, a.cache_tokens) ? block_row(a.cache, b, tb) : -1;
        if (brow < 0 && tid == 0 && t0 == tb) atomicOr(a.err, kErrBadMetadata);  // the block is written as zeros
        const int64_t src = brow < 0 ? 0 : brow + (t0 - tb);  // a block's rows are contiguous (a page holds whole blocks)
        const int64_t dst = static_cast<int64_t>(slot) * a.slot_rows + t0;
        const int live_rows = brow < 0 ? 0 : max(0, min(kWidenPos, L - t0));
        const uint8_t* k8 = a.k8 + src * H * kHeadDim;
        const uint8_t* v8 = a.v8 + src * H * kHeadDim;
        uint16_t* kw = a.kw + dst * H * kHeadDim;
        uint16_t* vw = a.vw + dst * H * kHeadDim;
        for (int c0 = tid; c0 < unit_chunks; c0 += kWidenBatch * kWidenThreads) {
            uint4 kx[kWidenBatch], vx[kWidenBatch];  // every load of the batch in flight before a store
#pragma unroll
            for (int j = 0; j < kWidenBatch; ++j) {
                const int c = c0 + j * kWidenThreads;
                const bool live = c < live_rows * row_chunks;
                kx[j] = live ? ld_stream_v4(k8 + c * 16) : make_uint4(0, 0, 0, 0);
                vx[j] = live ? ld_stream_v4(v8 + c * 16) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < kWidenBatch; ++j) {
                const int c = c0 + j * kWidenThreads;
                if (c >= unit_chunks) break;
                const uint2 k0 = widen_i8x4(kx[j].x), k1 = widen_i8x4(kx[j].y), k2 = widen_i8x4(kx[j].z),
                            k3 = widen_i8x4(kx[j].w);
                const uint2 v0 = widen_i8x4(vx[j].x), v1 = widen_i8x4(vx[j].y), v2 = widen_i8x4(vx[j].z),
                            v3 = widen_i8x4(vx[j].w);
                uint4* kd = reinterpret_cast<uint4*>(kw + static_cast<int64_t>(c) * 16);
                uint4* vd = reinterpret_cast<uint4*>(vw + static_cast<int64_t>(c) * 16);
                kd[0] = make_uint4(k0.x, k0.y, k1.x, k1.y);
                kd[1] = make_uint4(k2.x, k2.y, k3.x, k3.y);
                vd[0] = make_uint4(v0.x, v0.y, v1.x, v1.y);
                vd[1] = make_uint4(v2.x, v2.y, v3.x, v3.y);
            }
        }
        for (int c = tid; c < kWidenPos * H; c += kWidenThreads) {  // scales head-major: [H][rows]
            const bool live = c < live_rows * H;
            const int pos = c / H, h = c - pos * H;
            const int64_t o = static_cast<int64_t>(h) * wide_rows + dst + pos;
            a.ksw[o] = live ? a.k_scale[src * H + c] : 0.f;
            a.vsw[o] = live ? a.v_scale[src * H + c] : 0.f;
        }
    }
}

cudaError_t run_widen_kv(const WidenArgs& a, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>(a.num_seqs) * (a.slot_rows / kWidenPos);
    const int64_t cap = 4 * static_cast<int64_t>(device_sm_count());
    const int grid = static_cast<int>(units < cap ? (units > 0 ? units : 1) : cap);
    const size_t smem = static_cast<size_t>(a.num_seqs) * sizeof(int32_t);
    widen_kv_kernel<<<grid, kWidenThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace msa
