// CTA-wide top-k block selection with the forced local block.
//
// Rule ("MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120)", "What this fixes":
// each GQA group keeps 16 blocks ranked by their maximum index score, the
// current position's block always among them; PR #1388 "minimax_m3: a CUDA
// backend ...": the selection is made per row and key head): keep the local
// block J plus the (top_k - 1) best blocks
// j < J under (pooled score descending, block index ascending); keep every
// block 0..J when J < top_k; list the kept blocks ascending.
//
// Each candidate j is a distinct 64-bit key (ordered score, ~j), so the
// result does not depend on thread order:
//   1. every thread takes the largest score among its strided candidates; up
//      to kRegRounds x kChunk scores per thread are loaded at once and kept
//      in registers (longer lists are read in rounds of kChunk, and read
//      again for the gather);
//   2. every warp sorts its 32 per-thread maxima (bitonic, shuffles, on the
//      32-bit ordered score) and takes the k-th largest: a lower bound of the
//      k-th largest score overall (k distinct blocks reach it); tau = the
//      largest bound over the warps;
//   3. the blocks scoring >= tau (a few dozen for typical data) are written
//      to shared memory at offsets from warp prefix sums (no atomics), then
//      ranked exactly by counting on their 64-bit keys; the k best are placed
//      by rank;
//   4. if more than kCandCap blocks reach tau (adversarial ties), k rounds of
//      CTA-wide arg-max give the same answer.
#pragma once

#include "common.cuh"

namespace msa {

constexpr int kCandCap = 512;
constexpr int kChunk = 8;      // pooled scores per thread and load round
constexpr int kRegRounds = 4;  // rounds kept in registers (J <= 4 x 8 x NT): every load issued at once

template <int NT>
struct SelectSmem {
    uint32_t warp_tau[NT / 32];
    int32_t warp_cnt[NT / 32];
    uint64_t cand[kCandCap];
    uint64_t red[NT / 32];
    uint64_t tau;
    int32_t picked[kMaxTopK];
};

// Largest key among candidates j < J with key < below (0 if none).
template <int NT>
__device__ __forceinline__ uint64_t cta_argmax_below(const float* pooled, int J, uint64_t below, SelectSmem<NT>& sm) {
    uint64_t best = 0;
    for (int j = threadIdx.x; j < J; j += NT) {
        uint64_t key = block_key(pooled[j], j);
        if (key < below && key > best) best = key;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
    }
    if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = best;
    __syncthreads();
    uint64_t r = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) r = sm.red[w] > r ? sm.red[w] : r;
    __syncthreads();
    return r;
}

// Ranks pooled[0..J): returns others = min(top_k - 1, J), with sm.picked[k]
// the block of rank k (k < others; every block 0..J-1 when others == J, in
// order) visible to every thread.  All NT threads call it; pooled may point
// to global or shared memory (generic loads only).
template <int NT>
__device__ int cta_select_ranked(const float* pooled, int J, int top_k, SelectSmem<NT>& sm) {
    const int tid = threadIdx.x;
    const int others = min(top_k - 1, J);
    if (others == J) {  // every causal block is kept
        if (tid < others) sm.picked[tid] = tid;
        __syncthreads();
        return others;
    }
    // 1. per-thread maxima of the ordered scores (0 below every real score's code)
    const bool in_regs = J <= kRegRounds * kChunk * NT;
    uint32_t mine = 0;
    float v0[kRegRounds][kChunk];
    const int rounds = (J + kChunk * NT - 1) / (kChunk * NT);  // used rounds (uniform branches below)
    if (in_regs) {
#pragma unroll
        for (int rr = 0; rr < kRegRounds; ++rr)
            if (rr < rounds) {
#pragma unroll
                for (int i = 0; i < kChunk; ++i) {  // independent loads, all in flight together
                    const int j = (rr * kChunk + i) * NT + tid;
                    v0[rr][i] = j < J ? pooled[j] : 0.f;  // generic load: pooled may be shared memory
                }
            }
#pragma unroll
        for (int rr = 0; rr < kRegRounds; ++rr)
            if (rr < rounds) {
#pragma unroll
                for (int i = 0; i < kChunk; ++i) {
                    const int j = (rr * kChunk + i) * NT + tid;
                    if (j < J) mine = max(mine, ordered_bits(v0[rr][i]));
                }
            }
    } else {
        for (int base = 0; base < J; base += kChunk * NT) {
            float v[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const int j = base + i * NT + tid;
                v[i] = j < J ? pooled[j] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const int j = base + i * NT + tid;
                if (j < J) mine = max(mine, ordered_bits(v[i]));
            }
        }
    }
    // 2. per-warp bound: sort the 32 maxima descending, take the others-th;
    // warp 0 always holds min(J, 32) >= others candidates, so tau > 0
    const int lane = tid & 31, warp = tid >> 5;
    {
        uint32_t key = mine;
#pragma unroll
        for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
            for (int jj = k >> 1; jj > 0; jj >>= 1) {
                const uint32_t other = __shfl_xor_sync(0xffffffffu, key, jj);
                const bool keep_max = ((lane & k) == 0) == ((lane & jj) == 0);
                key = keep_max ? max(other, key) : min(other, key);
            }
        const uint32_t bound = __shfl_sync(0xffffffffu, key, others - 1);
        if (lane == 0) sm.warp_tau[warp] = bound;
    }
    __syncthreads();
    uint32_t tau = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) tau = max(tau, sm.warp_tau[w]);
    // 3. candidates: blocks with ordered score >= tau, written at offsets from
    // an inclusive scan of the per-thread counts within each warp and the warp
    // totals across warps (deterministic, no atomics)
    int cnt = 0;
    if (in_regs) {
#pragma unroll
        for (int rr = 0; rr < kRegRounds; ++rr)
            if (rr < rounds) {
#pragma unroll
                for (int i = 0; i < kChunk; ++i) {
                    const int j = (rr * kChunk + i) * NT + tid;
                    cnt += (j < J && ordered_bits(v0[rr][i]) >= tau) ? 1 : 0;
                }
            }
    } else {
        for (int j = tid; j < J; j += NT) cnt += ordered_bits(pooled[j]) >= tau ? 1 : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) sm.warp_cnt[warp] = incl;
    __syncthreads();
    int n = 0, off = incl - cnt;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        off += w < warp ? sm.warp_cnt[w] : 0;
        n += sm.warp_cnt[w];
    }
    if (n <= kCandCap && cnt > 0) {
        if (in_regs) {
#pragma unroll
            for (int rr = 0; rr < kRegRounds; ++rr)
                if (rr < rounds) {
#pragma unroll
                    for (int i = 0; i < kChunk; ++i) {
                        const int j = (rr * kChunk + i) * NT + tid;
                        if (j < J && ordered_bits(v0[rr][i]) >= tau) sm.cand[off++] = block_key(v0[rr][i], j);
                    }
                }
        } else {
            for (int j = tid; j < J; j += NT) {
                const float m = pooled[j];
                if (ordered_bits(m) >= tau) sm.cand[off++] = block_key(m, j);
            }
        }
    }
    __syncthreads();
    if (n <= kCandCap) {
        for (int c = tid; c < n; c += NT) {
            const uint64_t key = sm.cand[c];
            int r0 = 0, r1 = 0, r2 = 0, r3 = 0;  // four independent counts per pass
            int u = 0;
            for (; u + 4 <= n; u += 4) {
                r0 += sm.cand[u] > key;
                r1 += sm.cand[u + 1] > key;
                r2 += sm.cand[u + 2] > key;
                r3 += sm.cand[u + 3] > key;
            }
            for (; u < n; ++u) r0 += sm.cand[u] > key;
            const int rank = r0 + r1 + r2 + r3;
            if (rank < others) sm.picked[rank] = key_block(key);
        }
        __syncthreads();
    } else {
        uint64_t below = ~0ull;
        for (int i = 0; i < others; ++i) {
            below = cta_argmax_below<NT>(pooled, J, below, sm);
            if (tid == 0) sm.picked[i] = key_block(below);
        }
        __syncthreads();
    }
    return others;
}

// Selects from pooled[0..J) (+ the local block J): writes the kept blocks
// ascending to sel[0..top_k) (-1 padded; sel may be shared or global memory,
// written by threads < top_k) and returns nsel.
template <int NT>
__device__ int cta_select(const float* pooled, int J, int top_k, int* sel, SelectSmem<NT>& sm) {
    const int tid = threadIdx.x;
    const int others = cta_select_ranked<NT>(pooled, J, top_k, sm);
    // picked[0..others) + J, ascending (J is the largest)
    if (tid <= others) {
        int v = tid < others ? sm.picked[tid] : J;
        int pos = 0;
        for (int u = 0; u < others; ++u) pos += sm.picked[u] < v;
        if (tid == others) pos = others;
        sel[pos] = v;
    } else if (tid < top_k) {
        sel[tid] = -1;
    }
    __syncthreads();
    return others + 1;
}


}  // namespace msa
