// Prompt-chunk stage 3 on tcgen05: attention of the G query heads of one KV
// head over the row's kept blocks, with tensor-memory accumulators.
//
// PR #1388 "minimax_m3: a CUDA backend for MiniMax-M3.1-Flash ...", prompt-
// tile commit: a tile holds the 16 query heads of one key head; the heads
// share their row's block selection, so each key/value block is read once
// for all of them.  The row's selection is used as it stands (a tile never
// attends to a block the row did not keep).
//
// Work item = (query row, KV head), 16 kept blocks = 8 pairs of 64 keys.  The
// MMAs are transposed so that the 16 heads are the N dimension and the keys
// (or head dims) the M = 128 dimension:
//   S^T[128 keys, 16 heads]  = K_pair[128 keys, 128 dims] . Q^T        per pair
//   O^T[128 dims, 32]       += V_pair^T[128 dims, 128 keys] . [P_hi; P_lo]^T
// K and V pairs arrive by TMA (128-byte swizzle) in a 4-stage ring; V is read
// as an MN-major operand straight from its [key][dim] tile.  All 8 pairs'
// S^T (128 TMEM columns) are computed first, so the softmax is exact in one
// pass (no running rescale): thread t of the four softmax warps owns key t
// of every pair, reduces per-head maxima and sums across the CTA, and writes
// P as bf16 hi and lo parts (N = 32: heads 0-15 hi, 16-31 lo) so the
// weights keep ~16 significant bits.  The epilogue adds the two halves of
// O^T, divides by the sums and stores out[row, h*G+g, :].
//
// Warp roles: warps 0-3 softmax and epilogue, warp 4 TMA producer, warp 5
// MMA issuer and tensor-memory owner.  Items are strided over a grid of one
// CTA per SM.
#include "common.cuh"
#include "internal.h"

namespace msa {

constexpr int kPaThreads = 192;
constexpr int kPaStages = 4;
constexpr int kPairBytes = 2 * 2 * 64 * 64 * 2;  // [dim half][2 blocks x 64 keys][64 dims] bf16 = 32 KB
constexpr int kQBytes = 2 * 16 * 64 * 2;         // [dim half][16 heads][64 dims] = 4 KB
constexpr int kPChunkBytes = 32 * 64 * 2;        // [32 rows: hi heads, lo heads][64 keys] = 4 KB
constexpr int kTmemCols = 256;
constexpr int kOCol = 128;                       // O^T columns [128, 160)

struct __align__(1024) AttendSmem {
    uint8_t stage[kPaStages][kPairBytes];
    uint8_t p[16][kPChunkBytes];                 // 16 chunks of 64 keys
    uint8_t q[2][kQBytes];
    uint64_t full[kPaStages];
    uint64_t empty[kPaStages];
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t s_full;
    uint64_t p_full;
    uint64_t o_full;
    float red[4][16];
    float rowmax[16];
    float rowsum[16];
    uint32_t tmem_base;
};

struct Item {
    int r, h, p, nsel;
    int64_t start;
    int blk[kMaxTopK];
};

// Decodes work item `it`; false when the item is skipped (a row of a decode
// sequence on the fused path, or inconsistent metadata / selection).
__device__ bool load_item(const PrefillAttendArgs& a, int it, Item& x, bool& bad) {
    bad = false;
    x.r = it / a.H;
    x.h = it - x.r * a.H;
    int lo = 0, hi = a.num_seqs;  // largest b with cu_rows[b] <= r
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.cu_rows[mid] <= x.r) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int n = a.cu_rows[b + 1] - a.cu_rows[b];
    if (a.only_multi_row && n <= 1) return false;
    const int L = a.cache_lens[b];
    x.start = a.cache_starts[b];
    x.p = L - n + (x.r - a.cu_rows[b]);
    if (x.r < a.cu_rows[b] || x.r >= a.cu_rows[b + 1] || L < 1 || L > a.max_cache_len || x.p < 0 || x.start < 0 ||
        x.start + L > a.cache_tokens) {
        bad = true;
        return false;
    }
    const int J = x.p / kBlock;
    x.nsel = a.nsel[static_cast<int64_t>(x.r) * a.H + x.h];
    if (x.nsel < 1 || x.nsel > a.top_k) {
        bad = true;
        return false;
    }
    const int32_t* s = a.sel + (static_cast<int64_t>(x.r) * a.H + x.h) * a.top_k;
    for (int i = 0; i < kMaxTopK; ++i) {
        x.blk[i] = i < x.nsel ? s[i] : 0;
        if (i < x.nsel && (x.blk[i] < 0 || x.blk[i] > J)) {
            bad = true;
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(kPaThreads, 1) prefill_attend_kernel(const __grid_constant__ CUtensorMap q_map,
                                                                       const __grid_constant__ CUtensorMap k_map,
                                                                       const __grid_constant__ CUtensorMap v_map,
                                                                       const PrefillAttendArgs a) {
    extern __shared__ uint8_t smem_raw[];
    AttendSmem& sm = *reinterpret_cast<AttendSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_items = a.total_rows * a.H;

    if (tid == 0) {
        for (int s = 0; s < kPaStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.q_full[s], 1);
            mbar_init(&sm.q_empty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.p_full, 128);
        mbar_init(&sm.o_full, 1);
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(&sm.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 4) {
        // ---------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&q_map);
            prefetch_tmap(&k_map);
            prefetch_tmap(&v_map);
            uint32_t g = 0, it = 0;
            bool alive = true;
            for (int item = blockIdx.x; alive && item < n_items; item += gridDim.x) {
                Item x;
                bool bad;
                if (!load_item(a, item, x, bad)) continue;
                const int qb = it & 1;
                if (it >= 2 && !mbar_wait(&sm.q_empty[qb], ((it >> 1) - 1) & 1, a.err)) break;
                mbar_arrive_expect_tx(&sm.q_full[qb], kQBytes);
                const int hq0 = x.h * a.G;
                tma_load_3d(sm.q[qb], &q_map, &sm.q_full[qb], 0, hq0, x.r);
                tma_load_3d(sm.q[qb] + kQBytes / 2, &q_map, &sm.q_full[qb], 64, hq0, x.r);
                const int npairs = (x.nsel + 1) >> 1;
                for (int pass = 0; pass < 2 && alive; ++pass) {
                    const CUtensorMap* map = pass == 0 ? &k_map : &v_map;
                    for (int q = 0; q < npairs; ++q, ++g) {
                        const int s = g % kPaStages;
                        if (g >= kPaStages && !mbar_wait(&sm.empty[s], ((g / kPaStages) - 1) & 1, a.err)) {
                            alive = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&sm.full[s], kPairBytes);
                        for (int half = 0; half < 2; ++half) {
                            const int blk = x.blk[min(2 * q + half, x.nsel - 1)];
                            const int tok = static_cast<int>(x.start + static_cast<int64_t>(blk) * kBlock);
                            uint8_t* dst = sm.stage[s] + half * 8192;
                            tma_load_3d(dst, map, &sm.full[s], 0, x.h, tok);
                            tma_load_3d(dst + 16384, map, &sm.full[s], 64, x.h, tok);
                        }
                    }
                }
                ++it;
            }
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 16, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, 32, 1, 0);
            uint32_t g = 0, it = 0;
            bool alive = true;
            for (int item = blockIdx.x; alive && item < n_items; item += gridDim.x) {
                Item x;
                bool bad;
                if (!load_item(a, item, x, bad)) continue;
                const int qb = it & 1;
                const int npairs = (x.nsel + 1) >> 1;
                if (!mbar_wait(&sm.q_full[qb], (it >> 1) & 1, a.err)) break;
                const uint32_t q_addr = smem_u32(sm.q[qb]);
                for (int q = 0; q < npairs; ++q, ++g) {  // S^T per pair
                    const int s = g % kPaStages;
                    if (!mbar_wait(&sm.full[s], (g / kPaStages) & 1, a.err)) { alive = false; break; }
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(sm.stage[s]);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint64_t ad = smem_desc_sw128(k_addr + off, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(q_addr + (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32, 16, 1024);
                        tc_mma_ss(tmem + q * 16, ad, bd, idesc_s, kk > 0);
                    }
                    tc_commit(&sm.empty[s]);
                }
                if (!alive) break;
                tc_commit(&sm.q_empty[qb]);
                tc_commit(&sm.s_full);
                if (!mbar_wait(&sm.p_full, it & 1, a.err)) break;
                tc_fence_after();
                for (int q = 0; q < npairs; ++q, ++g) {  // O^T += V^T P^T per pair
                    const int s = g % kPaStages;
                    if (!mbar_wait(&sm.full[s], (g / kPaStages) & 1, a.err)) { alive = false; break; }
                    tc_fence_after();
                    const uint32_t v_addr = smem_u32(sm.stage[s]);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {  // 16 keys per step
                        const uint64_t ad = smem_desc_sw128(v_addr + kk * 2048, 16384, 1024);
                        const int chunk = 2 * q + (kk >> 2);
                        const uint64_t bd = smem_desc_sw128(smem_u32(sm.p[chunk]) + (kk & 3) * 32, 16, 1024);
                        tc_mma_ss(tmem + kOCol, ad, bd, idesc_o, (q > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&sm.empty[s]);
                }
                if (!alive) break;
                tc_commit(&sm.o_full);
                ++it;
            }
        }
    } else {
        // ---------------- softmax + epilogue (128 threads; thread = TMEM lane)
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const int key_in_blk = tid & 63, half = tid >> 6;
        uint32_t it = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            Item x;
            bool bad;
            if (!load_item(a, item, x, bad)) {
                if (bad && tid == 0) atomicOr(a.err, kErrBadMetadata);
                continue;
            }
            const int npairs = (x.nsel + 1) >> 1;
            if (!mbar_wait(&sm.s_full, it & 1, a.err)) break;
            tc_fence_after();
            // pass 1: per-head maxima of the raw scores over valid keys
            float mx[16];
#pragma unroll
            for (int g = 0; g < 16; ++g) mx[g] = -INFINITY;
            for (int q = 0; q < npairs; ++q) {
                uint32_t v[16];
                tmem_ld16(lane_addr + q * 16, v);
                tmem_ld_wait();
                const int idx = 2 * q + half;
                const bool valid = idx < x.nsel && x.blk[idx] * kBlock + key_in_blk <= x.p;
                if (valid) {
#pragma unroll
                    for (int g = 0; g < 16; ++g) mx[g] = fmaxf(mx[g], __uint_as_float(v[g]));
                }
            }
#pragma unroll
            for (int g = 0; g < 16; ++g) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], o));
            }
            if (lane < 16) {
                float m = mx[0];
#pragma unroll
                for (int g = 1; g < 16; ++g) m = lane == g ? mx[g] : m;
                sm.red[warp][lane] = m;
            }
            named_sync_softmax();
            float ms[16];
#pragma unroll
            for (int g = 0; g < 16; ++g)
                ms[g] = fmaxf(fmaxf(sm.red[0][g], sm.red[1][g]), fmaxf(sm.red[2][g], sm.red[3][g])) * a.scale_log2;
            named_sync_softmax();
            // pass 2: P = 2^(s*scale*log2e - max), hi/lo bf16 parts, sums
            float sum[16];
#pragma unroll
            for (int g = 0; g < 16; ++g) sum[g] = 0.f;
            for (int q = 0; q < npairs; ++q) {
                uint32_t v[16];
                tmem_ld16(lane_addr + q * 16, v);
                tmem_ld_wait();
                const int idx = 2 * q + half;
                const bool valid = idx < x.nsel && x.blk[idx] * kBlock + key_in_blk <= x.p;
                uint8_t* chunk = sm.p[2 * q + half];
                const int ch = key_in_blk >> 3, within = (key_in_blk & 7) * 2;
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                    const float pr = valid ? exp2f(fmaf(__uint_as_float(v[g]), a.scale_log2, -ms[g])) : 0.f;
                    sum[g] += pr;
                    const __nv_bfloat16 hi_b = __float2bfloat16_rn(pr);
                    const __nv_bfloat16 lo_b = __float2bfloat16_rn(pr - __bfloat162float(hi_b));
                    const uint32_t sw = static_cast<uint32_t>((ch ^ (g & 7)) << 4) + within;
                    *reinterpret_cast<__nv_bfloat16*>(chunk + g * 128 + sw) = hi_b;
                    *reinterpret_cast<__nv_bfloat16*>(chunk + (16 + g) * 128 + sw) = lo_b;
                }
            }
            fence_proxy_async_smem();  // P is read by the tensor cores
#pragma unroll
            for (int g = 0; g < 16; ++g) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum[g] += __shfl_xor_sync(0xffffffffu, sum[g], o);
            }
            if (lane < 16) {
                float m = sum[0];
#pragma unroll
                for (int g = 1; g < 16; ++g) m = lane == g ? sum[g] : m;
                sm.red[warp][lane] = m;
            }
            named_sync_softmax();
            if (tid < 16) sm.rowsum[tid] = sm.red[0][tid] + sm.red[1][tid] + sm.red[2][tid] + sm.red[3][tid];
            tc_fence_before();
            mbar_arrive(&sm.p_full);
            // epilogue: out[r, h*G + g, d] = (O_hi + O_lo)[d, g] / sum[g]
            if (!mbar_wait(&sm.o_full, it & 1, a.err)) break;
            tc_fence_after();
            uint32_t ohi[16], olo[16];
            tmem_ld16(lane_addr + kOCol, ohi);
            tmem_ld16(lane_addr + kOCol + 16, olo);
            tmem_ld_wait();
            named_sync_softmax();  // rowsum visible
            const int d = tid;
            const int64_t base = (static_cast<int64_t>(x.r) * a.H * a.G + static_cast<int64_t>(x.h) * a.G) * kHeadDim + d;
            for (int g = 0; g < a.G; ++g) {
                const float o = (__uint_as_float(ohi[g]) + __uint_as_float(olo[g])) / sm.rowsum[g];
                if (a.out_bf16)
                    reinterpret_cast<__nv_bfloat16*>(a.out)[base + static_cast<int64_t>(g) * kHeadDim] = __float2bfloat16_rn(o);
                else
                    reinterpret_cast<float*>(a.out)[base + static_cast<int64_t>(g) * kHeadDim] = o;
            }
            tc_fence_before();
            ++it;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

cudaError_t run_prefill_attend(const PrefillAttendArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(AttendSmem) + 1024;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_attend_kernel), smem);
    if (e != cudaSuccess) return e;
    const int64_t items = static_cast<int64_t>(a.total_rows) * a.H;
    const int grid = static_cast<int>(items < device_sm_count() ? items : device_sm_count());
    prefill_attend_kernel<<<grid, kPaThreads, smem, stream>>>(*a.q_map, *a.k_map, *a.v_map, a);
    return cudaGetLastError();
}

}  // namespace msa
