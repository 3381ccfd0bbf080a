// Decode stage 1+2a: lightning-indexer scan with the block max-pool fused in.
//
// For every sequence of the decode family (1 to 8 query rows, row i of n at
// p = L - n + i) and every KV head h, computes the pooled index score of
// every block j for each row:
//     m_j = max_{t in block j, t <= p}  iq[r,h,:] . ik[t,h,:]
// ("MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120)", "What this fixes":
// blocks are scored by their largest index score; PR #1388 "minimax_m3: a
// CUDA backend ...": index scores are taken per row and key head).  Only the pooled scores (4 bytes per block
// and head) leave the kernel; the per-position scores live in registers.
//
// The scan is HBM-bound: each cached position carries H x 64 bf16 index-key
// values (128 B per head) that are read exactly once.  Work unit = one
// 64-position block of one sequence with all H heads: H x 8 KB of contiguous
// memory (token-major cache).  One CTA per SM takes an even share of all
// units of all decode sequences (the split is computed on the device from
// the per-sequence lengths, so ragged batches balance).  A producer lane
// streams units into a ring of shared-memory stages with TMA tile loads (one
// 64-position x 64-dim box per head, 128-byte swizzle, mbarrier completion),
// keeping up to kStages units (192 KB) in flight per SM; consumer warp w
// owns stage w and reduces whole units on its own, so the loop has no
// CTA-wide barrier.  The dot products run on the tensor cores (mma.sync
// m16n8k16: A = 16 positions x 16 index dims from ldmatrix, B = the index
// query in column 0), about 50 instructions per head and block instead of
// ~500 on the FP32 pipes; fp32 accumulation keeps integer scores exact.
#include "common.cuh"
#include "internal.h"

namespace msa {

// kShared: one index key per position for all heads (a unit is one 8 KB box,
// read once for the H heads' queries), else one key per head (H boxes).
template <int H, bool kShared>
struct ScanCfg {
    static constexpr int kHeadBytes = kBlock * kIndexDim * 2;                 // 8 KB: [64 pos][64 dims]
    static constexpr int kKeyHeads = kShared ? 1 : H;
    static constexpr int kUnitBytes = kKeyHeads * kHeadBytes;
    static constexpr int kStages = kShared ? 16 : ((H == 8) ? 3 : 6);         // <= 192 KB of ring
    static constexpr int kConsumers = kStages;                                // one warp per stage
    static constexpr int kThreads = 32 * (kConsumers + 1);                    // + producer warp
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct ScanSeqState {
    int b = -1, L = 0, r = 0, n = 1;  // sequence, cache length, first row, rows
};

// Advance to the sequence holding unit u and refresh its metadata.
__device__ __forceinline__ bool scan_locate(const ScanArgs& a, const int32_t* prefix, int64_t u, int& b,
                                            ScanSeqState& st) {
    while (u >= prefix[b + 1]) ++b;
    if (b != st.b) {
        st.b = b;
        const int r = a.cu_rows[b];
        const int nr = min(max(a.cu_rows[b + 1] - r, 1), kDecodeMaxRows);
        const int L = min(max(a.cache_lens[b], 0), a.max_cache_len);
        // more rows than the pooled-score slots of a sequence (max_rows_per_seq understated) would
        // write into the next sequence's slots or past the buffer: inconsistent, like the rest
        const bool ok = r >= 0 && r + nr <= a.total_rows && L >= nr && nr <= a.rows_per_seq &&
                        seq_rows_ok(a.cache, b, L, a.cache_tokens);
        st.L = ok ? L : 0;  // inconsistent metadata: the sequence is skipped (the attention sets the error word)
        st.n = ok ? nr : 1;
        st.r = ok ? r : 0;
        return true;
    }
    return false;
}

template <int H, bool kShared>
__global__ void __launch_bounds__(ScanCfg<H, kShared>::kThreads, 1) decode_scan_kernel(const __grid_constant__ CUtensorMap ik_map,
                                                                             const ScanArgs a) {
    using Cfg = ScanCfg<H, kShared>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + Cfg::kStages * Cfg::kUnitBytes);
    uint64_t* empty = full + Cfg::kStages;
    int32_t* prefix = reinterpret_cast<int32_t*>(empty + Cfg::kStages);  // [num_seqs + 1]
    __shared__ int warp_tot[Cfg::kThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
        prefetch_tmap(&ik_map);
    }
    // Launched as a programmatic dependent of whatever kernel precedes it on the
    // stream: only the set-up above may overlap that kernel; every input read and
    // every write comes after it has completed and its memory is visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The attention kernel that follows uses these words; clear them here.
    if (blockIdx.x == 0)
        for (int i = tid; i < a.n_clear; i += Cfg::kThreads) a.clear_words[i] = 0;
    // Units per sequence: ceil(L/64) for decode sequences, 0 otherwise
    // (block-wide exclusive scan in chunks of kThreads).
    int carry = 0;
    for (int base = 0; base < a.num_seqs; base += Cfg::kThreads) {
        const int b = base + tid;
        int units = 0;
        const int nrows = b < a.num_seqs ? a.cu_rows[b + 1] - a.cu_rows[b] : 0;
        if (nrows >= 1 && nrows <= kDecodeMaxRows) {
            const int L = min(max(a.cache_lens[b], 0), a.max_cache_len);
            units = (L + kBlock - 1) / kBlock;
        }
        int incl = units;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int before = 0, chunk_total = 0;
        for (int w = 0; w < Cfg::kThreads / 32; ++w) {
            if (w < warp) before += warp_tot[w];
            chunk_total += warp_tot[w];
        }
        if (b < a.num_seqs) prefix[b] = carry + before + incl - units;
        __syncthreads();
        carry += chunk_total;
    }
    if (tid == 0) prefix[a.num_seqs] = carry;
    __syncthreads();
    if (blockIdx.x == 0 && a.drow_prefix != nullptr) {
        // exclusive prefix of decode-family rows per sequence: the decode attention's grid has
        // one entry per such row and finds the row's sequence here (same chunked block scan)
        int carry2 = 0;
        for (int base = 0; base < a.num_seqs; base += Cfg::kThreads) {
            const int b = base + tid;
            const int nr = b < a.num_seqs ? a.cu_rows[b + 1] - a.cu_rows[b] : 0;
            const int rows = nr >= 1 && nr <= kDecodeMaxRows ? nr : 0;
            int incl = rows;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (lane == 31) warp_tot[warp] = incl;
            __syncthreads();
            int before = 0, chunk_total = 0;
            for (int w = 0; w < Cfg::kThreads / 32; ++w) {
                if (w < warp) before += warp_tot[w];
                chunk_total += warp_tot[w];
            }
            if (b < a.num_seqs) a.drow_prefix[b] = carry2 + before + incl - rows;
            __syncthreads();
            carry2 += chunk_total;
        }
        if (tid == 0) a.drow_prefix[a.num_seqs] = carry2;
    }
    // the attention kernel may be scheduled now; it waits for this grid to
    // finish before it reads the pooled scores
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int64_t total = carry;
    const int64_t u0 = total * blockIdx.x / gridDim.x;
    const int64_t u1 = total * (blockIdx.x + 1) / gridDim.x;
    const int n = static_cast<int>(u1 - u0);
    if (n <= 0) return;
    int b0 = 0;
    {
        int lo = 0, hi = a.num_seqs;  // largest b with prefix[b] <= u0
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= u0) lo = mid; else hi = mid;
        }
        b0 = lo;
    }

    if (warp == Cfg::kConsumers) {
        // ---------------- producer: one lane streams units into the ring
        if (lane == 0) {
            int b = b0;
            ScanSeqState st;
            int armed = 0;  // stages armed so far (ring positions 0 .. armed-1)
            for (int i = 0; i < n; ++i) {
                const int64_t u = u0 + i;
                scan_locate(a, prefix, u, b, st);
                const int j = static_cast<int>(u - prefix[b]);
                const int npos = max(0, min(kBlock, st.L - j * kBlock));
                const int s = i % Cfg::kStages;
                if (i >= Cfg::kStages && !mbar_wait(&empty[s], ((i / Cfg::kStages) - 1) & 1, a.err)) break;
                if (npos > 0) {
                    // whole 64-position boxes; rows past the sequence are masked by the consumer
                    // and rows past the cache are zero-filled by the copy engine
                    mbar_arrive_expect_tx(&full[s], Cfg::kUnitBytes);
                    int64_t row = block_row(a.cache, b, static_cast<int64_t>(j) * kBlock);
                    if (row < 0) {  // page outside the pool
                        atomicOr(a.err, kErrBadMetadata);
                        row = 0;
                    }
                    const int tok = static_cast<int>(row);
#pragma unroll
                    for (int h = 0; h < Cfg::kKeyHeads; ++h)
                        tma_load_3d(ring + s * Cfg::kUnitBytes + h * Cfg::kHeadBytes, &ik_map, &full[s], 0, h, tok);
                } else {
                    mbar_arrive_expect_tx(&full[s], 0);
                }
                armed = i + 1;
            }
            // no copy of this lane may still be in flight when the CTA ends (after a timed-out
            // wait of a consumer, too): wait, bounded, for the last phase armed on every stage
            for (int s = 0; s < Cfg::kStages && s < armed; ++s)
                mbar_wait(&full[s], ((s + Cfg::kStages * ((armed - 1 - s) / Cfg::kStages)) / Cfg::kStages) & 1, a.err);
        }
        return;
    }

    // ---------------- consumer warp `warp` owns stage `warp`
    // B fragment of mma.m16n8k16 (col-major 16 x 8): lane (grp = lane/4,
    // tig = lane%4) holds B[2tig, 2tig+1][grp] and B[2tig+8, 2tig+9][grp].
    // Column i < n is the index query of the sequence's row i (the other
    // columns are zero), so one pass over the index keys serves all its rows;
    // accumulator lane (grp, tig) holds columns 2tig and 2tig+1 of positions
    // 16mt + grp and 16mt + grp + 8.
    const int grp = lane >> 2, tig = lane & 3;
    int b = b0;
    ScanSeqState st;
    const uint32_t stage = smem_u32(ring + warp * Cfg::kUnitBytes);
    for (int i = warp; i < n; i += Cfg::kStages) {
        const int64_t u = u0 + i;
        scan_locate(a, prefix, u, b, st);
        // this lane's B column: row grp of the sequence (if it exists)
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(
            a.iq + static_cast<int64_t>(st.r + (grp < st.n ? grp : 0)) * H * kIndexDim);
        const int j = static_cast<int>(u - prefix[b]);
        // valid positions of this block for the lane's two columns (rows 2tig, 2tig+1
        // at p = L - n + row): npos = p + 1 - 64 j, clamped to [0, 64]
        const int last0 = st.L - st.n + 2 * tig + 1 - j * kBlock;
        const int npos0 = 2 * tig < st.n ? max(0, min(kBlock, last0)) : 0;
        const int npos1 = 2 * tig + 1 < st.n ? max(0, min(kBlock, last0 + 1)) : 0;
        if (!mbar_wait(&full[warp], (i / Cfg::kStages) & 1, a.err)) break;
        if constexpr (kShared) {
            // one key tile for every head: the B columns are the (row, head) pairs,
            // column c = h * n + i, eight per pass
            const int ncols = st.n * H;
            for (int c0 = 0; c0 < ncols; c0 += 8) {
                const int cb = c0 + grp;  // this lane's B column
                uint32_t bq[4][2];
                if (cb < ncols) {
                    const int hb = cb / st.n, ib = cb - hb * st.n;
                    const uint32_t* qc = reinterpret_cast<const uint32_t*>(
                        a.iq + (static_cast<int64_t>(st.r + ib) * H + hb) * kIndexDim);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        bq[kk][0] = __ldg(qc + kk * 8 + tig);
                        bq[kk][1] = __ldg(qc + kk * 8 + 4 + tig);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) bq[kk][0] = bq[kk][1] = 0u;
                }
                float c[4][4];
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) c[mt][0] = c[mt][1] = c[mt][2] = c[mt][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        const int mi = lane >> 3;
                        const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
                        const int chunk = kk * 2 + (mi >> 1);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(stage + row * 128 + ((chunk ^ (row & 7)) << 4), a0, a1, a2, a3);
                        mma_bf16_16816(c[mt], a0, a1, a2, a3, bq[kk][0], bq[kk][1]);
                    }
                // accumulator columns of this lane: c0 + 2tig (e = 0) and c0 + 2tig + 1 (e = 1)
                int npe[2], he[2], ie[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int ce = c0 + 2 * tig + e;
                    he[e] = ce / st.n;
                    ie[e] = ce - he[e] * st.n;
                    npe[e] = ce < ncols ? max(0, min(kBlock, st.L - st.n + ie[e] + 1 - j * kBlock)) : 0;
                }
                float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    const int t0 = mt * 16 + grp, t1 = t0 + 8;
                    if (t0 < npe[0]) m0 = fmaxf(m0, c[mt][0]);
                    if (t1 < npe[0]) m0 = fmaxf(m0, c[mt][2]);
                    if (t0 < npe[1]) m1 = fmaxf(m1, c[mt][1]);
                    if (t1 < npe[1]) m1 = fmaxf(m1, c[mt][3]);
                }
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
                }
                if (grp == 0) {
                    const float me[2] = {m0, m1};
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (npe[e] > 0)
                            a.pooled[((static_cast<int64_t>(b) * a.rows_per_seq + ie[e]) * H + he[e]) * a.max_blocks + j] =
                                me[e];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[warp]);  // stage reusable
            continue;
        }
        if constexpr (!kShared) {  // one key tile per head
#pragma unroll 1
        for (int h = 0; h < H; ++h) {
            uint32_t bq[4][2];  // this head's index queries as B fragments (L1-resident rows)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                bq[kk][0] = grp < st.n ? __ldg(q32 + h * 32 + kk * 8 + tig) : 0u;
                bq[kk][1] = grp < st.n ? __ldg(q32 + h * 32 + kk * 8 + 4 + tig) : 0u;
            }
            float c[4][4];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) c[mt][0] = c[mt][1] = c[mt][2] = c[mt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    const int mi = lane >> 3;
                    const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
                    const int chunk = kk * 2 + (mi >> 1);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(stage + h * Cfg::kHeadBytes + row * 128 + ((chunk ^ (row & 7)) << 4), a0,
                            a1, a2, a3);
                    mma_bf16_16816(c[mt], a0, a1, a2, a3, bq[kk][0], bq[kk][1]);
                }
            // block maxima of columns 2tig (m0) and 2tig+1 (m1) over the valid positions
            float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int t0 = mt * 16 + grp, t1 = t0 + 8;
                if (t0 < npos0) m0 = fmaxf(m0, c[mt][0]);
                if (t1 < npos0) m0 = fmaxf(m0, c[mt][2]);
                if (t0 < npos1) m1 = fmaxf(m1, c[mt][1]);
                if (t1 < npos1) m1 = fmaxf(m1, c[mt][3]);
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
            }
            if (grp == 0) {  // lanes 0-3 store rows 2tig and 2tig+1
                float* pooled = a.pooled + (static_cast<int64_t>(b) * a.rows_per_seq * H + h) * a.max_blocks + j;
                const int64_t row_stride = static_cast<int64_t>(H) * a.max_blocks;
                if (npos0 > 0) pooled[(2 * tig) * row_stride] = m0;
                if (npos1 > 0) pooled[(2 * tig + 1) * row_stride] = m1;
            }
        }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[warp]);  // stage reusable
    }
}

template <int H, bool kShared>
static cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream) {
    using Cfg = ScanCfg<H, kShared>;
    const size_t smem = 1024 + static_cast<size_t>(Cfg::kStages) * Cfg::kUnitBytes + 2 * Cfg::kStages * sizeof(uint64_t) +
                        static_cast<size_t>(a.num_seqs + 1) * sizeof(int32_t);
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(decode_scan_kernel<H, kShared>), smem);
    if (e != cudaSuccess) return e;
    int64_t grid = device_sm_count();
    if (a.unit_bound < grid) grid = a.unit_bound > 0 ? a.unit_bound : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;  // set-up overlaps the previous kernel's tail
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_scan_kernel<H, kShared>, *a.ik_map, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t run_decode_scan(const ScanArgs& a, cudaStream_t stream) {
    switch (a.H) {
        case 1: return launch_scan<1, false>(a, stream);
        case 2: return a.ik_shared ? launch_scan<2, true>(a, stream) : launch_scan<2, false>(a, stream);
        case 4: return a.ik_shared ? launch_scan<4, true>(a, stream) : launch_scan<4, false>(a, stream);
        case 8: return a.ik_shared ? launch_scan<8, true>(a, stream) : launch_scan<8, false>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace msa
