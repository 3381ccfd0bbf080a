// Decode stage 2b+3 as one thread-block cluster per (query row, KV head) of
// the decode family (sequences with up to kDecodeMaxRows rows).
//
// PR #1388 "minimax_m3: a CUDA backend for MiniMax-M3.1-Flash ...", native
// Metal family commit: a decode row attends to its chosen blocks in partial
// results that are merged afterwards.  Here the partials never leave the
// chip:
//   - the 8 CTAs of a cluster each take two of the (up to 16) kept blocks,
//     stage their K and V by TMA (128-byte swizzle) and compute S = Q K^T
//     and O = P V for the group's 16 query heads on mma.sync (P split into
//     bf16 hi + lo parts so the weights keep ~16 significant bits);
//   - when a batch has more (row, head) problems than clusters of 8 fit on
//     the GPU at once, clusters of 4 CTAs take four blocks each, in two
//     rounds of two through the same tiles, the softmax carried from round
//     to round with a running max (the partial O rescaled by 2^(m - m'));
//     one wave of clusters of 4 ends sooner than two waves of clusters of 8;
//   - each CTA stores the (m, l, O) rows of its heads' partials straight
//     into the shared memory of the CTA that finishes them (head g: CTA
//     g / (16 / cluster size); distributed shared memory, remote stores: no
//     round trip); after one cluster barrier each CTA combines its heads from
//     its own shared memory:
//         M = max m_c,  L = sum l_c 2^(m_c - M),  out = sum O_c 2^(m_c - M) / L
//   - the kept blocks come from the pooled index scores (every CTA runs the
//     same deterministic selection) or from a given list;
//   - an int8 key/value cache (PR #1388, native Metal family commit: int8
//     values with a scale per position and head) lands by TMA as int8 tiles
//     that every thread rewrites row by row, in place, as bf16 (exact: the
//     integers have at most 8 significant bits); the key scale multiplies the
//     row's scores and the value scale its softmax weights before P V, so the
//     MMAs are the same as for a bf16 cache.
// Launched after the index scan as a programmatic dependent launch: q and
// the sequence metadata are read before waiting for the scan to finish.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace msa {

constexpr int kClThreads = 128;

struct __align__(1024) ClusterSmem {
    uint16_t k[2][2][64 * 64];  // [block][dim half][key][64 dims], 128B-swizzled by TMA
    uint16_t v[2][2][64 * 64];
    uint16_t q[16 * 128];       // [head][dim], 16-byte chunks XOR-swizzled by row
    uint16_t p[2][16 * 128];    // [hi/lo][head][128 keys], same swizzle
    float recv_o[16][128];  // partial outputs of my heads: row c * heads-per-CTA + slot from source CTA c
    float recv_ml[16][2];   // their (max in the log2 domain, sum)
    float wmax[4][16];
    float wsum[4][16];
    float kvscale[2][2][64];         // int8 cache: [key/value][block][key] scales of this CTA's blocks
    uint64_t bar_k;  // the round's K tiles landed
    uint64_t bar_v;  // the round's V tiles landed
    int32_t sel[kMaxTopK];
    int32_t nsel;
    int32_t meta_ok;
    SelectSmem<kClThreads> select;
};

__device__ __forceinline__ uint32_t cl_swz(int row, int chunk, int row_bytes) {
    return row * row_bytes + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void cl_ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void cl_ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                             uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void cl_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster; release/acquire orders shared-memory
// writes before the barrier with reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of `p` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
    return out;
}
__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float x, float y) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y) : "memory");
}
// Split cluster barrier: arrive early, wait just before the first remote
// shared-memory access (every peer has then started).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// grid (kCl, H, rows), cluster (kCl, 1, 1): CTA `rank` of the cluster of (row, KV head h) takes
// kept blocks rank + kCl * i, two per round (kCl = 8: one round; kCl = 4: two rounds through the
// same tiles, the softmax carried over with a running max), and finishes heads kHpc * rank ...
template <bool kSelGiven, bool kInt8, int kCl>
__global__ void __launch_bounds__(kClThreads, 2) decode_cluster_kernel(const __grid_constant__ CUtensorMap k_map,
                                                                    const __grid_constant__ CUtensorMap v_map,
                                                                    const DecodeAttendArgs a) {
    static_assert(kCl == 8 || kCl == 4, "clusters of 8 or 4 CTAs");
    constexpr int kBlk = kMaxTopK / kCl;  // kept blocks per CTA
    constexpr int kRounds = kBlk / 2;     // two blocks (64 KB of K and V) per round
    constexpr int kHpc = 16 / kCl;        // heads each CTA combines
    extern __shared__ uint8_t smem_raw[];
    ClusterSmem& sm = *reinterpret_cast<ClusterSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int rank = static_cast<int>(cluster_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, G = a.G;
    const int h = blockIdx.y;
    int b, row_in_seq;
    if (a.drow_prefix != nullptr) {
        // compact grid (fused path): blockIdx.z is a decode-family row; its sequence comes from
        // the prefix of rows the index scan wrote, so this wait comes first
        pdl_wait();
        const int z = blockIdx.z, B = a.num_seqs;
        const int total = a.drow_prefix[B];
        if (z == 0 && h == 0 && rank == 0 && tid == 0 && total > static_cast<int>(gridDim.z))
            atomicOr(a.err, kErrBadMetadata);  // the host's row count is below the device metadata's
        if (z >= total) return;  // a host count above the device's: nothing to do
        int lo = 0, hi = B;  // largest b with drow_prefix[b] <= z
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (a.drow_prefix[mid] <= z) lo = mid; else hi = mid;
        }
        b = lo;
        row_in_seq = z - a.drow_prefix[b];
    } else {  // one entry per row slot: b * RS + i is row i of sequence b
        b = blockIdx.z / a.rows_per_seq;
        row_in_seq = blockIdx.z - b * a.rows_per_seq;
    }
    const int row_slot = b * a.rows_per_seq + row_in_seq;  // the row's pooled-score slot

    // ---- prologue: only inputs that no earlier kernel of the step writes
    const int nrows = a.cu_rows[b + 1] - a.cu_rows[b];
    // not a decode-family sequence, or no such row (the whole cluster returns)
    if (nrows < 1 || nrows > kDecodeMaxRows || row_in_seq >= nrows) return;
    const int r = a.cu_rows[b] + row_in_seq;
    const int L = a.cache_lens[b];
    // nrows > rows_per_seq: more rows than the grid and the pooled scores have slots for
    const bool meta_ok = !(r < 0 || r >= a.total_rows || L < nrows || L > a.max_cache_len || nrows > a.rows_per_seq) &&
                         seq_rows_ok(a.cache, b, L, a.cache_tokens);
    if (tid == 0) {
        mbar_init(&sm.bar_k, 4);  // one arrival from each of warps 0-3 (with the bytes it copies)
        mbar_init(&sm.bar_v, 4);
        fence_mbar_init();
    }
    if (tid == 32) {  // the K/V descriptors ride along with the wait, not behind the selection
        prefetch_tmap(&k_map);
        prefetch_tmap(&v_map);
    }
    if (meta_ok) {
        const uint16_t* qrow = a.q + (static_cast<int64_t>(r) * H * G + static_cast<int64_t>(h) * G) * kHeadDim;
        for (int c = tid; c < 16 * 16; c += kClThreads) {  // 16 heads x 16 chunks of 8 dims
            const int g = c >> 4, ch = c & 15;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (g < G) val = *reinterpret_cast<const uint4*>(qrow + g * kHeadDim + ch * 8);
            *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sm.q) + cl_swz(g, ch, 256)) = val;
        }
        if constexpr (kSelGiven) {
            if (tid < kMaxTopK)
                sm.sel[tid] = tid < a.top_k ? a.sel_in[(static_cast<int64_t>(r) * H + h) * a.top_k + tid] : -1;
            if (tid == 0) sm.nsel = min(max(a.nsel_in[static_cast<int64_t>(r) * H + h], 0), a.top_k);
        }
    }
    // a given count of kept blocks (the same in every thread of the cluster)
    const int nsel_given = kSelGiven && meta_ok ? a.nsel_in[static_cast<int64_t>(r) * H + h] : 1;
    pdl_wait();  // the index scan (pooled scores, error word) is complete and visible
    // A kernel launched after this one as a programmatic dependent may start now.  The
    // scan's header clears (tickets of the prompt indexer) have landed by this point;
    // a dependent that reads anything this grid writes waits for it to finish first.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!meta_ok) {
        if (tid == 0 && rank == 0) atomicOr(a.err, kErrBadMetadata);
        return;  // the whole cluster returns: before any cluster barrier
    }
    if (nsel_given < 1 || nsel_given > a.top_k) {
        if (tid == 0 && rank == 0) atomicOr(a.err, kErrBadMetadata);
        if (nsel_given < 1) {  // no kept block: the softmax is empty; the outputs are zeros
            for (int t = tid; t < kHpc * kHeadDim / 2; t += kClThreads) {  // CTA `rank` owns heads kHpc * rank ...
                const int g = kHpc * rank + t / (kHeadDim / 2), d = (t % (kHeadDim / 2)) * 2;
                if (g < G) {
                    const int64_t oi = (static_cast<int64_t>(r) * H * G + static_cast<int64_t>(h) * G + g) * kHeadDim + d;
                    if (a.out_bf16)
                        *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + oi) = pack_bf16x2(0.f, 0.f);
                    else
                        *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + oi) = make_float2(0.f, 0.f);
                }
            }
            return;  // every CTA of the cluster takes this branch, before any cluster barrier
        }
    }
    cluster_arrive_relaxed();  // matched by cluster_wait() before the first remote store
    const int p = L - nrows + row_in_seq;  // this row's position
    const int J = p / kBlock;
    // ---- the kept blocks: k < nsel, block kept(k); this CTA takes k = rank + kCl * i, two a round
    int nsel, others = 0;
    if constexpr (kSelGiven) {
        __syncthreads();  // the given list (read before the wait) visible to every thread
        nsel = sm.nsel;
    } else {
        // the fused selection ranks the blocks; the kept list is [best first ..., J] and
        // the copies go out right after the ranking (the caller's ascending list is written
        // while they are in flight)
        const float* pooled = a.pooled + (static_cast<int64_t>(row_slot) * H + h) * a.max_blocks;
        others = cta_select_ranked<kClThreads>(pooled, J, a.top_k, sm.select);
        nsel = others + 1;
    }
    auto kept = [&](int k) { return kSelGiven ? sm.sel[k] : (k < others ? sm.select.picked[k] : J); };
    int nmy = 0;
    int blk[kBlk];
#pragma unroll
    for (int i = 0; i < kBlk; ++i) {
        blk[i] = J;
        if (rank + kCl * i < nsel) {
            ++nmy;
            blk[i] = kept(rank + kCl * i);
            if (blk[i] < 0 || blk[i] > J) {  // a given selection outside the causal range
                if (tid == 0) atomicOr(a.err, kErrBadMetadata);
                blk[i] = J;
            }
        }
    }

    const int grp = lane >> 2, tig = lane & 3;
    const int my_blk = warp >> 1, key0 = (warp & 1) * 32;  // the warp's block in a round, first key in it
    // running softmax state of heads grp and grp + 8 over this CTA's rounds (the same in every
    // warp): max (log2 domain) and sum; O[heads, 32w .. 32w+32) in the MMA accumulators
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
    float o[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    int late_phase = -1;  // a copy that did not land in time: its phase, waited for again at the end
    int k_armed = -1;     // last phase of the K barrier with copies armed (round r arms phase r)
    // Warps 0-3 issue a round's copies, each arming the barrier with its own bytes first (warps
    // without a copy arrive without bytes): one thread issues TMA boxes at a bounded rate, so
    // four issuers land the 64 KB sooner than one.  K goes first, so that S and the softmax
    // overlap the V transfer, and a later round's K leaves as soon as the last round's S has read
    // the K tiles.  bf16: warp w copies dims 64 (w & 1) .. of block w / 2; int8 (one 128-dim box
    // a tile): warp w copies the K (w < 2) or V tile of block w & 1.  Called by lane 0 of warps
    // 0-3; every call arrives once on its barrier.
    auto copy_row = [&](int bi) {
        int64_t row = block_row(a.cache, b, static_cast<int64_t>(bi) * kBlock);
        if (row < 0) {  // page outside the pool
            atomicOr(a.err, kErrBadMetadata);
            row = 0;
        }
        return static_cast<int>(row);
    };
    auto issue_k = [&](int nr, int bA, int bB) {
        const int i = kInt8 ? (warp & 1) : (warp >> 1);
        if (i < nr && (!kInt8 || warp < 2)) {
            const int tok = copy_row(i == 0 ? bA : bB);
            if constexpr (kInt8) {  // one int8 tile per block into the upper 8 KB, widened in place below
                mbar_arrive_expect_tx(&sm.bar_k, 64 * 128);
                tma_load_3d(sm.k[i][1], &k_map, &sm.bar_k, 0, h, tok);
            } else {
                const int half = warp & 1;
                mbar_arrive_expect_tx(&sm.bar_k, 64 * 64 * 2);
                tma_load_3d(sm.k[i][half], &k_map, &sm.bar_k, 64 * half, h, tok);
            }
        } else {
            mbar_arrive(&sm.bar_k);
        }
    };
    auto issue_v = [&](int nr, int bA, int bB) {
        const int i = kInt8 ? (warp & 1) : (warp >> 1);
        if (i < nr && (!kInt8 || warp >= 2)) {
            const int tok = copy_row(i == 0 ? bA : bB);
            if constexpr (kInt8) {
                mbar_arrive_expect_tx(&sm.bar_v, 64 * 128);
                tma_load_3d(sm.v[i][1], &v_map, &sm.bar_v, 0, h, tok);
            } else {
                const int half = warp & 1;
                mbar_arrive_expect_tx(&sm.bar_v, 64 * 64 * 2);
                tma_load_3d(sm.v[i][half], &v_map, &sm.bar_v, 64 * half, h, tok);
            }
        } else {
            mbar_arrive(&sm.bar_v);
        }
    };
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
        const int nr = min(max(nmy - 2 * rd, 0), 2);  // this round's blocks (uniform over the CTA)
        const int bA = blk[2 * rd], bB = blk[2 * rd + 1];
        if (rd > 0) __syncthreads();  // the V tiles, P and the row statistics of the last round are read
        if (lane == 0 && warp < 4) {
            if (rd == 0) issue_k(nr, bA, bB);  // a later round's K left after the last round's S
            issue_v(nr, bA, bB);
        }
        if (rd == 0) k_armed = 0;
        if (!kSelGiven && rd == 0 && rank == 0 && a.sel_out != nullptr && tid < a.top_k) {
            // the kept blocks ascending, for the caller, while the first copies are in flight
            const int64_t o = (static_cast<int64_t>(r) * H + h) * a.top_k;
            if (tid < nsel) {
                const int v = kept(tid);
                int pos = 0;
                for (int u = 0; u < nsel; ++u) pos += kept(u) < v;
                a.sel_out[o + pos] = v;
            } else {
                a.sel_out[o + tid] = -1;
            }
            if (tid == 0) a.nsel_out[static_cast<int64_t>(r) * H + h] = nsel;
        }
        if constexpr (kInt8) {
            // scales of the round's keys (thread = block tid / 64, key tid % 64); keys past p are
            // masked and may lie past the sequence's cache rows, so they are not read (scale 0,
            // as for a block this CTA does not have)
            const int i = tid >> 6, key = tid & 63;
            const int bi = i == 0 ? bA : bB;
            float ks = 0.f, vs = 0.f;
            if (i < nr && bi * kBlock + key <= p) {
                const int64_t row = block_row(a.cache, b, static_cast<int64_t>(bi) * kBlock);
                if (row >= 0) {
                    const int64_t si = (row + key) * H + h;
                    ks = a.k_scale[si];
                    vs = a.v_scale[si];
                }
            }
            sm.kvscale[0][i][key] = ks;
            sm.kvscale[1][i][key] = vs;
        }
        if (nr == 0) break;  // no block left for this CTA (uniform)
        // the K tiles (an int8 cache: K and V, widened together below)
        if (!__syncthreads_and(mbar_wait(&sm.bar_k, rd & 1, a.err) &&
                               (!kInt8 || mbar_wait(&sm.bar_v, rd & 1, a.err)))) {
            late_phase = rd & 1;  // copy never landed: no more keys
            break;
        }
        if constexpr (kInt8) {
            // every thread widens whole key rows (K rows then V rows of the round's blocks)
            for (int rr = tid; rr < nr * 2 * 64; rr += kClThreads) {
                const bool is_v = rr >= nr * 64;
                const int r2 = is_v ? rr - nr * 64 : rr;
                convert_i8_row(reinterpret_cast<uint8_t*>(is_v ? sm.v[r2 >> 6][0] : sm.k[r2 >> 6][0]), r2 & 63);
            }
            __syncthreads();  // bf16 tiles and scales visible to every warp
        }

        // ---- S = Q K^T: warp w owns keys [32w, 32w+32) of the round's 128 (block w/2)
        const bool warp_live = my_blk < nr;
        const int wblk = my_blk == 0 ? bA : bB;
        float s[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        if (warp_live) {
            const uint32_t q_base = smem_u32(sm.q);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // 16 dims per step
                const int mi = lane >> 3;
                uint32_t a0, a1, a2, a3;
                cl_ldsm_x4(q_base + cl_swz((mi & 1) * 8 + (lane & 7), kk * 2 + (mi >> 1), 256), a0, a1, a2, a3);
                const int dim = kk * 16 + (mi & 1) * 8;
                const uint32_t kb = smem_u32(sm.k[my_blk][dim >> 6]);
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {  // two 8-key tiles per ldmatrix
                    const int key = key0 + pp * 16 + (mi >> 1) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    cl_ldsm_x4(kb + cl_swz(key, (dim & 63) >> 3, 128), b0, b1, b2, b3);
                    cl_mma(s[pp * 2 + 0], a0, a1, a2, a3, b0, b1);
                    cl_mma(s[pp * 2 + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        // scale (log2 domain; times the key's scale for an int8 cache), causal mask inside the
        // local block, row maxima
        float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + nt * 8 + tig * 2 + (e & 1);
                const bool valid = warp_live && wblk * kBlock + key <= p;
                const float f = kInt8 ? a.scale_log2 * sm.kvscale[0][my_blk][key] : a.scale_log2;
                s[nt][e] = valid ? s[nt][e] * f : -INFINITY;
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
        if constexpr (kRounds > 1) {
            if (rd + 1 < kRounds) {  // every warp has read the K tiles: the next round's K leaves now
                if (lane == 0 && warp < 4)
                    issue_k(min(max(nmy - 2 * (rd + 1), 0), 2), blk[2 * rd + 2], blk[2 * rd + 3]);
                k_armed = rd + 1;
            }
        }
        // new running maxima; the old sums and outputs are rescaled to them
        float mnew[2], alpha[2], lsum[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int hg = grp + 8 * i;
            const float mr = fmaxf(fmaxf(sm.wmax[0][hg], sm.wmax[1][hg]), fmaxf(sm.wmax[2][hg], sm.wmax[3][hg]));
            if constexpr (kRounds > 1) {
                mnew[i] = fmaxf(mrun[i], mr);
                alpha[i] = mrun[i] == -INFINITY ? 0.f : exp2f(mrun[i] - mnew[i]);
            } else {  // one round: nothing to carry over
                mnew[i] = mr;
                alpha[i] = 0.f;
            }
        }
        // a row with no valid key so far gets P = 0
        const float msafe[2] = {mnew[0] == -INFINITY ? 0.f : mnew[0], mnew[1] == -INFINITY ? 0.f : mnew[1]};
        uint8_t* phi = reinterpret_cast<uint8_t*>(sm.p[0]);
        uint8_t* plo = reinterpret_cast<uint8_t*>(sm.p[1]);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const float p0 = exp2f(s[nt][0] - msafe[0]), p1 = exp2f(s[nt][1] - msafe[0]);
            const float p2 = exp2f(s[nt][2] - msafe[1]), p3 = exp2f(s[nt][3] - msafe[1]);
            lsum[0] += p0 + p1;
            lsum[1] += p2 + p3;
            const int key = warp * 32 + nt * 8 + tig * 2;  // key index among the round's 128
            // int8 cache: the value scale of each key folds into its weight (the sum keeps the weight)
            const float vs0 = kInt8 ? sm.kvscale[1][key >> 6][key & 63] : 1.f;
            const float vs1 = kInt8 ? sm.kvscale[1][key >> 6][(key + 1) & 63] : 1.f;
            const float w0 = p0 * vs0, w1 = p1 * vs1, w2 = p2 * vs0, w3 = p3 * vs1;
            const int chunk = key >> 3, within = (key & 7) * 2;
            const uint32_t h01 = pack_bf16x2(w0, w1), h23 = pack_bf16x2(w2, w3);
            *reinterpret_cast<uint32_t*>(phi + cl_swz(grp, chunk, 256) + within) = h01;
            *reinterpret_cast<uint32_t*>(phi + cl_swz(grp + 8, chunk, 256) + within) = h23;
            *reinterpret_cast<uint32_t*>(plo + cl_swz(grp, chunk, 256) + within) =
                pack_bf16x2(w0 - bf16_lo(h01), w1 - bf16_hi(h01));
            *reinterpret_cast<uint32_t*>(plo + cl_swz(grp + 8, chunk, 256) + within) =
                pack_bf16x2(w2 - bf16_lo(h23), w3 - bf16_hi(h23));
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
        // P and the row sums written; a bf16 cache's V tiles landed
        if (!__syncthreads_and(kInt8 || mbar_wait(&sm.bar_v, rd & 1, a.err))) {
            late_phase = rd & 1;  // copy never landed: no more keys (the output is flagged)
            break;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int hg = grp + 8 * i;
            const float lr = sm.wsum[0][hg] + sm.wsum[1][hg] + sm.wsum[2][hg] + sm.wsum[3][hg];
            lrun[i] = kRounds > 1 ? lrun[i] * alpha[i] + lr : lr;
            mrun[i] = mnew[i];
        }
        if constexpr (kRounds > 1) {
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {  // accumulator rows grp (c0, c1) and grp + 8 (c2, c3)
                o[nt][0] *= alpha[0];
                o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1];
                o[nt][3] *= alpha[1];
            }
        }

        // ---- O[:, 32w .. 32w+32) += P V over the round's 64 * nr keys
        for (int kk = 0; kk < 4 * nr; ++kk) {  // 16 keys per step
            const int mi = lane >> 3;
            const int row = (mi & 1) * 8 + (lane & 7);
            uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
            cl_ldsm_x4(smem_u32(sm.p[0]) + cl_swz(row, kk * 2 + (mi >> 1), 256), a0, a1, a2, a3);
            cl_ldsm_x4(smem_u32(sm.p[1]) + cl_swz(row, kk * 2 + (mi >> 1), 256), l0, l1, l2, l3);
            const int vb = kk >> 2;  // block of these keys
#pragma unroll
            for (int np = 0; np < 2; ++np) {  // pairs of 8-dim tiles
                const int key = (kk & 3) * 16 + (mi & 1) * 8 + (lane & 7);
                const int dim = warp * 32 + np * 16 + (mi >> 1) * 8;
                uint32_t b0, b1, b2, b3;
                cl_ldsm_x4_t(smem_u32(sm.v[vb][dim >> 6]) + cl_swz(key, (dim & 63) >> 3, 128), b0, b1, b2, b3);
                cl_mma(o[np * 2 + 0], a0, a1, a2, a3, b0, b1);
                cl_mma(o[np * 2 + 1], a0, a1, a2, a3, b2, b3);
                cl_mma(o[np * 2 + 0], l0, l1, l2, l3, b0, b1);
                cl_mma(o[np * 2 + 1], l0, l1, l2, l3, b2, b3);
            }
        }
    }
    // ---- push my partial rows to their owners: head g is finished by CTA g / kHpc
    cluster_wait();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int g = grp + 8 * half;
        if (g < G) {
            const int owner = g / kHpc, slot = g % kHpc;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int dim = warp * 32 + nt * 8 + tig * 2;
                st_cluster_f32x2(map_to_rank(&sm.recv_o[rank * kHpc + slot][dim], owner), o[nt][2 * half],
                                 o[nt][2 * half + 1]);
            }
            if (warp == 0 && tig == 0)  // the (max, sum) of head g, the same in every warp
                st_cluster_f32x2(map_to_rank(&sm.recv_ml[rank * kHpc + slot][0], owner), mrun[half], lrun[half]);
        }
    }
    cluster_sync();  // all pushes have landed; no remote access follows

    // ---- combine my heads kHpc * rank .. + kHpc - 1; thread t owns kHpc dims of one
    constexpr int kTpHead = kClThreads / kHpc;  // threads per head
    const int slot = tid / kTpHead;
    const int g = kHpc * rank + slot;
    const int d = (tid % kTpHead) * kHpc;
    if (g < G) {
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kCl; ++c) M = fmaxf(M, sm.recv_ml[c * kHpc + slot][0]);
        float Ls = 0.f, ov[kHpc];
#pragma unroll
        for (int j = 0; j < kHpc; ++j) ov[j] = 0.f;
#pragma unroll
        for (int c = 0; c < kCl; ++c) {
            const float mc = sm.recv_ml[c * kHpc + slot][0];
            const float w = mc == -INFINITY ? 0.f : exp2f(mc - M);
            Ls = fmaf(w, sm.recv_ml[c * kHpc + slot][1], Ls);
#pragma unroll
            for (int j = 0; j < kHpc; j += 2) {  // two dims per load
                const float2 oc = *reinterpret_cast<const float2*>(&sm.recv_o[c * kHpc + slot][d + j]);
                ov[j] = fmaf(w, oc.x, ov[j]);
                ov[j + 1] = fmaf(w, oc.y, ov[j + 1]);
            }
        }
        const float inv = 1.f / Ls;
        const int64_t oi = (static_cast<int64_t>(r) * H * G + static_cast<int64_t>(h) * G + g) * kHeadDim + d;
#pragma unroll
        for (int j = 0; j < kHpc; j += 2) {
            if (a.out_bf16)
                *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + oi + j) =
                    pack_bf16x2(ov[j] * inv, ov[j + 1] * inv);
            else
                *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + oi + j) =
                    make_float2(ov[j] * inv, ov[j + 1] * inv);
        }
    }
    if (late_phase >= 0 && tid == 0) {  // the copies still in flight land before the CTA exits
        mbar_wait(&sm.bar_k, k_armed & 1, nullptr);  // the last K phase armed (the earlier ones completed)
        mbar_wait(&sm.bar_v, late_phase, nullptr);
    }
}

// Shared memory a CTA asks for: what it uses, or (one CTA per SM) more than half of an SM's
// 228 KB, so that no two CTAs share an SM and each takes in its 64 KB of K and V alone.
constexpr size_t kClSmem = sizeof(ClusterSmem) + 1024;
constexpr size_t kClSmemAlone = 120 * 1024;
static_assert(kClSmem <= kClSmemAlone && 2 * (kClSmemAlone + 1024) > 228 * 1024, "one CTA per SM");

template <bool kSelGiven, bool kInt8, int kCl>
static cudaError_t launch_cluster(const DecodeAttendArgs& a, int rows, bool after_scan, size_t smem,
                                  cudaStream_t stream) {
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(decode_cluster_kernel<kSelGiven, kInt8, kCl>), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCl, a.H, rows);
    cfg.blockDim = dim3(kClThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_scan ? 2 : 1;  // overlap the prologue with the index scan's tail
    e = cudaLaunchKernelEx(&cfg, decode_cluster_kernel<kSelGiven, kInt8, kCl>, *a.k_map, *a.v_map, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Clusters of 8 CTAs of this kernel, each CTA with `alone` ? kClSmemAlone : kClSmem bytes of
// shared memory, that the current device runs at once (queried once per device; 0 if the
// query fails).
static int clusters_of_8_at_once(bool alone) {
    static int counts[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int& c = counts[alone][dev & 63];
    if (c == 0) {
        const size_t smem = alone ? kClSmemAlone : kClSmem;
        if (ensure_smem_limit(reinterpret_cast<const void*>(decode_cluster_kernel<false, false, 8>), smem) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(8, 1, 1);
        cfg.blockDim = dim3(kClThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 8;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, decode_cluster_kernel<false, false, 8>, &cfg) != cudaSuccess) {
            cudaGetLastError();  // clear the query's error
            return 0;
        }
        c = n > 0 ? n : -1;
    }
    return c > 0 ? c : 0;
}

cudaError_t run_decode_cluster(const DecodeAttendArgs& a, bool after_scan, cudaStream_t stream) {
    const bool given = a.pooled == nullptr;
    const int rows = a.drow_prefix != nullptr ? a.decode_rows : a.num_seqs * a.rows_per_seq;
    // Clusters of 8 finish a (row, head) soonest, one CTA per SM when they all fit that way;
    // when there are more problems than clusters of 8 fit at once, clusters of 4 (two rounds a
    // CTA) run them in fewer waves.
    const int64_t problems = static_cast<int64_t>(rows) * a.H;
    const int cap_alone = clusters_of_8_at_once(true);
    const int cap = clusters_of_8_at_once(false);
    const bool alone = cap_alone > 0 && problems <= cap_alone;
    const bool four = !alone && cap > 0 && problems > cap;
    const size_t smem = alone ? kClSmemAlone : kClSmem;
    if (a.kv_int8) {
        if (given) return four ? launch_cluster<true, true, 4>(a, rows, after_scan, smem, stream)
                               : launch_cluster<true, true, 8>(a, rows, after_scan, smem, stream);
        return four ? launch_cluster<false, true, 4>(a, rows, after_scan, smem, stream)
                    : launch_cluster<false, true, 8>(a, rows, after_scan, smem, stream);
    }
    if (given) return four ? launch_cluster<true, false, 4>(a, rows, after_scan, smem, stream)
                           : launch_cluster<true, false, 8>(a, rows, after_scan, smem, stream);
    return four ? launch_cluster<false, false, 4>(a, rows, after_scan, smem, stream)
                : launch_cluster<false, false, 8>(a, rows, after_scan, smem, stream);
}

}  // namespace msa
