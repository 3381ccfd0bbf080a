// Prompt-chunk stages 1+2 on tcgen05: lightning-indexer scores as a tensor-
// core GEMM with the block max-pool and a running top-k in its epilogue.
//
// PR #1388 "minimax_m3: a CUDA backend for MiniMax-M3.1-Flash ...": index
// scores and the top-16 block selection are made per row and key head;
// "MiniMax-M3 on 4x RTX PRO 6000 Blackwell (SM120)", "What this fixes": blocks
// are ranked by their largest index score and the current position's block
// is always kept.
//
// One CTA = one tile of 128 query rows of one sequence and one KV head (and,
// when the tiles alone would leave SMs idle, one of up to kIdxMaxSplit
// ranges of the positions; the last range to finish merges the ranges' lists
// of the 15 best blocks).  It streams the index keys in tiles of 256 positions:
//     D[128 rows, 256 positions] = iq[128, 64] . ik[256, 64]^T   (fp32, TMEM)
// one tcgen05.mma (M=128, N=256, K=16) per 16 index dims.  The accumulator is
// double-buffered in tensor memory (2 x 256 columns) so the MMA of tile n+1
// overlaps the epilogue of tile n.  Epilogue: thread i owns row i (TMEM lane
// i) and max-pools each 64-column block with one reduction load from tensor
// memory (tcgen05.ld.red .max: the block's maximum arrives with its values,
// no per-column compares), then inserts blocks j < J into a sorted register
// list of the 15 best (pooled score desc, j asc).  Blocks j < J lie wholly
// at positions <= p; the local block J is forced and needs no score.
// Scores are never written to memory.
//
// Warp roles: warps 0-7 epilogue (two per TMEM lane quarter, each taking two
// of a tile's four blocks), warp 8 TMA producer, warp 9 MMA issuer and
// tensor-memory owner.
#include "common.cuh"
#include "internal.h"

namespace msa {

constexpr int kIdxThreads = 320;  // 8 epilogue warps, producer, MMA issuer
constexpr int kIdxRows = 128;     // M
constexpr int kIdxCols = 256;     // N, positions per tile
constexpr int kIdxStages = 4;     // index-key tile ring
constexpr int kIdxTileBytes = kIdxCols * kIndexDim * 2;  // 32 KB
constexpr int kIdxABytes = kIdxRows * kIndexDim * 2;     // 16 KB

struct __align__(1024) IndexSmem {
    uint8_t b[kIdxStages][kIdxTileBytes];
    uint8_t a[kIdxABytes];
    uint64_t full[kIdxStages];
    uint64_t empty[kIdxStages];
    uint64_t a_full;
    uint64_t drain;  // the MMA issuer's last MMAs done before tensor memory is freed
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_base;
    int32_t seq, row0, nrows, ntiles, p0, L;
    int32_t n0, n1;  // this split's 256-position tiles [n0, n1)
    int32_t last;    // this CTA merges the splits' lists
    uint64_t half_list[kIdxRows][16];  // the second epilogue half's best blocks per row

};

// Which (sequence, row tile) CTA `tile` handles; false when beyond the end.
// Tiles of a sequence with n rows (n > kDecodeMaxRows):
// ceil(n / 128).  Walks the sequences (num_seqs is small).
__device__ bool find_tile(const PrefillIndexArgs& a, int tile, int& b, int& i0, int& n) {
    int acc = 0;
    for (int s = 0; s < a.num_seqs; ++s) {
        const int rows = a.cu_rows[s + 1] - a.cu_rows[s];
        if (rows <= kDecodeMaxRows) continue;  // the decode kernels take these
        const int t = (rows + kIdxRows - 1) / kIdxRows;
        if (tile < acc + t) {
            b = s;
            i0 = (tile - acc) * kIdxRows;
            n = rows;
            return true;
        }
        acc += t;
    }
    return false;
}

// Barrier of the eight epilogue warps (threads 0-255) only.
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// A thread's running list of its row's best blocks: key inserted into best[0..14]
// (descending; key 0 = none, every block's key is larger; keys are distinct).  As the
// list is sorted, "key goes above slot i" is one comparison per slot, all independent,
// and each slot's new value is a select on the old list: slot i keeps its key, takes
// the new one (the first slot it beats) or takes its upper neighbour's.  Depth ~4
// instead of a chain of 14 dependent compare-and-swaps, for about as many instructions.
__device__ __forceinline__ void insert_top(uint64_t (&best)[16], uint64_t key) {
    if (key <= best[14]) return;
    bool above[15];
#pragma unroll
    for (int i = 0; i < 15; ++i) above[i] = key > best[i];
#pragma unroll
    for (int i = 14; i > 0; --i) best[i] = above[i] ? (above[i - 1] ? best[i - 1] : key) : best[i];
    best[0] = above[0] ? key : best[0];
}

// Merging whole lists, at the end of a row, uses bitonic networks instead of 15
// insertions one after another: 16 maxima and four stages of eight independent
// compare-and-swaps.  All indices are compile-time constants, so the lists stay in
// registers.

// Compare-and-swap: the larger key to a.
__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
    const uint64_t hi = a > b ? a : b;
    b = a > b ? b : a;
    a = hi;
}

// best := the 16 largest keys of best and b, descending (both given descending;
// best[15] and b[15] may be 0).  The elementwise maximum of best and b reversed
// is a bitonic sequence holding them; the bitonic merge (four stages) sorts it.
__device__ __forceinline__ void merge16_desc(uint64_t (&best)[16], const uint64_t (&b)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) best[i] = best[i] > b[15 - i] ? best[i] : b[15 - i];
#pragma unroll
    for (int stride = 8; stride > 0; stride >>= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int l = i ^ stride;
            if (l > i) cas_desc(best[i], best[l]);
        }
}

// Bitonic sort of 16 block indices into ascending order.
__device__ __forceinline__ void sort16_asc(int (&v)[16]) {
#pragma unroll
    for (int size = 2; size <= 16; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int l = i ^ stride;
                if (l > i) {
                    const bool up = (i & size) == 0;  // ascending run
                    const int lo = min(v[i], v[l]), hi = max(v[i], v[l]);
                    v[i] = up ? lo : hi;
                    v[l] = up ? hi : lo;
                }
            }
}

// Launched as a programmatic dependent of the decode attention (mixed batches), this
// kernel reads nothing that grid writes, so it starts at once; but every working CTA
// (and CTA 0 in any case) waits for that grid to finish before it exits, so this grid
// cannot finish first and work queued after it on the stream also comes after the
// decode attention.  A no-op in an ordinary launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__global__ void __launch_bounds__(kIdxThreads, 1) prefill_index_kernel(const __grid_constant__ CUtensorMap iq_map,
                                                                       const __grid_constant__ CUtensorMap ik_map,
                                                                       const PrefillIndexArgs a) {
    extern __shared__ uint8_t smem_raw[];
    IndexSmem& sm = *reinterpret_cast<IndexSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;

    if (tid == 0) {
        int b = 0, i0 = 0, n = 0;
        sm.seq = -1;
        if (find_tile(a, blockIdx.x, b, i0, n)) {
            const int L = a.cache_lens[b];
            const int r0 = a.cu_rows[b] + i0;
            const int nr = min(kIdxRows, n - i0);
            const bool ok = L >= n && L <= a.max_cache_len && seq_rows_ok(a.cache, b, L, a.cache_tokens) &&
                            r0 >= 0 && r0 + nr <= a.total_rows;
            if (ok) {
                sm.seq = b;
                sm.row0 = r0;
                sm.nrows = nr;
                sm.L = L;
                sm.p0 = L - n + i0;                              // position of the tile's first row
                const int pmax = sm.p0 + nr - 1;
                sm.ntiles = (pmax + kIdxCols) / kIdxCols;        // tiles covering positions 0..pmax
                sm.n0 = static_cast<int>(static_cast<int64_t>(sm.ntiles) * blockIdx.z / a.nsplit);
                sm.n1 = static_cast<int>(static_cast<int64_t>(sm.ntiles) * (blockIdx.z + 1) / a.nsplit);
            } else {
                atomicOr(a.err, kErrBadMetadata);
            }
        }
        for (int s = 0; s < kIdxStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.a_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.acc_full[s], 1);
            mbar_init(&sm.acc_empty[s], 256);  // every epilogue thread
        }
        mbar_init(&sm.drain, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (sm.seq < 0) {  // no tile here: leave the SM to working CTAs, but CTA 0 always waits
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) grid_dependency_wait();
        return;
    }
    if (warp == 9) tmem_alloc(&sm.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const int n0 = sm.n0, n1 = sm.n1;  // this split's tiles

    if (warp == 8) {
        // ---------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&iq_map);
            prefetch_tmap(&ik_map);
            const int key_head = a.ik_shared ? 0 : h;  // a shared index key is head 0 of ik
            mbar_arrive_expect_tx(&sm.a_full, kIdxABytes);
            tma_load_3d(sm.a, &iq_map, &sm.a_full, 0, h, sm.row0);
            int armed = 0;  // ring positions armed so far
            for (int n = n0; n < n1; ++n) {
                const int i = n - n0;  // ring position
                const int s = i % kIdxStages;
                if (i >= kIdxStages && !mbar_wait(&sm.empty[s], ((i / kIdxStages) - 1) & 1, a.err)) break;
                armed = i + 1;
                if (a.cache.table == nullptr) {  // contiguous: the tile is one 256-position box
                    mbar_arrive_expect_tx(&sm.full[s], kIdxTileBytes);
                    tma_load_3d(sm.b[s], &ik_map, &sm.full[s], 0, key_head,
                                static_cast<int>(a.cache.starts[sm.seq] + static_cast<int64_t>(n) * kIdxCols));
                    continue;
                }
                // paged: one 64-position box per block (blocks sit on separate pages);
                // blocks at or past L are not loaded (their positions are masked)
                int64_t rows[kIdxCols / kBlock];
                int nbox = 0;
#pragma unroll
                for (int qq = 0; qq < kIdxCols / kBlock; ++qq) {
                    const int64_t t = static_cast<int64_t>(n) * kIdxCols + qq * kBlock;
                    rows[qq] = -1;
                    if (t < sm.L) {
                        rows[qq] = block_row(a.cache, sm.seq, t);
                        if (rows[qq] < 0) {  // page outside the pool
                            atomicOr(a.err, kErrBadMetadata);
                            rows[qq] = 0;
                        }
                        ++nbox;
                    }
                }
                mbar_arrive_expect_tx(&sm.full[s], nbox * (kIdxTileBytes / (kIdxCols / kBlock)));
#pragma unroll
                for (int qq = 0; qq < kIdxCols / kBlock; ++qq)
                    if (rows[qq] >= 0)
                        tma_load_3d(sm.b[s] + qq * (kIdxTileBytes / (kIdxCols / kBlock)), &ik_map, &sm.full[s], 0, key_head,
                                    static_cast<int>(rows[qq]));
            }
            // no copy of this lane may still be in flight when the CTA ends (after a timed-out
            // wait elsewhere, too): wait, bounded, for the last phase armed on every slot
            mbar_wait(&sm.a_full, 0, a.err);
            for (int s = 0; s < kIdxStages && s < armed; ++s)
                mbar_wait(&sm.full[s], ((s + kIdxStages * ((armed - 1 - s) / kIdxStages)) / kIdxStages) & 1, a.err);
        }
    } else if (warp == 9) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kIdxRows, kIdxCols, 0, 0);
            bool ok = mbar_wait(&sm.a_full, 0, a.err);
            bool issued = false;
            const uint32_t a_addr = smem_u32(sm.a);
            for (int n = n0; ok && n < n1; ++n) {
                const int i = n - n0;
                const int s = i % kIdxStages, acc = i & 1;
                if (!mbar_wait(&sm.full[s], (i / kIdxStages) & 1, a.err)) break;
                if (i >= 2 && !mbar_wait(&sm.acc_empty[acc], ((i >> 1) - 1) & 1, a.err)) break;
                tc_fence_after();
                const uint32_t b_addr = smem_u32(sm.b[s]);
#pragma unroll
                for (int k = 0; k < kIndexDim / 16; ++k) {
                    const uint64_t ad = smem_desc_sw128(a_addr + k * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(b_addr + k * 32, 16, 1024);
                    tc_mma_ss(tmem + acc * kIdxCols, ad, bd, idesc, k > 0);
                }
                issued = true;
                tc_commit(&sm.empty[s]);
                tc_commit(&sm.acc_full[acc]);
            }
            if (issued) {  // this thread's MMAs are done before tensor memory is freed
                tc_commit(&sm.drain);
                mbar_wait(&sm.drain, 0, a.err);
            }
        }
    } else {
        // ---------------- epilogue: warps w and w+4 share TMEM lane quarter w; a thread
        // owns one row and half of each tile's blocks (blocks 2 half, 2 half + 1)
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;  // TMEM lane
        bool live = row < sm.nrows;
        const int p = sm.p0 + row;
        const int J = p / kBlock;
        // best[0..14]: the 15 best keys so far, descending; best[15] stays 0 (a slot for the
        // merges below)
        uint64_t best[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) best[i] = 0;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        for (int n = n0; n < n1; ++n) {
            const int acc = (n - n0) & 1;
            if (!mbar_wait(&sm.acc_full[acc], ((n - n0) >> 1) & 1, a.err)) break;
            tc_fence_after();
#pragma unroll 1
            for (int jb = half * 2; jb < half * 2 + 2; ++jb) {
                const int j = n * (kIdxCols / kBlock) + jb;
                float m;  // the block's pooled score: the maximum of its 64 columns, taken by the TMEM load
                tmem_ld_max64(lane_addr + acc * kIdxCols + jb * kBlock, m);
                tmem_ld_wait();
                if (!live || j >= J) continue;  // the local block is forced; later blocks are in the future
                insert_top(best, block_key(m, j));
            }
            tc_fence_before();
            mbar_arrive(&sm.acc_empty[acc]);
        }
        // the two halves' lists of a row into one (blocks are disjoint)
        if (half == 1 && live) {
#pragma unroll
            for (int i = 0; i < 16; ++i) sm.half_list[row][i] = best[i];
        }
        epilogue_sync();
        if (half == 0 && live) {
            uint64_t other[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) other[i] = sm.half_list[row][i];
            merge16_desc(best, other);
        }
        if (half == 1) live = false;  // half 0 finishes the row
        if (a.nsplit > 1) {
            // publish this split's list; the last split of the (row tile, head) to
            // arrive merges all lists (each block lies in exactly one split's range)
            if (live) {
                uint64_t* mine =
                    a.cand + ((static_cast<int64_t>(sm.row0 + row) * a.H + h) * a.nsplit + blockIdx.z) * 15;
#pragma unroll
                for (int i = 0; i < 15; ++i) mine[i] = best[i];
            }
            __threadfence();
            epilogue_sync();
            if (tid == 0) sm.last = atomicAdd(a.tickets + static_cast<int64_t>(blockIdx.x) * a.H + h, 1) == a.nsplit - 1;
            epilogue_sync();
            if (!sm.last) {
                live = false;
            } else {
                __threadfence();
                if (live) {
                    // the other splits' lists (15 keys each, descending), the next one loading
                    // while the current one is merged
                    const uint64_t* lists = a.cand + (static_cast<int64_t>(sm.row0 + row) * a.H + h) * a.nsplit * 15;
                    const int me = static_cast<int>(blockIdx.z);
                    int sp = me == 0 ? 1 : 0;  // the first other split (nsplit >= 2)
                    uint64_t cur[16], nxt[16];
                    cur[15] = nxt[15] = 0;
#pragma unroll
                    for (int i = 0; i < 15; ++i) cur[i] = __ldcg(lists + sp * 15 + i);
                    while (true) {
                        int sn = sp + 1;
                        if (sn == me) ++sn;
                        const bool more = sn < a.nsplit;
                        if (more) {
#pragma unroll
                            for (int i = 0; i < 15; ++i) nxt[i] = __ldcg(lists + sn * 15 + i);
                        }
                        merge16_desc(best, cur);
                        if (!more) break;
#pragma unroll
                        for (int i = 0; i < 15; ++i) cur[i] = nxt[i];
                        sp = sn;
                    }
                }
            }
        }
        if (live) {
            // kept blocks: the best min(top_k-1, J) plus J, ascending, -1 padded
            const int others = min(a.top_k - 1, J);
            int v[16];
#pragma unroll
            for (int i = 0; i < 15; ++i) v[i] = i < others ? key_block(best[i]) : 0x7fffffff;
            v[15] = 0x7fffffff;
            if (others < 16) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (i == others) v[i] = J;
            }
            sort16_asc(v);
            const int r = sm.row0 + row;
            int32_t* out = a.sel + (static_cast<int64_t>(r) * a.H + h) * a.top_k;
#pragma unroll
            for (int i = 0; i < kMaxTopK; ++i)  // unrolled: v stays in registers
                if (i < a.top_k) out[i] = v[i] == 0x7fffffff ? -1 : v[i];
            a.nsel[static_cast<int64_t>(r) * a.H + h] = others + 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    grid_dependency_wait();
}

cudaError_t run_prefill_index(const PrefillIndexArgs& a, bool after_decode, cudaStream_t stream) {
    const size_t smem = sizeof(IndexSmem) + 1024;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_index_kernel), smem);
    if (e != cudaSuccess) return e;
    const int tiles = (a.total_rows + kIdxRows - 1) / kIdxRows + a.num_seqs;  // upper bound
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, a.H, a.nsplit);
    cfg.blockDim = dim3(kIdxThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // only behind the decode attention, whose outputs this kernel does not read; as the
    // first kernel of a call it would overlap whatever the caller wrote iq or ik with
    cfg.numAttrs = after_decode ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, prefill_index_kernel, *a.iq_map, *a.ik_map, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace msa
