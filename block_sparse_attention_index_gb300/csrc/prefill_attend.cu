// Prompt-chunk stage 3 on tcgen05: attention of the G query heads of one KV
// head over the row's kept blocks, with tensor-memory accumulators.
//
// PR #1388 "minimax_m3: a CUDA backend for MiniMax-M3.1-Flash ...", prompt-
// tile commit: the 16 query heads of a key head use the same chosen blocks,
// so one read of a key or value block serves them all.  Each row keeps its
// own selection here: a work item never touches a block its row did not
// choose.
//
// Work item = (query row, KV head), up to 16 kept blocks = 8 pairs of 64
// keys.  The MMAs are transposed so that the 16 heads are the N dimension and
// the keys (or head dims) the M = 128 dimension:
//   S^T[128 keys, 16 heads]  = K_pair[128 keys, 128 dims] . Q^T        per pair
//   O^T[128 dims, 32]       += V_pair^T[128 dims, 128 keys] . [P_hi; P_lo]^T
// K and V pairs arrive by TMA (128-byte swizzle) in two 3-stage rings, each
// fed by its own producer warp, so K pairs of the next items keep loading
// while V pairs wait for the softmax of the current one; V is read as an
// MN-major operand straight from its [key][dim] tile.  Slot i of the V ring
// and slot i of the P ring belong to the same PV pair and share one barrier
// (the V bytes plus one arrival per softmax warp), so the PV issuer tests one
// barrier per pair: on these small-N MMAs each barrier test costs the issuing
// thread a few hundred cycles, about as long as the pair's eight MMAs.  All pairs' S^T
// (128 TMEM columns) are computed before the softmax, so it is exact with a
// single max (no running rescale); P is written as bf16 hi and lo parts (N =
// 32: heads 0-15 hi, 16-31 lo, ~16 significant bits) pair by pair into a
// small ring (three slots) that the PV MMAs drain.  P is stored key-major (one 64-byte row
// per key, 64-byte swizzle), the MN-major form of the B operand, so a thread
// writes its key's 32 values with four 16-byte stores.
//
// Items overlap: S and O are double-buffered in tensor memory (2 x 128 + 2 x
// 32 columns), so the tensor cores compute S of item i+1 while the softmax
// warps work on item i, and the epilogue warps store item i while the
// softmax warps start item i+1.  S and PV MMAs are issued by two threads of
// their own (tcgen05.commit tracks each thread's MMAs separately), so the
// tensor pipe runs one's MMAs while the other waits on a barrier; each
// producer loads its pairs in item order.
//
// Warp roles: 0-7 softmax (warps w and w+4 share TMEM lane quarter w and
// take heads 0-7 and 8-15), 8-11 epilogue, 12 K producer, 13 V producer,
// 14 S issuer and tensor-memory owner, 15 PV issuer, 16 item decoder (the
// whole warp reads a row's selection and resolves its cache rows, up to six
// items ahead, so the producers never wait on metadata loads).  Items are
// strided over a grid of one CTA per SM.
//
// int8 key/value cache (PR #1388, native Metal family commit: keys and values
// cached as int8 with a scale per position and head): the producers land each
// block as one int8 tile in the upper half of its ring slot, and eight more
// warps widen the tiles in place to the same bf16 layout (17-20: K pairs and
// the item's key and value scales, 21-24: V pairs; a lane widens one key row
// of each pair), so the MMAs are those of a bf16 cache.  The softmax multiplies each key's scores by its key scale
// and its weights by its value scale before P enters the PV MMAs (the row
// sum keeps the plain weights).  The K ring has two slots here, which leaves
// room for the scales of two items.  When a chunk's rows keep many key rows
// per position, the positions are widened once per call beforehand
// (run_widen_kv: bf16 integers and head-major scales in the workspace) and a
// third form loads those bf16 tiles directly; four warps (17-20) only stage
// each item's scales.
//
// The softmax's cross-lane reductions use one redux.sync.max.f32 per head for
// the maxima and (bf16 form) a reduce-scatter by halving exchanges for the
// row sums; its per-head maxima and sums go through separate shared arrays,
// so two 256-thread barriers an item suffice.
#include "common.cuh"
#include "internal.h"

namespace msa {

// Key/value forms: bf16 caches; int8 caches whose tiles the kernel widens
// (eight converter warps, 17-20 for K and the scales, 21-24 for V); int8
// caches widened beforehand (run_widen_kv: bf16 tiles of the integers, scales
// beside them; warps 17-20 only stage the scales).  Both int8 forms have a
// shorter K ring, which leaves room for the scales of two items.
enum KvForm { kKvBf16 = 0, kKvInt8 = 1, kKvWidened = 2 };
template <int kKv>
struct PaCfg {
    static constexpr int kConverters = kKv == kKvInt8 ? 8 : (kKv == kKvWidened ? 4 : 0);
    static constexpr int kThreads = 544 + 32 * kConverters;
    static constexpr int kKStages = kKv != kKvBf16 ? 2 : 3;  // K pairs ring (its own producer warp)
    static constexpr int kPvStages = 3;              // V pairs + P pairs ring: slot i holds both operands of one PV pair
    // info ring readers: K and V producers, S and PV issuers, softmax warps, epilogue warps, converters
    static constexpr int kInfoReaders = 2 + 2 + 8 + 4 + kConverters;
    static constexpr int kScaleFloats = kKv != kKvBf16 ? 2 * 2 * kMaxTopK * 64 : 1;  // [item parity][key/value][block][key]
};
constexpr int kPairBytes = 2 * 2 * 64 * 64 * 2;  // [dim half][2 blocks x 64 keys][64 dims] bf16 = 32 KB
constexpr int kQBytes = 2 * 16 * 64 * 2;         // [dim half][16 heads][64 dims] = 4 KB
constexpr int kPSlotBytes = 128 * 32 * 2;        // one pair: [128 keys][32 = 16 hi + 16 lo heads] bf16 = 8 KB
constexpr int kTmemCols = 512;
constexpr int kSCol = 0;                         // S^T buffers: columns [0,128) and [128,256)
constexpr int kOCol = 256;                       // O^T buffers: columns [256,288) and [288,320)
constexpr int kInfoSlots = 6;                    // decoded items published by the K producer

// One decoded work item, shared through shared memory so that only the
// decoder warp walks the sequence metadata and reads the selection.
struct ItemInfo {
    int32_t r, h, p, nsel, end;
    int32_t b;                // sequence
    int32_t blk[kMaxTopK];    // kept blocks
    int32_t row[kMaxTopK];    // their first cache rows
};

template <int kKv>
struct __align__(1024) AttendSmem {
    static constexpr int kKStages = PaCfg<kKv>::kKStages, kPvStages = PaCfg<kKv>::kPvStages;
    uint8_t kst[kKStages][kPairBytes];
    uint8_t vst[kPvStages][kPairBytes];
    uint8_t p[kPvStages][kPSlotBytes];
    uint8_t q[2][kQBytes];
    float sc[PaCfg<kKv>::kScaleFloats];  // int8 cache: key and value scales of two items
    uint64_t kfull[kKStages];
    uint64_t kempty[kKStages];
    uint64_t kraw[kKStages];       // int8 cache: the K pair's int8 tiles landed
    uint64_t vraw[kPvStages];      // int8 cache: the V pair's int8 tiles landed
    uint64_t sc_full[2];           // int8 cache: an item's scales written
    uint64_t sc_empty[2];          // int8 cache: the softmax is done with them
    uint64_t pv_full[kPvStages];   // V pair ready (bf16) and the 8 softmax warps wrote P
    uint64_t pv_empty[kPvStages];  // PV pair done: V and P slot free
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t o_full[2];
    uint64_t o_empty[2];
    uint64_t rs_full[2];
    uint64_t rs_empty[2];
    uint64_t drain[2];  // S and PV issuers: their last MMAs done before the CTA frees tensor memory
    uint64_t info_full[kInfoSlots];
    uint64_t info_empty[kInfoSlots];
    ItemInfo info[kInfoSlots];
    float red_max[4][16];  // per lane quarter: the heads' maxima, then (a separate array, so that no
    float red_sum[4][16];  // barrier guards the reuse) their sums
    float rowsum[2][16];
    uint32_t tmem_base;
};

static_assert(sizeof(AttendSmem<kKvBf16>) + 1024 <= 227 * 1024, "prompt-chunk attention exceeds 227 KB of shared memory");
static_assert(sizeof(AttendSmem<kKvInt8>) + 1024 <= 227 * 1024, "prompt-chunk attention (int8) exceeds 227 KB of shared memory");
static_assert(sizeof(AttendSmem<kKvWidened>) + 1024 <= 227 * 1024, "prompt-chunk attention (widened) exceeds 227 KB");

// One work item as decoded by a warp: the row, KV head, position, number of
// kept blocks and sequence (the same in every lane), and kept block `lane`
// with its first cache row (lanes < nsel).
struct WarpItem {
    int r, h, p, nsel, b;
    int blk, row;
};

// Decodes work item `it` with all 32 lanes (lane i reads kept block i and
// resolves its cache row, so the loads of a row's blocks go out together).
// False when the item is skipped: a row of a decode-family sequence on the
// fused path, or (with `bad` set in every lane) inconsistent metadata or
// selection.  Every branch depends only on values that all lanes share.
__device__ bool decode_item_warp(const PrefillAttendArgs& a, int it, int lane, WarpItem& x, bool& bad) {
    bad = false;
    x.r = it / a.H;
    x.h = it - x.r * a.H;
    int lo = 0, hi = a.num_seqs;  // largest b with cu_rows[b] <= r
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.cu_rows[mid] <= x.r) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int c0 = a.cu_rows[b], c1 = a.cu_rows[b + 1];
    const int n = c1 - c0;
    if (a.only_multi_row && n <= kDecodeMaxRows) return false;  // taken by the decode kernels
    const int L = a.cache_lens[b];
    x.b = b;
    x.p = L - n + (x.r - c0);
    if (x.r < c0 || x.r >= c1 || L < 1 || L > a.max_cache_len || x.p < 0 ||
        !seq_rows_ok(a.cache, b, L, a.cache_tokens)) {
        bad = true;
        return false;
    }
    const int J = x.p / kBlock;
    x.nsel = a.nsel[static_cast<int64_t>(x.r) * a.H + x.h];
    if (x.nsel < 1 || x.nsel > a.top_k) {
        bad = true;
        return false;
    }
    const bool mine = lane < x.nsel;  // nsel <= top_k <= kMaxTopK <= 32
    x.blk = mine ? a.sel[(static_cast<int64_t>(x.r) * a.H + x.h) * a.top_k + lane] : 0;
    bool lane_bad = mine && (x.blk < 0 || x.blk > J);
    int64_t row = 0;
    if (mine && !lane_bad) {
        const int64_t t = static_cast<int64_t>(x.blk) * kBlock;
        row = a.cache.table == nullptr ? a.cache.starts[b] + t : block_row(a.cache, b, t);
        lane_bad = row < 0;  // page outside the pool
    }
    x.row = static_cast<int>(row);
    if (__any_sync(0xffffffffu, lane_bad)) {
        bad = true;
        return false;
    }
    return true;
}

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The same barrier, returning the AND of p over the 256 softmax threads (so that a decision to stop,
// taken after a bounded wait gave up, is the same in every thread and none waits at a later barrier
// for threads that left).
__device__ __forceinline__ bool named_sync_softmax_and(bool p) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred q, o;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred o, 1, 256, q;\n\t"
                 "selp.u32 %0, 1, 0, o;\n\t}"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(p))
                 : "memory");
    return r != 0;
}

// Sums of v[0..7] over the warp's 32 lanes by halving exchanges (a reduce-scatter: 9 shuffles
// instead of 8 x 5): lane l returns the sum of v[(l >> 2) & 7].
__device__ __forceinline__ float warp_sum8_scatter(const float (&v)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4];  // after the exchange over lane bit 4: value (b4 ? 4 : 0) + i
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = (b4 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 4], 16);
    float c[2];  // over bit 3: value (b4 ? 4 : 0) + (b3 ? 2 : 0) + i
#pragma unroll
    for (int i = 0; i < 2; ++i) c[i] = (b3 ? a[i + 2] : a[i]) + __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[i + 2], 8);
    float d = (b2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, b2 ? c[0] : c[1], 4);  // over bit 2
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    return d;
}

// Maximum of v over the 32 lanes of the warp, in every lane (one warp reduction instruction of the
// sm_100 family; NaN inputs are ignored as by fmaxf, -inf stays -inf).
__device__ __forceinline__ float warp_max_f32(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


template <int kKv>
__global__ void __launch_bounds__(PaCfg<kKv>::kThreads, 1) prefill_attend_kernel(const __grid_constant__ CUtensorMap q_map,
                                                                     const __grid_constant__ CUtensorMap k_map,
                                                                     const __grid_constant__ CUtensorMap v_map,
                                                                     const PrefillAttendArgs a) {
    using Cfg = PaCfg<kKv>;
    constexpr bool kInt8 = kKv != kKvBf16;   // scores and weights times the int8 scales
    constexpr bool kWiden = kKv == kKvInt8;  // int8 tiles widened here
    constexpr int kKStages = Cfg::kKStages, kPvStages = Cfg::kPvStages;
    extern __shared__ uint8_t smem_raw[];
    AttendSmem<kKv>& sm =
        *reinterpret_cast<AttendSmem<kKv>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_items = a.total_rows * a.H;

    if (tid == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&sm.kfull[s], kWiden ? 4 : 1);  // the K producer's bytes, or the four K converter warps
            mbar_init(&sm.kempty[s], 1);
            mbar_init(&sm.kraw[s], 1);
        }
        for (int s = 0; s < kPvStages; ++s) {
            // V bytes (producer) or the four V converter warps, + one arrival per softmax warp
            mbar_init(&sm.pv_full[s], (kWiden ? 4 : 1) + 8);
            mbar_init(&sm.pv_empty[s], 1);
            mbar_init(&sm.vraw[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.sc_full[s], 4);
            mbar_init(&sm.sc_empty[s], 8);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.q_full[s], 1);
            mbar_init(&sm.q_empty[s], 1);
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.s_empty[s], 8);
            mbar_init(&sm.o_full[s], 1);
            mbar_init(&sm.o_empty[s], 4);
            mbar_init(&sm.rs_full[s], 8);
            mbar_init(&sm.rs_empty[s], 4);
        }
        for (int s = 0; s < 2; ++s) mbar_init(&sm.drain[s], 1);
        for (int s = 0; s < kInfoSlots; ++s) {
            mbar_init(&sm.info_full[s], 32);  // every lane of the decoder warp (each releases its own writes)
            mbar_init(&sm.info_empty[s], Cfg::kInfoReaders);
        }
        fence_mbar_init();
    }
    if (warp == 14) tmem_alloc(&sm.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 16) {
        // ---------------- item decoder: decodes this CTA's items with the whole warp and
        // publishes them in the info ring, up to kInfoSlots items ahead of the producers
        uint32_t n = 0;
        bool alive = true;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            WarpItem x;
            bool bad;
            if (!decode_item_warp(a, item, lane, x, bad)) {
                if (bad && lane == 0) atomicOr(a.err, kErrBadMetadata);
                continue;
            }
            const int slot = n % kInfoSlots;
            int free_slot = 1;
            if (lane == 0 && n >= kInfoSlots) free_slot = mbar_wait(&sm.info_empty[slot], ((n / kInfoSlots) - 1) & 1, a.err);
            if (!__shfl_sync(0xffffffffu, free_slot, 0)) {
                alive = false;
                break;
            }
            ItemInfo& inf = sm.info[slot];
            if (lane == 0) {
                inf.r = x.r;
                inf.h = x.h;
                inf.p = x.p;
                inf.nsel = x.nsel;
                inf.b = x.b;
                inf.end = 0;
            }
            if (lane < kMaxTopK) {
                inf.blk[lane] = x.blk;
                inf.row[lane] = x.row;
            }
            mbar_arrive(&sm.info_full[slot]);  // every lane: release of its own fields
            ++n;
        }
        // end marker (also after an abandoned loop, so that every reader stops)
        const int slot = n % kInfoSlots;
        int free_slot = alive ? 1 : 0;
        if (lane == 0 && alive && n >= kInfoSlots)
            free_slot = mbar_wait(&sm.info_empty[slot], ((n / kInfoSlots) - 1) & 1, a.err);
        if (__shfl_sync(0xffffffffu, free_slot, 0)) {
            if (lane == 0) sm.info[slot].end = 1;
            mbar_arrive(&sm.info_full[slot]);
        }
    } else if (warp == 12) {
        // ---------------- K producer: Q(i) and the K pairs of S(i), in item order
        if (lane == 0) {
            prefetch_tmap(&q_map);
            prefetch_tmap(&k_map);
            uint32_t g = 0, q_armed = 0;
            bool alive = true;
            for (uint32_t n = 0; alive; ++n) {
                const int slot = n % kInfoSlots;
                if (!mbar_wait(&sm.info_full[slot], (n / kInfoSlots) & 1, a.err)) break;
                const ItemInfo& inf = sm.info[slot];
                if (inf.end) break;
                const int qb = n & 1;
                if (n >= 2 && !mbar_wait(&sm.q_empty[qb], ((n >> 1) - 1) & 1, a.err)) break;
                mbar_arrive_expect_tx(&sm.q_full[qb], kQBytes);
                ++q_armed;
                const int hq0 = inf.h * a.G;
                tma_load_3d(sm.q[qb], &q_map, &sm.q_full[qb], 0, hq0, inf.r);
                tma_load_3d(sm.q[qb] + kQBytes / 2, &q_map, &sm.q_full[qb], 64, hq0, inf.r);
                const int nsel = inf.nsel, npairs = (nsel + 1) >> 1;
                for (int q = 0; q < npairs; ++q, ++g) {
                    const int s = g % kKStages;
                    if (g >= static_cast<uint32_t>(kKStages) &&
                        !mbar_wait(&sm.kempty[s], ((g / kKStages) - 1) & 1, a.err)) {
                        alive = false;
                        break;
                    }
                    uint64_t* kbar = kWiden ? &sm.kraw[s] : &sm.kfull[s];
                    mbar_arrive_expect_tx(kbar, kWiden ? kPairBytes / 2 : kPairBytes);
                    for (int half = 0; half < 2; ++half) {
                        const int tok = inf.row[min(2 * q + half, nsel - 1)];
                        if constexpr (kWiden) {  // one int8 tile per block, in the slot's upper half
                            tma_load_3d(sm.kst[s] + 16384 + half * 8192, &k_map, kbar, 0, inf.h, tok);
                        } else {
                            tma_load_3d(sm.kst[s] + half * 8192, &k_map, kbar, 0, inf.h, tok);
                            tma_load_3d(sm.kst[s] + half * 8192 + 16384, &k_map, kbar, 64, inf.h, tok);
                        }
                    }
                }
                mbar_arrive(&sm.info_empty[slot]);
            }
            // no copy of this thread may still be in flight when the CTA ends (after a
            // timed-out wait elsewhere, too): wait, bounded, for the last phase armed on
            // every slot
            for (uint32_t s = 0; s < kKStages; ++s)
                if (g > s)
                    mbar_wait(kWiden ? &sm.kraw[s] : &sm.kfull[s], ((s + kKStages * ((g - 1 - s) / kKStages)) / kKStages) & 1,
                              a.err);
            for (uint32_t b = 0; b < 2; ++b)
                if (q_armed > b) mbar_wait(&sm.q_full[b], ((b + 2 * ((q_armed - 1 - b) / 2)) >> 1) & 1, a.err);
        }
    } else if (warp == 13) {
        // ---------------- V producer: the V pairs of PV(i), in item order
        if (lane == 0) {
            prefetch_tmap(&v_map);
            uint32_t g = 0;
            for (uint32_t n = 0;; ++n) {
                const int slot = n % kInfoSlots;
                if (!mbar_wait(&sm.info_full[slot], (n / kInfoSlots) & 1, a.err)) break;
                const ItemInfo& inf = sm.info[slot];
                if (inf.end) break;
                const int npairs = (inf.nsel + 1) >> 1;
                bool alive = true;
                for (int q = 0; q < npairs; ++q, ++g) {
                    const int s = g % kPvStages;
                    if (g >= static_cast<uint32_t>(kPvStages) &&
                        !mbar_wait(&sm.pv_empty[s], ((g / kPvStages) - 1) & 1, a.err)) {
                        alive = false;
                        break;
                    }
                    uint64_t* vbar = kWiden ? &sm.vraw[s] : &sm.pv_full[s];
                    mbar_arrive_expect_tx(vbar, kWiden ? kPairBytes / 2 : kPairBytes);
                    for (int half = 0; half < 2; ++half) {
                        const int tok = inf.row[min(2 * q + half, inf.nsel - 1)];
                        if constexpr (kWiden) {
                            tma_load_3d(sm.vst[s] + 16384 + half * 8192, &v_map, vbar, 0, inf.h, tok);
                        } else {
                            tma_load_3d(sm.vst[s] + half * 8192, &v_map, vbar, 0, inf.h, tok);
                            tma_load_3d(sm.vst[s] + half * 8192 + 16384, &v_map, vbar, 64, inf.h, tok);
                        }
                    }
                }
                mbar_arrive(&sm.info_empty[slot]);
                if (!alive) break;
            }
            for (uint32_t s = 0; s < kPvStages; ++s)  // as for K: no copy left in flight
                if (g > s)
                    mbar_wait(kWiden ? &sm.vraw[s] : &sm.pv_full[s],
                              ((s + kPvStages * ((g - 1 - s) / kPvStages)) / kPvStages) & 1, a.err);
        }
    } else if (warp == 14) {
        // ---------------- S issuer (tensor-memory owner): S^T(i) = K_pair . Q^T per pair
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 16, 0, 0);
            // Descriptor bases, built once: the start-address field counts 16-byte
            // units in the low bits, so a k-step adds (byte offset >> 4).
            uint64_t kdesc[kKStages], qdesc[2];
#pragma unroll
            for (int i = 0; i < kKStages; ++i) kdesc[i] = smem_desc_sw128(smem_u32(sm.kst[i]), 16, 1024);
#pragma unroll
            for (int i = 0; i < 2; ++i) qdesc[i] = smem_desc_sw128(smem_u32(sm.q[i]), 16, 1024);
            uint32_t g = 0;
            bool issued = false;
            for (uint32_t n = 0;; ++n) {
                const int slot = n % kInfoSlots;
                if (!mbar_wait(&sm.info_full[slot], (n / kInfoSlots) & 1, a.err)) break;
                if (sm.info[slot].end) break;
                const int npairs = (sm.info[slot].nsel + 1) >> 1;
                mbar_arrive(&sm.info_empty[slot]);
                const int qb = n & 1, sb = n & 1;
                if (!mbar_wait(&sm.q_full[qb], (n >> 1) & 1, a.err)) break;
                if (n >= 2 && !mbar_wait(&sm.s_empty[sb], ((n >> 1) - 1) & 1, a.err)) break;
                const uint64_t qb_desc = qdesc[qb];
                bool alive = true;
                for (int q = 0; q < npairs; ++q, ++g) {
                    const int s = g % kKStages;
                    if (!mbar_wait(&sm.kfull[s], (g / kKStages) & 1, a.err)) { alive = false; break; }
                    tc_fence_after();
                    const uint64_t kb = kdesc[s];
                    const uint32_t d_tmem = tmem + kSCol + sb * 128 + q * 16;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {  // 16 dims per step
                        const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint32_t qoff = (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32;
                        tc_mma_ss(d_tmem, kb + static_cast<uint64_t>(koff >> 4), qb_desc + static_cast<uint64_t>(qoff >> 4),
                                  idesc_s, kk > 0);
                    }
                    issued = true;
                    tc_commit(&sm.kempty[s]);
                }
                if (!alive) break;
                tc_commit(&sm.q_empty[qb]);
                tc_commit(&sm.s_full[sb]);
            }
            if (issued) {  // this thread's MMAs are done before tensor memory is freed
                tc_commit(&sm.drain[0]);
                mbar_wait(&sm.drain[0], 0, a.err);
            }
        }
    } else if (warp == 15) {
        // ---------------- PV issuer: O^T(i) += V_pair^T . [P_hi; P_lo]^T per pair.  A
        // second issuing thread, so that its barrier waits and those of the S
        // issuer overlap each other's MMAs.
        if (lane == 0) {
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, 32, 1, 1);
            uint64_t vdesc[kPvStages], pdesc[kPvStages];
#pragma unroll
            for (int i = 0; i < kPvStages; ++i) {
                vdesc[i] = smem_desc_sw128(smem_u32(sm.vst[i]), 16384, 1024);
                pdesc[i] = smem_desc_sw64(smem_u32(sm.p[i]), 8192, 512);
            }
            uint32_t g = 0;
            bool issued = false;
            for (uint32_t n = 0;; ++n) {
                const int slot = n % kInfoSlots;
                if (!mbar_wait(&sm.info_full[slot], (n / kInfoSlots) & 1, a.err)) break;
                if (sm.info[slot].end) break;
                const int npairs = (sm.info[slot].nsel + 1) >> 1;
                mbar_arrive(&sm.info_empty[slot]);
                const int ob = n & 1;
                if (n >= 2 && !mbar_wait(&sm.o_empty[ob], ((n >> 1) - 1) & 1, a.err)) break;
                const uint32_t d_tmem = tmem + kOCol + ob * 32;
                bool alive = true;
                for (int q = 0; q < npairs; ++q, ++g) {
                    const int s = g % kPvStages;
                    if (!mbar_wait(&sm.pv_full[s], (g / kPvStages) & 1, a.err)) { alive = false; break; }
                    tc_fence_after();
                    const uint64_t vb = vdesc[s], pb = pdesc[s];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // 16 keys per step: V rows +2 KB, P rows +1 KB
                        tc_mma_ss(d_tmem, vb + static_cast<uint64_t>(kk * 2048 >> 4), pb + static_cast<uint64_t>(kk * 1024 >> 4),
                                  idesc_o, (q > 0 || kk > 0) ? 1u : 0u);
                    issued = true;
                    tc_commit(&sm.pv_empty[s]);
                }
                if (!alive) break;
                tc_commit(&sm.o_full[ob]);
            }
            if (issued) {
                tc_commit(&sm.drain[1]);
                mbar_wait(&sm.drain[1], 0, a.err);
            }
        }
    } else if (warp < 8) {
        // ---------------- softmax (256 threads; row = TMEM lane = key of a pair; warp
        // w takes lane quarter w & 3 and heads 8 * (w >> 2) .. + 7)
        const int quarter = warp & 3, hh = warp >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const int key_in_blk = row & 63, half = row >> 6;
        uint32_t pc = 0;
        for (uint32_t n = 0;; ++n) {
            const int slot = n % kInfoSlots;
            if (!mbar_wait(&sm.info_full[slot], (n / kInfoSlots) & 1, a.err)) break;
            const ItemInfo& inf = sm.info[slot];
            if (inf.end) break;
            const int nsel = inf.nsel, pos = inf.p;
            const int npairs = (nsel + 1) >> 1;
            // key validity per pair: the pair's block on this row's half exists and t <= p
            uint32_t valid_mask = 0;
            for (int q = 0; q < npairs; ++q) {
                const int idx = 2 * q + half;
                if (idx < nsel && inf.blk[idx] * kBlock + key_in_blk <= pos) valid_mask |= 1u << q;
            }
            const int sb = n & 1;
            // int8 cache: this item's key and value scales ([block][key], pair q's half-`half`
            // block is block 2q + half), written by the K converter warps
            const float* sck = sm.sc + (kInt8 ? sb * 2 * kMaxTopK * 64 : 0);
            const float* scv = sck + (kInt8 ? kMaxTopK * 64 : 0);
            if (kInt8 && !mbar_wait(&sm.sc_full[sb], (n >> 1) & 1, a.err)) break;
            if (!mbar_wait(&sm.s_full[sb], (n >> 1) & 1, a.err)) break;
            tc_fence_after();
            const uint32_t s_addr = lane_addr + kSCol + sb * 128 + hh * 8;
            // pass 1: per-head maxima of the raw scores over valid keys
            float mx[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) mx[g] = -INFINITY;
            for (int q0 = 0; q0 < npairs; q0 += 4) {  // four pairs per TMEM round trip
                uint32_t v[4][8];
#pragma unroll
                for (int k = 0; k < 4; ++k) tmem_ld8(s_addr + (q0 + k) * 16, v[k]);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (valid_mask & (1u << (q0 + k))) {
                        const float ks = kInt8 ? sck[(2 * (q0 + k) + half) * 64 + key_in_blk] : 1.f;
#pragma unroll
                        for (int g = 0; g < 8; ++g) mx[g] = fmaxf(mx[g], __uint_as_float(v[k][g]) * ks);
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < 8; ++g) mx[g] = warp_max_f32(mx[g]);  // over the warp's 32 keys
            if (lane < 8) {
                float m = mx[0];
#pragma unroll
                for (int g = 1; g < 8; ++g) m = lane == g ? mx[g] : m;
                sm.red_max[quarter][hh * 8 + lane] = m;
            }
            named_sync_softmax();
            float ms[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int hg = hh * 8 + g;
                ms[g] = fmaxf(fmaxf(sm.red_max[0][hg], sm.red_max[1][hg]), fmaxf(sm.red_max[2][hg], sm.red_max[3][hg])) *
                        a.scale_log2;
            }
            // (red_max is written again only in the next item, after the barrier that closes this one)
            // pass 2: P = 2^(s*scale*log2e - max) as bf16 hi + lo, pair by pair
            float sum[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) sum[g] = 0.f;
            bool alive2 = true;
            for (int q0 = 0; q0 < npairs && alive2; q0 += 4) {  // four pairs per TMEM round trip
                uint32_t vv[4][8];
#pragma unroll
                for (int k = 0; k < 4; ++k) tmem_ld8(s_addr + (q0 + k) * 16, vv[k]);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int q = q0 + k;
                    if (q >= npairs) break;
                    const int ps = pc % kPvStages;
                    if (pc >= kPvStages && !mbar_wait(&sm.pv_empty[ps], ((pc / kPvStages) - 1) & 1, a.err)) {
                        alive2 = false;
                        break;
                    }
                    const bool valid = (valid_mask >> q) & 1u;
                    // int8 cache: scores times the key's scale; weights times the value's scale
                    const float ks = kInt8 && valid ? sck[(2 * q + half) * 64 + key_in_blk] : 1.f;
                    const float vs = kInt8 && valid ? scv[(2 * q + half) * 64 + key_in_blk] : 1.f;
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int g2 = 0; g2 < 4; ++g2) {
                        const float p0 =
                            valid ? exp2f(fmaf(__uint_as_float(vv[k][2 * g2]) * ks, a.scale_log2, -ms[2 * g2])) : 0.f;
                        const float p1 =
                            valid ? exp2f(fmaf(__uint_as_float(vv[k][2 * g2 + 1]) * ks, a.scale_log2, -ms[2 * g2 + 1]))
                                  : 0.f;
                        sum[2 * g2] += p0;
                        sum[2 * g2 + 1] += p1;
                        const float w0 = p0 * vs, w1 = p1 * vs;
                        hi[g2] = pack_bf16x2(w0, w1);
                        lo[g2] = pack_bf16x2(w0 - bf16_lo(hi[g2]), w1 - bf16_hi(hi[g2]));
                    }
                    // row `row` of the slot: 4 chunks of 16 bytes (hi 0-7, hi 8-15, lo 0-7,
                    // lo 8-15), chunk c at position c ^ ((row >> 1) & 3); this warp writes
                    // chunks hh (hi) and 2 + hh (lo)
                    uint8_t* rp = sm.p[ps] + row * 64;
                    const int sw = (row >> 1) & 3;
                    *reinterpret_cast<uint4*>(rp + ((hh ^ sw) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(rp + (((2 + hh) ^ sw) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    fence_proxy_async_smem();  // P is read by the tensor cores
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.pv_full[ps]);
                    ++pc;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_empty[sb]);  // S(n) fully read
            if (kInt8 && lane == 0) mbar_arrive(&sm.sc_empty[sb]);  // the item's scales are no longer read
            if constexpr (!kInt8) {  // (measured: the int8 forms, at 80 registers, ran slower with it)
                const float hs = warp_sum8_scatter(sum, lane);  // lanes 4g .. 4g + 3: head g's sum
                if ((lane & 3) == 0) sm.red_sum[quarter][hh * 8 + (lane >> 2)] = hs;
            } else {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) sum[g] += __shfl_xor_sync(0xffffffffu, sum[g], o);
                }
                if (lane < 8) {
                    float m = sum[0];
#pragma unroll
                    for (int g = 1; g < 8; ++g) m = lane == g ? sum[g] : m;
                    sm.red_sum[quarter][hh * 8 + lane] = m;
                }
            }
            alive2 = named_sync_softmax_and(alive2);  // every thread stops together
            if (n >= 2) mbar_wait(&sm.rs_empty[sb], ((n >> 1) - 1) & 1, a.err);
            if (tid < 16)
                sm.rowsum[sb][tid] = sm.red_sum[0][tid] + sm.red_sum[1][tid] + sm.red_sum[2][tid] + sm.red_sum[3][tid];
            // red_sum is written again only after the next item's first barrier; warp 0's row sums
            // are ordered before its lane 0's arrival below
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.rs_full[sb]);
                mbar_arrive(&sm.info_empty[slot]);
            }
            if (!alive2) break;
        }
    } else if (kInt8 && warp >= 17) {
        // ---------------- int8 converters: warps 17-20 widen the K pairs (warp 17 + j takes keys
        // 32 (j & 1) .. + 31 of block j / 2 of every pair) and write the item's key and value
        // scales, warps 21-24 the V pairs; each lane widens one key row in place.  Tiles widened
        // beforehand: warps 17-20 write the scales only.
        const int cw = warp - 17;
        const bool is_k = cw < 4;
        const int part = cw & 3;  // block part >> 1, keys 32 (part & 1) ..
        uint32_t g = 0;
        bool alive = true;
        for (uint32_t n = 0; alive; ++n) {
            const int slot = n % kInfoSlots;
            if (!mbar_wait(&sm.info_full[slot], (n / kInfoSlots) & 1, a.err)) break;
            const ItemInfo& inf = sm.info[slot];
            if (inf.end) break;
            const int nsel = inf.nsel, npairs = (nsel + 1) >> 1;
            if (is_k) {
                // scales of the item's keys (block bi of the pair list, keys past p read as 0);
                // warp 17 + j takes blocks j, j + 4, ...
                const int sb = n & 1;
                if (n >= 2 && !mbar_wait(&sm.sc_empty[sb], ((n >> 1) - 1) & 1, a.err)) break;
                float* sck = sm.sc + sb * 2 * kMaxTopK * 64;
                float* scv = sck + kMaxTopK * 64;
                for (int bi = part; bi < 2 * npairs; bi += 4) {
                    const int idx = min(bi, nsel - 1);
                    const int64_t row0 = inf.row[idx];
                    const int t0 = inf.blk[idx] * kBlock;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const int key = lane + 32 * kk;
                        float ks = 0.f, vs = 0.f;
                        if (t0 + key <= inf.p) {  // the widened copy keeps its scales head-major
                            const int64_t si = kKv == kKvWidened ? inf.h * a.cache_tokens + row0 + key
                                                                 : (row0 + key) * a.H + inf.h;
                            ks = a.k_scale[si];
                            vs = a.v_scale[si];
                        }
                        sck[bi * 64 + key] = ks;
                        scv[bi * 64 + key] = vs;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.sc_full[sb]);
            }
            for (int q = 0; kWiden && q < npairs; ++q, ++g) {
                const int s = is_k ? static_cast<int>(g % kKStages) : static_cast<int>(g % kPvStages);
                const uint32_t ph = is_k ? (g / kKStages) & 1 : (g / kPvStages) & 1;
                if (!mbar_wait(is_k ? &sm.kraw[s] : &sm.vraw[s], ph, a.err)) {
                    alive = false;
                    break;
                }
                uint8_t* area = (is_k ? sm.kst[s] : sm.vst[s]) + (part >> 1) * 8192;
                convert_i8_row(area, (part & 1) * 32 + lane, 16384);
                fence_proxy_async_smem();  // the tensor cores read the bf16 tile
                __syncwarp();
                if (lane == 0) mbar_arrive(is_k ? &sm.kfull[s] : &sm.pv_full[s]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.info_empty[slot]);
        }
    } else {
        // ---------------- epilogue (warps 4-7; thread = TMEM lane = output dim)
        const int quarter = warp - 8;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const int d = quarter * 32 + lane;
        for (uint32_t n = 0;; ++n) {
            const int slot = n % kInfoSlots;
            if (!mbar_wait(&sm.info_full[slot], (n / kInfoSlots) & 1, a.err)) break;
            if (sm.info[slot].end) break;
            const int r = sm.info[slot].r, h = sm.info[slot].h;
            const int ob = n & 1;
            if (!mbar_wait(&sm.o_full[ob], (n >> 1) & 1, a.err)) break;
            tc_fence_after();
            uint32_t ohi[16], olo[16];
            tmem_ld16(lane_addr + kOCol + ob * 32, ohi);
            tmem_ld16(lane_addr + kOCol + ob * 32 + 16, olo);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_empty[ob]);
            if (!mbar_wait(&sm.rs_full[ob], (n >> 1) & 1, a.err)) break;
            float inv[16];
#pragma unroll
            for (int g = 0; g < 16; ++g) inv[g] = 1.f / sm.rowsum[ob][g];
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.rs_empty[ob]);
                mbar_arrive(&sm.info_empty[slot]);
            }
            const int64_t base = (static_cast<int64_t>(r) * a.H * a.G + static_cast<int64_t>(h) * a.G) * kHeadDim + d;
#pragma unroll
            for (int g = 0; g < 16; ++g) {
                if (g < a.G) {
                    const float o = (__uint_as_float(ohi[g]) + __uint_as_float(olo[g])) * inv[g];
                    if (a.out_bf16)
                        reinterpret_cast<__nv_bfloat16*>(a.out)[base + static_cast<int64_t>(g) * kHeadDim] =
                            __float2bfloat16_rn(o);
                    else
                        reinterpret_cast<float*>(a.out)[base + static_cast<int64_t>(g) * kHeadDim] = o;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 14) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int kKv>
static cudaError_t launch_prefill_attend(const PrefillAttendArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(AttendSmem<kKv>) + 1024;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_attend_kernel<kKv>), smem);
    if (e != cudaSuccess) return e;
    const int64_t items = static_cast<int64_t>(a.total_rows) * a.H;
    const int grid = static_cast<int>(items < device_sm_count() ? items : device_sm_count());
    prefill_attend_kernel<kKv><<<grid, PaCfg<kKv>::kThreads, smem, stream>>>(*a.q_map, *a.k_map, *a.v_map, a);
    return cudaGetLastError();
}

cudaError_t run_prefill_attend(const PrefillAttendArgs& a, cudaStream_t stream) {
    if (a.kv_int8 == 2) return launch_prefill_attend<kKvWidened>(a, stream);
    return a.kv_int8 ? launch_prefill_attend<kKvInt8>(a, stream) : launch_prefill_attend<kKvBf16>(a, stream);
}

}  // namespace msa
