// prefill.cu -- causal (or bidirectional) GQA prefill attention on sm_103a:
// TMA-staged tiles, tcgen05 MMA with fp32 accumulators in TMEM, online
// softmax in registers, causal tile skipping and a persistent
// longest-first schedule.
//
// Mapping of the chowfi/kernels README ("What helped most") onto GB300:
//  * item 3, skip the masked half: a query tile only visits KV tiles up to
//    and including its diagonal tile; only the diagonal tile is masked;
//  * item 4, largest blocks first: work items are ordered by their number of
//    KV tiles, descending, and dealt to persistent CTAs (one per SM) in a
//    snake order so every CTA ends with the short items;
//  * item 5, exp2 softmax: log2(e)/sqrt(128) is folded into one FFMA per score
//    ahead of the MUFU ex2;
//  * item 2, GQA: the 4 query heads of a KV group are adjacent in the item
//    order, so their K/V tiles are L2 hits for one another.
//
// One work item = one query head x 256 query rows, held as two 128-row Q
// tiles (A and B) that share every K/V tile loaded into shared memory.
// Roles (384 threads, three warpgroups):
//   warps 0-3  softmax of tile A (thread r owns TMEM lane / query row r)
//   warps 4-7  softmax of tile B
//   warp  8    TMA producer: Q tiles, then K_j, V_j into a 4-slot ring
//   warp  9    TMEM allocator and tcgen05.mma issuer (one thread)
//   warp  10   ring bookkeeping: K/V residency checks and slot release
//   warp  11   idle (completes the third warpgroup, whose registers
//              setmaxnreg hands to the softmax warps)
// TMEM (512 columns x 128 lanes, fp32):
//   S_A [0,128)  S_B [128,256)  O_A [256,384)  O_B [384,512)
//   P_t (bf16, two per column) overwrites the first 64 columns of S_t.
// MMA issue per KV tile j, two batches of 16 MMAs:  [PV_A(j), S_A(j+1)],
// [PV_B(j), S_B(j+1)]: while one tile's softmax runs, the tensor core works
// on the other's.  The issuing thread waits once per batch (on that tile's
// P) and commits once per batch (S complete); the ring warp adds the
// "K/V resident" condition to the same barrier and returns ring slots once a
// completed S_B implies every MMA that read them is done.  O's completion is
// signalled once per item (for the epilogue): S_t(j) follows PV_t(j-1) in
// the in-order tensor pipe, so a completed S_t(j) already implies that O is
// complete for the softmax's rescale.
// Row maxima of full tiles come out of the TMEM load itself (tcgen05.ld.red
// .max, per thread over each 32 loaded columns); only a masked diagonal or
// ragged tile takes its maximum in registers after masking.
// O is rescaled only when a row maximum grows by more than 2^8 (the final
// O / l uses the same stale maximum, so the result is unchanged).
// The epilogue (softmax warps) stages each warp's 32 output rows in shared
// memory and writes them as 128-byte row segments.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kBM = 128;                       // query rows per tile
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kTiles = 2;                      // Q tiles per work item
constexpr int kStages = 4;                     // K/V ring slots
constexpr int kTileBytes = kBM * kD * 2;       // 32 KB
constexpr int kHalfBytes = kTileBytes / 2;     // [128 rows][64 dims], 16 KB
constexpr int kSoftmaxWarps = 4 * kTiles;
constexpr int kWarpLoad = kSoftmaxWarps;       // 8
constexpr int kWarpMma = kSoftmaxWarps + 1;    // 9
constexpr int kWarpRing = kSoftmaxWarps + 2;   // 10
// 12 warps = three warpgroups: softmax A, softmax B, and producer + MMA +
// ring + one idle warp.  At launch every thread gets 168 registers (384 x 168 =
// 64512); the third group lowers itself to 104 and the softmax groups raise
// themselves to 200 (256 x 200 + 128 x 104 = 64512, exactly what the third
// group gives up; per SMSP one warp of each group: (200 + 200 + 104) x 32 =
// 16128 of 16384).
constexpr int kThreads = (kSoftmaxWarps + 4) * 32;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 104;
constexpr int kQBytes = kTiles * kTileBytes;
constexpr int kRingBytes = kStages * kTileBytes;
// q_full, q_empty, kv_full[4], kv_empty[4], s_full[2], p_full[2], o_full[2],
// drain
constexpr int kNumBars = 2 + 2 * kStages + 3 * kTiles + 1;
// epilogue staging: per softmax warp, 32 rows x 64 columns of bf16 output
constexpr int kStageWarpBytes = 32 * 64 * 2;
constexpr int kStageBytes = kSoftmaxWarps * kStageWarpBytes;
// packed batches up to this many sequences use the compact item order (Work)
constexpr int kCompactBatch = 64;
constexpr int kTabBytes = kCompactBatch * 8;
constexpr int kCursorBytes = 16 * (kSoftmaxWarps + 4);  // one slot per warp
constexpr size_t kSmemBytes =
    1024 + kQBytes + kRingBytes + kStageBytes + kTabBytes + kCursorBytes + kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint32_t kTmemCols = 512;

static_assert(kBM == kPrefillBoxRows && kBN == kPrefillBoxRows, "tensor-map box");

constexpr uint32_t kIdescS = umma_idesc_bf16(kBM, kBN, 0, 0);  // Q.K^T, both K-major
constexpr uint32_t kIdescO = umma_idesc_bf16(kBM, kD, 0, 1);   // P.V, V MN-major
constexpr float kScaleLog2 = 1.4426950408889634f * 0.08838834764831845f;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

struct Bars {
    uint32_t base;
    __device__ uint32_t q_full() const { return base; }
    __device__ uint32_t q_empty() const { return base + 8; }
    __device__ uint32_t kv_full(int s) const { return base + 16 + 8 * s; }
    __device__ uint32_t kv_empty(int s) const { return base + 16 + 8 * kStages + 8 * s; }
    __device__ uint32_t s_full(int t) const { return base + 16 + 16 * kStages + 8 * t; }
    __device__ uint32_t p_full(int t) const { return base + 32 + 16 * kStages + 8 * t; }
    __device__ uint32_t o_full(int t) const { return base + 48 + 16 * kStages + 8 * t; }
    // the MMA issuer's last commit: every MMA it issued has completed
    __device__ uint32_t drain() const { return base + 64 + 16 * kStages; }
};

// Work decomposition shared by every role.  The batch is B packed
// sequences (sequence s spans rows cu[s] .. cu[s+1]-1 of q, k, v and out;
// B = 1 with no cu array is the single-sequence case).  Item idx -> (block
// b of 256 rows, sequence, head): blocks with the most KV tiles first, the
// heads of one sequence adjacent (the 4 heads of a KV group share K/V in L2).
// Items whose block lies past the end of their sequence are skipped by every
// role alike.
struct Item {
    int b, h, start, len, T;
};

// 256-row blocks of a sequence of `len` rows.
__device__ __forceinline__ int blocks_of(int len) { return ((len + kBM - 1) / kBM + 1) / 2; }

// Items (block b, sequence, head), dealt longest first: block-major with b
// descending (causal) or ascending.  A packed batch of at most
// kCompactBatch sequences comes with a shared-memory table {start, len} per
// sequence and skips the blocks past each sequence's end, so the empty items
// a mixed-length batch would otherwise leave in some CTAs' share are gone
// (schedule balance on lengths 8192..256: 0.83 -> 0.99); its order is b
// descending, then sequence, then head.  Each role warp walks its items in
// increasing index order, which its cursor relies on: (cb, cbase, ck) = block
// cb holds items cbase .. cbase + hq*ck - 1, kept in a per-warp shared-memory
// slot after the table (every lane of a warp computes the same values).
template <bool kVarlen, bool kCompact>
struct Work {
    const int *cu;
    uint32_t tab;  // compact order: shared address of {start, len} per sequence, else 0
    int B, total, n_blocks, n_items, causal, hq, group;
    __device__ Work(const int *cu_, uint32_t tab_, int B_, int max_len, int total_,
                    int causal_, int hq_, int group_)
        : cu(cu_), tab(tab_), B(B_), total(total_), causal(causal_), hq(hq_), group(group_) {
        n_blocks = ((max_len + kBM - 1) / kBM + 1) / 2;
        if (kCompact) {
            int blocks = 0;
            for (int s = 0; s < B; ++s) blocks += blocks_of(len_of(s));
            n_items = blocks * hq;
            const uint32_t c = cursor();
            st_shared_v4(c, uint32_t(n_blocks), 0u, 0u, 0u);
        } else {
            n_items = n_blocks * B * hq;
        }
    }
    __device__ int len_of(int s) const { return ld_shared_s32(tab + 8 * s + 4); }
    __device__ uint32_t cursor() const { return tab + kTabBytes + 16 * (threadIdx.x >> 5); }
    // sequences with more than b blocks
    __device__ int count(int b) const {
        int c = 0;
        for (int s = 0; s < B; ++s) c += blocks_of(len_of(s)) > b;
        return c;
    }
    // Item of round `r` for CTA `c` (snake order over the grid).
    __device__ int item(int r, int c, int G) const {
        return r * G + ((r & 1) ? (G - 1 - c) : c);
    }
    // Compact order (see above).  The cursor is only a cache: walking from the
    // initial state is always correct, so the lanes of a warp may interleave
    // their reads and writes of the slot in any order (all compute the same
    // state for the same index; a lane that reads an already advanced state
    // finds its item in it directly).
    __device__ bool resolve_compact(int idx, Item &it) const {
        const uint32_t c = cursor();
        const uint4 cur = ld_shared_v4(c);
        int cb = int(cur.x), cbase = int(cur.y), ck = int(cur.z);
        while (idx >= cbase + hq * ck) {
            cbase += hq * ck;
            if (--cb < 0) return false;
            ck = count(cb);
        }
        st_shared_v4(c, uint32_t(cb), uint32_t(cbase), uint32_t(ck), 0u);
        const int off = idx - cbase, rank = off / hq;
        it.h = off - rank * hq;
        it.b = cb;
        int s = 0;
        for (int seen = 0; s < B; ++s)
            if (blocks_of(len_of(s)) > cb) {
                if (seen == rank) break;
                ++seen;
            }
        it.start = ld_shared_s32(tab + 8 * s);
        it.len = len_of(s);
        it.T = (it.len + kBM - 1) / kBM;
        return true;
    }
    // false: nothing to do for this item (past its sequence, or a malformed
    // cu array, which also sets kErrBadSeqlens)
    __device__ bool resolve(int idx, Item &it, unsigned *err) const {
        if (kCompact) return resolve_compact(idx, it);
        const int per_block = B * hq;
        it.b = causal ? n_blocks - 1 - idx / per_block : idx / per_block;
        const int rem = idx % per_block;
        const int seq = rem / hq;
        it.h = rem % hq;
        if (kVarlen) {
            it.start = __ldg(cu + seq);
            it.len = __ldg(cu + seq + 1) - it.start;
            if (it.start < 0 || it.len < 0 || it.start + it.len > total ||
                it.len > n_blocks * 2 * kBM) {
                atomicOr(err, kErrBadSeqlens);
                return false;
            }
        } else {
            it.start = 0;
            it.len = total;
        }
        it.T = (it.len + kBM - 1) / kBM;
        return 2 * it.b < it.T;
    }
    // KV tiles visited by tile t (0 = A, 1 = B) of the item.
    __device__ int n_kv(const Item &it, int t) const {
        if (!causal) return it.T;
        const int n = 2 * it.b + t + 1;
        return n < it.T ? n : it.T;
    }
};

// Bounded wait shared by a whole warp: every lane polls; if any lane gives up
// (timeout or another role's abort) the warp gives up together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned *err,
                                          unsigned code, volatile int *abort) {
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const long long t0 = clock64();
        while (!(ok = mbar_try_wait(bar, parity))) {
            if (*abort || clock64() - t0 > kWaitLimitCycles) break;
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        if ((threadIdx.x & 31) == 0) {
            atomicOr(err, code);
            *abort = 1;
        }
    }
    return ok;
}
// Same for a single thread (producer / MMA issuer).
__device__ __forceinline__ bool lone_wait(uint32_t bar, uint32_t parity, unsigned *err,
                                          unsigned code, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort || clock64() - t0 > kWaitLimitCycles) {
            atomicOr(err, code);
            *abort = 1;
            return false;
        }
    }
    return true;
}

// Shared-memory matrix descriptors, split into their two 32-bit words so the
// issuing thread only adds a constant to the low word per MMA.  Low word:
// start address >> 4 (bits 0-13) and leading byte offset >> 4 (bits 16-29);
// high word: stride byte offset >> 4, descriptor version 1, 128-byte
// swizzle (the fields of umma_desc_sw128).  Start addresses stay below
// 256 KB, so adding (offset >> 4) to the low word never carries out of the
// address field.
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
    return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
constexpr uint32_t kDescHi = ((1024u >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);  // SBO 1 KB
__device__ __forceinline__ uint64_t desc(uint32_t lo) {
    return (uint64_t(kDescHi) << 32) | lo;
}
// 16-dim K step kk of a K-major [128 rows][128 dims] tile stored as two
// swizzled [128][64] halves (kHalfBytes apart), 32 bytes per step inside a
// half, 8-row groups 1 KB apart (SBO): offset in 16-byte units.
__host__ __device__ constexpr uint32_t kmajor_step(int kk) {
    return uint32_t(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
}
// V as the MN-major B operand: 16-key step kk = 16 rows of 128 B; the two
// 64-dim halves are kHalfBytes apart (LBO), 8-key groups 1 KB apart (SBO).
__host__ __device__ constexpr uint32_t v_step(int kk) { return uint32_t((kk * 2048) >> 4); }

template <bool kVarlen, bool kCompact>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap,
               const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, __nv_bfloat16 *__restrict__ out,
               float *__restrict__ lse, const int *__restrict__ cu_seqlens, int B,
               int max_len, int total, int causal, int hq, int group, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sRing = sQ + kQBytes;
    const uint32_t sStage = sRing + kRingBytes;
    int2 *seq_tab = reinterpret_cast<int2 *>(smem + kQBytes + kRingBytes + kStageBytes);
    uint64_t *bar_mem =
        reinterpret_cast<uint64_t *>(smem + kQBytes + kRingBytes + kStageBytes + kTabBytes +
                                     kCursorBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mem + kNumBars);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const Bars bars{smem_u32(bar_mem)};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;

    if (threadIdx.x == 0) {
        mbar_init(bars.q_full(), 1);
        mbar_init(bars.q_empty(), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bars.kv_full(s), 1);
            mbar_init(bars.kv_empty(s), 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bars.s_full(t), 1);
            mbar_init(bars.p_full(t), 4 + 1);  // the tile's softmax warps + ring warp
            mbar_init(bars.o_full(t), 1);
        }
        mbar_init(bars.drain(), 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpLoad && lane == 0) {
        prefetch_tmap(&qmap);
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the preceding kernel on the
    // stream: the set-up above overlapped its tail; wait for its results
    // before reading q/k/v or writing out.  The next kernel may launch now
    // (it waits for this grid in the same way).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (kCompact) {  // B <= kCompactBatch (the host's choice)
        const int max_rows = (((max_len + kBM - 1) / kBM + 1) / 2) * 2 * kBM;
        for (int s = threadIdx.x; s < B; s += blockDim.x) {
            const int st = __ldg(cu_seqlens + s), en = __ldg(cu_seqlens + s + 1);
            int len = en - st;
            if (st < 0 || len < 0 || en > total || len > max_rows) {
                atomicOr(err, kErrBadSeqlens);  // malformed: the sequence gets no items
                len = 0;
            }
            seq_tab[s] = make_int2(st, len);
        }
        __syncthreads();
    }
    const Work<kVarlen, kCompact> work(cu_seqlens, kCompact ? smem_u32(seq_tab) : 0u, B,
                                       max_len, total, causal, hq,
                       group);

    if (warp >= kSoftmaxWarps) {
        // producer / MMA warpgroup: give registers to the softmax groups
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther) : "memory");
    if (warp == kWarpLoad) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            int kv = 0, n = 0;  // K/V tiles and Q pairs issued
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int idx = work.item(r, cta, G);
                if (idx >= work.n_items) break;
                Item it;
                if (!work.resolve(idx, it, err)) continue;
                const int h = it.h, g = h / work.group;
                if (n > 0 && !(ok = lone_wait(bars.q_empty(), (n - 1) & 1, err,
                                              kErrWaitEmpty, abort)))
                    break;
                ++n;
                mbar_arrive_expect_tx(bars.q_full(), kQBytes);
                for (int t = 0; t < kTiles; ++t) {
                    const int row = it.start + (2 * it.b + t) * kBM;
                    const uint32_t dst = sQ + t * kTileBytes;
                    tma_load_3d(dst, &qmap, bars.q_full(), 0, h, row, pol_q);
                    tma_load_3d(dst + kHalfBytes, &qmap, bars.q_full(), 64, h, row, pol_q);
                }
                const int nkv = work.n_kv(it, 1);
                for (int j = 0; j < nkv && ok; ++j) {
                    for (int which = 0; which < 2; ++which, ++kv) {
                        const int s = kv % kStages;
                        if (kv >= kStages &&
                            !(ok = lone_wait(bars.kv_empty(s), ((kv / kStages) & 1) ^ 1, err,
                                             kErrWaitEmpty, abort)))
                            break;
                        const CUtensorMap *m = which ? &vmap : &kmap;
                        const uint32_t dst = sRing + s * kTileBytes;
                        mbar_arrive_expect_tx(bars.kv_full(s), kTileBytes);
                        const int krow = it.start + j * kBN;
                        tma_load_3d(dst, m, bars.kv_full(s), 0, g, krow, pol_kv);
                        tma_load_3d(dst + kHalfBytes, m, bars.kv_full(s), 64, g, krow, pol_kv);
                    }
                }
            }
            // No copy may still be landing in shared memory when the CTA
            // exits: wait (bounded, regardless of an abort) for the last Q
            // tiles and K/V tiles this thread issued.  Normally they have all
            // been consumed already; after a wait that gave up, some may still
            // be in flight.
            for (int i = kv > kStages ? kv - kStages : 0; i < kv; ++i)
                mbar_wait(bars.kv_full(i % kStages), (i / kStages) & 1, err, kErrWaitFull);
            if (n > 0) mbar_wait(bars.q_full(), (n - 1) & 1, err, kErrWaitFull);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------ MMA issuer
        // Per KV step this thread polls only p_full(A) and p_full(B) (which
        // also carry "K/V resident", from the ring warp) and commits only
        // s_full(A) and s_full(B).  A shared-memory poll right after a commit
        // stalls this thread for about one MMA, and the tensor pipe queues
        // only a few MMAs, so every extra poll between batches idles it.
        if (lane == 0) {
            int kv = 0;  // ring index of the next K/V tile (K_0 V_0 K_1 V_1 ...)
            int p_cnt[kTiles] = {0, 0};
            bool ok = true;
            // descriptor low words: Q tiles A and B, ring slot 0 as a K-major
            // (LBO 16 B) and as an MN-major V (LBO = kHalfBytes) operand
            const uint32_t q_lo[kTiles] = {desc_lo(sQ, 16), desc_lo(sQ + kTileBytes, 16)};
            const uint32_t k_lo0 = desc_lo(sRing, 16), v_lo0 = desc_lo(sRing, kHalfBytes);
            constexpr uint32_t kSlotStep = kTileBytes >> 4;
            auto issue_s = [&](int t, int slot) {
                const uint32_t d = tmem + kBN * t;
                const uint32_t k_lo = k_lo0 + uint32_t(slot) * kSlotStep;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_ss(d, desc(q_lo[t] + kmajor_step(kk)), desc(k_lo + kmajor_step(kk)),
                            kIdescS, kk > 0);
                umma_commit(bars.s_full(t));
            };
            auto issue_pv = [&](int t, int slot, bool first) {
                const uint32_t d = tmem + 2 * kBN + kD * t;
                const uint32_t p = tmem + kBN * t;
                const uint32_t v_lo = v_lo0 + uint32_t(slot) * kSlotStep;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    umma_ts(d, p + kk * 8, desc(v_lo + v_step(kk)), kIdescO, (!first || kk > 0));
            };
            auto wait_p = [&](int t) {
                if (!lone_wait(bars.p_full(t), p_cnt[t] & 1, err, kErrWaitSoftmax, abort))
                    return false;
                ++p_cnt[t];
                tc_fence_after();
                return true;
            };
            for (int r = 0, n = 0; ok; ++r) {
                const int idx = work.item(r, cta, G);
                if (idx >= work.n_items) break;
                Item it;
                if (!work.resolve(idx, it, err)) continue;
                const int nA = work.n_kv(it, 0), nB = work.n_kv(it, 1);
                if (!(ok = lone_wait(bars.q_full(), n & 1, err, kErrWaitFull, abort))) break;
                ++n;
                // K_0 -> S_A(0), S_B(0)
                if (!(ok = lone_wait(bars.kv_full(kv % kStages), (kv / kStages) & 1, err,
                                     kErrWaitFull, abort)))
                    break;
                tc_fence_after();
                issue_s(0, kv % kStages);
                issue_s(1, kv % kStages);
                ++kv;
                if (nB == 1) umma_commit(bars.q_empty());
                // step j: [PV_A(j), S_A(j+1)] then [PV_B(j), S_B(j+1)];
                // kv indexes V_j, kv + 1 is K_{j+1}
                for (int j = 0; j < nB; ++j) {
                    const int vt = kv % kStages, kt = (kv + 1) % kStages;
                    if (j < nA) {
                        if (!(ok = wait_p(0))) break;
                        issue_pv(0, vt, j == 0);
                        if (j + 1 < nA)
                            issue_s(0, kt);
                        else
                            umma_commit(bars.o_full(0));
                    }
                    if (!(ok = wait_p(1))) break;
                    issue_pv(1, vt, j == 0);
                    if (j + 1 < nB) {
                        issue_s(1, kt);
                        kv += 2;
                        if (j + 2 == nB) umma_commit(bars.q_empty());
                    } else {
                        umma_commit(bars.o_full(1));
                        kv += 1;
                    }
                }
            }
        }
    } else if (warp == kWarpRing) {
        // ------------------------------------------------------ ring warp
        // Keeps K/V bookkeeping off the softmax and MMA critical paths.  Per
        // KV step j it waits until V_j and K_{j+1} are resident and adds the
        // fifth arrival to p_full(A) / p_full(B), so a completed p_full means
        // "P ready and operands resident".  Then, as soon as S_B(j) has
        // completed (and with it every MMA issued before it, all reads of K_j
        // and V_{j-1}), those two slots go back to the producer: a softmax
        // earlier than waiting for P_B(j), which keeps the refill's ~1100-cycle
        // TMA latency off the MMA's wait for P_A(j+1).  The item's last V goes
        // back once its final PV has completed.
        if (lane == 0) {
            int kv = 0;  // ring index, as counted by the producer
            int p_cnt[kTiles] = {0, 0};
            int o_cnt = 0, s_cnt = 0;
            bool ok = true;
            auto wait_ring = [&](int i) {
                return lone_wait(bars.kv_full(i % kStages), (i / kStages) & 1, err, kErrWaitFull,
                                 abort);
            };
            // Until S_B of this step has completed.  Either barrier proves it:
            // s_full(B) completing that phase, or p_full(B) completing this
            // step's phase (its softmax has seen S_B).  s_full(B) can only be
            // two phases ahead (its parity then reads "not complete" again)
            // once p_full(B) has completed, and p_full(B) cannot run ahead of
            // this warp, whose arrival each of its phases needs.
            auto wait_sb = [&](int pb) {
                const long long t0 = clock64();
                while (!mbar_test_wait(bars.s_full(1), s_cnt & 1) &&
                       !mbar_test_wait(bars.p_full(1), pb & 1)) {
                    if (*abort || clock64() - t0 > kWaitLimitCycles) {
                        atomicOr(err, kErrWaitMma);
                        *abort = 1;
                        return false;
                    }
                    __nanosleep(32);
                }
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int idx = work.item(r, cta, G);
                if (idx >= work.n_items) break;
                Item it;
                if (!work.resolve(idx, it, err)) continue;
                const int nA = work.n_kv(it, 0), nB = work.n_kv(it, 1);
                const int k0 = kv;  // K_0; V_j = k0 + 2j + 1, K_j = k0 + 2j
                for (int j = 0; j < nB && ok; ++j) {
                    if (!(ok = wait_ring(k0 + 2 * j + 1))) break;
                    if (j + 1 < nB && !(ok = wait_ring(k0 + 2 * j + 2))) break;
                    if (j < nA) mbar_arrive(bars.p_full(0));
                    mbar_arrive(bars.p_full(1));
                    if (!(ok = wait_sb(p_cnt[1]))) break;
                    ++s_cnt;
                    mbar_arrive(bars.kv_empty((k0 + 2 * j) % kStages));                 // K_j
                    if (j > 0) mbar_arrive(bars.kv_empty((k0 + 2 * j - 1) % kStages));  // V_{j-1}
                    // one arrival per phase: wait for the phases to complete
                    if (j < nA) {
                        if (!(ok = lone_wait(bars.p_full(0), p_cnt[0] & 1, err, kErrWaitSoftmax,
                                             abort)))
                            break;
                        ++p_cnt[0];
                    }
                    if (!(ok = lone_wait(bars.p_full(1), p_cnt[1] & 1, err, kErrWaitSoftmax,
                                         abort)))
                        break;
                    ++p_cnt[1];
                }
                if (!ok) break;
                if (!(ok = lone_wait(bars.o_full(1), o_cnt & 1, err, kErrWaitMma, abort))) break;
                ++o_cnt;
                mbar_arrive(bars.kv_empty((k0 + 2 * nB - 1) % kStages));  // V_{nB-1}
                kv = k0 + 2 * nB;
            }
        }
    }  // warp 11 has no role
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax) : "memory");
        // ------------------------------------------------------ softmax
        const int t = warp >> 2;             // 0 = tile A, 1 = tile B
        const int r = (warp & 3) * 32 + lane; // row inside the tile = TMEM lane
        const uint32_t lane_field = uint32_t((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_field + kBN * t;
        const uint32_t o_tm = tmem + lane_field + 2 * kBN + kD * t;
        int s_cnt = 0, o_cnt = 0;
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int idx = work.item(rr, cta, G);
            if (idx >= work.n_items) break;
            Item it;
            if (!work.resolve(idx, it, err)) continue;
            const int h = it.h, len = it.len;
            const int qt = 2 * it.b + t;
            const int n = work.n_kv(it, t);
            const int row = qt * kBM + r;  // row inside the sequence
            float m_run = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                if (!(ok = warp_wait(bars.s_full(t), s_cnt & 1, err, kErrWaitMma, abort)))
                    break;
                ++s_cnt;
                tc_fence_after();
                // S_t(j), with each row's maximum over every 32 columns
                // reduced by the TMEM load itself
                uint32_t sv[kBN];
                float part_max[kBN / 32];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c)
                    tmem_ld32_max(s_tm + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c),
                                  part_max[c]);
                tmem_wait_ld();
                // keys kbase + c with c <= lim are visible to this row
                const int kbase = j * kBN;
                int lim = len - 1 - kbase;
                if (causal && row - kbase < lim) lim = row - kbase;
                float mx = fmaxf(fmax3(part_max[0], part_max[1], part_max[2]), part_max[3]);
                if (lim < kBN - 1) {
                    // diagonal or ragged last tile: mask, then take the row
                    // maximum over the visible keys only (8 chains of 3-input max)
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c > lim) sv[c] = __float_as_uint(-INFINITY);
                    float mx8[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        mx8[c] = fmaxf(__uint_as_float(sv[c]), __uint_as_float(sv[c + 8]));
#pragma unroll
                    for (int c = 16; c < kBN; c += 16)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            mx8[e] = fmax3(mx8[e], __uint_as_float(sv[c + e]),
                                           __uint_as_float(sv[c + 8 + e]));
                    mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
                }
                const float m_new = fmaxf(m_run, mx * kScaleLog2);
                float alpha = 1.f;
                bool resc = false;
                if (j == 0) {
                    m_run = m_new;
                } else if (m_new > m_run + kRescaleLog2) {
                    alpha = ex2(m_run - m_new);
                    m_run = m_new;
                    l *= alpha;
                    resc = true;
                }
                // p = 2^(s*scale*log2e - m): one packed FFMA per two scores,
                // one MUFU ex2 per score, row sum in 4 packed accumulators
                const float2 scale2 = make_float2(kScaleLog2, kScaleLog2);
                const float2 neg_m2 = make_float2(-m_run, -m_run);
                float2 sum2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) sum2[e] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < kBN; c += 2) {
                    const float2 x = ffma2(make_float2(__uint_as_float(sv[c]),
                                                       __uint_as_float(sv[c + 1])),
                                           scale2, neg_m2);
                    const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                    sum2[(c >> 1) & 3] = fadd2(sum2[(c >> 1) & 3], pp);
                    sv[c >> 1] = pack_bf16(pp.x, pp.y);
                }
                const float2 s01 = fadd2(sum2[0], sum2[1]), s23 = fadd2(sum2[2], sum2[3]);
                l += (s01.x + s01.y) + (s23.x + s23.y);
                tmem_st32(s_tm, *reinterpret_cast<uint32_t(*)[32]>(sv));
                tmem_st32(s_tm + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
                tmem_wait_st();
                if (j > 0) {
                    // S_t(j) was issued after PV_t(j-1), so O is complete here
                    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                        for (int c = 0; c < kD / 32; ++c) {
                            uint32_t ov[32];
                            tmem_ld32(o_tm + 32 * c, ov);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                            tmem_st32(o_tm + 32 * c, ov);
                        }
                        tmem_wait_st();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.p_full(t));
            }
            if (!ok) break;
            // epilogue: out = O / l (bf16), rows past S are not stored
            if (!(ok = warp_wait(bars.o_full(t), o_cnt & 1, err, kErrWaitMma, abort))) break;
            ++o_cnt;
            tc_fence_after();
            const float inv = 1.f / l;
            if (lse != nullptr && row < len)  // ln sum_j exp(s_j) = ln2 * (m + log2 l)
                lse[size_t(h) * total + it.start + row] = (m_run + __log2f(l)) * kLn2;
            // Each thread holds one row; stored directly, every warp store
            // would touch 32 rows.  So each half (64 columns) goes through
            // this warp's staging buffer (16-byte chunk k of row r at chunk
            // k ^ (r & 7): conflict-free both ways) and leaves as 128-byte row
            // segments, four rows per warp store.
            const uint32_t stage = sStage + uint32_t(warp) * kStageWarpBytes;
            const int row0 = qt * kBM + (warp & 3) * 32;  // this warp's first row
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(o_tm + 64 * half + 32 * c, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[16 * c + e] = pack_bf16(__uint_as_float(ov[2 * e]) * inv,
                                                   __uint_as_float(ov[2 * e + 1]) * inv);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    st_shared_v4(stage + lane * 128 + ((k ^ (lane & 7)) << 4), pk[4 * k],
                                 pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int sr = 4 * i + (lane >> 3), k = lane & 7;
                    const uint4 v = ld_shared_v4(stage + sr * 128 + ((k ^ (sr & 7)) << 4));
                    if (row0 + sr < len)
                        *reinterpret_cast<uint4 *>(
                            out + (size_t(it.start + row0 + sr) * work.hq + h) * kD + 64 * half +
                            8 * k) = v;
                }
                __syncwarp();
            }
            tc_fence_before();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        // Normally every MMA has completed here (the epilogue waited for the
        // last ones).  After a wait gave up, some may still be running: the
        // issuing thread's commit tells when they are done, and tensor memory
        // is freed only then.
        if (*abort && lane == 0) {
            umma_commit(bars.drain());
            mbar_wait(bars.drain(), 0, err, kErrWaitMma);
        }
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kVarlen, bool kCompact>
cudaError_t launch(const CUtensorMap &qmap, const CUtensorMap &kmap, const CUtensorMap &vmap,
                   void *out, float *lse, const int *cu_seqlens, int B, int max_len, int total,
                   int causal, int hq, int hkv, int num_sms, unsigned *err,
                   cudaStream_t stream) {
    // The shared-memory attribute is per device: set once per device, by
    // whichever host thread gets there first (the others wait for it).
    static std::once_flag once[kMaxDevices];
    static cudaError_t configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        configured[dev] = cudaFuncSetAttribute(prefill_kernel<kVarlen, kCompact>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               int(kSmemBytes));
    });
    if ((e = configured[dev]) != cudaSuccess) return e;
    const long long n_items = ((max_len + kBM - 1) / kBM + 1) / 2 * (long long)B * hq;
    const int grid = n_items < num_sms ? int(n_items) : num_sms;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<kVarlen, kCompact>, qmap, kmap, vmap,
                              static_cast<__nv_bfloat16 *>(out), lse, cu_seqlens, B, max_len,
                              total, causal, hq, hq / hkv, err);
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, void *out, float *lse,
                           const int *cu_seqlens, int B, int max_len, int total, int causal,
                           int hq, int hkv, int num_sms, unsigned *err, cudaStream_t stream) {
    // one sequence: the instantiation without per-sequence offsets
    if (cu_seqlens == nullptr)
        return launch<false, false>(qmap, kmap, vmap, out, lse, nullptr, 1, total, total,
                                    causal, hq, hkv, num_sms, err, stream);
    // A batch whose rows fill batch x max_seqlen has every sequence at the
    // maximum length, so no empty blocks to skip: the plain order, whose
    // kernel carries no compact-order code.  Mixed lengths (up to
    // kCompactBatch sequences) take the compact order.
    if (B <= kCompactBatch && static_cast<long long>(B) * max_len != total)
        return launch<true, true>(qmap, kmap, vmap, out, lse, cu_seqlens, B, max_len, total,
                                  causal, hq, hkv, num_sms, err, stream);
    return launch<true, false>(qmap, kmap, vmap, out, lse, cu_seqlens, B, max_len, total,
                               causal, hq, hkv, num_sms, err, stream);
}

}  // namespace gqa
