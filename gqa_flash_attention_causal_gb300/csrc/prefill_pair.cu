// prefill_pair.cu -- causal (or bidirectional) GQA prefill on CTA pairs
// (sm_103a): the prefill of prefill.cu with every tcgen05 MMA spanning the
// two SMs of a cluster of two CTAs (cta_group::2).
//
// The chowfi/kernels README ("What helped most", item 2) reads K and V once
// for all the query heads of a group.  Here the two CTAs of a pair work on
// two query heads of the same KV group over the same 256 query rows, and
// share each K/V tile: an MMA of M = 256 rows (128 in each CTA's tensor
// memory) takes its B operand half from each CTA's shared memory, so a CTA
// stages only half of every K tile (64 keys) and half of every V tile (64
// dims), and its tensor core reads half the B bytes per FLOP that it reads in
// the single-CTA kernel.
//
// Work item = two query heads h0, h0 + 1 (one KV head) x 256 query rows,
// CTA c taking head h0 + c as two 128-row Q tiles A and B -- exactly the
// single-CTA kernel's item, so both CTAs mask the same causal diagonal and
// walk the same KV tiles.  Needs an even number of query heads per KV head.
//
// Roles per CTA (384 threads, as in prefill.cu):
//   warps 0-3 / 4-7  softmax of Q tile A / B (thread = TMEM lane = row)
//   warp  8          TMA producer: this CTA's Q tiles and K/V halves
//   warp  9          TMEM allocation for the pair; in CTA 0 (the leader) the
//                    one thread that issues every MMA of the pair
//   warp  10         in CTA 0: ring bookkeeping for both CTAs
// Barriers: CTA 0 owns the ones the MMA issuer waits on (q_full, kv_full,
// p_full); CTA 1's producer and softmax warps arrive on them remotely.  Each
// commit of the issuer arrives on s_full / o_full / q_empty in both CTAs;
// ring slots return to both producers from CTA 0's ring warp.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kBM = 128;                     // query rows per CTA tile
constexpr int kBN = 128;                     // keys per KV tile
constexpr int kTiles = 2;                    // Q tiles per CTA
constexpr int kStages = 8;                   // ring slots, half a K or V tile each
constexpr int kTileBytes = kBM * kD * 2;     // Q tile, 32 KB
constexpr int kQHalf = kTileBytes / 2;       // [128 rows][64 dims]
constexpr int kSlotBytes = 16384;            // K half [64 keys][128 dims] or V half [128][64]
constexpr int kKHalf = kSlotBytes / 2;       // [64 keys][64 dims]
constexpr int kSoftmaxWarps = 4 * kTiles;
constexpr int kWarpLoad = kSoftmaxWarps;     // 8
constexpr int kWarpMma = kSoftmaxWarps + 1;  // 9
constexpr int kWarpRing = kSoftmaxWarps + 2; // 10
constexpr int kThreads = (kSoftmaxWarps + 4) * 32;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 104;
constexpr int kQBytes = kTiles * kTileBytes;
constexpr int kRingBytes = kStages * kSlotBytes;
// q_full, q_empty, kv_full[8], kv_empty[8], s_full[2], p_full[2], o_full[2],
// drain
constexpr int kNumBars = 2 + 2 * kStages + 3 * kTiles + 1;
constexpr int kStageWarpBytes = 32 * 64 * 2;
constexpr int kStageBytes = kSoftmaxWarps * kStageWarpBytes;
// + TMEM address, abort flag, the two producers' copy counts (leader's copy)
constexpr size_t kSmemBytes = 1024 + kQBytes + kRingBytes + kStageBytes + kNumBars * 8 + 32;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint32_t kTmemCols = 512;
constexpr int kItemRows = 2 * kBM;  // query rows per work item

static_assert(kBM == kPrefillBoxRows && kBN / 2 == kPairKBoxRows, "tensor-map boxes");

// M = 256 over the pair (128 rows per CTA), N = 128
constexpr uint32_t kIdescS = umma_idesc_bf16(2 * kBM, kBN, 0, 0);  // Q.K^T, K-major
constexpr uint32_t kIdescO = umma_idesc_bf16(2 * kBM, kD, 0, 1);   // P.V, V MN-major
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

// Items (256-row block b, head pair h0 = 2p, 2p + 1) of one sequence of S
// rows, dealt to the CTA pairs longest first (b descending when causal) in a
// snake order; the head pairs of one KV head are adjacent.
struct PairWork {
    int S, T, n_blocks, n_items, causal, hp;
    __device__ PairWork(int S_, int causal_, int hq) : S(S_), causal(causal_), hp(hq / 2) {
        T = (S + kBM - 1) / kBM;
        n_blocks = (S + kItemRows - 1) / kItemRows;
        n_items = n_blocks * hp;
    }
    __device__ int item(int r, int p, int G) const {
        return r * G + ((r & 1) ? (G - 1 - p) : p);
    }
    // block b and the pair's first query head h0
    __device__ void resolve(int idx, int &b, int &h0) const {
        b = causal ? n_blocks - 1 - idx / hp : idx / hp;
        h0 = 2 * (idx % hp);
    }
    // KV tiles visited by Q tile t of block b (up to its diagonal)
    __device__ int n_kv(int b, int t) const {
        if (!causal) return T;
        const int n = 2 * b + t + 1;
        return n < T ? n : T;
    }
};

// The CTA's abort flag and the peer's (as a cluster address): a role that
// gives up tells both CTAs, so neither waits on the other for long.
struct Abort {
    volatile int *own;
    uint32_t peer;
    __device__ void raise() const {
        *own = 1;
        st_shared_cluster_u32(peer, 1u);
    }
};

// Bounded waits (about one second, or until either CTA aborts).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned *err,
                                          unsigned code, const Abort &ab) {
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
        const long long t0 = clock64();
        while (!(ok = mbar_try_wait(bar, parity))) {
            if (*ab.own || clock64() - t0 > kWaitLimitCycles) break;
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && (threadIdx.x & 31) == 0) {
        atomicOr(err, code);
        ab.raise();
    }
    return ok;
}
__device__ __forceinline__ bool lone_wait(uint32_t bar, uint32_t parity, unsigned *err,
                                          unsigned code, const Abort &ab) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*ab.own || clock64() - t0 > kWaitLimitCycles) {
            atomicOr(err, code);
            ab.raise();
            return false;
        }
    }
    return true;
}

// Descriptor words, as in prefill.cu: the high word is constant (SBO 1 KB,
// version 1, 128-byte swizzle), the issuing thread adds a step to the low
// word per MMA.
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
    return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
constexpr uint32_t kDescHi = ((1024u >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint64_t desc(uint32_t lo) { return (uint64_t(kDescHi) << 32) | lo; }
// 16-dim step kk of a K-major tile stored as two swizzled 64-dim halves
// `half` bytes apart (Q: 16 KB, a K half tile: 8 KB), 32 bytes per step.
__host__ __device__ constexpr uint32_t kmajor_step(int kk, int half) {
    return uint32_t(((kk >> 2) * half + (kk & 3) * 32) >> 4);
}
// V half as the MN-major B operand: 16-key step = 16 rows of 128 bytes.
__host__ __device__ constexpr uint32_t v_step(int kk) { return uint32_t((kk * 2048) >> 4); }

__global__ void __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, __nv_bfloat16 *__restrict__ out,
                    float *__restrict__ lse, int S, int causal, int hq, int group,
                    unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sRing = sQ + kQBytes;
    const uint32_t sStage = sRing + kRingBytes;
    uint64_t *bar_mem = reinterpret_cast<uint64_t *>(smem + kQBytes + kRingBytes + kStageBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mem + kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // [K/V copies, Q copies] issued by CTA 0's and CTA 1's producers (read in CTA 0)
    volatile uint32_t *copies = tmem_slot + 2;
    const Bars bars{smem_u32(bar_mem)};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int G = gridDim.x >> 1, pair = blockIdx.x >> 1;

    if (threadIdx.x == 0) {
        mbar_init(bars.q_full(), 2);  // both producers (leader's copy is used)
        mbar_init(bars.q_empty(), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bars.kv_full(s), 2);
            mbar_init(bars.kv_empty(s), 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bars.s_full(t), 1);
            mbar_init(bars.p_full(t), 2 * 4 + 1);  // both CTAs' softmax warps + ring warp
            mbar_init(bars.o_full(t), 1);
        }
        mbar_init(bars.drain(), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == kWarpLoad && lane == 0) {
        prefetch_tmap(&qmap);
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const Abort ab{abort_flag, mapa_shared(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u)};
    const PairWork work(S, causal, hq);

    if (warp >= kSoftmaxWarps) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther) : "memory");
        if (warp == kWarpLoad && lane == 0) {
            // -------------------------------------------------- TMA producer
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            const uint32_t c_q_full = mapa_shared(bars.q_full(), 0);
            int kv = 0, n = 0;  // K/V halves and Q pairs issued
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int idx = work.item(r, pair, G);
                if (idx >= work.n_items) break;
                int b, h0;
                work.resolve(idx, b, h0);
                const int h = h0 + int(rank), g = h0 / group;
                if (n > 0 &&
                    !(ok = lone_wait(bars.q_empty(), (n - 1) & 1, err, kErrWaitEmpty, ab)))
                    break;
                ++n;
                mbar_arrive_expect_tx_cluster(c_q_full, kQBytes);
                for (int t = 0; t < kTiles; ++t) {
                    const int row = (2 * b + t) * kBM;
                    const uint32_t dst = sQ + t * kTileBytes;
                    tma_load_3d_pair(dst, &qmap, c_q_full, 0, h, row, pol_q);
                    tma_load_3d_pair(dst + kQHalf, &qmap, c_q_full, 64, h, row, pol_q);
                }
                const int nkv = work.n_kv(b, 1);
                for (int j = 0; j < nkv && ok; ++j) {
                    for (int which = 0; which < 2; ++which, ++kv) {
                        const int s = kv % kStages;
                        if (kv >= kStages &&
                            !(ok = lone_wait(bars.kv_empty(s), ((kv / kStages) & 1) ^ 1, err,
                                             kErrWaitEmpty, ab)))
                            break;
                        const uint32_t dst = sRing + s * kSlotBytes;
                        const uint32_t cb = mapa_shared(bars.kv_full(s), 0);
                        mbar_arrive_expect_tx_cluster(cb, kSlotBytes);
                        if (which == 0) {  // K: keys 64*rank .. +63 of tile j, all dims
                            const int krow = j * kBN + int(rank) * (kBN / 2);
                            tma_load_3d_pair(dst, &kmap, cb, 0, g, krow, pol_kv);
                            tma_load_3d_pair(dst + kKHalf, &kmap, cb, 64, g, krow, pol_kv);
                        } else {  // V: dims 64*rank .. +63 of tile j, all keys
                            tma_load_3d_pair(dst, &vmap, cb, 64 * int(rank), g, j * kBN, pol_kv);
                        }
                    }
                }
            }
            // CTA 0 drains both producers' copies at the end (they complete on
            // its barriers): tell it how many this one issued.
            const uint32_t c_copies = mapa_shared(smem_u32(const_cast<uint32_t *>(copies)), 0);
            st_shared_cluster_u32(c_copies + 8 * rank, uint32_t(kv));
            st_shared_cluster_u32(c_copies + 8 * rank + 4, uint32_t(n));
        } else if (warp == kWarpMma && leader && lane == 0) {
            // -------------------------------------------------- MMA issuer (pair)
            int kv = 0;
            int p_cnt[kTiles] = {0, 0};
            bool ok = true;
            const uint32_t q_lo[kTiles] = {desc_lo(sQ, 16), desc_lo(sQ + kTileBytes, 16)};
            const uint32_t k_lo0 = desc_lo(sRing, 16), v_lo0 = desc_lo(sRing, kSlotBytes);
            constexpr uint32_t kSlotStep = kSlotBytes >> 4;
            auto issue_s = [&](int t, int slot) {
                const uint32_t d = tmem + kBN * t;
                const uint32_t k_lo = k_lo0 + uint32_t(slot) * kSlotStep;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    umma_ss_pair(d, desc(q_lo[t] + kmajor_step(kk, kQHalf)),
                                 desc(k_lo + kmajor_step(kk, kKHalf)), kIdescS, kk > 0);
                umma_commit_pair(bars.s_full(t));
            };
            auto issue_pv = [&](int t, int slot, bool first) {
                const uint32_t d = tmem + 2 * kBN + kD * t;
                const uint32_t p = tmem + kBN * t;
                const uint32_t v_lo = v_lo0 + uint32_t(slot) * kSlotStep;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    umma_ts_pair(d, p + kk * 8, desc(v_lo + v_step(kk)), kIdescO,
                                 (!first || kk > 0));
            };
            auto wait_p = [&](int t) {
                if (!lone_wait(bars.p_full(t), p_cnt[t] & 1, err, kErrWaitSoftmax, ab))
                    return false;
                ++p_cnt[t];
                tc_fence_after();
                return true;
            };
            for (int r = 0, n = 0; ok; ++r) {
                const int idx = work.item(r, pair, G);
                if (idx >= work.n_items) break;
                int b, h0;
                work.resolve(idx, b, h0);
                const int nA = work.n_kv(b, 0), nB = work.n_kv(b, 1);
                if (!(ok = lone_wait(bars.q_full(), n & 1, err, kErrWaitFull, ab))) break;
                ++n;
                if (!(ok = lone_wait(bars.kv_full(kv % kStages), (kv / kStages) & 1, err,
                                     kErrWaitFull, ab)))
                    break;
                tc_fence_after();
                issue_s(0, kv % kStages);
                issue_s(1, kv % kStages);
                ++kv;
                if (nB == 1) umma_commit_pair(bars.q_empty());
                for (int j = 0; j < nB; ++j) {
                    const int vt = kv % kStages, kt = (kv + 1) % kStages;
                    if (j < nA) {
                        if (!(ok = wait_p(0))) break;
                        issue_pv(0, vt, j == 0);
                        if (j + 1 < nA)
                            issue_s(0, kt);
                        else
                            umma_commit_pair(bars.o_full(0));
                    }
                    if (!(ok = wait_p(1))) break;
                    issue_pv(1, vt, j == 0);
                    if (j + 1 < nB) {
                        issue_s(1, kt);
                        kv += 2;
                        if (j + 2 == nB) umma_commit_pair(bars.q_empty());
                    } else {
                        umma_commit_pair(bars.o_full(1));
                        kv += 1;
                    }
                }
            }
        } else if (warp == kWarpRing && leader && lane == 0) {
            // -------------------------------------------------- ring warp (pair)
            // As in prefill.cu: adds "V_j and K_{j+1} resident in both CTAs"
            // to p_full and returns slots once S_B(j) has completed -- here to
            // both CTAs' producers.
            const uint32_t peer = rank ^ 1u;
            int kv = 0;
            int p_cnt[kTiles] = {0, 0};
            int s_cnt = 0, o_cnt = 0;
            bool ok = true;
            auto wait_ring = [&](int i) {
                return lone_wait(bars.kv_full(i % kStages), (i / kStages) & 1, err, kErrWaitFull,
                                 ab);
            };
            auto release = [&](int i) {
                const uint32_t e = bars.kv_empty(i % kStages);
                mbar_arrive(e);
                mbar_arrive_cluster(mapa_shared(e, peer));
            };
            auto wait_sb = [&](int pb) {
                const long long t0 = clock64();
                while (!mbar_test_wait(bars.s_full(1), s_cnt & 1) &&
                       !mbar_test_wait(bars.p_full(1), pb & 1)) {
                    if (*ab.own || clock64() - t0 > kWaitLimitCycles) {
                        atomicOr(err, kErrWaitMma);
                        ab.raise();
                        return false;
                    }
                    __nanosleep(32);
                }
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int idx = work.item(r, pair, G);
                if (idx >= work.n_items) break;
                int b, h0;
                work.resolve(idx, b, h0);
                const int nA = work.n_kv(b, 0), nB = work.n_kv(b, 1);
                const int k0 = kv;
                for (int j = 0; j < nB && ok; ++j) {
                    if (!(ok = wait_ring(k0 + 2 * j + 1))) break;
                    if (j + 1 < nB && !(ok = wait_ring(k0 + 2 * j + 2))) break;
                    if (j < nA) mbar_arrive(bars.p_full(0));
                    mbar_arrive(bars.p_full(1));
                    if (!(ok = wait_sb(p_cnt[1]))) break;
                    ++s_cnt;
                    release(k0 + 2 * j);                  // K_j
                    if (j > 0) release(k0 + 2 * j - 1);   // V_{j-1}
                    if (j < nA) {
                        if (!(ok = lone_wait(bars.p_full(0), p_cnt[0] & 1, err, kErrWaitSoftmax,
                                             ab)))
                            break;
                        ++p_cnt[0];
                    }
                    if (!(ok = lone_wait(bars.p_full(1), p_cnt[1] & 1, err, kErrWaitSoftmax, ab)))
                        break;
                    ++p_cnt[1];
                }
                if (!ok) break;
                if (!(ok = lone_wait(bars.o_full(1), o_cnt & 1, err, kErrWaitMma, ab))) break;
                ++o_cnt;
                release(k0 + 2 * nB - 1);  // V_{nB-1}
                kv = k0 + 2 * nB;
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax) : "memory");
        // ------------------------------------------------------ softmax
        const int t = warp >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_field = uint32_t((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_field + kBN * t;
        const uint32_t o_tm = tmem + lane_field + 2 * kBN + kD * t;
        const uint32_t c_p_full = mapa_shared(bars.p_full(t), 0);
        int s_cnt = 0, o_cnt = 0;
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int idx = work.item(rr, pair, G);
            if (idx >= work.n_items) break;
            int b, h0;
            work.resolve(idx, b, h0);
            const int h = h0 + int(rank);
            const int qt = 2 * b + t;  // this CTA's 128-row tile
            const int n = work.n_kv(b, t);
            const int row = qt * kBM + r;
            float m_run = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                if (!(ok = warp_wait(bars.s_full(t), s_cnt & 1, err, kErrWaitMma, ab))) break;
                ++s_cnt;
                tc_fence_after();
                uint32_t sv[kBN];
                float part_max[kBN / 32];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c)
                    tmem_ld32_max(s_tm + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c),
                                  part_max[c]);
                tmem_wait_ld();
                // keys kbase + c with c <= lim are visible to this row
                const int kbase = j * kBN;
                int lim = S - 1 - kbase;
                if (causal && row - kbase < lim) lim = row - kbase;
                float mx = fmaxf(fmax3(part_max[0], part_max[1], part_max[2]), part_max[3]);
                if (lim < kBN - 1) {
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
                if (lane == 0) mbar_arrive_cluster(c_p_full);
            }
            if (!ok) break;
            if (!(ok = warp_wait(bars.o_full(t), o_cnt & 1, err, kErrWaitMma, ab))) break;
            ++o_cnt;
            tc_fence_after();
            const float inv = 1.f / l;
            if (lse != nullptr && row < S)
                lse[size_t(h) * S + row] = (m_run + __log2f(l)) * kLn2;
            const uint32_t stage = sStage + uint32_t(warp) * kStageWarpBytes;
            const int row0 = qt * kBM + (warp & 3) * 32;
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
                    if (row0 + sr < S)
                        *reinterpret_cast<uint4 *>(out + (size_t(row0 + sr) * hq + h) * kD +
                                                   64 * half + 8 * k) = v;
                }
                __syncwarp();
            }
            tc_fence_before();
        }
    }

    // Neither CTA leaves (or frees the pair's tensor memory) while the other
    // may still run MMAs on it, arrive on its barriers, or have copies landing
    // in its shared memory.  Both producers' copies complete on CTA 0's
    // barriers: once both have stopped issuing (first cluster barrier), CTA 0
    // supplies the arrival of any phase that only one producer joined (the
    // other gave up first; the two issue the same sequence, and one can lead
    // by at most a ring's worth of K/V halves and one Q pair) and waits,
    // bounded, for every phase either issued that may not have completed.
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    // Normally every MMA has completed here (the epilogues waited for the
    // last ones).  After a wait gave up, some may still be running: the
    // issuing thread's commit tells when they are done, and tensor memory is
    // freed (below) only then.
    if (leader && warp == kWarpMma && lane == 0 && *abort_flag) {
        tc_fence_after();
        umma_commit_pair(bars.drain());
        mbar_wait(bars.drain(), 0, err, kErrWaitMma);
    }
    if (leader && warp == kWarpLoad && lane == 0) {
        const int kv0 = int(copies[0]), n0 = int(copies[1]);
        const int kv1 = int(copies[2]), n1 = int(copies[3]);
        const int kv_lo = min(kv0, kv1), kv_hi = max(kv0, kv1);
        const int n_lo = min(n0, n1), n_hi = max(n0, n1);
        // phases both joined, then the lone ones (their slots' previous
        // phases, both joined, are complete by then)
        for (int i = kv_lo > kStages ? kv_lo - kStages : 0; i < kv_lo; ++i)
            mbar_wait(bars.kv_full(i % kStages), (i / kStages) & 1, err, kErrWaitFull);
        if (n_lo > 0) mbar_wait(bars.q_full(), (n_lo - 1) & 1, err, kErrWaitFull);
        for (int i = kv_lo; i < kv_hi; ++i) {
            mbar_arrive(bars.kv_full(i % kStages));
            mbar_wait(bars.kv_full(i % kStages), (i / kStages) & 1, err, kErrWaitFull);
        }
        for (int i = n_lo; i < n_hi; ++i) {
            mbar_arrive(bars.q_full());
            mbar_wait(bars.q_full(), i & 1, err, kErrWaitFull);
        }
    }
    __syncwarp();
    cluster_sync();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill_pair(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, void *out, float *lse, int S,
                                int causal, int hq, int hkv, unsigned *err,
                                cudaStream_t stream) {
    // Per device, once: the shared-memory attribute and how many pairs can be
    // resident at a time (the persistent grid's size).
    static std::once_flag once[kMaxDevices];
    static cudaError_t configured[kMaxDevices];
    static int max_pairs[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    std::call_once(once[dev], [dev, &cfg] {
        cudaError_t r = cudaFuncSetAttribute(prefill_pair_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(kSmemBytes));
        int n = 0;
        if (r == cudaSuccess) {
            cudaLaunchConfig_t q = cfg;
            q.numAttrs = 1;  // the cluster shape only
            q.gridDim = dim3(2);
            r = cudaOccupancyMaxActiveClusters(&n, prefill_pair_kernel, &q);
        }
        if (r == cudaSuccess && n < 1) r = cudaErrorInvalidConfiguration;
        max_pairs[dev] = n;
        configured[dev] = r;
    });
    if ((e = configured[dev]) != cudaSuccess) return e;
    if ((hq / hkv) % 2 != 0) return cudaErrorInvalidValue;  // heads are paired within a group
    const long long n_items = (long long)((S + kItemRows - 1) / kItemRows) * (hq / 2);
    const int pairs = n_items < max_pairs[dev] ? int(n_items) : max_pairs[dev];
    cfg.gridDim = dim3(2 * pairs);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, prefill_pair_kernel, qmap, kmap, vmap,
                              static_cast<__nv_bfloat16 *>(out), lse, S, causal, hq, hq / hkv,
                              err);
}

}  // namespace gqa
