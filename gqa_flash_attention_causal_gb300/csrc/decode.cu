// decode.cu -- single-token GQA decode against a KV cache: split-KV kernel
// plus log-sum-exp combine kernel (sm_103a).
//
// What the chowfi/kernels README ("What helped most", items 1, 2 and 5)
// describes for decode, restated for GB300:
//  * one decode token is too little work for the GPU, so the KV length is cut
//    into chunks that run in parallel on every SM and are merged afterwards
//    (item 1: split-KV);
//  * the 4 query heads of a group read their shared K/V once, not 4 times
//    (item 2: GQA packing): one CTA owns (chunk, KV head) and computes all 4
//    query heads from one pass over that chunk;
//  * K/V are read exactly once, so their loads carry an L2 evict-first hint
//    (item 5: cache hints for read-once data);
//  * softmax in base 2 with log2(e) folded into the score scale (item 5).
//
// The work is HBM-bound (4 flops per byte), so the design goal is keeping
// enough bytes in flight: K/V tiles stream through a 6-stage TMA ring (192 KB
// in flight per SM), one CTA per SM, and each CTA starts its first six
// stages on their way into L2 before it waits for the preceding kernel (a
// programmatic dependent launch), so a call's stream overlaps the previous
// kernel's tail.  The 16-key x 128-dim x head-group
// products go through warp-level bf16 MMA (m16n8k16, the group's heads in
// its 8 N columns; other head layouts take groups of up to 16 as two N
// tiles) with fp32 accumulation: one ldmatrix + one MMA replaces 256 scalar
// FMAs, which keeps instruction issue far below the memory time.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

constexpr int kWarps = 4;                        // compute warps per CTA
constexpr int kStageKeys = 16 * kWarps;          // 64 keys per stage
constexpr int kStages = 6;                       // TMA ring depth
constexpr int kHalfBytes = kStageKeys * 128;     // 64 keys x 64 dims x 2 B
constexpr int kTileBytes = 2 * kHalfBytes;       // K (or V) tile, 16 KB
constexpr int kStageBytes = 2 * kTileBytes;      // K + V, 32 KB
constexpr int kThreads = (kWarps + 1) * 32;      // + one TMA producer warp
constexpr int kCtasPerSm = 1;
// query heads per KV head the kernel handles: up to two N tiles of the warp
// MMA's 8 columns
constexpr int kMaxGroup = 16;
// Shared memory of the instantiation with kNT tiles: the ring, the
// cross-warp merge buffers for 8 * kNT heads, the barriers.
constexpr size_t smem_bytes(int nt) {
    return 1024 /*align slack*/ + size_t(kStages) * kStageBytes +
           size_t(kWarps) * 8 * nt * kD * 4 + 2 * kWarps * 8 * nt * 4 + 2 * kStages * 8;
}
constexpr size_t kSmemBytes = smem_bytes(2);  // the largest
static_assert(smem_bytes(1) < kSmemBytes, "one-tile instantiations stay smaller");

static_assert(kStageKeys == kDecodeBoxRows, "tensor-map box must match a stage");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kMaxGroup == kDecodeMaxGroup, "host limit and kernel buffers agree");

// log2(e) / sqrt(128): scores are kept in the base-2 domain.
constexpr float kScaleLog2 = 1.4426950408889634f * 0.08838834764831845f;

// kFixedGroup > 0: the query heads per KV head are a compile-time constant
// (the 32/8 layout); 0: they come from `group_arg` (1..8 * kNT).  kNT: N
// tiles of 8 query heads per MMA step (1, or 2 for groups of 9..16).
template <int kFixedGroup, int kNT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap,
                    const __nv_bfloat16 *__restrict__ q, const int *__restrict__ seqlens,
                    int Lmax, int chunk, int hq, int group_arg, float *__restrict__ part_o,
                    float *__restrict__ part_lse, unsigned *err) {
    const int group = kFixedGroup > 0 ? kFixedGroup : group_arg;
    constexpr int kMG = 8 * kNT;  // heads the merge buffers hold
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *cmb_o = reinterpret_cast<float *>(smem + kStages * kStageBytes);
    float *cmb_m = cmb_o + kWarps * kMG * kD;
    float *cmb_l = cmb_m + kWarps * kMG;
    uint64_t *bars = reinterpret_cast<uint64_t *>(cmb_l + kWarps * kMG);
    const uint32_t tiles = smem_u32(smem);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);

    const int split = blockIdx.x, g = blockIdx.y, seq = blockIdx.z;
    const int n_split = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's chunk of sequence `seq`, whose cache holds rows
    // seq*Lmax .. seq*Lmax + L - 1 of the tensor maps
    const int row0 = seq * Lmax;
    q += size_t(seq) * hq * kD;
    part_o += size_t(seq) * n_split * hq * kD;
    part_lse += size_t(seq) * n_split * hq;

    // Let the combine kernel (a programmatic dependent) get scheduled now; it
    // still waits for this whole grid to finish before reading its results.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kWarps);
        }
        fence_barrier_init();
    }
    if (threadIdx.x == kWarps * 32) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
        // Start this CTA's first stages on their way into L2 while the
        // preceding kernel finishes.  A prefetch only fills L2, the point of
        // coherence every SM reads through, so it cannot hand out data older
        // than what that kernel writes; the loads into shared memory still
        // wait for it below.  With per-sequence lengths (known only after
        // the wait) nothing is prefetched.
        if (seqlens == nullptr) {
            const int k0 = split * chunk;
            const int n_pre =
                min(kStages, (min(Lmax, k0 + chunk) - k0 + kStageKeys - 1) / kStageKeys);
            for (int it = 0; it < n_pre; ++it) {
                const int row = row0 + k0 + it * kStageKeys;
                tma_prefetch_3d(&kmap, 0, g, row);
                tma_prefetch_3d(&kmap, 64, g, row);
                tma_prefetch_3d(&vmap, 0, g, row);
                tma_prefetch_3d(&vmap, 64, g, row);
            }
        }
    }
    __syncthreads();
    // Launched as a programmatic dependent of whatever kernel precedes it on
    // the stream: everything above overlapped that kernel's tail; from here
    // on its results (q, the caches, the lengths) are complete and visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int L = Lmax;
    if (seqlens != nullptr) {
        L = __ldg(seqlens + seq);
        if (L < 1 || L > Lmax) {  // not computed; the combine skips it too
            if (threadIdx.x == 0) atomicOr(err, kErrBadSeqlens);
            L = 0;
        }
    }
    const int key0 = split * chunk;
    const int key_end = min(L, key0 + chunk);
    const int n_iter = key_end > key0 ? (key_end - key0 + kStageKeys - 1) / kStageKeys : 0;

    if (warp == kWarps) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int s = it % kStages;
                if (it >= kStages &&
                    !mbar_wait(empty0 + 8 * s, ((it / kStages) & 1) ^ 1, err, kErrWaitEmpty))
                    break;
                const uint32_t full = full0 + 8 * s, dst = tiles + s * kStageBytes;
                const int row = row0 + key0 + it * kStageKeys;
                mbar_arrive_expect_tx(full, kStageBytes);
                tma_load_3d(dst, &kmap, full, 0, g, row, pol);
                tma_load_3d(dst + kHalfBytes, &kmap, full, 64, g, row, pol);
                tma_load_3d(dst + kTileBytes, &vmap, full, 0, g, row, pol);
                tma_load_3d(dst + kTileBytes + kHalfBytes, &vmap, full, 64, g, row, pol);
                issued = it + 1;
            }
            // No copy may still be landing in shared memory when the CTA
            // exits: wait (bounded) for the stages this thread filled last.
            // Normally the compute warps have waited for them already; after
            // a wait that gave up, some may still be in flight.
            for (int it = issued > kStages ? issued - kStages : 0; it < issued; ++it)
                mbar_wait(full0 + 8 * (it % kStages), (it / kStages) & 1, err, kErrWaitFull);
        }
        return;  // the producer takes no part in the merge below
    }

    // -------------------------------------------------------- compute warps
    // Mapping (m16n8k16 fragments, gi = lane/4, ti = lane%4), per N tile nt
    // of 8 query heads (group heads nt*8 .. nt*8+7; kNT tiles hold groups of
    // up to 8 * kNT, missing heads are zero columns):
    //   S^T[key][head] = K[key][d] . Q^T[d][head]   (A = K via ldmatrix, B = Q^T)
    //   O^T[d][head]  += V^T[d][key] . P^T[key][head]  (A = V^T via
    //   ldmatrix.trans, B = P^T from the S^T fragment by movmatrix.trans)
    // Every K and V fragment loaded from shared memory serves all N tiles.
    // A lane owns heads nt*8 + 2ti and nt*8 + 2ti + 1 in both products, so the
    // running max, sum and O rescale stay in registers.
    const int gi = lane >> 2, ti = lane & 3;
    uint32_t qf[kNT][8][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int hg = nt * 8 + gi;  // head of this B column inside the group
            if (hg < group) {
                const uint32_t *qh = reinterpret_cast<const uint32_t *>(
                    q + (g * group + hg) * kD + 16 * kk + 2 * ti);
                qf[nt][kk][0] = __ldg(qh);
                qf[nt][kk][1] = __ldg(qh + 4);
            } else {
                qf[nt][kk][0] = qf[nt][kk][1] = 0u;
            }
        }
    float o[kNT][8][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
            o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
    float m[kNT][2], l[kNT][2];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
    }
    const int kb = warp * 16;  // this warp's 16 keys inside a stage

    for (int it = 0; it < n_iter; ++it) {
        const int s = it % kStages;
        if (!mbar_wait(full0 + 8 * s, (it / kStages) & 1, err, kErrWaitFull)) break;
        const uint32_t kt = tiles + s * kStageBytes, vt = kt + kTileBytes;

        float c[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
        {
            const uint32_t row = kb + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(sw128(kt + (kk >> 2) * kHalfBytes, row, 2 * (kk & 3) + (lane >> 4)),
                        a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt)
                    mma_bf16_16816(c[nt][0], c[nt][1], c[nt][2], c[nt][3], a0, a1, a2, a3,
                                   qf[nt][kk][0], qf[nt][kk][1]);
            }
        }
        const int key_a = key0 + it * kStageKeys + kb + gi, key_b = key_a + 8;
        uint32_t b[kNT][2];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
            float x0 = c[nt][0] * kScaleLog2, x1 = c[nt][1] * kScaleLog2;
            float x2 = c[nt][2] * kScaleLog2, x3 = c[nt][3] * kScaleLog2;
            if (key_a >= L) x0 = x1 = -INFINITY;
            if (key_b >= L) x2 = x3 = -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
            const float r0 = mn0 == -INFINITY ? 0.f : mn0;  // all keys so far masked
            const float r1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ex2(m[nt][0] - r0), al1 = ex2(m[nt][1] - r1);
            const float p0 = ex2(x0 - r0), p1 = ex2(x1 - r1);
            const float p2 = ex2(x2 - r0), p3 = ex2(x3 - r1);
            l[nt][0] = l[nt][0] * al0 + (p0 + p2);
            l[nt][1] = l[nt][1] * al1 + (p1 + p3);
            m[nt][0] = mn0;
            m[nt][1] = mn1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[nt][mt][0] *= al0;
                o[nt][mt][1] *= al1;
                o[nt][mt][2] *= al0;
                o[nt][mt][3] *= al1;
            }
            b[nt][0] = movmatrix_t(pack_bf16(p0, p1));  // keys 0..7
            b[nt][1] = movmatrix_t(pack_bf16(p2, p3));  // keys 8..15
        }
        {
            const int mi = lane >> 3;
            const uint32_t row = kb + (lane & 7) + (mi >> 1) * 8;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int dc = 2 * mt + (mi & 1);  // 16-byte chunk along d
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(sw128(vt + (dc >> 3) * kHalfBytes, row, dc & 7), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt)
                    mma_bf16_16816(o[nt][mt][0], o[nt][mt][1], o[nt][mt][2], o[nt][mt][3], a0,
                                   a1, a2, a3, b[nt][0], b[nt][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }

    if (n_iter == 0) {  // no keys here: a partial that carries no weight
        const int t = threadIdx.x;
        const int d0 = (t & 31) * 4;
        for (int n = t >> 5; n < group; n += kWarps) {
            const int h = g * group + n;
            *reinterpret_cast<float4 *>(part_o + (size_t(split) * hq + h) * kD + d0) =
                make_float4(0.f, 0.f, 0.f, 0.f);
            if (d0 == 0) part_lse[split * hq + h] = -INFINITY;
        }
        return;
    }

    // ------------------------------------------- merge the 4 warps' states
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
            l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
        }
        const int h0 = nt * 8 + 2 * ti, h1 = h0 + 1;  // this lane's heads in the group
        if (h0 < group) {
            float *w0 = cmb_o + (warp * kMG + h0) * kD;
            float *w1 = cmb_o + (warp * kMG + h1) * kD;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int d = 16 * mt + gi;
                w0[d] = o[nt][mt][0];
                w1[d] = o[nt][mt][1];
                w0[d + 8] = o[nt][mt][2];
                w1[d + 8] = o[nt][mt][3];
            }
            if (gi == 0) {
                cmb_m[warp * kMG + h0] = m[nt][0];
                cmb_m[warp * kMG + h1] = m[nt][1];
                cmb_l[warp * kMG + h0] = l[nt][0];
                cmb_l[warp * kMG + h1] = l[nt][1];
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");

    const int t = threadIdx.x;            // 0..127: query head n, dims d0..d0+3
    const int d0 = (t & 31) * 4;
    for (int n = t >> 5; n < group; n += kWarps) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cmb_m[w * kMG + n]);
        float den = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = cmb_m[w * kMG + n];
            const float f = mw == -INFINITY ? 0.f : ex2(mw - M);
            den += f * cmb_l[w * kMG + n];
            const float4 v =
                *reinterpret_cast<const float4 *>(cmb_o + (w * kMG + n) * kD + d0);
            acc[0] += f * v.x;
            acc[1] += f * v.y;
            acc[2] += f * v.z;
            acc[3] += f * v.w;
        }
        const float inv = 1.f / den;
        const int h = g * group + n;
        *reinterpret_cast<float4 *>(part_o + (size_t(split) * hq + h) * kD + d0) =
            make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
        if (d0 == 0) part_lse[split * hq + h] = M + __log2f(den);
    }
}

// Merge the chunk results of every query head: with per-chunk normalised
// outputs O_c and base-2 log-sum-exp values lse_c,
//   out = sum_c 2^(lse_c - M) O_c / sum_c 2^(lse_c - M),  M = max_c lse_c.
// One CTA per query head; warp w merges chunks w, w+8, ... (lane = 4 dims)
// with a running maximum, then warp 0 merges the 8 warps' states.
constexpr int kCmbWarps = 8;
constexpr int kCmbUnroll = 4;

__global__ void __launch_bounds__(kCmbWarps * 32)
decode_combine_kernel(const float *__restrict__ part_o,
                      const float *__restrict__ part_lse, int n_split, int hq,
                      __nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
                      const int *__restrict__ seqlens, int Lmax) {
    // The next kernel on the stream may be scheduled now (it waits for this
    // grid's completion before touching its results).  This kernel is a
    // programmatic dependent of the split kernel: wait until its results are
    // visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float s_m[kCmbWarps], s_den[kCmbWarps];
    __shared__ float4 s_acc[kCmbWarps][32];
    const int h = blockIdx.x, seq = blockIdx.y;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (seqlens != nullptr) {
        const int L = __ldg(seqlens + seq);
        if (L < 1 || L > Lmax) return;  // flagged by the split kernel; out untouched
    }
    part_o += size_t(seq) * n_split * hq * kD;
    part_lse += size_t(seq) * n_split * hq;
    out += size_t(seq) * hq * kD;
    if (lse != nullptr) lse += size_t(seq) * hq;
    const int d0 = lane * 4;
    float m = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = w; s0 < n_split; s0 += kCmbWarps * kCmbUnroll) {
        float l[kCmbUnroll];
        float4 o[kCmbUnroll];
#pragma unroll
        for (int u = 0; u < kCmbUnroll; ++u) {  // issue every load first
            const int s = s0 + u * kCmbWarps;
            if (s < n_split) {
                l[u] = __ldcg(part_lse + s * hq + h);
                o[u] = __ldcg(reinterpret_cast<const float4 *>(
                    part_o + (size_t(s) * hq + h) * kD + d0));
            }
        }
#pragma unroll
        for (int u = 0; u < kCmbUnroll; ++u) {
            if (s0 + u * kCmbWarps >= n_split) break;
            if (l[u] == -INFINITY) continue;  // a chunk past the sequence's end
            if (l[u] > m) {
                const float sc = ex2(m - l[u]);  // 0 while m is -inf
                den *= sc;
                acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
                m = l[u];
            }
            const float wt = ex2(l[u] - m);
            den += wt;
            acc.x += wt * o[u].x; acc.y += wt * o[u].y;
            acc.z += wt * o[u].z; acc.w += wt * o[u].w;
        }
    }
    if (lane == 0) {
        s_m[w] = m;
        s_den[w] = den;
    }
    s_acc[w][lane] = acc;
    __syncthreads();
    if (w != 0) return;
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kCmbWarps; ++i) M = fmaxf(M, s_m[i]);
    float tden = 0.f;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kCmbWarps; ++i) {
        if (s_m[i] == -INFINITY) continue;  // a warp with no chunk
        const float f = ex2(s_m[i] - M);
        tden += f * s_den[i];
        const float4 a = s_acc[i][lane];
        t.x += f * a.x; t.y += f * a.y; t.z += f * a.z; t.w += f * a.w;
    }
    const float inv = 1.f / tden;
    if (lse != nullptr && lane == 0)  // base-2 chunk values -> natural log
        lse[h] = (M + __log2f(tden)) * 0.6931471805599453f;
    uint2 pk;
    pk.x = pack_bf16(t.x * inv, t.y * inv);
    pk.y = pack_bf16(t.z * inv, t.w * inv);
    *reinterpret_cast<uint2 *>(out + h * kD + d0) = pk;
}

}  // namespace

DecodePlan decode_plan(int Lmax, int batch, int num_sms, int hq, int hkv) {
    const int max_split = (Lmax + kStageKeys - 1) / kStageKeys;
    // one wave of (split, KV head, sequence) CTAs
    int n = int(num_sms * kCtasPerSm / (static_cast<long long>(hkv) * batch));
    if (n < 1) n = 1;
    if (n > max_split) n = max_split;
    int chunk = (Lmax + n - 1) / n;
    chunk = (chunk + kStageKeys - 1) / kStageKeys * kStageKeys;
    DecodePlan p;
    p.chunk = chunk;
    p.n_split = (Lmax + chunk - 1) / chunk;
    p.batch = batch;
    p.hq = hq;
    p.hkv = hkv;
    return p;
}

size_t decode_workspace_bytes(const DecodePlan &p) {
    const size_t parts = size_t(p.n_split) * p.batch;
    const size_t o = parts * p.hq * kD * sizeof(float);
    const size_t lse = parts * p.hq * sizeof(float);
    return o + ((lse + 255) / 256) * 256;
}

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap,
                          const void *q, void *out, float *lse, const int *seqlens, int Lmax,
                          const DecodePlan &plan, void *workspace, unsigned *err,
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
        cudaError_t r = cudaFuncSetAttribute(decode_split_kernel<kGroup, 1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem_bytes(1)));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(decode_split_kernel<0, 1>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(smem_bytes(1)));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(decode_split_kernel<0, 2>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(smem_bytes(2)));
        configured[dev] = r;
    });
    if ((e = configured[dev]) != cudaSuccess) return e;
    const int group = plan.hq / plan.hkv;
    float *part_o = static_cast<float *>(workspace);
    float *part_lse = part_o + size_t(plan.n_split) * plan.batch * plan.hq * kD;

    // Both kernels are programmatic dependents of their predecessor on the
    // stream: their launch and set-up overlap it, and each waits
    // (griddepcontrol.wait) before reading anything the predecessor wrote.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.n_split, plan.hkv, plan.batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes(group <= 8 ? 1 : 2);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg,
                           group == kGroup ? decode_split_kernel<kGroup, 1>
                           : group <= 8    ? decode_split_kernel<0, 1>
                                           : decode_split_kernel<0, 2>,
                           kmap, vmap, static_cast<const __nv_bfloat16 *>(q), seqlens, Lmax,
                           plan.chunk, plan.hq, group, part_o, part_lse, err);
    if (e != cudaSuccess) return e;

    cfg.gridDim = dim3(plan.hq, plan.batch);
    cfg.blockDim = dim3(kCmbWarps * 32);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel,
                              static_cast<const float *>(part_o),
                              static_cast<const float *>(part_lse), plan.n_split, plan.hq,
                              static_cast<__nv_bfloat16 *>(out), lse, seqlens, Lmax);
}

}  // namespace gqa
