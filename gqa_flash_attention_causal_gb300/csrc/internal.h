// internal.h -- declarations shared by the host C-ABI layer and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace gqa {

constexpr int kHq = 32;    // query heads
constexpr int kHkv = 8;    // KV heads
constexpr int kGroup = 4;  // query heads per KV head
constexpr int kD = 128;    // head dim
constexpr int kMaxDevices = 64;

// ------------------------------------------------------------------ decode
// Split plan: each sequence's cache (Lmax rows) is cut into n_split chunks
// of `chunk` keys (a multiple of the 64-key stage); CTA (split, g, seq)
// handles chunk `split` of KV head g of sequence seq for its hq / hkv query
// heads (at most 8).
struct DecodePlan {
    int n_split;
    int chunk;
    int batch;
    int hq = kHq;
    int hkv = kHkv;
};
constexpr int kDecodeMaxGroup = 16;  // query heads per KV head the decode supports
DecodePlan decode_plan(int Lmax, int batch, int num_sms, int hq = kHq, int hkv = kHkv);
size_t decode_workspace_bytes(const DecodePlan &p);

// q, out [batch][hq][128]; caches [batch][Lmax][hkv][128] behind the tensor
// maps (the plan's head counts); sequence s attends to its first seqlens[s]
// rows (seqlens null: all Lmax rows).  lse (may be null): [batch][hq] fp32
// natural-log log-sum-exp.
cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap,
                          const void *q, void *out, float *lse, const int *seqlens, int Lmax,
                          const DecodePlan &plan, void *workspace, unsigned *err,
                          cudaStream_t stream);

// Box sizes the kernels expect in their tensor maps (rows of 64 bf16 each).
constexpr int kDecodeBoxRows = 64;
constexpr int kPrefillBoxRows = 128;

// ------------------------------------------------------------------ prefill
// B packed sequences, sequence s at rows cu_seqlens[s] .. cu_seqlens[s+1]-1 of
// `total` rows (cu_seqlens null: one sequence of `total` rows); max_len bounds
// every sequence's length.  hq query heads share hkv KV heads (query head h
// reads KV head h / (hq / hkv)); q, out [total][hq][128], k, v
// [total][hkv][128].  lse (may be null): [hq][total] fp32, natural-log
// log-sum-exp of each row's scores.
cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, void *out, float *lse,
                           const int *cu_seqlens, int B, int max_len, int total, int causal,
                           int hq, int hkv, int num_sms, unsigned *err, cudaStream_t stream);

// Paired-CTA prefill of one sequence (prefill_pair.cu): q, out [S][hq][128],
// k, v [S][hkv][128]; the tensor maps' boxes are kPrefillBoxRows rows for q
// and v and kPairKBoxRows rows for k.  lse as for launch_prefill.
constexpr int kPairKBoxRows = 64;
cudaError_t launch_prefill_pair(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, void *out, float *lse, int S,
                                int causal, int hq, int hkv, unsigned *err,
                                cudaStream_t stream);

// ------------------------------------------------------------------ self-test
// Error bit the self-test kernel's deliberately expiring wait sets.
constexpr unsigned kErrSelfTestBit = 1u << 31;
cudaError_t launch_wait_timeout_selftest(unsigned *err, cudaStream_t stream);

}  // namespace gqa
