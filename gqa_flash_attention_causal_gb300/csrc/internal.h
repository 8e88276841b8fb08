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
// handles chunk `split` of KV head g of sequence seq for its 4 query heads.
struct DecodePlan {
    int n_split;
    int chunk;
    int batch;
};
DecodePlan decode_plan(int Lmax, int batch, int num_sms);
size_t decode_workspace_bytes(const DecodePlan &p);

// q, out [batch][32][128]; caches [batch][Lmax][8][128] behind the tensor
// maps; sequence s attends to its first seqlens[s] rows (seqlens null:
// all Lmax rows).  lse (may be null): [batch][32] fp32 natural-log
// log-sum-exp.
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
// every sequence's length.  lse (may be null): [32][total] fp32, natural-log
// log-sum-exp of each row's scores.
cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, void *out, float *lse,
                           const int *cu_seqlens, int B, int max_len, int total, int causal,
                           int num_sms, unsigned *err, cudaStream_t stream);

// ------------------------------------------------------------------ self-test
// Error bit the self-test kernel's deliberately expiring wait sets.
constexpr unsigned kErrSelfTestBit = 1u << 31;
cudaError_t launch_wait_timeout_selftest(unsigned *err, cudaStream_t stream);

}  // namespace gqa
