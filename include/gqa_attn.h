/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) grouped-query attention forward
 * library: causal prefill over a whole prompt and single-token decode against
 * a KV cache.
 *
 * The operation (chowfi/kernels README, "Result" section and the settings
 * line under its table): the attention step of a Llama-3-8B-size model,
 * forward only, bf16, batch 1, 32 query heads sharing 8 KV heads, head size
 * 128.  For query head h the KV head is g = h / 4 (4 query heads per group):
 *
 *     out[i,h,:] = sum_{j in J(i)} softmax_j( q[i,h,:] . k[j,g,:] / sqrt(128) ) v[j,g,:]
 *
 * Prefill: J(i) = {0..i} when causal ("Skip the masked half in prefill":
 * causal attention ignores future tokens), {0..S-1} otherwise.
 * Decode: one new query against every one of the L cached positions.
 * Products and sums accumulate in fp32; the output is rounded to bf16 (RNE).
 *
 * Conventions shared by every call:
 *  - Geometry is fixed: batch 1, 32 query heads, 8 KV heads, head dim 128.
 *  - Tensors are bf16, contiguous, sequence-major (BSHD):
 *      prefill  q, out [1][S][32][128]   k, v [1][S][8][128]
 *      decode   q, out [1][1][32][128]   kcache, vcache [1][L][8][128]
 *  - Every pointer is a DEVICE pointer on the current CUDA device, owned by
 *    the caller, 16-byte aligned; inputs are only read, out is only written.
 *    The library keeps no reference to them after the call returns.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream): the
 *    result is valid once the stream reaches that point.  No call
 *    synchronises the host, except where noted.
 *  - Errors are status codes; no call throws.  A validation error launches
 *    nothing and leaves `out` untouched.
 *  - The current device must be a compute-capability 10.3 GPU (GB300).
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_ATTN_NUM_Q_HEADS 32
#define GQA_ATTN_NUM_KV_HEADS 8
#define GQA_ATTN_HEAD_DIM 128

typedef enum {
    GQA_OK = 0,
    GQA_ERR_NULL = 1,      /* a required pointer is NULL                      */
    GQA_ERR_ALIGN = 2,     /* a pointer is not 16-byte aligned                */
    GQA_ERR_SHAPE = 3,     /* S or L < 1, or too large for 32-bit indexing    */
    GQA_ERR_DEVICE = 4,    /* current device is not compute capability 10.3   */
    GQA_ERR_WORKSPACE = 5, /* caller workspace NULL, misaligned or too small  */
    GQA_ERR_TIMEOUT = 6,   /* a bounded device-side wait ran out (see below)  */
    GQA_ERR_CUDA = 7,      /* a CUDA runtime or driver call failed            */
    GQA_ERR_POINTER = 8    /* a pointer is not device memory of this device   */
} gqa_status;

/*
 * Causal (or, with causal = 0, bidirectional) prefill attention.
 * q, out: [1][S][32][128] bf16; k, v: [1][S][8][128] bf16; 1 <= S <= 2^20.
 * Persistent tcgen05/TMA kernel; fully masked causal tiles are skipped.
 * Needs no workspace.  Returns GQA_OK once the kernel is enqueued.
 */
gqa_status gqa_attn_prefill(const void *q, const void *k, const void *v,
                            void *out, int S, int causal, cudaStream_t stream);

/*
 * gqa_attn_prefill that also returns, for every query row and head, the
 * natural-log log-sum-exp of that row's scaled scores,
 *     lse[h][i] = ln sum_{j in J(i)} exp( q[i,h,:] . k[j,g,:] / sqrt(128) ),
 * the normaliser of the softmax (what a backward pass or a merge of
 * attention over separate key ranges needs).  lse: [32][S] fp32 device
 * memory, 4-byte aligned, written only for rows < S.
 */
gqa_status gqa_attn_prefill_lse(const void *q, const void *k, const void *v,
                                void *out, float *lse, int S, int causal,
                                cudaStream_t stream);

/*
 * Prefill of a batch of `batch` independent sequences packed along the
 * sequence axis (the layout variable-length serving uses): sequence s
 * occupies rows cu_seqlens[s] .. cu_seqlens[s+1]-1 of
 *     q, out [total][32][128] bf16,   k, v [total][8][128] bf16,
 * and attends only within itself (causal or not).  cu_seqlens: batch+1
 * non-decreasing int32 offsets in DEVICE memory with cu_seqlens[0] = 0 and
 * cu_seqlens[batch] = total; max_seqlen (host) >= every sequence's length,
 * <= 2^20; total <= 2^24.  lse (may be NULL): [32][total] fp32, natural-log
 * log-sum-exp of every row, as gqa_attn_prefill_lse.  A sequence whose
 * offsets fall outside [0, total] or whose length exceeds max_seqlen is not
 * computed and sets bit 5 of the device error word (gqa_attn_device_error).
 * With batch = 1 and cu_seqlens = {0, S} it computes gqa_attn_prefill.
 */
gqa_status gqa_attn_prefill_varlen(const void *q, const void *k, const void *v,
                                   void *out, float *lse, const int *cu_seqlens,
                                   int batch, int max_seqlen, int total, int causal,
                                   cudaStream_t stream);

/*
 * Prefill for other head layouts (the pages' model is the 32 / 8 case; the
 * pages have no counterpart for other counts): num_q_heads query heads share
 * num_kv_heads KV heads, query head h reading KV head
 * h / (num_q_heads / num_kv_heads); head dim 128.  Otherwise exactly
 * gqa_attn_prefill_varlen with the head counts in place of 32 and 8:
 *     q, out [total][num_q_heads][128],  k, v [total][num_kv_heads][128]
 * bf16, lse (may be NULL) [num_q_heads][total] fp32.  cu_seqlens may be NULL
 * for a single sequence (then batch = 1 and max_seqlen = total).
 * 1 <= num_kv_heads <= num_q_heads <= 256, num_q_heads a multiple of
 * num_kv_heads (num_kv_heads = num_q_heads: multi-head attention;
 * num_kv_heads = 1: multi-query attention); otherwise GQA_ERR_SHAPE.
 */
gqa_status gqa_attn_prefill_heads(const void *q, const void *k, const void *v,
                                  void *out, float *lse, const int *cu_seqlens,
                                  int batch, int max_seqlen, int total,
                                  int num_q_heads, int num_kv_heads, int causal,
                                  cudaStream_t stream);

/*
 * gqa_attn_prefill (and, with lse non-NULL, gqa_attn_prefill_lse) computed by
 * the paired-CTA kernel: the CTAs run as clusters of two on the two SMs of a
 * TPC, the two CTAs of a pair compute two query heads of one KV group over
 * the same rows, and every tcgen05 MMA spans both SMs' tensor memory
 * (M = 256 rows, 128 per CTA), each CTA staging half of every K and V tile,
 * so that the pair reads each K/V tile into shared memory once for both
 * heads (chowfi/kernels README, "What helped most", item 2: read K and V once
 * for the query heads of a group).  Same arguments, layouts, limits and
 * result as gqa_attn_prefill_lse with lse optional (the same fp32
 * accumulation order: the output is identical to gqa_attn_prefill's).
 * A device that cannot hold one two-CTA cluster of this kernel gives
 * GQA_ERR_CUDA and nothing is launched.
 */
gqa_status gqa_attn_prefill_pair(const void *q, const void *k, const void *v,
                                 void *out, float *lse, int S, int causal,
                                 cudaStream_t stream);

/*
 * Decode: one query token against a KV cache of length L (every cached
 * position is attended).  q, out: [1][1][32][128] bf16; kcache, vcache:
 * [1][L][8][128] bf16; 1 <= L <= 2^26.
 * The KV length is split into chunks processed in parallel (each chunk reads
 * its K/V once for all 4 query heads of a group), and a second kernel merges
 * the chunk results with a log-sum-exp combine.  The per-chunk partial
 * results live in a library-owned workspace allocated per device on the
 * first call (cudaMalloc; not inside stream capture) and reused afterwards:
 * calls on different streams of one device must not overlap in time.
 */
gqa_status gqa_attn_decode(const void *q, const void *kcache,
                           const void *vcache, void *out, int L,
                           cudaStream_t stream);

/* gqa_attn_decode that also returns lse[h] = ln sum_j exp(q[h,:] . k[j,g,:] /
 * sqrt(128)) for the 32 query heads: [32] fp32 device memory, 4-byte aligned. */
gqa_status gqa_attn_decode_lse(const void *q, const void *kcache,
                               const void *vcache, void *out, float *lse, int L,
                               cudaStream_t stream);

/*
 * Decode of a batch: `batch` independent query tokens, sequence s with its
 * own cache of max_len rows,
 *     q, out [batch][32][128] bf16,   kcache, vcache [batch][max_len][8][128] bf16,
 * attending to the first seqlens[s] rows of its cache (1 <= seqlens[s] <=
 * max_len; seqlens: batch int32 in DEVICE memory, or NULL for all max_len
 * rows).  lse (may be NULL): [batch][32] fp32 as gqa_attn_decode_lse.
 * Chunks of every sequence run in one wave across the SMs and are merged
 * per sequence.  A sequence whose length is outside [1, max_len] is not
 * computed (its out rows are left untouched) and sets bit 5 of the device
 * error word.  Uses (and if needed grows) the library-owned workspace of
 * gqa_attn_decode.  1 <= max_len <= 2^26, batch * max_len <= 2^30.
 */
gqa_status gqa_attn_decode_batched(const void *q, const void *kcache,
                                   const void *vcache, void *out, float *lse,
                                   const int *seqlens, int batch, int max_len,
                                   cudaStream_t stream);

/*
 * Decode for other head layouts (the pages have no counterpart): exactly
 * gqa_attn_decode_batched with num_q_heads / num_kv_heads in place of 32 / 8:
 *     q, out [batch][num_q_heads][128],  caches [batch][max_len][num_kv_heads][128]
 * bf16, lse (may be NULL) [batch][num_q_heads] fp32.  The query heads of a
 * KV head are computed together from one pass over its cache, which holds
 * at most 16 of them: 1 <= num_kv_heads <= num_q_heads <= 256,
 * num_q_heads a multiple of num_kv_heads and num_q_heads / num_kv_heads
 * <= 16; otherwise GQA_ERR_SHAPE.
 */
gqa_status gqa_attn_decode_heads(const void *q, const void *kcache,
                                 const void *vcache, void *out, float *lse,
                                 const int *seqlens, int batch, int max_len,
                                 int num_q_heads, int num_kv_heads,
                                 cudaStream_t stream);

/* Bytes of device workspace gqa_attn_decode_ws needs for length L (0 if L
 * is out of range). */
size_t gqa_attn_decode_workspace_bytes(int L);

/*
 * gqa_attn_decode with a caller-owned device workspace of at least
 * gqa_attn_decode_workspace_bytes(L) bytes, 16-byte aligned.  Allocates
 * nothing, so it may be captured in a CUDA graph (tested).  The workspace
 * must not be used by anything else until the call has completed on `stream`.
 */
gqa_status gqa_attn_decode_ws(const void *q, const void *kcache,
                              const void *vcache, void *out, int L,
                              void *workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/*
 * gqa_attn_decode for callers that cannot allocate device memory: it calls
 * no cudaMalloc, cudaFree or other allocating routine.  (The pages have no
 * counterpart; this is a deployment need.)  Such callers include serving
 * processes whose device memory is entirely handed to their own pool (for
 * instance a KV-cache pool sized to all free HBM, where one more cudaMalloc
 * fails or fragments the pool) and processes running under a fixed device
 * memory budget that forbids allocations after start-up.
 *
 * Arguments, layouts and results are those of gqa_attn_decode; the caller
 * still passes the inputs and the output.  The per-chunk partial results go
 * to a fixed 1 MiB scratch array compiled into the library (every GPU that
 * loads the library holds one copy until the process exits).
 *  - The first call on a device looks up that device's copy of the array
 *    (once per device); make that first call before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    partials: calls that overlap in time on the GPU (e.g. on two streams)
 *    race and give wrong results.  Nothing in it needs to start at zero:
 *    each call writes every partial it reads.
 *  - If length L would need more scratch than 1 MiB on this device (more
 *    than 63 chunks; a 152-SM GB300 uses at most 38), the call returns
 *    GQA_ERR_WORKSPACE and launches nothing.
 */
gqa_status gqa_attn_decode_noalloc(const void *q, const void *kcache,
                                   const void *vcache, void *out, int L,
                                   cudaStream_t stream);

/* The decode's split plan for cache length L, batch and SM count, computed on
 * the host without touching a device: every sequence's cache is cut into
 * *n_split chunks of *chunk keys (a multiple of 64).  Returns 1, or 0 on
 * out-of-range arguments. */
int gqa_attn_decode_plan(int L, int batch, int num_sms, int *n_split, int *chunk);

/* Number of KV chunks (splits) the decode uses for length L on the current
 * device; 0 if L is out of range.  Exposed for tests and the bench. */
int gqa_attn_decode_num_splits(int L);

/* Number of CUDA kernel launches one call makes (prefill: 1; decode: 2). */
int gqa_attn_launches_per_call(int is_decode);

/*
 * Device-side error word of the current device.  Every device-side wait in
 * the kernels is bounded (about a second); on expiry the kernel sets a bit
 * here, abandons its work and exits cleanly instead of hanging.  This call
 * synchronises the device, writes the word to *flags (0 = no error) and,
 * if clear != 0, resets it.  Returns GQA_ERR_TIMEOUT if the word is
 * non-zero, GQA_OK otherwise.
 */
gqa_status gqa_attn_device_error(unsigned int *flags, int clear);

/*
 * Self-test of the failure path behind GQA_ERR_TIMEOUT (the pages have no
 * counterpart).  Launches a one-CTA kernel on the legacy default stream that
 * waits, through the same bounded wait the kernels use, on a barrier that
 * nothing arrives at.  The wait gives up after its limit (about a second),
 * sets bit 31 of the device error word and returns; no fault, no trap, and
 * the context stays usable.  Synchronises the device, clears the word before
 * and after, and stores the word the kernel left in *flags.  Returns
 * GQA_ERR_TIMEOUT when the wait ran out as designed.
 */
gqa_status gqa_attn_selftest_wait_timeout(unsigned int *flags);

/* Text of the most recent failing CUDA call made by this library on the
 * calling host thread (the reason behind a GQA_ERR_CUDA), or "" if none.
 * The string is owned by the library and valid until the thread's next
 * call into it. */
const char *gqa_attn_last_error_string(void);

/* Static description of a status code. */
const char *gqa_attn_status_string(gqa_status status);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
