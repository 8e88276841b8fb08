// gqa_attn.cu -- host side of the C ABI declared in include/gqa_attn.h:
// argument validation, per-device state (SM count, error word, decode
// workspace), TMA tensor-map encoding and kernel dispatch.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"

using gqa::kD;
using gqa::kHkv;
using gqa::kHq;
using gqa::kMaxDevices;

// Fixed scratch of gqa_attn_decode_noalloc: the decode's per-chunk partial
// results live here instead of in allocated memory.  1 MiB holds the
// partials of up to 63 chunks (a 152-SM GB300 uses at most 38).  Every GPU
// that loads this library holds one copy until the process exits, and all
// calls on a device share it.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {

// Per-device word the kernels OR their error bits into (bounded waits that
// ran out).  Read and cleared through gqa_attn_device_error().
__device__ unsigned g_device_error;

constexpr int kMaxPrefillLen = 1 << 20;
constexpr int kMaxPrefillTotal = 1 << 24;  // rows of a packed batch
constexpr int kMaxDecodeLen = 1 << 26;
constexpr long long kMaxDecodeRows = 1ll << 30;  // batch x cache rows
constexpr int kMaxHeads = 256;                  // query heads of the *_heads entries

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    unsigned *err = nullptr;       // device address of g_device_error
    void *workspace = nullptr;     // decode partials (library-owned)
    size_t workspace_bytes = 0;
    void *scratch = nullptr;       // device address of g_decode_scratch
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Text of the last failing CUDA call on this host thread.
thread_local char t_last_error[160] = "";

void note_error(const char *what, cudaError_t e) {
    snprintf(t_last_error, sizeof t_last_error, "%s: %s (%d)", what, cudaGetErrorString(e),
             int(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Current device's state, probing it on first use.
gqa_status current_device(DeviceState **out) {
    int dev = -1;
    const cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess) {
        note_error("cudaGetDevice", ge);
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GQA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess) {
            cudaGetLastError();
            return GQA_ERR_CUDA;
        }
        d.supported = (major == 10 && minor == 3);
        if (d.supported &&
            cudaGetSymbolAddress(reinterpret_cast<void **>(&d.err), g_device_error) !=
                cudaSuccess) {
            cudaGetLastError();
            return GQA_ERR_CUDA;
        }
        d.probed = true;
    }
    if (!d.supported) return GQA_ERR_DEVICE;
    *out = &d;
    return GQA_OK;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Device memory of the current device (plain or managed)?
gqa_status check_device_ptr(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_POINTER;
    }
    int dev = -1;
    cudaGetDevice(&dev);
    if (a.type == cudaMemoryTypeDevice && a.device == dev) return GQA_OK;
    if (a.type == cudaMemoryTypeManaged) return GQA_OK;
    return GQA_ERR_POINTER;
}

// [rows][heads][128] bf16 tensor, boxes of box_rows x 1 head x 64 dims,
// 128-byte swizzle (the layout the kernels' shared-memory tiles assume).
gqa_status encode_bshd(CUtensorMap *m, const void *base, int rows, int heads, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return GQA_ERR_CUDA;
    const cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(heads), cuuint64_t(rows)};
    const cuuint64_t strides[2] = {cuuint64_t(kD) * 2, cuuint64_t(heads) * kD * 2};
    const cuuint32_t box[3] = {64u, 1u, cuuint32_t(box_rows)};
    const cuuint32_t estride[3] = {1u, 1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(t_last_error, sizeof t_last_error, "cuTensorMapEncodeTiled: CUresult %d",
                 int(r));
        return GQA_ERR_CUDA;
    }
    return GQA_OK;
}

gqa_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return GQA_OK;
    note_error("kernel launch", e);
    cudaGetLastError();
    return GQA_ERR_CUDA;
}

// Validation shared by both decode entry points; launches nothing.
gqa_status decode_args(const void *q, const void *kc, const void *vc, void *out, int L,
                       DeviceState **dev) {
    if (!q || !kc || !vc || !out) return GQA_ERR_NULL;
    if (misaligned(q) || misaligned(kc) || misaligned(vc) || misaligned(out))
        return GQA_ERR_ALIGN;
    if (L < 1 || L > kMaxDecodeLen) return GQA_ERR_SHAPE;
    gqa_status st = current_device(dev);
    if (st != GQA_OK) return st;
    for (const void *p : {q, kc, vc, static_cast<const void *>(out)}) {
        st = check_device_ptr(p);
        if (st != GQA_OK) return st;
    }
    return GQA_OK;
}

// Device address of this device's copy of g_decode_scratch.  In host code the
// array's name only stands for the symbol, so the address is looked up once
// per device, with that device current, and cached.
gqa_status decode_scratch(DeviceState *dev, void **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!dev->scratch) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GQA_ERR_CUDA;
        }
        dev->scratch = p;
    }
    *out = dev->scratch;
    return GQA_OK;
}

gqa_status run_decode(const void *q, const void *kc, const void *vc, void *out, float *lse,
                      const int *seqlens, int Lmax, const gqa::DecodePlan &plan, void *ws,
                      unsigned *err, cudaStream_t stream) {
    CUtensorMap kmap, vmap;
    const int rows = Lmax * plan.batch;
    gqa_status st = encode_bshd(&kmap, kc, rows, plan.hkv, gqa::kDecodeBoxRows);
    if (st == GQA_OK) st = encode_bshd(&vmap, vc, rows, plan.hkv, gqa::kDecodeBoxRows);
    if (st != GQA_OK) return st;
    return from_cuda(gqa::launch_decode(kmap, vmap, q, out, lse, seqlens, Lmax, plan, ws, err,
                                        stream));
}

// Library-owned decode workspace of at least `need` bytes on this device
// (grown with cudaMalloc when a larger batch needs it; never inside capture).
gqa_status library_workspace(DeviceState *dev, size_t need, void **ws) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev->workspace_bytes < need) {
        // at least the largest single-sequence plan, so batch 1 never regrows
        const gqa::DecodePlan most = gqa::decode_plan(kMaxDecodeLen, 1, dev->num_sms);
        size_t bytes = gqa::decode_workspace_bytes(most);
        if (bytes < need) bytes = need;
        void *p = nullptr;
        const cudaError_t e = cudaMalloc(&p, bytes);
        if (e != cudaSuccess) {
            note_error("cudaMalloc (decode workspace)", e);
            cudaGetLastError();
            return GQA_ERR_CUDA;
        }
        if (dev->workspace) cudaFree(dev->workspace);
        dev->workspace = p;
        dev->workspace_bytes = bytes;
    }
    *ws = dev->workspace;
    return GQA_OK;
}

}  // namespace

extern "C" {

// Shared by every prefill entry: B packed sequences over `total` rows (cu
// null: one sequence of `total` rows).
static gqa_status prefill_impl(const void *q, const void *k, const void *v, void *out,
                               float *lse, const int *cu, int B, int max_len, int total,
                               int causal, int hq, int hkv, cudaStream_t stream) {
    if (!q || !k || !v || !out) return GQA_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out))
        return GQA_ERR_ALIGN;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return GQA_ERR_ALIGN;
    if (cu && (reinterpret_cast<uintptr_t>(cu) & 3u)) return GQA_ERR_ALIGN;
    if (B < 1 || max_len < 1 || max_len > kMaxPrefillLen || total < 1 ||
        total > kMaxPrefillTotal)
        return GQA_ERR_SHAPE;
    if (hkv < 1 || hq < hkv || hq > kMaxHeads || hq % hkv != 0) return GQA_ERR_SHAPE;
    const long long blocks = ((max_len + 127) / 128 + 1) / 2;
    if (blocks * B * hq > 0x7fffffffLL) return GQA_ERR_SHAPE;
    DeviceState *dev = nullptr;
    gqa_status st = current_device(&dev);
    if (st != GQA_OK) return st;
    for (const void *p : {q, k, v, static_cast<const void *>(out)}) {
        st = check_device_ptr(p);
        if (st != GQA_OK) return st;
    }
    if (lse && (st = check_device_ptr(lse)) != GQA_OK) return st;
    if (cu && (st = check_device_ptr(cu)) != GQA_OK) return st;
    CUtensorMap qmap, kmap, vmap;
    st = encode_bshd(&qmap, q, total, hq, gqa::kPrefillBoxRows);
    if (st == GQA_OK) st = encode_bshd(&kmap, k, total, hkv, gqa::kPrefillBoxRows);
    if (st == GQA_OK) st = encode_bshd(&vmap, v, total, hkv, gqa::kPrefillBoxRows);
    if (st != GQA_OK) return st;
    return from_cuda(gqa::launch_prefill(qmap, kmap, vmap, out, lse, cu, B, max_len, total,
                                         causal ? 1 : 0, hq, hkv, dev->num_sms, dev->err,
                                         stream));
}

gqa_status gqa_attn_prefill(const void *q, const void *k, const void *v, void *out, int S,
                            int causal, cudaStream_t stream) {
    return prefill_impl(q, k, v, out, nullptr, nullptr, 1, S, S, causal, kHq, kHkv, stream);
}

gqa_status gqa_attn_prefill_lse(const void *q, const void *k, const void *v, void *out,
                                float *lse, int S, int causal, cudaStream_t stream) {
    if (!lse) return GQA_ERR_NULL;
    return prefill_impl(q, k, v, out, lse, nullptr, 1, S, S, causal, kHq, kHkv, stream);
}

gqa_status gqa_attn_prefill_varlen(const void *q, const void *k, const void *v, void *out,
                                   float *lse, const int *cu_seqlens, int batch,
                                   int max_seqlen, int total, int causal,
                                   cudaStream_t stream) {
    if (!cu_seqlens) return GQA_ERR_NULL;
    return prefill_impl(q, k, v, out, lse, cu_seqlens, batch, max_seqlen, total, causal, kHq,
                        kHkv, stream);
}

gqa_status gqa_attn_prefill_heads(const void *q, const void *k, const void *v, void *out,
                                  float *lse, const int *cu_seqlens, int batch, int max_seqlen,
                                  int total, int num_q_heads, int num_kv_heads, int causal,
                                  cudaStream_t stream) {
    if (!cu_seqlens && batch != 1) return GQA_ERR_SHAPE;
    if (!cu_seqlens && max_seqlen != total) return GQA_ERR_SHAPE;
    return prefill_impl(q, k, v, out, lse, cu_seqlens, batch, max_seqlen, total, causal,
                        num_q_heads, num_kv_heads, stream);
}

gqa_status gqa_attn_prefill_pair(const void *q, const void *k, const void *v, void *out,
                                 float *lse, int S, int causal, cudaStream_t stream) {
    if (!q || !k || !v || !out) return GQA_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out))
        return GQA_ERR_ALIGN;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return GQA_ERR_ALIGN;
    if (S < 1 || S > kMaxPrefillLen) return GQA_ERR_SHAPE;
    DeviceState *dev = nullptr;
    gqa_status st = current_device(&dev);
    if (st != GQA_OK) return st;
    for (const void *p : {q, k, v, static_cast<const void *>(out)}) {
        st = check_device_ptr(p);
        if (st != GQA_OK) return st;
    }
    if (lse && (st = check_device_ptr(lse)) != GQA_OK) return st;
    CUtensorMap qmap, kmap, vmap;
    st = encode_bshd(&qmap, q, S, kHq, gqa::kPrefillBoxRows);
    if (st == GQA_OK) st = encode_bshd(&kmap, k, S, kHkv, gqa::kPairKBoxRows);
    if (st == GQA_OK) st = encode_bshd(&vmap, v, S, kHkv, gqa::kPrefillBoxRows);
    if (st != GQA_OK) return st;
    return from_cuda(gqa::launch_prefill_pair(qmap, kmap, vmap, out, lse, S, causal ? 1 : 0,
                                              kHq, kHkv, dev->err, stream));
}

size_t gqa_attn_decode_workspace_bytes(int L) {
    if (L < 1 || L > kMaxDecodeLen) return 0;
    DeviceState *dev = nullptr;
    if (current_device(&dev) != GQA_OK) return 0;
    return gqa::decode_workspace_bytes(gqa::decode_plan(L, 1, dev->num_sms));
}

int gqa_attn_decode_plan(int L, int batch, int num_sms, int *n_split, int *chunk) {
    if (!n_split || !chunk || L < 1 || L > kMaxDecodeLen || batch < 1 || num_sms < 1)
        return 0;
    const gqa::DecodePlan p = gqa::decode_plan(L, batch, num_sms);
    *n_split = p.n_split;
    *chunk = p.chunk;
    return 1;
}

int gqa_attn_decode_num_splits(int L) {
    if (L < 1 || L > kMaxDecodeLen) return 0;
    DeviceState *dev = nullptr;
    if (current_device(&dev) != GQA_OK) return 0;
    return gqa::decode_plan(L, 1, dev->num_sms).n_split;
}

gqa_status gqa_attn_decode_ws(const void *q, const void *kcache, const void *vcache,
                              void *out, int L, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    DeviceState *dev = nullptr;
    gqa_status st = decode_args(q, kcache, vcache, out, L, &dev);
    if (st != GQA_OK) return st;
    const gqa::DecodePlan plan = gqa::decode_plan(L, 1, dev->num_sms);
    if (!workspace || misaligned(workspace) ||
        workspace_bytes < gqa::decode_workspace_bytes(plan))
        return GQA_ERR_WORKSPACE;
    st = check_device_ptr(workspace);
    if (st != GQA_OK) return GQA_ERR_WORKSPACE;
    return run_decode(q, kcache, vcache, out, nullptr, nullptr, L, plan, workspace, dev->err,
                      stream);
}

static gqa_status decode_impl(const void *q, const void *kcache, const void *vcache, void *out,
                              float *lse, int L, cudaStream_t stream) {
    DeviceState *dev = nullptr;
    gqa_status st = decode_args(q, kcache, vcache, out, L, &dev);
    if (st != GQA_OK) return st;
    if (lse && (st = check_device_ptr(lse)) != GQA_OK) return st;
    const gqa::DecodePlan plan = gqa::decode_plan(L, 1, dev->num_sms);
    void *ws = nullptr;
    st = library_workspace(dev, gqa::decode_workspace_bytes(plan), &ws);
    if (st != GQA_OK) return st;
    return run_decode(q, kcache, vcache, out, lse, nullptr, L, plan, ws, dev->err, stream);
}

gqa_status gqa_attn_decode(const void *q, const void *kcache, const void *vcache, void *out,
                           int L, cudaStream_t stream) {
    return decode_impl(q, kcache, vcache, out, nullptr, L, stream);
}

gqa_status gqa_attn_decode_lse(const void *q, const void *kcache, const void *vcache, void *out,
                               float *lse, int L, cudaStream_t stream) {
    if (!lse) return GQA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return GQA_ERR_ALIGN;
    return decode_impl(q, kcache, vcache, out, lse, L, stream);
}

static gqa_status decode_batched_impl(const void *q, const void *kcache, const void *vcache,
                                      void *out, float *lse, const int *seqlens, int batch,
                                      int max_len, int hq, int hkv, cudaStream_t stream) {
    if (!q || !kcache || !vcache || !out) return GQA_ERR_NULL;
    if (misaligned(q) || misaligned(kcache) || misaligned(vcache) || misaligned(out))
        return GQA_ERR_ALIGN;
    if ((lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
        (seqlens && (reinterpret_cast<uintptr_t>(seqlens) & 3u)))
        return GQA_ERR_ALIGN;
    if (batch < 1 || max_len < 1 || max_len > kMaxDecodeLen ||
        (long long)batch * max_len > kMaxDecodeRows)
        return GQA_ERR_SHAPE;
    if (hkv < 1 || hq < hkv || hq > kMaxHeads || hq % hkv != 0 ||
        hq / hkv > gqa::kDecodeMaxGroup)
        return GQA_ERR_SHAPE;
    DeviceState *dev = nullptr;
    gqa_status st = current_device(&dev);
    if (st != GQA_OK) return st;
    for (const void *p : {q, kcache, vcache, static_cast<const void *>(out)}) {
        st = check_device_ptr(p);
        if (st != GQA_OK) return st;
    }
    if (lse && (st = check_device_ptr(lse)) != GQA_OK) return st;
    if (seqlens && (st = check_device_ptr(seqlens)) != GQA_OK) return st;
    const gqa::DecodePlan plan = gqa::decode_plan(max_len, batch, dev->num_sms, hq, hkv);
    void *ws = nullptr;
    st = library_workspace(dev, gqa::decode_workspace_bytes(plan), &ws);
    if (st != GQA_OK) return st;
    return run_decode(q, kcache, vcache, out, lse, seqlens, max_len, plan, ws, dev->err,
                      stream);
}

gqa_status gqa_attn_decode_batched(const void *q, const void *kcache, const void *vcache,
                                   void *out, float *lse, const int *seqlens, int batch,
                                   int max_len, cudaStream_t stream) {
    return decode_batched_impl(q, kcache, vcache, out, lse, seqlens, batch, max_len, kHq, kHkv,
                               stream);
}

gqa_status gqa_attn_decode_heads(const void *q, const void *kcache, const void *vcache,
                                 void *out, float *lse, const int *seqlens, int batch,
                                 int max_len, int num_q_heads, int num_kv_heads,
                                 cudaStream_t stream) {
    return decode_batched_impl(q, kcache, vcache, out, lse, seqlens, batch, max_len,
                               num_q_heads, num_kv_heads, stream);
}

gqa_status gqa_attn_decode_noalloc(const void *q, const void *kcache, const void *vcache,
                                   void *out, int L, cudaStream_t stream) {
    DeviceState *dev = nullptr;
    gqa_status st = decode_args(q, kcache, vcache, out, L, &dev);
    if (st != GQA_OK) return st;
    const gqa::DecodePlan plan = gqa::decode_plan(L, 1, dev->num_sms);
    if (gqa::decode_workspace_bytes(plan) > kNoAllocScratchBytes) return GQA_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = decode_scratch(dev, &scratch);
    if (st != GQA_OK) return st;
    return run_decode(q, kcache, vcache, out, nullptr, nullptr, L, plan, scratch, dev->err,
                      stream);
}

int gqa_attn_launches_per_call(int is_decode) { return is_decode ? 2 : 1; }

gqa_status gqa_attn_device_error(unsigned int *flags, int clear) {
    if (!flags) return GQA_ERR_NULL;
    DeviceState *dev = nullptr;
    gqa_status st = current_device(&dev);
    if (st != GQA_OK) return st;
    unsigned word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, dev->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GQA_ERR_CUDA;
    }
    if (clear && word) {
        const unsigned zero = 0;
        if (cudaMemcpy(dev->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return GQA_ERR_CUDA;
        }
    }
    *flags = word;
    return word ? GQA_ERR_TIMEOUT : GQA_OK;
}

gqa_status gqa_attn_selftest_wait_timeout(unsigned int *flags) {
    if (!flags) return GQA_ERR_NULL;
    unsigned before = 0;
    gqa_status st = gqa_attn_device_error(&before, 1);  // start from a clear word
    if (st != GQA_OK && st != GQA_ERR_TIMEOUT) return st;
    DeviceState *dev = nullptr;
    st = current_device(&dev);
    if (st != GQA_OK) return st;
    st = from_cuda(gqa::launch_wait_timeout_selftest(dev->err, 0));
    if (st != GQA_OK) return st;
    return gqa_attn_device_error(flags, 1);
}

const char *gqa_attn_last_error_string(void) { return t_last_error; }

const char *gqa_attn_status_string(gqa_status s) {
    switch (s) {
    case GQA_OK: return "ok";
    case GQA_ERR_NULL: return "a required pointer is NULL";
    case GQA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case GQA_ERR_SHAPE: return "sequence length out of range";
    case GQA_ERR_DEVICE: return "current device is not compute capability 10.3 (GB300)";
    case GQA_ERR_WORKSPACE: return "workspace NULL, misaligned or too small";
    case GQA_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case GQA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case GQA_ERR_POINTER: return "a pointer is not device memory of the current device";
    }
    return "unknown status";
}

}  // extern "C"
