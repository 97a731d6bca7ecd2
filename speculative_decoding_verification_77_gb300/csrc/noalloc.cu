// spec_verify_attn_noalloc: dense verification attention for callers that
// cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: serving engines
// that reserve almost all of HBM for the KV cache when they start and forbid
// allocations afterwards (a late cudaMalloc can fail, or stall the device while
// the allocator synchronises), and hosts that reach the library through a
// plain C callback with no allocator of their own. This entry point keeps the
// split-KV partials and the status word in a fixed, file-scope device array
// instead, so it allocates nothing: no cudaMalloc, no cudaFree, no allocating
// library call. It computes what spec_verify_attn computes, within the same
// parity tolerances, but always through the warp-level tensor-core cache
// kernel (mma.sync) and the merge kernel, not the tcgen05 cache kernel that
// spec_verify_attn picks where the shape allows: the results agree within
// tolerance, not bit for bit, and the speed differs.
#include <mutex>

#include "common.cuh"

namespace specverify {

namespace {

// Built-in scratch: status word (first 256 bytes), then o partials, then lse
// partials, carved exactly like a caller's workspace. Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void *g_scratch_addr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of the scratch array on the current device (set up once per
// device, with that device current). The array's name in host code is only a
// host-side stand-in, so the kernels must be given this address instead. The
// result of the first lookup is kept for the process, a failure included: a
// device whose lookup failed keeps returning that error.
cudaError_t scratch_address(int dev, void **out) {
    std::call_once(g_scratch_once[dev], [dev] {
        void *p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        g_scratch_addr[dev] = p;
    });
    *out = g_scratch_addr[dev];
    return g_scratch_err[dev];
}

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

}  // namespace specverify

using namespace specverify;

extern "C" spec_status_t spec_verify_attn_noalloc(
    const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache, int64_t kv_stride_b,
    int64_t kv_stride_h, int64_t kv_stride_t, const uint16_t *k_draft, const uint16_t *v_draft,
    const int32_t *parent, int B, int N, int Hq, int Hkv, int d, int L, const int32_t *ctx_lens,
    float scale, float *out, float *lse, int32_t *status_out, void *stream) {
    // host checks (the same as spec_verify_attn's)
    if (!q || !out || !lse) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || N > 4096 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || L < 0) return SPEC_ERR_INVALID_ARG;
    if (L > 0 && (!k_cache || !v_cache)) return SPEC_ERR_INVALID_ARG;
    if ((k_draft == nullptr) != (v_draft == nullptr)) return SPEC_ERR_INVALID_ARG;
    if (k_draft && !parent) return SPEC_ERR_INVALID_ARG;
    if (kv_stride_b < 0 || kv_stride_h < 0 || kv_stride_t < 0 || kv_stride_b % 8 || kv_stride_h % 8 ||
        kv_stride_t % 8)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_draft, 16) ||
        !aligned(v_draft, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(parent, 4) ||
        !aligned(ctx_lens, 4) || !aligned(status_out, 4))
        return SPEC_ERR_INVALID_ARG;
    if (!(scale == scale)) return SPEC_ERR_INVALID_ARG;
    if (d != kHeadDim) return SPEC_ERR_UNSUPPORTED;
    if ((int64_t)B * N * Hq > (int64_t)1 << 31) return SPEC_ERR_INVALID_ARG;
    // the split plan numbers tiles in 32-bit arithmetic (the same guard as spec_verify_attn)
    if ((int64_t)B * Hkv * (((int64_t)(Hq / Hkv) * N + 63) / 64) * ((int64_t)L / 64 + 1) >= ((int64_t)1 << 31))
        return SPEC_ERR_UNSUPPORTED;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SPEC_ERR_UNSUPPORTED;
    }
    if (major != 10 || minor != 3) return SPEC_ERR_UNSUPPORTED;

    // the problem must fit the built-in scratch
    const SplitPlan plan = make_plan(B, N, Hq, Hkv, L, mma_rows_per_unit(), mma_tile_tokens(), sms * 2);
    if (plan_workspace_bytes(plan, d) > kNoAllocScratchBytes) return SPEC_ERR_WORKSPACE;

    void *base = nullptr;
    if (const cudaError_t e = scratch_address(dev, &base); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    if (base == nullptr) return SPEC_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(base);

    VerifyArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.k_cache = reinterpret_cast<const __nv_bfloat16 *>(k_cache);
    a.v_cache = reinterpret_cast<const __nv_bfloat16 *>(v_cache);
    a.sb = kv_stride_b; a.sh = kv_stride_h; a.st = kv_stride_t;
    a.k_draft = reinterpret_cast<const __nv_bfloat16 *>(k_draft);
    a.v_draft = reinterpret_cast<const __nv_bfloat16 *>(v_draft);
    a.parent = parent;
    a.ctx_lens = ctx_lens;
    a.idx = nullptr;
    a.budget = 0;
    a.B = B; a.N = N; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.L = L;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    a.status = reinterpret_cast<uint32_t *>(ws);
    a.table = nullptr;
    a.table_ld = 0;
    a.block_size = 0;
    a.num_blocks = 0;
    a.idx_resolved = 0;
    a.out_bf16 = 0;
    a.kv_fp8 = 0;
    a.k_scale = nullptr;
    a.v_scale = nullptr;
    a.o_part = reinterpret_cast<float *>(ws + kHeaderBytes);
    a.lse_part = reinterpret_cast<float *>(ws + kHeaderBytes +
                                           align_up((size_t)plan.slots * plan.BM * d * sizeof(float), 256));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the scratch keeps the previous call's contents: the status word must start at zero;
    // every partial slot the merge reads is written by this call's cache kernel first
    if (const cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    if (const cudaError_t e = launch_cache_attn_mma(a, plan, false, s, nullptr, nullptr); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    if (const cudaError_t e = launch_merge_tree(a, plan, s); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    if (status_out) {
        if (const cudaError_t e = cudaMemcpyAsync(status_out, a.status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
            e != cudaSuccess)
            return (spec_status_t)cuda_failure(e);
    }
    return SPEC_OK;
}
