// C ABI of libspecverify.so: argument checks, workspace carve-up, dispatch.
// Every declaration and its contract is in include/specverify.h.
#include <mutex>

#include "common.cuh"

namespace specverify {

namespace {

thread_local uint64_t g_launches = 0;

// Clears a verify call's status word. Launched with programmatic stream serialisation, it
// may start while the previous grid runs (a selection lets it), so it writes only once that
// grid is complete; it lets the cache kernel behind it start its set-up at once, and that
// kernel waits for this grid before it can record an error or read the index set.
__global__ void status_reset_kernel(uint32_t *status) {
    griddep_launch_dependents();
    griddep_wait();
    if (threadIdx.x == 0) *status = 0u;
}

thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_stop = nullptr;
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

struct DeviceInfo {
    int ok;   // -1 unknown, 0 unsupported, 1 compute capability 10.3
    int sms;  // multiprocessor count
};
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

// Current device's properties (cached per device). Returns SPEC_OK on a cc 10.3 device.
spec_status_t current_device(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SPEC_ERR_UNSUPPORTED;
    }
    std::call_once(g_dev_once[dev], [dev] {
        int major = 0, minor = 0, sms = 0;
        bool good = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
                    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
        cudaGetLastError();
        g_dev[dev].ok = good && major == 10 && minor == 3 ? 1 : 0;
        g_dev[dev].sms = sms > 0 ? sms : 0;
    });
    *out = g_dev[dev];
    return out->ok == 1 ? SPEC_OK : SPEC_ERR_UNSUPPORTED;
}

// SM count used for sizing: the current device's, else 160 (an upper bound for GB300 parts).
int sizing_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
        return sms;
    cudaGetLastError();
    return 160;
}

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

constexpr int kMmaCtasPerSm = 2;

SplitPlan verify_plan(int B, int N, int Hq, int Hkv, int L_eff, int sms) {
    return make_plan(B, N, Hq, Hkv, L_eff, mma_rows_per_unit(), mma_tile_tokens(), sms * kMmaCtasPerSm);
}

// Workspace that covers either cache kernel's plan, plus (after the partials) room for
// the resolved index rows of a paged sparse call, [B, L_eff] int32.
size_t verify_bytes_any(int B, int N, int Hq, int Hkv, int d, int L_eff, int sms) {
    const size_t a = plan_workspace_bytes(verify_plan(B, N, Hq, Hkv, L_eff, sms), d);
    // the slot count does not depend on balancing, so the dense plan sizes both kinds
    const size_t b = plan_workspace_bytes(make_plan_tc(B, N, Hq, Hkv, L_eff, sms, false), d);
    return std::max(a, b) + align_up((size_t)B * L_eff * sizeof(int32_t), 256);
}

// The extended call's options: where a paged call's cache lives (all zero for a contiguous
// cache), and an fp8 cache's scales.
struct ExtArgs {
    const int32_t *table = nullptr;
    int64_t table_ld = 0;
    int block_size = 0;
    int64_t num_blocks = 0;
    bool kv_fp8 = false;
    const float *k_scale = nullptr;
    const float *v_scale = nullptr;
};

spec_status_t verify_common(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                            int64_t sb, int64_t sh, int64_t st, const uint16_t *k_draft,
                            const uint16_t *v_draft, const int32_t *parent, int B, int N, int Hq,
                            int Hkv, int d, int L, const int32_t *ctx_lens, float scale,
                            const int32_t *idx, int budget, bool sparse, float *out, float *lse,
                            void *workspace, size_t ws_bytes, void *stream, const ExtArgs &pg = ExtArgs(),
                            bool out_bf16 = false) {
    // host checks, before anything is enqueued
    if (!q || !out || !lse || !workspace) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || N > 4096 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || L < 0) return SPEC_ERR_INVALID_ARG;
    if (L > 0 && (!k_cache || !v_cache)) return SPEC_ERR_INVALID_ARG;
    if ((k_draft == nullptr) != (v_draft == nullptr)) return SPEC_ERR_INVALID_ARG;
    if (k_draft && !parent) return SPEC_ERR_INVALID_ARG;
    if (sparse && (!idx || budget < 1)) return SPEC_ERR_INVALID_ARG;
    if (sb < 0 || sh < 0 || st < 0 || sb % 8 || sh % 8 || st % 8) return SPEC_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_draft, 16) ||
        !aligned(v_draft, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(workspace, 256) ||
        !aligned(parent, 4) || !aligned(idx, 4) || !aligned(ctx_lens, 4))
        return SPEC_ERR_INVALID_ARG;
    if (!(scale == scale)) return SPEC_ERR_INVALID_ARG;
    if (d != kHeadDim) return SPEC_ERR_UNSUPPORTED;
    if ((int64_t)B * N * Hq > (int64_t)1 << 31) return SPEC_ERR_INVALID_ARG;
    if (pg.kv_fp8) {  // E4M3 codes: one byte an element, rows copied 16 bytes at a time
        if (L > 0 && (!pg.k_scale || !pg.v_scale || !aligned(pg.k_scale, 4) || !aligned(pg.v_scale, 4)))
            return SPEC_ERR_INVALID_ARG;
        if (sb % 16 || sh % 16 || st % 16) return SPEC_ERR_INVALID_ARG;
    }
    if (pg.table) {  // paged cache
        if (pg.block_size < 1 || pg.num_blocks < 0 || st < 1 || !aligned(pg.table, 4) ||
            pg.table_ld < ((int64_t)L + pg.block_size - 1) / pg.block_size)
            return SPEC_ERR_INVALID_ARG;
        // sparse: index entries become pool rows blk * (sb / st) + o, numbered in 32 bits
        if (sparse && (sb % st != 0 || pg.num_blocks * (sb / st) + pg.block_size > INT32_MAX))
            return SPEC_ERR_UNSUPPORTED;
    }
    DeviceInfo dev;
    if (spec_status_t s = current_device(&dev)) return s;

    const int L_eff = sparse ? budget : L;
    // the split plan numbers tiles in 32-bit arithmetic
    if ((int64_t)B * Hkv * (((int64_t)(Hq / Hkv) * N + 63) / 64) * ((int64_t)L_eff / 64 + 1) >= ((int64_t)1 << 31))
        return SPEC_ERR_UNSUPPORTED;
    if (ws_bytes < verify_bytes_any(B, N, Hq, Hkv, d, L_eff, dev.sms)) return SPEC_ERR_WORKSPACE;

    VerifyArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.k_cache = reinterpret_cast<const __nv_bfloat16 *>(k_cache);
    a.v_cache = reinterpret_cast<const __nv_bfloat16 *>(v_cache);
    a.sb = sb; a.sh = sh; a.st = st;
    a.k_draft = reinterpret_cast<const __nv_bfloat16 *>(k_draft);
    a.v_draft = reinterpret_cast<const __nv_bfloat16 *>(v_draft);
    a.parent = parent;
    a.ctx_lens = ctx_lens;
    a.idx = sparse ? idx : nullptr;
    a.budget = sparse ? budget : 0;
    a.B = B; a.N = N; a.Hq = Hq; a.Hkv = Hkv; a.G = Hq / Hkv; a.L = L;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.status = reinterpret_cast<uint32_t *>(ws);
    a.table = pg.table;
    a.table_ld = pg.table_ld;
    a.block_size = pg.block_size;
    a.num_blocks = pg.num_blocks;
    a.idx_resolved = 0;
    a.out_bf16 = out_bf16 ? 1 : 0;
    a.kv_fp8 = pg.kv_fp8 ? 1 : 0;
    a.k_scale = pg.k_scale;
    a.v_scale = pg.v_scale;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(32);
        cfg.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (const cudaError_t e = cudaLaunchKernelEx(&cfg, status_reset_kernel, a.status); e != cudaSuccess)
            return (spec_status_t)cuda_failure(e);
    }
    count_launches(1);
    if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    if (pg.table && sparse) {
        // the index set resolved to pool rows (checked there), at the end of the workspace;
        // the gather kernels then read the pool as one cache of row stride st
        const size_t rows_bytes = align_up((size_t)B * budget * sizeof(int32_t), 256);
        int32_t *rows = reinterpret_cast<int32_t *>(ws + (ws_bytes - rows_bytes) / 256 * 256);
        if (const cudaError_t e = launch_resolve_paged_idx(a, rows, s); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
        a.idx = rows;
        a.idx_resolved = 1;
        a.table = nullptr;
        a.sb = 0;
    }
    cudaEvent_t ev0 = g_prof_start && g_prof_stop ? g_prof_start : nullptr;
    cudaEvent_t ev1 = ev0 ? g_prof_stop : nullptr;
    // the tcgen05 kernel when the shape allows it (its TMA maps, its 16-byte row gathers);
    // the other shapes: the warp-level tensor-core kernel
    SplitPlan plan;
    bool launched = false;
    if (tc_supported(a)) {
        plan = make_plan_tc(B, N, Hq, Hkv, L_eff, dev.sms, sparse);
        a.o_part = reinterpret_cast<float *>(ws + kHeaderBytes);
        a.lse_part = reinterpret_cast<float *>(ws + kHeaderBytes + plan_o_bytes(plan, d));
        if (const cudaError_t e = launch_cache_attn_tc(a, plan, s, ev0, ev1, &launched); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    }
    if (!launched) {
        plan = verify_plan(B, N, Hq, Hkv, L_eff, dev.sms);
        a.o_part = reinterpret_cast<float *>(ws + kHeaderBytes);
        a.lse_part = reinterpret_cast<float *>(ws + kHeaderBytes + plan_o_bytes(plan, d));
        if (const cudaError_t e = launch_cache_attn_mma(a, plan, sparse, s, ev0, ev1); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    }
    if (const cudaError_t e = launch_merge_tree(a, plan, s); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    return SPEC_OK;
}

}  // namespace

void count_launches(int n) { g_launches += (uint64_t)n; }

int cuda_failure(cudaError_t e) {
    g_last_cuda_error = e;
    return SPEC_ERR_CUDA;
}

}  // namespace specverify

using namespace specverify;

extern "C" {

const char *spec_status_string(int status) {
    switch (status) {
        case SPEC_OK: return "SPEC_OK";
        case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
        case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
        case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
        case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
        case SPEC_ERR_BAD_INPUT: return "SPEC_ERR_BAD_INPUT";
        case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
        default: return "SPEC_ERR_UNKNOWN";
    }
}

size_t spec_select_workspace_size(int B, int L, int budget) {
    (void)B; (void)L; (void)budget;
    return kHeaderBytes;
}

spec_status_t spec_select_topk(const float *draft_score, const float *target_score, int64_t ld,
                               int B, int L, const int32_t *ctx_lens, int sink, int window,
                               int top_m, int budget, int32_t *idx, int32_t *count,
                               void *workspace, size_t ws_bytes, void *stream) {
    if (!draft_score || !target_score || !idx || !workspace) return SPEC_ERR_INVALID_ARG;
    if (B < 0 || L < 1 || L > 1572864 || ld < L || sink < 0 || window < 0 || top_m < 0 ||
        budget < 1 || (int64_t)sink + window > budget)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(draft_score, 4) || !aligned(target_score, 4) || !aligned(idx, 4) ||
        !aligned(count, 4) || !aligned(ctx_lens, 4) || !aligned(workspace, 256))
        return SPEC_ERR_INVALID_ARG;
    if (ws_bytes < spec_select_workspace_size(B, L, budget)) return SPEC_ERR_WORKSPACE;
    DeviceInfo dev;
    if (spec_status_t s = current_device(&dev)) return s;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *status = static_cast<uint32_t *>(workspace);
    // the kernel writes the status word itself; with no sequence there is no kernel
    if (B == 0) {
        if (const cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s); e != cudaSuccess)
            return (spec_status_t)cuda_failure(e);
        return SPEC_OK;
    }
    if (const cudaError_t e = launch_select_topk(draft_score, target_score, ld, B, L, ctx_lens, sink, window,
                                                 top_m, budget, idx, count, status, s);
        e != cudaSuccess)
        return (spec_status_t)cuda_failure(e);
    return SPEC_OK;
}

size_t spec_verify_workspace_size(int B, int N, int Hq, int Hkv, int d, int L_or_budget) {
    if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1 || L_or_budget < 0) return 0;
    return verify_bytes_any(B, N, Hq, Hkv, d, L_or_budget, sizing_sms());
}

int spec_split_plan(int B, int N, int Hq, int Hkv, int L_or_budget, int sms, int sparse, int32_t *starts,
                    int max_starts, int32_t *info) {
    if (B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || L_or_budget < 0 || sms < 1 || !starts || !info)
        return -(int)SPEC_ERR_INVALID_ARG;
    // the verify calls' bound on the plan's 32-bit tile numbering
    if ((int64_t)B * Hkv * (((int64_t)(Hq / Hkv) * N + 63) / 64) * ((int64_t)L_or_budget / 64 + 1) >=
        ((int64_t)1 << 31))
        return -(int)SPEC_ERR_UNSUPPORTED;
    const SplitPlan p = make_plan_tc(B, N, Hq, Hkv, L_or_budget, sms, sparse != 0);
    if (max_starts < p.ctas + 1) return -(int)SPEC_ERR_INVALID_ARG;
    for (int c = 0; c <= p.ctas; ++c) starts[c] = (int32_t)plan_start(p, c);
    info[0] = p.units;
    info[1] = p.tiles_per_unit;
    info[2] = p.row_groups;
    info[3] = p.BM;
    info[4] = p.split_tiles;
    info[5] = p.pipes;
    info[6] = (int32_t)p.slots;
    info[7] = p.uniform;
    return p.ctas;
}

spec_status_t spec_verify_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                               int64_t kv_stride_b, int64_t kv_stride_h, int64_t kv_stride_t,
                               const uint16_t *k_draft, const uint16_t *v_draft,
                               const int32_t *parent, int B, int N, int Hq, int Hkv, int d, int L,
                               const int32_t *ctx_lens, float scale, float *out, float *lse,
                               void *workspace, size_t ws_bytes, void *stream) {
    return verify_common(q, k_cache, v_cache, kv_stride_b, kv_stride_h, kv_stride_t, k_draft, v_draft,
                         parent, B, N, Hq, Hkv, d, L, ctx_lens, scale, nullptr, 0, false, out, lse,
                         workspace, ws_bytes, stream);
}

spec_status_t spec_verify_attn_sparse(const uint16_t *q, const uint16_t *k_cache,
                                      const uint16_t *v_cache, int64_t kv_stride_b,
                                      int64_t kv_stride_h, int64_t kv_stride_t,
                                      const uint16_t *k_draft, const uint16_t *v_draft,
                                      const int32_t *parent, int B, int N, int Hq, int Hkv, int d,
                                      int L, const int32_t *ctx_lens, float scale,
                                      const int32_t *idx, int budget, float *out, float *lse,
                                      void *workspace, size_t ws_bytes, void *stream) {
    return verify_common(q, k_cache, v_cache, kv_stride_b, kv_stride_h, kv_stride_t, k_draft, v_draft,
                         parent, B, N, Hq, Hkv, d, L, ctx_lens, scale, idx, budget, true, out, lse,
                         workspace, ws_bytes, stream);
}

spec_status_t spec_verify_attn_ex(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                  int64_t kv_stride_b, int64_t kv_stride_h, int64_t kv_stride_t,
                                  const uint16_t *k_draft, const uint16_t *v_draft, const int32_t *parent, int B,
                                  int N, int Hq, int Hkv, int d, int L, const int32_t *ctx_lens, float scale,
                                  const int32_t *idx, int budget, const spec_verify_ext *ext, void *out, float *lse,
                                  void *workspace, size_t ws_bytes, void *stream) {
    ExtArgs pg;
    bool bf16 = false;
    if (ext) {
        if (ext->out_dtype != SPEC_OUT_F32 && ext->out_dtype != SPEC_OUT_BF16) return SPEC_ERR_INVALID_ARG;
        if (ext->kv_dtype != SPEC_KV_BF16 && ext->kv_dtype != SPEC_KV_E4M3) return SPEC_ERR_INVALID_ARG;
        bf16 = ext->out_dtype == SPEC_OUT_BF16;
        pg.table = ext->block_table;
        pg.table_ld = ext->table_ld;
        pg.block_size = ext->block_size;
        pg.num_blocks = ext->num_blocks;
        pg.kv_fp8 = ext->kv_dtype == SPEC_KV_E4M3;
        pg.k_scale = ext->k_scale;
        pg.v_scale = ext->v_scale;
    }
    return verify_common(q, k_cache, v_cache, kv_stride_b, kv_stride_h, kv_stride_t, k_draft, v_draft, parent, B, N,
                         Hq, Hkv, d, L, ctx_lens, scale, idx, budget, idx != nullptr, static_cast<float *>(out), lse,
                         workspace, ws_bytes, stream, pg, bf16);
}

spec_status_t spec_lse_merge(const float *o_a, const float *lse_a, const float *o_b,
                             const float *lse_b, float *out, float *lse_out, int64_t rows, int d,
                             void *stream) {
    if (!o_a || !lse_a || !o_b || !lse_b || !out || !lse_out || rows < 0 || d < 1)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(o_a, 4) || !aligned(o_b, 4) || !aligned(out, 4) || !aligned(lse_a, 4) ||
        !aligned(lse_b, 4) || !aligned(lse_out, 4))
        return SPEC_ERR_INVALID_ARG;
    if (rows > (int64_t)INT32_MAX * 8) return SPEC_ERR_INVALID_ARG;  // one warp per row, 8 per block
    DeviceInfo dev;
    if (spec_status_t s = current_device(&dev)) return s;
    if (const cudaError_t e = launch_lse_merge2(o_a, lse_a, o_b, lse_b, out, lse_out, rows, d,
                                               static_cast<cudaStream_t>(stream));
        e != cudaSuccess)
        return (spec_status_t)cuda_failure(e);
    return SPEC_OK;
}

spec_status_t spec_read_device_status(const void *workspace, void *stream) {
    if (!workspace) return SPEC_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (const cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s); e != cudaSuccess)
        return (spec_status_t)cuda_failure(e);
    if (const cudaError_t e = cudaStreamSynchronize(s); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    return static_cast<spec_status_t>(v);
}

const char *spec_last_cuda_error(void) {
    return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

void spec_profile_events(void *start_event, void *stop_event) {
    g_prof_start = static_cast<cudaEvent_t>(start_event);
    g_prof_stop = static_cast<cudaEvent_t>(stop_event);
}

uint64_t spec_kernel_launches(void) { return g_launches; }

}  // extern "C"
