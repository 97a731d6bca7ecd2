// spec_accept_commit: greedy acceptance of the draft tree and commit of the
// accepted draft K/V rows into the cache.
//
// The target verifies the draft tokens, and the accepted ones join the cache
// while the rejected ones are dropped (Dustin "Workflow di Verifica", steps
// 4-5), under greedy decoding (BASTION "Risultati Sperimentali"). The rule taken
// for "accepted": from the root, the next accepted node is the lowest-index child
// whose draft token equals the target's greedy token after the current node; the
// walk stops when no child matches, and the target's token after the last
// accepted node is the bonus token. The accepted nodes' draft K/V rows are copied
// in path order to cache positions ctx, ctx + 1, ... and ctx advances.
//
// One CTA per sequence: the CTA stages the sequence's parents, tokens and target
// tokens in shared memory with coalesced loads, warp 0 walks the tree there (a
// ballot over each 32-node window finds the lowest matching child), then the CTA
// copies the rows 16 bytes at a time. The work is a few kilobytes per sequence:
// a single launch, bound by its latency, with one round trip to memory before
// the walk instead of several per accepted node.
#include "common.cuh"

namespace specverify {

namespace {

constexpr int kAcceptThreads = 256;
constexpr int kAcceptMaxN = 4096;

__global__ void __launch_bounds__(kAcceptThreads)
accept_commit_kernel(const int32_t *__restrict__ draft_token, const int32_t *__restrict__ parent,
                     const int32_t *__restrict__ target_next, int N, int32_t *__restrict__ path,
                     int32_t *__restrict__ accept_len, int32_t *__restrict__ bonus, __nv_bfloat16 *__restrict__ k_cache,
                     __nv_bfloat16 *__restrict__ v_cache, int64_t sb, int64_t sh, int64_t st,
                     const __nv_bfloat16 *__restrict__ k_draft, const __nv_bfloat16 *__restrict__ v_draft, int Hkv,
                     int L, int32_t *ctx_lens, int32_t *status) {
    extern __shared__ int32_t s_buf[];  // parents [N], tokens [N], target tokens [N + 1], path [N]
    __shared__ int s_len;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    int32_t *par = s_buf, *tok = s_buf + N, *tn = s_buf + 2 * N, *s_path = s_buf + 3 * N + 1;
    for (int i = tid; i < N; i += kAcceptThreads) {
        par[i] = parent[(int64_t)b * N + i];
        tok[i] = draft_token[(int64_t)b * N + i];
    }
    for (int i = tid; i <= N; i += kAcceptThreads) tn[i] = target_next[(int64_t)b * (N + 1) + i];
    __syncthreads();
    if (tid < 32) {
        // a parent outside [-1, i) never makes node i a child (the walk only looks
        // past the current node); it is reported
        bool bad = false;
        for (int i = lane; i < N; i += 32) {
            const int p = par[i];
            bad |= p < -1 || p >= i;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0 && status) atomicMax(status, (int32_t)SPEC_ERR_BAD_INPUT);
        int cur = -1, n = 0;
        while (true) {
            const int want = tn[cur + 1];
            int nxt = -1;
            for (int base = cur + 1; base < N; base += 32) {
                const int c = base + lane;
                const bool m = c < N && par[c] == cur && tok[c] == want;
                const unsigned bal = __ballot_sync(0xffffffffu, m);
                if (bal) {
                    nxt = base + __ffs((int)bal) - 1;
                    break;
                }
            }
            if (nxt < 0) break;
            if (lane == 0) s_path[n] = nxt;
            ++n;
            cur = nxt;
        }
        __syncwarp();
        int32_t *pb = path + (int64_t)b * N;
        for (int j = lane; j < N; j += 32) pb[j] = j < n ? s_path[j] : -1;
        if (lane == 0) {
            accept_len[b] = n;
            bonus[b] = tn[cur + 1];
            s_len = n;
        }
    }
    __syncthreads();
    if (k_cache == nullptr) return;
    const int n = s_len;
    const int c0 = ctx_lens[b];
    const bool ctx_ok = c0 >= 0 && c0 <= L;
    const int fit = ctx_ok ? min(n, L - c0) : 0;
    if (tid == 0 && status && (!ctx_ok || fit < n)) atomicMax(status, (int32_t)SPEC_ERR_BAD_INPUT);
    // chunk x: row j of the path, KV head h, K or V, 16-byte chunk ch of the 256-byte
    // row; each thread loads kCopyBatch chunks before storing them, so the copy takes a
    // round trip to memory per batch rather than per chunk
    constexpr int kCopyBatch = 8;
    const int chunks = fit * Hkv * 2 * 16;
    auto locate = [&](int x, __nv_bfloat16 *&dst, const __nv_bfloat16 *&src) {
        const int ch = x & 15;
        const int r = x >> 4;
        const int kv = r & 1;
        const int h = (r >> 1) % Hkv;
        const int j = (r >> 1) / Hkv;
        const int node = s_path[j];
        dst = (kv ? v_cache : k_cache) + (int64_t)b * sb + (int64_t)h * sh + (int64_t)(c0 + j) * st + ch * 8;
        src = (kv ? v_draft : k_draft) + (((int64_t)b * N + node) * Hkv + h) * kHeadDim + ch * 8;
    };
    for (int x0 = tid; x0 < chunks; x0 += kAcceptThreads * kCopyBatch) {
        uint4 v[kCopyBatch];
        __nv_bfloat16 *dst[kCopyBatch];
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u) {
            const int x = x0 + u * kAcceptThreads;
            const __nv_bfloat16 *src = nullptr;
            dst[u] = nullptr;
            if (x < chunks) {
                locate(x, dst[u], src);
                v[u] = *reinterpret_cast<const uint4 *>(src);
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyBatch; ++u)
            if (dst[u]) *reinterpret_cast<uint4 *>(dst[u]) = v[u];
    }
    __syncthreads();  // every thread has read ctx_lens[b]
    if (tid == 0 && ctx_ok) ctx_lens[b] = c0 + fit;
}

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

}  // namespace specverify

using namespace specverify;

extern "C" spec_status_t spec_accept_commit(const int32_t *draft_token, const int32_t *parent,
                                            const int32_t *target_next, int B, int N, int32_t *accept_path,
                                            int32_t *accept_len, int32_t *bonus_token, uint16_t *k_cache,
                                            uint16_t *v_cache, int64_t kv_stride_b, int64_t kv_stride_h,
                                            int64_t kv_stride_t, const uint16_t *k_draft, const uint16_t *v_draft,
                                            int Hkv, int d, int L, int32_t *ctx_lens, int32_t *status, void *stream) {
    if (!draft_token || !parent || !target_next || !accept_path || !accept_len || !bonus_token)
        return SPEC_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || N > kAcceptMaxN) return SPEC_ERR_INVALID_ARG;
    if (!aligned(draft_token, 4) || !aligned(parent, 4) || !aligned(target_next, 4) || !aligned(accept_path, 4) ||
        !aligned(accept_len, 4) || !aligned(bonus_token, 4) || !aligned(status, 4))
        return SPEC_ERR_INVALID_ARG;
    const bool commit = k_cache || v_cache || k_draft || v_draft || ctx_lens;
    if (commit) {
        if (!k_cache || !v_cache || !k_draft || !v_draft || !ctx_lens) return SPEC_ERR_INVALID_ARG;
        if (Hkv < 1 || L < 0) return SPEC_ERR_INVALID_ARG;
        if (kv_stride_b < 0 || kv_stride_h < 0 || kv_stride_t < 0 || kv_stride_b % 8 || kv_stride_h % 8 ||
            kv_stride_t % 8)
            return SPEC_ERR_INVALID_ARG;
        if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_draft, 16) || !aligned(v_draft, 16) ||
            !aligned(ctx_lens, 4))
            return SPEC_ERR_INVALID_ARG;
        if (d != kHeadDim) return SPEC_ERR_UNSUPPORTED;
    }
    const size_t smem = (size_t)(4 * N + 1) * sizeof(int32_t);
    static PerDeviceOnce attr_once;
    const cudaError_t attr = once_per_device(attr_once, [] {
        return kernel_attributes(accept_commit_kernel, (int)((4 * kAcceptMaxN + 1) * sizeof(int32_t)));
    });
    if (attr != cudaSuccess) return (spec_status_t)cuda_failure(attr);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (status) {
        if (const cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), s); e != cudaSuccess)
            return (spec_status_t)cuda_failure(e);
    }
    accept_commit_kernel<<<(unsigned)B, kAcceptThreads, smem, s>>>(
        draft_token, parent, target_next, N, accept_path, accept_len, bonus_token,
        reinterpret_cast<__nv_bfloat16 *>(commit ? k_cache : nullptr), reinterpret_cast<__nv_bfloat16 *>(v_cache),
        kv_stride_b, kv_stride_h, kv_stride_t, reinterpret_cast<const __nv_bfloat16 *>(k_draft),
        reinterpret_cast<const __nv_bfloat16 *>(v_draft), Hkv, L, ctx_lens, status);
    count_launches(1);
    if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    return SPEC_OK;
}
