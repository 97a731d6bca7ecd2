// spec_importance_scores: target-historical importance of every cache token,
// the input the next step's selection reads as its target score.
//
// The pages fuse the target's historical attention with the drafter's and
// score only on a few semantic retrieval heads (Dustin "Metodologia", sections
// 1-2), without saying how heads and queries combine. Taken here: the score of
// cache token t of sequence b is the sum, over the listed query heads h and the
// N draft queries i, of the final attention probability of row (b, i, h) on t,
// exp(scale q[b,i,h] . k[b, h / G, t] - lse[b,i,h]), with lse as the verify call
// returns it. Rows with lse = -inf (nothing attended) add nothing.
//
// A second pass over the K rows of the listed heads, after the verify call. The
// tensor-core form (importance_tc.cu) takes the call when the listed heads'
// queries fit its staging (heads x queries padded to 16 <= 256 rows); this file
// keeps the portable form for the other shapes: one thread per token, the token's
// K row in registers, each head's queries and lse staged in shared memory and
// read as broadcasts, fp32 dot products on the FMA pipe.
#include "common.cuh"

namespace specverify {

namespace {

constexpr int kImpThreads = 256;
constexpr int kImpMaxN = 512;  // queries staged per head: N x 256 B + N x 4 B of shared memory

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
    const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *y = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 fx = __bfloat1622float2(x[j]), fy = __bfloat1622float2(y[j]);
        acc = fmaf(fx.x, fy.x, acc);
        acc = fmaf(fx.y, fy.y, acc);
    }
    return acc;
}

__global__ void __launch_bounds__(kImpThreads)
importance_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k_cache, int64_t sb,
                  int64_t sh, int64_t st, const float *__restrict__ lse, const int32_t *__restrict__ heads, int nh,
                  int N, int Hq, int Hkv, int L, const int32_t *__restrict__ ctx_lens, float scale,
                  float *__restrict__ score, int64_t ld, int32_t *status) {
    extern __shared__ __align__(16) uint8_t s_raw[];
    uint4 *s_q = reinterpret_cast<uint4 *>(s_raw);                          // [N][16] chunks of 8 bf16
    float *s_lse = reinterpret_cast<float *>(s_raw + (size_t)N * 256);     // [N]
    const int b = blockIdx.y;
    const int t = blockIdx.x * kImpThreads + threadIdx.x;
    int n_ctx = L;
    if (ctx_lens) {
        const int c = ctx_lens[b];
        n_ctx = c < 0 ? 0 : (c > L ? L : c);
    }
    const int G = Hq / Hkv;
    float acc = 0.f;
    for (int hi = 0; hi < nh; ++hi) {
        const int h = heads[hi];
        if (h < 0 || h >= Hq) {  // a head index out of range adds nothing; it is reported
            if (threadIdx.x == 0 && blockIdx.x == 0 && status) atomicMax(status, (int32_t)SPEC_ERR_BAD_INPUT);
            continue;
        }
        __syncthreads();  // the previous head's queries are no longer read
        for (int x = threadIdx.x; x < N * 16; x += kImpThreads) {
            const int i = x >> 4, ch = x & 15;
            s_q[x] = *reinterpret_cast<const uint4 *>(q + (((int64_t)b * N + i) * Hq + h) * kHeadDim + ch * 8);
        }
        for (int i = threadIdx.x; i < N; i += kImpThreads) s_lse[i] = lse[((int64_t)b * N + i) * Hq + h];
        __syncthreads();
        if (t < n_ctx) {
            const __nv_bfloat16 *kr = k_cache + (int64_t)b * sb + (int64_t)(h / G) * sh + (int64_t)t * st;
            uint4 kv[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) kv[c] = *reinterpret_cast<const uint4 *>(kr + c * 8);
            for (int i = 0; i < N; ++i) {
                const float l = s_lse[i];
                if (!(l > -INFINITY)) continue;  // the row attends nothing (or lse is NaN)
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < 16; ++c) dot = dot8(s_q[i * 16 + c], kv[c], dot);
                acc += expf(scale * dot - l);
            }
        }
    }
    if (t < L) score[(int64_t)b * ld + t] = t < n_ctx ? acc : 0.f;
}

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

}  // namespace specverify

using namespace specverify;

extern "C" spec_status_t spec_importance_scores(const uint16_t *q, const uint16_t *k_cache, int64_t kv_stride_b,
                                                int64_t kv_stride_h, int64_t kv_stride_t, const float *lse,
                                                const int32_t *heads, int nh, int B, int N, int Hq, int Hkv, int d,
                                                int L, const int32_t *ctx_lens, float scale, float *score,
                                                int64_t ld, int32_t *status, void *stream) {
    if (!q || !lse || !score || (nh > 0 && !heads)) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || B > 65535 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || L < 0 || nh < 0 || ld < L)
        return SPEC_ERR_INVALID_ARG;
    if (L > 0 && !k_cache) return SPEC_ERR_INVALID_ARG;
    if (kv_stride_b < 0 || kv_stride_h < 0 || kv_stride_t < 0 || kv_stride_b % 8 || kv_stride_h % 8 ||
        kv_stride_t % 8)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(lse, 4) || !aligned(heads, 4) || !aligned(score, 4) ||
        !aligned(ctx_lens, 4) || !aligned(status, 4))
        return SPEC_ERR_INVALID_ARG;
    if (!(scale == scale)) return SPEC_ERR_INVALID_ARG;
    if (d != kHeadDim || N > kImpMaxN) return SPEC_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L > 0 && nh > 0) {  // the tensor-core form where the shape allows it (it writes the status word)
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return (spec_status_t)cuda_failure(cudaGetLastError());
        cudaError_t e;
        if (launch_importance_tc(reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k_cache),
                                 kv_stride_b, kv_stride_h, kv_stride_t, lse, heads, nh, B, N, Hq, Hkv, L, ctx_lens, scale,
                                 score, ld, status, sms, s, &e))
            return e == cudaSuccess ? SPEC_OK : (spec_status_t)cuda_failure(e);
    }
    if (status) {
        if (const cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), s); e != cudaSuccess)
            return (spec_status_t)cuda_failure(e);
    }
    if (L == 0) return SPEC_OK;
    const size_t smem = (size_t)N * 256 + (size_t)N * sizeof(float);
    static PerDeviceOnce attr_once;
    const cudaError_t attr = once_per_device(
        attr_once, [] { return kernel_attributes(importance_kernel, (int)(kImpMaxN * 256 + kImpMaxN * 4)); });
    if (attr != cudaSuccess) return (spec_status_t)cuda_failure(attr);
    const dim3 grid((unsigned)((L + kImpThreads - 1) / kImpThreads), (unsigned)B);
    importance_kernel<<<grid, kImpThreads, smem, s>>>(
        reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k_cache), kv_stride_b,
        kv_stride_h, kv_stride_t, lse, heads, nh, N, Hq, Hkv, L, ctx_lens, scale, score, ld, status);
    count_launches(1);
    if (const cudaError_t e = cudaGetLastError(); e != cudaSuccess) return (spec_status_t)cuda_failure(e);
    return SPEC_OK;
}
