// Target-historical importance scores on the 5th-generation tensor core.
//
// score[b, t] = sum over the listed query heads h and the N draft queries i of
// exp(scale q[b,i,h] . k[b, h / G, t] - lse[b,i,h]) (Dustin "Metodologia",
// sections 1-2: the target's attention on a few semantic retrieval heads; the
// heads and queries are summed). For each 128-token tile of the cache and each
// listed head, one MMA computes S^T = K_tile Q_h^T (M = 128 tokens, N = the
// head's draft queries, K = d) into TMEM, so each accumulator lane is one token:
// the thread that owns the lane sums its row's probabilities with no exchange.
//
// One CTA per (range of tiles, sequence): warp 0 streams the K tiles of the
// listed heads' KV heads through a ring of up to 6 slots by TMA (128-byte swizzle,
// the layout the tensor core reads; as many slots as the shared memory left by the
// queries holds), warp 1 issues the MMAs (tile-major, head-minor) into two TMEM
// accumulators, and warps 2-9 turn each accumulator into probabilities and add them
// to their token's score: two warps per TMEM lane quarter, each over half of the
// queries, whose sums meet in shared memory at the tile's end. The
// queries of every listed head and their lse (in base 2) are staged once per
// CTA; thread 0 issues the queries' and the first ring's K loads as soon as the
// barriers exist, so the rest of the set-up overlaps them. Every wait is bounded;
// one that gives up records SPEC_ERR_TIMEOUT and the CTA drains and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace specverify {

namespace {

using namespace sm100;

constexpr int IT_T = 128;                // tokens per tile
constexpr int IT_RING_MAX = 6;           // K tile slots at most (the launch sizes the ring)
constexpr int IT_SLOT = IT_T * kHeadDim * 2;  // 32 KiB
constexpr int IT_MAX_ROWS = 256;         // listed heads x padded queries staged
constexpr int IT_EPI_WARPS = 8;          // two per TMEM lane quarter, one per half of the queries
constexpr int IT_THREADS = 64 + 32 * IT_EPI_WARPS;
constexpr int IT_WARP_PRODUCER = 0, IT_WARP_MMA = 1, IT_WARP_EPI0 = 2;
constexpr long long IT_WAIT_LIMIT = 4000000000LL;  // ~2 s
constexpr int IT_SMEM_MAX = 232448;

struct ItBars {
    uint64_t q_full;
    uint64_t kv_full[IT_RING_MAX], kv_empty[IT_RING_MAX];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(ItBars) <= 256, "barrier block");

// smem (from a 1024-byte aligned base): [Q rows: nh*npad x 256 B, two 64-column halves,
// rounded up to 1 KiB] [ring: `ring` slots of 32 KiB] [lse2: IT_MAX_ROWS floats]
// [pair sums: 2 x IT_T floats] [bars]. The launch takes as many slots as fit.
constexpr int IT_TAIL_BYTES = IT_MAX_ROWS * 4 + 2 * IT_T * 4 + 256;

struct ItParams {
    int nh, npad;       // listed heads, queries per head padded to a multiple of 16
    int tiles_per_cta;  // cache tiles per CTA
    int ring;           // K tile slots (<= IT_RING_MAX)
    uint32_t q_bytes;   // the Q area (1 KiB multiple)
    uint32_t col_stride;  // TMEM columns per accumulator: npad rounded up to 32 (whole 32-column reads)
    uint32_t tmem_cols;
};

__host__ __device__ constexpr int it_smem_bytes(uint32_t q_bytes, int ring) {
    return (int)q_bytes + ring * IT_SLOT + IT_TAIL_BYTES + 1024;  // + alignment slack
}

__device__ __forceinline__ bool it_wait(ItBars &bs, uint64_t *bar, uint32_t parity, int32_t *status) {
    if (*(volatile uint32_t *)&bs.abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
        if (*(volatile uint32_t *)&bs.abort) return false;
        if (clock64() - t0 > IT_WAIT_LIMIT) {
            atomicExch(&bs.abort, 1u);
            if (status) atomicMax(status, (int32_t)SPEC_ERR_TIMEOUT);
            return false;
        }
    }
}
__device__ __forceinline__ void it_drain(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity) && clock64() - t0 < IT_WAIT_LIMIT) {
    }
}

// Every listed head's queries: rows b*N .. b*N + npad of head h, two column halves (one thread).
__device__ __forceinline__ void it_load_q(ItBars &bs, uint8_t *sQ, const CUtensorMap *tm_q, const int32_t *heads,
                                          const ItParams &ip, int Hq, int row0) {
    mbar_arrive_expect_tx(&bs.q_full, (uint32_t)(ip.nh * ip.npad * kHeadDim * 2));
    for (int j = 0; j < ip.nh; ++j) {
        const int h = min(max(__ldg(heads + j), 0), Hq - 1);  // a bad head's rows are never used
        for (int kh = 0; kh < 2; ++kh)
            tma_load_3d(sQ + kh * (ip.nh * ip.npad * 128) + j * ip.npad * 128, tm_q, &bs.q_full, kh * 64, h, row0);
    }
}

// Item n (tile tile0 + n / nh, listed head n % nh): the tile's 128 K rows of the head's KV
// head into ring slot n % ring, whose previous use the caller has seen consumed (one thread).
__device__ __forceinline__ void it_load_k(ItBars &bs, uint8_t *sRing, const CUtensorMap *tm_k, const int32_t *heads,
                                          const ItParams &ip, int G, int Hq, int b, int tile0, int n) {
    const int t = tile0 + n / ip.nh, j = n % ip.nh;
    const int hk = min(max(__ldg(heads + j), 0), Hq - 1) / G;
    const int slot = n % ip.ring;
    uint8_t *dst = sRing + slot * IT_SLOT;
    mbar_arrive_expect_tx(&bs.kv_full[slot], IT_SLOT);
    tma_load_4d(dst, tm_k, &bs.kv_full[slot], 0, t * IT_T, hk, b);
    tma_load_4d(dst + IT_SLOT / 2, tm_k, &bs.kv_full[slot], 64, t * IT_T, hk, b);
}

__global__ void __launch_bounds__(IT_THREADS, 1)
importance_tc_kernel(const float *__restrict__ lse, const int32_t *__restrict__ heads, int N, int Hq, int Hkv,
                     int L, const int32_t *__restrict__ ctx_lens, float scale, float *__restrict__ score, int64_t ld,
                     int32_t *status, const ItParams ip, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k) {
    extern __shared__ uint8_t it_raw[];
    uint8_t *smem = it_raw + ((1024 - (smem_u32(it_raw) & 1023)) & 1023);
    const int ring = ip.ring;
    uint8_t *sQ = smem;
    uint8_t *sRing = smem + ip.q_bytes;
    float *sLse2 = reinterpret_cast<float *>(sRing + ring * IT_SLOT);
    float *sPair = sLse2 + IT_MAX_ROWS;  // [tile parity][token of the tile]
    ItBars &bs = *reinterpret_cast<ItBars *>(sPair + 2 * IT_T);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int G = Hq / Hkv;
    const int tile0 = blockIdx.x * ip.tiles_per_cta;
    const int ntiles_all = (L + IT_T - 1) / IT_T;
    const int ntiles = min(ip.tiles_per_cta, ntiles_all - tile0);
    const int nitems = ntiles * ip.nh;
    int n_ctx = L;
    if (ctx_lens) {
        const int c = ctx_lens[b];
        n_ctx = c < 0 ? 0 : (c > L ? L : c);
    }

    if (threadIdx.x == 0) {
        mbar_init(&bs.q_full, 1);
        for (int i = 0; i < ring; ++i) {
            mbar_init(&bs.kv_full[i], 1);
            mbar_init(&bs.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bs.acc_full[i], 1);
            mbar_init(&bs.acc_empty[i], IT_EPI_WARPS);
        }
        mbar_init(&bs.mma_done, 1);
        bs.abort = 0;
        fence_mbar_init();
        // the queries and the ring's first K tiles go out before the rest of the set-up
        // (the lse staging's loads, the TMEM allocation), which then overlaps them
        if (nitems > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            it_load_q(bs, sQ, &tm_q, heads, ip, Hq, b * N);
            for (int n = 0; n < nitems && n < ring; ++n) it_load_k(bs, sRing, &tm_k, heads, ip, G, Hq, b, tile0, n);
        }
    }
    // lse of every listed head's queries, in base 2; rows past N, or whose lse is -inf or
    // NaN (nothing attended), get +inf so that they add exp2(-inf) = 0
    for (int r = threadIdx.x; r < ip.nh * ip.npad; r += IT_THREADS) {
        const int j = r / ip.npad, i = r % ip.npad;
        const int h = __ldg(heads + j);
        float v = INFINITY;
        if (i < N && h >= 0 && h < Hq) {
            const float l = __ldg(lse + ((int64_t)b * N + i) * Hq + h);
            if (l > -INFINITY) v = l * 1.4426950408889634f;
        }
        sLse2[r] = v;
    }
    // the status word, written whole by the first CTA (no clearing memset before the launch):
    // SPEC_ERR_BAD_INPUT if a listed head is outside [0, Hq) (its rows add nothing), else
    // SPEC_OK; a wait that gives up later raises it to SPEC_ERR_TIMEOUT
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 32) {
        bool bad = false;
        for (int j = threadIdx.x; j < ip.nh; j += 32) {
            const int h = __ldg(heads + j);
            bad |= h < 0 || h >= Hq;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (threadIdx.x == 0 && status) *status = bad ? (int32_t)SPEC_ERR_BAD_INPUT : (int32_t)SPEC_OK;
    }
    if (warp == IT_WARP_PRODUCER) {
        tmem_alloc(&bs.tmem_base, ip.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bs.tmem_base;

    if (warp == IT_WARP_PRODUCER) {
        if (lane == 0 && nitems > 0) {
            // the queries and items 0 .. ring-1 were issued at the start
            bool ok = true;
            for (int n = ring; ok && n < nitems; ++n) {
                if (!(ok = it_wait(bs, &bs.kv_empty[n % ring], ((n / ring) - 1) & 1, status))) break;
                it_load_k(bs, sRing, &tm_k, heads, ip, G, Hq, b, tile0, n);
            }
            // drain the copies still in flight
            for (int n = nitems > ring ? nitems - ring : 0; n < nitems; ++n)
                it_drain(&bs.kv_full[n % ring], (n / ring) & 1);
            it_drain(&bs.q_full, 0);
        }
        __syncwarp();
    } else if (warp == IT_WARP_MMA) {
        bool ok = nitems > 0 && __all_sync(0xffffffffu, it_wait(bs, &bs.q_full, 0, status));
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, ip.npad, false);
        const uint64_t dk0 = desc_sw128(smem_u32(sRing), 16, 1024);
        const uint32_t qhalf = (uint32_t)(ip.nh * ip.npad * 128);  // bytes to the second column half
        for (int n = 0; ok && n < nitems; ++n) {
            const int j = n % ip.nh, slot = n % ring, buf = n & 1;
            if (!(ok = __all_sync(0xffffffffu, it_wait(bs, &bs.kv_full[slot], (n / ring) & 1, status)))) break;
            if (n >= 2 && !(ok = __all_sync(0xffffffffu, it_wait(bs, &bs.acc_empty[buf], ((n >> 1) - 1) & 1, status))))
                break;
            tc_fence_after();
            const uint64_t dk = dk0 + (uint64_t)slot * (IT_SLOT >> 4);
            const uint64_t dq = desc_sw128(smem_u32(sQ) + (uint32_t)(j * ip.npad * 128), 16, 1024);
            const uint32_t d_tmem = tmem + (uint32_t)buf * ip.col_stride;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_ss_elect(d_tmem, dk + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2),
                             dq + (uint64_t)((ks >> 2) * (qhalf >> 4) + (ks & 3) * 2), idesc, ks > 0 ? 1u : 0u);
            mma_commit_elect(&bs.kv_empty[slot]);
            mma_commit_elect(&bs.acc_full[buf]);
        }
        mma_commit_elect(&bs.mma_done);
        it_drain(&bs.mma_done, 0);
    } else {
        // epilogue: a warp may only read the TMEM lane quarter of its index mod 4, so warp w
        // takes lanes 32 (w & 3) .. + 31 = those tokens of the tile; warps 2-5 take the query
        // columns [0, 32) + 64 k, warps 6-9 [32, 64) + 64 k, and at the tile's end the second
        // half hands its sums to the first through shared memory
        const int lg = warp & 3, half = (warp - IT_WARP_EPI0) >> 2;
        const uint32_t lane_addr = (uint32_t)(lg * 32) << 16;
        const float sl2 = scale * 1.4426950408889634f;
        bool ok = true;
        float acc = 0.f;
        for (int n = 0; n < nitems; ++n) {
            const int j = n % ip.nh, buf = n & 1;
            ok = __all_sync(0xffffffffu, ok && it_wait(bs, &bs.acc_full[buf], (n >> 1) & 1, status));
            tc_fence_after();
            if (ok) {
                const float *l2 = sLse2 + j * ip.npad;
                for (int c0 = 32 * half; c0 < N; c0 += 64) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_addr + (uint32_t)buf * ip.col_stride + (uint32_t)c0, r);
                    tmem_wait_ld();
                    const int cn = min(32, N - c0);
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (c < cn) acc += ex2(__uint_as_float(r[c]) * sl2 - l2[c0 + c]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bs.acc_empty[buf]);
            if (j == ip.nh - 1) {  // the tile's last head: its tokens' scores are complete
                const int tl = n / ip.nh;
                float *pair = sPair + (tl & 1) * IT_T + lg * 32 + lane;
                if (half) *pair = acc;
                // the 8 epilogue warps; a buffer is rewritten two tiles later, after the next
                // barrier, which its reader has passed only once it has read it
                asm volatile("bar.sync 1, %0;" ::"n"(32 * IT_EPI_WARPS) : "memory");
                if (!half) {
                    const int t = (tile0 + tl) * IT_T + lg * 32 + lane;
                    if (t < L) score[(int64_t)b * ld + t] = (ok && t < n_ctx) ? acc + *pair : 0.f;
                }
                acc = 0.f;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == IT_WARP_PRODUCER) tmem_dealloc(tmem, ip.tmem_cols);
}

bool it_encode(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
               const cuuint32_t *box) {
    static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        const bool found = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                            &q) == cudaSuccess &&
                           q == cudaDriverEntryPointSuccess;
        cudaGetLastError();
        return found ? reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn) : nullptr;
    }();
    if (!encode) return false;
    cuuint32_t elem[4] = {1, 1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box,
                  elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The tensor-core form when the shape allows it (listed heads x queries padded to 16 fit
// 256 staged rows, 16-byte aligned strides); returns false (nothing launched) otherwise.
bool launch_importance_tc(const __nv_bfloat16 *q, const __nv_bfloat16 *k_cache, int64_t sb, int64_t sh, int64_t st,
                          const float *lse, const int32_t *heads, int nh, int B, int N, int Hq, int Hkv, int L,
                          const int32_t *ctx_lens, float scale, float *score, int64_t ld, int32_t *status,
                          int sms, cudaStream_t s, cudaError_t *err) {
    *err = cudaSuccess;
    const int npad = (N + 15) / 16 * 16;
    if (nh < 1 || L < 1 || npad > 256 || nh * npad > IT_MAX_ROWS || sb % 8 || sh % 8 || st % 8 ||
        (int64_t)B * N > INT32_MAX)
        return false;
    CUtensorMap mq, mk;
    {  // q [B*N, Hq, d]: box = 64 columns x 1 head x npad queries
        const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)Hq, (cuuint64_t)B * N};
        const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)Hq * kHeadDim * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)npad};
        if (!it_encode(&mq, q, 3, dims, strides, box)) return false;
    }
    {  // the cache [B, Hkv, L, d] with the caller's strides: box = 64 columns x 128 tokens
        const cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)L, (cuuint64_t)Hkv, (cuuint64_t)B};
        const cuuint64_t strides[3] = {(cuuint64_t)st * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)IT_T, 1, 1};
        if (!it_encode(&mk, k_cache, 4, dims, strides, box)) return false;
    }
    static PerDeviceOnce attr_once;
    *err = once_per_device(attr_once, [] { return kernel_attributes(importance_tc_kernel, IT_SMEM_MAX); });
    if (*err != cudaSuccess) return true;
    ItParams ip;
    ip.nh = nh;
    ip.npad = npad;
    ip.q_bytes = (uint32_t)((nh * npad * kHeadDim * 2 + 1023) / 1024 * 1024);
    ip.ring = std::min(IT_RING_MAX, (int)((IT_SMEM_MAX - it_smem_bytes(ip.q_bytes, 0)) / IT_SLOT));
    const int ntiles = (L + IT_T - 1) / IT_T;
    // about one CTA per SM over the whole batch
    const int ctas_per_seq = std::max(1, std::min(ntiles, (sms + B - 1) / B));
    ip.tiles_per_cta = (ntiles + ctas_per_seq - 1) / ctas_per_seq;
    ip.col_stride = (uint32_t)(npad + 31) / 32 * 32;
    ip.tmem_cols = 32;
    while (ip.tmem_cols < 2 * ip.col_stride) ip.tmem_cols <<= 1;
    const dim3 grid((unsigned)((ntiles + ip.tiles_per_cta - 1) / ip.tiles_per_cta), (unsigned)B);
    importance_tc_kernel<<<grid, IT_THREADS, it_smem_bytes(ip.q_bytes, ip.ring), s>>>(lse, heads, N, Hq, Hkv, L, ctx_lens, scale, score, ld,
                                                          status, ip, mq, mk);
    count_launches(1);
    *err = cudaGetLastError();
    return true;
}

}  // namespace specverify
