// Cache part of verification attention, warp-level tensor-core (mma.sync) path.
//
// Computes, for every unit (b, h_kv, group of 64 query rows) and every range
// of KV tiles given by the split plan, the normalised partial attention of the
// unit's rows (query heads of h_kv x draft nodes, packed together) over the
// cache tokens of that range, with no mask other than "token exists":
//   dense  - cache tokens 0 .. n-1 (full-cache verification, Dustin
//            "Definizione del Problema"; the unmasked cache part of LongSpec
//            section 2.C);
//   sparse - the cache rows listed in idx[b] (Dustin "Workflow di Verifica",
//            steps 3-4: the compressed cache is the selected rows of the full
//            cache, gathered on the fly; nothing is copied or evicted).
// Partials go to slot (cta + unit) of the workspace and are merged by
// log-sum-exp with the tree part afterwards.
//
// Layout: 4 warps, each owning 16 query rows; 64-token K/V tiles double
// buffered in shared memory by cp.async (16-byte, XOR-swizzled rows); S = QK^T
// and O += PV with mma.m16n8k16 bf16 -> fp32; online softmax in base 2.
//
// fp8 cache (FP8): the rows are E4M3 codes, 128 bytes each, double buffered by
// cp.async in a staging area; before a tile is used, the CTA converts its codes
// into the bf16 tile layout above (every E4M3 number is exact in bf16), and the
// per-(sequence, KV head) scales enter as a factor of the softmax scale (K) and
// of the partial's normalisation (V), so the MMAs stay bf16.
#include "common.cuh"

namespace specverify {

namespace {

constexpr int BM = 64;       // query rows per CTA
constexpr int BN = 64;       // tokens per tile
constexpr int D = kHeadDim;  // 128
constexpr int STAGES = 2;
constexpr int THREADS = 128;
constexpr int TILE_BYTES = BN * D * 2;  // 16 KiB
constexpr int SMEM_BYTES = BM * D * 2 + STAGES * 2 * TILE_BYTES + STAGES * BN;
// fp8: the first stage's K|V area holds the converted bf16 tile, the second the staged codes
constexpr int ROW8_BYTES = D;                 // 128 codes
constexpr int TILE8_BYTES = BN * ROW8_BYTES;  // 8 KiB
static_assert(STAGES * 2 * TILE8_BYTES <= 2 * TILE_BYTES, "staged codes fit one stage's area");

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a [rows][128] bf16 tile
    return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 -> the 16 bytes are zero-filled, nothing is read
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}


// Token held by cache position p of sequence b, or -1 when the position is
// masked. Sparse: p indexes idx[b]; an entry is used iff it is in [0, n) and
// above the previous entry; anything but -1 padding that is unused is flagged.
template <bool SPARSE>
__device__ __forceinline__ int cache_token(const VerifyArgs &a, int b, int n, int p, bool report) {
    if (!SPARSE) return p < n ? p : -1;
    return sparse_token(a, b, n, p, report);
}

template <bool SPARSE, bool FP8>
__global__ void __launch_bounds__(THREADS, 2) cache_attn_mma_kernel(VerifyArgs a, SplitPlan p) {
    griddep_launch_dependents();  // the merge may be scheduled as this grid's CTAs drain
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + BM * D * 2;  // [stage][K|V][BN][D]
    uint8_t *sValid = sKV + STAGES * 2 * TILE_BYTES;
    uint8_t *sCodes = sKV + 2 * TILE_BYTES;  // fp8: [stage][K|V][BN][128 codes]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int M = a.G * a.N;
    const float sl2 = a.scale * 1.4426950408889634f;  // scores in base 2

    const int64_t g0 = plan_start(p, blockIdx.x), g1 = plan_start(p, blockIdx.x + 1);
    for (int64_t u = g0 / p.tiles_per_unit; u * p.tiles_per_unit < g1; ++u) {
        const int64_t ub = u * p.tiles_per_unit;
        const int tb = (int)((g0 > ub ? g0 : ub) - ub);
        const int te = (int)((g1 < ub + p.tiles_per_unit ? g1 : ub + p.tiles_per_unit) - ub);
        int b, hk, rg;
        plan_unit_coords(p, a.Hkv, u, b, hk, rg);
        const int n = context_len(a, b);
        // fp8: the K scale joins the softmax scale, the V scale the partial's normalisation
        const float sl2u = FP8 ? sl2 * __ldg(a.k_scale + (int64_t)b * a.Hkv + hk) : sl2;
        const float vscale = FP8 ? __ldg(a.v_scale + (int64_t)b * a.Hkv + hk) : 1.f;

        // Q rows of this unit -> shared memory (zero rows past G*N)
        __syncthreads();
        for (int c = tid; c < BM * 16; c += THREADS) {
            const int row = c >> 4, ch = c & 15;
            const int rfull = rg * BM + row;
            const bool ok = rfull < M;
            const int nn = ok ? rfull / a.G : 0, gg = ok ? rfull % a.G : 0;
            const __nv_bfloat16 *src = a.q + (((int64_t)b * a.N + nn) * a.Hq + hk * a.G + gg) * D + ch * 8;
            cp_async16(smem_addr(sQ + swz(row, ch)), ok ? (const void *)src : (const void *)a.q, ok);
        }
        cp_async_commit();

        auto load_tile = [&](int tile, int stage) {
            if (FP8) {  // 8 chunks of 16 codes a row, unswizzled in the staging area
                uint8_t *sK8 = sCodes + (stage * 2) * TILE8_BYTES;
                uint8_t *sV8 = sK8 + TILE8_BYTES;
                const uint8_t *k8 = reinterpret_cast<const uint8_t *>(a.k_cache);
                const uint8_t *v8 = reinterpret_cast<const uint8_t *>(a.v_cache);
                for (int c = tid; c < BN * 8; c += THREADS) {
                    const int row = c >> 3, ch = c & 7;
                    const int t = cache_token<SPARSE>(a, b, n, tile * BN + row, ch == 0);
                    const int64_t roff = t >= 0 ? cache_row_offset(a, b, hk, t, ch == 0) : -1;
                    const bool ok = roff >= 0;
                    const int64_t off = roff + ch * 16;  // one byte an element
                    cp_async16(smem_addr(sK8 + row * ROW8_BYTES + ch * 16), ok ? (const void *)(k8 + off) : (const void *)a.q, ok);
                    cp_async16(smem_addr(sV8 + row * ROW8_BYTES + ch * 16), ok ? (const void *)(v8 + off) : (const void *)a.q, ok);
                    if (ch == 0) sValid[stage * BN + row] = ok;
                }
                cp_async_commit();
                return;
            }
            uint8_t *sK = sKV + (stage * 2) * TILE_BYTES;
            uint8_t *sV = sK + TILE_BYTES;
            for (int c = tid; c < BN * 16; c += THREADS) {
                const int row = c >> 4, ch = c & 15;
                const int t = cache_token<SPARSE>(a, b, n, tile * BN + row, ch == 0);
                // the row's offset (paged: through the block table); a row that does not
                // exist is masked like an unused one
                const int64_t roff = t >= 0 ? cache_row_offset(a, b, hk, t, ch == 0) : -1;
                const bool ok = roff >= 0;
                // a masked row is zero-filled; its (unread) source is a valid address
                const int64_t off = roff + ch * 8;
                cp_async16(smem_addr(sK + swz(row, ch)), ok ? (const void *)(a.k_cache + off) : (const void *)a.q, ok);
                cp_async16(smem_addr(sV + swz(row, ch)), ok ? (const void *)(a.v_cache + off) : (const void *)a.q, ok);
                if (ch == 0) sValid[stage * BN + row] = ok;
            }
            cp_async_commit();
        };

        const int ntile = te - tb;
        load_tile(tb, 0);
        if (ntile > 1) load_tile(tb + 1, 1);

        float acc[16][4];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
        uint32_t qf[8][4];

        for (int it = 0; it < ntile; ++it) {
            if (it + 1 < ntile) cp_async_wait<1>(); else cp_async_wait<0>();
            __syncthreads();
            if (it == 0) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int row = warp * 16 + (lane & 15);
                    ldmatrix_x4(smem_addr(sQ + swz(row, ks * 2 + (lane >> 4))), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
                }
            }
            const int stage = it % STAGES;
            const uint8_t *sK = sKV + (FP8 ? 0 : stage * 2) * TILE_BYTES;
            const uint8_t *sV = sK + TILE_BYTES;
            const uint8_t *valid = sValid + stage * BN;
            if (FP8) {  // the staged codes -> the bf16 tile (16 codes = two 16-byte bf16 chunks)
                const uint8_t *sK8 = sCodes + (stage * 2) * TILE8_BYTES;
                for (int c = tid; c < 2 * BN * 8; c += THREADS) {
                    const int kv = c >= BN * 8, cc = c - kv * BN * 8;
                    const int row = cc >> 3, ch = cc & 7;
                    const uint4 codes = *reinterpret_cast<const uint4 *>(sK8 + kv * TILE8_BYTES + row * ROW8_BYTES + ch * 16);
                    uint8_t *dst = sKV + kv * TILE_BYTES;
                    uint4 lo, hi;
                    e4m3x16_to_bf16x16(codes, lo, hi);
                    *reinterpret_cast<uint4 *>(dst + swz(row, 2 * ch)) = lo;
                    *reinterpret_cast<uint4 *>(dst + swz(row, 2 * ch + 1)) = hi;
                }
                __syncthreads();
            }

            // S = Q K^T for this warp's 16 rows x 64 tokens
            float s[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int tok = np * 16 + ((lane >> 4) << 3) + (lane & 7);
                    const int ch = ks * 2 + ((lane >> 3) & 1);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(smem_addr(sK + swz(tok, ch)), b0, b1, b2, b3);
                    mma_bf16(s[2 * np], qf[ks], b0, b1);
                    mma_bf16(s[2 * np + 1], qf[ks], b2, b3);
                }
            }
            // online softmax (rows gq and gq+8 of the warp)
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int j = nt * 8 + tq * 2;
                const bool v0 = valid[j], v1 = valid[j + 1];
                s[nt][0] = v0 ? s[nt][0] * sl2u : -INFINITY;
                s[nt][1] = v1 ? s[nt][1] * sl2u : -INFINITY;
                s[nt][2] = v0 ? s[nt][2] * sl2u : -INFINITY;
                s[nt][3] = v1 ? s[nt][3] * sl2u : -INFINITY;
                mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
                mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
            }
            float alpha[2], muse[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mnew = fmaxf(mrow[r], mx[r]);
                muse[r] = mnew == -INFINITY ? 0.f : mnew;
                alpha[r] = exp2f(mrow[r] - muse[r]);
                mrow[r] = mnew;
                lrow[r] *= alpha[r];
            }
            uint32_t pf[4][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const float p0 = exp2f(s[nt][0] - muse[0]), p1 = exp2f(s[nt][1] - muse[0]);
                const float p2 = exp2f(s[nt][2] - muse[1]), p3 = exp2f(s[nt][3] - muse[1]);
                lrow[0] += p0 + p1;
                lrow[1] += p2 + p3;
                pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
                pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                acc[i][0] *= alpha[0]; acc[i][1] *= alpha[0];
                acc[i][2] *= alpha[1]; acc[i][3] *= alpha[1];
            }
            // O += P V
#pragma unroll
            for (int kj = 0; kj < 4; ++kj) {
                const uint32_t af[4] = {pf[kj][0], pf[kj][1], pf[kj][2], pf[kj][3]};
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    const int tok = kj * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
                    const int ch = dp * 2 + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_t(smem_addr(sV + swz(tok, ch)), b0, b1, b2, b3);
                    mma_bf16(acc[2 * dp], af, b0, b1);
                    mma_bf16(acc[2 * dp + 1], af, b2, b3);
                }
            }
            __syncthreads();
            if (it + 2 < ntile) load_tile(tb + it + 2, stage);
        }

        // epilogue: normalised partial and its natural-log lse -> slot (cta + unit)
        const int64_t slot = (int64_t)blockIdx.x + u;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float l = lrow[r];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            const int row = warp * 16 + gq + r * 8;
            if (rg * BM + row >= M) continue;
            const float inv = l > 0.f ? vscale / l : 0.f;
            float *dst = a.o_part + (slot * BM + row) * D;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                *reinterpret_cast<float2 *>(dst + nt * 8 + tq * 2) =
                    make_float2(acc[nt][r * 2] * inv, acc[nt][r * 2 + 1] * inv);
            if (tq == 0)
                a.lse_part[slot * BM + row] = l > 0.f ? (mrow[r] + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
    }
}

}  // namespace

int mma_rows_per_unit() { return BM; }
int mma_tile_tokens() { return BN; }

cudaError_t launch_cache_attn_mma(const VerifyArgs &a, const SplitPlan &p, bool sparse,
                                  cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1) {
    auto kern = a.kv_fp8 ? (sparse ? cache_attn_mma_kernel<true, true> : cache_attn_mma_kernel<false, true>)
                         : (sparse ? cache_attn_mma_kernel<true, false> : cache_attn_mma_kernel<false, false>);
    static PerDeviceOnce attr_once;
    cudaError_t e = once_per_device(attr_once, [] {
        cudaError_t r = cudaSuccess;
        for (auto k : {cache_attn_mma_kernel<false, false>, cache_attn_mma_kernel<true, false>,
                       cache_attn_mma_kernel<false, true>, cache_attn_mma_kernel<true, true>})
            if (r == cudaSuccess) r = kernel_attributes(k, SMEM_BYTES);
        return r;
    });
    if (e != cudaSuccess) return e;
    if (ev0) cudaEventRecord(ev0, s);
    kern<<<p.ctas, THREADS, SMEM_BYTES, s>>>(a, p);
    e = cudaGetLastError();
    if (ev1) cudaEventRecord(ev1, s);
    count_launches(1);
    return e;
}

}  // namespace specverify
