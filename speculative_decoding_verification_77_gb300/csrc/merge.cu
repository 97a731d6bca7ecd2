// Log-sum-exp reduction of the split-KV partials, fused with the tree-masked
// draft block (LongSpec section 2.C: cache part without mask + speculative part
// with the tree mask, combined exactly by log-sum-exp), and the exported
// two-part merge.
#include "common.cuh"

namespace specverify {

namespace {

__device__ __forceinline__ float4 load_bf16x4(const __nv_bfloat16 *p) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// Reductions over the lanes that hold the same row j = lane % GB (lane bits >= log2 GB).
template <int GB>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = 16; o >= GB; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
template <int GB>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = 16; o >= GB; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Reduce-scatter across the warp: lane l holds V partial sums p[0..V) (V a
// power of two, at most 32) and gets back the warp-wide sum of entry l % V. Each
// halving step keeps the half of the entries whose index bit matches the lane's
// and adds the partner's copy of that half; the lane bits above log2 V are then
// summed with plain butterflies. 31 shuffles for V = 32 instead of 32 x 5.
template <int V>
__device__ __forceinline__ float reduce_scatter(float (&p)[V], int lane) {
#pragma unroll
    for (int h = V / 2; h >= 1; h >>= 1) {
        const bool up = (lane & h) != 0;
#pragma unroll
        for (int t = 0; t < h; ++t) {
            const float keep = up ? p[t + h] : p[t];
            const float send = up ? p[t] : p[t + h];
            p[t] = keep + __shfl_xor_sync(0xffffffffu, send, h);
        }
    }
    float x = p[0];
#pragma unroll
    for (int o = 16; o >= V; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// GB consecutive floats of a warp's weight scratch (p aligned to GB floats).
template <int GB>
__device__ __forceinline__ void load_weights(const float *p, float (&w)[GB]) {
    if constexpr (GB >= 4) {
#pragma unroll
        for (int c = 0; c < GB; c += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(p + c);
            w[c] = v.x; w[c + 1] = v.y; w[c + 2] = v.z; w[c + 3] = v.w;
        }
    } else if constexpr (GB == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = p[0];
    }
}

// Running log-sum-exp state of GB rows held by one warp (lane holds columns
// 4*lane .. 4*lane+3 of every row). Terms arrive in batches of up to 32/GB:
// lane q holds the natural-log weight of term q / GB for row q % GB.
template <int GB>
struct RowsLse {
    float m[GB], s[GB];  // warp-uniform running max and sum of every row
    float4 acc[GB];
    float m_mine;        // m[lane % GB], kept in step without indexing m by a lane-dependent value
    __device__ __forceinline__ RowsLse() : m_mine(-INFINITY) {
#pragma unroll
        for (int j = 0; j < GB; ++j) { m[j] = -INFINITY; s[j] = 0.f; acc[j] = make_float4(0.f, 0.f, 0.f, 0.f); }
    }
    // fold a batch into the running maxima; returns this lane's weight exp(w - m[lane % GB])
    __device__ __forceinline__ float begin_batch(float w, int lane) {
        const float bm = group_max<GB>(w);
#pragma unroll
        for (int j = 0; j < GB; ++j) {
            const float bmj = __shfl_sync(0xffffffffu, bm, j);
            if (bmj > m[j]) {
                const float c = __expf(m[j] - bmj);  // m == -inf -> 0
                acc[j].x *= c; acc[j].y *= c; acc[j].z *= c; acc[j].w *= c;
                s[j] *= c;
                m[j] = bmj;
            }
        }
        m_mine = fmaxf(m_mine, bm);
        const float e = w == -INFINITY ? 0.f : __expf(w - m_mine);
        const float es = group_sum<GB>(e);
#pragma unroll
        for (int j = 0; j < GB; ++j) s[j] += __shfl_sync(0xffffffffu, es, j);
        return e;
    }
    __device__ __forceinline__ void add(int j, float e, float4 x) {
        acc[j].x += e * x.x; acc[j].y += e * x.y; acc[j].z += e * x.z; acc[j].w += e * x.w;
    }
};

// One warp per (b, i, h_kv, block of GB query heads); lane holds columns
// 4*lane .. 4*lane+3 of the GB output rows, which are consecutive in `out` and
// in every partial slot. Terms of each row: (b) the draft keys the tree mask
// lets node i see (itself and its ancestors), weighted by their logits, and
// (a) the normalised partials of every CTA and pipe that covered the unit,
// weighted by their lse. The tree part reads nothing the cache kernel writes,
// so it runs first and, under programmatic dependent launch, overlaps the
// cache kernel's last CTAs; the wait for the partials comes after it. The
// ancestor walk runs over the parent row staged in shared memory, and each
// batch of draft K/V rows (shared by the GB heads) and of partials is loaded
// in one go, so a warp makes a handful of round trips to memory. The logits of
// a batch come out of one reduce-scatter, and the batch's weights reach every
// lane through a 32-float scratch of the warp in shared memory.
template <int GB>
__global__ void __launch_bounds__(256) merge_tree_kernel(VerifyArgs a, SplitPlan p) {
    extern __shared__ int32_t parent_smem[];  // [warps per block][N]
    __shared__ __align__(16) float w_smem[8][32];  // [warp][term * GB + head]: a batch's weights
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nblk = a.G / GB;
    const int warps = a.B * a.N * a.Hkv * nblk;
    if (warp >= warps) return;
    const int gb = warp % nblk;
    const int t1 = warp / nblk;
    const int hk = t1 % a.Hkv;
    const int bi = t1 / a.Hkv;  // b * N + i
    const int i = bi % a.N, b = bi / a.N;
    const int h0 = hk * a.G + gb * GB;
    const int64_t out_row0 = (int64_t)bi * a.Hq + h0;
    constexpr int PER_BATCH = 32 / GB;                 // lse terms per shuffle batch
    constexpr int TB = PER_BATCH < 8 ? PER_BATCH : 8;  // draft rows loaded per batch
    constexpr int U = GB >= 8 ? 2 : (GB == 4 ? 4 : 8); // partial rows loaded per chunk
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);

    RowsLse<GB> st;
    float *wsc = w_smem[threadIdx.x >> 5];
    // (b) speculative part: node i and its ancestors, TB at a time
    if (a.k_draft) {
        int32_t *ps = parent_smem + (threadIdx.x >> 5) * a.N;
        const int32_t *par = a.parent + (int64_t)b * a.N;
        for (int t = lane; t <= i; t += 32) ps[t] = __ldg(par + t);
        float4 qv[GB];
#pragma unroll
        for (int j = 0; j < GB; ++j) qv[j] = load_bf16x4(a.q + (out_row0 + j) * kHeadDim + 4 * lane);
        const int64_t node_stride = (int64_t)a.Hkv * kHeadDim;
        const __nv_bfloat16 *kd = a.k_draft + ((int64_t)b * a.N * a.Hkv + hk) * kHeadDim + 4 * lane;
        const __nv_bfloat16 *vd = a.v_draft + ((int64_t)b * a.N * a.Hkv + hk) * kHeadDim + 4 * lane;
        __syncwarp();
        int j = i;
        while (j >= 0) {
            int mine = -1, nb = 0;
            while (nb < TB && j >= 0) {  // lane nb records the next ancestor
                if (lane == nb) mine = j;
                ++nb;
                const int pj = ps[j];
                if (pj < -1 || pj >= j) {  // not a tree in topological order: stop here
                    if (lane == 0) flag_status(a.status, SPEC_ERR_BAD_INPUT);
                    j = -1;
                } else {
                    j = pj;
                }
            }
            float4 kr[TB], vr[TB];
#pragma unroll
            for (int d = 0; d < TB; ++d) {
                const int node = __shfl_sync(0xffffffffu, mine, d);
                kr[d] = d < nb ? load_bf16x4(kd + node * node_stride) : zero4;
                vr[d] = d < nb ? load_bf16x4(vd + node * node_stride) : zero4;
            }
            // lane d*GB + jj gets the logit of ancestor d for head jj (padding rows: -inf)
            constexpr int V = TB * GB;
            float pd[V];
#pragma unroll
            for (int d = 0; d < TB; ++d)
#pragma unroll
                for (int jj = 0; jj < GB; ++jj)
                    pd[d * GB + jj] = qv[jj].x * kr[d].x + qv[jj].y * kr[d].y + qv[jj].z * kr[d].z + qv[jj].w * kr[d].w;
            float logit = reduce_scatter<V>(pd, lane) * a.scale;
            if (lane >= V || (lane & (V - 1)) / GB >= nb) logit = -INFINITY;
            const float e = st.begin_batch(logit, lane);
            wsc[lane] = e;
            __syncwarp();
#pragma unroll
            for (int d = 0; d < TB; ++d) {  // padding rows are zero with weight zero
                float wd[GB];
                load_weights<GB>(wsc + d * GB, wd);
#pragma unroll
                for (int jj = 0; jj < GB; ++jj) st.add(jj, wd[jj], vr[d]);
            }
            __syncwarp();  // the scratch is read before the next batch overwrites it
        }
    }

    // (a) cache part: wait until the cache kernel's partials are complete and visible
    griddep_wait();
    const int rfull = i * a.G + gb * GB;  // first unit row of the block (a multiple of GB)
    const int rg = rfull / p.BM, ru = rfull - rg * p.BM;
    const int u = (int)plan_unit(p, a.Hkv, b, hk, rg);
    const int h_lo = p.split_tiles ? 0 : ru / p.slot_rows;
    const int nh_shift = p.split_tiles && p.pipes == 2 ? 1 : 0;  // one or two pipe slots per CTA
    const int r = p.split_tiles ? ru : ru % p.slot_rows;
    const int c_lo = (int)plan_cta_of(p, (int64_t)u * p.tiles_per_unit);
    const int c_hi = (int)plan_cta_of(p, (int64_t)(u + 1) * p.tiles_per_unit - 1);
    const int n_parts = (c_hi - c_lo + 1) << nh_shift;
    const int64_t row0 = ((int64_t)(c_lo + u) * p.pipes + h_lo) * p.slot_rows + r;
    const int64_t cta_stride = (int64_t)p.pipes * p.slot_rows;
    auto part_row = [&](int k) -> int64_t {
        return row0 + (k >> nh_shift) * cta_stride + (k & nh_shift) * p.slot_rows;
    };
    for (int k0 = 0; k0 < n_parts; k0 += PER_BATCH) {
        const int nb = min(PER_BATCH, n_parts - k0);
        const int kq = lane / GB, jq = lane & (GB - 1);
        const float w = kq < nb ? a.lse_part[part_row(k0 + kq) + jq] : -INFINITY;
        float e = 0.f;
        for (int d0 = 0; d0 < nb; d0 += U) {
            float4 x[U][GB];
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                const float *src = a.o_part + part_row(k0 + d0 + uu) * kHeadDim + 4 * lane;
#pragma unroll
                for (int jj = 0; jj < GB; ++jj)
                    x[uu][jj] = d0 + uu < nb ? *reinterpret_cast<const float4 *>(src + jj * kHeadDim) : zero4;
            }
            if (d0 == 0) {  // after the first chunk's loads are issued
                e = st.begin_batch(w, lane);
                wsc[lane] = e;
                __syncwarp();
            }
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                if (d0 + uu < nb) {
                    float wk[GB];
                    load_weights<GB>(wsc + (d0 + uu) * GB, wk);
#pragma unroll
                    for (int jj = 0; jj < GB; ++jj)
                        if (wk[jj] != 0.f) st.add(jj, wk[jj], x[uu][jj]);  // an empty partial may hold anything
                }
            }
        }
        __syncwarp();  // the scratch is read before the next batch overwrites it
    }
#pragma unroll
    for (int j = 0; j < GB; ++j) {
        float4 o = zero4;
        float l = -INFINITY;
        if (st.s[j] > 0.f) {
            const float inv = 1.f / st.s[j];
            o = make_float4(st.acc[j].x * inv, st.acc[j].y * inv, st.acc[j].z * inv, st.acc[j].w * inv);
            l = st.m[j] + __logf(st.s[j]);
        }
        const int64_t e0 = (out_row0 + j) * kHeadDim + 4 * lane;  // first of this lane's 4 elements
        if (a.out_bf16) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
            uint2 w;
            w.x = *reinterpret_cast<const uint32_t *>(&lo);
            w.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + e0) = w;
        } else {
            *reinterpret_cast<float4 *>(a.out + e0) = o;
        }
        if (lane == 0) a.lse[out_row0 + j] = l;
    }
}

// Exported two-part merge: one warp per row, any d. With VEC (d a multiple of 4, every
// row 16-byte aligned) a lane moves 4 consecutive floats per load and store, so a row of
// d = 128 is one float4 per lane and part; the two lse loads and the first row loads are
// issued together. In place (out == o_a, lse_out == lse_a) is allowed: every lane reads its
// own elements before writing them, and the lse values are read by all lanes before lane 0
// writes the row's lse.
template <bool VEC>
__global__ void __launch_bounds__(256) lse_merge2_kernel(const float *o_a, const float *lse_a,
                                                         const float *o_b, const float *lse_b,
                                                         float *out, float *lse_out, int64_t rows,
                                                         int d) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float la = lse_a[row], lb = lse_b[row];
    const float *pa = o_a + row * d, *pb = o_b + row * d;
    float *po = out + row * d;
    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), y0 = x0;
    if (VEC && 4 * lane < d) {  // the first float4 of each part, in flight with the lse loads
        x0 = *reinterpret_cast<const float4 *>(pa + 4 * lane);
        y0 = *reinterpret_cast<const float4 *>(pb + 4 * lane);
    }
    __syncwarp();  // every lane has read the lse values before lane 0 may overwrite them in place
    const float m = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f, l = -INFINITY;
    if (m != -INFINITY) {
        const float ea = __expf(la - m), eb = __expf(lb - m);
        const float inv = 1.f / (ea + eb);
        wa = ea * inv;
        wb = eb * inv;
        l = m + __logf(ea + eb);
    }
    if (isnan(la) || isnan(lb)) { wa = wb = l = NAN; }
    auto mix = [&](float x, float y) { return (wa == 0.f ? 0.f : wa * x) + (wb == 0.f ? 0.f : wb * y); };
    if (VEC) {
        for (int c = 4 * lane; c < d; c += 128) {
            float4 x = x0, y = y0;
            if (c != 4 * lane) {
                x = *reinterpret_cast<const float4 *>(pa + c);
                y = *reinterpret_cast<const float4 *>(pb + c);
            }
            *reinterpret_cast<float4 *>(po + c) = make_float4(mix(x.x, y.x), mix(x.y, y.y), mix(x.z, y.z), mix(x.w, y.w));
        }
    } else {
        for (int c = lane; c < d; c += 32) po[c] = mix(pa[c], pb[c]);
    }
    if (lane == 0) lse_out[row] = l;
}

}  // namespace

// Attributes of the merge kernels, set once per device: shared memory for the largest N
// (8 warps x 4096 parents).
cudaError_t merge_attributes() {
    constexpr int kMaxMergeSmem = 8 * 4096 * (int)sizeof(int32_t);
    static PerDeviceOnce attr_once;
    return once_per_device(attr_once, [] {
        cudaError_t r = kernel_attributes(merge_tree_kernel<8>, kMaxMergeSmem);
        if (r == cudaSuccess) r = kernel_attributes(merge_tree_kernel<4>, kMaxMergeSmem);
        if (r == cudaSuccess) r = kernel_attributes(merge_tree_kernel<2>, kMaxMergeSmem);
        if (r == cudaSuccess) r = kernel_attributes(merge_tree_kernel<1>, kMaxMergeSmem);
        if (r == cudaSuccess) r = kernel_attributes(lse_merge2_kernel<true>, 0);
        if (r == cudaSuccess) r = kernel_attributes(lse_merge2_kernel<false>, 0);
        return r;
    });
}

cudaError_t launch_merge_tree(const VerifyArgs &a, const SplitPlan &p, cudaStream_t s) {
    // heads per warp: the largest of 8, 4, 2, 1 that divides G, halved while that leaves
    // fewer than ~10 warps per SM to hide the latency of each warp's chain of loads
    constexpr int64_t kMinWarps = 1536;
    int gb = a.G % 8 == 0 ? 8 : a.G % 4 == 0 ? 4 : a.G % 2 == 0 ? 2 : 1;
    while (gb > 1 && (int64_t)a.B * a.N * a.Hkv * (a.G / gb) < kMinWarps) gb >>= 1;
    const int64_t warps = (int64_t)a.B * a.N * a.Hkv * (a.G / gb);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps * 32 + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = (size_t)8 * a.N * sizeof(int32_t);  // a parent row per warp
    cfg.stream = s;
    // programmatic dependent launch: the blocks may start while the cache kernel drains;
    // griddepcontrol.wait inside the kernel orders the reads of its partials
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = merge_attributes();
    if (e != cudaSuccess) return e;
    switch (gb) {
        case 8: e = cudaLaunchKernelEx(&cfg, merge_tree_kernel<8>, a, p); break;
        case 4: e = cudaLaunchKernelEx(&cfg, merge_tree_kernel<4>, a, p); break;
        case 2: e = cudaLaunchKernelEx(&cfg, merge_tree_kernel<2>, a, p); break;
        default: e = cudaLaunchKernelEx(&cfg, merge_tree_kernel<1>, a, p); break;
    }
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_lse_merge2(const float *o_a, const float *lse_a, const float *o_b,
                              const float *lse_b, float *out, float *lse_out, int64_t rows, int d,
                              cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    if (const cudaError_t e = merge_attributes(); e != cudaSuccess) return e;
    const int64_t blocks = (rows * 32 + 255) / 256;
    const bool vec = d % 4 == 0 && ((reinterpret_cast<uintptr_t>(o_a) | reinterpret_cast<uintptr_t>(o_b) |
                                     reinterpret_cast<uintptr_t>(out)) & 15) == 0;
    if (vec)
        lse_merge2_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(o_a, lse_a, o_b, lse_b, out, lse_out, rows, d);
    else
        lse_merge2_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(o_a, lse_a, o_b, lse_b, out, lse_out, rows, d);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace specverify
