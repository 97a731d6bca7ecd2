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

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Running log-sum-exp state of a warp, fed in batches of up to 32 terms: lane d
// holds the natural-log weight of term d of the batch; a term's row (4 columns
// per lane) is loaded once its weight is known, and the loads of a batch are
// independent, so they are in flight together.
struct WarpLse {
    float m = -INFINITY, s = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);

    // folds the batch max into m; returns this lane's weight exp(w - m)
    __device__ __forceinline__ float begin_batch(float w) {
        const float bm = warp_max(w);
        if (bm > m) {
            const float c = __expf(m - bm);  // m == -inf -> 0
            acc.x *= c; acc.y *= c; acc.z *= c; acc.w *= c;
            s *= c;
            m = bm;
        }
        const float e = w == -INFINITY ? 0.f : __expf(w - m);
        s += warp_sum(e);
        return e;
    }
    __device__ __forceinline__ void add(float e, float4 x) {
        acc.x += e * x.x; acc.y += e * x.y; acc.z += e * x.z; acc.w += e * x.w;
    }
};

// One warp per output row (b, i, h); lane holds columns 4*lane .. 4*lane+3.
// Terms: (a) the normalised partials of every CTA and pipe that covered the
// row's unit, weighted by their lse; (b) the draft keys the tree mask lets the
// row see (node i and its ancestors), weighted by their logits.
__global__ void __launch_bounds__(256) merge_tree_kernel(VerifyArgs a, SplitPlan p) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int rows = a.B * a.N * a.Hq;
    if (warp >= rows) return;
    const int h = warp % a.Hq;
    const int bi = warp / a.Hq;  // b * N + i
    const int i = bi % a.N, b = bi / a.N;
    const int hk = h / a.G, g = h - hk * a.G;
    const int rfull = i * a.G + g;
    const int rg = rfull / p.BM, ru = rfull - rg * p.BM;
    const int u = (b * a.Hkv + hk) * p.row_groups + rg;
    // which pipe slots hold this row, and the row inside a slot
    const int h_lo = p.split_tiles ? 0 : ru / p.slot_rows;
    const int nh_shift = p.split_tiles && p.pipes == 2 ? 1 : 0;  // one or two pipe slots per CTA
    const int r = p.split_tiles ? ru : ru % p.slot_rows;
    const int c_lo = (int)plan_cta_of(p, (int64_t)u * p.tiles_per_unit);
    const int c_hi = (int)plan_cta_of(p, (int64_t)(u + 1) * p.tiles_per_unit - 1);
    const int n_parts = (c_hi - c_lo + 1) << nh_shift;
    const int64_t row0 = ((int64_t)(c_lo + u) * p.pipes + h_lo) * p.slot_rows + r;
    const int64_t cta_stride = (int64_t)p.pipes * p.slot_rows;

    WarpLse st;
    // (a) cache part
    for (int k0 = 0; k0 < n_parts; k0 += 32) {
        const int nb = min(32, n_parts - k0);
        const int k = k0 + lane;
        const float w = lane < nb ? a.lse_part[row0 + (k >> nh_shift) * cta_stride + (k & nh_shift) * p.slot_rows]
                                  : -INFINITY;
        const float e = st.begin_batch(w);
#pragma unroll 4
        for (int d = 0; d < nb; ++d) {
            const float ed = __shfl_sync(0xffffffffu, e, d);
            const int kd = k0 + d;
            const int64_t row = row0 + (kd >> nh_shift) * cta_stride + (kd & nh_shift) * p.slot_rows;
            if (ed != 0.f) st.add(ed, *reinterpret_cast<const float4 *>(a.o_part + row * kHeadDim + 4 * lane));
        }
    }
    // (b) speculative part, walking node i's ancestors 32 at a time
    if (a.k_draft) {
        const float4 qv = load_bf16x4(a.q + (int64_t)warp * kHeadDim + 4 * lane);
        const int32_t *par = a.parent + (int64_t)b * a.N;
        const int64_t node_stride = (int64_t)a.Hkv * kHeadDim;
        const __nv_bfloat16 *kd = a.k_draft + ((int64_t)b * a.N * a.Hkv + hk) * kHeadDim + 4 * lane;
        const __nv_bfloat16 *vd = a.v_draft + ((int64_t)b * a.N * a.Hkv + hk) * kHeadDim + 4 * lane;
        int j = i;
        while (j >= 0) {
            int mine = -1, nb = 0;
            while (nb < 32 && j >= 0) {  // lane nb records the next ancestor
                if (lane == nb) mine = j;
                ++nb;
                const int pj = __ldg(par + j);
                if (pj < -1 || pj >= j) {  // not a tree in topological order: stop here
                    if (lane == 0) flag_status(a.status, SPEC_ERR_BAD_INPUT);
                    j = -1;
                } else {
                    j = pj;
                }
            }
            float logit = -INFINITY;
#pragma unroll 4
            for (int d = 0; d < nb; ++d) {
                const int node = __shfl_sync(0xffffffffu, mine, d);
                const float4 kv = load_bf16x4(kd + node * node_stride);
                const float dot = warp_sum(qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w) * a.scale;
                if (lane == d) logit = dot;
            }
            const float e = st.begin_batch(logit);
#pragma unroll 4
            for (int d = 0; d < nb; ++d) {
                const float ed = __shfl_sync(0xffffffffu, e, d);
                const int node = __shfl_sync(0xffffffffu, mine, d);
                st.add(ed, load_bf16x4(vd + node * node_stride));
            }
        }
    }
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = -INFINITY;
    if (st.s > 0.f) {
        const float inv = 1.f / st.s;
        o = make_float4(st.acc.x * inv, st.acc.y * inv, st.acc.z * inv, st.acc.w * inv);
        l = st.m + __logf(st.s);
    }
    *reinterpret_cast<float4 *>(a.out + (int64_t)warp * kHeadDim + 4 * lane) = o;
    if (lane == 0) a.lse[warp] = l;
}

// Exported two-part merge: one warp per row, any d.
__global__ void __launch_bounds__(256) lse_merge2_kernel(const float *o_a, const float *lse_a,
                                                         const float *o_b, const float *lse_b,
                                                         float *out, float *lse_out, int64_t rows,
                                                         int d) {
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float la = lse_a[row], lb = lse_b[row];
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
    const float *pa = o_a + row * d, *pb = o_b + row * d;
    float *po = out + row * d;
    for (int c = lane; c < d; c += 32) {
        const float x = pa[c], y = pb[c];
        po[c] = (wa == 0.f ? 0.f : wa * x) + (wb == 0.f ? 0.f : wb * y);
    }
    if (lane == 0) lse_out[row] = l;
}

}  // namespace

cudaError_t launch_merge_tree(const VerifyArgs &a, const SplitPlan &p, cudaStream_t s) {
    const int64_t rows = (int64_t)a.B * a.N * a.Hq;
    const int64_t blocks = (rows * 32 + 255) / 256;
    merge_tree_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, p);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_lse_merge2(const float *o_a, const float *lse_a, const float *o_b,
                              const float *lse_b, float *out, float *lse_out, int64_t rows, int d,
                              cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows * 32 + 255) / 256;
    lse_merge2_kernel<<<(unsigned)blocks, 256, 0, s>>>(o_a, lse_a, o_b, lse_b, out, lse_out, rows, d);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace specverify
