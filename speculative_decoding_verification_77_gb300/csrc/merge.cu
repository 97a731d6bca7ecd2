// Log-sum-exp reduction of the split-KV partials, fused with the tree-masked
// draft block (LongSpec section 2.C: cache part without mask + speculative part
// with the tree mask, combined exactly by log-sum-exp), and the exported
// two-part merge.
#include "common.cuh"

namespace specverify {

namespace {

struct OnlineRow {
    float m = -INFINITY;  // running max of the natural-log weights
    float s = 0.f;        // running sum of exp(weight - m)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);

    // add a term exp(w) * x (x = 4 components of the row held by this lane)
    __device__ __forceinline__ void add(float w, float4 x) {
        if (w == -INFINITY) return;
        if (w > m) {
            float c = __expf(m - w);  // m == -inf -> 0
            acc.x *= c; acc.y *= c; acc.z *= c; acc.w *= c;
            s *= c;
            m = w;
        }
        float e = __expf(w - m);
        acc.x += e * x.x; acc.y += e * x.y; acc.z += e * x.z; acc.w += e * x.w;
        s += e;
    }
};

__device__ __forceinline__ float4 load_bf16x4(const __nv_bfloat16 *p) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One warp per output row (b, i, h); lane holds columns 4*lane .. 4*lane+3.
__global__ void __launch_bounds__(256) merge_tree_kernel(VerifyArgs a, SplitPlan p) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)a.B * a.N * a.Hq;
    if (warp >= rows) return;
    const int h = warp % a.Hq;
    const int i = (warp / a.Hq) % a.N;
    const int b = warp / (a.Hq * a.N);
    const int hk = h / a.G, g = h % a.G;
    const int rfull = i * a.G + g;
    const int rg = rfull / p.BM, ru = rfull % p.BM;
    const int64_t u = ((int64_t)b * a.Hkv + hk) * p.row_groups + rg;
    // which pipe slots hold this row, and the row inside a slot
    const int h_lo = p.split_tiles ? 0 : ru / p.slot_rows;
    const int h_hi = p.split_tiles ? p.pipes - 1 : h_lo;
    const int r = p.split_tiles ? ru : ru % p.slot_rows;

    OnlineRow st;
    // cache part: the normalised partials of every CTA (and pipe) that covered this unit
    const int64_t c_lo = plan_cta_of(p, u * p.tiles_per_unit);
    const int64_t c_hi = plan_cta_of(p, (u + 1) * p.tiles_per_unit - 1);
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        for (int hh = h_lo; hh <= h_hi; ++hh) {
            const int64_t slot = (c + u) * p.pipes + hh;
            const float w = a.lse_part[slot * p.slot_rows + r];
            const float4 o =
                *reinterpret_cast<const float4 *>(a.o_part + (slot * p.slot_rows + r) * kHeadDim + 4 * lane);
            st.add(w, o);
        }
    }
    // speculative part: node i and its ancestors (tree mask)
    if (a.k_draft) {
        const float4 qv = load_bf16x4(a.q + (((int64_t)b * a.N + i) * a.Hq + h) * kHeadDim + 4 * lane);
        const int32_t *par = a.parent + (int64_t)b * a.N;
        int j = i;
        while (true) {
            const int64_t kv_off = (((int64_t)b * a.N + j) * a.Hkv + hk) * kHeadDim + 4 * lane;
            const float4 kv = load_bf16x4(a.k_draft + kv_off);
            float dot = qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
            dot = warp_sum(dot);
            st.add(dot * a.scale, load_bf16x4(a.v_draft + kv_off));
            const int pj = __ldg(par + j);
            if (pj == -1) break;
            if (pj < -1 || pj >= j) {  // not a tree in topological order: stop here
                if (lane == 0) flag_status(a.status, SPEC_ERR_BAD_INPUT);
                break;
            }
            j = pj;
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
