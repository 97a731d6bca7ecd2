// Hybrid top-k selection of the verification set I_verify: one thread-block
// cluster of CL CTAs per sequence (4 up to 65536 tokens, 8 up to 131072), keys
// in registers.
//
// Dustin, "Metodologia" section 1: keep an attention-sink prefix and a window
// of recent tokens, then fill the rest of a fixed budget in tiers - the top-m
// tokens by the draft-lookahead score, then the best remaining tokens by the
// target-historical score - and emit the set in ascending token order.
//
// CTA r of the cluster owns tokens [2048 Q r, 2048 Q (r + 1)); its warp w the
// Q quads of 128 tokens from 2048 Q r + 128 Q w, and lane l the 4 consecutive
// tokens 128 q + 4 l .. + 3 of quad q. Both tiers' keys (32-bit order-
// preserving keys of the fp32 scores) stay in registers, loaded 16 bytes at a
// time where the rows allow it, so CL SMs share the reading of a sequence. With
// one CTA per SM, a GB300 runs 15 clusters of 8 at a time but many more of 4:
// the smaller cluster keeps a batch of 16 sequences in one wave.
//
// Each tier is an exact radix select in up to three digit passes (11, 11 and
// 10 bits), stopping as soon as the chosen bin holds exactly the keys still
// needed. A pass costs one cluster barrier: every CTA histograms its own keys in
// shared memory (two 16-bit counts per word), and after the barrier every CTA
// reads the CL histograms of the cluster through distributed shared memory (one
// 8-byte read per peer and thread, 4 bins) and finds the same digit from the
// same totals, with two CTA barriers and no further exchange. The histograms
// alternate between two buffers, so a pass never overwrites a buffer that a peer
// may still be reading; each pass clears the buffer the next one fills.
// Each CTA then posts its counts of keys above and equal to the threshold to
// every CTA: tier 1's ride on tier 2's first barrier, tier 2's take one last
// exchange, and from them every CTA knows the members of the CTAs before it (ties
// at the final key go by index: CTA, warp and lane prefixes) and the ascending
// emission finds its positions with no further exchange.
#include "common.cuh"
#include "sm100.cuh"

namespace specverify {

namespace {

using namespace sm100;

constexpr int kMaxCL = 8;     // CTAs per sequence (one cluster), at most
constexpr int kThrL = 512;
constexpr int kWarpsL = kThrL / 32;
constexpr int kBinsL = 2048;  // 11-bit digits
static_assert(kBinsL == 4 * kThrL, "four bins per thread in the digit search");

// Order-preserving key: larger score -> larger key; -0 == +0; NaN -> 0, below
// every number (the smallest key of a number, -inf, is 0x007fffff).
__device__ __forceinline__ uint32_t okey(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the lanes of a warp; *total = the warp's sum.
__device__ __forceinline__ uint32_t warp_excl(uint32_t v, uint32_t *total) {
    const int lane = threadIdx.x & 31;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

__device__ __forceinline__ uint2 dsmem_ld64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

struct ClSmem {
    uint32_t hist[2][kBinsL / 2];  // this CTA's histogram of the current pass (bin 2w + h in half h
                                   // of word w, 16 bits each), two buffers
    uint32_t xc[2][kMaxCL][2];     // per tier, per CTA of the cluster: (members above the
                                   // threshold, keys equal to it), stored there by that CTA
    uint32_t wtot[kWarpsL];
    uint32_t bc[4];
};

// This CTA's per-tier counts (above, equal) into slot [tier][rank] of every CTA of the
// cluster (itself included); they are read locally after the next cluster barrier.
template <int CL>
__device__ __forceinline__ void cl_post(ClSmem &sm, int tier, uint32_t rank, uint32_t above, uint32_t equal) {
    if (threadIdx.x < 2 * CL) {
        const uint32_t r = threadIdx.x >> 1;
        dsmem_st(dsmem_map(&sm.xc[tier][rank][threadIdx.x & 1], r), (threadIdx.x & 1) ? equal : above);
    }
}

// Members of tier `tier` in CTA r: those above the threshold, then the first `need`
// (by index) of those equal to it, CTA by CTA.
__device__ __forceinline__ uint32_t cl_members(const ClSmem &sm, int tier, int r, uint32_t need) {
    uint32_t eq_before = 0u;
    for (int x = 0; x < r; ++x) eq_before += sm.xc[tier][x][1];
    const uint32_t eq = sm.xc[tier][r][1];
    const uint32_t t = eq_before >= need ? 0u : (need - eq_before < eq ? need - eq_before : eq);
    return sm.xc[tier][r][0] + t;
}

// digit of pass p: key bits [31..21], [20..10], [9..0]
__device__ __forceinline__ int cshift(int p) { return p == 0 ? 21 : (p == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t chi_mask(int p) { return p == 0 ? 0u : (p == 1 ? 0xffe00000u : 0xfffffc00u); }
__device__ __forceinline__ uint32_t cdigit_mask(int p) { return p == 2 ? 0x3ffu : 0x7ffu; }

// Warp-uniform count per warp -> the sum over the warps before this one; *total = CTA sum.
__device__ __forceinline__ uint32_t cta_warps_before(uint32_t wcount, ClSmem &sm, uint32_t *total) {
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sm.wtot[warp] = wcount;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarpsL; ++w) {
        const uint32_t x = sm.wtot[w];
        all += x;
        before += w < warp ? x : 0u;
    }
    __syncthreads();
    *total = all;
    return before;
}

// One tier's digit search: the threshold key of the top k (1 <= k <= candidates of the
// sequence) among the candidates `cand` (bit 4 q + e of this thread) under the keys
// key[4 q + e], resolved above *res_shift, with *need = how many candidates agreeing
// with it there belong to the top k, and *all_eq = whether that is all of them. `ph`
// counts the passes made so far (histogram buffer ph & 1).
template <int CL, int Q>
__device__ uint32_t cl_digits(const uint32_t (&key)[4 * Q], uint32_t cand, uint32_t k, ClSmem &sm, int &ph,
                              uint32_t *need, int *res_shift, bool *all_eq) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t prefix = 0u, kr = k;
    int shift = 21;
    bool whole = false;
    for (int p = 0; p < 3; ++p) {
        shift = cshift(p);
        const uint32_t him = chi_mask(p), dm = cdigit_mask(p);
        uint32_t *hist = sm.hist[ph & 1];  // zeroed (at the start, or during the previous pass)
        ++ph;
#pragma unroll
        for (int j = 0; j < 4 * Q; ++j)
            if (((cand >> j) & 1u) && (key[j] & him) == (prefix & him)) {
                const uint32_t bin = (key[j] >> shift) & dm;  // at most 2048 Q <= 16384 per bin: no carry
                atomicAdd(&hist[bin >> 1], 1u << (16 * (bin & 1)));
            }
        cluster_sync();  // every CTA's histogram of this pass is complete and visible
        // bins 2047 - 4 tid .. 2044 - 4 tid (descending) summed over the cluster: words
        // 1023 - 2 tid (bins 2047 / 2046 in the high / low half) and 1022 - 2 tid (2045 / 2044)
        uint32_t cnt[4] = {0u, 0u, 0u, 0u};
        const uint32_t off = (uint32_t)(kBinsL / 2 - 2 - 2 * tid);
#pragma unroll
        for (int r = 0; r < CL; ++r) {
            const uint2 v = dsmem_ld64(dsmem_map(hist + off, (uint32_t)r));
            cnt[0] += v.y >> 16;
            cnt[1] += v.y & 0xffffu;
            cnt[2] += v.x >> 16;
            cnt[3] += v.x & 0xffffu;
        }
        // the other buffer, last read by the peers in the previous pass (they have all passed
        // this pass's barrier), is cleared for the next pass
        reinterpret_cast<uint2 *>(sm.hist[ph & 1])[tid] = make_uint2(0u, 0u);
        const uint32_t own = cnt[0] + cnt[1] + cnt[2] + cnt[3];
        uint32_t wsum;
        uint32_t before = warp_excl(own, &wsum);
        if (lane == 0) sm.wtot[wid] = wsum;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < kWarpsL; ++w) before += w < wid ? sm.wtot[w] : 0u;
        if (before < kr && before + own >= kr) {  // exactly one thread
            uint32_t cum = before;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (cum + cnt[j] >= kr) {
                    sm.bc[1] = (uint32_t)(kBinsL - 1 - (4 * tid + j));
                    sm.bc[2] = kr - cum;
                    sm.bc[3] = cnt[j] == kr - cum ? 1u : 0u;
                    break;
                }
                cum += cnt[j];
            }
        }
        __syncthreads();
        prefix |= sm.bc[1] << shift;
        kr = sm.bc[2];
        whole = sm.bc[3] != 0u;
        if (whole) break;  // the lower digits cannot change the set
    }
    *need = kr;
    *res_shift = shift;
    *all_eq = whole;
    return prefix;
}

// This thread's keys above the threshold (*above) and equal to it (*equal), both at
// the resolution above `shift`.
template <int Q>
__device__ __forceinline__ void cl_split(const uint32_t (&key)[4 * Q], uint32_t cand, uint32_t thr, int shift,
                                         uint32_t *above, uint32_t *equal) {
    const uint32_t thr_hi = thr >> shift;
    uint32_t a = 0u, e = 0u;
#pragma unroll
    for (int j = 0; j < 4 * Q; ++j) {
        if (!((cand >> j) & 1u)) continue;
        const uint32_t hi = key[j] >> shift;
        if (hi > thr_hi) a |= 1u << j;
        else if (hi == thr_hi) e |= 1u << j;
    }
    *above = a;
    *equal = e;
}

// The first `take` (by index) of the equal keys in `eqbits`, `run` being the equal
// keys of the lower CTAs and warps of this CTA (uniform in the warp).
template <int Q>
__device__ __forceinline__ uint32_t cl_first_equal(uint32_t eqbits, uint32_t run, uint32_t take) {
    uint32_t bits = 0u;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const uint32_t e4 = (eqbits >> (4 * q)) & 0xfu;
        uint32_t qtot;
        uint32_t r = run + warp_excl(__popc(e4), &qtot);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((e4 >> e) & 1u) {
                if (r < take) bits |= 1u << (4 * q + e);
                ++r;
            }
        run += qtot;
    }
    return bits;
}

template <bool VEC>
__device__ __forceinline__ float4 load_quad(const float *src, int t, int n) {
    float4 v;
    if (VEC && t + 4 <= n) {
        v = __ldg(reinterpret_cast<const float4 *>(src + t));
    } else {
        v.x = t < n ? __ldg(src + t) : 0.f;
        v.y = t + 1 < n ? __ldg(src + t + 1) : 0.f;
        v.z = t + 2 < n ? __ldg(src + t + 2) : 0.f;
        v.w = t + 3 < n ? __ldg(src + t + 3) : 0.f;
    }
    return v;
}

// Both tiers' keys of this thread (a null row is skipped): every load is issued before
// the first conversion, the raw bits parked in the key registers.
template <int Q, bool VEC>
__device__ __forceinline__ void load_keys_both(uint32_t (&dk)[4 * Q], uint32_t (&tk)[4 * Q], const float *ds,
                                               const float *ts, int seg0, int n) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int t = seg0 + 128 * q + 4 * lane;
        const float4 a = ds ? load_quad<VEC>(ds, t, n) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 c = ts ? load_quad<VEC>(ts, t, n) : make_float4(0.f, 0.f, 0.f, 0.f);
        dk[4 * q] = __float_as_uint(a.x); dk[4 * q + 1] = __float_as_uint(a.y);
        dk[4 * q + 2] = __float_as_uint(a.z); dk[4 * q + 3] = __float_as_uint(a.w);
        tk[4 * q] = __float_as_uint(c.x); tk[4 * q + 1] = __float_as_uint(c.y);
        tk[4 * q + 2] = __float_as_uint(c.z); tk[4 * q + 3] = __float_as_uint(c.w);
    }
#pragma unroll
    for (int j = 0; j < 4 * Q; ++j) {
        dk[j] = okey(__uint_as_float(dk[j]));
        tk[j] = okey(__uint_as_float(tk[j]));
    }
}

template <int CL, int Q, bool VEC>
__global__ void __launch_bounds__(kThrL, 1)
select_cl_kernel(const float *__restrict__ draft, const float *__restrict__ target, int64_t ld, int L,
                 const int32_t *__restrict__ ctx_lens, int sink, int window, int top_m, int budget,
                 int32_t *__restrict__ idx, int32_t *__restrict__ count, uint32_t *status) {
    static_assert(4 * Q <= 32, "one bit per token of a thread in a 32-bit mask");
    __shared__ __align__(16) ClSmem sm;
    // the verify call behind this selection may launch now: its kernels do their set-up on
    // the SMs the clusters leave free and wait for this grid before they read the index set
    griddep_launch_dependents();
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.x / CL;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    select_status_block0(ctx_lens, (int)(gridDim.x / CL), L, status);
    int n = L;
    if (ctx_lens) {  // a length outside [0, L] is clamped (and reported by block 0)
        n = ctx_lens[b];
        n = n < 0 ? 0 : (n > L ? L : n);
    }
    int32_t *out = idx + (int64_t)b * budget;
    if (budget >= n) {  // the whole context fits: verify in full (uniform over the cluster)
        for (int j = (int)rank * kThrL + tid; j < budget; j += CL * kThrL) out[j] = j < n ? j : -1;
        if (count && rank == 0 && tid == 0) count[b] = n;
        return;
    }
    const float *ds = draft + (int64_t)b * ld;
    const float *ts = target + (int64_t)b * ld;
    const int s0 = sink < n ? sink : n;
    const int w0n = window < n - s0 ? window : n - s0;
    const int lo = s0, hi = n - w0n;  // candidates: [lo, hi)
    const int left = budget - s0 - w0n;
    int m = top_m < left ? top_m : left;
    if (m > hi - lo) m = hi - lo;
    const int f = left - m;
    const int seg0 = (int)rank * 2048 * Q + warp * 128 * Q;  // this warp's first token

    uint32_t dk[4 * Q], tk[4 * Q];
    load_keys_both<Q, VEC>(dk, tk, m > 0 ? ds : nullptr, f > 0 ? ts : nullptr, seg0, n);
    // both histogram buffers start cleared; each pass clears the other one for the next
    reinterpret_cast<uint2 *>(sm.hist[0])[tid] = make_uint2(0u, 0u);
    reinterpret_cast<uint2 *>(sm.hist[1])[tid] = make_uint2(0u, 0u);
    __syncthreads();
    uint32_t nmask = 0u, cmask = 0u;  // bit 4 q + e: in the context, a candidate
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = seg0 + 128 * q + 4 * lane + e;
            nmask |= (uint32_t)(t < n) << (4 * q + e);
            cmask |= (uint32_t)(t >= lo && t < hi) << (4 * q + e);
        }

    // Each tier: the digit search, then this thread's keys above the threshold and equal
    // to it; the CTA's counts of both go to every CTA (cl_post) ahead of the next cluster
    // barrier. Ties at the final key go by index, so a tier that takes only part of the
    // keys equal to its threshold needs the counts of the lower CTAs first: that barrier
    // then comes at once. Otherwise tier 1's counts ride on tier 2's first barrier, and
    // the last exchange settles the rest. After that last barrier no CTA reads or writes
    // another's shared memory, so every CTA may exit once it is done.
    int ph = 0;
    uint32_t dbits = 0u, fbits = 0u;
    uint32_t need1 = 0u, need2 = 0u;
    bool posted = false;  // counts posted and not yet followed by a cluster barrier
    if (m > 0) {  // tier 1: top-m by draft score
        int shift;
        bool all_eq;
        uint32_t above, equal, wa, we, cta_a, cta_e;
        const uint32_t thr = cl_digits<CL, Q>(dk, cmask, (uint32_t)m, sm, ph, &need1, &shift, &all_eq);
        cl_split<Q>(dk, cmask, thr, shift, &above, &equal);
        (void)warp_excl(__popc(above), &wa);
        (void)warp_excl(__popc(equal), &we);
        (void)cta_warps_before(wa, sm, &cta_a);
        const uint32_t warp_e = cta_warps_before(we, sm, &cta_e);
        cl_post<CL>(sm, 0, rank, cta_a, cta_e);
        posted = true;
        if (all_eq) {
            dbits = above | equal;
        } else {
            cluster_sync();
            posted = false;
            uint32_t eb = 0u;
            for (int r = 0; r < (int)rank; ++r) eb += sm.xc[0][r][1];
            dbits = above | cl_first_equal<Q>(equal, eb + warp_e, need1);
        }
    }
    if (f > 0) {  // tier 2: fill by target score among the rest (its first barrier also
                  // delivers tier 1's posted counts)
        const uint32_t fcand = cmask & ~dbits;
        int shift;
        bool all_eq;
        uint32_t above, equal, wa, we, cta_a, cta_e;
        const uint32_t thr = cl_digits<CL, Q>(tk, fcand, (uint32_t)f, sm, ph, &need2, &shift, &all_eq);
        posted = false;
        cl_split<Q>(tk, fcand, thr, shift, &above, &equal);
        (void)warp_excl(__popc(above), &wa);
        (void)warp_excl(__popc(equal), &we);
        (void)cta_warps_before(wa, sm, &cta_a);
        const uint32_t warp_e = cta_warps_before(we, sm, &cta_e);
        cl_post<CL>(sm, 1, rank, cta_a, cta_e);
        cluster_sync();  // the last exchange
        uint32_t eb = 0u;
        for (int r = 0; r < (int)rank; ++r) eb += sm.xc[1][r][1];
        fbits = above | (all_eq ? equal : cl_first_equal<Q>(equal, eb + warp_e, need2));
    } else if (posted) {
        cluster_sync();  // tier 1's counts, for the emission (the last exchange)
    }

    // emission: sink u window u tiers, ascending. Position of this CTA's first token: the
    // sink and window tokens and the tier members of the CTAs before it.
    uint32_t pos = 0u;
    const int tok_cta = 2048 * Q;
    for (int r = 0; r < (int)rank; ++r) {
        const int c0 = r * tok_cta, c1 = c0 + tok_cta;
        const int sinkw = max(0, min(c1, lo) - c0) + max(0, min(c1, n) - max(c0, hi));
        pos += (uint32_t)sinkw + (m > 0 ? cl_members(sm, 0, r, need1) : 0u) + (f > 0 ? cl_members(sm, 1, r, need2) : 0u);
    }
    const uint32_t sel = (nmask & ~cmask) | dbits | fbits;
    uint32_t wsel, cta_sel;
    (void)warp_excl(__popc(sel), &wsel);
    pos += cta_warps_before(wsel, sm, &cta_sel);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const uint32_t s4 = (sel >> (4 * q)) & 0xfu;
        uint32_t qtot;
        uint32_t p = pos + warp_excl(__popc(s4), &qtot);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((s4 >> e) & 1u) {
                if (p < (uint32_t)budget) out[p] = seg0 + 128 * q + 4 * lane + e;
                ++p;
            }
        pos += qtot;
    }
    if (count && rank == 0 && tid == 0) count[b] = budget;
}

template <int CL, int Q, bool VEC>
cudaError_t launch_cl(const float *ds, const float *ts, int64_t ld, int B, int L, const int32_t *ctx_lens, int sink,
                      int window, int top_m, int budget, int32_t *idx, int32_t *count, uint32_t *status,
                      cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B * CL);
    cfg.blockDim = dim3(kThrL);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_cl_kernel<CL, Q, VEC>, ds, ts, ld, L, ctx_lens, sink, window, top_m,
                              budget, idx, count, status);
}

}  // namespace

// One cluster per sequence (4 CTAs up to 65536 tokens, 8 up to 131072), keys in
// registers; returns false (nothing launched) for longer contexts.
bool launch_select_cluster_reg(const float *ds, const float *ts, int64_t ld, int B, int L, const int32_t *ctx_lens,
                               int sink, int window, int top_m, int budget, int32_t *idx, int32_t *count,
                               uint32_t *status, cudaStream_t s, cudaError_t *err) {
    *err = cudaSuccess;
    if (L > 8 * 2048 * 8) return false;
    // 16-byte loads when both score rows start on 16-byte boundaries
    const bool vec = ld % 4 == 0 && (uintptr_t)ds % 16 == 0 && (uintptr_t)ts % 16 == 0;
    auto go = [&](auto launch) {
        *err = launch(ds, ts, ld, B, L, ctx_lens, sink, window, top_m, budget, idx, count, status, s);
    };
    if (L <= 4 * 2048) {
        vec ? go(launch_cl<4, 1, true>) : go(launch_cl<4, 1, false>);
    } else if (L <= 4 * 2048 * 2) {
        vec ? go(launch_cl<4, 2, true>) : go(launch_cl<4, 2, false>);
    } else if (L <= 4 * 2048 * 4) {
        vec ? go(launch_cl<4, 4, true>) : go(launch_cl<4, 4, false>);
    } else if (L <= 4 * 2048 * 8) {
        vec ? go(launch_cl<4, 8, true>) : go(launch_cl<4, 8, false>);
    } else {
        vec ? go(launch_cl<8, 8, true>) : go(launch_cl<8, 8, false>);
    }
    count_launches(1);
    if (*err == cudaSuccess) *err = cudaGetLastError();
    return true;
}

}  // namespace specverify
