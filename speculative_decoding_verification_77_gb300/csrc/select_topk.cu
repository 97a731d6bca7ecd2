// Hybrid top-k selection of the verification set I_verify.
//
// Dustin, "Metodologia" section 1: keep an attention-sink prefix and a window
// of recent tokens, then fill the rest of a fixed budget in tiers - the top-m
// tokens by the draft-lookahead score, then the best remaining tokens by the
// target-historical score. The result is emitted in ascending token order.
//
// One CTA of 1024 threads per sequence. Each tier is an exact radix select on
// a 32-bit order-preserving key of the fp32 score (four 8-bit digit passes,
// warp-aggregated shared-memory histograms), which yields the threshold key
// and how many tokens equal to it are still needed; an ordered block scan
// then gives those equal tokens to the lowest indices. The draft tier is kept
// as a bitmap in shared memory (one bit per token), so L <= 1,572,864.
#include "common.cuh"

namespace specverify {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Order-preserving key: larger score -> larger key; -0 == +0; NaN -> 0, below
// every number (the smallest key of a number, -inf, is 0x007fffff).
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelectSmem {
    uint32_t hist[256];
    uint32_t warp_tot[kWarps];
    uint32_t bcast[4];
};

// Exclusive block scan of one value per thread; returns the prefix, *total = sum.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, SelectSmem &sm, uint32_t *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        uint32_t t = sm.warp_tot[lane];
        uint32_t s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        sm.warp_tot[lane] = s - t;  // exclusive prefix of the warp totals
        if (lane == 31) sm.bcast[0] = s;
    }
    __syncthreads();
    const uint32_t r = sm.warp_tot[wid] + x - v;
    *total = sm.bcast[0];
    __syncthreads();
    return r;
}

__device__ __forceinline__ bool bit_set(const uint32_t *bits, int t) {
    return (bits[t >> 5] >> (t & 31)) & 1u;
}

// k-th largest key (k >= 1) among tokens t in [lo, hi) not in `exclude`.
// Returns the key; *need = how many tokens with exactly that key belong to the top k.
__device__ uint32_t radix_select(const float *score, int lo, int hi, const uint32_t *exclude,
                                 uint32_t k, SelectSmem &sm, uint32_t *need) {
    uint32_t prefix = 0u;
    uint32_t kr = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kThreads) sm.hist[i] = 0u;
        __syncthreads();
        const uint32_t hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
        for (int base = lo; base < hi; base += kThreads) {
            const int t = base + threadIdx.x;
            int digit = -1;
            if (t < hi && !(exclude && bit_set(exclude, t))) {
                const uint32_t key = order_key(__ldg(score + t));
                if ((key & hi_mask) == (prefix & hi_mask)) digit = (key >> shift) & 0xffu;
            }
            // one shared atomic per distinct digit in the warp
            const unsigned peers = __match_any_sync(0xffffffffu, digit);
            const int leader = __ffs(peers) - 1;
            if (digit >= 0 && (threadIdx.x & 31) == leader) atomicAdd(&sm.hist[digit], __popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l owns digits 255-8l .. 248-8l (descending order of digits)
            const int lane = threadIdx.x;
            uint32_t own = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) own += sm.hist[255 - 8 * lane - j];
            uint32_t incl = own;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - own;
            const unsigned hit = __ballot_sync(0xffffffffu, excl < kr && incl >= kr);
            const int owner = __ffs(hit) - 1;  // exactly one lane when kr <= candidates
            if (lane == owner) {
                uint32_t cum = excl;
                for (int j = 0; j < 8; ++j) {
                    const int dgt = 255 - 8 * lane - j;
                    const uint32_t c = sm.hist[dgt];
                    if (cum + c >= kr) {
                        sm.bcast[1] = (uint32_t)dgt;
                        sm.bcast[2] = kr - cum;
                        break;
                    }
                    cum += c;
                }
            }
        }
        __syncthreads();
        prefix |= sm.bcast[1] << shift;
        kr = sm.bcast[2];
        __syncthreads();
    }
    *need = kr;
    return prefix;
}

// Marks into `out_bits` (words owned per thread) the top-k of [lo, hi) \ exclude:
// keys above `thr`, plus the first `need` tokens (by index) whose key equals `thr`.
__device__ void mark_tier(const float *score, int lo, int hi, const uint32_t *exclude,
                          uint32_t thr, uint32_t need, uint32_t *out_bits, int w0, int w1,
                          SelectSmem &sm) {
    uint32_t eq = 0;
    for (int w = w0; w < w1; ++w) {
        for (int j = 0; j < 32; ++j) {
            const int t = w * 32 + j;
            if (t < lo || t >= hi || (exclude && bit_set(exclude, t))) continue;
            eq += order_key(__ldg(score + t)) == thr;
        }
    }
    uint32_t total;
    uint32_t rank = block_exclusive_scan(eq, sm, &total);
    for (int w = w0; w < w1; ++w) {
        uint32_t word = 0;
        for (int j = 0; j < 32; ++j) {
            const int t = w * 32 + j;
            if (t < lo || t >= hi || (exclude && bit_set(exclude, t))) continue;
            const uint32_t key = order_key(__ldg(score + t));
            bool take = key > thr;
            if (key == thr) {
                take = rank < need;
                ++rank;
            }
            word |= (uint32_t)take << j;
        }
        out_bits[w] = word;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
select_topk_kernel(const float *__restrict__ draft, const float *__restrict__ target, int64_t ld,
                   int L, const int32_t *__restrict__ ctx_lens, int sink, int window, int top_m,
                   int budget, int32_t *__restrict__ idx, int32_t *__restrict__ count,
                   uint32_t *status) {
    extern __shared__ __align__(16) uint32_t dyn[];
    __shared__ SelectSmem sm;
    const int b = blockIdx.x;
    int n = L;
    if (ctx_lens) {
        n = ctx_lens[b];
        if (n < 0 || n > L) {
            if (threadIdx.x == 0) flag_status(status, SPEC_ERR_BAD_INPUT);
            n = n < 0 ? 0 : L;
        }
    }
    int32_t *out = idx + (int64_t)b * budget;
    if (budget >= n) {  // the whole context fits: verify in full
        for (int j = threadIdx.x; j < budget; j += kThreads) out[j] = j < n ? j : -1;
        if (count && threadIdx.x == 0) count[b] = n;
        return;
    }
    const float *ds = draft + (int64_t)b * ld;
    const float *ts = target + (int64_t)b * ld;
    const int s0 = sink < n ? sink : n;
    const int w0n = window < n - s0 ? window : n - s0;
    const int lo = s0, hi = n - w0n;
    int left = budget - s0 - w0n;
    int m = top_m < left ? top_m : left;
    if (m > hi - lo) m = hi - lo;
    const int f = left - m;

    const int nwords = (n + 31) >> 5;
    const int wpt = (nwords + kThreads - 1) / kThreads;
    const int wa = threadIdx.x * wpt;
    const int wb = min(wa + wpt, nwords);
    uint32_t *dbits = dyn;  // [nwords] draft-tier membership

    // tier 1: top-m by draft score
    if (m > 0) {
        uint32_t need;
        const uint32_t thr = radix_select(ds, lo, hi, nullptr, (uint32_t)m, sm, &need);
        mark_tier(ds, lo, hi, nullptr, thr, need, dbits, wa, wb, sm);
    } else {
        for (int w = wa; w < wb; ++w) dbits[w] = 0u;
    }
    __syncthreads();
    // tier 2: fill by target score among the rest; reuse each thread's own words
    uint32_t thr_f = 0, need_f = 0;
    if (f > 0) thr_f = radix_select(ts, lo, hi, dbits, (uint32_t)f, sm, &need_f);
    // final ordered pass: selected = sink u window u D u F, emitted ascending
    uint32_t eq = 0;
    if (f > 0) {
        for (int w = wa; w < wb; ++w)
            for (int j = 0; j < 32; ++j) {
                const int t = w * 32 + j;
                if (t < lo || t >= hi || bit_set(dbits, t)) continue;
                eq += order_key(__ldg(ts + t)) == thr_f;
            }
    }
    uint32_t eq_total;
    uint32_t eq_rank = block_exclusive_scan(eq, sm, &eq_total);
    // count selected per thread, in index order
    uint32_t sel = 0;
    uint32_t r2 = eq_rank;
    for (int w = wa; w < wb; ++w)
        for (int j = 0; j < 32; ++j) {
            const int t = w * 32 + j;
            if (t >= n) continue;
            bool take;
            if (t < lo || t >= hi) take = true;
            else if (bit_set(dbits, t)) take = true;
            else if (f > 0) {
                const uint32_t key = order_key(__ldg(ts + t));
                take = key > thr_f;
                if (key == thr_f) { take = r2 < need_f; ++r2; }
            } else take = false;
            sel += take;
        }
    uint32_t total;
    uint32_t pos = block_exclusive_scan(sel, sm, &total);
    r2 = eq_rank;
    for (int w = wa; w < wb; ++w)
        for (int j = 0; j < 32; ++j) {
            const int t = w * 32 + j;
            if (t >= n) continue;
            bool take;
            if (t < lo || t >= hi) take = true;
            else if (bit_set(dbits, t)) take = true;
            else if (f > 0) {
                const uint32_t key = order_key(__ldg(ts + t));
                take = key > thr_f;
                if (key == thr_f) { take = r2 < need_f; ++r2; }
            } else take = false;
            if (take && pos < (uint32_t)budget) out[pos++] = t;
        }
    for (int j = (int)total + threadIdx.x; j < budget; j += kThreads) out[j] = -1;
    if (count && threadIdx.x == 0) count[b] = (int32_t)(total < (uint32_t)budget ? total : budget);
}

}  // namespace

cudaError_t launch_select_topk(const float *ds, const float *ts, int64_t ld, int B, int L,
                               const int32_t *ctx_lens, int sink, int window, int top_m,
                               int budget, int32_t *idx, int32_t *count, uint32_t *status,
                               cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    const size_t smem = (size_t)((L + 31) / 32) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    select_topk_kernel<<<B, kThreads, smem, s>>>(ds, ts, ld, L, ctx_lens, sink, window, top_m, budget,
                                                 idx, count, status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace specverify
