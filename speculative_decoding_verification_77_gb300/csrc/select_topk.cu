// Hybrid top-k selection of the verification set I_verify.
//
// Dustin, "Metodologia" section 1: keep an attention-sink prefix and a window
// of recent tokens, then fill the rest of a fixed budget in tiers - the top-m
// tokens by the draft-lookahead score, then the best remaining tokens by the
// target-historical score. The result is emitted in ascending token order.
//
// Contexts longer than 131072 tokens (shorter ones go to select_cl.cu): one
// thread-block cluster of 8 CTAs per sequence; CTA r owns a contiguous
// chunk of the context, and inside it warp w owns a contiguous segment that it
// walks 32 tokens at a time (coalesced loads, one bitmap word per step). Each
// tier is an exact radix select on a 32-bit order-preserving key of the fp32
// score in three digit passes (11, 11, 10 bits): every CTA histograms its
// chunk in shared memory and adds the non-empty bins into the CTA that owns
// them through distributed shared memory; after a cluster barrier every CTA
// reads all totals and finds the same digit. The select yields the threshold
// key and how many tokens equal to it are still needed; those go to the
// lowest indices, ranked by warp ballots with CTA and warp prefixes. Tier
// members are kept as a bitmap in shared memory (one bit per token of the
// chunk), and the final ascending emission is one more ballot pass over it.
#include "common.cuh"
#include "sm100.cuh"

namespace specverify {

namespace {

using namespace sm100;

constexpr int kCtas = 8;  // CTAs per sequence (one cluster)
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;  // 11-bit digits
constexpr int kSlice = kBins / kCtas;  // bins whose cluster total lives in each CTA
constexpr int kPassesPerTier = 3;
constexpr int kMaxL = 1572864;  // longest context the entry point accepts
static_assert(kBins == 4 * kThreads, "four bins per thread in the digit search");

// Order-preserving key: larger score -> larger key; -0 == +0; NaN -> 0, below
// every number (the smallest key of a number, -inf, is 0x007fffff).
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// digit of pass p: key bits [31..21], [20..10], [9..0]
__device__ __forceinline__ int pass_shift(int p) { return p == 0 ? 21 : (p == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t pass_hi_mask(int p) { return p == 0 ? 0u : (p == 1 ? 0xffe00000u : 0xfffffc00u); }
__device__ __forceinline__ uint32_t pass_digit_mask(int p) { return p == 2 ? 0x3ffu : 0x7ffu; }

struct SelectSmem {
    uint32_t hist[kBins];                      // this CTA's histogram of the current pass
    uint32_t acc[2 * kPassesPerTier][kSlice];  // cluster totals of the owned bins, one buffer per pass
    uint32_t xcnt[3][kCtas];                   // per-CTA counts, written by every CTA of the cluster
    uint32_t warp_tot[kWarps];
    uint32_t bcast[4];
};

// Tokens per CTA for a context of n: ceil(n / kCtas) rounded up to a multiple
// of 4 * kThreads, so every warp walks a multiple of four 32-token rounds.
__host__ __device__ __forceinline__ int chunk_tokens(int n) {
    return ((n + kCtas - 1) / kCtas + 4 * kThreads - 1) / (4 * kThreads) * (4 * kThreads);
}

// The chunk of one CTA: tokens [base, base + C) of the context [0, n), warp w
// owning [seg0, seg0 + 32 * rounds).
struct Chunk {
    int n, lo, hi;  // context length and the candidate range [lo, hi) (outside sink and window)
    int seg0, rounds;  // rounds: a multiple of 4
};

// Keys of rounds kk0 .. kk0+3 of this lane: from the warp's staged copy in
// shared memory, or straight from the scores (four loads in flight).
template <bool STAGED>
__device__ __forceinline__ void fetch4(uint32_t (&key)[4], const float *score, const uint32_t *staged,
                                       const Chunk &c, int kk0, int lane) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int kk = kk0 + u;
        const int t = c.seg0 + kk * 32 + lane;
        if (STAGED) key[u] = staged[kk * 32 + lane];
        else key[u] = t < c.n ? order_key(__ldg(score + t)) : 0u;
    }
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive block scan of one value per thread; returns the prefix, *total = sum.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, SelectSmem &sm, uint32_t *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        const uint32_t t = lane < kWarps ? sm.warp_tot[lane] : 0u;
        uint32_t s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) sm.warp_tot[lane] = s - t;  // exclusive prefix of the warp totals
        if (lane == 31) sm.bcast[0] = s;
    }
    __syncthreads();
    const uint32_t r = sm.warp_tot[wid] + x - v;
    *total = sm.bcast[0];
    __syncthreads();
    return r;
}

// Warp-uniform count per warp -> the sum over the warps before this one; *total = CTA sum.
__device__ __forceinline__ uint32_t warp_prefix(uint32_t wcount, SelectSmem &sm, uint32_t *total) {
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sm.warp_tot[warp] = wcount;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t x = sm.warp_tot[w];
        all += x;
        before += w < warp ? x : 0u;
    }
    __syncthreads();
    *total = all;
    return before;
}

// CTA-uniform value v of every CTA of the cluster -> the sum over the CTAs
// before this one; *total = cluster sum. One cluster barrier.
__device__ __forceinline__ uint32_t cluster_exchange(uint32_t v, int ph, uint32_t rank, SelectSmem &sm,
                                                     uint32_t *total) {
    if (threadIdx.x < kCtas) dsmem_st(dsmem_map(&sm.xcnt[ph][rank], threadIdx.x), v);
    cluster_sync();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int q = 0; q < kCtas; ++q) {
        const uint32_t x = sm.xcnt[ph][q];
        all += x;
        before += q < (int)rank ? x : 0u;
    }
    *total = all;
    return before;
}

__device__ __forceinline__ bool candidate(const Chunk &c, int t, const uint32_t *excl, int word, int lane) {
    return t >= c.lo && t < c.hi && !(excl && ((excl[word] >> lane) & 1u));
}

// k-th largest key (1 <= k <= candidates) among the candidates of the whole
// sequence not marked in `excl`, resolved to the bits above *res_shift: the key
// is returned with the bits below *res_shift zero, and *need = how many tokens
// whose key agrees with it above *res_shift belong to the top k. The digit
// passes stop early when the chosen bin holds exactly the keys still needed:
// then all of them are in the top k whatever their lower bits. Every CTA of the
// cluster returns the same values (they come from the cluster totals). Uses acc
// buffers buf .. buf + 2.
template <bool STAGED>
__device__ uint32_t cluster_select(const float *score, const uint32_t *staged, const Chunk &c,
                                   const uint32_t *excl, uint32_t k, SelectSmem &sm, int buf, uint32_t *need,
                                   int *res_shift) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, kr = k;
    int last_shift = 0;
    for (int p = 0; p < kPassesPerTier; ++p) {
        const int shift = pass_shift(p);
        const uint32_t him = pass_hi_mask(p), dm = pass_digit_mask(p);
        for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0u;
        __syncthreads();
        for (int kk0 = 0; kk0 < c.rounds; kk0 += 4) {
            uint32_t key[4];
            fetch4<STAGED>(key, score, staged, c, kk0, lane);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int t = c.seg0 + (kk0 + u) * 32 + lane;
                if (candidate(c, t, excl, warp * c.rounds + kk0 + u, lane) && (key[u] & him) == (prefix & him))
                    atomicAdd(&sm.hist[(key[u] >> shift) & dm], 1u);
            }
        }
        __syncthreads();
        uint32_t *acc = sm.acc[buf + p];
        for (int i = tid; i < kBins; i += kThreads) {
            const uint32_t v = sm.hist[i];
            if (v) dsmem_red_add(dsmem_map(&acc[i % kSlice], i / kSlice), v);
        }
        cluster_sync();
        // cluster totals, four bins per thread in descending digit order
        uint32_t cnt[4], own = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = kBins - 1 - (4 * tid + j);
            cnt[j] = dsmem_ld(dsmem_map(&acc[d % kSlice], d / kSlice));
            own += cnt[j];
        }
        uint32_t total;
        const uint32_t before = block_exclusive_scan(own, sm, &total);
        if (before < kr && before + own >= kr) {  // exactly one thread
            uint32_t cum = before;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (cum + cnt[j] >= kr) {
                    sm.bcast[1] = (uint32_t)(kBins - 1 - (4 * tid + j));
                    sm.bcast[2] = kr - cum;
                    sm.bcast[3] = cnt[j] == kr - cum ? 1u : 0u;  // the whole bin is needed
                    break;
                }
                cum += cnt[j];
            }
        }
        __syncthreads();
        prefix |= sm.bcast[1] << shift;
        kr = sm.bcast[2];
        const bool whole_bin = sm.bcast[3] != 0u;
        __syncthreads();
        last_shift = shift;
        if (whole_bin) break;  // the lower digits cannot change the set
    }
    *need = kr;
    *res_shift = last_shift;
    return prefix;
}

// ORs into `bits` the top-k of the candidates not already in `excl`: keys
// above `thr`, plus the first `need` tokens (by index, over the whole
// sequence) whose key equals `thr`, keys compared above bit `shift`. `excl`
// may alias `bits`: each warp reads and writes only its own words, a word's
// read before its write.
template <bool STAGED>
__device__ void mark_tier(const float *score, const uint32_t *staged, const Chunk &c, const uint32_t *excl,
                          uint32_t *bits, uint32_t thr, uint32_t need, int shift, int ph, uint32_t rank,
                          SelectSmem &sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t thr_hi = thr >> shift;
    uint32_t weq = 0;
    for (int kk0 = 0; kk0 < c.rounds; kk0 += 4) {
        uint32_t key[4];
        fetch4<STAGED>(key, score, staged, c, kk0, lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = c.seg0 + (kk0 + u) * 32 + lane;
            const bool eq = candidate(c, t, excl, warp * c.rounds + kk0 + u, lane) && (key[u] >> shift) == thr_hi;
            weq += __popc(__ballot_sync(0xffffffffu, eq));
        }
    }
    uint32_t cta_eq, eq_all;
    const uint32_t warp_before = warp_prefix(weq, sm, &cta_eq);
    const uint32_t cta_before = cluster_exchange(cta_eq, ph, rank, sm, &eq_all);
    const bool all_eq = need >= eq_all;
    uint32_t run = cta_before + warp_before;  // rank of this warp's next equal key
    for (int kk0 = 0; kk0 < c.rounds; kk0 += 4) {
        uint32_t key[4];
        fetch4<STAGED>(key, score, staged, c, kk0, lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = c.seg0 + (kk0 + u) * 32 + lane;
            const int word = warp * c.rounds + kk0 + u;
            const bool cand = candidate(c, t, excl, word, lane);
            const uint32_t hi = key[u] >> shift;
            const bool eq = cand && hi == thr_hi;
            const unsigned eqm = __ballot_sync(0xffffffffu, eq);
            const bool take = cand && (hi > thr_hi || (eq && (all_eq || run + __popc(eqm & lanemask_lt()) < need)));
            const unsigned w = __ballot_sync(0xffffffffu, take);
            if (lane == 0) bits[word] |= w;
            run += __popc(eqm);
        }
    }
}

// Copies this warp's keys of `score` into its staged segment.
__device__ __forceinline__ void stage_keys(const float *score, uint32_t *staged, const Chunk &c, int lane) {
    for (int kk0 = 0; kk0 < c.rounds; kk0 += 4) {
        uint32_t key[4];
        fetch4<false>(key, score, nullptr, c, kk0, lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) staged[(kk0 + u) * 32 + lane] = key[u];
    }
    __syncwarp();
}

template <bool STAGED>
__global__ void __cluster_dims__(kCtas, 1, 1) __launch_bounds__(kThreads, 1)
select_topk_kernel(const float *__restrict__ draft, const float *__restrict__ target, int64_t ld, int L,
                   const int32_t *__restrict__ ctx_lens, int sink, int window, int top_m, int budget,
                   int32_t *__restrict__ idx, int32_t *__restrict__ count, uint32_t *status) {
    extern __shared__ __align__(16) uint32_t dyn[];
    griddep_launch_dependents();  // as in the cluster selection: the verify call may start its set-up
    SelectSmem &sm = *reinterpret_cast<SelectSmem *>(dyn);
    uint32_t *bits = dyn + sizeof(SelectSmem) / sizeof(uint32_t);  // [C / 32] tier membership
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.x / kCtas;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    select_status_block0(ctx_lens, (int)(gridDim.x / kCtas), L, status);
    int n = L;
    if (ctx_lens) {  // a length outside [0, L] is clamped (and reported by block 0)
        n = ctx_lens[b];
        n = n < 0 ? 0 : (n > L ? L : n);
    }
    int32_t *out = idx + (int64_t)b * budget;
    if (budget >= n) {  // the whole context fits: verify in full (uniform over the cluster)
        for (int j = (int)rank * kThreads + tid; j < budget; j += kCtas * kThreads) out[j] = j < n ? j : -1;
        if (count && rank == 0 && tid == 0) count[b] = n;
        return;
    }
    const float *ds = draft + (int64_t)b * ld;
    const float *ts = target + (int64_t)b * ld;
    const int s0 = sink < n ? sink : n;
    const int w0n = window < n - s0 ? window : n - s0;
    Chunk c;
    c.n = n;
    c.lo = s0;
    c.hi = n - w0n;
    const int left = budget - s0 - w0n;
    int m = top_m < left ? top_m : left;
    if (m > c.hi - c.lo) m = c.hi - c.lo;
    const int f = left - m;
    const int C = chunk_tokens(n);
    c.rounds = C / kThreads;
    c.seg0 = (int)rank * C + warp * c.rounds * 32;
    const int nwords = kWarps * c.rounds;
    // staged keys: [C] after the bitmap, warp w's segment at w * 32 * rounds
    uint32_t *staged = bits + chunk_tokens(L) / 32 + warp * c.rounds * 32;

    for (int i = tid; i < 2 * kPassesPerTier * kSlice; i += kThreads) (&sm.acc[0][0])[i] = 0u;
    for (int i = tid; i < nwords; i += kThreads) bits[i] = 0u;
    cluster_sync();  // peers are running and their totals are zero before any remote add

    int buf = 0;
    if (m > 0) {  // tier 1: top-m by draft score
        if (STAGED) stage_keys(ds, staged, c, lane);
        uint32_t need;
        int shift;
        const uint32_t thr = cluster_select<STAGED>(ds, staged, c, nullptr, (uint32_t)m, sm, buf, &need, &shift);
        buf += kPassesPerTier;
        mark_tier<STAGED>(ds, staged, c, nullptr, bits, thr, need, shift, 0, rank, sm);
        __syncthreads();
    }
    if (f > 0) {  // tier 2: fill by target score among the rest
        if (STAGED) stage_keys(ts, staged, c, lane);
        uint32_t need;
        int shift;
        const uint32_t thr = cluster_select<STAGED>(ts, staged, c, bits, (uint32_t)f, sm, buf, &need, &shift);
        mark_tier<STAGED>(ts, staged, c, bits, bits, thr, need, shift, 1, rank, sm);
        __syncthreads();
    }
    // emission: sink u window u tiers, ascending
    uint32_t wsel = 0;
    for (int kk = 0; kk < c.rounds; ++kk) {
        const int t = c.seg0 + kk * 32 + lane;
        const bool sel = t < n && (t < c.lo || t >= c.hi || ((bits[warp * c.rounds + kk] >> lane) & 1u));
        wsel += __popc(__ballot_sync(0xffffffffu, sel));
    }
    uint32_t cta_sel, all_sel;
    const uint32_t warp_before = warp_prefix(wsel, sm, &cta_sel);
    const uint32_t cta_before = cluster_exchange(cta_sel, 2, rank, sm, &all_sel);
    uint32_t pos = cta_before + warp_before;
    for (int kk = 0; kk < c.rounds; ++kk) {
        const int t = c.seg0 + kk * 32 + lane;
        const bool sel = t < n && (t < c.lo || t >= c.hi || ((bits[warp * c.rounds + kk] >> lane) & 1u));
        const unsigned msk = __ballot_sync(0xffffffffu, sel);
        const uint32_t p = pos + __popc(msk & lanemask_lt());
        if (sel && p < (uint32_t)budget) out[p] = t;
        pos += __popc(msk);
    }
    for (int j = (int)all_sel + (int)rank * kThreads + tid; j < budget; j += kCtas * kThreads) out[j] = -1;
    if (count && rank == 0 && tid == 0) count[b] = (int32_t)(all_sel < (uint32_t)budget ? all_sel : budget);
}

}  // namespace

cudaError_t launch_select_topk(const float *ds, const float *ts, int64_t ld, int B, int L,
                               const int32_t *ctx_lens, int sink, int window, int top_m,
                               int budget, int32_t *idx, int32_t *count, uint32_t *status,
                               cudaStream_t s) {
    if (B == 0) return cudaSuccess;
    cudaError_t sub_err;
    // up to 131072 tokens: a 4- or 8-CTA cluster per sequence with the keys in registers
    if (launch_select_cluster_reg(ds, ts, ld, B, L, ctx_lens, sink, window, top_m, budget, idx, count, status, s,
                                  &sub_err))
        return sub_err;
    const size_t C = (size_t)chunk_tokens(L);
    const size_t base = sizeof(SelectSmem) + C / 32 * sizeof(uint32_t);
    const size_t staged = base + C * sizeof(uint32_t);
    // keys staged in shared memory while the chunk fits (L up to about 360k), else read from L2 each pass
    const bool use_staged = staged <= 200 * 1024;
    const size_t smem = use_staged ? staged : base;
    auto kern = use_staged ? select_topk_kernel<true> : select_topk_kernel<false>;
    // attributes for the largest shared memory either variant can need, set once per device
    static PerDeviceOnce attr_once;
    const cudaError_t attr = once_per_device(attr_once, [] {
        cudaError_t e = kernel_attributes(select_topk_kernel<true>, 200 * 1024);
        if (e == cudaSuccess) {
            const size_t Cmax = (size_t)chunk_tokens(kMaxL);
            e = kernel_attributes(select_topk_kernel<false>, (int)(sizeof(SelectSmem) + Cmax / 32 * sizeof(uint32_t)));
        }
        return e;
    });
    if (attr != cudaSuccess) return attr;
    kern<<<(unsigned)B * kCtas, kThreads, smem, s>>>(ds, ts, ld, L, ctx_lens, sink, window, top_m, budget, idx,
                                                     count, status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace specverify
