// Internal helpers shared by the CUDA translation units of libspecverify.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <stdint.h>

#include "../../include/specverify.h"

namespace specverify {

constexpr int kHeadDim = 128;
constexpr size_t kHeaderBytes = 256;  // status word + reserved, at the start of every workspace

// Status word handling (device side). Never traps: the most severe code wins.
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start before the previous kernel on the
// stream ends; griddepcontrol.wait blocks until that kernel has completed and
// its writes are visible. launch_dependents lets the dependent grid be
// scheduled once every CTA of this grid has issued it (or exited).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void flag_status(uint32_t *status, uint32_t code) {
    if (status) atomicMax(status, code);
}

// Status word of a selection call, written whole by block 0 of the grid (the other
// blocks never write it, so no clearing memset has to come first): SPEC_ERR_BAD_INPUT
// if a context length of the B sequences is outside [0, L], else SPEC_OK. Every
// thread of block 0 calls it.
__device__ __forceinline__ void select_status_block0(const int32_t *ctx_lens, int B, int L, uint32_t *status) {
    if (blockIdx.x != 0) return;
    int bad = 0;
    if (ctx_lens)
        for (int b = threadIdx.x; b < B; b += blockDim.x) bad |= ctx_lens[b] < 0 || ctx_lens[b] > L;
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0 && status) *status = bad ? (uint32_t)SPEC_ERR_BAD_INPUT : (uint32_t)SPEC_OK;
}

// ---------------------------------------------------------------------------
// Split-KV work plan.
//
// The cache part is cut into "units" (b, h_kv, row group) of up to BM query
// rows each, every unit into tiles of `tile` KV positions. The units' tiles
// are laid end to end (unit-major) and cut into `ctas` contiguous ranges, one
// per CTA, so every SM gets about the same work whatever B, Hkv and L are.
// CTA c covers global tiles [start(c), start(c+1)); for each unit u its range
// touches, it writes one normalised partial (o, lse) into slot c + u. Along
// the range both c and u only grow, so c + u is unique per (c, u) pair and the
// slots number ctas + units - 1.
//
// Uniform plans give every CTA q or q + 1 tiles. Balanced plans (the tcgen05
// kernel) charge a CTA for each extra unit its range enters, since starting a
// unit costs about kUnitSwitchTiles tiles of time (Q reload, pipeline refill,
// a partial written out), and cut the ranges so that tiles plus those charges
// are even; their starts are kept in the plan.
constexpr int kPlanMaxCtas = 512;
constexpr int kUnitSwitchTiles = 4;

struct SplitPlan {
    int BM;             // query rows per unit (rows of one CTA's tile)
    int tile;           // KV positions per tile
    int row_groups;     // ceil(G*N / BM)
    int bh;             // B * Hkv
    int units;          // B * Hkv * row_groups, row group first (plan_unit)
    int tiles_per_unit; // ceil(L_eff / tile), at least 1
    int ctas;           // CTAs of the cache kernel
    int64_t total;      // units * tiles_per_unit
    int64_t slots;      // (ctas + units - 1) * pipes
    int pipes;          // partial slots per (cta, unit) pair
    int slot_rows;      // rows per slot
    int split_tiles;    // 1: the pipes cover alternate tiles of the same rows (both slots per row);
                        // 0: pipe h covers rows [h*slot_rows, (h+1)*slot_rows) of the unit
    int q, rem;         // uniform plans: total = q * ctas + rem
    int uniform;        // 1: q / rem arithmetic; 0: the starts below
    int32_t starts[kPlanMaxCtas + 1];  // balanced plans: start(c), start(ctas) = total
};

// Uniform: CTA c covers q or q+1 tiles, the first `rem` CTAs taking q+1 (q = total
// / ctas, rem = total % ctas). All in 32-bit arithmetic (total < 2^31 is checked on
// the host).
__host__ __device__ __forceinline__ int64_t plan_start(const SplitPlan &p, int64_t c) {
    const int ci = (int)c;
    if (!p.uniform) return p.starts[ci];
    return (int64_t)ci * p.q + (ci < p.rem ? ci : p.rem);
}
// The CTA whose range holds global tile g (0 <= g < total).
__host__ __device__ __forceinline__ int64_t plan_cta_of(const SplitPlan &p, int64_t g) {
    const int gi = (int)g;
    if (!p.uniform) {  // the last c with starts[c] <= g; empty ranges only follow the last tile
        int lo = 0, hi = p.ctas - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.starts[mid] <= gi) lo = mid;
            else hi = mid - 1;
        }
        return lo;
    }
    const int big = p.rem * (p.q + 1);
    return gi < big ? gi / (p.q + 1) : p.rem + (gi - big) / p.q;
}

// Greedy cut of the tiles into contiguous ranges whose cost (tiles plus
// kUnitSwitchTiles for every unit a range enters after its first) stays within
// `budget`; returns the number of ranges used and fills starts[0..used).
inline int plan_cut(int64_t total, int tiles_per_unit, int64_t budget, int max_ranges, int32_t *starts) {
    int64_t g = 0;
    int used = 0;
    while (g < total) {
        if (used == max_ranges) return max_ranges + 1;  // does not fit
        starts[used++] = (int32_t)g;
        int64_t cost = 0, pos = g;
        while (pos < total) {
            const int64_t avail = tiles_per_unit - pos % tiles_per_unit;
            const int64_t extra = pos == g ? 0 : kUnitSwitchTiles;
            const int64_t take = std::min<int64_t>(avail, budget - cost - extra);
            if (take <= 0) break;
            cost += extra + take;
            pos += take;
            if (take < avail) break;
        }
        if (pos == g) return max_ranges + 1;  // budget below one tile
        g = pos;
    }
    return used;
}

// Turns a uniform plan into a balanced one: the smallest budget whose greedy cut
// fits the plan's CTAs (trailing CTAs get empty ranges at the end).
inline void plan_balance(SplitPlan &p) {
    if (p.ctas > kPlanMaxCtas || p.total < 2 * (int64_t)p.ctas) return;  // too few tiles to matter
    int64_t lo = (p.total + p.ctas - 1) / p.ctas, hi = lo + 2 * kUnitSwitchTiles + 2;
    while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (plan_cut(p.total, p.tiles_per_unit, mid, p.ctas, p.starts) <= p.ctas) hi = mid;
        else lo = mid + 1;
    }
    const int used = plan_cut(p.total, p.tiles_per_unit, lo, p.ctas, p.starts);
    if (used > p.ctas) return;  // keep the uniform plan
    for (int c = used; c <= p.ctas; ++c) p.starts[c] = (int32_t)p.total;
    p.uniform = 0;
}

inline SplitPlan make_plan(int B, int N, int Hq, int Hkv, int L_eff, int BM, int tile, int max_ctas) {
    SplitPlan p;
    const int G = Hq / Hkv;
    p.BM = BM;
    p.tile = tile;
    p.row_groups = (G * N + BM - 1) / BM;
    p.bh = B * Hkv;
    p.units = B * Hkv * p.row_groups;
    p.tiles_per_unit = L_eff > 0 ? (L_eff + tile - 1) / tile : 1;
    p.total = (int64_t)p.units * p.tiles_per_unit;
    p.ctas = (int)(p.total < max_ctas ? p.total : max_ctas);
    if (p.ctas > kPlanMaxCtas) p.ctas = kPlanMaxCtas;
    if (p.ctas < 1) p.ctas = 1;
    p.uniform = 1;
    p.q = (int)(p.total / p.ctas);
    p.rem = (int)(p.total % p.ctas);
    p.pipes = 1;
    p.slot_rows = BM;
    p.split_tiles = 0;
    p.slots = (int64_t)p.ctas + p.units - 1;
    return p;
}

// Plan of the tensor-core cache kernel: units of 256 query rows (128 when G*N <= 128),
// 128-token tiles, one CTA per SM, two pipes of 128 rows each writing their own slots.
// With more than one row group per (b, h_kv), each row group gets its own block of CTAs and
// every block the same uniform cut (the blocks then read the same tiles in step, from L2 after
// the first). Otherwise dense plans are balanced against the cost of entering a unit, and
// sparse ones (gathered tiles, where a unit switch costs less than the SMs a balanced cut
// leaves idle) stay uniform.
inline SplitPlan make_plan_tc(int B, int N, int Hq, int Hkv, int L_eff, int sms, bool sparse) {
    const int M = (Hq / Hkv) * N;
    SplitPlan p = make_plan(B, N, Hq, Hkv, L_eff, M > 128 ? 256 : 128, 128, sms);
    p.pipes = 2;
    p.slot_rows = 128;
    p.split_tiles = M <= 128 ? 1 : 0;
    p.slots = ((int64_t)p.ctas + p.units - 1) * 2;
    if (p.row_groups > 1 && p.ctas >= p.row_groups && p.ctas <= kPlanMaxCtas) {
        // one block of CTAs per row group (the CTAs the row groups do not divide stay idle), the
        // same uniform cut in every block: the CTAs of one head's row groups walk the same tiles
        // at the same time. Dense and sparse calls take the same CTA count (one workspace size).
        const int per = p.ctas / p.row_groups;
        p.ctas = per * p.row_groups;
        p.slots = ((int64_t)p.ctas + p.units - 1) * 2;
        const int64_t blk = p.total / p.row_groups;
        for (int c = 0; c < p.ctas; ++c) {
            const int r = c / per, i = c % per;
            const int64_t q = blk / per, rem = blk % per;
            p.starts[c] = (int32_t)(r * blk + i * q + (i < rem ? i : rem));
        }
        p.starts[p.ctas] = (int32_t)p.total;
        p.uniform = 0;
    } else if (!sparse) {
        plan_balance(p);
    }
    return p;
}

// Unit numbering: u = rg * B * Hkv + b * Hkv + h_kv. The row groups of one (b, h_kv) lie B * Hkv
// units apart, so that with one block of CTAs per row group (make_plan_tc) the CTAs that cover
// them stream the same K/V tiles at the same time and share them through L2.
__host__ __device__ __forceinline__ int64_t plan_unit(const SplitPlan &p, int Hkv, int b, int hk, int rg) {
    return (int64_t)rg * p.bh + (int64_t)b * Hkv + hk;
}
__host__ __device__ __forceinline__ void plan_unit_coords(const SplitPlan &p, int Hkv, int64_t u, int &b, int &hk,
                                                          int &rg) {
    rg = (int)(u / p.bh);
    const int bh = (int)(u - (int64_t)rg * p.bh);
    b = bh / Hkv;
    hk = bh - b * Hkv;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace carve-up for the verify calls: header | o partials | lse partials.
inline size_t plan_o_bytes(const SplitPlan &p, int d) {
    return align_up((size_t)p.slots * p.slot_rows * d * sizeof(float), 256);
}
inline size_t plan_workspace_bytes(const SplitPlan &p, int d) {
    return kHeaderBytes + plan_o_bytes(p, d) + align_up((size_t)p.slots * p.slot_rows * sizeof(float), 256);
}

struct VerifyArgs {
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_cache;
    const __nv_bfloat16 *v_cache;
    int64_t sb, sh, st;  // cache strides in elements
    const __nv_bfloat16 *k_draft;
    const __nv_bfloat16 *v_draft;
    const int32_t *parent;
    const int32_t *ctx_lens;
    const int32_t *idx;  // sparse only
    int budget;          // sparse only
    int B, N, Hq, Hkv, G, L;
    float scale;
    float *out;
    float *lse;
    uint32_t *status;
    float *o_part;    // [slots][BM][d]
    float *lse_part;  // [slots][BM]
    // paged cache (table != nullptr): token t of sequence b is row t % block_size of pool
    // block table[b * table_ld + t / block_size]; sb is then the pool's block stride
    const int32_t *table;
    int64_t table_ld;
    int block_size;
    int64_t num_blocks;
    int idx_resolved;  // sparse: idx holds validated pool rows (entry >= 0: used), see paged.cu
    int out_bf16;      // out is bf16 [B, N, Hq, d] (rounded to nearest even) instead of fp32
    // fp8 cache: k_cache / v_cache hold E4M3 codes (one byte an element, element strides);
    // the value is the code's number times k_scale / v_scale [b * Hkv + h] (fp32)
    int kv_fp8;
    const float *k_scale;
    const float *v_scale;
};

// Two E4M3 codes (the lower byte first) -> the bf16 pair of the same numbers (exact: E4M3 ->
// f16 is exact, and so is f16 -> f32 -> bf16 for every E4M3 number).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    const __nv_bfloat162 v = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Sixteen E4M3 codes (byte j of the uint4 = element j) -> sixteen bf16 of the same numbers,
// elements 0-7 in lo and 8-15 in hi (exact for every code, NaN included).
__device__ __forceinline__ void e4m3x16_to_bf16x16(const uint4 codes, uint4 &lo, uint4 &hi) {
    lo.x = e4m3x2_to_bf16x2(codes.x & 0xffffu);
    lo.y = e4m3x2_to_bf16x2(codes.x >> 16);
    lo.z = e4m3x2_to_bf16x2(codes.y & 0xffffu);
    lo.w = e4m3x2_to_bf16x2(codes.y >> 16);
    hi.x = e4m3x2_to_bf16x2(codes.z & 0xffffu);
    hi.y = e4m3x2_to_bf16x2(codes.z >> 16);
    hi.z = e4m3x2_to_bf16x2(codes.w & 0xffffu);
    hi.w = e4m3x2_to_bf16x2(codes.w >> 16);
}

// Context length of sequence b, clamped to [0, L]; out-of-range values flag bad input.
__device__ __forceinline__ int context_len(const VerifyArgs &a, int b) {
    if (!a.ctx_lens) return a.L;
    int n = __ldg(a.ctx_lens + b);
    if (n < 0 || n > a.L) {
        flag_status(a.status, SPEC_ERR_BAD_INPUT);
        n = n < 0 ? 0 : a.L;
    }
    return n;
}

// Token behind index slot j of sequence b in sparse mode, or -1 when the slot
// is unused: past the budget, -1 padding, outside [0, n), or not above the
// previous slot's token. Unused entries other than -1 padding are bad input.
__device__ __forceinline__ int sparse_token(const VerifyArgs &a, int b, int n, int j, bool report) {
    if (j >= a.budget) return -1;
    const int32_t *ib = a.idx + (int64_t)b * a.budget;
    const int t = __ldg(ib + j);
    if (a.idx_resolved) return t >= 0 ? t : -1;  // checked (and reported) when it was resolved
    const bool ok = t >= 0 && t < n && (j == 0 || t > __ldg(ib + j - 1));
    if (!ok && t != -1 && report) flag_status(a.status, SPEC_ERR_BAD_INPUT);
    return ok ? t : -1;
}

// The same rule split in two, so that the loads can be issued a tile early:
// the raw entries of slot j and of slot j - 1 ...
struct IdxPair {
    int cur, prev;
};
__device__ __forceinline__ IdxPair sparse_raw(const VerifyArgs &a, int b, int j) {
    IdxPair r{-1, -1};
    if (j < a.budget) {
        const int32_t *ib = a.idx + (int64_t)b * a.budget;
        r.cur = __ldg(ib + j);
        r.prev = j > 0 ? __ldg(ib + j - 1) : -1;
    }
    return r;
}
// ... then the token (or -1) once they have arrived.
__device__ __forceinline__ int sparse_resolve(const VerifyArgs &a, IdxPair r, int j, int n, bool report) {
    if (j >= a.budget) return -1;
    if (a.idx_resolved) return r.cur >= 0 ? r.cur : -1;  // checked (and reported) when it was resolved
    const bool ok = r.cur >= 0 && r.cur < n && (j == 0 || r.cur > r.prev);
    if (!ok && r.cur != -1 && report) flag_status(a.status, SPEC_ERR_BAD_INPUT);
    return ok ? r.cur : -1;
}

// Element offset of the cache row of token t (sequence b, KV head hk), or -1 when the
// row does not exist (paged: its block entry is outside the pool, recorded as bad input
// when `report`).
__device__ __forceinline__ int64_t cache_row_offset(const VerifyArgs &a, int b, int hk, int t, bool report) {
    if (!a.table) return (int64_t)b * a.sb + (int64_t)hk * a.sh + (int64_t)t * a.st;
    const int64_t blk = __ldg(a.table + (int64_t)b * a.table_ld + t / a.block_size);
    if (blk < 0 || blk >= a.num_blocks) {
        if (report) flag_status(a.status, SPEC_ERR_BAD_INPUT);
        return -1;
    }
    return blk * a.sb + (int64_t)hk * a.sh + (int64_t)(t % a.block_size) * a.st;
}

// Tiling of the mma.sync cache kernel (query rows per unit, tokens per tile).
int mma_rows_per_unit();
int mma_tile_tokens();

// Kernel attributes: the dynamic shared memory a kernel may use beyond the
// 48 KiB default. The setting belongs to the current device's context, so the
// launchers make it once per device, with that device current (once_per_device).
template <class Kernel>
cudaError_t kernel_attributes(Kernel kern, int dyn_smem) {
    if (dyn_smem <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
}

// Per-device one-time set-up: f() runs once for each device index, the first time
// a launcher runs with that device current, and its result is kept for that device.
constexpr int kMaxDevices = 64;
struct PerDeviceOnce {
    std::once_flag once[kMaxDevices];
    cudaError_t err[kMaxDevices] = {};
};
template <class F>
cudaError_t once_per_device(PerDeviceOnce &st, F f) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return cudaErrorInvalidDevice;
    }
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(st.once[dev], [&] { st.err[dev] = f(); });
    return st.err[dev];
}

// Records a failed CUDA call for spec_last_cuda_error() (this host thread) and
// returns SPEC_ERR_CUDA.
int cuda_failure(cudaError_t e);

// Host-side launchers (one per translation unit).
cudaError_t launch_cache_attn_mma(const VerifyArgs &a, const SplitPlan &p, bool sparse,
                                  cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1);
cudaError_t launch_merge_tree(const VerifyArgs &a, const SplitPlan &p, cudaStream_t s);
bool tc_supported(const VerifyArgs &a);
cudaError_t launch_cache_attn_tc(const VerifyArgs &a, const SplitPlan &p, cudaStream_t s, cudaEvent_t ev0,
                                 cudaEvent_t ev1, bool *launched);
cudaError_t launch_lse_merge2(const float *o_a, const float *lse_a, const float *o_b,
                              const float *lse_b, float *out, float *lse_out, int64_t rows, int d,
                              cudaStream_t s);
bool launch_select_cluster_reg(const float *ds, const float *ts, int64_t ld, int B, int L, const int32_t *ctx_lens,
                               int sink, int window, int top_m, int budget, int32_t *idx, int32_t *count,
                               uint32_t *status, cudaStream_t s, cudaError_t *err);
// Paged sparse calls: idx [B, budget] -> the pool rows of its used entries (-1 otherwise),
// see paged.cu.
cudaError_t launch_resolve_paged_idx(const VerifyArgs &a, int32_t *rows_out, cudaStream_t s);
cudaError_t launch_select_topk(const float *ds, const float *ts, int64_t ld, int B, int L,
                               const int32_t *ctx_lens, int sink, int window, int top_m,
                               int budget, int32_t *idx, int32_t *count, uint32_t *status,
                               cudaStream_t s);

// Importance scores on the tensor core; false (nothing launched) for shapes it does not take.
bool launch_importance_tc(const __nv_bfloat16 *q, const __nv_bfloat16 *k_cache, int64_t sb, int64_t sh, int64_t st,
                          const float *lse, const int32_t *heads, int nh, int B, int N, int Hq, int Hkv, int L,
                          const int32_t *ctx_lens, float scale, float *score, int64_t ld, int32_t *status,
                          int sms, cudaStream_t s, cudaError_t *err);

// Kernel-launch counter (per host thread), see spec_kernel_launches().
void count_launches(int n);

}  // namespace specverify
