// Cache part of verification attention on the 5th-generation tensor core
// (tcgen05 + TMEM + TMA), for the full cache (dense) and for the selected
// index set (sparse).
//
// What it computes is the same normalised split-KV partial as the warp-level
// kernel: for every unit (b, h_kv, group of query rows: the query heads of
// h_kv times the draft nodes, packed together) and every range of 128-token
// KV tiles of the split plan, softmax(scale * Q K^T) V over the cache tokens of
// that range, with no mask but "token < n" (the cache part needs none, LongSpec
// section 2.C). Partials are merged by log-sum-exp with the tree part later.
//
// Sparse (Dustin, "Workflow di Verifica"): tile t holds index slots
// [128 t, 128 t + 128) of idx[b]; a slot whose entry is unused (padding, out of
// the context, not ascending) is a zero row in shared memory and a masked
// column of S.
//
// Design (one CTA per SM, persistent over its balanced range of tiles):
//   warp 8      producer: the unit's Q rows by TMA (3-D map over [B*N, Hq, d],
//               so query heads x draft nodes land as consecutive rows), then a
//               5-slot ring of K and V tiles, 128-byte swizzle. Dense: TMA
//               (4-D map over [B, Hkv, L, d] with the caller's strides). Sparse:
//               the whole warp gathers the rows with 16-byte cp.async into the
//               same swizzled layout, two rows of 256 bytes per instruction;
//               every lane then arms an arrival on the slot's barrier that fires
//               when its copies have landed (32 arrivals complete the slot), so
//               the producer never waits for its own copies. The MMA warp fences
//               the async proxy after the wait, before the tensor core reads the
//               slot.
//   warp 9      MMA issuer (one thread): S_h = Q_h K^T (A and B from shared
//               memory) and O_h += P_h V (P from TMEM, V MN-major from shared
//               memory), fp32 accumulators in TMEM, tcgen05.commit to mbarriers.
//   warps 0-3,  softmax for pipe 0 / pipe 1: thread i owns TMEM lane i = query
//   warps 4-7   row i; loads its S row, takes the online max in base 2, writes
//               P = 2^(x - m) as bf16 back over S for the PV MMA. The O
//               accumulator is only rescaled when the running max grows by more
//               than 2^8 (exact: l and O always share the same reference max).
// Two pipes ping-pong on the tensor core. With more than 128 query rows per
// unit the pipes take rows 0-127 and 128-255 of every tile; with at most 128
// rows they take alternate tiles of the same rows and each writes its own
// partial. TMEM (512 columns): S_0, S_1, O_0, O_1, 128 columns each.
// Every wait on an mbarrier is bounded; a wait that gives up records
// SPEC_ERR_TIMEOUT, the CTA drains its in-flight copies and MMAs, frees TMEM
// and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace specverify {

namespace {

using namespace sm100;

constexpr int D = kHeadDim;
constexpr int T = 128;                // tokens per tile
constexpr int RING = 5;               // K/V slots
constexpr int SLOT_BYTES = T * D * 2; // 32 KiB: one K or V tile
constexpr int HALF_BYTES = SLOT_BYTES / 2;
constexpr int Q_BYTES = 256 * D * 2;  // 64 KiB
constexpr int SMEM_RING = Q_BYTES;
constexpr int SMEM_BAR = SMEM_RING + RING * SLOT_BYTES;  // 229376
constexpr int SMEM_BYTES = SMEM_BAR + 256 + 1024;        // + barriers + alignment slack
constexpr int THREADS = 320;
constexpr int WARP_PRODUCER = 8, WARP_MMA = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 128, true);
constexpr long long WAIT_LIMIT_CYCLES = 4000000000LL;  // ~2 s

struct Bars {
    uint64_t q_full[2], q_empty[2];  // Q buffers (two only when the pipes share <= 128 rows)
    uint64_t kv_full[RING], kv_empty[RING];
    uint64_t s_full[2], p_full[2], o_done[2], o_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block fits its reservation");
static_assert(SMEM_BYTES <= 232448, "dynamic shared memory fits one CTA per SM");

struct TcParams {
    int split_tiles;  // 1: pipes take alternate tiles of the same <=128 rows
    int M;            // G * N query rows per (b, h_kv)
};

// Bounded wait: false (and the abort flag set) if the phase does not complete in time.
__device__ __forceinline__ bool wait_bar(Bars &bs, uint64_t *bar, uint32_t parity, uint32_t *status) {
    if (*(volatile uint32_t *)&bs.abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000)) return true;  // sleeps in hardware, no spinning
        if (*(volatile uint32_t *)&bs.abort) return false;
        if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
            atomicExch(&bs.abort, 1u);
            flag_status(status, SPEC_ERR_TIMEOUT);
            return false;
        }
    }
}

// Wait used while draining after an abort: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity) && clock64() - t0 < WAIT_LIMIT_CYCLES) {
    }
}

// Segment of the CTA's tile range inside one unit.
struct Seg {
    int64_t u;
    int tb, te;  // tiles [tb, te) of the unit
    int b, hk, rg;
    int cnt[2];  // tiles per pipe
};

__device__ __forceinline__ void seg_decode(const VerifyArgs &a, const SplitPlan &p, int split_tiles, int64_t u,
                                           int64_t g0, int64_t g1, Seg &s) {
    const int64_t ub = u * p.tiles_per_unit;
    s.u = u;
    s.tb = (int)((g0 > ub ? g0 : ub) - ub);
    s.te = (int)((g1 < ub + p.tiles_per_unit ? g1 : ub + p.tiles_per_unit) - ub);
    s.rg = (int)(u % p.row_groups);
    s.hk = (int)((u / p.row_groups) % a.Hkv);
    s.b = (int)(u / ((int64_t)p.row_groups * a.Hkv));
    const int nt = s.te - s.tb;
    s.cnt[0] = split_tiles ? (nt + 1) / 2 : nt;
    s.cnt[1] = split_tiles ? nt / 2 : nt;
}
__device__ __forceinline__ int seg_tile(const Seg &s, int split_tiles, int h, int i) {
    return split_tiles ? s.tb + 2 * i + h : s.tb + i;
}

// Q buffers: with more than 128 rows per unit the pipes read rows 0-127 and
// 128-255 of one 64 KiB buffer; with at most 128 they share rows 0-127, and the
// two 32 KiB halves serve alternate units, so that the next unit's Q loads while
// the current one is still in use. Segment seg_i uses buffer seg_i % nqb for the
// (seg_i / nqb)-th time.
__device__ __forceinline__ void q_buffer(int split_tiles, int seg_i, int &qb, uint32_t &use) {
    const int nqb = split_tiles ? 2 : 1;
    qb = seg_i % nqb;
    use = (uint32_t)(seg_i / nqb);
}

// TMA of the unit's Q rows into buffer qb (one thread).
__device__ __forceinline__ void load_q(const CUtensorMap *tm_q, uint8_t *sQ, uint64_t *bar, int split_tiles, int qb,
                                       const Seg &s, int BM, int G, int N) {
    const int npipe_q = split_tiles ? 1 : 2;
    mbar_arrive_expect_tx(bar, npipe_q * 2 * 16384);
    for (int h = 0; h < npipe_q; ++h) {
        const int n0 = (s.rg * BM + 128 * h) / G;
        const int half = split_tiles ? qb : h;  // 16 KiB row block inside each 32 KiB column half
        for (int kh = 0; kh < 2; ++kh)
            tma_load_3d(sQ + kh * 32768 + half * 16384, tm_q, bar, kh * 64, s.hk * G, s.b * N + n0);
    }
}

// Drain (one thread): the Q loads still in flight, the last of each buffer.
__device__ __forceinline__ void drain_q(Bars &bs, int split_tiles, int q_loads) {
    const int nqb = split_tiles ? 2 : 1;
    for (int i = q_loads > nqb ? q_loads - nqb : 0; i < q_loads; ++i) {
        int qb;
        uint32_t quse;
        q_buffer(split_tiles, i, qb, quse);
        drain_wait(&bs.q_full[qb], quse & 1);
    }
}

template <bool SPARSE>
__global__ void __launch_bounds__(THREADS, 1)
cache_attn_tc_kernel(const VerifyArgs a, const SplitPlan p, const TcParams tp,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    griddep_launch_dependents();  // the merge may be scheduled as this grid's CTAs drain
    // the 128-byte swizzle needs 1024-byte aligned tiles; SMEM_BYTES has 1 KiB of slack for it
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *sQ = smem;
    uint8_t *sRing = smem + SMEM_RING;
    Bars &bs = *reinterpret_cast<Bars *>(smem + SMEM_BAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split_tiles = tp.split_tiles;
    const int BM = p.BM;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bs.q_full[i], 1);
            mbar_init(&bs.q_empty[i], 1);
        }
        for (int i = 0; i < RING; ++i) {
            mbar_init(&bs.kv_full[i], SPARSE ? 32 : 1);  // sparse: one arrival per gathering lane
            mbar_init(&bs.kv_empty[i], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bs.s_full[h], 1);
            mbar_init(&bs.p_full[h], 4);
            mbar_init(&bs.o_done[h], 1);
            mbar_init(&bs.o_empty[h], 4);
        }
        mbar_init(&bs.mma_done, 1);
        bs.abort = 0;
        fence_mbar_init();
    }
    if (warp == WARP_PRODUCER) {
        tmem_alloc(&bs.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bs.tmem_base;

    const int64_t g0 = plan_start(p, blockIdx.x), g1 = plan_start(p, blockIdx.x + 1);
    const int64_t u_first = g0 / p.tiles_per_unit;

    if (SPARSE && warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ gather producer
        if (lane == 0) tma_prefetch_desc(&tm_q);
        int64_t item = 0;  // K/V tiles issued (same in all lanes)
        int seg_i = 0;
        bool ok = true;
        // Copy pattern: in step v (0..31), lane l copies 16-byte chunk c = l & 7 of both
        // 128-byte halves of tile row r = 4v + (l >> 3): every instruction moves four whole
        // 128-byte lines. Row r lands at r * 128 bytes of each half, its chunks permuted by
        // the 128-byte swizzle (c ^ (r & 7), and r & 7 = 4 (v & 1) + (l >> 3)).
        const int rs = lane >> 3, c8 = lane & 7;
        const uint32_t xo0 = (uint32_t)((c8 ^ rs) << 4), xo1 = (uint32_t)((c8 ^ (4 + rs)) << 4);
        const int64_t row_bytes = a.st * 2;
        for (int64_t u = u_first; ok && u * p.tiles_per_unit < g1; ++u, ++seg_i) {
            Seg s;
            seg_decode(a, p, split_tiles, u, g0, g1, s);
            {  // the unit's Q rows, as in the dense producer
                int qb;
                uint32_t quse;
                q_buffer(split_tiles, seg_i, qb, quse);
                if (quse > 0 &&
                    !(ok = __all_sync(0xffffffffu, wait_bar(bs, &bs.q_empty[qb], (quse - 1) & 1, a.status))))
                    break;
                if (lane == 0) load_q(&tm_q, sQ, &bs.q_full[qb], split_tiles, qb, s, BM, a.G, a.N);
            }
            const int n_ctx = context_len(a, s.b);
            const char *kbase = reinterpret_cast<const char *>(a.k_cache + s.b * a.sb + s.hk * a.sh);
            const char *vbase = reinterpret_cast<const char *>(a.v_cache + s.b * a.sb + s.hk * a.sh);
            IdxPair raw[4];  // index entries of the next tile, loaded one tile ahead
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) raw[u4] = sparse_raw(a, s.b, s.tb * T + 32 * u4 + lane);
            for (int t = s.tb; ok && t < s.te; ++t) {
                int tok[4];  // token of index slot 128 t + 32 u + lane, or -1
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) tok[u4] = sparse_resolve(a, raw[u4], t * T + 32 * u4 + lane, n_ctx, true);
                if (t + 1 < s.te) {
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) raw[u4] = sparse_raw(a, s.b, (t + 1) * T + 32 * u4 + lane);
                }
                int tkr[32];  // token of tile row 4v + rs, or -1
#pragma unroll
                for (int v = 0; v < 32; ++v) tkr[v] = __shfl_sync(0xffffffffu, tok[v >> 3], (4 * v + rs) & 31);
                for (int kv = 0; kv < 2; ++kv) {
                    const int slot = (int)(item % RING);
                    const int64_t use = item / RING;
                    if (use > 0 &&
                        !(ok = __all_sync(0xffffffffu, wait_bar(bs, &bs.kv_empty[slot], (uint32_t)((use - 1) & 1), a.status))))
                        break;
                    const char *base = (kv ? vbase : kbase) + c8 * 16;
                    const uint32_t d0 = smem_u32(sRing + slot * SLOT_BYTES) + (uint32_t)rs * 128u;
#pragma unroll
                    for (int v = 0; v < 32; ++v) {
                        const bool ok_row = tkr[v] >= 0;
                        const char *src = ok_row ? base + (int64_t)tkr[v] * row_bytes : reinterpret_cast<const char *>(a.q);
                        const uint32_t d = d0 + (uint32_t)v * 512u + ((v & 1) ? xo1 : xo0);
                        cp_async16_zfill(d, src, ok_row);                    // columns 0-63
                        cp_async16_zfill(d + HALF_BYTES, src + 128, ok_row);  // columns 64-127
                    }
                    cp_async_mbar_arrive_noinc(&bs.kv_full[slot]);
                    ++item;
                }
            }
        }
        cp_async_wait_all();  // the drain: no copy is left in flight
        if (lane == 0) drain_q(bs, split_tiles, seg_i);
        __syncwarp();
    } else if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int64_t item = 0;  // K/V tiles loaded so far (K and V count separately)
            int q_loads = 0;
            bool ok = true;
            for (int64_t u = u_first; ok && u * p.tiles_per_unit < g1; ++u, ++q_loads) {
                Seg s;
                seg_decode(a, p, split_tiles, u, g0, g1, s);
                // the unit's Q rows, once the QK MMAs of the unit that last used the buffer are
                // done with it (the previous unit, or with two buffers the one before)
                int qb;
                uint32_t quse;
                q_buffer(split_tiles, q_loads, qb, quse);
                if (quse > 0 && !(ok = wait_bar(bs, &bs.q_empty[qb], (quse - 1) & 1, a.status))) break;
                load_q(&tm_q, sQ, &bs.q_full[qb], split_tiles, qb, s, BM, a.G, a.N);
                // K and V tiles in order: tile tb: K, V; tile tb+1: K, V; ...
                for (int t = s.tb; t < s.te; ++t) {
                    for (int kv = 0; kv < 2; ++kv, ++item) {
                        const int slot = (int)(item % RING);
                        const int64_t use = item / RING;
                        if (use > 0 && !(ok = wait_bar(bs, &bs.kv_empty[slot], (uint32_t)((use - 1) & 1), a.status)))
                            break;
                        uint8_t *dst = sRing + slot * SLOT_BYTES;
                        mbar_arrive_expect_tx(&bs.kv_full[slot], SLOT_BYTES);
                        const CUtensorMap *m = kv == 0 ? &tm_k : &tm_v;
                        tma_load_4d(dst, m, &bs.kv_full[slot], 0, t * T, s.hk, s.b);
                        tma_load_4d(dst + HALF_BYTES, m, &bs.kv_full[slot], 64, t * T, s.hk, s.b);
                    }
                    if (!ok) break;
                }
            }
            // drain: wait for the last copies still in flight (consumed ones return at once)
            const int64_t first = item > RING ? item - RING : 0;
            for (int64_t n = first; n < item; ++n) drain_wait(&bs.kv_full[n % RING], (uint32_t)((n / RING) & 1));
            drain_q(bs, split_tiles, q_loads);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the issue loop (its operands stay warp-uniform); one elected
        // lane issues each tcgen05 instruction.
        {
            uint32_t item_base = 0;
            int seg_i = 0;
            uint32_t pv_count[2] = {0, 0};   // PV MMAs issued per pipe
            uint32_t pipe_segs[2] = {0, 0};  // segments in which the pipe produced a partial
            bool ok = true;
            // Descriptors are built once; every MMA only adds compile-time offsets (16-byte
            // units), which keeps the single issuing thread's instruction stream short.
            const uint64_t dq_base = desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dk0 = desc_sw128(smem_u32(sRing), 16, 1024);
            const uint64_t dv0 = desc_sw128(smem_u32(sRing), 16384, 1024);
            for (int64_t u = u_first; ok && u * p.tiles_per_unit < g1; ++u, ++seg_i) {
                Seg s;
                seg_decode(a, p, split_tiles, u, g0, g1, s);
                int qb;
                uint32_t quse;
                q_buffer(split_tiles, seg_i, qb, quse);
                if (!(ok = __all_sync(0xffffffffu, wait_bar(bs, &bs.q_full[qb], quse & 1, a.status)))) break;
                // Q of pipe h: its own 128-row block (more than 128 rows) or this unit's buffer
                const uint64_t dq0 = dq_base + (split_tiles ? (uint64_t)qb * (16384u >> 4) : 0u);
                const uint64_t dq1 = split_tiles ? dq0 : dq_base + (16384u >> 4);
                tc_fence_after();
                const int qk_total = s.cnt[0] + s.cnt[1];
                int qk_done = 0;
                auto issue_qk = [&](int h, int i) -> bool {
                    const uint32_t n = item_base + 2u * (uint32_t)(seg_tile(s, split_tiles, h, i) - s.tb);
                    const uint32_t slot = n % RING;
                    // pipe 1 of a shared tile reuses the K tile pipe 0 already waited for
                    if ((split_tiles || h == 0) && !__all_sync(0xffffffffu, wait_bar(bs, &bs.kv_full[slot], (n / RING) & 1u, a.status)))
                        return false;
                    if (SPARSE) fence_proxy_async_smem();  // the slot was written by cp.async (generic proxy)
                    const uint64_t dq = h ? dq1 : dq0;
                    const uint64_t dk = dk0 + (uint64_t)slot * (SLOT_BYTES >> 4);
                    const uint32_t d_tmem = tmem + 128u * h;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ss_elect(d_tmem, dq + (uint64_t)((ks >> 2) * 2048 + (ks & 3) * 2),
                               dk + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2), IDESC_QK, ks > 0 ? 1u : 0u);
                    mma_commit_elect(&bs.s_full[h]);
                    if (split_tiles || h == 1) mma_commit_elect(&bs.kv_empty[slot]);
                    if (++qk_done == qk_total) mma_commit_elect(&bs.q_empty[qb]);
                    return true;
                };
                auto issue_pv = [&](int h, int i) -> bool {
                    if (!__all_sync(0xffffffffu, wait_bar(bs, &bs.p_full[h], pv_count[h] & 1, a.status))) return false;
                    if (i == 0 && pipe_segs[h] > 0 &&
                        !__all_sync(0xffffffffu, wait_bar(bs, &bs.o_empty[h], (pipe_segs[h] - 1) & 1, a.status)))
                        return false;
                    const uint32_t n = item_base + 2u * (uint32_t)(seg_tile(s, split_tiles, h, i) - s.tb) + 1u;
                    const uint32_t slot = n % RING;
                    if ((split_tiles || h == 0) && !__all_sync(0xffffffffu, wait_bar(bs, &bs.kv_full[slot], (n / RING) & 1u, a.status)))
                        return false;
                    if (SPARSE) fence_proxy_async_smem();  // the slot was written by cp.async (generic proxy)
                    tc_fence_after();  // P_h was written to TMEM by the softmax warps
                    const uint64_t dv = dv0 + (uint64_t)slot * (SLOT_BYTES >> 4);
                    const uint32_t d_tmem = tmem + 256u + 128u * h, a_tmem = tmem + 128u * h;
                    const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts_elect(d_tmem, a_tmem + 8u * ks, dv + (uint64_t)(ks * 128), IDESC_PV, ks > 0 ? 1u : acc0);
                    if (split_tiles || h == 1) mma_commit_elect(&bs.kv_empty[slot]);
                    if (i == s.cnt[h] - 1) mma_commit_elect(&bs.o_done[h]);  // the unit's O_h is final
                    ++pv_count[h];
                    return true;
                };
                for (int h = 0; ok && h < 2; ++h)
                    if (s.cnt[h] > 0) ok = issue_qk(h, 0);
                const int n_iter = s.cnt[0];
                for (int i = 0; ok && i < n_iter; ++i)
                    for (int h = 0; ok && h < 2; ++h) {
                        if (i >= s.cnt[h]) continue;
                        ok = issue_pv(h, i);
                        if (ok && i + 1 < s.cnt[h]) ok = issue_qk(h, i + 1);
                    }
                for (int h = 0; h < 2; ++h)
                    if (s.cnt[h] > 0) ++pipe_segs[h];
                item_base += 2u * (uint32_t)(s.te - s.tb);
            }
            // drain: every MMA issued so far must complete before TMEM is freed
            mma_commit_elect(&bs.mma_done);
            drain_wait(&bs.mma_done, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int h = warp >> 2;            // pipe
        const int lg = warp & 3;            // TMEM lane group of this warp
        const int row = lg * 32 + lane;     // row of the pipe = TMEM lane
        const uint32_t lane_addr = (uint32_t)(lg * 32) << 16;
        const uint32_t s_col = 128u * h, o_col = 256u + 128u * h;
        const float sl2 = a.scale * 1.4426950408889634f;  // scores in base 2
        uint32_t s_count = 0, epi_count = 0;
        bool ok = true;
        for (int64_t u = u_first; u * p.tiles_per_unit < g1; ++u) {
            Seg s;
            seg_decode(a, p, split_tiles, u, g0, g1, s);
            const int row0 = s.rg * BM + (split_tiles ? 0 : 128 * h);  // first unit row of this pipe
            const int real_rows = min(max(tp.M - row0, 0), 128);
            const bool warp_rows = lg * 32 < real_rows;
            const int64_t slot = (((int64_t)blockIdx.x + u) << 1) + h;
            float *orow = a.o_part + (slot * 128 + row) * D;
            float *lrow = a.lse_part + slot * 128 + row;
            if (s.cnt[h] == 0) {  // this pipe got no tile of the unit: an empty partial
                if (row < real_rows) {
                    for (int c = 0; c < D; c += 4) *reinterpret_cast<float4 *>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                    *lrow = -INFINITY;
                }
                continue;
            }
            const int n_ctx = context_len(a, s.b);
            float m_ref = -INFINITY, l = 0.f;
            IdxPair raw[4];  // sparse: index entries of this pipe's next tile, loaded one tile ahead
            if (SPARSE && warp_rows) {
                const int t0 = seg_tile(s, split_tiles, h, 0);
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) raw[u4] = sparse_raw(a, s.b, t0 * T + 32 * u4 + lane);
            }
            for (int k = 0; k < s.cnt[h]; ++k) {
                const int t = seg_tile(s, split_tiles, h, k);
                uint32_t vmask[4] = {~0u, ~0u, ~0u, ~0u};  // sparse: used index slots of the tile
                if (SPARSE && warp_rows) {
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4)
                        vmask[u4] = __ballot_sync(0xffffffffu,
                                                  sparse_resolve(a, raw[u4], t * T + 32 * u4 + lane, n_ctx, false) >= 0);
                    if (k + 1 < s.cnt[h]) {
                        const int tn = seg_tile(s, split_tiles, h, k + 1);
#pragma unroll
                        for (int u4 = 0; u4 < 4; ++u4) raw[u4] = sparse_raw(a, s.b, tn * T + 32 * u4 + lane);
                    }
                }
                ok = __all_sync(0xffffffffu, ok && wait_bar(bs, &bs.s_full[h], s_count & 1, a.status));
                ++s_count;
                tc_fence_after();
                if (ok && warp_rows) {
                    uint32_t r[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_addr + s_col + 32u * c, r[c]);
                    tmem_wait_ld();
                    if (SPARSE) {
                        if ((vmask[0] & vmask[1] & vmask[2] & vmask[3]) != ~0u) {  // warp-uniform
#pragma unroll
                            for (int c = 0; c < 4; ++c)
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (!((vmask[c] >> j) & 1u)) r[c][j] = __float_as_uint(-INFINITY);
                        }
                    } else {
                        const int valid = min(max(n_ctx - t * T, 0), T);  // tokens of this tile inside the context
                        if (valid < T) {  // tail tile (warp-uniform): mask the tokens past the context
#pragma unroll
                            for (int c = 0; c < 4; ++c)
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (32 * c + j >= valid) r[c][j] = __float_as_uint(-INFINITY);
                        }
                    }
                    // row max of the raw scores (scale > 0): eight independent chains of
                    // three-operand max, then a short tree
                    float mx8[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mx8[q] = fmaxf(__uint_as_float(r[q >> 1][(q & 1) * 16]), __uint_as_float(r[q >> 1][(q & 1) * 16 + 1]));
#pragma unroll
                    for (int q = 0; q < 8; ++q)
#pragma unroll
                        for (int j = 2; j < 16; j += 2)
                            mx8[q] = fmax3(mx8[q], __uint_as_float(r[q >> 1][(q & 1) * 16 + j]),
                                           __uint_as_float(r[q >> 1][(q & 1) * 16 + j + 1]));
                    float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                    mx *= sl2;  // base-2 units
                    // move the reference max only when it grows by more than 2^8
                    bool rescale_o = false;
                    float factor = 1.f;
                    if (mx > m_ref + 8.f) {
                        factor = ex2(m_ref - mx);  // m_ref = -inf -> 0
                        rescale_o = l > 0.f;
                        l *= factor;
                        m_ref = mx;
                    }
                    // p = 2^(s * sl2 - m_ref), two columns per fp32x2 instruction
                    const float mref = m_ref == -INFINITY ? 0.f : m_ref;
                    const uint64_t scale2 = pack2(sl2, sl2), shift2 = pack2(-mref, -mref);
                    uint64_t sum2[4] = {pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f)};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float x0, x1;
                            unpack2(ffma2(pack2(__uint_as_float(r[c][2 * j]), __uint_as_float(r[c][2 * j + 1])),
                                          scale2, shift2),
                                    x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            sum2[j & 3] = fadd2(sum2[j & 3], pack2(p0, p1));
                            __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
                            pk[j] = *reinterpret_cast<uint32_t *>(&v);
                        }
                        tmem_st16(tmem + lane_addr + s_col + 16u * c, pk);
                    }
                    float sa, sb;
                    unpack2(fadd2(fadd2(sum2[0], sum2[1]), fadd2(sum2[2], sum2[3])), sa, sb);
                    l += sa + sb;
                    tmem_wait_st();
                    if (__any_sync(0xffffffffu, rescale_o) && k > 0) {
                        // O holds the previous tiles. Their PV has completed: the commit that
                        // signalled this S_h came after it from the same issuing thread. Rescale
                        // this warp's rows (after P is built, so the score registers are free).
                        const float f = rescale_o ? factor : 1.f;
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tmem + lane_addr + o_col + 32u * c, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
                            tmem_st32(tmem + lane_addr + o_col + 32u * c, o);
                        }
                        tmem_wait_st();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bs.p_full[h]);
            }
            // epilogue: O / l and lse of this pipe's rows -> partial slot
            ok = __all_sync(0xffffffffu, ok && wait_bar(bs, &bs.o_done[h], epi_count & 1, a.status));
            ++epi_count;
            tc_fence_after();
            if (ok && warp_rows) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_addr + o_col + 32u * c, o);
                    tmem_wait_ld();
                    if (row < real_rows) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(orow + 32 * c + j) =
                                make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                                            __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
                    }
                }
                if (row < real_rows) *lrow = l > 0.f ? (m_ref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bs.o_empty[h]);
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_PRODUCER) tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------- host side

bool encode_map(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                const cuuint32_t *box) {
    static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        const bool found = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                            cudaEnableDefault, &q) == cudaSuccess &&
                           q == cudaDriverEntryPointSuccess;
        cudaGetLastError();
        return found ? reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn) : nullptr;
    }();
    if (!encode) return false;
    cuuint32_t elem[4] = {1, 1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims,
                        strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const VerifyArgs &a) {
    // the softmax takes the row max of the raw scores, which needs scale > 0
    if (!(a.G >= 1 && a.G <= 128 && (128 % a.G) == 0 && a.scale > 0.f)) return false;
    if (a.idx)  // gathered rows are copied 16 bytes at a time: every row start 16-byte aligned
        return a.budget >= 1 && a.sb % 8 == 0 && a.sh % 8 == 0 && a.st % 8 == 0;
    return a.L >= 1;
}

cudaError_t launch_cache_attn_tc(const VerifyArgs &a, const SplitPlan &p, cudaStream_t s, cudaEvent_t ev0,
                                 cudaEvent_t ev1, bool *launched) {
    *launched = false;
    CUtensorMap mq, mk, mv;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.Hq, (cuuint64_t)a.B * a.N};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)a.G, (cuuint32_t)(128 / a.G)};
        if (!encode_map(&mq, a.q, 3, dims, strides, box)) return cudaSuccess;
    }
    const bool sparse = a.idx != nullptr;
    if (sparse) {  // rows are gathered with cp.async; the K/V maps are not read
        mk = mq;
        mv = mq;
    } else {
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.L, (cuuint64_t)a.Hkv, (cuuint64_t)a.B};
        const cuuint64_t strides[3] = {(cuuint64_t)a.st * 2, (cuuint64_t)a.sh * 2, (cuuint64_t)a.sb * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)T, 1, 1};
        if (!encode_map(&mk, a.k_cache, 4, dims, strides, box)) return cudaSuccess;
        if (!encode_map(&mv, a.v_cache, 4, dims, strides, box)) return cudaSuccess;
    }
    TcParams tp;
    tp.M = a.G * a.N;
    tp.split_tiles = tp.M <= 128 ? 1 : 0;
    auto kern = sparse ? cache_attn_tc_kernel<true> : cache_attn_tc_kernel<false>;
    static const cudaError_t attr_dense = kernel_attributes(cache_attn_tc_kernel<false>, SMEM_BYTES);
    static const cudaError_t attr_sparse = kernel_attributes(cache_attn_tc_kernel<true>, SMEM_BYTES);
    cudaError_t e = sparse ? attr_sparse : attr_dense;
    if (e != cudaSuccess) return e;
    if (ev0) cudaEventRecord(ev0, s);
    kern<<<p.ctas, THREADS, SMEM_BYTES, s>>>(a, p, tp, mq, mk, mv);
    e = cudaGetLastError();
    if (ev1) cudaEventRecord(ev1, s);
    count_launches(1);
    *launched = true;
    return e;
}

}  // namespace specverify
