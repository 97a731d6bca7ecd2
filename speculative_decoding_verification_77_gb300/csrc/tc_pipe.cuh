// Pipeline pieces shared by the tcgen05 cache kernels: the mbarrier block, the
// bounded waits, the walk over a CTA's units (segments), the Q buffers and the
// two K/V producers (TMA for the dense cache, a cp.async row gather for the
// index set) that fill the ring of 128-token K and V tiles in the 128-byte
// swizzled K-major layout the tensor core reads.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace specverify {
namespace tcpipe {

using namespace sm100;

constexpr int T = 128;                       // tokens per tile
constexpr int RING = 5;                      // K/V slots
constexpr int SLOT_BYTES = T * kHeadDim * 2; // 32 KiB: one K or V tile
constexpr int HALF_BYTES = SLOT_BYTES / 2;   // 64 of the 128 columns
constexpr long long WAIT_LIMIT_CYCLES = 4000000000LL;  // ~2 s

// fp8 cache: the producer warp only requests the codes; converter warps (10-15) each turn
// a sixth of every staged tile into a slot of a ring of FP8_KR bf16 tiles. The staging
// (FP8_STAGES tiles of codes, 16 KiB each) takes the room of the bf16 ring's other slots.
constexpr int FP8_CONVERTERS = 6;
constexpr int FP8_KR = 4;
constexpr int FP8_STAGES = 2;
static_assert(2 * FP8_KR + FP8_STAGES <= 2 * RING, "fp8 ring and staging fit the bf16 ring's room");

struct Bars {
    uint64_t q_full[2], q_empty[2];  // Q buffers (two only when the pipes share the rows)
    uint64_t kv_full[RING], kv_empty[RING];
    uint64_t s_full[2], p_full[2], o_done[2], o_empty[2];
    uint64_t st_full[FP8_STAGES];   // fp8 cache: the staged codes of an item have landed
    uint64_t st_empty[FP8_STAGES];  // fp8 cache: every converter has read the staged codes
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block fits its reservation");

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
    plan_unit_coords(p, a.Hkv, u, s.b, s.hk, s.rg);
    const int nt = s.te - s.tb;
    s.cnt[0] = split_tiles ? (nt + 1) / 2 : nt;
    s.cnt[1] = split_tiles ? nt / 2 : nt;
}
__device__ __forceinline__ int seg_tile(const Seg &s, int split_tiles, int h, int i) {
    return split_tiles ? s.tb + 2 * i + h : s.tb + i;
}

// Q buffers: when the two pipes read different rows of a unit there is one
// buffer; when they share the rows (alternate tiles) two buffers serve
// alternate units, so that the next unit's Q loads while the current one is
// still in use. Segment seg_i uses buffer seg_i % nqb for the (seg_i / nqb)-th
// time.
__device__ __forceinline__ void q_buffer(int split_tiles, int seg_i, int &qb, uint32_t &use) {
    const int nqb = split_tiles ? 2 : 1;
    qb = seg_i % nqb;
    use = (uint32_t)(seg_i / nqb);
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

// Gather producer (the whole warp): the K and V rows named by idx[b] of every
// tile of the CTA's range, and each unit's Q through qload(seg, buffer, bar)
// (called by lane 0).
template <class QLoad>
__device__ __forceinline__ void produce_sparse(Bars &bs, uint8_t *sRing, const CUtensorMap *tm_q, const VerifyArgs &a,
                                               const SplitPlan &p, int split_tiles, int64_t u_first, int64_t g0,
                                               int64_t g1, int lane, QLoad qload) {
    if (lane == 0) tma_prefetch_desc(tm_q);
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
            if (lane == 0) qload(s, qb, &bs.q_full[qb]);
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
}

// fp8 cache: part `part` of FP8_CONVERTERS of one K or V tile of E4M3 codes (128 rows of 128
// codes, row r at r * 128) converted by the 32 lanes of a warp into the bf16 tile the TMA
// would have written (two 16 KiB column halves; row r of a half at r * 128 bytes, its 16-byte
// chunk q at (q ^ (r & 7)) * 16, the 128-byte swizzle of a 1024-byte aligned tile). Part p
// takes the 16-code chunks lane + 32 k for k = p, p + FP8_CONVERTERS, ...
__device__ __forceinline__ void convert_e4m3_tile(const uint8_t *src, uint8_t *dst, int lane, int part) {
#pragma unroll 2
    for (int k = part; k < 32; k += FP8_CONVERTERS) {
        const int c = lane + 32 * k;  // 16 codes: row c >> 3, columns 16 (c & 7) .. + 15
        const int r = c >> 3, m = c & 7;
        const uint4 codes = *reinterpret_cast<const uint4 *>(src + c * 16);
        uint4 lo, hi;
        e4m3x16_to_bf16x16(codes, lo, hi);
        uint8_t *row = dst + (m >> 2) * HALF_BYTES + r * 128;
        const int q0 = 2 * (m & 3);
        *reinterpret_cast<uint4 *>(row + ((q0 ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(row + (((q0 + 1) ^ (r & 7)) << 4)) = hi;
    }
}

// fp8 cache: a converter warp, part `part` of every item of the CTA's range (item n: K of tile
// g0 + n / 2 for even n, V for odd). Per item: wait for its staged codes and its ring slot,
// convert, fence the generic-proxy stores for the tensor core, and (lane 0) arrive on the slot
// and on the staging buffer.
__device__ __forceinline__ void convert_items(Bars &bs, uint8_t *sRing, const uint8_t *sStage, int64_t g0, int64_t g1,
                                              int lane, int part, uint32_t *status) {
    const int64_t nitems = 2 * (g1 - g0);
    for (int64_t n = 0; n < nitems; ++n) {
        const int sb = (int)(n % FP8_STAGES);
        if (!__all_sync(0xffffffffu, wait_bar(bs, &bs.st_full[sb], (uint32_t)((n / FP8_STAGES) & 1), status))) break;
        const int slot = (int)(n % FP8_KR);
        const int64_t use = n / FP8_KR;
        if (use > 0 &&
            !__all_sync(0xffffffffu, wait_bar(bs, &bs.kv_empty[slot], (uint32_t)((use - 1) & 1), status)))
            break;
        convert_e4m3_tile(sStage + sb * (T * kHeadDim), sRing + slot * SLOT_BYTES, lane, part);
        fence_proxy_async_smem();  // the tensor core reads what these generic stores wrote
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bs.kv_full[slot]);
            mbar_arrive(&bs.st_empty[sb]);
        }
    }
}

// fp8 producer (one thread): the E4M3 codes of every K and V tile of the CTA's range by TMA
// into FP8_STAGES staging buffers (item m into buffer m % FP8_STAGES, once every converter
// has arrived on that buffer's st_empty for item m - FP8_STAGES), and each unit's Q through
// qload(seg, buffer, bar) before the unit's first item.
template <class QLoad>
__device__ __forceinline__ void produce_dense_fp8(Bars &bs, uint8_t *sStage, const CUtensorMap *tm_q,
                                                  const CUtensorMap *tm_k, const CUtensorMap *tm_v, const VerifyArgs &a,
                                                  const SplitPlan &p, int split_tiles, int64_t u_first, int64_t g0,
                                                  int64_t g1, QLoad qload) {
    constexpr uint32_t STAGE_BYTES = T * kHeadDim;  // 16 KiB of codes
    tma_prefetch_desc(tm_q);
    tma_prefetch_desc(tm_k);
    tma_prefetch_desc(tm_v);
    int64_t m = 0;  // items requested so far
    int q_loads = 0;
    bool ok = true;
    for (int64_t u = u_first; ok && u * p.tiles_per_unit < g1; ++u, ++q_loads) {
        Seg s;
        seg_decode(a, p, split_tiles, u, g0, g1, s);
        int qb;
        uint32_t quse;
        q_buffer(split_tiles, q_loads, qb, quse);
        if (quse > 0 && !(ok = wait_bar(bs, &bs.q_empty[qb], (quse - 1) & 1, a.status))) break;
        qload(s, qb, &bs.q_full[qb]);
        for (int t = s.tb; ok && t < s.te; ++t) {
            for (int kv = 0; kv < 2; ++kv, ++m) {
                const int sb = (int)(m % FP8_STAGES);
                if (m >= FP8_STAGES &&
                    !(ok = wait_bar(bs, &bs.st_empty[sb], (uint32_t)((m / FP8_STAGES - 1) & 1), a.status)))
                    break;
                uint64_t *bar = &bs.st_full[sb];
                mbar_arrive_expect_tx(bar, STAGE_BYTES);
                tma_load_4d(sStage + sb * STAGE_BYTES, kv ? tm_v : tm_k, bar, 0, t * T, s.hk, s.b);
            }
        }
    }
    // the drain: the last FP8_STAGES loads (one per buffer) have landed before the CTA ends
    for (int64_t i = m > FP8_STAGES ? m - FP8_STAGES : 0; i < m; ++i)
        drain_wait(&bs.st_full[i % FP8_STAGES], (uint32_t)((i / FP8_STAGES) & 1));
    drain_q(bs, split_tiles, q_loads);
}

// TMA producer (one thread): the K and V tiles of the CTA's range, and each
// unit's Q through qload(seg, buffer, bar).
template <bool PAGED, class QLoad>
__device__ __forceinline__ void produce_dense(Bars &bs, uint8_t *sRing, const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                                              const CUtensorMap *tm_v, const VerifyArgs &a, const SplitPlan &p,
                                              int split_tiles, int64_t u_first, int64_t g0, int64_t g1, QLoad qload) {
    tma_prefetch_desc(tm_q);
    tma_prefetch_desc(tm_k);
    tma_prefetch_desc(tm_v);
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
        qload(s, qb, &bs.q_full[qb]);
        // paged cache: the pool block of each tile (a tile lies in one block), loaded four
        // tiles ahead of its use
        auto block_of = [&](int t) -> int {
            if (!PAGED || t >= s.te) return 0;
            return __ldg(a.table + (int64_t)s.b * a.table_ld + (int64_t)t * T / a.block_size);
        };
        int blk0 = block_of(s.tb), blk1 = block_of(s.tb + 1), blk2 = block_of(s.tb + 2), blk3 = block_of(s.tb + 3);
        // K and V tiles in order: tile tb: K, V; tile tb+1: K, V; ...
        for (int t = s.tb; t < s.te; ++t) {
            const int blk = blk0;
            blk0 = blk1;
            blk1 = blk2;
            blk2 = blk3;
            blk3 = block_of(t + 4);
            for (int kv = 0; kv < 2; ++kv, ++item) {
                const int slot = (int)(item % RING);
                const int64_t use = item / RING;
                if (use > 0 && !(ok = wait_bar(bs, &bs.kv_empty[slot], (uint32_t)((use - 1) & 1), a.status)))
                    break;
                uint8_t *dst = sRing + slot * SLOT_BYTES;
                mbar_arrive_expect_tx(&bs.kv_full[slot], SLOT_BYTES);
                const CUtensorMap *m = kv == 0 ? tm_k : tm_v;
                if (PAGED) {  // pool map [blocks, Hkv, block_size, d]: a block entry outside the pool
                                // reads the zero fill (the softmax masks that tile)
                    const int o = (int)((int64_t)t * T % a.block_size);
                    tma_load_4d(dst, m, &bs.kv_full[slot], 0, o, s.hk, blk);
                    tma_load_4d(dst + HALF_BYTES, m, &bs.kv_full[slot], 64, o, s.hk, blk);
                } else {
                    tma_load_4d(dst, m, &bs.kv_full[slot], 0, t * T, s.hk, s.b);
                    tma_load_4d(dst + HALF_BYTES, m, &bs.kv_full[slot], 64, t * T, s.hk, s.b);
                }
            }
            if (!ok) break;
        }
    }
    // drain: wait for the last copies still in flight (consumed ones return at once)
    const int64_t first = item > RING ? item - RING : 0;
    for (int64_t n = first; n < item; ++n) drain_wait(&bs.kv_full[n % RING], (uint32_t)((n / RING) & 1));
    drain_q(bs, split_tiles, q_loads);
}

}  // namespace tcpipe
}  // namespace specverify
