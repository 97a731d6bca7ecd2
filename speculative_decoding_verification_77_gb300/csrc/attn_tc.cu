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
// fp8 cache (dense, contiguous; 512 threads): the producer brings each K or
// V tile as E4M3 codes by TMA into one of two staging buffers; warps 10-15
// each convert a sixth of it into the bf16 ring (4 slots), fence the async
// proxy and arrive on the slot and the staging buffer; the unit's K scale
// joins the softmax scale and its V scale the final normalisation. Warps 8-15
// give registers back (setmaxnreg) to the two softmax warpgroups.
// Every wait on an mbarrier is bounded; a wait that gives up records
// SPEC_ERR_TIMEOUT, the CTA drains its in-flight copies and MMAs, frees TMEM
// and returns.
#include "tc_pipe.cuh"

namespace specverify {

namespace {

using namespace sm100;
using namespace tcpipe;

constexpr int D = kHeadDim;
constexpr int Q_BYTES = 256 * D * 2;  // 64 KiB
constexpr int SMEM_RING = Q_BYTES;
constexpr int SMEM_BAR = SMEM_RING + RING * SLOT_BYTES;  // 229376
constexpr int SMEM_BYTES = SMEM_BAR + 256 + 1024;        // + barriers + alignment slack
constexpr int THREADS = 320;
constexpr int WARP_PRODUCER = 8, WARP_MMA = 9;
// fp8 cache: the converter warps follow the MMA warp
constexpr int THREADS_FP8 = THREADS + 32 * FP8_CONVERTERS;
// 512 threads start with 128 registers each; two warpgroups at 176 and two at 80 use them all
constexpr uint32_t FP8_REGS_SOFTMAX = 176, FP8_REGS_OTHER = 80;
static_assert(THREADS_FP8 == 512 && 256 * (FP8_REGS_SOFTMAX + FP8_REGS_OTHER) == 65536,
              "the register split adds up to the launch's registers");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 128, true);

static_assert(SMEM_BYTES <= 232448, "dynamic shared memory fits one CTA per SM");

struct TcParams {
    int split_tiles;  // 1: pipes take alternate tiles of the same <=128 rows
    int M;            // G * N query rows per (b, h_kv)
};

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

template <bool SPARSE, bool PAGED, bool FP8>
__global__ void __launch_bounds__(FP8 ? THREADS_FP8 : THREADS, 1)
cache_attn_tc_kernel(const VerifyArgs a, const SplitPlan p, const TcParams tp,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    griddep_launch_dependents();  // the merge may be scheduled as this grid's CTAs drain
    // the 128-byte swizzle needs 1024-byte aligned tiles; SMEM_BYTES has 1 KiB of slack for it
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *sQ = smem;
    uint8_t *sRing = smem + SMEM_RING;
    // fp8 cache: a ring of FP8_KR bf16 tiles, then the staging of FP8_STAGES tiles of codes
    constexpr int KRING = FP8 ? FP8_KR : RING;
    uint8_t *sStage = sRing + KRING * SLOT_BYTES;
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
            // sparse: one arrival per gathering lane; fp8: one per converter warp
            mbar_init(&bs.kv_full[i], SPARSE ? 32 : FP8 ? FP8_CONVERTERS : 1);
            mbar_init(&bs.kv_empty[i], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&bs.s_full[h], 1);
            mbar_init(&bs.p_full[h], 4);
            mbar_init(&bs.o_done[h], 1);
            mbar_init(&bs.o_empty[h], 4);
        }
        for (int i = 0; i < FP8_STAGES; ++i) {
            mbar_init(&bs.st_full[i], 1);
            mbar_init(&bs.st_empty[i], FP8_CONVERTERS);
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
    // launched early behind the status word's reset kernel: wait for it before anything can
    // record an error there (the set-up above overlaps it)
    griddep_wait();
    const uint32_t tmem = bs.tmem_base;

    const int64_t g0 = plan_start(p, blockIdx.x), g1 = plan_start(p, blockIdx.x + 1);
    const int64_t u_first = g0 / p.tiles_per_unit;

    // Q of a unit into buffer qb (one thread)
    auto qload = [&](const Seg &sg, int qb, uint64_t *bar) { load_q(&tm_q, sQ, bar, split_tiles, qb, sg, BM, a.G, a.N); };
    if (warp >= WARP_PRODUCER) {
        // fp8: this warpgroup and the next (loader, issuer, converters) give registers to the softmax
        if (FP8) setmaxnreg_dec<FP8_REGS_OTHER>();
        if (SPARSE && warp == WARP_PRODUCER) {
            // ------------------------------------------------------------ gather producer
            produce_sparse(bs, sRing, &tm_q, a, p, split_tiles, u_first, g0, g1, lane, qload);
            __syncwarp();
        } else if (warp == WARP_PRODUCER) {
            // ------------------------------------------------------------ TMA producer
            if (FP8) {
                if (lane == 0) produce_dense_fp8(bs, sStage, &tm_q, &tm_k, &tm_v, a, p, split_tiles, u_first, g0, g1, qload);
            } else if (lane == 0)
                produce_dense<PAGED>(bs, sRing, &tm_q, &tm_k, &tm_v, a, p, split_tiles, u_first, g0, g1, qload);
            __syncwarp();
        } else if (FP8 && warp > WARP_MMA) {
            // ------------------------------------------------------------ fp8 converters
            convert_items(bs, sRing, sStage, g0, g1, lane, warp - WARP_MMA - 1, a.status);
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
                        const uint32_t slot = n % KRING;
                        // pipe 1 of a shared tile reuses the K tile pipe 0 already waited for
                        if ((split_tiles || h == 0) && !__all_sync(0xffffffffu, wait_bar(bs, &bs.kv_full[slot], (n / KRING) & 1u, a.status)))
                            return false;
                        if (SPARSE || FP8) fence_proxy_async_smem();  // the slot was written by the generic proxy
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
                        const uint32_t slot = n % KRING;
                        if ((split_tiles || h == 0) && !__all_sync(0xffffffffu, wait_bar(bs, &bs.kv_full[slot], (n / KRING) & 1u, a.status)))
                            return false;
                        if (SPARSE || FP8) fence_proxy_async_smem();  // the slot was written by the generic proxy
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
        }
    } else {
        if (FP8) setmaxnreg_inc<FP8_REGS_SOFTMAX>();
        // ------------------------------------------------------------ softmax warps
        const int h = warp >> 2;            // pipe
        const int lg = warp & 3;            // TMEM lane group of this warp
        const int row = lg * 32 + lane;     // row of the pipe = TMEM lane
        const uint32_t lane_addr = (uint32_t)(lg * 32) << 16;
        const uint32_t s_col = 128u * h, o_col = 256u + 128u * h;
        const float sl2_base = a.scale * 1.4426950408889634f;  // scores in base 2
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
            // fp8 cache: the unit's K scale joins the softmax scale, its V scale the normalisation
            const float sl2 = FP8 ? sl2_base * __ldg(a.k_scale + (int64_t)s.b * a.Hkv + s.hk) : sl2_base;
            const float vscale = FP8 ? __ldg(a.v_scale + (int64_t)s.b * a.Hkv + s.hk) : 1.f;
            float m_ref = -INFINITY, l = 0.f;
            IdxPair raw[4];  // sparse: index entries of this pipe's next tile, loaded one tile ahead
            if (SPARSE && warp_rows) {
                const int t0 = seg_tile(s, split_tiles, h, 0);
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) raw[u4] = sparse_raw(a, s.b, t0 * T + 32 * u4 + lane);
            }
            // dense, paged cache: the pool block of this pipe's next tile, loaded one tile ahead
            auto block_of = [&](int t) -> int {
                return __ldg(a.table + (int64_t)s.b * a.table_ld + (int64_t)t * T / a.block_size);
            };
            int blk_next = (PAGED && warp_rows) ? block_of(seg_tile(s, split_tiles, h, 0)) : 0;
            for (int k = 0; k < s.cnt[h]; ++k) {
                const int t = seg_tile(s, split_tiles, h, k);
                uint32_t vmask[4] = {~0u, ~0u, ~0u, ~0u};  // sparse: used index slots of the tile
                bool bad_block = false;                     // dense, paged: the tile's block is not in the pool
                if (PAGED && warp_rows) {
                    bad_block = blk_next < 0 || blk_next >= a.num_blocks;
                    if (k + 1 < s.cnt[h]) blk_next = block_of(seg_tile(s, split_tiles, h, k + 1));
                    if (bad_block && t * T < n_ctx && lane == 0) flag_status(a.status, SPEC_ERR_BAD_INPUT);
                }
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
                        // tokens of this tile inside the context (none when its block is not in the pool)
                        const int valid = bad_block ? 0 : min(max(n_ctx - t * T, 0), T);
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
                const float inv = l > 0.f ? vscale / l : 0.f;
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

// bf16 tiles in the 128-byte swizzle the tensor core reads, or (codes) unswizzled bytes.
bool encode_map(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                const cuuint32_t *box, bool codes = false) {
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
    CUresult r = encode(map, codes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, codes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const VerifyArgs &a) {
    // fp8 cache: the dense contiguous case (its codes are converted to bf16 tiles by the producer)
    if (a.kv_fp8 && (a.idx || a.table)) return false;
    // the softmax takes the row max of the raw scores, which needs scale > 0
    if (!(a.G >= 1 && a.G <= 128 && (128 % a.G) == 0 && a.scale > 0.f)) return false;
    if (a.idx)  // gathered rows are copied 16 bytes at a time: every row start 16-byte aligned
        return a.budget >= 1 && a.sb % 8 == 0 && a.sh % 8 == 0 && a.st % 8 == 0;
    // paged: a 128-token tile must lie in one block, and the block coordinate is 32-bit
    if (a.table && (a.block_size % T != 0 || a.num_blocks < 1 || a.num_blocks > INT32_MAX)) return false;
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
    } else if (a.kv_fp8) {
        // E4M3 codes [B, Hkv, L, d], one byte an element: 128 x 128-byte boxes into the staging,
        // unswizzled (the warp converts them into the swizzled bf16 tile)
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)a.L, (cuuint64_t)a.Hkv, (cuuint64_t)a.B};
        const cuuint64_t strides[3] = {(cuuint64_t)a.st, (cuuint64_t)a.sh, (cuuint64_t)a.sb};
        const cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)T, 1, 1};
        if (!encode_map(&mk, a.k_cache, 4, dims, strides, box, true)) return cudaSuccess;
        if (!encode_map(&mv, a.v_cache, 4, dims, strides, box, true)) return cudaSuccess;
    } else {
        // contiguous cache [B, Hkv, L, d] or (paged) the pool [blocks, Hkv, block_size, d]
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)(a.table ? a.block_size : a.L), (cuuint64_t)a.Hkv,
                                    (cuuint64_t)(a.table ? a.num_blocks : a.B)};
        const cuuint64_t strides[3] = {(cuuint64_t)a.st * 2, (cuuint64_t)a.sh * 2, (cuuint64_t)a.sb * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)T, 1, 1};
        if (!encode_map(&mk, a.k_cache, 4, dims, strides, box)) return cudaSuccess;
        if (!encode_map(&mv, a.v_cache, 4, dims, strides, box)) return cudaSuccess;
    }
    TcParams tp;
    tp.M = a.G * a.N;
    tp.split_tiles = tp.M <= 128 ? 1 : 0;
    auto kern = sparse ? cache_attn_tc_kernel<true, false, false>
                : a.table  ? cache_attn_tc_kernel<false, true, false>
                : a.kv_fp8 ? cache_attn_tc_kernel<false, false, true>
                           : cache_attn_tc_kernel<false, false, false>;
    static PerDeviceOnce attr_once;
    cudaError_t e = once_per_device(attr_once, [] {
        cudaError_t r = cudaSuccess;
        for (auto k : {cache_attn_tc_kernel<false, false, false>, cache_attn_tc_kernel<false, true, false>,
                       cache_attn_tc_kernel<true, false, false>, cache_attn_tc_kernel<false, false, true>})
            if (r == cudaSuccess) r = kernel_attributes(k, SMEM_BYTES);
        return r;
    });
    if (e != cudaSuccess) return e;
    if (ev0) cudaEventRecord(ev0, s);
    {  // programmatic stream serialisation: the CTAs may start while the previous kernel runs
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)p.ctas);
        cfg.blockDim = dim3(a.kv_fp8 && !sparse && !a.table ? THREADS_FP8 : THREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.stream = s;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, a, p, tp, mq, mk, mv);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (ev1) cudaEventRecord(ev1, s);
    count_launches(1);
    *launched = true;
    return e;
}

}  // namespace specverify
