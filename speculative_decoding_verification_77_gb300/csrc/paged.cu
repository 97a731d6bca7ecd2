// Paged KV cache: the index set of a sparse call resolved to pool rows.
//
// A paged cache (a layout the source pages do not use: the same cache stored in
// fixed-size blocks of a pool, found through a per-sequence block table) needs
// no change in the gather kernels if every used index entry is translated once
// into the pool row that holds it. Pool rows are numbered as if the pool were
// one long cache of row stride st: block blk, row o is row blk * (sblk / st) + o
// (the caller's block stride is a multiple of its row stride). The translation
// also performs the checks of a sparse index entry (inside the context, above the
// previous entry; -1 padding) and of its block entry (inside the pool); an entry
// that fails either becomes -1 and, unless it was -1 padding, is reported as bad
// input. The kernels then read the translated list as already checked.
#include "common.cuh"

namespace specverify {

namespace {

__global__ void __launch_bounds__(256) resolve_paged_idx_kernel(VerifyArgs a, int32_t *rows_out, int64_t row_step) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= a.budget) return;
    const int n = context_len(a, b);
    const int32_t *ib = a.idx + (int64_t)b * a.budget;
    const int t = __ldg(ib + j);
    int32_t r = -1;
    if (t >= 0 && t < n && (j == 0 || t > __ldg(ib + j - 1))) {
        const int64_t blk = __ldg(a.table + (int64_t)b * a.table_ld + t / a.block_size);
        if (blk >= 0 && blk < a.num_blocks) r = (int32_t)(blk * row_step + t % a.block_size);
        else flag_status(a.status, SPEC_ERR_BAD_INPUT);
    } else if (t != -1) {
        flag_status(a.status, SPEC_ERR_BAD_INPUT);
    }
    rows_out[(int64_t)b * a.budget + j] = r;
}

}  // namespace

cudaError_t launch_resolve_paged_idx(const VerifyArgs &a, int32_t *rows_out, cudaStream_t s) {
    const dim3 grid((unsigned)((a.budget + 255) / 256), (unsigned)a.B);
    resolve_paged_idx_kernel<<<grid, 256, 0, s>>>(a, rows_out, a.sb / a.st);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace specverify
