// Content validation: every rule of gqa_validate / gqa_validate_attend, one
// CTA per batch row.
#include "gqa_common.cuh"
#include "gqa_launch.h"

namespace gqa {
namespace {

// One CTA per batch row: every rule of the public header's gqa_validate.
// L is the last slot the call touches: lengths[b] for the decode step (the
// append slot), lengths[b] - 1 for the read-only attend, lengths[b] + q_len - 1
// for a multi-token step (cu_q non-null; a row without tokens is checked as
// if it touched slot max(lengths[b] - 1, 0) of a paged table).
__global__ void __launch_bounds__(256) validate_kernel(const int32_t *lengths, const int32_t *slot_ids,
                                                       const int32_t *block_table, int B, int R, int Smax,
                                                       int num_blocks, int block_size, int max_blocks,
                                                       int attend, const int32_t *cu_q, int T,
                                                       int32_t *result)
{
    const int b = blockIdx.x;
    long long L = (long long)lengths[b] - attend;
    bool bad = false;
    if (cu_q) {
        const long long q0 = cu_q[b], q1 = cu_q[b + 1];
        if (threadIdx.x == 0 && ((b == 0 && q0 != 0) || (b == B - 1 && q1 != T) || q1 < q0))
            bad = true;
        const long long Lb = lengths[b];
        if (!block_table) {
            if (threadIdx.x == 0 && (Lb < 0 || Lb + (q1 - q0) > Smax))
                bad = true;
            L = 0;   // the range checks are done
        } else {
            const long long l = Lb + (q1 - q0) - 1;
            L = Lb < 0 ? -1 : (l < 0 ? 0 : l);
        }
    }
    if (!block_table) {
        if (threadIdx.x == 0) {
            if (L < 0 || L > Smax - 1)
                bad = true;
            if (!slot_ids && B > R)
                bad = true;
            if (slot_ids && (slot_ids[b] < 0 || slot_ids[b] >= R))
                bad = true;
        }
        if (slot_ids) {
            const int mine = slot_ids[b];
            for (int c = threadIdx.x; c < b; c += blockDim.x)
                if (slot_ids[c] == mine)
                    bad = true;
        }
    } else {
        const int32_t *row = block_table + (long long)b * max_blocks;
        if (threadIdx.x == 0 && (L < 0 || L >= (long long)max_blocks * block_size))
            bad = true;
        const long long need = (L >= 0) ? L / block_size : -1;
        for (int i = threadIdx.x; i < max_blocks; i += blockDim.x) {
            const int e = row[i];
            if (e == -1) {
                if (i <= need)
                    bad = true;
                continue;
            }
            if (e < 0 || e >= num_blocks)
                bad = true;
            for (int k = 0; k < i; ++k)
                if (row[k] == e)
                    bad = true;
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0)
        atomicOr(result, 1);
}

}  // namespace

cudaError_t validate_launch(const int32_t *lengths, const int32_t *slot_ids,
                            const int32_t *block_table, int B, int R, int Smax,
                            int num_blocks, int block_size, int max_blocks, int attend,
                            const int32_t *cu_q, int T, int32_t *d_result, cudaStream_t st)
{
    validate_kernel<<<B, 256, 0, st>>>(lengths, slot_ids, block_table, B, R, Smax, num_blocks,
                                       block_size, max_blocks, attend, cu_q, T, d_result);
    return cudaGetLastError();
}

}  // namespace gqa
