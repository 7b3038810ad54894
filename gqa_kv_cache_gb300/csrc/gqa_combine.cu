// Split combine (log-sum-exp merge of per-CTA partial softmax states) and
// the content-validation kernel.
#include "gqa_common.cuh"
#include "gqa_launch.h"

namespace gqa {
namespace {

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One CTA per unit u = b * Hkv + kvh. A unit whose tiles lie in one decode
// CTA was finished by that CTA and is skipped here. Otherwise CTAs
// first..last each left (m_i, l_i, o_i) at partial index u + i, and
//   M = max_i m_i,  o = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i
// (m in base-2 units).
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p)
{
    // With programmatic dependent launch this CTA may start while the decode
    // grid still runs; wait for its completion and memory before reading.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int u = blockIdx.x;
    const int b = u / p.Hkv, kvh = u % p.Hkv;
    const int L = __ldg(p.lengths + b);
    const int nt = row_tiles(p, L);
    const long long N = p.ws_total[0];
    const long long first_tile = p.ws_rowpre[b] + (long long)kvh * nt;
    const long long C = working_ctas(N, p.grid);
    const int first = cta_of_tile(first_tile, N, C);
    const int last = cta_of_tile(first_tile + nt - 1, N, C);
    if (first == last)
        return;
    const int G = p.G, D = p.D;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
        for (int i = first; i <= last; ++i)
            M = fmaxf(M, p.ws_ml[(((long long)u + i) * G + g) * 2]);
        float num = 0.f, den = 0.f;
        for (int i = first; i <= last; ++i) {
            const long long P = (long long)u + i;
            const float a = ex2(p.ws_ml[(P * G + g) * 2] - M);
            num = fmaf(a, p.ws_o[(P * G + g) * D + d], num);
            den = fmaf(a, p.ws_ml[(P * G + g) * 2 + 1], den);
        }
        p.out[((long long)b * p.Hq + kvh * G + g) * D + d] = num / den;
    }
}

// One CTA per batch row: every rule of the public header's gqa_validate.
__global__ void __launch_bounds__(256) validate_kernel(const int32_t *lengths, const int32_t *slot_ids,
                                                       const int32_t *block_table, int B, int R, int Smax,
                                                       int num_blocks, int block_size, int max_blocks,
                                                       int32_t *result)
{
    const int b = blockIdx.x;
    const long long L = lengths[b];
    bool bad = false;
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

cudaError_t combine_launch(const DecodeParams &p, cudaStream_t st, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B * p.Hkv);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

cudaError_t validate_launch(const int32_t *lengths, const int32_t *slot_ids,
                            const int32_t *block_table, int B, int R, int Smax,
                            int num_blocks, int block_size, int max_blocks,
                            int32_t *d_result, cudaStream_t st)
{
    validate_kernel<<<B, 256, 0, st>>>(lengths, slot_ids, block_table, B, R, Smax, num_blocks,
                                       block_size, max_blocks, d_result);
    return cudaGetLastError();
}

}  // namespace gqa
