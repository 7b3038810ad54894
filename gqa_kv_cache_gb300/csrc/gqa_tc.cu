// Tensor-core decode kernel, single-token instantiations (the decode step and
// the read-only attend); the kernel is in gqa_tc_kernel.cuh. This unit is
// compiled without the multi-token branches of the schedule.
#define GQA_MULTI_TOKEN 0
#include "gqa_tc_kernel.cuh"

namespace gqa {

bool tc_supports(bool bf16, int D, int G, bool paged, int block_size)
{
    // bf16: a bfloat16 or E4M3 cache (the kernel's two forms)
    if (!bf16 || D != kD || G < 1 || G > kGMax)
        return false;
    if (paged) {
        // blocks land on 1024-byte boundaries of the swizzled ring
        if (block_size < 8 || (block_size & (block_size - 1)))
            return false;
    }
    return true;
}

int tc_tile() { return kTile; }
int tc_ctas_per_sm(bool kv8, int unit_rows) { return (kv8 && unit_rows <= kGMax) ? kCtasPerSmKV8 : kCtasPerSm; }

cudaError_t tc_launch(const DecodeParams &p, const TcMaps &maps, cudaStream_t st)
{
    const bool win = p.window > 0;
    if (p.cu_q)     // multi-token steps (bfloat16 query)
        return tc_launch_multi(p, maps, st);
    if (p.kv8) {    // E4M3 cache
        if (p.q_bf16)
            return win ? launch_q<false, true, false, true>(p, maps, st)
                       : launch_q<false, false, false, true>(p, maps, st);
        return win ? launch_q<true, true, false, true>(p, maps, st) : launch_q<true, false, false, true>(p, maps, st);
    }
    if (p.q_bf16)
        return win ? launch_q<false, true, false>(p, maps, st) : launch_q<false, false, false>(p, maps, st);
    return win ? launch_q<true, true, false>(p, maps, st) : launch_q<true, false, false>(p, maps, st);
}

}  // namespace gqa
