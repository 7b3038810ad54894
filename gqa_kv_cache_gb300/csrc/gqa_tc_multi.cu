// Tensor-core decode kernel, multi-token instantiations (bfloat16 query over a
// bfloat16 or E4M3 cache); the kernels are in gqa_tc_kernel.cuh (mma.sync)
// and gqa_tc5_kernel.cuh (tcgen05, units of 17 to 32 rows over bf16).
#include "gqa_tc5_kernel.cuh"

namespace gqa {

cudaError_t tc_launch_multi(const DecodeParams &p, const TcMaps &maps, cudaStream_t st)
{
    if (!p.q_bf16)
        return cudaErrorInvalidValue;
    const bool win = p.window > 0;
    // units of more than 8 query rows keep the rows on the M = 16 side: up
    // to 16 one M tile per warp, up to 32 two warps per M tile
    if (p.G > 16) {
        if (p.kv8)
            return win ? launch_q<false, true, true, true, 32>(p, maps, st)
                       : launch_q<false, false, true, true, 32>(p, maps, st);
        return win ? launch_q<false, true, true, false, 32>(p, maps, st)
                   : launch_q<false, false, true, false, 32>(p, maps, st);
    }
    if (p.G > 8) {
        if (p.kv8)
            return win ? launch_q<false, true, true, true, 16>(p, maps, st)
                       : launch_q<false, false, true, true, 16>(p, maps, st);
        return win ? launch_q<false, true, true, false, 16>(p, maps, st)
                   : launch_q<false, false, true, false, 16>(p, maps, st);
    }
    if (p.kv8)
        return win ? launch_q<false, true, true, true, 0>(p, maps, st)
                   : launch_q<false, false, true, true, 0>(p, maps, st);
    return win ? launch_q<false, true, true, false, 0>(p, maps, st)
               : launch_q<false, false, true, false, 0>(p, maps, st);
}

bool tc5_takes(const DecodeParams &p) { return p.q_bf16 && !p.kv8 && p.G > 16 && p.G <= kT5Rows; }

cudaError_t tc5_launch_multi(const DecodeParams &p, const TcMaps &maps, cudaStream_t st)
{
    if (!tc5_takes(p))
        return tc_launch_multi(p, maps, st);
    return p.window > 0 ? launch_t5<true>(p, maps, st) : launch_t5<false>(p, maps, st);
}

}  // namespace gqa
