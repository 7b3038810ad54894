// Tensor-core decode kernel, multi-token instantiations (bfloat16 query over a
// bfloat16 or E4M3 cache); the kernel is in gqa_tc_kernel.cuh.
#include "gqa_tc_kernel.cuh"

namespace gqa {

cudaError_t tc_launch_multi(const DecodeParams &p, const TcMaps &maps, cudaStream_t st)
{
    if (!p.q_bf16)
        return cudaErrorInvalidValue;
    if (p.kv8)
        return p.window > 0 ? launch_q<false, true, true, true>(p, maps, st)
                            : launch_q<false, false, true, true>(p, maps, st);
    return p.window > 0 ? launch_q<false, true, true>(p, maps, st) : launch_q<false, false, true>(p, maps, st);
}

}  // namespace gqa
