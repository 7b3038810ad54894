// CUDA-core decode kernel instantiations: float, D in {1, 2, 4, 8, 16}
// (the kernel is in gqa_simt_kernel.cuh).
#include "gqa_simt_kernel.cuh"

namespace gqa {

cudaError_t GQA_SIMT_FN(simt_launch_f32_small)(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm)
{
    switch (D) {
    case 1: return launch_g<float, 1, kSimtGen>(G, p, st, per_sm);
    case 2: return launch_g<float, 2, kSimtGen>(G, p, st, per_sm);
    case 4: return launch_g<float, 4, kSimtGen>(G, p, st, per_sm);
    case 8: return launch_g<float, 8, kSimtGen>(G, p, st, per_sm);
    case 16: return launch_g<float, 16, kSimtGen>(G, p, st, per_sm);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gqa
