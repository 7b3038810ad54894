// CUDA-core decode kernel instantiations: __nv_bfloat16, D in {32, 64, 128, 256}
// (the kernel is in gqa_simt_kernel.cuh).
#include "gqa_simt_kernel.cuh"

namespace gqa {

cudaError_t GQA_SIMT_FN(simt_launch_bf16_large)(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm)
{
    switch (D) {
    case 32: return launch_g<__nv_bfloat16, 32, kSimtGen>(G, p, st, per_sm);
    case 64: return launch_g<__nv_bfloat16, 64, kSimtGen>(G, p, st, per_sm);
    case 128: return launch_g<__nv_bfloat16, 128, kSimtGen>(G, p, st, per_sm);
    case 256: return launch_g<__nv_bfloat16, 256, kSimtGen>(G, p, st, per_sm);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gqa
