// Decode kernel for small caches (one CTA per unit, the unit staged in shared
// memory): sizing, the choice of instantiation and the launch. The kernel is
// in gqa_unit_kernel.cuh.
#include "gqa_unit_kernel.cuh"

namespace gqa {

namespace {

constexpr size_t kUnitSmemMax = 200 * 1024;   // dynamic shared memory a CTA may take

int padded_g(int G) { return G <= 2 ? G : (G <= 4 ? 4 : (G <= 6 ? 6 : 8)); }

}  // namespace

size_t unit_smem_bytes(bool bf16, int D, int G, long long cap_rows)
{
    const size_t es = bf16 ? 2 : 4;
    const size_t stage = 2 * (size_t)cap_rows * (size_t)D * es;
    const size_t merge = (size_t)kUnitWarps * (size_t)padded_g(G) * (size_t)D * 4;
    return stage > merge ? stage : merge;
}

bool unit_supports(bool bf16, int D, int G, long long cap_rows)
{
    if (G < 1 || G > 8 || cap_rows < 1)
        return false;
    if (D != 32 && D != 64 && D != 128 && D != 256)
        return false;
    return unit_smem_bytes(bf16, D, G, cap_rows) <= kUnitSmemMax;
}

// Resident CTAs of the instantiation per SM with its shared memory (0 on error).
int unit_ctas_per_sm(bool bf16, int D, int G, long long cap_rows)
{
    const size_t smem = unit_smem_bytes(bf16, D, G, cap_rows);
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
    const int gp = padded_g(G);
#define GQA_UNIT_OCC(T, DD)                                                                                 \
    if (D == DD) {                                                                                          \
        const void *f = gp == 1   ? (const void *)unit_decode_kernel<T, DD, 1>                              \
                        : gp == 2 ? (const void *)unit_decode_kernel<T, DD, 2>                              \
                        : gp == 4 ? (const void *)unit_decode_kernel<T, DD, 4>                              \
                        : gp == 6 ? (const void *)unit_decode_kernel<T, DD, 6>                              \
                                  : (const void *)unit_decode_kernel<T, DD, 8>;                             \
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);                \
        if (e == cudaSuccess)                                                                               \
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kUnitThreads, smem);                   \
    }
    if (bf16) {
        GQA_UNIT_OCC(__nv_bfloat16, 32) GQA_UNIT_OCC(__nv_bfloat16, 64) GQA_UNIT_OCC(__nv_bfloat16, 128)
        GQA_UNIT_OCC(__nv_bfloat16, 256)
    } else {
        GQA_UNIT_OCC(float, 32) GQA_UNIT_OCC(float, 64) GQA_UNIT_OCC(float, 128) GQA_UNIT_OCC(float, 256)
    }
#undef GQA_UNIT_OCC
    return e == cudaSuccess ? n : 0;
}

cudaError_t unit_launch(const DecodeParams &p, bool bf16, long long cap_rows, cudaStream_t st)
{
    const size_t smem = unit_smem_bytes(bf16, p.D, p.G, cap_rows);
    switch (p.D) {
    case 32: return bf16 ? unit_launch_g<__nv_bfloat16, 32>(&p, smem, st) : unit_launch_g<float, 32>(&p, smem, st);
    case 64: return bf16 ? unit_launch_g<__nv_bfloat16, 64>(&p, smem, st) : unit_launch_g<float, 64>(&p, smem, st);
    case 128: return bf16 ? unit_launch_g<__nv_bfloat16, 128>(&p, smem, st) : unit_launch_g<float, 128>(&p, smem, st);
    case 256: return bf16 ? unit_launch_g<__nv_bfloat16, 256>(&p, smem, st) : unit_launch_g<float, 256>(&p, smem, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gqa
