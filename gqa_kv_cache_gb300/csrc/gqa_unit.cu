// Decode kernel for small caches (one cluster of CTAs per unit, the unit
// staged in their shared memory): sizing, the cluster size, the choice of
// instantiation and the launch. The kernel is in gqa_unit_kernel.cuh.
#include "gqa_unit_kernel.cuh"

namespace gqa {

namespace {

constexpr size_t kUnitSmemMax = 200 * 1024;   // dynamic shared memory a CTA may take
constexpr long long kUnitMinRows = 32;          // staged rows a CTA at least, when a unit is split
// Capacity bytes of all units up to which a dense step stages every row's
// whole capacity before its length is known (under a microsecond of HBM
// time, spent to hide one HBM round trip).
constexpr long long kUnitSpecBytes = 4LL << 20;

int padded_g(int G) { return G <= 2 ? G : (G <= 4 ? 4 : (G <= 6 ? 6 : 8)); }

}  // namespace

// Dynamic shared memory of a CTA staging `rows` rows of K and of V in a
// cluster of `cl` CTAs: the staging area (which later holds the warps'
// states), then for cl > 1 the cluster's CTA states (the kernel's
// unit_stage_bytes layout; a lone CTA keeps its state on the warps' states).
size_t unit_smem_bytes(bool bf16, int D, int G, long long rows, int cl)
{
    const size_t es = bf16 ? 2 : 4, gp = (size_t)padded_g(G);
    const size_t stage = 2 * (size_t)rows * (size_t)D * es;
    const size_t warps = (size_t)kUnitWarps * gp * (size_t)D * 4;
    return ((stage > warps ? stage : warps) + 15) / 16 * 16 + (cl > 1 ? (size_t)cl * gp * (size_t)D * 4 : 0);
}

// CTAs a unit: the units spread over the SMs, so that more SMs copy at once
// (a power of two up to the portable cluster size, and no CTA with fewer
// than kUnitMinRows of the capacity's rows).
int unit_cluster(long long cap_rows, long long units, int sms)
{
    int cl = 1;
    while (cl < kUnitMaxCluster && units * (cl * 2) <= sms && (cap_rows + cl * 2 - 1) / (cl * 2) >= kUnitMinRows)
        cl *= 2;
    return cl;
}

bool unit_supports(bool bf16, int D, int G, long long cap_rows)
{
    if (G < 1 || G > 8 || cap_rows < 1)
        return false;
    if (D != 32 && D != 64 && D != 128 && D != 256)
        return false;
    return unit_smem_bytes(bf16, D, G, cap_rows, 1) <= kUnitSmemMax;
}

// Resident CTAs of the instantiation per SM with its shared memory (0 on error).
int unit_ctas_per_sm(bool bf16, int D, int G, long long cap_rows)
{
    const size_t smem = unit_smem_bytes(bf16, D, G, cap_rows, 1);
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

cudaError_t unit_launch(const DecodeParams &p, bool bf16, long long cap_rows, int sms, cudaStream_t st)
{
    const long long units = (long long)p.B * p.Hkv;
    const int cl = unit_cluster(cap_rows, units, sms);
    const int rows = (int)((cap_rows + cl - 1) / cl);
    const size_t smem = unit_smem_bytes(bf16, p.D, p.G, rows, cl);
    const long long cap_bytes = units * cap_rows * 2 * p.D * (bf16 ? 2 : 4);
    const bool spec = !p.paged && !p.slot_ids && p.window <= 0 && cap_bytes <= kUnitSpecBytes;
#define GQA_UNIT_LAUNCH(DD)                                                                                 \
    case DD:                                                                                                \
        return bf16 ? unit_launch_g<__nv_bfloat16, DD>(&p, cl, rows, spec, smem, st)                        \
                    : unit_launch_g<float, DD>(&p, cl, rows, spec, smem, st);
    switch (p.D) {
        GQA_UNIT_LAUNCH(32)
        GQA_UNIT_LAUNCH(64)
        GQA_UNIT_LAUNCH(128)
        GQA_UNIT_LAUNCH(256)
    }
#undef GQA_UNIT_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace gqa
