// CUDA-core decode kernel: host-side dispatch over the instantiations (the
// kernel itself is in gqa_simt_kernel.cuh, its instantiations in
// gqa_simt_{f32,bf16}_{small,large}[_plain].cu: the general form for
// multi-token steps and windows, the plain form for the rest).
#include "gqa_simt_kernel.cuh"

namespace gqa {
namespace {

cudaError_t launch_any(bool bf16, int D, int G, bool gen, const DecodeParams *p, cudaStream_t st, int *per_sm)
{
    if (gen) {
        if (bf16)
            return D <= 16 ? simt_launch_bf16_small(D, G, p, st, per_sm) : simt_launch_bf16_large(D, G, p, st, per_sm);
        return D <= 16 ? simt_launch_f32_small(D, G, p, st, per_sm) : simt_launch_f32_large(D, G, p, st, per_sm);
    }
    if (bf16)
        return D <= 16 ? simt_launch_bf16_small_plain(D, G, p, st, per_sm)
                       : simt_launch_bf16_large_plain(D, G, p, st, per_sm);
    return D <= 16 ? simt_launch_f32_small_plain(D, G, p, st, per_sm) : simt_launch_f32_large_plain(D, G, p, st, per_sm);
}

}  // namespace

bool simt_supports(int D, int G)
{
    return G >= 1 && G <= 8 && D >= 1 && D <= 256 && (D & (D - 1)) == 0;
}

int simt_tile() { return kSimtTile; }

// CTAs of the general form that fit on an SM (the grid of both forms: the
// plain form needs no more registers, and the workspace is sized by the grid)
int simt_ctas_per_sm(bool bf16, int D, int G)
{
    int n = 0;
    cudaError_t e = launch_any(bf16, D, G, true, nullptr, nullptr, &n);
    return (e == cudaSuccess && n > 0) ? n : 1;
}

cudaError_t simt_launch(const DecodeParams &p, bool bf16, cudaStream_t st)
{
    return launch_any(bf16, p.D, p.G, p.cu_q != nullptr || p.window > 0, &p, st, nullptr);
}

}  // namespace gqa
