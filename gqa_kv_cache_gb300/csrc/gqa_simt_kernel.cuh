// CUDA-core (FMA) decode kernel: the general path (float32 or bfloat16 cache,
// float32 or bfloat16 query, any power-of-two head width up to 256, group
// size up to 8, dense / slot_ids / paged addressing with any block size; the
// decode step and the read-only attend).
//
// One persistent CTA of 4 warps walks its contiguous share of the tile list
// (see gqa_common.cuh). Inside a tile, a group of LPS = D / VEC lanes owns
// one slot at a time, each lane VEC consecutive elements loaded with one
// 16-byte (or narrower) load; a warp holds 32 / LPS slots at once. Per slot
// the G partial dot products are summed across the lane group with xor
// shuffles, each lane group keeps its own online-softmax state (running
// base-2 max m, sum l, and its VEC columns of o for every head), and at the
// end of a unit segment the states of all lane groups and warps are merged
// with the log-sum-exp rule (finish_segment, which also merges the units cut
// by CTA boundaries). In the decode step the new token (slot L) is read from
// k_new/v_new directly and written into the cache by the lane group that
// reads it; no thread reads the cache at slot L, so the append cannot race.
// The read-only attend reads slot L from the cache and writes nothing but out.
// In a multi-token step every slot from the row's write offset on is a new
// token, read from k_new / v_new (and appended by the chunk that owns it), and
// each query row (token, head) is masked beyond its own token's position.
//
// GEN: the general form (multi-token steps, sliding windows). The plain
// single-token forms (decode step and attend without a window) are compiled
// without the per-row bounds and, in their own translation units, without the
// multi-token schedule branches (GQA_SIMT_GEN 0, GQA_MULTI_TOKEN 0): measured,
// the general code cost the plain step about 20 %.
#pragma once

#ifndef GQA_SIMT_GEN
#define GQA_SIMT_GEN 1
#endif
#if GQA_SIMT_GEN
#define GQA_SIMT_FN(name) name
#else
#define GQA_SIMT_FN(name) name##_plain
#endif

#include "gqa_common.cuh"
#include "gqa_launch.h"

namespace gqa {
namespace {

constexpr bool kSimtGen = GQA_SIMT_GEN;

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kSimtTile = 64;

template <typename T, int D>
struct SimtShape {
    static constexpr int kMinVec = 16 / (int)sizeof(T);  // elements in 16 bytes
    static constexpr int VEC = (D >= kMinVec * 32) ? D / 32 : (D < kMinVec ? D : kMinVec);
    static constexpr int LPS = D / VEC;                  // lanes per slot
    static constexpr int SPW = 32 / LPS;                 // slots per warp at once
    static constexpr int STREAMS = kWarps * SPW;         // slots per CTA at once
    static_assert(LPS >= 1 && LPS <= 32 && (LPS & (LPS - 1)) == 0, "D must be a power of two <= 256");
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// VEC elements at p (aligned to VEC * sizeof(T) bytes) widened to float.
template <typename T, int VEC>
__device__ __forceinline__ void load_vec(const T *p, float (&v)[VEC])
{
    constexpr int BYTES = VEC * (int)sizeof(T);
    uint32_t w[(BYTES + 3) / 4];
    if constexpr (BYTES == 32) {
        uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
        uint4 b = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (BYTES == 16) {
        uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    } else if constexpr (BYTES == 8) {
        uint2 a = __ldg(reinterpret_cast<const uint2 *>(p));
        w[0] = a.x; w[1] = a.y;
    } else if constexpr (BYTES == 4) {
        w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
    } else {
        w[0] = __ldg(reinterpret_cast<const unsigned short *>(p));
    }
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            v[e] = __uint_as_float(w[e]);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            v[e] = (e & 1) ? bf16_hi(w[e / 2]) : bf16_lo(w[e / 2]);
    }
}

// VEC query elements at element index i, in the query's own dtype.
template <int VEC>
__device__ __forceinline__ void load_q(const DecodeParams &p, long long i, float (&v)[VEC])
{
    if (p.q_bf16)
        load_vec<__nv_bfloat16, VEC>(static_cast<const __nv_bfloat16 *>(p.q) + i, v);
    else
        load_vec<float, VEC>(static_cast<const float *>(p.q) + i, v);
}

// Raw copy of VEC elements (the append is a bit copy).
template <typename T, int VEC>
__device__ __forceinline__ void copy_vec(T *dst, const T *src)
{
    constexpr int BYTES = VEC * (int)sizeof(T);
    if constexpr (BYTES == 32) {
        reinterpret_cast<uint4 *>(dst)[0] = __ldg(reinterpret_cast<const uint4 *>(src));
        reinterpret_cast<uint4 *>(dst)[1] = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
    } else if constexpr (BYTES == 16) {
        *reinterpret_cast<uint4 *>(dst) = __ldg(reinterpret_cast<const uint4 *>(src));
    } else if constexpr (BYTES == 8) {
        *reinterpret_cast<uint2 *>(dst) = __ldg(reinterpret_cast<const uint2 *>(src));
    } else if constexpr (BYTES == 4) {
        *reinterpret_cast<unsigned int *>(dst) = __ldg(reinterpret_cast<const unsigned int *>(src));
    } else {
        *reinterpret_cast<unsigned short *>(dst) = __ldg(reinterpret_cast<const unsigned short *>(src));
    }
}

// Merge softmax state (m2, l2, o2) into (m1, l1, o1); max in base-2 units.
template <int GP, int VEC>
__device__ __forceinline__ void merge_state(float (&m1)[GP], float (&l1)[GP], float (&o1)[GP][VEC],
                                            const float (&m2)[GP], const float (&l2)[GP],
                                            const float (&o2)[GP][VEC])
{
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        float M = fmaxf(m1[g], m2[g]);
        float a1 = (m1[g] == -INFINITY) ? 0.f : ex2(m1[g] - M);
        float a2 = (m2[g] == -INFINITY) ? 0.f : ex2(m2[g] - M);
        m1[g] = M;
        l1[g] = a1 * l1[g] + a2 * l2[g];
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            o1[g][e] = a1 * o1[g][e] + a2 * o2[g][e];
    }
}

template <typename T, int D, int GP, bool GEN>
__global__ void __launch_bounds__(kThreads) simt_decode_kernel(const DecodeParams p)
{
    using S = SimtShape<T, D>;
    constexpr int VEC = S::VEC, LPS = S::LPS, SPW = S::SPW, STREAMS = S::STREAMS;

    __shared__ long long sched[kThreads / 32 + 8];
    __shared__ TileWalk walk;
    __shared__ int sm_flag;
    __shared__ MergeBuf sm_merge;
    __shared__ float sm_m[kWarps][GP], sm_l[kWarps][GP];
    __shared__ __align__(16) float sm_o[kWarps][GP][D];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int lg = lane / LPS, li = lane % LPS;
    const int G = p.G;
    const T *kc = static_cast<const T *>(p.k_cache);
    const T *vc = static_cast<const T *>(p.v_cache);

    // programmatic dependent of the previous kernel: read no input before it is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    schedule_walk(p, sched, &walk, (int)sizeof(T));   // also prefetches the first tiles into L2
    TileCursor cur;
    bool in_b = false;
    bool more = walk_first(p, cur, walk, in_b);

    float q[GP][VEC];
    float m[GP], l[GP], o[GP][VEC];
    int lim[GP];                  // each query row's last attended slot
    int seg_first_t = 0;
    bool row_good = true;
    bool seg_start = true;
    int bad_local = 0;

    while (more) {
        const int b = cur.b, kvh = cur.kvh, L = cur.L;
        if (seg_start) {
            seg_first_t = cur.t;
            row_good = row_ok(p, b, L);
            if (!row_good && tid == 0 && cur.t == 0 && kvh == 0)
                report(p, row_error_bits(p, b, L));
            const bool multi = GEN && p.cu_q;
            const int qrows = multi ? p.Gh * cur.nq : G;   // query rows with data
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                m[g] = -INFINITY;
                l[g] = 0.f;
                if constexpr (GEN)
                    lim[g] = multi ? L - (cur.nq - 1 - g / p.Gh) : L;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    o[g][e] = 0.f;
                if (g < qrows) {
                    float tmp[VEC];
                    // row g: token tok, head kvh * Gh + g % Gh
                    const long long tok = multi ? cur.tokL - (cur.nq - 1 - g / p.Gh) : b;
                    load_q<VEC>(p, (tok * p.Hq + (long long)kvh * p.Gh + g % p.Gh) * D + li * VEC, tmp);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        q[g][e] = tmp[e] * p.scale_log2;
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        q[g][e] = 0.f;
                }
            }
            seg_start = false;
        }

        if (row_good) {
            const int s0 = tile_slot0(cur, p.tile);
            const int s1 = min(s0 + p.tile, L + 1);
            // slots from here on are new tokens (none in the read-only attend)
            const bool multi = GEN && p.cu_q;
            const int first_new = p.attend ? INT_MAX : (multi ? cur.Lb : L);
            // warp-uniform trip count: every lane takes part in the shuffles
            for (int jb = s0 + warp * SPW; jb < s1; jb += STREAMS) {
                const int j = jb + lg;
                float kv[VEC], vv[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    kv[e] = vv[e] = 0.f;
                bool use = false;
                if (j < first_new) {
                    // without a window every slot up to L is attended (j may
                    // pass s1 in the tile's last lane groups)
                    if (GEN ? attended(L, cur.lo, cur.P, j) : j <= L) {
                        long long off = slot_offset(p, b, kvh, j);
                        if (off < 0) {
                            bad_local = 1;
                        } else {
                            load_vec<T, VEC>(kc + off + li * VEC, kv);
                            load_vec<T, VEC>(vc + off + li * VEC, vv);
                            use = true;
                        }
                    }
                } else if (j <= L) {  // a new token, and its in-place append
                    const long long tok = multi ? cur.tokL - (L - j) : b;
                    const long long new_off = (tok * p.Hkv + kvh) * D + li * VEC;
                    load_vec<T, VEC>(static_cast<const T *>(p.k_new) + new_off, kv);
                    load_vec<T, VEC>(static_cast<const T *>(p.v_new) + new_off, vv);
                    use = true;
                    // appended by the unit that owns the token
                    long long off = (!multi || j > L - cur.nq) ? slot_offset(p, b, kvh, j) : -2;
                    if (off >= 0) {
                        copy_vec<T, VEC>(static_cast<T *>(p.k_cache) + off + li * VEC,
                                         static_cast<const T *>(p.k_new) + new_off);
                        copy_vec<T, VEC>(static_cast<T *>(p.v_cache) + off + li * VEC,
                                         static_cast<const T *>(p.v_new) + new_off);
                    } else if (off == -1) {
                        bad_local = 1;
                    }
                }
                float s[GP];
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        acc = fmaf(q[g][e], kv[e], acc);
#pragma unroll
                    for (int off = LPS / 2; off > 0; off >>= 1)
                        acc += __shfl_xor_sync(0xffffffffu, acc, off);
                    s[g] = acc;
                }
                if (use) {
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        // row g's own causal bound and window
                        if (GEN && (j > lim[g] || (p.window > 0 && j <= lim[g] - p.window && j >= cur.P)))
                            continue;
                        float mn = fmaxf(m[g], s[g]);
                        float alpha = ex2(m[g] - mn);  // m = -inf gives 0
                        float pj = ex2(s[g] - mn);
                        m[g] = mn;
                        l[g] = l[g] * alpha + pj;
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            o[g][e] = fmaf(pj, vv[e], o[g][e] * alpha);
                    }
                }
            }
        }

        const bool unit_done = (cur.t == cur.nr - 1);
        const bool cta_done = (cur.g + 1 == cur.end);
        if (unit_done || cta_done) {
            // lane groups of a warp -> one state
#pragma unroll
            for (int off = LPS; off < 32; off <<= 1) {
                float m2[GP], l2[GP], o2[GP][VEC];
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    m2[g] = __shfl_xor_sync(0xffffffffu, m[g], off);
                    l2[g] = __shfl_xor_sync(0xffffffffu, l[g], off);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        o2[g][e] = __shfl_xor_sync(0xffffffffu, o[g][e], off);
                }
                merge_state<GP, VEC>(m, l, o, m2, l2, o2);
            }
            if (lg == 0) {
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    if (li == 0) {
                        sm_m[warp][g] = m[g];
                        sm_l[warp][g] = l[g];
                    }
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        sm_o[warp][g][li * VEC + e] = o[g][e];
                }
            }
            const bool seg_bad = __syncthreads_or(bad_local) != 0;
            bad_local = 0;
            const bool bad = !row_good || seg_bad;
            if (bad && row_good && tid == 0)
                report(p, kBadBlock);
            // the plain form's cursor carries no chunk fields (output row b)
            finish_segment<kWarps, GP, D, D, GEN>(p, cur, walk, seg_first_t, bad, sm_m, sm_l, sm_o, &sm_flag, sm_merge, tid,
                                          kThreads, [] { __syncthreads(); });
            seg_start = true;
        }
        more = walk_next(p, cur, walk, in_b);
    }
}

// Either launches the instantiation for (T, D, GP) or, with p == nullptr,
// reports how many of its CTAs fit on one SM.
template <typename T, int D, int GP, bool GEN>
cudaError_t launch_one(const DecodeParams *p, cudaStream_t st, int *per_sm)
{
    if (!p) {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, simt_decode_kernel<T, D, GP, GEN>,
                                                             kThreads, 0);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p->grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, simt_decode_kernel<T, D, GP, GEN>, *p);
}

template <typename T, int D, bool GEN>
cudaError_t launch_g(int G, const DecodeParams *p, cudaStream_t st, int *per_sm)
{
    if (G == 1) return launch_one<T, D, 1, GEN>(p, st, per_sm);
    if (G == 2) return launch_one<T, D, 2, GEN>(p, st, per_sm);
    if (G <= 4) return launch_one<T, D, 4, GEN>(p, st, per_sm);
    if (G <= 6) return launch_one<T, D, 6, GEN>(p, st, per_sm);
    return launch_one<T, D, 8, GEN>(p, st, per_sm);
}

}  // namespace

// The instantiations are spread over several translation units (by dtype,
// head width and form) so that they compile in parallel; each defines one of
// these (the _plain ones: GEN = false).
cudaError_t simt_launch_f32_small(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);
cudaError_t simt_launch_f32_large(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);
cudaError_t simt_launch_bf16_small(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);
cudaError_t simt_launch_bf16_large(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);
cudaError_t simt_launch_f32_small_plain(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);
cudaError_t simt_launch_f32_large_plain(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);
cudaError_t simt_launch_bf16_small_plain(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);
cudaError_t simt_launch_bf16_large_plain(int D, int G, const DecodeParams *p, cudaStream_t st, int *per_sm);

}  // namespace gqa
