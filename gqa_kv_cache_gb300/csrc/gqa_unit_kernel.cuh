// Decode kernel for small caches: one CTA per (batch row, cache head) unit,
// the unit's attended slots staged whole in shared memory by bulk copies.
//
// When a row's capacity is a few hundred slots, the persistent kernels spend
// most of a step on their start (the schedule over all rows) and on merging
// the pieces of units cut between CTAs, and the CUDA-core kernel's slot loop
// waits on one global load after another. Here a unit never leaves its CTA:
//  * thread 0 reads the row's length (and slot id or block-table entries) and
//    issues one bulk copy (cp.async.bulk, completing on an mbarrier) per
//    contiguous run of attended cached slots of K and of V -- one per range
//    for a dense or slot-id cache (the prefix below a window's start, then the
//    window), one per block for a paged cache -- into rows of shared memory;
//  * meanwhile every lane loads its slice of the group's G query rows, and in
//    the decode step the new key / value are copied into the cache slot
//    lengths[b] (the append) and kept in registers by the lane group that
//    scores slot L;
//  * after the (bounded) wait, the eight warps score the staged slots from
//    shared memory with the CUDA-core kernel's lane layout (D / VEC lanes a
//    slot, VEC elements each, xor-shuffle dot products, an online softmax per
//    lane group), then the lane groups and warps are merged (log-sum-exp),
//    a sink logit is folded into the denominator, and the normalised output
//    is written. No workspace, no merge between CTAs, no schedule.
// Every staged slot is attended, so nothing is masked; slots outside the
// window and stale slots are never read.
#pragma once

#include "gqa_common.cuh"
#include "gqa_launch.h"

namespace gqa {
namespace {

constexpr int kUnitWarps = 8;
constexpr int kUnitThreads = kUnitWarps * 32;
constexpr long long kUnitWaitCycles = 4LL << 30;   // about 2 s at 2 GHz

template <typename T, int D>
struct UnitShape {
    static constexpr int kMinVec = 16 / (int)sizeof(T);  // elements in 16 bytes
    static constexpr int VEC = (D >= kMinVec * 32) ? D / 32 : (D < kMinVec ? D : kMinVec);
    static constexpr int LPS = D / VEC;                  // lanes per slot
    static constexpr int SPW = 32 / LPS;                 // slots per warp at once
    static constexpr int STREAMS = kUnitWarps * SPW;     // slots per CTA at once
    static constexpr int kRowBytes = D * (int)sizeof(T);
    static_assert(kRowBytes % 16 == 0, "rows must be whole 16-byte chunks for the bulk copies");
};

__device__ __forceinline__ float unit_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t unit_smem(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// VEC elements of T widened to float (p aligned to VEC * sizeof(T) bytes, a
// multiple of 4 bytes; 16 or more for the cache's own type).
template <typename T, int VEC>
__device__ __forceinline__ void unit_load(const T *p, float (&v)[VEC])
{
    constexpr int WORDS = VEC * (int)sizeof(T) / 4;
    uint32_t w[WORDS];
    const uint32_t *pw = reinterpret_cast<const uint32_t *>(p);
    if constexpr (WORDS >= 4) {
#pragma unroll
        for (int i = 0; i < WORDS; i += 4) {
            const uint4 a = *reinterpret_cast<const uint4 *>(pw + i);
            w[i] = a.x;
            w[i + 1] = a.y;
            w[i + 2] = a.z;
            w[i + 3] = a.w;
        }
    } else if constexpr (WORDS == 2) {
        const uint2 a = *reinterpret_cast<const uint2 *>(pw);
        w[0] = a.x;
        w[1] = a.y;
    } else {
        w[0] = *pw;
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

// Per-unit facts thread 0 finds and shares.
struct UnitInfo {
    int L;        // last attended slot (the query's position)
    int bad;      // content error bits of the row (0: good)
    int pe;       // staged prefix slots 0 .. pe-1 (below the window's start)
    int lo;       // first window slot (0 without a window)
    int n_cached; // staged cached slots: pe + the window's cached part
    int append;   // decode step: slot L holds the new token
};

template <typename T, int D, int GP>
__global__ void __launch_bounds__(kUnitThreads) unit_decode_kernel(const DecodeParams p)
{
    using S = UnitShape<T, D>;
    constexpr int VEC = S::VEC, LPS = S::LPS, SPW = S::SPW, STREAMS = S::STREAMS;
    constexpr int RB = S::kRowBytes;
    extern __shared__ __align__(128) uint8_t dyn[];   // K rows, then V rows (cap rows each)
    __shared__ uint64_t bar;
    __shared__ UnitInfo info;
    __shared__ int blk_bad;
    __shared__ float sm_m[kUnitWarps][GP], sm_l[kUnitWarps][GP];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int lg = lane / LPS, li = lane % LPS;
    const int u = blockIdx.x, b = u / p.Hkv, kvh = u % p.Hkv;
    const int G = p.G;
    const int cap = p.paged ? p.max_blocks * p.block_size : p.Smax;   // staging rows (host-checked)
    T *sk = reinterpret_cast<T *>(dyn);
    T *sv = reinterpret_cast<T *>(dyn + (size_t)cap * RB);
    const uint32_t bar_u = unit_smem(&bar);

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_u));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        blk_bad = 0;
    }
    // a programmatic dependent of the previous kernel: read no input before it is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        UnitInfo f;
        f.L = last_slot(p, b);
        f.bad = row_error_bits(p, b, f.L);
        f.append = !p.attend;
        f.lo = 0;
        f.pe = 0;
        f.n_cached = 0;
        if (!f.bad) {
            const int P = kept_prefix(p, b);
            const int last_cached = f.append ? f.L - 1 : f.L;
            if (p.window > 0) {
                f.lo = max(0, f.L - p.window + 1);
                f.pe = min(P, f.lo);
            }
            f.n_cached = f.pe + max(0, last_cached - f.lo + 1);
        }
        info = f;
    }
    __syncthreads();
    const UnitInfo f = info;

    // ---- stage the attended cached slots: bulk copies completing on `bar`
    if (!f.bad) {
        if (!p.paged) {
            if (tid == 0) {
                const long long row = p.slot_ids ? __ldg(p.slot_ids + b) : b;
                const T *kb = static_cast<const T *>(p.k_cache) + ((row * p.Hkv + kvh) * p.Smax) * (long long)D;
                const T *vb = static_cast<const T *>(p.v_cache) + ((row * p.Hkv + kvh) * p.Smax) * (long long)D;
                const uint32_t bytes = (uint32_t)f.n_cached * RB * 2u;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_u), "r"(bytes)
                             : "memory");
                // the prefix below the window, then the window's cached slots
                const int r0[2] = {0, f.lo}, n[2] = {f.pe, f.n_cached - f.pe}, dst[2] = {0, f.pe};
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    if (n[k] <= 0)
                        continue;
                    const uint32_t nb = (uint32_t)n[k] * RB;
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 ::"r"(unit_smem(sk) + dst[k] * RB), "l"(kb + (long long)r0[k] * D), "r"(nb), "r"(bar_u)
                                 : "memory");
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 ::"r"(unit_smem(sv) + dst[k] * RB), "l"(vb + (long long)r0[k] * D), "r"(nb), "r"(bar_u)
                                 : "memory");
                }
            }
        } else {
            // one copy per block and range piece, issued by the threads in
            // parallel; an unusable table entry makes the row bad
            const int bs = p.block_size;
            if (tid == 0)
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_u),
                             "r"((uint32_t)f.n_cached * RB * 2u)
                             : "memory");
            __syncthreads();   // the expected bytes are posted before any copy lands
            for (int k = 0; k < 2; ++k) {
                const int s0 = k ? f.lo : 0, n = k ? f.n_cached - f.pe : f.pe, d0 = k ? f.pe : 0;
                if (n <= 0)
                    continue;
                const int b0 = s0 / bs, b1 = (s0 + n - 1) / bs;
                for (int bi = b0 + tid; bi <= b1; bi += kUnitThreads) {
                    const int e = __ldg(p.block_table + (long long)b * p.max_blocks + bi);
                    const int a = max(s0, bi * bs), z = min(s0 + n, (bi + 1) * bs);   // slots [a, z)
                    const uint32_t nb = (uint32_t)(z - a) * RB;
                    if (e < 0 || e >= p.num_blocks) {
                        blk_bad = 1;
                        // nothing lands for these slots: complete their bytes by hand
                        asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar_u), "r"(2u * nb)
                                     : "memory");
                        continue;
                    }
                    const long long src = (((long long)e * p.Hkv + kvh) * bs + (a - bi * bs)) * D;
                    const int dr = d0 + (a - s0);
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 ::"r"(unit_smem(sk) + dr * RB), "l"(static_cast<const T *>(p.k_cache) + src), "r"(nb),
                                 "r"(bar_u)
                                 : "memory");
                    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                                 ::"r"(unit_smem(sv) + dr * RB), "l"(static_cast<const T *>(p.v_cache) + src), "r"(nb),
                                 "r"(bar_u)
                                 : "memory");
                }
            }
        }
    }

    // ---- the query slice of this lane (scores in base-2 units), the append
    float q[GP][VEC];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            q[g][e] = 0.f;
        if (g < G && !f.bad) {
            const long long qi = ((long long)b * p.Hq + (long long)kvh * G + g) * D + li * VEC;
            float tmp[VEC];
            if (p.q_bf16)
                unit_load<__nv_bfloat16, VEC>(static_cast<const __nv_bfloat16 *>(p.q) + qi, tmp);
            else
                unit_load<float, VEC>(static_cast<const float *>(p.q) + qi, tmp);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                q[g][e] = tmp[e] * p.scale_log2;
        }
    }
    // the new token: kept by the lane group that takes the last staged row
    const int n_rows = f.bad ? 0 : f.n_cached + (f.append ? 1 : 0);
    const long long new_off = ((long long)b * p.Hkv + kvh) * D;
    if (f.append && !f.bad && tid < 2 * (RB / 16)) {
        // the in-place append: 16-byte chunks of K (first half of the threads) and V
        const int c = tid % (RB / 16);
        const bool is_k = tid < RB / 16;
        const long long off = slot_offset(p, b, kvh, f.L);
        if (off >= 0) {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const T *>(is_k ? p.k_new : p.v_new) + new_off);
            reinterpret_cast<uint4 *>(static_cast<T *>(is_k ? p.k_cache : p.v_cache) + off)[c] = __ldg(src + c);
        } else if (c == 0) {
            blk_bad = 1;
        }
    }

    // ---- wait for the staged rows (bounded; the copies land whatever happens)
    int timed_out = 0;
    if (!f.bad && f.n_cached > 0) {
        uint32_t ok = 0;
        const long long t0 = clock64();
        while (true) {
            asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(ok)
                         : "r"(bar_u)
                         : "memory");
            if (ok || clock64() - t0 > kUnitWaitCycles)
                break;
        }
        timed_out = ok ? 0 : 1;
    }

    // ---- online softmax over the staged rows (row r < n_cached: shared
    // memory; the last row of the decode step: the new token)
    float m[GP], l[GP], o[GP][VEC];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            o[g][e] = 0.f;
    }
    // warp-uniform trip count: every lane takes part in the shuffles
    for (int rb = warp * SPW; rb < n_rows; rb += STREAMS) {
        const int r = rb + lg;
        float kv[VEC], vv[VEC];
        const bool use = r < n_rows;
        if (r < f.n_cached) {
            unit_load<T, VEC>(sk + (long long)r * D + li * VEC, kv);
            unit_load<T, VEC>(sv + (long long)r * D + li * VEC, vv);
        } else if (use) {
            unit_load<T, VEC>(static_cast<const T *>(p.k_new) + new_off + li * VEC, kv);
            unit_load<T, VEC>(static_cast<const T *>(p.v_new) + new_off + li * VEC, vv);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                kv[e] = vv[e] = 0.f;
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
                const float mn = fmaxf(m[g], s[g]);
                const float alpha = unit_ex2(m[g] - mn);   // m = -inf gives 0
                const float pj = unit_ex2(s[g] - mn);
                m[g] = mn;
                l[g] = l[g] * alpha + pj;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    o[g][e] = fmaf(pj, vv[e], o[g][e] * alpha);
            }
        }
    }
    // lane groups of a warp -> one state (log-sum-exp rule)
#pragma unroll
    for (int off = LPS; off < 32; off <<= 1) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m[g], off);
            const float l2 = __shfl_xor_sync(0xffffffffu, l[g], off);
            const float M = fmaxf(m[g], m2);
            const float a1 = (m[g] == -INFINITY) ? 0.f : unit_ex2(m[g] - M);
            const float a2 = (m2 == -INFINITY) ? 0.f : unit_ex2(m2 - M);
            m[g] = M;
            l[g] = a1 * l[g] + a2 * l2;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float o2 = __shfl_xor_sync(0xffffffffu, o[g][e], off);
                o[g][e] = a1 * o[g][e] + a2 * o2;
            }
        }
    }
    // warps -> shared memory (the staging area is free once every warp is done)
    __syncthreads();
    float *so = reinterpret_cast<float *>(dyn);   // [kUnitWarps][GP][D]
    if (lg == 0) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            if (li == 0) {
                sm_m[warp][g] = m[g];
                sm_l[warp][g] = l[g];
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                so[(warp * GP + g) * D + li * VEC + e] = o[g][e];
        }
    }
    const int any_timeout = __syncthreads_or(timed_out);
    const bool bad = f.bad || blk_bad || any_timeout;
    if (tid == 0) {
        if (f.bad)
            report(p, f.bad);
        else if (any_timeout)
            report(p, kTimeout);
        else if (blk_bad)
            report(p, kBadBlock);
    }
    const float qnan = __int_as_float(0x7fc00000);
    for (int idx = tid; idx < G * D; idx += kUnitThreads) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kUnitWarps; ++w)
            M = fmaxf(M, sm_m[w][g]);
        const float sk2 = p.sink ? sink_log2(p, kvh * G + g) : -INFINITY;
        M = fmaxf(M, sk2);
        float num = 0.f, den = (sk2 == -INFINITY) ? 0.f : unit_ex2(sk2 - M);
#pragma unroll
        for (int w = 0; w < kUnitWarps; ++w) {
            const float a = (sm_m[w][g] == -INFINITY) ? 0.f : unit_ex2(sm_m[w][g] - M);
            den = fmaf(a, sm_l[w][g], den);
            num = fmaf(a, so[(w * GP + g) * D + d], num);
        }
        p.out[((long long)b * p.Hq + (long long)kvh * G + g) * D + d] = bad ? qnan : num / den;
    }
}

// Launches the instantiation with `smem` bytes of dynamic shared memory (the
// attribute is set on every launch: it is per device, and this path is for
// small steps where the host call does not matter).
template <typename T, int D, int GP>
cudaError_t unit_launch_one(const DecodeParams *p, size_t smem, cudaStream_t st)
{
    const cudaError_t e = cudaFuncSetAttribute(unit_decode_kernel<T, D, GP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p->B * (unsigned)p->Hkv);
    cfg.blockDim = dim3(kUnitThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, unit_decode_kernel<T, D, GP>, *p);
}

template <typename T, int D>
cudaError_t unit_launch_g(const DecodeParams *p, size_t smem, cudaStream_t st)
{
    const int G = p->G;
    if (G == 1) return unit_launch_one<T, D, 1>(p, smem, st);
    if (G == 2) return unit_launch_one<T, D, 2>(p, smem, st);
    if (G <= 4) return unit_launch_one<T, D, 4>(p, smem, st);
    if (G <= 6) return unit_launch_one<T, D, 6>(p, smem, st);
    return unit_launch_one<T, D, 8>(p, smem, st);
}

}  // namespace
}  // namespace gqa
