// Decode kernel for small caches: one thread-block cluster per (batch row,
// cache head) unit, the unit's attended slots staged in the shared memory of
// its CTAs by bulk copies.
//
// When a row's capacity is a few hundred slots, the persistent kernels spend
// most of a step on their start (the schedule over all rows) and on merging
// the pieces of units cut between CTAs through global memory, and the
// CUDA-core kernel's slot loop waits on one global load after another. Here:
//  * the unit's staged rows -- its attended cached slots in order (the prefix
//    below a window's start, then the window), then in the decode step the
//    new token -- are shared out in contiguous parts, one per CTA of the
//    cluster (one CTA when the units already fill the SMs), so that several
//    SMs pull the unit from HBM at once;
//  * thread 0 of each CTA reads the row's length (and slot id) and issues one
//    bulk copy (cp.async.bulk, completing on an mbarrier) per contiguous run
//    of its part, of K and of V; for a paged cache the threads issue one copy
//    per block piece in parallel;
//  * meanwhile every lane loads its slice of the group's G query rows, and
//    the CTA holding the new token copies it into the cache slot lengths[b]
//    (the append);
//  * after the (bounded) wait, the eight warps score the staged slots from
//    shared memory with the CUDA-core kernel's lane layout (D / VEC lanes a
//    slot, VEC elements each, xor-shuffle dot products, an online softmax per
//    lane group), the lane groups and warps are merged (log-sum-exp) into one
//    state per CTA, and after a cluster barrier each CTA merges every CTA's
//    state for its share of the outputs through distributed shared memory,
//    folds in a sink logit and writes the normalised output. No workspace,
//    no global merge, no schedule.
// Every staged slot is attended, so nothing is masked; slots outside the
// window and stale slots are never read.
#pragma once

#include "gqa_common.cuh"
#include "gqa_launch.h"

namespace gqa {
namespace {

constexpr int kUnitWarps = 8;
constexpr int kUnitThreads = kUnitWarps * 32;
constexpr long long kUnitWaitCycles = 4LL << 30;   // about 2 s at 2 GHz: the limit of the drain after a timeout
constexpr int kUnitMaxCluster = 8;                  // CTAs a unit at most (the portable cluster size)

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
    int n_cached; // staged cached slots of the unit: pe + the window's cached part
    int append;   // decode step: the unit's last row is the new token
    int r0, r1;   // this CTA's rows of the unit's n_cached (+ 1 new) rows
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t n;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

// The cluster barrier in two halves: every thread of every CTA arrives, then
// waits for all the others. Release / acquire order the shared-memory writes
// before the arrival (this CTA's and remote ones) with the reads after the wait.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores v at the address of `local` in the shared memory of CTA `rank` of
// the cluster.
__device__ __forceinline__ void st_cluster(const void *local, uint32_t rank, float v)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(unit_smem(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_int(const void *local, uint32_t rank, int v)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(unit_smem(local)), "r"(rank));
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

// Bytes of the staging area of a CTA staging `rows` rows (K then V); it
// later holds the warps' states. In a cluster of several CTAs the CTA states
// follow it.
template <typename T, int D, int GP>
__host__ __device__ constexpr size_t unit_stage_bytes(int rows)
{
    const size_t stage = 2 * (size_t)rows * D * sizeof(T);
    const size_t warps = (size_t)kUnitWarps * GP * D * 4;
    return ((stage > warps ? stage : warps) + 15) / 16 * 16;
}

// Bounded wait for phase 0 of `bar`: false when it gave up after `limit`
// SM clock cycles (below 2^20 cycles with a one-nanosecond suspend hint, so
// a short limit is honoured to the cycle).
__device__ __forceinline__ bool unit_wait(uint32_t bar, long long limit)
{
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        if (limit < (1LL << 20))
            asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0, 1;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(ok)
                         : "r"(bar)
                         : "memory");
        else
            asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(ok)
                         : "r"(bar)
                         : "memory");
        if (ok)
            return true;
        if (clock64() - t0 > limit)
            return false;
    }
}

__device__ __forceinline__ void bulk_copy(const void *dst_smem, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(unit_smem(dst_smem)), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// One cluster of CTAs per (row, cache head) unit. The unit's staged rows (the
// attended cached slots in order, then in the decode step the new token) are
// shared out in contiguous parts, one per CTA of the cluster, so the copies
// into shared memory run on several SMs at once; each CTA merges its warps'
// states, and CTA 0 of the cluster merges the CTAs' states through
// distributed shared memory and writes the output.
template <typename T, int D, int GP>
__global__ void __launch_bounds__(kUnitThreads) unit_decode_kernel(const DecodeParams p, int rows_per_cta, bool spec)
{
    using S = UnitShape<T, D>;
    constexpr int VEC = S::VEC, LPS = S::LPS, SPW = S::SPW, STREAMS = S::STREAMS;
    constexpr int RB = S::kRowBytes;
    // dynamic: K rows, then V rows (rows_per_cta each); then (in a cluster)
    // [cluster][GP][D] CTA states (the unnormalised outputs), filled in CTA 0
    // by every CTA
    extern __shared__ __align__(128) uint8_t dyn[];
    __shared__ uint64_t bar;
    __shared__ uint64_t stall_bar;   // a barrier nothing completes (tests of the timeout path)
    __shared__ UnitInfo info;
    __shared__ int blk_bad;
    __shared__ float sm_m[kUnitWarps][GP], sm_l[kUnitWarps][GP];
    // CTA states in CTA 0: maximum, sum and error flag of every CTA
    __shared__ float pm[kUnitMaxCluster][GP], pl[kUnitMaxCluster][GP];
    __shared__ int pbad[kUnitMaxCluster];

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int lg = lane / LPS, li = lane % LPS;
    const uint32_t rank = cluster_rank(), ncta = cluster_size();
    const int u = blockIdx.x / ncta, b = u / p.Hkv, kvh = u % p.Hkv;
    const int G = p.G;
    T *sk = reinterpret_cast<T *>(dyn);
    T *sv = reinterpret_cast<T *>(dyn + (size_t)rows_per_cta * RB);
    // CTA states: after the staging area in a cluster (other CTAs store into
    // it while this one may still be staging or scoring); for a lone CTA on
    // its warps' states (state element i is written by the thread that alone
    // reads warp state element i of every warp)
    float *po = reinterpret_cast<float *>(dyn + (ncta > 1 ? unit_stage_bytes<T, D, GP>(rows_per_cta) : 0));
    const uint32_t bar_u = unit_smem(&bar);

    // `spec` (a dense cache without slot ids or window, the host's choice
    // when the whole capacity of every unit is a few MB): the CTA's rows are
    // its share of the row's capacity, rows [rank * rows_per_cta, ...), and
    // their copy starts before the row's length is read, so that the two HBM
    // round trips overlap. Rows at or past the length land too and are never
    // used (the copy may also meet the append of slot L: that row is not used
    // either). Otherwise the CTA's rows are an equal share of the unit's
    // staged rows, copied once the length is known.
    const int n_spec = spec ? max(0, min(rows_per_cta, p.Smax - (int)rank * rows_per_cta)) : 0;

    // first half of a cluster barrier: its wait, before the first store into
    // CTA 0, makes sure every CTA of the cluster has started
    cluster_arrive_relaxed();
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_u));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(unit_smem(&stall_bar)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        blk_bad = 0;
    }
    // a programmatic dependent of the previous kernel: read no input before it is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        if (n_spec > 0) {
            const long long off = (((long long)b * p.Hkv + kvh) * p.Smax + (long long)rank * rows_per_cta) * D;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_u),
                         "r"((uint32_t)n_spec * RB * 2u)
                         : "memory");
            bulk_copy(sk, static_cast<const T *>(p.k_cache) + off, (uint32_t)n_spec * RB, bar_u);
            bulk_copy(sv, static_cast<const T *>(p.v_cache) + off, (uint32_t)n_spec * RB, bar_u);
        }
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
        const int n_rows = f.bad ? 0 : f.n_cached + (f.append ? 1 : 0);
        const int part = spec ? rows_per_cta : (n_rows + (int)ncta - 1) / (int)ncta;
        f.r0 = min(n_rows, (int)rank * part);
        f.r1 = min(n_rows, f.r0 + part);
        // the copies of the CTA's cached rows, once the length is known: the
        // expected bytes posted before the barrier below, so before any copy
        // by another thread lands; dense ones issued here
        const int c0 = f.r0, c1 = min(f.r1, f.n_cached);
        if (!spec && c1 > c0) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_u),
                         "r"((uint32_t)(c1 - c0) * RB * 2u)
                         : "memory");
            if (!p.paged) {
                const long long row = p.slot_ids ? __ldg(p.slot_ids + b) : b;
                for (int k = 0; k < 2; ++k) {
                    // the rows of this part: staged indices [i0, i1), slots from s0
                    const int i0 = k ? max(c0, f.pe) : c0, i1 = k ? c1 : min(c1, f.pe);
                    if (i1 <= i0)
                        continue;
                    const int s0 = k ? f.lo + (i0 - f.pe) : i0, d0 = i0 - c0;
                    const long long off = ((row * p.Hkv + kvh) * p.Smax + s0) * (long long)D;
                    bulk_copy(sk + (long long)d0 * D, static_cast<const T *>(p.k_cache) + off,
                              (uint32_t)(i1 - i0) * RB, bar_u);
                    bulk_copy(sv + (long long)d0 * D, static_cast<const T *>(p.v_cache) + off,
                              (uint32_t)(i1 - i0) * RB, bar_u);
                }
            }
        }
        info = f;
    }
    __syncthreads();
    const UnitInfo f = info;
    // this CTA's cached rows [c0, c1) of the unit's staged order: index i is
    // slot i below the prefix end pe, else slot lo + (i - pe)
    const int c0 = f.r0, c1 = min(f.r1, f.n_cached);
    const bool staged = spec ? n_spec > 0 : c1 > c0;   // copies to wait for

    // ---- paged: one copy per block piece of the CTA's rows, issued by the
    // threads in parallel; an unusable table entry makes the row bad
    if (p.paged && c1 > c0) {
        for (int k = 0; k < 2; ++k) {
            const int i0 = k ? max(c0, f.pe) : c0, i1 = k ? c1 : min(c1, f.pe);
            if (i1 <= i0)
                continue;
            const int s0 = k ? f.lo + (i0 - f.pe) : i0, n = i1 - i0, d0 = i0 - c0;
            const int bs = p.block_size;
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
                bulk_copy(sk + (long long)dr * D, static_cast<const T *>(p.k_cache) + src, nb, bar_u);
                bulk_copy(sv + (long long)dr * D, static_cast<const T *>(p.v_cache) + src, nb, bar_u);
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
        if (g < G && f.r1 > f.r0) {
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
    // the new token: the CTA holding the unit's last row scores it from
    // k_new / v_new and appends it now, so the stores overlap the wait
    // (appending it at the end, after every CTA of the unit is known good,
    // cost pr1_fp32 0.2 us: a step that times out may therefore have
    // appended it); an unusable slot makes the unit bad
    const bool has_new = f.append && !f.bad && f.r1 > f.n_cached;
    const long long new_off = ((long long)b * p.Hkv + kvh) * D;
    if (has_new && tid < 2 * (RB / 16)) {
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

    // ---- wait for the staged rows, bounded by the launch's limit (tests of
    // the timeout path also wait on a barrier nothing completes, so the wait
    // runs out). A wait that ran out is followed by a drain with the full
    // limit, so that no copy still writes into shared memory when the CTA
    // exits.
    int timed_out = 0;
    if (staged) {
        bool ok = unit_wait(bar_u, p.wait_cycles);
        if (p.test_stall)
            ok = ok && unit_wait(unit_smem(&stall_bar), p.wait_cycles);
        if (!ok) {
            timed_out = 1;
            unit_wait(bar_u, kUnitWaitCycles);
        }
    }

    // ---- online softmax over this CTA's rows (cached rows from shared
    // memory; the new token from global memory)
    float m[GP], l[GP], o[GP][VEC];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            o[g][e] = 0.f;
    }
    const int n_mine = f.r1 - f.r0;
    // warp-uniform trip count: every lane takes part in the shuffles
    for (int rb = warp * SPW; rb < n_mine; rb += STREAMS) {
        const int r = rb + lg;            // local row
        float kv[VEC], vv[VEC];
        const bool use = r < n_mine;
        if (f.r0 + r < f.n_cached) {
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
    float *so = reinterpret_cast<float *>(dyn);                        // [kUnitWarps][GP][D]
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
    if (tid == 0) {
        if (f.bad && rank == 0)
            report(p, f.bad);
        else if (any_timeout)
            report(p, kTimeout);
        else if (blk_bad)
            report(p, kBadBlock);
    }
    // this CTA's state (the warps merged: maximum, sum, unnormalised output),
    // stored into CTA 0's slot `rank`
    cluster_wait();
    for (int idx = tid; idx < G * D; idx += kUnitThreads) {
        const int g = idx / D, d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kUnitWarps; ++w)
            M = fmaxf(M, sm_m[w][g]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kUnitWarps; ++w) {
            const float a = (sm_m[w][g] == -INFINITY) ? 0.f : unit_ex2(sm_m[w][g] - M);
            den = fmaf(a, sm_l[w][g], den);
            num = fmaf(a, so[(w * GP + g) * D + d], num);
        }
        st_cluster(po + (rank * GP + g) * D + d, 0, num);
        if (d == 0) {
            st_cluster(&pm[rank][g], 0, M);
            st_cluster(&pl[rank][g], 0, den);
        }
    }
    if (tid == 0)
        st_cluster_int(&pbad[rank], 0, blk_bad || any_timeout);
    cluster_arrive();
    cluster_wait();
    if (rank != 0)
        return;
    // CTA 0: every CTA's state merged (log-sum-exp rule) with the sink logit
    int any_bad = f.bad;
    for (uint32_t r = 0; r < ncta; ++r)
        any_bad |= pbad[r];
    const float qnan = __int_as_float(0x7fc00000);
    for (int idx = tid; idx < G * D; idx += kUnitThreads) {
        const int g = idx / D, d = idx - g * D;
        const float sk2 = p.sink ? sink_log2(p, kvh * G + g) : -INFINITY;
        float M = sk2;
        for (uint32_t r = 0; r < ncta; ++r)
            M = fmaxf(M, pm[r][g]);
        float num = 0.f, den = (sk2 == -INFINITY) ? 0.f : unit_ex2(sk2 - M);
        for (uint32_t r = 0; r < ncta; ++r) {
            const float a = (pm[r][g] == -INFINITY) ? 0.f : unit_ex2(pm[r][g] - M);
            den = fmaf(a, pl[r][g], den);
            num = fmaf(a, po[(r * GP + g) * D + d], num);
        }
        p.out[((long long)b * p.Hq + (long long)kvh * G + g) * D + d] = any_bad ? qnan : num / den;
    }
}

// Launches the instantiation: `cl` CTAs a cluster (one cluster per unit),
// each staging up to `rows` rows in `smem` bytes of dynamic shared memory,
// the copies started before the lengths are read when `spec`
// (the attribute is set on every launch: it is per device, and this path is
// for small steps where the host call does not matter).
template <typename T, int D, int GP>
cudaError_t unit_launch_one(const DecodeParams *p, int cl, int rows, bool spec, size_t smem, cudaStream_t st)
{
    const cudaError_t e = cudaFuncSetAttribute(unit_decode_kernel<T, D, GP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p->B * (unsigned)p->Hkv * (unsigned)cl);
    cfg.blockDim = dim3(kUnitThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, unit_decode_kernel<T, D, GP>, *p, rows, spec);
}

template <typename T, int D>
cudaError_t unit_launch_g(const DecodeParams *p, int cl, int rows, bool spec, size_t smem, cudaStream_t st)
{
    const int G = p->G;
    if (G == 1) return unit_launch_one<T, D, 1>(p, cl, rows, spec, smem, st);
    if (G == 2) return unit_launch_one<T, D, 2>(p, cl, rows, spec, smem, st);
    if (G <= 4) return unit_launch_one<T, D, 4>(p, cl, rows, spec, smem, st);
    if (G <= 6) return unit_launch_one<T, D, 6>(p, cl, rows, spec, smem, st);
    return unit_launch_one<T, D, 8>(p, cl, rows, spec, smem, st);
}

}  // namespace
}  // namespace gqa
