// Multi-token units of 17 to 32 query rows on the fifth-generation tensor
// cores: tcgen05.mma with its accumulators in tensor memory (TMEM), bf16
// query over a bf16 cache.
//
// With 32 query rows a tile's products are four times those of a
// single-token unit, and on the warp-level mma.sync path they, not HBM, set
// the pace. Here one thread issues them to the tensor core and they run
// beside everything else:
//  * S = Q K^T (M = 128, N = 64 slots, K = 128 dims, eight steps of 16): the
//    unit's 32 query rows are rows 0-31 of M (rows 32-127 are never read:
//    their A rows are whatever lies in shared memory after the query rows,
//    their accumulator lanes are never loaded); K comes straight from the TMA
//    ring, whose 128-byte-swizzled 64-dim halves are the K-major SW128 layout
//    of the B operand. Two S buffers in TMEM (64 columns each) alternate.
//  * two softmax warps (0 and 4, both on TMEM lanes 0-31): lane r holds
//    query row r, warp 0 its scores of slots 0-31 of the tile, warp 4 of
//    slots 32-63; the partial row maxima are exchanged through shared
//    memory, the rest (the lazy rescale, the weights) is per-thread work, no
//    shuffles. Each writes its half of row r's weights (bf16) into one of two
//    P buffers in the K-major SW128 layout, and rescales and reads back its
//    64 dims of O.
//  * O += P V (M = 128, N = 128 dims, K = 64 slots, four steps of 16): A = P,
//    B = the V tile of the ring as an MN-major SW128 operand (dims
//    contiguous: leading offset = the 64-dim half, stride = 8 slot rows).
//    O (128 columns) stays in TMEM for the unit segment; a rescale of a row
//    (its running maximum up by more than 8, rare after the first tiles) is
//    a load, a multiply and a store of that row by its own thread.
//  * the MMA warp also substitutes the new tokens into the ring rows of the
//    tiles that hold them (and appends the ones its chunk owns), and zeroes
//    the V rows of slots no row attends, before the products of such a tile
//    (0 * NaN would not be 0).
//  * a producer warp fills the ring (TMA, as in the mma.sync kernel; the
//    segment's first tile also brings the query rows, copied by the softmax
//    warp into the swizzled A operand).
// Ordering: full[s] (TMA landed) -> S(i) -> s_ready -> softmax(i) -> P(i),
// p_ready -> O += P(i) V(i) -> pv_done, and the commit after it frees the
// ring stage. P(i) waits for the product of tile i - 2 (same P buffer); a
// rescale for the product of tile i - 1. At a segment's end the softmax
// warp reads O and writes the output (a whole unit) or the partial state;
// a cut unit's arrival ticket and merge run in the same warp. The next
// segment's query copy is signalled only after that, so its first product
// (which overwrites O) cannot start earlier.
// Every wait is bounded and abort-aware, as in the mma.sync kernel; at the
// end the MMA warp waits (bounded) for a commit covering all its products,
// and the producer for its copies, before TMEM is freed and the CTA exits.
#pragma once

#include "gqa_tc_kernel.cuh"

namespace gqa {
namespace {

constexpr int kT5Rows = 32;                                    // query rows of a unit
constexpr int kT5Stages = 2;
constexpr int kT5QBytes = kT5Rows * kD * 2;                    // the unit's query rows in a stage
constexpr int kT5StageBytes = 4 * kHalfBytes + kT5QBytes;      // K lo, K hi, V lo, V hi, Q (40 KB)
// Operands in front of the ring: Q dims 0-63 and Q dims 64-127, rows 0-63
// of each (the unit's 32 query rows twice: 8 KB), then P buffers 0 and 1,
// rows 0-31 of each (4 KB); each is read as 128 rows (16 KB), the rest
// landing on what follows (never used).
constexpr int kT5QOp = 8192, kT5POp = 2 * kT5QOp;
constexpr int kT5OpBytes = kT5POp + 2 * 4096;
constexpr int kT5DynSmem = kT5OpBytes + kT5Stages * kT5StageBytes + 1024;
// softmax (warp 0: TMEM lanes 0-31, warp 1: lanes 32-63, the same query
// rows), MMA (2), producer (3)
constexpr int kT5Threads = 4 * 32;
constexpr uint32_t kT5Cols = 256;                              // TMEM: S0, S1 (64 each), O (128)
static_assert(kT5StageBytes % 1024 == 0, "stages must stay 1024-byte aligned for the swizzle");
static_assert(kT5POp + 4096 + 16384 <= kT5OpBytes + kT5Stages * kT5StageBytes, "operand windows");

struct T5Shared {
    uint64_t full[kT5Stages];
    uint64_t empty[kT5Stages];
    uint64_t s_ready[2], p_ready[2], pv_done[2];
    uint64_t q_ready;
    uint64_t mma_done;
    uint64_t stall;       // a barrier nothing completes (tests of the timeout path)
    int stage_bad[kT5Stages];
    int abort_flag;
    uint32_t tmem;
    float xm[2][2][32];   // [tile parity][softmax warp][row]: partial row maxima of a tile
    float xl[2][32];      // [softmax warp][row]: partial row sums at a segment's end
    long long sched[kMaxWarps + 8];
    TileWalk walk;
    MergeBufT<kT5Rows, merge_partials(kT5Rows)> merge;
};

// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start
// address, leading and stride byte offsets (sm_100 form).
__device__ __forceinline__ uint64_t t5_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;     // descriptor version
    d |= (uint64_t)2 << 61;     // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, M x N, B
// K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t t5_idesc(int M, int N, int b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void t5_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)acc)
                 : "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void t5_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Whether the phase of `bar` with this parity has completed (never blocks).
__device__ __forceinline__ bool t5_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ void t5_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void t5_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (lane i of the
// warp: TMEM lane base + i).
__device__ __forceinline__ void t5_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void t5_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                   "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                   "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                   "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                   "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                   "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
                   "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                   "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
                   "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                   "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// The softmax and MMA warps (0, 1 and 2).
__device__ __forceinline__ void t5_end_sync() { asm volatile("bar.sync 1, 96;" ::: "memory"); }

// The two softmax warps (0 and 1): a barrier that also returns whether v
// held in any of their threads.
__device__ __forceinline__ bool t5_softmax_or(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, 2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v)
                 : "memory");
    return r != 0;
}

template <bool WIN>
__global__ void __launch_bounds__(kT5Threads, 2)
    tc5_multi_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                     const __grid_constant__ CUtensorMap mk16, const __grid_constant__ CUtensorMap mv16)
{
    extern __shared__ uint8_t dyn_smem[];
    __shared__ T5Shared sh;
    uint8_t *opnd = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = opnd + kT5OpBytes;
    const uint32_t op_u32 = smem_u32(opnd), ring_u32 = smem_u32(ring);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    if (tid == 0) {
        for (int s = 0; s < kT5Stages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 1);
            sh.stage_bad[s] = 0;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sh.s_ready[b]), 1);
            mbar_init(smem_u32(&sh.p_ready[b]), 2);   // both softmax warps
            mbar_init(smem_u32(&sh.pv_done[b]), 1);
        }
        mbar_init(smem_u32(&sh.q_ready), 1);
        mbar_init(smem_u32(&sh.mma_done), 1);
        mbar_init(smem_u32(&sh.stall), 1);
        sh.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem)),
                     "r"(kT5Cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        t5_fence_before();
    }
    if (warp == 3 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mv)) : "memory");
        if (!p.paged) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mk16)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mv16)) : "memory");
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    schedule_walk(p, sh.sched, &sh.walk, 2);   // contains __syncthreads (publishes the TMEM address too)
    t5_fence_after();
    const TileWalk &walk = sh.walk;
    const uint32_t tmem = sh.tmem;
    const __nv_bfloat16 *knew = static_cast<const __nv_bfloat16 *>(p.k_new);
    const __nv_bfloat16 *vnew = static_cast<const __nv_bfloat16 *>(p.v_new);

    if (warp == 3) {
        // ------------------------------------------------------ producer --
        uint64_t policy;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        TileCursor cur;
        bool in_b = false;
        bool more = walk_first(p, cur, walk, in_b);
        long long range_start = cur.g;
        int stage = 0;
        uint32_t phase = 0;
        const int bs = p.block_size;
        const int nblk = p.paged ? (bs < kTile ? kTile / bs : 1) : 1;
        const int box_rows = p.paged ? (bs < kTile ? bs : kTile) : kTile;
        struct Plan {
            int z, y;
            bool bad_entry, good;
            int rows;   // the tile's box height (warp-uniform)
        };
        auto plan = [&](const TileCursor &c) {
            Plan r{-1, 0, false, row_ok(p, c.b, c.L), box_rows};
            if (!r.good)
                return r;
            const int slot0 = WIN ? tile_slot0(c, kTile) : c.t * kTile;
            const int rb = real_row(p, c.b);
            if (!p.paged) {
                // a dense cache: one box for a tile read whole, else a small
                // box per part that holds a slot the step reads
                const int s = slot0 + lane * kDenseBoxRows;
                const bool need = lane < kTile / kDenseBoxRows && s <= c.L &&
                                  (!WIN || s + kDenseBoxRows - 1 >= c.lo || s < c.P);
                const unsigned parts = __ballot_sync(0xffffffffu, need);
                const bool whole = parts == (1u << (kTile / kDenseBoxRows)) - 1u;
                r.rows = whole ? kTile : kDenseBoxRows;
                if (whole ? lane == 0 : need) {
                    const int row = p.slot_ids ? __ldg(p.slot_ids + rb) : rb;
                    r.z = row * p.Hkv + c.kvh;
                    r.y = s;
                }
            } else if (lane < nblk) {
                const int s = slot0 + lane * box_rows;
                if (s <= c.L && (!WIN || s + box_rows - 1 >= c.lo || s < c.P)) {
                    const int e = __ldg(p.block_table + (long long)rb * p.max_blocks + s / bs);
                    if (e >= 0 && e < p.num_blocks) {
                        r.z = e * p.Hkv + c.kvh;
                        r.y = s % bs;
                    } else {
                        r.bad_entry = true;
                    }
                }
            }
            return r;
        };
        int issued = 0;
        Plan pl = more ? plan(cur) : Plan{-1, 0, false, false};
        while (more) {
            if (__any_sync(0xffffffffu, *((volatile int *)&sh.abort_flag) != 0))
                break;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&sh.empty[stage]), phase ^ 1, kWaitCycles, &sh.abort_flag))) {
                if (lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                    report(p, kTimeout);
                    atomicExch(&sh.abort_flag, 1);
                }
                break;
            }
            const unsigned copying = __ballot_sync(0xffffffffu, pl.z >= 0);
            const bool any_bad = __any_sync(0xffffffffu, pl.bad_entry);
            const bool seg_first = pl.good && (cur.t == 0 || cur.g == range_start);
            const uint32_t qbytes = seg_first ? (uint32_t)(p.Gh * cur.nq * kD * 2) : 0u;
            const uint32_t bytes = (uint32_t)__popc(copying) * 4u * (uint32_t)pl.rows * 128u + qbytes;
            const uint32_t fb = smem_u32(&sh.full[stage]);
            if (lane == 0) {
                sh.stage_bad[stage] = any_bad ? 1 : 0;
                mbar_arrive_tx(fb, bytes);
                if (qbytes) {
                    // one copy per token: its Gh heads are contiguous in q
                    const uint32_t qdst = ring_u32 + stage * kT5StageBytes + 4 * kHalfBytes;
                    const uint32_t tb = (uint32_t)(p.Gh * kD * 2);
                    for (int i = 0; i < cur.nq; ++i) {
                        const long long tok = cur.tokL - (cur.nq - 1 - i);
                        bulk_load(qdst + i * tb,
                                  static_cast<const uint8_t *>(p.q) + (tok * p.Hq + (long long)cur.kvh * p.Gh) * kD * 2,
                                  tb, fb);
                    }
                }
            }
            __syncwarp();
            if (pl.z >= 0) {
                if (pl.rows == box_rows) {   // a whole box (a paged block, a dense tile)
                    const uint32_t dst = ring_u32 + stage * kT5StageBytes + lane * box_rows * 128;
                    tma_load_3d(dst, &mk, 0, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + kHalfBytes, &mk, 64, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + 2 * kHalfBytes, &mv, 0, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + 3 * kHalfBytes, &mv, 64, pl.y, pl.z, fb, policy);
                } else {   // a part of a dense tile (the small-box maps)
                    const uint32_t dst = ring_u32 + stage * kT5StageBytes + lane * kDenseBoxRows * 128;
                    tma_load_3d(dst, &mk16, 0, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + kHalfBytes, &mk16, 64, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + 2 * kHalfBytes, &mv16, 0, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + 3 * kHalfBytes, &mv16, 64, pl.y, pl.z, fb, policy);
                }
            }
            ++issued;
            const bool was_b = in_b;
            more = walk_next(p, cur, walk, in_b);
            if (in_b != was_b)
                range_start = cur.g;
            if (more)
                pl = plan(cur);
            if (++stage == kT5Stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        asm volatile("griddepcontrol.launch_dependents;");
        // let every copy still in flight land before the warp exits (the last
        // min(stages, issued) stages are exactly those that can be)
        {
            int s = stage, ph = phase;
            for (int k = 0; k < kT5Stages && k < issued; ++k) {
                if (--s < 0) {
                    s = kT5Stages - 1;
                    ph ^= 1;
                }
                mbar_wait(smem_u32(&sh.full[s]), ph);
            }
        }
        return;
    }

    // Both other warps walk the same tiles in the same order.
    TileCursor cur;
    bool in_b = false;
    bool more = walk_first(p, cur, walk, in_b);
    long long range_start = cur.g;
    int stage = 0;
    uint32_t phase = 0;
    bool stall = p.test_stall != 0;     // the first wait also waits on sh.stall (runs out)
    const uint32_t idesc_s = t5_idesc(128, kTile, 0), idesc_o = t5_idesc(128, kD, 1);

    if (warp == 2) {
        // ----------------------------------------------------------- MMA --
        int i = 0;                           // tiles of this CTA so far
        bool pend = false, pend_acc = false; // a product O += P V still to issue
        int pend_i = 0, pend_stage = 0;
        uint32_t q_phase = 0;
        bool aborted = false;
        bool row_good = true;                // of the current segment's row
        auto issue_pv = [&](bool ready) {
            // O += P(pend_i) V(pend_i): waits for the weights of that tile
            // (unless already seen ready)
            const int bufp = pend_i & 1;
            bool ok = ready || (!aborted && __all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.p_ready[bufp]),
                                                                                (pend_i >> 1) & 1, p.wait_cycles,
                                                                                &sh.abort_flag)));
            if (!ok && !aborted && lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                report(p, kTimeout);
                atomicExch(&sh.abort_flag, 1);
            }
            aborted = aborted || !ok;
            if (ok && lane == 0) {
                t5_fence_after();
                const uint32_t pa = op_u32 + kT5POp + bufp * 4096;
                const uint32_t va = ring_u32 + pend_stage * kT5StageBytes + 2 * kHalfBytes;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    t5_mma(tmem + 128, t5_desc(pa + ks * 32, 16, 1024), t5_desc(va + ks * 2048, kHalfBytes, 1024),
                           idesc_o, pend_acc || ks > 0);
                t5_commit(smem_u32(&sh.pv_done[bufp]));
                t5_commit(smem_u32(&sh.empty[pend_stage]));   // the stage is free once this product is done
            }
            __syncwarp();
            pend = false;
        };
        while (more) {
            const int b = cur.b, kvh = cur.kvh, L = cur.L;
            const bool seg_first = cur.t == 0 || cur.g == range_start;
            bool have = false;
            if (!aborted && !__any_sync(0xffffffffu, *((volatile int *)&sh.abort_flag) != 0)) {
                // while tile i has not landed, the pending product is issued
                // as soon as its weights are ready (it frees its ring stage)
                // (bounded: past the limit the wait below gives up in turn)
                const uint32_t fb = smem_u32(&sh.full[stage]);
                const long long t0 = clock64();
                while (pend && !stall && !__all_sync(0xffffffffu, t5_test(fb, phase))) {
                    if (__all_sync(0xffffffffu, t5_test(smem_u32(&sh.p_ready[pend_i & 1]), (pend_i >> 1) & 1))) {
                        issue_pv(true);
                        break;
                    }
                    if (__any_sync(0xffffffffu, *((volatile int *)&sh.abort_flag) != 0 || clock64() - t0 > p.wait_cycles))
                        break;
                }
                bool ok = mbar_wait(fb, phase, p.wait_cycles, &sh.abort_flag);
                if (stall) {   // tests of the timeout path: a wait that nothing ends
                    ok = ok && mbar_wait(smem_u32(&sh.stall), 0, p.wait_cycles);
                    stall = false;
                }
                have = __all_sync(0xffffffffu, ok);
                if (!have && lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                    report(p, kTimeout);
                    atomicExch(&sh.abort_flag, 1);
                }
            }
            aborted = aborted || !have;
            // a segment's first product overwrites O: the previous segment's
            // last product goes first (the softmax warp reads O after it and
            // only then copies the next query)
            if (seg_first && pend)
                issue_pv(false);
            if (have && seg_first) {
                const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.q_ready), q_phase, p.wait_cycles,
                                                                  &sh.abort_flag));
                q_phase ^= 1;
                if (!ok && lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                    report(p, kTimeout);
                    atomicExch(&sh.abort_flag, 1);
                }
                aborted = aborted || !ok;
                have = have && ok;
            }
            if (seg_first)
                row_good = row_ok(p, b, L);
            const bool tile_bad = have ? sh.stage_bad[stage] != 0 : true;
            const int slot0 = WIN ? tile_slot0(cur, kTile) : cur.t * kTile;
            uint8_t *kring = ring + stage * kT5StageBytes;
            uint8_t *vring = kring + 2 * kHalfBytes;
            const bool newt = slot0 + kTile - 1 >= cur.Lb;
            const bool partial = newt || (WIN && slot0 < max(0, L - p.window + 1));
            if (have && row_good && !tile_bad && partial) {
                // rows holding new tokens: substituted from k_new / v_new (the
                // chunk that owns a token appends it); rows no query row
                // attends: zero V
                const int first_new = max(cur.Lb, slot0), last_new = min(L, slot0 + kTile - 1);
                for (int sn = first_new; sn <= last_new; ++sn) {
                    const int lr = sn - slot0;
                    const long long tok = cur.tokL - (L - sn);
                    const long long nidx = (tok * p.Hkv + kvh) * kD;
                    const int c = lane & 15;   // 16-byte chunk of the row
                    const uint4 *src = reinterpret_cast<const uint4 *>((lane < 16 ? knew : vnew) + nidx) + c;
                    const uint4 v = __ldg(src);
                    *reinterpret_cast<uint4 *>((lane < 16 ? kring : vring) + (c >> 3) * kHalfBytes + swz(lr, c & 7)) = v;
                    if (sn > L - cur.nq) {
                        const long long off = slot_offset(p, b, kvh, sn);
                        if (off >= 0) {
                            __nv_bfloat16 *cache = static_cast<__nv_bfloat16 *>(lane < 16 ? p.k_cache : p.v_cache);
                            reinterpret_cast<uint4 *>(cache + off)[c] = v;
                        }
                    }
                }
                for (int r = lane >> 4; r < kTile; r += 2) {
                    if (WIN ? !attended(L, cur.lo, cur.P, slot0 + r) : slot0 + r > L) {
                        const int c = lane & 15;
                        *reinterpret_cast<uint4 *>(vring + (c >> 3) * kHalfBytes + swz(r, c & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
            if (have) {
                // S(i) = Q K^T into S buffer i & 1 (its previous contents, of
                // tile i - 2, were read before the weights of i - 2 were
                // signalled, i.e. before the product of i - 2 was issued)
                if (lane == 0) {
                    t5_fence_after();
                    const uint32_t ka = ring_u32 + stage * kT5StageBytes;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t qo = (ks >> 2) * kT5QOp + (ks & 3) * 32, ko = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
                        t5_mma(tmem + (i & 1) * kTile, t5_desc(op_u32 + qo, 16, 1024), t5_desc(ka + ko, 16, 1024),
                               idesc_s, ks > 0);
                    }
                    t5_commit(smem_u32(&sh.s_ready[i & 1]));
                }
                __syncwarp();
            }
            if (pend)
                issue_pv(false);
            if (have) {
                pend = true;
                pend_i = i;
                pend_stage = stage;
                pend_acc = !seg_first;
            }
            ++i;
            const bool was_b = in_b;
            more = walk_next(p, cur, walk, in_b);
            if (in_b != was_b)
                range_start = cur.g;
            if (++stage == kT5Stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (pend)
            issue_pv(false);
        // every product issued has completed before TMEM is freed
        if (lane == 0)
            t5_commit(smem_u32(&sh.mma_done));
        __syncwarp();
        mbar_wait(smem_u32(&sh.mma_done), 0);
        t5_fence_before();
        t5_end_sync();
        return;
    }

    // ---------------------------------------------- softmax (warps 0 and 1) --
    // lane r: query row r of the unit, in TMEM lane r (warp 0) and lane
    // 32 + r (warp 1: the query rows are in A twice). Warp h takes slots
    // 32 h .. 32 h + 31 of every tile; they exchange their partial row maxima
    // every tile and their partial sums at a segment's end, so both keep the
    // same running maximum. Warp 0 also copies the query rows, rescales and
    // reads back O (rows 0-31), and takes a cut unit's ticket and merge.
    const int h = warp;
    const uint32_t tlane = (uint32_t)(32 * h) << 16;   // this warp's TMEM lanes
    const int r = lane;
    const float qnan = __int_as_float(0x7fc00000);
    int i = 0;
    int pv_seen[2] = {0, 0};             // products of each P buffer seen complete
    bool aborted = false;
    float m_run = -INFINITY, l_run = 0.f; // l_run: this warp's slots
    int lim = -1, lo_r = 0, seg_first_i = 0, seg_first_t = 0;
    bool seg_bad = false, row_good = true;
    // waits until the product of tile j (P buffer j & 1) is complete
    auto wait_pv = [&](int j) -> bool {
        const int bb = j & 1;
        if (pv_seen[bb] > (j >> 1))
            return true;
        const bool ok = !aborted && __all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.pv_done[bb]), (j >> 1) & 1,
                                                                        p.wait_cycles, &sh.abort_flag));
        if (ok) {
            pv_seen[bb] = (j >> 1) + 1;
            t5_fence_after();
        } else {
            if (!aborted && lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                report(p, kTimeout);
                atomicExch(&sh.abort_flag, 1);
            }
            aborted = true;
        }
        return ok;
    };
    while (more) {
        const int b = cur.b, kvh = cur.kvh, L = cur.L;
        const bool seg_first = cur.t == 0 || cur.g == range_start;
        bool have = false;
        if (!aborted && !__any_sync(0xffffffffu, *((volatile int *)&sh.abort_flag) != 0)) {
            bool ok = mbar_wait(smem_u32(&sh.full[stage]), phase, p.wait_cycles, &sh.abort_flag);
            if (stall) {
                ok = ok && mbar_wait(smem_u32(&sh.stall), 0, p.wait_cycles);
                stall = false;
            }
            have = __all_sync(0xffffffffu, ok);
            if (!have && lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                report(p, kTimeout);
                atomicExch(&sh.abort_flag, 1);
            }
        }
        aborted = aborted || !have;
        const int qrows = p.Gh * cur.nq;
        if (seg_first) {
            seg_first_i = i;
            seg_first_t = cur.t;
            row_good = row_ok(p, b, L);
            if (!row_good && h == 0 && lane == 0 && cur.t == 0 && kvh == 0)
                report(p, row_error_bits(p, b, L));
            seg_bad = false;
            m_run = -INFINITY;
            l_run = 0.f;
            // row r is token r / Gh of the chunk and attends up to its own position
            lim = r < qrows ? L - (cur.nq - 1 - r / p.Gh) : -1;
            lo_r = WIN ? max(0, lim - p.window + 1) : 0;
            if (have && h == 0) {
                // the query rows into the A operand (K-major, 128-byte swizzle),
                // as rows r and 32 + r
                const uint8_t *qs = ring + stage * kT5StageBytes + 4 * kHalfBytes + r * (kD * 2);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 v = r < qrows ? *reinterpret_cast<const uint4 *>(qs + c * 16) : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(opnd + (c >> 3) * kT5QOp + swz(r, c & 7)) = v;
                    *reinterpret_cast<uint4 *>(opnd + (c >> 3) * kT5QOp + swz(32 + r, c & 7)) = v;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&sh.q_ready));
            }
        }
        const bool tile_bad = have ? sh.stage_bad[stage] != 0 : true;
        seg_bad = seg_bad || tile_bad || aborted;
        const int slot0 = WIN ? tile_slot0(cur, kTile) : cur.t * kTile;
        const bool newt = slot0 + kTile - 1 >= cur.Lb;
        const bool partial = newt || (WIN && slot0 < max(0, L - p.window + 1));
        const int sb = i & 1;
        bool s_ok = false;
        if (have) {
            s_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.s_ready[sb]), (i >> 1) & 1, p.wait_cycles,
                                                     &sh.abort_flag));
            if (!s_ok && lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                report(p, kTimeout);
                atomicExch(&sh.abort_flag, 1);
            }
            aborted = aborted || !s_ok;
            seg_bad = seg_bad || !s_ok;
        }
        // this warp's 32 raw scores of row r; masked (-inf) only on the tiles
        // that hold slots outside some row's softmax (a warp-uniform branch)
        float x[32];
        float pm = -INFINITY;
        if (s_ok) {
            t5_fence_after();
            t5_ld32(tmem + tlane + sb * kTile + 32 * h, x);
            if (partial || lim < 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int sl = slot0 + 32 * h + j;
                    const bool on = lim >= 0 && (WIN ? attended(lim, lo_r, cur.P, sl) : sl <= lim);
                    x[j] = on ? x[j] : -INFINITY;
                }
            }
            float mt[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                mt[j] = fmaxf(fmaxf(x[4 * j], x[4 * j + 1]), fmaxf(x[4 * j + 2], x[4 * j + 3]));
#pragma unroll
            for (int w = 4; w > 0; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j)
                    mt[j] = fmaxf(mt[j], mt[j + w]);
            pm = mt[0];
        }
        // the row maximum over both warps' slots (every tile, both warps)
        sh.xm[sb][h][lane] = pm;
        t5_softmax_or(false);
        const float mx = fmaxf(pm, sh.xm[sb][1 - h][lane]) * p.scale_log2;   // the scale is positive
        if (s_ok) {
            // lazy rescale: a row's running maximum moves only by more than
            // 8. The decision is per row (lane) and the same in both warps;
            // warp 0 rescales O, warp-wide (TMEM accesses and the wait): when
            // any row must, each lane by its own factor (1 for rows that keep
            // their maximum).
            const bool raise = mx > m_run + 8.f;
            const bool scale_o = raise && m_run != -INFINITY && i > seg_first_i;   // O holds tiles up to i - 1
            const float alpha = scale_o ? fast_ex2(m_run - mx) : 1.f;
            if (h == 0 && __any_sync(0xffffffffu, scale_o) && wait_pv(i - 1)) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float o[32];
                    t5_ld32(tmem + 128 + c * 32, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        o[j] *= alpha;
                    t5_st32(tmem + 128 + c * 32, o);
                }
            }
            if (raise) {
                l_run = scale_o ? l_run * alpha : 0.f;
                m_run = mx;
            }
            // the weights 2^(s scale - m) in bf16, into this warp's half of
            // P buffer sb once the product of tile i - 2 has read it; their
            // sum in float32
            uint32_t pk[16];
            float ps[4] = {0.f, 0.f, 0.f, 0.f};
            const float nm = m_run == -INFINITY ? 0.f : -m_run;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float a = x[2 * j] == -INFINITY ? 0.f : fast_ex2(fmaf(x[2 * j], p.scale_log2, nm));
                const float c = x[2 * j + 1] == -INFINITY ? 0.f : fast_ex2(fmaf(x[2 * j + 1], p.scale_log2, nm));
                pk[j] = pack_bf16(a, c);
                ps[j & 3] += a + c;
            }
            l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            if (i >= 2)
                wait_pv(i - 2);
            uint8_t *pb = opnd + kT5POp + sb * 4096;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4 *>(pb + swz(r, 4 * h + c)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            t5_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&sh.p_ready[sb]));
        }

        const bool unit_done = (cur.t == cur.nr - 1);
        const bool range_done = (cur.g + 1 == cur.end);
        if (unit_done || range_done) {
            // ---- the segment's end: O of row r from TMEM (warp 0), then the
            // output (a whole unit) or the partial state
            const bool o_ok = s_ok && (h == 1 || wait_pv(i));
            sh.xl[h][lane] = l_run;
            const bool bad = t5_softmax_or(!row_good || seg_bad || !o_ok);   // both warps
            const bool whole = (seg_first_t == 0) && unit_done;
            const int G = p.G;
            const long long P = (long long)b * p.Hkv + kvh + blockIdx.x;
            float sc = 1.f;
            float M = m_run, den = l_run + sh.xl[1 - h][lane];
            if (whole) {
                const float sk = p.sink ? sink_log2(p, kvh * p.Gh + r % p.Gh) : -INFINITY;
                const float Mx = fmaxf(M, sk);
                const float a = (M == -INFINITY) ? 0.f : fast_ex2(M - Mx);
                den = a * den + ((sk == -INFINITY) ? 0.f : fast_ex2(sk - Mx));
                sc = a / den;
            } else if (r < G && h == 0) {
                p.ws_ml[(P * G + r) * 2 + 0] = bad ? qnan : M;
                p.ws_ml[(P * G + r) * 2 + 1] = bad ? qnan : den;
            }
            float *dst = nullptr;
            if (h == 0 && whole && r < qrows)
                dst = out_row<true>(p, cur, r, kD);
            else if (h == 0 && !whole && r < G)
                dst = p.ws_o + (P * G + r) * kD;
#pragma unroll 1
            for (int c = 0; c < (h == 0 ? 4 : 0); ++c) {
                float o[32];
                if (o_ok)
                    t5_ld32(tmem + 128 + c * 32, o);
                if (dst) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(dst + c * 32 + j) =
                            bad ? make_float4(qnan, qnan, qnan, qnan)
                                : make_float4(o[j] * sc, o[j + 1] * sc, o[j + 2] * sc, o[j + 3] * sc);
                }
            }
            if (bad && row_good && h == 0 && lane == 0)
                report(p, aborted ? kTimeout : kBadBlock);
            t5_fence_before();
            // both warps' stores before the ticket (and the sums read before
            // the next segment's end rewrites them)
            t5_softmax_or(false);
            if (!whole && h == 0) {
                // the arrival ticket and, in the last CTA of the unit, the merge
                const long long first_tile = cur.g - cur.t;
                FinJob j;
                j.stop = 0;
                j.first = cta_of_tile(first_tile, walk.N, walk.C);
                j.last = cta_of_tile(first_tile + cur.nr - 1, walk.N, walk.C);
                j.b = cur.b;
                j.kvh = cur.kvh;
                j.nq = cur.nq;
                j.tokL = cur.tokL;
                fin_ticket_merge<kT5Rows, true>(p, j, sh.merge, lane);
            }
        }
        ++i;
        const bool was_b = in_b;
        more = walk_next(p, cur, walk, in_b);
        if (in_b != was_b)
            range_start = cur.g;
        if (++stage == kT5Stages) {
            stage = 0;
            phase ^= 1;
        }
    }
    // the MMA warp has seen its last product complete, the other softmax warp
    // is done with TMEM: free it
    t5_fence_before();
    t5_end_sync();
    if (warp == 0) {
        t5_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kT5Cols) : "memory");
    }
}

template <bool WIN>
cudaError_t launch_t5(const DecodeParams &p, const TcMaps &maps, cudaStream_t st)
{
    static std::atomic<unsigned long long> attr_set{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(tc5_multi_kernel<WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kT5DynSmem);
        if (e != cudaSuccess)
            return e;
        attr_set.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kT5Threads);
    cfg.dynamicSmemBytes = kT5DynSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc5_multi_kernel<WIN>, p, maps.k, maps.v, maps.k16, maps.v16);
}

}  // namespace
}  // namespace gqa
