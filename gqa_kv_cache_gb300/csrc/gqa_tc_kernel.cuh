// Tensor-core decode kernel for bfloat16 or E4M3 (FP8) caches with D = 128 and
// G <= 8; the query is bfloat16 or float32.
//
// Data path (persistent CTAs, kCtasPerSm per SM):
//  * a producer warp walks the CTA's tiles (gqa_common.cuh) and streams every
//    64-slot tile of K and V from HBM into a kStages-deep shared-memory ring
//    with TMA tiled copies (cp.async.bulk.tensor, 128-byte swizzle, two
//    64-element halves per row), signalling an mbarrier per stage; for paged
//    caches each lane copies one block of the tile. The first tile of each
//    unit segment also brings the unit's G query rows (one bulk copy), so no
//    consumer ever waits on a global load. Table and row lookups for a tile
//    are issued one tile ahead, before the wait for a free stage.
//  * four consumer warps each take 16 slots of every tile and compute, on the
//    tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), with the
//    operands swapped so that the G <= 8 query rows are the N = 8 side:
//      S^T = K Q^T    M = the warp's 16 slots, N = 8 query rows (rows >= G
//                     are zero), K = 16 dims, 8 steps over D = 128 (two
//                     accumulator chains, even and odd steps); a float32
//                     query adds a second product with its bf16 remainders
//                     bf16(q - bf16(q)), so q enters with ~16 significant bits;
//      O^T += V^T P^T M = 16 dims (8 tiles over D), N = 8 query rows, K = 16
//                     slots; P^T is bf16(p) plus a second product with the
//                     remainders bf16(p - bf16(p)), so the weights keep ~16
//                     significant bits and the sum stays float32-accurate.
//    The K fragments come from ldmatrix, the V^T fragments from
//    ldmatrix.trans (the swizzle makes both conflict-free), and the score
//    fragment (slot, row pairs) becomes the P^T fragment (row, slot pairs)
//    with one movmatrix transpose per 8 slots. Compared with putting the
//    heads on the M = 16 side, no MMA row is padding: half the products and
//    half the accumulator registers.
//  * online softmax in float32 with base-2 scores (scale log2(e)/sqrt(D)
//    folded in), a lazy rescale (the running max is only raised when a score
//    exceeds it by more than 8, i.e. p <= 256), masking by selection so stale
//    slots (and slots outside a sliding window and kept prefix) never enter
//    the arithmetic, and the V rows of such slots zeroed in shared memory
//    before the product (0 * NaN would not be 0). A window skips whole tiles
//    (the schedule lists only tiles holding attended slots) and, for paged
//    caches, whole blocks.
//  * E4M3 caches (KV8): tiles arrive as bytes (half the traffic), and the
//    products run in f16 (every E4M3 value is an f16): K fragments come from a
//    b16 ldmatrix over the byte rows -- each lane gets four consecutive E4M3
//    values of a slot, two conversions make its part of the A fragment, and
//    the query fragments are gathered in the same permuted order of the 16
//    dims of a k-step (a dot product does not depend on the order); V^T
//    fragments come from ldmatrix.trans, whose byte pairs one byte permute
//    splits into (slot, slot + 1) pairs of an even and of an odd dim, the two
//    halves of one M = 16 tile (the dims are interleaved, undone in the
//    epilogue). The query is f16 (a float32 one split into hi + remainder), P
//    is f16; the K scale joins the score scale, the V scale multiplies the
//    accumulator before the epilogue, and the appended token is quantised
//    (float32 division by the scale, round to nearest even, saturating). With
//    its smaller stages the single-token E4M3 kernel runs three CTAs per SM
//    (2-stage rings, at most 128 registers a thread).
//  * multi-token steps (MULTI): a unit is a chunk of up to 32 / G tokens of a
//    row; its query rows are (token, head) pairs, gathered by one bulk copy
//    per token. Units of up to 8 rows take the products above (rows on the
//    N = 8 side); units of 9 to 16 rows keep the rows on the M = 16 side
//    (S = Q K^T, O += P V, the score fragment reused as the A fragment of P;
//    P in plain bf16, f16 over an E4M3 cache), each warp on its 16 slots of
//    a tile; units of 17 to 32 rows do the same with two warps per 16 query
//    rows, each on 32 slots of a tile (two passes of 16), so a row's KV is
//    streamed once for up to 32 rows; at the segment's end the warps holding
//    slots 32-63 hand their states to those holding slots 0-31, which merge
//    them in registers and write the output or partial. Each row is masked
//    beyond its own token's position and keeps its own softmax state, every
//    slot holding a new token is substituted from k_new / v_new as below
//    (quantised over an E4M3 cache), and the chunk appends its own tokens.
//    With 16 or 32 query rows the E4M3 ring takes 3 stages (two CTAs per
//    SM); with up to 8, the E4M3 kernel runs three CTAs per SM as for single
//    tokens.
//  * the new token (decode step only; the read-only attend reads slot L from
//    the cache like any other): in the tile that holds slot L the owning warp writes
//    k_new / v_new into the ring slot of row L (the TMA copy of the stale
//    cache row is discarded) and stores them into the cache at slot L. The
//    copy of that tile has landed before the store, and no other CTA loads
//    slot L, so the append cannot race with a read.
//  * at the end of each unit segment the four warp states are merged in
//    shared memory (finish_segment): a whole unit writes its output, a cut
//    unit its partial state, and the last CTA of a cut unit merges them.
// Two CTAs (three for the single-token E4M3 kernel) share each SM, so one
// CTA's segment epilogue overlaps the others' streaming.
// Every mbarrier wait is bounded. A wait that gives up sets GQA_STATUS_TIMEOUT
// and a CTA-wide abort flag: the producer stops issuing and waits (bounded)
// for its copies in flight; the consumer warps stop waiting and computing but
// keep walking their tiles and taking part in every barrier, writing NaN.
// The consumers' limit on a wait for a tile is a launch parameter (about 2 s
// by default), the producer's waits always keep the full limit. For tests of
// this path a launch can also make each consumer warp's first wait include a
// barrier that nothing completes, so that wait runs out after the (shortened)
// limit whatever the timing of the copies.
#pragma once

#include <cuda_fp16.h>

#include <atomic>
#include <type_traits>

#include "gqa_common.cuh"
#include "gqa_launch.h"

namespace gqa {
namespace {

#ifndef GQA_TC_STAGES
#define GQA_TC_STAGES 2
#endif
#ifndef GQA_TC_CTAS_PER_SM
#define GQA_TC_CTAS_PER_SM 2
#endif
#ifndef GQA_TC_KV8_CTAS_PER_SM
#define GQA_TC_KV8_CTAS_PER_SM 3
#endif

constexpr int kD = 128;
constexpr int kTile = 64;                             // slots per tile
constexpr int kStages = GQA_TC_STAGES;                // depth of one CTA's TMA ring (bf16)
constexpr int kCtasPerSm = GQA_TC_CTAS_PER_SM;        // resident CTAs per SM
constexpr int kCtasPerSmKV8 = GQA_TC_KV8_CTAS_PER_SM; // the same, single-token steps over an E4M3 cache
constexpr int kConsumerWarps = 4;
constexpr int kMaxWarps = kConsumerWarps + 2;          // consumers, producer, finisher
constexpr int kGMax = 8;
constexpr int kHalfBytes = kTile * 128;               // one 64-element half of a tile
constexpr long long kWaitCycles = 4LL << 30;          // ~2 s at 2 GHz

// Ring geometry for a bfloat16 (QF32 = false) or float32 query over a
// bfloat16 or E4M3 (KV8) cache.
template <bool QF32, bool KV8 = false, bool MULTI = false, int MR = 0>
struct Ring {
    static constexpr bool kMside = MULTI && MR > 0;   // units of up to MR (16 or 32) query rows
    static constexpr int kQElem = QF32 ? 4 : 2;
    static constexpr int kQRows = kMside ? MR : kGMax;               // query rows of a unit
    static constexpr int kQBytes = kQRows * kD * kQElem;             // the unit's query rows
    static constexpr int kKVBytes = KV8 ? kTile * kD : 2 * kHalfBytes; // K (or V) of one tile
    // single-token steps over an E4M3 cache: the new token's bf16 K and V rows
    // (2 x 256 bytes), copied by the producer into the stage of the tile that
    // holds slot L (measured: about 0.5 us off llama3_8b's step; over a bf16
    // cache it made no difference or cost time, so there the owning warp
    // loads them from global memory)
    static constexpr int kNewBytes = (!MULTI && KV8) ? 1024 : 0;
    static constexpr int kStageBytes = 2 * kKVBytes + kQBytes + kNewBytes;   // K (lo, hi), V (lo, hi), Q, new
    // E4M3: 4 stages at two CTAs per SM, 2 at three; 3 with the query rows
    // of a 16- or 32-row multi-token unit, so two CTAs still share an SM
    static constexpr int kNumStages = KV8 ? (kMside ? 3 : (kCtasPerSmKV8 >= 3 ? 2 : 4)) : kStages;
    static constexpr int kCtas = (KV8 && !kMside) ? kCtasPerSmKV8 : kCtasPerSm;   // resident CTAs per SM
    static constexpr int kDynSmem = kNumStages * kStageBytes + 1024;
    // Multi-token steps over a bfloat16 cache: a finisher warp takes the
    // arrival ticket (and the merge, when last) of every cut unit but the
    // CTA's last off the consumers' path (measured: llama3_8b q_len 4 91.5 ->
    // 84.0 us, paged q_len 3 811.8 -> 793.7 us). In the single-token kernels a
    // sixth warp made every CTA stream about 5 % slower and the steps 1-2 us
    // longer, and the E4M3 kernels at three CTAs per SM have no registers to
    // spare, so those keep the ticket on the consumers.
    static constexpr bool kFin = MULTI && !KV8;
    static constexpr int kThreads = (kConsumerWarps + 1 + (kFin ? 1 : 0)) * 32;
    static_assert(kStageBytes % 1024 == 0, "stages must stay 1024-byte aligned for the swizzle");
};

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, int count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// The same test with a suspend-time hint of `ns` nanoseconds: the thread
// sleeps at most about that long before the test answers.
__device__ __forceinline__ bool mbar_try_ns(uint32_t bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(ns)
                 : "memory");
    return ok != 0;
}

// Limits below this are honoured to the cycle: the wait then polls with a
// one-nanosecond suspend hint instead of letting a test sleep for the
// hardware's own time limit first.
constexpr long long kShortWait = 1LL << 20;

// Bounded wait: false when it gave up after `limit` SM clock cycles or, with
// `abort` given, as soon as *abort is set.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit = kWaitCycles,
                                          const int *abort = nullptr)
{
    if (limit < kShortWait) {
        const long long t0 = clock64();
        while (!mbar_try_ns(bar, parity, 1u)) {
            if (clock64() - t0 > limit || (abort && *((const volatile int *)abort)))
                return false;
        }
        return true;
    }
    if (mbar_try(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try(bar, parity)) {
        if (clock64() - t0 > limit || (abort && *((const volatile int *)abort)))
            return false;
    }
    return true;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 pair (lo in the low half) rounded to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// f16 pair (lo in the low half) rounded to nearest even.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float f16_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))); }
__device__ __forceinline__ float f16_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

// A float32 pair as f16 hi parts and f16 remainders: v = hi + lo to ~22 bits.
__device__ __forceinline__ void split_f16(float2 v, uint32_t &hi, uint32_t &lo)
{
    hi = pack_f16(v.x, v.y);
    lo = pack_f16(v.x - f16_lo(hi), v.y - f16_hi(hi));
}

// Four E4M3 bytes (the first in the low byte) as two f16 pairs; exact.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((unsigned short)(w & 0xffffu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((unsigned short)(w >> 16)));
}

// Sixteen consecutive bf16 values (two 16-byte words, the first value in the
// low half of a.x) divided by `scale` in float32 (round to nearest) and
// encoded as E4M3 (round to nearest even, saturating): sixteen bytes.
__device__ __forceinline__ uint4 quant_e4m3x16(uint4 a, uint4 b, float scale)
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float x0 = __fdiv_rn(__uint_as_float(w[i] << 16), scale);
        const float x1 = __fdiv_rn(__uint_as_float(w[i] & 0xffff0000u), scale);
        unsigned short q;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(x1), "f"(x0));
        o[i >> 1] |= (uint32_t)q << (16 * (i & 1));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// The 8x8 matrix of 16-bit values held in fragment layout (lane 4 r + c holds
// row r, columns 2 c and 2 c + 1) transposed in registers.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a)
{
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// A float32 pair as bf16 hi parts and bf16 remainders: v = hi + lo to ~16 bits.
__device__ __forceinline__ void split_bf16(float2 v, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16(v.x, v.y);
    lo = pack_bf16(v.x - __uint_as_float(hi << 16), v.y - __uint_as_float(hi & 0xffff0000u));
}

// Byte offset, within one 64-element half, of 16-byte chunk c8 of row r
// under the 128-byte swizzle (the half starts on a 1024-byte boundary).
__device__ __forceinline__ uint32_t swz(int r, int c8) { return (uint32_t)(r * 128 + ((c8 ^ (r & 7)) << 4)); }

// The consumers and the finisher warp hand over cut units through one job
// slot and two named barriers: 2 (a job is posted: the consumers arrive, the
// finisher waits) and 3 (the slot is free again: the finisher arrives, the
// consumers wait). The barriers also order the consumers' partial stores
// before the finisher's ticket.
constexpr int kFinBarThreads = (kConsumerWarps + 1) * 32;

struct FinJob {
    int stop;          // 1: no more jobs
    int first, last;   // CTAs whose ranges hold the unit's tiles
    int b, kvh, nq, tokL;
};

__device__ __forceinline__ void job_wait_posted() { asm volatile("bar.sync 2, %0;" ::"n"(kFinBarThreads) : "memory"); }
__device__ __forceinline__ void job_post() { asm volatile("bar.arrive 2, %0;" ::"n"(kFinBarThreads) : "memory"); }
__device__ __forceinline__ void job_wait_free() { asm volatile("bar.sync 3, %0;" ::"n"(kFinBarThreads) : "memory"); }
__device__ __forceinline__ void job_free() { asm volatile("bar.arrive 3, %0;" ::"n"(kFinBarThreads) : "memory"); }

// The finisher warp's handling of a cut unit (RW query rows at most): the
// arrival ticket and, in the last CTA of the unit to arrive, the merge of the
// K partials (log-sum-exp rule), the output, and the partials and counter
// back to zero. One warp: the partial outputs are read with all of a lane's
// loads of one partial (of up to 16 rows at a time) in flight at once, so a
// merge costs about one L2 round trip per partial and block of rows.
template <int RW, bool MULTI, int GR, int KM>
__device__ __noinline__ void fin_ticket_merge(const DecodeParams &p, const FinJob j, MergeBufT<GR, KM> &mb, int lane)
{
    constexpr int RB = RW > 16 ? 16 : RW;    // rows merged at a time (the registers of acc and v)
    constexpr int IT = RB * kD / (32 * 4);   // float4 per lane and partial
    const int G = p.G;
    const int u = j.b * p.Hkv + j.kvh;
    const int K = j.last - j.first + 1;
    int old = 0;
    if (lane == 0)
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.ws_cnt + u) : "memory");
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != K - 1)
        return;                              // other pieces still to come
    TileCursor c;
    c.b = j.b;
    c.kvh = j.kvh;
    c.nq = j.nq;
    c.tokL = j.tokL;
    const long long P0 = (long long)u + j.first;
    if (K <= KM) {
        // every partial's (m, l): weights and the denominator per query row
        for (int k = lane; k < K * G; k += 32) {
            mb.w[k] = __ldcg(p.ws_ml + (P0 * G + k) * 2);
            mb.l[k] = __ldcg(p.ws_ml + (P0 * G + k) * 2 + 1);
        }
        __syncwarp();
        if (lane < G) {
            float M = -INFINITY;
            for (int i = 0; i < K; ++i)
                M = fmaxf(M, mb.w[i * G + lane]);
            const float sk = p.sink ? sink_log2(p, j.kvh * p.Gh + lane % p.Gh) : -INFINITY;
            M = fmaxf(M, sk);
            float den = (sk == -INFINITY) ? 0.f : fast_ex2(sk - M);
            for (int i = 0; i < K; ++i) {
                const float a = fast_ex2(mb.w[i * G + lane] - M);
                mb.w[i * G + lane] = a;
                den = fmaf(a, mb.l[i * G + lane], den);
            }
            mb.inv_den[lane] = 1.f / den;
        }
    } else if (lane < G) {
        // more partials than the buffer holds: the maximum and the denominator
        // per row from every partial's (m, l) directly; the weights follow KM
        // partials at a time
        float M = -INFINITY;
        for (int i = 0; i < K; ++i)
            M = fmaxf(M, __ldcg(p.ws_ml + ((P0 + i) * G + lane) * 2));
        const float sk = p.sink ? sink_log2(p, j.kvh * p.Gh + lane % p.Gh) : -INFINITY;
        M = fmaxf(M, sk);
        float den = (sk == -INFINITY) ? 0.f : fast_ex2(sk - M);
        for (int i = 0; i < K; ++i) {
            const float *ml = p.ws_ml + ((P0 + i) * G + lane) * 2;
            den = fmaf(fast_ex2(__ldcg(ml) - M), __ldcg(ml + 1), den);
        }
        mb.M[lane] = M;
        mb.inv_den[lane] = 1.f / den;
    }
    __syncwarp();
    const int nrow = MULTI ? p.Gh * j.nq : G;
    for (int r0 = 0; r0 < G; r0 += RB) {
        const int base = r0 * kD;            // first element of this block of rows
        float4 acc[IT];
#pragma unroll
        for (int it = 0; it < IT; ++it)
            acc[it] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < K; c0 += KM) {
            const int kc = min(KM, K - c0);
            if (K > KM) {   // this chunk's weights (partial c0 + k / G, row k % G)
                __syncwarp();
                for (int k = lane; k < kc * G; k += 32)
                    mb.w[k] = fast_ex2(__ldcg(p.ws_ml + ((P0 + c0) * G + k) * 2) - mb.M[k % G]);
                __syncwarp();
            }
            for (int i = 0; i < kc; ++i) {
                float4 *po = reinterpret_cast<float4 *>(p.ws_o + (P0 + c0 + i) * G * kD + base);
                float4 v[IT];
#pragma unroll
                for (int it = 0; it < IT; ++it) {
                    const int idx = base + (it * 32 + lane) * 4;
                    v[it] = idx < G * kD ? __ldcg(po + it * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int it = 0; it < IT; ++it) {
                    const int idx = base + (it * 32 + lane) * 4;
                    if (idx < G * kD) {
                        const float a = mb.w[i * G + idx / kD];
                        acc[it].x = fmaf(a, v[it].x, acc[it].x);
                        acc[it].y = fmaf(a, v[it].y, acc[it].y);
                        acc[it].z = fmaf(a, v[it].z, acc[it].z);
                        acc[it].w = fmaf(a, v[it].w, acc[it].w);
                        po[it * 32 + lane] = make_float4(0.f, 0.f, 0.f, 0.f);   // consumed: zero-filled again
                    }
                }
            }
        }
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int idx = base + (it * 32 + lane) * 4;
            const int g = idx / kD;
            if (idx < G * kD && g < nrow) {
                const float sc = mb.inv_den[g];
                *reinterpret_cast<float4 *>(out_row<MULTI>(p, c, g, kD) + (idx - g * kD)) =
                    make_float4(acc[it].x * sc, acc[it].y * sc, acc[it].z * sc, acc[it].w * sc);
            }
        }
    }
    float *ml = p.ws_ml + P0 * G * 2;
    for (int k = lane; k < K * G * 2; k += 32)
        ml[k] = 0.f;
    if (lane == 0)
        p.ws_cnt[u] = 0;
    __syncwarp();
}

// Partials of a cut unit whose weights one pass through shared memory holds
// (more: that many at a time), by query rows of a unit.
constexpr int merge_partials(int rw) { return rw == kGMax ? kMergeMax : (rw == 16 ? 16 : 8); }

// The finisher warp's job slot and merge buffer (kernels with one).
template <int RW>
struct FinShared {
    FinJob job;
    MergeBufT<RW, merge_partials(RW)> merge;
};
struct NoFinShared {};

// NS ring stages; RW query rows per unit (8, or 16 or 32 for multi-token
// units); FIN: a finisher warp; SW warp states of SR rows each kept for the
// segment's end (the four warps' states of every row; 32-row units: the two
// warps holding slots 32-63 of rows 0-15 and 16-31, handed to the two holding
// slots 0-31).
template <int NS, int RW = kGMax, bool FIN = false, int SW = kConsumerWarps, int SR = RW>
struct Shared {
    static constexpr int kOPad = 4;   // rows 132 floats apart: the epilogue's stores are conflict-free
    uint64_t full[NS];
    uint64_t empty[NS];
    uint64_t stall;      // a barrier nothing completes (tests of the timeout path)
    int stage_bad[NS];
    int abort_flag;
    int last_flag;
    long long sched[kMaxWarps + 8];
    TileWalk walk;
    float m[SW][SR];
    float l[SW][SR];
    alignas(16) float o[SW][SR][kD + kOPad];  // rows padded: (near) conflict-free 8-byte stores
    MergeBufT<RW, merge_partials(RW)> merge;
    std::conditional_t<FIN, FinShared<RW>, NoFinShared> fin;
};

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// consumer_sync that also returns whether v was true in any consumer thread.
__device__ __forceinline__ bool consumer_sync_or(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(kConsumerWarps * 32)
                 : "memory");
    return r != 0;
}

// The two consumer warps 2 pr and 2 pr + 1 (32-row units: the pair that
// shares slots 32 pr .. 32 pr + 31 of every tile).
__device__ __forceinline__ void pair_sync(int pr)
{
    asm volatile("bar.sync %0, 64;" ::"r"(4 + pr) : "memory");
}


// WIN: a sliding window is in force. Without one the window fields of the
// cursor are never read, so they take no registers and no code. MULTI: a
// multi-token step (the chunk fields of the cursor are read only then). KV8:
// an E4M3 cache. MR: multi-token units of 9 to 16 (MR = 16) or of 17 to 32
// (MR = 32) query rows, which keep the rows on the M = 16 side of the
// products; units of up to 8 rows (and every single-token unit, MR = 0) put
// them on the N = 8 side.
template <bool QF32, bool WIN, bool MULTI, bool KV8, int MR>
__global__ void __launch_bounds__((Ring<QF32, KV8, MULTI, MR>::kThreads), (Ring<QF32, KV8, MULTI, MR>::kCtas))
    tc_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mk16,
                     const __grid_constant__ CUtensorMap mv16)
{
    using RG = Ring<QF32, KV8, MULTI, MR>;
    static_assert(!(MULTI && QF32), "multi-token steps take a bfloat16 query");
    static_assert(MR == 0 || (MULTI && (MR == 16 || MR == 32)), "16- and 32-row units are multi-token units");
    constexpr bool kMside = RG::kMside;              // query rows on the M = 16 side
    constexpr bool kM32 = kMside && MR == 32;        // two warps per 16 query rows, 32 slots each
    constexpr int kRW = kMside ? MR : kGMax;         // query rows of a unit
    constexpr int kSW = kM32 ? 2 : kConsumerWarps;   // warp states kept for the segment's end
    constexpr int kSR = kM32 ? 16 : kRW;             // rows of each
    using SharedT = Shared<RG::kNumStages, kRW, RG::kFin, kSW, kSR>;
    constexpr int kStageBytes = RG::kStageBytes;
    constexpr int kNS = RG::kNumStages;   // ring depth
    constexpr int kKVB = RG::kKVBytes;    // K (or V) bytes of one tile
    extern __shared__ uint8_t dyn_smem[];
    __shared__ SharedT sh;
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_u32 = smem_u32(ring);

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), kConsumerWarps);
            sh.stage_bad[s] = 0;
        }
        sh.abort_flag = 0;
        mbar_init(smem_u32(&sh.stall), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kConsumerWarps && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mv)) : "memory");
        if (!KV8 && !p.paged) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mk16)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mv16)) : "memory");
        }
    }
    // Launched as a programmatic dependent of the previous kernel on the
    // stream: everything above overlaps its tail; no input is read before it
    // has completed and its memory is visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    schedule_walk(p, sh.sched, &sh.walk, KV8 ? 1 : 2);   // contains __syncthreads
    const TileWalk &walk = sh.walk;

    const int G = p.G;
    const __nv_bfloat16 *knew = static_cast<const __nv_bfloat16 *>(p.k_new);
    const __nv_bfloat16 *vnew = static_cast<const __nv_bfloat16 *>(p.v_new);

    if (warp == kConsumerWarps) {
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
        const int nblk = p.paged ? (bs < kTile ? kTile / bs : 1) : 1;  // copies per half per tile
        const int box_rows = p.paged ? (bs < kTile ? bs : kTile) : kTile;
        // Where this lane copies tile `c` from: z (cache head row of the
        // tensor map) and y (first slot in it); z < 0: nothing; `rows`: the
        // tile's box height (warp-uniform). Computed one tile ahead, before
        // the wait for a free stage, so the table reads overlap the wait.
        struct Plan {
            int z, y;
            bool bad_entry, good;
            int rows;
        };
        auto plan = [&](const TileCursor &c) {
            Plan r{-1, 0, false, row_ok(p, c.b, c.L), box_rows};
            if (!r.good)
                return r;
            const int slot0 = WIN ? tile_slot0(c, kTile) : c.t * kTile;
            const int rb = MULTI ? real_row(p, c.b) : c.b;   // the batch row
            if (KV8 && !p.paged) {
                // an E4M3 dense cache: the whole tile (half the bytes of a
                // bf16 one; small boxes for partly read tiles measured slower
                // here: llama3_8b 44.5 against 43.4 us)
                if (lane == 0) {
                    const int row = p.slot_ids ? __ldg(p.slot_ids + rb) : rb;
                    r.z = row * p.Hkv + c.kvh;
                    r.y = slot0;
                }
            } else if (!p.paged) {
                // a dense cache: one box when every part of the tile holds a
                // slot the step reads, else a small box per part that does (a
                // unit's last tile, a window's first; the consumers mask and
                // zero the rest as in any such tile). ragged_slots 118.3 ->
                // 117.0 us, llama3_8b 63.7 -> 63.0 us; a small box for every
                // part of every tile was slower (ragged_slots 120.9 us)
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
                const int s = slot0 + lane * box_rows;  // first slot this lane copies
                // a block is copied when it holds an attended slot
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
            // every decision below is warp-uniform (the loop uses warp votes)
            if (__any_sync(0xffffffffu, *((volatile int *)&sh.abort_flag) != 0))
                break;
            // (a wait for a free stage also ends when the consumers have aborted)
            if (!__all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&sh.empty[stage]), phase ^ 1, kWaitCycles, &sh.abort_flag))) {
                if (lane == 0 && !*((volatile int *)&sh.abort_flag)) {
                    report(p, kTimeout);
                    atomicExch(&sh.abort_flag, 1);
                }
                break;
            }
            const int b = cur.b, kvh = cur.kvh;
            const unsigned copying = __ballot_sync(0xffffffffu, pl.z >= 0);
            const bool any_bad = __any_sync(0xffffffffu, pl.bad_entry);
            // the first tile of each of this CTA's unit segments also brings
            // the unit's G query rows (contiguous in q)
            const bool seg_first = pl.good && (cur.t == 0 || cur.g == range_start);
            const int qrows = MULTI ? p.Gh * cur.nq : G;   // query rows with data
            const uint32_t qbytes = seg_first ? (uint32_t)(qrows * kD * RG::kQElem) : 0u;
            // single-token decode over an E4M3 cache: the tile holding slot L
            // (the unit's last real tile) also brings the new token's K and V
            // rows, so the consumers quantise and append them from shared memory
            const bool newt = RG::kNewBytes > 0 && !p.attend && pl.good && cur.t == cur.nr - 1;
            const uint32_t nbytes = newt ? 2u * kD * 2u : 0u;
            const uint32_t bytes = (uint32_t)__popc(copying) * (KV8 ? 2u : 4u) *
                                       (uint32_t)(KV8 ? box_rows : pl.rows) * 128u + qbytes + nbytes;
            const uint32_t fb = smem_u32(&sh.full[stage]);
            if (lane == 0) {
                sh.stage_bad[stage] = any_bad ? 1 : 0;
                mbar_arrive_tx(fb, bytes);
                if constexpr (RG::kNewBytes > 0) {
                    if (newt) {
                        const uint32_t ndst = ring_u32 + stage * kStageBytes + 2 * kKVB + RG::kQBytes;
                        const long long nidx = ((long long)b * p.Hkv + kvh) * kD;
                        bulk_load(ndst, knew + nidx, kD * 2u, fb);
                        bulk_load(ndst + kD * 2u, vnew + nidx, kD * 2u, fb);
                    }
                }
                if (qbytes) {
                    const uint32_t qdst = ring_u32 + stage * kStageBytes + 2 * kKVB;
                    if constexpr (MULTI) {
                        // one copy per token: its Gh heads are contiguous in q
                        const uint32_t tb = (uint32_t)(p.Gh * kD * RG::kQElem);
                        for (int i = 0; i < cur.nq; ++i) {
                            const long long tok = cur.tokL - (cur.nq - 1 - i);
                            bulk_load(qdst + i * tb,
                                      static_cast<const uint8_t *>(p.q) +
                                          (tok * p.Hq + (long long)kvh * p.Gh) * kD * RG::kQElem,
                                      tb, fb);
                        }
                    } else {
                        bulk_load(qdst,
                                  static_cast<const uint8_t *>(p.q) +
                                      ((long long)b * p.Hq + (long long)kvh * G) * kD * RG::kQElem,
                                  qbytes, fb);
                    }
                }
            }
            __syncwarp();
            if (pl.z >= 0) {
                if constexpr (KV8) {   // rows of 128 one-byte elements: one box each
                    const uint32_t dst = ring_u32 + stage * kStageBytes + lane * box_rows * 128;
                    tma_load_3d(dst, &mk, 0, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + kKVB, &mv, 0, pl.y, pl.z, fb, policy);
                } else if (pl.rows == box_rows) {   // a whole box (a paged block, a dense tile)
                    const uint32_t dst = ring_u32 + stage * kStageBytes + lane * box_rows * 128;
                    tma_load_3d(dst, &mk, 0, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + kHalfBytes, &mk, 64, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + 2 * kHalfBytes, &mv, 0, pl.y, pl.z, fb, policy);
                    tma_load_3d(dst + 3 * kHalfBytes, &mv, 64, pl.y, pl.z, fb, policy);
                } else {   // a part of a dense tile (the small-box maps)
                    const uint32_t dst = ring_u32 + stage * kStageBytes + lane * kDenseBoxRows * 128;
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
            if (++stage == kNS) {
                stage = 0;
                phase ^= 1;
            }
        }
        // every tile is issued: the next kernel on the stream may start launching
        asm volatile("griddepcontrol.launch_dependents;");
        // Let every copy still in flight land before the producer exits, so
        // that no CTA can end while one of its copies is still writing into
        // its shared memory (consumers that gave up on a wait no longer hold
        // the CTA open until their tiles land). At most kNS stages are in
        // flight (a stage is refilled only after the consumers released it,
        // i.e. after its copies landed), and the last min(kNS, issued) issued
        // stages are exactly those; each wait keeps the full limit, whatever
        // the consumers' limit. Without an abort these waits end as the
        // tiles land, which the consumers wait for anyway.
        {
            int s = stage, ph = phase;
            for (int k = 0; k < kNS && k < issued; ++k) {
                if (--s < 0) {
                    s = kNS - 1;
                    ph ^= 1;
                }
                mbar_wait(smem_u32(&sh.full[s]), ph);
            }
        }
        return;
    }

    // --------------------------------------------------------- finisher --
    // Takes each cut unit the consumers hand over: the arrival ticket (whose
    // release must wait until this CTA's partial stores are visible at GPU
    // scope, about 2 us under full HBM load) and, in the last CTA of the unit
    // to arrive, the merge. The consumers meanwhile stream the next segment.
    if constexpr (RG::kFin) {
        if (warp == kConsumerWarps + 1) {
            job_free();                  // the slot starts free
            while (true) {
                job_wait_posted();
                const FinJob j = sh.fin.job;
                if (j.stop)
                    break;
                job_free();
                fin_ticket_merge<kRW, MULTI>(p, j, sh.fin.merge, lane);
            }
            return;
        }
    }

    // -------------------------------------------------------- consumers --
    const int g0 = lane >> 2, q4 = lane & 3;
    // this warp's 16 rows of every tile (the slots it substitutes and zeroes,
    // and, but for 32-row units, the slots it computes on)
    const int row0 = warp * 16;
    // 32-row units: query rows rq0 .. rq0 + 15 over slots 32 (warp >> 1) .. +31
    const int rq0 = kM32 ? 16 * (warp & 1) : 0;
    TileCursor cur;
    bool in_b = false;
    bool more = walk_first(p, cur, walk, in_b);
    int stage = 0;
    uint32_t phase = 0;
    // Q fragments of query row g0 (< G), 8 k-steps: the B operand of S^T = K Q^T
    // (single-token units, multi-token units of up to 8 rows) or rows 0-7 of
    // the A operand of S = Q K^T (16-row units)
    uint32_t qa[8][2];
    // float32 query: the remainders of row g0 (a second B operand);
    // 16-row units: query row g0 + 8 (A rows 8-15)
    uint32_t ql[8][2];
    // O: multi-token units, 16 n-tiles of 8 dims for rows g0 and g0 + 8;
    // single-token units, O^T in 8 m-tiles of 16 dims for rows 2 q4, 2 q4 + 1
    constexpr int kOT = kMside ? 16 : 8;
    float acc_o[kOT][4];
    float m_run = -INFINITY, l_run = 0.f;
    int seg_first_t = 0;
    int pre_cnt = -1;                    // thread 0: the unit's arrival count near the segment's end
    bool seg_start = true, row_good = true, aborted = false;
    bool stall = p.test_stall != 0;      // the first wait also waits on sh.stall (runs out)
    int seg_bad = 0;
    // multi-token units only: this lane's rows g0 and g0 + 8 (last slot,
    // window start, softmax state of the second), rows with data
    int lim = 0, lo_r = 0, lim1 = 0, lo_r1 = 0, qrows = G;
    float m_run1 = -INFINITY, l_run1 = 0.f;
    // E4M3 cache: the unit's score scale (with k_scale) and v_scale
    float ssc = p.scale_log2, vsc = 1.f;

    while (more) {
        const int b = cur.b, kvh = cur.kvh, L = cur.L;
        const bool first_of_seg = seg_start;
        if (seg_start) {
            seg_first_t = cur.t;
            row_good = row_ok(p, b, L);
            if (!row_good && tid == 0 && cur.t == 0 && kvh == 0)
                report(p, row_error_bits(p, b, L));
#pragma unroll
            for (int n = 0; n < kOT; ++n)
                acc_o[n][0] = acc_o[n][1] = acc_o[n][2] = acc_o[n][3] = 0.f;
            m_run = m_run1 = -INFINITY;
            l_run = l_run1 = 0.f;
            seg_bad = 0;
            seg_start = false;
            if constexpr (MULTI) {
                // this lane's two query rows (g0 and g0 + 8 on the M side, else
                // 2 q4 and 2 q4 + 1); row r is token r / Gh of the chunk and
                // attends up to its own position; rows without a token none
                const int ra = kMside ? rq0 + g0 : 2 * q4, rb = kMside ? rq0 + g0 + 8 : 2 * q4 + 1;
                qrows = p.Gh * cur.nq;
                lim = ra < qrows ? L - (cur.nq - 1 - ra / p.Gh) : -1;
                lim1 = rb < qrows ? L - (cur.nq - 1 - rb / p.Gh) : -1;
                if constexpr (WIN) {
                    lo_r = max(0, lim - p.window + 1);
                    lo_r1 = max(0, lim1 - p.window + 1);
                }
            }
            if constexpr (KV8) {
                ssc = p.scale_log2 * __ldg(p.k_scale + kvh);
                vsc = __ldg(p.v_scale + kvh);
            }
            pre_cnt = -1;
        }
        // One tile before the segment ends, thread 0 reads the unit's arrival
        // count (acquire): if every other piece has arrived by then, the
        // segment's end needs no ticket (finish_segment). The load's latency
        // hides behind the last tile.
        if (tid == 0 && (cur.t == cur.nr - 2 || cur.g + 2 == cur.end))
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];"
                         : "=r"(pre_cnt)
                         : "l"(p.ws_cnt + (long long)b * p.Hkv + kvh)
                         : "memory");

        // After an abort every warp keeps walking its tiles and taking part in
        // every barrier, but waits for and computes nothing (outputs NaN).
        // The outcome is made warp-uniform: a lane that gave up makes the
        // whole warp give up (the products below are warp-wide).
        bool have = false;
        if (!aborted && !__any_sync(0xffffffffu, *((volatile int *)&sh.abort_flag) != 0)) {
            bool ok = mbar_wait(smem_u32(&sh.full[stage]), phase, p.wait_cycles);
            if (stall) {   // tests of the timeout path: a wait that nothing ends
                ok = ok && mbar_wait(smem_u32(&sh.stall), 0, p.wait_cycles);
                stall = false;
            }
            have = __all_sync(0xffffffffu, ok);
            if (!have && lane == 0) {
                report(p, kTimeout);
                atomicExch(&sh.abort_flag, 1);
            }
        }
        aborted = aborted || !have;
        seg_bad |= aborted ? 1 : 0;

        const int slot0 = WIN ? tile_slot0(cur, kTile) : cur.t * kTile;
        const uint32_t kbase = ring_u32 + stage * kStageBytes;
        const uint32_t vbase = kbase + kKVB;
        uint8_t *kring = ring + stage * kStageBytes;
        uint8_t *vring = kring + kKVB;
        const int tile_bad = have ? sh.stage_bad[stage] : 1;
        seg_bad |= tile_bad;
        if (first_of_seg && have && row_good) {
            // Q fragments from the ring (rows g0 < G): dims 16ks + 2q4 (+1)
            // and 16ks + 8 + 2q4 (+1) of head g0
            if constexpr (QF32) {
                const float *qs = reinterpret_cast<const float *>(kring + 2 * kKVB) + g0 * kD;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qa[ks][0] = qa[ks][1] = ql[ks][0] = ql[ks][1] = 0u;
                    if (g0 < (MULTI ? qrows : G)) {
                        // over an E4M3 cache the k-step's dims are taken in the
                        // order the byte fragments of K deliver them (4 q4 .. +3)
                        const int d0 = KV8 ? 16 * ks + 4 * q4 : 16 * ks + 2 * q4;
                        const int d1 = KV8 ? 16 * ks + 4 * q4 + 2 : 16 * ks + 8 + 2 * q4;
                        const float2 v0 = *reinterpret_cast<const float2 *>(qs + d0);
                        const float2 v1 = *reinterpret_cast<const float2 *>(qs + d1);
                        if constexpr (KV8) {   // f16 products over an E4M3 cache
                            split_f16(v0, qa[ks][0], ql[ks][0]);
                            split_f16(v1, qa[ks][1], ql[ks][1]);
                        } else {
                            split_bf16(v0, qa[ks][0], ql[ks][0]);
                            split_bf16(v1, qa[ks][1], ql[ks][1]);
                        }
                    }
                }
            } else if constexpr (KV8) {
                // bf16 query as f16 (exact in the normal range); a multi-token
                // unit's row g0 + 8 is a query row of its own
                const uint8_t *qs = kring + 2 * kKVB + (rq0 + g0) * (kD * 2);
                const int nrow = MULTI ? qrows : G;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qa[ks][0] = qa[ks][1] = 0u;
                    if (rq0 + g0 < nrow) {
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(qs + (16 * ks + 4 * q4) * 2);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(qs + (16 * ks + 4 * q4 + 2) * 2);
                        qa[ks][0] = pack_f16(bf16_lo(w0), bf16_hi(w0));
                        qa[ks][1] = pack_f16(bf16_lo(w1), bf16_hi(w1));
                    }
                    if constexpr (kMside) {
                        ql[ks][0] = ql[ks][1] = 0u;
                        if (rq0 + g0 + 8 < nrow) {
                            const uint8_t *qs1 = qs + 8 * (kD * 2);
                            const uint32_t w0 = *reinterpret_cast<const uint32_t *>(qs1 + (16 * ks + 4 * q4) * 2);
                            const uint32_t w1 =
                                *reinterpret_cast<const uint32_t *>(qs1 + (16 * ks + 4 * q4 + 2) * 2);
                            ql[ks][0] = pack_f16(bf16_lo(w0), bf16_hi(w0));
                            ql[ks][1] = pack_f16(bf16_lo(w1), bf16_hi(w1));
                        }
                    }
                }
            } else {
                const uint8_t *qs = kring + 2 * kKVB + (rq0 + g0) * (kD * 2);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const bool on = rq0 + g0 < (MULTI ? qrows : G);
                    qa[ks][0] = on ? *reinterpret_cast<const uint32_t *>(qs + (16 * ks + 2 * q4) * 2) : 0u;
                    qa[ks][1] = on ? *reinterpret_cast<const uint32_t *>(qs + (16 * ks + 8 + 2 * q4) * 2) : 0u;
                    if constexpr (kMside) {   // row g0 + 8: a query row of its own
                        const bool on1 = rq0 + g0 + 8 < qrows;
                        const uint8_t *qs1 = qs + 8 * (kD * 2);
                        ql[ks][0] = on1 ? *reinterpret_cast<const uint32_t *>(qs1 + (16 * ks + 2 * q4) * 2) : 0u;
                        ql[ks][1] = on1 ? *reinterpret_cast<const uint32_t *>(qs1 + (16 * ks + 8 + 2 * q4) * 2) : 0u;
                    }
                }
            }
        }

        const bool last_tile = (cur.t == cur.nr - 1);
        // tiles holding new tokens: the last one; in a multi-token step
        // every tile reaching the row's write offset
        const bool newt = MULTI ? (slot0 + kTile - 1 >= cur.Lb) : last_tile;
        // tiles that hold slots outside some row's softmax: those, and,
        // with a window, those below the last row's window start
        const bool partial = newt || (WIN && slot0 < (MULTI ? max(0, L - p.window + 1) : cur.lo));
        const bool work = have && row_good && !tile_bad;
        {
            if (work && partial) {
                // new-token rows: substituted from k_new / v_new (and appended
                // by the unit owning the token); rows no query row attends:
                // zero V
                if constexpr (KV8 && MULTI) {
                    // this warp's rows holding new tokens, quantised into the
                    // ring; the unit that owns a token appends it (lanes 0-7:
                    // K, 8-15: V, sixteen elements each)
                    const int first_new = max(cur.Lb, slot0 + row0);
                    const int last_new = min(L, slot0 + row0 + 15);
                    const int c16 = lane & 7;
                    const bool is_k = lane < 8;
                    const float qsc = lane < 16 ? __ldg((is_k ? p.k_scale : p.v_scale) + kvh) : 1.f;
                    for (int sn = first_new; sn <= last_new && lane < 16; ++sn) {
                        const int lr = sn - slot0;
                        const long long tok = cur.tokL - (L - sn);
                        const long long nidx = (tok * p.Hkv + kvh) * kD;
                        const uint4 *src = reinterpret_cast<const uint4 *>((is_k ? knew : vnew) + nidx) + 2 * c16;
                        const uint4 q8 = quant_e4m3x16(__ldg(src), __ldg(src + 1), qsc);
                        *reinterpret_cast<uint4 *>((is_k ? kring : vring) + swz(lr, c16)) = q8;
                        if (sn > L - cur.nq) {
                            const long long off = slot_offset(p, b, kvh, sn);
                            if (off >= 0)
                                reinterpret_cast<uint4 *>(static_cast<uint8_t *>(is_k ? p.k_cache : p.v_cache) +
                                                          off)[c16] = q8;
                        }
                    }
                } else if constexpr (KV8) {
                    // row L of the last tile: the new token, quantised into the
                    // ring and appended to the cache (lanes 0-7: K, 8-15: V,
                    // sixteen elements each)
                    const int lr = L - slot0;
                    if (last_tile && !p.attend && lr >= row0 && lr < row0 + 16 && lane < 16) {
                        const int c16 = lane & 7;
                        const bool is_k = lane < 8;
                        // the new token's rows, brought into the stage by the producer
                        const uint4 *src = reinterpret_cast<const uint4 *>(kring + 2 * kKVB + RG::kQBytes +
                                                                           (is_k ? 0 : kD * 2)) + 2 * c16;
                        const uint4 q8 = quant_e4m3x16(src[0], src[1], __ldg((is_k ? p.k_scale : p.v_scale) + kvh));
                        *reinterpret_cast<uint4 *>((is_k ? kring : vring) + swz(lr, c16)) = q8;
                        const long long off = slot_offset(p, b, kvh, L);
                        if (off >= 0)
                            reinterpret_cast<uint4 *>(static_cast<uint8_t *>(is_k ? p.k_cache : p.v_cache) + off)[c16] = q8;
                    }
                } else if constexpr (MULTI) {
                    // this warp's rows holding new tokens
                    const int first_new = max(cur.Lb, slot0 + row0);
                    const int last_new = min(L, slot0 + row0 + 15);
                    for (int sn = first_new; sn <= last_new; ++sn) {
                        const int lr = sn - slot0;
                        const long long tok = cur.tokL - (L - sn);
                        const long long nidx = (tok * p.Hkv + kvh) * kD;
                        const int c = lane & 15;          // 16-byte chunk of the row
                        const int half = c >> 3, c8 = c & 7;
                        const uint4 *src = reinterpret_cast<const uint4 *>((lane < 16 ? knew : vnew) + nidx) + c;
                        const uint4 v = __ldg(src);
                        uint8_t *dst = (lane < 16 ? kring : vring) + half * kHalfBytes + swz(lr, c8);
                        *reinterpret_cast<uint4 *>(dst) = v;
                        // the in-place append, by the unit that owns the token
                        if (sn > L - cur.nq) {
                            const long long off = slot_offset(p, b, kvh, sn);
                            if (off >= 0) {
                                __nv_bfloat16 *cache = static_cast<__nv_bfloat16 *>(lane < 16 ? p.k_cache : p.v_cache);
                                reinterpret_cast<uint4 *>(cache + off)[c] = v;
                            }
                        }
                    }
                } else {
                    // row L of the last tile: the new token
                    const int lr = L - slot0;            // 0..63 in the last tile
                    if (last_tile && !p.attend && lr >= row0 && lr < row0 + 16) {
                        const long long nidx = ((long long)b * p.Hkv + kvh) * kD;
                        const int c = lane & 15;          // 16-byte chunk of the row
                        const int half = c >> 3, c8 = c & 7;
                        const uint4 *src = reinterpret_cast<const uint4 *>((lane < 16 ? knew : vnew) + nidx) + c;
                        const uint4 v = __ldg(src);
                        uint8_t *dst = (lane < 16 ? kring : vring) + half * kHalfBytes + swz(lr, c8);
                        *reinterpret_cast<uint4 *>(dst) = v;
                        // the in-place append
                        const long long off = slot_offset(p, b, kvh, L);
                        if (off >= 0) {
                            __nv_bfloat16 *cache = static_cast<__nv_bfloat16 *>(lane < 16 ? p.k_cache : p.v_cache);
                            reinterpret_cast<uint4 *>(cache + off)[c] = v;
                        }
                    }
                }
                if constexpr (KV8) {
                    for (int r = row0 + (lane >> 3); r < row0 + 16; r += 4) {
                        if (WIN ? !attended(L, cur.lo, cur.P, slot0 + r) : slot0 + r > L)
                            *reinterpret_cast<uint4 *>(vring + swz(r, lane & 7)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                } else {
                    for (int r = row0 + (lane >> 4); r < row0 + 16; r += 2) {
                        if (WIN ? !attended(L, cur.lo, cur.P, slot0 + r) : slot0 + r > L) {
                            const int c = lane & 15;
                            *reinterpret_cast<uint4 *>(vring + (c >> 3) * kHalfBytes + swz(r, c & 7)) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                __syncwarp();
            }
        }
        // 32-row units: a warp computes on slots that its pair partner
        // substituted or zeroed (whatever either warp's wait gave: both walk
        // the same tiles)
        if constexpr (kM32) {
            if (partial && row_good)
                pair_sync(warp >> 1);
        }
        if (work) {
            if constexpr (kMside) {
                // (32-row units over a bfloat16 cache: the passes one after the
                // other, fewer spills; measured paged q_len 3 578 -> 542 us.
                // Over an E4M3 cache the unrolled form is faster: 524 vs 600 us)
#pragma unroll(KV8 ? 2 : 1)
                for (int sb = 0; sb < (kM32 ? 2 : 1); ++sb) {
                    // the 16 slots of this pass: the warp's own (16-row units), or
                    // half sb of its 32 (32-row units)
                    const int crow = kM32 ? 32 * (warp >> 1) + 16 * sb : row0;
                    // ---- S = Q K^T for these 16 slots (two n-tiles of 8);
                    // rows g0 and g0 + 8 are query rows of their own; even and odd
                    // k-steps accumulate separately (shorter chains)
                    float s_acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    {
                        float s_odd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                        const int mi = lane >> 3, ri = lane & 7;
                        const int r = crow + 8 * (mi >> 1) + ri;
                        if constexpr (KV8) {
                            // matrix mi: slots 8 (mi >> 1) .. +7, k-step 2 kp + (mi & 1)
                            // (16 bytes of each row)
#pragma unroll
                            for (int kp = 0; kp < 4; ++kp) {
                                uint32_t kb[4];
                                ldsm_x4(kbase + swz(r, 2 * kp + (mi & 1)), kb);
#pragma unroll
                                for (int mm = 0; mm < 4; ++mm) {
                                    const int ks = 2 * kp + (mm & 1), nt = mm >> 1;
                                    uint32_t b0, b1;
                                    e4m3x4_to_f16(kb[mm], b0, b1);
                                    float(&acc)[2][4] = (ks & 1) ? s_odd : s_acc;
                                    mma_f16(acc[nt], qa[ks][0], ql[ks][0], qa[ks][1], ql[ks][1], b0, b1);
                                }
                            }
                        } else {
#pragma unroll
                            for (int ks = 0; ks < 8; ++ks) {
                                const int c = 2 * ks + (mi & 1);
                                uint32_t kb[4];
                                float(&acc)[2][4] = (ks & 1) ? s_odd : s_acc;
                                ldsm_x4(kbase + (c >> 3) * kHalfBytes + swz(r, c & 7), kb);
                                mma_bf16(acc[0], qa[ks][0], ql[ks][0], qa[ks][1], ql[ks][1], kb[0], kb[1]);
                                mma_bf16(acc[1], qa[ks][0], ql[ks][0], qa[ks][1], ql[ks][1], kb[2], kb[3]);
                            }
                        }
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                s_acc[nt][e] += s_odd[nt][e];
                    }
                    // two query rows per lane, g0 (c0, c1) and g0 + 8 (c2, c3), each
                    // with its own causal bound, window and softmax state; P in bf16
                    // (f16 over an E4M3 cache)
                    uint32_t pa[4];
                    const float ssl = KV8 ? ssc : p.scale_log2;
                    float x0[2][2], x1[2][2];
                    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int j = slot0 + crow + 8 * nt + 2 * q4 + e;
                            const bool on0 = WIN ? attended(lim, lo_r, cur.P, j) : j <= lim;
                            const bool on1 = WIN ? attended(lim1, lo_r1, cur.P, j) : j <= lim1;
                            x0[nt][e] = (!partial || on0) ? s_acc[nt][e] * ssl : -INFINITY;
                            x1[nt][e] = (!partial || on1) ? s_acc[nt][e + 2] * ssl : -INFINITY;
                            mx0 = fmaxf(mx0, x0[nt][e]);
                            mx1 = fmaxf(mx1, x1[nt][e]);
                        }
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                    if (mx0 > m_run + 8.f) {
                        const float alpha = (m_run == -INFINITY) ? 0.f : fast_ex2(m_run - mx0);
                        l_run *= alpha;
#pragma unroll
                        for (int n = 0; n < kOT; ++n) {
                            acc_o[n][0] *= alpha;
                            acc_o[n][1] *= alpha;
                        }
                        m_run = mx0;
                    }
                    if (mx1 > m_run1 + 8.f) {
                        const float alpha = (m_run1 == -INFINITY) ? 0.f : fast_ex2(m_run1 - mx1);
                        l_run1 *= alpha;
#pragma unroll
                        for (int n = 0; n < kOT; ++n) {
                            acc_o[n][2] *= alpha;
                            acc_o[n][3] *= alpha;
                        }
                        m_run1 = mx1;
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        float p0[2], p1[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            p0[e] = (x0[nt][e] == -INFINITY) ? 0.f : fast_ex2(x0[nt][e] - m_run);
                            p1[e] = (x1[nt][e] == -INFINITY) ? 0.f : fast_ex2(x1[nt][e] - m_run1);
                            l_run += p0[e];
                            l_run1 += p1[e];
                        }
                        // row g0: slots 8nt + 2q4, +1; then row g0 + 8
                        pa[2 * nt] = KV8 ? pack_f16(p0[0], p0[1]) : pack_bf16(p0[0], p0[1]);
                        pa[2 * nt + 1] = KV8 ? pack_f16(p1[0], p1[1]) : pack_bf16(p1[0], p1[1]);
                    }
                    // ---- O += P V (16 n-tiles of 8 dims)
                    {
                        const int mi = lane >> 3, ri = lane & 7;
                        const int r = crow + 8 * (mi & 1) + ri;
                        if constexpr (KV8) {
                            // matrix mi: slots 8 (mi & 1) .. +7, 16-dim block
                            // 2 bp + (mi >> 1); each lane gets bytes (s, d), (s, d+1),
                            // (s+1, d), (s+1, d+1) and splits them into the (s, s+1)
                            // pairs of dim d (even) and d + 1 (odd)
#pragma unroll
                            for (int bp = 0; bp < 4; ++bp) {
                                uint32_t vb[4];
                                ldsm_x4_t(vbase + swz(r, 2 * bp + (mi >> 1)), vb);
                                uint32_t ev[4], od[4];
#pragma unroll
                                for (int mm = 0; mm < 4; ++mm)
                                    e4m3x4_to_f16(__byte_perm(vb[mm], 0u, 0x3120u), ev[mm], od[mm]);
#pragma unroll
                                for (int hb = 0; hb < 2; ++hb) {   // block 2 bp + hb: matrices 2 hb (slots 0-7), 2 hb + 1
                                    const int blk = 2 * bp + hb;
                                    mma_f16(acc_o[2 * blk], pa[0], pa[1], pa[2], pa[3], ev[2 * hb], ev[2 * hb + 1]);
                                    mma_f16(acc_o[2 * blk + 1], pa[0], pa[1], pa[2], pa[3], od[2 * hb], od[2 * hb + 1]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int np = 0; np < 8; ++np) {
                                const int c = 2 * np + (mi >> 1);
                                uint32_t vb[4];
                                ldsm_x4_t(vbase + (c >> 3) * kHalfBytes + swz(r, c & 7), vb);
                                mma_bf16(acc_o[2 * np], pa[0], pa[1], pa[2], pa[3], vb[0], vb[1]);
                                mma_bf16(acc_o[2 * np + 1], pa[0], pa[1], pa[2], pa[3], vb[2], vb[3]);
                            }
                        }
                    }
                }
            } else {
                // ---- S^T = K Q^T: M = this warp's 16 slots, N = the 8 query
                // rows, K = 16 dims per step. Lane (g0, q4) holds the scores of
                // slots g0 (c0, c1) and g0 + 8 (c2, c3) for query rows 2 q4
                // (c0, c2) and 2 q4 + 1 (c1, c3). Even and odd k-steps
                // accumulate separately (shorter chains).
                float st[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    float st2[4] = {0.f, 0.f, 0.f, 0.f};
                    const int mi = lane >> 3, ri = lane & 7;
                    if constexpr (KV8) {
                        // matrix mi: slots 8 (mi >> 1) .. +7, byte chunk
                        // 2 kp + (mi & 1); each lane gets bytes 4 q4 .. +3 of its
                        // slot, i.e. the k-step's dims in the permuted order the
                        // query fragments use
                        const int r = row0 + 8 * (mi >> 1) + ri;
#pragma unroll
                        for (int kp = 0; kp < 4; ++kp) {
                            uint32_t kb[4];
                            ldsm_x4(kbase + swz(r, 2 * kp + (mi & 1)), kb);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int ks = 2 * kp + h;
                                uint32_t lo0, hi0, lo1, hi1;
                                e4m3x4_to_f16(kb[h], lo0, hi0);       // slots 0-7
                                e4m3x4_to_f16(kb[2 + h], lo1, hi1);   // slots 8-15
                                float(&acc)[4] = h ? st2 : st;
                                mma_f16(acc, lo0, lo1, hi0, hi1, qa[ks][0], qa[ks][1]);
                                if constexpr (QF32)   // the query remainders
                                    mma_f16(acc, lo0, lo1, hi0, hi1, ql[ks][0], ql[ks][1]);
                            }
                        }
                    } else {
                        // matrix mi: slots 8 (mi & 1) .. +7, dims 16 ks + 8 (mi >> 1) .. +7
                        const int r = row0 + 8 * (mi & 1) + ri;
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const int c = 2 * ks + (mi >> 1);
                            uint32_t kb[4];
                            ldsm_x4(kbase + (c >> 3) * kHalfBytes + swz(r, c & 7), kb);
                            float(&acc)[4] = (ks & 1) ? st2 : st;
                            mma_bf16(acc, kb[0], kb[1], kb[2], kb[3], qa[ks][0], qa[ks][1]);
                            if constexpr (QF32)   // the query remainders
                                mma_bf16(acc, kb[0], kb[1], kb[2], kb[3], ql[ks][0], ql[ks][1]);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        st[e] += st2[e];
                }
                // ---- masked online softmax (base 2) of rows 2 q4 (m_run) and
                // 2 q4 + 1 (m_run1); only the partial tiles (the last one, those
                // below a window's start) test slots. The row maxima need a
                // reduction over the eight lanes sharing q4, which the lazy
                // rescale makes rare: it runs only when some lane sees a score
                // above its row's running max + 8 (a warp vote).
                const float sl = KV8 ? ssc : p.scale_log2;
                const int j0 = slot0 + row0 + g0;
                bool on00, on01, on10, on11;   // (row 2 q4 + i, slot j0 + 8 k)
                if constexpr (MULTI) {         // each row its own causal bound and window
                    on00 = !partial || (WIN ? attended(lim, lo_r, cur.P, j0) : j0 <= lim);
                    on01 = !partial || (WIN ? attended(lim, lo_r, cur.P, j0 + 8) : j0 + 8 <= lim);
                    on10 = !partial || (WIN ? attended(lim1, lo_r1, cur.P, j0) : j0 <= lim1);
                    on11 = !partial || (WIN ? attended(lim1, lo_r1, cur.P, j0 + 8) : j0 + 8 <= lim1);
                } else {
                    on00 = on10 = !partial || (WIN ? attended(L, cur.lo, cur.P, j0) : j0 <= L);
                    on01 = on11 = !partial || (WIN ? attended(L, cur.lo, cur.P, j0 + 8) : j0 + 8 <= L);
                }
                const float x00 = on00 ? st[0] * sl : -INFINITY;   // row 2 q4,     slot g0
                const float x10 = on10 ? st[1] * sl : -INFINITY;   // row 2 q4 + 1, slot g0
                const float x01 = on01 ? st[2] * sl : -INFINITY;   // row 2 q4,     slot g0 + 8
                const float x11 = on11 ? st[3] * sl : -INFINITY;   // row 2 q4 + 1, slot g0 + 8
                float mx0 = fmaxf(x00, x01), mx1 = fmaxf(x10, x11);
                if (__any_sync(0xffffffffu, mx0 > m_run + 8.f || mx1 > m_run1 + 8.f)) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    if (mx0 > m_run + 8.f) {   // raise the running max (also from -inf)
                        const float alpha = (m_run == -INFINITY) ? 0.f : fast_ex2(m_run - mx0);
                        l_run *= alpha;
#pragma unroll
                        for (int n = 0; n < kOT; ++n) {
                            acc_o[n][0] *= alpha;
                            acc_o[n][2] *= alpha;
                        }
                        m_run = mx0;
                    }
                    if (mx1 > m_run1 + 8.f) {
                        const float alpha = (m_run1 == -INFINITY) ? 0.f : fast_ex2(m_run1 - mx1);
                        l_run1 *= alpha;
#pragma unroll
                        for (int n = 0; n < kOT; ++n) {
                            acc_o[n][1] *= alpha;
                            acc_o[n][3] *= alpha;
                        }
                        m_run1 = mx1;
                    }
                }
                const float p00 = (x00 == -INFINITY) ? 0.f : fast_ex2(x00 - m_run);
                const float p01 = (x01 == -INFINITY) ? 0.f : fast_ex2(x01 - m_run);
                const float p10 = (x10 == -INFINITY) ? 0.f : fast_ex2(x10 - m_run1);
                const float p11 = (x11 == -INFINITY) ? 0.f : fast_ex2(x11 - m_run1);
                l_run += p00 + p01;
                l_run1 += p10 + p11;
                // P^T as the B operand of the next product: the lane's pairs
                // (slot g0; rows 2 q4, 2 q4 + 1) transposed in registers into
                // (row g0; slots 2 q4, 2 q4 + 1), per half of the 16 slots. Over
                // a bf16 cache P enters as bf16 + a bf16 remainder (a second
                // product), so the weights keep ~16 significant bits and the
                // result does not depend on the split of a unit beyond float32
                // rounding; over an E4M3 cache as f16 (11 bits).
                uint32_t ph0, ph1, pl0 = 0u, pl1 = 0u;
                if constexpr (KV8) {
                    ph0 = pack_f16(p00, p10);
                    ph1 = pack_f16(p01, p11);
                } else {
                    split_bf16(make_float2(p00, p10), ph0, pl0);
                    split_bf16(make_float2(p01, p11), ph1, pl1);
                    pl0 = movmatrix_t(pl0);
                    pl1 = movmatrix_t(pl1);
                }
                const uint32_t pb0 = movmatrix_t(ph0), pb1 = movmatrix_t(ph1);
                // ---- O^T += V^T P^T: M = 16 dims per tile, N = the 8 query
                // rows, K = the 16 slots. Lane (g0, q4) accumulates rows 2 q4
                // (c0, c2) and 2 q4 + 1 (c1, c3).
                {
                    const int mi = lane >> 3, ri = lane & 7;
                    const int r = row0 + 8 * (mi & 1) + ri;
                    if constexpr (KV8) {
                        // matrix mi: slots 8 (mi & 1) .. +7, byte chunk
                        // 2 bp + (mi >> 1); each lane gets bytes (s, d), (s, d+1),
                        // (s+1, d), (s+1, d+1), d = 16 chunk + 2 g0, s = 2 q4, and
                        // one byte permute splits them into the (s, s+1) pairs of
                        // dim d (A rows 0-7) and dim d + 1 (A rows 8-15)
#pragma unroll
                        for (int bp = 0; bp < 4; ++bp) {
                            uint32_t vb[4];
                            ldsm_x4_t(vbase + swz(r, 2 * bp + (mi >> 1)), vb);
#pragma unroll
                            for (int hb = 0; hb < 2; ++hb) {   // chunk 2 bp + hb
                                uint32_t e0, o0, e1, o1;
                                e4m3x4_to_f16(__byte_perm(vb[2 * hb], 0u, 0x3120u), e0, o0);       // slots 0-7
                                e4m3x4_to_f16(__byte_perm(vb[2 * hb + 1], 0u, 0x3120u), e1, o1);   // slots 8-15
                                mma_f16(acc_o[2 * bp + hb], e0, o0, e1, o1, pb0, pb1);
                            }
                        }
                    } else {
                        // matrix mi: slots 8 (mi & 1) .. +7, dims 16 mt + 8 (mi >> 1) .. +7
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            const int c = 2 * mt + (mi >> 1);
                            uint32_t vb[4];
                            ldsm_x4_t(vbase + (c >> 3) * kHalfBytes + swz(r, c & 7), vb);
                            mma_bf16(acc_o[mt], vb[0], vb[2], vb[1], vb[3], pb0, pb1);
                            mma_bf16(acc_o[mt], vb[0], vb[2], vb[1], vb[3], pl0, pl1);   // the remainders
                        }
                    }
                }
            }
            if (partial)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0 && have)
            mbar_arrive(smem_u32(&sh.empty[stage]));
        if (++stage == kNS) {
            stage = 0;
            phase ^= 1;
        }

        const bool unit_done = (cur.t == cur.nr - 1);
        const bool range_done = (cur.g + 1 == cur.end);
        if (unit_done || range_done) {
            // a cut unit's arrival ticket (and the merge, when last) handed to the
            // finisher warp: not in the CTA's last segment, where nothing is left
            // to overlap with and four warps merge faster than one
            const bool to_fin = RG::kFin && !(range_done && (in_b || walk.b.g >= walk.b.end));
            auto post_job = [&] {
                if constexpr (RG::kFin) {
                    const long long first_tile = cur.g - cur.t;
                    job_wait_free();
                    if (tid == 0) {
                        FinJob j;
                        j.stop = 0;
                        j.first = cta_of_tile(first_tile, walk.N, walk.C);
                        j.last = cta_of_tile(first_tile + cur.nr - 1, walk.N, walk.C);
                        j.b = cur.b;
                        j.kvh = cur.kvh;
                        j.nq = MULTI ? cur.nq : 1;
                        j.tokL = MULTI ? cur.tokL : cur.b;
                        sh.fin.job = j;
                    }
                    job_post();
                }
            };
            if constexpr (kM32) {
                // ---- 32-row units: warps 2 and 3 (slots 32-63 of every tile)
                // hand their states of rows rq0 + g0 and rq0 + g0 + 8 to warps 0
                // and 1 (slots 0-31, the same rows), which merge them in registers
                // and write the output (a whole unit) or the partial state
                float l_tot = l_run, l_tot1 = l_run1;
                l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
                l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
                l_tot1 += __shfl_xor_sync(0xffffffffu, l_tot1, 1);
                l_tot1 += __shfl_xor_sync(0xffffffffu, l_tot1, 2);
                const float osc = KV8 ? vsc : 1.f;   // the V scale of an E4M3 cache
                // n-tile n holds dims dn(n) (c0, c2) and dn(n) + de (c1, c3)
                constexpr int de = KV8 ? 2 : 1;
                auto dn = [&](int n) { return KV8 ? 16 * (n >> 1) + 4 * q4 + (n & 1) : 8 * n + 2 * q4; };
                if (warp >= 2) {
                    const int sw = warp - 2;
                    if (q4 == 0) {
                        sh.m[sw][g0] = m_run;
                        sh.l[sw][g0] = l_tot;
                        sh.m[sw][g0 + 8] = m_run1;
                        sh.l[sw][g0 + 8] = l_tot1;
                    }
    #pragma unroll
                    for (int n = 0; n < kOT; ++n) {
                        const int d = dn(n);
                        sh.o[sw][g0][d] = acc_o[n][0] * osc;
                        sh.o[sw][g0][d + de] = acc_o[n][1] * osc;
                        sh.o[sw][g0 + 8][d] = acc_o[n][2] * osc;
                        sh.o[sw][g0 + 8][d + de] = acc_o[n][3] * osc;
                    }
                }
                const bool bad = consumer_sync_or(!row_good || seg_bad);
                const bool any_abort = consumer_sync_or(aborted);
                if (bad && row_good && tid == 0)
                    report(p, any_abort ? kTimeout : kBadBlock);
                const bool whole = (seg_first_t == 0) && unit_done;
                if (warp < 2) {
                    const int G = p.G;
                    const int nrow = p.Gh * cur.nq;           // query rows with an output
                    const long long P = (long long)cur.b * p.Hkv + cur.kvh + blockIdx.x;
                    const float qnan = __int_as_float(0x7fc00000);
                    float sc[2], wo[2], wl[2];                // per row: own weight, other's weight
                    int rr[2];
    #pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int gr = g0 + 8 * h;            // row within the warp's 16
                        const float ms = h ? m_run1 : m_run, ls = h ? l_tot1 : l_tot;
                        const float mo = sh.m[warp][gr], lo = sh.l[warp][gr];
                        float M = fmaxf(ms, mo);
                        const float as = (ms == -INFINITY) ? 0.f : fast_ex2(ms - M);
                        const float ao = (mo == -INFINITY) ? 0.f : fast_ex2(mo - M);
                        float den = as * ls + ao * lo;
                        rr[h] = rq0 + gr;
                        wl[h] = as * osc;
                        wo[h] = ao;
                        if (whole) {
                            // the normalisation, with the sink logit when given
                            const float sk = p.sink ? sink_log2(p, cur.kvh * p.Gh + rr[h] % p.Gh) : -INFINITY;
                            const float Mx = fmaxf(M, sk);
                            const float a = (M == -INFINITY) ? 0.f : fast_ex2(M - Mx);
                            den = a * den + ((sk == -INFINITY) ? 0.f : fast_ex2(sk - Mx));
                            sc[h] = a / den;
                        } else {
                            sc[h] = 1.f;
                            if (q4 == 0 && rr[h] < G) {
                                p.ws_ml[(P * G + rr[h]) * 2 + 0] = bad ? qnan : M;
                                p.ws_ml[(P * G + rr[h]) * 2 + 1] = bad ? qnan : den;
                            }
                        }
                    }
    #pragma unroll
                    for (int n = 0; n < kOT; ++n) {
                        const int d = dn(n);
    #pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int gr = g0 + 8 * h;
                            const float v0 = fmaf(wl[h], acc_o[n][2 * h], wo[h] * sh.o[warp][gr][d]) * sc[h];
                            const float v1 = fmaf(wl[h], acc_o[n][2 * h + 1], wo[h] * sh.o[warp][gr][d + de]) * sc[h];
                            float *dst = nullptr;
                            if (whole && rr[h] < nrow)
                                dst = out_row<MULTI>(p, cur, rr[h], kD);
                            else if (!whole && rr[h] < G)
                                dst = p.ws_o + (P * G + rr[h]) * kD;
                            if (dst) {
                                dst[d] = bad ? qnan : v0;
                                dst[d + de] = bad ? qnan : v1;
                            }
                        }
                    }
                }
                consumer_sync();   // the output or partial stores before the ticket
                if (!whole) {
                    if (to_fin) {
                        post_job();
                    } else {
                        const long long first_tile = cur.g - cur.t;
                        const int first = cta_of_tile(first_tile, walk.N, walk.C);
                        const int last = cta_of_tile(first_tile + cur.nr - 1, walk.N, walk.C);
                        unit_ticket_merge<kD, MULTI, !KV8>(p, cur, first, last, &sh.last_flag, sh.merge, tid,
                                                           kConsumerWarps * 32, [] { consumer_sync(); }, pre_cnt);
                    }
                }
            } else {
                // ---- merge the four warps' states and emit
                if constexpr (kMside) {   // rows g0 and g0 + 8, each its own query row
                    float l_tot = l_run;
                    l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
                    l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
                    float l_tot1 = l_run1;
                    l_tot1 += __shfl_xor_sync(0xffffffffu, l_tot1, 1);
                    l_tot1 += __shfl_xor_sync(0xffffffffu, l_tot1, 2);
                    if (q4 == 0) {
                        sh.m[warp][g0] = m_run;
                        sh.l[warp][g0] = l_tot;
                        sh.m[warp][g0 + 8] = m_run1;
                        sh.l[warp][g0 + 8] = l_tot1;
                    }
    #pragma unroll
                    for (int n = 0; n < kOT; ++n) {
                        if constexpr (KV8) {
                            // n-tile n = 2 blk + parity holds dims 16 blk + 4 q4 +
                            // parity (+2); times the V scale
                            const int d = 16 * (n >> 1) + 4 * q4 + (n & 1);
                            sh.o[warp][g0][d] = acc_o[n][0] * vsc;
                            sh.o[warp][g0][d + 2] = acc_o[n][1] * vsc;
                            sh.o[warp][g0 + 8][d] = acc_o[n][2] * vsc;
                            sh.o[warp][g0 + 8][d + 2] = acc_o[n][3] * vsc;
                        } else {
                            *reinterpret_cast<float2 *>(&sh.o[warp][g0][8 * n + 2 * q4]) =
                                make_float2(acc_o[n][0], acc_o[n][1]);
                            *reinterpret_cast<float2 *>(&sh.o[warp][g0 + 8][8 * n + 2 * q4]) =
                                make_float2(acc_o[n][2], acc_o[n][3]);
                        }
                    }
                } else {
                    // rows 2 q4 and 2 q4 + 1; the eight lanes sharing q4 hold
                    // different slots of them
                    float l_tot = l_run, l_tot1 = l_run1;
    #pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        l_tot += __shfl_xor_sync(0xffffffffu, l_tot, off);
                        l_tot1 += __shfl_xor_sync(0xffffffffu, l_tot1, off);
                    }
                    const int r0 = 2 * q4, r1 = r0 + 1;
                    if (g0 == 0) {
                        if (r0 < G) {
                            sh.m[warp][r0] = m_run;
                            sh.l[warp][r0] = l_tot;
                        }
                        if (r1 < G) {
                            sh.m[warp][r1] = m_run1;
                            sh.l[warp][r1] = l_tot1;
                        }
                    }
    #pragma unroll
                    for (int n = 0; n < kOT; ++n) {
                        if constexpr (KV8) {
                            // m-tile n: dims 16 n + 2 g0 (c0, c1) and + 1 (c2, c3);
                            // times the V scale
                            const int d = 16 * n + 2 * g0;
                            if (r0 < G)
                                *reinterpret_cast<float2 *>(&sh.o[warp][r0][d]) =
                                    make_float2(acc_o[n][0] * vsc, acc_o[n][2] * vsc);
                            if (r1 < G)
                                *reinterpret_cast<float2 *>(&sh.o[warp][r1][d]) =
                                    make_float2(acc_o[n][1] * vsc, acc_o[n][3] * vsc);
                        } else {
                            // m-tile n: dims 16 n + g0 (c0, c1) and + 8 (c2, c3)
                            const int d = 16 * n + g0;
                            if (r0 < G) {
                                sh.o[warp][r0][d] = acc_o[n][0];
                                sh.o[warp][r0][d + 8] = acc_o[n][2];
                            }
                            if (r1 < G) {
                                sh.o[warp][r1][d] = acc_o[n][1];
                                sh.o[warp][r1][d + 8] = acc_o[n][3];
                            }
                        }
                    }
                }
                consumer_sync();
                const bool bad = !row_good || seg_bad;
                if (bad && row_good && tid == 0)
                    report(p, aborted ? kTimeout : kBadBlock);
                if (to_fin) {
                    // the output (a whole unit) or the partial state; a cut unit's
                    // ticket and merge go to the finisher
                    if (!segment_out<kSW, kSR, kD, kD + SharedT::kOPad, MULTI>(
                            p, cur, seg_first_t, bad, sh.m, sh.l, sh.o, sh.merge, tid, kConsumerWarps * 32,
                            [] { consumer_sync(); }))
                        post_job();
                } else {
                    // the merge's preload of partial outputs costs registers: off
                    // for the E4M3 kernels (at their 128-register cap)
                    finish_segment<kSW, kSR, kD, kD + SharedT::kOPad, MULTI, !KV8>(
                        p, cur, walk, seg_first_t, bad, sh.m, sh.l, sh.o, &sh.last_flag, sh.merge, tid,
                        kConsumerWarps * 32, [] { consumer_sync(); }, pre_cnt);
                }
            }
            seg_start = true;
        }
        more = walk_next(p, cur, walk, in_b);
    }
    if constexpr (RG::kFin) {   // no more jobs
        job_wait_free();
        if (tid == 0)
            sh.fin.job.stop = 1;
        job_post();
    }
}


template <bool QF32, bool WIN, bool MULTI, bool KV8 = false, int MR = 0>
cudaError_t launch_q(const DecodeParams &p, const TcMaps &maps, cudaStream_t st)
{
    constexpr int kDynSmem = Ring<QF32, KV8, MULTI, MR>::kDynSmem;
    // The shared-memory limit is a per-device attribute of the kernel: set it
    // once on every device this instantiation is launched on (a bit per
    // device; devices beyond 64 set it on every launch).
    static std::atomic<unsigned long long> attr_set{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(tc_decode_kernel<QF32, WIN, MULTI, KV8, MR>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
        if (e != cudaSuccess)
            return e;
        attr_set.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(Ring<QF32, KV8, MULTI, MR>::kThreads);
    cfg.dynamicSmemBytes = kDynSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_decode_kernel<QF32, WIN, MULTI, KV8, MR>, p, maps.k, maps.v, maps.k16,
                              maps.v16);
}

}  // namespace

// The instantiations live in two translation units: the single-token kernels
// (gqa_tc.cu, compiled without the multi-token schedule code) and the
// multi-token kernels (gqa_tc_multi.cu).
cudaError_t tc_launch_multi(const DecodeParams &p, const TcMaps &maps, cudaStream_t st);

}  // namespace gqa
