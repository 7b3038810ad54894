// Device-side pieces shared by the decode kernels and the split combine:
// launch parameters, the persistent tile schedule, the workspace layout and
// small numeric helpers.
//
// Work decomposition. A unit is one (batch row b, cache head kvh) pair; unit
// u = b * Hkv + kvh. Its slots 0..L (L = lengths[b]; slot L is the new token)
// are cut into tiles of T slots, n_tiles(b) = ceil((L + 1) / T). The tiles of
// all units, in (b, kvh, tile) order, form one list of N tiles, and CTA i of
// a grid takes the contiguous range [floor(i N / C), floor((i+1) N / C)) with
// C = min(grid size, N), so every working CTA owns at least one tile (CTAs
// i >= C stay idle). Every CTA therefore streams the same number of KV bytes
// (to within one tile), whatever the length mix. A unit whose tiles fall inside one CTA is
// finished there (normalised output written directly); a unit cut by CTA
// boundaries leaves one partial softmax state per CTA, (m, l, o[D]) per head,
// and the combine kernel merges them (log-sum-exp merge). The partial of CTA
// i for unit u is stored at index u + i: along the (CTA, unit) pairs in
// order, u + i grows by one or two at every step, so the index is unique and
// fewer than B * Hkv + C partials exist.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gqa {

// Status bits (mirror the public header).
constexpr int kBadLength = 1;
constexpr int kBadSlotId = 2;
constexpr int kBadBlock = 4;
constexpr int kTimeout = 8;

struct DecodeParams {
    const void *q;      // (B, Hq, D)
    const void *k_new;  // (B, Hkv, D)
    const void *v_new;  // (B, Hkv, D)
    void *k_cache;      // dense (R, Hkv, Smax, D) or blocks (num_blocks, Hkv, bs, D)
    void *v_cache;
    const int32_t *lengths;
    const int32_t *slot_ids;     // dense only, may be null
    const int32_t *block_table;  // paged only
    float *out;                  // (B, Hq, D)
    int B, Hq, Hkv, G, D;
    int R, Smax;                                     // dense
    int paged, num_blocks, block_size, max_blocks;   // paged
    float scale_log2;  // log2(e) / sqrt(D): scores are kept in base-2 units
    int tile;          // T, slots per tile
    int grid;          // C, CTAs of the decode launch
    // workspace
    long long *ws_total;   // [1] N, written by CTA 0
    long long *ws_rowpre;  // [B + 1] tiles before row b (all heads), written by CTA 0
    float *ws_ml;          // [P][G][2] partial (m, l), base-2 max
    float *ws_o;           // [P][G][D] partial unnormalised output
    int32_t *status;       // sticky content-error bits, may be null
};

// Workspace layout (bytes from the workspace base), shared by host and device.
struct WorkspaceLayout {
    size_t off_total, off_rowpre, off_ml, off_o, bytes;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WorkspaceLayout workspace_layout(int B, int Hkv, int G, int D, int grid)
{
    WorkspaceLayout w;
    const size_t P = (size_t)B * Hkv + (size_t)grid;
    w.off_total = 0;
    w.off_rowpre = 256;
    w.off_ml = align_up(w.off_rowpre + sizeof(long long) * ((size_t)B + 1), 256);
    w.off_o = align_up(w.off_ml + sizeof(float) * P * G * 2, 256);
    w.bytes = align_up(w.off_o + sizeof(float) * P * G * D, 256);
    return w;
}

// Capacity of one row in slots: lengths[b] must be below it.
__host__ __device__ inline long long row_capacity(const DecodeParams &p)
{
    return p.paged ? (long long)p.max_blocks * p.block_size : (long long)p.Smax;
}

// Tiles of batch row b for ONE cache head. Rows with bad content get one tile,
// which only writes NaN.
__device__ __forceinline__ int row_tiles(const DecodeParams &p, int L)
{
    if (L < 0 || (long long)L >= row_capacity(p))
        return 1;
    return (L + p.tile) / p.tile;  // ceil((L + 1) / T)
}

// CTAs that share the N tiles: min(grid size, N).
__device__ __forceinline__ long long working_ctas(long long N, int grid)
{
    return N < grid ? N : (long long)grid;
}

// CTA that owns global tile x: the largest i with floor(i N / C) <= x.
__device__ __forceinline__ int cta_of_tile(long long x, long long N, long long C)
{
    return (int)(((x + 1) * C - 1) / N);
}

__device__ __forceinline__ void report(const DecodeParams &p, int bits)
{
    if (p.status)
        atomicOr(p.status, bits);
}

// Position of a CTA in the tile list.
struct TileCursor {
    long long g;      // global tile index
    long long end;    // one past this CTA's last tile
    int b, kvh, t;    // current row, head, tile within the unit
    int nt;           // tiles per head of row b
    int L;            // lengths[b]
};

// Finds this CTA's first tile. Every thread of the block must call it (it
// uses __syncthreads and `scratch`, >= 2 * blockDim.x + 8 long longs of shared
// memory). CTA 0 also publishes the row prefix and the total to the workspace
// for the combine kernel.
__device__ inline TileCursor schedule_start(const DecodeParams &p, long long *scratch)
{
    const int nthr = blockDim.x, tid = threadIdx.x;
    const int chunk = (p.B + nthr - 1) / nthr;
    const int r0 = min(p.B, tid * chunk), r1 = min(p.B, r0 + chunk);
    long long local = 0;
    for (int b = r0; b < r1; ++b)
        local += (long long)p.Hkv * row_tiles(p, __ldg(p.lengths + b));
    scratch[tid] = local;
    __syncthreads();
    // inclusive scan (Hillis-Steele) over the per-thread sums
    long long *a = scratch, *c = scratch + nthr;
    for (int off = 1; off < nthr; off <<= 1) {
        long long v = a[tid] + (tid >= off ? a[tid - off] : 0);
        __syncthreads();
        c[tid] = v;
        __syncthreads();
        long long *tmp = a; a = c; c = tmp;
    }
    const long long incl = a[tid];
    const long long excl = incl - local;
    const long long N = a[nthr - 1];
    long long *found = scratch + 2 * nthr;  // [0] b, [1] tiles before b
    const long long C = working_ctas(N, p.grid);
    const long long begin = blockIdx.x < C ? (long long)blockIdx.x * N / C : N;
    const long long end = blockIdx.x < C ? ((long long)blockIdx.x + 1) * N / C : N;
    if (tid == 0) {
        found[0] = p.B;
        found[1] = N;
    }
    __syncthreads();
    long long run = excl;
    for (int b = r0; b < r1; ++b) {
        long long n = (long long)p.Hkv * row_tiles(p, __ldg(p.lengths + b));
        if (blockIdx.x == 0)
            p.ws_rowpre[b] = run;
        if (begin >= run && begin < run + n) {
            found[0] = b;
            found[1] = run;
        }
        run += n;
    }
    if (blockIdx.x == 0 && tid == 0) {
        p.ws_rowpre[p.B] = N;
        p.ws_total[0] = N;
    }
    __syncthreads();
    TileCursor cur;
    cur.g = begin;
    cur.end = end;
    cur.b = (int)found[0];
    cur.kvh = 0;
    cur.t = 0;
    cur.nt = 1;
    cur.L = 0;
    if (begin < end) {
        cur.L = __ldg(p.lengths + cur.b);
        cur.nt = row_tiles(p, cur.L);
        long long within = begin - found[1];
        cur.kvh = (int)(within / cur.nt);
        cur.t = (int)(within % cur.nt);
    }
    __syncthreads();
    return cur;
}

__device__ __forceinline__ void advance(const DecodeParams &p, TileCursor &c)
{
    ++c.g;
    if (++c.t == c.nt) {
        c.t = 0;
        if (++c.kvh == p.Hkv) {
            c.kvh = 0;
            ++c.b;
            if (c.g < c.end) {
                c.L = __ldg(p.lengths + c.b);
                c.nt = row_tiles(p, c.L);
            }
        }
    }
}

// Row-level content check: length in range, slot id in range.
__device__ __forceinline__ bool row_ok(const DecodeParams &p, int b, int L)
{
    if (L < 0 || (long long)L >= row_capacity(p))
        return false;
    if (!p.paged && p.slot_ids) {
        int r = __ldg(p.slot_ids + b);
        if (r < 0 || r >= p.R)
            return false;
    }
    return true;
}

__device__ __forceinline__ int row_error_bits(const DecodeParams &p, int b, int L)
{
    if (L < 0 || (long long)L >= row_capacity(p))
        return kBadLength;
    if (!p.paged && p.slot_ids) {
        int r = __ldg(p.slot_ids + b);
        if (r < 0 || r >= p.R)
            return kBadSlotId;
    }
    return 0;
}

// Element offset of slot s of (b, kvh) in the dense cache, or -1 when the
// paged table entry that holds it is unusable.
__device__ __forceinline__ long long slot_offset(const DecodeParams &p, int b, int kvh, int s)
{
    if (!p.paged) {
        long long r = p.slot_ids ? __ldg(p.slot_ids + b) : b;
        return ((r * p.Hkv + kvh) * p.Smax + s) * (long long)p.D;
    }
    int blk = __ldg(p.block_table + (long long)b * p.max_blocks + s / p.block_size);
    if (blk < 0 || blk >= p.num_blocks)
        return -1;
    return (((long long)blk * p.Hkv + kvh) * p.block_size + s % p.block_size) * (long long)p.D;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace gqa
