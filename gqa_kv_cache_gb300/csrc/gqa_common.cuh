// Device-side pieces shared by the decode kernels: launch parameters, the
// persistent tile schedule, the in-kernel split merge, the workspace layout
// and small numeric helpers.
//
// Work decomposition. A unit is one (batch row b, cache head kvh) pair; unit
// u = b * Hkv + kvh. Its slots 0..L are attended: in the decode step
// L = lengths[b] and slot L is the new token; in the read-only attend
// L = lengths[b] - 1 (lengths counts the valid slots). With a sliding window
// W and a kept prefix P only the slots j <= L with j > L - W or j < P are
// attended, and only the tiles that hold such a slot are listed (the prefix
// tiles, then the window tiles: the tiles in between are skipped). They are cut into tiles of T slots, n_tiles(b) = ceil((L + 1) / T). The tiles of
// all units, in (b, kvh, tile) order, form one list of N tiles, and CTA i of
// a grid takes the contiguous range [floor(i N / C), floor((i+1) N / C)) with
// C = min(grid size, N), so every working CTA owns at least one tile (CTAs
// i >= C stay idle). Every CTA therefore streams the same number of KV bytes
// (to within one tile), whatever the length mix. A unit whose tiles fall
// inside one CTA is finished there (normalised output written directly); a
// unit cut by CTA boundaries leaves one partial softmax state per CTA,
// (m, l, o[D]) per head, and the last of those CTAs to finish (an arrival
// counter per unit in the workspace) merges them with the log-sum-exp rule,
// then clears the partials and resets the counter: no second kernel is needed
// and the workspace is zero-filled again after every call. The partial of CTA
// i for unit u is stored at index u + i: along the (CTA, unit) pairs in
// order, u + i grows by one or two at every step, so the index is unique and
// fewer than B * Hkv + C partials exist.
//
// Multi-token step. A batch row with q_len new tokens is cut into chunks of
// up to tpc tokens (tpc * Gh <= 8 query rows); each (row, chunk) is a
// virtual batch row, so B above counts B_real * max_chunks virtual rows and G
// counts the query rows of a unit, (token, head) pairs in token-major order.
// Chunk c of row b attends slots 0 .. L with L the position of its last
// token; row r (token i of the chunk) is masked beyond L - (nq - 1 - i).
// Every slot at or beyond the row's write offset Lb holds a new token: it is
// taken from k_new / v_new, never from the cache, and the chunk owning the
// token writes it into the cache (the append).
#pragma once

// GQA_MULTI_TOKEN 0 compiles the multi-token branches of the schedule out (a
// translation unit that instantiates single-token kernels only: their
// streaming loops then carry none of that code). The types shared with the
// host are the same either way.
#ifndef GQA_MULTI_TOKEN
#define GQA_MULTI_TOKEN 1
#endif

#include <climits>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace gqa {

// Status bits (mirror the public header).
constexpr int kBadLength = 1;
constexpr int kBadSlotId = 2;
constexpr int kBadBlock = 4;
constexpr int kTimeout = 8;
constexpr int kBadPrefix = 16;
constexpr int kBadQLen = 32;

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
    int attend;        // 1: read-only attend (no new token, nothing written but out)
    int q_bf16;        // query dtype: 1 bfloat16, 0 float32 (the cache has its own)
    int kv8;           // 1: E4M3 cache bytes (k_new / v_new then bfloat16)
    const float *k_scale, *v_scale;  // E4M3 cache: (Hkv) dequantisation scales
    int B, Hq, Hkv, G, D;
    int R, Smax;                                     // dense
    int paged, num_blocks, block_size, max_blocks;   // paged
    float scale_log2;  // log2(e) / sqrt(D): scores are kept in base-2 units
    // softmax modifiers
    const float *sink;               // (Hq) logits folded into the denominator, or null
    int window;                      // W > 0: only the last W positions (and the prefix); 0: all
    int kept_prefix;                 // P for every row when kept_prefix_rows is null
    const int32_t *kept_prefix_rows; // (B) P per row, or null
    // multi-token step (cu_q non-null; see above)
    const int32_t *cu_q;  // (B_real + 1) packed token offsets
    int T;                // packed tokens
    int Gh;               // query heads per cache head (G = Gh * tpc query rows)
    int tpc;              // tokens per chunk
    int max_chunks;       // chunks (virtual rows) per batch row
    int max_q;            // largest accepted q_len (tpc * max_chunks)
    int tile;          // T, slots per tile
    int pad_tiles;     // W, schedule-only tiles appended to every unit (see row_tiles)
    int grid;          // C, CTAs of the decode launch
    // workspace (zero-filled between calls)
    int *ws_cnt;       // [B * Hkv] arrival counters
    float *ws_ml;      // [P][G][2] partial (m, l), base-2 max
    float *ws_o;       // [P][G][D] partial unnormalised output
    int32_t *status;   // sticky content-error bits, may be null
    long long wait_cycles;  // consumer warps: SM clock cycles before a wait for a tile gives up
    int test_stall;         // 1: the consumers' first wait also waits on a barrier nothing completes
};

// Workspace layout (bytes from the workspace base), shared by host and device.
// The workspace is zero-filled before the first call and every call leaves it
// zero-filled: the last CTA of a cut unit resets the unit's counter and clears
// the partial states it merged.
struct WorkspaceLayout {
    size_t off_cnt, cnt_bytes, off_ml, off_o, bytes;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WorkspaceLayout workspace_layout(int B, int Hkv, int G, int D, int grid)
{
    WorkspaceLayout w;
    const size_t P = (size_t)B * Hkv + (size_t)grid;
    w.off_cnt = 0;
    w.cnt_bytes = align_up(sizeof(int) * (size_t)B * Hkv, 256);
    w.off_ml = w.off_cnt + w.cnt_bytes;
    w.off_o = align_up(w.off_ml + sizeof(float) * P * G * 2, 256);
    w.bytes = align_up(w.off_o + sizeof(float) * P * G * D, 256);
    return w;
}

// Last attended slot of row b: lengths[b] in the decode step (the append
// slot), lengths[b] - 1 in the read-only attend; -1 (a bad row) when the
// attend has no valid slot. (Single-token forms; see row_geom for chunks.)
__device__ __forceinline__ int last_slot(const DecodeParams &p, int b)
{
    const int n = __ldg(p.lengths + b);
    return p.attend ? (n > 0 ? n - 1 : -1) : n;
}

// Batch row of virtual row vb.
__device__ __forceinline__ int real_row(const DecodeParams &p, int vb)
{
#if GQA_MULTI_TOKEN
    return p.cu_q ? vb / p.max_chunks : vb;
#else
    return vb;
#endif
}

// The tokens of virtual row vb of a multi-token step: nq tokens (0: an empty
// chunk; -1: the row's token offsets are bad), i0 tokens of the row before
// them, tok0 the packed index of the row's first token, Lb its write offset.
struct ChunkInfo {
    int nq, i0, tok0, Lb;
};

#if GQA_MULTI_TOKEN
__device__ __forceinline__ ChunkInfo chunk_info(const DecodeParams &p, int vb)
{
    const int b = vb / p.max_chunks, c = vb % p.max_chunks;
    const int t0 = __ldg(p.cu_q + b), t1 = __ldg(p.cu_q + b + 1);
    ChunkInfo ci;
    ci.i0 = c * p.tpc;
    ci.tok0 = t0;
    ci.Lb = __ldg(p.lengths + b);
    const int qlen = t1 - t0;
    if (t0 < 0 || t1 > p.T || qlen < 0 || qlen > p.max_q)
        ci.nq = (c == 0) ? -1 : 0;
    else
        ci.nq = max(0, min(p.tpc, qlen - ci.i0));
    return ci;
}
#endif

// Capacity of one row in slots: the last attended slot must be below it.
__host__ __device__ inline long long row_capacity(const DecodeParams &p)
{
    return p.paged ? (long long)p.max_blocks * p.block_size : (long long)p.Smax;
}

// The kept prefix of virtual row vb (negative: a bad row).
__device__ __forceinline__ int kept_prefix(const DecodeParams &p, int vb)
{
    return p.kept_prefix_rows ? __ldg(p.kept_prefix_rows + real_row(p, vb)) : p.kept_prefix;
}

// Geometry of batch row b's tiles (the same for every cache head). Slot j is
// attended when j <= L and (j >= lo or j < P). The real tiles are the tiles at
// positions 0 .. tp-1 (those holding prefix slots below lo) and then
// tp + gap .. L / T (those holding window slots); without a window lo = 0,
// gap = 0 and all ceil((L + 1) / T) tiles are real. Rows with bad content get
// one tile, which only writes NaN.
// L of a multi-token row whose token offsets are bad (GQA_STATUS_BAD_QLEN).
constexpr int kBadQLenSlot = INT_MIN;

struct RowGeom {
    int L;    // last attended slot (< 0: a bad row; kBadQLenSlot: bad token offsets)
    int lo;   // first slot of the window (0 without one)
    int P;    // kept prefix
    int nr;   // real tiles (0: an empty chunk of a multi-token step)
    int tp;   // tiles holding prefix slots below lo
    int gap;  // tiles skipped between them and the window's first tile
    int nq;   // tokens (query rows / Gh) of the unit: 1 for a single-token form
    int tokL; // packed index of the token at slot L (single-token forms: b)
    int Lb;   // first slot holding a new token (single-token decode: L)
};

__device__ __forceinline__ bool geom_ok(const DecodeParams &p, int L, int P)
{
    return L >= 0 && (long long)L < row_capacity(p) && P >= 0;
}

// Two forms of one body: the schedule (once per kernel, on the critical path
// to the first copy) inlines it; the streaming loops' row changes call the
// out-of-line form, since inlining its window arithmetic there measurably
// slowed the loops (instruction fetch), while a call from the schedule costs
// a cold instruction fetch before the first byte moves.
__device__ __forceinline__ RowGeom row_geom_inl(const DecodeParams &p, int b)
{
    RowGeom r;
    r.P = kept_prefix(p, b);
    r.lo = 0;
    r.tp = 0;
    r.gap = 0;
#if GQA_MULTI_TOKEN
    if (p.cu_q) {
        const ChunkInfo ci = chunk_info(p, b);
        if (ci.nq == 0) {            // an empty chunk: no tiles at all
            r.L = r.Lb = r.tokL = r.nq = r.nr = 0;
            return r;
        }
        r.nq = max(ci.nq, 0);        // bad token offsets: one tile, no output rows
        r.L = ci.nq < 0 ? kBadQLenSlot : (ci.Lb < 0 ? -1 : ci.Lb + ci.i0 + ci.nq - 1);
        r.tokL = ci.tok0 + ci.i0 + ci.nq - 1;
        r.Lb = ci.Lb;
    } else
#endif
    {
        r.L = last_slot(p, b);
        r.nq = 1;
        r.tokL = b;
        r.Lb = r.L;
    }
    if (!geom_ok(p, r.L, r.P)) {
        r.nr = 1;
        return r;
    }
    const int T = p.tile;
    const int last_tile = r.L / T;
    if (p.window > 0) {
        // the window of the unit's first token (the lowest of its rows)
        r.lo = (int)max(0LL, (long long)r.L - (r.nq - 1) - p.window + 1);
        const int pe = min(r.P, r.lo);                 // prefix slots below the window
        r.tp = (pe + T - 1) / T;
        r.gap = max(0, r.lo / T - r.tp);
    }
    r.nr = last_tile + 1 - r.gap;
    return r;
}

static __device__ __noinline__ RowGeom row_geom(const DecodeParams &p, int b) { return row_geom_inl(p, b); }

// Whether slot j of a row with this geometry takes part in the softmax.
__device__ __forceinline__ bool attended(int L, int lo, int P, int j)
{
    return j <= L && (j >= lo || j < P);
}

// Tiles of one unit in the schedule: its real tiles plus W virtual ones that
// nobody loads or computes. Finishing a unit segment costs a CTA about as much
// time as streaming a few tiles; counting W extra tiles per unit gives the
// CTAs whose ranges cross more unit boundaries correspondingly fewer real
// tiles, so all CTAs finish together.
__device__ __forceinline__ int row_tiles(const DecodeParams &p, int b)
{
    const int nr = row_geom_inl(p, b).nr;   // schedule only
#if GQA_MULTI_TOKEN
    return nr ? nr + p.pad_tiles : 0;
#else
    return nr + p.pad_tiles;
#endif
}

// CTAs that share the N tiles: min(grid size, N).
__device__ __forceinline__ long long working_ctas(long long N, int grid)
{
    return N < grid ? N : (long long)grid;
}

// floor(a / c) for 0 <= a, 0 < c: a 32-bit division when both fit (the
// usual case; a 64-bit one is a long software sequence on the start and end
// paths of the kernels).
__device__ __forceinline__ long long div_floor(long long a, long long c)
{
    if (((unsigned long long)a | (unsigned long long)c) < (1ull << 32))
        return (long long)((unsigned)a / (unsigned)c);
    return a / c;
}

// CTA that owns global tile x: the largest i with floor(i N / C) <= x.
__device__ __forceinline__ int cta_of_tile(long long x, long long N, long long C)
{
    return (int)div_floor((x + 1) * C - 1, N);
}

__device__ __forceinline__ void report(const DecodeParams &p, int bits)
{
    if (p.status)
        atomicOr(p.status, bits);
}

// Position of a CTA in the tile list.
// (Kept small: it lives in registers through the whole streaming loop. The
// schedule's constants N and C live in the shared TileWalk.)
struct TileCursor {
    long long g;      // global tile index
    long long end;    // one past the last tile of the current range
    int b, kvh, t;    // current row, head, tile within the unit
    int nr;           // real tiles of the unit (t < nr holds data; the next
                      // pad_tiles schedule positions are virtual)
    int L;            // last attended slot of row b (last_slot)
    int lo, P;        // window start and kept prefix of row b (see RowGeom)
    int tp, gap;      // real tile t sits at tile position t (t < tp) or t + gap
    int nq, tokL, Lb; // multi-token unit: tokens, token at slot L, first new slot
};

__device__ __forceinline__ void set_row(const DecodeParams &p, TileCursor &c)
{
    const RowGeom r = row_geom(p, c.b);
    c.L = r.L;
    c.lo = r.lo;
    c.P = r.P;
    c.nr = r.nr;
    c.tp = r.tp;
    c.gap = r.gap;
#if GQA_MULTI_TOKEN
    c.nq = r.nq;
    c.tokL = r.tokL;
    c.Lb = r.Lb;
#endif
}

// First slot of the cursor's (real) tile.
__device__ __forceinline__ int tile_slot0(const TileCursor &c, int T)
{
    return (c.t < c.tp ? c.t : c.t + c.gap) * T;
}

// Cursor at global tile g, which lies in row b whose tiles start at `run`.
__device__ __forceinline__ TileCursor cursor_at(const DecodeParams &p, int b, long long run, long long g,
                                               long long end)
{
    TileCursor c;
    c.g = g;
    c.end = end;
    c.b = b;
    const RowGeom r = row_geom_inl(p, b);   // schedule only: inlined (see row_geom)
    c.L = r.L;
    c.lo = r.lo;
    c.P = r.P;
    c.nr = r.nr;
    c.tp = r.tp;
    c.gap = r.gap;
    c.nq = r.nq;
    c.tokL = r.tokL;
    c.Lb = r.Lb;
    const int nt = c.nr + p.pad_tiles;   // cursor_at is only used on rows with tiles
    const long long within = g - run;
    c.kvh = (int)div_floor(within, nt);
    c.t = (int)(within - (long long)c.kvh * nt);
    return c;
}

// The order in which a CTA walks its tile range [begin, end): first the
// segment that holds its last tile -- the head of a unit that usually
// continues in the next CTA -- as range `a` = [split, end), then the rest as
// range `b` = [begin, split). The units cut by CTA boundaries thus have all
// their partial states written early in the kernel (the next CTA starts with
// the same unit's tail), and the end of the kernel finishes whole units only.
// Held in shared memory (one copy per CTA).
struct TileWalk {
    TileCursor a, b;
    long long N, C;   // tiles in the list, CTAs sharing them
};

// L2 prefetch of the cached K and V rows of the first n tiles from cursor c
// (dense and slot-id caches of kv_es bytes per element; paged caches and
// kv_es = 0: nothing). Rows are clamped to the attended slots and the row's
// capacity; rows with a bad length or slot id are skipped. A hint only: the
// kernel's own copies read the same bytes.
__device__ __forceinline__ void prefetch_tiles(const DecodeParams &p, const TileCursor &c, int n, int kv_es)
{
    if (p.paged || kv_es == 0 || c.L < 0)
        return;
    int row = real_row(p, c.b);
    if (p.slot_ids) {
        row = __ldg(p.slot_ids + row);
        if (row < 0 || row >= p.R)
            return;
    }
    const int s0 = tile_slot0(c, p.tile);
    const int s1 = min(min(p.Smax, c.L + 1), s0 + n * p.tile);
    if (s1 <= s0)
        return;
    const size_t rowbytes = (size_t)p.D * kv_es;
    const size_t off = (((size_t)row * p.Hkv + c.kvh) * p.Smax + s0) * rowbytes;
    const size_t bytes = (size_t)(s1 - s0) * rowbytes;
    if ((bytes & 15) || (off & 15) || bytes >= (1u << 31))
        return;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char *>(p.k_cache) + off),
                 "r"((unsigned)bytes)
                 : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char *>(p.v_cache) + off),
                 "r"((unsigned)bytes)
                 : "memory");
}

// Every thread of the block must call it (it uses __syncthreads and
// `scratch`, >= blockDim.x / 32 + 8 long longs of shared memory; blockDim.x a
// multiple of 32). kv_es > 0: the threads that find the CTA's first tiles
// also prefetch them into L2 (prefetch_tiles), so HBM starts working before
// the walk is assembled and the first copies are issued. The row prefix is a block-wide scan of the per-row tile
// counts, recomputed by every CTA from `lengths` (no host round trip). The
// threads whose rows hold the CTA's first and last tiles build those two
// cursors (in `out`), and thread 0 then orders them into the walk: the start
// of the kernel is a chain of dependent steps, kept short. The walk is
// visible to all threads on return.
__device__ inline void schedule_walk(const DecodeParams &p, long long *scratch, TileWalk *out, int kv_es = 0)
{
    const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = nthr >> 5;
    const int chunk = (p.B + nthr - 1) / nthr;
    const int r0 = min(p.B, tid * chunk), r1 = min(p.B, r0 + chunk);
    long long local = 0, n0 = 0;        // tiles of this thread's rows, of its first row
    for (int b = r0; b < r1; ++b) {
        const long long n = (long long)p.Hkv * row_tiles(p, b);
        n0 = (b == r0) ? n : n0;
        local += n;
    }
    // inclusive scan: within the warp by shuffles, then over the warp totals
    long long incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off)
            incl += v;
    }
    long long *wsum = scratch;              // [nwarps]
    if (lane == 31)
        wsum[warp] = incl;
    __syncthreads();
    long long before = 0, N = 0;
    for (int w = 0; w < nwarps; ++w) {
        const long long v = wsum[w];
        before += (w < warp) ? v : 0;
        N += v;
    }
    incl += before;
    const long long excl = incl - local;
    const long long C = working_ctas(N, p.grid);
    const long long begin = blockIdx.x < C ? div_floor((long long)blockIdx.x * N, C) : N;
    const long long end = blockIdx.x < C ? div_floor(((long long)blockIdx.x + 1) * N, C) : N;
    const long long last = end - 1;
    if (begin < end && ((begin >= excl && begin < incl) || (last >= excl && last < incl))) {
        // this thread's rows hold the first tile (cursor -> out->b) and/or the
        // last one (-> out->a); each range's first 32 KB or so of K and V go
        // to L2 ahead of the copies (measured: deeper prefetches were slower)
        const int pf_tiles = kv_es == 1 ? 2 : 1;   // E4M3 tiles are half the bytes
        long long run = excl;
        for (int b = r0; b < r1; ++b) {
            const long long n = (b == r0) ? n0 : (long long)p.Hkv * row_tiles(p, b);
            if (begin >= run && begin < run + n) {
                const TileCursor c = cursor_at(p, b, run, begin, end);
                out->b = c;
                prefetch_tiles(p, c, pf_tiles, kv_es);
            }
            if (last >= run && last < run + n) {
                TileCursor c = cursor_at(p, b, run, last, end);
                out->a = c;
                if (last - c.t > begin) {   // range a, walked first, starts at the unit's tile 0
                    c.t = 0;
                    prefetch_tiles(p, c, pf_tiles, kv_es);
                }
            }
            run += n;
        }
    }
    __syncthreads();
    if (tid == 0) {
        TileWalk &w = *out;
        w.N = N;
        w.C = C;
        if (begin >= end) {
            TileCursor none;
            none.g = none.end = N;
            none.b = none.kvh = none.t = none.L = 0;
            none.lo = none.P = none.tp = none.gap = 0;
            none.nq = none.tokL = none.Lb = 0;
            none.nr = 1;
            w.a = w.b = none;
        } else {
            const TileCursor first = w.b;
            const TileCursor tail = w.a;
            const long long unit_start = last - tail.t;
            if (unit_start <= begin) {        // a single segment: walk it in order
                w.a = first;
                w.b = first;
                w.b.g = w.b.end = end;
            } else {
                w.a = tail;
                w.a.g = unit_start;
                w.a.t = 0;
                w.b = first;
                w.b.end = unit_start;
            }
        }
    }
    __syncthreads();
}

// The cursor's next row with tiles (empty chunks of a multi-token step hold
// none). Out of line: it runs once per row, and keeping its code out of the
// streaming loops keeps them short.
#if GQA_MULTI_TOKEN
static __device__ __noinline__ void next_row(const DecodeParams &p, TileCursor &c)
{
    do {
        ++c.b;
        set_row(p, c);
    } while (c.nr == 0);
}
#endif

__device__ __forceinline__ void advance(const DecodeParams &p, TileCursor &c)
{
    ++c.g;
    if (++c.t == c.nr + p.pad_tiles) {
        c.t = 0;
        if (++c.kvh == p.Hkv) {
            c.kvh = 0;
#if GQA_MULTI_TOKEN
            if (c.g < c.end)
                next_row(p, c);
            else
                ++c.b;
#else
            ++c.b;
            if (c.g < c.end)
                set_row(p, c);
#endif
        }
    }
}

// Moves past virtual tiles within the current part of the walk.
__device__ __forceinline__ void skip_virtual(const DecodeParams &p, TileCursor &c)
{
    while (c.g < c.end && c.t >= c.nr)
        advance(p, c);
}

// Next real tile of the walk: along the current range, then from range a into
// range b. False when the CTA has no tile left.
__device__ __forceinline__ bool walk_next(const DecodeParams &p, TileCursor &c, const TileWalk &w, bool &in_b)
{
    advance(p, c);
    skip_virtual(p, c);
    if (c.g < c.end)
        return true;
    if (!in_b && w.b.g < w.b.end) {
        c = w.b;
        in_b = true;
        skip_virtual(p, c);
        return c.g < c.end;
    }
    return false;
}

// First real tile of the walk; false when the CTA has none.
__device__ __forceinline__ bool walk_first(const DecodeParams &p, TileCursor &c, const TileWalk &w, bool &in_b)
{
    c = w.a;
    in_b = false;
    skip_virtual(p, c);
    if (c.g < c.end)
        return true;
    if (w.b.g < w.b.end) {
        c = w.b;
        in_b = true;
        skip_virtual(p, c);
        return c.g < c.end;
    }
    return false;
}

// Row-level content check: length in range, slot id in range.
// Content error bits of virtual row b whose last attended slot is L (0: a
// good row).
__device__ __forceinline__ int row_error_bits(const DecodeParams &p, int b, int L)
{
#if GQA_MULTI_TOKEN
    if (L == kBadQLenSlot)
        return kBadQLen;
#endif
    if (L < 0 || (long long)L >= row_capacity(p))
        return kBadLength;
    if (kept_prefix(p, b) < 0)
        return kBadPrefix;
    if (!p.paged && p.slot_ids) {
        int r = __ldg(p.slot_ids + real_row(p, b));
        if (r < 0 || r >= p.R)
            return kBadSlotId;
    }
    return 0;
}

__device__ __forceinline__ bool row_ok(const DecodeParams &p, int b, int L)
{
    return row_error_bits(p, b, L) == 0;
}

// Element offset of slot s of (b, kvh) in the dense cache, or -1 when the
// paged table entry that holds it is unusable.
__device__ __forceinline__ long long slot_offset(const DecodeParams &p, int vb, int kvh, int s)
{
    const int b = real_row(p, vb);
    if (!p.paged) {
        long long r = p.slot_ids ? __ldg(p.slot_ids + b) : b;
        return ((r * p.Hkv + kvh) * p.Smax + s) * (long long)p.D;
    }
    int blk = __ldg(p.block_table + (long long)b * p.max_blocks + s / p.block_size);
    if (blk < 0 || blk >= p.num_blocks)
        return -1;
    return (((long long)blk * p.Hkv + kvh) * p.block_size + s % p.block_size) * (long long)p.D;
}

__device__ __forceinline__ float fast_ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared-memory scratch of a segment's epilogue and of the in-kernel merge of
// a cut unit's partials.
constexpr int kMergeMax = 32;   // partials weighted in one pass through shared memory (more: in chunks)
constexpr int kMergeG = 8;      // query rows per unit (G <= 8)
constexpr int kMergeW = 4;      // warps whose states a segment merges
// For GR query rows per unit, up to KM partials merged through shared memory.
template <int GR, int KM>
struct MergeBufT {
    float a[kMergeW][GR];      // weight 2^(m_w - M) of each warp's state
    float M[GR], den[GR];
    float w[KM * GR];          // partial max, then its weight 2^(m_i - M)
    float l[KM * GR];
    float inv_den[GR];
};
using MergeBuf = MergeBufT<kMergeG, kMergeMax>;

// End of a unit segment. The NW per-warp states of the segment are in shared
// memory: sm_m[w][g] (base-2 running max, -inf for a warp that saw no slot),
// sm_l[w][g], sm_o[w][g][d] (rows padded to DP >= DD floats). All `nthr`
// calling threads take part; `sync` synchronises exactly them. The weights
// of the warp states are formed once per head, then the outputs are merged
// four at a time. A whole unit writes its normalised output. A cut unit
// writes its partial state, then takes an arrival ticket; the last CTA of the
// unit to arrive merges every partial (log-sum-exp rule), writes the output,
// zeroes the partials it merged and resets the unit's counter. A sink logit,
// when given, joins the final normalisation only (whole units here, cut units
// in the merge): it raises the maximum if larger and adds 2^(sink - M) to the
// denominator.
// Sink logit of query head h in base-2 units (the scores' units).
__device__ __forceinline__ float sink_log2(const DecodeParams &p, int h)
{
    return __ldg(p.sink + h) * 1.4426950408889634f;
}

// Output row of query row g of the cursor's unit: token tokL - (nq - 1 -
// g / Gh), head kvh * Gh + g % Gh; single-token forms (MULTI false): row b,
// head kvh * G + g, without touching the cursor's chunk fields (which then
// take no registers in the streaming loop).
template <bool MULTI>
__device__ __forceinline__ float *out_row(const DecodeParams &p, const TileCursor &c, int g, int DD)
{
    if constexpr (MULTI) {
        const long long tok = c.tokL - (c.nq - 1 - g / p.Gh);
        return p.out + (tok * p.Hq + (long long)c.kvh * p.Gh + g % p.Gh) * DD;
    } else {
        return p.out + ((long long)c.b * p.Hq + (long long)c.kvh * p.G + g) * DD;
    }
}

// First part of the end of a unit segment: the weights of the warp states,
// then the normalised output (the segment is the whole unit) or this CTA's
// partial state (a cut unit). Returns whether the unit was whole. Every
// calling thread takes part; ends with a sync().
template <int NW, int GP, int DD, int DP, bool MULTI, class Sync, int GR, int KM>
__device__ inline bool segment_out(const DecodeParams &p, const TileCursor &cur, int seg_first_t, bool bad,
                                   const float (&sm_m)[NW][GP], const float (&sm_l)[NW][GP],
                                   const float (&sm_o)[NW][GP][DP], MergeBufT<GR, KM> &mb, int tid, int nthr,
                                   Sync sync)
{
    static_assert(NW <= kMergeW && GP <= GR && DP >= DD, "merge buffer too small");
    const int G = p.G, b = cur.b, kvh = cur.kvh;
    const bool unit_done = (cur.t == cur.nr - 1);
    const bool whole = (seg_first_t == 0) && unit_done;
    const int u = b * p.Hkv + kvh;
    const long long P = (long long)u + blockIdx.x;
    const float qnan = __int_as_float(0x7fc00000);
    const int nrow = MULTI ? p.Gh * cur.nq : G;   // query rows with an output
    if (tid < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            M = fmaxf(M, sm_m[w][tid]);
        const float sk = (whole && p.sink) ? sink_log2(p, kvh * p.Gh + tid % p.Gh) : -INFINITY;
        M = fmaxf(M, sk);
        float den = (sk == -INFINITY) ? 0.f : fast_ex2(sk - M);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float a = (sm_m[w][tid] == -INFINITY) ? 0.f : fast_ex2(sm_m[w][tid] - M);
            mb.a[w][tid] = a;
            den = fmaf(a, sm_l[w][tid], den);
        }
        mb.M[tid] = M;
        mb.den[tid] = den;
        if (!whole) {
            p.ws_ml[(P * G + tid) * 2 + 0] = bad ? qnan : M;
            p.ws_ml[(P * G + tid) * 2 + 1] = bad ? qnan : den;
        }
    }
    sync();
    {
        constexpr int V = (DD % 4 == 0) ? 4 : 1;
        for (int idx = tid * V; idx < G * DD; idx += nthr * V) {
            const int g = idx / DD, d = idx % DD;
            float acc[V];
#pragma unroll
            for (int e = 0; e < V; ++e)
                acc[e] = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float a = mb.a[w][g];
                if constexpr (V == 4) {
                    const float4 o = *reinterpret_cast<const float4 *>(&sm_o[w][g][d]);
                    acc[0] = fmaf(a, o.x, acc[0]);
                    acc[1] = fmaf(a, o.y, acc[1]);
                    acc[2] = fmaf(a, o.z, acc[2]);
                    acc[3] = fmaf(a, o.w, acc[3]);
                } else {
                    acc[0] = fmaf(a, sm_o[w][g][d], acc[0]);
                }
            }
            if (whole) {
                const float inv = 1.f / mb.den[g];
#pragma unroll
                for (int e = 0; e < V; ++e)
                    acc[e] = bad ? qnan : acc[e] * inv;
                if (g < nrow) {
                    float *o = out_row<MULTI>(p, cur, g, DD) + d;
                    if constexpr (V == 4)
                        *reinterpret_cast<float4 *>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    else
                        *o = acc[0];
                }
            } else {
                float *po = p.ws_o + (P * G + g) * DD + d;
#pragma unroll
                for (int e = 0; e < V; ++e)
                    acc[e] = bad ? qnan : acc[e];
                if constexpr (V == 4)
                    *reinterpret_cast<float4 *>(po) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                else
                    *po = acc[0];
            }
        }
    }
    sync();
    return whole;
}

// Second part for a cut unit: the arrival ticket and, in the last CTA of the
// unit to arrive, the merge of every partial (log-sum-exp rule), the output,
// and the partials and counter back to zero. `cur` names the unit (b, kvh,
// and nq / tokL of a multi-token chunk); first..last are the CTAs whose
// ranges hold its tiles. The threads calling it must be ordered after the
// partial stores of this CTA (a barrier): thread 0's acquire-release ticket
// at GPU scope then publishes them (release is cumulative), and the last
// arriver's acquire plus the barrier order its reads after the stores of
// every other CTA of the unit.
template <int DD, bool MULTI, bool PRE2, class Sync, int GR, int KM>
__device__ inline void unit_ticket_merge(const DecodeParams &p, const TileCursor &cur, int first, int last,
                                         int *sm_flag, MergeBufT<GR, KM> &mb, int tid, int nthr, Sync sync,
                                         int pre_cnt)
{
    const int G = p.G, kvh = cur.kvh;
    const int u = cur.b * p.Hkv + kvh;
    const int nrow = MULTI ? p.Gh * cur.nq : G;   // query rows with an output
    if (tid == 0) {
        int old = pre_cnt;
        if (old != last - first)
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.ws_cnt + u) : "memory");
        *sm_flag = (old == last - first);
    }
    sync();
    if (*sm_flag) {
        const int K = last - first + 1;
        const long long P0 = (long long)u + first;
        if (K <= KM) {
            // one parallel load of every partial's (m, l), weights per head,
            // then independent (vector) loads of the partial outputs. PRE2: a
            // unit cut once (K = 2, the usual case) has this thread's first
            // two partial outputs loaded together with the (m, l) pairs, one
            // round trip to L2 instead of two on the kernel's last step (it
            // costs registers: kernels at their register cap leave it off).
            constexpr int V = (DD % 4 == 0) ? 4 : 1;
            const bool pre2 = PRE2 && (V == 4) && K == 2 && tid * V < G * DD;
            float4 pv0 = make_float4(0.f, 0.f, 0.f, 0.f), pv1 = pv0;
            if (pre2) {
                pv0 = __ldcg(reinterpret_cast<const float4 *>(p.ws_o + P0 * G * DD + tid * V));
                pv1 = __ldcg(reinterpret_cast<const float4 *>(p.ws_o + (P0 + 1) * G * DD + tid * V));
            }
            for (int k = tid; k < K * G; k += nthr) {
                mb.w[k] = __ldcg(p.ws_ml + (P0 * G + k) * 2);
                mb.l[k] = __ldcg(p.ws_ml + (P0 * G + k) * 2 + 1);
            }
            sync();
            if (tid < G) {
                float M = -INFINITY;
                for (int i = 0; i < K; ++i)
                    M = fmaxf(M, mb.w[i * G + tid]);
                const float sk = p.sink ? sink_log2(p, kvh * p.Gh + tid % p.Gh) : -INFINITY;
                M = fmaxf(M, sk);
                float den = (sk == -INFINITY) ? 0.f : fast_ex2(sk - M);
                for (int i = 0; i < K; ++i) {
                    const float a = fast_ex2(mb.w[i * G + tid] - M);
                    mb.w[i * G + tid] = a;
                    den = fmaf(a, mb.l[i * G + tid], den);
                }
                mb.inv_den[tid] = 1.f / den;
            }
            sync();
            for (int idx = tid * V; idx < G * DD; idx += nthr * V) {
                const int g = idx / DD;
                float acc[V];
#pragma unroll
                for (int e = 0; e < V; ++e)
                    acc[e] = 0.f;
                if constexpr (PRE2 && V == 4) {
                    if (pre2 && idx == tid * V) {   // the preloaded pair
                        const float a0 = mb.w[g], a1 = mb.w[G + g];
                        acc[0] = fmaf(a1, pv1.x, a0 * pv0.x);
                        acc[1] = fmaf(a1, pv1.y, a0 * pv0.y);
                        acc[2] = fmaf(a1, pv1.z, a0 * pv0.z);
                        acc[3] = fmaf(a1, pv1.w, a0 * pv0.w);
                        *reinterpret_cast<float4 *>(p.ws_o + P0 * G * DD + idx) = make_float4(0.f, 0.f, 0.f, 0.f);
                        *reinterpret_cast<float4 *>(p.ws_o + (P0 + 1) * G * DD + idx) =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                        if (g < nrow) {
                            float *o = out_row<MULTI>(p, cur, g, DD) + (idx - g * DD);
#pragma unroll
                            for (int e = 0; e < V; ++e)
                                o[e] = acc[e] * mb.inv_den[g];
                        }
                        continue;
                    }
                }
#pragma unroll 4
                for (int i = 0; i < K; ++i) {
                    const float a = mb.w[i * G + g];
                    float *po = p.ws_o + (P0 + i) * G * DD + idx;
                    if constexpr (V == 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(po));
                        acc[0] = fmaf(a, v.x, acc[0]);
                        acc[1] = fmaf(a, v.y, acc[1]);
                        acc[2] = fmaf(a, v.z, acc[2]);
                        acc[3] = fmaf(a, v.w, acc[3]);
                        *reinterpret_cast<float4 *>(po) = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else {
                        acc[0] = fmaf(a, __ldcg(po), acc[0]);
                        *po = 0.f;     // consumed: leave the workspace zero-filled
                    }
                }
                if (g < nrow) {
                    float *o = out_row<MULTI>(p, cur, g, DD) + (idx - g * DD);
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        o[e] = acc[e] * mb.inv_den[g];
                }
            }
        } else if constexpr (MULTI && PRE2) {
            // more partials than the buffer holds (multi-token units over a
            // bfloat16 cache: up to 32 rows): the maximum and the denominator
            // of each row first (every partial's (m, l) loaded directly), then
            // the outputs KM partials at a time, their weights through shared
            // memory and the sums in the output rows. long_context, 4 tokens a
            // row (each unit cut about 10 times): 246 us against 564 with the
            // element form below
            constexpr int V = (DD % 4 == 0) ? 4 : 1;
            for (int g = tid; g < G; g += nthr) {
                float M = -INFINITY;
                for (int i = 0; i < K; ++i)
                    M = fmaxf(M, __ldcg(p.ws_ml + ((P0 + i) * G + g) * 2));
                const float sk = p.sink ? sink_log2(p, kvh * p.Gh + g % p.Gh) : -INFINITY;
                M = fmaxf(M, sk);
                float den = (sk == -INFINITY) ? 0.f : fast_ex2(sk - M);
                for (int i = 0; i < K; ++i) {
                    const float *ml = p.ws_ml + ((P0 + i) * G + g) * 2;
                    den = fmaf(fast_ex2(__ldcg(ml) - M), __ldcg(ml + 1), den);
                }
                mb.M[g] = M;
                mb.inv_den[g] = 1.f / den;
            }
            for (int c0 = 0; c0 < K; c0 += KM) {
                const int kc = min(KM, K - c0);
                sync();   // the rows' maxima (first chunk); the previous chunk's weights read
                for (int k = tid; k < kc * G; k += nthr)   // partial c0 + k / G, row k % G
                    mb.w[k] = fast_ex2(__ldcg(p.ws_ml + ((P0 + c0) * G + k) * 2) - mb.M[k % G]);
                sync();
                for (int idx = tid * V; idx < G * DD; idx += nthr * V) {
                    const int g = idx / DD;
                    float acc[V];
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        acc[e] = 0.f;
#pragma unroll 4
                    for (int i = 0; i < kc; ++i) {
                        const float a = mb.w[i * G + g];
                        float *po = p.ws_o + (P0 + c0 + i) * G * DD + idx;
                        if constexpr (V == 4) {
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(po));
                            acc[0] = fmaf(a, v.x, acc[0]);
                            acc[1] = fmaf(a, v.y, acc[1]);
                            acc[2] = fmaf(a, v.z, acc[2]);
                            acc[3] = fmaf(a, v.w, acc[3]);
                            *reinterpret_cast<float4 *>(po) = make_float4(0.f, 0.f, 0.f, 0.f);
                        } else {
                            acc[0] = fmaf(a, __ldcg(po), acc[0]);
                            *po = 0.f;   // consumed: leave the workspace zero-filled
                        }
                    }
                    if (g < nrow) {
                        // this thread's own elements: the earlier chunks' sums
                        float *o = out_row<MULTI>(p, cur, g, DD) + (idx - g * DD);
#pragma unroll
                        for (int e = 0; e < V; ++e)
                            o[e] = fmaf(acc[e], mb.inv_den[g], c0 == 0 ? 0.f : o[e]);
                    }
                }
            }
        } else {
            // element by element, every partial's (m, l) read again per
            // element: few registers. Single-token units (at most 8 rows, and
            // only past 32 pieces), and the E4M3 kernels at their register cap
            // (their four-warp merge in this form: long_context 4 tokens a row
            // 300 us against 238 chunked, but the chunked form's spills cost
            // their common steps 3-5 %)
            for (int idx = tid; idx < G * DD; idx += nthr) {
                const int g = idx / DD, d = idx % DD;
                float M = -INFINITY;
                for (int i = 0; i < K; ++i)
                    M = fmaxf(M, __ldcg(p.ws_ml + ((P0 + i) * G + g) * 2));
                const float sk = p.sink ? sink_log2(p, kvh * p.Gh + g % p.Gh) : -INFINITY;
                M = fmaxf(M, sk);
                float num = 0.f, den = (sk == -INFINITY) ? 0.f : fast_ex2(sk - M);
                for (int i = 0; i < K; ++i) {
                    const long long Q = P0 + i;
                    const float a = fast_ex2(__ldcg(p.ws_ml + (Q * G + g) * 2) - M);
                    float *po = p.ws_o + (Q * G + g) * DD + d;
                    num = fmaf(a, __ldcg(po), num);
                    den = fmaf(a, __ldcg(p.ws_ml + (Q * G + g) * 2 + 1), den);
                    *po = 0.f;       // consumed: leave the workspace zero-filled
                }
                if (g < nrow)
                    out_row<MULTI>(p, cur, g, DD)[d] = num / den;
            }
        }
        sync();
        // the (m, l) pairs of partials u+first .. u+last are contiguous
        float *ml = p.ws_ml + P0 * G * 2;
        for (int k = tid; k < K * G * 2; k += nthr)
            ml[k] = 0.f;
        if (tid == 0)
            p.ws_cnt[u] = 0;
    }
    sync();
}

// MULTI: the unit may be a chunk of a multi-token step (any form then works).
// pre_cnt (thread 0 only): the unit's arrival count read with acquire
// semantics shortly before the segment's end, or -1. When it already shows
// every other piece of the unit arrived, this CTA is the last arriver: it
// skips the ticket's round trip and merges at once.
template <int NW, int GP, int DD, int DP, bool MULTI, bool PRE2 = false, class Sync, int GR, int KM>
__device__ inline void finish_segment(const DecodeParams &p, const TileCursor &cur, const TileWalk &walk,
                                      int seg_first_t,
                                      bool bad, const float (&sm_m)[NW][GP], const float (&sm_l)[NW][GP],
                                      const float (&sm_o)[NW][GP][DP], int *sm_flag, MergeBufT<GR, KM> &mb,
                                      int tid, int nthr, Sync sync, int pre_cnt = -1)
{
    if (segment_out<NW, GP, DD, DP, MULTI>(p, cur, seg_first_t, bad, sm_m, sm_l, sm_o, mb, tid, nthr, sync))
        return;
    const long long first_tile = cur.g - cur.t;
    const int first = cta_of_tile(first_tile, walk.N, walk.C);
    const int last = cta_of_tile(first_tile + cur.nr - 1, walk.N, walk.C);
    unit_ticket_merge<DD, MULTI, PRE2>(p, cur, first, last, sm_flag, mb, tid, nthr, sync, pre_cnt);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

}  // namespace gqa
