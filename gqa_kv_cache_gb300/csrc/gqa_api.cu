// The C ABI (include/gqa_decode.h): host-side argument checks, kernel
// choice, workspace sizing, TMA descriptor encoding, launches and tracing.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "gqa_decode.h"
#include "gqa_launch.h"

using namespace gqa;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultSchedPad = 3;
constexpr long long kDefaultWaitCycles = 4LL << 30;   // about 2 s at 2 GHz

int sm_count(int dev)
{
    static std::atomic<int> cache[kMaxDevices];   // zero-initialised (static storage)
    if (dev < 0 || dev >= kMaxDevices)
        return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Whether the small-cache kernel takes the step: single-token, a float32 or
// bfloat16 cache, and a row capacity whose K and V fit in shared memory
// (cap_rows < 0: capacity unknown, no).
bool unit_ok(gqa_dtype dt, int D, int G, long long cap_rows, bool multi)
{
    return !multi && cap_rows > 0 && (dt == GQA_DTYPE_F32 || dt == GQA_DTYPE_BF16) &&
           unit_supports(dt == GQA_DTYPE_BF16, D, G, cap_rows);
}

// Kernel the call will use (GQA_KERNEL_SIMT / _TC / _UNIT) or -1. AUTO takes
// the small-cache kernel when it applies and the units (B * Hkv, known > 0)
// fit in one wave of it; else the tensor-core kernel where it applies, else
// the CUDA-core one.
int pick_kernel(const gqa_options *opt, gqa_dtype dt, int D, int G, bool paged, int block_size,
                long long cap_rows = -1, bool multi = false, long long units = 0)
{
    // GQA_KERNEL_TC5 is the tensor-core kernel with one of its unit forms on
    // tcgen05 (chosen at the launch)
    const int want = opt ? (opt->kernel == GQA_KERNEL_TC5 ? GQA_KERNEL_TC : opt->kernel) : GQA_KERNEL_AUTO;
    const bool bf16 = dt == GQA_DTYPE_BF16 || dt == GQA_DTYPE_E4M3;   // the tensor-core kernel's caches
    const bool tc_ok = tc_supports(bf16, D, G, paged, block_size);
    const bool simt_ok = dt != GQA_DTYPE_E4M3 && simt_supports(D, G);
    const bool small_ok = unit_ok(dt, D, G, cap_rows, multi);
    if (want == GQA_KERNEL_TC)
        return tc_ok ? GQA_KERNEL_TC : -1;
    if (want == GQA_KERNEL_SIMT)
        return simt_ok ? GQA_KERNEL_SIMT : -1;
    if (want == GQA_KERNEL_UNIT)
        return small_ok ? GQA_KERNEL_UNIT : -1;
    if (want != GQA_KERNEL_AUTO)
        return -1;
    if (small_ok && units > 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) {
            const long long wave =
                (long long)sm_count(dev) * unit_ctas_per_sm(dt == GQA_DTYPE_BF16, D, G, cap_rows);
            if (units <= wave)
                return GQA_KERNEL_UNIT;
        }
    }
    if (tc_ok)
        return GQA_KERNEL_TC;
    return simt_ok ? GQA_KERNEL_SIMT : -1;
}

// Persistent grid: every SM holds as many CTAs as fit at once (cached per
// device and kernel instantiation).
int grid_for(int kernel, const gqa_options *opt, gqa_dtype dt, int D, int G)
{
    if (opt && opt->grid_ctas > 0)
        return opt->grid_ctas;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    const int sms = sm_count(dev);
    if (kernel == GQA_KERNEL_TC)
        return sms * tc_ctas_per_sm(dt == GQA_DTYPE_E4M3, G);   // G: query rows of a unit
    static std::mutex mu;
    static int cache[kMaxDevices][2][9][9] = {};
    int dlog = 0;
    while ((1 << dlog) < D && dlog < 8)
        ++dlog;
    const int bf = dt == GQA_DTYPE_BF16 ? 1 : 0;
    std::lock_guard<std::mutex> g(mu);
    int &c = cache[dev < kMaxDevices ? dev : 0][bf][dlog][G < 9 ? G : 8];
    if (!c)
        c = simt_ctas_per_sm(bf, D, G);
    return sms * c;
}

// ------------------------------------------------------------------ trace --

struct TraceRec {
    int kind;
    cudaEvent_t start, stop;
};

struct Trace {
    std::mutex mu;
    bool on = false;
    std::vector<TraceRec> pending;
    std::vector<cudaEvent_t> pool;
    cudaEvent_t get()
    {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
};

Trace &trace()
{
    static Trace t;
    return t;
}

struct TraceScope {
    bool on;
    int kind;
    cudaStream_t st;
    cudaEvent_t a = nullptr, b = nullptr;
    TraceScope(int k, cudaStream_t s) : on(trace().on), kind(k), st(s)
    {
        if (on) {
            std::lock_guard<std::mutex> g(trace().mu);
            a = trace().get();
            b = trace().get();
            cudaEventRecord(a, st);
        }
    }
    ~TraceScope()
    {
        if (on) {
            cudaEventRecord(b, st);
            std::lock_guard<std::mutex> g(trace().mu);
            trace().pending.push_back({kind, a, b});
        }
    }
};

// ------------------------------------------------------- tensor maps (TMA) --

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D map over a bf16 (es = 2) or E4M3 (es = 1) cache seen as (D,
// rows_per_head, heads_total): box (128 bytes of elements, box_rows, 1) with
// the 128-byte swizzle.
bool encode_cache_map(CUtensorMap *m, void *base, int D, long long rows_per_head,
                      long long heads_total, int box_rows, int es = 2)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows_per_head, (cuuint64_t)heads_total};
    cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)D * es * (cuuint64_t)rows_per_head};
    cuuint32_t box[3] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims,
              strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------- the step --

struct Shape {
    int B, Hq, Hkv, D;
    gqa_dtype dt;  // the cache (and k_new / v_new)
    bool paged;
    int R, Smax;
    int num_blocks, block_size, max_blocks;
    bool attend = false;          // read-only attend: no new token, nothing written but out
    gqa_dtype q_dt = GQA_DTYPE_F32;
    bool multi = false;           // multi-token step: T packed tokens, q_len <= max_q
    int T = 0, max_q = 1;
};

// How a multi-token step is cut into virtual rows: tokens per chunk (so that
// chunk rows G * tpc fit the query rows of a unit: 32 for the tensor-core
// kernel, 8 for the CUDA-core one) and chunks per batch row.
struct MultiCut {
    int tpc, chunks;
};

MultiCut multi_cut(int G, int max_q, int rows)
{
    MultiCut c;
    c.tpc = G >= rows ? 1 : rows / G;
    if (c.tpc > max_q)
        c.tpc = max_q > 0 ? max_q : 1;
    c.chunks = (max_q + c.tpc - 1) / c.tpc;
    if (c.chunks < 1)
        c.chunks = 1;
    return c;
}

bool valid_dtype(gqa_dtype d) { return d == GQA_DTYPE_F32 || d == GQA_DTYPE_BF16; }

gqa_status check_shape(const Shape &s)
{
    if (s.B < 0 || s.Hq < 1 || s.Hkv < 1 || s.D < 1 || s.Hq % s.Hkv != 0)
        return GQA_ERR_INVALID_ARGUMENT;
    if ((!valid_dtype(s.dt) && s.dt != GQA_DTYPE_E4M3) || !valid_dtype(s.q_dt))
        return GQA_ERR_INVALID_ARGUMENT;
    if (s.paged) {
        if (s.num_blocks < 1 || s.block_size < 1 || s.max_blocks < 1)
            return GQA_ERR_INVALID_ARGUMENT;
        if ((long long)s.max_blocks * s.block_size > (1LL << 31) - 1)
            return GQA_ERR_INVALID_ARGUMENT;
    } else {
        if (s.R < 0 || s.Smax < 1)
            return GQA_ERR_INVALID_ARGUMENT;
    }
    return GQA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gqa_status run_step(const Shape &s, const void *q, const void *k_new, const void *v_new, void *kc,
                    void *vc, const int32_t *lengths, const int32_t *slot_ids,
                    const int32_t *block_table, float *out, void *ws, size_t ws_bytes,
                    int32_t *d_status, void *stream, const gqa_options *opt,
                    const int32_t *cu_q = nullptr)
{
    gqa_status st = check_shape(s);
    if (st != GQA_OK)
        return st;
    if (s.multi && (s.T < 0 || s.max_q < 0 || !cu_q))
        return GQA_ERR_INVALID_ARGUMENT;
    const bool kv8 = s.dt == GQA_DTYPE_E4M3;
    if (kv8 && (!opt || !opt->k_scale || !opt->v_scale || (reinterpret_cast<uintptr_t>(opt->k_scale) & 3u) ||
                (reinterpret_cast<uintptr_t>(opt->v_scale) & 3u)))
        return GQA_ERR_INVALID_ARGUMENT;
    if (s.B == 0 || (s.multi && (s.T == 0 || s.max_q == 0)))
        return GQA_OK;
    if (!q || !kc || !vc || !lengths || !out || (s.paged && !block_table))
        return GQA_ERR_INVALID_ARGUMENT;
    if (!s.attend && (!k_new || !v_new))
        return GQA_ERR_INVALID_ARGUMENT;
    if (!s.paged && !slot_ids && s.R < s.B)
        return GQA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(out))
        return GQA_ERR_INVALID_ARGUMENT;
    if (opt && (opt->window < 0 || opt->kept_prefix < 0 || opt->wait_limit_cycles < 0 ||
                (reinterpret_cast<uintptr_t>(opt->head_sink) & 3u) ||
                (reinterpret_cast<uintptr_t>(opt->kept_prefix_rows) & 3u)))
        return GQA_ERR_INVALID_ARGUMENT;
    if (!s.attend && (!aligned16(k_new) || !aligned16(v_new)))
        return GQA_ERR_INVALID_ARGUMENT;
    const int Gh = s.Hq / s.Hkv;
    if (s.multi && Gh > 8)
        return GQA_ERR_UNSUPPORTED;
    const long long cap_rows = s.paged ? (long long)s.max_blocks * s.block_size : (long long)s.Smax;
    const int kernel = pick_kernel(opt, s.dt, s.D, Gh, s.paged, s.block_size, cap_rows, s.multi,
                                   (long long)s.B * s.Hkv);
    if (kernel < 0)
        return GQA_ERR_UNSUPPORTED;
    const MultiCut cut = s.multi ? multi_cut(Gh, s.max_q, kernel == GQA_KERNEL_TC ? 32 : 8) : MultiCut{1, 1};
    const int G = Gh * cut.tpc;             // query rows of a unit
    const int Bv = s.B * cut.chunks;        // (virtual) rows of the schedule
    const bool unit = kernel == GQA_KERNEL_UNIT;   // no schedule, no workspace
    const int grid = unit ? s.B * s.Hkv : grid_for(kernel, opt, s.dt, s.D, G);
    if (grid <= 0)
        return GQA_ERR_CUDA;
    const WorkspaceLayout lay = workspace_layout(Bv, s.Hkv, G, s.D, grid);
    if (!unit && (!ws || ws_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return GQA_ERR_WORKSPACE;

    DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.kv8 = kv8 ? 1 : 0;
    if (kv8) {
        p.k_scale = opt->k_scale;
        p.v_scale = opt->v_scale;
    }
    p.attend = s.attend ? 1 : 0;
    p.q_bf16 = s.q_dt == GQA_DTYPE_BF16 ? 1 : 0;
    p.k_new = s.attend ? nullptr : k_new;
    p.v_new = s.attend ? nullptr : v_new;
    p.k_cache = kc;
    p.v_cache = vc;
    p.lengths = lengths;
    p.slot_ids = s.paged ? nullptr : slot_ids;
    p.block_table = s.paged ? block_table : nullptr;
    p.out = out;
    p.B = Bv;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = G;
    p.Gh = Gh;
    p.tpc = cut.tpc;
    p.max_chunks = cut.chunks;
    p.cu_q = s.multi ? cu_q : nullptr;
    p.T = s.T;
    p.max_q = s.max_q;
    p.D = s.D;
    p.R = s.R;
    p.Smax = s.Smax;
    p.paged = s.paged ? 1 : 0;
    p.num_blocks = s.num_blocks;
    p.block_size = s.block_size;
    p.max_blocks = s.max_blocks;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.D));
    if (opt) {
        p.sink = opt->head_sink;
        p.window = opt->window;
        p.kept_prefix = opt->kept_prefix;
        p.kept_prefix_rows = opt->kept_prefix_rows;
    }
    p.tile = kernel == GQA_KERNEL_TC ? tc_tile() : simt_tile();
    // about the time a CTA spends finishing a sequence, in tiles of streaming
    p.pad_tiles = (opt && opt->sched_pad > 0) ? opt->sched_pad - 1 : kDefaultSchedPad;
    p.grid = grid;
    if (!unit) {
        char *w = static_cast<char *>(ws);
        p.ws_cnt = reinterpret_cast<int *>(w + lay.off_cnt);
        p.ws_ml = reinterpret_cast<float *>(w + lay.off_ml);
        p.ws_o = reinterpret_cast<float *>(w + lay.off_o);
    }
    p.status = d_status;
    p.wait_cycles = (opt && opt->wait_limit_cycles > 0) ? (long long)opt->wait_limit_cycles : kDefaultWaitCycles;
    p.test_stall = (opt && opt->test_stall) ? 1 : 0;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (kernel == GQA_KERNEL_TC) {
        TcMaps maps;
        const int T = p.tile;
        bool ok;
        const int es = kv8 ? 1 : 2;
        if (s.paged) {
            const int box = s.block_size < T ? s.block_size : T;
            ok = encode_cache_map(&maps.k, kc, s.D, s.block_size, (long long)s.num_blocks * s.Hkv, box, es) &&
                 encode_cache_map(&maps.v, vc, s.D, s.block_size, (long long)s.num_blocks * s.Hkv, box, es);
            maps.k16 = maps.k;   // not used with a paged cache
            maps.v16 = maps.v;
        } else {
            ok = encode_cache_map(&maps.k, kc, s.D, s.Smax, (long long)s.R * s.Hkv, T, es) &&
                 encode_cache_map(&maps.v, vc, s.D, s.Smax, (long long)s.R * s.Hkv, T, es) &&
                 encode_cache_map(&maps.k16, kc, s.D, s.Smax, (long long)s.R * s.Hkv, kDenseBoxRows, es) &&
                 encode_cache_map(&maps.v16, vc, s.D, s.Smax, (long long)s.R * s.Hkv, kDenseBoxRows, es);
        }
        if (!ok)
            return GQA_ERR_CUDA;
        // the opt-in tcgen05 form of 17- to 32-row multi-token units
        const bool t5 = opt && opt->kernel == GQA_KERNEL_TC5 && s.multi && tc5_takes(p);
        TraceScope ts(t5 ? 3 : 1, cs);
        e = t5 ? tc5_launch_multi(p, maps, cs) : tc_launch(p, maps, cs);
    } else if (unit) {
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return GQA_ERR_CUDA;
        TraceScope ts(2, cs);
        e = unit_launch(p, s.dt == GQA_DTYPE_BF16, cap_rows, sm_count(dev), cs);
    } else {
        TraceScope ts(0, cs);
        e = simt_launch(p, s.dt == GQA_DTYPE_BF16, cs);
    }
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *gqa_status_string(gqa_status s)
{
    switch (s) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported sizes (no kernel in this build)";
    case GQA_ERR_CUDA: return "CUDA runtime error";
    case GQA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GQA_ERR_TOO_LARGE: return "sizes need more scratch than gqa_decode_step_noalloc holds";
    }
    return "unknown status";
}

size_t gqa_workspace_bytes(int B, int Hq, int Hkv, int D, gqa_dtype dt, const gqa_options *opt)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv)
        return 0;
    const int G = Hq / Hkv;
    // the block size only matters for the paged form; 16 is the common case and
    // the workspace does not depend on it
    int kernel = pick_kernel(opt, dt, D, G, false, 16);
    if (opt && opt->kernel == GQA_KERNEL_UNIT)
        return 0;   // the small-cache kernel takes no workspace
    if (kernel < 0)
        return 0;
    int grid = grid_for(kernel, opt, dt, D, G);
    // AUTO may pick either kernel depending on the block size: size for the larger grid
    if ((!opt || opt->kernel == GQA_KERNEL_AUTO) && simt_supports(D, G)) {
        const int g2 = grid_for(GQA_KERNEL_SIMT, opt, dt, D, G);
        grid = grid > g2 ? grid : g2;
    }
    if (grid <= 0)
        return 0;
    return workspace_layout(B, Hkv, G, D, grid).bytes;
}

gqa_status gqa_decode_step_ex(const void *q, const void *k_new, const void *v_new, void *k_cache,
                              void *v_cache, const int32_t *lengths, const int32_t *slot_ids,
                              float *out, int B, int Hq, int Hkv, int D, int R, int Smax,
                              gqa_dtype dt, void *workspace, size_t workspace_bytes,
                              int32_t *d_status, void *stream, const gqa_options *opt)
{
    // over an E4M3 cache the query and the new key / value are bfloat16
    const gqa_dtype qdt = dt == GQA_DTYPE_E4M3 ? GQA_DTYPE_BF16 : dt;
    Shape s = {B, Hq, Hkv, D, dt, false, R, Smax, 0, 0, 0, false, qdt};
    return run_step(s, q, k_new, v_new, k_cache, v_cache, lengths, slot_ids, nullptr, out,
                    workspace, workspace_bytes, d_status, stream, opt);
}

gqa_status gqa_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache,
                           void *v_cache, const int32_t *lengths, const int32_t *slot_ids,
                           float *out, int B, int Hq, int Hkv, int D, int R, int Smax,
                           gqa_dtype dt, void *workspace, size_t workspace_bytes,
                           int32_t *d_status, void *stream)
{
    return gqa_decode_step_ex(q, k_new, v_new, k_cache, v_cache, lengths, slot_ids, out, B, Hq,
                              Hkv, D, R, Smax, dt, workspace, workspace_bytes, d_status, stream,
                              nullptr);
}

gqa_status gqa_decode_step_paged_ex(const void *q, const void *k_new, const void *v_new,
                                    void *k_blocks, void *v_blocks, const int32_t *block_table,
                                    const int32_t *lengths, float *out, int B, int Hq, int Hkv,
                                    int D, int num_blocks, int block_size, int max_blocks,
                                    gqa_dtype dt, void *workspace, size_t workspace_bytes,
                                    int32_t *d_status, void *stream, const gqa_options *opt)
{
    const gqa_dtype qdt = dt == GQA_DTYPE_E4M3 ? GQA_DTYPE_BF16 : dt;
    Shape s = {B, Hq, Hkv, D, dt, true, 0, 0, num_blocks, block_size, max_blocks, false, qdt};
    return run_step(s, q, k_new, v_new, k_blocks, v_blocks, lengths, nullptr, block_table, out,
                    workspace, workspace_bytes, d_status, stream, opt);
}

gqa_status gqa_decode_step_paged(const void *q, const void *k_new, const void *v_new,
                                 void *k_blocks, void *v_blocks, const int32_t *block_table,
                                 const int32_t *lengths, float *out, int B, int Hq, int Hkv, int D,
                                 int num_blocks, int block_size, int max_blocks, gqa_dtype dt,
                                 void *workspace, size_t workspace_bytes, int32_t *d_status,
                                 void *stream)
{
    return gqa_decode_step_paged_ex(q, k_new, v_new, k_blocks, v_blocks, block_table, lengths, out,
                                    B, Hq, Hkv, D, num_blocks, block_size, max_blocks, dt,
                                    workspace, workspace_bytes, d_status, stream, nullptr);
}

}  // extern "C"

namespace {

gqa_status validate_common(const int32_t *lengths, const int32_t *slot_ids, const int32_t *block_table,
                           int B, int R, int Smax, int num_blocks, int block_size, int max_blocks,
                           int attend, int32_t *d_result, void *stream, const int32_t *cu_q = nullptr,
                           int T = 0)
{
    if (B < 0 || !d_result)
        return GQA_ERR_INVALID_ARGUMENT;
    if (block_table) {
        if (num_blocks < 1 || block_size < 1 || max_blocks < 1)
            return GQA_ERR_INVALID_ARGUMENT;
    } else if (R < 0 || Smax < 1 || (!slot_ids && B > R)) {
        return GQA_ERR_INVALID_ARGUMENT;
    }
    if (B == 0)
        return GQA_OK;
    if (!lengths)
        return GQA_ERR_INVALID_ARGUMENT;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(d_result, 0, sizeof(int32_t), cs) != cudaSuccess)
        return GQA_ERR_CUDA;
    if (validate_launch(lengths, block_table ? nullptr : slot_ids, block_table, B, R, Smax,
                        num_blocks, block_size, max_blocks, attend, cu_q, T, d_result, cs) != cudaSuccess)
        return GQA_ERR_CUDA;
    int32_t h = 0;
    if (cudaMemcpyAsync(&h, d_result, sizeof h, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess)
        return GQA_ERR_CUDA;
    return h ? GQA_ERR_INVALID_ARGUMENT : GQA_OK;
}

}  // namespace

extern "C" {

gqa_status gqa_validate(const int32_t *lengths, const int32_t *slot_ids, const int32_t *block_table,
                        int B, int R, int Smax, int num_blocks, int block_size, int max_blocks,
                        int32_t *d_result, void *stream)
{
    return validate_common(lengths, slot_ids, block_table, B, R, Smax, num_blocks, block_size,
                           max_blocks, 0, d_result, stream);
}

gqa_status gqa_validate_attend(const int32_t *lengths, const int32_t *slot_ids,
                               const int32_t *block_table, int B, int R, int Smax, int num_blocks,
                               int block_size, int max_blocks, int32_t *d_result, void *stream)
{
    return validate_common(lengths, slot_ids, block_table, B, R, Smax, num_blocks, block_size,
                           max_blocks, 1, d_result, stream);
}

gqa_status gqa_validate_multi(const int32_t *lengths, const int32_t *cu_q, const int32_t *slot_ids,
                              const int32_t *block_table, int B, int T, int R, int Smax, int num_blocks,
                              int block_size, int max_blocks, int32_t *d_result, void *stream)
{
    if (!cu_q || T < 0)
        return GQA_ERR_INVALID_ARGUMENT;
    return validate_common(lengths, slot_ids, block_table, B, R, Smax, num_blocks, block_size,
                           max_blocks, 0, d_result, stream, cu_q, T);
}

size_t gqa_workspace_bytes_multi(int B, int Hq, int Hkv, int D, gqa_dtype dt, int max_q_len,
                                 const gqa_options *opt)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv || max_q_len < 0 || Hq / Hkv > 8)
        return 0;
    const int Gh = Hq / Hkv;
    // enough for whichever kernel the call will pick (AUTO may depend on the
    // paged block size): the larger of the two cuts' workspaces
    size_t bytes = 0;
    for (int k = GQA_KERNEL_SIMT; k <= GQA_KERNEL_TC; ++k) {
        const int want = opt ? (opt->kernel == GQA_KERNEL_TC5 ? GQA_KERNEL_TC : opt->kernel) : GQA_KERNEL_AUTO;
        if (want != GQA_KERNEL_AUTO && want != k)
            continue;
        gqa_options o = opt ? *opt : gqa_options{};
        o.kernel = k;
        if (pick_kernel(&o, dt, D, Gh, false, 16) != k)
            continue;
        const MultiCut cut = multi_cut(Gh, max_q_len, k == GQA_KERNEL_TC ? 32 : 8);
        const int G = Gh * cut.tpc;
        const int grid = grid_for(k, &o, dt, D, G);
        if (grid <= 0)
            continue;
        const size_t b = workspace_layout(B * cut.chunks, Hkv, G, D, grid).bytes;
        bytes = b > bytes ? b : bytes;
    }
    return bytes;
}

gqa_status gqa_decode_multi(const void *q, const void *k_new, const void *v_new, void *k_cache,
                            void *v_cache, const int32_t *lengths, const int32_t *cu_q,
                            const int32_t *slot_ids, float *out, int B, int T, int max_q_len, int Hq,
                            int Hkv, int D, int R, int Smax, gqa_dtype dt, void *workspace,
                            size_t workspace_bytes, int32_t *d_status, void *stream,
                            const gqa_options *opt)
{
    const gqa_dtype qdt = dt == GQA_DTYPE_E4M3 ? GQA_DTYPE_BF16 : dt;   // query and new tokens
    Shape s = {B, Hq, Hkv, D, dt, false, R, Smax, 0, 0, 0, false, qdt, true, T, max_q_len};
    return run_step(s, q, k_new, v_new, k_cache, v_cache, lengths, slot_ids, nullptr, out, workspace,
                    workspace_bytes, d_status, stream, opt, cu_q);
}

gqa_status gqa_decode_multi_paged(const void *q, const void *k_new, const void *v_new,
                                  void *k_blocks, void *v_blocks, const int32_t *block_table,
                                  const int32_t *lengths, const int32_t *cu_q, float *out, int B,
                                  int T, int max_q_len, int Hq, int Hkv, int D, int num_blocks,
                                  int block_size, int max_blocks, gqa_dtype dt, void *workspace,
                                  size_t workspace_bytes, int32_t *d_status, void *stream,
                                  const gqa_options *opt)
{
    const gqa_dtype qdt = dt == GQA_DTYPE_E4M3 ? GQA_DTYPE_BF16 : dt;
    Shape s = {B, Hq, Hkv, D, dt, true, 0, 0, num_blocks, block_size, max_blocks, false, qdt, true, T,
               max_q_len};
    return run_step(s, q, k_new, v_new, k_blocks, v_blocks, lengths, nullptr, block_table, out,
                    workspace, workspace_bytes, d_status, stream, opt, cu_q);
}

gqa_status gqa_attend(const void *q, gqa_dtype q_dtype, const void *k_cache, const void *v_cache,
                      const int32_t *lengths, const int32_t *slot_ids, float *out, int B, int Hq,
                      int Hkv, int D, int R, int Smax, gqa_dtype kv_dtype, void *workspace,
                      size_t workspace_bytes, int32_t *d_status, void *stream,
                      const gqa_options *opt)
{
    Shape s = {B, Hq, Hkv, D, kv_dtype, false, R, Smax, 0, 0, 0, true, q_dtype};
    // the kernels never write the cache in this mode
    return run_step(s, q, nullptr, nullptr, const_cast<void *>(k_cache), const_cast<void *>(v_cache),
                    lengths, slot_ids, nullptr, out, workspace, workspace_bytes, d_status, stream, opt);
}

gqa_status gqa_attend_paged(const void *q, gqa_dtype q_dtype, const void *k_blocks,
                            const void *v_blocks, const int32_t *block_table,
                            const int32_t *lengths, float *out, int B, int Hq, int Hkv, int D,
                            int num_blocks, int block_size, int max_blocks, gqa_dtype kv_dtype,
                            void *workspace, size_t workspace_bytes, int32_t *d_status,
                            void *stream, const gqa_options *opt)
{
    Shape s = {B, Hq, Hkv, D, kv_dtype, true, 0, 0, num_blocks, block_size, max_blocks, true, q_dtype};
    return run_step(s, q, nullptr, nullptr, const_cast<void *>(k_blocks), const_cast<void *>(v_blocks),
                    lengths, nullptr, block_table, out, workspace, workspace_bytes, d_status, stream,
                    opt);
}

int gqa_trace_enable(int on)
{
    std::lock_guard<std::mutex> g(trace().mu);
    int prev = trace().on ? 1 : 0;
    trace().on = on != 0;
    return prev;
}

gqa_status gqa_trace_collect(int n_kinds, int64_t *launches, double *ms)
{
    std::vector<TraceRec> recs;
    {
        std::lock_guard<std::mutex> g(trace().mu);
        recs.swap(trace().pending);
    }
    for (int k = 0; k < n_kinds; ++k) {
        if (launches) launches[k] = 0;
        if (ms) ms[k] = 0.0;
    }
    gqa_status st = GQA_OK;
    for (const TraceRec &r : recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
            st = GQA_ERR_CUDA;
        if (r.kind < n_kinds) {
            if (launches) launches[r.kind] += 1;
            if (ms) ms[r.kind] += t;
        }
        std::lock_guard<std::mutex> g(trace().mu);
        trace().pool.push_back(r.start);
        trace().pool.push_back(r.stop);
    }
    return st;
}

const char *gqa_kernel_name(int kind)
{
    switch (kind) {
    case 0: return "simt_decode_kernel";
    case 1: return "tc_decode_kernel";
    case 2: return "unit_decode_kernel";
    case 3: return "tc5_multi_kernel";
    }
    return "unknown";
}

gqa_status gqa_workspace_reset(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace)
        return GQA_ERR_INVALID_ARGUMENT;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GQA_OK
               : GQA_ERR_CUDA;
}

int gqa_version(void) { return 100; }

}  // extern "C"
