/*
 * gqa_decode.h — C ABI of the GB300 grouped-query-attention decode step.
 *
 * One decode step, for every batch row b of a batch of B sequences:
 *
 *   1. append: the new key and value of cache head kvh, k_new[b][kvh] and
 *      v_new[b][kvh], are written IN PLACE into slot lengths[b] of the row's
 *      cache ("groupQueryAttention", clika runtime: binding the present
 *      outputs to the past buffers appends in place, the decode perf path;
 *      "KV cache decode step", tensortonic: the new token takes position S
 *      after the S cached ones);
 *   2. attend: query head h (G = Hq/Hkv, cache head kvh = floor(h/G), the
 *      contiguous grouping of "Grouped-Query Decode Step", tensortonic,
 *      statement) scores slots j = 0..lengths[b] with s_j = q.K_j / sqrt(D),
 *      takes the softmax over those slots only (stale slots beyond the length
 *      get exactly zero weight, same page, statement and Requirements) and
 *      returns o = sum_j w_j V_j in float32.
 *
 * Scores, softmax and the weighted sum are computed in float32 from float32
 * or bfloat16 data ("Grouped-Query Decode Step", Requirements).
 *
 * The read-only attend (gqa_attend, gqa_attend_paged) is step 2 alone over
 * slots 0..lengths[b]-1, with lengths[b] counting the valid cached slots and
 * a query dtype of its own (a float32 query over a bfloat16 cache is that
 * page's contract); it writes nothing but its output.
 *
 * Conventions for every entry point:
 *  - Pointers marked (device) point to GPU memory of the current device;
 *    (host) to host memory. The library never allocates, frees or keeps any
 *    of them; the caller owns every buffer, including the workspace
 *    (the two-phase size-query-then-execute pattern of "aclnnMlaPrologV3
 *    WeightNz", CANN, calling sequence).
 *  - Tensors are dense and row-major in the shapes given; device pointers
 *    must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL: the legacy default stream). Calls are
 *    asynchronous on it unless stated otherwise.
 *  - Argument errors that the host can see (null pointers, shapes, dtype,
 *    workspace too small, unsupported sizes) return an error code before
 *    anything is launched, and nothing is written.
 *  - Content errors that only the device can see (a length out of range, a
 *    slot id out of range, a block-table entry out of range or -1 where a
 *    slot is needed) never fault: the affected batch row gets NaN outputs,
 *    its append is skipped when the append slot itself cannot be addressed,
 *    and a bit is OR-ed into *d_status (if d_status is not NULL).
 *    *d_status is sticky: the library never clears it. gqa_validate checks
 *    content completely (including duplicates) and synchronously.
 *  - B = 0 is valid: nothing is launched and GQA_OK is returned (empty
 *    tensors, "aclnnMlaPrologV3WeightNz", shape restrictions).
 *  - Results are deterministic: the same inputs and launch configuration give
 *    the same bits (no floating-point atomics).
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gqa_status {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARGUMENT = 1, /* bad shape/pointer/content (validate)      */
    GQA_ERR_UNSUPPORTED = 2,      /* a size this build has no kernel for       */
    GQA_ERR_CUDA = 3,             /* a CUDA runtime call failed                */
    GQA_ERR_WORKSPACE = 4,        /* workspace NULL or smaller than required   */
    GQA_ERR_TOO_LARGE = 5         /* sizes need more than the fixed scratch of
                                     gqa_decode_step_noalloc                   */
} gqa_status;

typedef enum gqa_dtype {
    GQA_DTYPE_F32 = 0,  /* float32  (decode step: q, k_new, v_new and the cache) */
    GQA_DTYPE_BF16 = 1, /* bfloat16 (decode step: q, k_new, v_new and the cache) */
    GQA_DTYPE_E4M3 = 2  /* a cache of OCP FP8 E4M3 bytes with per-cache-head float32
                           scales (gqa_options.k_scale / v_scale): K = k_scale[kvh] *
                           K8, V = v_scale[kvh] * V8 ("groupQueryAttention": kScale,
                           vScale). The decode step then takes bfloat16 q, k_new and
                           v_new and appends E4M3(float32(k_new) / k_scale[kvh]),
                           rounded to nearest even and saturated to +-448; the
                           read-only attend takes a float32 or bfloat16 query. Only
                           the tensor-core kernel takes it (D = 128, G <= 8; paged
                           block sizes a power of two >= 8); single-token steps. */
} gqa_dtype;

/* Bits OR-ed into *d_status by the kernels. */
enum {
    GQA_STATUS_BAD_LENGTH = 1,      /* lengths[b] < 0 (attend: < 1) or beyond the row's
                                       capacity                                           */
    GQA_STATUS_BAD_SLOT_ID = 2,     /* slot_ids[b] outside [0, R)                        */
    GQA_STATUS_BAD_BLOCK = 4,       /* block-table entry outside [0, num_blocks) or -1
                                       where a slot 0..lengths[b] lives                   */
    GQA_STATUS_TIMEOUT = 8,         /* a bounded on-chip wait gave up (never expected)    */
    GQA_STATUS_BAD_PREFIX = 16,     /* kept_prefix_rows[b] < 0                            */
    GQA_STATUS_BAD_QLEN = 32        /* multi-token: cu_q[b] / cu_q[b+1] outside [0, T],
                                       decreasing, or q_len above max_q_len             */
};

/* Kernel choice for the *_ex entry points. */
typedef enum gqa_kernel {
    GQA_KERNEL_AUTO = 0, /* the fastest kernel that supports the shapes                  */
    GQA_KERNEL_SIMT = 1, /* CUDA-core FMA kernel: any D in {1,2,4,...,256}, G <= 8,
                            float32 or bfloat16, any block size                          */
    GQA_KERNEL_TC = 2,   /* TMA ring + tensor-core kernel: bfloat16, D = 128, G <= 8,
                            block size a power of two >= 8                               */
    GQA_KERNEL_UNIT = 3  /* small caches: one CTA per (row, cache head), the row's attended
                            slots staged in shared memory by bulk copies, no workspace
                            used: float32 or bfloat16, D in {32, 64, 128, 256}, G <= 8,
                            2 * capacity * D * element size <= 200 KB (capacity = Smax,
                            or max_blocks * block_size); single-token steps (decode and
                            attend). AUTO takes it when those hold and the (row, head)
                            pairs fit in one wave of the GPU                             */,
    GQA_KERNEL_TC5 = 4   /* as GQA_KERNEL_TC, but multi-token units of 17 to 32 query rows
                            over a bfloat16 cache run on the tcgen05 tensor cores
                            (accumulators in tensor memory); never chosen by AUTO:
                            measured slower than GQA_KERNEL_TC for those units       */
} gqa_kernel;

/* Launch options (all zero = defaults). */
typedef struct gqa_options {
    int kernel;     /* a gqa_kernel                                                      */
    int grid_ctas;  /* 0: one persistent wave sized to the device; > 0: exactly this
                       many CTAs (each takes a contiguous share of the KV tiles; any
                       value gives the same output up to float32 rounding)             */
    int sched_pad;  /* 0: the default; k > 0: count k - 1 extra schedule-only tiles per
                       (row, cache head) when sharing the tiles among CTAs, which gives
                       CTAs that finish more sequences fewer tiles (no effect on
                       results beyond float32 rounding)                                 */
    /* Softmax modifiers ("groupQueryAttention": slidingWindow, kept_prefix,
     * head_sink). With the query at position L (the appended slot of the decode
     * step, the last valid slot of the attend), slot j <= L is attended when
     * window == 0, or j > L - window (the window positions up to and including
     * the query's own), or j < P (the row's kept prefix, used only with a
     * window). Only tiles (and paged blocks) holding attended slots are read;
     * the other slots' contents do not matter, and paged entries that hold no
     * attended slot (nor the appended one) may be -1. The sink of query head h
     * is one more logit in the softmax denominator, in the units of the scaled
     * scores: w_j = e^{s_j} / (e^{sink_h} + sum_{i attended} e^{s_i}).        */
    int window;       /* >= 0 (0: no window); < 0 is GQA_ERR_INVALID_ARGUMENT          */
    int kept_prefix;  /* P >= 0 for every row, used when kept_prefix_rows is NULL       */
    int wait_limit_cycles; /* 0: the default (about 2 s). c > 0: a tensor-core consumer
                       warp's wait for a tile to land gives up after c SM clock cycles;
                       its CTA then aborts (the units it touches get NaN, their appends
                       may be skipped, GQA_STATUS_TIMEOUT is set), every copy it issued
                       still lands before it exits, and the workspace is left
                       zero-filled. For tests of the timeout path; < 0 is
                       GQA_ERR_INVALID_ARGUMENT                                        */
    int test_stall;   /* 0: off. 1 (tests of the timeout path): every tensor-core
                       consumer warp's first wait for a tile also waits on an on-chip
                       barrier that nothing completes, so that wait runs out after
                       wait_limit_cycles (keep it short) and every CTA aborts as
                       described above                                                 */
    int reserved[1];
    const float *head_sink;          /* (device) (Hq,) float32 logits, or NULL          */
    const int32_t *kept_prefix_rows; /* (device) (B,) int32 P per batch row, or NULL;
                                        a negative entry makes that row bad
                                        (NaN, GQA_STATUS_BAD_PREFIX)                    */
    const float *k_scale;            /* (device) (Hkv,) float32: required with an
                                        E4M3 cache (GQA_DTYPE_E4M3), else ignored       */
    const float *v_scale;            /* (device) (Hkv,) float32, likewise               */
} gqa_options;

/* Human-readable name of a status code (static storage). */
const char *gqa_status_string(gqa_status s);

/*
 * Workspace bytes a decode step needs on the current device for these sizes
 * (one arrival counter per (row, cache head) and the float32 partial softmax
 * states of the sequences that several CTAs share). opt may be NULL. Returns
 * 0 for invalid sizes, and 0 when opt asks for GQA_KERNEL_UNIT (that kernel
 * takes no workspace: NULL may then be passed). Under GQA_KERNEL_AUTO the
 * size covers whichever kernel the call may take.
 *
 * The workspace must be zero-filled (gqa_workspace_reset or any memset)
 * before its first use; every call leaves it zero-filled again, whatever the
 * sizes of the next call. Zero it again after a call that reported
 * GQA_STATUS_TIMEOUT. One workspace serves one call at a time (calls that may
 * overlap on the GPU need different workspaces).
 */
size_t gqa_workspace_bytes(int B, int Hq, int Hkv, int D, gqa_dtype dt, const gqa_options *opt);

/* Zero-fills a workspace asynchronously on `stream` (a cudaMemsetAsync). */
gqa_status gqa_workspace_reset(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Dense or continuous-batch decode step.
 *
 *  q        (device) (B, Hq, D)          query of the new token
 *  k_new    (device) (B, Hkv, D)         new key   (appended at lengths[b])
 *  v_new    (device) (B, Hkv, D)         new value (appended at lengths[b])
 *  k_cache  (device) (R, Hkv, Smax, D)   key cache, written at one slot per (row, kvh)
 *  v_cache  (device) (R, Hkv, Smax, D)   value cache, same
 *  lengths  (device) (B,) int32          append slot = number of cached tokens of
 *                                        row b; 0 <= lengths[b] <= Smax-1. Not modified:
 *                                        the caller advances it.
 *  slot_ids (device) (B,) int32 or NULL  cache row of batch row b on a continuous
 *                                        [max_seqs = R, Hkv, Smax, D] cache: entries in
 *                                        [0, R), pairwise distinct ("groupQueryAttention",
 *                                        slot_ids). NULL: row b uses cache row b (R >= B).
 *  out      (device) (B, Hq, D) float32  attention output
 *  workspace(device) >= gqa_workspace_bytes(...) bytes, 256-byte aligned,
 *                                        zero-filled before its first use
 *  d_status (device) int32 or NULL       sticky content-error bits (see above)
 */
gqa_status gqa_decode_step(const void *q, const void *k_new, const void *v_new,
                           void *k_cache, void *v_cache, const int32_t *lengths,
                           const int32_t *slot_ids, float *out,
                           int B, int Hq, int Hkv, int D, int R, int Smax, gqa_dtype dt,
                           void *workspace, size_t workspace_bytes, int32_t *d_status,
                           void *stream);

/*
 * Paged decode step. The cache is a pool of blocks; slot s of batch row b
 * lives in block block_table[b][s / block_size] at offset s % block_size.
 *
 *  k_blocks    (device) (num_blocks, Hkv, block_size, D)
 *  v_blocks    (device) (num_blocks, Hkv, block_size, D)
 *  block_table (device) (B, max_blocks) int32: each entry -1 (unused tail pad) or
 *              a block in [0, num_blocks), no block twice in one row
 *              ("groupQueryAttention", paged block table); the entries holding
 *              slots 0..lengths[b] must be real blocks. A block named by two rows
 *              that receives this step's append is undefined (the pages leave it open).
 *  lengths     (device) (B,) int32, 0 <= lengths[b] < max_blocks * block_size.
 * Other arguments as in gqa_decode_step (there are no slot_ids: the block
 * table is the row map).
 */
gqa_status gqa_decode_step_paged(const void *q, const void *k_new, const void *v_new,
                                 void *k_blocks, void *v_blocks, const int32_t *block_table,
                                 const int32_t *lengths, float *out,
                                 int B, int Hq, int Hkv, int D,
                                 int num_blocks, int block_size, int max_blocks, gqa_dtype dt,
                                 void *workspace, size_t workspace_bytes, int32_t *d_status,
                                 void *stream);

/* The same two steps with launch options (kernel choice, CTA count). */
gqa_status gqa_decode_step_ex(const void *q, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, const int32_t *lengths,
                              const int32_t *slot_ids, float *out,
                              int B, int Hq, int Hkv, int D, int R, int Smax, gqa_dtype dt,
                              void *workspace, size_t workspace_bytes, int32_t *d_status,
                              void *stream, const gqa_options *opt);

gqa_status gqa_decode_step_paged_ex(const void *q, const void *k_new, const void *v_new,
                                    void *k_blocks, void *v_blocks, const int32_t *block_table,
                                    const int32_t *lengths, float *out,
                                    int B, int Hq, int Hkv, int D,
                                    int num_blocks, int block_size, int max_blocks, gqa_dtype dt,
                                    void *workspace, size_t workspace_bytes, int32_t *d_status,
                                    void *stream, const gqa_options *opt);

/*
 * Content validation, complete and SYNCHRONOUS (it waits for `stream`):
 * lengths in range; slot_ids in range and distinct; every block-table entry
 * -1 or in range, no repeats within a row, real blocks for slots
 * 0..lengths[b] ("groupQueryAttention": the table is validated whole before
 * any read). Pass block_table = NULL for the dense / slot_ids form (then
 * num_blocks, block_size and max_blocks are ignored) and slot_ids = NULL for
 * the plain dense form; with a block table, slot_ids, R and Smax are ignored.
 * Runs on the GPU; d_result (device) is one int32 of caller memory that the
 * call overwrites. Returns GQA_OK or GQA_ERR_INVALID_ARGUMENT (or an error of
 * the call itself).
 */
gqa_status gqa_validate(const int32_t *lengths, const int32_t *slot_ids,
                        const int32_t *block_table, int B, int R, int Smax,
                        int num_blocks, int block_size, int max_blocks,
                        int32_t *d_result, void *stream);

/*
 * Read-only attend over a dense or continuous-batch cache: every query head h
 * attends slots 0..lengths[b]-1 of cache head floor(h/G) of its row, with the
 * same scores, softmax and float32 output as the decode step, and nothing is
 * appended or written besides `out` ("groupQueryAttention": a read-only attend
 * passes no key or value and takes no present outputs, attention_over_cache;
 * "Grouped-Query Decode Step", statement and Constraints: lengths counts the
 * valid slots, the new token already among them, 1 <= lengths[b] <= S; the
 * query is float32 and the caches float32 or bfloat16).
 *
 *  q        (device) (B, Hq, D) of q_dtype (float32 or bfloat16)
 *  k_cache  (device) (R, Hkv, Smax, D) of kv_dtype, only read
 *  v_cache  (device) (R, Hkv, Smax, D) of kv_dtype, only read
 *  lengths  (device) (B,) int32, 1 <= lengths[b] <= Smax: valid slots of row b
 *  slot_ids (device) (B,) int32 or NULL, as in gqa_decode_step
 *  out      (device) (B, Hq, D) float32
 *  workspace, d_status, stream: as in gqa_decode_step (the same
 *           gqa_workspace_bytes, computed with kv_dtype); opt may be NULL.
 * A bad length (< 1 or > Smax) or slot id gives that row NaN outputs and sets
 * its status bit. The tensor-core kernel takes a bfloat16 cache with D = 128
 * and G <= 8 and either query dtype; everything else runs on the CUDA-core
 * kernel.
 */
gqa_status gqa_attend(const void *q, gqa_dtype q_dtype, const void *k_cache, const void *v_cache,
                      const int32_t *lengths, const int32_t *slot_ids, float *out,
                      int B, int Hq, int Hkv, int D, int R, int Smax, gqa_dtype kv_dtype,
                      void *workspace, size_t workspace_bytes, int32_t *d_status, void *stream,
                      const gqa_options *opt);

/*
 * Read-only attend over a paged cache (blocks and table as in
 * gqa_decode_step_paged); 1 <= lengths[b] <= max_blocks * block_size and the
 * entries holding slots 0..lengths[b]-1 must be real blocks.
 */
gqa_status gqa_attend_paged(const void *q, gqa_dtype q_dtype, const void *k_blocks,
                            const void *v_blocks, const int32_t *block_table,
                            const int32_t *lengths, float *out,
                            int B, int Hq, int Hkv, int D,
                            int num_blocks, int block_size, int max_blocks, gqa_dtype kv_dtype,
                            void *workspace, size_t workspace_bytes, int32_t *d_status,
                            void *stream, const gqa_options *opt);

/*
 * gqa_validate for the read-only attend's reading of lengths: the same rules
 * with 1 <= lengths[b] <= capacity and real blocks for slots
 * 0..lengths[b]-1. Synchronous; same arguments and results.
 */
gqa_status gqa_validate_attend(const int32_t *lengths, const int32_t *slot_ids,
                               const int32_t *block_table, int B, int R, int Smax,
                               int num_blocks, int block_size, int max_blocks,
                               int32_t *d_result, void *stream);

/*
 * Multi-token step (speculative or chunked decode): batch row b brings
 * q_len[b] = cu_q[b+1] - cu_q[b] new tokens, the packed rows cu_q[b] ..
 * cu_q[b+1]-1 of q, k_new, v_new and out. They are appended in place at slots
 * lengths[b] .. lengths[b] + q_len[b] - 1, and the query heads of token i
 * attend slots 0 .. lengths[b] + i of their cache head, the new tokens up to
 * their own included ("groupQueryAttention": q/k/v are packed [sum S,
 * heads * head_dim]; each row's write offset is cu_seqlens_k[b] - q_len[b],
 * i.e. lengths[b]; the append is in place; keys beyond the query's own
 * position are outside the causal bound). q_len = 1 everywhere is exactly
 * gqa_decode_step.
 *
 *  q        (device) (T, Hq, D)          queries of the new tokens
 *  k_new    (device) (T, Hkv, D)         their keys   (appended)
 *  v_new    (device) (T, Hkv, D)         their values (appended)
 *  lengths  (device) (B,) int32          write offset of row b (tokens already cached);
 *                                        0 <= lengths[b], lengths[b] + q_len[b] <= capacity
 *  cu_q     (device) (B + 1,) int32      cu_q[0] = 0, nondecreasing, cu_q[B] = T
 *  max_q_len (host)  bound on every q_len[b] (sizes the schedule and workspace;
 *                    a larger q_len makes the row bad: GQA_STATUS_BAD_QLEN and
 *                    its outputs are not written)
 *  out      (device) (T, Hq, D) float32
 *  Other arguments as in gqa_decode_step / gqa_decode_step_paged (the same
 *  softmax modifiers apply, each token with its own position). The workspace
 *  is gqa_workspace_bytes_multi(...). A bad row (length, slot id, block) gets
 *  NaN outputs for its tokens and its appends are skipped where their slots
 *  cannot be addressed. Rows with q_len = 0 are left alone.
 * Kernels: up to 16 / G tokens of a row (G = Hq / Hkv <= 8; 8 / G on the
 * CUDA-core kernel) share one pass over the cache; longer runs are cut into
 * chunks, each streaming the cache again. Over an E4M3 cache (tensor-core
 * kernel only) q, k_new and v_new are bfloat16, opt carries k_scale / v_scale
 * and each appended token is quantised as in gqa_decode_step.
 */
size_t gqa_workspace_bytes_multi(int B, int Hq, int Hkv, int D, gqa_dtype dt, int max_q_len,
                                 const gqa_options *opt);

gqa_status gqa_decode_multi(const void *q, const void *k_new, const void *v_new,
                            void *k_cache, void *v_cache, const int32_t *lengths,
                            const int32_t *cu_q, const int32_t *slot_ids, float *out,
                            int B, int T, int max_q_len, int Hq, int Hkv, int D, int R, int Smax,
                            gqa_dtype dt, void *workspace, size_t workspace_bytes,
                            int32_t *d_status, void *stream, const gqa_options *opt);

gqa_status gqa_decode_multi_paged(const void *q, const void *k_new, const void *v_new,
                                  void *k_blocks, void *v_blocks, const int32_t *block_table,
                                  const int32_t *lengths, const int32_t *cu_q, float *out,
                                  int B, int T, int max_q_len, int Hq, int Hkv, int D,
                                  int num_blocks, int block_size, int max_blocks, gqa_dtype dt,
                                  void *workspace, size_t workspace_bytes, int32_t *d_status,
                                  void *stream, const gqa_options *opt);

/*
 * gqa_validate for a multi-token step: the cu_q rules above, 0 <= lengths[b],
 * lengths[b] + q_len[b] <= Smax (dense) and, paged, the table rules with real
 * blocks for slots 0 .. lengths[b] + q_len[b] - 1. Synchronous.
 */
gqa_status gqa_validate_multi(const int32_t *lengths, const int32_t *cu_q, const int32_t *slot_ids,
                              const int32_t *block_table, int B, int T, int R, int Smax,
                              int num_blocks, int block_size, int max_blocks, int32_t *d_result,
                              void *stream);

/*
 * Kernel timing trace. When enabled, every decode call records CUDA events
 * around the kernel it launches; gqa_trace_collect waits for them and
 * returns, per kernel kind, the launches and total milliseconds since the
 * previous collect. Kinds: 0 = SIMT decode, 1 = tensor-core decode, 2 = the
 * small-cache decode, 3 = the tcgen05 form of 17- to 32-row multi-token
 * units (each decode step is exactly one kernel launch); gqa_kernel_name
 * gives each kind's kernel name. Meant for benchmarks.
 */
int gqa_trace_enable(int on);
gqa_status gqa_trace_collect(int n_kinds, int64_t *launches, double *ms);
const char *gqa_kernel_name(int kind);

/*
 * The dense / continuous-batch decode step without a workspace argument, for
 * callers that cannot allocate device memory (for example a plugin host that
 * gives an operator no scratch and forbids allocation while it runs, or a
 * plain C caller without a device allocator). The pages have no counterpart:
 * this is a deployment convenience.
 *
 * Arguments as in gqa_decode_step. The scratch is a fixed array of
 * gqa_noalloc_scratch_bytes() (8 MiB) inside the library, held by every GPU
 * that loads the library until the process exits; sizes whose workspace
 * (gqa_workspace_bytes) exceeds it return GQA_ERR_TOO_LARGE before any launch.
 * The call allocates nothing. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture. The address is kept for the life of
 * the process: do not use this entry point on a device after cudaDeviceReset
 * (or anything else that destroys its primary context) in the same process.
 * All calls share the array: calls whose kernels overlap on the GPU race and
 * must be serialised by the caller.
 */
size_t gqa_noalloc_scratch_bytes(void);
gqa_status gqa_decode_step_noalloc(const void *q, const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *lengths,
                                   const int32_t *slot_ids, float *out,
                                   int B, int Hq, int Hkv, int D, int R, int Smax, gqa_dtype dt,
                                   int32_t *d_status, void *stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int gqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
