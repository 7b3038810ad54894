/*
 * GQA decode-step oracle: plain float64 loops on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code with the CUDA library.
 *
 * What it computes, for every batch row b (all of it written out, no blocking,
 * fusion or reordering):
 *
 *   r   = slot_ids[b] if slot_ids are given, else b           (cache row)
 *   L   = lengths[b]                                         (append slot)
 *   cache[r][kvh][L] = k_new[b][kvh], v_new[b][kvh]          (bit copy, in place)
 *   for each query head h, with G = Hq / Hkv and kvh = floor(h / G):
 *     s_j = (q[b][h] . K[r][kvh][j]) / sqrt(D)        for j = 0 .. L
 *     m   = max_j s_j
 *     w_j = exp(s_j - m) / sum_i exp(s_i - m)
 *     o   = sum_j w_j V[r][kvh][j]
 *
 * The read-only attend (orc_attend_*) is the same computation with no new
 * token and no write: n = lengths[b] is the number of valid cached slots and
 * slots 0 .. n-1 are attended; the query may be float32 over a bfloat16 cache.
 *
 * The multi-token step (orc_decode_multi_*) appends the q_len[b] =
 * cu_q[b+1] - cu_q[b] new tokens of row b (packed rows cu_q[b] .. cu_q[b+1]-1
 * of q, k_new, v_new and out) at slots lengths[b] + i, and query token i
 * attends slots 0 .. lengths[b] + i (the causal bound); q_len = 1 everywhere
 * is the decode step.
 *
 * A quantised cache (kv dtype ORC_E4M3) holds OCP FP8 E4M3 bytes with one
 * float32 scale per cache head for K and one for V: K = k_scale[kvh] * K8,
 * V = v_scale[kvh] * V8. The query and the new keys / values keep their own
 * dtype (new_dtype); the append stores E4M3(float32(k_new) / k_scale), rounded
 * to nearest even and saturated to the largest finite value.
 *
 * Optional softmax modifiers (orc_mods, any entry point), with the query at
 * position L (the new token, or the last valid slot of the attend):
 *   window W > 0   slot j is attended only if L - W < j (the W positions up
 *                  to and including the query's own) ...
 *   kept prefix P  ... or if j < P (the sequence's first P keys);
 *   sink           one more logit per query head in the denominator:
 *                  w_j = exp(s_j) / (exp(sink_h) + sum_{i attended} exp(s_i)).
 *
 * Sources (web pages, by title and part):
 *  - "KV cache decode step" (tensortonic cs336-l10), problem statement: the new
 *    key and value take position S after the S cached positions, each KV head
 *    serves a contiguous group of G = Hq/Hkv query heads, and the softmax runs
 *    over every position including the new token, with the 1/sqrt(D) scale.
 *  - "Grouped-Query Decode Step" (tensortonic, JAX), statement and formula:
 *    query head h reads cache head floor(h/G); only the slots below the row's
 *    length get weight, stale slots get exactly zero; s_j = q.K_j/sqrt(D),
 *    w_j = e^{s_j} / sum e^{s_m}, o = sum w_j V_j; computed in float32 from
 *    bfloat16 caches (Requirements), here in float64.
 *  - "groupQueryAttention" (clika runtime), description: the in-place append,
 *    slot_ids as a row map on a [max_seqs, Hkv, max_seq, D] cache (entries in
 *    [0, max_seqs), no two rows sharing one), and the paged block table
 *    ([B, max_blocks], entries -1 or in [0, num_blocks), no repeats within a
 *    row, validated whole before any read, INVALID_ARGUMENT otherwise); a
 *    read-only attend (no key or value given) reads the cache and writes
 *    nothing ("use attention_over_cache").
 *  - "Grouped-Query Decode Step", Constraints: the query is float32 while the
 *    caches are float32 or bfloat16, and every length lies in [1, S]: this is
 *    the read-only attend's contract.
 *  - "groupQueryAttention", description: head_sink is a per-head virtual
 *    logit folded into the softmax denominator; kept_prefix keeps each
 *    sequence's first P keys attended beside the sliding window, a key is
 *    attended when it is inside the first P keys or inside the window (the
 *    window alone without P), and a negative P is refused. The packed
 *    (hidden-folded, [sum S, heads * head_dim]) q/k/v and the write offset of
 *    each row, cu_seqlens_k[b] - q_len[b], give the multi-token form.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - lengths[b] is the append slot (the number of tokens already cached), and
 *    slots 0 .. lengths[b] inclusive are attended: the first page's S per row.
 *  - dense: 0 <= lengths[b] <= Smax - 1. paged: 0 <= lengths[b] and
 *    lengths[b] < max_blocks * block_size, and the table entries covering
 *    slots 0 .. lengths[b] are not -1.
 *  - the window holds the W positions ending at the query's own (so W = 1
 *    attends the query's own key only); the sink is a logit in the same units
 *    as s_j (already scaled, not multiplied by 1/sqrt(D)); a kept prefix has
 *    no effect without a window; window < 0 is refused like a negative P.
 *  - quantised cache ("groupQueryAttention" names kScale / vScale and says
 *    nothing more): per-cache-head float32 scales, E4M3 bytes, dequantised
 *    value = scale * decoded byte; the new key / value is divided by the
 *    scale in float32 (round to nearest) and encoded round-to-nearest-even
 *    with saturation to +-448; NaN encodes to 0x7F.
 *  - multi-token: lengths[b] is the write offset (tokens already cached), so
 *    cu_seqlens_k[b] = lengths[b] + q_len[b]; cu_q[0] = 0, cu_q nondecreasing,
 *    cu_q[B] = T; 0 <= lengths[b] and lengths[b] + q_len[b] <= capacity; a
 *    row with q_len = 0 has nothing to do.
 *  - read-only attend: 1 <= lengths[b] <= Smax (dense) or
 *    <= max_blocks * block_size (paged, entries covering slots
 *    0 .. lengths[b]-1 not -1); zero valid slots has no softmax and is
 *    rejected like any other bad length.
 *  - subtracting the maximum before exp is the textbook rearrangement of the
 *    same quotient; it changes no value beyond rounding.
 *  - bfloat16 values are the upper 16 bits of an IEEE binary32; widening them
 *    to double is exact.
 */
#define _GNU_SOURCE
#include <limits.h>
#include <math.h>
#include <sched.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };
enum { ORC_OK = 0, ORC_INVALID_ARGUMENT = 1 };

/* Softmax modifiers and the scales of a quantised cache; a NULL orc_mods
 * pointer means none of them. */
typedef struct {
    const float *head_sink;         /* (Hq,) logits, or NULL: no sink          */
    int window;                     /* 0: no window; > 0: W                    */
    int kept_prefix;                /* P for every row (rows NULL), >= 0       */
    const int32_t *kept_prefix_rows;/* (B,) P per batch row, or NULL           */
    const float *k_scale, *v_scale; /* (Hkv,) E4M3 cache scales                */
    int new_dtype;                  /* E4M3 cache: dtype of q, k_new, v_new    */
} orc_mods;

/* ------------------------------------------------------------- E4M3 ----
 * OCP 8-bit floating point, E4M3: sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits; no infinities; S.1111.111 is NaN; exponent field 0 holds
 * the subnormals m/8 * 2^-6; the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t c)
{
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return (c & 0x80) ? -v : v;
}

/* Nearest E4M3 code to x, ties to the even code (mantissa bit 0 clear),
 * magnitudes at or above 448 saturated to 448, NaN to 0x7F. The finite
 * non-negative codes 0x00 .. 0x7E are increasing in value, so the nearest
 * one is found by a scan. */
uint8_t orc_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int lo = 0;
    while (lo < 0x7E && orc_e4m3_decode((uint8_t)(lo + 1)) <= a)
        ++lo;                              /* largest code with value <= a */
    if (orc_e4m3_decode((uint8_t)lo) == a)
        return sign | (uint8_t)lo;
    const int hi = lo + 1;
    const double dl = a - orc_e4m3_decode((uint8_t)lo), dh = orc_e4m3_decode((uint8_t)hi) - a;
    const int pick = dl < dh ? lo : (dh < dl ? hi : ((lo & 1) ? hi : lo));
    return sign | (uint8_t)pick;
}

/* One element of a float32 or bfloat16 array, widened exactly to double. */
static double elem(const void *base, size_t i, int dtype)
{
    if (dtype == ORC_F32) {
        return (double)((const float *)base)[i];
    }
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int usable_dtype(int dtype) { return dtype == ORC_F32 || dtype == ORC_BF16; }

static size_t esize(int dtype) { return dtype == ORC_F32 ? 4 : (dtype == ORC_E4M3 ? 1 : 2); }

static void copy_vec(void *dst, size_t dst_i, const void *src, size_t src_i, int D, int dtype)
{
    size_t es = esize(dtype);
    memcpy((char *)dst + dst_i * es, (const char *)src + src_i * es, (size_t)D * es);
}

/* ---------------------------------------------------------------- checks -- */

/* The highest slot a row touches: lengths[b] for the decode step (the append
 * slot), lengths[b] - 1 for the read-only attend (the last valid slot). */
static long long last_slot(const int32_t *lengths, int b, int attend)
{
    return (long long)lengths[b] - (attend ? 1 : 0);
}

/* Dense / slot_ids form: every touched slot in [0, Smax-1]; slot_ids in [0, R)
 * and pairwise distinct; without slot_ids the cache must hold a row per batch
 * row. */
static int validate_dense(const int32_t *lengths, const int32_t *slot_ids, int B, int R, int Smax,
                          int attend)
{
    if (B < 0 || R < 0 || Smax < 1)
        return ORC_INVALID_ARGUMENT;
    for (int b = 0; b < B; ++b)
        if (last_slot(lengths, b, attend) < 0 || last_slot(lengths, b, attend) > Smax - 1)
            return ORC_INVALID_ARGUMENT;
    if (!slot_ids)
        return B <= R ? ORC_OK : ORC_INVALID_ARGUMENT;
    for (int b = 0; b < B; ++b) {
        if (slot_ids[b] < 0 || slot_ids[b] >= R)
            return ORC_INVALID_ARGUMENT;
        for (int c = 0; c < b; ++c)
            if (slot_ids[c] == slot_ids[b])
                return ORC_INVALID_ARGUMENT;
    }
    return ORC_OK;
}

int orc_validate_dense(const int32_t *lengths, const int32_t *slot_ids, int B, int R, int Smax)
{
    return validate_dense(lengths, slot_ids, B, R, Smax, 0);
}

int orc_validate_attend_dense(const int32_t *lengths, const int32_t *slot_ids, int B, int R,
                              int Smax)
{
    return validate_dense(lengths, slot_ids, B, R, Smax, 1);
}

/* Paged form: every table entry is -1 or in [0, num_blocks); no block repeats
 * within a row; each touched slot fits the table and the entries that hold
 * slots 0 .. last touched slot are real blocks. */
static int validate_paged(const int32_t *lengths, const int32_t *block_table, int B,
                          int num_blocks, int block_size, int max_blocks, int attend)
{
    if (B < 0 || num_blocks < 1 || block_size < 1 || max_blocks < 1)
        return ORC_INVALID_ARGUMENT;
    for (int b = 0; b < B; ++b) {
        const int32_t *row = block_table + (size_t)b * max_blocks;
        for (int i = 0; i < max_blocks; ++i) {
            if (row[i] == -1)
                continue;
            if (row[i] < 0 || row[i] >= num_blocks)
                return ORC_INVALID_ARGUMENT;
            for (int k = 0; k < i; ++k)
                if (row[k] == row[i])
                    return ORC_INVALID_ARGUMENT;
        }
        long long last = last_slot(lengths, b, attend);
        if (last < 0 || last >= (long long)max_blocks * block_size)
            return ORC_INVALID_ARGUMENT;
        for (long long i = 0; i <= last / block_size; ++i)
            if (row[i] == -1)
                return ORC_INVALID_ARGUMENT;
    }
    return ORC_OK;
}

int orc_validate_paged(const int32_t *lengths, const int32_t *block_table, int B,
                       int num_blocks, int block_size, int max_blocks)
{
    return validate_paged(lengths, block_table, B, num_blocks, block_size, max_blocks, 0);
}

int orc_validate_attend_paged(const int32_t *lengths, const int32_t *block_table, int B,
                              int num_blocks, int block_size, int max_blocks)
{
    return validate_paged(lengths, block_table, B, num_blocks, block_size, max_blocks, 1);
}

/* ------------------------------------------------------------ addressing -- */

/* Where slot s of cache head kvh of batch row b lives, as an element index of
 * the first of its D values. */
typedef struct {
    int paged;
    /* dense */
    const int32_t *slot_ids;
    int Hkv, D, Smax;
    /* paged */
    const int32_t *block_table;
    int block_size, max_blocks;
} layout;

static size_t slot_index(const layout *lay, int b, int kvh, int s)
{
    if (!lay->paged) {
        size_t r = lay->slot_ids ? (size_t)lay->slot_ids[b] : (size_t)b;
        return ((r * lay->Hkv + kvh) * lay->Smax + s) * lay->D;
    }
    size_t blk = (size_t)lay->block_table[(size_t)b * lay->max_blocks + s / lay->block_size];
    return ((blk * lay->Hkv + kvh) * lay->block_size + (size_t)(s % lay->block_size)) * lay->D;
}

/* ----------------------------------------------------------------- step -- */

typedef struct {
    int q_dtype, kv_dtype;   /* the decode step has one dtype for all */
    int new_dtype;           /* k_new / v_new (differs from kv_dtype for an E4M3 cache) */
    int attend;              /* 1: read-only attend over slots 0 .. lengths[b]-1 */
    const void *q, *k_new, *v_new;
    void *k_cache, *v_cache;
    const int32_t *lengths;
    layout lay;
    int B, Hq, Hkv, D;
    int do_append;
    double *out;       /* (B, Hq, D); multi-token: (T, Hq, D) */
    const orc_mods *mods;  /* NULL: plain softmax */
    const int32_t *cu_q;   /* multi-token: (B + 1) token offsets, else NULL */
    const int32_t *rows; /* batch rows to compute */
    int nrows;
    /* work distribution over (row, kvh) pairs */
    int next;
    pthread_mutex_t mu;
} job;

/* Whether slot j (0 <= j <= L, the query at position L) of batch row b takes
 * part in the softmax: always without a window; with one, inside the window
 * or the kept prefix. */
static int attended(const job *J, int b, int L, int j)
{
    const orc_mods *M = J->mods;
    if (!M || M->window <= 0)
        return 1;
    if (j > L - M->window)
        return 1;
    const int P = M->kept_prefix_rows ? M->kept_prefix_rows[b] : M->kept_prefix;
    return j < P;
}

static int mods_ok(const orc_mods *M, int B)
{
    if (!M)
        return 1;
    if ((M->k_scale == NULL) != (M->v_scale == NULL))
        return 0;
    if (M->window < 0 || (!M->kept_prefix_rows && M->kept_prefix < 0))
        return 0;
    if (M->kept_prefix_rows)
        for (int b = 0; b < B; ++b)
            if (M->kept_prefix_rows[b] < 0)
                return 0;
    return 1;
}

/* The job's dtypes: q_dtype for the query; the cache's kv_dtype; the new
 * keys / values share the cache dtype, except over an E4M3 cache, which takes
 * their dtype and its scales from mods. 0 when the combination is invalid. */
static int setup_dtypes(job *J, int q_dtype, int kv_dtype, const orc_mods *mods)
{
    J->q_dtype = q_dtype;
    J->kv_dtype = kv_dtype;
    J->new_dtype = kv_dtype;
    if (kv_dtype == ORC_E4M3) {
        if (!mods || !mods->k_scale || !usable_dtype(mods->new_dtype))
            return 0;
        J->new_dtype = mods->new_dtype;
    } else if (!usable_dtype(kv_dtype)) {
        return 0;
    }
    return usable_dtype(q_dtype);
}

/* Element d of slot j of a cache (the dequantised value for E4M3). */
static double cache_elem(const job *J, const void *cache, const float *scale, size_t i, int kvh)
{
    if (J->kv_dtype == ORC_E4M3)
        return (double)scale[kvh] * orc_e4m3_decode(((const uint8_t *)cache)[i]);
    return elem(cache, i, J->kv_dtype);
}

/* The value an append stores for new element x of cache head kvh, as the
 * cache then reads it back. */
static double stored_new(const job *J, const void *news, const float *scale, size_t i, int kvh)
{
    const double x = elem(news, i, J->new_dtype);
    if (J->kv_dtype != ORC_E4M3)
        return x;
    const float y = (float)x / scale[kvh];     /* float32 division, round to nearest */
    return (double)scale[kvh] * orc_e4m3_decode(orc_e4m3_encode(y));
}

/* Append of D new elements into a cache slot. */
static void append_vec(const job *J, void *cache, size_t dst, const void *news, size_t src,
                       const float *scale, int kvh)
{
    if (J->kv_dtype != ORC_E4M3) {
        copy_vec(cache, dst, news, src, J->D, J->kv_dtype);
        return;
    }
    for (int d = 0; d < J->D; ++d) {
        const float y = (float)elem(news, src + d, J->new_dtype) / scale[kvh];
        ((uint8_t *)cache)[dst + d] = orc_e4m3_encode(y);
    }
}

/* Element index of the new key / value of token `tok`, cache head kvh. */
static size_t new_index(const job *J, int tok, int kvh)
{
    return ((size_t)tok * J->Hkv + kvh) * J->D;
}

/* The G query heads of token `tok` (its rows of q and out) over the attended
 * slots 0 .. L of (batch row b, cache head kvh). Slots at or beyond first_new
 * are read from the new keys / values of tokens new_tok0, new_tok0 + 1, ...
 * (the tokens a step without append did not write into the cache). */
static void attend_heads(job *J, int b, int kvh, int L, int tok, int first_new, int new_tok0)
{
    const int D = J->D, G = J->Hq / J->Hkv;
    const float *KS = J->mods ? J->mods->k_scale : NULL, *VS = J->mods ? J->mods->v_scale : NULL;
    double *s = (double *)malloc(sizeof(double) * (size_t)(L + 1));
    for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;           /* floor(h / G) == kvh */
        const size_t q_i = ((size_t)tok * J->Hq + h) * D;

        /* scores over slots 0 .. L */
        for (int j = 0; j <= L; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) {
                double kd = (j >= first_new)
                                ? stored_new(J, J->k_new, KS, new_index(J, new_tok0 + j - first_new, kvh) + d, kvh)
                                : cache_elem(J, J->k_cache, KS, slot_index(&J->lay, b, kvh, j) + d, kvh);
                dot += elem(J->q, q_i + d, J->q_dtype) * kd;
            }
            s[j] = dot / sqrt((double)D);
        }

        /* softmax over the attended slots (the valid ones, cut to the window
         * and the kept prefix when given), the sink as one more logit */
        const float *sink = J->mods ? J->mods->head_sink : NULL;
        double m = -INFINITY;
        for (int j = 0; j <= L; ++j)
            if (attended(J, b, L, j) && s[j] > m)
                m = s[j];
        if (sink && (double)sink[h] > m)
            m = (double)sink[h];
        double Z = sink ? exp((double)sink[h] - m) : 0.0;
        for (int j = 0; j <= L; ++j)
            if (attended(J, b, L, j))
                Z += exp(s[j] - m);

        /* weighted sum of values */
        double *o = J->out + q_i;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int j = 0; j <= L; ++j) {
            if (!attended(J, b, L, j))
                continue;
            double w = exp(s[j] - m) / Z;
            for (int d = 0; d < D; ++d) {
                double vd = (j >= first_new)
                                ? stored_new(J, J->v_new, VS, new_index(J, new_tok0 + j - first_new, kvh) + d, kvh)
                                : cache_elem(J, J->v_cache, VS, slot_index(&J->lay, b, kvh, j) + d, kvh);
                o[d] += w * vd;
            }
        }
    }
    free(s);
}

/* One (batch row, cache head) pair: append (decode step), then the G query
 * heads over the attended slots 0 .. L. */
static void one_pair(job *J, int b, int kvh)
{
    const float *KS = J->mods ? J->mods->k_scale : NULL, *VS = J->mods ? J->mods->v_scale : NULL;
    if (J->cu_q) {
        /* multi-token: tokens t0 .. t0 + nq - 1 take slots Lb .. Lb + nq - 1,
         * and token i attends slots 0 .. Lb + i */
        const int t0 = J->cu_q[b], nq = J->cu_q[b + 1] - t0, Lb = J->lengths[b];
        if (J->do_append)
            for (int i = 0; i < nq; ++i) {
                size_t dst = slot_index(&J->lay, b, kvh, Lb + i);
                append_vec(J, J->k_cache, dst, J->k_new, new_index(J, t0 + i, kvh), KS, kvh);
                append_vec(J, J->v_cache, dst, J->v_new, new_index(J, t0 + i, kvh), VS, kvh);
            }
        for (int i = 0; i < nq; ++i)
            attend_heads(J, b, kvh, Lb + i, t0 + i, J->do_append ? INT_MAX : Lb, t0);
        return;
    }
    const int L = J->attend ? J->lengths[b] - 1 : J->lengths[b];   /* last attended slot */
    const int from_new = !J->attend && !J->do_append;  /* slot L read from k_new / v_new */

    if (!J->attend && J->do_append) {
        size_t dst = slot_index(&J->lay, b, kvh, L);
        append_vec(J, J->k_cache, dst, J->k_new, new_index(J, b, kvh), KS, kvh);
        append_vec(J, J->v_cache, dst, J->v_new, new_index(J, b, kvh), VS, kvh);
    }
    attend_heads(J, b, kvh, L, b, from_new ? L : INT_MAX, b);
}

static void *worker(void *arg)
{
    job *J = (job *)arg;
    const int total = J->nrows * J->Hkv;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int t = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (t >= total)
            break;
        one_pair(J, J->rows[t / J->Hkv], t % J->Hkv);
    }
    return NULL;
}

static int run(job *J, int nthreads)
{
    int *all = NULL;
    if (!J->rows) {
        all = (int *)malloc(sizeof(int) * (size_t)(J->B > 0 ? J->B : 1));
        for (int b = 0; b < J->B; ++b)
            all[b] = b;
        J->rows = all;
        J->nrows = J->B;
    }
    if (nthreads < 1)
        nthreads = 1;
    J->next = 0;
    pthread_mutex_init(&J->mu, NULL);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i)
        pthread_create(&tid[i], NULL, worker, J);
    for (int i = 0; i < nthreads; ++i)
        pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&J->mu);
    free(all);
    return nthreads;
}

static int usable_shape(int B, int Hq, int Hkv, int D)
{
    return B >= 0 && Hq >= 1 && Hkv >= 1 && D >= 1 && Hq % Hkv == 0;
}

/* Dense or slot_ids cache (R, Hkv, Smax, D). rows/nrows pick the batch rows to
 * compute (NULL: all); out rows that are not picked are left untouched.
 * do_append = 0 computes the same output without writing the cache (slot L
 * then reads k_new / v_new, which is what the append would have put there).
 * Returns ORC_OK or ORC_INVALID_ARGUMENT; *threads_used gets the thread count. */
int orc_decode_dense(int dtype, const void *q, const void *k_new, const void *v_new,
                     void *k_cache, void *v_cache, const int32_t *lengths, const int32_t *slot_ids,
                     int B, int Hq, int Hkv, int D, int R, int Smax,
                     const int32_t *rows, int nrows, int do_append, double *out,
                     const orc_mods *mods, int nthreads, int *threads_used)
{
    if (!usable_shape(B, Hq, Hkv, D) || !mods_ok(mods, B))
        return ORC_INVALID_ARGUMENT;
    if (orc_validate_dense(lengths, slot_ids, B, R, Smax) != ORC_OK)
        return ORC_INVALID_ARGUMENT;
    job J;
    memset(&J, 0, sizeof J);
    if (!setup_dtypes(&J, dtype == ORC_E4M3 && mods ? mods->new_dtype : dtype, dtype, mods))
        return ORC_INVALID_ARGUMENT;
    J.q = q; J.k_new = k_new; J.v_new = v_new;
    J.k_cache = k_cache; J.v_cache = v_cache;
    J.lengths = lengths;
    J.lay.paged = 0; J.lay.slot_ids = slot_ids;
    J.lay.Hkv = Hkv; J.lay.D = D; J.lay.Smax = Smax;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.do_append = do_append;
    J.out = out;
    J.mods = mods;
    J.rows = (const int32_t *)rows; J.nrows = nrows;
    int n = run(&J, nthreads);
    if (threads_used)
        *threads_used = n;
    return ORC_OK;
}

/* Paged cache: blocks (num_blocks, Hkv, block_size, D), block table
 * (B, max_blocks). Same contract as orc_decode_dense otherwise. */
int orc_decode_paged(int dtype, const void *q, const void *k_new, const void *v_new,
                     void *k_blocks, void *v_blocks, const int32_t *block_table,
                     const int32_t *lengths, int B, int Hq, int Hkv, int D,
                     int num_blocks, int block_size, int max_blocks,
                     const int32_t *rows, int nrows, int do_append, double *out,
                     const orc_mods *mods, int nthreads, int *threads_used)
{
    if (!usable_shape(B, Hq, Hkv, D) || !mods_ok(mods, B))
        return ORC_INVALID_ARGUMENT;
    if (orc_validate_paged(lengths, block_table, B, num_blocks, block_size, max_blocks) != ORC_OK)
        return ORC_INVALID_ARGUMENT;
    job J;
    memset(&J, 0, sizeof J);
    if (!setup_dtypes(&J, dtype == ORC_E4M3 && mods ? mods->new_dtype : dtype, dtype, mods))
        return ORC_INVALID_ARGUMENT;
    J.q = q; J.k_new = k_new; J.v_new = v_new;
    J.k_cache = k_blocks; J.v_cache = v_blocks;
    J.lengths = lengths;
    J.lay.paged = 1; J.lay.block_table = block_table;
    J.lay.Hkv = Hkv; J.lay.D = D;
    J.lay.block_size = block_size; J.lay.max_blocks = max_blocks;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.do_append = do_append;
    J.out = out;
    J.mods = mods;
    J.rows = (const int32_t *)rows; J.nrows = nrows;
    int n = run(&J, nthreads);
    if (threads_used)
        *threads_used = n;
    return ORC_OK;
}


/* Read-only attend on a dense or slot_ids cache (R, Hkv, Smax, D): slots
 * 0 .. lengths[b]-1 of the row, nothing written. q_dtype and kv_dtype are
 * each ORC_F32 or ORC_BF16. rows/nrows as in orc_decode_dense. */
int orc_attend_dense(int q_dtype, int kv_dtype, const void *q, const void *k_cache,
                     const void *v_cache, const int32_t *lengths, const int32_t *slot_ids,
                     int B, int Hq, int Hkv, int D, int R, int Smax,
                     const int32_t *rows, int nrows, double *out, const orc_mods *mods,
                     int nthreads, int *threads_used)
{
    if (!usable_shape(B, Hq, Hkv, D) || !mods_ok(mods, B))
        return ORC_INVALID_ARGUMENT;
    if (orc_validate_attend_dense(lengths, slot_ids, B, R, Smax) != ORC_OK)
        return ORC_INVALID_ARGUMENT;
    job J;
    memset(&J, 0, sizeof J);
    if (!setup_dtypes(&J, q_dtype, kv_dtype, mods))
        return ORC_INVALID_ARGUMENT;
    J.attend = 1;
    J.q = q;
    J.k_cache = (void *)k_cache; J.v_cache = (void *)v_cache;   /* only read */
    J.lengths = lengths;
    J.lay.paged = 0; J.lay.slot_ids = slot_ids;
    J.lay.Hkv = Hkv; J.lay.D = D; J.lay.Smax = Smax;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.out = out;
    J.mods = mods;
    J.rows = (const int32_t *)rows; J.nrows = nrows;
    int n = run(&J, nthreads);
    if (threads_used)
        *threads_used = n;
    return ORC_OK;
}

/* Read-only attend on a paged cache; same contract as orc_attend_dense. */
int orc_attend_paged(int q_dtype, int kv_dtype, const void *q, const void *k_blocks,
                     const void *v_blocks, const int32_t *block_table, const int32_t *lengths,
                     int B, int Hq, int Hkv, int D, int num_blocks, int block_size, int max_blocks,
                     const int32_t *rows, int nrows, double *out, const orc_mods *mods,
                     int nthreads, int *threads_used)
{
    if (!usable_shape(B, Hq, Hkv, D) || !mods_ok(mods, B))
        return ORC_INVALID_ARGUMENT;
    if (orc_validate_attend_paged(lengths, block_table, B, num_blocks, block_size, max_blocks)
        != ORC_OK)
        return ORC_INVALID_ARGUMENT;
    job J;
    memset(&J, 0, sizeof J);
    if (!setup_dtypes(&J, q_dtype, kv_dtype, mods))
        return ORC_INVALID_ARGUMENT;
    J.attend = 1;
    J.q = q;
    J.k_cache = (void *)k_blocks; J.v_cache = (void *)v_blocks;
    J.lengths = lengths;
    J.lay.paged = 1; J.lay.block_table = block_table;
    J.lay.Hkv = Hkv; J.lay.D = D;
    J.lay.block_size = block_size; J.lay.max_blocks = max_blocks;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.out = out;
    J.mods = mods;
    J.rows = (const int32_t *)rows; J.nrows = nrows;
    int n = run(&J, nthreads);
    if (threads_used)
        *threads_used = n;
    return ORC_OK;
}

/* Multi-token checks: cu_q[0] = 0, nondecreasing, cu_q[B] = T; every row
 * 0 <= lengths[b] and lengths[b] + q_len[b] <= capacity. */
static int validate_cu_q(const int32_t *cu_q, int B, int T)
{
    if (B < 0 || T < 0 || cu_q[0] != 0 || cu_q[B] != T)
        return ORC_INVALID_ARGUMENT;
    for (int b = 0; b < B; ++b)
        if (cu_q[b + 1] < cu_q[b])
            return ORC_INVALID_ARGUMENT;
    return ORC_OK;
}

int orc_validate_multi_dense(const int32_t *lengths, const int32_t *cu_q, const int32_t *slot_ids,
                             int B, int T, int R, int Smax)
{
    if (validate_cu_q(cu_q, B, T) != ORC_OK)
        return ORC_INVALID_ARGUMENT;
    for (int b = 0; b < B; ++b)
        if (lengths[b] < 0 || (long long)lengths[b] + (cu_q[b + 1] - cu_q[b]) > Smax)
            return ORC_INVALID_ARGUMENT;
    /* the slot_ids / row rules of the decode step, with the lengths checked above */
    int32_t *zero = (int32_t *)calloc((size_t)(B > 0 ? B : 1), sizeof(int32_t));
    int st = orc_validate_dense(zero, slot_ids, B, R, Smax);
    free(zero);
    return st;
}

int orc_validate_multi_paged(const int32_t *lengths, const int32_t *cu_q, const int32_t *block_table,
                             int B, int T, int num_blocks, int block_size, int max_blocks)
{
    if (validate_cu_q(cu_q, B, T) != ORC_OK)
        return ORC_INVALID_ARGUMENT;
    /* the table rules of the decode step, with the last touched slot
     * lengths[b] + q_len[b] - 1 (rows without tokens touch none) */
    int32_t *last = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    for (int b = 0; b < B; ++b) {
        const long long l = (long long)lengths[b] + (cu_q[b + 1] - cu_q[b]) - 1;
        last[b] = lengths[b] < 0 ? -1 : (l < 0 ? 0 : (l > INT_MAX ? INT_MAX : (int32_t)l));
    }
    int st = orc_validate_paged(last, block_table, B, num_blocks, block_size, max_blocks);
    free(last);
    return st;
}

/* Multi-token step on a dense or slot_ids cache. q (T, Hq, D), k_new / v_new
 * (T, Hkv, D), out (T, Hq, D); cu_q (B + 1). do_append = 0 computes the same
 * outputs without writing the cache. */
int orc_decode_multi_dense(int dtype, const void *q, const void *k_new, const void *v_new,
                           void *k_cache, void *v_cache, const int32_t *lengths, const int32_t *cu_q,
                           const int32_t *slot_ids, int B, int T, int Hq, int Hkv, int D, int R,
                           int Smax, int do_append, double *out, const orc_mods *mods, int nthreads,
                           int *threads_used)
{
    if (!usable_shape(B, Hq, Hkv, D) || !mods_ok(mods, B))
        return ORC_INVALID_ARGUMENT;
    if (orc_validate_multi_dense(lengths, cu_q, slot_ids, B, T, R, Smax) != ORC_OK)
        return ORC_INVALID_ARGUMENT;
    job J;
    memset(&J, 0, sizeof J);
    if (!setup_dtypes(&J, dtype == ORC_E4M3 && mods ? mods->new_dtype : dtype, dtype, mods))
        return ORC_INVALID_ARGUMENT;
    J.q = q; J.k_new = k_new; J.v_new = v_new;
    J.k_cache = k_cache; J.v_cache = v_cache;
    J.lengths = lengths;
    J.cu_q = cu_q;
    J.lay.paged = 0; J.lay.slot_ids = slot_ids;
    J.lay.Hkv = Hkv; J.lay.D = D; J.lay.Smax = Smax;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.do_append = do_append;
    J.out = out;
    J.mods = mods;
    int n = run(&J, nthreads);
    if (threads_used)
        *threads_used = n;
    return ORC_OK;
}

/* Multi-token step on a paged cache; same contract otherwise. */
int orc_decode_multi_paged(int dtype, const void *q, const void *k_new, const void *v_new,
                           void *k_blocks, void *v_blocks, const int32_t *block_table,
                           const int32_t *lengths, const int32_t *cu_q, int B, int T, int Hq, int Hkv,
                           int D, int num_blocks, int block_size, int max_blocks, int do_append,
                           double *out, const orc_mods *mods, int nthreads, int *threads_used)
{
    if (!usable_shape(B, Hq, Hkv, D) || !mods_ok(mods, B))
        return ORC_INVALID_ARGUMENT;
    if (orc_validate_multi_paged(lengths, cu_q, block_table, B, T, num_blocks, block_size, max_blocks) !=
        ORC_OK)
        return ORC_INVALID_ARGUMENT;
    job J;
    memset(&J, 0, sizeof J);
    if (!setup_dtypes(&J, dtype == ORC_E4M3 && mods ? mods->new_dtype : dtype, dtype, mods))
        return ORC_INVALID_ARGUMENT;
    J.q = q; J.k_new = k_new; J.v_new = v_new;
    J.k_cache = k_blocks; J.v_cache = v_blocks;
    J.lengths = lengths;
    J.cu_q = cu_q;
    J.lay.paged = 1; J.lay.block_table = block_table;
    J.lay.Hkv = Hkv; J.lay.D = D;
    J.lay.block_size = block_size; J.lay.max_blocks = max_blocks;
    J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.do_append = do_append;
    J.out = out;
    J.mods = mods;
    int n = run(&J, nthreads);
    if (threads_used)
        *threads_used = n;
    return ORC_OK;
}

/* Cores this process may run on (the default thread count). */
int orc_default_threads(void)
{
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof set, &set) == 0 && CPU_COUNT(&set) > 0)
        return CPU_COUNT(&set);
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
