/*
 * Float64 reference ("oracle") for paged grouped-query attention over a
 * block-arena KV cache.  TEST INFRASTRUCTURE ONLY: tests, the smoke check and
 * the benchmark's CPU-baseline leg call it; the library never does.
 *
 * What it follows (pages "Building Kshipra", part 3, kshipra-3):
 *  - section 1 "Block-Arena KV Cache": KV rows live in fixed-size blocks of
 *    one preallocated arena; a sequence's logical block j is the physical
 *    block block_tables[s][j]; a token at position p sits in slot p % bs of
 *    logical block p / bs.
 *  - section 4 "Chunked Prefill": RoPE at absolute positions (a chunk after
 *    P cached tokens starts at position P); the causal mask lets a query at
 *    position p see keys 0..p of its own sequence; the block-wise online
 *    softmax is stated to equal dense masked attention.  The oracle computes
 *    that dense definition directly: explicit mask, row maximum, exponentials,
 *    normalisation, weighted sum of V, all in float64.
 *  - The attention reads its keys and values the way section 1 lays them out:
 *    every raw K/V row is first written into the oracle's own arena (every
 *    slot starts as a NaN pattern) at slot j % bs of physical block
 *    block_tables[s][j / bs], then gathered back through the same tables; a
 *    gathered NaN, a block id outside the arena, or a slot written twice with
 *    different bits (two sequences' rows aliased) is an error.  A second route
 *    reads the rows in logical order, for cross-checking the first.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - RoPE pairs element i with i + d/2 ("rotate half"), frequency
 *    theta^(-2i/d), angle = position * frequency, float64 libm cos/sin.
 *  - Attention uses the exact float64 rotation.  The rotated key stored in the
 *    arena (and the stored q_rot) is the float32 rotation: cos/sin rounded to
 *    float32, separately rounded float32 products, one float32 add or
 *    subtract (no fused multiply-add), then one rounding (nearest, ties to
 *    even) to the storage type.
 *  - scale is a caller input (1/sqrt(d) in every workload).
 *
 * Nothing here is shared with the CUDA library: conversions, RoPE and the
 * attention loop are written out independently.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* ---------------------------------------------------------------------- */
/* IEEE bit conversions                                                    */
/* ---------------------------------------------------------------------- */

static double small_float_to_f64(uint16_t h, int ebits, int mbits) {
    int sign = (h >> (ebits + mbits)) & 1;
    int e = (h >> mbits) & ((1 << ebits) - 1);
    int f = h & ((1 << mbits) - 1);
    int bias = (1 << (ebits - 1)) - 1;
    double v;
    if (e == (1 << ebits) - 1)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, 1 - bias - mbits);
    else
        v = ldexp((double)(f | (1 << mbits)), e - bias - mbits);
    return sign ? -v : v;
}

/* Round a double to a small binary float (ebits exponent bits, mbits
 * fraction bits) in one step: nearest, ties to even; overflow to infinity;
 * gradual underflow to subnormals. */
static uint16_t f64_to_small_float(double x, int ebits, int mbits) {
    uint64_t b;
    memcpy(&b, &x, sizeof b);
    uint16_t sign = (uint16_t)((b >> 63) << (ebits + mbits));
    uint64_t ab = b & 0x7FFFFFFFFFFFFFFFull;
    int emax_field = (1 << ebits) - 1;
    int bias = (1 << (ebits - 1)) - 1;
    if (ab > 0x7FF0000000000000ull) /* NaN -> quiet NaN */
        return (uint16_t)(sign | (emax_field << mbits) | (1u << (mbits - 1)));
    if (ab == 0x7FF0000000000000ull) /* infinity */
        return (uint16_t)(sign | (emax_field << mbits));
    int e = (int)(ab >> 52);
    if (e == 0) /* zero or double subnormal: far below any target subnormal */
        return sign;
    uint64_t m = (ab & ((1ull << 52) - 1)) | (1ull << 52); /* 53-bit significand */
    int te = (e - 1023) + bias;                             /* target biased exponent */
    if (te >= emax_field)
        return (uint16_t)(sign | (emax_field << mbits));
    int shift;
    int normal = te >= 1;
    if (normal)
        shift = 52 - mbits;
    else
        shift = 52 - mbits + (1 - te);
    if (shift >= 54) /* below half the smallest subnormal */
        return sign;
    uint64_t kept = m >> shift;
    uint64_t rem = m & ((1ull << shift) - 1);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (kept & 1)))
        kept++;
    uint64_t bits;
    if (normal) /* kept carries the implicit bit; a carry bumps the exponent */
        bits = ((uint64_t)(te - 1) << mbits) + kept;
    else /* subnormal; kept == 2^mbits is the smallest normal */
        bits = kept;
    return (uint16_t)(sign | bits);
}

double oracle_f16_to_f64(uint16_t h) { return small_float_to_f64(h, 5, 10); }
double oracle_bf16_to_f64(uint16_t h) { return small_float_to_f64(h, 8, 7); }
uint16_t oracle_f64_to_f16(double x) { return f64_to_small_float(x, 5, 10); }
uint16_t oracle_f64_to_bf16(double x) { return f64_to_small_float(x, 8, 7); }

static double to_f64(uint16_t h, int dtype) {
    return dtype == ORACLE_BF16 ? oracle_bf16_to_f64(h) : oracle_f16_to_f64(h);
}

static uint16_t from_f64(double x, int dtype) {
    return dtype == ORACLE_BF16 ? oracle_f64_to_bf16(x) : oracle_f64_to_f16(x);
}

/* Bulk helpers for tests (exhaustive and random checks). */
void oracle_decode_bits(const uint16_t* in, double* out, long n, int dtype) {
    for (long i = 0; i < n; ++i) out[i] = to_f64(in[i], dtype);
}

void oracle_encode_bits(const double* in, uint16_t* out, long n, int dtype) {
    for (long i = 0; i < n; ++i) out[i] = from_f64(in[i], dtype);
}

/* ---------------------------------------------------------------------- */
/* RoPE (section 4: absolute positions)                                    */
/* ---------------------------------------------------------------------- */

/* cos and sin of position * theta^(-2i/d) for pair i of a d-wide head. */
static void rope_angle(long pos, int i, int d, double theta, double* c, double* s) {
    double freq = pow(theta, -2.0 * (double)i / (double)d);
    double ang = (double)pos * freq;
    *c = cos(ang);
    *s = sin(ang);
}

/* Table [max_pos][d/2][2] of (cos, sin). */
int oracle_rope_table(double* out, int max_pos, int d, double theta) {
    if (!out || max_pos < 0 || d <= 0 || (d & 1)) return 1;
    for (long p = 0; p < max_pos; ++p)
        for (int i = 0; i < d / 2; ++i)
            rope_angle(p, i, d, theta, &out[(p * (d / 2) + i) * 2], &out[(p * (d / 2) + i) * 2 + 1]);
    return 0;
}

/* Rotate one head row x[d] (float64) at position pos into y[d]:
 *   y_i       = x_i * c - x_{i+d/2} * s
 *   y_{i+d/2} = x_{i+d/2} * c + x_i * s
 * Products are separate roundings, then one add/subtract (built without
 * floating-point contraction). */
static void rope_row(const double* x, double* y, long pos, int d, double theta) {
    int h = d / 2;
    for (int i = 0; i < h; ++i) {
        double c, s;
        rope_angle(pos, i, d, theta, &c, &s);
        double a = x[i], b = x[i + h];
        double ac = a * c, bs = b * s, bc = b * c, as = a * s;
        y[i] = ac - bs;
        y[i + h] = bc + as;
    }
}

/* The stored rotation (arena keys and q_rot): cos and sin from the float64
 * angle rounded once to float32, the pair rotated with separately rounded
 * float32 products and one float32 add/subtract (built without contraction),
 * then rounded once to the storage type by the caller. */
static void rope_row_f32(const float* x, float* y, long pos, int d, double theta) {
    int h = d / 2;
    for (int i = 0; i < h; ++i) {
        double c, s;
        rope_angle(pos, i, d, theta, &c, &s);
        float cf = (float)c, sf = (float)s;
        float a = x[i], b = x[i + h];
        float ac = a * cf, bs = b * sf, bc = b * cf, as = a * sf;
        y[i] = ac - bs;
        y[i + h] = bc + as;
    }
}

/* Expected bits of rotated rows: rows[n][H][d] at positions pos[n], rounded
 * once to the storage type.  Used for q_rot and for the rotated keys. */
int oracle_rope_rows(const uint16_t* rows, uint16_t* out, const int32_t* pos, long n, int H, int d,
                     double theta, int dtype) {
    if (d <= 0 || (d & 1) || d > 1024) return 1;
    float x[1024], y[1024];
    for (long t = 0; t < n; ++t)
        for (int hh = 0; hh < H; ++hh) {
            const uint16_t* r = rows + ((size_t)t * H + hh) * d;
            for (int i = 0; i < d; ++i) x[i] = (float)to_f64(r[i], dtype);
            rope_row_f32(x, y, pos[t], d, theta);
            uint16_t* o = out + ((size_t)t * H + hh) * d;
            for (int i = 0; i < d; ++i) o[i] = from_f64((double)y[i], dtype);
        }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Arena image (section 1: fixed-size blocks, block tables)                */
/* ---------------------------------------------------------------------- */

/* Expected arena contents after appending rows k_rows/v_rows[T][Hkv][d] of
 * the sequences described by query_start_loc[S+1] at positions[T].
 * Arena layout: [num_blocks][Hkv][bs][d].  The caller fills both arenas with
 * its sentinel first; slots no row maps to keep it.  Returns 0, or 2 when a
 * row's block-table entry is outside [0, num_blocks). */
int oracle_arena_image(uint16_t* k_arena, uint16_t* v_arena, const uint16_t* k_rows, const uint16_t* v_rows,
                       const int32_t* query_start_loc, const int32_t* positions, int num_seqs,
                       const int32_t* block_tables, int max_blocks_per_seq, int num_blocks, int Hkv, int bs,
                       int d, double theta, int dtype) {
    if (d <= 0 || (d & 1) || d > 1024) return 1;
    float x[1024], y[1024];
    for (int s = 0; s < num_seqs; ++s)
        for (int t = query_start_loc[s]; t < query_start_loc[s + 1]; ++t) {
            long p = positions[t];
            if (p < 0 || p / bs >= max_blocks_per_seq) return 2;
            int blk = block_tables[(size_t)s * max_blocks_per_seq + p / bs];
            int slot = (int)(p % bs);
            if (blk < 0 || blk >= num_blocks) return 2;
            for (int h = 0; h < Hkv; ++h) {
                size_t src = ((size_t)t * Hkv + h) * d;
                size_t dst = (((size_t)blk * Hkv + h) * bs + slot) * d;
                for (int i = 0; i < d; ++i) x[i] = (float)to_f64(k_rows[src + i], dtype);
                rope_row_f32(x, y, p, d, theta);
                for (int i = 0; i < d; ++i) k_arena[dst + i] = from_f64((double)y[i], dtype);
                memcpy(v_arena + dst, v_rows + src, (size_t)d * sizeof(uint16_t));
            }
        }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Dense masked softmax attention (section 4), float64                     */
/* ---------------------------------------------------------------------- */

typedef struct {
    double* out;                 /* [n_out][Hq][d] */
    const int32_t* out_tokens;   /* [n_out] token index of each output row */
    int n_out;
    const uint16_t* q;           /* [T][Hq][d] raw (unrotated) queries */
    const uint16_t* k_all;       /* [sum ctx][Hkv][d] raw keys, logical order */
    const uint16_t* v_all;
    const int64_t* kv_start;     /* [S+1] first row of each sequence in k_all/v_all */
    const int32_t* qsl;          /* [S+1] query_start_loc */
    const int32_t* positions;    /* [T] */
    const int32_t* context_lens; /* [S] */
    /* the oracle's own arena [num_blocks][Hkv][bs][d] (raw bits) and the
     * tables that address it; NULL arena: read k_all/v_all in logical order */
    const uint16_t* arena_k;
    const uint16_t* arena_v;
    const int32_t* block_tables; /* [S][max_blocks] */
    int max_blocks, bs, num_blocks;
    int S, Hq, Hkv, d, dtype;
    double theta, scale;
    int* task_seq;               /* tasks are (sequence, kv head) pairs */
    int* task_head;
    int n_tasks;
    int next_task;               /* shared counter */
    int status;
} attn_job;

static int seq_of_token(const int32_t* qsl, int S, int t) {
    for (int s = 0; s < S; ++s)
        if (t >= qsl[s] && t < qsl[s + 1]) return s;
    return -1;
}

static void attention_task(attn_job* J, int s, int g) {
    int d = J->d, Hq = J->Hq, Hkv = J->Hkv, G = Hq / Hkv;
    long ctx = J->context_lens[s];
    double* K = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * d);
    double* V = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * d);
    double* w = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
    char* visible = (char*)malloc((size_t)(ctx > 0 ? ctx : 1));
    double x[1024], qr[1024];
    if (!K || !V || !w || !visible) {
        J->status = 3;
        free(K); free(V); free(w); free(visible);
        return;
    }
    /* rotated keys and values of this (sequence, kv head), every position:
     * gathered from the arena through the block table (section 1), or read
     * in logical order on the cross-check route */
    for (long j = 0; j < ctx; ++j) {
        const uint16_t *kr, *vr;
        if (J->arena_k) {
            int blk = J->block_tables[(size_t)s * J->max_blocks + j / J->bs];
            size_t slot = (((size_t)blk * Hkv + g) * J->bs + (size_t)(j % J->bs)) * d;
            kr = J->arena_k + slot;
            vr = J->arena_v + slot;
        } else {
            size_t src = ((size_t)(J->kv_start[s] + j) * Hkv + g) * d;
            kr = J->k_all + src;
            vr = J->v_all + src;
        }
        for (int i = 0; i < d; ++i) x[i] = to_f64(kr[i], J->dtype);
        for (int i = 0; i < d; ++i) V[(size_t)j * d + i] = to_f64(vr[i], J->dtype);
        for (int i = 0; i < d; ++i)
            if (isnan(x[i]) || isnan(V[(size_t)j * d + i])) J->status = 6; /* a NaN was gathered */
        rope_row(x, K + (size_t)j * d, j, d, J->theta);
    }
    for (int r = 0; r < J->n_out; ++r) {
        int t = J->out_tokens[r];
        if (seq_of_token(J->qsl, J->S, t) != s) continue;
        long pos = J->positions[t];
        if (pos < 0 || pos >= ctx) { J->status = 4; continue; }
        /* explicit causal mask: key j is visible to this query iff j <= pos */
        for (long j = 0; j < ctx; ++j) visible[j] = (char)(j <= pos);
        for (int hh = g * G; hh < (g + 1) * G; ++hh) {
            size_t qo = ((size_t)t * Hq + hh) * d;
            for (int i = 0; i < d; ++i) x[i] = to_f64(J->q[qo + i], J->dtype);
            rope_row(x, qr, pos, d, J->theta);
            double mx = -INFINITY;
            for (long j = 0; j < ctx; ++j) {
                if (!visible[j]) { w[j] = -INFINITY; continue; }
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += qr[i] * K[(size_t)j * d + i];
                w[j] = J->scale * acc;
                if (w[j] > mx) mx = w[j];
            }
            double sum = 0.0;
            for (long j = 0; j < ctx; ++j) {
                w[j] = visible[j] ? exp(w[j] - mx) : 0.0;
                sum += w[j];
            }
            double* o = J->out + ((size_t)r * Hq + hh) * d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            for (long j = 0; j < ctx; ++j) {
                if (!visible[j]) continue;
                double pj = w[j] / sum;
                for (int i = 0; i < d; ++i) o[i] += pj * V[(size_t)j * d + i];
            }
        }
    }
    free(K); free(V); free(w); free(visible);
}

static void* attention_worker(void* arg) {
    attn_job* J = (attn_job*)arg;
    for (;;) {
        int k = __atomic_fetch_add(&J->next_task, 1, __ATOMIC_RELAXED);
        if (k >= J->n_tasks) break;
        attention_task(J, J->task_seq[k], J->task_head[k]);
    }
    return NULL;
}

/* The arena every slot of which starts as the NaN pattern ARENA_EMPTY
 * (a NaN in binary16 and in bfloat16); the raw K/V rows of each listed
 * sequence are written to slot j % bs of block block_tables[s][j / bs]
 * (section 1).  Returns 0; 2 a block id outside [0, num_blocks) or a
 * logical block past the table; 5 a slot written twice with different bits
 * (rows of different positions or sequences aliased); 3 out of memory. */
#define ARENA_EMPTY 0x7FC1u

static int arena_fill(uint16_t** ak, uint16_t** av, const char* want, const uint16_t* k_all, const uint16_t* v_all,
                      const int64_t* kv_start, const int32_t* context_lens, const int32_t* block_tables,
                      int max_blocks, int num_seqs, int num_blocks, int Hkv, int bs, int d) {
    size_t n = (size_t)num_blocks * Hkv * bs * d;
    uint16_t* K = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
    uint16_t* V = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
    if (!K || !V) { free(K); free(V); return 3; }
    for (size_t i = 0; i < n; ++i) K[i] = V[i] = (uint16_t)ARENA_EMPTY;
    *ak = K;
    *av = V;
    for (int s = 0; s < num_seqs; ++s) {
        if (!want[s]) continue;
        for (long j = 0; j < context_lens[s]; ++j) {
            if (j / bs >= max_blocks) return 2;
            int blk = block_tables[(size_t)s * max_blocks + j / bs];
            if (blk < 0 || blk >= num_blocks) return 2;
            for (int h = 0; h < Hkv; ++h) {
                size_t src = ((size_t)(kv_start[s] + j) * Hkv + h) * d;
                size_t dst = (((size_t)blk * Hkv + h) * bs + (size_t)(j % bs)) * d;
                size_t row = (size_t)d * sizeof(uint16_t);
                if (K[dst] != (uint16_t)ARENA_EMPTY) { /* written before: must hold the same row */
                    if (memcmp(K + dst, k_all + src, row) || memcmp(V + dst, v_all + src, row)) return 5;
                    continue;
                }
                memcpy(K + dst, k_all + src, row);
                memcpy(V + dst, v_all + src, row);
            }
        }
    }
    return 0;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* out[r][h][:] = softmax-weighted sum of V for query token out_tokens[r]
 * (all T tokens when out_tokens is NULL, then n_out = T), every q head.
 * With block_tables given, keys and values go through the oracle's own
 * arena of num_blocks blocks of bs slots (written, then gathered, through
 * the tables); with block_tables NULL they are read in logical order.
 * Returns 0; 1 bad shape; 2 a block id outside the arena; 3 out of memory;
 * 4 a position outside [0, ctx); 5 aliased arena slots; 6 a NaN gathered. */
int oracle_attention(double* out, const int32_t* out_tokens, int n_out, const uint16_t* q,
                     const uint16_t* k_all, const uint16_t* v_all, const int64_t* kv_start,
                     const int32_t* query_start_loc, const int32_t* positions, const int32_t* context_lens,
                     const int32_t* block_tables, int max_blocks, int block_size, int num_blocks,
                     int num_seqs, int num_tokens, int Hq, int Hkv, int d, double theta, double scale,
                     int dtype, int nthreads) {
    if (Hkv <= 0 || Hq % Hkv || d <= 0 || (d & 1) || d > 1024 || num_seqs < 0) return 1;
    if (block_tables && (max_blocks <= 0 || block_size <= 0 || num_blocks <= 0)) return 1;
    int32_t* all = NULL;
    if (!out_tokens) {
        all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_tokens > 0 ? num_tokens : 1));
        if (!all) return 3;
        for (int t = 0; t < num_tokens; ++t) all[t] = t;
        out_tokens = all;
        n_out = num_tokens;
    }
    attn_job J;
    memset(&J, 0, sizeof J);
    J.out = out; J.out_tokens = out_tokens; J.n_out = n_out; J.q = q; J.k_all = k_all; J.v_all = v_all;
    J.kv_start = kv_start; J.qsl = query_start_loc; J.positions = positions; J.context_lens = context_lens;
    J.S = num_seqs; J.Hq = Hq; J.Hkv = Hkv; J.d = d; J.dtype = dtype; J.theta = theta; J.scale = scale;
    /* one task per (sequence, kv head) that owns at least one requested token */
    char* want = (char*)calloc((size_t)(num_seqs > 0 ? num_seqs : 1), 1);
    J.task_seq = (int*)malloc(sizeof(int) * (size_t)(num_seqs > 0 ? num_seqs : 1) * Hkv);
    J.task_head = (int*)malloc(sizeof(int) * (size_t)(num_seqs > 0 ? num_seqs : 1) * Hkv);
    if (!want || !J.task_seq || !J.task_head) {
        free(want); free(J.task_seq); free(J.task_head); free(all);
        return 3;
    }
    for (int r = 0; r < n_out; ++r) {
        int s = seq_of_token(query_start_loc, num_seqs, out_tokens[r]);
        if (s >= 0) want[s] = 1;
    }
    for (int s = 0; s < num_seqs; ++s)
        if (want[s])
            for (int g = 0; g < Hkv; ++g) {
                J.task_seq[J.n_tasks] = s;
                J.task_head[J.n_tasks] = g;
                J.n_tasks++;
            }
    uint16_t *ak = NULL, *av = NULL;
    if (block_tables) {
        int rc = arena_fill(&ak, &av, want, k_all, v_all, kv_start, context_lens, block_tables, max_blocks,
                            num_seqs, num_blocks, Hkv, block_size, d);
        if (rc) {
            free(ak); free(av); free(want); free(J.task_seq); free(J.task_head); free(all);
            return rc;
        }
        J.arena_k = ak; J.arena_v = av; J.block_tables = block_tables;
        J.max_blocks = max_blocks; J.bs = block_size; J.num_blocks = num_blocks;
    }
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > J.n_tasks) nthreads = J.n_tasks > 0 ? J.n_tasks : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 1; th && i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, attention_worker, &J) == 0) started = i;
        else break;
    attention_worker(&J);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th); free(want); free(J.task_seq); free(J.task_head); free(all); free(ak); free(av);
    return J.status;
}
