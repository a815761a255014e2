/*
 * FP64 CPU oracle for single-token paged-KV GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header or constant with the CUDA path.
 *
 * What it computes (the definition, written out; not an algorithm):
 *
 *   "Paged Attention Kernel Architecture for BI-V100", section 1 (Problem
 *   Definition): for one decode query, output[h, d] = softmax(Q[h] . K[t]^T
 *   scaled) . V[t], with K and V stored in pages reached through a block table.
 *
 *   The paging layout, the per-sequence length and the GQA head map are the
 *   ones of the "Add Cuda Kernel" tutorial (RL.cu), include/kernels/
 *   attention.cuh, "Paged Attention - Decode" and the kernel body that walks
 *   the block table in src/kernels/attention.cu:
 *     q            [num_seqs, H_q, D]
 *     k/v cache    [num_blocks, H_kv, block_size, D]
 *     block_tables [num_seqs, max_blocks_per_seq]   logical page -> physical block
 *     seq_lens     [num_seqs]                      tokens t < seq_lens[s] are attended
 *     kv head      g = h * H_kv / H_q              (integer division)
 *   and the caller supplies the softmax scale.
 *
 *   For each (s, h):
 *     K_t = k_cache[bt[s, t / BS], g, t % BS, :]      t in [0, L)
 *     z_t = scale * sum_d q[s,h,d] * K_t[d]
 *     M   = max_t z_t
 *     w_t = exp(z_t - M)
 *     out[s,h,:] = (sum_t w_t V_t) / (sum_t w_t)
 *
 *   Every bf16 input is widened exactly to double; all arithmetic is double;
 *   scale is the float the caller passes, widened to double.  L = 0 gives a
 *   zero row (the pages never define an empty softmax; this is the reading
 *   the library documents), and so does a multi-token query that sees no
 *   token: parity unpinned for both (no page fixes the value).
 *
 *   FP8 caches (the nvfp4-megamoe README, "Stage D: FP8 Paged KV Gather" and
 *   "FP8 KV Quantize/Dequant": e4m3 values with a dequant scale per position)
 *   hold e4m3 bytes in the same layout plus one float per (block, KV head,
 *   slot) for K and for V; an element is its e4m3 value times that float:
 *     K_t[d] = e4m3(k8[bt[s, t / BS], g, t % BS, d]) * k_scale[bt[s, t / BS], g, t % BS]
 *   and everything else is the definition above.  e4m3 is the OCP 8-bit
 *   format with 1 sign bit, 4 exponent bits (bias 7) and 3 mantissa bits,
 *   subnormals at exponent 0, no infinities, S.1111.111 = NaN (max 448).
 *
 *   The x-packed caches ("Paged Attention Kernel Architecture for BI-V100",
 *   section 3, Paged K/V Gather) hold the same bf16 values in another order:
 *     key cache    [num_blocks, H_kv, D / x, block_size, x],  x = 16 / 2 = 8
 *     value cache  [num_blocks, H_kv, D, block_size]
 *   so K_t[d] = kx[bt[s, t / BS], g, d / 8, t % BS, d % 8] and
 *      V_t[d] = vt[bt[s, t / BS], g, d, t % BS];
 *   everything else is the definition above.
 *
 *   Multi-token decode (AstrAI's CUDA Kernels page: the prefill path over a
 *   ragged batch, "Q Scheduling and KV Addressing", with qo_indptr, and the
 *   wrappers' is_causal; "Python Wrappers"): sequence s owns the query rows
 *   qo_indptr[s] .. qo_indptr[s+1] - 1 of q ([total_q, H_q, D]), its last
 *   q_len = qo_indptr[s+1] - qo_indptr[s] tokens, all of them already in the
 *   cache (L = seq_lens[s] counts them).  With the causal mask, query i sees the
 *   tokens t <= L - q_len + i (its own position and everything before); without
 *   it, all L tokens.  Each query row is the definition above over the tokens
 *   it sees; a row that sees none is zero.
 *
 *   FP8 cache write (nvfp4-megamoe README, "FP8 KV Quantize/Dequant" and "Paged
 *   KV cache read/write"; the pages fix neither the row float nor the
 *   rounding, so this is a reading): a bf16 row x of D values is stored as the
 *   e4m3 codes of x[d] / f, with f = max_d |x[d]| / 448 computed in float32
 *   (f = 1 for an all-zero row) and each quotient a float32 division; the code
 *   is the e4m3 value nearest the quotient, a tie going to the code whose
 *   mantissa is even, and a magnitude beyond 448 takes 448's code.  The
 *   decision is taken in float32, the precision the library's kernel uses.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARGS -1
#define ORACLE_ERR_HEADS -2
#define ORACLE_ERR_LEN -3
#define ORACLE_ERR_BLOCK -4
#define ORACLE_ERR_NOMEM -5

static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The e4m3 value of one byte, decoded from its bit fields. */
static double e4m3_value(uint8_t b) {
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* A paged K/V cache pair: bf16 elements, or e4m3 bytes with a float per row. */
typedef struct {
    const uint16_t* k16;
    const uint16_t* v16;
    const uint8_t* k8;
    const uint8_t* v8;
    const float* k_scale; /* [num_blocks * H_kv * BS] */
    const float* v_scale;
    const uint16_t* kx;   /* x-packed bf16 K [num_blocks, H_kv, D / 8, BS, 8] */
    const uint16_t* vt;   /* D-major bf16 V [num_blocks, H_kv, D, BS] */
    int BS;               /* block size (x-packed layout only) */
} Cache;

/* Element d of cache row `row` = (block * H_kv + g) * BS + slot. */
static double cache_k(const Cache* c, size_t row, int d, int D) {
    if (c->k16) return widen_bf16(c->k16[row * D + d]);
    if (c->kx) {
        const size_t head = row / (size_t)c->BS, slot = row % (size_t)c->BS;
        return widen_bf16(c->kx[((head * (size_t)(D / 8) + (size_t)(d / 8)) * c->BS + slot) * 8 +
                                (size_t)(d % 8)]);
    }
    return e4m3_value(c->k8[row * D + d]) * (double)c->k_scale[row];
}
static double cache_v(const Cache* c, size_t row, int d, int D) {
    if (c->v16) return widen_bf16(c->v16[row * D + d]);
    if (c->vt) {
        const size_t head = row / (size_t)c->BS, slot = row % (size_t)c->BS;
        return widen_bf16(c->vt[(head * (size_t)D + (size_t)d) * c->BS + slot]);
    }
    return e4m3_value(c->v8[row * D + d]) * (double)c->v_scale[row];
}

/* Validate the sequence lengths and every block-table entry a sequence uses. */
static int check_inputs(const int32_t* bt, const int32_t* seq_lens, int num_seqs, int H_q,
                        int H_kv, int D, int max_blocks, int BS, long long num_blocks) {
    if (num_seqs < 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || max_blocks <= 0 || BS <= 0)
        return ORACLE_ERR_ARGS;
    if (H_q % H_kv != 0) return ORACLE_ERR_HEADS;
    for (int s = 0; s < num_seqs; ++s) {
        const long long L = seq_lens[s];
        if (L < 0 || L > (long long)max_blocks * BS) return ORACLE_ERR_LEN;
        const long long pages = (L + BS - 1) / BS;
        for (long long p = 0; p < pages; ++p) {
            const long long b = bt[(size_t)s * max_blocks + p];
            if (b < 0 || b >= num_blocks) return ORACLE_ERR_BLOCK;
        }
    }
    return ORACLE_OK;
}

/*
 * Softmax pieces of one (s, h) row over the token range [t0, t1):
 *   M = max_t z_t,  l = sum_t exp(z_t - M),  o[d] = sum_t exp(z_t - M) V_t[d].
 * An empty range gives M = -inf, l = 0, o = 0.  z is scratch of >= t1 - t0 doubles.
 */
static int kv_head(int h, int H_q, int H_kv) { return (int)(((long long)h * H_kv) / H_q); }

static void row_pieces(const uint16_t* qrow, const Cache* c, const int32_t* bt, int s, int g,
                       int H_kv, int D, int max_blocks, int BS, double scale, int t0, int t1,
                       double* z, double* M_out, double* l_out, double* o) {

    for (int d = 0; d < D; ++d) o[d] = 0.0;
    *l_out = 0.0;
    *M_out = -INFINITY;
    if (t1 <= t0) return;

    /* z_t = scale * q . K_t, K_t reached through the block table */
    for (int t = t0; t < t1; ++t) {
        const size_t pb = (size_t)bt[(size_t)s * max_blocks + t / BS];
        const size_t krow = (pb * H_kv + g) * BS + (size_t)(t % BS);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen_bf16(qrow[d]) * cache_k(c, krow, d, D);
        z[t - t0] = scale * dot;
    }

    double M = z[0];
    for (int t = t0 + 1; t < t1; ++t)
        if (z[t - t0] > M) M = z[t - t0];
    double l = 0.0;
    for (int t = t0; t < t1; ++t) {
        const double w = exp(z[t - t0] - M);
        l += w;
        const size_t pb = (size_t)bt[(size_t)s * max_blocks + t / BS];
        const size_t vrow = (pb * H_kv + g) * BS + (size_t)(t % BS);
        for (int d = 0; d < D; ++d) o[d] += w * cache_v(c, vrow, d, D);
    }
    *M_out = M;
    *l_out = l;
}

/* One (s, h) row of the definition: out = o / l over the whole sequence. */
static void attend_row(const uint16_t* q, const Cache* c, const int32_t* bt,
                       const int32_t* seq_lens, int s, int h, int H_q, int H_kv, int D,
                       int max_blocks, int BS, double scale, double* z, double* out_row) {
    double M, l;
    const int g = kv_head(h, H_q, H_kv);
    const uint16_t* qrow = q + ((size_t)s * H_q + h) * D;
    row_pieces(qrow, c, bt, s, g, H_kv, D, max_blocks, BS, scale, 0, seq_lens[s], z, &M, &l,
               out_row);
    if (l > 0.0)
        for (int d = 0; d < D; ++d) out_row[d] /= l;
}

/*
 * Rows listed in `pairs` ([num_pairs][2] = (s, h)); out is [num_pairs, D].
 * num_threads <= 0 uses the OpenMP default.  Returns 0 or a negative code.
 */
static int decode_pairs(const uint16_t* q, const Cache* c, const int32_t* block_tables,
                        const int32_t* seq_lens, int num_seqs, int H_q, int H_kv, int D,
                        int max_blocks_per_seq, int block_size, long long num_blocks,
                        float scale, const int32_t* pairs, int num_pairs, double* out,
                        int num_threads) {
    int rc = check_inputs(block_tables, seq_lens, num_seqs, H_q, H_kv, D, max_blocks_per_seq,
                          block_size, num_blocks);
    if (rc != ORACLE_OK) return rc;
    for (int i = 0; i < num_pairs; ++i) {
        if (pairs[2 * i] < 0 || pairs[2 * i] >= num_seqs || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= H_q)
            return ORACLE_ERR_ARGS;
    }
    int Lmax = 1;
    for (int s = 0; s < num_seqs; ++s)
        if (seq_lens[s] > Lmax) Lmax = seq_lens[s];
    const double sc = (double)scale;
    int failed = 0;

#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)Lmax);
        /* every thread reaches the work-sharing loop; one without scratch skips its rows */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int i = 0; i < num_pairs; ++i) {
            if (!z) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                failed = 1;
                continue;
            }
            attend_row(q, c, block_tables, seq_lens, pairs[2 * i], pairs[2 * i + 1], H_q, H_kv,
                       D, max_blocks_per_seq, block_size, sc, z, out + (size_t)i * D);
        }
        free(z);
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

int oracle_decode_pairs(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                        int H_q, int H_kv, int D, int max_blocks_per_seq, int block_size,
                        long long num_blocks, float scale, const int32_t* pairs, int num_pairs,
                        double* out, int num_threads) {
    const Cache c = {k_cache, v_cache, NULL, NULL, NULL, NULL, NULL, NULL, 0};
    return decode_pairs(q, &c, block_tables, seq_lens, num_seqs, H_q, H_kv, D,
                        max_blocks_per_seq, block_size, num_blocks, scale, pairs, num_pairs, out,
                        num_threads);
}

/* The same rows over FP8 caches (e4m3 bytes and per-row dequant floats). */
int oracle_decode_fp8_pairs(const uint16_t* q, const uint8_t* k8, const uint8_t* v8,
                            const float* k_scale, const float* v_scale,
                            const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                            int H_q, int H_kv, int D, int max_blocks_per_seq, int block_size,
                            long long num_blocks, float scale, const int32_t* pairs,
                            int num_pairs, double* out, int num_threads) {
    if (!k8 || !v8 || !k_scale || !v_scale) return ORACLE_ERR_ARGS;
    const Cache c = {NULL, NULL, k8, v8, k_scale, v_scale, NULL, NULL, 0};
    return decode_pairs(q, &c, block_tables, seq_lens, num_seqs, H_q, H_kv, D,
                        max_blocks_per_seq, block_size, num_blocks, scale, pairs, num_pairs, out,
                        num_threads);
}

/* The same rows over x-packed K and D-major V (bf16; head_dim a multiple of 8). */
int oracle_decode_xpacked_pairs(const uint16_t* q, const uint16_t* kx, const uint16_t* vt,
                                const int32_t* block_tables, const int32_t* seq_lens,
                                int num_seqs, int H_q, int H_kv, int D, int max_blocks_per_seq,
                                int block_size, long long num_blocks, float scale,
                                const int32_t* pairs, int num_pairs, double* out,
                                int num_threads) {
    if (!kx || !vt || D % 8 != 0) return ORACLE_ERR_ARGS;
    const Cache c = {NULL, NULL, NULL, NULL, NULL, NULL, kx, vt, block_size};
    return decode_pairs(q, &c, block_tables, seq_lens, num_seqs, H_q, H_kv, D,
                        max_blocks_per_seq, block_size, num_blocks, scale, pairs, num_pairs, out,
                        num_threads);
}

/* e4m3 values of the 256 byte codes (for checking the decoder). */
void oracle_e4m3_table(double* out) {
    for (int b = 0; b < 256; ++b) out[b] = e4m3_value((uint8_t)b);
}

/* Every row: out is [num_seqs, H_q, D]. */
int oracle_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                  const int32_t* block_tables, const int32_t* seq_lens, int num_seqs, int H_q,
                  int H_kv, int D, int max_blocks_per_seq, int block_size, long long num_blocks,
                  float scale, double* out, int num_threads) {
    if (num_seqs < 0 || H_q <= 0) return ORACLE_ERR_ARGS;
    const size_t n = (size_t)num_seqs * H_q;
    int32_t* pairs = (int32_t*)malloc(sizeof(int32_t) * 2 * (n ? n : 1));
    if (!pairs) return ORACLE_ERR_NOMEM;
    for (size_t i = 0; i < n; ++i) {
        pairs[2 * i] = (int32_t)(i / H_q);
        pairs[2 * i + 1] = (int32_t)(i % H_q);
    }
    int rc = oracle_decode_pairs(q, k_cache, v_cache, block_tables, seq_lens, num_seqs, H_q, H_kv,
                                 D, max_blocks_per_seq, block_size, num_blocks, scale, pairs,
                                 (int)n, out, num_threads);
    free(pairs);
    return rc;
}

/* Threads the OpenMP runtime would use by default (0 when built without it). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 0;
#endif
}

/*
 * Softmax pieces (M, l, o) of rows (s, h) over token ranges: ranges is
 * [num_pairs][2] = (t0, t1) with 0 <= t0 <= t1 <= seq_lens[s].  These are the
 * per-partition states that the split-KV design of "Paged Attention Kernel
 * Architecture for BI-V100" (section 2, Level 1 and Level 3) merges.
 */
int oracle_partial_pairs(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                         int H_q, int H_kv, int D, int max_blocks_per_seq, int block_size,
                         long long num_blocks, float scale, const int32_t* pairs,
                         const int32_t* ranges, int num_pairs, double* M, double* l, double* o) {
    int rc = check_inputs(block_tables, seq_lens, num_seqs, H_q, H_kv, D, max_blocks_per_seq,
                          block_size, num_blocks);
    if (rc != ORACLE_OK) return rc;
    int Lmax = 1;
    for (int i = 0; i < num_pairs; ++i) {
        const int s = pairs[2 * i], h = pairs[2 * i + 1];
        const int t0 = ranges[2 * i], t1 = ranges[2 * i + 1];
        if (s < 0 || s >= num_seqs || h < 0 || h >= H_q) return ORACLE_ERR_ARGS;
        if (t0 < 0 || t1 < t0 || t1 > seq_lens[s]) return ORACLE_ERR_ARGS;
        if (t1 - t0 > Lmax) Lmax = t1 - t0;
    }
    double* z = (double*)malloc(sizeof(double) * (size_t)Lmax);
    if (!z) return ORACLE_ERR_NOMEM;
    const Cache c = {k_cache, v_cache, NULL, NULL, NULL, NULL, NULL, NULL, 0};
    for (int i = 0; i < num_pairs; ++i) {
        const int s = pairs[2 * i], h = pairs[2 * i + 1];
        row_pieces(q + ((size_t)s * H_q + h) * D, &c, block_tables, s, kv_head(h, H_q, H_kv), H_kv,
                   D, max_blocks_per_seq, block_size, (double)scale, ranges[2 * i],
                   ranges[2 * i + 1], z, M + i, l + i, o + (size_t)i * D);
    }
    free(z);
    return ORACLE_OK;
}

/*
 * Multi-token decode: q and out are [total_q, H_q, D] with total_q =
 * qo_indptr[num_seqs]; qo_indptr [num_seqs + 1] is non-decreasing from 0 and
 * q_len <= L for every sequence.  causal != 0 applies the causal mask.
 */
int oracle_decode_multi(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* qo_indptr, const int32_t* block_tables,
                        const int32_t* seq_lens, int num_seqs, int H_q, int H_kv, int D,
                        int max_blocks_per_seq, int block_size, long long num_blocks,
                        float scale, int causal, double* out, int num_threads) {
    int rc = check_inputs(block_tables, seq_lens, num_seqs, H_q, H_kv, D, max_blocks_per_seq,
                          block_size, num_blocks);
    if (rc != ORACLE_OK) return rc;
    if (!qo_indptr || qo_indptr[0] != 0) return ORACLE_ERR_ARGS;
    int Lmax = 1;
    for (int s = 0; s < num_seqs; ++s) {
        const int ql = qo_indptr[s + 1] - qo_indptr[s];
        if (ql < 0 || ql > seq_lens[s]) return ORACLE_ERR_ARGS;
        if (seq_lens[s] > Lmax) Lmax = seq_lens[s];
    }
    const Cache c = {k_cache, v_cache, NULL, NULL, NULL, NULL, NULL, NULL, 0};
    const double sc = (double)scale;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)Lmax);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int s = 0; s < num_seqs; ++s) {
            if (!z) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                failed = 1;
                continue;
            }
            const int L = seq_lens[s];
            const int ql = qo_indptr[s + 1] - qo_indptr[s];
            for (int i = 0; i < ql; ++i) {
                const int seen = causal ? L - ql + i + 1 : L;  /* tokens t < seen */
                const size_t r = (size_t)qo_indptr[s] + (size_t)i;
                for (int h = 0; h < H_q; ++h) {
                    double M, l;
                    double* orow = out + (r * H_q + h) * D;
                    row_pieces(q + (r * H_q + h) * D, &c, block_tables, s, kv_head(h, H_q, H_kv),
                               H_kv, D, max_blocks_per_seq, block_size, sc, 0, seen, z, &M, &l,
                               orow);
                    if (l > 0.0)
                        for (int d = 0; d < D; ++d) orow[d] /= l;
                }
            }
        }
        free(z);
    }
    return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * e4m3 code of a float32 value (the FP8 cache write above): the finite code
 * whose value is nearest |v|, searched over all of them, ties to the even code,
 * the sign carried over; NaN gives 0x7F.
 */
static uint8_t e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

void oracle_e4m3_encode(const float* x, int n, uint8_t* out) {
    for (int i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

/* Quantize n_rows bf16 rows of D values: codes [n_rows, D], one float per row. */
void oracle_quantize_rows_e4m3(const uint16_t* rows, int n_rows, int D, uint8_t* codes,
                               float* f_out) {
    for (int r = 0; r < n_rows; ++r) {
        const uint16_t* x = rows + (size_t)r * D;
        float amax = 0.0f;
        for (int d = 0; d < D; ++d) {
            const float a = fabsf((float)widen_bf16(x[d]));
            if (a > amax) amax = a;
        }
        const float f = amax > 0.0f ? amax / 448.0f : 1.0f;
        for (int d = 0; d < D; ++d)
            codes[(size_t)r * D + d] = e4m3_encode((float)widen_bf16(x[d]) / f);
        f_out[r] = f;
    }
}
