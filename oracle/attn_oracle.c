/*
 * fp64 CPU oracle for single-query (n_q = 1) decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, calls or includes this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes is the plain definition that split-KV flash-decoding reaches
 * (up to floating-point reduction order).  The pages name the pieces without writing
 * the formula out: the decode op emits a log-sum-exp "LSE channel" next to its output
 * ("Rolling-KV -- overflow throughput evaluations", section 3), partial windows keep
 * "the online-softmax maximum, numerator, and denominator and are merged afterward"
 * ("KVARN KV Performance optimizations", item 9), and the window is attended on the
 * device while the host tail is streamed once (rolling_kv, section 5c).  For sequence
 * s and query head h, with G = n_head / n_head_kv and KV head g = floor(h / G):
 *
 *     valid(s) = { plan[s][i] : 0 <= i < seq_len[s], plan[s][i] != -1 }
 *                (or { 0 .. seq_len[s]-1 } of sequence s's own cache when no plan)
 *     x_c      = scale * sum_d q[s][h][d] * K[c][g][d]
 *     m        = max_c x_c
 *     l        = sum_c exp(x_c - m)
 *     O[s][h]  = sum_c exp(x_c - m) * V[c][g][:] / l
 *     LSE[s][h]= m + ln(l)                      (natural logarithm)
 *
 * An empty valid set gives O = 0 and LSE = -inf.  Every stored element is turned into
 * its exact fp64 value first: f16 by the IEEE 754 binary16 definition, Q8_0 as
 * d * qs with d an f16 scale shared by 32 consecutive head_dim elements, Q4_0 as
 * d * (n - 8) with n an unsigned 4-bit value and d an f16 scale per 32 elements.  The
 * pages name the q4_0 type (the mixed "q8_0K/q4_0V" cache of the Rolling-KV evaluation's
 * resident-compression anchors, and a q4_0 cache in its section 5a) without its bytes;
 * the reading taken is the llama.cpp q4_0 block -- 32 elements share one f16 scale and
 * 16 bytes, byte j of a block holding element j in its low nibble and element j + 16 in
 * its high nibble -- with the values and the scales kept in two planes:
 *     values uint8 [cells][Hk][D/2] (block b of a row = bytes 16b .. 16b+15),
 *     scales f16   [cells][Hk][D/32].
 *
 * The merge follows the same definition over partial results:
 *     M = max_p LSE_p;  w_p = exp(LSE_p - M);
 *     O = sum_p w_p O_p / sum_p w_p;  LSE = M + ln(sum_p w_p);
 * parts whose LSE is -inf carry no cells and are ignored (their O is not read).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_KV_F16 0
#define ORACLE_KV_Q8_0 1
#define ORACLE_KV_F64 2
#define ORACLE_KV_Q4_0 3

/* IEEE 754 binary16 -> binary64, from the format's definition (exact). */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);               /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)frac / 1024.0, expo - 15);
    }
    return sign ? -v : v;
}

/* All 65536 binary16 values, filled once from oracle_f16_to_f64 before any parallel work
 * (a cache of the definition above, so that large cases run in seconds). */
static double f16_table[65536];
static int f16_table_ready = 0;

static void f16_table_init(void) {
    if (f16_table_ready) return;
    for (int i = 0; i < 65536; ++i) f16_table[i] = oracle_f16_to_f64((uint16_t)i);
    f16_table_ready = 1;
}

/* One K or V source: element (cell, kv_head, dim) -> exact fp64 value. */
typedef struct {
    int kind;
    const void* data;        /* f16 bits / int8 / double [cells][Hk][D]; Q4_0: uint8 [cells][Hk][D/2] */
    const uint16_t* scale;   /* Q8_0 and Q4_0: f16 bits [cells][Hk][D/32] */
} kv_source;

static double kv_value(const kv_source* src, int64_t cell, int g, int d, int Hk, int D) {
    int64_t idx = (cell * Hk + g) * (int64_t)D + d;
    switch (src->kind) {
    case ORACLE_KV_F16:
        return f16_table[((const uint16_t*)src->data)[idx]];
    case ORACLE_KV_Q8_0: {
        double qs = (double)((const int8_t*)src->data)[idx];
        int64_t sidx = (cell * Hk + g) * (int64_t)(D / 32) + d / 32;
        return f16_table[src->scale[sidx]] * qs;
    }
    case ORACLE_KV_Q4_0: {
        int j = d % 32;                             /* position inside the 32-element block */
        int64_t byte_idx = (cell * Hk + g) * (int64_t)(D / 2) + 16 * (d / 32) + j % 16;
        unsigned byte = ((const uint8_t*)src->data)[byte_idx];
        unsigned n = (j < 16) ? (byte & 15u) : (byte >> 4);
        int64_t sidx = (cell * Hk + g) * (int64_t)(D / 32) + d / 32;
        return f16_table[src->scale[sidx]] * ((double)n - 8.0);
    }
    default:
        return ((const double*)src->data)[idx];
    }
}

/*
 * q: f16 bits [S][H][D] (q_is_f64 = 0) or double [S][H][D] (q_is_f64 = 1).
 * K/V: one cache of per_seq_cells rows per sequence when plan == NULL (sequence s
 *      starts at row s * per_seq_cells), or one unified cache of n_cells_phys rows
 *      addressed through plan[s][0 .. seq_len[s]) when plan != NULL.
 * out: double [S][H][D]; lse: double [S][H].
 * Returns 0, or -1 for an argument the definition does not cover (a plan entry
 * outside [-1, n_cells_phys), a length beyond the cache or the plan row).
 */
static int oracle_decode(const void* q, int q_is_f64, const kv_source* K, const kv_source* V,
                         int64_t n_cells_phys, int64_t per_seq_cells,
                         const int32_t* plan, int64_t plan_stride, const int64_t* seq_lens,
                         int S, int H, int Hk, int D, double scale,
                         double* out, double* lse, int n_threads) {
    if (S < 0 || H <= 0 || Hk <= 0 || D <= 0 || H % Hk != 0) return -1;
    int G = H / Hk;
    f16_table_init();
    for (int s = 0; s < S; ++s) {
        if (seq_lens[s] < 0) return -1;
        if (plan) {
            if (seq_lens[s] > plan_stride) return -1;
            for (int64_t i = 0; i < seq_lens[s]; ++i) {
                int32_t c = plan[s * plan_stride + i];
                if (c != -1 && (c < 0 || c >= n_cells_phys)) return -1;
            }
        } else if (seq_lens[s] > per_seq_cells) {
            return -1;
        }
    }
    int failed = 0;
    int64_t rows = (int64_t)S * H;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1)
    for (int64_t row = 0; row < rows; ++row) {
        int s = (int)(row / H), h = (int)(row % H), g = h / G;
        int64_t L = seq_lens[s];
        int64_t* cells = (int64_t*)malloc(sizeof(int64_t) * (L > 0 ? L : 1));
        double* x = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
        double* qd = (double*)malloc(sizeof(double) * D);
        if (!cells || !x || !qd) {
#pragma omp atomic write
            failed = 1;
            free(cells); free(x); free(qd);
            continue;
        }
        /* the valid set */
        int64_t n = 0;
        for (int64_t i = 0; i < L; ++i) {
            if (plan) {
                int32_t c = plan[s * plan_stride + i];
                if (c != -1) cells[n++] = c;
            } else {
                cells[n++] = (int64_t)s * per_seq_cells + i;
            }
        }
        for (int d = 0; d < D; ++d) {
            int64_t qi = (row) * D + d;
            qd[d] = q_is_f64 ? ((const double*)q)[qi] : oracle_f16_to_f64(((const uint16_t*)q)[qi]);
        }
        double* o = out + row * D;
        if (n == 0) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            lse[row] = -INFINITY;
        } else {
            /* scores */
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qd[d] * kv_value(K, cells[j], g, d, Hk, D);
                x[j] = scale * acc;
                if (x[j] > m) m = x[j];
            }
            /* softmax-weighted sum of V rows */
            double l = 0.0;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double p = exp(x[j] - m);
                l += p;
                for (int d = 0; d < D; ++d) o[d] += p * kv_value(V, cells[j], g, d, Hk, D);
            }
            for (int d = 0; d < D; ++d) o[d] /= l;
            lse[row] = m + log(l);
        }
        free(cells); free(x); free(qd);
    }
    return failed ? -1 : 0;
}

int oracle_decode_f16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      int64_t n_cells_phys, int64_t per_seq_cells,
                      const int32_t* plan, int64_t plan_stride, const int64_t* seq_lens,
                      int S, int H, int Hk, int D, double scale,
                      double* out, double* lse, int n_threads) {
    kv_source K = {ORACLE_KV_F16, k, NULL}, V = {ORACLE_KV_F16, v, NULL};
    return oracle_decode(q, 0, &K, &V, n_cells_phys, per_seq_cells, plan, plan_stride, seq_lens,
                         S, H, Hk, D, scale, out, lse, n_threads);
}

int oracle_decode_q8_0(const uint16_t* q, const int8_t* k_qs, const uint16_t* k_d,
                       const int8_t* v_qs, const uint16_t* v_d,
                       int64_t n_cells_phys, int64_t per_seq_cells,
                       const int32_t* plan, int64_t plan_stride, const int64_t* seq_lens,
                       int S, int H, int Hk, int D, double scale,
                       double* out, double* lse, int n_threads) {
    if (D % 32 != 0) return -1;
    kv_source K = {ORACLE_KV_Q8_0, k_qs, k_d}, V = {ORACLE_KV_Q8_0, v_qs, v_d};
    return oracle_decode(q, 0, &K, &V, n_cells_phys, per_seq_cells, plan, plan_stride, seq_lens,
                         S, H, Hk, D, scale, out, lse, n_threads);
}

/* Q8_0 keys and Q4_0 values (the mixed cache); values uint8 [cells][Hk][D/2]. */
int oracle_decode_q8_0_q4_0(const uint16_t* q, const int8_t* k_qs, const uint16_t* k_d,
                            const uint8_t* v_q4, const uint16_t* v_d,
                            int64_t n_cells_phys, int64_t per_seq_cells,
                            const int32_t* plan, int64_t plan_stride, const int64_t* seq_lens,
                            int S, int H, int Hk, int D, double scale,
                            double* out, double* lse, int n_threads) {
    if (D % 32 != 0) return -1;
    kv_source K = {ORACLE_KV_Q8_0, k_qs, k_d}, V = {ORACLE_KV_Q4_0, v_q4, v_d};
    return oracle_decode(q, 0, &K, &V, n_cells_phys, per_seq_cells, plan, plan_stride, seq_lens,
                         S, H, Hk, D, scale, out, lse, n_threads);
}

/* Q4_0 keys and values. */
int oracle_decode_q4_0(const uint16_t* q, const uint8_t* k_q4, const uint16_t* k_d,
                       const uint8_t* v_q4, const uint16_t* v_d,
                       int64_t n_cells_phys, int64_t per_seq_cells,
                       const int32_t* plan, int64_t plan_stride, const int64_t* seq_lens,
                       int S, int H, int Hk, int D, double scale,
                       double* out, double* lse, int n_threads) {
    if (D % 32 != 0) return -1;
    kv_source K = {ORACLE_KV_Q4_0, k_q4, k_d}, V = {ORACLE_KV_Q4_0, v_q4, v_d};
    return oracle_decode(q, 0, &K, &V, n_cells_phys, per_seq_cells, plan, plan_stride, seq_lens,
                         S, H, Hk, D, scale, out, lse, n_threads);
}

/* fp64 inputs throughout (used to pin the front ends against explicitly converted data). */
int oracle_decode_f64(const double* q, const double* k, const double* v,
                      int64_t n_cells_phys, int64_t per_seq_cells,
                      const int32_t* plan, int64_t plan_stride, const int64_t* seq_lens,
                      int S, int H, int Hk, int D, double scale,
                      double* out, double* lse, int n_threads) {
    kv_source K = {ORACLE_KV_F64, k, NULL}, V = {ORACLE_KV_F64, v, NULL};
    return oracle_decode(q, 1, &K, &V, n_cells_phys, per_seq_cells, plan, plan_stride, seq_lens,
                         S, H, Hk, D, scale, out, lse, n_threads);
}

/* parts: double [P][R][D], lses: double [P][R] -> out [R][D], lse [R]. */
int oracle_merge(const double* parts, const double* lses, int P, int R, int D,
                 double* out, double* lse) {
    if (P < 0 || R < 0 || D <= 0) return -1;
    for (int r = 0; r < R; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < P; ++p) {
            double x = lses[(int64_t)p * R + r];
            if (x > M) M = x;
        }
        double* o = out + (int64_t)r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int p = 0; p < P; ++p) {
            double x = lses[(int64_t)p * R + r];
            if (x == -INFINITY) continue;
            double w = exp(x - M);
            wsum += w;
            const double* op = parts + ((int64_t)p * R + r) * D;
            for (int d = 0; d < D; ++d) o[d] += w * op[d];
        }
        for (int d = 0; d < D; ++d) o[d] /= wsum;
        lse[r] = M + log(wsum);
    }
    return 0;
}
