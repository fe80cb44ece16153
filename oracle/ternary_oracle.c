/*
 * ternary_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the ternary-weight
 * linear layer computes.  It exists so that the CUDA path can be checked
 * against something written independently of it; nothing in the product
 * (the CUDA library and its Python binding) includes, links or calls this
 * file.  Only tests/, the smoke check in __graft_entry__.py and the CPU
 * baseline leg of bench.py may load it.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战"
 *        (trdm.cn/news/729035)
 *          §1.1  values {-1,0,+1}; 128 consecutive weights share one fp16 scale
 *          §3.1  packing rule: 00->0, 01->+1, 10->-1, 11 reserved and read as 0;
 *                four weights per byte, little-endian, first weight in the
 *                lowest two bits; scale blocks cut contiguously along K
 *          §4.2  y = x W^T with x[M,K], W packed as [N,K/4] u8,
 *                scale[N,K/128]; the scale multiplies the block sum at the
 *                block boundary
 *   [P2] the Qwen2.5-7B ternary-in-vLLM write-up (m.nxbn.cn/news/169761)
 *          §2.2  same code table; the four 2-bit fields of a byte are read
 *                low bits first
 *          §3.2  per-output-channel scale [N] multiplies row n
 *                (scale.view(-1,1), i.e. broadcast along K)
 *          §4.2  Y[m,n] = scale[n] * sum_k t[n,k] * X[m,k]
 *          §2.3  packing needs the input width K to be a multiple of 4; an
 *                export whose K is not pads each row up to whole bytes, and
 *                the padding fields must be cut off after unpacking.  Read
 *                here as: a row of K weights takes ceil(K/4) bytes, fields
 *                at k >= K are padding, pack writes them as 00, unpack and
 *                every product skip them (they are not weights, so an 11
 *                there is not counted as reserved)
 *
 * Precision: everything is fp64.  The callers convert fp16 / bf16 inputs to
 * fp64 exactly before calling in, so the only rounding here is the fp64
 * summation, which is far below any tolerance used against the GPU.
 *
 * Threading: oracle_linear_f64 may split the output rows n over POSIX
 * threads.  Every y[m,n] is still computed by one thread in the order written
 * below; threads only decide which n each of them takes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

/* [P1] §3.1, [P2] §2.2: the value a 2-bit code stands for. */
int oracle_trit(unsigned code)
{
    switch (code) {
    case 0: return 0;   /* 00 -> 0                       */
    case 1: return 1;   /* 01 -> +1                      */
    case 2: return -1;  /* 10 -> -1                      */
    case 3: return 0;   /* 11 -> reserved, read as 0     */
    default: return 0;
    }
}

/* Bytes per packed row of K weights ([P2] §2.3: whole bytes, padded). */
static int64_t row_bytes(int64_t K)
{
    return (K + 3) / 4;
}

/* The 2-bit code of weight k in a packed row: byte k/4, field k%4, where
 * field j occupies bits [2j+1 : 2j] ([P1] §3.1 "first weight in the lowest
 * two bits", [P2] §2.2 "from low bits to high bits"). */
static unsigned code_of(const uint8_t *row, int64_t k)
{
    unsigned byte = row[k / 4];
    unsigned field = (unsigned)(k % 4);
    return (byte >> (2u * field)) & 3u;
}

/* packed [N, ceil(K/4)] u8 -> t [N, K] int8 in {-1,0,+1}.
 * reserved_count (nullable) receives the number of 11 fields seen among the
 * K weights of each row (padding fields are not looked at). */
void oracle_unpack(const uint8_t *packed, int8_t *t, int64_t N, int64_t K,
                   int64_t *reserved_count)
{
    int64_t reserved = 0;
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t *row = packed + n * row_bytes(K);
        for (int64_t k = 0; k < K; ++k) {
            unsigned c = code_of(row, k);
            if (c == 3) ++reserved;
            t[n * K + k] = (int8_t)oracle_trit(c);
        }
    }
    if (reserved_count) *reserved_count = reserved;
}

/* The inverse of the code table for the three legal values. */
static unsigned code_for(int v, int *ok)
{
    *ok = 1;
    if (v == 0) return 0u;
    if (v == 1) return 1u;
    if (v == -1) return 2u;
    *ok = 0;
    return 0u;      /* an illegal value is written as 00 and counted */
}

/* t [N, K] int8 -> packed [N, ceil(K/4)] u8.  Never writes the reserved code
 * 11; padding fields (k >= K) are written as 00.
 * Returns the number of entries outside {-1,0,+1}. */
int64_t oracle_pack(const int8_t *t, uint8_t *packed, int64_t N, int64_t K)
{
    int64_t invalid = 0;
    const int64_t Kq = row_bytes(K);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < Kq; ++i) {
            unsigned byte = 0;
            for (unsigned j = 0; j < 4; ++j) {
                const int64_t k = 4 * i + j;
                if (k >= K) break; /* padding: 00 */
                int ok;
                unsigned c = code_for(t[n * K + k], &ok);
                if (!ok) ++invalid;
                byte |= c << (2u * j);
            }
            packed[n * Kq + i] = (uint8_t)byte;
        }
    }
    return invalid;
}

/*
 * y[m,n] for the ternary linear layer, in fp64.
 *
 *   group_size == 0  (per-channel, [P2] §3.2, §4.2):
 *       y[m,n] = s[n] * sum_{k<K} t[n,k] * x[m,k]
 *   group_size == G > 0  (per-group along K, [P1] §1.1, §3.1, §4.2):
 *       y[m,n] = sum_{g<K/G} s[n,g] * ( sum_{k in [gG, gG+G)} t[n,k] * x[m,k] )
 *
 * x: [M,K] fp64 row-major; scale: [N] or [N, K/G] fp64 row-major;
 * packed: [N, ceil(K/4)] u8; y: [M,N] fp64 row-major.
 */
typedef struct {
    const double *x;
    const uint8_t *packed;
    const double *scale;
    int64_t group_size, M, N, K;
    double *y;
    int64_t n_begin, n_end;
} lin_job;

static void *linear_rows(void *arg)
{
    lin_job *j = (lin_job *)arg;
    const int64_t K = j->K, M = j->M, N = j->N;
    int8_t *trow = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    for (int64_t n = j->n_begin; n < j->n_end; ++n) {
        /* decode row n once with the code table */
        oracle_unpack(j->packed + n * row_bytes(K), trow, 1, K, NULL);
        for (int64_t m = 0; m < M; ++m) {
            const double *xm = j->x + m * K;
            double y;
            if (j->group_size == 0) {
                double dot = 0.0;
                for (int64_t k = 0; k < K; ++k) dot += (double)trow[k] * xm[k];
                y = j->scale[n] * dot;
            } else {
                const int64_t G = j->group_size, ng = K / G;
                y = 0.0;
                for (int64_t g = 0; g < ng; ++g) {
                    double part = 0.0;
                    for (int64_t k = g * G; k < (g + 1) * G; ++k)
                        part += (double)trow[k] * xm[k];
                    y += j->scale[n * ng + g] * part;
                }
            }
            j->y[m * N + n] = y;
        }
    }
    free(trow);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments. nthreads <= 1 runs inline. */
int oracle_linear_f64(const double *x, const uint8_t *packed, const double *scale,
                      int64_t group_size, double *y, int64_t M, int64_t N,
                      int64_t K, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (group_size < 0 || (group_size > 0 && K % group_size != 0)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = (int)(N > 0 ? N : 1);
    lin_job *jobs = (lin_job *)calloc((size_t)nthreads, sizeof(lin_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].x = x; jobs[i].packed = packed; jobs[i].scale = scale;
        jobs[i].group_size = group_size; jobs[i].M = M; jobs[i].N = N;
        jobs[i].K = K; jobs[i].y = y;
        jobs[i].n_begin = N * i / nthreads;
        jobs[i].n_end = N * (i + 1) / nthreads;
    }
    if (nthreads == 1) {
        linear_rows(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&tid[i], NULL, linear_rows, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) pthread_join(tid[i], NULL);
    }
    free(jobs);
    free(tid);
    return 0;
}

/*
 * Gated product of a stacked gate/up layer: the pages quantise the gate, up
 * and down projections of a Qwen2.5-7B-architecture MLP ("三元量化模型接入vLLM：
 * 从逆向加载到Kernel优化的完整实战" §1.1, §1.3) but do not write out its
 * activation; that architecture's MLP feeds down_proj with silu(gate) * up,
 * silu(v) = v / (1 + exp(-v)).
 *   packed / scale hold 2N rows: gate rows [0, N), then up rows [N, 2N);
 *   h[m, j] = silu(g[m, j]) * u[m, j] with g, u the fp64 results of
 *   oracle_linear_f64 over those rows.  h is [M, N].  Returns 0, or -1 on bad
 *   arguments (as oracle_linear_f64) or when memory runs out.
 */
int oracle_silu_mul_f64(const double *x, const uint8_t *packed, const double *scale,
                        int64_t group_size, double *h, int64_t M, int64_t N, int64_t K,
                        int nthreads)
{
    if (M < 0 || N < 0) return -1;
    double *y = (double *)malloc((size_t)(M * 2 * N > 0 ? M * 2 * N : 1) * sizeof(double));
    if (!y) return -1;
    int rc = oracle_linear_f64(x, packed, scale, group_size, y, M, 2 * N, K, nthreads);
    if (rc == 0) {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t j = 0; j < N; ++j) {
                const double g = y[m * 2 * N + j], u = y[m * 2 * N + N + j];
                h[m * N + j] = g / (1.0 + exp(-g)) * u;
            }
    }
    free(y);
    return rc;
}

/*
 * Zero-block map for skipping all-zero weight blocks ([P1] §6: ternary weights
 * often come with sparse structure, and a mask of all-zero blocks lets the
 * kernel skip them).  Block (rb, kb) covers rows [128*rb, 128*rb + 128) and
 * weights k in [64*kb, 64*kb + 64), clipped to [0, N) x [0, K).  Its bit is 1
 * when any weight in it decodes to a non-zero value with the code table above
 * (so a block of 00 and 11 codes only is a zero block).
 *   mask: uint32 [ceil(N/128)][ceil(ceil(K/64)/32)], bit kb%32 of word kb/32.
 *   packed: [N, ceil(K/4)]; padding fields are not weights and never light a
 *   block.
 * Returns the number of zero blocks.
 */
int64_t oracle_block_mask(const uint8_t *packed, int64_t N, int64_t K, uint32_t *mask)
{
    const int64_t RB = (N + 127) / 128, KB = (K + 63) / 64, W = (KB + 31) / 32;
    int64_t zero = 0;
    for (int64_t i = 0; i < RB * W; ++i) mask[i] = 0u;
    for (int64_t rb = 0; rb < RB; ++rb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            int live = 0;
            for (int64_t n = 128 * rb; n < 128 * rb + 128 && n < N && !live; ++n) {
                const uint8_t *row = packed + n * row_bytes(K);
                for (int64_t k = 64 * kb; k < 64 * kb + 64 && k < K; ++k) {
                    if (oracle_trit(code_of(row, k)) != 0) {
                        live = 1;
                        break;
                    }
                }
            }
            if (live) mask[rb * W + kb / 32] |= 1u << (kb % 32);
            else ++zero;
        }
    }
    return zero;
}
