/*
 * CPU oracle for paged KV attention.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, obviously correct statement of what the paged
 * attention path computes.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA kernels.
 *
 * Every value is decoded from its 16-bit storage pattern into fp64 and all
 * arithmetic is fp64.  Nothing is blocked, fused, partitioned or reordered
 * beyond the plain definitions below:
 *
 *  - Address translation ("vLLM 在 CANN 上的推理优化", section "vLLM 的
 *    PagedAttention 数据结构", the read_kv sketch): logical token index idx of
 *    a sequence lives in logical block idx / block_size at offset
 *    idx % block_size; the block table maps the logical block to a physical
 *    block of the pool.  The slot of a token is
 *    physical_block * block_size + offset.
 *
 *  - Cache write ("vLLM-Ascend 原理", section 2.3 step "KV 写缓存" and
 *    section 2.4 step "KV 追加写"): the new k and v of a token are copied into
 *    its slot; K and V are separate pools (Model Runner V2 notes, section 4.1)
 *    laid out [num_blocks, block_size, num_kv_heads, head_dim] (CANN page,
 *    PagedAttentionKernel sketch, "kv_pool" comment).
 *
 *  - Attention ("vLLM-Ascend 原理", section 2.3, "因果自注意力"): the query at
 *    position i attends to the keys at positions 0..i, softmax, weighted sum of
 *    the values.  For decode (section 2.4, "分页自注意力") the single new query
 *    sits at position seq_len-1 and attends to the whole prefix read through
 *    the block table.  With grouped-query attention several q heads share one
 *    kv head; q head h reads kv head h / (num_q_heads / num_kv_heads).
 *    The softmax is written in its two-pass form: M = max_t s_t,
 *    out = sum_t exp(s_t - M) v_t / sum_t exp(s_t - M), s_t = scale * q.k_t.
 *
 * Readings where the pages are silent: seq_len counts the new token(s);
 * slot < 0 means "no write"; a decode row with seq_len == 0 yields zeros;
 * table entries past ceil(seq_len / block_size) are never read.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_F16 = 0, OR_BF16 = 1 };
enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_TABLE = 2, OR_ERR_SLOT = 3, OR_ERR_NOMEM = 4 };

/* binary16 (IEEE 754-2008, 3.6): 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits.  exponent 0: subnormal f * 2^-24; exponent 31: inf/NaN. */
static double decode_f16(uint16_t h) {
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x400 | f), e - 25);
    return sign ? -v : v;
}

/* bfloat16: the 16 most significant bits of a binary32 (1 sign, 8 exponent
 * bits with bias 127, 7 fraction bits).  Decoded here from the fields. */
static double decode_bf16(uint16_t h) {
    int sign = h >> 15;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);            /* f * 2^(1-127-7) */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x80 | f), e - 134); /* (128+f) * 2^(e-127-7) */
    return sign ? -v : v;
}

/* OCP 8-bit floating point E4M3, "FN" variant: 1 sign bit, 4 exponent bits
 * (bias 7), 3 fraction bits.  Exponent 0: subnormal f * 2^-9.  The patterns
 * S.1111.111 are NaN; there is no infinity; the largest finite value is 448. */
static double decode_e4m3(uint8_t c) {
    int sign = c >> 7;
    int e = (c >> 3) & 0xf;
    int f = c & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8 | f), e - 10);   /* (8+f) * 2^(e-7-3) */
    return sign ? -v : v;
}

/* Nearest E4M3 code to x: round to nearest, ties to the even code (even
 * fraction), saturating to +-448 beyond the finite range; NaN -> NaN.  Found by
 * comparing x with every non-negative finite code (plain and slow). */
static uint8_t encode_e4m3(float xf) {
    double x = (double)xf;
    if (x != x) return 0x7f;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)((neg << 7) | 0x7e);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 0x7f; ++c) {           /* 0x7f is NaN */
        double d = fabs(decode_e4m3((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best_d = d;
            best = c;
        }
    }
    return (uint8_t)((neg << 7) | best);
}

static double g_tab_e4m3[256];
static double g_tab_f16[65536];
static double g_tab_bf16[65536];
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

static void build_tables(void) {
    for (int i = 0; i < 65536; ++i) {
        g_tab_f16[i] = decode_f16((uint16_t)i);
        g_tab_bf16[i] = decode_bf16((uint16_t)i);
    }
    for (int i = 0; i < 256; ++i) g_tab_e4m3[i] = decode_e4m3((uint8_t)i);
}

static const double* table_e4m3(void) {
    pthread_once(&g_once, build_tables);
    return g_tab_e4m3;
}

static const double* table_for(int dtype) {
    pthread_once(&g_once, build_tables);
    return dtype == OR_BF16 ? g_tab_bf16 : g_tab_f16;
}

static int default_threads(int n) {
    if (n > 0) return n;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

/* ------------------------------------------------------------------------ */

int oracle_decode_values(const uint16_t* in, double* out, int64_t n, int dtype) {
    if (dtype != OR_F16 && dtype != OR_BF16) return OR_ERR_ARG;
    const double* tab = table_for(dtype);
    for (int64_t i = 0; i < n; ++i) out[i] = tab[in[i]];
    return OR_OK;
}

/* Slot of every new token.  Sequence b's new tokens are its last q_lens[b]
 * positions, seq_lens[b]-q_lens[b] .. seq_lens[b]-1, packed sequence after
 * sequence into slots[]. */
int oracle_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                        const int32_t* seq_lens, const int32_t* q_lens, int B,
                        int block_size, int num_blocks) {
    if (block_size <= 0 || B < 0) return OR_ERR_ARG;
    int64_t row = 0;
    for (int b = 0; b < B; ++b) {
        int n = seq_lens[b], ql = q_lens[b];
        if (ql < 0 || ql > n) return OR_ERR_ARG;
        for (int i = 0; i < ql; ++i) {
            int64_t idx = (int64_t)n - ql + i;        /* logical token index */
            int64_t logical_block = idx / block_size;
            int64_t offset = idx % block_size;
            if (logical_block >= max_blocks) return OR_ERR_TABLE;
            int64_t phys = block_tables[(int64_t)b * max_blocks + logical_block];
            if (phys < 0 || phys >= num_blocks) return OR_ERR_TABLE;
            slots[row++] = phys * block_size + offset;
        }
    }
    return OR_OK;
}

/* cache[slot / bs][slot % bs][h][:] = key[t][h][:] for every t with slot >= 0 */
int oracle_kv_write(const uint16_t* key, const uint16_t* value, uint16_t* k_cache,
                    uint16_t* v_cache, const int64_t* slots, int64_t T, int num_blocks,
                    int num_kv_heads, int head_dim, int block_size) {
    int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_slots) return OR_ERR_SLOT;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t dst = ((blk * block_size + off) * num_kv_heads + h) * head_dim + d;
                int64_t src = (t * num_kv_heads + h) * head_dim + d;
                k_cache[dst] = key[src];
                v_cache[dst] = value[src];
            }
        }
    }
    return OR_OK;
}

/* E4M3 codes -> fp64 values; fp32 values -> E4M3 codes (rules above). */
int oracle_decode_e4m3(const uint8_t* in, double* out, int64_t n) {
    const double* tab = table_e4m3();
    for (int64_t i = 0; i < n; ++i) out[i] = tab[in[i]];
    return OR_OK;
}

int oracle_encode_e4m3(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = encode_e4m3(in[i]);
    return OR_OK;
}

/* Quantising cache write ("vLLM-Ascend 原理", section 4 "量化": the k and v of
 * a decode step are quantised as they are written into the cache).  Each new
 * element is decoded from its fp16/bf16 pattern, multiplied in fp32 by the
 * fp32 reciprocal scale, and stored as its E4M3 code.  E4M3 pools are
 * head-major ([block][head][offset][d], the library's FP8 layout):
 *   cache[slot / bs][h][slot % bs][d] = e4m3(float(x) * inv_scale). */
int oracle_kv_write_fp8(const uint16_t* key, const uint16_t* value, uint8_t* k_cache, uint8_t* v_cache,
                        const int64_t* slots, int64_t T, int num_blocks, int num_kv_heads, int head_dim,
                        int block_size, int src_dtype, float k_inv_scale, float v_inv_scale) {
    if (src_dtype != OR_F16 && src_dtype != OR_BF16) return OR_ERR_ARG;
    const double* tab = table_for(src_dtype);
    int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_slots) return OR_ERR_SLOT;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t blk = slot / block_size, off = slot % block_size;
                int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim + d;
                int64_t src = (t * num_kv_heads + h) * head_dim + d;
                float kx = (float)tab[key[src]];     /* exact: fp16/bf16 values are floats */
                float vx = (float)tab[value[src]];
                volatile float kq = kx * k_inv_scale; /* one fp32 rounding, no contraction */
                volatile float vq = vx * v_inv_scale;
                k_cache[dst] = encode_e4m3(kq);
                v_cache[dst] = encode_e4m3(vq);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */

typedef struct {
    /* problem */
    const uint16_t *q, *k_cache, *v_cache;
    const uint8_t *k8, *v8;                     /* E4M3 cache (k_cache/v_cache unused) */
    double k_scale, v_scale;                    /* dequantisation scales of the E4M3 cache */
    const double* tab8;
    const int32_t *block_tables, *seq_lens;
    const int64_t *row_seq, *row_pos, *row_qrow; /* per computed row: seq, position, q row */
    int64_t n_rows;
    int max_blocks, Hq, Hkv, D, block_size, num_blocks;
    double scale;
    const double* tab;
    double* out;                                /* [n_rows, Hq, D] */
    int max_len;
    /* work split */
    int64_t u_begin, u_end;                     /* units = row * Hq + h */
    int status;
} job_t;

/* One query (row, head): walk the block table token by token. */
static int attend_one(const job_t* J, int64_t r, int h, double* s, double* qd, double* acc) {
    const int D = J->D, bs = J->block_size;
    const int G = J->Hq / J->Hkv, g = h / G;
    const int64_t b = J->row_seq[r];
    const int64_t pos = J->row_pos[r];
    double* o = J->out + (r * J->Hq + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (pos < 0) return OR_OK;                   /* empty context: zeros */
    const int64_t n = pos + 1;                   /* keys 0..pos inclusive */
    const uint16_t* qp = J->q + (J->row_qrow[r] * J->Hq + h) * D;
    for (int d = 0; d < D; ++d) qd[d] = J->tab[qp[d]];
    double M = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        int64_t lb = t / bs, off = t % bs;
        if (lb >= J->max_blocks) return OR_ERR_TABLE;
        int64_t phys = J->block_tables[b * J->max_blocks + lb];
        if (phys < 0 || phys >= J->num_blocks) return OR_ERR_TABLE;
        const int64_t koff = ((phys * bs + off) * J->Hkv + g) * D;
        double dot = 0.0;
        if (J->k8) {
            const uint8_t* kp = J->k8 + ((phys * J->Hkv + g) * bs + off) * D;   /* head-major */
            for (int d = 0; d < D; ++d) dot += qd[d] * (J->tab8[kp[d]] * J->k_scale);
        } else {
            const uint16_t* kp = J->k_cache + koff;
            for (int d = 0; d < D; ++d) dot += qd[d] * J->tab[kp[d]];
        }
        s[t] = J->scale * dot;
        if (s[t] > M) M = s[t];
    }
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    double L = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        int64_t lb = t / bs, off = t % bs;
        int64_t phys = J->block_tables[b * J->max_blocks + lb];
        const int64_t voff = ((phys * bs + off) * J->Hkv + g) * D;
        double w = exp(s[t] - M);
        L += w;
        if (J->v8) {
            const uint8_t* vp = J->v8 + ((phys * J->Hkv + g) * bs + off) * D;   /* head-major */
            for (int d = 0; d < D; ++d) acc[d] += w * (J->tab8[vp[d]] * J->v_scale);
        } else {
            const uint16_t* vp = J->v_cache + voff;
            for (int d = 0; d < D; ++d) acc[d] += w * J->tab[vp[d]];
        }
    }
    for (int d = 0; d < D; ++d) o[d] = acc[d] / L;
    return OR_OK;
}

static void* worker(void* arg) {
    job_t* J = (job_t*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)(J->max_len > 0 ? J->max_len : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)J->D);
    double* acc = (double*)malloc(sizeof(double) * (size_t)J->D);
    if (!s || !qd || !acc) {
        J->status = OR_ERR_NOMEM;
    } else {
        for (int64_t u = J->u_begin; u < J->u_end; ++u) {
            int rc = attend_one(J, u / J->Hq, (int)(u % J->Hq), s, qd, acc);
            if (rc) { J->status = rc; break; }
        }
    }
    free(s); free(qd); free(acc);
    return NULL;
}

static int run_rows(const job_t* proto, int num_threads) {
    int64_t units = proto->n_rows * proto->Hq;
    int nt = default_threads(num_threads);
    if (nt > units) nt = units > 0 ? (int)units : 1;
    job_t* jobs = (job_t*)calloc((size_t)nt, sizeof(job_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return OR_ERR_NOMEM; }
    for (int i = 0; i < nt; ++i) {
        jobs[i] = *proto;
        jobs[i].u_begin = units * i / nt;
        jobs[i].u_end = units * (i + 1) / nt;
        jobs[i].status = OR_OK;
    }
    int status = OR_OK;
    if (nt == 1) {
        worker(&jobs[0]);
    } else {
        for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, worker, &jobs[i]);
        for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    }
    for (int i = 0; i < nt; ++i) if (jobs[i].status) status = jobs[i].status;
    free(jobs); free(th);
    return status;
}

static int check_common(int B, int Hq, int Hkv, int D, int block_size, int dtype) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return OR_ERR_ARG;
    if (Hq % Hkv) return OR_ERR_ARG;
    if (dtype != OR_F16 && dtype != OR_BF16) return OR_ERR_ARG;
    return OR_OK;
}

/* Decode: one query per sequence, q [B, Hq, D] -> out [n, Hq, D] fp64.
 * sel (optional, n entries) picks which sequences to compute; NULL = all B. */
int oracle_paged_attention_decode(double* out, const uint16_t* q, const uint16_t* k_cache,
                                  const uint16_t* v_cache, const int32_t* block_tables,
                                  int max_blocks, const int32_t* seq_lens, int B, int num_blocks,
                                  int Hq, int Hkv, int D, int block_size, double scale,
                                  int dtype, const int64_t* sel, int64_t n_sel, int num_threads) {
    int rc = check_common(B, Hq, Hkv, D, block_size, dtype);
    if (rc) return rc;
    int64_t n = sel ? n_sel : B;
    int64_t* rs = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1) * 3);
    if (!rs) return OR_ERR_NOMEM;
    int64_t *row_seq = rs, *row_pos = rs + n, *row_q = rs + 2 * n;
    int max_len = 1;
    for (int64_t r = 0; r < n; ++r) {
        int64_t b = sel ? sel[r] : r;
        if (b < 0 || b >= B) { free(rs); return OR_ERR_ARG; }
        row_seq[r] = b;
        row_pos[r] = (int64_t)seq_lens[b] - 1;
        row_q[r] = b;
        if (seq_lens[b] > max_len) max_len = seq_lens[b];
    }
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k_cache = k_cache; J.v_cache = v_cache; J.block_tables = block_tables;
    J.seq_lens = seq_lens; J.row_seq = row_seq; J.row_pos = row_pos; J.row_qrow = row_q;
    J.n_rows = n; J.max_blocks = max_blocks; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.block_size = block_size; J.num_blocks = num_blocks; J.scale = scale;
    J.tab = table_for(dtype); J.out = out; J.max_len = max_len;
    rc = run_rows(&J, num_threads);
    free(rs);
    return rc;
}

/* The rows of a varlen call: row i of sequence b sits at position
 * seq_lens[b] - q_lens[b] + i and sees positions 0..that position
 * ("vLLM-Ascend 原理", section 2.3, causal self-attention; section 2.4: a
 * later chunk reads what earlier chunks wrote).  sel (optional) lists the q
 * rows to compute.  Fills J's row arrays; *buf is freed by the caller. */
static int prefill_rows(job_t* J, int64_t** buf, const int32_t* seq_lens, const int32_t* q_lens, int B,
                        const int64_t* sel, int64_t n_sel) {
    *buf = NULL;
    int64_t T = 0;
    for (int b = 0; b < B; ++b) {
        if (q_lens[b] < 0 || q_lens[b] > seq_lens[b]) return OR_ERR_ARG;
        T += q_lens[b];
    }
    int64_t n = sel ? n_sel : T;
    /* per packed row: sequence, position; per computed row: sequence, position, q row */
    int64_t* m = (int64_t*)malloc(sizeof(int64_t) * (size_t)((T > 0 ? T : 1) * 2 + (n > 0 ? n : 1) * 3));
    if (!m) return OR_ERR_NOMEM;
    int64_t *seq_of = m, *pos_of = m + T;
    int64_t *row_seq = m + 2 * T, *row_pos = row_seq + n, *row_q = row_seq + 2 * n;
    int64_t r = 0;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < q_lens[b]; ++i, ++r) {
            seq_of[r] = b;
            pos_of[r] = (int64_t)seq_lens[b] - q_lens[b] + i;
        }
    int max_len = 1;
    for (int64_t k = 0; k < n; ++k) {
        int64_t qr = sel ? sel[k] : k;
        if (qr < 0 || qr >= T) { free(m); return OR_ERR_ARG; }
        row_seq[k] = seq_of[qr];
        row_pos[k] = pos_of[qr];
        row_q[k] = qr;
        if (pos_of[qr] + 1 > max_len) max_len = (int)(pos_of[qr] + 1);
    }
    J->row_seq = row_seq; J->row_pos = row_pos; J->row_qrow = row_q;
    J->n_rows = n; J->max_len = max_len;
    *buf = m;
    return OR_OK;
}

/* Varlen causal attention over the paged cache.  q [T, Hq, D], rows packed
 * per sequence (q_lens[b] rows each); out is [n, Hq, D] fp64 (n = T, or the
 * sel rows). */
int oracle_paged_attention_prefill(double* out, const uint16_t* q, const uint16_t* k_cache,
                                   const uint16_t* v_cache, const int32_t* block_tables,
                                   int max_blocks, const int32_t* seq_lens,
                                   const int32_t* q_lens, int B, int num_blocks, int Hq, int Hkv,
                                   int D, int block_size, double scale, int dtype,
                                   const int64_t* sel, int64_t n_sel, int num_threads) {
    int rc = check_common(B, Hq, Hkv, D, block_size, dtype);
    if (rc) return rc;
    job_t J;
    memset(&J, 0, sizeof J);
    int64_t* buf = NULL;
    rc = prefill_rows(&J, &buf, seq_lens, q_lens, B, sel, n_sel);
    if (rc) return rc;
    J.q = q; J.k_cache = k_cache; J.v_cache = v_cache; J.block_tables = block_tables;
    J.seq_lens = seq_lens; J.max_blocks = max_blocks; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.block_size = block_size; J.num_blocks = num_blocks; J.scale = scale;
    J.tab = table_for(dtype); J.out = out;
    rc = run_rows(&J, num_threads);
    free(buf);
    return rc;
}

/* Varlen causal attention over a head-major E4M3 cache: the rows of
 * oracle_paged_attention_prefill, the keys and values of
 * oracle_paged_attention_decode_fp8 (k_t = e4m3(code) * k_scale,
 * v_t = e4m3(code) * v_scale; "vLLM-Ascend 原理", section 4 "量化": the cache
 * itself is quantised, so prefill chunks and speculative-verify rows read it
 * the same way decode rows do). */
int oracle_paged_attention_prefill_fp8(double* out, const uint16_t* q, const uint8_t* k_cache,
                                       const uint8_t* v_cache, const int32_t* block_tables, int max_blocks,
                                       const int32_t* seq_lens, const int32_t* q_lens, int B, int num_blocks,
                                       int Hq, int Hkv, int D, int block_size, double scale, int q_dtype,
                                       double k_scale, double v_scale, const int64_t* sel, int64_t n_sel,
                                       int num_threads) {
    int rc = check_common(B, Hq, Hkv, D, block_size, q_dtype);
    if (rc) return rc;
    job_t J;
    memset(&J, 0, sizeof J);
    int64_t* buf = NULL;
    rc = prefill_rows(&J, &buf, seq_lens, q_lens, B, sel, n_sel);
    if (rc) return rc;
    J.q = q; J.k8 = k_cache; J.v8 = v_cache; J.k_scale = k_scale; J.v_scale = v_scale;
    J.tab8 = table_e4m3(); J.block_tables = block_tables;
    J.seq_lens = seq_lens; J.max_blocks = max_blocks; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.block_size = block_size; J.num_blocks = num_blocks; J.scale = scale;
    J.tab = table_for(q_dtype); J.out = out;
    rc = run_rows(&J, num_threads);
    free(buf);
    return rc;
}

/* Decode attention over a head-major E4M3 cache ([block][head][offset][d]):
 * k_t = e4m3(code) * k_scale and
 * v_t = e4m3(code) * v_scale ("vLLM-Ascend 原理", section 4 "量化": blocks
 * are dequantised after being read through the block table), then the same
 * two-pass softmax as oracle_paged_attention_decode, in fp64. */
int oracle_paged_attention_decode_fp8(double* out, const uint16_t* q, const uint8_t* k_cache,
                                      const uint8_t* v_cache, const int32_t* block_tables, int max_blocks,
                                      const int32_t* seq_lens, int B, int num_blocks, int Hq, int Hkv, int D,
                                      int block_size, double scale, int q_dtype, double k_scale, double v_scale,
                                      const int64_t* sel, int64_t n_sel, int num_threads) {
    int rc = check_common(B, Hq, Hkv, D, block_size, q_dtype);
    if (rc) return rc;
    int64_t n = sel ? n_sel : B;
    int64_t* rs = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1) * 3);
    if (!rs) return OR_ERR_NOMEM;
    int64_t *row_seq = rs, *row_pos = rs + n, *row_q = rs + 2 * n;
    int max_len = 1;
    for (int64_t r = 0; r < n; ++r) {
        int64_t b = sel ? sel[r] : r;
        if (b < 0 || b >= B) { free(rs); return OR_ERR_ARG; }
        row_seq[r] = b;
        row_pos[r] = (int64_t)seq_lens[b] - 1;
        row_q[r] = b;
        if (seq_lens[b] > max_len) max_len = seq_lens[b];
    }
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k8 = k_cache; J.v8 = v_cache; J.k_scale = k_scale; J.v_scale = v_scale;
    J.tab8 = table_e4m3(); J.block_tables = block_tables;
    J.seq_lens = seq_lens; J.row_seq = row_seq; J.row_pos = row_pos; J.row_qrow = row_q;
    J.n_rows = n; J.max_blocks = max_blocks; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.block_size = block_size; J.num_blocks = num_blocks; J.scale = scale;
    J.tab = table_for(q_dtype); J.out = out; J.max_len = max_len;
    rc = run_rows(&J, num_threads);
    free(rs);
    return rc;
}

int oracle_num_threads(int requested) { return default_threads(requested); }
