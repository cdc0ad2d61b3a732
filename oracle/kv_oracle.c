/*
 * kv_oracle.c -- float64 CPU oracle for the decode step over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference arm may load this code.  It shares nothing with the
 * CUDA library (no header, helper, table or constant): every step below is the
 * plain definition, written out so that it can be checked against the pages by
 * eye.  Sources, by page and section:
 *
 *  [P1] xuewyang.github.io/posts/kv -- "Prefill and decode" (the new token's K/V
 *       are appended first, then the query attends over all cached tokens),
 *       "A toy vLLM: continuous batching with a paged cache" and "Reading the
 *       code: a warehouse of lockers" (token pos goes to table entry pos / BLOCK,
 *       slot pos % BLOCK; the gather reassembles the contiguous cache).
 *  [P2] brunomaga.github.io "inference-prefill-decode-roofline-cache" --
 *       "PagedAttention: memory management for the KV cache" (PagedKVCache.append
 *       and paged_decode_attention: scores q.K / sqrt(h), masked softmax, @ V).
 *  [P3] learn.mohebi.ai "LLM inference serving: KV cache, batching, paging and
 *       speculative decoding" -- section 3 notation (g = a / n_kv query heads per
 *       KV head) and "PagedAttention (4.1-4.3)" (block-by-block reads merged by
 *       the online-softmax update; split-KV decoding in section 6).
 *  [P4] 4yush.com "The KV cache and the systems around it" -- "Why the keys and
 *       values never change": with `start` cached tokens and T new ones, new token
 *       r sits at position start + r and sees keys 0 .. start + r.
 *  [P5] kongchang.com "Core Mechanics of LLM Inference Serving" -- GQA: 32 query
 *       heads in 8 groups of 4 sharing one KV head.
 *  [P1] again, "MLA: how does decode get full-size keys and values back?" -- the
 *       absorbed form of multi-head latent attention: every head scores one shared
 *       cached vector (latent + rotary key) and averages its latent part.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes): query head h uses KV head h / g (contiguous groups); the
 * context length counts the appended token; the split-KV merge is the standard
 * log-sum-exp identity; the fp8 cache is OCP e4m3fn, code = RNE_sat(fl32(x /
 * scale)), decoded as code * scale.
 *
 * Everything floating-point is double, except the one step the fp8 format
 * fixes in single precision (the quotient x / scale that is then rounded to
 * e4m3), so that the encoder's integer decision is taken in the same precision
 * as the device's.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVO_BF16 0
#define KVO_FP8_E4M3 1

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* bf16: 1 sign, 8 exponent (bias 127), 7 mantissa bits -- the top half of an
 * IEEE binary32.  Decoded from the fields, not by reinterpreting memory. */
double kvo_bf16_value(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int e = (bits >> 7) & 0xFF;
    int m = bits & 0x7F;
    double v;
    if (e == 0xFF) {
        v = m ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, -126 - 7);              /* subnormal: m/128 * 2^-126 */
    } else {
        v = ldexp(1.0 + (double)m / 128.0, e - 127);
    }
    return sign ? -v : v;
}

/* e4m3fn (OCP FP8): 1 sign, 4 exponent (bias 7), 3 mantissa bits.  No
 * infinities; S.1111.111 is NaN; largest finite magnitude 1.75 * 2^8 = 448;
 * subnormals m/8 * 2^-6 (smallest 2^-9). */
double kvo_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round-half-to-even of a non-negative double to an integer. */
static double round_half_even(double x)
{
    double f = floor(x);
    double r = x - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Encode a binary32 value as e4m3fn: round to nearest, ties to even, and
 * saturate magnitudes above 448 to 448 (the largest finite code); NaN -> NaN. */
uint8_t kvo_e4m3_from_float(float xf)
{
    double x = (double)xf;                   /* exact */
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return 0x7F | sign;
    double a = fabs(x);
    if (a > 448.0)
        return sign | 0x7E;                  /* e = 15, m = 6: 448 */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9 */
        double n = round_half_even(a * 512.0);      /* exact scaling by 2^9 */
        /* n == 8 is the smallest normal 2^-6, whose code is also 8 */
        return sign | (uint8_t)n;
    }
    int ex;
    (void)frexp(a, &ex);                     /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                          /* a in [2^e, 2^(e+1)) */
    double n = round_half_even(ldexp(a, 3 - e));    /* in [8, 16] */
    if (n == 16.0) { n = 8.0; e += 1; }
    int field = e + 7;
    int mant = (int)n - 8;
    if (field > 15 || (field == 15 && mant == 7))
        return sign | 0x7E;                  /* rounded past 448: saturate */
    return sign | (uint8_t)((field << 3) | mant);
}

/* The fp8 cache stores code = e4m3(fl32(x / scale)), x the bf16 input. */
uint8_t kvo_e4m3_quantize(uint16_t x_bf16, float scale)
{
    float x = (float)kvo_bf16_value(x_bf16);     /* exact in binary32 */
    volatile float q = x / scale;                /* one correctly rounded binary32 division */
    return kvo_e4m3_from_float(q);
}

/* Value of stored element i of a pool row, as the cache defines it. */
static double stored_value(const uint8_t* base, int dtype, size_t i, double scale)
{
    if (dtype == KVO_BF16) {
        uint16_t b;
        memcpy(&b, base + 2 * i, 2);
        return kvo_bf16_value(b);
    }
    return kvo_e4m3_value(base[i]) * scale;
}

/* ------------------------------------------------------------------------- */
/* Append: the expected pool image ([P1] write_kv, [P2] PagedKVCache.append)  */
/* ------------------------------------------------------------------------- */

/*
 * For token i: seq = token_seq ? token_seq[i] : i; pos = token_pos ?
 * token_pos[i] : context_lens[seq] - 1.  Table entry pos / block_size names the
 * physical block, slot pos % block_size the row in it; the K and V of every
 * kv head of the token are written there.  bf16 entries are copied bit for bit;
 * fp8 entries are quantised per kv head.
 * Returns the number of tokens whose address was invalid (those are skipped).
 */
int kvo_append(uint8_t* k_pool, uint8_t* v_pool, int dtype, int num_blocks, int block_size,
               int kv_heads, int head_dim, const uint16_t* k_new, const uint16_t* v_new,
               int num_tokens, const int32_t* token_seq, const int32_t* token_pos,
               const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
               int batch, const float* k_scale, const float* v_scale)
{
    int bad = 0;
    size_t eb = (dtype == KVO_BF16) ? 2 : 1;
    size_t row = (size_t)kv_heads * head_dim;        /* elements per token */
    for (int i = 0; i < num_tokens; ++i) {
        int seq = token_seq ? token_seq[i] : i;
        if (seq < 0 || seq >= batch) { ++bad; continue; }
        int pos = token_pos ? token_pos[i] : context_lens[seq] - 1;
        if (pos < 0 || pos / block_size >= max_blocks) { ++bad; continue; }
        int entry = pos / block_size;
        int slot = pos % block_size;
        int block = block_tables[(size_t)seq * max_blocks + entry];
        if (block < 0 || block >= num_blocks) { ++bad; continue; }
        size_t dst = ((size_t)block * block_size + slot) * row;
        for (int h = 0; h < kv_heads; ++h) {
            for (int c = 0; c < head_dim; ++c) {
                size_t s = (size_t)i * row + (size_t)h * head_dim + c;
                size_t o = dst + (size_t)h * head_dim + c;
                if (dtype == KVO_BF16) {
                    memcpy(k_pool + 2 * o, &k_new[s], 2);
                    memcpy(v_pool + 2 * o, &v_new[s], 2);
                } else {
                    k_pool[o] = kvo_e4m3_quantize(k_new[s], k_scale[h]);
                    v_pool[o] = kvo_e4m3_quantize(v_new[s], v_scale[h]);
                }
            }
        }
        (void)eb;
    }
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Gather ([P1] read_kv): follow the table, line the slots up, drop the tail  */
/* ------------------------------------------------------------------------- */

/* out: double [ctx, kv_heads, head_dim], token t from block table_row[t / bs]
 * at slot t % bs.  Returns -1 if an entry is outside the pool. */
int kvo_gather(const uint8_t* pool, int dtype, int num_blocks, int block_size, int kv_heads,
               int head_dim, const int32_t* table_row, int ctx, const float* scale, double* out)
{
    size_t eb = (dtype == KVO_BF16) ? 2 : 1;
    size_t row = (size_t)kv_heads * head_dim;
    for (int t = 0; t < ctx; ++t) {
        int block = table_row[t / block_size];
        if (block < 0 || block >= num_blocks) return -1;
        const uint8_t* src = pool + ((size_t)block * block_size + (t % block_size)) * row * eb;
        for (int h = 0; h < kv_heads; ++h)
            for (int c = 0; c < head_dim; ++c)
                out[(size_t)t * row + (size_t)h * head_dim + c] =
                    stored_value(src, dtype, (size_t)h * head_dim + c,
                                 dtype == KVO_BF16 ? 1.0 : (double)scale[h]);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Attention of one query over a contiguous cache ([P2] paged_decode_attention) */
/* ------------------------------------------------------------------------- */

/*
 * q: [q_heads, d]; k, v: [ctx, kv_heads, d].  For every query head h, with
 * kv = h / g (g = q_heads / kv_heads):
 *   s_t = scale * sum_c q[h,c] k[t,kv,c]          (t < ctx)
 *   m   = max_t s_t,   w_t = exp(s_t - m)
 *   out[h,:] = sum_t w_t v[t,kv,:] / sum_t w_t,   lse[h] = m + log sum_t w_t
 * ctx == 0 leaves out = 0 and lse = -inf (an empty sequence attends to nothing).
 */
void kvo_attend(const double* q, int q_heads, int kv_heads, int head_dim, const double* k,
                const double* v, int ctx, double scale, double* out, double* lse)
{
    int g = q_heads / kv_heads;
    size_t row = (size_t)kv_heads * head_dim;
    double* s = (double*)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
    for (int h = 0; h < q_heads; ++h) {
        int kv = h / g;
        const double* qh = q + (size_t)h * head_dim;
        double* oh = out + (size_t)h * head_dim;
        for (int c = 0; c < head_dim; ++c) oh[c] = 0.0;
        if (ctx <= 0) { if (lse) lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int t = 0; t < ctx; ++t) {
            const double* kt = k + (size_t)t * row + (size_t)kv * head_dim;
            double dot = 0.0;
            for (int c = 0; c < head_dim; ++c) dot += qh[c] * kt[c];
            s[t] = scale * dot;
            if (s[t] > m) m = s[t];
        }
        double l = 0.0;
        for (int t = 0; t < ctx; ++t) {
            double w = exp(s[t] - m);
            const double* vt = v + (size_t)t * row + (size_t)kv * head_dim;
            for (int c = 0; c < head_dim; ++c) oh[c] += w * vt[c];
            l += w;
        }
        for (int c = 0; c < head_dim; ++c) oh[c] /= l;
        if (lse) lse[h] = m + log(l);
    }
    free(s);
}

/*
 * Split-KV form: the tokens are cut into chunks [j*S, (j+1)*S) counted from
 * token 0; chunk j gives (o_j = normalised output, m_j = its max score, l_j =
 * sum exp(s - m_j)); the chunks are merged by the log-sum-exp identity
 *   M = max_j m_j,  w_j = l_j exp(m_j - M),  out = sum_j w_j o_j / sum_j w_j,
 *   lse = M + log sum_j w_j.
 * Chunks with no tokens carry (m = -inf, l = 0) and are skipped.  This is a
 * self-check of the identity, not a separate definition of the result.
 */
void kvo_attend_split(const double* q, int q_heads, int kv_heads, int head_dim,
                      const double* k, const double* v, int ctx, double scale,
                      int split_tokens, int num_chunks, double* out, double* lse)
{
    int g = q_heads / kv_heads;
    size_t row = (size_t)kv_heads * head_dim;
    double* o = (double*)calloc((size_t)num_chunks * head_dim, sizeof(double));
    double* m = (double*)malloc(sizeof(double) * num_chunks);
    double* l = (double*)malloc(sizeof(double) * num_chunks);
    double* sc = (double*)malloc(sizeof(double) * (split_tokens > 0 ? split_tokens : 1));
    for (int h = 0; h < q_heads; ++h) {
        int kv = h / g;
        const double* qh = q + (size_t)h * head_dim;
        for (int j = 0; j < num_chunks; ++j) {
            int t0 = j * split_tokens, t1 = t0 + split_tokens;
            if (t1 > ctx) t1 = ctx;
            double* oj = o + (size_t)j * head_dim;
            for (int c = 0; c < head_dim; ++c) oj[c] = 0.0;
            m[j] = -INFINITY; l[j] = 0.0;
            if (t0 >= t1) continue;
            for (int t = t0; t < t1; ++t) {
                const double* kt = k + (size_t)t * row + (size_t)kv * head_dim;
                double dot = 0.0;
                for (int c = 0; c < head_dim; ++c) dot += qh[c] * kt[c];
                sc[t - t0] = scale * dot;
                if (sc[t - t0] > m[j]) m[j] = sc[t - t0];
            }
            for (int t = t0; t < t1; ++t) {
                double w = exp(sc[t - t0] - m[j]);
                const double* vt = v + (size_t)t * row + (size_t)kv * head_dim;
                for (int c = 0; c < head_dim; ++c) oj[c] += w * vt[c];
                l[j] += w;
            }
            for (int c = 0; c < head_dim; ++c) oj[c] /= l[j];
        }
        double M = -INFINITY;
        for (int j = 0; j < num_chunks; ++j) if (l[j] > 0.0 && m[j] > M) M = m[j];
        double* oh = out + (size_t)h * head_dim;
        for (int c = 0; c < head_dim; ++c) oh[c] = 0.0;
        if (M == -INFINITY) { if (lse) lse[h] = -INFINITY; continue; }
        double wsum = 0.0;
        for (int j = 0; j < num_chunks; ++j) {
            if (l[j] <= 0.0) continue;
            double w = l[j] * exp(m[j] - M);
            for (int c = 0; c < head_dim; ++c) oh[c] += w * o[(size_t)j * head_dim + c];
            wsum += w;
        }
        for (int c = 0; c < head_dim; ++c) oh[c] /= wsum;
        if (lse) lse[h] = M + log(wsum);
    }
    free(o); free(m); free(l); free(sc);
}

/* ------------------------------------------------------------------------- */
/* Batched decode over contiguous per-sequence data (the oracle's own layout) */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t* q; int batch, q_heads, kv_heads, head_dim;
    const uint16_t* k; const uint16_t* v; const int64_t* seq_start; const int32_t* ctx;
    int dtype; const float* k_scale; const float* v_scale; double scale;
    const int32_t* seq_list; int n_list;
    double* out; double* lse;
    int next;                    /* shared work counter */
    pthread_mutex_t lock;
} decode_job;

/* Cache value of element (t, h, c) of sequence b, as the cache stores it:
 * bf16 exactly, or the dequantised fp8 code (quantised here, with the
 * oracle's own encoder, from the same bf16 input the kernel receives). */
static void load_sequence(const decode_job* J, int b, double* kd, double* vd)
{
    size_t row = (size_t)J->kv_heads * J->head_dim;
    size_t n = (size_t)J->ctx[b] * row;
    const uint16_t* ks = J->k + (size_t)J->seq_start[b] * row;
    const uint16_t* vs = J->v + (size_t)J->seq_start[b] * row;
    for (size_t i = 0; i < n; ++i) {
        int h = (int)((i % row) / J->head_dim);
        if (J->dtype == KVO_BF16) {
            kd[i] = kvo_bf16_value(ks[i]);
            vd[i] = kvo_bf16_value(vs[i]);
        } else {
            kd[i] = kvo_e4m3_value(kvo_e4m3_quantize(ks[i], J->k_scale[h])) * (double)J->k_scale[h];
            vd[i] = kvo_e4m3_value(kvo_e4m3_quantize(vs[i], J->v_scale[h])) * (double)J->v_scale[h];
        }
    }
}

static void* decode_worker(void* arg)
{
    decode_job* J = (decode_job*)arg;
    size_t row = (size_t)J->kv_heads * J->head_dim;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int idx = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (idx >= J->n_list) break;
        int b = J->seq_list ? J->seq_list[idx] : idx;
        int ctx = J->ctx[b];
        size_t n = (size_t)(ctx > 0 ? ctx : 1) * row;
        double* kd = (double*)malloc(sizeof(double) * n);
        double* vd = (double*)malloc(sizeof(double) * n);
        double* qd = (double*)malloc(sizeof(double) * (size_t)J->q_heads * J->head_dim);
        if (ctx > 0) load_sequence(J, b, kd, vd);
        for (int i = 0; i < J->q_heads * J->head_dim; ++i)
            qd[i] = kvo_bf16_value(J->q[(size_t)b * J->q_heads * J->head_dim + i]);
        kvo_attend(qd, J->q_heads, J->kv_heads, J->head_dim, kd, vd, ctx, J->scale,
                   J->out + (size_t)idx * J->q_heads * J->head_dim,
                   J->lse ? J->lse + (size_t)idx * J->q_heads : NULL);
        free(kd); free(vd); free(qd);
    }
    return NULL;
}

/*
 * Decode for the sequences listed in seq_list (or all `batch` when NULL):
 * q bf16 [batch, q_heads, d]; k, v bf16 [total_tokens, kv_heads, d] with
 * sequence b's tokens at rows seq_start[b] .. seq_start[b] + ctx[b] - 1.
 * Results go to out [n_list, q_heads, d] and lse [n_list, q_heads] in list
 * order.  Work is spread over `threads` POSIX threads, one sequence at a time.
 */
int kvo_decode(const uint16_t* q, int batch, int q_heads, int kv_heads, int head_dim,
               const uint16_t* k, const uint16_t* v, const int64_t* seq_start,
               const int32_t* context_lens, int dtype, const float* k_scale,
               const float* v_scale, double scale, const int32_t* seq_list, int n_list,
               double* out, double* lse, int threads)
{
    if (kv_heads <= 0 || q_heads % kv_heads != 0) return -1;
    decode_job J;
    J.q = q; J.batch = batch; J.q_heads = q_heads; J.kv_heads = kv_heads; J.head_dim = head_dim;
    J.k = k; J.v = v; J.seq_start = seq_start; J.ctx = context_lens;
    J.dtype = dtype; J.k_scale = k_scale; J.v_scale = v_scale; J.scale = scale;
    J.seq_list = seq_list; J.n_list = seq_list ? n_list : batch;
    J.out = out; J.lse = lse; J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    pthread_t tid[256];
    for (int i = 1; i < threads; ++i) pthread_create(&tid[i], NULL, decode_worker, &J);
    decode_worker(&J);
    for (int i = 1; i < threads; ++i) pthread_join(tid[i], NULL);
    pthread_mutex_destroy(&J.lock);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Several new tokens per sequence ([P1] "A KV cache in PyTorch": attn_cached  */
/* with the shifted mask tril(diagonal = T - t); 4yush.com "Why the keys and   */
/* values never change": the new token r is at position start + r and sees    */
/* keys 0 .. start + r)                                                        */
/* ------------------------------------------------------------------------- */

/*
 * q: bf16 [batch, q_heads, q_len, d]; the sequence's last q_len cached tokens
 * are the new ones, so query i sits at position ctx - q_len + i and attends
 * over the contiguous prefix of ctx - q_len + i + 1 tokens.  Results in list
 * order: out [n_list, q_heads, q_len, d], lse [n_list, q_heads, q_len].
 * A query whose position is negative (ctx < q_len) attends to nothing.
 */
int kvo_decode_multi(const uint16_t* q, int batch, int q_heads, int q_len, int kv_heads,
                     int head_dim, const uint16_t* k, const uint16_t* v,
                     const int64_t* seq_start, const int32_t* context_lens, int dtype,
                     const float* k_scale, const float* v_scale, double scale,
                     const int32_t* seq_list, int n_list, double* out, double* lse)
{
    if (kv_heads <= 0 || q_heads % kv_heads != 0 || q_len <= 0) return -1;
    decode_job J;
    J.q = q; J.batch = batch; J.q_heads = q_heads; J.kv_heads = kv_heads; J.head_dim = head_dim;
    J.k = k; J.v = v; J.seq_start = seq_start; J.ctx = context_lens;
    J.dtype = dtype; J.k_scale = k_scale; J.v_scale = v_scale; J.scale = scale;
    int n = seq_list ? n_list : batch;
    size_t row = (size_t)kv_heads * head_dim;
    double* qi = (double*)malloc(sizeof(double) * (size_t)q_heads * head_dim);
    double* oi = (double*)malloc(sizeof(double) * (size_t)q_heads * head_dim);
    double* li = (double*)malloc(sizeof(double) * (size_t)q_heads);
    for (int idx = 0; idx < n; ++idx) {
        int b = seq_list ? seq_list[idx] : idx;
        int ctx = context_lens[b];
        size_t cnt = (size_t)(ctx > 0 ? ctx : 1) * row;
        double* kd = (double*)malloc(sizeof(double) * cnt);
        double* vd = (double*)malloc(sizeof(double) * cnt);
        if (ctx > 0) load_sequence(&J, b, kd, vd);
        for (int i = 0; i < q_len; ++i) {
            int visible = ctx - q_len + i + 1;          /* keys 0 .. position of query i */
            if (visible < 0) visible = 0;
            for (int h = 0; h < q_heads; ++h)
                for (int c = 0; c < head_dim; ++c)
                    qi[(size_t)h * head_dim + c] = kvo_bf16_value(
                        q[(((size_t)b * q_heads + h) * q_len + i) * head_dim + c]);
            kvo_attend(qi, q_heads, kv_heads, head_dim, kd, vd, visible, scale, oi, li);
            for (int h = 0; h < q_heads; ++h) {
                for (int c = 0; c < head_dim; ++c)
                    out[(((size_t)idx * q_heads + h) * q_len + i) * head_dim + c] =
                        oi[(size_t)h * head_dim + c];
                if (lse) lse[((size_t)idx * q_heads + h) * q_len + i] = li[h];
            }
        }
        free(kd); free(vd);
    }
    free(qi); free(oi); free(li);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Multi-head latent attention, absorbed form ([P1] "MLA: how does decode get */
/* full-size keys and values back?"; [P3] section "Smaller caches").  Each    */
/* token caches one vector c_t of dl latent numbers followed by dr numbers of */
/* the rotary key, shared by all heads.  With W_UK folded into the query and  */
/* W_UV applied after the attention, head h scores every cached vector with   */
/* its whole query and averages only the latent part:                        */
/*   s_t = scale * sum_{c < dl + dr} q[h,c] c_t[c]                            */
/*   out[h, :] = sum_t exp(s_t - m) c_t[0 .. dl-1] / sum_t exp(s_t - m)        */
/*   lse[h] = m + log sum_t exp(s_t - m),  m = max_t s_t                      */
/* ------------------------------------------------------------------------- */
void kvo_mla_attend(const double* q, int q_heads, int dl, int dr, const double* cache, int ctx,
                    double scale, double* out, double* lse)
{
    int dk = dl + dr;
    double* s = (double*)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
    for (int h = 0; h < q_heads; ++h) {
        const double* qh = q + (size_t)h * dk;
        double* oh = out + (size_t)h * dl;
        for (int c = 0; c < dl; ++c) oh[c] = 0.0;
        if (ctx <= 0) { if (lse) lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int t = 0; t < ctx; ++t) {
            const double* ct = cache + (size_t)t * dk;
            double dot = 0.0;
            for (int c = 0; c < dk; ++c) dot += qh[c] * ct[c];
            s[t] = scale * dot;
            if (s[t] > m) m = s[t];
        }
        double l = 0.0;
        for (int t = 0; t < ctx; ++t) {
            double w = exp(s[t] - m);
            const double* ct = cache + (size_t)t * dk;
            for (int c = 0; c < dl; ++c) oh[c] += w * ct[c];
            l += w;
        }
        for (int c = 0; c < dl; ++c) oh[c] /= l;
        if (lse) lse[h] = m + log(l);
    }
    free(s);
}

/*
 * Batch of MLA decodes: q bf16 [batch, q_heads, dl + dr] (the absorbed queries),
 * cache bf16 [total_tokens, dl + dr] with sequence b's tokens at rows
 * seq_start[b] .. seq_start[b] + ctx[b] - 1.  Results for the listed sequences
 * (all when seq_list is NULL) in list order: out [n, q_heads, dl], lse [n, q_heads].
 */
int kvo_mla_decode(const uint16_t* q, int batch, int q_heads, int dl, int dr,
                   const uint16_t* cache, const int64_t* seq_start, const int32_t* context_lens,
                   double scale, const int32_t* seq_list, int n_list, double* out, double* lse)
{
    if (q_heads <= 0 || dl <= 0 || dr < 0) return -1;
    int dk = dl + dr;
    int n = seq_list ? n_list : batch;
    double* qd = (double*)malloc(sizeof(double) * (size_t)q_heads * dk);
    for (int idx = 0; idx < n; ++idx) {
        int b = seq_list ? seq_list[idx] : idx;
        int ctx = context_lens[b];
        size_t cnt = (size_t)(ctx > 0 ? ctx : 1) * dk;
        double* cd = (double*)malloc(sizeof(double) * cnt);
        for (size_t i = 0; ctx > 0 && i < (size_t)ctx * dk; ++i)
            cd[i] = kvo_bf16_value(cache[(size_t)seq_start[b] * dk + i]);
        for (int i = 0; i < q_heads * dk; ++i)
            qd[i] = kvo_bf16_value(q[(size_t)b * q_heads * dk + i]);
        kvo_mla_attend(qd, q_heads, dl, dr, cd, ctx, scale, out + (size_t)idx * q_heads * dl,
                       lse ? lse + (size_t)idx * q_heads : NULL);
        free(cd);
    }
    free(qd);
    return 0;
}
