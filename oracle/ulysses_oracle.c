/*
 * Oracle for the Ulysses DistributedAttention forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, single-threaded, deliberately slow C (fp64 arithmetic, no BLAS, no OpenMP,
 * no -ffast-math).  It shares no code, header, table or constant with the CUDA library;
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg call it.
 *
 * What it computes, and the passages it follows:
 *
 *  - AllToAll, by its definition: every rank cuts its input into P chunks, sends chunk i
 *    to rank i, and lays the chunks it receives out in the order of the sending rank
 *    ("大模型分布式训练通信原语及其应用", section 5 "AllToAll（全交换）", definition and
 *    the two-rank example).
 *  - All-to-all #1 (seq -> head): each rank splits its [b, s/P, h, d] tensor along the
 *    head axis into P parts, part j goes to rank j, and each rank concatenates the parts
 *    it receives along the sequence axis in source-rank order
 *    ("02 · DeepSpeed-Ulysses", section 2 "all-to-all 的转置与重分布", send/receive
 *    listing; the batch axis is carried through unchanged).
 *  - All-to-all #2 (head -> seq): the inverse -- split along the sequence axis, concat
 *    along the head axis (same page, same section; section 1 figure caption: the two
 *    exchanges are inverses).
 *  - Local attention: for every local head, softmax(Q K^T / sqrt(d)) V over the full
 *    sequence ("DeepSpeed-Ulysses 深度解析", section "核心设计：沿序列切分 + 两次
 *    All-to-All", step 4), with the causal mask taken on global query/key positions
 *    ("长上下文训练中的 SP 与 CP", section "Ring Attention：Q 留在本地，KV 沿环传递",
 *    causal paragraph) and grouped K/V heads: local query head hh reads local K/V head
 *    hh / (h_q / h_kv).
 *
 * Element types for attention inputs: 0 = binary32, 1 = bfloat16 (the upper 16 bits of a
 * binary32), 2 = binary64.  Decoding is exact; all arithmetic is in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NO_MEMORY 2

typedef unsigned char u8;

/* ------------------------------------------------------------------ AllToAll */

/* send[i*P + j] is rank i's chunk j; after the call recv[j*P + i] holds it. */
void orc_all_to_all(int P, size_t chunk_bytes, const void* const* send, void* const* recv) {
    for (int i = 0; i < P; ++i)
        for (int j = 0; j < P; ++j)
            memcpy(recv[(size_t)j * P + i], send[(size_t)i * P + j], chunk_bytes);
}

/* View x as [outer][n][inner] bytes and cut the middle axis into P equal parts. */
static void split_middle(const u8* x, size_t outer, size_t n, size_t inner, int P, u8* const* parts) {
    size_t np = n / (size_t)P;
    for (int p = 0; p < P; ++p)
        for (size_t o = 0; o < outer; ++o)
            memcpy(parts[p] + o * np * inner, x + (o * n + (size_t)p * np) * inner, np * inner);
}

/* Inverse of split_middle: P parts [outer][np][inner] -> [outer][P*np][inner]. */
static void concat_middle(const u8* const* parts, int P, size_t outer, size_t np, size_t inner, u8* y) {
    size_t n = np * (size_t)P;
    for (int p = 0; p < P; ++p)
        for (size_t o = 0; o < outer; ++o)
            memcpy(y + (o * n + (size_t)p * np) * inner, parts[p] + o * np * inner, np * inner);
}

static u8** alloc_chunks(int P, size_t chunk_bytes) {
    u8** c = (u8**)calloc((size_t)P * P, sizeof(u8*));
    if (!c) return NULL;
    for (size_t i = 0; i < (size_t)P * P; ++i) {
        c[i] = (u8*)malloc(chunk_bytes ? chunk_bytes : 1);
        if (!c[i]) {
            for (size_t k = 0; k < i; ++k) free(c[k]);
            free(c);
            return NULL;
        }
    }
    return c;
}

static void free_chunks(u8** c, int P) {
    if (!c) return;
    for (size_t i = 0; i < (size_t)P * P; ++i) free(c[i]);
    free(c);
}

static int shape_ok(int P, int b, int s, int h, int d, int e) {
    return P >= 1 && b >= 0 && s >= 0 && h >= 1 && d >= 1 && e >= 1 && s % P == 0 && h % P == 0;
}

/*
 * All-to-all #1: in_seq[j] is rank j's [b][s/P][h][d] tensor (element size e bytes);
 * out_head[r] receives rank r's [b][s][h/P][d] tensor.
 */
int orc_seq2head(int P, int b, int s, int h, int d, int e, const void* const* in_seq, void* const* out_head) {
    if (!shape_ok(P, b, s, h, d, e)) return ORC_BAD_ARG;
    size_t S = (size_t)s / P, H = (size_t)h / P;
    size_t chunk = (size_t)b * S * H * d * e;
    u8** send = alloc_chunks(P, chunk);
    u8** recv = alloc_chunks(P, chunk);
    if (!send || !recv) { free_chunks(send, P); free_chunks(recv, P); return ORC_NO_MEMORY; }
    /* each rank j: split [b*S][h][d] along heads into P parts [b*S][H][d] */
    for (int j = 0; j < P; ++j)
        split_middle((const u8*)in_seq[j], (size_t)b * S, (size_t)h, (size_t)d * e, P, send + (size_t)j * P);
    orc_all_to_all(P, chunk, (const void* const*)send, (void* const*)recv);
    /* each rank r: concat the parts from ranks 0..P-1 ([b][S][H*d] each) along seq */
    for (int r = 0; r < P; ++r)
        concat_middle((const u8* const*)(recv + (size_t)r * P), P, (size_t)b, S, H * d * e, (u8*)out_head[r]);
    free_chunks(send, P);
    free_chunks(recv, P);
    return ORC_OK;
}

/*
 * All-to-all #2: in_head[r] is rank r's [b][s][h/P][d] tensor; out_seq[j] receives rank
 * j's [b][s/P][h][d] tensor.
 */
int orc_head2seq(int P, int b, int s, int h, int d, int e, const void* const* in_head, void* const* out_seq) {
    if (!shape_ok(P, b, s, h, d, e)) return ORC_BAD_ARG;
    size_t S = (size_t)s / P, H = (size_t)h / P;
    size_t chunk = (size_t)b * S * H * d * e;
    u8** send = alloc_chunks(P, chunk);
    u8** recv = alloc_chunks(P, chunk);
    if (!send || !recv) { free_chunks(send, P); free_chunks(recv, P); return ORC_NO_MEMORY; }
    /* each rank r: split [b][s][H*d] along seq into P parts [b][S][H*d] */
    for (int r = 0; r < P; ++r)
        split_middle((const u8*)in_head[r], (size_t)b, (size_t)s, H * d * e, P, send + (size_t)r * P);
    orc_all_to_all(P, chunk, (const void* const*)send, (void* const*)recv);
    /* each rank j: concat the parts from ranks 0..P-1 ([b*S][H][d] each) along heads */
    for (int j = 0; j < P; ++j)
        concat_middle((const u8* const*)(recv + (size_t)j * P), P, (size_t)b * S, H, (size_t)d * e, (u8*)out_seq[j]);
    free_chunks(send, P);
    free_chunks(recv, P);
    return ORC_OK;
}

/* ---------------------------------------------------------------- attention */

static double load_elem(const void* base, size_t idx, int dtype) {
    if (dtype == 0) {
        float f;
        memcpy(&f, (const u8*)base + idx * 4, 4);
        return (double)f;
    }
    if (dtype == 1) {
        uint16_t hbits;
        memcpy(&hbits, (const u8*)base + idx * 2, 2);
        uint32_t w = (uint32_t)hbits << 16;
        float f;
        memcpy(&f, &w, 4);
        return (double)f;
    }
    double x;
    memcpy(&x, (const u8*)base + idx * 8, 8);
    return x;
}

/*
 * One query row of softmax(q K^T / sqrt(d)) V.  q_at(c) is element c of the query;
 * key/value rows j are read through the supplied index of their first element.
 * Keys j > i are masked when causal.  Writes d doubles to out.  If no key is visible the
 * row is defined as zero (unreachable for self-attention: the diagonal is visible).
 */
static void attend_row(int s, int d, int causal, int i,
                       const void* qb, size_t q_off, int qdt,
                       const void* kb, const size_t* k_off, const void* vb, const size_t* v_off, int kvdt,
                       double* scores, double* out) {
    double scale = 1.0 / sqrt((double)d);
    int n = causal ? (i + 1 < s ? i + 1 : s) : s;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += load_elem(qb, q_off + (size_t)c, qdt) * load_elem(kb, k_off[j] + (size_t)c, kvdt);
        scores[j] = acc * scale;
        if (scores[j] > m) m = scores[j];
    }
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (n == 0) return;
    double l = 0.0;
    for (int j = 0; j < n; ++j) {
        double p = exp(scores[j] - m);
        scores[j] = p;
        l += p;
    }
    for (int j = 0; j < n; ++j) {
        double w = scores[j] / l;
        for (int c = 0; c < d; ++c) out[c] += w * load_elem(vb, v_off[j] + (size_t)c, kvdt);
    }
}

/*
 * Local attention of one rank in head layout: q [b][s][hq][d], k/v [b][s][hkv][d],
 * out [b][s][hq][d] in double.  hq % hkv == 0.
 */
int orc_attention(int b, int s, int hq, int hkv, int d, int causal, int dtype,
                  const void* q, const void* k, const void* v, double* out) {
    if (b < 0 || s < 0 || hq < 1 || hkv < 1 || d < 1 || hq % hkv) return ORC_BAD_ARG;
    int g = hq / hkv;
    double* scores = (double*)malloc(sizeof(double) * (s ? s : 1));
    size_t* koff = (size_t*)malloc(sizeof(size_t) * (s ? s : 1));
    size_t* voff = (size_t*)malloc(sizeof(size_t) * (s ? s : 1));
    if (!scores || !koff || !voff) { free(scores); free(koff); free(voff); return ORC_NO_MEMORY; }
    for (int bb = 0; bb < b; ++bb)
        for (int hh = 0; hh < hq; ++hh) {
            int kh = hh / g;
            for (int j = 0; j < s; ++j) {
                koff[j] = (((size_t)bb * s + j) * hkv + kh) * d;
                voff[j] = koff[j];
            }
            for (int i = 0; i < s; ++i) {
                size_t qo = (((size_t)bb * s + i) * hq + hh) * d;
                attend_row(s, d, causal, i, q, qo, dtype, k, koff, v, voff, dtype, scores, out + qo);
            }
        }
    free(scores);
    free(koff);
    free(voff);
    return ORC_OK;
}

/*
 * Sampled rows of the whole forward, read straight from the seq-partitioned inputs.
 * Output row n is rank j's O_seq[b][t][gh][:] with (j, b, t, gh) = sample[4n..4n+3].
 * By all-to-all #2 that row is head-layout rank r = gh / (hq/P), local head gh % (hq/P),
 * token i = j*s/P + t; by all-to-all #1 its query is Q_seq[j][b][t][gh] and its keys and
 * values at token i' are rank (i' / (s/P))'s rows i' % (s/P) at kv head
 * r*(hkv/P) + (gh % (hq/P)) / g.  This is the same pipeline written per element, for
 * problem sizes whose full fp64 evaluation is out of reach.
 */
int orc_dist_attn_rows(int P, int b, int s, int hq, int hkv, int d, int causal, int dtype,
                       const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                       int n_samples, const int* sample, double* out) {
    if (P < 1 || s % P || hq % P || hkv % P || hq % hkv || d < 1) return ORC_BAD_ARG;
    int S = s / P, Hq = hq / P, Hk = hkv / P, g = hq / hkv;
    double* scores = (double*)malloc(sizeof(double) * (s ? s : 1));
    if (!scores) return ORC_NO_MEMORY;
    for (int n = 0; n < n_samples; ++n) {
        int j = sample[4 * n], bb = sample[4 * n + 1], t = sample[4 * n + 2], gh = sample[4 * n + 3];
        if (j < 0 || j >= P || bb < 0 || bb >= b || t < 0 || t >= S || gh < 0 || gh >= hq) {
            free(scores);
            return ORC_BAD_ARG;
        }
        int r = gh / Hq, hh = gh % Hq;
        int kv_head = r * Hk + hh / g;
        int i = j * S + t;
        int nvis = causal ? i + 1 : s;
        const void* qb = q_seq[j];
        size_t qo = (((size_t)bb * S + t) * hq + gh) * d;
        double scale = 1.0 / sqrt((double)d);
        double m = -INFINITY;
        for (int jj = 0; jj < nvis; ++jj) {
            int src = jj / S, tt = jj % S;
            size_t ko = (((size_t)bb * S + tt) * hkv + kv_head) * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += load_elem(qb, qo + (size_t)c, dtype) * load_elem(k_seq[src], ko + (size_t)c, dtype);
            scores[jj] = acc * scale;
            if (scores[jj] > m) m = scores[jj];
        }
        double l = 0.0;
        for (int jj = 0; jj < nvis; ++jj) {
            scores[jj] = exp(scores[jj] - m);
            l += scores[jj];
        }
        double* o = out + (size_t)n * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int jj = 0; jj < nvis; ++jj) {
            int src = jj / S, tt = jj % S;
            size_t vo = (((size_t)bb * S + tt) * hkv + kv_head) * d;
            double w = scores[jj] / l;
            for (int c = 0; c < d; ++c) o[c] += w * load_elem(v_seq[src], vo + (size_t)c, dtype);
        }
    }
    free(scores);
    return ORC_OK;
}

/* ----------------------------------------------------------------- backward */

/*
 * Per-row log-sum-exp of the scaled, masked scores of one rank's local attention, in
 * natural-log units: lse[bb][hh][i] = log sum_j exp(q_i . k_j / sqrt(d)).  The training
 * forward saves it so the backward can rebuild the softmax weights.
 */
int orc_attention_lse(int b, int s, int hq, int hkv, int d, int causal, int dtype,
                      const void* q, const void* k, double* lse) {
    if (b < 0 || s < 0 || hq < 1 || hkv < 1 || d < 1 || hq % hkv) return ORC_BAD_ARG;
    int g = hq / hkv;
    double scale = 1.0 / sqrt((double)d);
    double* sc = (double*)malloc(sizeof(double) * (s ? s : 1));
    if (!sc) return ORC_NO_MEMORY;
    for (int bb = 0; bb < b; ++bb)
        for (int hh = 0; hh < hq; ++hh) {
            int kh = hh / g;
            for (int i = 0; i < s; ++i) {
                int n = causal ? i + 1 : s;
                double m = -INFINITY;
                for (int j = 0; j < n; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += load_elem(q, (((size_t)bb * s + i) * hq + hh) * d + c, dtype) *
                               load_elem(k, (((size_t)bb * s + j) * hkv + kh) * d + c, dtype);
                    sc[j] = acc * scale;
                    if (sc[j] > m) m = sc[j];
                }
                double l = 0.0;
                for (int j = 0; j < n; ++j) l += exp(sc[j] - m);
                lse[((size_t)bb * hq + hh) * s + i] = m + log(l);
            }
        }
    free(sc);
    return ORC_OK;
}

/*
 * Gradient of one rank's local attention O = softmax(Q K^T / sqrt(d)) V (head layout),
 * given dO: with P the softmax weights of a row, D_i = sum_c dO_ic O_ic,
 *   dV_j += sum_i P_ij dO_i,   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i = sum_j dS_ij k_j / sqrt(d),   dK_j += sum_i dS_ij q_i / sqrt(d).
 * This is the derivative of the plain definition (the "ordinary attention backward" of
 * "02 · DeepSpeed-Ulysses", section 5).  Grouped K/V heads sum the contributions of their
 * g query heads.  dq [b][s][hq][d], dk/dv [b][s][hkv][d], all double, overwritten.
 */
int orc_attention_bwd(int b, int s, int hq, int hkv, int d, int causal, int dtype,
                      const void* q, const void* k, const void* v, const void* dout,
                      double* dq, double* dk, double* dv) {
    if (b < 0 || s < 0 || hq < 1 || hkv < 1 || d < 1 || hq % hkv) return ORC_BAD_ARG;
    int g = hq / hkv;
    double scale = 1.0 / sqrt((double)d);
    size_t nq = (size_t)b * s * hq * d, nk = (size_t)b * s * hkv * d;
    for (size_t x = 0; x < nq; ++x) dq[x] = 0.0;
    for (size_t x = 0; x < nk; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
    double* p = (double*)malloc(sizeof(double) * (s ? s : 1));
    double* o = (double*)malloc(sizeof(double) * (d ? d : 1));
    if (!p || !o) { free(p); free(o); return ORC_NO_MEMORY; }
    for (int bb = 0; bb < b; ++bb)
        for (int hh = 0; hh < hq; ++hh) {
            int kh = hh / g;
            for (int i = 0; i < s; ++i) {
                int n = causal ? i + 1 : s;
                size_t qo = (((size_t)bb * s + i) * hq + hh) * d;
                /* softmax weights of row i */
                double m = -INFINITY;
                for (int j = 0; j < n; ++j) {
                    size_t ko = (((size_t)bb * s + j) * hkv + kh) * d;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += load_elem(q, qo + c, dtype) * load_elem(k, ko + c, dtype);
                    p[j] = acc * scale;
                    if (p[j] > m) m = p[j];
                }
                double l = 0.0;
                for (int j = 0; j < n; ++j) { p[j] = exp(p[j] - m); l += p[j]; }
                for (int j = 0; j < n; ++j) p[j] /= l;
                /* output row and D_i */
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                for (int j = 0; j < n; ++j) {
                    size_t vo = (((size_t)bb * s + j) * hkv + kh) * d;
                    for (int c = 0; c < d; ++c) o[c] += p[j] * load_elem(v, vo + c, dtype);
                }
                double Di = 0.0;
                for (int c = 0; c < d; ++c) Di += load_elem(dout, qo + c, dtype) * o[c];
                for (int j = 0; j < n; ++j) {
                    size_t ko = (((size_t)bb * s + j) * hkv + kh) * d;
                    double dp = 0.0;
                    for (int c = 0; c < d; ++c) dp += load_elem(dout, qo + c, dtype) * load_elem(v, ko + c, dtype);
                    double ds = p[j] * (dp - Di);
                    for (int c = 0; c < d; ++c) {
                        dv[ko + c] += p[j] * load_elem(dout, qo + c, dtype);
                        dq[qo + c] += ds * load_elem(k, ko + c, dtype) * scale;
                        dk[ko + c] += ds * load_elem(q, qo + c, dtype) * scale;
                    }
                }
            }
        }
    free(p);
    free(o);
    return ORC_OK;
}

/* ------------------------------------------------- Ulysses x Ring (USP, a2a + p2p) */

/* n separately allocated buffers of `bytes` each (NULL if any allocation fails). */
static u8** alloc_bufs(int n, size_t bytes) {
    u8** c = (u8**)calloc((size_t)n, sizeof(u8*));
    if (!c) return NULL;
    for (int i = 0; i < n; ++i) {
        c[i] = (u8*)malloc(bytes ? bytes : 1);
        if (!c[i]) {
            for (int k = 0; k < i; ++k) free(c[k]);
            free(c);
            return NULL;
        }
    }
    return c;
}

static void free_bufs(u8** c, int n) {
    for (int i = 0; i < n; ++i) free(c[i]);
    free(c);
}

/*
 * The two-level forward: P = Pu * Pr ranks, rank j = g*Pu + u holds tokens
 * [j*s/P, (j+1)*s/P) of every head ("长上下文训练中的 SP 与 CP", section "组合与配置：区分算法
 * 组合和并行维度", subsection "Ulysses + Ring：组合两种 Attention 路线": 256K tokens over
 * Ulysses degree 4 x Ring degree 2; "02 · DeepSpeed-Ulysses", section 4 "a2a+p2p 分层 CP":
 * inner a2a, outer p2p ring, the product of the two sizes is the CP size).
 *  1. Inside ring group g (ranks g*Pu .. g*Pu+Pu-1, which together hold the contiguous
 *     segment g of L = s/Pr tokens) all-to-all #1: rank (g, u) gets all L tokens of the
 *     segment for heads [u*hq/Pu, (u+1)*hq/Pu) (and the matching K/V heads).
 *  2. Ring across the Pr groups among the ranks with the same u: rank (g, u) keeps its Q
 *     and processes the K/V segments in the order g, g-1, ..., g-Pr+1 (mod Pr), the blocks
 *     arriving from the neighbour ("Ring Attention：Q 留在本地，KV 沿环传递", the four-rank
 *     example).  Each query row keeps the online-softmax state (m, l, A), starting at
 *     (-inf, 0, 0); a block of scores S raises m to m' = max(m, rowmax S), rescales
 *     l and A by exp(m - m'), adds sum exp(S - m') and sum exp(S - m') v; at the end
 *     O = A / l (same section, online-softmax paragraph).  Causal, on global positions:
 *     blocks after the query segment are skipped, in the query's own segment only keys
 *     at or before the query count (a lower-triangular block), earlier blocks count in
 *     full (same section, causal paragraph).
 *  3. Inside the group, all-to-all #2 back to the sequence split.
 * Inputs: P pointers to [b][s/P][h][d] of `dtype`; out: P pointers to double [b][s/P][hq][d].
 */
int orc_usp_fwd(int Pu, int Pr, int b, int s, int hq, int hkv, int d, int causal, int dtype,
                const void* const* q_seq, const void* const* k_seq, const void* const* v_seq, double* const* out) {
    if (Pu < 1 || Pr < 1 || b < 1 || s < 1 || d < 1 || hq < 1 || hkv < 1) return ORC_BAD_ARG;
    const int P = Pu * Pr;
    if (s % P || hq % Pu || hkv % Pu || hq % hkv) return ORC_BAD_ARG;
    const int e = dtype == 0 ? 4 : (dtype == 1 ? 2 : 8);
    const int L = s / Pr, Hq = hq / Pu, Hk = hkv / Pu, g_q = hq / hkv;
    const size_t qh_bytes = (size_t)b * L * Hq * d * e, kh_bytes = (size_t)b * L * Hk * d * e;
    u8** qh = alloc_bufs(P, qh_bytes);
    u8** kh = alloc_bufs(P, kh_bytes);
    u8** vh = alloc_bufs(P, kh_bytes);
    u8** oh = alloc_bufs(P, (size_t)b * L * Hq * d * sizeof(double));
    double* A = (double*)malloc(sizeof(double) * d);
    double* sc = (double*)malloc(sizeof(double) * L);
    int rc = ORC_OK;
    if (!qh || !kh || !vh || !oh || !A || !sc) rc = ORC_NO_MEMORY;
    /* 1. all-to-all #1 inside every ring group */
    for (int g = 0; g < Pr && rc == ORC_OK; ++g) {
        rc = orc_seq2head(Pu, b, L, hq, d, e, q_seq + g * Pu, (void* const*)(qh + g * Pu));
        if (rc == ORC_OK) rc = orc_seq2head(Pu, b, L, hkv, d, e, k_seq + g * Pu, (void* const*)(kh + g * Pu));
        if (rc == ORC_OK) rc = orc_seq2head(Pu, b, L, hkv, d, e, v_seq + g * Pu, (void* const*)(vh + g * Pu));
    }
    /* 2. the ring, per rank (g, u), query row by query row */
    const double scale = 1.0 / sqrt((double)d);
    for (int g = 0; g < Pr && rc == ORC_OK; ++g)
        for (int u = 0; u < Pu; ++u) {
            const int me = g * Pu + u;
            for (int bb = 0; bb < b; ++bb)
                for (int hh = 0; hh < Hq; ++hh)
                    for (int i = 0; i < L; ++i) {
                        const size_t qo = (((size_t)bb * L + i) * Hq + hh) * d;
                        double m = -INFINITY, l = 0.0;
                        for (int c = 0; c < d; ++c) A[c] = 0.0;
                        for (int t = 0; t < Pr; ++t) {
                            const int src = ((g - t) % Pr + Pr) % Pr; /* block received at step t */
                            if (causal && src > g) continue;       /* after the query segment */
                            const int nk = (causal && src == g) ? i + 1 : L;
                            const u8* kb = kh[src * Pu + u];
                            const u8* vb = vh[src * Pu + u];
                            double bmax = -INFINITY;
                            for (int j = 0; j < nk; ++j) {
                                const size_t ko = (((size_t)bb * L + j) * Hk + hh / g_q) * d;
                                double acc = 0.0;
                                for (int c = 0; c < d; ++c)
                                    acc += load_elem(qh[me], qo + c, dtype) * load_elem(kb, ko + c, dtype);
                                sc[j] = acc * scale;
                                if (sc[j] > bmax) bmax = sc[j];
                            }
                            const double mn = bmax > m ? bmax : m;
                            const double f = exp(m - mn); /* 0 while nothing was seen */
                            l *= f;
                            for (int c = 0; c < d; ++c) A[c] *= f;
                            for (int j = 0; j < nk; ++j) {
                                const double p = exp(sc[j] - mn);
                                const size_t vo = (((size_t)bb * L + j) * Hk + hh / g_q) * d;
                                l += p;
                                for (int c = 0; c < d; ++c) A[c] += p * load_elem(vb, vo + c, dtype);
                            }
                            m = mn;
                        }
                        double* o = (double*)oh[me] + qo;
                        for (int c = 0; c < d; ++c) o[c] = l > 0.0 ? A[c] / l : 0.0;
                    }
        }
    /* 3. all-to-all #2 inside every ring group */
    for (int g = 0; g < Pr && rc == ORC_OK; ++g)
        rc = orc_head2seq(Pu, b, L, hq, d, (int)sizeof(double), (const void* const*)(oh + g * Pu),
                          (void* const*)(out + g * Pu));
    free(A);
    free(sc);
    if (qh) free_bufs(qh, P);
    if (kh) free_bufs(kh, P);
    if (vh) free_bufs(vh, P);
    if (oh) free_bufs(oh, P);
    return rc;
}

/* --------------------------------------------------------- sampled gradient rows */

/*
 * Selected rows of the local attention gradient, for sizes whose full evaluation is out
 * of reach.  The definitions are those of orc_attention_bwd, evaluated per row:
 *   dQ_i = sum_j P_ij (dP_ij - D_i) k_j / sqrt(d)            (query row i of head hh)
 *   dV_j = sum_hh sum_i P_ij dO_i,  dK_j = sum_hh sum_i P_ij (dP_ij - D_i) q_i / sqrt(d)
 * with P_ij = exp(q_i.k_j/sqrt(d) - L_i), L_i the row's log-sum-exp, D_i = dO_i . O_i
 * (O the exact output) and, for key rows, the sum over the query heads hh that read
 * K/V head kvh.  One pass over a (batch, query head) computes L_i and D_i of every row.
 * qs[3n..3n+2] = (bb, i, hh) for dq row n; ks[3n..3n+2] = (bb, j, kvh) for dk/dv row n.
 * Head layout inputs as orc_attention_bwd; outputs double [n][d].
 */
int orc_attention_bwd_rows(int b, int s, int hq, int hkv, int d, int causal, int dtype,
                           const void* q, const void* k, const void* v, const void* dout,
                           int nq, const int* qs, int nk, const int* ks,
                           double* dq, double* dk, double* dv) {
    if (b < 1 || s < 1 || hq < 1 || hkv < 1 || d < 1 || hq % hkv) return ORC_BAD_ARG;
    const int g = hq / hkv;
    const double scale = 1.0 / sqrt((double)d);
    double* L = (double*)malloc(sizeof(double) * s);
    double* D = (double*)malloc(sizeof(double) * s);
    double* sc = (double*)malloc(sizeof(double) * s);
    double* o = (double*)malloc(sizeof(double) * d);
    if (!L || !D || !sc || !o) {
        free(L); free(D); free(sc); free(o);
        return ORC_NO_MEMORY;
    }
#define QI(bb, i, hh, c) load_elem(q, ((((size_t)(bb) * s + (i)) * hq + (hh)) * d + (c)), dtype)
#define DOI(bb, i, hh, c) load_elem(dout, ((((size_t)(bb) * s + (i)) * hq + (hh)) * d + (c)), dtype)
#define KJ(bb, j, kh, c) load_elem(k, ((((size_t)(bb) * s + (j)) * hkv + (kh)) * d + (c)), dtype)
#define VJ(bb, j, kh, c) load_elem(v, ((((size_t)(bb) * s + (j)) * hkv + (kh)) * d + (c)), dtype)
    /* the (batch, query head) pairs any request needs */
    for (int n = 0; n < nq + nk; ++n) {
        const int* smp = n < nq ? qs + 3 * n : ks + 3 * (n - nq);
        if (smp[0] < 0 || smp[0] >= b || smp[1] < 0 || smp[1] >= s || smp[2] < 0 ||
            smp[2] >= (n < nq ? hq : hkv)) {
            free(L); free(D); free(sc); free(o);
            return ORC_BAD_ARG;
        }
    }
    for (int n = 0; n < nq; ++n)
        for (int c = 0; c < d; ++c) dq[(size_t)n * d + c] = 0.0;
    for (int n = 0; n < nk; ++n)
        for (int c = 0; c < d; ++c) dk[(size_t)n * d + c] = dv[(size_t)n * d + c] = 0.0;
    for (int bb = 0; bb < b; ++bb)
        for (int hh = 0; hh < hq; ++hh) {
            const int kh = hh / g;
            int needed = 0;
            for (int n = 0; n < nq; ++n) needed |= qs[3 * n] == bb && qs[3 * n + 2] == hh;
            for (int n = 0; n < nk; ++n) needed |= ks[3 * n] == bb && ks[3 * n + 2] == kh;
            if (!needed) continue;
            /* L_i and D_i of every query row of this (batch, head) */
            for (int i = 0; i < s; ++i) {
                const int nv = causal ? i + 1 : s;
                double m = -INFINITY;
                for (int j = 0; j < nv; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += QI(bb, i, hh, c) * KJ(bb, j, kh, c);
                    sc[j] = acc * scale;
                    if (sc[j] > m) m = sc[j];
                }
                double l = 0.0;
                for (int j = 0; j < nv; ++j) l += exp(sc[j] - m);
                L[i] = m + log(l);
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                for (int j = 0; j < nv; ++j) {
                    const double w = exp(sc[j] - L[i]);
                    for (int c = 0; c < d; ++c) o[c] += w * VJ(bb, j, kh, c);
                }
                double dd = 0.0;
                for (int c = 0; c < d; ++c) dd += DOI(bb, i, hh, c) * o[c];
                D[i] = dd;
            }
            /* requested query rows of this head */
            for (int n = 0; n < nq; ++n) {
                if (qs[3 * n] != bb || qs[3 * n + 2] != hh) continue;
                const int i = qs[3 * n + 1], nv = causal ? i + 1 : s;
                for (int j = 0; j < nv; ++j) {
                    double sij = 0.0, dpij = 0.0;
                    for (int c = 0; c < d; ++c) {
                        sij += QI(bb, i, hh, c) * KJ(bb, j, kh, c);
                        dpij += DOI(bb, i, hh, c) * VJ(bb, j, kh, c);
                    }
                    const double pij = exp(sij * scale - L[i]);
                    const double ds = pij * (dpij - D[i]);
                    for (int c = 0; c < d; ++c) dq[(size_t)n * d + c] += ds * KJ(bb, j, kh, c) * scale;
                }
            }
            /* requested key rows of this head's K/V head: this head's share */
            for (int n = 0; n < nk; ++n) {
                if (ks[3 * n] != bb || ks[3 * n + 2] != kh) continue;
                const int j = ks[3 * n + 1];
                for (int i = causal ? j : 0; i < s; ++i) {
                    double sij = 0.0, dpij = 0.0;
                    for (int c = 0; c < d; ++c) {
                        sij += QI(bb, i, hh, c) * KJ(bb, j, kh, c);
                        dpij += DOI(bb, i, hh, c) * VJ(bb, j, kh, c);
                    }
                    const double pij = exp(sij * scale - L[i]);
                    const double ds = pij * (dpij - D[i]);
                    for (int c = 0; c < d; ++c) {
                        dv[(size_t)n * d + c] += pij * DOI(bb, i, hh, c);
                        dk[(size_t)n * d + c] += ds * QI(bb, i, hh, c) * scale;
                    }
                }
            }
        }
#undef QI
#undef DOI
#undef KJ
#undef VJ
    free(L);
    free(D);
    free(sc);
    free(o);
    return ORC_OK;
}

/* ------------------------------------------------- magnitudes of the gradient terms */

/*
 * For every gradient element of the local attention backward, the sum of the absolute
 * values of the terms that orc_attention_bwd adds up for it -- the quantity that bounds
 * the effect of rounding those terms (each term rounded with relative error u moves the
 * sum by at most u times this magnitude; the textbook error bound of a sum of rounded
 * products).  With P_ij, dP_ij = dO_i . v_j, D_i = dO_i . O_i and dS_ij = P_ij (dP_ij - D_i)
 * as in orc_attention_bwd ("02 · DeepSpeed-Ulysses", section 5: the ordinary attention
 * backward), and
 *   E_i = sum_c |dO_ic| (|O_ic| + sum_j P_ij |v_jc|),
 * the bound on |D_i - D~_i| in units of u when every O_ic is known only to within
 * u (|O_ic| + sum_j P_ij |v_jc|) -- an output formed from rounded weights P_ij and then
 * rounded itself:
 *   mq_ic = sum_j (|dS_ij| + P_ij E_i) |k_jc| / sqrt(d)
 *   mk_jc = sum_hh sum_i (|dS_ij| + P_ij E_i) |q_ic| / sqrt(d)
 *   mv_jc = sum_hh sum_i P_ij |dO_ic|
 * (grouped heads: key rows sum over the query heads hh that read K/V head kvh, exactly as
 * the gradients do).  Same layouts and arguments as orc_attention_bwd.
 */
int orc_attention_bwd_magnitudes(int b, int s, int hq, int hkv, int d, int causal, int dtype,
                                 const void* q, const void* k, const void* v, const void* dout,
                                 double* mq, double* mk, double* mv) {
    if (b < 0 || s < 0 || hq < 1 || hkv < 1 || d < 1 || hq % hkv) return ORC_BAD_ARG;
    int g = hq / hkv;
    double scale = 1.0 / sqrt((double)d);
    size_t nq = (size_t)b * s * hq * d, nk = (size_t)b * s * hkv * d;
    for (size_t x = 0; x < nq; ++x) mq[x] = 0.0;
    for (size_t x = 0; x < nk; ++x) { mk[x] = 0.0; mv[x] = 0.0; }
    double* p = (double*)malloc(sizeof(double) * (s ? s : 1));
    double* o = (double*)malloc(sizeof(double) * (d ? d : 1));
    double* oa = (double*)malloc(sizeof(double) * (d ? d : 1));
    if (!p || !o || !oa) { free(p); free(o); free(oa); return ORC_NO_MEMORY; }
    for (int bb = 0; bb < b; ++bb)
        for (int hh = 0; hh < hq; ++hh) {
            int kh = hh / g;
            for (int i = 0; i < s; ++i) {
                int n = causal ? i + 1 : s;
                size_t qo = (((size_t)bb * s + i) * hq + hh) * d;
                double m = -INFINITY;
                for (int j = 0; j < n; ++j) {
                    size_t ko = (((size_t)bb * s + j) * hkv + kh) * d;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += load_elem(q, qo + c, dtype) * load_elem(k, ko + c, dtype);
                    p[j] = acc * scale;
                    if (p[j] > m) m = p[j];
                }
                double l = 0.0;
                for (int j = 0; j < n; ++j) { p[j] = exp(p[j] - m); l += p[j]; }
                for (int j = 0; j < n; ++j) p[j] /= l;
                /* O_i and sum_j P_ij |v_j| */
                for (int c = 0; c < d; ++c) { o[c] = 0.0; oa[c] = 0.0; }
                for (int j = 0; j < n; ++j) {
                    size_t vo = (((size_t)bb * s + j) * hkv + kh) * d;
                    for (int c = 0; c < d; ++c) {
                        double vv = load_elem(v, vo + c, dtype);
                        o[c] += p[j] * vv;
                        oa[c] += p[j] * fabs(vv);
                    }
                }
                double Di = 0.0, Ei = 0.0;
                for (int c = 0; c < d; ++c) {
                    double g_c = load_elem(dout, qo + c, dtype);
                    Di += g_c * o[c];
                    Ei += fabs(g_c) * (fabs(o[c]) + oa[c]);
                }
                for (int j = 0; j < n; ++j) {
                    size_t ko = (((size_t)bb * s + j) * hkv + kh) * d;
                    double dp = 0.0;
                    for (int c = 0; c < d; ++c) dp += load_elem(dout, qo + c, dtype) * load_elem(v, ko + c, dtype);
                    double w = fabs(p[j] * (dp - Di)) + p[j] * Ei;
                    for (int c = 0; c < d; ++c) {
                        mv[ko + c] += p[j] * fabs(load_elem(dout, qo + c, dtype));
                        mq[qo + c] += w * fabs(load_elem(k, ko + c, dtype)) * scale;
                        mk[ko + c] += w * fabs(load_elem(q, qo + c, dtype)) * scale;
                    }
                }
            }
        }
    free(p);
    free(o);
    free(oa);
    return ORC_OK;
}
