/*
 * infllmv2_oracle.c -- fp64 CPU oracle for InfLLM v2 block-sparse attention.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library; the CUDA library never links it and
 * shares no code, header or table with it.
 *
 * It restates, step by step and with no blocking, fusion or reordering, the
 * method the pages describe:
 *   - "MiniCPM4: 如何在手机电脑上高效运行大语言模型" (xugj520.cn), section 1.1
 *     "InfLLM v2": text split into blocks, overlapping semantic kernels of 32
 *     tokens with stride 16, each query keeps its top-K relevant blocks, the
 *     opening tokens and the sliding-window tokens are always kept, and
 *     attention is computed on the kept blocks only; the tree-speculative
 *     verification mask is a uint64 bit set per draft token.
 *   - "MiniCPM40极速狂飙端侧模型的比赛结束了" (shadowrocket9.top), section
 *     "InfLLM v2：重新定义注意力机制": 64-token blocks, top-64 blocks, dense
 *     attention below 8192 tokens; deployment guide: sparse_config
 *     {topk, block_size, dense_len}.
 * Where the pages leave a step open, the reading taken is stated beside it
 * (R1..R11 in the design notes use the same numbering).
 *
 * Number types: inputs are bf16 bit patterns widened exactly to double; all
 * arithmetic is double.  The semantic-kernel representation is stored as bf16
 * (reading R4), rounded once from the exact fp64 mean.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* integer parameters, in this order */
enum { P_BLOCK = 0, P_KSIZE, P_KSTRIDE, P_TOPK, P_NINIT, P_NLOCAL, P_DENSE_LEN, P_COUNT };

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_CAPACITY (-2)

static double bf16_value(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even.
 * frexp gives |x| = m * 2^e with m in [0.5, 1); scaling m by 2^8 puts the
 * eight kept bits left of the binary point and nearbyint rounds the rest
 * in the default (nearest-even) mode.  Normal range only (reading R9). */
static uint16_t bf16_round(double x) {
    if (x == 0.0) return signbit(x) ? 0x8000u : 0u;
    int e;
    double m = frexp(fabs(x), &e);
    double r = ldexp(nearbyint(m * 256.0), e - 8);
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t h = (uint16_t)(u >> 16);
    return signbit(x) ? (uint16_t)(h | 0x8000u) : h;
}

void orc_bf16_round(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_round(x[i]);
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Number of complete semantic kernels among the first L tokens: kernel j covers
 * tokens [j*s, j*s + c - 1]. */
static int64_t n_kernels(int64_t L, int64_t c, int64_t s) {
    return L < c ? 0 : (L - c) / s + 1;
}

/*
 * Step 1 -- semantic kernels (section 1.1 "InfLLM v2", semantic-kernel item):
 *   kern[b,h,j,:] = bf16( (1/c) * sum_{i=j*s}^{j*s+c-1} K[b,h,i,:] )
 * for every kernel complete within the first kv_len[b] tokens.
 * K: [B,H,L_max,d] bf16; kern: [B,H,M_max,d] bf16; kern_exact (nullable): same
 * shape in double, the mean before rounding.
 */
int orc_kernel_pool(const uint16_t* K, int64_t B, int64_t H, int64_t L_max, int64_t d,
                    const int32_t* kv_len, int32_t c, int32_t s, uint16_t* kern,
                    double* kern_exact, int64_t M_max) {
    if (c <= 0 || s <= 0) return ORC_ERR_ARG;
    for (int64_t b = 0; b < B; ++b) {
        if (kv_len[b] < 0 || kv_len[b] > L_max) return ORC_ERR_ARG;
        if (n_kernels(kv_len[b], c, s) > M_max) return ORC_ERR_CAPACITY;
    }
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            int64_t M = n_kernels(kv_len[b], c, s);
            for (int64_t j = 0; j < M; ++j) {
                for (int64_t x = 0; x < d; ++x) {
                    double sum = 0.0;
                    for (int64_t i = j * s; i < j * s + c; ++i)
                        sum += bf16_value(K[((b * H + h) * L_max + i) * d + x]);
                    double mean = sum / (double)c;
                    int64_t o = ((b * H + h) * M_max + j) * d + x;
                    kern[o] = bf16_round(mean);
                    if (kern_exact) kern_exact[o] = mean;
                }
            }
        }
    }
    return ORC_OK;
}

/* Position of query t: a causal chunk is the last Tq tokens of the cache
 * (reading R10); decode is the chunk with Tq = 1; a tree draft comes after the
 * whole cache, so it sees every cached token and every cached kernel. */
static int64_t query_pos(int64_t kv_len, int64_t Tq, int64_t t, int tree) {
    return tree ? kv_len - 1 : kv_len - Tq + t;
}

/*
 * Step 2 -- block scores (section 1.1, "dynamic block selection"; the max over
 * overlapping kernels and over the heads of a GQA group, so that a group
 * shares one selection):
 *   s(t,h,j)  = q[t,h] . kern[j]                    (unscaled, reading R7)
 *   S[t,g,b]  = max_{h in group g} max_{j overlaps b, j visible to t} s(t,h,j)
 * kernel j overlaps block b iff they share a token (reading R6):
 *   j*s < (b+1)*B_s  and  j*s + c > b*B_s
 * kernel j is visible to the query at position p iff j*s + c - 1 <= p (R2).
 * S has layout [B, Hkv, n_t, nblk_max]; blocks past the query's own block, and
 * blocks with no visible overlapping kernel, hold -inf.
 * q: [B,Tq,Hq,d]; kern: [B,Hkv,M_max,d]; t_list: the n_t queries to score.
 */
int orc_block_scores(const uint16_t* q, const uint16_t* kern, const int32_t* kv_len, int64_t B,
                     int64_t Tq, int64_t Hq, int64_t Hkv, int64_t d, int64_t M_max, int32_t tree,
                     const int32_t* ip, const int32_t* t_list, int64_t n_t, int64_t nblk_max,
                     double* S) {
    const int64_t bs = ip[P_BLOCK], c = ip[P_KSIZE], s = ip[P_KSTRIDE];
    if (Hkv <= 0 || Hq % Hkv != 0 || bs <= 0 || c <= 0 || s <= 0) return ORC_ERR_ARG;
    const int64_t G = Hq / Hkv;
    for (int64_t b = 0; b < B; ++b) {
        if (n_kernels(kv_len[b], c, s) > M_max) return ORC_ERR_CAPACITY;
        for (int64_t ti = 0; ti < n_t; ++ti) {
            int64_t pos = query_pos(kv_len[b], Tq, t_list[ti], tree);
            if (pos < 0 || pos / bs >= nblk_max) return ORC_ERR_CAPACITY;
        }
    }
#pragma omp parallel for collapse(4) schedule(dynamic, 16)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t g = 0; g < Hkv; ++g) {
            for (int64_t ti = 0; ti < n_t; ++ti) {
                for (int64_t blk = 0; blk < nblk_max; ++blk) {
                    const int64_t t = t_list[ti];
                    const int64_t pos = query_pos(kv_len[b], Tq, t, tree);
                    const int64_t bt = pos / bs;
                    const int64_t M = n_kernels(kv_len[b], c, s);
                    double* row = S + ((b * Hkv + g) * n_t + ti) * nblk_max;
                    double best = -INFINITY;
                    if (blk <= bt) {
                        for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                            const uint16_t* qv = q + ((b * Tq + t) * Hq + h) * d;
                            /* scan a window that holds every kernel sharing a token with the
                             * block; the overlap test below is the definition */
                            int64_t j0 = blk * bs - c < 0 ? 0 : (blk * bs - c) / s;
                            int64_t j1 = (blk + 1) * bs / s + 1;
                            if (j1 > M) j1 = M;
                            for (int64_t j = j0; j < j1; ++j) {
                                int overlaps = (j * s < (blk + 1) * bs) && (j * s + c > blk * bs);
                                int visible = (j * s + c - 1 <= pos);
                                if (!overlaps || !visible) continue;
                                const uint16_t* kv = kern + ((b * Hkv + g) * M_max + j) * d;
                                double dot = 0.0;
                                for (int64_t x = 0; x < d; ++x) dot += bf16_value(qv[x]) * bf16_value(kv[x]);
                                if (dot > best) best = dot;
                            }
                        }
                    }
                    row[blk] = best;
                }
            }
        }
    }
    return ORC_OK;
}

typedef struct {
    double score;
    int32_t block;
} cand_t;

/* Order for top-k: higher score first; equal scores go to the lower block
 * index (reading R8).  -inf scores compare equal and fall back to the index. */
static int cand_cmp(const void* pa, const void* pb) {
    const cand_t* a = (const cand_t*)pa;
    const cand_t* b = (const cand_t*)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->block > b->block) - (a->block < b->block);
}

/*
 * Step 3 -- selection (section 1.1 "dynamic block selection" and "local
 * retention"; the dense switch below dense_len from the 64-token/top-64 page):
 *   bt = the query's own block; forced F = {0..n_init-1} u {bt-n_local+1..bt},
 *   clipped to [0, bt]; candidates C = {0..bt} \ F; keep the first min(k,|C|)
 *   of C in (score desc, index asc) order; Selected = F u kept (reading R1).
 *   If kv_len < dense_len the selection is every block 0..bt (reading R5).
 * idx: [B,Hkv,n_t,S_max] ascending, padded with -1; counts: [B,Hkv,n_t].
 * kth/next (nullable): the score of the last kept candidate and of the first
 * candidate left out (NaN where there is none), for the near-tie report.
 */
int orc_select(const double* S, const int32_t* kv_len, int64_t B, int64_t Hkv, int64_t Tq,
               int32_t tree, const int32_t* ip, const int32_t* t_list, int64_t n_t,
               int64_t nblk_max, int64_t S_max, int32_t* idx, int32_t* counts, double* kth,
               double* next) {
    const int64_t bs = ip[P_BLOCK], k = ip[P_TOPK], n_i = ip[P_NINIT], n_l = ip[P_NLOCAL];
    const int64_t dense_len = ip[P_DENSE_LEN];
    if (bs <= 0 || k < 0 || n_i < 0 || n_l < 1) return ORC_ERR_ARG;
    int err = ORC_OK;
#pragma omp parallel for collapse(3) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t g = 0; g < Hkv; ++g) {
            for (int64_t ti = 0; ti < n_t; ++ti) {
                const int64_t row_id = (b * Hkv + g) * n_t + ti;
                const double* row = S + row_id * nblk_max;
                const int64_t pos = query_pos(kv_len[b], Tq, t_list[ti], tree);
                const int64_t bt = pos / bs;
                char* chosen = (char*)calloc((size_t)(bt + 1), 1);
                cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(bt + 1));
                int64_t nc = 0;
                double kth_s = NAN, next_s = NAN;
                if (kv_len[b] < dense_len) {
                    for (int64_t blk = 0; blk <= bt; ++blk) chosen[blk] = 1;
                } else {
                    for (int64_t blk = 0; blk <= bt; ++blk) {
                        int forced = (blk < n_i) || (blk > bt - n_l);
                        if (forced) chosen[blk] = 1;
                        else { cand[nc].score = row[blk]; cand[nc].block = (int32_t)blk; ++nc; }
                    }
                    qsort(cand, (size_t)nc, sizeof(cand_t), cand_cmp);
                    int64_t take = nc < k ? nc : k;
                    for (int64_t r = 0; r < take; ++r) chosen[cand[r].block] = 1;
                    if (take > 0) kth_s = cand[take - 1].score;
                    if (take < nc) next_s = cand[take].score;
                }
                int64_t cnt = 0;
                int32_t* out = idx + row_id * S_max;
                for (int64_t blk = 0; blk <= bt; ++blk) {
                    if (!chosen[blk]) continue;
                    if (cnt < S_max) out[cnt] = (int32_t)blk;
                    ++cnt;
                }
                if (cnt > S_max) {
#pragma omp atomic write
                    err = ORC_ERR_CAPACITY;
                }
                for (int64_t r = cnt; r < S_max; ++r) out[r] = -1;
                counts[row_id] = (int32_t)cnt;
                if (kth) kth[row_id] = kth_s;
                if (next) next[row_id] = next_s;
                free(chosen);
                free(cand);
            }
        }
    }
    return err;
}

/*
 * Step 4 -- attention on the selected blocks only (section 1.1, "only the key
 * blocks' attention is computed"), one exact softmax per (query, head):
 *   keys T(t) = { x : block(x) selected, x <= pos(t), x < kv_len }
 *   tree drafts: every cached token of a selected block, plus draft j iff bit
 *   j of tree_mask[b,t] is set (section 1.1, technical-details note on the
 *   uint64 mask).
 *   z_x = scale * q.k_x ; o = sum_x exp(z_x - m) v_x / sum_x exp(z_x - m) ;
 *   lse = m + log(sum_x exp(z_x - m)), m = max_x z_x.
 * q: [B,Tq,Hq,d]; k/v cache: [B,Hkv,L_max,d]; draft k/v: [B,Hkv,Tq,d] or NULL;
 * tree_mask: [B,Tq] or NULL; idx/counts: as written by orc_select for the same
 * t_list (NULL idx = every block up to the query's own: dense causal).
 * o: [B,n_t,Hq,d]; lse: [B,Hq,n_t] (nullable).  scale <= 0 means 1/sqrt(d).
 */
int orc_attention(const uint16_t* q, const uint16_t* kc, const uint16_t* vc, const int32_t* kv_len,
                  const uint16_t* dk, const uint16_t* dv, const uint64_t* tree_mask,
                  const int32_t* idx, const int32_t* counts, int64_t S_max, int64_t B, int64_t Tq,
                  int64_t Hq, int64_t Hkv, int64_t d, int64_t L_max, const int32_t* ip, double scale,
                  const int32_t* t_list, int64_t n_t, double* o, double* lse) {
    const int64_t bs = ip[P_BLOCK];
    if (Hkv <= 0 || Hq % Hkv != 0 || bs <= 0) return ORC_ERR_ARG;
    if (tree_mask && (!dk || !dv || Tq > 64)) return ORC_ERR_ARG;
    const int64_t G = Hq / Hkv;
    const int tree = tree_mask != NULL;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)d);
    int err = ORC_OK;
#pragma omp parallel for collapse(3) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t ti = 0; ti < n_t; ++ti) {
            for (int64_t h = 0; h < Hq; ++h) {
                const int64_t t = t_list[ti];
                const int64_t g = h / G;
                const int64_t L = kv_len[b];
                const int64_t pos = query_pos(L, Tq, t, tree);
                const uint16_t* qv = q + ((b * Tq + t) * Hq + h) * d;
                const int64_t row_id = (b * Hkv + g) * n_t + ti;
                int64_t nsel = idx ? counts[row_id] : pos / bs + 1;
                /* keys gathered as (pointer to k, pointer to v) pairs */
                int64_t cap = nsel * bs + (tree ? Tq : 0);
                const uint16_t** kp = (const uint16_t**)malloc(sizeof(void*) * (size_t)(cap + 1));
                const uint16_t** vp = (const uint16_t**)malloc(sizeof(void*) * (size_t)(cap + 1));
                int64_t nk = 0;
                for (int64_t r = 0; r < nsel; ++r) {
                    int64_t blk = idx ? idx[row_id * S_max + r] : r;
                    if (blk < 0) {
#pragma omp atomic write
                        err = ORC_ERR_ARG;
                        continue;
                    }
                    for (int64_t x = blk * bs; x < (blk + 1) * bs; ++x) {
                        if (x >= L || x > pos) break;
                        kp[nk] = kc + ((b * Hkv + g) * L_max + x) * d;
                        vp[nk] = vc + ((b * Hkv + g) * L_max + x) * d;
                        ++nk;
                    }
                }
                if (tree) {
                    uint64_t m = tree_mask[b * Tq + t];
                    for (int64_t j = 0; j < Tq; ++j) {
                        if (!((m >> j) & 1u)) continue;
                        kp[nk] = dk + ((b * Hkv + g) * Tq + j) * d;
                        vp[nk] = dv + ((b * Hkv + g) * Tq + j) * d;
                        ++nk;
                    }
                }
                double* z = (double*)malloc(sizeof(double) * (size_t)(nk + 1));
                double zmax = -INFINITY;
                for (int64_t n = 0; n < nk; ++n) {
                    double dot = 0.0;
                    for (int64_t x = 0; x < d; ++x) dot += bf16_value(qv[x]) * bf16_value(kp[n][x]);
                    z[n] = scale * dot;
                    if (z[n] > zmax) zmax = z[n];
                }
                double denom = 0.0;
                for (int64_t n = 0; n < nk; ++n) {
                    z[n] = exp(z[n] - zmax); /* unnormalised weight of key n */
                    denom += z[n];
                }
                double* orow = o + ((b * n_t + ti) * Hq + h) * d;
                for (int64_t x = 0; x < d; ++x) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < nk; ++n) acc += z[n] * bf16_value(vp[n][x]);
                    orow[x] = nk ? acc / denom : 0.0;
                }
                if (lse) lse[(b * Hq + h) * n_t + ti] = nk ? zmax + log(denom) : -INFINITY;
                free(z);
                free(kp);
                free(vp);
            }
        }
    }
    return err;
}

/* ---------------------------------------------------------------------------------------------
 * Backward of the attention step ("MiniCPM4：如何在手机电脑上高效运行大语言模型", section 1.1: InfLLM
 * v2 is trainable sparse attention; the selection is a discrete choice, so gradients flow through
 * the attention over the selected keys with the selection held fixed).
 *
 * Both functions below take fp64 inputs (q [B,Tq,Hq,d]; caches [B,Hkv,L_max,d]) so that the
 * backward can be checked against finite differences of the forward; chunk layout only (query t
 * of a chunk sits at kv_len - Tq + t), no draft tree.  The key set of (b, t, h) is the same as in
 * orc_attention: tokens x <= pos of the selected blocks (every block from 0 to pos when idx is
 * NULL).
 */
static int64_t gather_keys(int64_t b, int64_t t, int64_t g, int64_t Tq, int64_t Hkv, int64_t L,
                           int64_t bs, const int32_t* idx, const int32_t* counts, int64_t S_max,
                           int64_t* keys) {
    const int64_t pos = L - Tq + t;
    const int64_t row_id = (b * Hkv + g) * Tq + t;
    const int64_t nsel = idx ? counts[row_id] : pos / bs + 1;
    int64_t nk = 0;
    for (int64_t r = 0; r < nsel; ++r) {
        const int64_t blk = idx ? idx[row_id * S_max + r] : r;
        if (blk < 0) return -1;
        for (int64_t x = blk * bs; x < (blk + 1) * bs; ++x) {
            if (x >= L || x > pos) break;
            keys[nk++] = x;
        }
    }
    return nk;
}

/* o = softmax(scale * q k^T) v over each row's keys, in fp64 (o [B,Tq,Hq,d], lse [B,Hq,Tq]). */
int orc_attention_f64(const double* q, const double* kc, const double* vc, const int32_t* kv_len,
                      const int32_t* idx, const int32_t* counts, int64_t S_max, int64_t B, int64_t Tq,
                      int64_t Hq, int64_t Hkv, int64_t d, int64_t L_max, const int32_t* ip, double scale,
                      double* o, double* lse) {
    const int64_t bs = ip[P_BLOCK];
    if (Hkv <= 0 || Hq % Hkv != 0 || bs <= 0) return ORC_ERR_ARG;
    const int64_t G = Hq / Hkv;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)d);
    int err = ORC_OK;
#pragma omp parallel for collapse(3) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < Tq; ++t)
            for (int64_t h = 0; h < Hq; ++h) {
                const int64_t g = h / G, L = kv_len[b];
                int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(L + 1));
                double* z = (double*)malloc(sizeof(double) * (size_t)(L + 1));
                const int64_t nk = gather_keys(b, t, g, Tq, Hkv, L, bs, idx, counts, S_max, keys);
                if (nk < 0) {
#pragma omp atomic write
                    err = ORC_ERR_ARG;
                }
                const double* qv = q + ((b * Tq + t) * Hq + h) * d;
                double zmax = -INFINITY, denom = 0.0;
                for (int64_t n = 0; n < nk; ++n) {
                    const double* kv = kc + ((b * Hkv + g) * L_max + keys[n]) * d;
                    double dot = 0.0;
                    for (int64_t x = 0; x < d; ++x) dot += qv[x] * kv[x];
                    z[n] = scale * dot;
                    if (z[n] > zmax) zmax = z[n];
                }
                for (int64_t n = 0; n < nk; ++n) {
                    z[n] = exp(z[n] - zmax);
                    denom += z[n];
                }
                double* orow = o + ((b * Tq + t) * Hq + h) * d;
                for (int64_t x = 0; x < d; ++x) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < nk; ++n) acc += z[n] * vc[((b * Hkv + g) * L_max + keys[n]) * d + x];
                    orow[x] = nk > 0 ? acc / denom : 0.0;
                }
                if (lse) lse[(b * Hq + h) * Tq + t] = nk > 0 ? zmax + log(denom) : -INFINITY;
                free(z);
                free(keys);
            }
    return err;
}

/* Gradients of sum(dout * o) for orc_attention_f64 with the selection fixed.  Per row, with p
 * the softmax weights and a_n = dout . v_n:
 *   dv_n += p_n dout;  dz_n = p_n (a_n - sum_m p_m a_m);  dq += scale sum_n dz_n k_n;
 *   dk_n += scale dz_n q.
 * dq [B,Tq,Hq,d]; dk, dv [B,Hkv,L_max,d], summed over the heads of a group and over the rows
 * (rows of one (b, g) run in order, so the sums need no atomics). */
int orc_attention_bwd(const double* q, const double* kc, const double* vc, const int32_t* kv_len,
                      const int32_t* idx, const int32_t* counts, int64_t S_max, int64_t B, int64_t Tq,
                      int64_t Hq, int64_t Hkv, int64_t d, int64_t L_max, const int32_t* ip, double scale,
                      const double* dout, double* dq, double* dk, double* dv) {
    const int64_t bs = ip[P_BLOCK];
    if (Hkv <= 0 || Hq % Hkv != 0 || bs <= 0) return ORC_ERR_ARG;
    const int64_t G = Hq / Hkv;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)d);
    memset(dq, 0, sizeof(double) * (size_t)(B * Tq * Hq * d));
    memset(dk, 0, sizeof(double) * (size_t)(B * Hkv * L_max * d));
    memset(dv, 0, sizeof(double) * (size_t)(B * Hkv * L_max * d));
    int err = ORC_OK;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g) {
            const int64_t L = kv_len[b];
            int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(L + 1));
            double* p = (double*)malloc(sizeof(double) * (size_t)(L + 1));
            double* a = (double*)malloc(sizeof(double) * (size_t)(L + 1));
            for (int64_t t = 0; t < Tq; ++t)
                for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                    const int64_t nk = gather_keys(b, t, g, Tq, Hkv, L, bs, idx, counts, S_max, keys);
                    if (nk < 0) {
#pragma omp atomic write
                        err = ORC_ERR_ARG;
                        continue;
                    }
                    const double* qv = q + ((b * Tq + t) * Hq + h) * d;
                    const double* dov = dout + ((b * Tq + t) * Hq + h) * d;
                    double zmax = -INFINITY, denom = 0.0;
                    for (int64_t n = 0; n < nk; ++n) {
                        const double* kv = kc + ((b * Hkv + g) * L_max + keys[n]) * d;
                        double dot = 0.0;
                        for (int64_t x = 0; x < d; ++x) dot += qv[x] * kv[x];
                        p[n] = scale * dot;
                        if (p[n] > zmax) zmax = p[n];
                    }
                    for (int64_t n = 0; n < nk; ++n) {
                        p[n] = exp(p[n] - zmax);
                        denom += p[n];
                    }
                    double pa = 0.0;
                    for (int64_t n = 0; n < nk; ++n) {
                        p[n] /= denom;
                        const double* vv = vc + ((b * Hkv + g) * L_max + keys[n]) * d;
                        double dot = 0.0;
                        for (int64_t x = 0; x < d; ++x) dot += dov[x] * vv[x];
                        a[n] = dot;
                        pa += p[n] * dot;
                    }
                    double* dqv = dq + ((b * Tq + t) * Hq + h) * d;
                    for (int64_t n = 0; n < nk; ++n) {
                        const double dz = p[n] * (a[n] - pa);
                        const int64_t row = ((b * Hkv + g) * L_max + keys[n]) * d;
                        for (int64_t x = 0; x < d; ++x) {
                            dqv[x] += scale * dz * kc[row + x];
                            dk[row + x] += scale * dz * qv[x];
                            dv[row + x] += p[n] * dov[x];
                        }
                    }
                }
            free(a);
            free(p);
            free(keys);
        }
    return err;
}
