/*
 * Hybrid Tree Attention: CPU fp64 oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do. It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes ("LongSpec: Long-Context Lossless Speculative Decoding with
 * Efficient Drafting and Verification", Korean summary section 2.C "Fast Tree
 * Attention" and Dutch summary Methodologie section 3 "Hybrid Tree
 * Attention"): the verification attention
 * of the T speculative-tree queries over the cached prefix followed by the tree
 * itself. The method splits this into an unmasked cached part and a masked
 * speculative part and merges them exactly; the oracle does NOT split. It
 * evaluates the single softmax over the union of both key sets, which is the
 * result the split method claims to reproduce exactly.
 *
 *   visible keys of query (b, t, hq):
 *       cache token j for 0 <= j < cache_lens[b]
 *       tree token  j for j in anc*(t), the ancestor-or-self set of node t
 *   s_j  = scale * <q, k_j>            (bf16 inputs widened exactly to double)
 *   m    = max_j s_j
 *   l    = sum_j exp(s_j - m)
 *   O    = sum_j exp(s_j - m) v_j / l
 *   LSE  = m + ln l                    (natural log)
 *
 * The tree mask follows "LogitSpec: Accelerating Retrieval-based Speculative
 * Decoding via Next Next Token Speculation", section 2 (Method), workflow
 * step 2 "draft tree construction and verification": the target verifies
 * every branch at once,
 * so a node may see its own root path and nothing else of the tree. The
 * oracle builds it by walking each node's parent chain on its own.
 *
 * Layouts (row-major, bf16 passed as raw uint16 bit patterns):
 *   q        [B][T][Hq][d]
 *   k_cache  [B][Hkv][Lmax][d]      v_cache the same
 *   k_spec   [B][Hkv][T][d]         v_spec  the same
 *   mask     [B][T][W] uint32, W = ceil(T/32), bit j%32 of word j/32
 *   o        [rows][d] double,  lse [rows] double
 * Query head hq reads KV head hq / (Hq/Hkv).
 *
 * Every function here has an independent pin in the test suite (brute force,
 * closed forms, library routines, invariants); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct oracle_dims {
    int32_t B, T, Hq, Hkv, d;
    int64_t Lmax;
    double scale; /* 0 selects 1/sqrt(d) */
} oracle_dims;

/* bf16 -> double: the bf16 bit pattern is the top half of an IEEE binary32. */
static double bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_mask_words(int32_t T) { return (T + 31) / 32; }

/*
 * Ancestor-or-self mask by independent parent-chain walks.
 * A tree is valid when parents[0] == -1 and -1 <= parents[i] < i for every i
 * (topological order; more than one root is allowed). A walk that would leave
 * that rule aborts. Returns 0 when every tree is valid, otherwise the number
 * of invalid trees; the rows of an invalid tree are all zero.
 */
int oracle_build_mask(const int32_t *parents, int32_t B, int32_t T, uint32_t *mask) {
    const int W = oracle_mask_words(T);
    int bad_trees = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parents + (int64_t)b * T;
        uint32_t *rows = mask + (int64_t)b * T * W;
        memset(rows, 0, sizeof(uint32_t) * (size_t)T * (size_t)W);
        int bad = 0;
        for (int i = 0; i < T && !bad; ++i) {
            int32_t p = par[i];
            if (p < -1 || p >= i) bad = 1;
        }
        if (bad) {
            ++bad_trees;
            continue;
        }
        for (int i = 0; i < T; ++i) {
            uint32_t *row = rows + (int64_t)i * W;
            int32_t j = i;
            int steps = 0;
            while (j != -1 && steps <= T) {
                row[j / 32] |= 1u << (j % 32);
                j = par[j];
                ++steps;
            }
        }
    }
    return bad_trees;
}

/*
 * Monolithic masked attention for a list of query rows.
 * row_ids[k] = (b*T + t)*Hq + hq; a NULL row_ids means every row in order.
 * A row with no visible key (empty prefix and empty mask row) gets
 * LSE = -inf and O = 0, the limit of an empty softmax sum.
 */
void oracle_attention(const oracle_dims *dm,
                      const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *cache_lens,
                      const uint16_t *k_spec, const uint16_t *v_spec,
                      const uint32_t *mask,
                      const int64_t *row_ids, int64_t n_rows,
                      double *o, double *lse) {
    const int B = dm->B, T = dm->T, Hq = dm->Hq, Hkv = dm->Hkv, d = dm->d;
    const int64_t Lmax = dm->Lmax;
    const int G = Hq / Hkv;
    const int W = oracle_mask_words(T);
    const double scale = dm->scale != 0.0 ? dm->scale : 1.0 / sqrt((double)d);
    (void)B;

#pragma omp parallel
    {
        /* per-thread scratch: one score per visible key */
        int64_t max_keys = Lmax + T;
        double *s = (double *)malloc(sizeof(double) * (size_t)max_keys);
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            const int64_t rid = row_ids ? row_ids[r] : r;
            const int hq = (int)(rid % Hq);
            const int t = (int)((rid / Hq) % T);
            const int b = (int)(rid / ((int64_t)Hq * T));
            const int kvh = hq / G;
            const int64_t L = cache_lens[b];
            const uint16_t *qr = q + rid * d;
            for (int c = 0; c < d; ++c) qd[c] = bf16_to_double(qr[c]);

            const uint16_t *kc = k_cache + ((int64_t)b * Hkv + kvh) * Lmax * d;
            const uint16_t *vc = v_cache + ((int64_t)b * Hkv + kvh) * Lmax * d;
            const uint16_t *ks = k_spec + ((int64_t)b * Hkv + kvh) * T * d;
            const uint16_t *vs = v_spec + ((int64_t)b * Hkv + kvh) * T * d;
            const uint32_t *mrow = mask + ((int64_t)b * T + t) * W;

            /* scores: cache keys first, then the visible tree keys */
            int64_t n = 0;
            double m = -INFINITY;
            for (int64_t j = 0; j < L; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += qd[c] * bf16_to_double(kc[j * d + c]);
                s[n] = scale * acc;
                if (s[n] > m) m = s[n];
                ++n;
            }
            for (int j = 0; j < T; ++j) {
                if (!((mrow[j / 32] >> (j % 32)) & 1u)) continue;
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += qd[c] * bf16_to_double(ks[(int64_t)j * d + c]);
                s[n] = scale * acc;
                if (s[n] > m) m = s[n];
                ++n;
            }

            double *orow = o + r * d;
            for (int c = 0; c < d; ++c) orow[c] = 0.0;
            if (n == 0) {
                lse[r] = -INFINITY;
                continue;
            }
            double l = 0.0;
            int64_t idx = 0;
            for (int64_t j = 0; j < L; ++j, ++idx) {
                double p = exp(s[idx] - m);
                l += p;
                for (int c = 0; c < d; ++c) orow[c] += p * bf16_to_double(vc[j * d + c]);
            }
            for (int j = 0; j < T; ++j) {
                if (!((mrow[j / 32] >> (j % 32)) & 1u)) continue;
                double p = exp(s[idx] - m);
                l += p;
                for (int c = 0; c < d; ++c) orow[c] += p * bf16_to_double(vs[(int64_t)j * d + c]);
                ++idx;
            }
            for (int c = 0; c < d; ++c) orow[c] /= l;
            lse[r] = m + log(l);
        }
        free(s);
        free(qd);
    }
}

/* Threads the OpenMP runtime will use for oracle_attention. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
