/*
 * oracle.c -- plain CPU reference of the gradient-averaging hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Single-threaded, no SIMD, no
 * blocking or reordering beyond what the cited definitions state.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ===================================================================== */
/* Philox4x32 [S]: a 4-word counter and a 2-word key; each round multiplies
 * words 0 and 2 by the two round multipliers, mixes the high halves with
 * words 1 and 3 and the key, and the key is advanced by the two Weyl
 * increments between rounds.  The constants are the ones the SC'11 paper
 * publishes for the 4x32 variant.                                          */
/* ===================================================================== */
#define PHILOX_MUL_A 0xD2511F53u
#define PHILOX_MUL_B 0xCD9E8D57u
#define PHILOX_WEYL_A 0x9E3779B9u
#define PHILOX_WEYL_B 0xBB67AE85u

void oracle_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds,
                       uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < rounds; ++r) {
        if (r > 0) {
            k0 += PHILOX_WEYL_A;
            k1 += PHILOX_WEYL_B;
        }
        uint64_t prod_a = (uint64_t)PHILOX_MUL_A * (uint64_t)c0;
        uint64_t prod_b = (uint64_t)PHILOX_MUL_B * (uint64_t)c2;
        uint32_t hi_a = (uint32_t)(prod_a >> 32), lo_a = (uint32_t)prod_a;
        uint32_t hi_b = (uint32_t)(prod_b >> 32), lo_b = (uint32_t)prod_b;
        uint32_t n0 = hi_b ^ c1 ^ k0;
        uint32_t n1 = lo_b;
        uint32_t n2 = hi_a ^ c3 ^ k1;
        uint32_t n3 = lo_a;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* ===================================================================== */
/* Ring all-reduce [H] "The Ring-Allreduce Algorithm", [R] sections 4, 5, 7 */
/* ===================================================================== */

/* The buffer is cut into p chunks.  The pages only give the case where p
 * divides n; for other n every chunk but the trailing ones has ceil(n/p)
 * elements and the trailing chunks are short or empty.                    */
int64_t oracle_ring_chunk_len(int64_t n, int p) { return (n + p - 1) / p; }

static int64_t chunk_begin(int64_t n, int p, int c) {
    int64_t b = (int64_t)c * oracle_ring_chunk_len(n, p);
    return b < n ? b : n;
}
static int64_t chunk_end(int64_t n, int p, int c) { return chunk_begin(n, p, c + 1); }
static int ring_mod(int a, int p) { return ((a % p) + p) % p; }

int oracle_ring_schedule_f32(float *const *bufs, int p, int64_t n, int op, int phases,
                             int64_t *sent_elems, int *steps) {
    if (p < 1 || n < 0 || (op != ORACLE_SUM && op != ORACLE_AVG)) return -1;
    int64_t clen = oracle_ring_chunk_len(n, p);
    /* one chunk-sized "wire" slot per sender, so that every worker's send of
     * a step is taken before any worker's receive of that step is applied */
    float *wire = (float *)malloc(sizeof(float) * (size_t)(clen > 0 ? clen : 1) * (size_t)p);
    if (!wire) return -1;
    for (int w = 0; w < p; ++w)
        if (sent_elems) sent_elems[w] = 0;
    int nsteps = 0;

    /* Phase 1, scatter-reduce: at step s worker i sends chunk (i - s) mod p
     * to worker i + 1, which adds it into its own copy of that chunk. */
    for (int s = 0; s < p - 1; ++s) {
        for (int i = 0; i < p; ++i) {
            int c = ring_mod(i - s, p);
            int64_t b = chunk_begin(n, p, c), e = chunk_end(n, p, c);
            memcpy(wire + (size_t)i * (size_t)clen, bufs[i] + b, sizeof(float) * (size_t)(e - b));
            if (sent_elems) sent_elems[i] += e - b;
        }
        for (int i = 0; i < p; ++i) {
            int from = ring_mod(i - 1, p);
            int c = ring_mod(i - s - 1, p);
            int64_t b = chunk_begin(n, p, c), e = chunk_end(n, p, c);
            const float *recv = wire + (size_t)from * (size_t)clen;
            for (int64_t k = b; k < e; ++k) bufs[i][k] = bufs[i][k] + recv[k - b];
        }
        ++nsteps;
    }
    if (phases == 2) {
        /* Phase 2, all-gather: at step s worker i sends its finished chunk
         * (i - s + 1) mod p to worker i + 1, which overwrites its copy. */
        for (int s = 0; s < p - 1; ++s) {
            for (int i = 0; i < p; ++i) {
                int c = ring_mod(i - s + 1, p);
                int64_t b = chunk_begin(n, p, c), e = chunk_end(n, p, c);
                memcpy(wire + (size_t)i * (size_t)clen, bufs[i] + b,
                       sizeof(float) * (size_t)(e - b));
                if (sent_elems) sent_elems[i] += e - b;
            }
            for (int i = 0; i < p; ++i) {
                int from = ring_mod(i - 1, p);
                int c = ring_mod(i - s, p);
                int64_t b = chunk_begin(n, p, c), e = chunk_end(n, p, c);
                memcpy(bufs[i] + b, wire + (size_t)from * (size_t)clen,
                       sizeof(float) * (size_t)(e - b));
            }
            ++nsteps;
        }
        /* The average is the sum divided element-wise by the worker count. */
        if (op == ORACLE_AVG) {
            float fp = (float)p;
            for (int i = 0; i < p; ++i)
                for (int64_t k = 0; k < n; ++k) bufs[i][k] = bufs[i][k] / fp;
        }
    }
    free(wire);
    if (steps) *steps = nsteps;
    return 0;
}

/* Chunk c leaves worker c at step 0 and picks up one addend per hop, so an
 * element of chunk c is x_c + x_{c+1} + ... + x_{c+p-1} (indices mod p),
 * added left to right in fp32.  IEEE addition is commutative, so this is
 * bit for bit the value the literal schedule produces. */
static float fold_one_f32(const float *const *x, int p, int64_t n, int op, int64_t k) {
    int c = (int)(k / oracle_ring_chunk_len(n, p));
    float s = x[c][k];
    for (int j = 1; j < p; ++j) s = s + x[(c + j) % p][k];
    if (op == ORACLE_AVG) s = s / (float)p;
    return s;
}

int oracle_ring_fold_f32(const float *const *x, int p, int64_t n, int op, float *out) {
    if (p < 1 || n < 0) return -1;
    for (int64_t k = 0; k < n; ++k) out[k] = fold_one_f32(x, p, n, op, k);
    return 0;
}

int oracle_ring_fold_f32_at(const float *const *x, int p, int64_t n, int op,
                            const int64_t *idx, int64_t count, float *out) {
    if (p < 1 || n < 0) return -1;
    for (int64_t k = 0; k < count; ++k) {
        if (idx[k] < 0 || idx[k] >= n) return -1;
        out[k] = fold_one_f32(x, p, n, op, idx[k]);
    }
    return 0;
}

/* bf16 is the top 16 bits of an IEEE binary32: widening is a shift. */
float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even.  NaN stays NaN (its
 * payload is not specified here). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* The same rounding over n values (out[k] = oracle_f32_to_bf16(in[k])). */
void oracle_f32_to_bf16_n(const float *in, int64_t n, uint16_t *out) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_f32_to_bf16(in[k]);
}

static float fold_one_bf16(const uint16_t *const *x, int p, int64_t n, int op, int64_t k) {
    int c = (int)(k / oracle_ring_chunk_len(n, p));
    float s = oracle_bf16_to_f32(x[c][k]);
    for (int j = 1; j < p; ++j) s = s + oracle_bf16_to_f32(x[(c + j) % p][k]);
    if (op == ORACLE_AVG) s = s / (float)p;
    return s;
}

int oracle_ring_fold_bf16(const uint16_t *const *x, int p, int64_t n, int op, uint16_t *out,
                          float *out_f32) {
    if (p < 1 || n < 0) return -1;
    for (int64_t k = 0; k < n; ++k) {
        float s = fold_one_bf16(x, p, n, op, k);
        if (out_f32) out_f32[k] = s;
        out[k] = oracle_f32_to_bf16(s);
    }
    return 0;
}

int oracle_ring_fold_bf16_at(const uint16_t *const *x, int p, int64_t n, int op,
                             const int64_t *idx, int64_t count, uint16_t *out) {
    if (p < 1 || n < 0) return -1;
    for (int64_t k = 0; k < count; ++k) {
        if (idx[k] < 0 || idx[k] >= n) return -1;
        out[k] = oracle_f32_to_bf16(fold_one_bf16(x, p, n, op, idx[k]));
    }
    return 0;
}

/* bf16 buffers on the literal schedule: the values on the wire are the fp32
 * partial sums; the result is rounded to bf16 once, at the end. */
int oracle_ring_schedule_bf16(uint16_t *const *bufs, int p, int64_t n, int op,
                              int64_t *sent_elems, int *steps) {
    if (p < 1 || n < 0) return -1;
    float **work = (float **)calloc((size_t)p, sizeof(float *));
    if (!work) return -1;
    int rc = 0;
    for (int i = 0; i < p; ++i) {
        work[i] = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
        if (!work[i]) rc = -1;
    }
    if (rc == 0) {
        for (int i = 0; i < p; ++i)
            for (int64_t k = 0; k < n; ++k) work[i][k] = oracle_bf16_to_f32(bufs[i][k]);
        rc = oracle_ring_schedule_f32(work, p, n, op, 2, sent_elems, steps);
        if (rc == 0)
            for (int i = 0; i < p; ++i)
                for (int64_t k = 0; k < n; ++k) bufs[i][k] = oracle_f32_to_bf16(work[i][k]);
    }
    for (int i = 0; i < p; ++i) free(work[i]);
    free(work);
    return rc;
}

int oracle_ring_fold_f32_samples(const float *vals, int p, int64_t n, int op, const int64_t *e,
                                 int64_t count, float *out) {
    if (p < 1 || n < 0) return -1;
    for (int64_t k = 0; k < count; ++k) {
        if (e[k] < 0 || e[k] >= n) return -1;
        int c = (int)(e[k] / oracle_ring_chunk_len(n, p));
        float s = vals[(int64_t)c * count + k];
        for (int j = 1; j < p; ++j) s = s + vals[(int64_t)((c + j) % p) * count + k];
        if (op == ORACLE_AVG) s = s / (float)p;
        out[k] = s;
    }
    return 0;
}

int oracle_ring_fold_bf16_samples(const uint16_t *vals, int p, int64_t n, int op,
                                  const int64_t *e, int64_t count, uint16_t *out) {
    if (p < 1 || n < 0) return -1;
    for (int64_t k = 0; k < count; ++k) {
        if (e[k] < 0 || e[k] >= n) return -1;
        int c = (int)(e[k] / oracle_ring_chunk_len(n, p));
        float s = oracle_bf16_to_f32(vals[(int64_t)c * count + k]);
        for (int j = 1; j < p; ++j) s = s + oracle_bf16_to_f32(vals[(int64_t)((c + j) % p) * count + k]);
        if (op == ORACLE_AVG) s = s / (float)p;
        out[k] = oracle_f32_to_bf16(s);
    }
    return 0;
}

/* ===================================================================== */
/* Bidirectional dual ring [R] section 11, exercise 1                     */
/* ===================================================================== */
/* 2p sub-chunks of ceil(n / 2p) elements (trailing ones short or empty).
 * Clockwise ring (next = i + 1) on sub-chunks 0..p-1, exactly the single
 * ring's schedule; counter-clockwise ring (next = i - 1) on p..2p-1: at
 * scatter step s worker i sends sub-chunk p + (i + s) mod p to worker i - 1,
 * which adds it into its own copy; at gather step s it sends
 * p + (i + s - 1) mod p, which the receiver copies.                       */
int64_t oracle_bidir_subchunk_len(int64_t n, int p) { return (n + 2 * (int64_t)p - 1) / (2 * (int64_t)p); }

static int64_t sub_begin(int64_t n, int p, int k) {
    int64_t b = (int64_t)k * oracle_bidir_subchunk_len(n, p);
    return b < n ? b : n;
}
static int64_t sub_end(int64_t n, int p, int k) { return sub_begin(n, p, k + 1); }

int oracle_bidir_schedule_f32(float *const *bufs, int p, int64_t n, int op, int64_t *sent_elems,
                              int *steps) {
    if (p < 1 || p > 64 || n < 0 || (op != ORACLE_SUM && op != ORACLE_AVG)) return -1;
    int64_t slen = oracle_bidir_subchunk_len(n, p);
    size_t slot = (size_t)(slen > 0 ? slen : 1);
    float *cw = (float *)malloc(sizeof(float) * slot * (size_t)p);
    float *ccw = (float *)malloc(sizeof(float) * slot * (size_t)p);
    if (!cw || !ccw) {
        free(cw);
        free(ccw);
        return -1;
    }
    for (int w = 0; w < p; ++w)
        if (sent_elems) sent_elems[w] = 0;
    int nsteps = 0;
    for (int phase = 0; phase < 2; ++phase) {
        for (int s = 0; s < p - 1; ++s) {
            /* every worker's two sends of this step, taken before any receive */
            int cw_send[64], ccw_send[64];
            for (int i = 0; i < p; ++i) {
                cw_send[i] = phase == 0 ? ring_mod(i - s, p) : ring_mod(i - s + 1, p);
                ccw_send[i] = p + (phase == 0 ? ring_mod(i + s, p) : ring_mod(i + s - 1, p));
                int64_t b0 = sub_begin(n, p, cw_send[i]), e0 = sub_end(n, p, cw_send[i]);
                int64_t b1 = sub_begin(n, p, ccw_send[i]), e1 = sub_end(n, p, ccw_send[i]);
                memcpy(cw + (size_t)i * slot, bufs[i] + b0, sizeof(float) * (size_t)(e0 - b0));
                memcpy(ccw + (size_t)i * slot, bufs[i] + b1, sizeof(float) * (size_t)(e1 - b1));
                if (sent_elems) sent_elems[i] += (e0 - b0) + (e1 - b1);
            }
            for (int i = 0; i < p; ++i) {
                int from_cw = ring_mod(i - 1, p), from_ccw = ring_mod(i + 1, p);
                int k0 = cw_send[from_cw], k1 = ccw_send[from_ccw];
                int64_t b0 = sub_begin(n, p, k0), e0 = sub_end(n, p, k0);
                int64_t b1 = sub_begin(n, p, k1), e1 = sub_end(n, p, k1);
                const float *r0 = cw + (size_t)from_cw * slot, *r1 = ccw + (size_t)from_ccw * slot;
                for (int64_t k = b0; k < e0; ++k) bufs[i][k] = phase == 0 ? bufs[i][k] + r0[k - b0] : r0[k - b0];
                for (int64_t k = b1; k < e1; ++k) bufs[i][k] = phase == 0 ? bufs[i][k] + r1[k - b1] : r1[k - b1];
            }
            ++nsteps;
        }
    }
    if (op == ORACLE_AVG) {
        float fp = (float)p;
        for (int i = 0; i < p; ++i)
            for (int64_t k = 0; k < n; ++k) bufs[i][k] = bufs[i][k] / fp;
    }
    free(cw);
    free(ccw);
    if (steps) *steps = nsteps;
    return 0;
}

/* Closed form: an element of clockwise sub-chunk c is x_c + x_{c+1} + ...;
 * one of counter-clockwise sub-chunk p + c is x_c + x_{c-1} + ... (mod p). */
int oracle_bidir_fold_f32(const float *const *x, int p, int64_t n, int op, float *out) {
    if (p < 1 || n < 0 || p > 64) return -1;
    int64_t slen = oracle_bidir_subchunk_len(n, p);
    for (int64_t k = 0; k < n; ++k) {
        int sub = (int)(k / slen);
        int c = sub < p ? sub : sub - p;
        int dir = sub < p ? 1 : -1;
        float s = x[c][k];
        for (int j = 1; j < p; ++j) s = s + x[ring_mod(c + dir * j, p)][k];
        if (op == ORACLE_AVG) s = s / (float)p;
        out[k] = s;
    }
    return 0;
}

int oracle_bidir_fold_f32_samples(const float *vals, int p, int64_t n, int op, const int64_t *e,
                                  int64_t count, float *out) {
    if (p < 1 || n < 0 || p > 64) return -1;
    int64_t slen = oracle_bidir_subchunk_len(n, p);
    for (int64_t k = 0; k < count; ++k) {
        if (e[k] < 0 || e[k] >= n) return -1;
        int sub = (int)(e[k] / slen);
        int c = sub < p ? sub : sub - p;
        int dir = sub < p ? 1 : -1;
        float s = vals[(int64_t)c * count + k];
        for (int j = 1; j < p; ++j) s = s + vals[(int64_t)ring_mod(c + dir * j, p) * count + k];
        if (op == ORACLE_AVG) s = s / (float)p;
        out[k] = s;
    }
    return 0;
}

/* ===================================================================== */
/* Double binary tree [R] "Design Alternatives & Collective Comparison    */
/* Matrix: Ring vs. Tree vs. NVLS"; construction [ST]                     */
/* ===================================================================== */
/* The tutorial compares the ring with the double-binary-tree all-reduce
 * (two complementary trees, each carrying half the data; about 2 log2(p)
 * latency steps; about 2M bytes sent per rank) but prints no construction.
 * Reading: the two-tree scheme of [ST].  Tree 1 is the in-order binary tree
 * on the labels 1..p: the root of a run of labels is the label in it with
 * the most trailing zero bits, and its left and right subtrees are built
 * the same way on the labels below and above it.  Label l hosts rank l - 1.
 * Tree 2 has the same shape; label l hosts rank p - l when p is even (the
 * mirror image) and rank (l - 2) mod p when p is odd (shifted by one).
 * Elements [0, ceil(n/2)) are reduced on tree 1, the rest on tree 2.  A
 * node's partial sum is its own value plus its left child's partial sum,
 * then plus its right child's (fp32); the root divides by p for AVG and the
 * value is broadcast down the same tree.                                  */
static int low_zeros(int v) {
    int k = 0;
    while ((v & 1) == 0) {
        v >>= 1;
        ++k;
    }
    return k;
}

/* Builds the run lo..hi of labels; returns its root label (0: empty run). */
static int build_run(int lo, int hi, int up, int *par, int *lc, int *rc) {
    if (lo > hi) return 0;
    int root = lo;
    for (int l = lo + 1; l <= hi; ++l)
        if (low_zeros(l) > low_zeros(root)) root = l;
    par[root] = up;
    lc[root] = build_run(lo, root - 1, root, par, lc, rc);
    rc[root] = build_run(root + 1, hi, root, par, lc, rc);
    return root;
}

static int host_rank(int p, int tree, int label) {
    if (tree == 0) return label - 1;
    if (p % 2 == 0) return p - label;
    return ((label - 2) % p + p) % p;
}

int oracle_dbtree_build(int p, int tree, int32_t *parent, int32_t *left, int32_t *right) {
    if (p < 1 || p > 64 || (tree != 0 && tree != 1)) return -1;
    int par[65], lc[65], rc[65];
    int root = build_run(1, p, 0, par, lc, rc);
    for (int l = 1; l <= p; ++l) {
        int r = host_rank(p, tree, l);
        parent[r] = par[l] ? host_rank(p, tree, par[l]) : -1;
        left[r] = lc[l] ? host_rank(p, tree, lc[l]) : -1;
        right[r] = rc[l] ? host_rank(p, tree, rc[l]) : -1;
    }
    return host_rank(p, tree, root);
}

int64_t oracle_dbtree_half(int64_t n) { return (n + 1) / 2; }

/* partial sum of the subtree under rank r; v[w] = worker w's value */
static float subtree_sum(const float *v, const int32_t *left, const int32_t *right, int r) {
    float s = v[r];
    if (left[r] >= 0) s = s + subtree_sum(v, left, right, left[r]);
    if (right[r] >= 0) s = s + subtree_sum(v, left, right, right[r]);
    return s;
}

struct dbtrees {
    int32_t parent[2][64], left[2][64], right[2][64];
    int root[2];
};

static int dbtrees_make(int p, struct dbtrees *t) {
    for (int k = 0; k < 2; ++k) {
        t->root[k] = oracle_dbtree_build(p, k, t->parent[k], t->left[k], t->right[k]);
        if (t->root[k] < 0) return -1;
    }
    return 0;
}

static float dbtree_value(const struct dbtrees *t, int p, int64_t n, int op, int64_t k, const float *v) {
    int tr = k < oracle_dbtree_half(n) ? 0 : 1;
    float s = subtree_sum(v, t->left[tr], t->right[tr], t->root[tr]);
    if (op == ORACLE_AVG) s = s / (float)p;
    return s;
}

int oracle_dbtree_fold_f32(const float *const *x, int p, int64_t n, int op, float *out) {
    struct dbtrees t;
    if (n < 0 || (op != ORACLE_SUM && op != ORACLE_AVG) || dbtrees_make(p, &t)) return -1;
    float v[64];
    for (int64_t k = 0; k < n; ++k) {
        for (int w = 0; w < p; ++w) v[w] = x[w][k];
        out[k] = dbtree_value(&t, p, n, op, k, v);
    }
    return 0;
}

int oracle_dbtree_fold_bf16(const uint16_t *const *x, int p, int64_t n, int op, uint16_t *out) {
    struct dbtrees t;
    if (n < 0 || (op != ORACLE_SUM && op != ORACLE_AVG) || dbtrees_make(p, &t)) return -1;
    float v[64];
    for (int64_t k = 0; k < n; ++k) {
        for (int w = 0; w < p; ++w) v[w] = oracle_bf16_to_f32(x[w][k]);
        out[k] = oracle_f32_to_bf16(dbtree_value(&t, p, n, op, k, v));
    }
    return 0;
}

/* sampled forms: vals[w * count + j] = worker w's value at element e[j] */
int oracle_dbtree_fold_f32_samples(const float *vals, int p, int64_t n, int op, const int64_t *e,
                                   int64_t count, float *out) {
    struct dbtrees t;
    if (n < 0 || (op != ORACLE_SUM && op != ORACLE_AVG) || dbtrees_make(p, &t)) return -1;
    float v[64];
    for (int64_t j = 0; j < count; ++j) {
        if (e[j] < 0 || e[j] >= n) return -1;
        for (int w = 0; w < p; ++w) v[w] = vals[(int64_t)w * count + j];
        out[j] = dbtree_value(&t, p, n, op, e[j], v);
    }
    return 0;
}

int oracle_dbtree_fold_bf16_samples(const uint16_t *vals, int p, int64_t n, int op, const int64_t *e,
                                    int64_t count, uint16_t *out) {
    struct dbtrees t;
    if (n < 0 || (op != ORACLE_SUM && op != ORACLE_AVG) || dbtrees_make(p, &t)) return -1;
    float v[64];
    for (int64_t j = 0; j < count; ++j) {
        if (e[j] < 0 || e[j] >= n) return -1;
        for (int w = 0; w < p; ++w) v[w] = oracle_bf16_to_f32(vals[(int64_t)w * count + j]);
        out[j] = oracle_f32_to_bf16(dbtree_value(&t, p, n, op, e[j], v));
    }
    return 0;
}

/* Literal schedule, in place on p fp32 buffers, the two trees side by side
 * in synchronous steps.  Reduce: a rank whose children have all delivered
 * adds their partial sums into its own half (left child's first), and sends
 * the result to its parent at the next step.  The root divides by p (AVG).
 * Broadcast: a rank that holds the result copies it to its children at the
 * next step.  *steps: synchronous steps taken; sent_elems[w]: elements rank
 * w put on the wire. */
int oracle_dbtree_schedule_f32(float *const *bufs, int p, int64_t n, int op, int64_t *sent_elems,
                               int *steps) {
    struct dbtrees t;
    if (n < 0 || (op != ORACLE_SUM && op != ORACLE_AVG) || dbtrees_make(p, &t)) return -1;
    const int64_t h = oracle_dbtree_half(n);
    const int64_t beg[2] = {0, h}, len[2] = {h, n - h};
    const size_t slot = (size_t)(h > 0 ? h : 1);
    float *inbox = (float *)malloc(sizeof(float) * slot * 2 * 2 * (size_t)p); /* [tree][rank][side] */
    if (!inbox) return -1;
    int got[2][64][2], ready[2][64], sent[2][64];
    for (int w = 0; w < p; ++w)
        if (sent_elems) sent_elems[w] = 0;
    for (int k = 0; k < 2; ++k)
        for (int r = 0; r < p; ++r) {
            got[k][r][0] = got[k][r][1] = 0;
            ready[k][r] = t.left[k][r] < 0 && t.right[k][r] < 0; /* a leaf's partial is its own value */
            sent[k][r] = 0;
        }
    int nsteps = 0;
    while (!ready[0][t.root[0]] || !ready[1][t.root[1]]) {
        for (int k = 0; k < 2; ++k) /* every send of this step, then every receive */
            for (int r = 0; r < p; ++r) {
                if (r == t.root[k] || !ready[k][r] || sent[k][r]) continue;
                int up = t.parent[k][r], side = t.left[k][up] == r ? 0 : 1;
                float *box = inbox + (((size_t)k * (size_t)p + (size_t)up) * 2 + (size_t)side) * slot;
                memcpy(box, bufs[r] + beg[k], sizeof(float) * (size_t)len[k]);
                got[k][up][side] = 1;
                sent[k][r] = 1;
                if (sent_elems) sent_elems[r] += len[k];
            }
        for (int k = 0; k < 2; ++k)
            for (int r = 0; r < p; ++r) {
                if (ready[k][r]) continue;
                if ((t.left[k][r] >= 0 && !got[k][r][0]) || (t.right[k][r] >= 0 && !got[k][r][1])) continue;
                for (int side = 0; side < 2; ++side) {
                    if ((side == 0 ? t.left[k][r] : t.right[k][r]) < 0) continue;
                    const float *box = inbox + (((size_t)k * (size_t)p + (size_t)r) * 2 + (size_t)side) * slot;
                    for (int64_t j = 0; j < len[k]; ++j) bufs[r][beg[k] + j] = bufs[r][beg[k] + j] + box[j];
                }
                ready[k][r] = 1;
            }
        ++nsteps;
    }
    free(inbox);
    for (int k = 0; k < 2; ++k)
        if (op == ORACLE_AVG)
            for (int64_t j = 0; j < len[k]; ++j)
                bufs[t.root[k]][beg[k] + j] = bufs[t.root[k]][beg[k] + j] / (float)p;
    int have[2][64], pending = 0;
    for (int k = 0; k < 2; ++k)
        for (int r = 0; r < p; ++r) {
            have[k][r] = r == t.root[k];
            pending += !have[k][r];
        }
    while (pending > 0) {
        int had[2][64];
        memcpy(had, have, sizeof(had));
        for (int k = 0; k < 2; ++k)
            for (int r = 0; r < p; ++r) {
                if (!had[k][r]) continue;
                for (int side = 0; side < 2; ++side) {
                    int c = side == 0 ? t.left[k][r] : t.right[k][r];
                    if (c < 0 || have[k][c]) continue;
                    memcpy(bufs[c] + beg[k], bufs[r] + beg[k], sizeof(float) * (size_t)len[k]);
                    have[k][c] = 1;
                    --pending;
                    if (sent_elems) sent_elems[r] += len[k];
                }
            }
        ++nsteps;
    }
    if (steps) *steps = nsteps;
    return 0;
}

/* ===================================================================== */
/* Tensor Fusion [H] "Tensor Fusion", steps 1-6                           */
/* ===================================================================== */
static int dtype_bytes(int32_t dt) {
    if (dt == ORACLE_F32) return 4;
    if (dt == ORACLE_BF16) return 2;
    return -1;
}

/* Tensors are taken in list (ready) order.  A tensor joins the open buffer
 * when it has the buffer's dtype and fits in the room left (its start
 * rounded up to align_bytes); otherwise the open buffer is closed and a new
 * one starts with this tensor.  A tensor larger than the capacity gets a
 * buffer to itself.                                                         */
int oracle_fusion_plan(const int64_t *numel, const int32_t *dtype, int count,
                       int64_t capacity_bytes, int align_bytes, int32_t *seg_buffer,
                       int64_t *seg_offset, int64_t *buf_numel) {
    if (count < 0 || capacity_bytes <= 0 || align_bytes <= 0) return -1;
    int nbuf = 0;
    int32_t open_dtype = -1;
    int64_t used = 0; /* bytes used in the open buffer */
    for (int i = 0; i < count; ++i) {
        int es = dtype_bytes(dtype[i]);
        if (es < 0 || numel[i] < 0 || align_bytes % es != 0) return -1;
        int64_t bytes = numel[i] * es;
        int64_t start = (used + align_bytes - 1) / align_bytes * align_bytes;
        int fits = nbuf > 0 && dtype[i] == open_dtype && start + bytes <= capacity_bytes;
        if (!fits) {
            ++nbuf;
            open_dtype = dtype[i];
            start = 0;
        }
        seg_buffer[i] = nbuf - 1;
        seg_offset[i] = start / es;
        used = start + bytes;
        buf_numel[nbuf - 1] = used / es;
    }
    return nbuf;
}

int oracle_fusion_pack(const void *const *src, const int32_t *seg_buffer,
                       const int64_t *seg_offset, const int64_t *numel, int count, int buffer,
                       void *fusion_buf, int64_t buf_numel, int elem_bytes) {
    if (elem_bytes <= 0 || buf_numel < 0) return -1;
    unsigned char *dst = (unsigned char *)fusion_buf;
    memset(dst, 0, (size_t)(buf_numel * elem_bytes));
    for (int i = 0; i < count; ++i) {
        if (seg_buffer[i] != buffer) continue;
        if (seg_offset[i] + numel[i] > buf_numel) return -1;
        memcpy(dst + seg_offset[i] * elem_bytes, src[i], (size_t)(numel[i] * elem_bytes));
    }
    return 0;
}

int oracle_fusion_unpack(const void *fusion_buf, const int32_t *seg_buffer,
                         const int64_t *seg_offset, const int64_t *numel, int count, int buffer,
                         void *const *dst, int elem_bytes) {
    if (elem_bytes <= 0) return -1;
    const unsigned char *src = (const unsigned char *)fusion_buf;
    for (int i = 0; i < count; ++i) {
        if (seg_buffer[i] != buffer) continue;
        memcpy(dst[i], src + seg_offset[i] * elem_bytes, (size_t)(numel[i] * elem_bytes));
    }
    return 0;
}

/* ===================================================================== */
/* Uniform THC [T] section 4, Algorithm 1                                 */
/* ===================================================================== */

/* Preliminary round: the global smallest and largest entry over all
 * workers.  NaN entries are skipped. */
void oracle_thc_range(const float *const *x, int p, int64_t n, float *m, float *M) {
    float lo = INFINITY, hi = -INFINITY;
    for (int w = 0; w < p; ++w)
        for (int64_t k = 0; k < n; ++k) {
            float v = x[w][k];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
    *m = lo;
    *M = hi;
}

/* The 2^b quantization values are q_j = m + j (M - m) / L, L = 2^b - 1.
 * The position of a value on that grid, in fp32: (x - m) times the fp32
 * scale L / (M - m), clamped to [0, L]. */
float oracle_thc_position(float x, float m, float M, int b) {
    const float L = (float)((1u << b) - 1u);
    if (M == m) return 0.0f;
    float range = M - m;
    float scale = L / range;
    float d = x - m;
    float t = d * scale;
    if (t < 0.0f) t = 0.0f;
    if (t > L) t = L;
    return t;
}

/* Stochastic quantization: a value between q_j and q_{j+1} goes up to
 * q_{j+1} with probability equal to its fractional position f and down to
 * q_j otherwise, which makes it unbiased.  The uniform draw u comes from
 * the Philox4x32-10 stream keyed by the 64-bit seed: counter
 * (e/4 low word, e/4 high word, worker, 0), output word e mod 4, of which
 * the low 23 bits are read as u = bits / 2^23 in [0, 1).  Up iff u < f. */
uint32_t oracle_thc_index(float x, float m, float M, int b, uint64_t seed, int worker,
                          int64_t e) {
    float t = oracle_thc_position(x, m, M, b);
    float j = floorf(t);
    float f = t - j;
    uint64_t q = (uint64_t)e >> 2;
    uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), (uint32_t)worker, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    oracle_philox4x32(ctr, key, 10, r);
    uint32_t bits = r[e & 3] & 0x7FFFFFu;
    float u = (float)bits / 8388608.0f; /* exact: bits < 2^23 */
    return (uint32_t)j + (u < f ? 1u : 0u);
}

static int valid_bits(int b) { return b == 1 || b == 2 || b == 4 || b == 8; }

/* Indices are packed least significant bits first: element e sits in
 * word e / (32 / b) at bit (e mod (32 / b)) * b; the last word is padded
 * with zero indices. */
int oracle_thc_encode(const float *x, int64_t n, float m, float M, int b, uint64_t seed,
                      int worker, uint32_t *packed) {
    if (!valid_bits(b) || n < 0) return -1;
    int per_word = 32 / b;
    int64_t nwords = (n + per_word - 1) / per_word;
    for (int64_t k = 0; k < nwords; ++k) packed[k] = 0u;
    for (int64_t e = 0; e < n; ++e) {
        uint32_t idx = oracle_thc_index(x[e], m, M, b, seed, worker, e);
        packed[e / per_word] |= idx << ((e % per_word) * b);
    }
    return 0;
}

int oracle_thc_unpack(const uint32_t *packed, int64_t n, int b, uint8_t *idx) {
    if (!valid_bits(b) || n < 0) return -1;
    int per_word = 32 / b;
    uint32_t mask = (1u << b) - 1u;
    for (int64_t e = 0; e < n; ++e)
        idx[e] = (uint8_t)((packed[e / per_word] >> ((e % per_word) * b)) & mask);
    return 0;
}

/* The PS sums the workers' index vectors as integers; nothing is decoded. */
int oracle_thc_aggregate(const uint32_t *const *packed, int p, int64_t n, int b,
                         uint16_t *sums) {
    if (!valid_bits(b) || n < 0 || p < 1) return -1;
    if ((int64_t)p * ((1 << b) - 1) > 65535) return -1;
    int per_word = 32 / b;
    uint32_t mask = (1u << b) - 1u;
    for (int64_t e = 0; e < n; ++e) {
        uint32_t s = 0;
        for (int w = 0; w < p; ++w) s += (packed[w][e / per_word] >> ((e % per_word) * b)) & mask;
        sums[e] = (uint16_t)s;
    }
    return 0;
}

/* Each worker divides the index sum by the number of workers and maps the
 * average index back onto the grid: avg = m + (S / p) (M - m) / L, in fp64. */
int oracle_thc_decode(const uint16_t *sums, int64_t n, float m, float M, int b, int p,
                      double *avg) {
    if (!valid_bits(b) || n < 0 || p < 1) return -1;
    double L = (double)((1 << b) - 1);
    double step = ((double)M - (double)m) / L;
    for (int64_t e = 0; e < n; ++e) avg[e] = (double)m + ((double)sums[e] / (double)p) * step;
    return 0;
}

int oracle_thc_allreduce_samples(const float *vals, int p, const int64_t *e, int64_t count, int b,
                                 uint64_t seed, float m, float M, uint8_t *idx, double *avg) {
    if (!valid_bits(b) || p < 1 || count < 0) return -1;
    double L = (double)((1 << b) - 1);
    double step = ((double)M - (double)m) / L;
    for (int64_t k = 0; k < count; ++k) {
        uint32_t s = 0;
        for (int w = 0; w < p; ++w) {
            uint32_t i = oracle_thc_index(vals[(int64_t)w * count + k], m, M, b, seed, w, e[k]);
            if (idx) idx[(int64_t)w * count + k] = (uint8_t)i;
            s += i;
        }
        avg[k] = (double)m + ((double)s / (double)p) * step;
    }
    return 0;
}

int oracle_thc_allreduce_masked(const float *const *x, int p, uint64_t arrived, int64_t n, int b,
                                uint64_t seed, float m, float M, double *avg, uint32_t *const *packed) {
    if (!valid_bits(b) || n < 0 || p < 1 || p > 64) return -1;
    int p_eff = 0;
    for (int w = 0; w < p; ++w) p_eff += (int)((arrived >> w) & 1u);
    if (p_eff == 0) return -1;
    double L = (double)((1 << b) - 1);
    double step = ((double)M - (double)m) / L;
    for (int w = 0; w < p; ++w) {
        if (!((arrived >> w) & 1u) || !packed) continue;
        if (oracle_thc_encode(x[w], n, m, M, b, seed, w, packed[w]) != 0) return -1;
    }
    for (int64_t e = 0; e < n; ++e) {
        uint32_t s = 0;
        for (int w = 0; w < p; ++w)
            if ((arrived >> w) & 1u) s += oracle_thc_index(x[w][e], m, M, b, seed, w, e);
        avg[e] = (double)m + ((double)s / (double)p_eff) * step;
    }
    return 0;
}

int oracle_thc_allreduce(const float *const *x, int p, int64_t n, int b, uint64_t seed,
                         float m, float M, double *avg, uint32_t *const *packed) {
    if (!valid_bits(b) || n < 0 || p < 1) return -1;
    int per_word = 32 / b;
    int64_t nwords = (n + per_word - 1) / per_word;
    uint32_t **pk = (uint32_t **)calloc((size_t)p, sizeof(uint32_t *));
    uint16_t *sums = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1));
    int rc = (pk && sums) ? 0 : -1;
    for (int w = 0; w < p && rc == 0; ++w) {
        pk[w] = packed ? packed[w]
                       : (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(nwords > 0 ? nwords : 1));
        if (!pk[w]) rc = -1;
        else rc = oracle_thc_encode(x[w], n, m, M, b, seed, w, pk[w]);
    }
    if (rc == 0) rc = oracle_thc_aggregate((const uint32_t *const *)pk, p, n, b, sums);
    if (rc == 0) rc = oracle_thc_decode(sums, n, m, M, b, p, avg);
    if (pk && !packed)
        for (int w = 0; w < p; ++w) free(pk[w]);
    free(pk);
    free(sums);
    return rc;
}

/* ===================================================================== */
/* Non-uniform THC [T] section 5, Algorithm 2                             */
/* ===================================================================== */
/* With granularity g >= 2^b - 1 the grid is m + k (M - m) / g, k = 0..g,
 * but a worker may only send the 2^b grid points whose k is a table value
 * T[z].  It rounds stochastically between the two neighbouring allowed
 * points (unbiased), sends the table index z, the PS looks each index up in
 * T and sums the looked-up values, and each worker divides that sum by the
 * number of workers and maps it back: avg = m + (Y / p) (M - m) / g.  With
 * g = 2^b - 1 and T the identity this is exactly uniform THC.            */
int oracle_nuhc_check_table(const uint16_t *table, int b, int g) {
    if (!valid_bits(b)) return -1;
    int L = (1 << b) - 1;
    if (g < L || table[0] != 0 || table[L] != g) return -1;
    for (int z = 0; z < L; ++z)
        if (table[z + 1] <= table[z]) return -1;
    return 0;
}

float oracle_nuhc_position(float x, float m, float M, int g) {
    const float G = (float)g;
    if (M == m) return 0.0f;
    float range = M - m;
    float scale = G / range;
    float d = x - m;
    float t = d * scale;
    if (t < 0.0f) t = 0.0f;
    if (t > G) t = G;
    return t;
}

uint32_t oracle_nuhc_index(float x, float m, float M, int b, int g, const uint16_t *table,
                           uint64_t seed, int worker, int64_t e) {
    int L = (1 << b) - 1;
    float t = oracle_nuhc_position(x, m, M, g);
    /* the allowed grid points around t: table[z] <= t <= table[z + 1] */
    int z = 0;
    while (z < L - 1 && t >= (float)table[z + 1]) ++z;
    float lo = (float)table[z], hi = (float)table[z + 1];
    /* rounds up to table[z + 1] with probability (t - lo) / (hi - lo): up iff
     * u (hi - lo) < t - lo, compared exactly in double (t - lo is exact in
     * float, the product has at most 37 significant bits) */
    uint64_t q = (uint64_t)e >> 2;
    uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), (uint32_t)worker, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    oracle_philox4x32(ctr, key, 10, r);
    float u = (float)(r[e & 3] & 0x7FFFFFu) / 8388608.0f;
    double a = (double)(t - lo), d = (double)(hi - lo);
    return (uint32_t)z + ((double)u * d < a ? 1u : 0u);
}

int oracle_nuhc_encode(const float *x, int64_t n, float m, float M, int b, int g,
                       const uint16_t *table, uint64_t seed, int worker, uint32_t *packed) {
    if (oracle_nuhc_check_table(table, b, g) != 0 || n < 0) return -1;
    int per_word = 32 / b;
    int64_t nwords = (n + per_word - 1) / per_word;
    for (int64_t k = 0; k < nwords; ++k) packed[k] = 0u;
    for (int64_t e = 0; e < n; ++e) {
        uint32_t idx = oracle_nuhc_index(x[e], m, M, b, g, table, seed, worker, e);
        packed[e / per_word] |= idx << ((e % per_word) * b);
    }
    return 0;
}

/* The same encoding of a run of a longer vector: x[k] is element e0 + k
 * (e0 a whole number of packed words into the vector), so the draws are
 * those of the whole vector's encoding and packed[j] is its word
 * e0 / (32 / b) + j. */
int oracle_nuhc_encode_at(const float *x, int64_t n, int64_t e0, float m, float M, int b, int g,
                          const uint16_t *table, uint64_t seed, int worker, uint32_t *packed) {
    if (oracle_nuhc_check_table(table, b, g) != 0 || n < 0 || e0 < 0) return -1;
    int per_word = 32 / b;
    if (e0 % per_word != 0) return -1;
    int64_t nwords = (n + per_word - 1) / per_word;
    for (int64_t k = 0; k < nwords; ++k) packed[k] = 0u;
    for (int64_t k = 0; k < n; ++k) {
        uint32_t idx = oracle_nuhc_index(x[k], m, M, b, g, table, seed, worker, e0 + k);
        packed[k / per_word] |= idx << ((k % per_word) * b);
    }
    return 0;
}

int oracle_nuhc_aggregate(const uint32_t *const *packed, int p, int64_t n, int b,
                          const uint16_t *table, uint16_t *sums) {
    if (!valid_bits(b) || n < 0 || p < 1) return -1;
    int L = (1 << b) - 1;
    if ((int64_t)p * table[L] > 65535) return -1;
    int per_word = 32 / b;
    uint32_t mask = (1u << b) - 1u;
    for (int64_t e = 0; e < n; ++e) {
        uint32_t s = 0;
        for (int w = 0; w < p; ++w) s += table[(packed[w][e / per_word] >> ((e % per_word) * b)) & mask];
        sums[e] = (uint16_t)s;
    }
    return 0;
}

int oracle_nuhc_decode(const uint16_t *sums, int64_t n, float m, float M, int g, int p,
                       double *avg) {
    if (g < 1 || n < 0 || p < 1) return -1;
    double step = ((double)M - (double)m) / (double)g;
    for (int64_t e = 0; e < n; ++e) avg[e] = (double)m + ((double)sums[e] / (double)p) * step;
    return 0;
}

/* ===================================================================== */
/* Randomized Hadamard Transform [T] section 5                            */
/* ===================================================================== */
static int is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

int oracle_rht_signs(int64_t n, uint64_t seed, int8_t *d) {
    if (n < 0) return -1;
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    for (int64_t i = 0; i < n; ++i) {
        uint64_t q = (uint64_t)i >> 7;
        uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), 0xFFFFFFFFu, 0u};
        uint32_t r[4];
        oracle_philox4x32(ctr, key, 10, r);
        uint32_t bit = (r[(i >> 5) & 3] >> (i & 31)) & 1u;
        d[i] = bit ? (int8_t)-1 : (int8_t)1;
    }
    return 0;
}

/* In-place fast Walsh-Hadamard transform (unnormalised): for each stride h
 * = 1, 2, 4, ..., pairs (a, b) at distance h become (a + b, a - b).  This is
 * H_n x for the Sylvester construction H_2n = [[H_n, H_n], [H_n, -H_n]]. */
static void fwht(double *v, int64_t n) {
    for (int64_t h = 1; h < n; h <<= 1)
        for (int64_t i = 0; i < n; i += 2 * h)
            for (int64_t j = i; j < i + h; ++j) {
                double a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
}

int oracle_rht(const double *in, int64_t n, uint64_t seed, int inverse, double *out) {
    if (!is_pow2(n)) return -1;
    int8_t *d = (int8_t *)malloc((size_t)n);
    if (!d) return -1;
    oracle_rht_signs(n, seed, d);
    double scale = 1.0 / sqrt((double)n);
    for (int64_t i = 0; i < n; ++i) out[i] = inverse ? in[i] : in[i] * d[i];
    fwht(out, n);
    for (int64_t i = 0; i < n; ++i) out[i] = (inverse ? out[i] * d[i] : out[i]) * scale;
    free(d);
    return 0;
}

void oracle_ef_apply(const float *grad, const float *e, float *x, int64_t n) {
    for (int64_t i = 0; i < n; ++i) x[i] = grad[i] + e[i];
}

void oracle_ef_update(float *e, const float *x, const float *x_hat, int64_t n) {
    for (int64_t i = 0; i < n; ++i) e[i] = x[i] - x_hat[i];
}

void oracle_rht_norm_range(const double *const *x, int p, int64_t n, double t_p, double *m,
                           double *M) {
    double l = 0.0;
    for (int w = 0; w < p; ++w) {
        double s = 0.0;
        for (int64_t i = 0; i < n; ++i) s += x[w][i] * x[w][i];
        if (sqrt(s) > l) l = sqrt(s);
    }
    *M = t_p / sqrt((double)n) * l;
    *m = -*M;
}

/* ===================================================================== */
/* NMSE [T] section 2: ||x - x_hat||^2 / ||x||^2, accumulated in fp64.     */
/* ===================================================================== */
double oracle_nmse(const float *x, const float *x_hat, int64_t n) {
    double num = 0.0, den = 0.0;
    for (int64_t k = 0; k < n; ++k) {
        double d = (double)x[k] - (double)x_hat[k];
        num += d * d;
        den += (double)x[k] * (double)x[k];
    }
    if (den == 0.0) return NAN;
    return num / den;
}

double oracle_nmse_f64(const double *x, const double *x_hat, int64_t n) {
    double num = 0.0, den = 0.0;
    for (int64_t k = 0; k < n; ++k) {
        double d = x[k] - x_hat[k];
        num += d * d;
        den += x[k] * x[k];
    }
    if (den == 0.0) return NAN;
    return num / den;
}

/* ===================================================================== */
/* Wire-vector checksum (silent data corruption check of the packed       */
/* indices): s1 = sum w_i, s2 = sum (i + 1) w_i over the 32-bit words,    */
/* both mod 2^32; returns (s2 << 32) | s1.                                */
/* ===================================================================== */
uint64_t oracle_checksum(const uint32_t *w, int64_t n) {
    uint32_t s1 = 0, s2 = 0;
    for (int64_t i = 0; i < n; ++i) {
        s1 += w[i];
        s2 += (uint32_t)(i + 1) * w[i];
    }
    return ((uint64_t)s2 << 32) | s1;
}
