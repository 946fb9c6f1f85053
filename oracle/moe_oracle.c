/*
 * moe_oracle.c -- CPU oracle for the MoE token path (route, dispatch layout,
 * pack, receiver permute, stand-in expert, weighted combine).
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use this file.  The CUDA library never includes, links or
 * calls it, and it shares no code with the CUDA library: every definition
 * below is written out again from the pages.
 *
 * Style: plain single-threaded loops in the order the definitions are stated,
 * double precision for every floating-point sum, no blocking and no fusion.
 *
 * Sources (cited by page and section):
 *   [a2a]  "a2a-backends", vincentzed.com/writing/a2a-backends
 *   [b1g]  "Beyond One GPU: Tensor, Pipeline and Expert Parallelism, and Split
 *          Prefill and Decode", ishwarj.com/writings/llm-inference-7-beyond-one-gpu
 *
 * Parity pins: every function here is checked by the CPU test suite against
 * values the pages print, closed forms, invariants or brute force (see the
 * tests named after each function).  No function is unpinned.
 *
 * Layout conventions (shared with the C-ABI only through its documentation):
 *   S sources, T tokens per source, k experts per token, E experts, P
 *   partitions of L = E/P contiguous experts, H bf16 elements per row.
 *   ids/weights: [S][T][k]; token_slot: [S][T][P]; send: [S][cap_send][H].
 *   Status bits: bit 1 = inconsistent index input, bit 2 = capacity
 *   overflow, bit 3 = expert id >= E.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/*
 * ORC_MUTANT n (n > 0) plants one deliberate mistake, numbered below; the
 * test suite builds such mutants to show that its pins reject them.  The
 * normal build has ORC_MUTANT 0 and none of them.
 */
#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

#define ORC_BIT_INCONSISTENT (1u << 1)
#define ORC_BIT_CAPACITY     (1u << 2)
#define ORC_BIT_BAD_ID       (1u << 3)

/* ---------------------------------------------------------------- bf16 -- */

/* A bfloat16 bit pattern is the upper half of the float32 with the same value. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to bfloat16, to nearest with ties to even, in ONE rounding
 * (no detour through float32, which would round twice).
 * bfloat16 keeps 8 significant bits and float32's exponent range: a normal
 * value in [2^(e-1), 2^e) has quantum 2^(e-8); below 2^-126 the quantum is
 * fixed at 2^-133.  Values that round to 2^128 or beyond become infinity.
 */
uint16_t oracle_bf16_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return 0x7FC0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80u;
    int ex;
    frexp(a, &ex);               /* a in [2^(ex-1), 2^ex) */
    int qe = ex - 8;
    if (qe < -133)
        qe = -133;
    double q = ldexp(1.0, qe);
#if ORC_MUTANT == 1
    double r = floor(a / q) * q;     /* mutant 1: truncates instead of rounding */
#else
    double r = nearbyint(a / q) * q; /* a/q is exact; default mode: ties to even */
#endif
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80u;
    float f = (float)r;          /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------- closed form, [a2a] 1.3 */

/* Binomial coefficient C(n, r) as a double (multiplicative formula). */
static double binom(int n, int r)
{
    if (r < 0 || r > n)
        return 0.0;
    double c = 1.0;
    for (int i = 1; i <= r; i++)
        c = c * (double)(n - r + i) / (double)i;
    return c;
}

/*
 * [a2a] 1.3: a GPU holding E/G of E experts misses all k picks of a uniform
 * router with probability C(E - E/G, k) / C(E, k); a token therefore needs
 * G * (1 - C(E - E/G, k) / C(E, k)) GPUs on average.
 */
double oracle_expected_copies(int E, int G, int k)
{
#if ORC_MUTANT == 6
    return (double)G * (1.0 - binom(E - G, k) / binom(E, k));   /* mutant 6 */
#else
    return (double)G * (1.0 - binom(E - E / G, k) / binom(E, k));
#endif
}

/* ------------------------------------------------------- route, [a2a] 1.1 */

typedef struct {
    float v;
    int32_t id;
} orc_cand;

/* Larger logit first; equal logits: lower expert id first. */
static int cand_cmp(const void *pa, const void *pb)
{
    const orc_cand *a = (const orc_cand *)pa, *b = (const orc_cand *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
#if ORC_MUTANT == 2
    return (a->id < b->id) - (a->id > b->id);   /* mutant 2: ties to the higher id */
#else
    return (a->id > b->id) - (a->id < b->id);
#endif
}

/*
 * [a2a] 1.1: the router gives every token the ids of its chosen experts and
 * one weight per expert.  Chosen experts: the k largest logits, by sorting
 * the whole row (descending, ties to the lower id).  Weights: softmax over
 * the k chosen logits, w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max), in
 * double.  logits [N][E] -> ids [N][k], w [N][k]; N = S*T rows.
 */
int oracle_route_topk(const float *logits, int64_t N, int E, int k,
                      int32_t *ids, double *w)
{
    if (k < 1 || k > E)
        return -1;
    orc_cand *c = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)E);
    if (!c)
        return -2;
    for (int64_t n = 0; n < N; n++) {
        const float *row = logits + n * (int64_t)E;
        for (int e = 0; e < E; e++) {
            c[e].v = row[e];
            c[e].id = e;
        }
        qsort(c, (size_t)E, sizeof(orc_cand), cand_cmp);
        double lmax = (double)c[0].v, denom = 0.0;
#if ORC_MUTANT == 3
        for (int j = 0; j < E; j++)                 /* mutant 3: softmax over every logit */
#else
        for (int j = 0; j < k; j++)
#endif
            denom += exp((double)c[j].v - lmax);
        for (int j = 0; j < k; j++) {
            ids[n * k + j] = c[j].id;
            w[n * k + j] = exp((double)c[j].v - lmax) / denom;
        }
    }
    free(c);
    return 0;
}

/* ---------------------------------------------- dispatch layout, [a2a] 1.3 */

/*
 * Expert e lives on partition e / L with L = E / P: contiguous blocks of
 * experts per GPU, [a2a] 2.1 (local ids first_local .. first_local+num_local)
 * and the 48-of-384 split of [a2a] 1.1.
 *
 * A token is copied once to every partition holding at least one of its
 * experts ([a2a] 1.1 Figure 1, 1.3 third answer, 3.2 first step).  Ids < 0
 * are "not routed" and skipped; ids >= E are skipped and flagged.
 *
 *   expert_counts[s][e]  = #{(t, j) : ids[s][t][j] == e}
 *   expert_rank[s][t][j] = #{(t', j') before (t, j) in (token, slot) order :
 *                            ids[s][t'][j'] == ids[s][t][j]}, or -1 if skipped
 *                          (the pair's place in its expert's run of source s;
 *                          the receiver's runs in [a2a] 1.5 / 3.3 are built
 *                          from it)
 *   part_counts[s][p]    = #{t : token t hits partition p}
 *   part_offsets[s][0]   = 0, part_offsets[s][p+1] = part_offsets[s][p] + part_counts[s][p]
 *   token_slot[s][t][p]  = part_offsets[s][p] + #{t' < t : t' hits p}, or -1
 *
 * Rows of one partition's region are in ascending token order.
 */
int oracle_dispatch_layout(const int32_t *ids, int S, int64_t T, int k, int E, int P,
                           int32_t *expert_counts, int32_t *expert_rank, int32_t *part_counts,
                           int32_t *part_offsets, int32_t *token_slot,
                           uint32_t *status)
{
    if (P < 1 || E % P != 0)
        return -1;
    const int L = E / P;
    char *hit = (char *)malloc((size_t)P);
    int32_t *seen = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!hit || !seen) {
        free(hit);
        free(seen);
        return -2;
    }
    for (int s = 0; s < S; s++) {
        for (int e = 0; e < E; e++)
            expert_counts[s * E + e] = 0;
        for (int p = 0; p < P; p++)
            part_counts[s * P + p] = 0;
        /* pass 1: counts */
        for (int64_t t = 0; t < T; t++) {
            memset(hit, 0, (size_t)P);
            for (int j = 0; j < k; j++) {
                int32_t e = ids[((int64_t)s * T + t) * k + j];
                if (e < 0)
                    continue;
                if (e >= E) {
                    *status |= ORC_BIT_BAD_ID;
                    continue;
                }
                expert_counts[s * E + e] += 1;
#if ORC_MUTANT == 4
                hit[e % P] = 1;                     /* mutant 4: experts dealt round robin */
#else
                hit[e / L] = 1;
#endif
            }
            for (int p = 0; p < P; p++)
                part_counts[s * P + p] += hit[p];
        }
        part_offsets[s * (P + 1) + 0] = 0;
        for (int p = 0; p < P; p++)
            part_offsets[s * (P + 1) + p + 1] = part_offsets[s * (P + 1) + p] + part_counts[s * P + p];
        /* ranks: walk the pairs in (token, slot) order; a pair's rank is how
         * many pairs of this source with the same expert were seen before it */
        for (int e = 0; e < E; e++)
            seen[e] = 0;
        for (int64_t t = 0; t < T; t++) {
            for (int j = 0; j < k; j++) {
                int64_t q = ((int64_t)s * T + t) * k + j;
                int32_t e = ids[q];
                if (e < 0 || e >= E) {
                    expert_rank[q] = -1;
                    continue;
                }
                expert_rank[q] = seen[e]++;
            }
        }
        /* pass 2: slots, ascending token order within each partition */
        for (int p = 0; p < P; p++) {
            int32_t next = part_offsets[s * (P + 1) + p];
            for (int64_t t = 0; t < T; t++) {
                int h = 0;
                for (int j = 0; j < k; j++) {
                    int32_t e = ids[((int64_t)s * T + t) * k + j];
#if ORC_MUTANT == 4
                    if (e >= 0 && e < E && e % P == p)
#else
                    if (e >= 0 && e < E && e / L == p)
#endif
                        h = 1;
                }
#if ORC_MUTANT == 5
                token_slot[((int64_t)s * T + t) * P + p] = h ? ++next : -1;   /* mutant 5 */
#else
                token_slot[((int64_t)s * T + t) * P + p] = h ? next++ : -1;
#endif
            }
        }
    }
    free(hit);
    free(seen);
    return 0;
}

/* ------------------------------------------------- pack, [a2a] 3.2, 5.1 */

/*
 * Sender side of dispatch: each (token, partition) with a slot gets a bit copy
 * of the token's row in that partition's region of the send buffer
 * ([a2a] 3.2 fourth step, 5.1 "a region for every sender", 6.1 one copy per
 * GPU that needs the token).  send_src[s][slot] = t is the source token of
 * the row; unused entries of send_src are -1.  A slot >= cap_send has no room
 * ([a2a] 4.1, 9.2 the cap): it is dropped and flagged.
 */
int oracle_dispatch_pack(const uint16_t *x, int S, int64_t T, int H, int P,
                         const int32_t *token_slot, int64_t cap_send,
                         uint16_t *send, int32_t *send_src, uint32_t *status)
{
    for (int s = 0; s < S; s++) {
        for (int64_t r = 0; r < cap_send; r++)
            send_src[(int64_t)s * cap_send + r] = -1;
        for (int64_t t = 0; t < T; t++) {
            for (int p = 0; p < P; p++) {
                int32_t slot = token_slot[((int64_t)s * T + t) * P + p];
                if (slot < 0)
                    continue;
                if (slot >= cap_send) {
                    *status |= ORC_BIT_CAPACITY;
                    continue;
                }
                memcpy(send + ((int64_t)s * cap_send + slot) * H,
                       x + ((int64_t)s * T + t) * H, sizeof(uint16_t) * (size_t)H);
                send_src[(int64_t)s * cap_send + slot] = (int32_t)t;
            }
        }
    }
    return 0;
}

/* ------------------------------------ receiver permute, [a2a] 1.5, 3.3, 5.1 */

/*
 * Receiver side: one row per (token, local expert), grouped by expert in
 * runs ([a2a] 1.5 contiguous layout; 3.3 "5 rows become 7"; 5.1 the copy
 * epilogue with do_expand and device-side offsets).
 *
 * The receiving set R is one partition (recv_part >= 0) or all of them (-1).
 * For each expert e in ascending order, cnt_e counts the pairs (s, t, j) with
 * ids[s][t][j] == e and part(e) in R; runs are padded to a multiple of
 * `align` rows ([a2a] 1.5: DeepGEMM pads each run to a multiple of 128):
 *   expert_offsets[0] = 0
 *   expert_offsets[e+1] = expert_offsets[e] + (part(e) in R ? ceil(cnt_e/align)*align : 0)
 * Within a run, pairs are in ascending (s, t, j) order (a stable sort of the
 * pairs by expert id).  The pair's row is a copy of its token's row in the
 * send region of partition part(e): send[s][token_slot[s][t][part(e)]].
 *
 *   pair_row[s][t][j] = row of the pair, or -1 (not in R, id < 0, or row >= cap_recv)
 *   recv_pair[row]    = (s*T + t)*k + j for pair rows, -1 for padding rows and
 *                       for rows >= expert_offsets[E]
 *   recv[row]         = the copy; padding rows are zero
 *
 * Flags: row >= cap_recv (dropped) or source slot >= cap_send -> capacity;
 * source slot < 0 for a routed pair -> inconsistent input (row is zeroed);
 * id >= E -> bad id (skipped).
 */
int oracle_permute_to_experts(const uint16_t *send, const int32_t *token_slot,
                              const int32_t *ids, int S, int64_t T, int k, int E, int P,
                              int H, int recv_part, int align, int64_t cap_send,
                              int64_t cap_recv, uint16_t *recv, int32_t *expert_offsets,
                              int32_t *pair_row, int32_t *recv_pair, uint32_t *status)
{
    if (P < 1 || E % P != 0 || align < 1 || recv_part < -1 || recv_part >= P)
        return -1;
    const int L = E / P;
    const int64_t npairs = (int64_t)S * T * k;
    int64_t *cnt = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    int64_t *fill = (int64_t *)calloc((size_t)E, sizeof(int64_t));
    if (!cnt || !fill) {
        free(cnt);
        free(fill);
        return -2;
    }
    /* counts per expert over the receiving set */
    for (int64_t q = 0; q < npairs; q++) {
        int32_t e = ids[q];
        if (e >= E)
            *status |= ORC_BIT_BAD_ID;
        if (e < 0 || e >= E)
            continue;
        if (recv_part >= 0 && e / L != recv_part)
            continue;
        cnt[e]++;
    }
    /* padded run offsets */
    int64_t off = 0;
    for (int e = 0; e < E; e++) {
        expert_offsets[e] = (int32_t)off;
        int in_r = (recv_part < 0) || (e / L == recv_part);
        if (in_r)
            off += (cnt[e] + align - 1) / align * align;
    }
    expert_offsets[E] = (int32_t)off;
    const int64_t total = off;
    /* every row starts as padding */
    for (int64_t r = 0; r < cap_recv; r++)
        recv_pair[r] = -1;
    for (int64_t r = 0; r < total && r < cap_recv; r++)
        memset(recv + r * H, 0, sizeof(uint16_t) * (size_t)H);
    /* pairs in ascending (s, t, j) order go to the end of their expert's run */
    for (int s = 0; s < S; s++) {
        for (int64_t t = 0; t < T; t++) {
            for (int j = 0; j < k; j++) {
                int64_t q = ((int64_t)s * T + t) * k + j;
                int32_t e = ids[q];
                pair_row[q] = -1;
                if (e < 0 || e >= E)
                    continue;
                int p = e / L;
                if (recv_part >= 0 && p != recv_part)
                    continue;
                int64_t row = expert_offsets[e] + fill[e];
                fill[e]++;
                if (row >= cap_recv) {
                    *status |= ORC_BIT_CAPACITY;
                    continue;
                }
                pair_row[q] = (int32_t)row;
                recv_pair[row] = (int32_t)q;
                int32_t slot = token_slot[((int64_t)s * T + t) * P + p];
                if (slot < 0) {
                    *status |= ORC_BIT_INCONSISTENT;
                    continue; /* row stays zero */
                }
                if (slot >= cap_send) {
                    *status |= ORC_BIT_CAPACITY;
                    continue; /* row stays zero */
                }
                memcpy(recv + row * H, send + ((int64_t)s * cap_send + slot) * H,
                       sizeof(uint16_t) * (size_t)H);
            }
        }
    }
    free(cnt);
    free(fill);
    return 0;
}

/* ------------------------------------------- masked layout, [a2a] 4.1-4.2 */

/*
 * The masked receive layout of DeepEP's low-latency mode ([a2a] 4.1: a region
 * per (local expert, sender) with room for the cap; 4.2: the receiver packs
 * each expert's rows together and writes a per-expert count, the output has a
 * fixed shape, 48 x 8 x 128 rows for the decode example; 5.2: SGLang's masked
 * kernel expects these fixed-size blocks).
 *
 * Every expert of the receiving set gets a block of block_rows rows; block b
 * holds expert e = b (recv_part < 0) or e = recv_part*L + b.  The pairs of
 * expert e, in ascending (s, t, j) order, fill the block from row 0; pairs
 * past the block's end are dropped (pair_row -1, capacity flag).
 *   masked_counts[b]            = rows of the block in use (<= block_rows)
 *   recv[b*block_rows + i]      = send[s][token_slot[s][t][part(e)]] of the i-th pair
 *   pair_row[s][t][j]           = its row, or -1
 *   recv_pair[b*block_rows + i] = (s*T + t)*k + j for used rows, -1 otherwise
 * Rows past masked_counts[b] are not written.  Missing source slots behave as
 * in the contiguous layout (zero row, flagged).
 */
int oracle_permute_masked(const uint16_t *send, const int32_t *token_slot, const int32_t *ids,
                          int S, int64_t T, int k, int E, int P, int H, int recv_part,
                          int64_t block_rows, int64_t cap_send, uint16_t *recv,
                          int32_t *masked_counts, int32_t *pair_row, int32_t *recv_pair,
                          uint32_t *status)
{
    if (P < 1 || E % P != 0 || recv_part < -1 || recv_part >= P || block_rows < 0)
        return -1;
    const int L = E / P;
    const int nb = recv_part < 0 ? E : L;
    const int e0 = recv_part < 0 ? 0 : recv_part * L;
    for (int b = 0; b < nb; b++)
        masked_counts[b] = 0;
    for (int64_t r = 0; r < (int64_t)nb * block_rows; r++)
        recv_pair[r] = -1;
    for (int s = 0; s < S; s++) {
        for (int64_t t = 0; t < T; t++) {
            for (int j = 0; j < k; j++) {
                int64_t q = ((int64_t)s * T + t) * k + j;
                int32_t e = ids[q];
                pair_row[q] = -1;
                if (e >= E)
                    *status |= ORC_BIT_BAD_ID;
                if (e < 0 || e >= E || e < e0 || e >= e0 + nb)
                    continue;
                int b = e - e0;
                if (masked_counts[b] >= block_rows) {
                    *status |= ORC_BIT_CAPACITY;
                    continue;
                }
                int64_t row = (int64_t)b * block_rows + masked_counts[b];
                masked_counts[b]++;
                pair_row[q] = (int32_t)row;
                recv_pair[row] = (int32_t)q;
                int32_t slot = token_slot[((int64_t)s * T + t) * P + e / L];
                if (slot < 0 || slot >= cap_send) {
                    *status |= (slot < 0) ? ORC_BIT_INCONSISTENT : ORC_BIT_CAPACITY;
                    memset(recv + row * H, 0, sizeof(uint16_t) * (size_t)H);
                    continue;
                }
                memcpy(recv + row * H, send + ((int64_t)s * cap_send + slot) * H,
                       sizeof(uint16_t) * (size_t)H);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------ stand-in expert -- */

/*
 * Stand-in for the expert kernel (not part of the method; the pages time
 * dispatch and combine without it, [a2a] 8.1): every row of expert e's run is
 * multiplied by the scalar scale[e] and rounded once to bfloat16.  Rows at or
 * beyond min(expert_offsets[E], cap_recv) are not written.
 */
int oracle_expert_scale(const uint16_t *recv, const int32_t *expert_offsets,
                        const float *scale, int E, int H, int64_t cap_recv, uint16_t *y)
{
    for (int e = 0; e < E; e++) {
        for (int64_t r = expert_offsets[e]; r < expert_offsets[e + 1] && r < cap_recv; r++) {
            for (int h = 0; h < H; h++) {
                double v = oracle_bf16_to_double(recv[r * H + h]) * (double)scale[e];
                y[r * H + h] = oracle_bf16_from_double(v);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------ combine, [a2a] 7.1 */

/*
 * [a2a] 1.1 / 7.1: the MoE output of a token is the sum of its experts'
 * outputs, each multiplied by its router weight; the home side adds in (at
 * least) 32-bit floats ([a2a] 7.1, FlashInfer) and the result travels as
 * bf16 ([a2a] 7.2).  Here the sum is taken in double and rounded once:
 *   out[s][t][h] = bf16( sum_{j : pair_row >= 0} w[s][t][j] * y[pair_row[s][t][j]][h] )
 * A token with no valid pair gets +0.
 */
int oracle_combine(const uint16_t *y, const int32_t *pair_row, const float *w,
                   int S, int64_t T, int k, int H, uint16_t *out)
{
    double *acc = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (!acc)
        return -2;
    for (int64_t n = 0; n < (int64_t)S * T; n++) {
        for (int h = 0; h < H; h++)
            acc[h] = 0.0;
#if ORC_MUTANT == 7
        for (int j = 0; j < k - 1; j++) {          /* mutant 7: the last choice is dropped */
#else
        for (int j = 0; j < k; j++) {
#endif
            int32_t r = pair_row[n * k + j];
            if (r < 0)
                continue;
#if ORC_MUTANT == 8
            double wj = 1.0;                        /* mutant 8: weights not applied */
#else
            double wj = (double)w[n * k + j];
#endif
            for (int h = 0; h < H; h++)
                acc[h] += wj * oracle_bf16_to_double(y[(int64_t)r * H + h]);
        }
        for (int h = 0; h < H; h++)
            out[n * H + h] = oracle_bf16_from_double(acc[h]);
    }
    free(acc);
    return 0;
}

/* --------------------------------------------- two-stage combine, [a2a] 7.1 */

/*
 * [a2a] 7.1 splits a token's weighted sum into a sum over the experts that sit
 * on one GPU (stage 1, before the rows travel back; DeepEP's combine and
 * FlashInfer's routed kernel pre-add there) and a sum over the GPUs at home
 * (stage 2, in 32-bit floats for FlashInfer).  Each token then returns as many
 * rows as it sent: one per destination partition.  Rows travel as bf16
 * ([a2a] 7.2), so stage 1 rounds once to bf16.
 *
 * Stage 1, for every (s, t, p) with p in the receiving set and a send slot
 * 0 <= slot < cap_send:
 *   ret[s][slot] = bf16( sum over j with part(ids[s][t][j]) == p and
 *                        pair_row >= 0 of w[s][t][j] * y[pair_row] )   (double sum)
 * Stage 2:
 *   out[s][t] = bf16( sum over p with 0 <= token_slot[s][t][p] < cap_send of
 *                     ret[s][token_slot[s][t][p]] )                  (double sum)
 * A token without slots gets +0.  Slots >= cap_send flag capacity.
 */
int oracle_combine_stage1(const uint16_t *y, const int32_t *pair_row, const float *w,
                          const int32_t *ids, const int32_t *token_slot, int S, int64_t T, int k,
                          int E, int P, int H, int recv_part, int64_t cap_send, uint16_t *ret,
                          uint32_t *status)
{
    if (P < 1 || E % P != 0 || recv_part < -1 || recv_part >= P)
        return -1;
    const int L = E / P;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (!acc)
        return -2;
    for (int s = 0; s < S; s++) {
        for (int64_t t = 0; t < T; t++) {
            const int64_t n = (int64_t)s * T + t;
            for (int p = 0; p < P; p++) {
                if (recv_part >= 0 && p != recv_part)
                    continue;
                int32_t slot = token_slot[n * P + p];
                if (slot < 0)
                    continue;
                if (slot >= cap_send) {
                    *status |= ORC_BIT_CAPACITY;
                    continue;
                }
                for (int h = 0; h < H; h++)
                    acc[h] = 0.0;
                for (int j = 0; j < k; j++) {
                    int32_t e = ids[n * k + j], r = pair_row[n * k + j];
#if ORC_MUTANT == 13
                    if (e < 0 || e >= E || r < 0)   /* mutant 13: other partitions' experts too */
#else
                    if (e < 0 || e >= E || e / L != p || r < 0)
#endif
                        continue;
                    double wj = (double)w[n * k + j];
                    for (int h = 0; h < H; h++)
                        acc[h] += wj * oracle_bf16_to_double(y[(int64_t)r * H + h]);
                }
                for (int h = 0; h < H; h++)
                    ret[((int64_t)s * cap_send + slot) * H + h] = oracle_bf16_from_double(acc[h]);
            }
        }
    }
    free(acc);
    return 0;
}

int oracle_combine_stage2(const uint16_t *ret, const int32_t *token_slot, int S, int64_t T,
                          int P, int H, int64_t cap_send, uint16_t *out, uint32_t *status)
{
    double *acc = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (!acc)
        return -2;
    for (int s = 0; s < S; s++) {
        for (int64_t t = 0; t < T; t++) {
            const int64_t n = (int64_t)s * T + t;
            for (int h = 0; h < H; h++)
                acc[h] = 0.0;
            for (int p = 0; p < P; p++) {
                int32_t slot = token_slot[n * P + p];
                if (slot < 0)
                    continue;
                if (slot >= cap_send) {
                    *status |= ORC_BIT_CAPACITY;
                    continue;
                }
                for (int h = 0; h < H; h++)
                    acc[h] += oracle_bf16_to_double(ret[((int64_t)s * cap_send + slot) * H + h]);
            }
            for (int h = 0; h < H; h++)
                out[n * H + h] = oracle_bf16_from_double(acc[h]);
        }
    }
    free(acc);
    return 0;
}

/* ---------------------------------------- FP8 dispatch rows, [a2a] 7.2 */

/*
 * [a2a] 7.2: expert kernels that quantize their input anyway can take rows
 * already quantized, so a token is converted before it is sent; an FP8 row of
 * DeepSeek-V4.1-Flash is 5,280 bytes: 5,120 one-byte values plus a one-byte
 * scale for every 32 values.  The pages fix the sizes, not the encoding; the
 * reading taken here is the OCP microscaling format MXFP8: E4M3 elements and
 * an E8M0 (power-of-two) scale per block of 32 values.
 *
 * E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities,
 * S.1111.111 is NaN): normal values (1 + m/8) * 2^e for e in [-6, 8] up to
 * 448, subnormals (m/8) * 2^-6.  Conversion: round to nearest, ties to even,
 * on that grid; magnitudes above 448 saturate to 448.
 */
uint8_t oracle_e4m3_from_double(double v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    if (isnan(v))
        return 0x7Fu;
    double a = fabs(v);
    if (a >= 448.0)
        return sign | 0x7Eu;
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);                       /* a in [2^(ex-1), 2^ex) */
    int e = ex - 1;
    if (e < -6)
        e = -6;                          /* subnormal range shares the 2^-9 quantum */
    double q = ldexp(1.0, e - 3);
    double r = nearbyint(a / q) * q;     /* ties to even */
    if (r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    /* encode r */
    int er;
    frexp(r, &er);
    int eu = er - 1;                     /* r in [2^eu, 2^(eu+1)) */
    if (eu < -6) {                       /* subnormal: r = m * 2^-9 */
        int m = (int)nearbyint(r / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int m = (int)nearbyint((r / ldexp(1.0, eu) - 1.0) * 8.0);
    return sign | (uint8_t)(((eu + 7) << 3) | m);
}

double oracle_e4m3_to_double(uint8_t b)
{
    int sign = b >> 7, E = (b >> 3) & 0xF, m = b & 7;
    if (E == 15 && m == 7)
        return NAN;
    double v = (E == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, E - 7);
    return sign ? -v : v;
}

/*
 * One MXFP8 block of 32 bf16 values: shared exponent
 *   X = 2^(floor(log2(max |v|)) - 8)        (8 = exponent of E4M3's largest power of two)
 * clamped to [2^-127, 2^127], stored as the E8M0 byte (exponent + 127); each
 * element is e4m3(v / X).  An all-zero block gets the smallest scale (byte 0).
 */
void oracle_quantize_mxfp8_block(const uint16_t *v, uint8_t *codes, uint8_t *scale)
{
    double amax = 0.0;
    for (int i = 0; i < 32; i++) {
        double a = fabs(oracle_bf16_to_double(v[i]));
        if (a > amax)
            amax = a;
    }
    int se = -127;
    if (amax > 0.0) {
        int ex;
        frexp(amax, &ex);                /* amax in [2^(ex-1), 2^ex) */
#if ORC_MUTANT == 9
        se = (ex - 1) - 7;                        /* mutant 9: scale one binade too high */
#else
        se = (ex - 1) - 8;
#endif
        if (se < -127)
            se = -127;
        if (se > 127)
            se = 127;
    }
    *scale = (uint8_t)(se + 127);
    for (int i = 0; i < 32; i++)
        codes[i] = oracle_e4m3_from_double(ldexp(oracle_bf16_to_double(v[i]), -se));
}

/*
 * Pack with the rows quantized on the way ([a2a] 7.2).  A quantized row is one
 * record of H + H/32 bytes, the page's 5,280 bytes for H = 5,120: the H E4M3
 * codes, then the H/32 E8M0 block scales.  Every (token, partition) slot gets
 * the token's record at send_q[s][slot][0 .. H + H/32); send_src and the
 * capacity rule are those of oracle_dispatch_pack.  H must be a multiple of 32.
 */
int oracle_dispatch_pack_mxfp8(const uint16_t *x, int S, int64_t T, int H, int P,
                               const int32_t *token_slot, int64_t cap_send, uint8_t *send_q,
                               int32_t *send_src, uint32_t *status)
{
    if (H % 32 != 0)
        return -1;
    const int nb = H / 32;
    const int64_t rb = (int64_t)H + nb;
    uint8_t *q = (uint8_t *)malloc((size_t)rb);
    if (!q)
        return -2;
    for (int s = 0; s < S; s++) {
        for (int64_t r = 0; r < cap_send; r++)
            send_src[(int64_t)s * cap_send + r] = -1;
        for (int64_t t = 0; t < T; t++) {
            const uint16_t *row = x + ((int64_t)s * T + t) * H;
            for (int b = 0; b < nb; b++)
                oracle_quantize_mxfp8_block(row + 32 * b, q + 32 * b, q + H + b);
            for (int p = 0; p < P; p++) {
                int32_t slot = token_slot[((int64_t)s * T + t) * P + p];
                if (slot < 0)
                    continue;
                if (slot >= cap_send) {
                    *status |= ORC_BIT_CAPACITY;
                    continue;
                }
                memcpy(send_q + ((int64_t)s * cap_send + slot) * rb, q, (size_t)rb);
                send_src[(int64_t)s * cap_send + slot] = (int32_t)t;
            }
        }
    }
    free(q);
    return 0;
}

/*
 * Stand-in expert on quantized rows: the receiver dequantizes each value of a
 * record (code times 2^(scale byte - 127)) and applies the same per-expert
 * scale as oracle_expert_scale, rounding once to bf16:
 *   y[r][h] = bf16( s_e * e4m3(code[r][h]) * 2^(scale[r][h/32] - 127) )
 * for the rows r of expert e's run.  recv_q rows are H + H/32 bytes.
 */
int oracle_expert_scale_mxfp8(const uint8_t *recv_q, const int32_t *expert_offsets,
                              const float *scale, int E, int H, int64_t cap_recv, uint16_t *y)
{
    if (H % 32 != 0)
        return -1;
    const int64_t rb = (int64_t)H + H / 32;
    for (int e = 0; e < E; e++) {
        for (int64_t r = expert_offsets[e]; r < expert_offsets[e + 1] && r < cap_recv; r++) {
            const uint8_t *rec = recv_q + r * rb;
            for (int h = 0; h < H; h++) {
                double v = oracle_e4m3_to_double(rec[h]) * ldexp(1.0, (int)rec[H + h / 32] - 127);
                y[r * H + h] = oracle_bf16_from_double(v * (double)scale[e]);
            }
        }
    }
    return 0;
}

/* ------------------------------------------ expert placement, [b1g] 6 -- */

/*
 * Share of copy c of an expert with `load` pairs and n copies when the r-th
 * pair goes to copy r mod n: the number of r in [0, load) with r % n == c.
 */
static int64_t oracle_copy_share(int64_t load, int n, int c)
{
    return load > c ? (load - c + n - 1) / n : 0;
}

/*
 * [b1g] 6, "The fix: place experts by load, and copy the hot ones":
 *  1. placement by load -- the heaviest expert first, each on the least
 *     loaded partition (GPU) that still has one of its E/P regular slots;
 *  2. redundant copies -- every partition has R spare slots; repeatedly take
 *     the busiest partition, its busiest expert (largest share), and copy it
 *     to the least loaded partition with a free spare slot; the expert's
 *     pairs are then split evenly over its copies.  A copy is kept only if
 *     it does not make a new busiest partition, i.e. the receiving
 *     partition's new load stays below the old maximum; the first copy that
 *     fails this test ends the loop, as does running out of spare slots.
 * Readings: loads are integer pair counts and the even split is the one the
 * layout implements (share of copy c = #{r < load : r mod n = c}); ties go to
 * the lower expert id and the lower partition; a partition never holds two
 * copies of one expert.
 * Physical slots: partition p owns slots [p*Lp, (p+1)*Lp), Lp = E/P + R,
 * filled in the order experts arrive there (regular slots first, then the
 * copies).  Outputs: copy_offsets[E+1] and copy_slots[] (CSR of each
 * expert's slots, original first, copies in the order they were made),
 * slot_expert[P*Lp] (-1 = empty), part_load[P] (loads after the copies).
 */
int oracle_plan_placement(const int64_t *load, int E, int P, int R, int32_t *copy_offsets,
                          int32_t *copy_slots, int32_t *slot_expert, int64_t *part_load)
{
    if (E < 1 || P < 1 || E % P != 0 || R < 0)
        return -1;
    const int Lb = E / P, Lp = E / P + R;
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    int *ncopy = (int *)calloc((size_t)E, sizeof(int));
    int32_t *slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)E * (size_t)(P + 1));
    int *used = (int *)calloc((size_t)P, sizeof(int));
    if (!order || !ncopy || !slots || !used)
        return -2;
    for (int i = 0; i < P * Lp; i++)
        slot_expert[i] = -1;
    /* 1. heaviest first (selection by scanning: ties to the lower id) */
    char *taken = (char *)calloc((size_t)E, 1);
    for (int i = 0; i < E; i++) {
        int best = -1;
        for (int e = 0; e < E; e++)
            if (!taken[e] && (best < 0 || load[e] > load[best]))
                best = e;
        taken[best] = 1;
        order[i] = best;
    }
    free(taken);
    for (int p = 0; p < P; p++)
        part_load[p] = 0;
    for (int i = 0; i < E; i++) {
        const int e = order[i];
        int q = -1;
        for (int p = 0; p < P; p++)
            if (used[p] < Lb && (q < 0 || part_load[p] < part_load[q]))
                q = p;
        const int s = q * Lp + used[q]++;
        slot_expert[s] = e;
        slots[(size_t)e * (P + 1)] = s;
        ncopy[e] = 1;
        part_load[q] += load[e];
    }
    /* 2. copies */
    for (;;) {
        /* loads from the current copies */
        for (int p = 0; p < P; p++)
            part_load[p] = 0;
        for (int e = 0; e < E; e++)
            for (int c = 0; c < ncopy[e]; c++)
                part_load[slots[(size_t)e * (P + 1) + c] / Lp] += oracle_copy_share(load[e], ncopy[e], c);
        int g = 0;
        for (int p = 1; p < P; p++)
            if (part_load[p] > part_load[g])
                g = p;
        int best = -1;
        int64_t best_share = -1;
        for (int e = 0; e < E; e++)
            for (int c = 0; c < ncopy[e]; c++)
                if (slots[(size_t)e * (P + 1) + c] / Lp == g) {
                    const int64_t sh = oracle_copy_share(load[e], ncopy[e], c);
                    if (sh > best_share) {
                        best_share = sh;
                        best = e;
                    }
                }
        if (best < 0)
            break;
        int tgt = -1;
        for (int p = 0; p < P; p++) {
            if (used[p] >= Lp)
                continue;
            int holds = 0;
            for (int c = 0; c < ncopy[best]; c++)
                if (slots[(size_t)best * (P + 1) + c] / Lp == p)
                    holds = 1;
            if (holds)
                continue;
            if (tgt < 0 || part_load[p] < part_load[tgt])
                tgt = p;
        }
        if (tgt < 0)
            break;
        /* the receiving partition's load with one more copy of `best` */
        const int n1 = ncopy[best] + 1;
        const int64_t new_tgt = part_load[tgt] + oracle_copy_share(load[best], n1, n1 - 1);
#if ORC_MUTANT == 11
        if (!(new_tgt <= part_load[g]))           /* mutant 11: keeps a copy that ties */
#else
        if (!(new_tgt < part_load[g]))
#endif
            break;
        const int s = tgt * Lp + used[tgt]++;
        slot_expert[s] = best;
        slots[(size_t)best * (P + 1) + ncopy[best]] = s;
        ncopy[best] = n1;
    }
    /* final loads and the CSR */
    for (int p = 0; p < P; p++)
        part_load[p] = 0;
    int o = 0;
    for (int e = 0; e < E; e++) {
        copy_offsets[e] = o;
        for (int c = 0; c < ncopy[e]; c++) {
            const int32_t s = slots[(size_t)e * (P + 1) + c];
            copy_slots[o++] = s;
            part_load[s / Lp] += oracle_copy_share(load[e], ncopy[e], c);
        }
    }
    copy_offsets[E] = o;
    free(order);
    free(ncopy);
    free(slots);
    free(used);
    return 0;
}

/*
 * Physical expert of every pair under a placement ([b1g] 6: the expert's
 * pairs are split evenly over its copies): for each source, the r-th pair of
 * logical expert e in (t, j) order goes to copy r mod n_e, i.e.
 *   phys[s][t][j] = copy_slots[copy_offsets[e] + (r mod n_e)].
 * Ids < 0 stay -1 (not routed); ids >= E become E_phys (an invalid physical
 * id, so the layout that follows flags it).
 */
int oracle_map_replicas(const int32_t *ids, int S, int64_t T, int k, int E,
                        const int32_t *copy_offsets, const int32_t *copy_slots, int E_phys,
                        int32_t *phys)
{
    int64_t *seen = (int64_t *)malloc(sizeof(int64_t) * (size_t)E);
    if (!seen)
        return -2;
    for (int s = 0; s < S; s++) {
        for (int e = 0; e < E; e++)
            seen[e] = 0;
        for (int64_t t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                const int64_t i = ((int64_t)s * T + t) * k + j;
                const int32_t e = ids[i];
                if (e < 0) {
                    phys[i] = -1;
                } else if (e >= E) {
                    phys[i] = E_phys;
                } else {
                    const int n = copy_offsets[e + 1] - copy_offsets[e];
#if ORC_MUTANT == 12
                    phys[i] = copy_slots[copy_offsets[e] + (int)(t % n)];   /* mutant 12 */
#else
                    phys[i] = copy_slots[copy_offsets[e] + (int)(seen[e] % n)];
#endif
                    seen[e]++;
                }
            }
    }
    free(seen);
    return 0;
}

/* --------------------------------------- routed payload, [a2a] 6.1, 7.1 -- */

/*
 * [a2a] 6.1: next to the hidden state the sender writes the token's expert
 * ids and weights (payloads = hidden state, top-k ids, top-k weights), so the
 * receiver need not group anything.  Rows go where oracle_dispatch_pack puts
 * them; every written row also gets the token's k ids and weights:
 *   send_ids[s][slot][j] = ids[s][t][j],  send_w[s][slot][j] = w[s][t][j]
 * Rows no slot names are empty and carry the invalid id -1 and weight 0
 * ([a2a] 6.3: empty slots are marked with an invalid expert id).
 */
int oracle_dispatch_pack_routed(const uint16_t *x, const int32_t *ids, const float *w, int S,
                                int64_t T, int H, int k, int P, const int32_t *token_slot,
                                int64_t cap_send, uint16_t *send, int32_t *send_src,
                                int32_t *send_ids, float *send_w, uint32_t *status)
{
    int rc = oracle_dispatch_pack(x, S, T, H, P, token_slot, cap_send, send, send_src, status);
    if (rc != 0)
        return rc;
    for (int s = 0; s < S; s++)
        for (int64_t r = 0; r < cap_send; r++) {
            const int64_t row = (int64_t)s * cap_send + r;
            const int32_t t = send_src[row];
            for (int j = 0; j < k; j++) {
                send_ids[row * k + j] = t < 0 ? -1 : ids[((int64_t)s * T + t) * k + j];
                send_w[row * k + j] = t < 0 ? 0.0f : w[((int64_t)s * T + t) * k + j];
            }
        }
    return 0;
}

/*
 * [a2a] 6.1 / 7.1: the routed expert kernel takes the rows in arrival order,
 * reads each row's ids, runs the experts of its own GPU and already produces
 * the weighted sum over them -- stage 1 of the combine -- in that GPU's
 * workspace.  With the stand-in expert (y = bf16(x * scale[e]); identity
 * when scale is NULL), for every row r of partition p's region of source s,
 * r in [part_offsets[s][p], part_offsets[s][p+1]), p in the receiving set:
 *   ret[s][r] = bf16( sum over ascending j with send_ids[s][r][j] in p
 *                     of send_w[s][r][j] * y_j ),   y_j = bf16(send[s][r] * scale[e_j])
 * summed in double.  Other rows of ret are not written; ids >= E are skipped
 * and flagged.
 */
int oracle_routed_expert_stage1(const uint16_t *send, const int32_t *send_ids, const float *send_w,
                                const int32_t *part_offsets, int S, int64_t cap_send, int k,
                                int E, int P, int H, int recv_part, const float *scale,
                                uint16_t *ret, uint32_t *status)
{
    if (P < 1 || E % P != 0 || recv_part < -1 || recv_part >= P)
        return -1;
    const int L = E / P;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (!acc)
        return -2;
    for (int s = 0; s < S; s++)
        for (int p = 0; p < P; p++) {
            if (recv_part >= 0 && p != recv_part)
                continue;
            const int32_t *po = part_offsets + (int64_t)s * (P + 1);
            for (int64_t r = po[p]; r < po[p + 1] && r < cap_send; r++) {
                const int64_t row = (int64_t)s * cap_send + r;
                for (int h = 0; h < H; h++)
                    acc[h] = 0.0;
                for (int j = 0; j < k; j++) {
                    const int32_t e = send_ids[row * k + j];
                    if (e >= E)
                        *status |= ORC_BIT_BAD_ID;
                    if (e < 0 || e >= E || e / L != p)
                        continue;
                    const double wj = (double)send_w[row * k + j];
                    for (int h = 0; h < H; h++) {
                        double v = oracle_bf16_to_double(send[row * H + h]);
                        if (scale)
                            v = oracle_bf16_to_double(oracle_bf16_from_double(v * (double)scale[e]));
                        acc[h] += wj * v;
                    }
                }
                for (int h = 0; h < H; h++)
                    ret[row * H + h] = oracle_bf16_from_double(acc[h]);
            }
        }
    free(acc);
    return 0;
}

/* --------------------------------------------- NVFP4 rows, [a2a] 7.2 -- */

/*
 * E2M1 (4 bits: sign, 2 exponent bits with bias 1, 1 mantissa bit): the
 * magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6.  Encoding rounds to the
 * nearest magnitude, ties to the even code (mantissa bit 0), magnitudes
 * above 6 become 6, and the sign is kept (also for zero).
 */
static const double oracle_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_to_double(uint8_t c)
{
    const double m = oracle_e2m1_mag[c & 7];
    return (c & 8) ? -m : m;
}

uint8_t oracle_e2m1_from_double(double v)
{
    const uint8_t sign = signbit(v) ? 8u : 0u;
    double a = fabs(v);
    if (a >= 6.0)
        return sign | 7u;
    int best = 0;
    for (int c = 1; c < 8; c++) {
        const double d = fabs(oracle_e2m1_mag[c] - a), db = fabs(oracle_e2m1_mag[best] - a);
#if ORC_MUTANT == 10
        if (d < db || (d == db && (c & 1) == 1))  /* mutant 10: ties to the odd code */
#else
        if (d < db || (d == db && (c & 1) == 0))
#endif
            best = c;
    }
    return sign | (uint8_t)best;
}

/*
 * One NVFP4 block of 16 bf16 values ([a2a] 7.2: a one-byte scale for every 16
 * values).  Reading (the page gives only the size): NVIDIA's NVFP4 -- E2M1
 * values, an E4M3 scale per 16 values and one fp32 scale g for the whole
 * tensor (given by the caller; it is not part of a row):
 *   s = e4m3( fp32(amax / fp32(6 g)) ),   code_i = e2m1( fp32(v_i / fp32(s g)) )
 * and all codes 0 when s is 0.  Every product and quotient is taken in fp32:
 * they decide integer codes, and fp32 is the precision of the GPU kernel.
 * Codes are packed two per byte, element 2i in the low nibble.
 */
void oracle_quantize_nvfp4_block(const uint16_t *v, float g, uint8_t *codes, uint8_t *scale)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; i++) {
        const float a = (float)fabs(oracle_bf16_to_double(v[i]));
        if (a > amax)
            amax = a;
    }
#if ORC_MUTANT == 14
    const float d = 6.0f;                         /* mutant 14: the tensor scale is ignored */
#else
    const float d = 6.0f * g;
#endif
    const float t = amax / d;
    *scale = oracle_e4m3_from_double((double)t);
    const float sg = (float)oracle_e4m3_to_double(*scale) * g;
    for (int i = 0; i < 8; i++) {
        uint8_t c[2];
        for (int h = 0; h < 2; h++) {
            const float x = (float)oracle_bf16_to_double(v[2 * i + h]);
            c[h] = sg == 0.0f ? 0u : oracle_e2m1_from_double((double)(x / sg));
        }
        codes[i] = (uint8_t)(c[0] | (c[1] << 4));
    }
}

/*
 * Pack with NVFP4 records ([a2a] 7.2): a record is H/2 bytes of codes
 * followed by H/16 bytes of block scales -- 2,880 bytes for H = 5,120, the
 * page's NVFP4 row.  Placement, send_src and capacity as oracle_dispatch_pack.
 * H must be a multiple of 16.
 */
int oracle_dispatch_pack_nvfp4(const uint16_t *x, int S, int64_t T, int H, int P, float g,
                               const int32_t *token_slot, int64_t cap_send, uint8_t *send_q,
                               int32_t *send_src, uint32_t *status)
{
    if (H % 16 != 0)
        return -1;
    const int nb = H / 16;
    const int64_t rb = (int64_t)H / 2 + nb;
    uint8_t *q = (uint8_t *)malloc((size_t)rb);
    if (!q)
        return -2;
    for (int s = 0; s < S; s++) {
        for (int64_t r = 0; r < cap_send; r++)
            send_src[(int64_t)s * cap_send + r] = -1;
        for (int64_t t = 0; t < T; t++) {
            const uint16_t *row = x + ((int64_t)s * T + t) * H;
            for (int b = 0; b < nb; b++)
                oracle_quantize_nvfp4_block(row + 16 * b, g, q + 8 * b, q + H / 2 + b);
            for (int p = 0; p < P; p++) {
                int32_t slot = token_slot[((int64_t)s * T + t) * P + p];
                if (slot < 0)
                    continue;
                if (slot >= cap_send) {
                    *status |= ORC_BIT_CAPACITY;
                    continue;
                }
                memcpy(send_q + ((int64_t)s * cap_send + slot) * rb, q, (size_t)rb);
                send_src[(int64_t)s * cap_send + slot] = (int32_t)t;
            }
        }
    }
    free(q);
    return 0;
}

/*
 * Stand-in expert on NVFP4 records (as oracle_expert_scale_mxfp8):
 *   y[r][h] = bf16( s_e * e2m1(code[r][h]) * e4m3(scale[r][h/16]) * g )
 */
int oracle_expert_scale_nvfp4(const uint8_t *recv_q, const int32_t *expert_offsets,
                              const float *scale, int E, int H, float g, int64_t cap_recv,
                              uint16_t *y)
{
    if (H % 16 != 0)
        return -1;
    const int64_t rb = (int64_t)H / 2 + H / 16;
    for (int e = 0; e < E; e++) {
        for (int64_t r = expert_offsets[e]; r < expert_offsets[e + 1] && r < cap_recv; r++) {
            const uint8_t *rec = recv_q + r * rb;
            for (int h = 0; h < H; h++) {
                const uint8_t c = (uint8_t)((rec[h / 2] >> (4 * (h & 1))) & 0xF);
                const double v = oracle_e2m1_to_double(c) * oracle_e4m3_to_double(rec[H / 2 + h / 16]) *
                                  (double)g;
                y[r * H + h] = oracle_bf16_from_double(v * (double)scale[e]);
            }
        }
    }
    return 0;
}
