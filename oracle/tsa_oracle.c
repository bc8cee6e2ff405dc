/*
 * tsa_oracle.c -- CPU oracle for topology-scheduled sparse attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline / reference leg may load this library.  It
 * shares no code, header, table or constant with the CUDA library under
 * topology_scheduled_gb300/csrc; the two are compared only through their
 * outputs on the same seeded inputs.
 *
 * Everything here is plain, slow and written to be checked by eye against the
 * pages it follows:
 *
 *   [PR] "Add topology-derived sparse attention kernel" (triton-lang/kernels#22),
 *        Summary: a forward-only scheduled-attention kernel over causal CSR block
 *        schedules; schedules built from sink blocks, local-window blocks and a
 *        0D-persistence salience over key-block centroids; [seq, dim] and
 *        [batch, heads, seq, dim] inputs sharing one CSR.
 *   [PORT] the same PR's GitHub mirror page, the port note ("A port of the
 *        Triton kernel merged as triton-lang/kernels#22"): the kernel is checked
 *        against dense masked attention; the block loop keeps a running maximum
 *        and denominator and rescales by exp(m_prev - m_new); salience is the
 *        elder rule, exactly one block scores zero, and on a size tie the
 *        absorbed component depends on index order.
 *   [SCHED] the same mirror page, the world-model commit's schedule.py bullet:
 *        the block salience is reproduced from MST edges instead of all pairs.
 *   [GATE] the same mirror page, the later commit about a forget gate's exact
 *        zeros feeding the merged CSR kernel: segment boundaries as a CSR
 *        schedule, with block counts at S 4096 and block 64 of 2,080 (dense),
 *        288 (fixed 512-token segments), 160 (fixed 256-token segments) and
 *        478 (random boundaries at 0.0024 flags per token, mean of 200 draws).
 *
 * Where the pages leave a step open, the reading taken is stated at the step.
 * All floating point is IEEE binary64; compile with -ffp-contract=off so that
 * no multiply-add is fused except where fma() is written out.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* ------------------------------------------------------------------------ */
/* Element decoding (exact widening of the 16-bit inputs to binary64).       */
/* ------------------------------------------------------------------------ */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(0x400 | m), e - 25); /* (1024+m) * 2^(e-15-10) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double bf16_bits_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133); /* subnormal: m * 2^(1-127-7) */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(0x80 | m), e - 134); /* (128+m) * 2^(e-127-7) */
    return sign ? -v : v;
}

static double g_table[2][65536];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;

static void build_tables(void)
{
    for (int i = 0; i < 65536; ++i) {
        g_table[ORACLE_F16][i] = half_bits_to_double((uint16_t)i);
        g_table[ORACLE_BF16][i] = bf16_bits_to_double((uint16_t)i);
    }
}

static const double *decode_table(int dtype)
{
    pthread_once(&g_table_once, build_tables);
    return g_table[dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_F16];
}

/* Decode n 16-bit values of the given dtype to binary64. */
int oracle_decode(const uint16_t *x, int64_t n, int dtype, double *out)
{
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return 1;
    const double *t = decode_table(dtype);
    for (int64_t i = 0; i < n; ++i) out[i] = t[x[i]];
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dense causal CSR  ([PR] Summary "dense causal CSR layout"; Local          */
/* benchmark: the dense CSR path visits every causal block).                 */
/* ------------------------------------------------------------------------ */

/* Row i holds every key block 0..i, so row_ptr[i] = i(i+1)/2. */
int oracle_dense_causal_csr(int64_t nb, int32_t *row_ptr, int32_t *col_idx)
{
    int64_t e = 0;
    row_ptr[0] = 0;
    for (int64_t i = 0; i < nb; ++i) {
        for (int64_t j = 0; j <= i; ++j) col_idx[e++] = (int32_t)j;
        row_ptr[i + 1] = (int32_t)e;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Key-block centroids ([PR] Summary: salience "over key-block centroids").  */
/* ------------------------------------------------------------------------ */

/*
 * K is [L][S][D] (L = batch*heads lanes, one shared schedule).  Reading: the
 * point cloud is the mean key of each block, averaged over the lanes too:
 *
 *   C[b][d] = ( sum_{l=0}^{L-1} ( sum_{t=0}^{n_b-1} K[l][b*block+t][d] ) ) / (n_b*L)
 *
 * with both sums taken in ascending order, one binary64 accumulator each, and
 * one correctly rounded division at the end.  There are nb = ceil(S / block)
 * blocks; n_b = block except for a partial last block, which holds the
 * S - (nb-1)*block tokens that exist (the pages do not say; the mean over the
 * tokens a block holds is the plainest reading).
 */
int oracle_centroids(const uint16_t *K, int dtype, int64_t L, int64_t S, int64_t D,
                     int64_t block, double *C)
{
    if (block <= 0 || S <= 0) return 1;
    const double *tab = decode_table(dtype);
    int64_t nb = (S + block - 1) / block;
    double *part = (double *)malloc(sizeof(double) * (size_t)D);
    double *total = (double *)malloc(sizeof(double) * (size_t)D);
    if (!part || !total) { free(part); free(total); return 2; }
    for (int64_t b = 0; b < nb; ++b) {
        const int64_t n_b = (b + 1) * block <= S ? block : S - b * block;
        const double denom = (double)(n_b * L);
        for (int64_t d = 0; d < D; ++d) total[d] = 0.0;
        for (int64_t l = 0; l < L; ++l) {
            for (int64_t d = 0; d < D; ++d) part[d] = 0.0;
            for (int64_t t = 0; t < n_b; ++t) {
                const uint16_t *row = K + ((l * S) + b * block + t) * D;
                for (int64_t d = 0; d < D; ++d) part[d] = part[d] + tab[row[d]];
            }
            for (int64_t d = 0; d < D; ++d) total[d] = total[d] + part[d];
        }
        for (int64_t d = 0; d < D; ++d) C[b * D + d] = total[d] / denom;
    }
    free(part);
    free(total);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Merge distances.                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Reading: the distance is Euclidean; every comparison uses its square,
 *   d2(u,v) = sum_{d=0}^{D-1} (C[u][d] - C[v][d])^2,
 * in binary64 with one fixed order of summation (the pages fix none):
 *   P_j = the terms d = j, j + 32, j + 64, ... (d < D) accumulated in ascending
 *         d from +0 with one fused multiply-add each, for j = 0 .. 31;
 *   then halving: P_j = P_j + P_{j+w} for j < w, w = 16, 8, 4, 2, 1; d2 = P_0.
 * (An empty P_j is +0, and adding +0 changes no sum.)
 */
static double pair_d2(const double *C, int64_t D, int64_t u, int64_t v)
{
    double part[32];
    for (int j = 0; j < 32; ++j) {
        double acc = 0.0;
        for (int64_t d = j; d < D; d += 32) {
            double delta = C[u * D + d] - C[v * D + d];
            acc = fma(delta, delta, acc);
        }
        part[j] = acc;
    }
    for (int w = 16; w >= 1; w /= 2)
        for (int j = 0; j < w; ++j) part[j] = part[j] + part[j + w];
    return part[0];
}

int oracle_pairwise_d2(const double *C, int64_t nb, int64_t D, double *D2)
{
    for (int64_t u = 0; u < nb; ++u)
        for (int64_t v = 0; v < nb; ++v) D2[u * nb + v] = (u == v) ? 0.0 : pair_d2(C, D, u, v);
    return 0;
}

typedef struct {
    double d2;
    int32_t u, v; /* u before v in the block order below */
} edge_t;

/*
 * Block order used to break ties.
 *
 * Index rule ([PORT]: on a size tie the absorbed component "depends on index
 * order"): blocks compare by index.
 *
 * Content rule (the fix the port note asks for: a tie-break on centroid
 * content rather than index).  Reading: blocks compare by their centroid
 * vectors, coordinate by coordinate in ascending d, each coordinate in IEEE
 * 754 totalOrder (for finite values: numeric order, with -0 before +0); only
 * blocks with bit-identical centroids fall back to index order.  The oracle
 * requires finite centroids.
 */
static const double *g_order_C; /* qsort has no context argument */
static int64_t g_order_D;
static int g_order_content;

static int coord_cmp(double x, double y)
{
    if (x < y) return -1;
    if (x > y) return 1;
    if (signbit(x) != signbit(y)) return signbit(x) ? -1 : 1;
    return 0;
}

static int block_cmp(int32_t u, int32_t v)
{
    if (g_order_content) {
        for (int64_t d = 0; d < g_order_D; ++d) {
            int c = coord_cmp(g_order_C[u * g_order_D + d], g_order_C[v * g_order_D + d]);
            if (c != 0) return c;
        }
    }
    return u < v ? -1 : (u > v ? 1 : 0);
}

/* Reading: edges are ordered strictly by (d2, earlier endpoint, later endpoint). */
static int edge_cmp(const void *pa, const void *pb)
{
    const edge_t *a = (const edge_t *)pa, *b = (const edge_t *)pb;
    if (a->d2 < b->d2) return -1;
    if (a->d2 > b->d2) return 1;
    int c = block_cmp(a->u, b->u);
    if (c != 0) return c;
    return block_cmp(a->v, b->v);
}

static int32_t dsu_find(int32_t *parent, int32_t x)
{
    int32_t r = x;
    while (parent[r] != r) r = parent[r];
    while (parent[x] != r) { /* path compression never changes a root */
        int32_t nx = parent[x];
        parent[x] = r;
        x = nx;
    }
    return r;
}

/*
 * 0D persistence salience by the elder rule ([PORT]; [SCHED]).
 *
 * Kruskal over all nb(nb-1)/2 centroid pairs in the strict edge order.  Each
 * edge that joins two components merges them: the component with fewer blocks
 * is absorbed; on a size tie the component whose representative (root) comes
 * later in the block order is absorbed.  The absorbed component's root -- the
 * one block of that component never written before -- receives the edge's d2
 * as its salience; the survivor's root stays the root of the union.  The block
 * that is never absorbed keeps salience 0.
 *
 * Outputs: sal_sq[nb] (squared merge distance per block) and, optionally, the
 * nb-1 accepted (MST) edges in the order they were accepted.
 */
static int salience_kruskal(const double *C, int64_t nb, int64_t D, int content, double *sal_sq,
                            int32_t *mst_u, int32_t *mst_v, double *mst_d2)
{
    if (nb <= 0) return 1;
    g_order_C = C;
    g_order_D = D;
    g_order_content = content;
    int64_t ne = nb * (nb - 1) / 2;
    edge_t *edges = (edge_t *)malloc(sizeof(edge_t) * (size_t)(ne > 0 ? ne : 1));
    int32_t *parent = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb);
    int64_t *size = (int64_t *)malloc(sizeof(int64_t) * (size_t)nb);
    if (!edges || !parent || !size) { free(edges); free(parent); free(size); return 2; }
    int64_t e = 0;
    for (int64_t u = 0; u < nb; ++u)
        for (int64_t v = u + 1; v < nb; ++v) {
            edges[e].d2 = pair_d2(C, D, u, v);
            int before = block_cmp((int32_t)u, (int32_t)v) < 0;
            edges[e].u = (int32_t)(before ? u : v);
            edges[e].v = (int32_t)(before ? v : u);
            ++e;
        }
    qsort(edges, (size_t)ne, sizeof(edge_t), edge_cmp);
    for (int64_t i = 0; i < nb; ++i) {
        parent[i] = (int32_t)i;
        size[i] = 1;
        sal_sq[i] = 0.0;
    }
    int64_t accepted = 0;
    for (int64_t k = 0; k < ne && accepted < nb - 1; ++k) {
        int32_t ra = dsu_find(parent, edges[k].u);
        int32_t rb = dsu_find(parent, edges[k].v);
        if (ra == rb) continue;
        int32_t absorbed, survivor;
        if (size[ra] < size[rb]) { absorbed = ra; survivor = rb; }
        else if (size[rb] < size[ra]) { absorbed = rb; survivor = ra; }
        else if (block_cmp(ra, rb) > 0) { absorbed = ra; survivor = rb; }
        else { absorbed = rb; survivor = ra; }
        sal_sq[absorbed] = edges[k].d2;
        parent[absorbed] = survivor;
        size[survivor] += size[absorbed];
        if (mst_u) mst_u[accepted] = edges[k].u;
        if (mst_v) mst_v[accepted] = edges[k].v;
        if (mst_d2) mst_d2[accepted] = edges[k].d2;
        ++accepted;
    }
    free(edges);
    free(parent);
    free(size);
    return 0;
}

/* Index rule: size ties and equal distances are broken by block index. */
int oracle_salience(const double *C, int64_t nb, int64_t D, double *sal_sq,
                    int32_t *mst_u, int32_t *mst_v, double *mst_d2)
{
    return salience_kruskal(C, nb, D, 0, sal_sq, mst_u, mst_v, mst_d2);
}

/* Content rule: the same ties are broken by centroid content (block order above). */
int oracle_salience_content(const double *C, int64_t nb, int64_t D, double *sal_sq,
                            int32_t *mst_u, int32_t *mst_v, double *mst_d2)
{
    return salience_kruskal(C, nb, D, 1, sal_sq, mst_u, mst_v, mst_d2);
}

/* ------------------------------------------------------------------------ */
/* Topology CSR ([PR] Summary: sink blocks, local-window blocks and top-k    */
/* blocks by salience; one row per query block).                             */
/* ------------------------------------------------------------------------ */

static const double *g_sort_sal; /* qsort has no context argument */

/* Order of the top-k selection: larger salience first, lower index on ties. */
static int topk_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    double sa = g_sort_sal[a], sb = g_sort_sal[b];
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return a < b ? -1 : (a > b ? 1 : 0);
}

/*
 * Row i (query block i) holds, sorted ascending without repeats:
 *   sink blocks   { j : j < sink, j <= i }
 *   local window  { j : max(0, i - local_radius) <= j <= i }
 *   top-k         the topk blocks j <= i of largest salience (ties: lower j)
 * Reading: the top-k candidates are all causal blocks, including blocks that
 * are already sink or local, so a row may add fewer than topk new blocks.
 * Returns 3 if col_cap is too small.
 */
int oracle_topology_csr(const double *sal_sq, int64_t nb, int64_t sink, int64_t local_radius,
                        int64_t topk, int32_t *row_ptr, int32_t *col_idx, int64_t col_cap)
{
    if (nb <= 0 || sink < 0 || local_radius < 0 || topk < 0) return 1;
    unsigned char *mark = (unsigned char *)malloc((size_t)nb);
    int32_t *cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb);
    if (!mark || !cand) { free(mark); free(cand); return 2; }
    int64_t e = 0;
    row_ptr[0] = 0;
    g_sort_sal = sal_sq;
    for (int64_t i = 0; i < nb; ++i) {
        memset(mark, 0, (size_t)nb);
        for (int64_t j = 0; j < sink && j <= i; ++j) mark[j] = 1;
        for (int64_t j = (i - local_radius > 0 ? i - local_radius : 0); j <= i; ++j) mark[j] = 1;
        for (int64_t j = 0; j <= i; ++j) cand[j] = (int32_t)j;
        qsort(cand, (size_t)(i + 1), sizeof(int32_t), topk_cmp);
        for (int64_t t = 0; t < topk && t <= i; ++t) mark[cand[t]] = 1;
        for (int64_t j = 0; j <= i; ++j) {
            if (!mark[j]) continue;
            if (e >= col_cap) { free(mark); free(cand); return 3; }
            col_idx[e++] = (int32_t)j;
        }
        row_ptr[i + 1] = (int32_t)e;
    }
    free(mark);
    free(cand);
    return 0;
}

/* The whole builder: centroids -> salience -> topology CSR.  content selects
 * the tie rule of the salience (0: index, 1: centroid content). */
int oracle_build_schedule_tie(const uint16_t *K, int dtype, int64_t L, int64_t S, int64_t D,
                              int64_t block, int64_t sink, int64_t local_radius, int64_t topk,
                              int content, int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                              double *sal_sq)
{
    if (block <= 0 || S <= 0) return 1;
    int64_t nb = (S + block - 1) / block;  /* a partial last block is a block too */
    double *C = (double *)malloc(sizeof(double) * (size_t)(nb * D));
    if (!C) return 2;
    int rc = oracle_centroids(K, dtype, L, S, D, block, C);
    if (rc == 0) rc = salience_kruskal(C, nb, D, content, sal_sq, NULL, NULL, NULL);
    if (rc == 0) rc = oracle_topology_csr(sal_sq, nb, sink, local_radius, topk, row_ptr, col_idx, col_cap);
    free(C);
    return rc;
}

int oracle_build_schedule(const uint16_t *K, int dtype, int64_t L, int64_t S, int64_t D,
                          int64_t block, int64_t sink, int64_t local_radius, int64_t topk,
                          int32_t *row_ptr, int32_t *col_idx, int64_t col_cap, double *sal_sq)
{
    return oracle_build_schedule_tie(K, dtype, L, S, D, block, sink, local_radius, topk, 0,
                                     row_ptr, col_idx, col_cap, sal_sq);
}

/* ------------------------------------------------------------------------ */
/* Segment schedules ([GATE]: segment boundaries run through the CSR kernel). */
/* ------------------------------------------------------------------------ */

/*
 * Reading: `starts` lists the tokens that begin a new segment, strictly
 * ascending in [0, S); token 0 always begins one.  Query token q may attend to
 * key token k iff k <= q and no segment begins in (k, q], i.e. s(q) <= k <= q
 * with s(q) the last segment start <= q.  Row i of the block schedule holds
 * every key block that contains a key allowed to some query token of block i.
 * When every start is a multiple of `block` the block schedule allows exactly
 * the token pairs of the segment mask; otherwise it is the smallest block
 * schedule that covers it.  Returns 3 if col_cap is too small.
 */
int oracle_segment_csr(int64_t S, int64_t block, const int64_t *starts, int64_t n_starts,
                       int32_t *row_ptr, int32_t *col_idx, int64_t col_cap)
{
    if (S <= 0 || block <= 0 || S % block != 0 || n_starts < 0) return 1;
    for (int64_t k = 0; k < n_starts; ++k) {
        if (starts[k] < 0 || starts[k] >= S) return 1;
        if (k > 0 && starts[k] <= starts[k - 1]) return 1;
    }
    int64_t nb = S / block;
    unsigned char *mark = (unsigned char *)calloc((size_t)(nb * nb), 1);
    if (!mark) return 2;
    int64_t next = 0, seg = 0;
    for (int64_t q = 0; q < S; ++q) {
        while (next < n_starts && starts[next] <= q) seg = starts[next++];
        for (int64_t k = seg; k <= q; ++k) mark[(q / block) * nb + k / block] = 1;
    }
    int64_t e = 0;
    row_ptr[0] = 0;
    for (int64_t i = 0; i < nb; ++i) {
        for (int64_t j = 0; j < nb; ++j) {
            if (!mark[i * nb + j]) continue;
            if (e >= col_cap) { free(mark); return 3; }
            col_idx[e++] = (int32_t)j;
        }
        row_ptr[i + 1] = (int32_t)e;
    }
    free(mark);
    return 0;
}

/* Fixed segments of seg_tokens tokens: starts at seg_tokens, 2 seg_tokens, ... */
int oracle_fixed_segment_csr(int64_t S, int64_t block, int64_t seg_tokens, int32_t *row_ptr,
                             int32_t *col_idx, int64_t col_cap)
{
    if (seg_tokens <= 0 || S <= 0) return 1;
    int64_t n = (S - 1) / seg_tokens;
    int64_t *starts = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!starts) return 2;
    for (int64_t k = 0; k < n; ++k) starts[k] = (k + 1) * seg_tokens;
    int rc = oracle_segment_csr(S, block, starts, n, row_ptr, col_idx, col_cap);
    free(starts);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Masked attention ([PR] Summary; [PORT]: checked against dense masked      */
/* attention).                                                               */
/* ------------------------------------------------------------------------ */

/*
 * For lane l and query token q in query block i = q / block, the allowed keys
 * are A(q) = { k : k / block is in row i of the CSR, k <= q } (the token-level
 * causal rule applies in every visited block; it only bites on the diagonal).
 *
 *   O[l][q][:] = sum_{k in A(q)} softmax_k(scale * <Q[l][q], K[l][k]>) V[l][k][:]
 *
 * computed in binary64 as max-subtracted two-pass softmax.  A query with no
 * allowed key gets O = 0 (reading).
 */
typedef struct {
    const uint16_t *Q, *K, *V;
    const double *tab;
    int64_t S, D, block;
    double scale;
    const int32_t *row_ptr, *col_idx;
    const int64_t *lane, *tok;
    double *out;
    double *lse; /* optional: log-sum-exp of the scaled scores per row */
    int online;
    int64_t begin, end;
} attn_job_t;

static void attention_one_twopass(const attn_job_t *J, int64_t l, int64_t q, double *o,
                                  double *s, int64_t *keys, double *lse)
{
    const int64_t D = J->D, S = J->S, block = J->block;
    const double *tab = J->tab;
    const uint16_t *qrow = J->Q + (l * S + q) * D;
    int64_t i = q / block, n = 0;
    for (int32_t e = J->row_ptr[i]; e < J->row_ptr[i + 1]; ++e) {
        int64_t j = J->col_idx[e];
        for (int64_t k = j * block; k < (j + 1) * block; ++k)
            if (k <= q) keys[n++] = k;
    }
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    if (lse) *lse = -INFINITY;
    if (n == 0) return;
    double m = -INFINITY;
    for (int64_t a = 0; a < n; ++a) {
        const uint16_t *krow = J->K + (l * S + keys[a]) * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += tab[qrow[d]] * tab[krow[d]];
        s[a] = J->scale * dot;
        if (s[a] > m) m = s[a];
    }
    double den = 0.0;
    for (int64_t a = 0; a < n; ++a) {
        s[a] = exp(s[a] - m);
        den += s[a];
    }
    if (lse) *lse = m + log(den);
    for (int64_t a = 0; a < n; ++a) {
        const uint16_t *vrow = J->V + (l * S + keys[a]) * D;
        double w = s[a] / den;
        for (int64_t d = 0; d < D; ++d) o[d] += w * tab[vrow[d]];
    }
}

/*
 * The same quantity by the pages' single pass ([PORT]): walk the row's key
 * blocks in order keeping a running maximum m and denominator den; when a
 * block raises the maximum, rescale den and the accumulator by exp(m_prev - m_new).
 */
static void attention_one_online(const attn_job_t *J, int64_t l, int64_t q, double *o,
                                 double *s)
{
    const int64_t D = J->D, S = J->S, block = J->block;
    const double *tab = J->tab;
    const uint16_t *qrow = J->Q + (l * S + q) * D;
    int64_t i = q / block;
    double m = -INFINITY, den = 0.0;
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    for (int32_t e = J->row_ptr[i]; e < J->row_ptr[i + 1]; ++e) {
        int64_t j = J->col_idx[e];
        int64_t n = 0;
        double bmax = -INFINITY;
        for (int64_t k = j * block; k < (j + 1) * block && k <= q; ++k) {
            const uint16_t *krow = J->K + (l * S + k) * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += tab[qrow[d]] * tab[krow[d]];
            s[n] = J->scale * dot;
            if (s[n] > bmax) bmax = s[n];
            ++n;
        }
        if (n == 0) continue;
        double m_new = bmax > m ? bmax : m;
        double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        den *= alpha;
        for (int64_t d = 0; d < D; ++d) o[d] *= alpha;
        for (int64_t a = 0; a < n; ++a) {
            double p = exp(s[a] - m_new);
            den += p;
            const uint16_t *vrow = J->V + (l * S + j * block + a) * D;
            for (int64_t d = 0; d < D; ++d) o[d] += p * tab[vrow[d]];
        }
        m = m_new;
    }
    if (den > 0.0)
        for (int64_t d = 0; d < D; ++d) o[d] /= den;
}

static void *attention_worker(void *arg)
{
    attn_job_t *J = (attn_job_t *)arg;
    int64_t S = J->S;
    double *s = (double *)malloc(sizeof(double) * (size_t)S);
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)S);
    if (s && keys) {
        for (int64_t r = J->begin; r < J->end; ++r) {
            double *o = J->out + r * J->D;
            if (J->online)
                attention_one_online(J, J->lane[r], J->tok[r], o, s);
            else
                attention_one_twopass(J, J->lane[r], J->tok[r], o, s, keys,
                                      J->lse ? J->lse + r : NULL);
        }
    }
    free(s);
    free(keys);
    return NULL;
}

/*
 * Evaluate O for n (lane, token) pairs.  Q, K, V are [L][S][D] 16-bit values of
 * the given dtype; out is [n][D] binary64.  Rows are independent, so they are
 * split into nthreads contiguous chunks; the result does not depend on nthreads.
 * lse (optional, two-pass form only) receives log(sum_k exp(scale <Q_q, K_k>))
 * over the allowed keys, -inf for a row without keys.
 */
int oracle_attention_lse(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype,
                         int64_t L, int64_t S, int64_t D, int64_t block, double scale,
                         const int32_t *row_ptr, const int32_t *col_idx, int64_t n,
                         const int64_t *lane, const int64_t *tok, double *out, double *lse,
                         int online, int nthreads);

int oracle_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype,
                     int64_t L, int64_t S, int64_t D, int64_t block, double scale,
                     const int32_t *row_ptr, const int32_t *col_idx, int64_t n,
                     const int64_t *lane, const int64_t *tok, double *out, int online,
                     int nthreads)
{
    return oracle_attention_lse(Q, K, V, dtype, L, S, D, block, scale, row_ptr, col_idx, n, lane,
                                tok, out, NULL, online, nthreads);
}

int oracle_attention_lse(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int dtype,
                         int64_t L, int64_t S, int64_t D, int64_t block, double scale,
                         const int32_t *row_ptr, const int32_t *col_idx, int64_t n,
                         const int64_t *lane, const int64_t *tok, double *out, double *lse,
                         int online, int nthreads)
{
    if (lse && online) return 1;
    /* S need not be a multiple of block: keys k < S only (k <= q < S) */
    if (block <= 0 || S <= 0 || L <= 0 || D <= 0) return 1;
    for (int64_t r = 0; r < n; ++r)
        if (lane[r] < 0 || lane[r] >= L || tok[r] < 0 || tok[r] >= S) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    attn_job_t base;
    base.Q = Q; base.K = K; base.V = V;
    base.tab = decode_table(dtype);
    base.S = S; base.D = D; base.block = block; base.scale = scale;
    base.row_ptr = row_ptr; base.col_idx = col_idx;
    base.lane = lane; base.tok = tok; base.out = out; base.lse = lse; base.online = online;
    attn_job_t jobs[256];
    pthread_t th[256];
    int started[256];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].begin = t * chunk < n ? t * chunk : n;
        jobs[t].end = (t + 1) * chunk < n ? (t + 1) * chunk : n;
        started[t] = 0;
        if (t > 0 && jobs[t].begin < jobs[t].end)
            started[t] = pthread_create(&th[t], NULL, attention_worker, &jobs[t]) == 0;
    }
    attention_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        else if (jobs[t].begin < jobs[t].end) attention_worker(&jobs[t]);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward pass of the masked attention above (the step after the forward   */
/* kernel; the mirror page's segment-boundary record notes that the merged   */
/* kernel has none).  It is the chain rule of the forward definition, with   */
/* the same allowed sets A(q).                                               */
/* ------------------------------------------------------------------------ */

/*
 * For lane l, with p_qk = softmax_k(scale <Q_q, K_k>) over k in A(q) and
 * O_q = sum_k p_qk V_k, the gradients of a loss with dL/dO = dO are
 *
 *   dV_k  = sum_{q : k in A(q)} p_qk dO_q
 *   dP_qk = <dO_q, V_k>,   Delta_q = <dO_q, O_q> = sum_k p_qk dP_qk
 *   dS_qk = p_qk (dP_qk - Delta_q)
 *   dQ_q  = scale sum_k dS_qk K_k,   dK_k = scale sum_{q : k in A(q)} dS_qk Q_q
 *
 * all in binary64 from the exactly widened 16-bit inputs.  A query without
 * allowed keys contributes nothing.  Lanes are independent; each lane runs in
 * one thread, queries in ascending order, so the result does not depend on
 * nthreads.
 */
typedef struct {
    const uint16_t *Q, *K, *V, *dO;
    const double *tab;
    int64_t S, D, block;
    double scale;
    const int32_t *row_ptr, *col_idx;
    double *dQ, *dK, *dV;
    int64_t lane_begin, lane_end;
} bwd_job_t;

static void backward_lane(const bwd_job_t *J, int64_t l, double *p, int64_t *keys, double *o)
{
    const int64_t S = J->S, D = J->D, block = J->block;
    const double *tab = J->tab;
    double *dQ = J->dQ + l * S * D, *dK = J->dK + l * S * D, *dV = J->dV + l * S * D;
    for (int64_t x = 0; x < S * D; ++x) dQ[x] = dK[x] = dV[x] = 0.0;
    for (int64_t q = 0; q < S; ++q) {
        const uint16_t *qrow = J->Q + (l * S + q) * D;
        const uint16_t *dorow = J->dO + (l * S + q) * D;
        int64_t i = q / block, n = 0;
        for (int32_t e = J->row_ptr[i]; e < J->row_ptr[i + 1]; ++e) {
            int64_t j = J->col_idx[e];
            for (int64_t k = j * block; k < (j + 1) * block; ++k)
                if (k <= q) keys[n++] = k;
        }
        if (n == 0) continue;
        double m = -INFINITY;
        for (int64_t a = 0; a < n; ++a) {
            const uint16_t *krow = J->K + (l * S + keys[a]) * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += tab[qrow[d]] * tab[krow[d]];
            p[a] = J->scale * dot;
            if (p[a] > m) m = p[a];
        }
        double den = 0.0;
        for (int64_t a = 0; a < n; ++a) {
            p[a] = exp(p[a] - m);
            den += p[a];
        }
        for (int64_t a = 0; a < n; ++a) p[a] /= den;
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t a = 0; a < n; ++a) {
            const uint16_t *vrow = J->V + (l * S + keys[a]) * D;
            for (int64_t d = 0; d < D; ++d) o[d] += p[a] * tab[vrow[d]];
        }
        double delta = 0.0;
        for (int64_t d = 0; d < D; ++d) delta += tab[dorow[d]] * o[d];
        for (int64_t a = 0; a < n; ++a) {
            const int64_t k = keys[a];
            const uint16_t *krow = J->K + (l * S + k) * D;
            const uint16_t *vrow = J->V + (l * S + k) * D;
            double dp = 0.0;
            for (int64_t d = 0; d < D; ++d) dp += tab[dorow[d]] * tab[vrow[d]];
            const double ds = p[a] * (dp - delta);
            for (int64_t d = 0; d < D; ++d) {
                dQ[q * D + d] += J->scale * ds * tab[krow[d]];
                dK[k * D + d] += J->scale * ds * tab[qrow[d]];
                dV[k * D + d] += p[a] * tab[dorow[d]];
            }
        }
    }
}

static void *backward_worker(void *arg)
{
    bwd_job_t *J = (bwd_job_t *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->S);
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)J->S);
    double *o = (double *)malloc(sizeof(double) * (size_t)J->D);
    if (p && keys && o)
        for (int64_t l = J->lane_begin; l < J->lane_end; ++l) backward_lane(J, l, p, keys, o);
    free(p);
    free(keys);
    free(o);
    return NULL;
}

/* dQ, dK, dV are [L][S][D] binary64 outputs; dO is [L][S][D] 16-bit like Q. */
int oracle_attention_backward(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                              const uint16_t *dO, int dtype, int64_t L, int64_t S, int64_t D,
                              int64_t block, double scale, const int32_t *row_ptr,
                              const int32_t *col_idx, double *dQ, double *dK, double *dV,
                              int nthreads)
{
    /* S need not be a multiple of block: row i = q / block of a query q < S only reaches
     * keys k <= q < S, so a partial last block needs nothing else. */
    if (block <= 0 || S <= 0 || L <= 0 || D <= 0) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > L) nthreads = (int)L;
    bwd_job_t base;
    base.Q = Q; base.K = K; base.V = V; base.dO = dO;
    base.tab = decode_table(dtype);
    base.S = S; base.D = D; base.block = block; base.scale = scale;
    base.row_ptr = row_ptr; base.col_idx = col_idx;
    base.dQ = dQ; base.dK = dK; base.dV = dV;
    bwd_job_t jobs[256];
    pthread_t th[256];
    int started[256];
    int64_t chunk = (L + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].lane_begin = t * chunk < L ? t * chunk : L;
        jobs[t].lane_end = (t + 1) * chunk < L ? (t + 1) * chunk : L;
        started[t] = 0;
        if (t > 0 && jobs[t].lane_begin < jobs[t].lane_end)
            started[t] = pthread_create(&th[t], NULL, backward_worker, &jobs[t]) == 0;
    }
    backward_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        else if (jobs[t].lane_begin < jobs[t].lane_end) backward_worker(&jobs[t]);
    }
    return 0;
}
