/*
 * spec_oracle.c -- CPU oracle for the tree-verification step of lossless greedy
 * speculative decoding on a hybrid Gated-DeltaNet / attention target.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or constant with the CUDA path, and the CUDA
 * path never calls it.
 *
 * Source of every definition below: the paper digest "SpecPilot: Autonomous
 * Algorithm Discovery and Systems Optimization for Speculative Decoding"
 * (rainbus.top), cited by its section names:
 *   [SD]    prerequisites / speculative decoding   -- greedy acceptance rule,
 *           tau in [1, m+1], one bonus token;
 *   [LAT]   prerequisites / parallel drafter        -- per-position top-16
 *           candidates with scores form the lattice;
 *   [TREE]  prerequisites / draft-tree verification -- every node sees only its
 *           ancestors; accept the longest root path matching the target argmax
 *           plus a bonus; nodes added greedily by path log-prob up to N;
 *   [GDN]   prerequisites / hybrid recurrent target -- the gated delta rule
 *           h_t = a_t (I - b_t k_t k_t^T) h_{t-1} + b_t k_t v_t^T,
 *           o_t = h_t^T q_t;
 *   [NOV]   technical novelty + Figure 6 ("Best-first tree on a hybrid
 *           target") -- best-first tree with edges scored log p(child|parent);
 *           node states recomputed along root paths, no per-node snapshots;
 *   [BATCH] technical novelty, batching -- a node budget shared by the batch
 *           (the target GEMM's 192-node plateau) and the number of draft
 *           positions chosen per request (16/12/8);
 *   [MARK]  prerequisites / parallel drafter -- DSpark's Markov head conditions
 *           each position on the previous token:
 *           l_s(y) = bases(y) + <W1[x_{s-1}], W2[y]>.
 * and the speculative-decoding tutorial (mlqm.cn, news/131545):
 *   [RS]    section 2.3, the acceptance rule at temperature > 0: a draft token
 *           x with draft probability q(x) and target probability p(x) is kept
 *           with probability min(1, p(x)/q(x)); otherwise a token is drawn from
 *           max(0, p - q), renormalised, and the output follows p exactly.
 *
 * Precision: every floating-point result is accumulated in double from the
 * exact values of the (bf16 or fp32) inputs.  The one exception is the tree
 * key, a root-path sum of fp32 edge scores, which the readings below fix as an
 * fp32 sum; it is computed in float on purpose.
 *
 * Readings of points the page leaves open (listed again in the design notes):
 *   R1  N counts draft nodes; the root (the pending bonus token) is one more
 *       verified row, so a tree has T = 1 + min(N, sum_d K^d) rows.
 *   R2  The best-first key is the fp32 sum of edge scores along the root path.
 *   R3  Ties: score desc, depth asc, parent index asc, rank asc.  Argmax takes
 *       the lowest index; a repeated child token takes the lowest node index.
 *   R7  q has no 1/sqrt(d_k) scale; alpha arrives directly; qk-head of v-head
 *       j is j / (Hv / Hk).
 *   R8  Attention scale 1/sqrt(D); q-head h reads kv-head h / (Hq / Hkv).
 *   R9  Commit: the state after the last accepted node becomes the committed
 *       state; the tree K/V rows of the accepted path are appended.
 *   R14 Markov edges: a child y of a parent with token x at lattice position d
 *       has l = base_d(y) + <W1[x], W2[y]> (fp32: the dot product as a chain
 *       of fused multiply-adds in index order, then one add) and edge score
 *       l - LSE, the log-sum-exp over the position's K candidates under the
 *       same parent (fp32: M = max l, Z = sum in index order of exp32(l - M),
 *       LSE = M + log32(Z)).  exp32 and log32 are the fp32 functions defined
 *       below, so the scores are fixed to the bit.  Children of a parent are
 *       ranked by (edge desc, candidate index asc).
 *   R15 Stochastic acceptance: the tree's drafts are fixed tokens (q is a point
 *       mass), so at a node with children x_1..x_k the [RS] rule keeps x_i with
 *       probability p'(x_i), p' being p with the earlier children removed and
 *       renormalised, and otherwise draws the bonus from p without all of
 *       them.  That is the same law as drawing y ~ p at the node and moving to
 *       the child whose token is y (y is the bonus when there is none).  The
 *       draw from p = softmax(l / theta) is a two-level Gumbel-max over chunks
 *       of 4096 tokens (orc_sample_row), with Gumbel noise from Philox4x32-10
 *       keyed by the 64-bit seed and counted by (index, row, request,
 *       kv_len).  The walk is then C6 with the draws in place of the argmax.
 *   R12 Shared budget: request b drafts from its first m_b lattice positions;
 *       the batch's draft nodes are inserted best-first over the frontiers of
 *       all requests together (key: score desc, then request index asc, then
 *       the R3 order), each request holding at most N drafts, until the budget
 *       is spent or every frontier is empty.
 *
 * Layouts (all row-major, outermost first):
 *   lattice     tok int32 [B][m][K], score f32 [B][m][K]
 *   tree        node_* [B][T], anc uint64 [B][T][2] (bit a of node n set iff
 *               node a is n or an ancestor of n), n_nodes [B]
 *   gdn         h0 double [B][Hv][dk][dv]; q,k [B][T][Hk][dk]; v [B][T][Hv][dv];
 *               alpha, beta f32 [B][T][Hv]; o double [B][T][Hv][dv]
 *   attention   q [B][T][Hq][D]; k_tree, v_tree [B][T][Hkv][D];
 *               k_cache, v_cache [B][Lmax][Hkv][D]; kv_len int32 [B];
 *               o double [B][T][Hq][D]
 *   logits      [rows][V]
 * Element type of q/k/v/logits/caches: io_bf16 = 1 -> raw bf16 bits (uint16),
 * io_bf16 = 0 -> float.
 *
 * Return value of every entry point: 0 on success, a negative number when the
 * input breaks a precondition (documented per function).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_ANC_WORDS 2   /* trees hold at most 128 rows */
#define ORC_LN2 0.69314718055994530941723212145818   /* ln 2 */
#define ORC_SQRT2 1.4142135623730950488016887242097  /* sqrt 2 */
#define ORC_MAX_ROWS 128

/* ---- element access ---------------------------------------------------- */

/* Exact widening of one stored element to double. */
static double orc_elem(const void *base, size_t idx, int io_bf16)
{
    if (io_bf16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

/* ---- C1/C2: lattice canonicalisation and best-first tree [LAT][TREE][NOV] */

/* One frontier entry: the child with lattice rank `rank` of inserted node
 * `parent`. */
typedef struct {
    int parent;
    int rank;
    int depth;
    float score;
} orc_cand;

/* Strict total order of R3: a precedes b. */
static int orc_cand_before(const orc_cand *a, const orc_cand *b)
{
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    if (a->parent != b->parent) return a->parent < b->parent;
    return a->rank < b->rank;
}

/*
 * orc_tree_build: best-first draft tree over a lattice [TREE][NOV].
 *
 * Per request: candidates of each position are stable-sorted by score
 * (descending, input index ascending); a candidate's rank is its sorted
 * position.  Node 0 is the root (token root_tok, depth 0, score 0, parent -1).
 * The frontier holds every child of every inserted node of depth < m; the
 * child of rank r of node p has depth d_p + 1, token and score taken from the
 * rank-r candidate of lattice position d_p (0-based, i.e. depth d_p + 1), and
 * key fl32(score_p + edge score).  Until N drafts are inserted or the frontier
 * is empty, the frontier entry first in the R3 order becomes the next node.
 *
 * Rows n >= n_nodes[b] are padding: tok/parent/depth/rank = -1, score 0,
 * anc 0.  Requires 1 <= m, 1 <= K, 0 <= N, N + 1 <= 128 (returns -1
 * otherwise) and distinct tokens within a position (returns -2 otherwise).
 */
int orc_tree_build(int B, int m, int K, int N,
                   const int32_t *lat_tok, const float *lat_score,
                   const int32_t *root_tok,
                   int32_t *node_tok, int32_t *node_parent, int32_t *node_depth,
                   int32_t *node_rank, float *node_score, uint64_t *node_anc,
                   int32_t *n_nodes)
{
    if (B < 0 || m < 1 || K < 1 || N < 0 || N + 1 > ORC_MAX_ROWS) return -1;
    const int T = N + 1;
    int *order = (int *)malloc(sizeof(int) * (size_t)m * (size_t)K);
    orc_cand *front = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(T * K + K));
    if (!order || !front) { free(order); free(front); return -3; }
    int rc = 0;

    for (int b = 0; b < B && rc == 0; ++b) {
        const int32_t *tok = lat_tok + (size_t)b * m * K;
        const float *sc = lat_score + (size_t)b * m * K;

        /* canonical order per position: insertion sort is stable */
        for (int s = 0; s < m; ++s) {
            int *o = order + (size_t)s * K;
            for (int i = 0; i < K; ++i) {
                int j = i;
                while (j > 0 && sc[s * K + i] > sc[s * K + o[j - 1]]) {
                    o[j] = o[j - 1];
                    --j;
                }
                o[j] = i;
            }
            for (int i = 0; i < K; ++i)
                for (int j = i + 1; j < K; ++j)
                    if (tok[s * K + i] == tok[s * K + j]) rc = -2;
        }
        if (rc) break;

        int32_t *ntok = node_tok + (size_t)b * T, *npar = node_parent + (size_t)b * T;
        int32_t *ndep = node_depth + (size_t)b * T, *nrank = node_rank + (size_t)b * T;
        float *nsc = node_score + (size_t)b * T;
        uint64_t *nanc = node_anc + (size_t)b * T * ORC_ANC_WORDS;
        for (int n = 0; n < T; ++n) {
            ntok[n] = -1; npar[n] = -1; ndep[n] = -1; nrank[n] = -1; nsc[n] = 0.0f;
            for (int w = 0; w < ORC_ANC_WORDS; ++w) nanc[n * ORC_ANC_WORDS + w] = 0;
        }

        ntok[0] = root_tok[b]; npar[0] = -1; ndep[0] = 0; nrank[0] = -1; nsc[0] = 0.0f;
        nanc[0] = 1ull;
        int count = 1, nfront = 0;
        for (int r = 0; r < K; ++r) {            /* children of the root */
            orc_cand c = { 0, r, 1, nsc[0] + sc[0 * K + order[r]] };
            front[nfront++] = c;
        }
        while (count < T && nfront > 0) {
            int best = 0;
            for (int i = 1; i < nfront; ++i)
                if (orc_cand_before(&front[i], &front[best])) best = i;
            orc_cand c = front[best];
            front[best] = front[--nfront];

            const int n = count++;
            const int s = c.depth - 1;           /* lattice position of depth d */
            ntok[n] = tok[s * K + order[s * K + c.rank]];
            npar[n] = c.parent;
            ndep[n] = c.depth;
            nrank[n] = c.rank;
            nsc[n] = c.score;
            for (int w = 0; w < ORC_ANC_WORDS; ++w)
                nanc[n * ORC_ANC_WORDS + w] = nanc[c.parent * ORC_ANC_WORDS + w];
            nanc[n * ORC_ANC_WORDS + n / 64] |= 1ull << (n % 64);

            if (c.depth < m) {
                for (int r = 0; r < K; ++r) {
                    float e = sc[c.depth * K + order[c.depth * K + r]];
                    orc_cand ch = { n, r, c.depth + 1, nsc[n] + e };
                    front[nfront++] = ch;
                }
            }
        }
        n_nodes[b] = count;
    }
    free(order);
    free(front);
    return rc;
}

/*
 * orc_tree_build_ragged: best-first draft trees of a batch that shares a node
 * budget [BATCH][TREE][NOV], reading R12.
 *
 * m_req[b] in [1, m] lattice positions per request; budget = total draft
 * nodes over the batch (budget < 0: no shared budget, every request up to N).
 * The frontier is one list over all requests; the entry first in the order
 * (score desc, request asc, depth asc, parent asc, rank asc) becomes the next
 * node of its request, unless that request already holds N drafts, in which
 * case the entry is dropped.  Outputs and padding rows as orc_tree_build.
 * Returns -1 on bad sizes or m_req, -2 on a repeated token, -3 on allocation.
 */
int orc_tree_build_ragged(int B, int m, int K, int N, const int32_t *m_req, int budget,
                          const int32_t *lat_tok, const float *lat_score,
                          const int32_t *root_tok,
                          int32_t *node_tok, int32_t *node_parent, int32_t *node_depth,
                          int32_t *node_rank, float *node_score, uint64_t *node_anc,
                          int32_t *n_nodes)
{
    if (B < 0 || m < 1 || K < 1 || N < 0 || N + 1 > ORC_MAX_ROWS) return -1;
    for (int b = 0; b < B; ++b)
        if (m_req[b] < 1 || m_req[b] > m) return -1;
    const int T = N + 1;
    int *order = (int *)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1) * m * K);
    orc_cand *front = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(B > 0 ? B : 1) * (T * K + K));
    int *front_req = (int *)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1) * (T * K + K));
    if (!order || !front || !front_req) { free(order); free(front); free(front_req); return -3; }
    int rc = 0, nfront = 0;

    for (int b = 0; b < B && rc == 0; ++b) {
        const int32_t *tok = lat_tok + (size_t)b * m * K;
        const float *sc = lat_score + (size_t)b * m * K;
        for (int s = 0; s < m; ++s) {            /* canonical order per position */
            int *o = order + ((size_t)b * m + s) * K;
            for (int i = 0; i < K; ++i) {
                int j = i;
                while (j > 0 && sc[s * K + i] > sc[s * K + o[j - 1]]) {
                    o[j] = o[j - 1];
                    --j;
                }
                o[j] = i;
            }
            for (int i = 0; i < K; ++i)
                for (int j = i + 1; j < K; ++j)
                    if (tok[s * K + i] == tok[s * K + j]) rc = -2;
        }
        int32_t *ntok = node_tok + (size_t)b * T, *npar = node_parent + (size_t)b * T;
        int32_t *ndep = node_depth + (size_t)b * T, *nrank = node_rank + (size_t)b * T;
        float *nsc = node_score + (size_t)b * T;
        uint64_t *nanc = node_anc + (size_t)b * T * ORC_ANC_WORDS;
        for (int n = 0; n < T; ++n) {
            ntok[n] = -1; npar[n] = -1; ndep[n] = -1; nrank[n] = -1; nsc[n] = 0.0f;
            for (int w = 0; w < ORC_ANC_WORDS; ++w) nanc[n * ORC_ANC_WORDS + w] = 0;
        }
        ntok[0] = root_tok[b]; ndep[0] = 0; nanc[0] = 1ull;
        n_nodes[b] = 1;
        for (int r = 0; r < K; ++r) {            /* children of the root: 0 + edge (R2) */
            orc_cand c = { 0, r, 1, nsc[0] + sc[order[(size_t)b * m * K + r]] };
            front_req[nfront] = b;
            front[nfront++] = c;
        }
    }
    int used = 0;
    while (rc == 0 && nfront > 0 && (budget < 0 || used < budget)) {
        int best = 0;
        for (int i = 1; i < nfront; ++i) {
            const orc_cand *a = &front[i], *c = &front[best];
            int before;
            if (a->score != c->score) before = a->score > c->score;
            else if (front_req[i] != front_req[best]) before = front_req[i] < front_req[best];
            else before = orc_cand_before(a, c);
            if (before) best = i;
        }
        const orc_cand c = front[best];
        const int b = front_req[best];
        front[best] = front[nfront - 1];
        front_req[best] = front_req[nfront - 1];
        --nfront;
        if (n_nodes[b] >= T) continue;           /* request full: drop the entry */

        const int32_t *tok = lat_tok + (size_t)b * m * K;
        const float *sc = lat_score + (size_t)b * m * K;
        const int *ord = order + (size_t)b * m * K;
        int32_t *ntok = node_tok + (size_t)b * T, *npar = node_parent + (size_t)b * T;
        int32_t *ndep = node_depth + (size_t)b * T, *nrank = node_rank + (size_t)b * T;
        float *nsc = node_score + (size_t)b * T;
        uint64_t *nanc = node_anc + (size_t)b * T * ORC_ANC_WORDS;
        const int n = n_nodes[b]++;
        ++used;
        const int s = c.depth - 1;
        ntok[n] = tok[s * K + ord[s * K + c.rank]];
        npar[n] = c.parent;
        ndep[n] = c.depth;
        nrank[n] = c.rank;
        nsc[n] = c.score;
        for (int w = 0; w < ORC_ANC_WORDS; ++w)
            nanc[n * ORC_ANC_WORDS + w] = nanc[c.parent * ORC_ANC_WORDS + w];
        nanc[n * ORC_ANC_WORDS + n / 64] |= 1ull << (n % 64);
        if (c.depth < m_req[b]) {
            for (int r = 0; r < K; ++r) {
                orc_cand ch = { n, r, c.depth + 1, nsc[n] + sc[c.depth * K + ord[c.depth * K + r]] };
                front_req[nfront] = b;
                front[nfront++] = ch;
            }
        }
    }
    free(order);
    free(front);
    free(front_req);
    return rc;
}

/* ---- R14: Markov-head edge scores [MARK][NOV] ----------------------------
 *
 * exp32(x), x <= 0: Cody-Waite reduction x = n ln2 + r with ln2 split into a
 * 9-bit head 355/512 and the fp32 rounding of the rest, n = rint(x / ln2) (the
 * product with fp32(1/ln2) rounded to fp32), e^r by its Taylor polynomial to
 * degree 7 (Horner, fused multiply-adds, coefficients fp32(1/k!)), times 2^n;
 * x < -86 gives 0.
 * log32(z), z >= 1: z = f 2^e with f in [1, 2), halved (e + 1) when f > fp32
 * (sqrt 2); log f = 2 atanh(s), s = (f - 1) / (f + 1), by the odd series to
 * s^13 (Horner in s^2, coefficients fp32(1/k)); log z = e ln2 + log f.
 */
static float orc_exp32(float x)
{
    if (x < -86.0f) return 0.0f;
    const float inv_ln2 = (float)(1.0 / ORC_LN2);
    const float ln2_hi = 355.0f / 512.0f;
    const float ln2_lo = (float)(ORC_LN2 - 355.0 / 512.0);
    const float n = rintf(x * inv_ln2);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    float p = (float)(1.0 / 5040.0);
    p = fmaf(p, r, (float)(1.0 / 720.0));
    p = fmaf(p, r, (float)(1.0 / 120.0));
    p = fmaf(p, r, (float)(1.0 / 24.0));
    p = fmaf(p, r, (float)(1.0 / 6.0));
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    const uint32_t bits = (uint32_t)((int)n + 127) << 23;   /* 2^n, n in [-125, 0] */
    float scale;
    memcpy(&scale, &bits, sizeof scale);
    return p * scale;
}

static float orc_log32(float z)
{
    uint32_t bits;
    memcpy(&bits, &z, sizeof bits);
    int e = (int)((bits >> 23) & 0xffu) - 127;
    const uint32_t fb = (bits & 0x7fffffu) | 0x3f800000u;
    float f;
    memcpy(&f, &fb, sizeof f);
    if (f > (float)ORC_SQRT2) { f = f * 0.5f; e += 1; }
    const float s = (f - 1.0f) / (f + 1.0f);
    const float s2 = s * s;
    float t = (float)(1.0 / 13.0);
    t = fmaf(t, s2, (float)(1.0 / 11.0));
    t = fmaf(t, s2, (float)(1.0 / 9.0));
    t = fmaf(t, s2, (float)(1.0 / 7.0));
    t = fmaf(t, s2, (float)(1.0 / 5.0));
    t = fmaf(t, s2, (float)(1.0 / 3.0));
    t = fmaf(t, s2, 1.0f);
    const float lf = (2.0f * s) * t;
    const float ef = (float)e;
    return fmaf(ef, 355.0f / 512.0f, fmaf(ef, (float)(ORC_LN2 - 355.0 / 512.0), lf));
}

/* Edge scores of the K candidates (tokens tok[K], bases base[K]) under a
 * parent with token x (R14); W1, W2 f32 [V][R]. */
static void orc_markov_edges_row(int K, int R, int x, const int32_t *tok, const float *base,
                                 const float *W1, const float *W2, float *edge)
{
    float M = -INFINITY;
    for (int i = 0; i < K; ++i) {
        float dot = 0.0f;
        for (int k = 0; k < R; ++k)
            dot = fmaf(W1[(size_t)x * R + k], W2[(size_t)tok[i] * R + k], dot);
        edge[i] = base[i] + dot;
        if (edge[i] > M) M = edge[i];
    }
    float Z = 0.0f;
    for (int i = 0; i < K; ++i) Z = Z + orc_exp32(edge[i] - M);
    const float lse = M + orc_log32(Z);
    for (int i = 0; i < K; ++i) edge[i] = edge[i] - lse;
}

/* Exported for the pins: exp32/log32 of n values, and one edge row. */
int orc_exp32_log32(int n, const float *x, float *ex, const float *z, float *lz)
{
    for (int i = 0; i < n; ++i) { ex[i] = orc_exp32(x[i]); lz[i] = orc_log32(z[i]); }
    return 0;
}

int orc_markov_edges(int K, int R, int x, const int32_t *tok, const float *base,
                     const float *W1, const float *W2, float *edge)
{
    if (K < 1 || R < 0) return -1;
    orc_markov_edges_row(K, R, x, tok, base, W1, W2, edge);
    return 0;
}

/*
 * orc_tree_build_markov: best-first draft tree whose edge scores depend on the
 * parent's token [MARK][TREE][NOV], reading R14.
 *
 * lat_tok int32 [B][m][K], lat_base f32 [B][m][K] (the drafter's base logits),
 * W1, W2 f32 [V][R].  When node n (token x, depth d < m) is inserted, its
 * children are the K candidates of lattice position d with edge scores
 * R14(x, d), ranked by (edge desc, index asc); the child of rank r has key
 * fl32(score_n + edge).  Frontier order, padding rows and return codes as
 * orc_tree_build.
 */
int orc_tree_build_markov(int B, int m, int K, int N, int R, const int32_t *lat_tok,
                          const float *lat_base, const float *W1, const float *W2,
                          const int32_t *root_tok,
                          int32_t *node_tok, int32_t *node_parent, int32_t *node_depth,
                          int32_t *node_rank, float *node_score, uint64_t *node_anc,
                          int32_t *n_nodes)
{
    if (B < 0 || m < 1 || K < 1 || N < 0 || N + 1 > ORC_MAX_ROWS || R < 0) return -1;
    const int T = N + 1;
    float *cedge = (float *)malloc(sizeof(float) * (size_t)T * K);   /* [T][K] by rank */
    int *cidx = (int *)malloc(sizeof(int) * (size_t)T * K);          /* [T][K] by rank */
    float *row = (float *)malloc(sizeof(float) * (size_t)K);
    orc_cand *front = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(T * K + K));
    if (!cedge || !cidx || !row || !front) {
        free(cedge); free(cidx); free(row); free(front);
        return -3;
    }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        const int32_t *tok = lat_tok + (size_t)b * m * K;
        const float *base = lat_base + (size_t)b * m * K;
        for (int s = 0; s < m; ++s)
            for (int i = 0; i < K; ++i)
                for (int j = i + 1; j < K; ++j)
                    if (tok[s * K + i] == tok[s * K + j]) rc = -2;
        if (rc) break;
        int32_t *ntok = node_tok + (size_t)b * T, *npar = node_parent + (size_t)b * T;
        int32_t *ndep = node_depth + (size_t)b * T, *nrank = node_rank + (size_t)b * T;
        float *nsc = node_score + (size_t)b * T;
        uint64_t *nanc = node_anc + (size_t)b * T * ORC_ANC_WORDS;
        for (int n = 0; n < T; ++n) {
            ntok[n] = -1; npar[n] = -1; ndep[n] = -1; nrank[n] = -1; nsc[n] = 0.0f;
            for (int w = 0; w < ORC_ANC_WORDS; ++w) nanc[n * ORC_ANC_WORDS + w] = 0;
        }
        ntok[0] = root_tok[b]; ndep[0] = 0; nanc[0] = 1ull;
        int count = 1, nfront = 0;
        /* the children of node n, ranked: edges R14(token of n, its depth) */
        #define ORC_OFFER(n_)                                                              \
            do {                                                                           \
                const int d_ = ndep[n_];                                                   \
                orc_markov_edges_row(K, R, ntok[n_], tok + d_ * K, base + d_ * K, W1, W2, row); \
                int *o_ = cidx + (size_t)(n_) * K;                                         \
                for (int i_ = 0; i_ < K; ++i_) {                                           \
                    int j_ = i_;                                                           \
                    while (j_ > 0 && row[i_] > row[o_[j_ - 1]]) { o_[j_] = o_[j_ - 1]; --j_; } \
                    o_[j_] = i_;                                                           \
                }                                                                          \
                for (int r_ = 0; r_ < K; ++r_) {                                           \
                    cedge[(size_t)(n_) * K + r_] = row[o_[r_]];                            \
                    orc_cand c_ = { n_, r_, d_ + 1, nsc[n_] + row[o_[r_]] };               \
                    front[nfront++] = c_;                                                  \
                }                                                                          \
            } while (0)
        ORC_OFFER(0);
        while (count < T && nfront > 0) {
            int best = 0;
            for (int i = 1; i < nfront; ++i)
                if (orc_cand_before(&front[i], &front[best])) best = i;
            orc_cand c = front[best];
            front[best] = front[--nfront];
            const int n = count++;
            const int s = c.depth - 1;
            ntok[n] = tok[s * K + cidx[(size_t)c.parent * K + c.rank]];
            npar[n] = c.parent;
            ndep[n] = c.depth;
            nrank[n] = c.rank;
            nsc[n] = c.score;
            for (int w = 0; w < ORC_ANC_WORDS; ++w)
                nanc[n * ORC_ANC_WORDS + w] = nanc[c.parent * ORC_ANC_WORDS + w];
            nanc[n * ORC_ANC_WORDS + n / 64] |= 1ull << (n % 64);
            if (c.depth < m) ORC_OFFER(n);
        }
        #undef ORC_OFFER
        n_nodes[b] = count;
    }
    free(cedge); free(cidx); free(row); free(front);
    return rc;
}

/* Root path of node n (root first); returns its length (depth + 1). */
static int orc_root_path(const int32_t *parent, int n, int *path)
{
    int len = 0, x = n;
    while (x >= 0) { path[len++] = x; x = parent[x]; }
    for (int i = 0; i < len / 2; ++i) {
        int t = path[i]; path[i] = path[len - 1 - i]; path[len - 1 - i] = t;
    }
    return len;
}

/* ---- C3: Gated DeltaNet along root paths [GDN][NOV] --------------------- */

/*
 * One gated-delta step on a dk x dv state held in double:
 *   u = h^T k;  h <- alpha (h - beta k u^T) + beta k v^T,
 * which is h <- alpha (I - beta k k^T) h + beta k v^T written out.
 */
static void orc_gdn_step(double *h, int dk, int dv, const double *k,
                         const double *v, double alpha, double beta, double *u)
{
    for (int c = 0; c < dv; ++c) {
        double acc = 0.0;
        for (int r = 0; r < dk; ++r) acc += h[(size_t)r * dv + c] * k[r];
        u[c] = acc;
    }
    for (int r = 0; r < dk; ++r)
        for (int c = 0; c < dv; ++c) {
            double x = h[(size_t)r * dv + c];
            h[(size_t)r * dv + c] = alpha * (x - beta * k[r] * u[c]) + beta * k[r] * v[c];
        }
}

/*
 * orc_gdn_tree: output of every tree node of one GDN layer.
 *
 * For node n, v-head j (qk-head i = j / (Hv/Hk)) and root path
 * 0 = p_0, ..., p_l = n: start from h = h0[b][j], apply the gated-delta step
 * of every node on the path in root-to-leaf order (the root's own row
 * included), then o[b][n][j] = h^T q_n.  This is the sequential linear-chain
 * decode of the node's root path; nothing is shared between nodes.
 * Padding rows (n >= n_nodes[b]) get o = 0.  Requires Hv % Hk == 0.
 */
int orc_gdn_tree(int B, int T, int Hk, int Hv, int dk, int dv,
                 const int32_t *node_parent, const int32_t *n_nodes,
                 const double *h0, const void *q, const void *k, const void *v,
                 int io_bf16, const float *alpha, const float *beta, double *o)
{
    if (Hk <= 0 || Hv % Hk != 0 || T > ORC_MAX_ROWS) return -1;
    const int grp = Hv / Hk;
    double *h = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
    double *qq = (double *)malloc(sizeof(double) * (size_t)dk);
    double *vv = (double *)malloc(sizeof(double) * (size_t)dv);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    int path[ORC_MAX_ROWS];
    if (!h || !kk || !qq || !vv || !u) { free(h); free(kk); free(qq); free(vv); free(u); return -3; }

    for (int b = 0; b < B; ++b) {
        const int32_t *par = node_parent + (size_t)b * T;
        for (int n = 0; n < T; ++n) {
            for (int j = 0; j < Hv; ++j) {
                double *out = o + (((size_t)b * T + n) * Hv + j) * dv;
                if (n >= n_nodes[b]) { for (int c = 0; c < dv; ++c) out[c] = 0.0; continue; }
                const int i = j / grp;
                memcpy(h, h0 + ((size_t)b * Hv + j) * dk * dv, sizeof(double) * (size_t)dk * dv);
                const int len = orc_root_path(par, n, path);
                for (int s = 0; s < len; ++s) {
                    const int t = path[s];
                    for (int r = 0; r < dk; ++r)
                        kk[r] = orc_elem(k, (((size_t)b * T + t) * Hk + i) * dk + r, io_bf16);
                    for (int c = 0; c < dv; ++c)
                        vv[c] = orc_elem(v, (((size_t)b * T + t) * Hv + j) * dv + c, io_bf16);
                    const double a = alpha[((size_t)b * T + t) * Hv + j];
                    const double be = beta[((size_t)b * T + t) * Hv + j];
                    orc_gdn_step(h, dk, dv, kk, vv, a, be, u);
                }
                for (int r = 0; r < dk; ++r)
                    qq[r] = orc_elem(q, (((size_t)b * T + n) * Hk + i) * dk + r, io_bf16);
                for (int c = 0; c < dv; ++c) {
                    double acc = 0.0;
                    for (int r = 0; r < dk; ++r) acc += h[(size_t)r * dv + c] * qq[r];
                    out[c] = acc;
                }
            }
        }
    }
    free(h); free(kk); free(qq); free(vv); free(u);
    return 0;
}

/* ---- C4: tree-ancestor-masked attention [TREE] --------------------------- */

/*
 * orc_attn_tree: for node n and q-head h (kv-head g = h / (Hq/Hkv)) the
 * visible keys are the cache rows [0, kv_len[b]) and the tree rows a with bit
 * a set in anc[b][n] (the node and its ancestors).  Scores are
 * <q, k_x> / sqrt(D); o = sum_x softmax(s)_x v_x.  Padding rows get o = 0.
 * Requires Hq % Hkv == 0 and 0 <= kv_len[b] <= Lmax.
 */
int orc_attn_tree(int B, int T, int Hq, int Hkv, int D, int Lmax,
                  const int32_t *n_nodes, const uint64_t *node_anc,
                  const void *q, const void *k_tree, const void *v_tree,
                  const void *k_cache, const void *v_cache, const int32_t *kv_len,
                  int io_bf16, double *o)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || T > ORC_MAX_ROWS) return -1;
    for (int b = 0; b < B; ++b)
        if (kv_len[b] < 0 || kv_len[b] > Lmax) return -1;
    const int grp = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)D);
    double *qq = (double *)malloc(sizeof(double) * (size_t)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)(Lmax + T));
    if (!qq || !s) { free(qq); free(s); return -3; }

    for (int b = 0; b < B; ++b) {
        const int L = kv_len[b];
        for (int n = 0; n < T; ++n) {
            const uint64_t *anc = node_anc + ((size_t)b * T + n) * ORC_ANC_WORDS;
            for (int hq = 0; hq < Hq; ++hq) {
                double *out = o + (((size_t)b * T + n) * Hq + hq) * D;
                for (int d = 0; d < D; ++d) out[d] = 0.0;
                if (n >= n_nodes[b]) continue;
                const int g = hq / grp;
                for (int d = 0; d < D; ++d)
                    qq[d] = orc_elem(q, (((size_t)b * T + n) * Hq + hq) * D + d, io_bf16);

                /* scores over the visible set: cache rows, then tree rows */
                int nv = 0;
                double mx = -INFINITY;
                for (int x = 0; x < L; ++x) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += qq[d] * orc_elem(k_cache, (((size_t)b * Lmax + x) * Hkv + g) * D + d, io_bf16);
                    s[nv] = acc * scale;
                    if (s[nv] > mx) mx = s[nv];
                    ++nv;
                }
                for (int a = 0; a < n_nodes[b]; ++a) {
                    if (!((anc[a / 64] >> (a % 64)) & 1ull)) continue;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += qq[d] * orc_elem(k_tree, (((size_t)b * T + a) * Hkv + g) * D + d, io_bf16);
                    s[nv] = acc * scale;
                    if (s[nv] > mx) mx = s[nv];
                    ++nv;
                }

                double den = 0.0;
                for (int x = 0; x < nv; ++x) { s[x] = exp(s[x] - mx); den += s[x]; }
                nv = 0;
                for (int x = 0; x < L; ++x, ++nv)
                    for (int d = 0; d < D; ++d)
                        out[d] += s[nv] * orc_elem(v_cache, (((size_t)b * Lmax + x) * Hkv + g) * D + d, io_bf16);
                for (int a = 0; a < n_nodes[b]; ++a) {
                    if (!((anc[a / 64] >> (a % 64)) & 1ull)) continue;
                    for (int d = 0; d < D; ++d)
                        out[d] += s[nv] * orc_elem(v_tree, (((size_t)b * T + a) * Hkv + g) * D + d, io_bf16);
                    ++nv;
                }
                for (int d = 0; d < D; ++d) out[d] /= den;
            }
        }
    }
    free(qq);
    free(s);
    return 0;
}

/* ---- C5: vocabulary argmax [SD] ----------------------------------------- */

/*
 * orc_argmax: first index of the maximum of each row, values compared as
 * floats after widening.  margin[row] = max - (largest value at any other
 * index); it is +inf for V == 1.
 */
int orc_argmax(int rows, int V, const void *logits, int io_bf16,
               int32_t *idx, float *margin)
{
    if (V < 1) return -1;
    for (int r = 0; r < rows; ++r) {
        int best = 0;
        float bv = (float)orc_elem(logits, (size_t)r * V, io_bf16);
        for (int x = 1; x < V; ++x) {
            float f = (float)orc_elem(logits, (size_t)r * V + x, io_bf16);
            if (f > bv) { bv = f; best = x; }
        }
        double second = -INFINITY;
        for (int x = 0; x < V; ++x) {
            if (x == best) continue;
            double f = orc_elem(logits, (size_t)r * V + x, io_bf16);
            if (f > second) second = f;
        }
        idx[r] = best;
        if (margin) margin[r] = (float)((double)bv - second);
    }
    return 0;
}

/* ---- R15: the target's draw at each row, for stochastic acceptance [RS] -- */

/*
 * Philox4x32-10, from its definition in J. Salmon, M. Moraes, R. Dror and
 * D. Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011): ten
 * rounds of
 *   (hi0, lo0) = 64-bit product 0xD2511F53 * c0,
 *   (hi1, lo1) = 64-bit product 0xCD9E8D57 * c2,
 *   c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),
 * the key (k0, k1) growing by (0x9E3779B9, 0xBB67AE85) before every round but
 * the first.
 */
static void orc_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

int orc_philox4x32_10(int n, const uint32_t *ctr, const uint32_t *key, uint32_t *out)
{
    for (int i = 0; i < n; ++i) orc_philox(ctr + 4 * (size_t)i, key + 2 * (size_t)i, out + 4 * (size_t)i);
    return 0;
}

/* Gumbel noise of one 32-bit word: U = (floor(x / 2^9) + 1/2) / 2^23, which
 * lies in (0, 1) and is exact in float; g = -ln(-ln U). */
static double orc_gumbel(uint32_t x)
{
    const double u = ((double)(x >> 9) + 0.5) / 8388608.0;
    return -log(-log(u));
}

/* Noise of index i (a token, or a chunk when `chunk_space`) of tree row t of
 * request b at cache position pos: word i % 4 of Philox4x32-10 with counter
 * (i / 4, t or t + 2^31, b, pos) and key (low, high 32 bits of seed). */
static double orc_noise(uint64_t seed, uint32_t i, int chunk_space, uint32_t t, uint32_t b,
                        uint32_t pos)
{
    const uint32_t ctr[4] = {i >> 2, chunk_space ? (t | 0x80000000u) : t, b, pos};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox(ctr, key, w);
    return orc_gumbel(w[i & 3]);
}

/*
 * One draw from softmax(l / theta) over the V logits of tree row t of request
 * b (cache position pos), by the two-level Gumbel-max of R15:
 *   chunk c holds tokens [c C, min(V, (c+1) C));
 *   lambda_c = log sum_{v in c} exp(l_v / theta);
 *   c* = the chunk with the largest lambda_c + g_chunk(c) (lowest c on ties);
 *   v* = the token of c* with the largest l_v / theta + g_token(v) (lowest v).
 * P(v*) = P(c*) P(v* | c*) = exp(l_v / theta) / sum_u exp(l_u / theta).
 * *margin = the smaller of the two top-2 gaps (chunk scores; token scores in
 * c*), +inf when a level has one entry.  With alt >= 0, gaps[0] = the best
 * chunk score minus the score of alt's chunk and gaps[1] = the best token
 * score in alt's chunk minus alt's score (both 0 when alt is the draw).
 */
static int orc_sample_row(int V, const void *logits, int io_bf16, size_t row_off, double theta,
                          uint64_t seed, uint32_t t, uint32_t b, uint32_t pos, int C,
                          int alt, int *out, double *margin, double *gaps)
{
    const int nc = (V + C - 1) / C;
    double *score = (double *)malloc(sizeof(double) * (size_t)nc);
    if (!score) return -3;
    for (int c = 0; c < nc; ++c) {
        const int lo = c * C, hi = lo + C < V ? lo + C : V;
        double M = -INFINITY;
        for (int v = lo; v < hi; ++v) {
            const double l = orc_elem(logits, row_off + v, io_bf16) / theta;
            if (l > M) M = l;
        }
        double S = 0.0;
        for (int v = lo; v < hi; ++v) S += exp(orc_elem(logits, row_off + v, io_bf16) / theta - M);
        score[c] = M + log(S) + orc_noise(seed, (uint32_t)c, 1, t, b, pos);
    }
    int cs = 0;
    for (int c = 1; c < nc; ++c) if (score[c] > score[cs]) cs = c;
    double second = INFINITY;
    if (nc > 1) {
        double s2 = -INFINITY;
        for (int c = 0; c < nc; ++c) if (c != cs && score[c] > s2) s2 = score[c];
        second = score[cs] - s2;
    }
    /* the token level inside chunk c: best token, top-2 gap, alt's gap */
    int best = -1;
    double gap_tok = INFINITY;
    for (int pass = 0; pass < 2; ++pass) {
        const int c = pass == 0 ? cs : (alt >= 0 ? alt / C : -1);
        if (c < 0 || c >= nc) break;
        const int lo = c * C, hi = lo + C < V ? lo + C : V;
        int bv = -1;
        double b1 = -INFINITY, b2 = -INFINITY, za = -INFINITY;
        for (int v = lo; v < hi; ++v) {
            const double z = orc_elem(logits, row_off + v, io_bf16) / theta +
                             orc_noise(seed, (uint32_t)v, 0, t, b, pos);
            if (z > b1) { b2 = b1; b1 = z; bv = v; }
            else if (z > b2) b2 = z;
            if (v == alt) za = z;
        }
        if (pass == 0) {
            best = bv;
            gap_tok = hi - lo > 1 ? b1 - b2 : INFINITY;
        } else if (gaps) {
            gaps[0] = score[cs] - score[c];
            gaps[1] = b1 - za;
        }
    }
    *out = best;
    if (margin) *margin = second < gap_tok ? second : gap_tok;
    free(score);
    return 0;
}

/*
 * orc_sample_rows: the draw of every row t < n_nodes[b] of every request
 * (cache position kv_len[b]); padding rows get -1 and margin +inf.
 * logits [B][T][V].  Returns -1 on bad sizes or theta <= 0.
 */
int orc_sample_rows(int B, int T, int V, const void *logits, int io_bf16,
                    const int32_t *n_nodes, const int32_t *kv_len, double theta,
                    uint64_t seed, int chunk, int32_t *sample, double *margin)
{
    if (V < 1 || chunk < 1 || !(theta > 0.0)) return -1;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const size_t r = (size_t)b * T + t;
            if (t >= n_nodes[b]) { sample[r] = -1; margin[r] = INFINITY; continue; }
            int v;
            const int rc = orc_sample_row(V, logits, io_bf16, r * (size_t)V, theta, seed,
                                          (uint32_t)t, (uint32_t)b, (uint32_t)kv_len[b], chunk,
                                          -1, &v, &margin[r], NULL);
            if (rc) return rc;
            sample[r] = v;
        }
    return 0;
}

/* Gaps of the token `alt` in one row's draw (see orc_sample_row): how far it
 * falls behind the draw at the chunk and at the token level. */
int orc_sample_gaps(int V, const void *row_logits, int io_bf16, int t, int b, int pos,
                    double theta, uint64_t seed, int chunk, int alt, double *gaps)
{
    if (V < 1 || chunk < 1 || !(theta > 0.0) || alt < 0 || alt >= V) return -1;
    int v;
    return orc_sample_row(V, row_logits, io_bf16, 0, theta, seed, (uint32_t)t, (uint32_t)b,
                          (uint32_t)pos, chunk, alt, &v, NULL, gaps);
}

/* ---- C6: greedy acceptance of the longest matching root path [SD][TREE] -- */

/*
 * orc_accept: starting at the root, repeatedly look up the target argmax t of
 * the current row and move to the child of the current node whose token is t
 * (lowest node index when tokens repeat); stop when there is none.
 * tau = number of nodes on the accepted path (root included) in [1, m+1];
 * accept_nodes[b][0..tau) = the path; out_tok[b][0..tau) = tokens of the
 * accepted drafts followed by the bonus token (the argmax of the last accepted
 * row); slots >= tau hold -1.  new_root[b] = the bonus token.
 * argmax is [B][T].
 */
int orc_accept(int B, int T, int m,
               const int32_t *node_tok, const int32_t *node_parent,
               const int32_t *n_nodes, const int32_t *argmax,
               int32_t *accept_len, int32_t *accept_nodes, int32_t *out_tok,
               int32_t *new_root)
{
    for (int b = 0; b < B; ++b) {
        const int32_t *tok = node_tok + (size_t)b * T, *par = node_parent + (size_t)b * T;
        const int32_t *am = argmax + (size_t)b * T;
        int32_t *path = accept_nodes + (size_t)b * (m + 1), *ot = out_tok + (size_t)b * (m + 1);
        for (int i = 0; i <= m; ++i) { path[i] = -1; ot[i] = -1; }
        int cur = 0, len = 0;
        path[len++] = 0;
        for (;;) {
            const int t = am[cur];
            int next = -1;
            for (int c = 0; c < n_nodes[b]; ++c)
                if (par[c] == cur && tok[c] == t) { next = c; break; }
            if (next < 0 || len > m) break;
            ot[len - 1] = tok[next];
            path[len++] = next;
            cur = next;
        }
        ot[len - 1] = am[cur];
        accept_len[b] = len;
        new_root[b] = am[cur];
    }
    return 0;
}

/* ---- C7: commit of the accepted path [GDN][NOV] -------------------------- */

/*
 * orc_commit_gdn: h[b][j] <- the state after applying the gated-delta steps
 * of accept_nodes[b][0..tau) in order (root first) to h[b][j], for one GDN
 * layer.  Inputs as in orc_gdn_tree; h is updated in place (double).
 */
int orc_commit_gdn(int B, int T, int m, int Hk, int Hv, int dk, int dv,
                   const int32_t *accept_len, const int32_t *accept_nodes,
                   double *h, const void *k, const void *v, int io_bf16,
                   const float *alpha, const float *beta)
{
    if (Hk <= 0 || Hv % Hk != 0) return -1;
    const int grp = Hv / Hk;
    double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
    double *vv = (double *)malloc(sizeof(double) * (size_t)dv);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!kk || !vv || !u) { free(kk); free(vv); free(u); return -3; }
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < Hv; ++j) {
            const int i = j / grp;
            double *hj = h + ((size_t)b * Hv + j) * dk * dv;
            for (int s = 0; s < accept_len[b]; ++s) {
                const int t = accept_nodes[(size_t)b * (m + 1) + s];
                for (int r = 0; r < dk; ++r)
                    kk[r] = orc_elem(k, (((size_t)b * T + t) * Hk + i) * dk + r, io_bf16);
                for (int c = 0; c < dv; ++c)
                    vv[c] = orc_elem(v, (((size_t)b * T + t) * Hv + j) * dv + c, io_bf16);
                orc_gdn_step(hj, dk, dv, kk, vv, alpha[((size_t)b * T + t) * Hv + j],
                             beta[((size_t)b * T + t) * Hv + j], u);
            }
        }
    }
    free(kk); free(vv); free(u);
    return 0;
}

/*
 * orc_commit_kv: for one attention layer, copy the tree K/V rows of the
 * accepted path to cache rows [kv_len[b], kv_len[b] + tau) (raw element
 * copies, bit-exact).  kv_len is NOT advanced here: the caller advances it
 * once after every layer is committed.  Returns -4 (and copies nothing for
 * any request) if some kv_len[b] + tau > Lmax.
 */
int orc_commit_kv(int B, int T, int m, int Hkv, int D, int Lmax,
                  const int32_t *accept_len, const int32_t *accept_nodes,
                  const void *k_tree, const void *v_tree, void *k_cache, void *v_cache,
                  const int32_t *kv_len, int io_bf16)
{
    const size_t esz = io_bf16 ? 2 : 4;
    const size_t row = (size_t)Hkv * D * esz;
    for (int b = 0; b < B; ++b)
        if (kv_len[b] + accept_len[b] > Lmax) return -4;
    for (int b = 0; b < B; ++b) {
        for (int s = 0; s < accept_len[b]; ++s) {
            const int t = accept_nodes[(size_t)b * (m + 1) + s];
            const size_t dst = ((size_t)b * Lmax + kv_len[b] + s) * row;
            const size_t src = ((size_t)b * T + t) * row;
            memcpy((char *)k_cache + dst, (const char *)k_tree + src, row);
            memcpy((char *)v_cache + dst, (const char *)v_tree + src, row);
        }
    }
    return 0;
}
