/*
 * spec_tree.h -- C ABI of libspectree: the tree-verification step of lossless
 * greedy speculative decoding on a hybrid Gated-DeltaNet / attention target,
 * as hand-written CUDA kernels for one NVIDIA GB300 (sm_103a).
 *
 * The operations are those of the paper digest "SpecPilot: Autonomous
 * Algorithm Discovery and Systems Optimization for Speculative Decoding"
 * (rainbus.top); each entry point names the section it implements.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer to a caller-owned, contiguous,
 *    row-major buffer in the layout stated next to it, unless it says "host".
 *    The library allocates no memory and keeps no state between calls, with
 *    one exception: attn_tree_verify_noalloc's scratch, a static device array
 *    of the library's module (one per device) whose address the library
 *    caches after that call's first use on a device.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL means the legacy default stream).  Calls on different streams must
 *    use different buffers and workspaces.
 *  - Notation: B requests, m lattice positions, K candidates per position,
 *    N draft nodes, T = N + 1 tree rows (the root, i.e. the pending bonus
 *    token, plus N drafts).  Hk/Hv GDN q-k/v heads of dims dk/dv; Hq/Hkv
 *    attention query/key-value heads of dim D; Lmax cache rows per request;
 *    V vocabulary.  "io" below means the element type cfg->io_dtype selects:
 *    bfloat16 (SPEC_IO_BF16) or float (SPEC_IO_F32).
 *  - Limits (else ST_EINVAL): 1 <= B; 1 <= m <= 64; 1 <= K <= 32;
 *    0 <= N <= 127; dk, dv in {64, 128}; Hv % Hk == 0; D in {64, 128};
 *    Hq % Hkv == 0; 1 <= V; every pointer non-NULL and 16-byte aligned.
 *  - Host return value: an ST_* code.  Errors found on the device while the
 *    kernels run (cache overflow, a malformed lattice) are OR-ed into the
 *    device status word at the start of the workspace; read it with
 *    spec_status_read.
 *  - The workspace `ws` is caller-owned device memory of at least
 *    spec_workspace_bytes(cfg) bytes, zero-filled ONCE after allocation; every
 *    call leaves its internal counters at zero again.  One workspace serves
 *    one stream at a time.  Its layout (how the attention's keys are chunked,
 *    how the logits scan is split) follows the SM count of the device the
 *    calls run on: size it with that device current, and use it on that
 *    device (or one with the same SM count).
 */
#ifndef SPEC_TREE_H
#define SPEC_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_TREE_ABI_VERSION 1
#define SPEC_ANC_WORDS 2     /* ancestor bitmask words per tree row (T <= 128) */
#define SPEC_MAX_ROWS 128
#define SPEC_MAX_K 32
#define SPEC_MAX_M 64

/* Host return codes. */
enum {
    ST_OK = 0,           /* launched */
    ST_EINVAL = 1,       /* NULL or misaligned pointer, shape outside the limits */
    ST_EUNSUPPORTED = 2, /* unsupported dtype or head dimension */
    ST_ECUDA = 3,        /* a CUDA launch or copy failed (cudaGetLastError) */
    ST_EOVERFLOW = 4,    /* device status: kv_len + tau > Lmax for some request */
    ST_TIMEOUT = 5,      /* device status: a bounded device-side wait gave up */
    ST_ESCRATCH = 6      /* shape needs more than the fixed static scratch of
                            attn_tree_verify_noalloc */
};

/* Bits of the device status word (uint32 at byte 0 of the workspace). */
/* Tokens per vocabulary chunk of the sampled acceptance's two-level draw. */
#define SPEC_SAMPLE_CHUNK 4096

#define SPEC_DEV_OVERFLOW 0x1u  /* a request's commit was skipped: no room in the cache */
#define SPEC_DEV_BADLAT   0x2u  /* a lattice position repeats a token or has a NaN score */
#define SPEC_DEV_TIMEOUT  0x4u  /* a bounded device-side wait gave up */
#define SPEC_DEV_BADREQ   0x8u  /* a per-request position count was outside [1, m] (clamped) */
#define SPEC_DEV_BADLOGIT 0x10u /* a sampled row had no finite score (NaN / inf logits) */
#define SPEC_DEV_RANGE    0x20u /* attention: an output of a real tree row is not finite.  With
                                   bf16 I/O the attention keeps V and the split-KV partials in
                                   fp16, so a V value beyond fp16's range (|v| > 65504) among
                                   the keys the row sees (cache rows below kv_len, its tree
                                   ancestors) gives this, as do non-finite inputs there. */

enum { SPEC_IO_F32 = 0, SPEC_IO_BF16 = 1 };

/* Problem shape; passed by host pointer, read during the call only. */
typedef struct spec_cfg {
    int32_t B, m, K, N;
    int32_t Hk, Hv, dk, dv;          /* GDN */
    int32_t Hq, Hkv, D;              /* attention */
    int32_t Lmax;                    /* KV cache rows per request */
    int32_t V;                       /* vocabulary */
    int32_t n_gdn_layers, n_attn_layers;
    int32_t io_dtype;                /* SPEC_IO_BF16 or SPEC_IO_F32 */
} spec_cfg;

/* A draft tree per request, T = N + 1 rows in insertion order (a parent
 * always precedes its children).  Rows n >= n_nodes[b] are padding:
 * tok = parent = depth = rank = -1, score = 0, anc = 0. */
typedef struct spec_tree {
    int32_t *node_tok;      /* [B][T] token of the row (row 0: the root token) */
    int32_t *node_parent;   /* [B][T] parent row, -1 for the root */
    int32_t *node_depth;    /* [B][T] 0 for the root */
    int32_t *node_rank;     /* [B][T] rank of the token among its position's candidates, -1 root */
    float   *node_score;    /* [B][T] fp32 root-path sum of edge scores, 0 for the root */
    uint64_t *node_anc;     /* [B][T][2] bit a set iff row a is the row or one of its ancestors */
    int32_t *n_nodes;       /* [B] rows in use, 1 + min(N, sum_d K^d) */
} spec_tree;

/* Stacked per-layer buffers that accept_and_commit reads and updates.  Each
 * is the concatenation over layers (layer outermost) of the buffer the
 * matching verify call used for that layer. */
typedef struct spec_commit_io {
    float *h0;              /* [n_gdn][B][Hv][dk][dv] fp32 committed state, updated in place */
    const void *gdn_k;      /* [n_gdn][B][T][Hk][dk] io */
    const void *gdn_v;      /* [n_gdn][B][T][Hv][dv] io */
    const float *alpha;     /* [n_gdn][B][T][Hv] */
    const float *beta;      /* [n_gdn][B][T][Hv] */
    const void *k_tree;     /* [n_attn][B][T][Hkv][D] io */
    const void *v_tree;     /* [n_attn][B][T][Hkv][D] io */
    void *k_cache;          /* [n_attn][B][Lmax][Hkv][D] io, rows appended */
    void *v_cache;          /* [n_attn][B][Lmax][Hkv][D] io, rows appended */
    int32_t *kv_len;        /* [B] valid cache rows, advanced by tau */
    int32_t *root_tok;      /* [B] replaced by the bonus token */
} spec_commit_io;

/* Outputs of the acceptance. */
typedef struct spec_accept {
    int32_t *argmax;        /* [B][T] target argmax of each row, -1 on padding rows */
    int32_t *accept_len;    /* [B] tau in [1, m+1]: accepted drafts + 1 */
    int32_t *accept_nodes;  /* [B][m+1] accepted root path (row 0 first), -1 beyond tau */
    int32_t *out_tok;       /* [B][m+1] emitted tokens: accepted drafts then the bonus, -1 beyond tau */
} spec_accept;

/* Sampled acceptance (temperature > 0). */
typedef struct spec_sampling {
    float temperature;      /* > 0 and finite */
    uint32_t reserved;      /* must be 0 */
    uint64_t seed;          /* Philox4x32-10 key: (low 32 bits, high 32 bits) */
} spec_sampling;

/* Bytes of device workspace the calls below need for `cfg` on the current
 * device (0 on an invalid cfg, or when no device is visible). */
size_t spec_workspace_bytes(const spec_cfg *cfg);

/* The same for a device with `num_sms` SMs (host only: no device needed; 0 on
 * an invalid cfg or num_sms < 1).  The calls lay the workspace out for the SM
 * count of the device they run on, so size with that device's count. */
size_t spec_workspace_bytes_for_sms(const spec_cfg *cfg, int num_sms);

/*
 * spec_tree_build -- best-first draft tree over the drafter's lattice.
 * Digest: prerequisites / parallel drafter (per-position top-k candidates and
 * scores form a lattice), prerequisites / draft-tree verification (nodes are
 * added greedily by root-path log-prob up to N) and technical novelty,
 * Figure 6 (best-first tree, edges scored log p(child | parent)).
 *
 * Candidates of each position are ordered by score (descending), then input
 * index; a candidate's rank is its place in that order.  Row 0 is the root
 * (token root_tok[b], depth 0, score 0).  A child (p, r) of an inserted row p
 * of depth < m takes the rank-r candidate of lattice position depth(p) and the
 * key fl32(score_p + edge score).  N times (or until no child is left) the
 * child first in the order (key desc, depth asc, parent asc, rank asc) becomes
 * the next row.  Scores must be finite; a position must not repeat a token
 * (else SPEC_DEV_BADLAT is raised and that request's tree is unspecified).
 *   lat_tok   [B][m][K] int32     lat_score [B][m][K] float
 *   root_tok  [B] int32           out       tree buffers for T = N + 1 rows
 */
int spec_tree_build(const spec_cfg *cfg, const int32_t *lat_tok, const float *lat_score,
                    const int32_t *root_tok, const spec_tree *out, void *ws, void *stream);

/*
 * gdn_tree_verify -- outputs of one Gated-DeltaNet layer for every tree row.
 * Digest: prerequisites / hybrid recurrent target (gated delta rule
 * h_t = alpha_t (I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T,
 * o_t = h_t^T q_t) and technical novelty (each node's state is recomputed
 * along its root path from the committed state, without per-node snapshots).
 *
 * For row n and v-head j (q-k head j / (Hv/Hk)): start from h0[b][j], apply
 * the step of every row on n's root path (root first, n last) and output
 * o[b][n][j] = h^T q_n.  Padding rows get 0.  No state is written.
 *   h0    [B][Hv][dk][dv] float          q, k [B][T][Hk][dk] io
 *   v     [B][T][Hv][dv] io              alpha, beta [B][T][Hv] float
 *   o     [B][T][Hv][dv] io (output)
 *   c_opt NULL, or [B][T][Hv][dv] float: per-row write vectors
 *         c_n = beta_n v_n - alpha_n beta_n h_parent^T k_n (output)
 */
int gdn_tree_verify(const spec_cfg *cfg, const spec_tree *tree, const float *h0,
                    const void *q, const void *k, const void *v, const float *alpha,
                    const float *beta, void *o, float *c_opt, void *ws, void *stream);

/*
 * attn_tree_verify -- tree-ancestor-masked attention of one layer.
 * Digest: prerequisites / draft-tree verification (every node sees only its
 * ancestors).
 *
 * Row n, q-head h (kv-head h / (Hq/Hkv)) attends to cache rows
 * [0, kv_len[b]) and to the tree rows that are n or its ancestors:
 * o = softmax(q K^T / sqrt(D)) V, fp32 accumulation.  Padding rows get 0.
 * Requires 0 <= kv_len[b] <= Lmax (checked against Lmax on the device).
 *   q [B][T][Hq][D] io      k_tree, v_tree [B][T][Hkv][D] io
 *   k_cache, v_cache [B][Lmax][Hkv][D] io     kv_len [B] int32
 *   o [B][T][Hq][D] io (output)
 */
int attn_tree_verify(const spec_cfg *cfg, const spec_tree *tree, const void *q,
                     const void *k_tree, const void *v_tree, const void *k_cache,
                     const void *v_cache, const int32_t *kv_len, void *o, void *ws,
                     void *stream);

/*
 * accept_and_commit -- greedy acceptance and commit of the accepted path.
 * Digest: prerequisites / speculative decoding (accept the longest prefix equal
 * to the target argmax plus one bonus token, tau in [1, m+1]) and draft-tree
 * verification (the longest matching root path); the commit recomputes the
 * state along the accepted root path (technical novelty).
 *
 * (i) argmax[b][n] = first index of the maximum of logits[b][n][:].
 * (ii) From the root, move to the child whose token equals the current row's
 * argmax (lowest row index on repeats) while one exists; tau = rows on the path.
 * out_tok = tokens of the accepted drafts, then the bonus (argmax of the last
 * accepted row).  (iii) Unless kv_len[b] + tau > Lmax (then SPEC_DEV_OVERFLOW
 * is raised and request b is left uncommitted): every GDN layer's h0 advances
 * over the tau path rows, every attention layer's cache rows
 * [kv_len, kv_len + tau) receive the path rows' tree K/V, kv_len += tau and
 * root_tok = bonus.
 *   logits [B][T][V] io
 */
int accept_and_commit(const spec_cfg *cfg, const spec_tree *tree, const void *logits,
                      const spec_commit_io *io, const spec_accept *out, void *ws,
                      void *stream);

/*
 * accept_and_commit_sampled -- accept_and_commit at temperature > 0.
 * Speculative-decoding tutorial (mlqm.cn), section 2.3: a draft x with draft
 * probability q(x) is kept with probability min(1, p(x)/q(x)), else a token
 * is drawn from max(0, p - q) renormalised, and the output follows the
 * target's p exactly.  The tree's drafts are fixed tokens (q a point mass), so
 * at a node the rule keeps child x with the probability of x under p with the
 * earlier children removed; that is the law of drawing y from p at the row and
 * moving to the child whose token is y.  So step (i) of accept_and_commit
 * becomes a draw per row, and (ii)-(iii) are unchanged:
 *   p = softmax(logits[b][n][:] / temperature);
 *   chunk c = tokens [c C, min(V, (c+1) C)), C = SPEC_SAMPLE_CHUNK;
 *   c* = argmax_c log(sum_{v in c} exp(l_v / temperature)) + G(c)  (lowest c on ties)
 *   draw = argmax_{v in c*} l_v / temperature + G(v)                  (lowest v on ties)
 *   G(i) = -ln(-ln U), U = (floor(x / 2^9) + 1/2) 2^-23, x = word i % 4 of
 *   Philox4x32-10 with key (seed low, seed high) and counter
 *   (i / 4, n (+ 2^31 for chunks), b, kv_len[b]);
 * argmax[b][n] of `out` receives the draw.  A row whose scores are all NaN
 * (NaN or +inf logits) draws the first token of its first chunk and raises
 * SPEC_DEV_BADLOGIT.  The result is a draw from p (in
 * exact arithmetic); draws whose top-2 score gap is within float rounding can
 * differ from a float64 evaluation of the same definition.
 * ST_EINVAL when temperature is not > 0 and finite or reserved != 0.
 */
int accept_and_commit_sampled(const spec_cfg *cfg, const spec_tree *tree, const void *logits,
                              const spec_sampling *smp, const spec_commit_io *io,
                              const spec_accept *out, void *ws, void *stream);

/* Per-layer verify buffers of a whole step, stacked with the layer outermost
 * (layer l of gdn_q is the q that gdn_tree_verify would get for layer l). */
typedef struct spec_step_io {
    const void *gdn_q;      /* [n_gdn][B][T][Hk][dk] io */
    void *gdn_o;            /* [n_gdn][B][T][Hv][dv] io (output) */
    float *gdn_c;           /* NULL, or [n_gdn][B][T][Hv][dv] float (output) */
    const void *attn_q;     /* [n_attn][B][T][Hq][D] io */
    void *attn_o;           /* [n_attn][B][T][Hq][D] io (output) */
} spec_step_io;

/*
 * spec_verify_step -- one whole verify step: spec_tree_build into `tree`,
 * gdn_tree_verify for every GDN layer, attn_tree_verify for every attention
 * layer, then accept_and_commit; the results equal those of the four calls
 * made in that order on `stream`.  (Digest sections as for the four calls.)
 *
 * The kernels are launched in that fixed order with programmatic dependent
 * launch, so each one stages the inputs that do not depend on its
 * predecessor (state slices, cache blocks, logits) while the predecessor
 * finishes.  Per-layer inputs come from `step` (q) and `io` (everything the
 * commit also needs); outputs go to `step`, `tree`, `out` and the state in
 * `io`.  Needs spec_workspace_bytes(cfg) of workspace like the other calls.
 */
int spec_verify_step(const spec_cfg *cfg, const int32_t *lat_tok, const float *lat_score,
                     const spec_tree *tree, const spec_step_io *step, const void *logits,
                     const spec_commit_io *io, const spec_accept *out, void *ws, void *stream);

/*
 * spec_tree_build_ragged -- best-first draft trees of a batch with per-request
 * draft positions and a node budget shared by the batch.
 * Digest: technical novelty, batching (one node budget shared across the
 * batch, at the target GEMM's 192-node plateau; 16/12/8 draft positions chosen
 * per request), with the tree rules of spec_tree_build.
 *
 * Request b drafts from its first m_req[b] lattice positions (its nodes have
 * depth <= m_req[b]).  With node_budget >= 0 the batch keeps node_budget draft
 * nodes in all: the ones first in the order (score desc, request asc, then the
 * per-tree order), i.e. best-first over every request's frontier together,
 * each request holding at most N; every request keeps a prefix of its own
 * best-first order.  node_budget < 0: no shared budget (each request up to N).
 *   m_req  NULL (all m) or device int32 [B], values in [1, m]; an out-of-range
 *          value is clamped and sets SPEC_DEV_BADREQ.
 * Other arguments, outputs and padding rows as spec_tree_build.  The budget
 * step needs 4 (B (N + 1) + 2 B) bytes of shared memory in one CTA: more than
 * 200 KB returns ST_EUNSUPPORTED.  One more launch than spec_tree_build when
 * node_budget >= 0.
 */
int spec_tree_build_ragged(const spec_cfg *cfg, const int32_t *lat_tok, const float *lat_score,
                           const int32_t *root_tok, const int32_t *m_req, int node_budget,
                           const spec_tree *out, void *ws, void *stream);

/*
 * spec_tree_build_markov -- best-first draft tree whose edge scores depend on
 * the parent's token (a drafter with a Markov head).
 * Digest: prerequisites / parallel drafter (DSpark's Markov head:
 * l_s(y) = bases(y) + <W1[x_{s-1}], W2[y]>) and technical novelty, Figure 6
 * (edges scored log p(child | parent)).
 *
 * Candidate i of lattice position d under a parent with token x scores
 *   l_i = base_i + W1[x] . W2[y_i]      (fp32: one fused multiply-add chain over
 *                                        k = 0..R-1, then one add)
 *   e_i = l_i - (M + log32(sum_i exp32(l_i - M))),  M = max_i l_i
 * (the sum in index order; exp32 / log32 are fp32 functions fixed by their
 * algorithm: Cody-Waite reduction by ln 2 split as 355/512 + fp32(ln 2 -
 * 355/512), rint(x fp32(1/ln 2)), Taylor to degree 7 with coefficients
 * fp32(1/k!) by fused multiply-adds, times 2^n; exponent split, f halved when
 * above fp32(sqrt 2), s = (f - 1) / (f + 1), 2 s times the series in s^2 to
 * s^12 with coefficients fp32(1/k), plus e ln 2 as two fused multiply-adds;
 * exp32 is 0 below -86).  A parent's children are ranked by (e desc, index
 * asc); a child's key is fl32(parent key + e); insertion as spec_tree_build.
 *   lat_tok int32 [B][m][K]; lat_base f32 [B][m][K] the drafter's base logits;
 *   W1, W2 f32 [V][R] the head's two tables (R <= 1024; NULL allowed when R=0);
 *   root_tok, out, ws as spec_tree_build.  A NaN edge, or a token (or root
 *   token) outside [0, V), sets SPEC_DEV_BADLAT (such a token reads head row 0;
 *   that request's tree is unspecified).
 * Shared memory: 16 (1 + (m-1) K) K bytes of table entries plus
 * 4 (2 m K + 1) (R + 4) of staged head rows (R + 1 when R is not a multiple
 * of 4) plus 8 m K + 4 of tokens and bases; more than 200 KB returns
 * ST_EUNSUPPORTED.
 */
int spec_tree_build_markov(const spec_cfg *cfg, const int32_t *lat_tok, const float *lat_base,
                           const float *W1, const float *W2, int R, const int32_t *root_tok,
                           const spec_tree *out, void *ws, void *stream);

/*
 * spec_verify_step_sampled -- spec_verify_step with the acceptance of
 * accept_and_commit_sampled; the same number of launches.
 */
int spec_verify_step_sampled(const spec_cfg *cfg, const int32_t *lat_tok, const float *lat_score,
                             const spec_sampling *smp, const spec_tree *tree,
                             const spec_step_io *step, const void *logits,
                             const spec_commit_io *io, const spec_accept *out, void *ws,
                             void *stream);

/*
 * spec_verify_step_ragged -- spec_verify_step with the trees of
 * spec_tree_build_ragged (per-request draft positions, shared node budget);
 * the rest of the step treats the rows a request did not keep as padding rows.
 * One more launch than spec_verify_step when node_budget >= 0.
 */
int spec_verify_step_ragged(const spec_cfg *cfg, const int32_t *lat_tok, const float *lat_score,
                            const int32_t *m_req, int node_budget, const spec_tree *tree,
                            const spec_step_io *step, const void *logits,
                            const spec_commit_io *io, const spec_accept *out, void *ws,
                            void *stream);

/*
 * spec_verify_step_markov -- spec_verify_step with the tree of
 * spec_tree_build_markov (lat_base: the drafter's base logits; W1, W2, R: its
 * Markov head); the same number of launches as spec_verify_step.
 */
int spec_verify_step_markov(const spec_cfg *cfg, const int32_t *lat_tok, const float *lat_base,
                            const float *W1, const float *W2, int R, const spec_tree *tree,
                            const spec_step_io *step, const void *logits,
                            const spec_commit_io *io, const spec_accept *out, void *ws,
                            void *stream);

/*
 * spec_verify_step_persistent -- spec_verify_step whose argmax, acceptance,
 * KV append and every GDN layer's verify + commit run as one persistent,
 * cooperative launch after the tree and the attention layers.  Digest:
 * technical novelty (states recomputed along the root path, no per-node
 * snapshots) with the sections of the four calls.
 *
 * A GDN (layer, request, v-head) item keeps its fp32 state in shared memory
 * through the verify, waits for its request's acceptance (a flag raised by the
 * request's last argmax item, which also appends the KV rows and advances
 * kv_len / root_tok) and writes the state after the accepted path,
 *   h = A h0 + sum_s dec(p_s -> p_last) k_{p_s} c_{p_s}^T,
 * over h0: the state is read from HBM once and written once.  Every argmax
 * item precedes every GDN item in the work queue and never waits; each wait
 * is bounded (about a second: SPEC_DEV_TIMEOUT, that state left uncommitted).
 * Results equal spec_verify_step's within float rounding (the commit sums the
 * path's rank-one terms instead of stepping the recurrence).
 * Supported: bf16 I/O, d_k = d_v = 128, T <= 32, at least one GDN layer
 * (else ST_EUNSUPPORTED).  Launches: spec_step_launches_persistent(cfg).
 */
int spec_verify_step_persistent(const spec_cfg *cfg, const int32_t *lat_tok,
                                const float *lat_score, const spec_tree *tree,
                                const spec_step_io *step, const void *logits,
                                const spec_commit_io *io, const spec_accept *out, void *ws,
                                void *stream);

/* Number of kernel launches one spec_verify_step(cfg) call makes (host only;
 * -1 on an invalid cfg): for sizing graphs and counting launches.  The same
 * for spec_verify_step_ragged and _markov (the ragged step adds one launch
 * for the budget selection when a budget is given).  With an attention layer
 * and at most 64 logits rows (B x (N + 1)) the argmax + acceptance shares the
 * last merge's launch; spec_verify_step_sampled then makes one launch more
 * (its acceptance is always a launch of its own). */
int spec_step_launches(const spec_cfg *cfg);

/* The same for spec_verify_step_persistent (-1 when unsupported). */
int spec_step_launches_persistent(const spec_cfg *cfg);

/* Copy the device status word into *host_status (host pointer) and wait for
 * `stream`.  Returns ST_OK, or ST_ECUDA if the copy failed. */
int spec_status_read(const void *ws, uint32_t *host_status, void *stream);

/* Zero the device status word on `stream`. */
int spec_status_clear(void *ws, void *stream);

/* Static description of an ST_* code (never NULL). */
const char *spec_status_string(int code);

/* SPEC_TREE_ABI_VERSION of the loaded library. */
int spec_abi_version(void);

/*
 * spec_wait_probe -- diagnostic; the pages describe no such call.  Launches one
 * CTA that waits on a shared-memory mbarrier with the same bounded wait the
 * tensor-core kernels use.  With satisfy = 0 nothing ever arrives, so after
 * about limit_us microseconds (SM cycles at the 2070 MHz maximum clock) the
 * wait gives up and ORs SPEC_DEV_TIMEOUT into the status word of `ws`; with
 * satisfy != 0 the barrier completes first and the status is untouched.
 * Either way the kernel returns normally and the context stays usable.
 *   limit_us in [1, 1000000]; ws as for the other calls (only its status word
 *   is touched).  Returns ST_EINVAL on a bad limit or NULL/misaligned ws.
 */
int spec_wait_probe(uint32_t limit_us, int satisfy, void *ws, void *stream);

/*
 * attn_tree_verify_noalloc -- attn_tree_verify without a caller workspace.
 * The pages describe no such call (their method has no counterpart): it is a
 * library convenience for callers that own no device allocator where they
 * launch the op (a custom op inside a host runtime that owns all device
 * memory, a serving loop that must not call into an allocator).  Neither the
 * call nor anything it calls allocates device or host memory.
 *
 * Arguments, layouts and results are those of attn_tree_verify (the same
 * kernels run), except:
 *   - the scratch (status word + split-KV partials) is a static device array
 *     of SPEC_NOALLOC_SCRATCH_BYTES inside the library, one per device; a
 *     shape whose partials do not fit returns ST_ESCRATCH before any device
 *     work (with Hkv = 8, D = 128, bf16, T <= 32: one request up to Lmax ~ 61K,
 *     two up to ~ 28K, four up to ~ 12K);
 *   - dev_status: NULL, or a 4-byte-aligned device word the call ORs its
 *     SPEC_DEV_* bits into (the caller zeroes it when it wants); each call
 *     clears the scratch status word on its stream before its kernels (a
 *     memset, no allocation) and moves its bits to dev_status after them.
 * Returns the codes attn_tree_verify returns for an invalid cfg, tree or
 * pointer (ST_EINVAL, or ST_EUNSUPPORTED for an unsupported io_dtype).
 * The first call on a device (with that device current) sets up: it looks up
 * the array's address and clears its status word synchronously, so make it
 * before any stream capture or latency-critical section.  The address stays
 * cached for the life of the process: make no call after a cudaDeviceReset of
 * that device.  All calls on one device share the one scratch array: calls
 * that overlap in time (other streams, other host threads, other layers in
 * flight) race on it and give wrong results; order them on one stream or
 * serialise them.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (8u << 20)
int attn_tree_verify_noalloc(const spec_cfg *cfg, const spec_tree *tree, const void *q,
                             const void *k_tree, const void *v_tree, const void *k_cache,
                             const void *v_cache, const int32_t *kv_len, void *o,
                             uint32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_TREE_H */
