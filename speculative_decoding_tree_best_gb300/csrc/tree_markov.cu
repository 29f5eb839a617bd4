// tree_markov.cu -- best-first draft tree whose edge scores depend on the
// parent's token (a drafter with a Markov head).
//
// Digest "SpecPilot ...": prerequisites / parallel drafter (DSpark's Markov
// head conditions each position on the previous token:
// l_s(y) = bases(y) + <W1[x_{s-1}], W2[y]>) and technical novelty, Figure 6
// (best-first tree, edges scored log p(child | parent)).
//
// Edge score of candidate i of lattice position d under a parent with token x:
//     l_i  = base_i + (W1[x] . W2[y_i])     the dot product as one chain of
//                                           fused multiply-adds, k = 0..R-1
//     M    = max_i l_i,  Z = sum_i exp32(l_i - M)   (sum in index order)
//     e_i  = l_i - (M + log32(Z))
// with exp32 / log32 the fp32 functions below (Cody-Waite reduction by ln 2
// and the Taylor polynomial to degree 7; exponent split and the atanh series
// to s^13), every operation an explicitly rounded intrinsic, so the scores are
// fixed to the bit.  Children of a parent are ranked by (e desc, index asc).
//
// One CTA per request: 1024 threads (512 when T > 64).
//  A. All warps stage the rows of W1 and W2 the tables need (every candidate's
//     and the root's) in shared memory, every load in flight before the
//     stores, then fill the tables.  A table row is (position d, parent): the
//     root for d = 0, candidate p of position d-1 otherwise, so row
//     rho = 0 or 1 + (d-1) K + p.  A group of 16 or 32 lanes computes one row:
//     lane i the dot product and l_i, the group the maximum, every lane the
//     ordered sum (read back from shared memory in index order) and the
//     log-sum-exp, each lane its edge and its rank.  Per entry (row, rank): edge, token, the row of that
//     child's own children, and the first (best) edge among them.
//  B. Warp 0 inserts nodes best-first exactly as tree_build.cu does, row x in
//     lane x % 32, slot x / 32.  Each row offers its best remaining child; the
//     offers are compared with two warp-wide max reductions (key, then depth
//     and parent among equal keys).  The child lookups go through the row's
//     table row instead of a position's ranked list; both entries an insertion
//     reads are loaded warp-wide before the (predicated) updates.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace spec {

namespace {

// Threads per CTA: 1024 while the insertion's per-lane slots fit in 64
// registers (T <= 64), else 512.
constexpr int kMarkovThreadsMax = 1024;

__device__ __forceinline__ float exp32(float x) {
    if (x < -86.0f) return 0.0f;
    const float inv_ln2 = (float)(1.0 / 0.69314718055994530941723212145818);
    const float ln2_hi = 355.0f / 512.0f;
    const float ln2_lo = (float)(0.69314718055994530941723212145818 - 355.0 / 512.0);
    const float n = rintf(__fmul_rn(x, inv_ln2));
    float r = __fmaf_rn(-n, ln2_hi, x);
    r = __fmaf_rn(-n, ln2_lo, r);
    float p = (float)(1.0 / 5040.0);
    p = __fmaf_rn(p, r, (float)(1.0 / 720.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 120.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 24.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 6.0));
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const float scale = __uint_as_float(static_cast<uint32_t>(static_cast<int>(n) + 127) << 23);
    return __fmul_rn(p, scale);
}

__device__ __forceinline__ float log32(float z) {
    const uint32_t bits = __float_as_uint(z);
    int e = static_cast<int>((bits >> 23) & 0xffu) - 127;
    float f = __uint_as_float((bits & 0x7fffffu) | 0x3f800000u);
    if (f > (float)1.4142135623730950488016887242097) {
        f = __fmul_rn(f, 0.5f);
        e += 1;
    }
    const float s = __fdiv_rn(__fsub_rn(f, 1.0f), __fadd_rn(f, 1.0f));
    const float s2 = __fmul_rn(s, s);
    float t = (float)(1.0 / 13.0);
    t = __fmaf_rn(t, s2, (float)(1.0 / 11.0));
    t = __fmaf_rn(t, s2, (float)(1.0 / 9.0));
    t = __fmaf_rn(t, s2, (float)(1.0 / 7.0));
    t = __fmaf_rn(t, s2, (float)(1.0 / 5.0));
    t = __fmaf_rn(t, s2, (float)(1.0 / 3.0));
    t = __fmaf_rn(t, s2, 1.0f);
    const float lf = __fmul_rn(__fmul_rn(2.0f, s), t);
    const float ef = static_cast<float>(e);
    return __fmaf_rn(ef, 355.0f / 512.0f,
                     __fmaf_rn(ef, (float)(0.69314718055994530941723212145818 - 355.0 / 512.0), lf));
}

// Order-preserving map of a finite float to uint32 (-0 folded into +0).
__device__ __forceinline__ uint32_t ord_key(float f) {
    if (f == 0.0f) f = 0.0f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Among offers with equal keys: smaller child depth first, then smaller parent.
__device__ __forceinline__ uint32_t tie_rank(int child_depth, int parent) {
    return (static_cast<uint32_t>(255 - child_depth) << 8) | static_cast<uint32_t>(255 - parent);
}

// One table entry (row, rank): 16 bytes, so that the insertion reads an entry
// with one shared-memory load.
struct MEnt {
    float edge;       // edge score of the rank-th child
    float first;      // the first (best) edge among that child's children (0: none)
    int32_t tok;      // its token
    int32_t crow;     // the table row of its children (-1: none)
};

__host__ __device__ inline size_t markov_rows(int m, int K) { return 1 + (size_t)(m - 1) * K; }

// Row stride of the staged head rows in floats: R + 4 when R is a multiple of
// 4 (16-byte loads; the 8 lanes of a load phase then start 4 banks apart),
// else R + 1 (the lanes of a group, each reading its own W2 row at the same
// k, hit distinct banks).
__host__ __device__ inline int markov_stride(int R) { return (R & 3) == 0 ? R + 4 : R + 1; }

// table entries, the staged head rows (W1 of every candidate and the root, W2
// of every candidate), then the lattice's tokens (and the root) and bases
__host__ __device__ inline size_t markov_smem(int m, int K, int R) {
    const size_t e = markov_rows(m, K) * K;
    return sizeof(MEnt) * e + sizeof(float) * (size_t)(2 * m * K + 1) * markov_stride(R) +
           sizeof(int32_t) * (size_t)(m * K + 1) + sizeof(float) * (size_t)m * K;
}

// Phase A for lane groups of G lanes (G >= K): fills every table row's entries
// except `first`.  Returns true when an edge is NaN.
// xs: 64 floats of scratch per warp (the group's exp terms, then its edges),
// read back in index order with 16-byte broadcast loads.
template <int G>
__device__ __forceinline__ bool markov_fill(const spec_cfg& c, int R, int RP, int nthreads,
                                            const float* w1s, const float* w2s,
                                            const int32_t* tok_s, const float* base_s, MEnt* tb,
                                            float* xs_all) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = c.m, K = c.K;
    const int groups = (nthreads / 32) * (32 / G);
    const int grp = warp * (32 / G) + lane / G, gl = lane % G;
    float* xs = xs_all + warp * 64;
    const int g0 = lane & ~(G - 1);          // the group's first lane
    const int nrows = (int)markov_rows(m, K);
    const bool vec = (R & 3) == 0;           // RP = R + 4 then; R + 1 can be a multiple of 4 too
    bool bad = false;
    for (int rho0 = 0; rho0 < nrows; rho0 += groups) {
        const int rho = rho0 + grp;
        const bool act = rho < nrows && gl < K;
        // row rho: position d under parent p (the root for rho = 0)
        const int d = rho == 0 ? 0 : 1 + (rho - 1) / K;
        const int p = rho == 0 ? 0 : rho - 1 - (d - 1) * K;
        float l = -INFINITY;
        int y = 0;
        if (act) {
            y = tok_s[d * K + gl];
            const float* w1 = w1s + (size_t)(rho == 0 ? m * K : (d - 1) * K + p) * RP;
            const float* w2 = w2s + (size_t)(d * K + gl) * RP;
            float dot = 0.0f;
            if (vec) {
#pragma unroll 4
                for (int k = 0; k < R; k += 4) {
                    const float4 a = *reinterpret_cast<const float4*>(w1 + k);
                    const float4 v = *reinterpret_cast<const float4*>(w2 + k);
                    dot = __fmaf_rn(a.x, v.x, dot);
                    dot = __fmaf_rn(a.y, v.y, dot);
                    dot = __fmaf_rn(a.z, v.z, dot);
                    dot = __fmaf_rn(a.w, v.w, dot);
                }
            } else {
#pragma unroll 4
                for (int k = 0; k < R; ++k) dot = __fmaf_rn(w1[k], w2[k], dot);
            }
            l = __fadd_rn(base_s[d * K + gl], dot);
        }
        float M = l;
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o, G));
        // lanes past K add +0, which leaves the ordered sum unchanged
        xs[lane] = act ? exp32(__fsub_rn(l, M)) : 0.0f;
        __syncwarp();
        float Z = 0.0f;
#pragma unroll
        for (int j = 0; j < G; j += 4) {
            const float4 q = *reinterpret_cast<const float4*>(xs + g0 + j);
            Z = __fadd_rn(Z, q.x);
            Z = __fadd_rn(Z, q.y);
            Z = __fadd_rn(Z, q.z);
            Z = __fadd_rn(Z, q.w);
        }
        const float e = __fsub_rn(l, __fadd_rn(M, log32(Z)));
        xs[32 + lane] = e;
        __syncwarp();
        // lanes past K hold e = -inf and never outrank an active lane
        int rank = 0;
#pragma unroll
        for (int j = 0; j < G; j += 4) {
            const float4 q = *reinterpret_cast<const float4*>(xs + 32 + g0 + j);
            rank += (q.x > e || (q.x == e && j < gl)) ? 1 : 0;
            rank += (q.y > e || (q.y == e && j + 1 < gl)) ? 1 : 0;
            rank += (q.z > e || (q.z == e && j + 2 < gl)) ? 1 : 0;
            rank += (q.w > e || (q.w == e && j + 3 < gl)) ? 1 : 0;
        }
        __syncwarp();                        // the next pass rewrites xs
        if (act) {
            MEnt& t = tb[(size_t)rho * K + rank];
            t.edge = e;
            t.tok = y;
            // the child's own children: row 1 + d K + (candidate index)
            t.crow = d + 1 < m ? 1 + d * K + gl : -1;
        }
        bad |= act && !(e == e);           // a NaN base or weight
    }
    return bad;
}

template <int SLOTS, int NT>
__global__ void __launch_bounds__(NT)
tree_markov_kernel(spec_cfg c, int R, const int32_t* __restrict__ lat_tok,
                   const float* __restrict__ lat_base, const float* __restrict__ W1,
                   const float* __restrict__ W2, const int32_t* __restrict__ root_tok,
                   spec_tree out, void* ws) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = c.m, K = c.K, T = c.N + 1;
    const int E = (int)markov_rows(m, K) * K;
    MEnt* tb = reinterpret_cast<MEnt*>(smem);
    __shared__ __align__(16) float xs[(NT / 32) * 64];
    // staged head rows: w1s [m K + 1][RP] (candidate (d, i) at d K + i, the
    // root last), w2s [m K][RP]
    const int RP = markov_stride(R);
    float* w1s = reinterpret_cast<float*>(tb + E);
    float* w2s = w1s + (size_t)(m * K + 1) * RP;
    int32_t* tok_s = reinterpret_cast<int32_t*>(w2s + (size_t)m * K * RP);  // [m K] + root
    float* base_s = reinterpret_cast<float*>(tok_s + m * K + 1);          // [m K]

    pdl_wait();          // root_tok may come from the previous step's acceptance
    pdl_trigger();
    bool bad = false;
    for (int i = tid; i <= m * K; i += NT) {
        const int t = i < m * K ? lat_tok[(size_t)b * m * K + i] : root_tok[b];
        tok_s[i] = t;
        if (i < m * K) base_s[i] = lat_base[(size_t)b * m * K + i];
        bad |= t < 0 || t >= c.V;          // such a token reads head row 0 below
    }
    __syncthreads();
    const int root = tok_s[m * K];
    // every row of W1 and W2 the tables need: each thread issues up to 4 loads
    // before it stores any (16 bytes at a time when the rows allow it)
    {
        const int nw = 2 * m * K + 1;
        const bool vec = (R & 3) == 0 &&
            ((reinterpret_cast<uintptr_t>(W1) | reinterpret_cast<uintptr_t>(W2)) & 15u) == 0;
        const int per_row = vec ? R >> 2 : R;       // loads per row
        const int total = nw * per_row;
        for (int i0 = tid; i0 < total; i0 += 4 * NT) {
            float4 v[4];
            float* dst[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * NT;
                dst[u] = nullptr;
                if (i < total) {
                    const int row = i / per_row, k = i - row * per_row;
                    const bool first = row < m * K + 1;
                    int t = tok_s[first ? row : row - (m * K + 1)];
                    t = (t >= 0 && t < c.V) ? t : 0;
                    const float* src = (first ? W1 : W2) + (size_t)t * R;
                    dst[u] = (first ? w1s + (size_t)row * RP : w2s + (size_t)(row - (m * K + 1)) * RP);
                    if (vec) {
                        v[u] = reinterpret_cast<const float4*>(src)[k];
                        dst[u] += 4 * k;
                    } else {
                        v[u].x = src[k];
                        dst[u] += k;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (dst[u] == nullptr) continue;
                if (vec) *reinterpret_cast<float4*>(dst[u]) = v[u];
                else *dst[u] = v[u].x;
            }
        }
    }
    __syncthreads();

    // ---- A. tables: one row per lane group ------------------------------------------
    bad |= K <= 16 ? markov_fill<16>(c, R, RP, NT, w1s, w2s, tok_s, base_s, tb, xs)
                   : markov_fill<32>(c, R, RP, NT, w1s, w2s, tok_s, base_s, tb, xs);
    __syncthreads();
    for (int i = tid; i < E; i += NT) {
        const int cr = tb[i].crow;
        tb[i].first = cr >= 0 ? tb[(size_t)cr * K].edge : 0.0f;
    }
    if (__syncthreads_or(bad) && tid == 0) raise_status(ws, SPEC_DEV_BADLAT);
    if (warp != 0) return;

    // ---- B. best-first insertion: row x in lane x % 32, slot x / 32 ----------------
    int nd[SLOTS], nrow[SLOTS], nx[SLOTS], ntk[SLOTS], npar[SLOTS], nrk[SLOTS];
    float ns[SLOTS], cs[SLOTS];
    uint32_t co[SLOTS];
    uint64_t a0[SLOTS], a1[SLOTS];
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        nd[k] = 0; nrow[k] = -1; nx[k] = K; ntk[k] = -1; npar[k] = -1; nrk[k] = -1;
        ns[k] = 0.0f; cs[k] = 0.0f; co[k] = 0u; a0[k] = 0ull; a1[k] = 0ull;
    }
    if (lane == 0) {
        nrow[0] = 0; nx[0] = 0; ntk[0] = root; a0[0] = 1ull;
        cs[0] = __fadd_rn(0.0f, tb[0].edge);
        co[0] = ord_key(cs[0]);
    }
    int count = 1;
    while (count < T) {
        uint32_t bo = 0u, bt = 0u;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const uint32_t t = tie_rank(nd[k] + 1, lane + 32 * k);
            if (co[k] > bo || (co[k] == bo && co[k] != 0u && t > bt)) { bo = co[k]; bt = t; }
        }
        const uint32_t best_ord = __reduce_max_sync(0xffffffffu, bo);
        if (best_ord == 0u) break;                                  // frontier empty
        const uint32_t best_tie = __reduce_max_sync(0xffffffffu, bo == best_ord ? bt : 0u);
        const int pr = 255 - static_cast<int>(best_tie & 0xffu);    // parent row
        const int pl = pr & 31, pk = pr >> 5;
        const int n = count++;
        int d = 0, r = 0, rw = 0;
        float sc = 0.0f;
        uint64_t pa0 = 0ull, pa1 = 0ull;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k)
            if (k == pk) { d = nd[k]; r = nx[k]; rw = nrow[k]; sc = cs[k]; pa0 = a0[k]; pa1 = a1[k]; }
        d = __shfl_sync(0xffffffffu, d, pl);
        r = __shfl_sync(0xffffffffu, r, pl);
        rw = __shfl_sync(0xffffffffu, rw, pl);
        sc = __shfl_sync(0xffffffffu, sc, pl);
        pa0 = __shfl_sync(0xffffffffu, pa0, pl);
        pa1 = __shfl_sync(0xffffffffu, pa1, pl);
        // the offered child and the parent's next child: warp-uniform loads, both
        // in flight before either update
        const int ent = rw * K + r;
        const bool more = r + 1 < K;
        const MEnt ch = tb[ent];
        const float nxt = tb[more ? ent + 1 : ent].edge;
        const bool is_par = lane == pl, is_new = lane == (n & 31);
        const int nk = n >> 5;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            if (is_par && k == pk) {                                // the parent's next offer
                nx[k] = r + 1;
                cs[k] = __fadd_rn(ns[k], nxt);
                co[k] = more ? ord_key(cs[k]) : 0u;
            }
            if (is_new && k == nk) {                                // the new row
                nd[k] = d + 1; nrow[k] = ch.crow; nx[k] = 0; ns[k] = sc; npar[k] = pr; nrk[k] = r;
                ntk[k] = ch.tok;
                a0[k] = pa0 | (n < 64 ? 1ull << n : 0ull);
                a1[k] = pa1 | (n >= 64 ? 1ull << (n - 64) : 0ull);
                cs[k] = __fadd_rn(sc, ch.first);
                co[k] = ch.crow >= 0 ? ord_key(cs[k]) : 0u;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        const int x = lane + 32 * k;
        if (x < T) {
            const size_t o = (size_t)b * T + x;
            const bool used = x < count;
            out.node_tok[o] = used ? ntk[k] : -1;
            out.node_parent[o] = used ? npar[k] : -1;
            out.node_depth[o] = used ? nd[k] : -1;
            out.node_rank[o] = used ? nrk[k] : -1;
            out.node_score[o] = used ? ns[k] : 0.0f;
            out.node_anc[2 * o] = used ? a0[k] : 0ull;
            out.node_anc[2 * o + 1] = used ? a1[k] : 0ull;
        }
    }
    if (lane == 0) out.n_nodes[b] = count;
}

}  // namespace

size_t tree_markov_smem(const spec_cfg& c, int R) { return markov_smem(c.m, c.K, R); }

cudaError_t launch_tree_markov(const spec_cfg& c, const int32_t* lat_tok, const float* lat_base,
                               const float* W1, const float* W2, int R, const int32_t* root_tok,
                               const spec_tree& out, void* ws, cudaStream_t st, bool pdl) {
    const size_t smem = tree_markov_smem(c, R);
    if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
    const int T = c.N + 1;
    auto go = [&](auto kern, int nt) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        return launch_k(pdl, kern, dim3(c.B), dim3(nt), smem, st, c, R, lat_tok, lat_base, W1, W2,
                        root_tok, out, ws);
    };
    if (T <= 32) return go(tree_markov_kernel<1, kMarkovThreadsMax>, kMarkovThreadsMax);
    if (T <= 64) return go(tree_markov_kernel<2, kMarkovThreadsMax>, kMarkovThreadsMax);
    return go(tree_markov_kernel<4, kMarkovThreadsMax / 2>, kMarkovThreadsMax / 2);
}

}  // namespace spec
