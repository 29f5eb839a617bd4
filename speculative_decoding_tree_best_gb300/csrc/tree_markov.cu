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
// One CTA of 256 threads per request.
//  A. All warps fill the tables.  A table row is (position d, parent): the
//     root for d = 0, candidate p of position d-1 otherwise, so row
//     rho = 0 or 1 + (d-1) K + p.  A group of lanes computes one row: lane i
//     the dot product and l_i, the group the maximum, lane 0 the ordered sum
//     and the log-sum-exp, each lane its edge and its rank.  Per entry
//     (row, rank): edge, token, the row of that child's own children, and
//     the first (best) edge among them.
//  B. Warp 0 inserts nodes best-first exactly as tree_build.cu does, row x in
//     lane x % 32, slot x / 32.  Each row offers its best remaining child; the
//     offers are compared with two warp-wide max reductions (key, then depth
//     and parent among equal keys).  The child lookups go through the row's
//     table row instead of a position's ranked list.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace spec {

namespace {

constexpr int kMarkovThreads = 256;

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

struct MarkovTables {
    float* edge;      // [rows][K] edge score by rank
    int32_t* tok;     // [rows][K] token by rank
    int16_t* crow;    // [rows][K] table row of that child's children (-1: none)
    float* first;     // [rows][K] the first edge among that child's children (0: none)
};

__host__ __device__ inline size_t markov_rows(int m, int K) { return 1 + (size_t)(m - 1) * K; }

__host__ __device__ inline size_t markov_smem(int m, int K) {
    const size_t e = markov_rows(m, K) * K;
    return e * (4 + 4 + 4) + ((e * 2 + 15) & ~size_t(15));
}

template <int SLOTS>
__global__ void __launch_bounds__(kMarkovThreads)
tree_markov_kernel(spec_cfg c, int R, const int32_t* __restrict__ lat_tok,
                   const float* __restrict__ lat_base, const float* __restrict__ W1,
                   const float* __restrict__ W2, const int32_t* __restrict__ root_tok,
                   spec_tree out, void* ws) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = c.m, K = c.K, T = c.N + 1;
    const size_t E = markov_rows(m, K) * K;
    MarkovTables tb;
    tb.edge = reinterpret_cast<float*>(smem);
    tb.tok = reinterpret_cast<int32_t*>(tb.edge + E);
    tb.first = reinterpret_cast<float*>(tb.tok + E);
    tb.crow = reinterpret_cast<int16_t*>(tb.first + E);
    const int32_t* tok_b = lat_tok + (size_t)b * m * K;
    const float* base_b = lat_base + (size_t)b * m * K;

    pdl_wait();          // root_tok may come from the previous step's acceptance
    pdl_trigger();
    const int root = root_tok[b];

    // ---- A. tables: one row per lane group of G lanes ------------------------------
    const int G = K <= 16 ? 16 : 32;
    const int groups = (kMarkovThreads / 32) * (32 / G);
    const int grp = warp * (32 / G) + lane / G, gl = lane % G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (0xffffu << (lane & 16));
    const int nrows = (int)markov_rows(m, K);
    bool bad = false;
    for (int rho0 = 0; rho0 < nrows; rho0 += groups) {
        const int rho = rho0 + grp;
        const bool live = rho < nrows;
        const int d = rho == 0 ? 0 : 1 + (rho - 1) / K;
        const int p = rho == 0 ? 0 : (rho - 1) % K;
        const int x = rho == 0 ? root : (live ? tok_b[(d - 1) * K + p] : 0);
        const bool act = live && gl < K;
        const int y = act ? tok_b[d * K + gl] : 0;
        float l = -INFINITY;
        if (act) {
            float dot = 0.0f;
            const float* w1 = W1 + (size_t)x * R;
            const float* w2 = W2 + (size_t)y * R;
            for (int k = 0; k < R; ++k) dot = __fmaf_rn(w1[k], w2[k], dot);
            l = __fadd_rn(base_b[d * K + gl], dot);
        }
        float M = l;
        for (int o = G / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(gmask, M, o, G));
        const float ex = act ? exp32(__fsub_rn(l, M)) : 0.0f;
        float Z = 0.0f;
        for (int j = 0; j < K; ++j) Z = __fadd_rn(Z, __shfl_sync(gmask, ex, j, G));
        const float lse = __fadd_rn(M, log32(Z));
        const float e = __fsub_rn(l, lse);
        int rank = 0;
        for (int j = 0; j < K; ++j) {
            const float ej = __shfl_sync(gmask, e, j, G);
            rank += (ej > e || (ej == e && j < gl)) ? 1 : 0;
        }
        if (act) {
            tb.edge[(size_t)rho * K + rank] = e;
            tb.tok[(size_t)rho * K + rank] = y;
            // the child's own children: row 1 + d K + (candidate index)
            tb.crow[(size_t)rho * K + rank] = static_cast<int16_t>(d + 1 < m ? 1 + d * K + gl : -1);
        }
        bad |= act && !(e == e);           // a NaN base or weight
    }
    __syncthreads();
    for (size_t i = tid; i < E; i += kMarkovThreads) {
        const int cr = tb.crow[i];
        tb.first[i] = cr >= 0 ? tb.edge[(size_t)cr * K] : 0.0f;
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
        cs[0] = __fadd_rn(0.0f, tb.edge[0]);
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
        const size_t ent = (size_t)rw * K + r;                      // the offered child
        if (lane == pl) {                                           // the parent's next offer
#pragma unroll
            for (int k = 0; k < SLOTS; ++k)
                if (k == pk) {
                    nx[k] = r + 1;
                    if (r + 1 < K) {
                        cs[k] = __fadd_rn(ns[k], tb.edge[ent + 1]);
                        co[k] = ord_key(cs[k]);
                    } else {
                        co[k] = 0u;
                    }
                }
        }
        if (lane == (n & 31)) {                                     // the new row
            const int nk = n >> 5;
            const int crow = tb.crow[ent];
#pragma unroll
            for (int k = 0; k < SLOTS; ++k)
                if (k == nk) {
                    nd[k] = d + 1; nrow[k] = crow; nx[k] = 0; ns[k] = sc; npar[k] = pr; nrk[k] = r;
                    ntk[k] = tb.tok[ent];
                    a0[k] = pa0 | (n < 64 ? 1ull << n : 0ull);
                    a1[k] = pa1 | (n >= 64 ? 1ull << (n - 64) : 0ull);
                    if (crow >= 0) {
                        cs[k] = __fadd_rn(sc, tb.first[ent]);
                        co[k] = ord_key(cs[k]);
                    } else {
                        co[k] = 0u;
                    }
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

size_t tree_markov_smem(const spec_cfg& c) { return markov_smem(c.m, c.K); }

cudaError_t launch_tree_markov(const spec_cfg& c, const int32_t* lat_tok, const float* lat_base,
                               const float* W1, const float* W2, int R, const int32_t* root_tok,
                               const spec_tree& out, void* ws, cudaStream_t st, bool pdl) {
    const size_t smem = tree_markov_smem(c);
    if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
    const int T = c.N + 1;
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        return launch_k(pdl, kern, dim3(c.B), dim3(kMarkovThreads), smem, st, c, R, lat_tok,
                        lat_base, W1, W2, root_tok, out, ws);
    };
    if (T <= 32) return go(tree_markov_kernel<1>);
    if (T <= 64) return go(tree_markov_kernel<2>);
    return go(tree_markov_kernel<4>);
}

}  // namespace spec
