// tree_build.cu -- best-first draft tree over a drafter lattice.
//
// Digest "SpecPilot: Autonomous Algorithm Discovery and Systems Optimization
// for Speculative Decoding": prerequisites / parallel drafter (the lattice of
// per-position top-k candidates and scores), prerequisites / draft-tree
// verification (nodes added greedily by root-path log-prob up to N) and
// technical novelty, Figure 6 (best-first tree, edges log p(child | parent)).
//
// One warp builds one request's tree entirely in shared memory.
//  1. Each lattice position is ranked in registers: lane r holds candidate r
//     and counts the candidates that precede it (score desc, index asc).
//  2. Because a position's ranked scores are non-increasing and fp32 addition
//     is monotone, the best remaining child of any inserted node is its
//     lowest not-yet-inserted rank.  The frontier is therefore one candidate
//     per inserted node ("next rank"), not K per node.
//  3. Every lane caches the best candidate among the nodes it owns
//     (row % 32 == lane); one iteration is two warp-wide REDUX max operations
//     (score, then depth/parent among equal scores), one insertion by lane 0,
//     and a re-scan by the two lanes whose nodes changed.
#include "common.cuh"
#include "kernels.h"

namespace spec {

// Order-preserving map of a finite float to uint32 (-0 folded into +0, since
// the two compare equal).
__device__ __forceinline__ uint32_t ord_f32(float f) {
    if (f == 0.0f) f = 0.0f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Among candidates with equal scores: smaller depth first, then smaller parent.
__device__ __forceinline__ uint32_t tie_key(int depth, int parent) {
    return ((uint32_t)(255 - depth) << 8) | (uint32_t)(255 - parent);
}

__global__ void __launch_bounds__(32)
tree_build_kernel(spec_cfg c, const int32_t* __restrict__ lat_tok,
                  const float* __restrict__ lat_score, const int32_t* __restrict__ root_tok,
                  spec_tree out, void* ws) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    const int m = c.m, K = c.K, T = c.N + 1;

    uint64_t* n_anc = reinterpret_cast<uint64_t*>(smem);          // [T][2]
    int32_t* s_tok = reinterpret_cast<int32_t*>(n_anc + 2 * T);    // [m][K] ranked tokens
    float* s_sc = reinterpret_cast<float*>(s_tok + m * K);         // [m][K] ranked scores
    int32_t* n_tok = reinterpret_cast<int32_t*>(s_sc + m * K);     // [T]
    int32_t* n_par = n_tok + T;
    int32_t* n_dep = n_par + T;
    int32_t* n_rank = n_dep + T;
    int32_t* n_next = n_rank + T;                                  // next child rank to offer
    float* n_sc = reinterpret_cast<float*>(n_next + T);
    int32_t* r_tok = reinterpret_cast<int32_t*>(n_sc + T);          // [m][K] as given
    float* r_sc = reinterpret_cast<float*>(r_tok + m * K);          // [m][K] as given

    // ---- 1. stage the lattice (one round trip), then rank every position -------
    for (int i = lane; i < m * K; i += kWarp) {
        r_tok[i] = lat_tok[(size_t)b * m * K + i];
        r_sc[i] = lat_score[(size_t)b * m * K + i];
    }
    __syncwarp();
    bool bad = false;
    for (int s = 0; s < m; ++s) {
        int tok = 0;
        float sc = 0.0f;
        if (lane < K) {
            tok = r_tok[s * K + lane];
            sc = r_sc[s * K + lane];
            bad |= (sc != sc);
        }
        int rank = 0;
        for (int j = 0; j < K; ++j) {
            const float sj = __shfl_sync(0xffffffffu, sc, j);
            const int tj = __shfl_sync(0xffffffffu, tok, j);
            if (lane < K && j != lane) {
                rank += (sj > sc || (sj == sc && j < lane)) ? 1 : 0;
                bad |= (tj == tok);
            }
        }
        if (lane < K && rank < K) {
            s_tok[s * K + rank] = tok;
            s_sc[s * K + rank] = sc;
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(ws, SPEC_DEV_BADLAT);

    // ---- 2./3. best-first insertion ------------------------------------------
    if (lane == 0) {
        n_tok[0] = root_tok[b];
        n_par[0] = -1;
        n_dep[0] = 0;
        n_rank[0] = -1;
        n_next[0] = 0;
        n_sc[0] = 0.0f;
        n_anc[0] = 1ull;
        n_anc[1] = 0ull;
    }
    __syncwarp();

    uint32_t my_ord = 0, my_tie = 0;   // cached best candidate of this lane's nodes
    auto rescan = [&](int count) {
        my_ord = 0;
        my_tie = 0;
        for (int x = lane; x < count; x += kWarp) {
            const int d = n_dep[x], r = n_next[x];
            if (d < m && r < K) {
                const uint32_t o = ord_f32(n_sc[x] + s_sc[d * K + r]);
                const uint32_t t = tie_key(d + 1, x);
                if (o > my_ord || (o == my_ord && t > my_tie)) {
                    my_ord = o;
                    my_tie = t;
                }
            }
        }
    };
    int count = 1;
    rescan(count);
    while (count < T) {
        const uint32_t best_ord = __reduce_max_sync(0xffffffffu, my_ord);
        if (best_ord == 0u) break;                                  // frontier empty
        const uint32_t best_tie =
            __reduce_max_sync(0xffffffffu, my_ord == best_ord ? my_tie : 0u);
        const int p = 255 - (int)(best_tie & 0xffu);
        const int n = count;
        if (lane == 0) {
            const int d = n_dep[p], r = n_next[p];
            n_tok[n] = s_tok[d * K + r];
            n_par[n] = p;
            n_dep[n] = d + 1;
            n_rank[n] = r;
            n_next[n] = 0;
            n_sc[n] = n_sc[p] + s_sc[d * K + r];
            n_anc[2 * n] = n_anc[2 * p];
            n_anc[2 * n + 1] = n_anc[2 * p + 1];
            n_anc[2 * n + (n >> 6)] |= 1ull << (n & 63);
            n_next[p] = r + 1;
        }
        __syncwarp();
        ++count;
        if ((p & 31) == lane || (n & 31) == lane) rescan(count);
    }
    __syncwarp();

    // ---- write the tree ----------------------------------------------------------
    for (int x = lane; x < T; x += kWarp) {
        const size_t o = (size_t)b * T + x;
        const bool used = x < count;
        out.node_tok[o] = used ? n_tok[x] : -1;
        out.node_parent[o] = used ? n_par[x] : -1;
        out.node_depth[o] = used ? n_dep[x] : -1;
        out.node_rank[o] = used ? n_rank[x] : -1;
        out.node_score[o] = used ? n_sc[x] : 0.0f;
        out.node_anc[2 * o] = used ? n_anc[2 * x] : 0ull;
        out.node_anc[2 * o + 1] = used ? n_anc[2 * x + 1] : 0ull;
    }
    if (lane == 0) out.n_nodes[b] = count;
}

size_t tree_build_smem(const spec_cfg& c) {
    const int T = c.N + 1;
    return sizeof(uint64_t) * 2 * T + 2 * (sizeof(int32_t) + sizeof(float)) * (size_t)c.m * c.K +
           (5 * sizeof(int32_t) + sizeof(float)) * (size_t)T;
}

cudaError_t launch_tree_build(const spec_cfg& c, const int32_t* lat_tok, const float* lat_score,
                              const int32_t* root_tok, const spec_tree& out, void* ws,
                              cudaStream_t st) {
    const size_t smem = tree_build_smem(c);
    tree_build_kernel<<<c.B, 32, smem, st>>>(c, lat_tok, lat_score, root_tok, out, ws);
    return cudaGetLastError();
}

}  // namespace spec
