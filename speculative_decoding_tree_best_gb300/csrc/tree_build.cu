// tree_build.cu -- best-first draft tree over a drafter lattice.
//
// Digest "SpecPilot: Autonomous Algorithm Discovery and Systems Optimization
// for Speculative Decoding": prerequisites / parallel drafter (the lattice of
// per-position top-k candidates and scores), prerequisites / draft-tree
// verification (nodes added greedily by root-path log-prob up to N) and
// technical novelty, Figure 6 (best-first tree, edges log p(child | parent)).
//
// One warp builds one request's tree.
//  1. Every candidate is ranked in registers, 32 / K positions per warp pass:
//     its rank is the number of candidates of its position that precede it
//     (score desc, index asc), counted over shuffles within the position.
//  2. Because a position's ranked scores are non-increasing and fp32 addition
//     is monotone, the best remaining child of an inserted node is its lowest
//     not-yet-inserted rank, so the frontier is one candidate per inserted row.
//  3. Row x lives in the registers of lane x % 32 (slot x / 32, T <= 128).
//     Each lane caches its best candidate; one insertion is two warp-wide
//     REDUX max operations (score, then depth/parent among equal scores), a
//     few shuffles from the parent's lane to the new row's lane, and a
//     re-scan of at most four slots by the two lanes whose rows changed.  The
//     edge scores a row will need next are prefetched from shared memory after
//     each insertion, so the chain from one insertion to the next has no
//     shared-memory load.
#include "common.cuh"
#include "kernels.h"

namespace spec {

namespace {


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

// SLOTS = rows per lane: ceil(T / 32), 1 to 4.
template <int SLOTS>
__global__ void __launch_bounds__(32)
tree_build_kernel(spec_cfg c, const int32_t* __restrict__ lat_tok,
                  const float* __restrict__ lat_score, const int32_t* __restrict__ root_tok,
                  spec_tree out, void* ws, const int32_t* __restrict__ m_req) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int b = blockIdx.x;
    const int lane = threadIdx.x;
    const int m = c.m, K = c.K, T = c.N + 1;
    const int MK = m * K;
    // depth limit of this request: m_req[b] lattice positions (all m when absent)
    int mb = m;
    if (m_req != nullptr) {
        mb = m_req[b];
        if (mb < 1 || mb > m) {
            if (lane == 0) raise_status(ws, SPEC_DEV_BADREQ);
            mb = mb < 1 ? 1 : m;
        }
    }

    int32_t* s_tok = reinterpret_cast<int32_t*>(smem);      // [m][K] ranked tokens
    float* s_sc = reinterpret_cast<float*>(s_tok + MK);      // [m][K] ranked edge scores
    int32_t* r_tok = reinterpret_cast<int32_t*>(s_sc + MK);  // [m][K] as given
    float* r_sc = reinterpret_cast<float*>(r_tok + MK);      // [m][K] as given

    // ---- 1. stage (one round trip), then rank: 32 / K2 positions per warp pass --------
    pdl_wait();          // the previous step's acceptance wrote root_tok
    pdl_trigger();
    const int root = root_tok[b];
    for (int i = lane; i < MK; i += 32) {
        r_tok[i] = lat_tok[(size_t)b * MK + i];
        r_sc[i] = lat_score[(size_t)b * MK + i];
    }
    __syncwarp();
    int K2 = 1;
    while (K2 < K) K2 <<= 1;
    const int ppp = 32 / K2;                                 // positions per pass
    const int sub = lane / K2, ci = lane % K2;
    bool bad = false;
    for (int s0 = 0; s0 < m; s0 += ppp) {
        const int s = s0 + sub;
        const bool valid = s < m && ci < K;
        const float sc = valid ? r_sc[s * K + ci] : 0.0f;
        const int tk = valid ? r_tok[s * K + ci] : 0;
        bad |= valid && (sc != sc);
        int rank = 0;
#pragma unroll 8
        for (int jj = 0; jj < K; ++jj) {
            const float sj = __shfl_sync(0xffffffffu, sc, jj, K2);
            const int tj = __shfl_sync(0xffffffffu, tk, jj, K2);
            rank += (sj > sc || (sj == sc && jj < ci)) ? 1 : 0;
            bad |= valid && jj != ci && tj == tk;
        }
        if (valid && rank < K) {
            s_tok[s * K + rank] = tk;
            s_sc[s * K + rank] = sc;
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(ws, SPEC_DEV_BADLAT);
    __syncwarp();

    // ---- 2./3. best-first insertion, rows in registers ----------------------------
    // Per slot: depth nd, offered rank nx, score ns, offered child score cs and
    // its order key co (0 = nothing offered), nxt = edge score of the rank after
    // the offered one, fst = first edge score of the next position (the first
    // child of any new child of this row); both prefetched off the critical path.
    int nd[SLOTS], nx[SLOTS], ntk[SLOTS], npar[SLOTS], nrk[SLOTS];
    float ns[SLOTS], cs[SLOTS], nxt[SLOTS], fst[SLOTS];
    uint32_t co[SLOTS];
    uint64_t a0[SLOTS], a1[SLOTS];
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        nd[k] = m; nx[k] = K; ntk[k] = -1; npar[k] = -1; nrk[k] = -1;
        ns[k] = 0.0f; cs[k] = 0.0f; nxt[k] = 0.0f; fst[k] = 0.0f; co[k] = 0u;
        a0[k] = 0ull; a1[k] = 0ull;
    }
    auto prefetch = [&](int k) {
        const int d = nd[k];
        nxt[k] = (d < mb && nx[k] + 1 < K) ? s_sc[d * K + nx[k] + 1] : 0.0f;
        fst[k] = (d + 1 < mb) ? s_sc[(d + 1) * K] : 0.0f;
    };
    uint32_t bo = 0, bt = 0;   // this lane's best candidate (ord, tie)
    auto best_of_lane = [&]() {
        bo = 0u;
        bt = 0u;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const uint32_t t = tie_key(nd[k] + 1, lane + 32 * k);
            if (co[k] > bo || (co[k] == bo && co[k] != 0u && t > bt)) { bo = co[k]; bt = t; }
        }
    };
    if (lane == 0) {   // row 0: the root
        nd[0] = 0; nx[0] = 0; ntk[0] = root; ns[0] = 0.0f; a0[0] = 1ull;
        if (m > 0 && K > 0) {
            cs[0] = 0.0f + s_sc[0];
            co[0] = ord_f32(cs[0]);
        }
        prefetch(0);
    }
    best_of_lane();
    int count = 1;
    if constexpr (SLOTS == 1) {
        // Trees of up to 32 rows: row x lives in lane x, and an insertion is pure
        // data movement by shuffles and selects (no divergent branch).
        uint32_t bo1 = co[0];
        uint32_t bt1 = tie_key(nd[0] + 1, lane);
        while (count < T) {
            const uint32_t best_ord = __reduce_max_sync(0xffffffffu, bo1);
            if (best_ord == 0u) break;                              // frontier empty
            const uint32_t best_tie = __reduce_max_sync(0xffffffffu, bo1 == best_ord ? bt1 : 0u);
            const int p = 255 - (int)(best_tie & 0xffu);
            const int n = count++;
            const int d = __shfl_sync(0xffffffffu, nd[0], p);
            const int r = __shfl_sync(0xffffffffu, nx[0], p);
            const float sc = __shfl_sync(0xffffffffu, cs[0], p);
            const float fe = __shfl_sync(0xffffffffu, fst[0], p);
            const bool isp = lane == p, isn = lane == n;
            const float cs_p = ns[0] + nxt[0];
            const uint32_t co_p = (r + 1 < K) ? ord_f32(cs_p) : 0u;
            const float cs_n = sc + fe;
            const uint32_t co_n = (d + 1 < mb) ? ord_f32(cs_n) : 0u;
            nx[0] = isp ? r + 1 : (isn ? 0 : nx[0]);
            nd[0] = isn ? d + 1 : nd[0];
            ns[0] = isn ? sc : ns[0];
            npar[0] = isn ? p : npar[0];
            nrk[0] = isn ? r : nrk[0];
            cs[0] = isp ? cs_p : (isn ? cs_n : cs[0]);
            co[0] = isp ? co_p : (isn ? co_n : co[0]);
            bo1 = co[0];
            bt1 = tie_key(nd[0] + 1, lane);
            // off the critical path: ancestors, token, prefetched edge scores
            const uint64_t pa0 = __shfl_sync(0xffffffffu, a0[0], p);
            const uint64_t pa1 = __shfl_sync(0xffffffffu, a1[0], p);
            const int tkn = s_tok[d * K + r];
            a0[0] = isn ? (pa0 | (n < 64 ? 1ull << n : 0ull)) : a0[0];
            a1[0] = isn ? (pa1 | (n >= 64 ? 1ull << (n - 64) : 0ull)) : a1[0];
            ntk[0] = isn ? tkn : ntk[0];
            const int dd = nd[0];
            const int i_nxt = (dd < mb && nx[0] + 1 < K) ? dd * K + nx[0] + 1 : 0;
            const int i_fst = (dd + 1 < mb) ? (dd + 1) * K : 0;
            nxt[0] = s_sc[i_nxt];
            fst[0] = s_sc[i_fst];
        }
    } else {
        // Larger trees: row x lives in slot x / 32 of lane x % 32.  The same
        // branch-free step over every slot of every lane: the parent's slot is
        // picked by selects (its index is warp-uniform) before the shuffles.
        while (count < T) {
            const uint32_t best_ord = __reduce_max_sync(0xffffffffu, bo);
            if (best_ord == 0u) break;                              // frontier empty
            const uint32_t best_tie = __reduce_max_sync(0xffffffffu, bo == best_ord ? bt : 0u);
            const int p = 255 - (int)(best_tie & 0xffu);
            const int n = count++;
            const int pl = p & 31, pk = p >> 5, nl = n & 31, nk = n >> 5;
            int d = nd[0], r = nx[0];
            float sc = cs[0], fe = fst[0];
            uint64_t pa0 = a0[0], pa1 = a1[0];
#pragma unroll
            for (int k = 1; k < SLOTS; ++k) {
                const bool sel = k == pk;
                d = sel ? nd[k] : d;
                r = sel ? nx[k] : r;
                sc = sel ? cs[k] : sc;
                fe = sel ? fst[k] : fe;
                pa0 = sel ? a0[k] : pa0;
                pa1 = sel ? a1[k] : pa1;
            }
            d = __shfl_sync(0xffffffffu, d, pl);
            r = __shfl_sync(0xffffffffu, r, pl);
            sc = __shfl_sync(0xffffffffu, sc, pl);
            fe = __shfl_sync(0xffffffffu, fe, pl);
            const float cs_n = sc + fe;
            const uint32_t co_n = (d + 1 < mb) ? ord_f32(cs_n) : 0u;
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const bool isp = lane == pl && k == pk, isn = lane == nl && k == nk;
                const float cs_p = ns[k] + nxt[k];
                const uint32_t co_p = (r + 1 < K) ? ord_f32(cs_p) : 0u;
                nx[k] = isp ? r + 1 : (isn ? 0 : nx[k]);
                nd[k] = isn ? d + 1 : nd[k];
                ns[k] = isn ? sc : ns[k];
                npar[k] = isn ? p : npar[k];
                nrk[k] = isn ? r : nrk[k];
                cs[k] = isp ? cs_p : (isn ? cs_n : cs[k]);
                co[k] = isp ? co_p : (isn ? co_n : co[k]);
            }
            best_of_lane();
            // off the critical path: ancestors, token, the changed slots' edge scores
            pa0 = __shfl_sync(0xffffffffu, pa0, pl);
            pa1 = __shfl_sync(0xffffffffu, pa1, pl);
            const int tkn = s_tok[d * K + r];
            // slot pk of lane pl and slot nk of lane nl changed (the same lane
            // when p and n are 32 apart); each lane reloads both candidates
            int dp = nd[0], xp = nx[0], dn = nd[0], xn = nx[0];
#pragma unroll
            for (int k = 1; k < SLOTS; ++k) {
                dp = k == pk ? nd[k] : dp;
                xp = k == pk ? nx[k] : xp;
                dn = k == nk ? nd[k] : dn;
                xn = k == nk ? nx[k] : xn;
            }
            const float nxt_p = s_sc[(dp < mb && xp + 1 < K) ? dp * K + xp + 1 : 0];
            const float fst_p = s_sc[(dp + 1 < mb) ? (dp + 1) * K : 0];
            const float nxt_n = s_sc[(dn < mb && xn + 1 < K) ? dn * K + xn + 1 : 0];
            const float fst_n = s_sc[(dn + 1 < mb) ? (dn + 1) * K : 0];
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const bool isp = lane == pl && k == pk, isn = lane == nl && k == nk;
                a0[k] = isn ? (pa0 | (n < 64 ? 1ull << n : 0ull)) : a0[k];
                a1[k] = isn ? (pa1 | (n >= 64 ? 1ull << (n - 64) : 0ull)) : a1[k];
                ntk[k] = isn ? tkn : ntk[k];
                nxt[k] = isn ? nxt_n : (isp ? nxt_p : nxt[k]);
                fst[k] = isn ? fst_n : (isp ? fst_p : fst[k]);
            }
        }
    }

    // ---- write the tree ----------------------------------------------------------
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

// A node budget shared by the batch (digest, technical novelty: batching
// shares one node budget across requests).  Each request's tree was built
// best-first up to N drafts; the batch keeps the `budget` drafts first in the
// order (score desc, request asc, index asc), which is the best-first order
// over all frontiers together, and every request keeps a prefix of its own
// insertion order.  A draft's place in that order is its index within its
// request plus, for every other request, the count of that request's drafts
// that precede it (a binary search: a request's scores never increase along
// its insertion order).  One CTA; rows past a request's kept drafts become
// padding rows.
__global__ void __launch_bounds__(1024)
budget_select(spec_cfg c, spec_tree t, int budget) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int B = c.B, T = c.N + 1, N = c.N;
    float* s_sc = reinterpret_cast<float*>(smem);               // [B][T] scores
    int* s_n = reinterpret_cast<int*>(s_sc + (size_t)B * T);    // [B] rows built
    int* s_keep = s_n + B;                                      // [B] drafts kept
    pdl_wait();                  // the trees come from the launch just before
    pdl_trigger();
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int n = t.n_nodes[b];
        s_n[b] = n < 1 ? 1 : (n > T ? T : n);
        s_keep[b] = 0;
    }
    for (int i = threadIdx.x; i < B * T; i += blockDim.x) s_sc[i] = t.node_score[i];
    __syncthreads();
    for (int cand = threadIdx.x; cand < B * N; cand += blockDim.x) {
        const int b = cand / N, i = 1 + cand % N;
        if (i >= s_n[b]) continue;
        const float s = s_sc[b * T + i];
        int rank = i - 1;
        for (int b2 = 0; b2 < B && rank < budget; ++b2) {
            if (b2 == b) continue;
            // drafts of b2 before this one: score > s, or score == s when b2 < b
            const float* a = s_sc + b2 * T;
            int lo = 1, hi = s_n[b2];           // first j in [1, n) not preceding
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                const bool before = a[mid] > s || (a[mid] == s && b2 < b);
                if (before) lo = mid + 1; else hi = mid;
            }
            rank += lo - 1;
        }
        if (rank < budget) atomicMax(&s_keep[b], i);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < B * T; i += blockDim.x) {
        const int b = i / T, x = i % T;
        if (x > s_keep[b] && x < s_n[b]) {
            t.node_tok[i] = -1;
            t.node_parent[i] = -1;
            t.node_depth[i] = -1;
            t.node_rank[i] = -1;
            t.node_score[i] = 0.0f;
            t.node_anc[2 * (size_t)i] = 0ull;
            t.node_anc[2 * (size_t)i + 1] = 0ull;
        }
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) t.n_nodes[b] = 1 + s_keep[b];
}

}  // namespace

size_t tree_build_smem(const spec_cfg& c) {
    return 2 * (sizeof(int32_t) + sizeof(float)) * (size_t)c.m * c.K;
}

cudaError_t launch_tree_build(const spec_cfg& c, const int32_t* lat_tok, const float* lat_score,
                              const int32_t* root_tok, const spec_tree& out, void* ws,
                              cudaStream_t st, bool pdl, const int32_t* m_req) {
    const size_t smem = tree_build_smem(c);
    const int T = c.N + 1;
    if (T <= 32)
        return launch_k(pdl, tree_build_kernel<1>, dim3(c.B), dim3(32), smem, st, c, lat_tok,
                        lat_score, root_tok, out, ws, m_req);
    if (T <= 64)
        return launch_k(pdl, tree_build_kernel<2>, dim3(c.B), dim3(32), smem, st, c, lat_tok,
                        lat_score, root_tok, out, ws, m_req);
    if (T <= 96)
        return launch_k(pdl, tree_build_kernel<3>, dim3(c.B), dim3(32), smem, st, c, lat_tok,
                        lat_score, root_tok, out, ws, m_req);
    return launch_k(pdl, tree_build_kernel<4>, dim3(c.B), dim3(32), smem, st, c, lat_tok,
                    lat_score, root_tok, out, ws, m_req);
}

size_t budget_select_smem(const spec_cfg& c) {
    return sizeof(float) * (size_t)c.B * (c.N + 1) + 2 * sizeof(int) * (size_t)c.B;
}

cudaError_t launch_budget_select(const spec_cfg& c, const spec_tree& out, int budget,
                                 cudaStream_t st, bool pdl) {
    const size_t smem = budget_select_smem(c);
    if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(budget_select,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_k(pdl, budget_select, dim3(1), dim3(1024), smem, st, c, out, budget);
}

}  // namespace spec
