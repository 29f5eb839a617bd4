// gdn_tree.cu -- tree-masked Gated DeltaNet: every tree row's output with its
// state recomputed along its root path from the committed state.
//
// Digest "SpecPilot ...": prerequisites / hybrid recurrent target (gated delta
// rule h_t = a_t (I - b_t k_t k_t^T) h_{t-1} + b_t k_t v_t^T, o_t = h_t^T q_t)
// and technical novelty (recompute along the root path, no per-node
// snapshots of the d_k x d_v state).
//
// Formulation.  Writing c_t = b_t v_t - a_t b_t u_t with u_t = h_par^T k_t,
// one step is h_t = a_t h_par + k_t c_t^T, so along a root path
//     h_x = A_x h0 + sum_{a on path(x)} dec(a -> x) k_a c_a^T,
// with A_x the product of alpha over path(x) and dec(a -> x) the product of
// alpha over the nodes after a on path(x).  Hence
//     u_x = A_par Pk_x + sum_{a on path(par)} dec(a -> par) (k_a . k_x) c_a
//     o_x = A_x   Pq_x + sum_{a on path(x)}   dec(a -> x)   (k_a . q_x) c_a
// where Pk_x = h0^T k_x and Pq_x = h0^T q_x.  The only d_k x d_v work is the
// skinny product h0^T [K; Q] over all rows; every c_a is computed once and
// shared by all descendants of a (the root-path prefix sharing), and no
// d_k x d_v state is ever written.
//
// Every column of the state evolves independently, so a CTA owns 32 columns
// of one (request, v-head) state: it stages that 32-column slice of h0 in
// shared memory once, and all arithmetic is fp32.
#include "common.cuh"
#include "kernels.h"

namespace spec {

namespace {

constexpr int CB = 32;       // state columns per CTA
constexpr int NT = 256;      // threads per CTA (8 warps)
constexpr int NG = NT / 32;  // warps = row groups
constexpr int kChainMax = 17;  // per-thread chains for root paths of up to 17 rows (m <= 16)

// 16 bytes of I/O elements -> floats (8 bf16 or 4 fp32).
template <int IO>
__device__ __forceinline__ void unpack16(const uint4& u, float* f);
template <>
__device__ __forceinline__ void unpack16<SPEC_IO_BF16>(const uint4& u, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(h[e]);
        f[2 * e] = x.x;
        f[2 * e + 1] = x.y;
    }
}
template <>
__device__ __forceinline__ void unpack16<SPEC_IO_F32>(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}

struct GdnSmem {
    // offsets in floats/ints (4-byte words) from the start of dynamic smem
    int hs, kq, P, cv, vs, al, be, A, Ap, par, dep, pidx, wu, wo, total;
    int S;  // path slots per row
};

__host__ __device__ inline GdnSmem gdn_smem_layout(int T, int m, int DK) {
    GdnSmem L;
    int S = (m < T - 1 ? m : T - 1) + 1;
    L.S = S;
    int o = 0;
    L.hs = o;  o += DK * CB;
    L.kq = o;  o += 2 * T * (DK + 4);     // rows padded by 16 B: no bank conflicts across rows
    L.P = o;   o += 2 * T * CB;
    L.cv = o;  o += T * CB;
    L.vs = o;  o += T * CB;
    L.al = o;  o += T;
    L.be = o;  o += T;
    L.A = o;   o += T;
    L.Ap = o;  o += T;
    L.par = o; o += T;
    L.dep = o; o += T;
    L.pidx = o; o += T * S;
    L.wu = o;  o += T * S;
    L.wo = o;  o += T * S;
    L.total = o;
    return L;
}

// MAXD > 0: trees whose root paths hold at most MAXD rows use per-thread
// chains; MAXD == 0: level-synchronous recursion for deeper trees.
template <int IO, int DK, int MAXD>
__global__ void __launch_bounds__(NT)
gdn_tree_kernel(spec_cfg c, spec_tree tree, const float* __restrict__ h0,
                const typename io_t<IO>::T* __restrict__ q, const typename io_t<IO>::T* __restrict__ k,
                const typename io_t<IO>::T* __restrict__ v, const float* __restrict__ alpha,
                const float* __restrict__ beta, typename io_t<IO>::T* __restrict__ o,
                float* __restrict__ c_out, bool early) {
    extern __shared__ __align__(16) float sm[];
    const int T = c.N + 1, Hv = c.Hv, Hk = c.Hk, dv = c.dv;
    const int c0 = blockIdx.x * CB, j = blockIdx.y, b = blockIdx.z;
    const int ih = j / (Hv / Hk);
    const int tid = threadIdx.x, col = tid & 31, grp = tid >> 5;
    const GdnSmem L = gdn_smem_layout(T, c.m, DK);
    const int S = L.S;
    constexpr int KQS = DK + 4;             // k/q row stride in floats
    float* hs = sm + L.hs;
    float* kq = sm + L.kq;
    float* P = sm + L.P;
    float* cv = sm + L.cv;
    float* vs = sm + L.vs;
    float* al = sm + L.al;
    float* be = sm + L.be;
    float* A = sm + L.A;
    float* Ap = sm + L.Ap;
    int* par = reinterpret_cast<int*>(sm + L.par);
    int* dep = reinterpret_cast<int*>(sm + L.dep);
    int* pidx = reinterpret_cast<int*>(sm + L.pidx);
    float* wu = sm + L.wu;
    float* wo = sm + L.wo;

    // ---- before the tree exists: stage h0 slice, k/q/v rows and gates of all T
    // rows, then P = h0_slice^T [K; Q].  (Rows beyond the tree are padding and
    // their results are never used.)  Every global load of the first round is
    // issued into registers before any shared-memory store, so the CTA pays one
    // memory round trip, not one per loop iteration.
    using E = typename io_t<IO>::T;
    constexpr int HQ = DK * (CB / 4) / NT;           // h0 float4 per thread
    constexpr int KQR = 8;                           // k/q 16-byte chunks per thread per round
    constexpr int EPC = 16 / sizeof(E);              // elements per 16-byte chunk
    constexpr int KQC = DK / EPC;                    // chunks per k/q row
    constexpr int VC = CB / EPC;                     // chunks per v row slice
    const float* hsrc = h0 + ((size_t)b * Hv + j) * DK * dv + c0;
    float4 hreg[HQ];
#pragma unroll
    for (int i = 0; i < HQ; ++i) {
        const int idx = tid + i * NT, r = idx / (CB / 4), q4 = idx % (CB / 4);
        hreg[i] = *reinterpret_cast<const float4*>(hsrc + (size_t)r * dv + q4 * 4);
    }
    float t_al = 0.f, t_be = 0.f;
    if (tid < T) {
        t_al = alpha[((size_t)b * T + tid) * Hv + j];
        t_be = beta[((size_t)b * T + tid) * Hv + j];
    }
    uint4 vreg = make_uint4(0, 0, 0, 0);
    const bool has_v = tid < T * VC;
    if (has_v) {
        const int x = tid / VC, e0 = (tid % VC) * EPC;
        vreg = *reinterpret_cast<const uint4*>(v + (((size_t)b * T + x) * Hv + j) * dv + c0 + e0);
    }
    const int nkq = 2 * T * KQC;
    for (int base = 0; base < nkq; base += NT * KQR) {
        uint4 kreg[KQR];
#pragma unroll
        for (int i = 0; i < KQR; ++i) {
            const int idx = base + tid + i * NT;
            if (idx < nkq) {
                const int row = idx / KQC, ch = idx % KQC;
                const int x = row < T ? row : row - T;
                kreg[i] = *reinterpret_cast<const uint4*>(
                    (row < T ? k : q) + (((size_t)b * T + x) * Hk + ih) * DK + ch * EPC);
            }
        }
#pragma unroll
        for (int i = 0; i < KQR; ++i) {
            const int idx = base + tid + i * NT;
            if (idx < nkq) {
                const int row = idx / KQC, ch = idx % KQC;
                float f[EPC];
                unpack16<IO>(kreg[i], f);
#pragma unroll
                for (int e = 0; e < EPC; e += 4)
                    *reinterpret_cast<float4*>(kq + row * KQS + ch * EPC + e) =
                        make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < HQ; ++i) {
        const int idx = tid + i * NT, r = idx / (CB / 4), q4 = idx % (CB / 4);
        *reinterpret_cast<float4*>(hs + r * CB + q4 * 4) = hreg[i];
    }
    if (tid < T) {
        al[tid] = t_al;
        be[tid] = t_be;
    }
    if (has_v) {
        const int x = tid / VC, e0 = (tid % VC) * EPC;
        float f[EPC];
        unpack16<IO>(vreg, f);
#pragma unroll
        for (int e = 0; e < EPC; ++e) vs[x * CB + e0 + e] = f[e];
    }
    for (int x = NT + tid; x < T; x += NT) {       // more rows than threads
        al[x] = alpha[((size_t)b * T + x) * Hv + j];
        be[x] = beta[((size_t)b * T + x) * Hv + j];
    }
    for (int idx = NT + tid; idx < T * VC; idx += NT) {
        const int x = idx / VC, e0 = (idx % VC) * EPC;
        float f[EPC];
        unpack16<IO>(*reinterpret_cast<const uint4*>(v + (((size_t)b * T + x) * Hv + j) * dv + c0 + e0), f);
#pragma unroll
        for (int e = 0; e < EPC; ++e) vs[x * CB + e0 + e] = f[e];
    }
    __syncthreads();

    // ---- P = h0_slice^T [K; Q]: rows t = grp + 8 i, column col ------------------------
    for (int t0 = 0; t0 < 2 * T; t0 += 8 * NG) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int r = 0; r < DK; r += 4) {
            const float h_0 = hs[(r + 0) * CB + col], h_1 = hs[(r + 1) * CB + col];
            const float h_2 = hs[(r + 2) * CB + col], h_3 = hs[(r + 3) * CB + col];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = t0 + grp + NG * i;
                if (t < 2 * T) {
                    const float4 kk = *reinterpret_cast<const float4*>(kq + t * KQS + r);
                    acc[i] = fmaf(h_0, kk.x, fmaf(h_1, kk.y, fmaf(h_2, kk.z, fmaf(h_3, kk.w, acc[i]))));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = t0 + grp + NG * i;
            if (t < 2 * T) P[t * CB + col] = acc[i];
        }
    }

    // ---- the tree from here on.  early: it may come from the launch just before
    // this one; otherwise it is at least two launches back and no wait is needed
    // until the end.
    if (early) {
        pdl_wait();
        pdl_trigger();
    }
    int nn = tree.n_nodes[b];
    nn = nn < 1 ? 1 : (nn > T ? T : nn);     // a malformed tree must not index out of range
    for (int x = tid; x < nn; x += NT) {
        const int pp = tree.node_parent[(size_t)b * T + x];
        const int d = tree.node_depth[(size_t)b * T + x];
        par[x] = (pp >= 0 && pp < x) ? pp : -1;
        dep[x] = d < 0 ? 0 : (d >= S ? S - 1 : d);
    }
    __syncthreads();

    // ---- root paths and decay products (one thread per row) ------------------------
    for (int x = tid; x < nn; x += NT) {
        const int d = dep[x];
        int y = x;
        for (int s = d; s >= 0; --s) { pidx[x * S + s] = y; y = par[y] < 0 ? 0 : par[y]; }
        float acc = 1.0f;                       // dec(path[s] -> x)
        for (int s = d; s >= 0; --s) { wo[x * S + s] = acc; acc *= al[pidx[x * S + s]]; }
        A[x] = acc;
        acc = 1.0f;                             // dec(path[s] -> parent)
        for (int s = d - 1; s >= 0; --s) { wu[x * S + s] = acc; acc *= al[pidx[x * S + s]]; }
        Ap[x] = acc;
    }
    __syncthreads();

    // ---- Gram weights: wo *= k_a . q_x, wu *= k_a . k_x (one thread per pair) ---------
    for (int idx = tid; idx < nn * S; idx += NT) {
        const int x = idx / S, s = idx - x * S;
        const int d = dep[x];
        if (s > d) continue;
        const float4* ka = reinterpret_cast<const float4*>(kq + pidx[x * S + s] * KQS);
        const float4* kx = reinterpret_cast<const float4*>(kq + x * KQS);
        const float4* qx = reinterpret_cast<const float4*>(kq + (T + x) * KQS);
        float dq0 = 0.f, dq1 = 0.f, dk0 = 0.f, dk1 = 0.f;
#pragma unroll 8
        for (int e = 0; e < DK / 4; e += 2) {
            const float4 a0 = ka[e], a1 = ka[e + 1];
            const float4 q0 = qx[e], q1 = qx[e + 1];
            const float4 k0 = kx[e], k1 = kx[e + 1];
            dq0 = fmaf(a0.x, q0.x, fmaf(a0.y, q0.y, fmaf(a0.z, q0.z, fmaf(a0.w, q0.w, dq0))));
            dq1 = fmaf(a1.x, q1.x, fmaf(a1.y, q1.y, fmaf(a1.z, q1.z, fmaf(a1.w, q1.w, dq1))));
            dk0 = fmaf(a0.x, k0.x, fmaf(a0.y, k0.y, fmaf(a0.z, k0.z, fmaf(a0.w, k0.w, dk0))));
            dk1 = fmaf(a1.x, k1.x, fmaf(a1.y, k1.y, fmaf(a1.z, k1.z, fmaf(a1.w, k1.w, dk1))));
        }
        wo[x * S + s] *= dq0 + dq1;
        if (s < d) wu[x * S + s] *= dk0 + dk1;
    }

    __syncthreads();

    if constexpr (MAXD > 0) {
        // ---- write vectors and outputs, one (row, column) chain per thread ------------
        // Thread (x, col) walks x's root path y_0 = root .. y_d = x and rebuilds
        // c_{y_s} = beta v - alpha beta (A_par Pk + sum_{s'<s} wu[y_s][s'] c_{y_s'})
        // in registers; y_s's ancestors are y_0 .. y_{s-1}, so its weights are
        // indexed by the same path positions.  Work is redundant across
        // siblings (shorter than one barrier per tree level at these depths).
        for (int x = grp; x < T; x += NG) {
            float ox = 0.0f, cx = 0.0f;
            if (x < nn) {
                const int d = dep[x];
                float cc[MAXD];
                ox = A[x] * P[(T + x) * CB + col];
#pragma unroll
                for (int s = 0; s < MAXD; ++s) {
                    if (s > d) break;
                    const int y = pidx[x * S + s];
                    float u = Ap[y] * P[y * CB + col];
#pragma unroll
                    for (int s2 = 0; s2 < s; ++s2) u = fmaf(wu[y * S + s2], cc[s2], u);
                    cc[s] = be[y] * vs[y * CB + col] - al[y] * be[y] * u;
                    ox = fmaf(wo[x * S + s], cc[s], ox);
                    cx = cc[s];
                }
            }
            const size_t oi = (((size_t)b * T + x) * Hv + j) * dv + c0 + col;
            io_t<IO>::st(o, oi, ox);
            if (c_out) c_out[oi] = cx;
        }
        if (!early) {
            pdl_wait();
            pdl_trigger();
        }
        return;
    }

    // ---- write vectors c_x, level by level (ancestors first) --------------------------
    const int maxd = c.m < nn - 1 ? c.m : nn - 1;
    for (int d = 0; d <= maxd; ++d) {
        for (int x = grp; x < nn; x += NG) {
            if (dep[x] != d) continue;
            float u = Ap[x] * P[x * CB + col];
            for (int s = 0; s < d; ++s) u = fmaf(wu[x * S + s], cv[pidx[x * S + s] * CB + col], u);
            cv[x * CB + col] = be[x] * vs[x * CB + col] - al[x] * be[x] * u;
        }
        __syncthreads();
    }

    // ---- outputs -------------------------------------------------------------------
    for (int x = grp; x < T; x += NG) {
        float ox = 0.0f, cx = 0.0f;
        if (x < nn) {
            ox = A[x] * P[(T + x) * CB + col];
            const int d = dep[x];
            for (int s = 0; s <= d; ++s) ox = fmaf(wo[x * S + s], cv[pidx[x * S + s] * CB + col], ox);
            cx = cv[x * CB + col];
        }
        const size_t oi = (((size_t)b * T + x) * Hv + j) * dv + c0 + col;
        io_t<IO>::st(o, oi, ox);
        if (c_out) c_out[oi] = cx;
    }
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }
}

template <int IO, int DK, int MAXD>
cudaError_t launch_one(const spec_cfg& c, const spec_tree& t, const float* h0, const void* q,
                       const void* k, const void* v, const float* alpha, const float* beta,
                       void* o, float* c_out, size_t smem, cudaStream_t st, bool pdl,
                       bool early) {
    using E = typename io_t<IO>::T;
    auto kern = gdn_tree_kernel<IO, DK, MAXD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(c.dv / CB, c.Hv, c.B);
    return launch_k(pdl, kern, grid, dim3(NT), smem, st, c, t, h0, static_cast<const E*>(q),
                      static_cast<const E*>(k), static_cast<const E*>(v), alpha, beta,
                      static_cast<E*>(o), c_out, early);
}

}  // namespace

size_t gdn_tree_smem(const spec_cfg& c) {
    return sizeof(float) * (size_t)gdn_smem_layout(c.N + 1, c.m, c.dk).total;
}

cudaError_t launch_gdn_tree(const spec_cfg& c, const spec_tree& t, const float* h0,
                            const void* q, const void* k, const void* v, const float* alpha,
                            const float* beta, void* o, float* c_out, void* ws, cudaStream_t st,
                            bool pdl, bool early) {
    if (gdn_state_supported(c))
        return launch_gdn_state(c, t, h0, q, k, v, alpha, beta, o, c_out, ws, st, pdl, early);
    const size_t smem = gdn_tree_smem(c);
    if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
    const int T = c.N + 1;
    const int S = (c.m < T - 1 ? c.m : T - 1) + 1;        // rows on the longest root path
    const bool chains = S <= kChainMax;
#define SPEC_GDN_LAUNCH(IO_, DK_)                                                              \
    return chains ? launch_one<IO_, DK_, kChainMax>(c, t, h0, q, k, v, alpha, beta, o, c_out, smem, st, pdl, early) \
                  : launch_one<IO_, DK_, 0>(c, t, h0, q, k, v, alpha, beta, o, c_out, smem, st, pdl, early)
    if (c.io_dtype == SPEC_IO_BF16) {
        if (c.dk == 128) { SPEC_GDN_LAUNCH(SPEC_IO_BF16, 128); }
        SPEC_GDN_LAUNCH(SPEC_IO_BF16, 64);
    }
    if (c.dk == 128) { SPEC_GDN_LAUNCH(SPEC_IO_F32, 128); }
    SPEC_GDN_LAUNCH(SPEC_IO_F32, 64);
#undef SPEC_GDN_LAUNCH
}

}  // namespace spec
