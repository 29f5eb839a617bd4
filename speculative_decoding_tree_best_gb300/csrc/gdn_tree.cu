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

template <int IO>
__device__ __forceinline__ void ld8(const typename io_t<IO>::T* p, float* f);
template <>
__device__ __forceinline__ void ld8<SPEC_IO_BF16>(const __nv_bfloat16* p, float* f) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(h[e]);
        f[2 * e] = x.x;
        f[2 * e + 1] = x.y;
    }
}
template <>
__device__ __forceinline__ void ld8<SPEC_IO_F32>(const float* p, float* f) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
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
    L.kq = o;  o += 2 * T * DK;
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

template <int IO, int DK>
__global__ void __launch_bounds__(NT)
gdn_tree_kernel(spec_cfg c, spec_tree tree, const float* __restrict__ h0,
                const typename io_t<IO>::T* __restrict__ q, const typename io_t<IO>::T* __restrict__ k,
                const typename io_t<IO>::T* __restrict__ v, const float* __restrict__ alpha,
                const float* __restrict__ beta, typename io_t<IO>::T* __restrict__ o,
                float* __restrict__ c_out) {
    extern __shared__ __align__(16) float sm[];
    const int T = c.N + 1, Hv = c.Hv, Hk = c.Hk, dv = c.dv;
    const int c0 = blockIdx.x * CB, j = blockIdx.y, b = blockIdx.z;
    const int ih = j / (Hv / Hk);
    const int tid = threadIdx.x, col = tid & 31, grp = tid >> 5;
    const GdnSmem L = gdn_smem_layout(T, c.m, DK);
    const int S = L.S;
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

    int nn = tree.n_nodes[b];
    nn = nn < 1 ? 1 : (nn > T ? T : nn);     // a malformed tree must not index out of range

    // ---- stage: tree, gates, h0 slice, k/q rows, v slice ---------------------------
    for (int x = tid; x < nn; x += NT) {
        const int p = tree.node_parent[(size_t)b * T + x];
        const int d = tree.node_depth[(size_t)b * T + x];
        par[x] = (p >= 0 && p < x) ? p : -1;
        dep[x] = d < 0 ? 0 : (d >= S ? S - 1 : d);
        al[x] = alpha[((size_t)b * T + x) * Hv + j];
        be[x] = beta[((size_t)b * T + x) * Hv + j];
    }
    {
        const float* hsrc = h0 + ((size_t)b * Hv + j) * DK * dv + c0;
        for (int idx = tid; idx < DK * (CB / 4); idx += NT) {
            const int r = idx / (CB / 4), q4 = idx % (CB / 4);
            *reinterpret_cast<float4*>(hs + r * CB + q4 * 4) =
                *reinterpret_cast<const float4*>(hsrc + (size_t)r * dv + q4 * 4);
        }
    }
    for (int idx = tid; idx < 2 * nn * (DK / 8); idx += NT) {
        const int row = idx / (DK / 8), e8 = (idx % (DK / 8)) * 8;
        const int x = row < nn ? row : row - nn;
        const auto* src = (row < nn ? k : q) + (((size_t)b * T + x) * Hk + ih) * DK + e8;
        float f[8];
        ld8<IO>(src, f);
        float4* dst = reinterpret_cast<float4*>(kq + row * DK + e8);
        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    for (int idx = tid; idx < nn * (CB / 8); idx += NT) {
        const int x = idx / (CB / 8), e8 = (idx % (CB / 8)) * 8;
        float f[8];
        ld8<IO>(v + (((size_t)b * T + x) * Hv + j) * dv + c0 + e8, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) vs[x * CB + e8 + e] = f[e];
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

    // ---- Gram weights: wo *= k_a . q_x, wu *= k_a . k_x (one warp per row) ------------
    {
        constexpr int EPL = DK / 32;  // elements per lane
        for (int x = grp; x < nn; x += NG) {
            float kx[EPL], qx[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                kx[e] = kq[x * DK + col + 32 * e];
                qx[e] = kq[(nn + x) * DK + col + 32 * e];
            }
            const int d = dep[x];
            for (int s = 0; s <= d; ++s) {
                const float* ka = kq + pidx[x * S + s] * DK;
                float dq = 0.0f, dk = 0.0f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const float a = ka[col + 32 * e];
                    dq = fmaf(a, qx[e], dq);
                    dk = fmaf(a, kx[e], dk);
                }
                dq = warp_sum(dq);
                dk = warp_sum(dk);
                if (col == 0) {
                    wo[x * S + s] *= dq;
                    if (s < d) wu[x * S + s] *= dk;
                }
            }
        }
    }

    // ---- P = h0_slice^T [K; Q]: rows t = grp + 8 i, column col ------------------------
    for (int t0 = 0; t0 < 2 * nn; t0 += 8 * NG) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int r = 0; r < DK; r += 4) {
            const float h_0 = hs[(r + 0) * CB + col], h_1 = hs[(r + 1) * CB + col];
            const float h_2 = hs[(r + 2) * CB + col], h_3 = hs[(r + 3) * CB + col];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = t0 + grp + NG * i;
                if (t < 2 * nn) {
                    const float4 kk = *reinterpret_cast<const float4*>(kq + t * DK + r);
                    acc[i] = fmaf(h_0, kk.x, fmaf(h_1, kk.y, fmaf(h_2, kk.z, fmaf(h_3, kk.w, acc[i]))));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = t0 + grp + NG * i;
            if (t < 2 * nn) P[t * CB + col] = acc[i];
        }
    }
    __syncthreads();

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
            ox = A[x] * P[(nn + x) * CB + col];
            const int d = dep[x];
            for (int s = 0; s <= d; ++s) ox = fmaf(wo[x * S + s], cv[pidx[x * S + s] * CB + col], ox);
            cx = cv[x * CB + col];
        }
        const size_t oi = (((size_t)b * T + x) * Hv + j) * dv + c0 + col;
        io_t<IO>::st(o, oi, ox);
        if (c_out) c_out[oi] = cx;
    }
}

template <int IO, int DK>
cudaError_t launch_one(const spec_cfg& c, const spec_tree& t, const float* h0, const void* q,
                       const void* k, const void* v, const float* alpha, const float* beta,
                       void* o, float* c_out, size_t smem, cudaStream_t st) {
    using E = typename io_t<IO>::T;
    auto kern = gdn_tree_kernel<IO, DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(c.dv / CB, c.Hv, c.B);
    kern<<<grid, NT, smem, st>>>(c, t, h0, static_cast<const E*>(q), static_cast<const E*>(k),
                                 static_cast<const E*>(v), alpha, beta, static_cast<E*>(o), c_out);
    return cudaGetLastError();
}

}  // namespace

size_t gdn_tree_smem(const spec_cfg& c) {
    return sizeof(float) * (size_t)gdn_smem_layout(c.N + 1, c.m, c.dk).total;
}

cudaError_t launch_gdn_tree(const spec_cfg& c, const spec_tree& t, const float* h0,
                            const void* q, const void* k, const void* v, const float* alpha,
                            const float* beta, void* o, float* c_out, cudaStream_t st) {
    const size_t smem = gdn_tree_smem(c);
    if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
    if (c.io_dtype == SPEC_IO_BF16) {
        return c.dk == 128 ? launch_one<SPEC_IO_BF16, 128>(c, t, h0, q, k, v, alpha, beta, o, c_out, smem, st)
                           : launch_one<SPEC_IO_BF16, 64>(c, t, h0, q, k, v, alpha, beta, o, c_out, smem, st);
    }
    return c.dk == 128 ? launch_one<SPEC_IO_F32, 128>(c, t, h0, q, k, v, alpha, beta, o, c_out, smem, st)
                       : launch_one<SPEC_IO_F32, 64>(c, t, h0, q, k, v, alpha, beta, o, c_out, smem, st);
}

}  // namespace spec
