// accept_commit.cu -- vocabulary argmax, greedy acceptance of the longest
// matching root path plus the bonus token, and commit of the accepted path.
//
// Digest "SpecPilot ...": prerequisites / speculative decoding (greedy: accept
// the longest prefix equal to the target argmax, plus one bonus token,
// tau in [1, m+1]), prerequisites / draft-tree verification (longest matching
// root path) and technical novelty (states recomputed along the root path).
//
// Two launches:
//  1. argmax_accept: every logits row is cut into `argmax_split` segments;
//     a CTA scans one segment with 16-byte loads (eight in flight per thread)
//     and reduces (value desc, index asc) with warp shuffles.  The last CTA to
//     finish a request (atomic ticket) runs its acceptance with one warp:
//     reduce the segments of each row, walk the tree with ballots over the
//     children, write the outputs, check the cache room and advance kv_len /
//     root_tok.
//  2. commit: GDN blocks apply the accepted rows' gated-delta steps to 32
//     columns of a state each (literal recurrence, fp32, the state slice held
//     in registers); KV blocks copy the accepted tree K/V rows into the cache.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace spec {

namespace {

constexpr int NT = 256;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// Acceptance of request b by one warp (lanes 0-31 of the calling CTA).
__device__ void accept_request(const spec_cfg& c, const spec_tree& tree, const spec_commit_io& io,
                               const spec_accept& out, void* ws, const WsLayout& w, int b) {
    __shared__ int sa[3 * SPEC_MAX_ROWS + SPEC_MAX_M + 1];
    const int T = c.N + 1, m = c.m, lane = threadIdx.x;
    int* am = sa;            // [T]
    int* tok = am + T;       // [T]
    int* par = tok + T;      // [T]
    int* path = par + T;     // [m + 1]
    int nn = tree.n_nodes[b];
    nn = nn < 1 ? 1 : (nn > T ? T : nn);
    const float2* part = ws_ptr<const float2>(ws, w.argmax_off);
    for (int t = lane; t < T; t += 32) {
        int a = -1;
        if (t < nn) {
            // all segment partials of the row in flight, then reduced
            float2 pp[kArgmaxSplit];
#pragma unroll
            for (int sp = 0; sp < kArgmaxSplit; ++sp)
                pp[sp] = sp < w.argmax_split ? part[((size_t)b * T + t) * kArgmaxSplit + sp]
                                             : make_float2(-INFINITY, __int_as_float(0x7fffffff));
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int sp = 0; sp < kArgmaxSplit; ++sp) {
                const int pi = __float_as_int(pp[sp].y);
                if (better(pp[sp].x, pi, bv, bi)) { bv = pp[sp].x; bi = pi; }
            }
            a = bi;
        }
        am[t] = a;
        tok[t] = tree.node_tok[(size_t)b * T + t];
        par[t] = tree.node_parent[(size_t)b * T + t];
        out.argmax[(size_t)b * T + t] = a;
    }
    __syncwarp();

    int cur = 0, len = 1;
    if (lane == 0) path[0] = 0;
    for (;;) {
        const int target = am[cur];
        int next = -1;
        for (int base = 0; base < nn && next < 0; base += 32) {
            const int x = base + lane;
            const bool hit = x < nn && par[x] == cur && tok[x] == target;
            const unsigned msk = __ballot_sync(0xffffffffu, hit);
            if (msk) next = base + __ffs(msk) - 1;
        }
        if (next < 0 || len > m) break;
        if (lane == 0) path[len] = next;
        ++len;
        cur = next;
    }
    __syncwarp();
    const int bonus = am[cur];
    for (int s = lane; s <= m; s += 32) {
        out.accept_nodes[(size_t)b * (m + 1) + s] = s < len ? path[s] : -1;
        int ot = -1;
        if (s < len - 1) ot = tok[path[s + 1]];
        else if (s == len - 1) ot = bonus;
        out.out_tok[(size_t)b * (m + 1) + s] = ot;
    }
    if (lane == 0) {
        out.accept_len[b] = len;
        const int L = io.kv_len[b];
        const bool ok = L >= 0 && L + len <= c.Lmax;
        int32_t* plan = ws_ptr<int32_t>(ws, w.plan_off) + 4 * b;
        plan[0] = ok ? len : 0;
        plan[1] = L;
        if (ok) {
            io.kv_len[b] = L + len;
            io.root_tok[b] = bonus;
        } else {
            raise_status(ws, SPEC_DEV_OVERFLOW);
        }
    }
}

// (max, first index) of logits row `row` over the segment [lo, hi), reduced
// over the CTA; valid in thread 0.
template <int IO>
__device__ void scan_segment(const typename io_t<IO>::T* __restrict__ rp, int V, int lo, int hi,
                             float& bv, int& bi) {
    using E = typename io_t<IO>::T;
    constexpr int VEC = 16 / sizeof(E);
    bv = -INFINITY;
    bi = 0x7fffffff;
    const bool vec_ok = (V % VEC) == 0 && ((reinterpret_cast<uintptr_t>(rp) & 15) == 0);
    if (vec_ok) {
        constexpr int U = 8;                  // 16-byte loads in flight per thread
        for (int e0 = lo + threadIdx.x * VEC; e0 < hi; e0 += U * NT * VEC) {
            uint4 u[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ek = e0 + k * NT * VEC;
                u[k] = ek < hi ? *reinterpret_cast<const uint4*>(rp + ek) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ek = e0 + k * NT * VEC;
                const E* ev = reinterpret_cast<const E*>(&u[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float x = io_t<IO>::ld(ev, e);
                    if (ek < hi && x > bv) { bv = x; bi = ek + e; }
                }
            }
        }
    } else {
        for (int e = lo + threadIdx.x; e < hi; e += NT) {
            const float x = io_t<IO>::ld(rp, e);
            if (x > bv) { bv = x; bi = e; }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    __shared__ float sv[NT / 32];
    __shared__ int si[NT / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int k = 1; k < NT / 32; ++k)
            if (better(sv[k], si[k], bv, bi)) { bv = sv[k]; bi = si[k]; }
}

template <int IO>
__global__ void __launch_bounds__(NT)
argmax_accept(spec_cfg c, const typename io_t<IO>::T* __restrict__ logits, spec_tree tree,
              spec_commit_io io, spec_accept acc, void* ws, WsLayout w) {
    using E = typename io_t<IO>::T;
    constexpr int VEC = 16 / sizeof(E);
    const int sp = blockIdx.x, row = blockIdx.y;
    const int T = c.N + 1, b = row / T, t = row % T;
    if (t < tree.n_nodes[b]) {                           // CTA-uniform
        int seg = (c.V + w.argmax_split - 1) / w.argmax_split;
        seg = (seg + VEC - 1) / VEC * VEC;
        const int lo = sp * seg, hi = min(c.V, lo + seg);
        float bv;
        int bi;
        scan_segment<IO>(logits + (size_t)row * c.V, c.V, lo, hi, bv, bi);
        if (threadIdx.x == 0)
            ws_ptr<float2>(ws, w.argmax_off)[(size_t)row * kArgmaxSplit + sp] =
                make_float2(bv, __int_as_float(bi));
    }
    // The acceptance reads the tree and rewrites kv_len: everything before this
    // launch must be done.
    pdl_wait();
    pdl_trigger();
    // Every CTA of the request takes a ticket; the last one runs the acceptance.
    __shared__ bool last;
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned int* tk = ws_ptr<unsigned int>(ws, w.acc_ticket_off) + b;
        const unsigned int done = atomicAdd(tk, 1u);
        last = done == (unsigned int)(T * w.argmax_split) - 1u;
        if (last) *tk = 0u;                 // leave the ticket at zero for the next call
    }
    __syncthreads();
    if (last && threadIdx.x < 32) {
        __threadfence();
        accept_request(c, tree, io, acc, ws, w, b);
    }
}

// Gated-delta steps of the accepted rows on 32 state columns (rows split over
// the CTA's 8 warps, held in registers), written back in place.
template <int IO, int DK>
__device__ __forceinline__ void commit_state(const spec_cfg& c, const spec_commit_io& io,
                                             const spec_accept& acc, const int32_t* plan,
                                             float* hr, float* h, int b, int j, int layer, int cb,
                                             float* sc) {
    using E = typename io_t<IO>::T;
    constexpr int CB = 32, NG = NT / 32, RPT = DK / NG;
    const int T = c.N + 1, m = c.m, tid = threadIdx.x;
    const int ih = j / (c.Hv / c.Hk), c0 = cb * CB, col = tid & 31, grp = tid >> 5;
    const int tau = plan[4 * b];
    if (tau == 0) return;
    float* ks = sc;                     // [tau][DK]
    float* vsm = ks + (m + 1) * DK;     // [tau][CB]
    float* ab = vsm + (m + 1) * CB;     // [tau][2]
    float* red = ab + 2 * (m + 1);      // [2][NG][CB]
    const E* kl = static_cast<const E*>(io.gdn_k) + (size_t)layer * c.B * T * c.Hk * DK;
    const E* vl = static_cast<const E*>(io.gdn_v) + (size_t)layer * c.B * T * c.Hv * c.dv;
    const float* al = io.alpha + (size_t)layer * c.B * T * c.Hv;
    const float* be = io.beta + (size_t)layer * c.B * T * c.Hv;
    const int32_t* nodes = acc.accept_nodes + (size_t)b * (m + 1);
    for (int idx = tid; idx < tau * DK; idx += NT) {
        const int s = idx / DK, r = idx % DK, x = nodes[s];
        ks[idx] = io_t<IO>::ld(kl, (((size_t)b * T + x) * c.Hk + ih) * DK + r);
    }
    for (int idx = tid; idx < tau * CB; idx += NT) {
        const int s = idx / CB, cc = idx % CB, x = nodes[s];
        vsm[idx] = io_t<IO>::ld(vl, (((size_t)b * T + x) * c.Hv + j) * c.dv + c0 + cc);
    }
    for (int s = tid; s < tau; s += NT) {
        const int x = nodes[s];
        ab[2 * s] = al[((size_t)b * T + x) * c.Hv + j];
        ab[2 * s + 1] = be[((size_t)b * T + x) * c.Hv + j];
    }
    __syncthreads();
    for (int s = 0; s < tau; ++s) {
        const float* kk = ks + s * DK + grp * RPT;
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) part = fmaf(hr[i], kk[i], part);
        float* rb = red + (s & 1) * NG * CB;
        rb[grp * CB + col] = part;
        __syncthreads();
        float u = 0.0f;
#pragma unroll
        for (int g2 = 0; g2 < NG; ++g2) u += rb[g2 * CB + col];
        const float a = ab[2 * s], bb = ab[2 * s + 1], vv = vsm[s * CB + col];
#pragma unroll
        for (int i = 0; i < RPT; ++i) hr[i] = a * (hr[i] - bb * kk[i] * u) + bb * kk[i] * vv;
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) h[(size_t)(grp * RPT + i) * c.dv + c0 + col] = hr[i];
}

// Copy the tree K/V row of accepted path slot s of (layer, request) into the
// cache; block id encodes (layer, request, slot).
template <int IO>
__device__ __forceinline__ void append_kv(const spec_cfg& c, const spec_commit_io& io,
                                          const spec_accept& acc, const int32_t* plan, int id) {
    using E = typename io_t<IO>::T;
    const int T = c.N + 1, m = c.m, tid = threadIdx.x;
    const int s = id % (m + 1); id /= (m + 1);
    const int b = id % c.B;
    const int layer = id / c.B;
    const int tau = plan[4 * b];
    if (s >= tau) return;
    const int L = plan[4 * b + 1];
    const int x = acc.accept_nodes[(size_t)b * (m + 1) + s];
    const size_t row = (size_t)c.Hkv * c.D * sizeof(E);          // bytes, multiple of 16
    const size_t src = (((size_t)layer * c.B + b) * T + x) * row;
    const size_t dst = (((size_t)layer * c.B + b) * c.Lmax + L + s) * row;
    const char* kt = static_cast<const char*>(io.k_tree);
    const char* vt = static_cast<const char*>(io.v_tree);
    char* kc = static_cast<char*>(io.k_cache);
    char* vc = static_cast<char*>(io.v_cache);
    for (size_t o = (size_t)tid * 16; o < row; o += NT * 16) {
        *reinterpret_cast<uint4*>(kc + dst + o) = *reinterpret_cast<const uint4*>(kt + src + o);
        *reinterpret_cast<uint4*>(vc + dst + o) = *reinterpret_cast<const uint4*>(vt + src + o);
    }
}

// early: the acceptance, or a GDN layer that still reads h0, may be the launch
// just before this one, so wait before anything else; otherwise both are at
// least two launches back and the wait moves to the end.
template <int IO, int DK>
__global__ void __launch_bounds__(NT)
commit_kernel(spec_cfg c, spec_commit_io io, spec_accept acc, void* ws, WsLayout w, int gdn_blocks,
              bool early) {
    extern __shared__ __align__(16) float sc[];
    const int32_t* plan = ws_ptr<const int32_t>(ws, w.plan_off);
    const int tid = threadIdx.x;
    if ((int)blockIdx.x < gdn_blocks) {
        constexpr int CB = 32, NG = NT / 32, RPT = DK / NG;
        const int nb = c.dv / CB;
        int id = blockIdx.x;
        const int cb = id % nb; id /= nb;
        const int j = id % c.Hv; id /= c.Hv;
        const int b = id % c.B;
        const int layer = id / c.B;
        const int c0 = cb * CB, col = tid & 31, grp = tid >> 5;
        // the state slice does not depend on the acceptance: load it first
        float* h = io.h0 + (size_t)layer * c.B * c.Hv * DK * c.dv + ((size_t)b * c.Hv + j) * DK * c.dv;
        float hr[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) hr[i] = h[(size_t)(grp * RPT + i) * c.dv + c0 + col];
        if (early) {
            pdl_wait();
            pdl_trigger();
        }
        commit_state<IO, DK>(c, io, acc, plan, hr, h, b, j, layer, cb, sc);
    } else {
        if (early) {
            pdl_wait();
            pdl_trigger();
        }
        append_kv<IO>(c, io, acc, plan, blockIdx.x - gdn_blocks);
    }
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }
}

template <int IO, int DK>
cudaError_t launch_commit_k(const spec_cfg& c, const spec_commit_io& io, const spec_accept& out,
                            void* ws, const WsLayout& w, cudaStream_t st, bool pdl, bool early) {
    const int gdn_blocks = c.n_gdn_layers * c.B * c.Hv * (c.dv / 32);
    const int kv_blocks = c.n_attn_layers * c.B * (c.m + 1);
    if (gdn_blocks + kv_blocks == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)(c.m + 1) * (DK + 32 + 2) + 2 * 8 * 32);
    auto kern = commit_kernel<IO, DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(pdl, kern, dim3(gdn_blocks + kv_blocks), dim3(NT), smem, st, c, io, out, ws, w,
                    gdn_blocks, early);
}

}  // namespace

cudaError_t launch_argmax_accept(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 const spec_commit_io& io, const spec_accept& out, void* ws,
                                 cudaStream_t st, bool pdl) {
    const WsLayout w = ws_layout(c);
    dim3 g1(w.argmax_split, c.B * (c.N + 1));
    return c.io_dtype == SPEC_IO_BF16
        ? launch_k(pdl, argmax_accept<SPEC_IO_BF16>, g1, dim3(NT), 0, st, c,
                   static_cast<const __nv_bfloat16*>(logits), t, io, out, ws, w)
        : launch_k(pdl, argmax_accept<SPEC_IO_F32>, g1, dim3(NT), 0, st, c,
                   static_cast<const float*>(logits), t, io, out, ws, w);
}

cudaError_t launch_commit(const spec_cfg& c, const spec_commit_io& io, const spec_accept& out,
                          void* ws, cudaStream_t st, bool pdl, bool early) {
    const WsLayout w = ws_layout(c);
    if (c.io_dtype == SPEC_IO_BF16)
        return c.dk == 128 ? launch_commit_k<SPEC_IO_BF16, 128>(c, io, out, ws, w, st, pdl, early)
                           : launch_commit_k<SPEC_IO_BF16, 64>(c, io, out, ws, w, st, pdl, early);
    return c.dk == 128 ? launch_commit_k<SPEC_IO_F32, 128>(c, io, out, ws, w, st, pdl, early)
                       : launch_commit_k<SPEC_IO_F32, 64>(c, io, out, ws, w, st, pdl, early);
}

cudaError_t launch_accept_commit(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 const spec_commit_io& io, const spec_accept& out, void* ws,
                                 cudaStream_t st, bool pdl) {
    cudaError_t e = launch_argmax_accept(c, t, logits, io, out, ws, st, pdl);
    if (e != cudaSuccess) return e;
    return launch_commit(c, io, out, ws, st, pdl, true);
}

}  // namespace spec
