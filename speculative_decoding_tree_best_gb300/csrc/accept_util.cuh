// accept_util.cuh -- the pieces of the acceptance shared by accept_commit.cu,
// verify_commit.cu and attn_tree.cu (the merge + acceptance launch): the
// vocabulary argmax of a logits segment, the greedy walk of one request, and
// one CTA of the argmax + acceptance launch.
//
// Digest "SpecPilot ...": prerequisites / speculative decoding (greedy: accept
// the longest prefix equal to the target argmax, plus one bonus token,
// tau in [1, m+1]) and prerequisites / draft-tree verification (longest
// matching root path).
#pragma once

#include "common.cuh"

namespace spec {
namespace acc {

constexpr int NT = 256;          // threads of a CTA that calls scan_segment

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// Acceptance of request b by one warp (lanes 0-31 of the calling CTA).  With
// `draws` the row tokens are the target's draws [B][T]; without, the argmax
// partials are reduced.
__device__ inline void accept_request(const spec_cfg& c, const spec_tree& tree, const spec_commit_io& io,
                               const spec_accept& out, void* ws, const WsLayout& w, int b,
                               const int32_t* draws = nullptr) {
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
        if (t < nn && draws) {
            a = __ldcg(draws + (size_t)b * T + t);    // written by other CTAs of this launch
        } else if (t < nn) {
            // all segment partials of the row in flight, then reduced
            float2 pp[kArgmaxSplit];
#pragma unroll
            for (int sp = 0; sp < kArgmaxSplit; ++sp)
                pp[sp] = sp < w.argmax_split
                             ? __ldcg(part + ((size_t)b * T + t) * kArgmaxSplit + sp)  // other CTAs'
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
// over the CTA; valid in thread 0.  U: 16-byte loads in flight per thread.
template <int IO, int U = 8>
__device__ inline void scan_segment(const typename io_t<IO>::T* __restrict__ rp, int V, int lo, int hi,
                             float& bv, int& bi) {
    using E = typename io_t<IO>::T;
    constexpr int VEC = 16 / sizeof(E);
    bv = -INFINITY;
    bi = 0x7fffffff;
    const bool vec_ok = (V % VEC) == 0 && ((reinterpret_cast<uintptr_t>(rp) & 15) == 0);
    if (vec_ok) {
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


// One CTA of the argmax + acceptance launch: segment `sp` of logits row `row`
// (request row / T, tree row row % T), reduced to (max, first index) in the
// workspace; the last CTA of a request (atomic ticket) runs its acceptance.
// tree_early: the launch that wrote the tree is at least two back, so n_nodes
// may be read before the wait.  trigger_first: the launches after this one
// read nothing it writes before their own waits, so they may start at once.
template <int IO>
__device__ inline void argmax_block(const spec_cfg& c, const typename io_t<IO>::T* __restrict__ logits,
                                    const spec_tree& tree, const spec_commit_io& io,
                                    const spec_accept& out, void* ws, const WsLayout& w,
                                    bool tree_early, bool trigger_first, int sp, int row) {
    using E = typename io_t<IO>::T;
    constexpr int VEC = 16 / sizeof(E);
    if (trigger_first) pdl_trigger();
    const int T = c.N + 1, b = row / T, t = row % T;
    // n_nodes may only be read before the wait when the launch that wrote the
    // tree is at least two back
    if (!tree_early) pdl_wait();
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
    if (!trigger_first) pdl_trigger();
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
        accept_request(c, tree, io, out, ws, w, b);
    }
}

}  // namespace acc
}  // namespace spec
