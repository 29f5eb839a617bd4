// attn_tree.cu -- tree-ancestor-masked attention of the tree rows over the KV
// cache plus their tree ancestors (split-KV, then a merge).
//
// Digest "SpecPilot ...": prerequisites / draft-tree verification (one target
// pass verifies the whole tree; every node sees only its ancestors).
//
// Work split.  The query rows of one (request, kv-head) are the G = Hq/Hkv
// q-heads of that group times the tree rows, row r = node * G + head_in_group,
// cut into 128-row tiles.  The keys are the cache rows [0, kv_len) cut into
// fixed chunks plus one extra "tree chunk" holding the T tree rows, where a
// key is visible to node x iff it is x or an ancestor of x.  Every
// (request, kv-head, tile, chunk) produces an un-normalised partial
// (O, running max, running sum); the merge rescales and sums the partials.
// Only the tree chunk depends on the tree, so the cache chunks (all the KV
// bytes) need nothing from spec_tree_build except n_nodes.
//
// This file holds the SIMT partial (fp32 I/O and head dim 64) and the merge;
// attn_tree_tc.cu holds the tcgen05 partial used for bf16 I/O, head dim 128.
#include <cuda_fp16.h>
#include <math.h>

#include "accept_util.cuh"
#include "common.cuh"
#include "kernels.h"

namespace spec {

namespace {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int kMergeGroup = 8;   // merge: chunk partials loaded per round trip

template <int IO, int D>
__global__ void __launch_bounds__(NT)
attn_partial_simt(spec_cfg c, spec_tree tree, const typename io_t<IO>::T* __restrict__ q,
                  const typename io_t<IO>::T* __restrict__ k_tree,
                  const typename io_t<IO>::T* __restrict__ v_tree,
                  const typename io_t<IO>::T* __restrict__ k_cache,
                  const typename io_t<IO>::T* __restrict__ v_cache,
                  const int32_t* __restrict__ kv_len, void* ws, WsLayout w) {
    constexpr int EPL = D / 32;
    const int ch = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int T = c.N + 1, G = c.Hq / c.Hkv, Hkv = c.Hkv;
    pdl_wait();
    pdl_trigger();
    int nn = tree.n_nodes[b];
    nn = nn < 1 ? 1 : (nn > T ? T : nn);
    int L = kv_len[b];
    L = L < 0 ? 0 : (L > c.Lmax ? c.Lmax : L);
    const bool tree_chunk = ch == w.n_split;
    int k0 = 0, k1 = 0;
    if (!tree_chunk) {
        k0 = ch * w.chunk;
        k1 = min(k0 + w.chunk, L);
        if (k0 >= L) {                       // no cache rows here: an empty partial
            float2* wML = ws_ptr<float2>(ws, w.attn_ml_off);
            for (int r = threadIdx.x; r < G * T; r += NT) {
                const size_t tile = (((size_t)b * Hkv + g) * w.n_mt + r / 128) * w.n_chunks + ch;
                wML[tile * 128 + r % 128] = make_float2(-INFINITY, 0.0f);
            }
            return;
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float scale = rsqrtf((float)D);
    using PT = typename io_t<IO>::PT;
    PT* wO = ws_ptr<PT>(ws, w.attn_o_off);
    float2* wML = ws_ptr<float2>(ws, w.attn_ml_off);

    for (int r = warp; r < G * nn; r += NW) {
        const int x = r / G, h = g * G + r % G;
        float qv[EPL], acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            qv[e] = io_t<IO>::ld(q, (((size_t)b * T + x) * c.Hq + h) * D + lane * EPL + e);
            acc[e] = 0.0f;
        }
        float mx = -INFINITY, sum = 0.0f;
        const uint64_t a0 = tree.node_anc[2 * ((size_t)b * T + x)];
        const uint64_t a1 = tree.node_anc[2 * ((size_t)b * T + x) + 1];
        const int kend = tree_chunk ? nn : k1;
        for (int key = tree_chunk ? 0 : k0; key < kend; ++key) {
            size_t base;
            const typename io_t<IO>::T *kp, *vp;
            if (tree_chunk) {
                const uint64_t word = key < 64 ? a0 : a1;
                if (!((word >> (key & 63)) & 1ull)) continue;
                base = (((size_t)b * T + key) * Hkv + g) * D;
                kp = k_tree;
                vp = v_tree;
            } else {
                base = (((size_t)b * c.Lmax + key) * Hkv + g) * D;
                kp = k_cache;
                vp = v_cache;
            }
            float s = 0.0f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) s = fmaf(qv[e], io_t<IO>::ld(kp, base + lane * EPL + e), s);
            s = warp_sum(s) * scale;
            const float mn = fmaxf(mx, s);
            const float corr = __expf(mx - mn);
            const float p = __expf(s - mn);
            sum = sum * corr + p;
#pragma unroll
            for (int e = 0; e < EPL; ++e)
                acc[e] = fmaf(p, io_t<IO>::ld(vp, base + lane * EPL + e), acc[e] * corr);
            mx = mn;
        }
        const int mt = r / 128, rr = r % 128;
        const size_t tile = (((size_t)b * Hkv + g) * w.n_mt + mt) * w.n_chunks + ch;
        const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) wO[(tile * 128 + rr) * D + lane * EPL + e] = static_cast<PT>(acc[e] * inv);
        if (lane == 0) wML[tile * 128 + rr] = make_float2(mx, sum);
    }
}

// One warp per query row (8 rows per CTA).  Each chunk left a normalised
// row O_c / l_c (fp16 for bf16 I/O, fp32 for fp32 I/O) and its (max m_c,
// sum l_c).  Lane i reads chunk i's
// (m, l); the warp forms the weights w_c = l_c exp(m_c - M) / sum and every
// lane sums its D/32 output columns over the chunks, all loads in flight.
// EPL consecutive partial elements -> floats (one 8- or 16-byte load).
template <int EPL>
__device__ __forceinline__ void load_partial(const __half* p, float* f) {
    if constexpr (EPL == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
        f[0] = a.x; f[1] = a.y;
    }
}
template <int EPL>
__device__ __forceinline__ void load_partial(const float* p, float* f) {
    if constexpr (EPL == 4) {
        const float4 a = *reinterpret_cast<const float4*>(p);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    } else {
        const float2 a = *reinterpret_cast<const float2*>(p);
        f[0] = a.x; f[1] = a.y;
    }
}

template <int IO, int D>
__device__ __forceinline__ void merge_row(const spec_cfg& c, const spec_tree& tree, void* ws,
                                          const WsLayout& w, typename io_t<IO>::T* __restrict__ o,
                                          int r, int g, int b, int lane);

template <int IO, int D>
__global__ void __launch_bounds__(NT, 3)
attn_merge(spec_cfg c, spec_tree tree, void* ws, WsLayout w, typename io_t<IO>::T* __restrict__ o,
           bool early) {
    const int g = blockIdx.y, b = blockIdx.z;
    const int T = c.N + 1, G = c.Hq / c.Hkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x * NW + warp;
    // early: the partials may come from the launch just before this one
    if (early) {
        pdl_wait();
        pdl_trigger();
    }
    if (r < G * T) merge_row<IO, D>(c, tree, ws, w, o, r, g, b, lane);
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }
}

template <int IO, int D>
__device__ __forceinline__ void merge_row(const spec_cfg& c, const spec_tree& tree, void* ws,
                                          const WsLayout& w, typename io_t<IO>::T* __restrict__ o,
                                          int r, int g, int b, int lane) {
    constexpr int EPL = D / 32;
    const int T = c.N + 1, G = c.Hq / c.Hkv;
    int nn = tree.n_nodes[b];
    nn = nn < 1 ? 1 : (nn > T ? T : nn);
    const int x = r / G, h = g * G + r % G, mt = r / 128, rr = r % 128;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.0f;
    if (x < nn) {
        using PT = typename io_t<IO>::PT;
        const PT* wO = ws_ptr<const PT>(ws, w.attn_o_off);
        const float2* wML = ws_ptr<const float2>(ws, w.attn_ml_off);
        const size_t tile0 = (((size_t)b * c.Hkv + g) * w.n_mt + mt) * w.n_chunks;
        // every chunk; chunks without keys left (max -inf, sum 0) and weigh 0
        const int nch = w.n_chunks;
        float m_run = -INFINITY, den_run = 0.0f;
        for (int base = 0; base < nch; base += 32) {           // rounds of 32 chunks
            const int i = base + lane;
            const int cnt = min(32, nch - base);
            // the first group's partial rows go out with the (max, sum) pairs: one
            // round trip.  Chunks without keys never wrote their rows; their
            // weight is 0 and a select (not a product) drops whatever is there.
            float raw[kMergeGroup][EPL];
#pragma unroll
            for (int k = 0; k < kMergeGroup; ++k) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) raw[k][e] = 0.0f;
                if (k < cnt)
                    load_partial<EPL>(wO + ((tile0 + base + k) * 128 + rr) * D + lane * EPL, raw[k]);
            }
            const float2 ml = i < nch ? wML[(tile0 + i) * 128 + rr] : make_float2(-INFINITY, 0.0f);
            float M = ml.x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            const float f = ml.y > 0.0f ? ml.y * __expf(ml.x - M) : 0.0f;  // unnormalised weight
            const float den_r = warp_sum(f);
            float gacc[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) gacc[e] = 0.0f;
#pragma unroll
            for (int k = 0; k < kMergeGroup; ++k) {
                const float fk = __shfl_sync(0xffffffffu, f, k);
#pragma unroll
                for (int e = 0; e < EPL; ++e) gacc[e] = fk > 0.0f ? fmaf(raw[k][e], fk, gacc[e]) : gacc[e];
            }
            // further groups (more than 8 chunks): loads only where the weight is non-zero
            for (int k0 = kMergeGroup; k0 < cnt; k0 += kMergeGroup) {
#pragma unroll
                for (int k = 0; k < kMergeGroup; ++k) {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) raw[k][e] = 0.0f;
                    const bool has = __shfl_sync(0xffffffffu, f, (k0 + k) & 31) > 0.0f;
                    if (k0 + k < cnt && has)
                        load_partial<EPL>(wO + ((tile0 + base + k0 + k) * 128 + rr) * D + lane * EPL,
                                          raw[k]);
                }
#pragma unroll
                for (int k = 0; k < kMergeGroup; ++k) {
                    const float fk = __shfl_sync(0xffffffffu, f, (k0 + k) & 31);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) gacc[e] = fmaf(raw[k][e], fk, gacc[e]);
                }
            }
            const float m_new = fmaxf(m_run, M);
            const float s_old = m_run == -INFINITY ? 0.0f : __expf(m_run - m_new);
            const float s_new = __expf(M - m_new);
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = acc[e] * s_old + gacc[e] * s_new;
            den_run = den_run * s_old + den_r * s_new;
            m_run = m_new;
        }
        const float inv = 1.0f / den_run;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= inv;
    }
    // a real row whose output is not finite: an fp16 V operand or partial out
    // of range (bf16 I/O), or non-finite inputs among the keys it sees
    bool bad = false;
#pragma unroll
    for (int e = 0; e < EPL; ++e) bad |= !(fabsf(acc[e]) <= 3.402823466e38f);
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(ws, SPEC_DEV_RANGE);
#pragma unroll
    for (int e = 0; e < EPL; ++e)
        io_t<IO>::st(o, (((size_t)b * T + x) * c.Hq + h) * D + lane * EPL + e, acc[e]);
}

// The last attention layer's merge and the argmax + acceptance in one launch
// (the step's merge and logits scan have no data in common): blocks
// [0, n_merge) are the merge's (merge_x row groups per (kv-head, request);
// they wait for the partials first, as the merge launched with early does),
// the others the argmax + acceptance CTAs in (segment, row) order (they let
// the next launch start at once, scan, and wait before their tickets).
template <int IO, int D>
__global__ void __launch_bounds__(NT, 3)
merge_accept(spec_cfg c, spec_tree tree, void* ws, WsLayout w, typename io_t<IO>::T* __restrict__ o,
             const typename io_t<IO>::T* __restrict__ logits, spec_commit_io io, spec_accept out,
             int n_merge, int merge_x) {
    const int id = blockIdx.x;
    if (id < n_merge) {
        const int bx = id % merge_x, g = (id / merge_x) % c.Hkv, b = id / (merge_x * c.Hkv);
        const int T = c.N + 1, G = c.Hq / c.Hkv;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int r = bx * NW + warp;
        pdl_wait();
        pdl_trigger();
        if (r < G * T) merge_row<IO, D>(c, tree, ws, w, o, r, g, b, lane);
    } else {
        const int a = id - n_merge;
        acc::argmax_block<IO>(c, logits, tree, io, out, ws, w, /*tree_early=*/true,
                              /*trigger_first=*/true, a % w.argmax_split, a / w.argmax_split);
    }
}

template <int IO, int D>
cudaError_t launch_partial(const spec_cfg& c, const spec_tree& t, const void* q, const void* kt,
                           const void* vt, const void* kc, const void* vc, const int32_t* kv_len,
                           void* ws, cudaStream_t st, bool pdl, int part_buf) {
    using E = typename io_t<IO>::T;
    const WsLayout w = with_attn_buf(ws_layout(c, device_sm_count()), part_buf);
    if (attn_tc_supported(c)) return launch_attn_tc(c, t, q, kt, vt, kc, vc, kv_len, ws, w, st, pdl);
    return launch_k(pdl, attn_partial_simt<IO, D>, dim3(w.n_chunks, c.Hkv, c.B), dim3(NT), 0, st,
                    c, t, static_cast<const E*>(q), static_cast<const E*>(kt),
                    static_cast<const E*>(vt), static_cast<const E*>(kc),
                    static_cast<const E*>(vc), kv_len, ws, w);
}

template <int IO, int D>
cudaError_t launch_merge(const spec_cfg& c, const spec_tree& t, void* o, void* ws, cudaStream_t st,
                         bool pdl, int part_buf, bool early) {
    using E = typename io_t<IO>::T;
    const WsLayout w = with_attn_buf(ws_layout(c, device_sm_count()), part_buf);
    const int G = c.Hq / c.Hkv;
    return launch_k(pdl, attn_merge<IO, D>, dim3((G * (c.N + 1) + NW - 1) / NW, c.Hkv, c.B),
                    dim3(NT), 0, st, c, t, ws, w, static_cast<E*>(o), early);
}

template <int IO, int D>
cudaError_t launch_merge_accept_k(const spec_cfg& c, const spec_tree& t, void* o, void* ws,
                                  cudaStream_t st, bool pdl, int part_buf, const void* logits,
                                  const spec_commit_io& io, const spec_accept& out) {
    using E = typename io_t<IO>::T;
    static_assert(NT == acc::NT, "the argmax CTAs run with the merge's block size");
    const WsLayout w = with_attn_buf(ws_layout(c, device_sm_count()), part_buf);
    const int G = c.Hq / c.Hkv;
    const int merge_x = (G * (c.N + 1) + NW - 1) / NW;
    const int n_merge = merge_x * c.Hkv * c.B;
    const int n_arg = w.argmax_split * c.B * (c.N + 1);
    return launch_k(pdl, merge_accept<IO, D>, dim3(n_merge + n_arg), dim3(NT), 0, st, c, t, ws, w,
                    static_cast<E*>(o), static_cast<const E*>(logits), io, out, n_merge, merge_x);
}

}  // namespace

#define SPEC_ATTN_DISPATCH(FN, ...)                                                      \
    if (c.io_dtype == SPEC_IO_BF16)                                                      \
        return c.D == 128 ? FN<SPEC_IO_BF16, 128>(__VA_ARGS__) : FN<SPEC_IO_BF16, 64>(__VA_ARGS__); \
    return c.D == 128 ? FN<SPEC_IO_F32, 128>(__VA_ARGS__) : FN<SPEC_IO_F32, 64>(__VA_ARGS__)

cudaError_t launch_attn_partial(const spec_cfg& c, const spec_tree& t, const void* q,
                                const void* k_tree, const void* v_tree, const void* k_cache,
                                const void* v_cache, const int32_t* kv_len, void* ws,
                                cudaStream_t st, bool pdl, int part_buf) {
    SPEC_ATTN_DISPATCH(launch_partial, c, t, q, k_tree, v_tree, k_cache, v_cache, kv_len, ws, st,
                       pdl, part_buf);
}

cudaError_t launch_attn_merge(const spec_cfg& c, const spec_tree& t, void* o, void* ws,
                              cudaStream_t st, bool pdl, int part_buf, bool early) {
    SPEC_ATTN_DISPATCH(launch_merge, c, t, o, ws, st, pdl, part_buf, early);
}
cudaError_t launch_merge_accept(const spec_cfg& c, const spec_tree& t, void* o, void* ws,
                                cudaStream_t st, bool pdl, int part_buf, const void* logits,
                                const spec_commit_io& io, const spec_accept& out) {
    SPEC_ATTN_DISPATCH(launch_merge_accept_k, c, t, o, ws, st, pdl, part_buf, logits, io, out);
}
#undef SPEC_ATTN_DISPATCH

cudaError_t launch_attn_tree(const spec_cfg& c, const spec_tree& t, const void* q,
                             const void* k_tree, const void* v_tree, const void* k_cache,
                             const void* v_cache, const int32_t* kv_len, void* o, void* ws,
                             cudaStream_t st, bool pdl, int part_buf) {
    cudaError_t e = launch_attn_partial(c, t, q, k_tree, v_tree, k_cache, v_cache, kv_len, ws, st,
                                        pdl, part_buf);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(c, t, o, ws, st, pdl, part_buf, true);
}

}  // namespace spec
