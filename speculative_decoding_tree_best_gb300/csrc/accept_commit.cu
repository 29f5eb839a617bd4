// accept_commit.cu -- vocabulary argmax, greedy acceptance of the longest
// matching root path plus the bonus token, and commit of the accepted path.
//
// Digest "SpecPilot ...": prerequisites / speculative decoding (greedy: accept
// the longest prefix equal to the target argmax, plus one bonus token,
// tau in [1, m+1]), prerequisites / draft-tree verification (longest matching
// root path) and technical novelty (states recomputed along the root path).
//
// Sampled acceptance (temperature > 0; the speculative-decoding tutorial
// (mlqm.cn), section 2.3): the drafts are fixed tokens, so the rejection rule
// keeps a child with the target's probability of its token after the earlier
// children are removed, which is the law of drawing y from
// softmax(logits / temperature) at the row and moving to the child whose
// token is y.  The draw replaces the argmax:
//  1'. sample_accept: warp w of CTA (x, row) scans vocabulary chunk 8 x + w
//     (SPEC_SAMPLE_CHUNK tokens, 16-byte loads) into (max, sum of exp); the
//     last CTA of the row (ticket) picks the chunk by Gumbel-max over the
//     chunks' log-masses, then the token inside it by Gumbel-max over its
//     logits / temperature (Philox4x32-10 noise, four tokens per block); the
//     last row of a request runs the acceptance walk on the draws.
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

#include "accept_util.cuh"
#include "common.cuh"
#include "kernels.h"

namespace spec {

namespace {

constexpr int NT = 256;
using acc::better;
using acc::accept_request;
using acc::scan_segment;

template <int IO>
__global__ void __launch_bounds__(NT)
argmax_accept(spec_cfg c, const typename io_t<IO>::T* __restrict__ logits, spec_tree tree,
              spec_commit_io io, spec_accept acc, void* ws, WsLayout w, bool tree_early,
              bool trigger_first) {
    acc::argmax_block<IO>(c, logits, tree, io, acc, ws, w, tree_early, trigger_first, blockIdx.x,
                          blockIdx.y);
}

// ---- sampled acceptance ------------------------------------------------------------

// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds of two 32x32 -> 64-bit products of
// words 0 and 2 by the round multipliers, the high halves mixed with words 1
// and 3 and the key; the key grows by the Weyl increments between rounds.
__device__ __forceinline__ void philox4x32_10(uint32_t& c0, uint32_t& c1, uint32_t& c2,
                                              uint32_t& c3, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
}

// Gumbel noise of one word: U = (floor(x / 2^9) + 1/2) 2^-23, exact in float
// and inside (0, 1); g = -ln(-ln U).  The inner log is the accurate logf: the
// winners have U near 1, where -ln U must keep its relative precision.  The
// outer one only needs a small absolute error, which the fast __logf has.
__device__ __forceinline__ float gumbel(uint32_t x) {
    const float u = (__uint2float_rn(x >> 9) + 0.5f) * (1.0f / 8388608.0f);
    return -__logf(-logf(u));
}

__device__ __forceinline__ uint32_t word_of(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                            int i) {
    return i == 0 ? c0 : (i == 1 ? c1 : (i == 2 ? c2 : c3));
}

// Merge of two (max, sum of exp((x - max) k)) pairs.
__device__ __forceinline__ void mass_merge(float& m, float& s, float om, float os, float k) {
    const float nm = fmaxf(m, om);
    if (nm == -INFINITY) return;                       // both empty
    s = (m == nm ? s : s * __expf((m - nm) * k)) + (om == nm ? os : os * __expf((om - nm) * k));
    m = nm;
}

// (max, sum of exp((x - max) / temperature)) of logits [lo, hi) by one warp.
template <int IO>
__device__ __forceinline__ float2 chunk_mass(const typename io_t<IO>::T* __restrict__ rp, int lo,
                                             int hi, bool vec_ok, float k, int lane) {
    using E = typename io_t<IO>::T;
    constexpr int VEC = 16 / sizeof(E);
    // 16-byte loads in flight per lane: a whole bf16 chunk (16 per lane) at once
    constexpr int U = VEC == 8 ? 16 : 8;
    float m = -INFINITY, s = 0.0f;
    if (vec_ok) {
        for (int e0 = lo + lane * VEC; e0 < hi; e0 += U * 32 * VEC) {
            uint4 u[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int ej = e0 + j * 32 * VEC;
                u[j] = ej < hi ? *reinterpret_cast<const uint4*>(rp + ej) : make_uint4(0, 0, 0, 0);
            }
            float bm = -INFINITY;
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const E* ev = reinterpret_cast<const E*>(&u[j]);
                if (e0 + j * 32 * VEC < hi)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) bm = fmaxf(bm, io_t<IO>::ld(ev, e));
            }
            const float nm = fmaxf(m, bm);
            if (nm == -INFINITY) continue;
            s = m == nm ? s : s * __expf((m - nm) * k);
            m = nm;
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const E* ev = reinterpret_cast<const E*>(&u[j]);
                if (e0 + j * 32 * VEC < hi)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) s += __expf((io_t<IO>::ld(ev, e) - m) * k);
            }
        }
    } else {
        for (int e = lo + lane; e < hi; e += 32) {
            const float x = io_t<IO>::ld(rp, e);
            mass_merge(m, s, x, 1.0f, k);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float os = __shfl_xor_sync(0xffffffffu, s, o);
        mass_merge(m, s, om, os, k);
    }
    return make_float2(m, s);
}

// CTA-wide (value desc, index asc) reduction; the result in every thread.
__device__ __forceinline__ void cta_best(float& bv, int& bi) {
    __shared__ float sv[NT / 32];
    __shared__ int si[NT / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();                                   // sv / si free from a previous use
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    __syncthreads();
    bv = sv[0];
    bi = si[0];
    for (int k = 1; k < NT / 32; ++k)
        if (better(sv[k], si[k], bv, bi)) { bv = sv[k]; bi = si[k]; }
}

// One CTA per SM at bf16 (a whole chunk's 16-byte loads in flight per lane
// keep ~64 KB per SM in flight, more than the bandwidth needs).
template <int IO>
__global__ void __launch_bounds__(NT)
sample_accept(spec_cfg c, const typename io_t<IO>::T* __restrict__ logits, spec_tree tree,
              spec_commit_io io, spec_accept acc, void* ws, WsLayout w, float inv_temp,
              uint32_t key0, uint32_t key1, bool tree_early, bool trigger_first) {
    using E = typename io_t<IO>::T;
    if (trigger_first) pdl_trigger();       // as in argmax_accept
    constexpr int VEC = 16 / sizeof(E);
    const int row = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = c.N + 1, b = row / T, t = row % T, V = c.V, nvc = w.n_vchunks;
    const E* rp = logits + (size_t)row * V;
    float2* part = ws_ptr<float2>(ws, w.samp_off) + (size_t)row * nvc;
    if (!tree_early) pdl_wait();
    const bool live = t < tree.n_nodes[b];             // CTA-uniform
    const bool vec_ok = (V % VEC) == 0 && ((reinterpret_cast<uintptr_t>(rp) & 15) == 0);

    // ---- 1. one vocabulary chunk per warp: (max, sum of exp) -------------------------
    const int ch = blockIdx.x * (NT / 32) + warp;
    if (live && ch < nvc) {
        const int lo = ch * SPEC_SAMPLE_CHUNK, hi = min(V, lo + SPEC_SAMPLE_CHUNK);
        const float2 ms = chunk_mass<IO>(rp, lo, hi, vec_ok, inv_temp, lane);
        if (lane == 0) part[ch] = ms;
    }
    // kv_len (the noise counter) and the acceptance need every earlier launch
    pdl_wait();
    if (!trigger_first) pdl_trigger();
    __shared__ bool last;
    if (tid == 0) {
        __threadfence();
        unsigned int* tk = ws_ptr<unsigned int>(ws, w.row_ticket_off) + row;
        const unsigned int done = atomicAdd(tk, 1u);
        last = done == gridDim.x - 1u;
        if (last) *tk = 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();

    // ---- 2. the row's draw (last CTA of the row) --------------------------------------
    int draw = -1;
    if (live) {
        const uint32_t pos = static_cast<uint32_t>(io.kv_len[b]);
        // chunk: Gumbel-max over the log-masses
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int q = tid; q < nvc; q += NT) {
            const float2 ms = __ldcg(part + q);          // written by other CTAs of this launch
            uint32_t c0 = static_cast<uint32_t>(q) >> 2, c1 = static_cast<uint32_t>(t) | 0x80000000u,
                     c2 = static_cast<uint32_t>(b), c3 = pos;
            philox4x32_10(c0, c1, c2, c3, key0, key1);
            const float sc = ms.x * inv_temp + logf(ms.y) + gumbel(word_of(c0, c1, c2, c3, q & 3));
            if (better(sc, q, bv, bi)) { bv = sc; bi = q; }
        }
        cta_best(bv, bi);
        bool bad = bi >= nvc;                          // every chunk score NaN
        if (bad) bi = 0;
        // token inside the chunk: Gumbel-max over logits / temperature, four
        // tokens per Philox block
        const int lo = bi * SPEC_SAMPLE_CHUNK, hi = min(V, lo + SPEC_SAMPLE_CHUNK);
        float tv = -INFINITY;
        int ti = 0x7fffffff;
        for (int q = (lo >> 2) + tid; 4 * q < hi; q += NT) {
            uint32_t c0 = static_cast<uint32_t>(q), c1 = static_cast<uint32_t>(t),
                     c2 = static_cast<uint32_t>(b), c3 = pos;
            philox4x32_10(c0, c1, c2, c3, key0, key1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int v = 4 * q + j;
                if (v < hi) {
                    const float z = io_t<IO>::ld(rp, v) * inv_temp + gumbel(word_of(c0, c1, c2, c3, j));
                    if (better(z, v, tv, ti)) { tv = z; ti = v; }
                }
            }
        }
        cta_best(tv, ti);
        if (ti >= hi) {                                // every token score NaN
            ti = lo;
            bad = true;
        }
        if (bad && tid == 0) raise_status(ws, SPEC_DEV_BADLOGIT);
        draw = ti;
    }
    int32_t* draws = ws_ptr<int32_t>(ws, w.samp_tok_off);
    if (tid == 0) draws[row] = draw;

    // ---- 3. the last row of the request runs the acceptance ---------------------------
    __shared__ bool last_row;
    if (tid == 0) {
        __threadfence();
        unsigned int* tk = ws_ptr<unsigned int>(ws, w.acc_ticket_off) + b;
        const unsigned int done = atomicAdd(tk, 1u);
        last_row = done == (unsigned int)T - 1u;
        if (last_row) *tk = 0u;
    }
    __syncthreads();
    if (last_row && tid < 32) {
        __threadfence();
        accept_request(c, tree, io, acc, ws, w, b, draws);
    }
}

// Gated-delta steps of the accepted rows on CB columns (from c0) of a d_k x d_v
// state: thread (row group g, column col) of the 4 CB threads holds rows
// [g DK/4, (g+1) DK/4) of column c0 + col in registers; written back in place.
template <int IO, int DK, int DV, int CB>
__device__ __forceinline__ void commit_state(const spec_cfg& c, const spec_commit_io& io,
                                             const spec_accept& acc, const int32_t* plan,
                                             float* hr, float* h, int b, int j, int layer, int c0,
                                             float* sc) {
    using E = typename io_t<IO>::T;
    constexpr int NTC = 4 * CB, RPT = DK / 4;
    const int T = c.N + 1, m = c.m, tid = threadIdx.x;
    const int ih = j / (c.Hv / c.Hk), col = tid % CB, grp = tid / CB;
    const int tau = plan[4 * b];
    if (tau == 0) return;
    float* ks = sc;                     // [tau][DK]
    float* vsm = ks + (m + 1) * DK;     // [tau][CB]
    float* ab = vsm + (m + 1) * CB;     // [tau][2]
    float* red = ab + 2 * (m + 1);      // [2][4][CB]
    const E* kl = static_cast<const E*>(io.gdn_k) + (size_t)layer * c.B * T * c.Hk * DK;
    const E* vl = static_cast<const E*>(io.gdn_v) + (size_t)layer * c.B * T * c.Hv * DV;
    const float* al = io.alpha + (size_t)layer * c.B * T * c.Hv;
    const float* be = io.beta + (size_t)layer * c.B * T * c.Hv;
    const int32_t* nodes = acc.accept_nodes + (size_t)b * (m + 1);
    for (int idx = tid; idx < tau * DK; idx += NTC) {
        const int s = idx / DK, r = idx % DK, x = nodes[s];
        ks[idx] = io_t<IO>::ld(kl, (((size_t)b * T + x) * c.Hk + ih) * DK + r);
    }
    for (int idx = tid; idx < tau * CB; idx += NTC) {
        const int s = idx / CB, r = idx % CB, x = nodes[s];
        vsm[idx] = io_t<IO>::ld(vl, (((size_t)b * T + x) * c.Hv + j) * DV + c0 + r);
    }
    for (int s = tid; s < tau; s += NTC) {
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
        float* rb = red + (s & 1) * 4 * CB;
        rb[grp * CB + col] = part;
        __syncthreads();
        const float u = (rb[col] + rb[CB + col]) + (rb[2 * CB + col] + rb[3 * CB + col]);
        const float a = ab[2 * s], bb = ab[2 * s + 1], vv = vsm[s * CB + col];
#pragma unroll
        for (int i = 0; i < RPT; ++i) hr[i] = a * (hr[i] - bb * kk[i] * u) + bb * kk[i] * vv;
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) h[(size_t)(grp * RPT + i) * DV + c0 + col] = hr[i];
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
    for (size_t o = (size_t)tid * 16; o < row; o += (size_t)blockDim.x * 16) {
        *reinterpret_cast<uint4*>(kc + dst + o) = *reinterpret_cast<const uint4*>(kt + src + o);
        *reinterpret_cast<uint4*>(vc + dst + o) = *reinterpret_cast<const uint4*>(vt + src + o);
    }
}

// early: the acceptance, or a GDN layer that still reads h0, may be the launch
// just before this one, so wait before anything else; otherwise both are at
// least two launches back and the wait moves to the end.  One block per CB
// columns of a GDN (layer, request, v-head) state (4 CB threads: the whole
// state when there are enough states to fill the GPU, 32 columns otherwise),
// then one block per KV row append.
template <int IO, int DK, int DV, int CB>
__global__ void __launch_bounds__(4 * CB)
commit_kernel(spec_cfg c, spec_commit_io io, spec_accept acc, void* ws, WsLayout w, int gdn_blocks,
              bool early) {
    extern __shared__ __align__(16) float sc[];
    const int32_t* plan = ws_ptr<const int32_t>(ws, w.plan_off);
    const int tid = threadIdx.x;
    if ((int)blockIdx.x < gdn_blocks) {
        constexpr int RPT = DK / 4;
        int id = blockIdx.x;
        const int c0 = (id % (DV / CB)) * CB; id /= DV / CB;
        const int j = id % c.Hv; id /= c.Hv;
        const int b = id % c.B;
        const int layer = id / c.B;
        const int col = tid % CB, grp = tid / CB;
        // the state does not depend on the acceptance: load it first
        float* h = io.h0 + (size_t)layer * c.B * c.Hv * DK * DV + ((size_t)b * c.Hv + j) * DK * DV;
        float hr[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) hr[i] = h[(size_t)(grp * RPT + i) * DV + c0 + col];
        if (early) {
            pdl_wait();
            pdl_trigger();
        }
        commit_state<IO, DK, DV, CB>(c, io, acc, plan, hr, h, b, j, layer, c0, sc);
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

template <int IO, int DK, int DV, int CB>
cudaError_t launch_commit_k(const spec_cfg& c, const spec_commit_io& io, const spec_accept& out,
                            void* ws, const WsLayout& w, cudaStream_t st, bool pdl, bool early) {
    const int gdn_blocks = c.n_gdn_layers * c.B * c.Hv * (DV / CB);
    const int kv_blocks = c.n_attn_layers * c.B * (c.m + 1);
    if (gdn_blocks + kv_blocks == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)(c.m + 1) * (DK + CB + 2) + 2 * 4 * CB);
    auto kern = commit_kernel<IO, DK, DV, CB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(pdl, kern, dim3(gdn_blocks + kv_blocks), dim3(4 * CB), smem, st, c, io, out, ws,
                    w, gdn_blocks, early);
}

}  // namespace

cudaError_t launch_argmax_accept(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 const spec_commit_io& io, const spec_accept& out, void* ws,
                                 cudaStream_t st, bool pdl, bool tree_early, bool trigger_first) {
    const WsLayout w = ws_layout(c, device_sm_count());
    dim3 g1(w.argmax_split, c.B * (c.N + 1));
    return c.io_dtype == SPEC_IO_BF16
        ? launch_k(pdl, argmax_accept<SPEC_IO_BF16>, g1, dim3(NT), 0, st, c,
                   static_cast<const __nv_bfloat16*>(logits), t, io, out, ws, w, tree_early,
                   trigger_first)
        : launch_k(pdl, argmax_accept<SPEC_IO_F32>, g1, dim3(NT), 0, st, c,
                   static_cast<const float*>(logits), t, io, out, ws, w, tree_early,
                   trigger_first);
}

cudaError_t launch_sample_accept(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 float temperature, uint64_t seed, const spec_commit_io& io,
                                 const spec_accept& out, void* ws, cudaStream_t st, bool pdl,
                                 bool tree_early, bool trigger_first) {
    const WsLayout w = ws_layout(c, device_sm_count());
    dim3 g1((w.n_vchunks + NT / 32 - 1) / (NT / 32), c.B * (c.N + 1));
    const float inv_temp = 1.0f / temperature;
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    return c.io_dtype == SPEC_IO_BF16
        ? launch_k(pdl, sample_accept<SPEC_IO_BF16>, g1, dim3(NT), 0, st, c,
                   static_cast<const __nv_bfloat16*>(logits), t, io, out, ws, w, inv_temp, k0, k1,
                   tree_early, trigger_first)
        : launch_k(pdl, sample_accept<SPEC_IO_F32>, g1, dim3(NT), 0, st, c,
                   static_cast<const float*>(logits), t, io, out, ws, w, inv_temp, k0, k1,
                   tree_early, trigger_first);
}

template <int IO>
static cudaError_t launch_commit_io(const spec_cfg& c, const spec_commit_io& io,
                                    const spec_accept& out, void* ws, const WsLayout& w,
                                    cudaStream_t st, bool pdl, bool early) {
    // whole states when they fill the GPU four times over, else 32-column slices
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const bool whole = (long)c.n_gdn_layers * c.B * c.Hv >= 4L * sms;
    if (c.dk == 128) {
        if (c.dv == 128)
            return whole ? launch_commit_k<IO, 128, 128, 128>(c, io, out, ws, w, st, pdl, early)
                         : launch_commit_k<IO, 128, 128, 32>(c, io, out, ws, w, st, pdl, early);
        return whole ? launch_commit_k<IO, 128, 64, 64>(c, io, out, ws, w, st, pdl, early)
                     : launch_commit_k<IO, 128, 64, 32>(c, io, out, ws, w, st, pdl, early);
    }
    if (c.dv == 128)
        return whole ? launch_commit_k<IO, 64, 128, 128>(c, io, out, ws, w, st, pdl, early)
                     : launch_commit_k<IO, 64, 128, 32>(c, io, out, ws, w, st, pdl, early);
    return whole ? launch_commit_k<IO, 64, 64, 64>(c, io, out, ws, w, st, pdl, early)
                 : launch_commit_k<IO, 64, 64, 32>(c, io, out, ws, w, st, pdl, early);
}

cudaError_t launch_commit(const spec_cfg& c, const spec_commit_io& io, const spec_accept& out,
                          void* ws, cudaStream_t st, bool pdl, bool early) {
    const WsLayout w = ws_layout(c, device_sm_count());
    return c.io_dtype == SPEC_IO_BF16
        ? launch_commit_io<SPEC_IO_BF16>(c, io, out, ws, w, st, pdl, early)
        : launch_commit_io<SPEC_IO_F32>(c, io, out, ws, w, st, pdl, early);
}

cudaError_t launch_accept_commit(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 const spec_commit_io& io, const spec_accept& out, void* ws,
                                 cudaStream_t st, bool pdl, const float* temperature,
                                 uint64_t seed) {
    cudaError_t e = temperature
        ? launch_sample_accept(c, t, logits, *temperature, seed, io, out, ws, st, pdl, false)
        : launch_argmax_accept(c, t, logits, io, out, ws, st, pdl, false);
    if (e != cudaSuccess) return e;
    return launch_commit(c, io, out, ws, st, pdl, true);
}

}  // namespace spec
