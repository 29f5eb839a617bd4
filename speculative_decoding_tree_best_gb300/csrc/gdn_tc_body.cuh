// gdn_tc_body.cuh -- one (request, v-head) item of the tree-masked Gated
// DeltaNet with the h0^T [K; Q] product on the tensor cores (tcgen05), bf16
// I/O, d_k = d_v = 128, trees of up to 32 rows.  Used by gdn_tree_tc.cu (one
// item per CTA) and by verify_commit.cu (a persistent CTA runs items in turn
// and commits the state it still holds once the request is accepted).
//
// Digest "SpecPilot ...": prerequisites / hybrid recurrent target (gated delta
// rule h_t = a_t (I - b_t k_t k_t^T) h_{t-1} + b_t k_t v_t^T, o_t = h_t^T q_t)
// and technical novelty (recompute along the root path, no per-node
// snapshots).  The formulation is the one of gdn_tree.cu:
//     u_x = A_par Pk_x + sum_{a on path(par)} dec(a -> par) (k_a . k_x) c_a
//     c_x = beta_x v_x - alpha_x beta_x u_x
//     o_x = A_x   Pq_x + sum_{a on path(x)}   dec(a -> x)   (k_a . q_x) c_a
// with P = h0^T [K; Q] the only d_k x d_v-sized work, and the state after a
// root path ending at x is h_x = A_x h0 + sum_{a on path(x)} dec(a -> x) k_a c_a^T.
//
// An item (256 threads):
//  1. threads read the fp32 state once and write it as two bf16 terms
//     (h = hi + lo, hi = bf16(h), lo = bf16(h - hi): ~16 significant bits, the
//     product keeps fp32 accuracy to ~2^-17) in the MN-major 128-byte-swizzled
//     layout, one half of the d_k rows at a time through one 32 KB buffer (the
//     second half's lines are prefetched into L2 meanwhile), optionally also
//     keeping the fp32 state in shared memory; TMA brings the K and Q rows of
//     the q-k head (K-major, 32 rows each) and the v rows;
//  2. one thread issues 2 x 4 tcgen05.mma for P per half (M = 128 state
//     columns, N = 64 rows of [K; Q], K = 16) and 8 more for the Gram rows
//     [K; Q] K^T; both accumulate in tensor memory;
//  3. P and the Gram rows move to shared memory (over the dead state terms);
//     with the tree, one thread per row turns its ancestor mask into dense
//     weight rows (decay x Gram entry on the root path, zero elsewhere); one
//     thread per state column then forms the write vectors and outputs of all
//     rows in index order (ancestors first) with the write vectors held in
//     registers: dense, fully unrolled FMA chains without dependent loads.
// Everything up to 3 needs no tree.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc_util.cuh"

namespace spec {
namespace gdn_tc {

using namespace tc;

constexpr int DKV = 128;                     // d_k = d_v
constexpr int NT = 256;
constexpr uint32_t A_PART = DKV * DKV;       // one bf16 term of half the state rows: 16 KB
constexpr int TPM = 32;                      // rows of a tree (padded)
constexpr int NM = 2 * TPM;                  // rows of [K; Q]
constexpr uint32_t kTmemCols = 128;          // P: 64 columns, Gram: 32 more

struct Layout {
    // byte offsets from the 1024-aligned shared-memory base.  The state goes
    // through the tensor cores in two halves of d_k rows, each as two bf16
    // terms (hi, lo).  After the MMAs the terms' space holds P [N][128] and
    // the dead K/Q tile the Gram rows G [N][TP] (fp32).  h32: the fp32 state
    // [128][128] when an item keeps it for a commit.
    uint32_t a_hi, a_lo, p, g, b, v, nodes, h32, bar, total;
};

__host__ __device__ inline Layout layout(bool keep_state) {
    Layout L;
    uint32_t o = 0;
    L.a_hi = o; o += A_PART;
    L.a_lo = o; o += A_PART;
    L.p = 0;                                             // P: 32 KB over both terms
    L.b = o;    o += 2u * NM * 128;                      // [2 halves][64 rows][64] bf16, swizzled
    L.g = L.b;                                           // G: 8 KB over the K/Q tile
    L.v = o;    o += 2u * TPM * 128;                     // [2 halves][32 rows][64] bf16
    L.nodes = o;
    o += 4u * (4 * TPM + 2 * TPM * TPM + TPM);           // al be A Ap | Wu Wo [TP][TP] | masks
    L.h32 = 0;
    if (keep_state) {
        L.h32 = (o + 15) / 16 * 16;
        o = L.h32 + 4u * DKV * DKV;
    }
    L.bar = (o + 7) / 8 * 8;
    o = L.bar + 24 + 16;                                 // 3 mbarriers, TMEM slot, abort flag, issued
    L.total = o + 1024;                                  // alignment slack
    return L;
}

__device__ __forceinline__ unsigned char* aligned_base(unsigned char* raw) {
    return reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Once per CTA (thread 0 / warp 1 / every thread as marked), before any item.
__device__ __forceinline__ uint32_t setup(unsigned char* sm, const Layout& L) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 3);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    __syncthreads();
    tc_fence_after();
    return *tmem_slot;
}

// Once per CTA after its last item (every thread).
__device__ __forceinline__ void teardown(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

struct Item {
    int j, b;                    // v-head, request
    int row0;                    // first TMA row of the request: (layer B + b) T
    const float* h0;             // the layer's state [B][Hv][128][128]
    const float* alpha;          // the layer's gates [B][T][Hv]
    const float* beta;
    __nv_bfloat16* o;            // the layer's outputs [B][T][Hv][128]
    float* c_out;                // NULL or [B][T][Hv][128]
};

struct NoEpilogue {
    __device__ __forceinline__ void operator()(int, int) const {}
};

// One item, called by all NT threads of the CTA.  ph: the parity of this
// item's phase of the three mbarriers (items alternate).  wait_before_tree:
// run the programmatic wait before the first read of the tree.  When L keeps
// the state, its fp32 copy is in L.h32 afterwards.  epi(col, nn) runs on
// threads 0..127 (state column col) after the rows; the column's write-vector
// entry of row x < nn is then at L.p + 4 (x 128 + col).  Returns false when a
// bounded wait gave up (SPEC_DEV_TIMEOUT raised; nothing in flight any more).
template <class Epi>
__device__ bool item(const CUtensorMap* mk, const CUtensorMap* mq, const CUtensorMap* mv,
                     const spec_cfg& c, const spec_tree& tree, const Item& it, void* ws,
                     unsigned char* sm, const Layout& L, uint32_t tmem, uint32_t ph,
                     bool wait_before_tree, Epi&& epi) {
    const int T = c.N + 1, Hv = c.Hv, Hk = c.Hk;
    const int j = it.j, b = it.b;
    const int ih = j / (Hv / Hk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar);      // [0] TMA, [1] MMA, [2] first half
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* issued = reinterpret_cast<volatile int*>(tmem_slot + 2);   // halves issued
    float* nodes = reinterpret_cast<float*>(sm + L.nodes);
    float* al = nodes;
    float* be = al + TPM;
    float* A = be + TPM;
    float* Ap = A + TPM;
    float* Wu = Ap + TPM;            // [x][a]: dec(a -> parent(x)) (k_a . k_x), a on path(parent(x))
    float* Wo = Wu + TPM * TPM;      // [x][a]: dec(a -> x) (k_a . q_x), a on path(x); 0 elsewhere
    uint32_t* ancm = reinterpret_cast<uint32_t*>(Wo + TPM * TPM);   // [x]: ancestors-or-self of x
    float* h32 = L.h32 ? reinterpret_cast<float*>(sm + L.h32) : nullptr;

    __syncthreads();                 // the previous item is done with shared memory
    if (tid == 0) {
        *abort_flag = 0;
        *issued = 0;
    }
    __syncthreads();

    // ---- 1. TMA: K and Q rows of q-k head ih (K-major), v rows of head j -----------
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 3u * 2u * TPM * 128);
        for (int h = 0; h < 2; ++h) {
            unsigned char* bh = sm + L.b + h * NM * 128;
            tma_load_3d(bh, mk, &bar[0], h * 64, ih, it.row0);
            tma_load_3d(bh + TPM * 128, mq, &bar[0], h * 64, ih, it.row0);
            tma_load_3d(sm + L.v + h * TPM * 128, mv, &bar[0], h * 64, j, it.row0);
        }
    }
    // ---- 1./2. the state as two bf16 terms, MN-major, 128-byte swizzle, one half of
    // the d_k rows at a time; the tensor cores form P = h0^T [K; Q] half by half
    // (two bf16 terms of h0) and the Gram rows G = [K; Q] K^T (exact bf16 products).
    const float* hsrc = it.h0 + ((size_t)b * Hv + j) * DKV * DKV;
    // 16-byte chunk = 8 consecutive columns of one row; 1024 chunks per half,
    // 4 per thread: chunk i of half hh is row 64 hh + (tid + i NT) / 16
    constexpr int CPT = DKV * 8 / NT;
    auto load_half = [&](int hh, float4* xr) {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int idx = tid + i * NT, r = 64 * hh + (idx >> 4), ch = idx & 15;
            xr[2 * i] = *reinterpret_cast<const float4*>(hsrc + r * DKV + ch * 8);
            xr[2 * i + 1] = *reinterpret_cast<const float4*>(hsrc + r * DKV + ch * 8 + 4);
        }
    };
    auto store_half = [&](int hh, const float4* xr) {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int idx = tid + i * NT, r = idx >> 4, ch = idx & 15;
            if (h32) {
                float4* d = reinterpret_cast<float4*>(h32 + (64 * hh + r) * DKV + ch * 8);
                d[0] = xr[2 * i];
                d[1] = xr[2 * i + 1];
            }
            const float xs[8] = {xr[2 * i].x, xr[2 * i].y, xr[2 * i].z, xr[2 * i].w,
                                 xr[2 * i + 1].x, xr[2 * i + 1].y, xr[2 * i + 1].z, xr[2 * i + 1].w};
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(xs[2 * e], xs[2 * e + 1]);
                const float2 hf = __bfloat1622float2(h2);
                const __nv_bfloat162 l2 = __floats2bfloat162_rn(xs[2 * e] - hf.x, xs[2 * e + 1] - hf.y);
                hw[e] = *reinterpret_cast<const uint32_t*>(&h2);
                lw[e] = *reinterpret_cast<const uint32_t*>(&l2);
            }
            const uint32_t off = (ch >> 3) * (A_PART / 2) + sw128_offset(r, (ch & 7) * 8);
            *reinterpret_cast<uint4*>(sm + L.a_hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(sm + L.a_lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
    };
    // the MMAs of half hh (and, after the second, the Gram rows); one thread
    auto issue_half = [&](int hh) {
        const uint32_t idP = idesc_bf16_f32(128, NM, /*a_mn=*/true, /*b_mn=*/false);
        const uint32_t b_s = smem_u32(sm + L.b);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const uint32_t a_s = smem_u32(sm + (part ? L.a_lo : L.a_hi));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sdesc_sw128(a_s + kk * 2048, A_PART / 2, 1024);
                const uint64_t bd = sdesc_sw128(b_s + hh * NM * 128 + kk * 32, 16, 1024);
                mma_bf16(tmem, ad, bd, idP, (hh | part | kk) != 0);
            }
        }
        if (hh == 1) {
            // Gram: A = the [K; Q] rows (M = 128 rows read, the first 64
            // meaningful), B = the K rows (N = 32); both K-major over d_k
            const uint32_t idG = idesc_bf16_f32(128, TPM, false, false);
#pragma unroll
            for (int ks = 0; ks < DKV / 16; ++ks) {
                const uint32_t off = (ks >> 2) * NM * 128 + (ks & 3) * 32;
                mma_bf16(tmem + NM, sdesc_sw128(b_s + off, 16, 1024),
                         sdesc_sw128(b_s + off, 16, 1024), idG, ks != 0);
            }
        }
        mma_commit(&bar[hh ? 1 : 2]);
        *issued = hh + 1;
    };
    float4 xr[2 * CPT];
    load_half(0, xr);
#pragma unroll
    for (int i = 0; i < CPT; ++i) {          // the second half's lines on their way to L2
        const int idx = tid + i * NT;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(hsrc + (64 + (idx >> 4)) * DKV + (idx & 15) * 8));
    }
    store_half(0, xr);
    if (tid < T) {
        al[tid] = it.alpha[((size_t)b * T + tid) * Hv + j];
        be[tid] = it.beta[((size_t)b * T + tid) * Hv + j];
    }
    fence_async_smem();
    __syncthreads();
    bool ok = true;
    if (warp == 1 && lane == 0) {
        ok = mbar_wait(&bar[0], ph, abort_flag);
        if (ok) {
            tc_fence_after();
            issue_half(0);
        }
    }
    load_half(1, xr);
    // the first half's MMAs have read the terms: write the second half over them
    if (!__syncthreads_and(ok && mbar_wait(&bar[2], ph, abort_flag))) {
        ok = false;
    } else {
        store_half(1, xr);
        fence_async_smem();
        __syncthreads();
        if (warp == 1 && lane == 0) {
            tc_fence_after();
            issue_half(1);
        }
    }
    // P -> smem [64][128] and G -> smem [64][32] (over the dead state terms); warp
    // w < 4 owns tensor-memory lanes 32w..32w+31
    float* P = reinterpret_cast<float*>(sm + L.p);
    float* Gs = reinterpret_cast<float*>(sm + L.g);
    if (warp < 4 && ok) {
        const bool w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[1], ph, abort_flag));
        if (w_ok) {
            tc_fence_after();
            const uint32_t la = (uint32_t)(warp * 32) << 16;
            const int col = warp * 32 + lane;
            float pv[32];
#pragma unroll
            for (int n0 = 0; n0 < NM; n0 += 32) {
                tmem_ld32(tmem + la + n0, pv);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) P[(n0 + i) * DKV + col] = pv[i];
            }
            if (warp < 2) {                      // Gram rows 0..63 live in lanes 0..63
                tmem_ld32(tmem + la + NM, pv);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) Gs[col * TPM + i] = pv[i];
            }
        } else {
            ok = false;
        }
    }
    if (!ok) {
        *abort_flag = 1;
        raise_status(ws, SPEC_DEV_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) {          // let the TMA copies and issued MMAs land before leaving
            int never = 0;
            mbar_wait(&bar[0], ph, &never);
            if (*issued >= 1) mbar_wait(&bar[2], ph, &never);
            if (*issued >= 2) mbar_wait(&bar[1], ph, &never);
        }
        __syncthreads();
        return false;
    }

    // ---- 3. the tree ----------------------------------------------------------------
    if (wait_before_tree) {
        pdl_wait();
        pdl_trigger();
    }
    int nn = tree.n_nodes[b];
    nn = nn < 1 ? 1 : (nn > T ? T : nn);
    // row x's ancestors-or-self are the set bits of its mask, in root-to-x order
    uint32_t anc = 0;
    if (tid < TPM) anc = tid < nn ? static_cast<uint32_t>(tree.node_anc[2 * ((size_t)b * T + tid)]) : 0u;
    for (int i = tid; i < 2 * TPM * TPM; i += NT) Wu[i] = 0.0f;   // Wu and Wo are adjacent
    __syncthreads();
    if (tid < nn) {                            // decays and Gram weights of row x
        const int x = tid;
        ancm[x] = anc;
        float acc = 1.0f;                      // dec(a -> x), walking from x up
        for (uint32_t m = anc; m; m &= ~(1u << (31 - __clz(m)))) {
            const int a = 31 - __clz(m);
            Wo[x * TPM + a] = acc * Gs[(TPM + x) * TPM + a];
            acc *= al[a];
        }
        A[x] = acc;
        acc = 1.0f;                            // dec(a -> parent(x)), a strict ancestor
        for (uint32_t m = anc & ~(1u << x); m; m &= ~(1u << (31 - __clz(m)))) {
            const int a = 31 - __clz(m);
            Wu[x * TPM + a] = acc * Gs[x * TPM + a];
            acc *= al[a];
        }
        Ap[x] = acc;
    }
    __syncthreads();

    // ---- write vectors and outputs: one state column per thread; the column's
    // write vectors of all rows stay in registers (rows in index order, a row's
    // ancestors come first), so every sum is a dense unrolled FMA chain over the
    // weight rows (zero off the root path).  Each row's write vector also goes
    // over its consumed P[K] entry (C[x][col] = c_x[col] at P[x][col]) for an
    // epilogue that commits the state.
    if (tid < DKV) {
        const int col = tid, vh = col >> 6, vc = col & 63;
        const __nv_bfloat16* vs = reinterpret_cast<const __nv_bfloat16*>(sm + L.v);
        float cc[TPM];
#pragma unroll
        for (int x = 0; x < TPM; ++x) {
            if (x >= nn) break;
            float u0 = Ap[x] * P[x * DKV + col], u1 = 0.0f;
            float o0 = 0.0f, o1 = 0.0f;
            const float4* wu4 = reinterpret_cast<const float4*>(Wu + x * TPM);
            const float4* wo4 = reinterpret_cast<const float4*>(Wo + x * TPM);
#pragma unroll
            for (int a4 = 0; a4 < TPM / 4; ++a4) {
                if (4 * a4 >= x) break;
                const float4 wu = wu4[a4], wo = wo4[a4];
                const float c0 = cc[4 * a4], c1 = 4 * a4 + 1 < x ? cc[4 * a4 + 1] : 0.0f;
                const float c2 = 4 * a4 + 2 < x ? cc[4 * a4 + 2] : 0.0f;
                const float c3 = 4 * a4 + 3 < x ? cc[4 * a4 + 3] : 0.0f;
                u0 = fmaf(wu.x, c0, fmaf(wu.z, c2, u0));
                u1 = fmaf(wu.y, c1, fmaf(wu.w, c3, u1));
                o0 = fmaf(wo.x, c0, fmaf(wo.z, c2, o0));
                o1 = fmaf(wo.y, c1, fmaf(wo.w, c3, o1));
            }
            const float vx = __bfloat162float(vs[(vh * TPM + x) * 64 + vc]);
            const float cx = be[x] * vx - al[x] * be[x] * (u0 + u1);
            cc[x] = cx;
            P[x * DKV + col] = cx;
            const float ox = fmaf(Wo[x * TPM + x], cx, fmaf(A[x], P[(TPM + x) * DKV + col], o0 + o1));
            const size_t oi = (((size_t)b * T + x) * Hv + j) * DKV + col;
            it.o[oi] = __float2bfloat16_rn(ox);
            if (it.c_out) it.c_out[oi] = cx;
        }
        epi(col, nn);
    } else {
        // padding rows x in [nn, T): zero outputs
        for (int i = tid - DKV; i < (T - nn) * DKV; i += NT - DKV) {
            const int x = nn + i / DKV, col = i % DKV;
            const size_t oi = (((size_t)b * T + x) * Hv + j) * DKV + col;
            it.o[oi] = __float2bfloat16_rn(0.0f);
            if (it.c_out) it.c_out[oi] = 0.0f;
        }
    }
    return true;
}

// ---- tensor maps ------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// bf16 rows [rows_total][H][128] as a 3-D tensor map, box {64, 1, box_rows}.
inline bool rows_map(CUtensorMap* m, const void* base, int H, int rows_total, int box_rows,
                     CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)DKV, (cuuint64_t)H, (cuuint64_t)rows_total};
    cuuint64_t str[2] = {(cuuint64_t)DKV * 2, (cuuint64_t)H * DKV * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdn_tc
}  // namespace spec
