// gdn_state.cu -- tree-masked Gated DeltaNet, bf16 I/O, d_k = d_v = 128, trees
// of up to 32 rows: one CTA per (request, v-head) state at a time.
//
// Digest "SpecPilot ...": prerequisites / hybrid recurrent target (gated delta
// rule h_t = a_t (I - b_t k_t k_t^T) h_{t-1} + b_t k_t v_t^T, o_t = h_t^T q_t)
// and technical novelty (recompute along the root path, no per-node
// snapshots).  With c_t = b_t v_t - a_t b_t u_t and u_t = h_par^T k_t, one step
// is h_t = a_t h_par + k_t c_t^T, so along a root path
//     c_x = b_x v_x - a_x b_x A_par Pk_x + sum_{a on path(par)} w_xa c_a
//     o_x = A_x Pq_x + sum_{a on path(x)} dec(a -> x) (k_a . q_x) c_a
// with w_xa = -a_x b_x dec(a -> par) (k_a . k_x) and P = h0^T [K; Q] the only
// d_k x d_v-sized work.  Every state column evolves on its own once P, the
// Gram rows [K; Q] K^T and the decays exist.  Eight warps in two warpgroups:
//
//  * warpgroup 1 (warps 4-7) splits the fp32 state (TMA-staged, 128 rows x
//    128 columns as two 64-column halves) into two bf16 terms (hi = h
//    truncated to bf16, lo = bf16(h - hi): ~16 significant bits), in place,
//    one 64-row half of d_k at a time, and after each half issues its tcgen05
//    products
//        D[col][x] += sum_k h0[k][col] [K; Q][x][k]    (state as MN-major A,
//                                                        M = 128 columns)
//    so that tensor-memory lane `col` holds that column's Pk_x, Pq_x.  Its
//    first thread also issues the next item's state and K/Q/v copies and
//    prefetches the item after into L2;
//  * warpgroup 0 (warps 0-3): thread 0 issues, once K and Q are in, the Gram
//    rows G = [K; Q] K^T (exact bf16 products) into tensor memory; warps 0/1
//    turn Gram row x (lane x) and the tree into the weight row of c_x (warp 0)
//    or o_x (warp 1): decay x Gram entry on the root path, zero elsewhere.
//    Then each of the four warps takes 32 state columns (its tensor-memory
//    lane quarter: one warp per SM sub-partition) and runs, one column per
//    lane, the write-vector recursion with the write vectors in registers
//    (right-looking: row x adds its weighted c_x into every later row, two
//    rows per packed FMA; a row without descendants is skipped; padding rows
//    carry zero weights).  The outputs O = C Wo^T + A Pq are three more
//    tcgen05 products (the write vectors and the o weights as bf16 hi/lo
//    terms, the write vectors as A in tensor memory), read back per column.
//
// About 107 KB of shared memory and 256 tensor-memory columns per CTA: two
// CTAs per SM, each with two states in flight (one being split while the
// other's rows run).
#include <cuda.h>

#include "common.cuh"
#include "gdn_tc_body.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace spec {

namespace {

using namespace tc;

constexpr int DKV = 128;                 // d_k = d_v
constexpr int HC = 64;                   // columns per state half (one TMA box, one MMA atom)
constexpr int NT = 256;                  // threads per CTA: two warpgroups
constexpr int TP = 32;                   // tree rows (padded)
// tensor-memory columns: P^T of two items (64 each: [K; Q] rows), the Gram
// rows, the write vectors split into two bf16 terms (two per column), and the
// outputs
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t TM_G = 128, TM_C = 160, TM_O = 192;

// byte offsets from the 1024-aligned base
constexpr uint32_t OFF_KQ = 0;                           // [2 halves][64 rows][64] bf16, swizzled
constexpr uint32_t HALF_ST = DKV * HC * 4;               // one column half of the state: 32 KB
constexpr uint32_t OFF_ST = OFF_KQ + 2 * 64 * 128;       // fp32 [2 column halves][128][64]; in
                                                         // place, per 64-row half kh of a
                                                         // column half: lo tile, then hi tile
constexpr uint32_t VBUF = 2 * TP * HC * 2;               // v of one item: [2 halves][32 rows][64]
constexpr uint32_t OFF_V = OFF_ST + 2 * HALF_ST;         // bf16, two items
constexpr uint32_t OFF_WU = OFF_V + 2 * VBUF;            // WuT[a][y]: c_a in c_y
constexpr uint32_t OFF_WO = OFF_WU + TP * TP * 4;        // Wo [x][hi a | lo a] bf16, swizzled:
                                                         // c_a in o_x
constexpr uint32_t OFF_SM = OFF_WO + TP * 128;           // al be [2][32], A ca [32] fp32
constexpr int NBAR = 7;
constexpr uint32_t OFF_BAR = OFF_SM + 6 * TP * 4;        // mbarriers, TMEM slot, abort flag
constexpr uint32_t SMEM_BYTES = OFF_BAR + 8 * NBAR + 16 + 1024;   // + alignment slack
constexpr uint32_t TX_KQV = 4 * TP * 128 + VBUF;         // K, Q (two halves each), v
constexpr uint32_t TX_ST = 2 * HALF_ST;                  // the state
constexpr uint32_t TILE = 64 * HC * 2;                   // one bf16 term of 64 d_k rows: 8 KB

// the Gram products read A rows 64..127 past each 64-row half of the K/Q tile:
// for the second half those rows are the staged state (valid shared memory)
static_assert(OFF_KQ + 64 * 128 + 128 * 128 <= OFF_ST + 2 * HALF_ST, "A rows stay in smem");
static_assert(OFF_BAR % 8 == 0 && OFF_WO % 1024 == 0 && OFF_ST % 1024 == 0, "alignment");
static_assert(2 * (SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");

__device__ __forceinline__ unsigned char* align1024(unsigned char* raw) {
    return reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

// (x, y) -> bf16x2 of x and y truncated to their upper 16 bits (x in the low half)
__device__ __forceinline__ uint32_t bf16x2_trunc(float x, float y) {
    return __byte_perm(__float_as_uint(x), __float_as_uint(y), 0x7632);
}
__device__ __forceinline__ float trunc_rest(float x) {
    return x - __uint_as_float(__float_as_uint(x) & 0xffff0000u);
}
// x as two bf16 terms hi + lo (hi = bf16(x), lo = bf16(x - hi): ~16 significant
// bits), packed with y's: (hi_x | hi_y << 16), (lo_x | lo_y << 16)
__device__ __forceinline__ void bf16x2_split(float x, float y, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ uint32_t bf16x2_rn(float x, float y) {
    __nv_bfloat162 t = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&t);
}

// named barrier over one warpgroup (id 1: warpgroup 1, id 2: warpgroup 0;
// 0 is __syncthreads)
__device__ __forceinline__ void wg_sync(int id) {
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

__device__ __forceinline__ bool wg_sync_and(int id, bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id)
        : "memory");
    return r != 0;
}

struct ItemIdx {
    int b, j, ih;
};
__device__ __forceinline__ ItemIdx decode(int it, const spec_cfg& c) {
    ItemIdx d;
    d.b = it / c.Hv;
    d.j = it % c.Hv;
    d.ih = d.j / (c.Hv / c.Hk);
    return d;
}

// A persistent grid of at most two CTAs per SM runs the items (request,
// v-head) it = blockIdx.x, blockIdx.x + gridDim.x, ...  Consecutive items of
// one request share K/Q rows (Hv / Hk v-heads per q-k head), so the CTAs
// running at one time share them in L2.  Per item k of a CTA, the four
// mbarriers [0] K/Q/v in, [1] state in, [2] state products done, [3] Gram
// rows done complete once (parity k & 1), as does [6], the output products.
// Item k's products go to the tensor-memory buffer k & 1, and [4 + (k & 1)]
// completes once all four row warps have read that buffer (parity
// (k >> 1) & 1).  Item k + 1's products wait for that (the start of item k's
// rows, not their end), which also keeps [2] from completing item k + 1
// before every row warp has waited for item k.  As soon as item k's products
// and Gram rows have read the staging buffer and the K/Q tile, item k + 1's
// state and K/Q/v copies start (v into the other of two buffers), so
// warpgroup 1 splits item k + 1's state while warpgroup 0 runs item k's
// rows.  early: the
// tree may come from the launch just before, so the programmatic wait
// precedes the first read of it; otherwise the wait ends the kernel.
__global__ void __launch_bounds__(NT, 2)
gdn_state_kernel(const __grid_constant__ CUtensorMap mh, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mv,
                 spec_cfg c, spec_tree tree, const float* __restrict__ alpha,
                 const float* __restrict__ beta, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ c_out, void* ws, bool early, int n_items) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = align1024(smem_raw);
    const int T = c.N + 1, Hv = c.Hv, G = gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* al2 = reinterpret_cast<float*>(sm + OFF_SM);    // [2][TP]: gates of items k, k + 1
    float* be2 = al2 + 2 * TP;
    float* A = be2 + 2 * TP;                               // [TP]
    float* ca = A + TP;                                    // -alpha_x beta_x A_par(x)
    const uint32_t kq_s = smem_u32(sm + OFF_KQ), st_s = smem_u32(sm + OFF_ST);

    auto load_gates = [&](int it, int buf) {               // the lanes of one warp
        const ItemIdx d = decode(it, c);
        al2[buf * TP + lane] = lane < T ? alpha[((size_t)d.b * T + lane) * Hv + d.j] : 0.0f;
        be2[buf * TP + lane] = lane < T ? beta[((size_t)d.b * T + lane) * Hv + d.j] : 0.0f;
    };
    // copies issued: thread 0 issues the first item's, thread 128 the rest (its
    // counts start at 1 so that (n - 1) & 1 is the parity of its last copy)
    int n_st = tid == 128 ? 1 : 0, n_kq = n_st;
    auto issue_state = [&](int it) {
        const ItemIdx d = decode(it, c);
        mbar_arrive_expect_tx(&bar[1], TX_ST);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            tma_load_2d(sm + OFF_ST + h * HALF_ST, &mh, &bar[1], h * HC, (d.b * Hv + d.j) * DKV);
        ++n_st;
    };
    auto issue_kqv = [&](int it, int kv) {             // kv: the item's index in this CTA
        const ItemIdx d = decode(it, c);
        const int row0 = d.b * T;
        mbar_arrive_expect_tx(&bar[0], TX_KQV);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_load_3d(sm + OFF_KQ + h * 64 * 128, &mk, &bar[0], h * 64, d.ih, row0);
            tma_load_3d(sm + OFF_KQ + h * 64 * 128 + TP * 128, &mq, &bar[0], h * 64, d.ih, row0);
            tma_load_3d(sm + OFF_V + (kv & 1) * VBUF + h * (VBUF / 2), &mv, &bar[0], h * HC, d.j,
                        row0);
        }
        ++n_kq;
    };
    auto prefetch_l2 = [&](int it) {       // the item's state and rows into L2
        const ItemIdx d = decode(it, c);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_prefetch_l2_2d(&mh, h * HC, (d.b * Hv + d.j) * DKV);
            tma_prefetch_l2_3d(&mk, h * 64, d.ih, d.b * T);
            tma_prefetch_l2_3d(&mq, h * 64, d.ih, d.b * T);
            tma_prefetch_l2_3d(&mv, h * HC, d.j, d.b * T);
        }
    };

    const int it0 = blockIdx.x;
    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bar[i], i == 4 || i == 5 ? 4 : 1);
        *abort_flag = 0;
        fence_mbar_init();
        issue_state(it0);
        issue_kqv(it0, 0);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    if (warp == 0) load_gates(it0, 0);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp >= 4) {
        // ---- state split and products (warpgroup 1) -------------------------------------
        const int t = tid - 128;               // 0..127
        const int t6 = t & 63;                 // 64 threads per column half
        const uint32_t hbase = OFF_ST + (t >> 6) * HALF_ST;
        const uint32_t idp = idesc_bf16_f32(128, 2 * TP, /*a_mn=*/true, /*b_mn=*/false);
        int n_p = 0;                           // product commits (thread 128)
        bool pending = false;                  // products issued, not yet committed
        int k = 0;
        for (int it = it0; it < n_items && ok; it += G, ++k) {
            const uint32_t ph = k & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[1], ph, abort_flag));
            // the next item's inputs start towards L2 while this one is split
            if (t == 0 && it + G < n_items) prefetch_l2(it + G);
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {
                // d_k rows 64 kh .. 64 kh + 63 of this thread's column half (16 KB of fp32);
                // unit u = t6 + 64 i: row 64 kh + u / 8, columns 8 (u % 8) .. + 7
                const float4* hs = reinterpret_cast<const float4*>(sm + hbase + kh * 2 * TILE);
                float4 xv[16];
                if (ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        xv[2 * i] = hs[2 * (t6 + 64 * i)];
                        xv[2 * i + 1] = hs[2 * (t6 + 64 * i) + 1];
                    }
                }
                ok = wg_sync_and(1, ok);       // the warpgroup holds its values
                if (!ok) break;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int u = t6 + 64 * i, kr = u >> 3, ch = u & 7;
                    const float4 a = xv[2 * i], e = xv[2 * i + 1];
                    const uint4 hi = make_uint4(bf16x2_trunc(a.x, a.y), bf16x2_trunc(a.z, a.w),
                                                bf16x2_trunc(e.x, e.y), bf16x2_trunc(e.z, e.w));
                    const uint4 lo = make_uint4(bf16x2_rn(trunc_rest(a.x), trunc_rest(a.y)),
                                                bf16x2_rn(trunc_rest(a.z), trunc_rest(a.w)),
                                                bf16x2_rn(trunc_rest(e.x), trunc_rest(e.y)),
                                                bf16x2_rn(trunc_rest(e.z), trunc_rest(e.w)));
                    const uint32_t off = sw128_offset(kr, ch * 8);
                    *reinterpret_cast<uint4*>(sm + hbase + kh * 2 * TILE + off) = lo;
                    *reinterpret_cast<uint4*>(sm + hbase + kh * 2 * TILE + TILE + off) = hi;
                }
                fence_async_smem();
                bool go = true;
                if (t == 0 && kh == 0) {
                    // item k - 1's P^T has been read -- so every row warp has seen item
                    // k - 1's products complete before item k's can complete (the
                    // products barrier never runs two phases ahead of a waiter) -- and
                    // this item's K/Q rows are in.  Item k writes the other buffer, so
                    // it waits only for the start of item k - 1's rows.
                    if (k >= 1) go = mbar_wait(&bar[4 + (ph ^ 1)], ((k - 1) >> 1) & 1, abort_flag);
                    go = go && mbar_wait(&bar[0], ph, abort_flag);
                }
                ok = wg_sync_and(1, go);
                if (!ok) break;
                if (t == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // columns 0..63 and, HALF_ST further, 64..127 (M = 128)
                            const uint32_t a_s = st_s + kh * 2 * TILE + part * TILE + kk * 2048;
                            const uint32_t b_s = kq_s + kh * 64 * 128 + kk * 32;
                            mma_bf16(tmem + 2 * TP * ph, sdesc_sw128(a_s, HALF_ST, 1024),
                                     sdesc_sw128(b_s, 16, 1024), idp, (kh | part | kk) != 0);
                        }
                    }
                    pending = true;
                }
            }
            if (t == 0 && pending) {
                mma_commit(&bar[2]);
                ++n_p;
                pending = false;
                if (ok && it + G < n_items) {
                    // the next item's copies once this item's products and Gram rows
                    // have read the staging buffer and the K/Q tile, and item k - 1's
                    // rows (the other v buffer) have read their inputs
                    bool free = mbar_wait(&bar[2], ph, abort_flag) &&
                                mbar_wait(&bar[3], ph, abort_flag);
                    if (k >= 1) free = free && mbar_wait(&bar[4 + (ph ^ 1)], ((k - 1) >> 1) & 1,
                                                         abort_flag);
                    if (free) {
                        issue_state(it + G);
                        issue_kqv(it + G, k + 1);
                    } else {
                        ok = false;
                    }
                }
            }
            ok = wg_sync_and(1, ok);           // the warpgroup leaves the loop together
            if (k == 0 && early) {
                pdl_wait();
                pdl_trigger();
            }
        }
        if (t == 0 && pending) {               // products left in flight by a failure
            mma_commit(&bar[2]);
            ++n_p;
        }
        if (!ok) *abort_flag = 1;
        if (t == 0 && n_p > 0) mbar_wait(&bar[2], (n_p - 1) & 1, nullptr);
    } else {
        // ---- Gram rows, weights, write vectors and outputs (warpgroup 0) ------------------
        int n_g = 0, n_o = 0;                  // Gram and output commits (thread 0)
        // the next item's tree rows and gates are loaded one item ahead (both loads
        // independent of each other); rows past n_nodes are masked at use
        auto tree_of = [&](int it, int& nn, uint32_t& anc) {
            const ItemIdx d = decode(it, c);
            nn = tree.n_nodes[d.b];
            anc = lane < T ? static_cast<uint32_t>(tree.node_anc[2 * ((size_t)d.b * T + lane)]) : 0u;
        };
        auto gates_of = [&](int it, float& a, float& bb) {
            const ItemIdx d = decode(it, c);
            a = lane < T ? alpha[((size_t)d.b * T + lane) * Hv + d.j] : 0.0f;
            bb = lane < T ? beta[((size_t)d.b * T + lane) * Hv + d.j] : 0.0f;
        };
        int nn_next = 0;
        uint32_t anc_next = 0;
        float al_next = 0.0f, be_next = 0.0f;
        if (early) {
            pdl_wait();
            pdl_trigger();
        }
        tree_of(it0, nn_next, anc_next);
        int k = 0;
        for (int it = it0; it < n_items; it += G, ++k) {
            const uint32_t ph = k & 1;
            const ItemIdx d = decode(it, c);
            const float* al = al2 + ph * TP;
            const float* be = be2 + ph * TP;
            const int nn = nn_next < 1 ? 1 : (nn_next > T ? T : nn_next);
            const uint32_t anc = lane < nn ? anc_next : 0u;
            const bool more = it + G < n_items;
            if (more) {                                         // in flight meanwhile
                tree_of(it + G, nn_next, anc_next);
                if (warp == 0) gates_of(it + G, al_next, be_next);
            }
            bool go = true;
            if (warp < 2) {
                if (tid == 0) {
                    go = mbar_wait(&bar[0], ph, abort_flag);
                    if (go) {
                        tc_fence_after();
                        const uint32_t idg = idesc_bf16_f32(128, TP, false, false);
#pragma unroll
                        for (int ks = 0; ks < DKV / 16; ++ks) {
                            const uint32_t off = (ks >> 2) * 64 * 128 + (ks & 3) * 32;
                            mma_bf16(tmem + TM_G, sdesc_sw128(kq_s + off, 16, 1024),
                                     sdesc_sw128(kq_s + off, 16, 1024), idg, ks != 0);
                        }
                    }
                    mma_commit(&bar[3]);
                    ++n_g;
                    if (!go) *abort_flag = 1;
                }
                go = __all_sync(0xffffffffu, mbar_wait(&bar[3], ph, abort_flag));
                if (go) {
                    // the weight rows (item k - 1's readers are done): lane x, Gram row x
                    float w[TP], alr[TP];
                    float acc = 1.0f;
                    tc_fence_after();
                    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + TM_G, w);
#pragma unroll
                    for (int a4 = 0; a4 < TP / 4; ++a4) {
                        const float4 t4 = *reinterpret_cast<const float4*>(al + 4 * a4);
                        alr[4 * a4] = t4.x;
                        alr[4 * a4 + 1] = t4.y;
                        alr[4 * a4 + 2] = t4.z;
                        alr[4 * a4 + 3] = t4.w;
                    }
                    tmem_wait_ld();
                    const uint32_t path = warp == 0 ? anc & ~(1u << lane) : anc;  // parent's / x's
#pragma unroll
                    for (int a = TP - 1; a >= 0; --a) {
                        const bool on = (path >> a) & 1u;
                        w[a] = on ? acc * w[a] : 0.0f;
                        acc = on ? acc * alr[a] : acc;
                    }
                    if (warp == 0) {
                        const float s = -al[lane] * be[lane];
                        float* WuT = reinterpret_cast<float*>(sm + OFF_WU);
#pragma unroll
                        for (int a = 0; a < TP; ++a) WuT[a * TP + lane] = s * w[a];
                        ca[lane] = s * acc;
                    } else {
                        // row x = lane of Wo as [hi(a = 0..31) | lo(a = 0..31)] bf16,
                        // K-major with the 128-byte swizzle (16-byte chunk j of row x
                        // at j ^ (x % 8))
#pragma unroll
                        for (int j = 0; j < TP / 8; ++j) {
                            uint4 hi, lo;
                            bf16x2_split(w[8 * j], w[8 * j + 1], hi.x, lo.x);
                            bf16x2_split(w[8 * j + 2], w[8 * j + 3], hi.y, lo.y);
                            bf16x2_split(w[8 * j + 4], w[8 * j + 5], hi.z, lo.z);
                            bf16x2_split(w[8 * j + 6], w[8 * j + 7], hi.w, lo.w);
                            *reinterpret_cast<uint4*>(sm + OFF_WO + lane * 128 +
                                                      ((j ^ (lane & 7)) << 4)) = hi;
                            *reinterpret_cast<uint4*>(sm + OFF_WO + lane * 128 +
                                                      (((j + 4) ^ (lane & 7)) << 4)) = lo;
                        }
                        fence_async_smem();
                        A[lane] = acc;
                    }
                }
            }
            go = go && mbar_wait(&bar[2], ph, abort_flag);
            ok = wg_sync_and(2, go && *abort_flag == 0);        // the weights are visible
            if (!ok) break;
            tc_fence_after();

            // one state column per lane: warp w owns columns 32 w .. 32 w + 31
            const int cl = warp * 32 + lane;   // column of the state = tensor-memory lane
            const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16) + 2 * TP * ph;
            float pk[TP];
            tmem_ld32(tl, pk);                 // Pk_x of this column, x = 0..31
            tmem_wait_ld();
            const float* WuT = reinterpret_cast<const float*>(sm + OFF_WU);
            const __nv_bfloat16* vs = reinterpret_cast<const __nv_bfloat16*>(
                sm + OFF_V + ph * VBUF + (cl >> 6) * (VBUF / 2)) + (cl & (HC - 1));
            float2 u[TP / 2];                  // rows 2p, 2p + 1
#pragma unroll
            for (int p = 0; p < TP / 2; ++p) {
                u[p].x = fmaf(be[2 * p], __bfloat162float(vs[(2 * p) * HC]), ca[2 * p] * pk[2 * p]);
                u[p].y = fmaf(be[2 * p + 1], __bfloat162float(vs[(2 * p + 1) * HC]),
                              ca[2 * p + 1] * pk[2 * p + 1]);
            }
            // rows with descendants (the strict ancestors of some row): a leaf's
            // weight row is zero, so its step is skipped (a warp-uniform branch)
            const uint32_t inner = __reduce_or_sync(0xffffffffu, anc & ~(1u << lane));
#pragma unroll
            for (int x = 0; x < TP - 1; ++x) {
                if (!((inner >> x) & 1u)) continue;
                float4 wq[TP / 4];
#pragma unroll
                for (int q = (x + 1) / 4; q < TP / 4; ++q)           // the row's weights first
                    wq[q] = *reinterpret_cast<const float4*>(WuT + x * TP + 4 * q);
                const float cx = (x & 1) ? u[x >> 1].y : u[x >> 1].x;   // final
                const float2 cxx = make_float2(cx, cx);
#pragma unroll
                for (int q = (x + 1) / 4; q < TP / 4; ++q) {         // rows 4q .. 4q + 3
                    if (4 * q > x) {
                        u[2 * q] = __ffma2_rn(make_float2(wq[q].x, wq[q].y), cxx, u[2 * q]);
                    } else if (4 * q + 1 > x) {
                        u[2 * q].y = fmaf(wq[q].y, cx, u[2 * q].y);
                    }
                    if (4 * q + 2 > x) {
                        u[2 * q + 1] = __ffma2_rn(make_float2(wq[q].z, wq[q].w), cxx, u[2 * q + 1]);
                    } else {
                        u[2 * q + 1].y = fmaf(wq[q].w, cx, u[2 * q + 1].y);
                    }
                }
            }
            // padding rows' write vectors read as zero (their inputs may be anything)
#pragma unroll
            for (int p = 0; p < TP / 2; ++p) {
                if (2 * p >= nn) u[p].x = 0.0f;
                if (2 * p + 1 >= nn) u[p].y = 0.0f;
            }
            const size_t rs = (size_t)Hv * DKV;                          // row stride
            const size_t ob = ((size_t)d.b * T * Hv + d.j) * DKV + cl;
            if (c_out) {
#pragma unroll
                for (int p = 0; p < TP / 2; ++p) {
                    if (2 * p < T) c_out[ob + (2 * p) * rs] = u[p].x;
                    if (2 * p + 1 < T) c_out[ob + (2 * p + 1) * rs] = u[p].y;
                }
            }
            // outputs on the tensor cores: O[col][x] = sum_a c[col][a] Wo[x][a] as three
            // bf16 products of the split terms (hi hi, lo hi, hi lo), the write vectors
            // of this warp's columns as A in tensor memory (lane = column; c hi in
            // columns TM_C .. + 15, c lo in the next 16)
            {
                uint32_t ch[TP / 2], clo[TP / 2];
#pragma unroll
                for (int p = 0; p < TP / 2; ++p) bf16x2_split(u[p].x, u[p].y, ch[p], clo[p]);
                const uint32_t tq = tmem + ((uint32_t)(warp * 32) << 16);
                tmem_st16(tq + TM_C, ch);
                tmem_st16(tq + TM_C + TP / 2, clo);
            }
            float pq[TP];
            tmem_ld32(tl + TP, pq);            // Pq_x of this column
            tmem_wait_ld();
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[4 + ph]);   // this P^T buffer is free again
            tc_fence_before();
            wg_sync(2);                        // every column's write vectors are in place
            if (tid == 0) {
                tc_fence_after();
                const uint32_t idt = idesc_bf16_f32(128, TP, false, false);
                const uint32_t wo_s = smem_u32(sm + OFF_WO);
#pragma unroll
                for (int m3 = 0; m3 < 3; ++m3) {
                    const uint32_t a_c = TM_C + (m3 == 1 ? TP / 2 : 0);   // c hi, c lo, c hi
                    const uint32_t b_w = wo_s + (m3 == 2 ? 2 * TP : 0);   // Wo hi, hi, lo
#pragma unroll
                    for (int s16 = 0; s16 < TP / 16; ++s16)             // K = 16 per product
                        mma_f16_tmem_a(tmem + TM_O, tmem + a_c + 8 * s16,
                                       sdesc_sw128(b_w + s16 * 32, 16, 1024), idt,
                                       (m3 | s16) != 0);
                }
                mma_commit(&bar[6]);
                ++n_o;
            }
            const bool o_ok = __all_sync(0xffffffffu, mbar_wait(&bar[6], ph, abort_flag));
            if (o_ok) {
                tc_fence_after();
                float ov[TP];
                tmem_ld32(tl - 2 * TP * ph + TM_O, ov);
                tmem_wait_ld();
                tc_fence_before();
                const size_t rs = (size_t)Hv * DKV;                      // row stride
                const size_t ob = ((size_t)d.b * T * Hv + d.j) * DKV + cl;
#pragma unroll
                for (int x4 = 0; x4 < TP / 4; ++x4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(A + 4 * x4);   // A_x
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int x = 4 * x4 + e;
                        if (x < T)
                            o[ob + x * rs] = __float2bfloat16_rn(
                                x < nn ? fmaf(av[e], pq[x], ov[x]) : 0.0f);
                    }
                }
            }
            // the next item's gates go to the other buffer (this item's readers are done)
            if (warp == 0 && more) {
                al2[(ph ^ 1) * TP + lane] = al_next;
                be2[(ph ^ 1) * TP + lane] = be_next;
            }
            ok = wg_sync_and(2, o_ok && *abort_flag == 0);
            if (!ok) break;
        }
        if (!ok) *abort_flag = 1;
        if (tid == 0 && n_g > 0) mbar_wait(&bar[3], (n_g - 1) & 1, nullptr);
        if (tid == 0 && n_o > 0) mbar_wait(&bar[6], (n_o - 1) & 1, nullptr);
    }

    // ---- teardown ------------------------------------------------------------------------
    ok = __syncthreads_and(ok && *abort_flag == 0);
    if (!ok) {
        raise_status(ws, SPEC_DEV_TIMEOUT);
        if (tid == 0 || tid == 128) {      // let the copies in flight land before leaving
            if (n_kq > 0) mbar_wait(&bar[0], (n_kq - 1) & 1, nullptr);
            if (n_st > 0) mbar_wait(&bar[1], (n_st - 1) & 1, nullptr);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }
}

// fp32 state [rows][128] as a 2-D tensor map, box {64 columns, 128 rows}.
bool state_map(CUtensorMap* m, const float* base, int rows) {
    gdn_tc::EncodeTiledFn enc = gdn_tc::encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)DKV, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)DKV * 4};
    cuuint32_t box[2] = {(cuuint32_t)HC, (cuuint32_t)DKV};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 rows [rows][H][128] as a 3-D tensor map, box {64 columns, 1, TP rows}.
bool vslice_map(CUtensorMap* m, const void* base, int H, int rows) {
    gdn_tc::EncodeTiledFn enc = gdn_tc::encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)DKV, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t str[2] = {(cuuint64_t)DKV * 2, (cuuint64_t)H * DKV * 2};
    cuuint32_t box[3] = {(cuuint32_t)HC, 1, (cuuint32_t)TP};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gdn_state_supported(const spec_cfg& c) {
    return c.io_dtype == SPEC_IO_BF16 && c.dk == DKV && c.dv == DKV && c.N + 1 <= TP &&
           gdn_tc::encode_fn() != nullptr;
}

cudaError_t launch_gdn_state(const spec_cfg& c, const spec_tree& t, const float* h0,
                             const void* q, const void* k, const void* v, const float* alpha,
                             const float* beta, void* o, float* c_out, void* ws, cudaStream_t st,
                             bool pdl, bool early) {
    const int T = c.N + 1;
    CUtensorMap mh, mk, mq, mv;
    if (!state_map(&mh, h0, c.B * c.Hv * DKV) ||
        !gdn_tc::rows_map(&mk, k, c.Hk, c.B * T, TP, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !gdn_tc::rows_map(&mq, q, c.Hk, c.B * T, TP, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !vslice_map(&mv, v, c.Hv, c.B * T))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_state_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int n_items = c.Hv * c.B;
    const int grid = n_items < 2 * sms ? n_items : 2 * sms;       // two CTAs per SM
    // without programmatic launch the tree is complete when the kernel starts
    return launch_k(pdl, gdn_state_kernel, dim3(grid), dim3(NT), SMEM_BYTES, st, mh, mk, mq, mv,
                    c, t, alpha, beta, static_cast<__nv_bfloat16*>(o), c_out, ws, early && pdl,
                    n_items);
}

}  // namespace spec
