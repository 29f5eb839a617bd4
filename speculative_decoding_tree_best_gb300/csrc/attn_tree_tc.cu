// attn_tree_tc.cu -- tensor-core (tcgen05) split-KV partial for tree attention,
// bf16 I/O, head dim 128.
//
// Digest "SpecPilot ...": prerequisites / draft-tree verification (one target
// pass verifies the tree; every node sees only its ancestors).
//
// One CTA = one (request, kv-head, 128-row query tile, key chunk).  The query
// tile holds the G = Hq/Hkv q-heads of the group for 128/G consecutive tree
// rows (row r = node * G + head_in_group), loaded once by TMA.  The chunk's
// keys stream through two-stage rings of 128-key K and V blocks (TMA, 128-byte
// swizzle); a K stage is refilled as soon as its S product is done, a V stage
// once its PV product is done.  Per block j:
//    S_j = Q K_j^T          tcgen05.mma (bf16, exact products), fp32 in tensor
//                           memory, two S buffers so S_{j+1} is ready while
//                           the softmax works on S_j
//    P_j = exp2(S_j c - m)  one thread per (row, 32 keys), written as fp16
//                           (11 significant bits; a bf16 P would cost ~1.7e-3
//                           relative error on O)
//    V_j -> fp16            the softmax threads convert V_j in place (the same
//                           swizzled layout), so PV runs as kind::f16 with f16
//                           operands
//    O += P_j V_j           tcgen05.mma, fp32 in tensor memory
// The MMA order is S_0, S_1, PV_0, S_2, PV_1, ...  The running maximum is only
// raised (and O rescaled in tensor memory) when a block's maximum exceeds it by
// more than 2^8, so P <= 256.  The chunk's output is stored normalised
// (O / sum) in fp16 with its (max, sum); |V| must stay below the fp16 range
// (65504).  Warp roles: warp 0 loads Q and the K ring, warp 1 issues the MMAs
// (one thread each), warp 2 loads the V ring, warps 3-18 run the softmax: four
// threads per query row (tensor-memory lane = row), each owning 32 of the 128
// key columns.  The partial (O, max, sum) goes to the workspace; attn_merge
// combines chunks.
//
// The cache chunks read nothing from the tree; only the tree chunk (the T
// tree rows as keys, masked by the ancestor bitmasks) does.
//
// Every mbarrier wait is bounded (about one second): on timeout the CTA raises
// SPEC_DEV_TIMEOUT, every role unwinds, and tensor memory is freed.
#include <cuda.h>
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace spec {

namespace {

using namespace tc;

constexpr int NB = 128;             // keys per block
constexpr int BM = 128;             // query rows per tile
constexpr int HD = 128;             // head dim
constexpr int NWG = 4;              // softmax warpgroups: thread (wg, row) owns 32 key columns
constexpr int CPT = 128 / NWG;      // key (and output) columns per softmax thread
constexpr int NSOFT = 128 * NWG;    // softmax threads
constexpr int NROLE = 3;            // warps 0-2: K loads, MMA issue, V loads
constexpr int NTHREADS = 32 * NROLE + NSOFT;
constexpr uint32_t TILE_BYTES = 128 * 128 * 2;   // one 128 x 128 16-bit tile (two 64-wide halves)
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;
constexpr uint32_t TMEM_COLS = 512;              // S0, S1, O (128 columns each), rounded up

// shared-memory map (offsets from the 1024-aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;                   // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE_BYTES;               // 2 stages
constexpr uint32_t OFF_P = OFF_V + 2 * TILE_BYTES;               // fp16 P, K-major
constexpr uint32_t OFF_RED = OFF_P + TILE_BYTES;                 // float [2][NWG][128] row maxima
constexpr uint32_t OFF_REDL = OFF_RED + 2 * NWG * 128 * 4;       // float [NWG][128] row sums
constexpr uint32_t OFF_BAR = OFF_REDL + NWG * 128 * 4;
enum { B_Q = 0, B_KF, B_VF = B_KF + 2, B_KE = B_VF + 2, B_VE = B_KE + 2, B_SFULL = B_VE + 2,
       B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE, NBARS };
constexpr uint32_t SMEM_BYTES = OFF_BAR + NBARS * 8 + 32 + 1024;  // + slack for alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// Barrier over `nthreads` threads with id `id` that also ANDs a predicate, so
// a pair of warps leaves a loop together.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Eight bf16 (one 16-byte chunk) to eight fp16, in place.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
        const __half2 h = __floats2half2_rn(lo, hi);
        w[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

struct TcParams {
    spec_cfg c;
    spec_tree tree;
    const int32_t* kv_len;
    void* ws;
    WsLayout w;
};

__global__ void __launch_bounds__(NTHREADS, 1)
attn_tc_partial(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mkc,
                const __grid_constant__ CUtensorMap mvc, const __grid_constant__ CUtensorMap mkt,
                const __grid_constant__ CUtensorMap mvt, const TcParams prm) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued_k = reinterpret_cast<int*>(tmem_slot + 2);       // K blocks the producer issued
    int* issued_v = reinterpret_cast<int*>(tmem_slot + 3);       // V blocks the producer issued

    const spec_cfg& c = prm.c;
    const WsLayout& w = prm.w;
    const int T = c.N + 1, G = c.Hq / c.Hkv;
    const int ch = blockIdx.x, g = blockIdx.y % c.Hkv, mt = blockIdx.y / c.Hkv, b = blockIdx.z;
    const bool tree_chunk = ch == w.n_split;
    int L = prm.kv_len[b];
    L = L < 0 ? 0 : (L > c.Lmax ? c.Lmax : L);
    int k0 = 0, k1 = T;
    if (!tree_chunk) {
        k0 = ch * w.chunk;
        if (k0 >= L) {
            // no cache rows here: leave an empty partial (max -inf, sum 0) so the
            // merge needs no kv_len, and exit (nothing allocated yet)
            float2* wML = ws_ptr<float2>(prm.ws, w.attn_ml_off);
            const size_t tile = (((size_t)b * c.Hkv + g) * w.n_mt + mt) * w.n_chunks + ch;
            for (int row = threadIdx.x; row < BM; row += NTHREADS)
                if (mt * BM + row < G * T) wML[tile * BM + row] = make_float2(-INFINITY, 0.0f);
            return;
        }
        k1 = min(k0 + w.chunk, L);
    }
    const int nblk = (k1 - k0 + NB - 1) / NB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bar[B_Q], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[B_KF + s], 1);
            mbar_init(&bar[B_VF + s], 1);
            mbar_init(&bar[B_KE + s], 1);
            mbar_init(&bar[B_VE + s], 1);
            mbar_init(&bar[B_SFULL + s], 1);
            mbar_init(&bar[B_SFREE + s], NSOFT);
        }
        mbar_init(&bar[B_PFULL], NSOFT);
        mbar_init(&bar[B_PVDONE], 1);
        *abort_flag = 0;
        *issued_k = 0;
        *issued_v = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(tree_chunk ? &mkt : &mkc);
        tma_prefetch_desc(tree_chunk ? &mvt : &mvc);
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + 256;                  // S buffers at +0 and +128
    bool ok = true;
    const CUtensorMap* mk = tree_chunk ? &mkt : &mkc;
    const CUtensorMap* mv = tree_chunk ? &mvt : &mvc;

    if (warp == 0) {
        // ------------------------------------------------------------ Q and the K ring
        if (lane == 0) {
            mbar_arrive_expect_tx(&bar[B_Q], TILE_BYTES);
            const int node0 = mt * (BM / G);
            for (int h = 0; h < 2; ++h)
                tma_load_3d(sm + OFF_Q + h * HALF_BYTES, &mq, &bar[B_Q], h * 64, g * G,
                            b * T + node0);
            for (int j = 0; j < nblk; ++j) {
                const int s = j & 1;
                // stage s is free once S_{j-2} is done
                if (j >= 2 && !mbar_wait(&bar[B_KE + s], ((j >> 1) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bar[B_KF + s], TILE_BYTES);
                for (int h = 0; h < 2; ++h)
                    tma_load_4d(sm + OFF_K + s * TILE_BYTES + h * HALF_BYTES, mk, &bar[B_KF + s],
                                h * 64, g, k0 + j * NB, b);
                *issued_k = j + 1;
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ the V ring
        if (lane == 0) {
            for (int j = 0; j < nblk; ++j) {
                const int s = j & 1;
                // stage s is free once PV_{j-2} is done
                if (j >= 2 && !mbar_wait(&bar[B_VE + s], ((j >> 1) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bar[B_VF + s], TILE_BYTES);
                for (int h = 0; h < 2; ++h)
                    tma_load_4d(sm + OFF_V + s * TILE_BYTES + h * HALF_BYTES, mv, &bar[B_VF + s],
                                h * 64, g, k0 + j * NB, b);
                *issued_v = j + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(128, NB, false, false);
            const uint32_t idPV = idesc_f16_f32(128, HD, false, true);
            const uint32_t q_s = smem_u32(sm + OFF_Q);
            const uint32_t p_s = smem_u32(sm + OFF_P);
            // S_i = Q K_i^T into S buffer i & 1
            auto issue_s = [&](int i) -> bool {
                const int s = i & 1;
                if (!mbar_wait(&bar[B_KF + s], (i >> 1) & 1, abort_flag)) return false;
                // the softmax has read S_{i-2} out of this buffer
                if (i >= 2 && !mbar_wait(&bar[B_SFREE + s], ((i >> 1) - 1) & 1, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t k_s = smem_u32(sm + OFF_K + s * TILE_BYTES);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint32_t off = (k >> 2) * HALF_BYTES + (k & 3) * 32;
                    mma_bf16(tmem + s * 128, sdesc_sw128(q_s + off, 16, 1024),
                             sdesc_sw128(k_s + off, 16, 1024), idS, k > 0);
                }
                mma_commit(&bar[B_SFULL + s]);
                mma_commit(&bar[B_KE + s]);
                return true;
            };
            ok = mbar_wait(&bar[B_Q], 0, abort_flag);
            if (ok) ok = issue_s(0);
            if (ok && nblk > 1) ok = issue_s(1);
            for (int j = 0; j < nblk && ok; ++j) {
                const int s = j & 1;
                // P_j written and V_j converted to fp16 by the softmax threads
                if (!mbar_wait(&bar[B_PFULL], j & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t v_s = smem_u32(sm + OFF_V + s * TILE_BYTES);
#pragma unroll
                for (int k = 0; k < NB / 16; ++k) {
                    const uint32_t offp = (k >> 2) * HALF_BYTES + (k & 3) * 32;
                    mma_f16(tO, sdesc_sw128(p_s + offp, 16, 1024),
                            sdesc_sw128(v_s + k * 2048, HALF_BYTES, 1024), idPV, (j > 0 || k > 0));
                }
                mma_commit(&bar[B_PVDONE]);
                mma_commit(&bar[B_VE + s]);
                if (j + 2 < nblk) ok = issue_s(j + 2);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        // Softmax warp sw = warp - NROLE: warpgroup wg = sw / 4 owns key (and
        // output) columns [CPT wg, CPT wg + CPT) of row lg * 32 + lane, where
        // lg = warp % 4 is the tensor-memory lane group the warp may access.
        // The NWG threads of a row swap partial maxima through shared memory
        // under a named barrier over the NWG warps of that lane group.
        const int st = threadIdx.x - 32 * NROLE;           // 0 .. NSOFT-1
        const int wg = (warp - NROLE) >> 2;
        const int lg = warp & 3;
        const int row = lg * 32 + lane;
        const int r = mt * BM + row;                     // query row within (request, kv-head)
        const int x = r / G;
        const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
        const int cb0 = wg * CPT;                        // first column of this thread
        const int grp_bar = 1 + lg;
        constexpr int GRP_THREADS = 32 * NWG;
        float* red = reinterpret_cast<float*>(sm + OFF_RED);
        float* redl = reinterpret_cast<float*>(sm + OFF_REDL);
        uint32_t visbits = 0xffffffffu;                  // tree chunk: visible keys among my columns
        if (tree_chunk) {
            pdl_wait();          // the tree may come from the launch just before
            int nn = prm.tree.n_nodes[b];
            nn = nn < 1 ? 1 : (nn > T ? T : nn);
            visbits = 0u;
            if (x < nn) {
                const uint64_t a = prm.tree.node_anc[2 * ((size_t)b * T + x) + (cb0 >> 6)];
                visbits = static_cast<uint32_t>(a >> (cb0 & 63));
                if (cb0 + CPT > nn) visbits &= (nn - cb0 <= 0) ? 0u : (0xffffffffu >> (32 - (nn - cb0)));
            }
        }
        const float sl2 = 1.4426950408889634f * rsqrtf((float)HD);   // log2(e) / sqrt(D)
        float m_ref = -INFINITY, l = 0.0f;                // m_ref in raw score units
        unsigned char* pbuf = sm + OFF_P;
        float sv[CPT];
        for (int j = 0; j < nblk; ++j) {
            const int s = j & 1;
            bool w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_SFULL + s], (j >> 1) & 1, abort_flag));
            float pm0 = -INFINITY, pm1 = -INFINITY, pm2 = -INFINITY, pm3 = -INFINITY;
            if (w_ok) {
                tc_fence_after();
                tmem_ld32(tmem + s * 128 + lane_addr + cb0, sv);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bar[B_SFREE + s]);
                // visibility: all columns of a full cache block are visible
                uint32_t vis = visbits;
                if (!tree_chunk) {
                    const int nvis = k1 - (k0 + j * NB + cb0);
                    vis = nvis >= CPT ? 0xffffffffu : (nvis <= 0 ? 0u : (0xffffffffu >> (32 - nvis)));
                }
                if (vis != 0xffffffffu) {
#pragma unroll
                    for (int i = 0; i < CPT; ++i) sv[i] = ((vis >> i) & 1u) ? sv[i] : -INFINITY;
                }
#pragma unroll
                for (int i = 0; i < CPT; i += 4) {
                    pm0 = fmaxf(pm0, sv[i]);
                    pm1 = fmaxf(pm1, sv[i + 1]);
                    pm2 = fmaxf(pm2, sv[i + 2]);
                    pm3 = fmaxf(pm3, sv[i + 3]);
                }
                red[((j & 1) * NWG + wg) * 128 + row] = fmaxf(fmaxf(pm0, pm1), fmaxf(pm2, pm3));
            }
            if (!bar_and(grp_bar, GRP_THREADS, w_ok)) { ok = false; break; }
            float mx = red[((j & 1) * NWG) * 128 + row];
#pragma unroll
            for (int k = 1; k < NWG; ++k) mx = fmaxf(mx, red[((j & 1) * NWG + k) * 128 + row]);
            float factor = 1.0f;
            bool rescale = false;
            if (j == 0) {
                m_ref = mx;
            } else if ((mx - m_ref) * sl2 > 8.0f) {
                factor = (m_ref == -INFINITY) ? 0.0f : ex2((m_ref - mx) * sl2);
                m_ref = mx;
                rescale = true;
            }
            const float mu = (m_ref == -INFINITY) ? 0.0f : m_ref * sl2;
            l *= factor;
            float l0 = 0.0f, l1 = 0.0f;
#pragma unroll
            for (int i = 0; i < CPT; i += 2) {
                sv[i] = ex2(fmaf(sv[i], sl2, -mu));
                sv[i + 1] = ex2(fmaf(sv[i + 1], sl2, -mu));
                l0 += sv[i];
                l1 += sv[i + 1];
            }
            l += l0 + l1;
            // V_j to fp16 in place: 16 bytes x 4 per thread
            w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_VF + s], (j >> 1) & 1, abort_flag));
            if (w_ok) {
                uint4* vs = reinterpret_cast<uint4*>(sm + OFF_V + s * TILE_BYTES);
                uint4 vv[TILE_BYTES / 16 / NSOFT];
#pragma unroll
                for (int i = 0; i < TILE_BYTES / 16 / NSOFT; ++i) vv[i] = vs[st + i * NSOFT];
#pragma unroll
                for (int i = 0; i < TILE_BYTES / 16 / NSOFT; ++i)
                    vs[st + i * NSOFT] = bf16x8_to_f16x8(vv[i]);
            }
            // P_j may only overwrite the P buffer once PV_{j-1} is done
            if (j >= 1 && w_ok)
                w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_PVDONE], (j - 1) & 1, abort_flag));
            if (!bar_and(grp_bar, GRP_THREADS, w_ok)) { ok = false; break; }
            if (j >= 1) tc_fence_after();
            if (__any_sync(0xffffffffu, rescale)) {
                float ov[32];
#pragma unroll
                for (int cc = 0; cc < CPT / 32; ++cc) {
                    tmem_ld32(tO + lane_addr + cb0 + cc * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= factor;
                    tmem_st32(tO + lane_addr + cb0 + cc * 32, ov);
                }
                tmem_wait_st();
            }
#pragma unroll
            for (int cb = 0; cb < CPT / 8; ++cb) {         // 16-byte chunks of 8 keys
                uint32_t hw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __half2 h2 = __floats2half2_rn(sv[cb * 8 + 2 * e], sv[cb * 8 + 2 * e + 1]);
                    hw[e] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                const int col = cb0 + cb * 8;              // key column within the block
                const uint32_t off = (col >> 6) * HALF_BYTES + sw128_offset(row, col & 63);
                *reinterpret_cast<uint4*>(pbuf + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[B_PFULL]);
        }
        if (ok) {
            const bool w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_PVDONE], (nblk - 1) & 1, abort_flag));
            ok = bar_and(grp_bar, GRP_THREADS, w_ok);
        }
        if (ok) {
            tc_fence_after();
            __half* wO = ws_ptr<__half>(prm.ws, w.attn_o_off);
            float2* wML = ws_ptr<float2>(prm.ws, w.attn_ml_off);
            const size_t tile = (((size_t)b * c.Hkv + g) * w.n_mt + mt) * w.n_chunks + ch;
            redl[wg * 128 + row] = l;
            bar_and(grp_bar, GRP_THREADS, true);
            float lt = 0.0f;
#pragma unroll
            for (int k = 0; k < NWG; ++k) lt += redl[k * 128 + row];
            const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
            float ov[32];
#pragma unroll
            for (int cc = 0; cc < CPT / 32; ++cc) {
                tmem_ld32(tO + lane_addr + cb0 + cc * 32, ov);
                tmem_wait_ld();
                if (r < G * T) {
                    uint4* dst = reinterpret_cast<uint4*>(wO + (tile * BM + row) * HD + cb0 + cc * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t hv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __half2 h2 = __floats2half2_rn(ov[8 * i + 2 * e] * inv,
                                                                 ov[8 * i + 2 * e + 1] * inv);
                            hv[e] = *reinterpret_cast<const uint32_t*>(&h2);
                        }
                        dst[i] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                    }
                }
            }
            if (wg == 0 && r < G * T)
                // partial max in natural-log units of the scaled score s / sqrt(D)
                wML[tile * BM + row] = make_float2(m_ref * rsqrtf((float)HD), lt);
        }
    }

    if (!ok) {
        *abort_flag = 1;
        raise_status(prm.ws, SPEC_DEV_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (*abort_flag && threadIdx.x == 0) {
        // let the TMA copies still in flight land before the CTA's shared memory
        // is released: wait (bounded) on the phases of the last issued blocks
        int never = 0;
        mbar_wait(&bar[B_Q], 0, &never);
        for (int j = max(0, *issued_k - 2); j < *issued_k; ++j)
            mbar_wait(&bar[B_KF + (j & 1)], (j >> 1) & 1, &never);
        for (int j = max(0, *issued_v - 2); j < *issued_v; ++j)
            mbar_wait(&bar[B_VF + (j & 1)], (j >> 1) & 1, &never);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// bf16 tensor map over `rank` dims (innermost first), box {64, box1, box2, 1}.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
               strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_tc_supported(const spec_cfg& c) {
    const int G = c.Hq / c.Hkv;
    return c.io_dtype == SPEC_IO_BF16 && c.D == HD && G >= 1 && G <= BM && (BM % G) == 0 &&
           c.N + 1 <= NB && encode_fn() != nullptr;
}

cudaError_t launch_attn_tc(const spec_cfg& c, const spec_tree& t, const void* q,
                           const void* k_tree, const void* v_tree, const void* k_cache,
                           const void* v_cache, const int32_t* kv_len, void* ws,
                           const WsLayout& w, cudaStream_t st, bool pdl) {
    const int T = c.N + 1, G = c.Hq / c.Hkv;
    const cuuint64_t e = 2;   // bytes per bf16
    CUtensorMap mq, mkc, mvc, mkt, mvt;
    {
        cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)c.Hq, (cuuint64_t)c.B * T};
        cuuint64_t str[2] = {HD * e, (cuuint64_t)c.Hq * HD * e};
        cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(BM / G)};
        if (!make_map(&mq, q, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)c.Hkv, (cuuint64_t)c.Lmax, (cuuint64_t)c.B};
        cuuint64_t str[3] = {HD * e, (cuuint64_t)c.Hkv * HD * e, (cuuint64_t)c.Lmax * c.Hkv * HD * e};
        cuuint32_t box[4] = {64, 1, NB, 1};
        if (!make_map(&mkc, k_cache, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!make_map(&mvc, v_cache, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)c.Hkv, (cuuint64_t)T, (cuuint64_t)c.B};
        cuuint64_t str[3] = {HD * e, (cuuint64_t)c.Hkv * HD * e, (cuuint64_t)T * c.Hkv * HD * e};
        cuuint32_t box[4] = {64, 1, NB, 1};
        if (!make_map(&mkt, k_tree, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!make_map(&mvt, v_tree, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    TcParams prm{c, t, kv_len, ws, w};
    cudaError_t err = cudaFuncSetAttribute(attn_tc_partial,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    dim3 grid(w.n_chunks, c.Hkv * w.n_mt, c.B);
    return launch_k(pdl, attn_tc_partial, grid, dim3(NTHREADS), SMEM_BYTES, st, mq, mkc, mvc, mkt,
                    mvt, prm);
}

}  // namespace spec
