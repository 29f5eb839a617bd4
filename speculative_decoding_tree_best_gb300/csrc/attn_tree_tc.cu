// attn_tree_tc.cu -- tensor-core (tcgen05) split-KV partial for tree attention,
// bf16 I/O, head dim 128.
//
// Digest "SpecPilot ...": prerequisites / draft-tree verification (one target
// pass verifies the tree; every node sees only its ancestors).
//
// A work unit = one (request, kv-head, 128-row query tile, key chunk) that
// holds keys.  The launch is persistent: one CTA per SM (at most), each running
// every grid-th unit, with its pipelines running from one unit into the next.
// The query tile holds the G = Hq/Hkv q-heads of the group for 128/G
// consecutive tree rows (row r = node * G + head_in_group), loaded by TMA once
// the previous unit's S products are done.  The keys stream through rings of
// 128-key K blocks (two stages) and V blocks (three stages), TMA with 128-byte
// swizzle, numbered across the CTA's units; a K stage is refilled as soon as
// its S product is done, a V stage once its PV product is done.  Per block j:
//    S_j = Q K_j^T          tcgen05.mma (bf16, exact products), fp32 in tensor
//                           memory, two S buffers so S_{j+1} is ready while
//                           the softmax works on S_j
//    P_j = exp2(S_j c - m)  one thread per (row, 32 keys), written as fp16
//                           (11 significant bits; a bf16 P would cost ~1.7e-3
//                           relative error on O) into one of two P buffers in
//                           tensor memory, so P_j is written while PV_{j-1}
//                           still reads P_{j-1}
//    V_j -> fp16            the softmax threads convert V_j in place (the same
//                           swizzled layout), so PV runs as kind::f16 with f16
//                           operands
//    O += P_j V_j           tcgen05.mma with A (P) read from tensor memory, fp32
//                           in tensor memory
// Keeping P out of shared memory leaves room for the third V stage: more
// bytes in flight per SM, which is what bounds the stream rate.
// The MMA order is S_0, S_1, PV_0, S_2, PV_1, ...  The running maximum is only
// raised (and O rescaled in tensor memory, after PV_{j-1} is done) when a
// block's maximum exceeds it by more than 2^8, so P <= 256.  The chunk's output is stored normalised
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
constexpr int NVS = 3;                                          // V ring stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE_BYTES;               // NVS stages
constexpr uint32_t OFF_RED = OFF_V + NVS * TILE_BYTES;           // float [2][NWG][128] row maxima
constexpr uint32_t OFF_REDL = OFF_RED + 2 * NWG * 128 * 4;       // float [NWG][128] row sums
constexpr uint32_t OFF_BAR = OFF_REDL + NWG * 128 * 4;
enum { B_Q = 0, B_QE, B_KF, B_VF = B_KF + 2, B_KE = B_VF + NVS, B_VE = B_KE + 2,
       B_SFULL = B_VE + NVS, B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVD = B_PFULL + 2,
       NBARS = B_PVD + 2 };
// Every barrier that a role may pass twice before another role's wait on it
// sees the first pass is split per buffer (S, P) or per stage (K, V): a
// parity wait must never be two phases behind.  P_{j+1} can be written before
// the MMA thread has seen P_j (two P buffers), hence one PFULL barrier per P
// buffer.
// tensor-memory columns: S buffers 0 and 128, O 256, fp16 P buffers 384 and 448
constexpr uint32_t TM_O = 256, TM_P = 384;
constexpr uint32_t OFF_UNITS = OFF_BAR + NBARS * 8 + 32;         // int [4 B + 1]: the unit map
constexpr uint32_t SMEM_LIMIT = 227 * 1024;

__host__ __device__ constexpr uint32_t smem_bytes(int B) {
    return OFF_UNITS + 4u * (4u * (uint32_t)B + 1u) + 1024;      // + slack for alignment
}

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

// The work units of one launch: the (request, kv-head, query tile, key chunk)
// tiles that hold keys, longest first: the full cache chunks (request by
// request), then the partial last chunks (by length, longest first), then the
// tree chunks (which wait for the tree).  Every role of every CTA decodes the
// same numbering from the per-request counts in shared memory.  Round r of
// the grid takes units [r grid, (r + 1) grid), dealt to the CTAs in
// alternating directions (a snake), which evens out the CTAs' loads; each
// CTA's K/V rings run across its units' boundaries.
struct Units {
    const int* fpre;    // [B + 1]: full chunks of requests < b
    const int* len;     // [B]: kv_len clamped to [0, Lmax]
    const int* pord;    // [requests with a partial chunk]: longest partial first
    int B, hg, n_mt, chunk, T, grid;
    int n_full, n_part, total;   // units per region (x hg), all units

    // the largest b with pre[b] <= q (pre non-decreasing, pre[0] = 0 <= q < pre[B])
    __device__ __forceinline__ static int find(const int* pre, int B, int q) {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= q) lo = mid;
            else hi = mid;
        }
        return lo;
    }
    // the k-th unit of CTA i; the last round runs forwards, so its units go
    // to the lowest CTAs (the highest are placed last: behind, say, the CTA
    // of the launch before)
    __device__ __forceinline__ int unit_of(int i, int k) const {
        const int last = (total - 1) / grid;
        return k * grid + (((last - k) & 1) ? grid - 1 - i : i);
    }
    // how many units CTA i runs
    __device__ __forceinline__ int count(int i) const {
        if (total <= 0) return 0;
        const int last = (total - 1) / grid, rem = total - last * grid;
        return last + (i < rem ? 1 : 0);
    }
};

struct Unit {
    int b, g, mt, ch;    // ch = n_split for the tree chunk
    int k0, k1, nblk;
    bool tree;
};

__device__ __forceinline__ Unit decode(const Units& U, int u, int n_split) {
    Unit r;
    int rem, q;
    if (u < U.n_full) {
        q = u / U.hg;
        rem = u % U.hg;
        r.b = Units::find(U.fpre, U.B, q);
        r.ch = q - U.fpre[r.b];
        r.k0 = r.ch * U.chunk;
        r.k1 = r.k0 + U.chunk;
        r.tree = false;
    } else if (u < U.n_full + U.n_part) {
        q = (u - U.n_full) / U.hg;
        rem = (u - U.n_full) % U.hg;
        r.b = U.pord[q];
        r.ch = U.fpre[r.b + 1] - U.fpre[r.b];
        r.k0 = r.ch * U.chunk;
        r.k1 = U.len[r.b];
        r.tree = false;
    } else {
        const int t = u - U.n_full - U.n_part;
        r.b = t / U.hg;
        rem = t % U.hg;
        r.ch = n_split;
        r.k0 = 0;
        r.k1 = U.T;
        r.tree = true;
    }
    r.g = rem / U.n_mt;
    r.mt = rem % U.n_mt;
    r.nblk = (r.k1 - r.k0 + NB - 1) / NB;
    return r;
}

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
    int* issued_q = reinterpret_cast<int*>(tmem_slot + 4);       // Q tiles the producer issued
    int* n_partial = reinterpret_cast<int*>(tmem_slot + 5);      // requests with a partial chunk
    int* upre = reinterpret_cast<int*>(sm + OFF_UNITS);   // fpre [B+1] | len [B] | pnb [B] | pord [B]

    const spec_cfg& c = prm.c;
    const WsLayout& w = prm.w;
    const int T = c.N + 1, G = c.Hq / c.Hkv, B = c.B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Units U;
    int* pnb = upre + (B + 1) + B;                              // partial chunk's blocks, or 0
    U.fpre = upre;
    U.len = upre + (B + 1);
    U.pord = pnb + B;
    U.B = B;
    U.grid = gridDim.x;
    U.n_mt = w.n_mt;
    U.hg = c.Hkv * w.n_mt;
    U.chunk = w.chunk;
    U.T = T;

    if (threadIdx.x == 0) {
        mbar_init(&bar[B_Q], 1);
        mbar_init(&bar[B_QE], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[B_KF + s], 1);
            mbar_init(&bar[B_KE + s], 1);
            mbar_init(&bar[B_SFULL + s], 1);
            mbar_init(&bar[B_SFREE + s], NSOFT);
            mbar_init(&bar[B_PVD + s], 1);
            mbar_init(&bar[B_PFULL + s], NSOFT);
        }
        for (int s = 0; s < NVS; ++s) {
            mbar_init(&bar[B_VF + s], 1);
            mbar_init(&bar[B_VE + s], 1);
        }
        *abort_flag = 0;
        *issued_k = 0;
        *issued_v = 0;
        *issued_q = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&mq);
            tma_prefetch_desc(&mkc);
            tma_prefetch_desc(&mvc);
            tma_prefetch_desc(&mkt);
            tma_prefetch_desc(&mvt);
        }
    } else if (warp == 2) {
        // per-request full chunks and their prefix sums, 32 requests at a time;
        // the requests with a partial last chunk, longest first (stable)
        int cf = 0;
        uint32_t present = 0;                            // partial lengths in blocks present
        if (lane == 0) upre[0] = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int b = b0 + lane;
            int L = 0;
            if (b < B) {
                L = prm.kv_len[b];
                L = L < 0 ? 0 : (L > c.Lmax ? c.Lmax : L);
            }
            int f = b < B ? L / w.chunk : 0;
            const int pn = (L % w.chunk + NB - 1) / NB;  // 0 .. chunk / NB
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int fo = __shfl_up_sync(0xffffffffu, f, o);
                if (lane >= o) f += fo;
            }
            if (b < B) {
                upre[b + 1] = cf + f;
                upre[B + 1 + b] = L;
                pnb[b] = pn;
                present |= 1u << pn;
            }
            cf += __shfl_sync(0xffffffffu, f, 31);
        }
        present = __reduce_or_sync(0xffffffffu, present) & ~1u;
        __syncwarp();
        int pos = 0;
        while (present) {
            const int v = 31 - __clz(present);
            present &= ~(1u << v);
            for (int b0 = 0; b0 < B; b0 += 32) {
                const int b = b0 + lane;
                const bool hit = b < B && pnb[b] == v;
                const uint32_t m = __ballot_sync(0xffffffffu, hit);
                if (hit) pnb[B + pos + __popc(m & ((1u << lane) - 1u))] = b;
                pos += __popc(m);
            }
        }
        if (lane == 0) *n_partial = pos;
    } else if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + TM_O;                 // S buffers at +0 and +128
    U.n_full = U.fpre[B] * U.hg;
    U.n_part = n_partial[0] * U.hg;
    U.total = U.n_full + U.n_part + B * U.hg;
    const int nu = U.count(blockIdx.x);

    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ Q tiles and the K ring
        if (lane == 0) {
            int J = 0;                                   // global block index of this CTA
            for (int k = 0; k < nu && ok; ++k) {
                const Unit un = decode(U, U.unit_of(blockIdx.x, k), w.n_split);
                const CUtensorMap* mk = un.tree ? &mkt : &mkc;
                for (int j = 0; j < un.nblk; ++j, ++J) {
                    const int s = J & 1;
                    // stage s is free once S_{J-2} is done
                    if (J >= 2 && !mbar_wait(&bar[B_KE + s], ((J >> 1) - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar[B_KF + s], TILE_BYTES);
                    for (int h = 0; h < 2; ++h)
                        tma_load_4d(sm + OFF_K + s * TILE_BYTES + h * HALF_BYTES, mk,
                                    &bar[B_KF + s], h * 64, un.g, un.k0 + j * NB, un.b);
                    *issued_k = J + 1;
                    if (j == 0) {
                        // the Q tile is free once the previous unit's S products are done
                        if (k >= 1 && !mbar_wait(&bar[B_QE], (k - 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&bar[B_Q], TILE_BYTES);
                        const int node0 = un.mt * (BM / G);
                        for (int h = 0; h < 2; ++h)
                            tma_load_3d(sm + OFF_Q + h * HALF_BYTES, &mq, &bar[B_Q], h * 64,
                                        un.g * G, un.b * T + node0);
                        *issued_q = k + 1;
                    }
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ the V ring
        if (lane == 0) {
            int J = 0;
            for (int k = 0; k < nu && ok; ++k) {
                const Unit un = decode(U, U.unit_of(blockIdx.x, k), w.n_split);
                const CUtensorMap* mv = un.tree ? &mvt : &mvc;
                for (int j = 0; j < un.nblk; ++j, ++J) {
                    const int s = J % NVS;
                    // stage s is free once PV_{J-NVS} is done
                    if (J >= NVS && !mbar_wait(&bar[B_VE + s], (J / NVS - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bar[B_VF + s], TILE_BYTES);
                    for (int h = 0; h < 2; ++h)
                        tma_load_4d(sm + OFF_V + s * TILE_BYTES + h * HALF_BYTES, mv,
                                    &bar[B_VF + s], h * 64, un.g, un.k0 + j * NB, un.b);
                    *issued_v = J + 1;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(128, NB, false, false);
            const uint32_t idPV = idesc_f16_f32(128, HD, false, true);
            const uint32_t q_s = smem_u32(sm + OFF_Q);
            int nj = 0;                                  // blocks of all this CTA's units
            for (int k = 0; k < nu; ++k) nj += decode(U, U.unit_of(blockIdx.x, k), w.n_split).nblk;
            // the S cursor: unit ks, block js of it, global block JS
            int ks = 0, js = 0, JS = 0;
            int s_nblk = nu > 0 ? decode(U, U.unit_of(blockIdx.x, 0), w.n_split).nblk : 0;
            // S_JS = Q K_JS^T into S buffer JS & 1, then advance the cursor
            auto issue_s = [&]() -> bool {
                const int s = JS & 1;
                if (js == 0 && !mbar_wait(&bar[B_Q], ks & 1, abort_flag)) return false;
                if (!mbar_wait(&bar[B_KF + s], (JS >> 1) & 1, abort_flag)) return false;
                // the softmax has read S_{JS-2} out of this buffer
                if (JS >= 2 && !mbar_wait(&bar[B_SFREE + s], ((JS >> 1) - 1) & 1, abort_flag))
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
                ++JS;
                if (++js == s_nblk) {                    // the unit's last S: its Q tile is free
                    mma_commit(&bar[B_QE]);
                    js = 0;
                    if (++ks < nu) s_nblk = decode(U, U.unit_of(blockIdx.x, ks), w.n_split).nblk;
                }
                return true;
            };
            // S runs up to two blocks ahead of PV (two S buffers), except that a
            // unit's first S, which waits for that unit's Q tile, is not issued
            // while the PV of the block before it is still pending
            auto catch_up = [&](int jp_done) -> bool {
                while (JS < nj && JS <= jp_done + 2) {
                    if (js == 0 && JS == jp_done + 2) break;
                    if (!issue_s()) return false;
                }
                return true;
            };
            ok = catch_up(-1);
            // the PV cursor: block jp of the current unit, global block J
            int kp = 0, jp = 0;
            int p_nblk = nu > 0 ? decode(U, U.unit_of(blockIdx.x, 0), w.n_split).nblk : 0;
            for (int J = 0; J < nj && ok; ++J) {
                const int s = J % NVS;
                // P_J written (tensor memory) and V_J converted to fp16 by the softmax threads
                if (!mbar_wait(&bar[B_PFULL + (J & 1)], (J >> 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t v_s = smem_u32(sm + OFF_V + s * TILE_BYTES);
                const uint32_t p_t = tmem + TM_P + (J & 1) * (NB / 2);
#pragma unroll
                for (int k = 0; k < NB / 16; ++k)
                    mma_f16_tmem_a(tO, p_t + k * 8, sdesc_sw128(v_s + k * 2048, HALF_BYTES, 1024),
                                   idPV, (jp > 0 || k > 0));
                mma_commit(&bar[B_PVD + (J & 1)]);
                mma_commit(&bar[B_VE + s]);
                ok = catch_up(J);
                if (++jp == p_nblk) {
                    jp = 0;
                    if (++kp < nu) p_nblk = decode(U, U.unit_of(blockIdx.x, kp), w.n_split).nblk;
                }
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
        const uint32_t lane_addr = static_cast<uint32_t>(lg * 32) << 16;
        const int cb0 = wg * CPT;                        // first column of this thread
        const int grp_bar = 1 + lg;
        constexpr int GRP_THREADS = 32 * NWG;
        float* red = reinterpret_cast<float*>(sm + OFF_RED);
        float* redl = reinterpret_cast<float*>(sm + OFF_REDL);
        const float sl2 = 1.4426950408889634f * rsqrtf((float)HD);   // log2(e) / sqrt(D)
        float sv[CPT];
        {
            // chunks past a request's KV length leave an empty partial (max
            // -inf, sum 0), so the merge needs no kv_len: one softmax warp per
            // (request, kv-head, tile, chunk), strided over the grid, while the
            // first loads are in flight
            float2* wML = ws_ptr<float2>(prm.ws, w.attn_ml_off);
            const int n_tiles = B * U.hg * w.n_split;
            for (int t = (int)blockIdx.x * (NSOFT / 32) + (st >> 5); t < n_tiles;
                 t += (int)gridDim.x * (NSOFT / 32)) {
                const int ch = t % w.n_split, bh = t / w.n_split;   // bh = b hg + g n_mt + mt
                if (ch * w.chunk < U.len[bh / U.hg]) continue;
                const size_t tile = (size_t)bh * w.n_chunks + ch;
                const int mt = bh % w.n_mt;
                for (int r = lane; r < BM; r += 32)
                    if (mt * BM + r < G * T) wML[tile * BM + r] = make_float2(-INFINITY, 0.0f);
            }
        }
        int J = 0;                                       // global block index
        for (int k = 0; k < nu && ok; ++k) {
            const Unit un = decode(U, U.unit_of(blockIdx.x, k), w.n_split);
            const int r = un.mt * BM + row;              // query row within (request, kv-head)
            const int x = r / G;
            uint32_t visbits = 0xffffffffu;              // tree chunk: visible keys among my columns
            int tree_rows = NB;                          // tree chunk: its real rows
            if (un.tree) {
                pdl_wait();      // the tree may come from the launch just before
                int nn = prm.tree.n_nodes[un.b];
                nn = nn < 1 ? 1 : (nn > T ? T : nn);
                tree_rows = nn;
                visbits = 0u;
                if (x < nn) {
                    const uint64_t a = prm.tree.node_anc[2 * ((size_t)un.b * T + x) + (cb0 >> 6)];
                    visbits = static_cast<uint32_t>(a >> (cb0 & 63));
                    if (cb0 + CPT > nn)
                        visbits &= (nn - cb0 <= 0) ? 0u : (0xffffffffu >> (32 - (nn - cb0)));
                }
            }
            float m_ref = -INFINITY, l = 0.0f;           // m_ref in raw score units
            for (int j = 0; j < un.nblk; ++j, ++J) {
                const int s = J & 1;
                bool w_ok = __all_sync(0xffffffffu,
                                       mbar_wait(&bar[B_SFULL + s], (J >> 1) & 1, abort_flag));
                float pm0 = -INFINITY, pm1 = -INFINITY, pm2 = -INFINITY, pm3 = -INFINITY;
                if (w_ok) {
                    tc_fence_after();
                    tmem_ld32(tmem + s * 128 + lane_addr + cb0, sv);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(&bar[B_SFREE + s]);
                    // visibility: all columns of a full cache block are visible
                    uint32_t vis = visbits;
                    if (!un.tree) {
                        const int nvis = un.k1 - (un.k0 + j * NB + cb0);
                        vis = nvis >= CPT ? 0xffffffffu
                                          : (nvis <= 0 ? 0u : (0xffffffffu >> (32 - nvis)));
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
                    red[(s * NWG + wg) * 128 + row] = fmaxf(fmaxf(pm0, pm1), fmaxf(pm2, pm3));
                }
                if (!bar_and(grp_bar, GRP_THREADS, w_ok)) { ok = false; break; }
                float mx = red[(s * NWG) * 128 + row];
#pragma unroll
                for (int q = 1; q < NWG; ++q) mx = fmaxf(mx, red[(s * NWG + q) * 128 + row]);
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
                // V_J to fp16 in place: 16 bytes x 4 per thread.  In a block with
                // fewer keys than rows (a chunk's last block, the tree block) the
                // rows past its keys (cache rows at or beyond kv_len, padding tree
                // rows) become 0: their P is 0, but 0 x inf or 0 x NaN in the
                // product would not be, and the caller's buffer there is
                // arbitrary.  In the 128-byte-swizzled halves a 16-byte chunk's
                // row is its index / 8 (the swizzle permutes chunks within a row).
                const int vst = J % NVS;
                const int vrows = un.tree ? tree_rows : un.k1 - (un.k0 + j * NB);
                w_ok = __all_sync(0xffffffffu,
                                  mbar_wait(&bar[B_VF + vst], (J / NVS) & 1, abort_flag));
                if (w_ok) {
                    uint4* vs = reinterpret_cast<uint4*>(sm + OFF_V + vst * TILE_BYTES);
                    uint4 vv[TILE_BYTES / 16 / NSOFT];
#pragma unroll
                    for (int i = 0; i < TILE_BYTES / 16 / NSOFT; ++i) vv[i] = vs[st + i * NSOFT];
                    if (vrows >= NB) {
#pragma unroll
                        for (int i = 0; i < TILE_BYTES / 16 / NSOFT; ++i)
                            vs[st + i * NSOFT] = bf16x8_to_f16x8(vv[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < TILE_BYTES / 16 / NSOFT; ++i) {
                            const int vr = ((st + i * NSOFT) >> 3) & (NB - 1);
                            vs[st + i * NSOFT] = vr < vrows ? bf16x8_to_f16x8(vv[i])
                                                            : make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                // P_J goes to tensor-memory buffer J & 1 once PV_{J-2}, which read
                // it, is done; O is rescaled only once PV_{J-1} is done too
                const bool any_rescale = __any_sync(0xffffffffu, rescale);
                if (J >= 2 && w_ok)
                    w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_PVD + (J & 1)],
                                                             ((J >> 1) - 1) & 1, abort_flag));
                if (any_rescale && w_ok)
                    w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_PVD + ((J - 1) & 1)],
                                                             ((J - 1) >> 1) & 1, abort_flag));
                if (!bar_and(grp_bar, GRP_THREADS, w_ok)) { ok = false; break; }
                tc_fence_after();
                if (any_rescale) {
                    float ov[32];
#pragma unroll
                    for (int cc = 0; cc < CPT / 32; ++cc) {
                        tmem_ld32(tO + lane_addr + cb0 + cc * 32, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] *= factor;
                        tmem_st32(tO + lane_addr + cb0 + cc * 32, ov);
                    }
                }
                {
                    uint32_t hw[CPT / 2];                  // keys 2i, 2i + 1 as one half2
#pragma unroll
                    for (int i = 0; i < CPT / 2; ++i) {
                        const __half2 h2 = __floats2half2_rn(sv[2 * i], sv[2 * i + 1]);
                        hw[i] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    tmem_st16(tmem + TM_P + (J & 1) * (NB / 2) + lane_addr + cb0 / 2, hw);
                }
                tmem_wait_st();
                fence_async_smem();                        // the converted V, for the MMA
                tc_fence_before();
                mbar_arrive(&bar[B_PFULL + (J & 1)]);
            }
            if (!ok) break;
            // the unit's output once its last PV is done
            {
                const bool w_ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_PVD + ((J - 1) & 1)],
                                                                   ((J - 1) >> 1) & 1, abort_flag));
                if (!bar_and(grp_bar, GRP_THREADS, w_ok)) { ok = false; break; }
            }
            tc_fence_after();
            __half* wO = ws_ptr<__half>(prm.ws, w.attn_o_off);
            float2* wML = ws_ptr<float2>(prm.ws, w.attn_ml_off);
            const size_t tile = (((size_t)un.b * c.Hkv + un.g) * w.n_mt + un.mt) * w.n_chunks + un.ch;
            redl[wg * 128 + row] = l;
            bar_and(grp_bar, GRP_THREADS, true);
            float lt = 0.0f;
#pragma unroll
            for (int q = 0; q < NWG; ++q) lt += redl[q * 128 + row];
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
            // the next unit's first PV overwrites O: every thread's reads of it are done
            tc_fence_before();
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
        // is released: wait (bounded) on the phases of the last issued loads
        int never = 0;
        if (*issued_q > 0) mbar_wait(&bar[B_Q], (*issued_q - 1) & 1, &never);
        for (int j = max(0, *issued_k - 2); j < *issued_k; ++j)
            mbar_wait(&bar[B_KF + (j & 1)], (j >> 1) & 1, &never);
        for (int j = max(0, *issued_v - NVS); j < *issued_v; ++j)
            mbar_wait(&bar[B_VF + j % NVS], (j / NVS) & 1, &never);
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
           c.N + 1 <= NB && smem_bytes(c.B) <= SMEM_LIMIT && encode_fn() != nullptr;
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
    const uint32_t smem = smem_bytes(c.B);
    cudaError_t err = cudaFuncSetAttribute(attn_tc_partial,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    // one CTA per SM at most (the units themselves are counted on the device
    // from kv_len): at most every tile of every chunk
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    const long units = (long)c.B * c.Hkv * w.n_mt * w.n_chunks;
    const int grid = (int)(units < sms ? units : sms);
    return launch_k(pdl, attn_tc_partial, dim3(grid), dim3(NTHREADS), smem, st, mq, mkc, mvc, mkt,
                    mvt, prm);
}

}  // namespace spec
