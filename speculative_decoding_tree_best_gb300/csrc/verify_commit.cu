// verify_commit.cu -- the fused, persistent verify + commit: one cooperative
// launch that runs the vocabulary argmax and acceptance of every request and
// the tensor-core GDN verify of every (layer, request, v-head), and commits
// each GDN state from shared memory once its request is accepted: the state
// is read from HBM once and written once.
//
// Digest "SpecPilot ...": prerequisites / speculative decoding (greedy
// acceptance, tau in [1, m+1]), prerequisites / draft-tree verification
// (longest matching root path), prerequisites / hybrid recurrent target (the
// gated delta rule) and technical novelty (states recomputed along the root
// path, no per-node snapshots).  The committed state of a request is the state
// after its accepted path p_0 (the root) .. p_{tau-1}:
//     h = A h0 + sum_s dec(p_s -> p_{tau-1}) k_{p_s} c_{p_s}^T,
// A the product of alpha over the path, dec(a -> x) the product of alpha over
// the path nodes after a, c the write vectors of the verify.
//
// Work items, taken in order from a device-wide queue by a grid of CTAs that
// all fit on the GPU at once (cooperative launch, one CTA per SM):
//  * argmax items (row, segment): the (max, first index) of a logits segment;
//    the request's last item (atomic ticket) runs the greedy walk, advances
//    kv_len / root_tok, raises the request's acceptance flag, then appends
//    the accepted tree K/V rows to every attention layer's cache;
//  * GDN items (layer, request, v-head): the item of gdn_tc_body.cuh keeping
//    the fp32 state in shared memory; after its outputs it waits for the
//    flag (bounded: SPEC_DEV_TIMEOUT and no commit when it gives up) and
//    writes the committed state over h0.  The request's last GDN item clears
//    the flag.
// Every argmax item precedes every GDN item in the queue and never waits, so
// all flags a GDN item can wait for are raised by CTAs that are running.
#include "accept_util.cuh"
#include "common.cuh"
#include "gdn_tc_body.cuh"
#include "kernels.h"

namespace spec {

namespace {

using namespace gdn_tc;

struct FusedArgs {
    spec_cfg c;
    spec_tree tree;
    spec_commit_io io;
    spec_accept acc;
    const __nv_bfloat16* logits;   // [B][T][V]
    __nv_bfloat16* gdn_o;          // [n_gdn][B][T][Hv][128]
    float* gdn_c;                  // NULL or as gdn_o, float
    void* ws;
    WsLayout w;                    // argmax_split = the segments per row here
    int n_arg;                     // argmax items (B T split)
    int n_items;                   // + GDN items (n_gdn B Hv)
    bool tree_wait;                // the tree is the previous launch
};

__device__ __forceinline__ void named_sync_128() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---- argmax item ----------------------------------------------------------------------
__device__ void argmax_item(const FusedArgs& a, int itm, uint32_t* flags) {
    using E = __nv_bfloat16;
    constexpr int VEC = 8;
    const spec_cfg& c = a.c;
    const WsLayout& w = a.w;
    const int split = w.argmax_split, T = c.N + 1, tid = threadIdx.x;
    const int row = itm / split, sp = itm % split, b = row / T, t = row % T;
    if (t < a.tree.n_nodes[b]) {                                 // CTA-uniform
        int seg = (c.V + split - 1) / split;
        seg = (seg + VEC - 1) / VEC * VEC;
        const int lo = sp * seg, hi = min(c.V, lo + seg);
        float bv;
        int bi;
        // a whole segment of the single-request split (~76 KB) in flight at once
        acc::scan_segment<SPEC_IO_BF16, 24>(a.logits + (size_t)row * c.V, c.V, lo, hi, bv, bi);
        if (tid == 0)
            ws_ptr<float2>(a.ws, w.argmax_off)[(size_t)row * kArgmaxSplit + sp] =
                make_float2(bv, __int_as_float(bi));
    }
    __shared__ bool last;
    if (tid == 0) {
        __threadfence();
        unsigned int* tk = ws_ptr<unsigned int>(a.ws, w.acc_ticket_off) + b;
        const unsigned int done = atomicAdd(tk, 1u);
        last = done == (unsigned int)(T * split) - 1u;
        if (last) *tk = 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (tid < 32) acc::accept_request(c, a.tree, a.io, a.acc, a.ws, w, b);
    __threadfence();
    __syncthreads();
    // the GDN commits need the plan only: raise the flag before the KV append
    if (tid == 0 && c.n_gdn_layers > 0) atomicExch(flags + b, 1u);     // after the fence: a release
    // the accepted tree K/V rows of every attention layer go to the cache
    const int32_t* plan = ws_ptr<const int32_t>(a.ws, w.plan_off) + 4 * b;
    const int tau = plan[0], L = plan[1];
    if (tau > 0 && c.n_attn_layers > 0) {
        const int m = c.m;
        const size_t rowb = (size_t)c.Hkv * c.D * sizeof(E);     // bytes, multiple of 16
        const size_t per = rowb / 16;
        const size_t total = (size_t)c.n_attn_layers * tau * per;
        const char* kt = static_cast<const char*>(a.io.k_tree);
        const char* vt = static_cast<const char*>(a.io.v_tree);
        char* kc = static_cast<char*>(a.io.k_cache);
        char* vc = static_cast<char*>(a.io.v_cache);
        for (size_t i = tid; i < total; i += NT) {
            const size_t q = i % per;
            const int s = (int)((i / per) % tau), layer = (int)(i / (per * tau));
            const int x = a.acc.accept_nodes[(size_t)b * (m + 1) + s];
            const size_t src = (((size_t)layer * c.B + b) * T + x) * rowb + 16 * q;
            const size_t dst = (((size_t)layer * c.B + b) * c.Lmax + L + s) * rowb + 16 * q;
            *reinterpret_cast<uint4*>(kc + dst) = *reinterpret_cast<const uint4*>(kt + src);
            *reinterpret_cast<uint4*>(vc + dst) = *reinterpret_cast<const uint4*>(vt + src);
        }
    }
}

// ---- the commit of one GDN item: threads 0..127, column col ------------------------------
struct Commit {
    const FusedArgs* a;
    unsigned char* sm;
    const Layout* L;
    const uint32_t* flags;
    int layer, b, j;

    __device__ void operator()(int col, int nn) const {
        const spec_cfg& c = a->c;
        const int T = c.N + 1, m = c.m;
        const int ih = j / (c.Hv / c.Hk);
        const float* al = reinterpret_cast<const float*>(sm + L->nodes);   // alpha of the rows
        const float* h32 = reinterpret_cast<const float*>(sm + L->h32);
        const float* C = reinterpret_cast<const float*>(sm + L->p);        // [x][128]: c_x
        float* ks = reinterpret_cast<float*>(sm + L->p) + TPM * DKV;       // [x][128]: k_x
        float* wv = reinterpret_cast<float*>(sm + L->v);   // [s]: dec(p_s -> last); [TPM]: A
        int* px = reinterpret_cast<int*>(wv + TPM + 1);                    // [s]: p_s
        volatile int* s_tau = reinterpret_cast<volatile int*>(sm + L->bar + 24 + 12);
        // the k rows of every tree row, on their way while the acceptance is
        // pending (the column's Q entries of P are consumed)
        const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(a->io.gdn_k) +
                                  ((size_t)layer * c.B + b) * T * c.Hk * DKV;
        {
            __nv_bfloat16 kr[TPM];             // every load in flight before the stores
#pragma unroll
            for (int x = 0; x < TPM; ++x)
                kr[x] = x < nn ? kb[((size_t)x * c.Hk + ih) * DKV + col] : __float2bfloat16_rn(0.0f);
#pragma unroll
            for (int x = 0; x < TPM; ++x)
                if (x < nn) ks[x * DKV + col] = __bfloat162float(kr[x]);
        }
        if (col == 0) {
            // the request's acceptance: a bounded wait on its flag
            const long long t0 = clock64();
            bool ok = true;
            while (ld_acquire(flags + b) == 0u) {
                if (clock64() - t0 > tc::kWaitCycles) {
                    ok = false;
                    break;
                }
                __nanosleep(64);
            }
            int tau = 0;
            if (ok) tau = __ldcg(ws_ptr<const int32_t>(a->ws, a->w.plan_off) + 4 * b);
            else raise_status(a->ws, SPEC_DEV_TIMEOUT);
            *s_tau = tau;
        }
        named_sync_128();
        const int tau = *s_tau;
        if (tau <= 0) return;                       // skipped (no room) or given up
        if (col < tau) px[col] = __ldcg(a->acc.accept_nodes + (size_t)b * (m + 1) + col);
        named_sync_128();
        if (col == 0) {               // decays from the last accepted node up
            float acc = 1.0f;
            for (int s = tau - 1; s >= 0; --s) {
                wv[s] = acc;
                acc *= al[px[s]];
            }
            wv[TPM] = acc;            // A: the product over the whole path
        }
        named_sync_128();
        // h[r][col] = A h0[r][col] + sum_s k_{p_s}[r] dec_s c_{p_s}[col], 32 rows at a time
        const float A = wv[TPM];
        float* dst = a->io.h0 + (size_t)layer * c.B * c.Hv * DKV * DKV +
                     ((size_t)b * c.Hv + j) * DKV * DKV;
        for (int r0 = 0; r0 < DKV; r0 += 32) {
            float h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = A * h32[(r0 + i) * DKV + col];
            for (int s = 0; s < tau; ++s) {
                const int x = px[s];
                const float w = wv[s] * C[x * DKV + col];
                const float4* k4 = reinterpret_cast<const float4*>(ks + x * DKV + r0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 kk = k4[i];
                    h[4 * i] = fmaf(kk.x, w, h[4 * i]);
                    h[4 * i + 1] = fmaf(kk.y, w, h[4 * i + 1]);
                    h[4 * i + 2] = fmaf(kk.z, w, h[4 * i + 2]);
                    h[4 * i + 3] = fmaf(kk.w, w, h[4 * i + 3]);
                }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[(size_t)(r0 + i) * DKV + col] = h[i];
        }
    }
};

__global__ void __launch_bounds__(NT, 1)
verify_commit_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mv, const FusedArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = aligned_base(smem_raw);
    const Layout L = layout(true);
    const spec_cfg& c = a.c;
    const int T = c.N + 1, tid = threadIdx.x;
    uint32_t* ctr = ws_ptr<uint32_t>(a.ws, a.w.fused_off);    // [0] queue, [1] CTAs out
    uint32_t* flags = ctr + 2;                                 // [B]
    uint32_t* gdone = flags + c.B;                             // [B]
    const uint32_t tmem = setup(sm, L);
    if (a.tree_wait) pdl_wait();
    const int per_layer = c.B * c.Hv;
    __shared__ int s_item;
    uint32_t gph = 0;                                          // GDN items run: barrier parity
    for (;;) {
        __syncthreads();
        if (tid == 0) s_item = (int)atomicAdd(ctr, 1u);
        __syncthreads();
        const int itm = s_item;
        if (itm >= a.n_items) break;
        if (itm < a.n_arg) {
            argmax_item(a, itm, flags);
            continue;
        }
        const int g = itm - a.n_arg;
        const int layer = g / per_layer, b = (g % per_layer) / c.Hv, j = g % c.Hv;
        Item it;
        it.j = j;
        it.b = b;
        it.row0 = (layer * c.B + b) * T;
        it.h0 = a.io.h0 + (size_t)layer * c.B * c.Hv * DKV * DKV;
        it.alpha = a.io.alpha + (size_t)layer * c.B * T * c.Hv;
        it.beta = a.io.beta + (size_t)layer * c.B * T * c.Hv;
        it.o = a.gdn_o + (size_t)layer * c.B * T * c.Hv * DKV;
        it.c_out = a.gdn_c ? a.gdn_c + (size_t)layer * c.B * T * c.Hv * DKV : nullptr;
        const Commit commit{&a, sm, &L, flags, layer, b, j};
        item(&mk, &mq, &mv, c, a.tree, it, a.ws, sm, L, tmem, gph & 1u, false, commit);
        ++gph;
        __syncthreads();
        if (tid == 0) {                  // the request's last GDN item clears its flag
            __threadfence();
            const uint32_t done = atomicAdd(gdone + b, 1u);
            if (done == (uint32_t)(c.n_gdn_layers * c.Hv) - 1u) {
                gdone[b] = 0u;
                atomicExch(flags + b, 0u);
            }
        }
    }
    teardown(tmem);
    if (tid == 0) {                      // the last CTA out leaves the queue at zero
        __threadfence();
        if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1u) {
            ctr[0] = 0u;
            ctr[1] = 0u;
        }
    }
}

}  // namespace

bool verify_commit_supported(const spec_cfg& c) {
    return c.io_dtype == SPEC_IO_BF16 && c.n_gdn_layers > 0 && c.dk == DKV && c.dv == DKV &&
           c.N + 1 <= TPM && (c.n_attn_layers == 0 || c.D % 8 == 0) &&
           layout(true).total <= 227u * 1024u;
}

cudaError_t launch_verify_commit(const spec_cfg& c, const spec_tree& t, const spec_step_io& step,
                                 const void* logits, const spec_commit_io& io,
                                 const spec_accept& out, void* ws, cudaStream_t st, bool pdl,
                                 bool tree_wait) {
    if (!verify_commit_supported(c)) return cudaErrorInvalidConfiguration;
    if (encode_fn() == nullptr) return cudaErrorNotSupported;     // no tensor-map encoder
    const int T = c.N + 1;
    const Layout L = layout(true);
    const int rows = c.n_gdn_layers * c.B * T;
    CUtensorMap mk, mq, mv;
    if (!rows_map(&mk, io.gdn_k, c.Hk, rows, TPM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !rows_map(&mq, step.gdn_q, c.Hk, rows, TPM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !rows_map(&mv, io.gdn_v, c.Hv, rows, TPM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(verify_commit_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, occ = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, verify_commit_kernel, NT,
                                                           L.total)) != cudaSuccess)
        return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int cap = sms * occ;
    const int n_gdn = c.n_gdn_layers * c.B * c.Hv;
    // argmax segments per row: fill the CTAs the GDN items leave free
    int split = (cap - n_gdn) / (c.B * T);
    split = split < 1 ? 1 : (split > kArgmaxSplit ? kArgmaxSplit : split);
    FusedArgs a;
    a.c = c;
    a.tree = t;
    a.io = io;
    a.acc = out;
    a.logits = static_cast<const __nv_bfloat16*>(logits);
    a.gdn_o = static_cast<__nv_bfloat16*>(step.gdn_o);
    a.gdn_c = step.gdn_c;
    a.ws = ws;
    a.w = ws_layout(c, device_sm_count());
    a.w.argmax_split = split;
    a.n_arg = c.B * T * split;
    a.n_items = a.n_arg + n_gdn;
    a.tree_wait = tree_wait;
    const int grid = a.n_items < cap ? a.n_items : cap;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, verify_commit_kernel, mk, mq, mv, a);
    if (e != cudaSuccess && pdl) {
        (void)cudaGetLastError();        // cooperative and programmatic together refused: plain order
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, verify_commit_kernel, mk, mq, mv, a);
    }
    return e;
}

}  // namespace spec
