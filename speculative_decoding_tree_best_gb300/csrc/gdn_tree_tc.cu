// gdn_tree_tc.cu -- tree-masked Gated DeltaNet with the h0^T [K; Q] product on
// the tensor cores (tcgen05), bf16 I/O, d_k = d_v = 128, trees of up to 32 rows
// (larger trees use gdn_tree.cu): one CTA per (request, v-head), the item of
// gdn_tc_body.cuh (which states the formulation and the stages).
//
// Digest "SpecPilot ...": prerequisites / hybrid recurrent target (gated delta
// rule) and technical novelty (recompute along the root path, no per-node
// snapshots).
#include "common.cuh"
#include "gdn_tc_body.cuh"
#include "kernels.h"

namespace spec {

namespace {

using namespace gdn_tc;

// One CTA = one (request, v-head) item; 66 KB of shared memory: three CTAs
// share an SM.  early: the tree may come from the launch just before, so the
// programmatic wait precedes the first read of it; otherwise it ends the kernel.
__global__ void __launch_bounds__(NT, 3)
gdn_tc_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mq,
              const __grid_constant__ CUtensorMap mv, spec_cfg c, spec_tree tree,
              const float* __restrict__ h0, const float* __restrict__ alpha,
              const float* __restrict__ beta, __nv_bfloat16* __restrict__ o,
              float* __restrict__ c_out, void* ws, bool early) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = aligned_base(smem_raw);
    const Layout L = layout(false);
    const uint32_t tmem = setup(sm, L);
    Item it;
    it.j = blockIdx.x;
    it.b = blockIdx.y;
    it.row0 = blockIdx.y * (c.N + 1);
    it.h0 = h0;
    it.alpha = alpha;
    it.beta = beta;
    it.o = o;
    it.c_out = c_out;
    const bool ok = item(&mk, &mq, &mv, c, tree, it, ws, sm, L, tmem, 0u, early, NoEpilogue{});
    teardown(tmem);
    if (!ok || !early) {
        pdl_wait();
        pdl_trigger();
    }
}

}  // namespace

bool gdn_tc_supported(const spec_cfg& c) {
    const int T = c.N + 1;
    return c.io_dtype == SPEC_IO_BF16 && c.dk == DKV && c.dv == DKV && T <= TPM &&
           layout(false).total <= 227u * 1024u && encode_fn() != nullptr;
}

cudaError_t launch_gdn_tc(const spec_cfg& c, const spec_tree& t, const float* h0, const void* q,
                          const void* k, const void* v, const float* alpha, const float* beta,
                          void* o, float* c_out, void* ws, cudaStream_t st, bool pdl, bool early) {
    const int T = c.N + 1;
    const Layout L = layout(false);
    CUtensorMap mk, mq, mv;
    if (!rows_map(&mk, k, c.Hk, c.B * T, TPM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !rows_map(&mq, q, c.Hk, c.B * T, TPM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !rows_map(&mv, v, c.Hv, c.B * T, TPM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gdn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L.total);
    if (e != cudaSuccess) return e;
    return launch_k(pdl, gdn_tc_kernel, dim3(c.Hv, c.B), dim3(NT), L.total, st, mk, mq, mv, c, t,
                    h0, alpha, beta, static_cast<__nv_bfloat16*>(o), c_out, ws, early);
}

}  // namespace spec
