// attn_noalloc.cu -- attn_tree_verify_noalloc: tree-masked attention whose
// scratch (the split-KV partials and the device status word) lives in a
// file-scope static device array instead of a caller-supplied workspace.
//
// Who needs it: callers that own no allocator on the path that launches the
// op -- e.g. a custom op inside a host runtime that hands its plug-ins only the
// tensors of the call (the runtime owns every byte of device memory and its
// enqueue hook must not allocate), or a serving loop whose latency budget
// rules out a trip through a caching allocator.  Such a caller can still pass
// its inputs and outputs; the scratch is reserved once, with the library's
// module, at a fixed size.
//
// The attention computed is exactly attn_tree_verify's (same kernels, same
// launch shapes), so results are identical to that call's.
#include <mutex>

#include "checks.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = SPEC_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Zero-initialised when the module loads; setup clears the status word once
// more.  Byte 0 holds the status word (the only part that must start at zero,
// and each call leaves it at zero again); the partials after it are written
// before they are read in every call.
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Address of this device's copy of the scratch array.  The first call on a
// device (with that device current) looks it up and clears the status word
// synchronously; later calls only read the cached pointer (which a device
// reset would leave stale: calls must not span a cudaDeviceReset).
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ST_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return ST_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr)
            return ST_ECUDA;
        if (cudaMemset(p, 0, sizeof(uint32_t)) != cudaSuccess) return ST_ECUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return ST_ECUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return ST_OK;
}

// Moves the status bits of the call from the scratch word to the caller's
// word (if any) and leaves the scratch word at zero.
__global__ void fold_status(unsigned int* scratch_status, unsigned int* dev_status) {
    const unsigned int s = atomicExch(scratch_status, 0u);
    if (dev_status != nullptr && s != 0u) atomicOr(dev_status, s);
}

// Bytes of scratch the attention of `c` touches: status word, argmax reserve
// (unused here) and partial buffer 0 of the workspace layout.
size_t attn_scratch_need(const spec_cfg& c) {
    const spec::WsLayout w = spec::ws_layout(c, spec::device_sm_count());
    const size_t tiles = (size_t)c.B * c.Hkv * w.n_mt * w.n_chunks;
    return w.attn_ml_off + sizeof(float) * 2 * tiles * 128;
}

}  // namespace

extern "C" int attn_tree_verify_noalloc(const spec_cfg* cfg, const spec_tree* tree, const void* q,
                                        const void* k_tree, const void* v_tree,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* kv_len, void* o, uint32_t* dev_status,
                                        void* stream) {
    // shape and pointer checks first (the codes attn_tree_verify returns):
    // nothing touches the device before them
    using spec::al16;
    int rc = spec::check_cfg(cfg);
    if (rc != ST_OK) return rc;
    if ((rc = spec::check_tree(tree)) != ST_OK) return rc;
    if (!al16(q) || !al16(k_tree) || !al16(v_tree) || !al16(k_cache) || !al16(v_cache) ||
        !al16(kv_len) || !al16(o))
        return ST_EINVAL;
    if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return ST_EINVAL;
    if (attn_scratch_need(*cfg) > kScratchBytes) return ST_ESCRATCH;
    void* scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != ST_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the status word starts this call at zero, whatever a failed call before
    // left in it (a memset, not an allocation)
    cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess)
        e = spec::launch_attn_tree(*cfg, *tree, q, k_tree, v_tree, k_cache, v_cache, kv_len, o,
                                   scratch, st);
    if (e == cudaSuccess) {
        fold_status<<<1, 1, 0, st>>>(static_cast<unsigned int*>(scratch),
                                     reinterpret_cast<unsigned int*>(dev_status));
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) return ST_OK;
    return e == cudaErrorInvalidConfiguration ? ST_EUNSUPPORTED : ST_ECUDA;
}
