// common.cuh -- shared device helpers and the workspace layout of libspectree.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "spec_tree.h"

namespace spec {

constexpr int kWarp = 32;

// ---- element I/O ------------------------------------------------------------
// IO = SPEC_IO_F32 or SPEC_IO_BF16; all arithmetic is fp32.
template <int IO> struct io_t;
template <> struct io_t<SPEC_IO_F32> {
    using T = float;
    using PT = float;    // attention split-KV partial element
    static __device__ __forceinline__ float ld(const T* p, size_t i) { return p[i]; }
    static __device__ __forceinline__ void st(T* p, size_t i, float x) { p[i] = x; }
};
template <> struct io_t<SPEC_IO_BF16> {
    using T = __nv_bfloat16;
    using PT = __half;   // attention split-KV partial element
    static __device__ __forceinline__ float ld(const T* p, size_t i) { return __bfloat162float(p[i]); }
    static __device__ __forceinline__ void st(T* p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---- programmatic dependent launch ------------------------------------------
// spec_verify_step launches every kernel of a step with programmatic stream
// serialization, in a fixed order.  Each kernel follows one rule: code before
// pdl_wait() reads only data that kernels two or more launches earlier in
// that order wrote (or inputs no kernel of the step writes), and
// pdl_trigger() comes after pdl_wait().  So when kernel N+1 starts, kernels
// up to N-1 have completed and kernel N+1 stages its inputs while kernel N
// finishes.  The four single-operation entry points launch conventionally
// (pdl = false), where pdl_wait() returns at once: they are safe in any order.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                   size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void raise_status(void* ws, uint32_t bits) {
    atomicOr(reinterpret_cast<unsigned int*>(ws), bits);
}

// ---- workspace layout ---------------------------------------------------------
// byte 0: device status word; then argmax partials, attention split-KV
// partials, the per-request commit plan written by the acceptance kernel, and
// the tickets and queues of the kernels that hand work between CTAs.
constexpr int kArgmaxSplit = 16;         // CTAs per logits row (upper bound)

struct WsLayout {
    size_t argmax_off;     // float2 [B][T][kArgmaxSplit]: (value, index bits)
    size_t attn_o_off;     // PT     [B][Hkv][n_mt][n_chunks][128][D]: O / l of the chunk,
                           // PT = fp16 for bf16 I/O, fp32 for fp32 I/O
    size_t attn_ml_off;    // float2 [B][Hkv][n_mt][n_chunks][128]: (max, sum)
    size_t attn_o_off1, attn_ml_off1;  // a second partial buffer: attention layer l uses l % 2
    size_t plan_off;       // int32  [B][4]: committed tau (0 = skip), old kv_len
    size_t acc_ticket_off; // uint32 [B]: argmax CTAs (or sampled rows) finished per request
    size_t samp_off;       // float2 [B][T][n_vchunks]: (max, sum of exp) per vocabulary chunk
    size_t samp_tok_off;   // int32  [B][T]: the target's draw of each row
    size_t row_ticket_off; // uint32 [B][T]: chunk-scan CTAs finished per row
    size_t fused_off;      // uint32 [2 + 2B]: persistent step's work queue, CTAs out,
                           // acceptance flags [B], GDN items committed [B]
    size_t total;
    int n_split;           // cache chunks per (request, kv-head)
    int chunk;             // cache rows per chunk
    int n_chunks;          // n_split + 1 (the tree chunk)
    int n_mt;              // 128-row query tiles per (request, kv-head)
    int argmax_split;      // CTAs per logits row
    int n_vchunks;         // vocabulary chunks of SPEC_SAMPLE_CHUNK tokens
};

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// SMs of the current device (0 when there is none or the query fails).  The
// workspace layout (chunking of the attention's keys, split of the logits
// scan) follows the device the calls run on.
static inline int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms > 0 ? sms : 0;
}

// Cache rows per chunk: about one CTA per SM over B x Hkv x tiles x chunks
// for small problems, chunks of 256 to 2048 rows (multiples of 128).  Larger
// chunks amortise each CTA's prologue (Q and the first K/V blocks in flight,
// the first softmax) over more blocks and leave the merge fewer partials; past
// 2048 the load imbalance between long and short requests costs more (batched
// and long-tree steps measured fastest at 2048 of 1024, 1536, 2048, 3072, 4096).
static inline WsLayout ws_layout(const spec_cfg& c, int num_sms) {
    WsLayout w{};
    if (num_sms < 1) num_sms = 1;
    const int T = c.N + 1;
    const int G = c.Hq / c.Hkv;
    w.n_mt = (G * T + 127) / 128;
    const long units = (long)c.B * c.Hkv * w.n_mt;
    long want = (num_sms + units - 1) / units;
    if (want < 1) want = 1;
    long chunk = (c.Lmax + want - 1) / want;
    chunk = (chunk + 127) / 128 * 128;
    if (chunk < 256) chunk = 256;
    if (chunk > 2048) chunk = 2048;
    w.chunk = (int)chunk;
    w.n_split = (int)((c.Lmax + chunk - 1) / chunk);
    if (w.n_split < 1) w.n_split = 1;
    w.n_chunks = w.n_split + 1;
    const long rows = (long)c.B * T;
    // logits-scan CTAs: about three per SM, two for small steps (at most 64
    // rows), which leaves room beside the scan for the launches that overlap
    // it (single step 37.5 -> 36.5 us, Markov 43.7 -> 42.3 us)
    int split = (int)(((rows <= 64 ? 2L : 3L) * num_sms + rows - 1) / rows);
    if (split > kArgmaxSplit) split = kArgmaxSplit;
    if (split < 1) split = 1;
    w.argmax_split = split;

    size_t off = 256;                                   // status word + reserve
    w.argmax_off = off;
    off = align_up(off + sizeof(float) * 2 * (size_t)c.B * T * kArgmaxSplit, 256);
    const size_t tiles = (size_t)c.B * c.Hkv * w.n_mt * w.n_chunks;
    w.attn_o_off = off;
    off = align_up(off + (c.io_dtype == SPEC_IO_BF16 ? 2 : 4) * tiles * 128 * (size_t)c.D, 256);
    w.attn_ml_off = off;
    off = align_up(off + sizeof(float) * 2 * tiles * 128, 256);
    if (c.n_attn_layers > 1) {
        w.attn_o_off1 = off;
        off = align_up(off + (w.attn_ml_off - w.attn_o_off), 256);
        w.attn_ml_off1 = off;
        off = align_up(off + sizeof(float) * 2 * tiles * 128, 256);
    } else {
        w.attn_o_off1 = w.attn_o_off;
        w.attn_ml_off1 = w.attn_ml_off;
    }
    w.plan_off = off;
    off = align_up(off + sizeof(int32_t) * 4 * (size_t)c.B, 256);
    w.acc_ticket_off = off;
    off = align_up(off + sizeof(uint32_t) * (size_t)c.B, 256);
    w.n_vchunks = (int)(((long)c.V + SPEC_SAMPLE_CHUNK - 1) / SPEC_SAMPLE_CHUNK);
    w.samp_off = off;
    off = align_up(off + sizeof(float) * 2 * (size_t)rows * w.n_vchunks, 256);
    w.samp_tok_off = off;
    off = align_up(off + sizeof(int32_t) * (size_t)rows, 256);
    w.row_ticket_off = off;
    off = align_up(off + sizeof(uint32_t) * (size_t)rows, 256);
    w.fused_off = off;
    off = align_up(off + sizeof(uint32_t) * (2 + 2 * (size_t)c.B), 256);
    w.total = off;
    return w;
}

// The layout with attention partial buffer `buf` (0 or 1) selected.
static inline WsLayout with_attn_buf(WsLayout w, int buf) {
    if (buf & 1) {
        w.attn_o_off = w.attn_o_off1;
        w.attn_ml_off = w.attn_ml_off1;
    }
    return w;
}

template <typename T> __host__ __device__ __forceinline__ T* ws_ptr(void* ws, size_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

}  // namespace spec
