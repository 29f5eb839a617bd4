// diag.cu -- spec_wait_probe: one bounded device wait, to show on a real GPU
// that a wait which runs out ends with SPEC_DEV_TIMEOUT in the status word and
// a usable context (no trap, no fault, no hang).  It uses the same bounded
// mbarrier wait as the tensor-core kernels.
#include "common.cuh"
#include "tc_util.cuh"

namespace {

using namespace spec::tc;

constexpr uint32_t kMaxProbeUs = 1000000;   // one second
constexpr long long kCyclesPerUs = 2070;    // GB300 maximum SM clock, MHz

__global__ void wait_probe_kernel(void* ws, long long limit, int satisfy) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (satisfy) mbar_arrive(&bar);            // completes phase 0
        // without `satisfy` nothing ever arrives: the wait must run out
        if (!mbar_wait(&bar, 0, &abort_flag, limit)) spec::raise_status(ws, SPEC_DEV_TIMEOUT);
    }
}

}  // namespace

extern "C" int spec_wait_probe(uint32_t limit_us, int satisfy, void* ws, void* stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return ST_EINVAL;
    if (limit_us == 0 || limit_us > kMaxProbeUs) return ST_EINVAL;
    wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        ws, (long long)limit_us * kCyclesPerUs, satisfy);
    return cudaGetLastError() == cudaSuccess ? ST_OK : ST_ECUDA;
}
