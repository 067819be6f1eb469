// bd_api.cu -- status handling and small shared host helpers of the C ABI.
#include <atomic>

#include "bd_internal.cuh"

namespace bd {

namespace {
std::atomic<unsigned long long> g_launches{0};
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n < 1) n = 1;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

}  // namespace bd

extern "C" bd_status bitdelta_device_status(void* workspace, void* stream) {
    if (!workspace) return BD_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return BD_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return BD_ERR_CUDA;
    if (word != 0 && cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return BD_ERR_CUDA;
    for (unsigned c = 1; c < 32; ++c)
        if (word & (1u << c)) return static_cast<bd_status>(c);
    return BD_OK;
}

extern "C" const char* bitdelta_status_string(bd_status s) {
    switch (s) {
        case BD_OK: return "ok";
        case BD_ERR_NULL: return "a required pointer is NULL";
        case BD_ERR_ALIGN: return "a pointer is not suitably aligned";
        case BD_ERR_SHAPE: return "invalid shape";
        case BD_ERR_DTYPE: return "unsupported dtype";
        case BD_ERR_VARIANT: return "variant id outside [-1, V)";
        case BD_ERR_WORKSPACE: return "workspace missing or too small";
        case BD_ERR_CUDA: return "CUDA runtime error";
        case BD_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case BD_ERR_UNSUPPORTED: return "kernel path does not support this shape";
    }
    return "unknown status";
}

extern "C" int bitdelta_abi_version(void) { return BITDELTA_ABI_VERSION; }

extern "C" uint64_t bitdelta_launch_count(void) {
    return bd::g_launches.load(std::memory_order_relaxed);
}

// ---------------------------------------------------------------------------
// Health check of the bounded waits the tensor-core kernels use: one thread
// waits on an mbarrier for `poll_limit` polls.  With arrive != 0 the barrier
// is completed first and the wait succeeds; otherwise nothing ever arrives,
// the wait gives up, and BD_ERR_TIMEOUT is OR-ed into the workspace status
// word (with where-code 99 in the diagnostic word) -- the device stays usable.
// ---------------------------------------------------------------------------
#include "bd_sm100.cuh"

namespace bd {
namespace {
__global__ void bounded_wait_kernel(unsigned* status, uint32_t poll_limit, int arrive) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    sm100::mbar_init(&bar, 1);
    sm100::fence_mbar_init();
    if (arrive) sm100::mbar_arrive(&bar);
    sm100::mbar_wait(&bar, 0, poll_limit, status, 99, status + 2);
}
}  // namespace
}  // namespace bd

extern "C" bd_status bitdelta_check_bounded_wait(void* workspace, uint32_t poll_limit, int arrive,
                                                 void* stream) {
    if (!workspace) return BD_ERR_NULL;
    if (!bd::aligned(workspace, 16)) return BD_ERR_ALIGN;
    if (poll_limit < 1 || poll_limit > (1u << 24)) return BD_ERR_SHAPE;
    bd::bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned*>(workspace), poll_limit, arrive);
    return bd::launch_status();
}
