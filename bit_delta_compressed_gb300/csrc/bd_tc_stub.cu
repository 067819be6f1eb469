// bd_tc_stub.cu -- tensor-core paths not yet present: every shape goes to the
// CUDA-core kernel, and asking for a tensor-core path explicitly is refused.
#include "bd_paths.cuh"

namespace bd {

size_t tc_scratch_bytes(int64_t, int64_t, int64_t, int32_t) { return 0; }
bd_path choose_path(const LinearArgs&) { return BD_PATH_SIMT; }
bool decode_tc_supported(const LinearArgs&) { return false; }
bool prefill_tc_supported(const LinearArgs&) { return false; }
bd_status launch_decode_tc(const LinearArgs&, const LinearWorkspace&, cudaStream_t) {
    return BD_ERR_UNSUPPORTED;
}
bd_status launch_prefill_tc(const LinearArgs&, const LinearWorkspace&, cudaStream_t) {
    return BD_ERR_UNSUPPORTED;
}

}  // namespace bd
