// bd_prefill_tc.cu -- path selection and the tensor-core prefill path.
#include "bd_tc_common.cuh"

namespace bd {

size_t decode_tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V);

size_t tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V) {
    return decode_tc_scratch_bytes(M, N, K, V);
}

bd_path choose_path(const LinearArgs& a) {
    if (decode_tc_supported(a)) return BD_PATH_DECODE_TC;
    return BD_PATH_SIMT;
}

bool prefill_tc_supported(const LinearArgs&) { return false; }

bd_status launch_prefill_tc(const LinearArgs&, const LinearWorkspace&, cudaStream_t) {
    return BD_ERR_UNSUPPORTED;
}

}  // namespace bd
