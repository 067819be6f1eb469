// bd_paths.cuh -- arguments shared by the linear's kernel paths.
#pragma once

#include "bd_internal.cuh"

namespace bd {

// Device pointers of every variant's packed sign bits, passed by value as a
// kernel parameter (no device-side pointer table to upload).
struct BitsTable {
    const uint8_t* p[BITDELTA_MAX_VARIANTS];
};

struct LinearArgs {
    const void* x;                   // bf16 [M, K]
    const int32_t* ids;              // [M]
    int64_t M, N, K;
    const void* w_base;              // bf16 [N, K]
    const float* alphas;             // [V], or [V, N] when alpha_rows
    int32_t alpha_rows;              // 1: one scale per (variant, output row)
    int32_t V;
    BitsTable bits;
    const uint32_t* const* bits_host;
    void* y;                         // [M, N]
    bd_dtype y_dtype;
};

// Scratch the tensor-core paths need inside the linear workspace.
size_t tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V);

bd_path choose_path(const LinearArgs& a);
bool decode_tc_supported(const LinearArgs& a);
bool prefill_tc_supported(const LinearArgs& a);
bool decode_fold_supported(const LinearArgs& a);
bool decode_weff_supported(const LinearArgs& a);
bd_status launch_decode_weff(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s);
size_t decode_fold_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V);
bd_status launch_decode_fold(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s);
bd_status launch_decode_tc(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s);
bd_status launch_prefill_tc(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s);
// W_eff of every variant present in the grouped batch, slot d of the plan at
// weff + d * N * K (bf16, nearest to the exact sum).
bd_status launch_reconstruct_plan(const LinearArgs& a, const SegPlan* plan, void* weff, cudaStream_t s);

}  // namespace bd
