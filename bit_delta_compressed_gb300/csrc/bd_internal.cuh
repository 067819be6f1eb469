// bd_internal.cuh -- helpers shared by the library's translation units.
//
// Workspace header (the first 256 bytes of every workspace):
//   u32 [0]  status word: device-detected errors, OR-ed as (1 << bd_status)
//   u32 [1]  compress: ticket of the last-block-done reduction
//   u32 [2]  diagnostic: where a bounded wait gave up (0 = never)
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "bitdelta.h"

namespace bd {

constexpr size_t kHeaderBytes = 256;
constexpr size_t kAlign = 256;

__host__ __device__ inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device-side error report into the workspace status word.
__device__ __forceinline__ void report(unsigned* status, bd_status code) {
    atomicOr(status, 1u << static_cast<unsigned>(code));
}

// bf16 bit patterns -> f32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 16-byte streaming load that skips L1 (data read exactly once).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Number of SMs of the current device (cached per device).
int sm_count();

// Kernels this library has enqueued since it was loaded (all devices and
// streams); bitdelta_launch_count() reads it.
void note_launch();

// Launch check, called once right after every kernel launch: counts the
// launch and returns BD_ERR_CUDA if it failed.
inline bd_status launch_status() {
    note_launch();
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

// ---- linear workspace layout (shared by the dispatcher and kernels) ----

// Segment plan of one grouped batch, written by the grouping kernel.
// Grouped positions: [0, n_base) base-model tokens (id -1), then every
// present variant's tokens in variant order, then invalid ids.  For the
// tensor-core decode path each present variant d also gets a zero-padded
// segment of pad16(cnt[d]) rows starting at row seg[d] of the sign operand,
// and the variants are cut into passes (groups) whose padded rows fit
// `group_budget`.
constexpr int kMaxGroups = BITDELTA_MAX_VARIANTS;
struct SegPlan {
    int32_t M;
    int32_t n_base;
    int32_t n_invalid;
    int32_t D;                                    // present variants
    int32_t P;                                    // sum of pad16(cnt)
    int32_t n_groups;
    int32_t var[BITDELTA_MAX_VARIANTS];           // variant id of present index d
    int32_t cnt[BITDELTA_MAX_VARIANTS];           // its token count
    int32_t off[BITDELTA_MAX_VARIANTS];           // grouped position of its first token
    int32_t seg[BITDELTA_MAX_VARIANTS];           // first padded row of its segment
    int32_t group_first[kMaxGroups + 1];          // present-index range of each pass
};

// Issue plan of the folded tensor-core decode kernel, also written by the
// grouping kernel.  The accumulator has one column per grouped position
// (pad16(M) columns, 16-column chunks).  Entry e is present variant e_slot
// (one run of grouped positions): it covers columns [e_col, e_col + e_n)
// with rows [e_row, e_row + e_n) of the sign operand (rows of other
// variants' tokens are zero there) and the +-1 tile of that variant.  Issuer
// group i expands and issues entries iss_e0[i], iss_e0[i] + kFoldIssuers, ...
// (iss_ne[i] of them), and zeroes and writes out the columns [iss_col[i],
// iss_col[i] + iss_n[i]).  The base product (all columns at once) has an
// issuer of its own.
constexpr int kFoldIssuers = 4;
constexpr int kFoldMaxSlots = 16;                       // present variants
constexpr int kFoldMaxEntries = kFoldMaxSlots;          // one entry per present variant
constexpr int kFoldMaxCols = 128;                       // pad16(M)
constexpr int kFoldSepEntries = 16;                     // entries whose +-1 tiles fit (two buffers)
struct FoldPlan {
    int32_t ok;                                   // 1 if the batch fits the folded kernel
    int32_t C;                                    // chunks of 16 columns
    int32_t R;                                    // rows of the sign operand (multiple of 16)
    int32_t n_entries;
    int32_t iss_col[kFoldIssuers], iss_n[kFoldIssuers], iss_e0[kFoldIssuers], iss_ne[kFoldIssuers];
    int32_t e_col[kFoldMaxEntries], e_n[kFoldMaxEntries], e_slot[kFoldMaxEntries], e_row[kFoldMaxEntries];
};

struct GroupView {
    int32_t* counts;     // [V + 2]: bucket 0 = id -1 (base), 1..V = variants, V+1 = invalid
    int32_t* offsets;    // [V + 3]: first grouped position of each bucket; [V + 2] = M
    int32_t* pos2tok;    // [M]: grouped position -> original token
    int32_t* pos_var;    // [M]: grouped position -> variant id (-1 base, -2 invalid)
    SegPlan* plan;
    FoldPlan* fold;
};

__host__ __device__ inline int pad16(int v) { return (v + 15) & ~15; }

struct LinearWorkspace {
    unsigned* status;
    GroupView g;
    size_t group_end;    // bytes up to the end of the grouping area
    void* tc_scratch;    // tensor-core paths: staged activations
    size_t tc_bytes;
    size_t total;
};

LinearWorkspace linear_workspace_layout(void* base, int64_t M, int64_t N, int64_t K, int32_t V);

// Padded sign rows one pass of the tensor-core decode kernel can hold in
// tensor memory next to the base accumulator of pad16(M) columns, and the
// most variants one pass takes (bounded by its shared-memory bits ring).
int decode_group_budget(int64_t M);
constexpr int kMaxPassVariants = 12;

}  // namespace bd
