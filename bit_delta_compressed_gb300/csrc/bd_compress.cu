// bd_compress.cu -- BitDelta compression on the GPU.
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section "The
// mathematical foundation": delta = W_ft - W_base, the per-matrix scale
// alpha = (1/n) * ||delta||_1 = mean|delta|, and one sign bit per entry;
// section "Infrastructure details": bits packed 8 per byte, alpha stored f32.
//
// One HBM pass.  Each thread takes 8 consecutive elements (one 16-byte bf16
// vector, or two f32 vectors, per input) and produces one output byte; a warp
// therefore reads 512 contiguous bytes per input per load and writes 32
// contiguous bytes of bits.  The bit is the exact comparison W_ft >= W_base
// (immune to rounding of the difference; zero and -0 deltas give 1).
//
// |delta| is summed in fp32 over at most 32 terms (four 8-term trees), then
// accumulated in fp64 per thread, reduced in fp64 per block into a partial,
// and the last block to finish (an atomic ticket) adds the partials in a fixed
// order and writes alpha = f32(sum / n).  Grid size depends only on the shape
// and the device, so the result is bit-reproducible on a given device.

#include "bd_internal.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;           // 8-element chunks per thread per iteration
constexpr int kMaxGrid = 4096;

template <bool kF32>
struct ChunkIn {
    uint4 v[kF32 ? 2 : 1];
};

// Bits of 8 elements (bit i <-> element i) and the fp32 sum of their |delta|.
__device__ __forceinline__ uint32_t chunk_bf16(const ChunkIn<false>& f, const ChunkIn<false>& b,
                                               float& abs_sum) {
    const uint32_t fw[4] = {f.v[0].x, f.v[0].y, f.v[0].z, f.v[0].w};
    const uint32_t bw[4] = {b.v[0].x, b.v[0].y, b.v[0].z, b.v[0].w};
    float d[8];
    uint32_t byte = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float f0 = bf16_lo(fw[i]), b0 = bf16_lo(bw[i]);
        const float f1 = bf16_hi(fw[i]), b1 = bf16_hi(bw[i]);
        byte |= static_cast<uint32_t>(f0 >= b0) << (2 * i);
        byte |= static_cast<uint32_t>(f1 >= b1) << (2 * i + 1);
        d[2 * i] = fabsf(f0 - b0);        // exact for bf16 operands of nearby exponents
        d[2 * i + 1] = fabsf(f1 - b1);
    }
    abs_sum = ((d[0] + d[1]) + (d[2] + d[3])) + ((d[4] + d[5]) + (d[6] + d[7]));
    return byte;
}

__device__ __forceinline__ uint32_t chunk_f32(const ChunkIn<true>& f, const ChunkIn<true>& b,
                                              float& abs_sum) {
    const float fv[8] = {__uint_as_float(f.v[0].x), __uint_as_float(f.v[0].y),
                         __uint_as_float(f.v[0].z), __uint_as_float(f.v[0].w),
                         __uint_as_float(f.v[1].x), __uint_as_float(f.v[1].y),
                         __uint_as_float(f.v[1].z), __uint_as_float(f.v[1].w)};
    const float bv[8] = {__uint_as_float(b.v[0].x), __uint_as_float(b.v[0].y),
                         __uint_as_float(b.v[0].z), __uint_as_float(b.v[0].w),
                         __uint_as_float(b.v[1].x), __uint_as_float(b.v[1].y),
                         __uint_as_float(b.v[1].z), __uint_as_float(b.v[1].w)};
    float d[8];
    uint32_t byte = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        byte |= static_cast<uint32_t>(fv[i] >= bv[i]) << i;
        d[i] = fabsf(fv[i] - bv[i]);
    }
    abs_sum = ((d[0] + d[1]) + (d[2] + d[3])) + ((d[4] + d[5]) + (d[6] + d[7]));
    return byte;
}

template <bool kF32>
__device__ __forceinline__ uint32_t chunk(const ChunkIn<kF32>& f, const ChunkIn<kF32>& b, float& s) {
    if constexpr (kF32) return chunk_f32(f, b, s);
    else return chunk_bf16(f, b, s);
}

template <bool kF32>
__device__ __forceinline__ ChunkIn<kF32> load_chunk(const uint4* p, int64_t c) {
    ChunkIn<kF32> r;
    constexpr int kV = kF32 ? 2 : 1;
#pragma unroll
    for (int v = 0; v < kV; ++v) r.v[v] = ld_stream(p + c * kV + v);
    return r;
}

// Deterministic fp64 block sum (fixed shuffle tree, fixed warp order).
__device__ __forceinline__ double block_sum(double v, double* smem) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    double r = 0.0;
    if (warp == 0) {
        r = (lane < (int)(blockDim.x >> 5)) ? smem[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_down_sync(0xffffffffu, r, o);
    }
    __syncthreads();
    return r;   // valid in thread 0
}

struct CompressArgs {
    const uint4* ft;
    const uint4* base;
    uint8_t* bits;         // one byte per 8-element chunk
    int64_t n_chunks;
    double* partials;      // [gridDim.x]
    unsigned* ticket;
    float* alpha_out;
    double n_elems;
};

template <bool kF32>
__global__ void __launch_bounds__(kThreads) compress_kernel(CompressArgs a) {
    __shared__ double red[kThreads / 32];
    __shared__ bool last_block;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    double acc = 0.0;
    for (; c + (kUnroll - 1) * stride < a.n_chunks; c += kUnroll * stride) {
        ChunkIn<kF32> f[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            f[u] = load_chunk<kF32>(a.ft, c + u * stride);
            b[u] = load_chunk<kF32>(a.base, c + u * stride);
        }
        float part = 0.f;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float s;
            a.bits[c + u * stride] = static_cast<uint8_t>(chunk<kF32>(f[u], b[u], s));
            part += s;
        }
        acc += static_cast<double>(part);
    }
    for (; c < a.n_chunks; c += stride) {
        float s;
        ChunkIn<kF32> f = load_chunk<kF32>(a.ft, c), b = load_chunk<kF32>(a.base, c);
        a.bits[c] = static_cast<uint8_t>(chunk<kF32>(f, b, s));
        acc += static_cast<double>(s);
    }
    const double blk = block_sum(acc, red);
    if (threadIdx.x == 0) {
        a.partials[blockIdx.x] = blk;
        __threadfence();
        const unsigned t = atomicAdd(a.ticket, 1u);
        last_block = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!last_block) return;
    __threadfence();
    double s = 0.0;
    for (int j = threadIdx.x; j < (int)gridDim.x; j += blockDim.x) s += __ldcg(a.partials + j);
    const double total = block_sum(s, red);
    if (threadIdx.x == 0) {
        *a.alpha_out = static_cast<float>(total / a.n_elems);
        *a.ticket = 0u;
    }
}

// Per-output-row scale: one block per row.
template <bool kF32>
__global__ void __launch_bounds__(kThreads) compress_rows_kernel(const uint4* ft, const uint4* base,
                                                                 uint8_t* bits, int64_t K,
                                                                 float* alpha_out) {
    __shared__ double red[kThreads / 32];
    const int64_t chunks_per_row = K / 8;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * chunks_per_row;
    float acc = 0.f;
    double acc64 = 0.0;
    int n = 0;
    for (int64_t c = threadIdx.x; c < chunks_per_row; c += blockDim.x) {
        float s;
        ChunkIn<kF32> f = load_chunk<kF32>(ft, row0 + c), b = load_chunk<kF32>(base, row0 + c);
        bits[row0 + c] = static_cast<uint8_t>(chunk<kF32>(f, b, s));
        acc += s;
        if (++n == kUnroll) { acc64 += acc; acc = 0.f; n = 0; }
    }
    acc64 += acc;
    const double total = block_sum(acc64, red);
    if (threadIdx.x == 0) alpha_out[blockIdx.x] = static_cast<float>(total / static_cast<double>(K));
}

int compress_grid(int64_t n_chunks, bool f32) {
    int occ = 0;
    if (f32) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_kernel<true>, kThreads, 0);
    else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, compress_kernel<false>, kThreads, 0);
    if (occ < 1) occ = 1;
    int64_t cap = static_cast<int64_t>(sm_count()) * occ;
    if (cap > kMaxGrid) cap = kMaxGrid;
    int64_t want = (n_chunks + static_cast<int64_t>(kThreads) * kUnroll - 1) /
                   (static_cast<int64_t>(kThreads) * kUnroll);
    if (want < 1) want = 1;
    return static_cast<int>(want < cap ? want : cap);
}

bd_status check_compress_args(const void* w_ft, const void* w_base, bd_dtype dt, int64_t N,
                              int64_t K, const float* alpha_out, const uint32_t* bits_out) {
    if (!w_ft || !w_base || !alpha_out || !bits_out) return BD_ERR_NULL;
    if (dt != BD_F32 && dt != BD_BF16) return BD_ERR_DTYPE;
    if (N < 1 || K < 32 || K % 32 != 0) return BD_ERR_SHAPE;
    if (N > (int64_t(1) << 40) / K) return BD_ERR_SHAPE;
    if (!aligned(w_ft, 16) || !aligned(w_base, 16) || !aligned(bits_out, 16) ||
        !aligned(alpha_out, 4))
        return BD_ERR_ALIGN;
    return BD_OK;
}

}  // namespace

}  // namespace bd

using namespace bd;

extern "C" size_t bitdelta_compress_workspace(int64_t N, int64_t K) {
    if (N < 1 || K < 32 || K % 32 != 0) return 0;
    return kHeaderBytes + round_up(sizeof(double) * kMaxGrid, kAlign);
}

extern "C" bd_status bitdelta_compress(const void* w_ft, const void* w_base, bd_dtype in_dtype,
                                       int64_t N, int64_t K, float* alpha_out, uint32_t* bits_out,
                                       void* workspace, size_t ws_bytes, void* stream) {
    bd_status st = check_compress_args(w_ft, w_base, in_dtype, N, K, alpha_out, bits_out);
    if (st != BD_OK) return st;
    if (!workspace) return BD_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return BD_ERR_ALIGN;
    if (ws_bytes < bitdelta_compress_workspace(N, K)) return BD_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* hdr = static_cast<unsigned*>(workspace);
    if (cudaMemsetAsync(hdr + 1, 0, sizeof(unsigned), s) != cudaSuccess) return BD_ERR_CUDA;
    const bool f32 = (in_dtype == BD_F32);
    CompressArgs a;
    a.ft = static_cast<const uint4*>(w_ft);
    a.base = static_cast<const uint4*>(w_base);
    a.bits = reinterpret_cast<uint8_t*>(bits_out);
    a.n_chunks = N * K / 8;
    a.partials = reinterpret_cast<double*>(static_cast<char*>(workspace) + kHeaderBytes);
    a.ticket = hdr + 1;
    a.alpha_out = alpha_out;
    a.n_elems = static_cast<double>(N) * static_cast<double>(K);
    const int grid = compress_grid(a.n_chunks, f32);
    if (f32) compress_kernel<true><<<grid, kThreads, 0, s>>>(a);
    else compress_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

extern "C" bd_status bitdelta_compress_rows(const void* w_ft, const void* w_base,
                                            bd_dtype in_dtype, int64_t N, int64_t K,
                                            float* alpha_out, uint32_t* bits_out, void* stream) {
    bd_status st = check_compress_args(w_ft, w_base, in_dtype, N, K, alpha_out, bits_out);
    if (st != BD_OK) return st;
    if (N > 0x7fffffff) return BD_ERR_SHAPE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint4* ft = static_cast<const uint4*>(w_ft);
    const uint4* bs = static_cast<const uint4*>(w_base);
    uint8_t* bits = reinterpret_cast<uint8_t*>(bits_out);
    if (in_dtype == BD_F32)
        compress_rows_kernel<true><<<static_cast<unsigned>(N), kThreads, 0, s>>>(ft, bs, bits, K, alpha_out);
    else
        compress_rows_kernel<false><<<static_cast<unsigned>(N), kThreads, 0, s>>>(ft, bs, bits, K, alpha_out);
    return launch_status();
}

// ---------------------------------------------------------------------------
// bitdelta_compress_noalloc: the same compression kernel, for callers that
// cannot allocate device memory.  Some hosts of this library run where
// cudaMalloc is off limits: inside an inference engine whose memory pool owns
// every byte of the device, in a plugin that must not grow the process's
// footprint, or in code on a path where an allocation would synchronise the
// device.  They still pass inputs and outputs; the kernel's only scratch (one
// fp64 partial per block plus the finishing ticket) lives in the static
// device array below instead of a caller workspace.
//
// The array is shared by every call on a device and keeps the previous call's
// contents; the ticket is cleared before each launch.  Two calls that overlap
// on the GPU (different streams, no ordering between them) race on it and
// give wrong results.  Every GPU that loads the library holds the array until
// the process exits.
// ---------------------------------------------------------------------------
namespace bd {
namespace {

constexpr int kNoAllocMaxBlocks = 2048;
constexpr size_t kNoAllocScratchBytes = kHeaderBytes + sizeof(double) * kNoAllocMaxBlocks;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the static scratch on the current device.  In host code
// the array's name stands for a host-side shadow, not device memory, so the
// address is looked up with the device current.  The lookup is repeated on
// every call (it allocates nothing and costs a table lookup once the module
// is loaded): a cached address would go stale if the primary context were
// reset and the module reloaded elsewhere.
bd_status noalloc_scratch(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return BD_ERR_CUDA;
    *out = p;
    return BD_OK;
}

}  // namespace
}  // namespace bd

extern "C" bd_status bitdelta_compress_noalloc(const void* w_ft, const void* w_base,
                                               bd_dtype in_dtype, int64_t N, int64_t K,
                                               float* alpha_out, uint32_t* bits_out,
                                               void* stream) {
    bd_status st = check_compress_args(w_ft, w_base, in_dtype, N, K, alpha_out, bits_out);
    if (st != BD_OK) return st;
    const bool f32 = (in_dtype == BD_F32);
    const int64_t n_chunks = N * K / 8;
    // at most one fp64 partial per block fits the array; the kernel's
    // grid-stride loop covers any matrix with fewer blocks
    int grid = compress_grid(n_chunks, f32);
    if (grid > kNoAllocMaxBlocks) grid = kNoAllocMaxBlocks;
    void* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != BD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* hdr = static_cast<unsigned*>(scratch);
    if (cudaMemsetAsync(hdr + 1, 0, sizeof(unsigned), s) != cudaSuccess) return BD_ERR_CUDA;
    CompressArgs a;
    a.ft = static_cast<const uint4*>(w_ft);
    a.base = static_cast<const uint4*>(w_base);
    a.bits = reinterpret_cast<uint8_t*>(bits_out);
    a.n_chunks = n_chunks;
    a.partials = reinterpret_cast<double*>(static_cast<char*>(scratch) + kHeaderBytes);
    a.ticket = hdr + 1;
    a.alpha_out = alpha_out;
    a.n_elems = static_cast<double>(N) * static_cast<double>(K);
    if (f32) compress_kernel<true><<<grid, kThreads, 0, s>>>(a);
    else compress_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}
