// bd_reconstruct.cu -- materialised effective weights of one variant.
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture" (the conceptual listing rebuilds
// W_eff = W_base + alpha * sign(delta) in the base dtype and hands it to a
// standard linear) and section "Latency profile" (reconstruction in prefill,
// then the standard matmul path).  The decode kernels never write W_eff.
// This file writes it once per variant: for callers (bitdelta_reconstruct,
// e.g. to run "reconstruct, then a library GEMM" beside the fused path) and
// for the prefill path, which materialises every present variant of a large
// batch and then multiplies without rebuilding W tiles in shared memory.
//
// W_eff[n,k] = bf16_rne(W_base[n,k] + a s[n,k]), a = alpha (one per matrix)
// or alpha[n] (one per output row), s = +1 for a stored 1 bit, -1 for a 0.
// The sum is formed in f32 together with its exact rounding error (Knuth's
// TwoSum), and the error decides the rounding to bf16 whenever the f32 sum
// lands exactly halfway between two bf16 values, so the result is the bf16
// nearest to the exact sum (ties to even) with no double rounding.
//
// HBM-bound: 2 bytes of W_base and 1/8 byte of bits read, 2 bytes written per
// weight.  Each thread handles 8 consecutive weights (one 16-byte load and
// store, one byte of bits); the grid strides over the matrix.
#include "bd_internal.cuh"
#include "bd_paths.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;

// Nearest bf16 (ties to even) of the exact value s + e, where s is a finite
// f32 and e the exact error of the f32 operation that produced s
// (|e| <= half an f32 ulp of s).
__device__ __forceinline__ uint32_t bf16_rne_exact(float s, float e) {
    const uint32_t u = __float_as_uint(s);
    const uint32_t low = u & 0xFFFFu;
    uint32_t t = u >> 16;                           // truncated towards zero (sign-magnitude)
    bool up;
    if (low != 0x8000u) {
        up = low > 0x8000u;
    } else if (e == 0.f) {
        up = (t & 1u) != 0u;                        // exact tie: to even
    } else {
        up = (e > 0.f) == (s > 0.f);                // the exact value lies beyond the midpoint
    }
    return t + (up ? 1u : 0u);
}

__device__ __forceinline__ uint32_t eff_pair(uint32_t w2, uint32_t bits2, float a) {
    uint32_t out = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float wb = __uint_as_float(h ? (w2 & 0xFFFF0000u) : (w2 << 16));
        const float d = ((bits2 >> h) & 1u) ? a : -a;
        const float s = wb + d;
        const float bb = s - wb;                    // TwoSum: exact error of s = wb + d
        const float e = (wb - (s - bb)) + (d - bb);
        out |= bf16_rne_exact(s, e) << (16 * h);
    }
    return out;
}

__global__ void __launch_bounds__(kThreads) reconstruct_kernel(const uint4* __restrict__ w_base,
                                                               const uint8_t* __restrict__ bits,
                                                               const float* __restrict__ alpha, int per_row,
                                                               int64_t chunks, int64_t chunks_per_row,
                                                               uint4* __restrict__ w_eff) {
    const float a0 = per_row ? 0.f : __ldg(alpha);
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float a = per_row ? __ldg(alpha + c / chunks_per_row) : a0;
        const uint4 w = __ldg(w_base + c);
        const uint32_t b = __ldg(bits + c);
        uint4 o;
        o.x = eff_pair(w.x, b, a);
        o.y = eff_pair(w.y, b >> 2, a);
        o.z = eff_pair(w.z, b >> 4, a);
        o.w = eff_pair(w.w, b >> 6, a);
        w_eff[c] = o;
    }
}

// Every variant present in a grouped batch (slot d of the segment plan):
// W_eff of variant plan->var[d] into weff + d * N * K.  Used by the prefill
// path, which then multiplies the tokens of slot d with it.
__global__ void __launch_bounds__(kThreads) reconstruct_plan_kernel(const uint4* __restrict__ w_base,
                                                                    BitsTable bt, const float* __restrict__ alphas,
                                                                    int alpha_rows, const SegPlan* __restrict__ plan,
                                                                    int64_t N, int64_t K, uint4* __restrict__ weff) {
    const int64_t chunks = N * K / 8, per_row = K / 8;
    const int D = plan->D;
    for (int d = 0; d < D; ++d) {
        const int v = plan->var[d];
        const uint8_t* bits = bt.p[v];
        uint4* out = weff + static_cast<int64_t>(d) * chunks;
        const float a0 = alpha_rows ? 0.f : __ldg(alphas + v);
        for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
             c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const float a = alpha_rows ? __ldg(alphas + static_cast<int64_t>(v) * N + c / per_row) : a0;
            const uint4 w = __ldg(w_base + c);
            const uint32_t b = __ldg(bits + c);
            uint4 o;
            o.x = eff_pair(w.x, b, a);
            o.y = eff_pair(w.y, b >> 2, a);
            o.z = eff_pair(w.z, b >> 4, a);
            o.w = eff_pair(w.w, b >> 6, a);
            out[c] = o;
        }
    }
}

}  // namespace

bd_status launch_reconstruct_plan(const LinearArgs& a, const SegPlan* plan, void* weff, cudaStream_t s) {
    const int64_t chunks = a.N * a.K / 8;
    int sms = sm_count();
    int64_t blocks = (chunks + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 16;
    if (blocks > cap) blocks = cap;
    reconstruct_plan_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        static_cast<const uint4*>(a.w_base), a.bits, a.alphas, a.alpha_rows, plan, a.N, a.K,
        static_cast<uint4*>(weff));
    return launch_status();
}

}  // namespace bd

using namespace bd;

extern "C" bd_status bitdelta_reconstruct(const void* w_base, const float* alpha, int32_t per_row,
                                          const uint32_t* bits, int64_t N, int64_t K, void* w_eff_out,
                                          void* stream) {
    if (N < 1 || K < 32 || K % 32 != 0 || N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return BD_ERR_SHAPE;
    if (!w_base || !alpha || !bits || !w_eff_out) return BD_ERR_NULL;
    if (!aligned(w_base, 16) || !aligned(w_eff_out, 16) || !aligned(bits, 4) || !aligned(alpha, 4))
        return BD_ERR_ALIGN;
    const int64_t chunks = N * K / 8;
    const char* wb = static_cast<const char*>(w_base);
    const char* we = static_cast<const char*>(w_eff_out);
    if (we < wb + N * K * 2 && wb < we + N * K * 2) return BD_ERR_ALIGN;   // overlapping buffers
    int sms = sm_count();
    int64_t blocks = (chunks + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 16;
    if (blocks > cap) blocks = cap;
    reconstruct_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(w_base), reinterpret_cast<const uint8_t*>(bits), alpha, per_row != 0, chunks,
        K / 8, static_cast<uint4*>(w_eff_out));
    return launch_status();
}
