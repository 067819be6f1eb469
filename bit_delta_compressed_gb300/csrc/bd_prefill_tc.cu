// bd_prefill_tc.cu -- tensor-core prefill path of the fused multi-variant
// linear.
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture" (reconstruction W_eff = W_base + alpha_v *
// sign(delta_v) on chip, fused with the matmul; the conceptual
// fused_bitdelta_linear listing builds w_eff in the base weights' dtype) and
// section "Latency profile" (the reconstruction cost is paid in prefill).
//
// With thousands of tokens per variant the work is a dense bf16 contraction
// per variant, so each W_eff tile is built once in shared memory and reused
// across the CTA's tokens on the tensor cores.  A CTA covers kRowTiles x 128
// weight rows and kTokTiles x 256 tokens (all 512 tensor-memory columns); the
// tile is sized for reuse: per 64-column block it loads 32 KB of W and 32 KB
// of activations from L2 for 8.4 MFLOP, and the L2-to-SM fill rate, not the
// tensor pipe, sets the pace:
//   * a TMA producer loads the W_base tile (256 rows x 64 columns) and the
//     token tile (256 grouped tokens x 64 columns) of one variant;
//   * builder warps (one thread per weight row) rewrite the W tile in
//     place as bf16(W_base + alpha_v * s_v) from the variant's sign bits,
//     then hand it to the tensor core (async-proxy fence + mbarrier);
//   * one thread issues tcgen05.mma (M = 128 weight rows per MMA, N = 256
//     tokens, one MMA per row tile and token tile per K step, fp32
//     accumulators in tensor memory);
//   * the builder warps then read the accumulator out and store y rows of
//     the tokens that belong to the variant.
// Tokens of the base model (id -1) use W_base unchanged.  When the average
// variant of the batch has >= 2048 tokens, every present variant's W_eff is
// first materialised in the workspace (nearest bf16, one HBM pass per
// variant) and the kernel loads those tiles ready-made: the in-tile rewrite
// costs about a quarter of the GEMM time, the pass 4.125 bytes per weight.
#include "bd_sm100.cuh"
#include "bd_tc_common.cuh"

namespace bd {

size_t decode_tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V);

namespace {

constexpr int kRowTiles = 2;        // 128-row MMA tiles per CTA (TMEM lanes = rows of one tile)
constexpr int kTokTiles = 1;        // 256-token MMA tiles per CTA
constexpr int kBM = 128;            // MMA M
constexpr int kBX = 256;            // MMA N, and tokens per activation TMA box
constexpr int kBN = kBM * kRowTiles;    // weight rows per CTA
constexpr int kBT = kBX * kTokTiles;    // tokens per CTA
constexpr int kBK = 64;
constexpr int kBuildWarps = 4 * kRowTiles;
constexpr int kThreads = 64 + 32 * kBuildWarps;   // warp 0 TMA, warp 1 MMA, then build + epilogue
constexpr int kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kStageBytes = kBN * 128 + kBT * 128;
constexpr int kStages = (225 * 1024) / kStageBytes < 4 ? (225 * 1024) / kStageBytes : 4;
static_assert(kRowTiles * kTokTiles * kBX <= kTmemCols, "accumulators must fit tensor memory");
static_assert(kStages >= 2, "at least two pipeline stages");

struct PrefillParams {
    CUtensorMap tm_w;                       // W_base [N, K]
    CUtensorMap tm_x;                       // grouped activations [Mpad, K]
    CUtensorMap tm_weff[BITDELTA_MAX_VARIANTS];  // materialised W_eff of plan slot d (when prebuilt)
    int prebuilt;                           // 1: W_eff tiles come ready from HBM, no rewrite
    const uint32_t* bits[BITDELTA_MAX_VARIANTS];
    const float* alphas;                        // [V], or [V, N] when alpha_rows
    int alpha_rows;
    const SegPlan* plan;
    const int32_t* pos2tok;
    void* y;
    unsigned* status;
    unsigned* diag;
    int M, N, K, n_wtiles, y_bf16;
};

// Token tile `jt` (in grouped order over base tokens then each variant) ->
// first grouped position, end position and variant id (-1 = base).
__device__ bool token_tile(const SegPlan& pl, int jt, int& pos0, int& pos_end, int& var, int& slot) {
    int nt = (pl.n_base + kBT - 1) / kBT;
    if (jt < nt) {
        pos0 = jt * kBT;
        pos_end = pl.n_base;
        var = -1;
        slot = -1;
        return true;
    }
    jt -= nt;
    for (int d = 0; d < pl.D; ++d) {
        nt = (pl.cnt[d] + kBT - 1) / kBT;
        if (jt < nt) {
            pos0 = pl.off[d] + jt * kBT;
            pos_end = pl.off[d] + pl.cnt[d];
            var = pl.var[d];
            slot = d;
            return true;
        }
        jt -= nt;
    }
    return false;
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
    using namespace sm100;
    extern __shared__ uint8_t dsmem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_full[kStages], bar_built[kStages], bar_empty[kStages], acc_full;
    __shared__ uint32_t tmem_base;
    __shared__ SegPlan pl;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    {
        const int* src = reinterpret_cast<const int*>(p.plan);
        int* dst = reinterpret_cast<int*>(&pl);
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(SegPlan) / 4); i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    // tile order: 8 weight tiles x all token tiles, then the next 8 weight
    // tiles, so concurrently running CTAs share W and token tiles in L2
    const int group_w = 8;
    const int jt_count = gridDim.x / p.n_wtiles;
    const int per_group = group_w * jt_count;
    const int grp = blockIdx.x / per_group, rem = blockIdx.x % per_group;
    const int wt_in = min(group_w, p.n_wtiles - grp * group_w);
    const int wt = grp * group_w + rem % wt_in;
    const int jt = rem / wt_in;
    int pos0 = 0, pos_end = 0, var = -1, slot = -1;
    if (wt >= p.n_wtiles || jt >= jt_count || !token_tile(pl, jt, pos0, pos_end, var, slot)) return;
    // W tiles: the variant's materialised W_eff (prebuilt), else W_base
    // rewritten in shared memory by the builder warps
    const bool use_weff = p.prebuilt && var >= 0;
    const CUtensorMap* tmw = use_weff ? &p.tm_weff[slot] : &p.tm_w;
    const int n0 = wt * kBN;
    const int nkb = p.K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_built[s], kBuildWarps);
            mbar_init(&bar_empty[s], 1);
        }
        mbar_init(&acc_full, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(tmw);
            prefetch_tensormap(&p.tm_x);
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kStages;
                if (!mbar_wait_sleep(&bar_empty[s], ((kb / kStages) & 1) ^ 1, kWaitLimit, p.status, 11, p.diag)) break;
                mbar_expect_tx(&bar_full[s], kStageBytes);
                uint8_t* st = base + s * kStageBytes;
                tma_load_2d(st, tmw, &bar_full[s], kb * kBK, n0);
                for (int h = 0; h < kBT / kBX; ++h)
                    tma_load_2d(st + kBN * 128 + h * kBX * 128, &p.tm_x, &bar_full[s], kb * kBK, pos0 + h * kBX);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kBM, kBX);
            bool ok = true;
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % kStages;
                if (!(ok = mbar_wait_sleep(&bar_built[s], (kb / kStages) & 1, kWaitLimit, p.status, 12, p.diag))) break;
                tc_fence_after();
                const uint32_t sa = smem_u32(base + s * kStageBytes);
                const uint32_t sb = sa + kBN * 128;
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16)
#pragma unroll
                    for (int rt = 0; rt < kRowTiles; ++rt)
#pragma unroll
                        for (int tt = 0; tt < kTokTiles; ++tt)
                            mma_ss(tmem + kBX * (rt * kTokTiles + tt), desc_sw128(sa + rt * kBM * 128 + 32 * k16),
                                   desc_sw128(sb + tt * kBX * 128 + 32 * k16), idesc, (kb > 0 || k16 > 0) ? 1u : 0u);
                mma_commit(&bar_empty[s]);
            }
            if (ok) mma_commit(&acc_full);
        }
    } else {
        // builder warps: thread r owns weight row r of the CTA's rows; warp
        // (q, rt) covers TMEM lane quarter q of row tile rt
        const int q = warp % 4;
        const int rt = (warp - 2) / 4;
        const int r = kBM * rt + 32 * q + lane;
        const int n = n0 + r;
        const bool row_ok = n < p.N;
        const uint32_t* bits = (var >= 0 && !use_weff) ? p.bits[var] : nullptr;
        const float alpha = var < 0 ? 0.f
                            : p.alpha_rows ? (row_ok ? p.alphas[static_cast<int64_t>(var) * p.N + n] : 0.f)
                                           : p.alphas[var];
        const uint32_t abits = __float_as_uint(alpha);
        const int words_per_row = p.K / 32;
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s = kb % kStages;
            uint2 wbits = make_uint2(0, 0);
            if (bits && row_ok) wbits = __ldg(reinterpret_cast<const uint2*>(bits + static_cast<int64_t>(n) * words_per_row) + kb);
            if (!(ok = mbar_wait_sleep(&bar_full[s], (kb / kStages) & 1, kWaitLimit, p.status, 13, p.diag))) break;
            if (bits) {
                uint8_t* row = base + s * kStageBytes + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {           // 16-byte chunk c = columns 8c..8c+7
                    uint4* ptr = reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4));
                    uint4 v = *ptr;
                    const uint32_t word = (c < 4) ? wbits.x : wbits.y;
                    const int b0 = (c & 3) * 8;
                    uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t bl = (word >> (b0 + 2 * i)) & 1u, bh = (word >> (b0 + 2 * i + 1)) & 1u;
                        const float lo = __uint_as_float(w4[i] << 16) + __uint_as_float(abits ^ ((bl ^ 1u) << 31));
                        const float hi = __uint_as_float(w4[i] & 0xFFFF0000u) + __uint_as_float(abits ^ ((bh ^ 1u) << 31));
                        __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
                        w4[i] = *reinterpret_cast<uint32_t*>(&pr);
                    }
                    *ptr = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_built[s]);
        }
        const bool acc_ok = ok && mbar_wait_sleep(&acc_full, 0, kWaitLimit, p.status, 14, p.diag);
        if (acc_ok && p.y_bf16 && p.N % 8 == 0) {
            // bf16 outputs: stage the tile as [token][row] in the (now idle)
            // pipeline memory, then write each token's kBN outputs as one
            // contiguous 16-byte-per-lane row of y
            tc_fence_after();
            const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
            const int ntok = min(kBT, pos_end - pos0);
            __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(base);
            for (int c0 = 0; c0 < ntok; c0 += 16) {
                uint32_t v[16];
                const int col = kBX * (rt * kTokTiles + c0 / kBX) + c0 % kBX;
                tmem_ld16(tmem + lane_addr + col, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) tile[(c0 + i) * kBN + r] = __float2bfloat16_rn(__uint_as_float(v[i]));
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kBuildWarps * 32) : "memory");
            const int rows = min(kBN, p.N - n0);
            for (int t = warp - 2; t < ntok; t += kBuildWarps) {
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.y) + static_cast<int64_t>(p.pos2tok[pos0 + t]) * p.N + n0;
                const __nv_bfloat16* src = tile + t * kBN;
                if (rows == kBN) {
                    static_assert(kBN == 32 * 8, "one 16-byte vector per lane per token row");
                    reinterpret_cast<uint4*>(dst)[lane] = reinterpret_cast<const uint4*>(src)[lane];
                } else {
                    for (int rr = lane; rr < rows; rr += 32) dst[rr] = src[rr];
                }
            }
        } else if (acc_ok) {
            tc_fence_after();
            const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
            for (int c0 = 0; c0 < kBT && pos0 + c0 < pos_end; c0 += 16) {
                uint32_t v[16];
                const int col = kBX * (rt * kTokTiles + c0 / kBX) + c0 % kBX;
                tmem_ld16(tmem + lane_addr + col, v);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int pos = pos0 + c0 + i;
                        if (pos >= pos_end) break;
                        const int64_t o = static_cast<int64_t>(p.pos2tok[pos]) * p.N + n;
                        const float val = __uint_as_float(v[i]);
                        if (p.y_bf16) static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(val);
                        else static_cast<float*>(p.y)[o] = val;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// invalid ids get zero rows
__global__ void zero_invalid_kernel(const SegPlan* plan, const int32_t* pos2tok, void* y, int N, int y_bf16) {
    const int M = plan->M, ninv = plan->n_invalid;
    for (int i = blockIdx.x; i < ninv; i += gridDim.x) {
        const int64_t t = pos2tok[M - ninv + i];
        for (int n = threadIdx.x; n < N; n += blockDim.x) {
            if (y_bf16) static_cast<__nv_bfloat16*>(y)[t * N + n] = __float2bfloat16_rn(0.f);
            else static_cast<float*>(y)[t * N + n] = 0.f;
        }
    }
}

// grouped copy of the activations (rows [0, Mpad); rows past the valid
// tokens are zero)
__global__ void __launch_bounds__(256) gather_x_kernel(const uint4* __restrict__ x, int K,
                                                       const SegPlan* __restrict__ plan,
                                                       const int32_t* __restrict__ pos2tok,
                                                       uint4* __restrict__ xg) {
    const int row = blockIdx.y;
    const int64_t vec = K / 8;
    const int n_valid = plan->M - plan->n_invalid;
    const int tok = row < n_valid ? pos2tok[row] : -1;
    for (int64_t i = blockIdx.x * blockDim.x + threadIdx.x; i < vec; i += gridDim.x * blockDim.x)
        xg[row * vec + i] = tok >= 0 ? __ldg(x + tok * vec + i) : make_uint4(0, 0, 0, 0);
}

// Materialise each present variant's W_eff before the GEMM when the average
// variant has at least this many tokens: rebuilding a W tile in shared memory
// costs about a quarter of the GEMM time, a reconstruction pass over HBM
// 4.125 bytes per weight, which is less from ~2000 tokens per variant on.
constexpr int64_t kMatTokensPerVariant = 2048;
constexpr int64_t kMatMaxBytes = int64_t(32) << 30;

int64_t mat_slots(int64_t M, int32_t V) { return V < M ? V : M; }

bool materialise(int64_t M, int64_t N, int64_t K, int32_t V) {
    const int64_t d = mat_slots(M, V);
    return d >= 1 && M / d >= kMatTokensPerVariant && d * N * K * 2 <= kMatMaxBytes;
}

size_t prefill_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V) {
    size_t b = round_up(static_cast<size_t>(pad16(static_cast<int>(M))) * K * 2, kAlign);
    if (materialise(M, N, K, V)) b += round_up(static_cast<size_t>(mat_slots(M, V) * N * K * 2), kAlign);
    return b;
}

}  // namespace

bool prefill_tc_supported(const LinearArgs& a) {
    return a.M >= 1 && a.M <= 65520 && a.K % kBK == 0 && a.N >= 1 && a.N < (int64_t(1) << 31) &&
           a.M * a.K < (int64_t(1) << 40);
}

size_t tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V) {
    size_t a = decode_tc_scratch_bytes(M, N, K, V);
    size_t b = (K % kBK == 0 && M >= 1 && M <= 65520) ? prefill_scratch_bytes(M, N, K, V) : 0;
    size_t c = decode_fold_scratch_bytes(M, N, K, V);
    size_t m = a > b ? a : b;
    return m > c ? m : c;
}

bd_status launch_prefill_tc(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s) {
    const int M = static_cast<int>(a.M), N = static_cast<int>(a.N), K = static_cast<int>(a.K);
    const int Mpad = pad16(M);
    if (prefill_scratch_bytes(a.M, a.N, a.K, a.V) > w.tc_bytes) return BD_ERR_WORKSPACE;
    uint16_t* xg = static_cast<uint16_t*>(w.tc_scratch);
    const bool mat = materialise(a.M, a.N, a.K, a.V);
    uint8_t* weff = static_cast<uint8_t*>(w.tc_scratch) +
                    round_up(static_cast<size_t>(Mpad) * a.K * 2, kAlign);
    if (mat && launch_reconstruct_plan(a, w.g.plan, weff, s) != BD_OK) return BD_ERR_CUDA;
    gather_x_kernel<<<dim3((K / 8 + 255) / 256 < 8 ? (K / 8 + 255) / 256 : 8, Mpad), 256, 0, s>>>(
        static_cast<const uint4*>(a.x), K, w.g.plan, w.g.pos2tok, reinterpret_cast<uint4*>(xg));
    if (launch_status() != BD_OK) return BD_ERR_CUDA;
    zero_invalid_kernel<<<8, 256, 0, s>>>(w.g.plan, w.g.pos2tok, a.y, N, a.y_dtype == BD_BF16);
    if (launch_status() != BD_OK) return BD_ERR_CUDA;
    PrefillParams p;
    memset(&p, 0, sizeof p);
    static_assert(kBN <= 256 && kBX <= 256, "TMA boxes are at most 256 rows");
    p.prebuilt = mat ? 1 : 0;
    if (mat)
        for (int64_t d = 0; d < mat_slots(a.M, a.V); ++d)
            if (!make_tmap_bf16_sw128(&p.tm_weff[d], weff + d * a.N * a.K * 2, a.N, a.K, kBN)) return BD_ERR_CUDA;
    if (!make_tmap_bf16_sw128(&p.tm_w, a.w_base, a.N, a.K, kBN) ||
        !make_tmap_bf16_sw128(&p.tm_x, xg, Mpad, a.K, kBX))
        return BD_ERR_CUDA;
    for (int v = 0; v < a.V; ++v) p.bits[v] = reinterpret_cast<const uint32_t*>(a.bits.p[v]);
    p.alphas = a.alphas;
    p.alpha_rows = a.alpha_rows;
    p.plan = w.g.plan;
    p.pos2tok = w.g.pos2tok;
    p.y = a.y;
    p.status = w.status;
    p.diag = w.status + 2;
    p.M = M;
    p.N = N;
    p.K = K;
    p.n_wtiles = (N + kBN - 1) / kBN;
    p.y_bf16 = (a.y_dtype == BD_BF16);
    // token tiles: at most one partial tile per present variant plus base tokens
    const int64_t d_max = a.V < a.M ? a.V : a.M;
    const int64_t jt = (a.M + kBT - 1) / kBT + d_max + 1;
    const int64_t grid = jt * p.n_wtiles;
    if (grid > 0x7fffffff) return BD_ERR_UNSUPPORTED;
    const int smem = kStages * kStageBytes + 1024;
    if (!set_smem_attr(reinterpret_cast<const void*>(prefill_tc_kernel), smem, 1)) return BD_ERR_CUDA;
    prefill_tc_kernel<<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p);
    return launch_status();
}

}  // namespace bd
