// bd_decode_weff.cu -- tensor-core decode path of the fused linear for a
// batch served by a single variant (V = 1: every token is that variant, the
// base model, or invalid).
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": the conceptual fused_bitdelta_linear listing
// rebuilds W_eff = W_base + alpha * sign(delta) from the base weights and the
// packed bits and hands it to a standard linear; the fused kernel does this
// on chip without writing W_eff to HBM.  With one variant there is one W_eff,
// so this kernel builds it the way the listing does -- bf16 tiles of
// W_base + alpha s in shared memory -- and multiplies them with the bf16
// activations as they are (no staging kernel, no grouping of the tokens):
//   E[n, t] = sum_k bf16(W[n,k] + alpha_n s[n,k]) x[t,k]   (variant tokens)
//   B[n, t] = sum_k W[n,k] x[t,k]                          (base-model tokens)
// alpha_n is the variant's scale (one per matrix, or one per row).  Rounding
// each reconstructed weight to bf16 is the listing's own arithmetic (about
// 2^-9 relative); the products accumulate in fp32.
//
// One CTA owns 128 output rows (tensor-memory lanes) and a slice of K; the
// slices of a row tile run as one thread-block cluster and are summed in
// shared memory.  Warps:
//   * 0: TMA producer: per 64-column block the W_base tile (128 x 64 bf16)
//     and the activation tile (pad16(M) x 64 bf16, rows past M read as
//     zero), 128-byte swizzle, four stages; per pair of blocks the 128-row x
//     4-word tile of packed bits;
//   * 1: MMA issuer: per block four bf16 MMAs (N = pad16(M)) of the W_eff tile
//     into E and, when the batch has base-model tokens, four of the W tile
//     into B;
//   * 2..17 (four threads per row, two 16-byte chunks each): builders --
//     each thread turns its chunks of the W tile into W_eff (same swizzled
//     positions, a buffer of its own in the stage) -- and finally the
//     epilogue, which writes E or B per token column.
// The producer starts at once: nothing it loads comes from earlier work on
// the stream except the activations, and the grouping of the tokens (which
// says which are base-model tokens) is read by the warps that need it.
#include "bd_sm100.cuh"
#include "bd_tc_common.cuh"

namespace bd {

namespace {

constexpr int kBN = 128;                        // output rows per CTA
constexpr int kBK = 64;                         // K per block
constexpr int kStages = 4;                      // W / W_eff / activation stages
constexpr int kBStages = 2;                     // bits stages (two blocks each)
constexpr int kBuilderWarps = 16;               // four per tensor-memory lane quarter; a row's 8 chunks over 4 threads
constexpr int kFirstBuilder = 2;                // warps 0, 1: TMA producer, MMA issuer
constexpr int kThreads = 32 * (kFirstBuilder + kBuilderWarps);
constexpr int kMaxM = 128;
constexpr int kMaxSplits = 8;                   // cluster size (portable limit)
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kWTile = kBN * 128;          // 16 KB
constexpr int kTmemCols = 256;                  // E at column 0, B at column 128

struct WeffParams {
    CUtensorMap tm_w;                           // W_base [N, K], box 128 x 64
    CUtensorMap tm_x;                           // x [M, K], box Mb x 64
    CUtensorMap tm_bits;                        // bits [N, K/32] u32, box 128 x 4 words
    const float* alphas;                        // [1], or [N] with per-row scales
    int alpha_rows;
    const SegPlan* plan;
    const int32_t* pos2tok;
    const int32_t* pos_var;
    void* y;
    unsigned* status;
    unsigned* diag;
    int M, N, K, Mb, splits, y_bf16;
};

// Shared-memory layout of a stage: W tile, W_eff tile, activation tile.
__host__ __device__ constexpr uint32_t stage_bytes(int Mb) { return 2 * kWTile + static_cast<uint32_t>(Mb) * 128u; }
__host__ __device__ constexpr uint32_t smem_bytes(int Mb) {
    return kStages * stage_bytes(Mb) + kBStages * 2048u + 1024u;
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(saddr), "r"(rank));
    return a;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Eight bf16 weights (one 16-byte chunk) plus +-a by eight sign bits, each
// rounded to the nearest bf16.
__device__ __forceinline__ uint4 add_signs(uint4 w, uint32_t bits8, float a) {
    uint32_t in[4] = {w.x, w.y, w.z, w.w}, out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = bf16_lo(in[i]) + ((bits8 >> (2 * i)) & 1u ? a : -a);
        const float hi = bf16_hi(in[i]) + ((bits8 >> (2 * i + 1)) & 1u ? a : -a);
        const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
        out[i] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(kThreads, 1) weff_decode_kernel(const __grid_constant__ WeffParams p) {
    using namespace sm100;
    extern __shared__ uint8_t dsmem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], built[kStages], empty[kStages], b_full[kBStages], b_empty[kBStages];
    __shared__ uint64_t acc_full;
    __shared__ uint32_t tmem_base;
    __shared__ int32_t var_of_tok[kMaxM];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Mb = p.Mb;
    const uint32_t sbytes = stage_bytes(Mb);
    uint8_t* bring = base + kStages * sbytes;
    const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
    const int n0 = tile * kBN;
    // K slices at even 64-column blocks: every bits copy (two blocks, 16
    // bytes a row) starts on a 16-byte boundary
    const int kb_total = p.K / kBK;
    const int npairs = (kb_total + 1) / 2;
    const int kb0 = 2 * static_cast<int>(static_cast<int64_t>(split) * npairs / p.splits);
    const int kb1 = min(kb_total, 2 * static_cast<int>(static_cast<int64_t>(split + 1) * npairs / p.splits));
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&built[s], kBuilderWarps);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], kBuilderWarps);
        }
        mbar_init(&acc_full, 1);
        fence_mbar_init();
    }
    // the producer (thread 0, which initialised the barriers) issues the
    // first stages at once; the tensor-memory allocation and the block
    // barrier below overlap their flight
    const uint32_t tx = kWTile + static_cast<uint32_t>(Mb) * 128u;
    const int early = nkb < kStages ? nkb : kStages;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&p.tm_w);
        prefetch_tensormap(&p.tm_x);
        prefetch_tensormap(&p.tm_bits);
        for (int i = 0; i < early; ++i) {
            if ((i & 1) == 0) {
                const int bs = (i >> 1) & 1;
                mbar_expect_tx(&b_full[bs], 2048u);
                tma_load_2d(bring + bs * 2048, &p.tm_bits, &b_full[bs], 2 * (kb0 + i), n0);
            }
            uint8_t* st = base + i * sbytes;
            mbar_expect_tx(&full[i], tx);
            tma_load_2d(st, &p.tm_w, &full[i], (kb0 + i) * kBK, n0);
            tma_load_2d(st + 2 * kWTile, &p.tm_x, &full[i], (kb0 + i) * kBK, 0);
        }
    }
    if (warp == 1) tmem_alloc(&tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int issued = early, bissued = (early + 1) / 2;
            for (int i = early; i < nkb; ++i) {
                const int s = i % kStages;
                if ((i & 1) == 0) {
                    const int m = i >> 1, bs = m & 1;
                    if (!mbar_wait_sleep(&b_empty[bs], ((m >> 1) & 1) ^ 1, kWaitLimit, p.status, 42, p.diag)) break;
                    mbar_expect_tx(&b_full[bs], 2048u);
                    tma_load_2d(bring + bs * 2048, &p.tm_bits, &b_full[bs], 2 * (kb0 + i), n0);
                    bissued = m + 1;
                }
                if (!mbar_wait_sleep(&empty[s], ((i / kStages) & 1) ^ 1, kWaitLimit, p.status, 41, p.diag)) break;
                uint8_t* st = base + s * sbytes;
                mbar_expect_tx(&full[s], tx);
                tma_load_2d(st, &p.tm_w, &full[s], (kb0 + i) * kBK, n0);
                tma_load_2d(st + 2 * kWTile, &p.tm_x, &full[s], (kb0 + i) * kBK, 0);
                issued = i + 1;
            }
            // every load issued has landed before the CTA may exit
            for (int s = 0; s < kStages && s < issued; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) % kStages);
                mbar_wait_sleep(&full[s], (last / kStages) & 1, kWaitLimit, p.status, 43, p.diag);
            }
            for (int s = 0; s < kBStages && s < bissued; ++s) {
                const int last = bissued - 1 - ((bissued - 1 - s) % kBStages);
                mbar_wait_sleep(&b_full[s], (last / kBStages) & 1, kWaitLimit, p.status, 44, p.diag);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = idesc_bf16(128, Mb);
        // base-model tokens need the product of the plain W tile too (the
        // load overlaps the producer's first copies)
        const bool with_base = __shfl_sync(0xffffffffu, lane == 0 ? p.plan->n_base : 0, 0) > 0;
        bool ok = true;
        for (int i = 0; i < nkb && ok; ++i) {
            const int s = i % kStages;
            ok = warp_wait(&full[s], (i / kStages) & 1, kWaitLimit, p.status, 49, p.diag);
            if (ok) ok = warp_wait(&built[s], (i / kStages) & 1, kWaitLimit, p.status, 45, p.diag);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {               // one lane issues the block's MMAs and commit in a row
                const uint32_t st = smem_u32(base + s * sbytes);
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16) {
                    const uint64_t bx = desc_sw128(st + 2 * kWTile + 32 * k16);
                    mma_ss(tmem, desc_sw128(st + kWTile + 32 * k16), bx, idesc, (i > 0 || k16 > 0) ? 1u : 0u);
                    if (with_base) mma_ss(tmem + 128, desc_sw128(st + 32 * k16), bx, idesc, (i > 0 || k16 > 0) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            __syncwarp();
        }
        __syncwarp();
        if (elect_one()) mma_commit(&acc_full);  // completes when every MMA issued has (also after an error)
        if (!ok && lane == 0) report(p.status, BD_ERR_TIMEOUT);
    } else {
        // ---------------- builders, then the epilogue ----------------
        const int bw = warp - kFirstBuilder;
        const int q4 = warp & 3;                            // tensor-memory lane quarter (warp % 4)
        const int h = bw >> 2;                              // chunks 2h, 2h+1 of the row
        const int r = 32 * q4 + lane;                       // tile row of this thread
        const int n = n0 + r;
        const float a = p.alpha_rows ? (n < p.N ? __ldg(p.alphas + n) : 0.f) : __ldg(p.alphas);
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kStages, m = i >> 1, half = i & 1, bs = m & 1;
            if (ok && half == 0) ok = warp_wait(&b_full[bs], (m >> 1) & 1, kWaitLimit, p.status, 46, p.diag);
            if (ok) ok = warp_wait(&full[s], (i / kStages) & 1, kWaitLimit, p.status, 47, p.diag);
            if (ok) {
                const uint8_t* wrow = base + s * sbytes + r * 128;
                uint8_t* erow = base + s * sbytes + kWTile + r * 128;
                // bits of columns 16h .. 16h+15 of this block
                const uint32_t word = reinterpret_cast<const uint32_t*>(bring + bs * 2048)[r * 4 + 2 * half + (h >> 1)];
                const uint32_t bits16 = word >> (16 * (h & 1));
                // 16-byte chunk c of the row (columns 8c .. 8c+7) sits at
                // chunk position c ^ (r & 7) under the 128-byte swizzle
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * h + cc;
                    const int pc = (c ^ (r & 7)) * 16;
                    const uint4 w = *reinterpret_cast<const uint4*>(wrow + pc);
                    *reinterpret_cast<uint4*>(erow + pc) = add_signs(w, (bits16 >> (8 * cc)) & 0xFFu, a);
                }
            }
            // the tensor core reads the W_eff tile through the async proxy
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&built[s]);
                if (half == 1 || i == nkb - 1) mbar_arrive(&b_empty[bs]);
            }
        }
        // ---- epilogue: E for variant tokens, B for base-model tokens ----
        // which token is which (the grouping's inverse), once every builder
        // is past its last block
        if (h == 0)
            for (int t = lane + 32 * q4; t < kMaxM; t += 128) var_of_tok[t] = -2;
        named_bar_sync(1, 32 * kBuilderWarps);
        for (int q = lane + 32 * bw; q < p.M; q += 32 * kBuilderWarps) var_of_tok[p.pos2tok[q]] = p.pos_var[q];
        named_bar_sync(1, 32 * kBuilderWarps);
        if (ok) ok = warp_wait(&acc_full, 0, kWaitLimit, p.status, 48, p.diag);
        tc_fence_after();
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q4) << 16;
        // the partial tile [Mb][128] f32 of a K slice lives in the stage ring,
        // idle once every MMA has completed
        float* psm = reinterpret_cast<float*>(base);
        for (int c0 = 16 * h; c0 < Mb && ok; c0 += 64) {
            uint32_t e[16], b[16];
            tmem_ld16(tmem + lane_addr + c0, e);
            tmem_ld16(tmem + lane_addr + 128 + c0, b);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = c0 + j;
                if (t >= p.M) break;
                const int v = var_of_tok[t];
                const float val = v == 0 ? __uint_as_float(e[j]) : (v == -1 ? __uint_as_float(b[j]) : 0.f);
                if (p.splits > 1) {
                    psm[t * kBN + r] = val;
                } else if (n < p.N) {
                    if (p.y_bf16) static_cast<__nv_bfloat16*>(p.y)[static_cast<int64_t>(t) * p.N + n] = __float2bfloat16_rn(val);
                    else static_cast<float*>(p.y)[static_cast<int64_t>(t) * p.N + n] = val;
                }
            }
        }
    }

    __syncthreads();
    if (p.splits > 1) {
        // the K slices of this row tile are the CTAs of one cluster (rank =
        // split): CTA `split` sums its share of the tile over the slices'
        // shared memory in the order 0, 1, 2, ... and writes y
        cluster_sync_all();
        const int rows = min(kBN, p.N - n0);
        const uint32_t psm_a = smem_u32(base);
        const int per_t = kBN / 4;
        const int total = p.M * per_t;
        const int g0 = static_cast<int>(static_cast<int64_t>(split) * total / p.splits);
        const int g1 = static_cast<int>(static_cast<int64_t>(split + 1) * total / p.splits);
        for (int gi = g0 + static_cast<int>(threadIdx.x); gi < g1; gi += blockDim.x) {
            const int t = gi / per_t, r4 = 4 * (gi % per_t);
            if (r4 >= rows) continue;
            const uint32_t off = psm_a + static_cast<uint32_t>(gi) * 16u;
            float4 acc = ld_cluster_f4(cluster_map(off, 0));
            for (int sl = 1; sl < p.splits; ++sl) {
                const float4 v = ld_cluster_f4(cluster_map(off, static_cast<uint32_t>(sl)));
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
            const int64_t o = static_cast<int64_t>(t) * p.N + n0 + r4;
            if (r4 + 4 <= rows && (p.N & 3) == 0) {
                if (p.y_bf16) {
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.y) + o) =
                        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
                } else {
                    *reinterpret_cast<float4*>(static_cast<float*>(p.y) + o) = acc;
                }
            } else {
                const float v4[4] = {acc.x, acc.y, acc.z, acc.w};
                for (int j = 0; j < 4 && r4 + j < rows; ++j) {
                    if (p.y_bf16) static_cast<__nv_bfloat16*>(p.y)[o + j] = __float2bfloat16_rn(v4[j]);
                    else static_cast<float*>(p.y)[o + j] = v4[j];
                }
            }
        }
        cluster_sync_all();                  // no CTA leaves while its tile is being read
    }
    if (warp == 1) {
        // every MMA has completed before the tensor memory is freed
        warp_wait(&acc_full, 0, kWaitLimit, p.status, 50, p.diag);
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Clusters of `s` CTAs (one per SM at this kernel's shared-memory size) that
// run at once: the GPCs' SM counts need not be multiples of s.  Cached per
// device; 0 if the query fails.
int cluster_capacity(int s, int smem) {
    static int cache[64][kMaxSplits + 1] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev][s] > 0) return cache[dev][s];
    if (s == 1) return cache[dev][1] = sm_count();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s * 64));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, weff_decode_kernel, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 0;
    }
    return cache[dev][s] = n;
}

// K slices per row tile (at most 8, the cluster size; each slice at least 8
// blocks): the fewest block-times on the busiest SM, counting whole waves of
// clusters -- waves x (blocks per slice + about six blocks' worth of fixed
// cost per CTA).  A 224-tile matrix (28672 rows) thus runs in slices of 64
// blocks rather than in two waves of 128.
int weff_splits(int64_t n_tiles, int kb_total, int smem) {
    constexpr int64_t kFixedBlocks = 6;
    int best = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= kMaxSplits && (s == 1 || kb_total / s >= 8); ++s) {
        const int cap = cluster_capacity(s, smem);          // clusters at once
        if (cap < 1) continue;
        const int64_t waves = (n_tiles + cap - 1) / cap;
        const int64_t cost = waves * ((kb_total + s - 1) / s + kFixedBlocks);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = s; }
    }
    return best;
}

}  // namespace

bool decode_weff_supported(const LinearArgs& a) {
    return a.V == 1 && a.M >= 1 && a.M <= kMaxM && a.K % kBK == 0 && a.K >= kBK && a.N >= 1 &&
           a.N < (int64_t(1) << 31) && a.K < (int64_t(1) << 31);
}

bd_status launch_decode_weff(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s) {
    const int M = static_cast<int>(a.M);
    const int Mb = pad16(M);
    const int64_t n_tiles = (a.N + kBN - 1) / kBN;
    const int smem = static_cast<int>(smem_bytes(Mb));
    if (!set_smem_attr(reinterpret_cast<const void*>(weff_decode_kernel), smem, 3)) return BD_ERR_CUDA;
    const int splits = weff_splits(n_tiles, static_cast<int>(a.K / kBK), smem);
    WeffParams p;
    memset(&p, 0, sizeof p);
    if (!make_tmap_bf16_sw128(&p.tm_w, a.w_base, a.N, a.K, kBN) ||
        !make_tmap_bf16_sw128(&p.tm_x, a.x, a.M, a.K, Mb) ||
        !make_tmap_bits(&p.tm_bits, a.bits.p[0], a.N, a.K / 32, kBN))
        return BD_ERR_CUDA;
    p.alphas = a.alphas;
    p.alpha_rows = a.alpha_rows;
    p.plan = w.g.plan;
    p.pos2tok = w.g.pos2tok;
    p.pos_var = w.g.pos_var;
    p.y = a.y;
    p.status = w.status;
    p.diag = w.status + 2;
    p.M = M;
    p.N = static_cast<int>(a.N);
    p.K = static_cast<int>(a.K);
    p.Mb = Mb;
    p.splits = splits;
    p.y_bf16 = (a.y_dtype == BD_BF16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_tiles * splits));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, weff_decode_kernel, p) != cudaSuccess) return BD_ERR_CUDA;
    return launch_status();
}

}  // namespace bd
