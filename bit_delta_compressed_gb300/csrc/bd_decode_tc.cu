// bd_decode_tc.cu -- tensor-core decode path of the fused multi-variant linear.
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": the base weights are read once and shared by every
// variant; each variant's delta arrives as packed sign bits and is expanded
// on chip, so W_eff = W_base + alpha_v * sign(delta_v) never exists in HBM.
//
// One CTA owns 128 output rows (the 128 lanes of tensor memory) and a slice
// of K (split-K; the slices of a row tile are summed in a fixed order by the
// CTA that finishes last).  For every 64-column K block:
//   * a TMA warp loads the W_base tile, the batch's activations in grouped
//     order (X_c, bf16) and the sign operand's activations (X_p);
//   * one issuer thread accumulates D_base += W * X_c^T (bf16, both operands
//     in shared memory, fp32 accumulator in tensor memory);
//   * eight expansion warps turn each present variant's sign bits into +-1
//     in fp8 e4m3 straight in tensor memory: for a 32-bit word w of bits,
//     register j = ((w << (7 - j)) & 0x80808080) ^ 0xB8B8B8B8 holds columns
//     j, j+8, j+16, j+24 (bit 1 -> +1.0, bit 0 -> -1.0): one shift and one
//     LOP3 per four weights;
//   * eight more issuer threads (variants split between them; their MMAs
//     overlap on the tensor pipe) accumulate D_sign[segment of v] +=
//     S_v * X_p^T with kind::f8f6f4, A from tensor memory;
//   * the epilogue writes y = D_base + alpha_v * 2^-sigma_t * D_sign.
// X_p holds each token's activations scaled by a power of two 2^sigma_t
// (largest magnitude in [128, 256)) and split exactly into two e4m3 terms,
// hi = rn(x 2^sigma) and lo = rn(x 2^sigma - hi): every element within 2^9
// of the token's largest magnitude is represented exactly, smaller ones to
// 2^-17 of that maximum.  The columns inside each 32-column group are
// permuted to match the register layout above.  Variants whose padded
// segments do not fit next to D_base are handled in further passes over the
// same K slice; those passes reload only X_p and bits, never W_base.
#include <cuda_fp8.h>

#include "bd_sm100.cuh"
#include "bd_tc_common.cuh"

namespace bd {

namespace {

constexpr int kBN = 128;                  // output rows per CTA (TMEM lanes)
constexpr int kBK = 64;                   // K per stage
constexpr int kWStages = 4;               // W_base tiles in flight (HBM)
constexpr int kXStages = 2;               // activation tiles in flight (L2)
constexpr int kIssuers = 8;               // sign-MMA issuer threads
constexpr int kSlotCols = 8;              // one 32-column word of e4m3 per row
constexpr int kStagingCols = kIssuers * 2 * kSlotCols;
constexpr int kBaseCol = kStagingCols;
constexpr int kTmemCols = 512;
constexpr int kBitStages = 2;             // bits stages, each two K blocks (16 bytes per row)
constexpr int kMaxM = 176;                // pad16(M) must fit next to one variant's segment
constexpr int kExpandWarps = 8;
constexpr int kThreads = 32 * (2 + kIssuers + kExpandWarps);   // 576
constexpr int kFirstIssuerWarp = 2;
constexpr int kFirstExpandWarp = 2 + kIssuers;
constexpr uint32_t kWaitLimit = 1u << 20;

struct DecodeParams {
    CUtensorMap tm_w;                     // W_base [N, K] bf16, box 128 rows
    CUtensorMap tm_xc;                    // X_c [Mb, K] bf16, box Mb rows
    CUtensorMap tm_xp;                    // X_p [P_bound, 2K] bytes (e4m3 hi|lo per 64-col block), box 16 rows
    CUtensorMap tm_xp128;                 // the same, box 128 rows
    CUtensorMap tm_bits[BITDELTA_MAX_VARIANTS];   // packed bits [N, K/32] u32, box 128 rows x 4 words
    const float* alphas;                        // [V], or [V, N] when alpha_rows
    int alpha_rows;
    const SegPlan* plan;
    const int32_t* pos2tok;
    const int32_t* sigma;                 // per token
    void* y;
    float* part;                          // [splits][M][N] when splits > 1
    unsigned* tickets;                    // [n_tiles]
    unsigned* status;
    unsigned* diag;
    int M, N, K, Mb, budget, splits, y_bf16;
    int cluster_reduce;                   // the K slices of a row tile form one cluster (2..8 slices, M <= 128)
};

constexpr uint32_t kBitsTile = kBN * 16;  // one variant, 128 rows x 4 words
constexpr uint32_t kWTile = kBN * 128;    // 128 rows x 64 bf16
static_assert(kWStages * kWTile >= 128 * kBN * 4, "the W ring holds a 128-token f32 partial tile");

// Shared memory: W ring | activation ring (X_c rows then X_p rows per stage)
// | bits ring (kMaxPassVariants tiles per stage).
struct SmemLayout {
    uint32_t w, x, x_stage, xp_off, bits, bits_stage, total;
};

__host__ __device__ inline SmemLayout smem_layout(int Mb, int budget) {
    SmemLayout L;
    L.w = 0;
    L.x = kWStages * kWTile;
    L.x_stage = (Mb + budget) * 128;
    L.xp_off = Mb * 128;
    L.bits = L.x + kXStages * L.x_stage;
    L.bits_stage = kMaxPassVariants * kBitsTile;
    L.total = L.bits + kBitStages * L.bits_stage;
    return L;
}

__device__ __forceinline__ float exp2i(int e) {      // exact 2^e, e in [-126, 127]
    return __int_as_float((127 + e) << 23);
}

// Distributed shared memory of a thread-block cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
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

// Output (token t, row n = n0 + r) of this CTA: its partial tile in shared
// memory (cluster reduction), its K slice's partial in HBM (ticket
// reduction), or y itself (one slice).
__device__ __forceinline__ void store_y(const DecodeParams& p, float* psm, int split, int t, int n, int r, float v) {
    if (p.cluster_reduce) {
        psm[t * kBN + r] = v;
    } else if (p.splits > 1) {
        p.part[(static_cast<int64_t>(split) * p.M + t) * p.N + n] = v;
    } else if (p.y_bf16) {
        static_cast<__nv_bfloat16*>(p.y)[static_cast<int64_t>(t) * p.N + n] = __float2bfloat16_rn(v);
    } else {
        static_cast<float*>(p.y)[static_cast<int64_t>(t) * p.N + n] = v;
    }
}

// Pass g of the plan: present-variant range and its padded rows.
struct PassInfo {
    int d0, d1, row0, rows;
};
__device__ __forceinline__ PassInfo pass_info(const SegPlan& pl, int g) {
    PassInfo q;
    q.d0 = pl.group_first[g];
    q.d1 = pl.group_first[g + 1];
    q.row0 = (q.d1 > q.d0) ? pl.seg[q.d0] : 0;
    q.rows = (q.d1 > q.d0) ? pl.seg[q.d1 - 1] + pad16(pl.cnt[q.d1 - 1]) - q.row0 : 0;
    return q;
}

// Variants of a pass handled by issuer i: local indices i, i + 8, ...
__device__ __forceinline__ int issuer_count(int nd, int i) { return nd > i ? (nd - i + kIssuers - 1) / kIssuers : 0; }

__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
    using namespace sm100;
    extern __shared__ uint8_t dsmem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t w_full[kWStages], w_empty[kWStages], x_full[kXStages], x_empty[kXStages];
    __shared__ uint64_t bits_full[kBitStages], bits_empty[kBitStages];
    __shared__ uint64_t tm_full[kIssuers][2], tm_empty[kIssuers][2];
    __shared__ uint64_t acc_full, acc_empty;
    __shared__ uint32_t tmem_base;
    __shared__ SegPlan pl;
    __shared__ int last_cta;
    __shared__ int32_t tok_s[kMaxM];            // grouped position -> token
    __shared__ float scale_s[kMaxM];            // grouped position -> alpha_v * 2^-sigma_t

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Mb = p.Mb;
    const SmemLayout L = smem_layout(Mb, p.budget);
    // cluster reduction: the partial tile [M][128] f32 lives in the W ring,
    // which no load or MMA touches after pass 0's MMAs have completed
    float* psm = reinterpret_cast<float*>(base + L.w);
    const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
    const int n0 = tile * kBN;
    const int kb_total = p.K / kBK;
    const int kb0 = static_cast<int>(static_cast<int64_t>(split) * kb_total / p.splits);
    const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * kb_total / p.splits);
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], 1);                     // the base issuer
        }
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&x_empty[s], 1 + kIssuers);         // every issuer releases every stage
        }
        for (int b = 0; b < kBitStages; ++b) {
            mbar_init(&bits_full[b], 1);
            mbar_init(&bits_empty[b], kExpandWarps);
        }
        for (int i = 0; i < kIssuers; ++i)
            for (int h = 0; h < 2; ++h) {
                mbar_init(&tm_full[i][h], 4);              // four lane-quarter warps per word
                mbar_init(&tm_empty[i][h], 1);
            }
        mbar_init(&acc_full, 1 + kIssuers);
        mbar_init(&acc_empty, kExpandWarps);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kTmemCols);
    // everything above overlaps the staging kernel; from here on its outputs
    // (activations, scales, tickets) are read
    asm volatile("griddepcontrol.wait;" ::: "memory");
    {   // copy the segment plan into shared memory
        const int* src = reinterpret_cast<const int*>(p.plan);
        int* dst = reinterpret_cast<int*>(&pl);
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(SegPlan) / 4); i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    // per grouped position: token and the epilogue's scale of the sign product
    for (int d = 0; d < pl.D; ++d) {
        const float alpha = p.alpha_rows ? 1.f : p.alphas[pl.var[d]];    // per-row scales: in the epilogue
        for (int j = threadIdx.x; j < pl.cnt[d]; j += blockDim.x) {
            const int pos = pl.off[d] + j;
            const int tok = p.pos2tok[pos];
            tok_s[pos] = tok;
            scale_s[pos] = alpha * exp2i(-p.sigma[tok]);
        }
    }
    for (int pos = threadIdx.x; pos < pl.n_base; pos += blockDim.x) tok_s[pos] = p.pos2tok[pos];
    for (int pos = p.M - pl.n_invalid + threadIdx.x; pos < p.M; pos += blockDim.x) tok_s[pos] = p.pos2tok[pos];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const int n_groups = pl.n_groups;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            prefetch_tensormap(&p.tm_w);
            prefetch_tensormap(&p.tm_xc);
            prefetch_tensormap(&p.tm_xp);
            prefetch_tensormap(&p.tm_xp128);
            uint32_t wt = 0, xt = 0, bt = 0;
            bool ok = true;
            for (int g = 0; g < n_groups && ok; ++g) {
                const PassInfo q = pass_info(pl, g);
                for (int kb = kb0; kb < kb1 && ok; ++kb) {
                    if (kb == kb0 || (kb & 1) == 0) {
                        // bits of every variant of the pass for the K-block pair kb & ~1
                        const int b = bt % kBitStages;
                        if (!(ok = mbar_wait_sleep(&bits_empty[b], ((bt / kBitStages) & 1) ^ 1, kWaitLimit, p.status, 8, p.diag))) break;
                        mbar_expect_tx(&bits_full[b], (q.d1 - q.d0) * kBitsTile);
                        uint8_t* sb = base + L.bits + b * L.bits_stage;
                        for (int d = q.d0; d < q.d1; ++d)
                            tma_load_2d(sb + (d - q.d0) * kBitsTile, &p.tm_bits[pl.var[d]], &bits_full[b],
                                        2 * (kb & ~1), n0);
                        ++bt;
                    }
                    if (g == 0) {
                        const int s = wt % kWStages;
                        if (!(ok = mbar_wait_sleep(&w_empty[s], ((wt / kWStages) & 1) ^ 1, kWaitLimit, p.status, 1, p.diag))) break;
                        mbar_expect_tx(&w_full[s], kWTile);
                        tma_load_2d(base + L.w + s * kWTile, &p.tm_w, &w_full[s], kb * kBK, n0);
                        ++wt;
                    }
                    const int s = xt % kXStages;
                    if (!(ok = mbar_wait_sleep(&x_empty[s], ((xt / kXStages) & 1) ^ 1, kWaitLimit, p.status, 10, p.diag))) break;
                    mbar_expect_tx(&x_full[s], q.rows * 128 + (g == 0 ? Mb * 128 : 0));
                    uint8_t* sx = base + L.x + s * L.x_stage;
                    if (g == 0) tma_load_2d(sx, &p.tm_xc, &x_full[s], kb * kBK, 0);
                    uint8_t* sxp = sx + L.xp_off;
                    int r = 0;
                    for (; r + 128 <= q.rows; r += 128)
                        tma_load_2d(sxp + r * 128, &p.tm_xp128, &x_full[s], kb * 128, q.row0 + r);
                    for (; r < q.rows; r += 16)
                        tma_load_2d(sxp + r * 128, &p.tm_xp, &x_full[s], kb * 128, q.row0 + r);
                    ++xt;
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- base-product issuer ----------------
        if (lane == 0) {
            uint32_t xt = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16(128, Mb);
            for (int g = 0; g < n_groups && ok; ++g) {
                for (int i = 0; i < nkb && ok; ++i, ++xt) {
                    const int s = xt % kXStages;
                    if (!(ok = mbar_wait_sleep(&x_full[s], (xt / kXStages) & 1, kWaitLimit, p.status, 2, p.diag))) break;
                    if (g == 0) {
                        const int ws = i % kWStages;
                        if (!(ok = mbar_wait_sleep(&w_full[ws], (i / kWStages) & 1, kWaitLimit, p.status, 11, p.diag))) break;
                        tc_fence_after();
                        const uint32_t sw = smem_u32(base + L.w + ws * kWTile);
                        const uint32_t sxc = smem_u32(base + L.x + s * L.x_stage);
#pragma unroll
                        for (int k16 = 0; k16 < 4; ++k16)
                            mma_ss(tmem + kBaseCol, desc_sw128(sw + 32 * k16), desc_sw128(sxc + 32 * k16), idesc,
                                   (i > 0 || k16 > 0) ? 1u : 0u);
                        mma_commit(&w_empty[ws]);
                    }
                    mma_commit(&x_empty[s]);
                }
                if (ok) mma_commit(&acc_full);
            }
        }
    } else if (warp < kFirstExpandWarp) {
        // ---------------- sign-product issuers ----------------
        if (lane == 0) {
            const int me = warp - kFirstIssuerWarp;
            uint32_t it = 0, u = 0;
            bool ok = true;
            for (int g = 0; g < n_groups && ok; ++g) {
                const PassInfo q = pass_info(pl, g);
                const int nd = q.d1 - q.d0;
                if (g > 0 && !(ok = mbar_wait_sleep(&acc_empty, (g - 1) & 1, kWaitLimit, p.status, 3, p.diag))) break;
                for (int i = 0; i < nkb && ok; ++i, ++it) {
                    const int s = it % kXStages;
                    if (!(ok = mbar_wait_sleep(&x_full[s], (it / kXStages) & 1, kWaitLimit, p.status, 4, p.diag))) break;
                    const uint32_t sxp = smem_u32(base + L.x + s * L.x_stage + L.xp_off);
                    for (int dl = me; dl < nd && ok; dl += kIssuers) {
                        const int d = q.d0 + dl;
                        const int segr = pl.seg[d] - q.row0;
                        const uint32_t dcol = kBaseCol + Mb + segr;
                        const uint32_t idesc = idesc_e4m3(128, pad16(pl.cnt[d]));
                        for (int h = 0; h < 2 && ok; ++h, ++u) {
                            if (!(ok = mbar_wait_sleep(&tm_full[me][h], (u >> 1) & 1, kWaitLimit, p.status, 5, p.diag))) break;
                            tc_fence_after();
                            const uint32_t a = tmem + me * 2 * kSlotCols + h * kSlotCols;
                            const uint32_t brow = sxp + segr * 128 + 32 * h;
                            mma_ts_f8(tmem + dcol, a, desc_sw128(brow), idesc, (i > 0 || h > 0) ? 1u : 0u);
                            mma_ts_f8(tmem + dcol, a, desc_sw128(brow + 64), idesc, 1u);
                            mma_commit(&tm_empty[me][h]);
                        }
                    }
                    mma_commit(&x_empty[s]);
                }
                if (ok) mma_commit(&acc_full);
            }
        }
    } else {
        // ---------------- expansion, then epilogue ----------------
        const int e = warp - kFirstExpandWarp;
        const int h = e / 4;                      // which 32-bit word of the 64-column block
        const int q4 = warp % 4;                  // TMEM lane quarter this warp may access
        const int r = 32 * q4 + lane;             // output row within the tile
        const int n = n0 + r;
        const bool row_ok = n < p.N;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q4) << 16;
        uint32_t ubase[kIssuers];                 // units given to each issuer in earlier passes
#pragma unroll
        for (int i = 0; i < kIssuers; ++i) ubase[i] = 0;
        uint32_t bt = 0;
        bool ok = true;
        for (int g = 0; g < n_groups && ok; ++g) {
            const PassInfo q = pass_info(pl, g);
            const int nd = q.d1 - q.d0;
            for (int i = 0; i < nkb && ok; ++i) {
                const int kb = kb0 + i;
                const int b = bt % kBitStages;
                if (i == 0 || (kb & 1) == 0) {
                    if (!(ok = mbar_wait_sleep(&bits_full[b], (bt / kBitStages) & 1, kWaitLimit, p.status, 9, p.diag))) break;
                }
                const uint32_t* sb = reinterpret_cast<const uint32_t*>(base + L.bits + b * L.bits_stage) +
                                     r * 4 + 2 * (kb & 1) + h;
                for (int dl = 0; dl < nd && ok; ++dl) {
                    const int iss = dl % kIssuers;
                    const uint32_t u = ubase[iss] + 2 * (i * issuer_count(nd, iss) + dl / kIssuers) + h;
                    const uint32_t w = sb[dl * (kBitsTile / 4)];
                    if (!(ok = mbar_wait_sleep(&tm_empty[iss][h], ((u >> 1) & 1) ^ 1, kWaitLimit, p.status, 6, p.diag))) break;
                    tc_fence_after();
                    uint32_t v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = ((w << (7 - j)) & 0x80808080u) ^ 0xB8B8B8B8u;
                    tmem_st8(tmem + lane_addr + iss * 2 * kSlotCols + h * kSlotCols, v);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tm_full[iss][h]);
                }
                if (i == nkb - 1 || (kb & 1) == 1) {        // done with this bits stage
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bits_empty[b]);
                    ++bt;
                }
            }
#pragma unroll
            for (int i = 0; i < kIssuers; ++i) ubase[i] += 2 * nkb * issuer_count(nd, i);
            if (!ok) break;
            // ---- epilogue of pass g ----
            if (!(ok = mbar_wait_sleep(&acc_full, g & 1, kWaitLimit, p.status, 7, p.diag))) break;
            tc_fence_after();
            if (g == 0) {
                for (int pos0 = 8 * h; pos0 < pl.n_base; pos0 += 16) {     // base-model tokens
                    uint32_t b[8];
                    tmem_ld8(tmem + lane_addr + kBaseCol + pos0, b);
                    tmem_ld_wait();
                    if (row_ok)
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            if (pos0 + t < pl.n_base) store_y(p, psm, split, tok_s[pos0 + t], n, r, __uint_as_float(b[t]));
                }
                if (row_ok && h == 0)                                          // invalid ids: zero rows
                    for (int pos = p.M - pl.n_invalid; pos < p.M; ++pos) store_y(p, psm, split, tok_s[pos], n, r, 0.f);
            }
            for (int d = q.d0; d < q.d1; ++d) {
                const int cnt = pl.cnt[d], off = pl.off[d];
                const float ar = (p.alpha_rows && row_ok) ? p.alphas[static_cast<int64_t>(pl.var[d]) * p.N + n] : 1.f;
                const uint32_t scol = kBaseCol + Mb + (pl.seg[d] - q.row0);
                for (int ci = h; 8 * ci < cnt; ci += 2) {
                    const int pos0 = off + 8 * ci;
                    uint32_t sg[8], bs[8];
                    tmem_ld8(tmem + lane_addr + scol + 8 * ci, sg);
#pragma unroll
                    for (int t = 0; t < 8; ++t) bs[t] = tmem_ld1(tmem + lane_addr + kBaseCol + pos0 + t);
                    tmem_ld_wait();
                    if (row_ok) {
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            if (8 * ci + t >= cnt) break;
                            store_y(p, psm, split, tok_s[pos0 + t], n, r,
                                    fmaf(ar * scale_s[pos0 + t], __uint_as_float(sg[t]), __uint_as_float(bs[t])));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty);
        }
    }

    __syncthreads();
    if (p.cluster_reduce) {
        // the K slices of this row tile are the CTAs of one cluster (rank =
        // split): CTA `split` sums its share of the tile over the slices'
        // shared memory in the order 0, 1, 2, ... and writes y
        cluster_sync_all();
        const int rows = min(kBN, p.N - n0);
        const uint32_t psm_a = smem_u32(psm);
        const int per_t = kBN / 4;                              // float4 groups per token
        const int total = p.M * per_t;
        const int g0 = static_cast<int>(static_cast<int64_t>(split) * total / p.splits);
        const int g1 = static_cast<int>(static_cast<int64_t>(split + 1) * total / p.splits);
        for (int gi = g0 + static_cast<int>(threadIdx.x); gi < g1; gi += blockDim.x) {
            const int t = gi / per_t, r4 = 4 * (gi % per_t);
            if (r4 >= rows) continue;
            const uint32_t off = psm_a + static_cast<uint32_t>(gi) * 16u;
            float4 acc = ld_cluster_f4(cluster_map(off, 0));
            for (int sl = 1; sl < p.splits; ++sl) {
                const float4 a = ld_cluster_f4(cluster_map(off, static_cast<uint32_t>(sl)));
                acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
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
        cluster_sync_all();            // no CTA leaves while its tile is being read
    } else if (p.splits > 1) {
        // deterministic split-K reduction by the CTA that finishes the tile last
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned t = atomicAdd(&p.tickets[tile], 1u);
            last_cta = (t == static_cast<unsigned>(p.splits - 1));
        }
        __syncthreads();
        if (last_cta) {
            __threadfence();
            const int rows = min(kBN, p.N - n0);
            if (rows == kBN && (p.N & 3) == 0) {
                // four outputs per thread, slices summed in order 0, 1, 2, ...
                // with four loads in flight
                const int nq = kBN / 4;
                const int64_t sq = static_cast<int64_t>(p.M) * p.N / 4;      // float4s per slice
                for (int idx = threadIdx.x; idx < p.M * nq; idx += blockDim.x) {
                    const int t = idx / nq, c4 = idx % nq;
                    const float4* src = reinterpret_cast<const float4*>(p.part + static_cast<int64_t>(t) * p.N + n0) + c4;
                    float4 acc = __ldcg(src);
                    int sl = 1;
                    for (; sl + 3 < p.splits; sl += 4) {
                        const float4 a0 = __ldcg(src + sl * sq), a1 = __ldcg(src + (sl + 1) * sq);
                        const float4 a2 = __ldcg(src + (sl + 2) * sq), a3 = __ldcg(src + (sl + 3) * sq);
                        acc.x = (((acc.x + a0.x) + a1.x) + a2.x) + a3.x;
                        acc.y = (((acc.y + a0.y) + a1.y) + a2.y) + a3.y;
                        acc.z = (((acc.z + a0.z) + a1.z) + a2.z) + a3.z;
                        acc.w = (((acc.w + a0.w) + a1.w) + a2.w) + a3.w;
                    }
                    for (; sl < p.splits; ++sl) {
                        const float4 a0 = __ldcg(src + sl * sq);
                        acc.x += a0.x; acc.y += a0.y; acc.z += a0.z; acc.w += a0.w;
                    }
                    const int64_t o = static_cast<int64_t>(t) * p.N + n0 + 4 * c4;
                    if (p.y_bf16) {
                        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
                        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.y) + o) =
                            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
                    } else {
                        *reinterpret_cast<float4*>(static_cast<float*>(p.y) + o) = acc;
                    }
                }
            } else {
                for (int idx = threadIdx.x; idx < p.M * rows; idx += blockDim.x) {
                    const int t = idx / rows, rr = idx % rows;
                    float acc = 0.f;
                    for (int s = 0; s < p.splits; ++s)
                        acc += __ldcg(p.part + (static_cast<int64_t>(s) * p.M + t) * p.N + n0 + rr);
                    const int64_t o = static_cast<int64_t>(t) * p.N + n0 + rr;
                    if (p.y_bf16) static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(acc);
                    else static_cast<float*>(p.y)[o] = acc;
                }
            }
            if (threadIdx.x == 0) p.tickets[tile] = 0u;
        }
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Staging for one linear (one block per staged row):
//   X_c [Mb, K] bf16: grouped order, zero rows past the valid tokens;
//   X_p [rows, 2K] bytes: each present variant's tokens in a 16-row
//       zero-padded segment; per 64-column block 64 bytes of hi then 64 of lo
//       (e4m3), byte 32w + 4j + b of a half holding column 32w + j + 8b, for
//       x * 2^sigma_t with sigma_t chosen so that max_k |x[t,k]| 2^sigma_t
//       lies in [128, 256) (0 for an all-zero row);
//   sigma[t] for every token with a sign segment; the split-K tickets zeroed.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3(float v) {
    return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(hr));
}

__global__ void __launch_bounds__(256) prep_kernel(const uint4* __restrict__ x, int K, int Mb,
                                                   const SegPlan* __restrict__ plan,
                                                   const int32_t* __restrict__ pos2tok, int32_t* __restrict__ sigma,
                                                   uint4* __restrict__ xc, uint4* __restrict__ xp,
                                                   unsigned* tickets, int n_tickets) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int rr = blockIdx.x;
    const int64_t vec_per_row = K / 8;
    if (rr == 0)
        for (int i = threadIdx.x; i < n_tickets; i += blockDim.x) tickets[i] = 0u;
    if (rr < Mb) {
        const int n_valid = plan->M - plan->n_invalid;
        const int tok = (rr < n_valid) ? pos2tok[rr] : -1;
        uint4* dst = xc + static_cast<int64_t>(rr) * vec_per_row;
        const uint4* src = x + static_cast<int64_t>(tok < 0 ? 0 : tok) * vec_per_row;
        for (int64_t i = threadIdx.x; i < vec_per_row; i += blockDim.x)
            dst[i] = tok >= 0 ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        return;
    }
    const int q = rr - Mb;
    if (q >= plan->P) return;                     // never loaded
    int tok = -1;
    {
        int d = 0;
        while (d + 1 < plan->D && plan->seg[d + 1] <= q) ++d;
        const int j = q - plan->seg[d];
        if (j < plan->cnt[d]) tok = pos2tok[plan->off[d] + j];
    }
    uint4* dst = xp + static_cast<int64_t>(q) * vec_per_row;
    if (tok < 0) {
        for (int64_t i = threadIdx.x; i < vec_per_row; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4* src = x + static_cast<int64_t>(tok) * vec_per_row;
    // sigma_t from the largest |x| of the row (bf16 bit patterns order like magnitudes)
    uint32_t mx = 0;
    for (int64_t i = threadIdx.x; i < vec_per_row; i += blockDim.x) {
        const uint4 v = __ldg(src + i);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) mx = max(mx, max(w4[k] & 0x7FFFu, (w4[k] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __shared__ uint32_t red[8];
    __shared__ int sig_s;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; ++i) mx = max(mx, red[i]);
        const int ex = static_cast<int>((mx >> 7) & 0xFF);      // biased exponent of the max
        int sg = 0;
        if (mx != 0 && ex != 0xFF) sg = 7 - (ex > 0 ? ex - 127 : -126);
        sg = max(-120, min(120, sg));
        sig_s = sg;
        sigma[tok] = sg;
    }
    __syncthreads();
    const float sc = exp2i(sig_s);
    for (int blk = threadIdx.x; blk < K / 64; blk += blockDim.x) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = __ldg(src + 8 * blk + i);
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) { hi[i] = 0; lo[i] = 0; }
#pragma unroll
        for (int c = 0; c < 64; ++c) {                     // source column c of the block
            const uint32_t bits16 = (c & 1) ? (w[c >> 1] >> 16) : (w[c >> 1] & 0xFFFFu);
            const float v = __uint_as_float(bits16 << 16) * sc;
            const uint32_t h8 = e4m3(v);
            const uint32_t l8 = e4m3(v - e4m3_to_f32(h8));
            const int wd = c >> 5, cc = c & 31;             // word, column within it
            const int jj = cc & 7, b = cc >> 3;             // register j, byte b
            const int byte = 32 * wd + 4 * jj + b;
            hi[byte >> 2] |= h8 << (8 * (byte & 3));
            lo[byte >> 2] |= l8 << (8 * (byte & 3));
        }
        uint4* o = dst + 8 * blk;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[i] = make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
            o[4 + i] = make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
        }
    }
}

int p_bound(int64_t M, int32_t V) {
    const int64_t d = V < M ? V : M;
    return pad16(static_cast<int>(M + 15 * d));
}

// K slices per row tile: minimise waves x (per-CTA fixed cost + K blocks per
// slice x time per K block), both in microseconds as measured on GB300 for a
// 128-token batch (the fixed cost covers set-up, pipeline fill, epilogue and
// the split-K reduction).
int choose_splits(int64_t n_tiles, int kb_total, int sms, int variants) {
    const double fixed_us = 6.0, kb_us = 0.3 + 0.07 * variants;
    int best = 1;
    double best_t = 1e30;
    for (int s = 1; s <= 64 && s <= kb_total; ++s) {
        const int64_t ctas = n_tiles * s;
        const int64_t waves = (ctas + sms - 1) / sms;
        const double t = static_cast<double>(waves) * (fixed_us + ((kb_total + s - 1) / s) * kb_us);
        if (t < best_t * 0.98) { best_t = t; best = s; }
    }
    return best;
}

struct DecodeScratch {
    uint16_t* xc;
    uint8_t* xp;
    int32_t* sigma;
    float* part;
    unsigned* tickets;
    size_t bytes;
};

DecodeScratch decode_scratch(void* base, int64_t M, int64_t N, int64_t K, int32_t V, int splits) {
    DecodeScratch d{};
    char* p = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* r = p ? p + off : nullptr;
        off += round_up(bytes, kAlign);
        return r;
    };
    const int Mb = pad16(static_cast<int>(M));
    d.xc = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(Mb) * K * 2));
    d.xp = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(p_bound(M, V)) * K * 2));
    d.sigma = reinterpret_cast<int32_t*>(take(static_cast<size_t>(M) * 4));
    const int64_t n_tiles = (N + kBN - 1) / kBN;
    d.part = splits > 1 ? reinterpret_cast<float*>(take(static_cast<size_t>(splits) * M * N * 4)) : nullptr;
    d.tickets = reinterpret_cast<unsigned*>(take(static_cast<size_t>(n_tiles) * 4));
    d.bytes = off;
    return d;
}

}  // namespace

int decode_group_budget(int64_t M) {
    const int b = kTmemCols - kBaseCol - pad16(static_cast<int>(M < 0 ? 0 : M));
    return b > 0 ? b : 0;
}

bool decode_tc_supported(const LinearArgs& a) {
    return a.M >= 1 && a.M <= kMaxM && a.K % kBK == 0 &&
           pad16(static_cast<int>(a.M)) <= decode_group_budget(a.M) && a.N >= 1 &&
           a.N < (int64_t(1) << 31);
}

size_t decode_tc_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V) {
    if (M < 1 || M > kMaxM || K % kBK != 0) return 0;
    const int64_t n_tiles = (N + kBN - 1) / kBN;
    const int splits = choose_splits(n_tiles, static_cast<int>(K / kBK), sm_count(), V < M ? V : static_cast<int>(M));
    return decode_scratch(nullptr, M, N, K, V, splits).bytes;
}

bd_status launch_decode_tc(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s) {
    const int M = static_cast<int>(a.M), N = static_cast<int>(a.N), K = static_cast<int>(a.K);
    const int Mb = pad16(M);
    const int budget = decode_group_budget(M);
    const int64_t n_tiles = (a.N + kBN - 1) / kBN;
    const int kb_total = K / kBK;
    const int splits = choose_splits(n_tiles, kb_total, sm_count(), a.V < M ? a.V : M);
    DecodeScratch sc = decode_scratch(w.tc_scratch, a.M, a.N, a.K, a.V, splits);
    if (sc.bytes > w.tc_bytes) return BD_ERR_WORKSPACE;
    const int prow = p_bound(a.M, a.V);

    prep_kernel<<<Mb + prow, 256, 0, s>>>(static_cast<const uint4*>(a.x), K, Mb, w.g.plan, w.g.pos2tok, sc.sigma,
                                          reinterpret_cast<uint4*>(sc.xc), reinterpret_cast<uint4*>(sc.xp),
                                          sc.tickets, splits > 1 ? static_cast<int>(n_tiles) : 0);
    if (launch_status() != BD_OK) return BD_ERR_CUDA;

    DecodeParams p;
    memset(&p, 0, sizeof p);
    if (!make_tmap_bf16_sw128(&p.tm_w, a.w_base, a.N, a.K, kBN) ||
        !make_tmap_bf16_sw128(&p.tm_xc, sc.xc, Mb, a.K, Mb) ||
        !make_tmap_u8_sw128(&p.tm_xp, sc.xp, prow, 2 * a.K, 16) ||
        !make_tmap_u8_sw128(&p.tm_xp128, sc.xp, prow, 2 * a.K, 128))
        return BD_ERR_CUDA;
    for (int v = 0; v < a.V; ++v)
        if (!make_tmap_bits(&p.tm_bits[v], a.bits.p[v], a.N, a.K / 32, kBN)) return BD_ERR_CUDA;
    p.alphas = a.alphas;
    p.alpha_rows = a.alpha_rows;
    p.plan = w.g.plan;
    p.pos2tok = w.g.pos2tok;
    p.sigma = sc.sigma;
    p.y = a.y;
    p.part = sc.part;
    p.tickets = sc.tickets;
    p.status = w.status;
    p.diag = w.status + 2;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Mb = Mb;
    p.budget = budget;
    p.splits = splits;
    p.y_bf16 = (a.y_dtype == BD_BF16);
    // the partial tile must fit the W ring: M <= 128 (128 x 128 f32 = 4 W tiles)
    p.cluster_reduce = (splits > 1 && splits <= 8 && M <= 128) ? 1 : 0;
    const SmemLayout L = smem_layout(Mb, budget);
    const int smem = static_cast<int>(L.total) + 1024;
    if (!set_smem_attr(reinterpret_cast<const void*>(decode_tc_kernel), smem, 0)) return BD_ERR_CUDA;
    // programmatic dependent launch: the kernel's set-up overlaps the staging
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_tiles * splits));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.cluster_reduce ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, decode_tc_kernel, p) != cudaSuccess) return BD_ERR_CUDA;
    return launch_status();
}

}  // namespace bd
