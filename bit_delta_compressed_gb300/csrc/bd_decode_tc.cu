// bd_decode_tc.cu -- tensor-core decode path of the fused multi-variant linear.
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": the base weights are read once and shared by every
// variant; each variant's delta arrives as packed sign bits and is expanded
// on chip, so W_eff = W_base + alpha_v * sign(delta_v) never exists in HBM.
//
// One CTA owns 128 output rows (the 128 lanes of tensor memory) and a slice
// of K (split-K; the slices of a row tile are summed in a fixed order by the
// CTA that finishes last).  Per 64-column K block:
//   * a TMA producer warp loads the W_base tile (128 x 64 bf16), the batch's
//     activations in grouped order (X_c, pad16(M) rows) and the activations
//     of this pass's variants in 16-row zero-padded segments with the K order
//     permuted inside every 32-column group (X_p);
//   * eight expansion warps turn each present variant's sign bits into a
//     +-1 bf16 tile straight in tensor memory: for a 32-bit word w of bits,
//     register j = ((w << (15 - j)) & 0x80008000) ^ 0xBF80BF80 holds columns j
//     and j + 16 (bit 1 -> +1.0, bit 0 -> -1.0), one shift and one LOP3 per
//     pair; X_p carries the same column order so the products line up;
//   * one thread issues the MMAs: D_base += W * X_c^T (A and B from shared
//     memory) and, per variant, D_sign[seg] += S_v * X_p[seg]^T (A from
//     tensor memory), both fp32 accumulators in tensor memory;
//   * the epilogue computes y = D_base + alpha_v * D_sign with the f32 alpha.
// Variants whose padded segments do not fit in tensor memory next to D_base
// are handled in further passes over the same K slice; those passes reload
// only X_p and bits, never W_base.
#include <mutex>

#include "bd_sm100.cuh"
#include "bd_tc_common.cuh"

namespace bd {

namespace {

constexpr int kBN = 128;                  // output rows per CTA (TMEM lanes)
constexpr int kBK = 64;                   // K per stage (one 128-byte swizzle atom)
constexpr int kStages = 2;
constexpr int kSlots = 3;                 // TMEM staging slots for the +-1 A tiles
constexpr int kSlotCols = 32;             // 64 bf16 per row = 32 TMEM columns
constexpr int kBaseCol = kSlots * kSlotCols;
constexpr int kTmemCols = 512;
constexpr int kBitRing = 3;               // K blocks of bits in flight per thread
constexpr int kMaxM = 208;               // pad16(M) must fit next to one variant's segment
constexpr int kThreads = 320;             // warp 0 TMA, warp 1 MMA, warps 2..9 expand/epilogue
constexpr int kExpandWarps = 8;
constexpr uint32_t kWaitLimit = 1u << 20;

struct DecodeParams {
    CUtensorMap tm_w;                     // W_base [N, K]
    CUtensorMap tm_xc;                    // X_c [Mb, K]
    CUtensorMap tm_xp;                    // X_p [P_bound, K]
    const uint32_t* bits[BITDELTA_MAX_VARIANTS];
    const float* alphas;
    const SegPlan* plan;
    const int32_t* pos2tok;
    void* y;
    float* part;                          // [splits][M][N] when splits > 1
    unsigned* tickets;                    // [n_tiles]
    unsigned* status;
    unsigned* diag;
    int M, N, K, Mb, budget, splits, y_bf16;
};

struct SmemLayout {
    uint32_t w, xc, xp, bits, total;
    int dmax;
};

__host__ __device__ inline SmemLayout smem_layout(int Mb, int budget) {
    SmemLayout L;
    const uint32_t w_bytes = kBN * 128, xc_bytes = Mb * 128, xp_bytes = budget * 128;
    L.w = 0;
    L.xc = L.w + kStages * w_bytes;
    L.xp = L.xc + kStages * xc_bytes;
    L.bits = L.xp + kStages * xp_bytes;
    L.dmax = budget / 16;
    L.total = L.bits + kBitRing * L.dmax * 2 * kBN * 4;
    return L;
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sm100::smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void store_y(const DecodeParams& p, int split, int t, int n, float v) {
    if (p.splits > 1) {
        p.part[(static_cast<int64_t>(split) * p.M + t) * p.N + n] = v;
    } else if (p.y_bf16) {
        static_cast<__nv_bfloat16*>(p.y)[static_cast<int64_t>(t) * p.N + n] = __float2bfloat16_rn(v);
    } else {
        static_cast<float*>(p.y)[static_cast<int64_t>(t) * p.N + n] = v;
    }
}

__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
    using namespace sm100;
    extern __shared__ uint8_t dsmem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_full[kStages], bar_empty[kStages], tm_full[kSlots], tm_empty[kSlots];
    __shared__ uint64_t acc_full, acc_empty;
    __shared__ uint32_t tmem_base;
    __shared__ SegPlan pl;
    __shared__ int last_cta;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Mb = p.Mb;
    const SmemLayout L = smem_layout(Mb, p.budget);
    const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
    const int n0 = tile * kBN;
    const int kb_total = p.K / kBK;
    const int kb0 = static_cast<int>(static_cast<int64_t>(split) * kb_total / p.splits);
    const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * kb_total / p.splits);
    const int nkb = kb1 - kb0;

    {   // copy the segment plan into shared memory
        const int* src = reinterpret_cast<const int*>(p.plan);
        int* dst = reinterpret_cast<int*>(&pl);
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(SegPlan) / 4); i += blockDim.x) dst[i] = src[i];
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&bar_full[s], 1); mbar_init(&bar_empty[s], 1); }
        for (int j = 0; j < kSlots; ++j) { mbar_init(&tm_full[j], kExpandWarps); mbar_init(&tm_empty[j], 1); }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, kExpandWarps);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kTmemCols);
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
            uint32_t it = 0;
            bool ok = true;
            for (int g = 0; g < n_groups && ok; ++g) {
                const int d0 = pl.group_first[g], d1 = pl.group_first[g + 1];
                const int row0 = (d1 > d0) ? pl.seg[d0] : 0;
                const int rows = (d1 > d0) ? pl.seg[d1 - 1] + pad16(pl.cnt[d1 - 1]) - row0 : 0;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!(ok = mbar_wait(&bar_empty[s], ((it / kStages) & 1) ^ 1, kWaitLimit, p.status, 1, p.diag))) break;
                    const uint32_t bytes = rows * 128 + (g == 0 ? kBN * 128 + Mb * 128 : 0);
                    mbar_expect_tx(&bar_full[s], bytes);
                    const int kc = kb * kBK;
                    uint8_t* sw = base + L.w + s * (kBN * 128);
                    uint8_t* sxc = base + L.xc + s * (Mb * 128);
                    uint8_t* sxp = base + L.xp + s * (p.budget * 128);
                    if (g == 0) {
                        tma_load_2d(sw, &p.tm_w, &bar_full[s], kc, n0);
                        for (int r = 0; r < Mb; r += 16) tma_load_2d(sxc + r * 128, &p.tm_xc, &bar_full[s], kc, r);
                    }
                    for (int r = 0; r < rows; r += 16) tma_load_2d(sxp + r * 128, &p.tm_xp, &bar_full[s], kc, row0 + r);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            uint32_t it = 0, c = 0;
            bool ok = true;
            const uint32_t idesc_base = idesc_bf16(128, Mb);
            for (int g = 0; g < n_groups && ok; ++g) {
                const int d0 = pl.group_first[g], d1 = pl.group_first[g + 1];
                const int row0 = (d1 > d0) ? pl.seg[d0] : 0;
                if (g > 0 && !(ok = mbar_wait(&acc_empty, (g - 1) & 1, kWaitLimit, p.status, 2, p.diag))) break;
                for (int i = 0; i < nkb && ok; ++i, ++it) {
                    const int s = it % kStages;
                    if (!(ok = mbar_wait(&bar_full[s], (it / kStages) & 1, kWaitLimit, p.status, 3, p.diag))) break;
                    tc_fence_after();
                    const uint32_t sw = smem_u32(base + L.w + s * (kBN * 128));
                    const uint32_t sxc = smem_u32(base + L.xc + s * (Mb * 128));
                    const uint32_t sxp = smem_u32(base + L.xp + s * (p.budget * 128));
                    if (g == 0) {
#pragma unroll
                        for (int k16 = 0; k16 < 4; ++k16)
                            mma_ss(tmem + kBaseCol, desc_sw128(sw + 32 * k16), desc_sw128(sxc + 32 * k16),
                                   idesc_base, (i > 0 || k16 > 0) ? 1u : 0u);
                    }
                    for (int d = d0; d < d1 && ok; ++d, ++c) {
                        const int j = c % kSlots;
                        if (!(ok = mbar_wait(&tm_full[j], (c / kSlots) & 1, kWaitLimit, p.status, 4, p.diag))) break;
                        tc_fence_after();
                        const int segr = pl.seg[d] - row0;
                        const uint32_t dcol = kBaseCol + Mb + segr;
                        const uint32_t idesc = idesc_bf16(128, pad16(pl.cnt[d]));
#pragma unroll
                        for (int k16 = 0; k16 < 4; ++k16)
                            mma_ts(tmem + dcol, tmem + j * kSlotCols + 8 * k16,
                                   desc_sw128(sxp + segr * 128 + 32 * k16), idesc,
                                   (i > 0 || k16 > 0) ? 1u : 0u);
                        mma_commit(&tm_empty[j]);
                    }
                    mma_commit(&bar_empty[s]);
                }
                if (ok) mma_commit(&acc_full);
            }
        }
    } else {
        // ---------------- expansion, then epilogue ----------------
        const int e = warp - 2;
        const int h = e / 4;                      // which 32-bit word of the 64-column block
        const int q = warp % 4;                   // TMEM lane quarter this warp may access
        const int r = 32 * q + lane;              // output row within the tile
        const int n = n0 + r;
        const bool row_ok = n < p.N;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        const int words_per_row = p.K / 32;
        uint32_t* ring = reinterpret_cast<uint32_t*>(base + L.bits);
        uint32_t c = 0;
        bool ok = true;
        for (int g = 0; g < n_groups && ok; ++g) {
            const int d0 = pl.group_first[g], d1 = pl.group_first[g + 1];
            const int nd = d1 - d0;
            const int row0 = (d1 > d0) ? pl.seg[d0] : 0;
            auto issue = [&](int i) {
                if (i < nkb && row_ok) {
                    const int slot = i % kBitRing;
                    for (int d = d0; d < d1; ++d) {
                        const uint32_t* src = p.bits[pl.var[d]] + static_cast<int64_t>(n) * words_per_row +
                                              2 * (kb0 + i) + h;
                        cp_async4(ring + ((slot * L.dmax + (d - d0)) * 2 + h) * kBN + r, src);
                    }
                }
                cp_async_commit();
            };
            for (int i = 0; i < kBitRing - 1; ++i) issue(i);
            for (int i = 0; i < nkb && ok; ++i) {
                issue(i + kBitRing - 1);
                cp_async_wait<kBitRing - 1>();
                const int slot = i % kBitRing;
                for (int d = d0; d < d1 && ok; ++d, ++c) {
                    const uint32_t w = row_ok ? ring[((slot * L.dmax + (d - d0)) * 2 + h) * kBN + r] : 0u;
                    const int j = c % kSlots;
                    if (!(ok = mbar_wait(&tm_empty[j], ((c / kSlots) & 1) ^ 1, kWaitLimit, p.status, 5, p.diag))) break;
                    tc_fence_after();
                    uint32_t v[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) v[jj] = ((w << (15 - jj)) & 0x80008000u) ^ 0xBF80BF80u;
                    tmem_st16(tmem + lane_addr + j * kSlotCols + 16 * h, v);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tm_full[j]);
                }
            }
            cp_async_wait<0>();
            (void)nd;
            if (!ok) break;
            // ---- epilogue of pass g ----
            if (!(ok = mbar_wait(&acc_full, g & 1, kWaitLimit, p.status, 6, p.diag))) break;
            tc_fence_after();
            if (g == 0) {
                // base-model tokens: y = D_base
                for (int pos0 = 16 * h; pos0 < pl.n_base; pos0 += 32) {
                    uint32_t b[16];
                    tmem_ld16(tmem + lane_addr + kBaseCol + pos0, b);
                    tmem_ld_wait();
                    if (row_ok)
                        for (int t = 0; t < 16 && pos0 + t < pl.n_base; ++t)
                            store_y(p, split, p.pos2tok[pos0 + t], n, __uint_as_float(b[t]));
                }
                // invalid ids: zero rows
                if (row_ok && h == 0)
                    for (int pos = p.M - pl.n_invalid; pos < p.M; ++pos) store_y(p, split, p.pos2tok[pos], n, 0.f);
            }
            for (int d = d0; d < d1; ++d) {
                const int cnt = pl.cnt[d], off = pl.off[d];
                const float alpha = p.alphas[pl.var[d]];
                const uint32_t scol = kBaseCol + Mb + (pl.seg[d] - row0);
                for (int ci = h; 16 * ci < cnt; ci += 2) {
                    const int pos0 = off + 16 * ci;
                    const int a0 = pos0 & ~15;          // aligned base chunk(s) covering pos0..pos0+15
                    uint32_t b0[16], b1[16], sg[16];
                    tmem_ld16(tmem + lane_addr + kBaseCol + a0, b0);
                    tmem_ld16(tmem + lane_addr + kBaseCol + a0 + 16, b1);
                    tmem_ld16(tmem + lane_addr + scol + 16 * ci, sg);
                    tmem_ld_wait();
                    if (row_ok) {
                        const int sh = pos0 - a0;
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            if (16 * ci + t >= cnt) break;
                            const int k = sh + t;
                            const float bv = __uint_as_float(k < 16 ? b0[k & 15] : b1[k & 15]);
                            store_y(p, split, p.pos2tok[pos0 + t], n, fmaf(alpha, __uint_as_float(sg[t]), bv));
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
    if (p.splits > 1) {
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
            for (int idx = threadIdx.x; idx < p.M * rows; idx += blockDim.x) {
                const int t = idx / rows, r = idx % rows;
                float acc = 0.f;
                for (int s = 0; s < p.splits; ++s)
                    acc += __ldcg(p.part + (static_cast<int64_t>(s) * p.M + t) * p.N + n0 + r);
                const int64_t o = static_cast<int64_t>(t) * p.N + n0 + r;
                if (p.y_bf16) static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(acc);
                else static_cast<float*>(p.y)[o] = acc;
            }
            if (threadIdx.x == 0) p.tickets[tile] = 0u;
        }
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Activation staging for one linear: X_c (grouped order, pad16(M) rows) and
// X_p (each present variant's tokens in a 16-row zero-padded segment, K
// permuted inside every 32-column group: output column 2j + h of the group
// holds input column j + 16h).  One thread per 32-column group of one row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) stage_x_kernel(const uint4* __restrict__ x, int M, int K, int Mb,
                                                      const SegPlan* __restrict__ plan,
                                                      const int32_t* __restrict__ pos2tok,
                                                      uint4* __restrict__ xc, uint4* __restrict__ xp,
                                                      int p_rows) {
    const int rr = blockIdx.y;
    const int grp = blockIdx.x * blockDim.x + threadIdx.x;      // 32-column group
    if (grp >= K / 32) return;
    const int64_t vec_per_row = K / 8;
    int tok = -1;
    bool perm = false;
    uint4* dst;
    if (rr < Mb) {
        const int n_valid = plan->M - plan->n_invalid;
        tok = (rr < n_valid) ? pos2tok[rr] : -1;
        dst = xc + static_cast<int64_t>(rr) * vec_per_row + 4 * grp;
    } else {
        const int q = rr - Mb;
        if (q >= p_rows) return;
        perm = true;
        dst = xp + static_cast<int64_t>(q) * vec_per_row + 4 * grp;
        if (q < plan->P) {
            int d = 0;
            while (d + 1 < plan->D && plan->seg[d + 1] <= q) ++d;
            const int j = q - plan->seg[d];
            if (j < plan->cnt[d]) tok = pos2tok[plan->off[d] + j];
        }
    }
    uint4 in[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (tok >= 0) {
        const uint4* src = x + static_cast<int64_t>(tok) * vec_per_row + 4 * grp;
#pragma unroll
        for (int i = 0; i < 4; ++i) in[i] = __ldg(src + i);
    }
    if (!perm) {
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = in[i];
        return;
    }
    const uint32_t w[16] = {in[0].x, in[0].y, in[0].z, in[0].w, in[1].x, in[1].y, in[1].z, in[1].w,
                            in[2].x, in[2].y, in[2].z, in[2].w, in[3].x, in[3].y, in[3].z, in[3].w};
    uint32_t o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)   // element j (low) and element j + 16 (high)
        o[j] = __byte_perm(w[j >> 1], w[8 + (j >> 1)], (j & 1) ? 0x7632 : 0x5410);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

int p_bound(int64_t M, int32_t V) {
    const int64_t d = V < M ? V : M;
    return pad16(static_cast<int>(M + 15 * d));
}

int choose_splits(int64_t n_tiles, int kb_total, int sms) {
    int best = 1;
    double best_eff = 0.0;
    for (int s = 1; s <= 64 && kb_total / s >= 4; ++s) {
        const int64_t ctas = n_tiles * s;
        const int64_t waves = (ctas + sms - 1) / sms;
        const double eff = static_cast<double>(ctas) / static_cast<double>(waves * sms);
        if (eff > best_eff + 0.02) { best_eff = eff; best = s; }
    }
    return best;
}

struct DecodeScratch {
    uint16_t* xc;
    uint16_t* xp;
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
    d.xp = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(p_bound(M, V)) * K * 2));
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
    const int splits = choose_splits(n_tiles, static_cast<int>(K / kBK), sm_count());
    return decode_scratch(nullptr, M, N, K, V, splits).bytes;
}

bd_status launch_decode_tc(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s) {
    const int M = static_cast<int>(a.M), N = static_cast<int>(a.N), K = static_cast<int>(a.K);
    const int Mb = pad16(M);
    const int budget = decode_group_budget(M);
    const int64_t n_tiles = (a.N + kBN - 1) / kBN;
    const int kb_total = K / kBK;
    const int splits = choose_splits(n_tiles, kb_total, sm_count());
    DecodeScratch sc = decode_scratch(w.tc_scratch, a.M, a.N, a.K, a.V, splits);
    if (sc.bytes > w.tc_bytes) return BD_ERR_WORKSPACE;
    const int prow = p_bound(a.M, a.V);

    dim3 sg((K / 32 + 255) / 256, Mb + prow);
    stage_x_kernel<<<sg, 256, 0, s>>>(static_cast<const uint4*>(a.x), M, K, Mb, w.g.plan, w.g.pos2tok,
                                      reinterpret_cast<uint4*>(sc.xc), reinterpret_cast<uint4*>(sc.xp), prow);
    if (launch_status() != BD_OK) return BD_ERR_CUDA;
    if (splits > 1 && cudaMemsetAsync(sc.tickets, 0, n_tiles * 4, s) != cudaSuccess) return BD_ERR_CUDA;

    DecodeParams p;
    memset(&p, 0, sizeof p);
    if (!make_tmap_bf16_sw128(&p.tm_w, a.w_base, a.N, a.K, kBN) ||
        !make_tmap_bf16_sw128(&p.tm_xc, sc.xc, Mb, a.K, 16) ||
        !make_tmap_bf16_sw128(&p.tm_xp, sc.xp, prow, a.K, 16))
        return BD_ERR_CUDA;
    for (int v = 0; v < a.V; ++v) p.bits[v] = reinterpret_cast<const uint32_t*>(a.bits.p[v]);
    p.alphas = a.alphas;
    p.plan = w.g.plan;
    p.pos2tok = w.g.pos2tok;
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
    const SmemLayout L = smem_layout(Mb, budget);
    const int smem = static_cast<int>(L.total) + 1024;
    if (!set_smem_attr(reinterpret_cast<const void*>(decode_tc_kernel), smem, 0)) return BD_ERR_CUDA;
    decode_tc_kernel<<<static_cast<unsigned>(n_tiles * splits), kThreads, smem, s>>>(p);
    return launch_status();
}

// ---------------------------------------------------------------------------
// host helpers shared with the prefill path
// ---------------------------------------------------------------------------
namespace {
std::mutex g_tc_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_smem_set[64][4] = {};
}  // namespace

bool make_tmap_bf16_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows) {
    {
        std::lock_guard<std::mutex> lock(g_tc_mutex);
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                 &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return false;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool set_smem_attr(const void* kernel, int bytes, int slot) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(g_tc_mutex);
    if (g_smem_set[dev][slot] >= bytes) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    g_smem_set[dev][slot] = bytes;
    return true;
}

}  // namespace bd
