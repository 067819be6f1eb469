// bd_decode_fold.cu -- folded tensor-core decode path of the fused
// multi-variant linear.
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": the base weights are read once and shared by every
// variant, each variant's delta arrives as packed sign bits and is expanded
// on chip, and W_eff = W_base + alpha_v * sign(delta_v) never exists in HBM.
//
// Per output row n and token t (grouped order) the kernel accumulates, in
// tensor memory,
//   B[n, t] = sum_k W[n,k] (x[t,k] 2^s_t)          (base accumulator)
//   S[n, t] = sum_k s_v[n,k] (x[t,k] 2^s_t)        (sign accumulator, v = v(t))
//   y[t, n] = 2^-s_t (B[n, t] + alpha_v S[n, t])
// where 2^s_t is a per-token power of two (exact) that puts the token's
// largest |x[t,k]| 2^s_t in [128, 256), and alpha_v is the variant's scale
// (one per matrix, or one per output row n).  The base operand is the bf16
// activation row scaled by 2^s_t (exact); the sign operand is x 2^s_t written
// as the sum of two e4m3 terms hi = rn(v), lo = rn(v - hi), which keeps about
// 8 significant bits of every element (the same order as the bf16
// activations themselves).  Each accumulator column belongs to one token and
// so to one variant: the sign accumulator is shared by all variants, tensor
// memory holds 2 x 128 accumulator columns and the rest is free for +-1
// tiles, and the scale is applied per column (and row) in the epilogue.
//
// One CTA owns 128 output rows (the 128 lanes of tensor memory) and a slice
// of K (split-K at even 64-column blocks; the slices of a row tile are summed
// in a fixed order, over the shared memory of a thread-block cluster of up to
// 16 CTAs, or from HBM partials by the CTA that finishes the tile last).
// Warps:
//   * 0, 1, 2 (producers, each with a ring of its own): W_base tiles
//     (128 x 64 bf16, 128-byte swizzle) from HBM by TMA; per 64-column block
//     the scaled activations X_c (pad16(M) rows) and the sign operand X_p (R
//     rows) from L2 in one bulk copy of a pre-swizzled stage image; per pair
//     of blocks one 128-row x 4-word tile of packed bits per present variant
//     from HBM by TMA;
//   * 3, the base issuer: per block four bf16 MMAs (N = pad16(M)) of the W
//     tile with X_c; the only consumer of the W ring;
//   * four issuer groups of five warps.  An entry is one present variant
//     (its run of grouped positions, the 16-token chunks it touches and its
//     rows of X_p; variant runs that share a chunk are separated by zero rows
//     in X_p); entry e belongs to group e % 4, so the groups' loads differ by
//     one entry at most.  A group's four expansion warps (one per
//     tensor-memory lane quarter) turn the bits of its entries into e4m3 +-1
//     tiles in tensor memory (two buffers) -- one shift and one LOP3 per four
//     weights: register j = ((w << (7 - j)) & 0x80808080) ^ 0xB8B8B8B8 holds
//     columns j, j+8, j+16, j+24 of a 32-bit word -- and arrive on a named
//     barrier; its issuer warp then issues, per 32-column K step, two e4m3
//     sign products (hi, lo) per entry: issue and hand-off latencies, not
//     the tensor core, bound a step (with single-lane issue one issuer warp
//     per group beats two: fewer warps contend for the schedulers and for
//     tensor memory).  Entries of different groups may add into the same accumulator
//     columns (each MMA's accumulation is atomic in the tensor pipe), so all
//     sign columns are zeroed before the first sign product; at the end each
//     group's expansion warps read a quarter of the columns of both
//     accumulators and write y.
// The columns inside each 32-column group of X_p are permuted to match the
// register layout above.  One elected lane of an issuer warp issues all of
// its MMAs and commits of a step in a row (an elect per MMA by the whole warp
// costs ~6% of the kernel's time, and a plain lane-0 branch far more).
// Waiting warps poll with one lane that suspends in mbarrier.try_wait, and
// the sign bits come by TMA: per-thread global loads or polling by whole
// warps slow the tensor-core issue of the whole SM.
#include <cuda_fp8.h>

#include "bd_sm100.cuh"
#include "bd_tc_common.cuh"

namespace bd {

namespace {

constexpr int kBN = 128;                        // output rows per CTA
constexpr int kBK = 64;                         // K per block
constexpr int kWMax = 4;                        // W_base ring stages (runtime: 3 or 4)
constexpr int kXMax = 2;                        // activation ring stages (runtime: 1 or 2)
constexpr int kBStages = 2;                     // bits ring stages, two 64-column blocks each
constexpr int kIss = kFoldIssuers;             // issuer groups
constexpr int kGroupIss = 1;                    // issuer warps per group (entries dealt in turn)
constexpr int kGroupWarps = 4 + kGroupIss;      // 4 expansion warps (one per lane quarter) + the issuers
constexpr int kBaseWarp = 3;                    // the base-product issuer
constexpr int kFirstGroup = 4;                  // warps 0, 1, 2: W, activation and bits producers
constexpr int kThreads = 32 * (kFirstGroup + kIss * kGroupWarps);
constexpr int kABufs = 2;                       // +-1 tile buffers per group
constexpr int kRegEntries = 6;                  // entries whose MMA operands an issuer keeps in registers
constexpr int kSCol0 = kFoldMaxCols;            // sign accumulator after the base accumulator
constexpr int kACol0 = 2 * kFoldMaxCols;        // +-1 tiles after both accumulators
constexpr int kAEntries = (512 - kACol0) / (8 * kABufs);   // entries whose tiles fit
constexpr int kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kWTile = kBN * 128;
static_assert(kAEntries >= kFoldSepEntries, "tensor memory budget");

struct FoldParams {
    CUtensorMap tm_w;                           // W_base [N, K] bf16, box 128 rows
    CUtensorMap tm_bits[BITDELTA_MAX_VARIANTS];  // packed bits [N, K/32] u32, box 128 rows x 4 words
    const SegPlan* plan;
    const FoldPlan* fold;
    const int32_t* pos2tok;
    const int32_t* pos_var;                     // grouped position -> variant (-1 base, -2 invalid)
    const float* alphas;                        // [V], or [V, N] when alpha_rows
    int alpha_rows;
    const int32_t* sexp;                        // [Mb] scale exponent s per grouped position
    void* y;
    float* part;                                // [splits][M][N] by grouped position
    unsigned* tickets;
    unsigned* status;
    unsigned* diag;
    const uint8_t* ximg;                        // per 64-column block, the stage image of X_c and X_p
    int M, N, K, Mb, Rmax, splits, y_bf16;
    int cluster_reduce;                         // the K slices of a row tile form one cluster (2..16 slices)
    int wstages, xstages, bslots;               // ring depths; variants per bits stage
};

__device__ __forceinline__ float pow2i(int e) {        // exact 2^e, e in [-126, 127]
    return __int_as_float((127 + e) << 23);
}

// Output (grouped position pos, row n = n0 + r) of this CTA: its partial
// tile in shared memory (cluster reduction), its K slice's partial in HBM
// (ticket reduction), or y itself (one slice).
__device__ __forceinline__ void store_out(const FoldParams& p, float* psm, int split, int pos, int tok, int n, int r,
                                          float v) {
    if (p.cluster_reduce) {
        psm[pos * kBN + r] = v;
    } else if (p.splits > 1) {
        p.part[(static_cast<int64_t>(split) * p.M + pos) * p.N + n] = v;
    } else if (p.y_bf16) {
        static_cast<__nv_bfloat16*>(p.y)[static_cast<int64_t>(tok) * p.N + n] = __float2bfloat16_rn(v);
    } else {
        static_cast<float*>(p.y)[static_cast<int64_t>(tok) * p.N + n] = v;
    }
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
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
constexpr int kGroupThreads = 32 * kGroupWarps;
// Named barrier of group g's +-1 tile buffer b (barrier 0 is __syncthreads).
__device__ __forceinline__ int group_bar(int g, int b) { return 1 + kABufs * g + b; }

// The base issuer: per 64-column block, the bf16 product of the W tile with
// all pad16(M) scaled activation rows into the base accumulator (one MMA per
// 16 columns of K, N = pad16(M)), then release the W and activation stages.
__device__ void base_issue(const FoldParams& p, uint32_t tmem, int nkb, uint8_t* wring, uint8_t* xring,
                           uint32_t xs_bytes, uint64_t* w_full, uint64_t* w_empty, uint64_t* x_full,
                           uint64_t* x_empty, uint64_t* acc_full, uint64_t* drain) {
    using namespace sm100;
    const uint32_t idb = idesc_bf16(128, p.Mb);
    bool ok = true;
    for (int i = 0; i < nkb && ok; ++i) {
        const int ws = i % p.wstages, xs = i % p.xstages;
        ok = warp_wait(&x_full[xs], (i / p.xstages) & 1, kWaitLimit, p.status, 26, p.diag);
        if (ok) ok = warp_wait(&w_full[ws], (i / p.wstages) & 1, kWaitLimit, p.status, 27, p.diag);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
            const uint32_t sw = smem_u32(wring + ws * kWTile);
            const uint32_t sx = smem_u32(xring + xs * xs_bytes);
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16)
                mma_ss(tmem, desc_sw128(sw + 32 * k16), desc_sw128(sx + 32 * k16), idb, (i > 0 || k16 > 0) ? 1u : 0u);
            mma_commit(&w_empty[ws]);
            mma_commit(&x_empty[xs]);
        }
        __syncwarp();
    }
    __syncwarp();
    if (elect_one()) {
        if (ok) mma_commit(acc_full);
        mma_commit(drain);                   // completes when every MMA of this warp has
    }
}

// The sign issuer warp of a group: per 32-column K step j of block i, wait
// for the group's tiles (named barrier), then issue the hi/lo sign products
// of its entries into the sign accumulator (zeroed by the expansion warps
// before the first step).  Every barrier is visited on every step, also
// after an error, so the group never blocks.
__device__ void group_issue(const FoldParams& p, const FoldPlan& fp, uint32_t tmem, uint32_t abase, int e0,
                            int ne, int g, int iss, int nkb, uint8_t* xring, uint32_t xs_bytes, uint64_t* x_full,
                            uint64_t* x_empty, uint64_t* ge, uint64_t* zeroed, uint64_t* acc_full, uint64_t* drain) {
    using namespace sm100;
    const int lane = threadIdx.x & 31;
    // The group's entries are e0 + kIss l, l = 0 .. ne - 1 (tile of entry l at
    // 8 l columns inside the group's buffer of ne tiles); this issuer takes
    // l = iss, iss + kGroupIss, ...
    const int own = ne > iss ? (ne - iss + kGroupIss - 1) / kGroupIss : 0;
    const bool work = own > 0;
    const int Mb = p.Mb;
    // Operands of up to kRegEntries entries live in registers: the D column,
    // the low word of the B descriptor at stage 0 and step 0 (the stage and
    // step add 16-byte units to the start-address field; every address stays
    // below 256 KB, so the field never carries), and the instruction descriptor.
    const bool in_regs = own <= kRegEntries;
    uint32_t r_d[kRegEntries], r_a[kRegEntries], r_b[kRegEntries], r_id[kRegEntries];
    const uint64_t xdesc = desc_sw128(smem_u32(xring));
    const uint32_t xdesc_lo = static_cast<uint32_t>(xdesc), xdesc_hi = static_cast<uint32_t>(xdesc >> 32);
#pragma unroll
    for (int k = 0; k < kRegEntries; ++k) {
        const int l = k < own ? iss + kGroupIss * k : 0;
        const int e = e0 + kIss * l;
        r_d[k] = tmem + kSCol0 + fp.e_col[e];
        r_a[k] = static_cast<uint32_t>(8 * l);
        r_b[k] = xdesc_lo + static_cast<uint32_t>(Mb + fp.e_row[e]) * 8u;
        r_id[k] = idesc_e4m3(128, fp.e_n[e]);
    }
    // entries of every group may share accumulator columns: all of them are
    // zeroed before the first sign product
    bool ok = warp_wait(zeroed, 0, kWaitLimit, p.status, 34, p.diag);
    for (int i = 0; i < nkb; ++i) {
        const int xs = i % p.xstages;
        for (int j = 0; j < 2; ++j) {
            named_sync(group_bar(g, j), kGroupThreads);
            // every group, also one without entries, waits for the stage it
            // releases: an early arrival would count towards a later phase
            if (ok && j == 0) ok = warp_wait(&x_full[xs], (i / p.xstages) & 1, kWaitLimit, p.status, 26, p.diag);
            if (!ok) continue;
            if (work && in_regs) {
                tc_fence_after();
                const uint32_t abuf = abase + j * 8 * ne;
                const uint32_t soff = (static_cast<uint32_t>(xs) * xs_bytes >> 4) + 2u * j;
                if (elect_one()) {
#pragma unroll
                    for (int k = 0; k < kRegEntries; ++k)
                        if (k < own) {
                            const uint32_t blo = r_b[k] + soff;
                            mma_ts_f8(r_d[k], abuf + r_a[k], (static_cast<uint64_t>(xdesc_hi) << 32) | blo, r_id[k], 1u);
                            mma_ts_f8(r_d[k], abuf + r_a[k], (static_cast<uint64_t>(xdesc_hi) << 32) | (blo + 4u), r_id[k], 1u);
                        }
                    mma_commit(&ge[j]);
                    if (j == 1) mma_commit(&x_empty[xs]);
                }
                __syncwarp();
            } else if (work) {
                tc_fence_after();
                const uint32_t sxp = smem_u32(xring + xs * xs_bytes) + Mb * 128;
                const uint32_t abuf = abase + j * 8 * ne;
                if (elect_one()) {
                    for (int l = iss; l < ne; l += kGroupIss) {
                        const int e = e0 + kIss * l;
                        const uint32_t d = tmem + kSCol0 + fp.e_col[e];
                        const uint32_t a = abuf + 8 * l;
                        const uint32_t brow = sxp + fp.e_row[e] * 128 + 32 * j;
                        const uint32_t id8 = idesc_e4m3(128, fp.e_n[e]);
                        mma_ts_f8(d, a, desc_sw128(brow), id8, 1u);
                        mma_ts_f8(d, a, desc_sw128(brow + 64), id8, 1u);
                    }
                    mma_commit(&ge[j]);
                    if (j == 1) mma_commit(&x_empty[xs]);
                }
                __syncwarp();
            } else {
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ge[j]);
                    if (j == 1) mbar_arrive(&x_empty[xs]);
                }
            }
        }
    }
    __syncwarp();
    if (work) {
        if (elect_one()) {
            if (ok) mma_commit(acc_full);
            mma_commit(drain);
        }
    } else if (lane == 0) {
        if (ok) mbar_arrive(acc_full);
        mbar_arrive(drain);
    }
}

// +-1 tile of one 32-column word of sign bits, e4m3: register j holds
// columns j, j+8, j+16, j+24 (bit 1 -> 0x38 = +1.0, bit 0 -> 0xB8 = -1.0).
__device__ __forceinline__ void store_signs(uint32_t taddr, uint32_t w) {
    uint32_t v[8];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) v[jj] = ((w << (7 - jj)) & 0x80808080u) ^ 0xB8B8B8B8u;
    sm100::tmem_st8(taddr, v);
}

// An expansion warp of a group (lane quarter q4): per 32-column K step, wait
// until the buffer's previous MMAs are done, write the group's +-1 tiles for
// its 32 rows from the bits tiles that TMA put in shared memory (128 rows x 4
// words per present variant, two 64-column blocks per stage), and arrive on
// the group's named barrier; at the end read the group's accumulator columns
// and write y = 2^-s_t D.
__device__ void group_expand(const FoldParams& p, const FoldPlan& fp, uint32_t tmem,
                             uint32_t abase, int e0, int ne, int g, int q4, int n0, int nkb, uint64_t* ge,
                             const uint8_t* bring, uint32_t bstage_bytes, uint64_t* b_full, uint64_t* b_empty,
                             uint64_t* zeroed, uint64_t* acc_full, const int32_t* tok_s, const float* scale_s, const int32_t* var_s,
                             const float* alpha_s, int split, int bcol, int bn, float* psm) {
    using namespace sm100;
    const int lane = threadIdx.x & 31;
    const int r = 32 * q4 + lane;
    const int n = n0 + r;
    const bool row_ok = n < p.N;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q4) << 16;
    {
        // the sign products all accumulate: start the group's columns at zero
        uint32_t z[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) z[jj] = 0u;
        for (int c = bcol; c < bcol + bn; c += 8) tmem_st8(tmem + lane_addr + kSCol0 + c, z);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(zeroed);
    }
    bool ok = true;
    for (int i = 0; i < nkb; ++i) {
        const int m = i >> 1, half = i & 1, bs = m & 1;
        if (ok && half == 0) ok = warp_wait(&b_full[bs], (m >> 1) & 1, kWaitLimit, p.status, 31, p.diag);
        const uint32_t* words = reinterpret_cast<const uint32_t*>(bring + bs * bstage_bytes) + r * 4 + 2 * half;
        for (int j = 0; j < 2; ++j) {
            if (ok) ok = warp_wait(&ge[j], (i & 1) ^ 1, kWaitLimit, p.status, 28, p.diag);
            if (ok) {
                tc_fence_after();
                const uint32_t col = abase + lane_addr + j * 8 * ne;
                // one 8-column store per tile: a warp writes its 32 lanes of
                // four tiles faster as four such stores than as one 32-column store
                for (int k = 0; k < ne; ++k) store_signs(col + 8 * k, words[fp.e_slot[e0 + kIss * k] * 512 + j]);
                tmem_st_wait();
            }
            tc_fence_before();
            named_arrive(group_bar(g, j), kGroupThreads);
        }
        if (half == 1 || i == nkb - 1) {             // done with this bits stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&b_empty[bs]);
        }
    }
    // ---- epilogue: y = 2^-s_t (B + alpha_v S) over the group's columns, alpha
    // the variant's scale (per matrix, or of this output row) ----
    if (ok) ok = warp_wait(acc_full, 0, kWaitLimit, p.status, 29, p.diag);
    if (!ok) return;
    tc_fence_after();
    for (int c0 = bcol; c0 < bcol + bn; c0 += 16) {
        uint32_t v[16], u[16];
        tmem_ld16(tmem + lane_addr + c0, v);
        tmem_ld16(tmem + lane_addr + kSCol0 + c0, u);
        // the chunk's coefficients, the same for every lane: broadcast loads,
        // eight positions at a time, the first eight issued before the wait
        // on the tensor-memory loads
        float a[8], sc[8];
        auto coefs = [&](int t0) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float4 a4 = reinterpret_cast<const float4*>(alpha_s + c0 + t0)[q];
                const float4 s4 = reinterpret_cast<const float4*>(scale_s + c0 + t0)[q];
                a[4 * q] = a4.x; a[4 * q + 1] = a4.y; a[4 * q + 2] = a4.z; a[4 * q + 3] = a4.w;
                sc[4 * q] = s4.x; sc[4 * q + 1] = s4.y; sc[4 * q + 2] = s4.z; sc[4 * q + 3] = s4.w;
            }
            if (p.alpha_rows && row_ok) {
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int vv = var_s[c0 + t0 + t];
                    a[t] = vv >= 0 ? __ldg(p.alphas + static_cast<int64_t>(vv) * p.N + n) : 0.f;
                }
            }
        };
        coefs(0);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h == 1) coefs(8);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                v[8 * h + t] = __float_as_uint(fmaf(a[t], __uint_as_float(u[8 * h + t]), __uint_as_float(v[8 * h + t])) * sc[t]);
        }
        if (row_ok) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const int pos = c0 + t;
                const float val = __uint_as_float(v[t]);
                if (pos < p.M) store_out(p, psm, split, pos, tok_s[pos], n, r, val);
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) fold_decode_kernel(const __grid_constant__ FoldParams p) {
    using namespace sm100;
    extern __shared__ uint8_t dsmem[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t w_full[kWMax], w_empty[kWMax], x_full[kXMax], x_empty[kXMax];
    __shared__ uint64_t b_full[kBStages], b_empty[kBStages];
    __shared__ uint64_t g_empty[kIss][kABufs], zeroed, acc_full, drain;
    __shared__ uint32_t tmem_base;
    __shared__ SegPlan pl;
    __shared__ FoldPlan fp;
    __shared__ int last_cta;
    __shared__ int32_t tok_s[kFoldMaxCols];
    __shared__ __align__(16) float scale_s[kFoldMaxCols];   // 2^-s_t, 0 for invalid and padding positions
    __shared__ int32_t var_s[kFoldMaxCols];
    __shared__ __align__(16) float alpha_s[kFoldMaxCols];   // per-matrix scale of the position's variant, 0 for base

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Mb = p.Mb;
    const uint32_t xs_bytes = static_cast<uint32_t>(Mb + p.Rmax) * 128u;
    const uint32_t bstage_bytes = static_cast<uint32_t>(p.bslots) * 2048u;
    uint8_t* wring = base;
    uint8_t* bring = wring + p.wstages * kWTile;
    uint8_t* xring = bring + kBStages * bstage_bytes;
    const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
    const int n0 = tile * kBN;
    // K slices are cut at even 64-column blocks, so every bits copy (two
    // blocks, 16 bytes a row) starts on a 16-byte boundary
    const int kb_total = p.K / kBK;
    const int npairs = (kb_total + 1) / 2;
    const int kb0 = 2 * static_cast<int>(static_cast<int64_t>(split) * npairs / p.splits);
    const int kb1 = min(kb_total, 2 * static_cast<int>(static_cast<int64_t>(split + 1) * npairs / p.splits));
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWMax; ++s) { mbar_init(&w_full[s], 1); mbar_init(&w_empty[s], 1); }
        for (int s = 0; s < kXMax; ++s) { mbar_init(&x_full[s], 1); mbar_init(&x_empty[s], kIss * kGroupIss + 1); }
        for (int s = 0; s < kBStages; ++s) { mbar_init(&b_full[s], 1); mbar_init(&b_empty[s], 4 * kIss); }
        for (int g = 0; g < kIss; ++g)
            for (int b = 0; b < kABufs; ++b) mbar_init(&g_empty[g][b], kGroupIss);
        mbar_init(&zeroed, 4 * kIss);
        mbar_init(&acc_full, kIss * kGroupIss + 1);
        mbar_init(&drain, kIss * kGroupIss + 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base, kTmemCols);
    // everything above overlaps the staging kernel; its outputs are read below
    asm volatile("griddepcontrol.wait;" ::: "memory");
    {
        const int* src = reinterpret_cast<const int*>(p.plan);
        int* dst = reinterpret_cast<int*>(&pl);
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(SegPlan) / 4); i += blockDim.x) dst[i] = src[i];
        const int* fsrc = reinterpret_cast<const int*>(p.fold);
        int* fdst = reinterpret_cast<int*>(&fp);
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(FoldPlan) / 4); i += blockDim.x) fdst[i] = fsrc[i];
    }
    for (int q = threadIdx.x; q < Mb; q += blockDim.x) {
        tok_s[q] = q < p.M ? p.pos2tok[q] : -1;
        var_s[q] = q < p.M ? p.pos_var[q] : -2;
        scale_s[q] = var_s[q] == -2 ? 0.f : pow2i(-p.sexp[q]);
        alpha_s[q] = (!p.alpha_rows && var_s[q] >= 0) ? p.alphas[var_s[q]] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    // the host only picks this kernel when the plan fits; anything else is a bug
    const bool plan_ok = fp.ok != 0 && fp.R <= p.Rmax && fp.C * 16 == Mb && pl.D <= kFoldMaxSlots &&
                         fp.n_entries <= kAEntries && pl.D <= p.bslots;
    if (!plan_ok && threadIdx.x == 0) report(p.status, BD_ERR_UNSUPPORTED);

    if (!plan_ok) {
        // nothing was issued; fall through to the teardown
    } else if (warp == 0) {
        // ---------------- TMA producer: W_base tiles (HBM) ----------------
        // W and the activations have rings of their own, so the W stream runs
        // its full depth ahead whatever the depth of the activation ring.
        if (lane == 0) {
            prefetch_tensormap(&p.tm_w);
            int issued = 0;
            for (int i = 0; i < nkb; ++i) {
                const int ws = i % p.wstages;
                if (!mbar_wait_sleep(&w_empty[ws], ((i / p.wstages) & 1) ^ 1, kWaitLimit, p.status, 21, p.diag)) break;
                mbar_expect_tx(&w_full[ws], kWTile);
                tma_load_2d(wring + ws * kWTile, &p.tm_w, &w_full[ws], (kb0 + i) * kBK, n0);
                issued = i + 1;
            }
            // wait (bounded) until every load issued has landed, so no copy is
            // still writing shared memory when the CTA exits
            for (int s = 0; s < p.wstages && s < issued; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) % p.wstages);
                mbar_wait_sleep(&w_full[s], (last / p.wstages) & 1, kWaitLimit, p.status, 23, p.diag);
            }
        }
    } else if (warp == 1) {
        // ---------------- bulk producer: activations (L2) ----------------
        // The staging kernel lays out, per 64-column block, the stage exactly
        // as it sits in shared memory (X_c rows, then X_p rows, 128-byte
        // swizzled), so one contiguous copy fills a stage: the copy engine's
        // cost is per copy and per box row far more than per byte.
        if (lane == 0) {
            const uint32_t bytes = static_cast<uint32_t>(Mb + fp.R) * 128u;
            int issued = 0;
            for (int i = 0; i < nkb; ++i) {
                const int kb = kb0 + i;
                const int xs = i % p.xstages;
                if (!mbar_wait_sleep(&x_empty[xs], ((i / p.xstages) & 1) ^ 1, kWaitLimit, p.status, 22, p.diag)) break;
                mbar_expect_tx(&x_full[xs], bytes);
                bulk_load(xring + xs * xs_bytes, p.ximg + static_cast<int64_t>(kb) * xs_bytes, bytes, &x_full[xs]);
                issued = i + 1;
            }
            for (int s = 0; s < p.xstages && s < issued; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) % p.xstages);
                mbar_wait_sleep(&x_full[s], (last / p.xstages) & 1, kWaitLimit, p.status, 24, p.diag);
            }
        }
    } else if (warp == 2) {
        // ---------------- TMA producer: sign bits (HBM) ----------------
        // one 128-row x 4-word tile per present variant and pair of blocks
        if (lane == 0) {
            const int D = pl.D;
            for (int d = 0; d < D; ++d) prefetch_tensormap(&p.tm_bits[pl.var[d]]);
            const int np = (nkb + 1) / 2;
            int issued = 0;
            for (int m = 0; m < np; ++m) {
                const int bs = m % kBStages;
                if (!mbar_wait_sleep(&b_empty[bs], ((m / kBStages) & 1) ^ 1, kWaitLimit, p.status, 32, p.diag)) break;
                if (D == 0) { mbar_arrive(&b_full[bs]); issued = m + 1; continue; }
                mbar_expect_tx(&b_full[bs], static_cast<uint32_t>(D) * 2048u);
                uint8_t* sb = bring + bs * bstage_bytes;
                for (int d = 0; d < D; ++d)
                    tma_load_2d(sb + d * 2048, &p.tm_bits[pl.var[d]], &b_full[bs], 2 * (kb0 + 2 * m), n0);
                issued = m + 1;
            }
            for (int s = 0; s < kBStages && s < issued; ++s) {
                const int last = issued - 1 - ((issued - 1 - s) % kBStages);
                mbar_wait_sleep(&b_full[s], (last / kBStages) & 1, kWaitLimit, p.status, 33, p.diag);
            }
        }
    } else if (warp == kBaseWarp) {
        base_issue(p, tmem, nkb, wring, xring, xs_bytes, w_full, w_empty, x_full, x_empty, &acc_full, &drain);
    } else {
        // ---------------- issuer groups ----------------
        // Group g: four expansion warps (one per tensor-memory lane quarter)
        // build the +-1 tiles of the group's own entries, then arrive on a
        // named barrier; the group's issuer warp waits on it and issues the
        // group's MMAs.  Each group owns a disjoint run of accumulator
        // columns, so groups never wait for one another.
        const int g = (warp - kFirstGroup) / kGroupWarps;
        const int gw = (warp - kFirstGroup) % kGroupWarps;
        const int bcol = fp.iss_col[g], bn = fp.iss_n[g];
        const int e0 = fp.iss_e0[g], ne = fp.iss_ne[g];
        int a0 = 0;                                 // first +-1 tile column of this group
        for (int h = 0; h < g; ++h) a0 += 8 * kABufs * fp.iss_ne[h];
        const uint32_t abase = tmem + kACol0 + a0;
        if (gw >= 4)
            group_issue(p, fp, tmem, abase, e0, ne, g, gw - 4, nkb, xring, xs_bytes, x_full, x_empty, g_empty[g], &zeroed,
                        &acc_full, &drain);
        else
            group_expand(p, fp, tmem, abase, e0, ne, g, warp % 4, n0, nkb, g_empty[g], bring, bstage_bytes,
                         b_full, b_empty, &zeroed, &acc_full, tok_s, scale_s, var_s, alpha_s, split, bcol, bn,
                         reinterpret_cast<float*>(base));
    }

    __syncthreads();
    if (plan_ok && p.cluster_reduce) {
        // the K slices of this row tile are the CTAs of one cluster (rank =
        // split), each holding its partial tile [Mb][128] f32 at the start of
        // its (now idle) pipeline memory: CTA `split` sums its share of the
        // tile over the slices' shared memory in the order 0, 1, 2, ... and
        // writes y
        cluster_sync_all();
        const int rows = min(kBN, p.N - n0);
        const uint32_t psm_a = smem_u32(base);
        const int per_t = kBN / 4;                              // float4 groups per grouped position
        const int total = p.M * per_t;
        const int g0 = static_cast<int>(static_cast<int64_t>(split) * total / p.splits);
        const int g1 = static_cast<int>(static_cast<int64_t>(split + 1) * total / p.splits);
        // two float4 groups per thread and pass, the slices read four at a
        // time before they are added (in order): the remote loads of a pass
        // are in flight together
        const int nt = static_cast<int>(blockDim.x);
        for (int gb = g0 + static_cast<int>(threadIdx.x); gb < g1; gb += 2 * nt) {
            const int gq[2] = {gb, gb + nt};
            float4 acc[2];
            bool live[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                live[h] = gq[h] < g1 && 4 * (gq[h] % per_t) < rows;
                acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (live[h]) acc[h] = ld_cluster_f4(cluster_map(psm_a + static_cast<uint32_t>(gq[h]) * 16u, 0));
            }
            for (int sl = 1; sl < p.splits; sl += 4) {
                float4 part[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (live[h] && sl + q < p.splits)
                            part[h][q] = ld_cluster_f4(cluster_map(psm_a + static_cast<uint32_t>(gq[h]) * 16u,
                                                                   static_cast<uint32_t>(sl + q)));
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (live[h] && sl + q < p.splits) {
                            acc[h].x += part[h][q].x; acc[h].y += part[h][q].y;
                            acc[h].z += part[h][q].z; acc[h].w += part[h][q].w;
                        }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!live[h]) continue;
                const int pos = gq[h] / per_t, r4 = 4 * (gq[h] % per_t);
                const int64_t o = static_cast<int64_t>(tok_s[pos]) * p.N + n0 + r4;
                const float4 a = acc[h];
                if (r4 + 4 <= rows && (p.N & 3) == 0) {
                    if (p.y_bf16) {
                        const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
                        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.y) + o) =
                            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
                    } else {
                        *reinterpret_cast<float4*>(static_cast<float*>(p.y) + o) = a;
                    }
                } else {
                    const float v4[4] = {a.x, a.y, a.z, a.w};
                    for (int j = 0; j < 4 && r4 + j < rows; ++j) {
                        if (p.y_bf16) static_cast<__nv_bfloat16*>(p.y)[o + j] = __float2bfloat16_rn(v4[j]);
                        else static_cast<float*>(p.y)[o + j] = v4[j];
                    }
                }
            }
        }
        cluster_sync_all();            // no CTA leaves while its tile is being read
    } else if (plan_ok && p.splits > 1) {
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
            const int64_t sstride = static_cast<int64_t>(p.M) * p.N;        // floats per slice
            if (rows == kBN && (p.N & 3) == 0) {
                // four outputs per thread, slices summed in order 0, 1, 2, ...
                // with four loads in flight
                const int nq = kBN / 4;
                const int64_t sq = sstride / 4;
                for (int idx = threadIdx.x; idx < p.M * nq; idx += blockDim.x) {
                    const int pos = idx / nq, c4 = idx % nq;
                    const float4* src = reinterpret_cast<const float4*>(p.part + static_cast<int64_t>(pos) * p.N + n0) + c4;
                    float4 acc = __ldcg(src);
                    int sl = 1;
                    for (; sl + 3 < p.splits; sl += 4) {
                        const float4 a = __ldcg(src + sl * sq), b = __ldcg(src + (sl + 1) * sq);
                        const float4 c = __ldcg(src + (sl + 2) * sq), d = __ldcg(src + (sl + 3) * sq);
                        acc.x = (((acc.x + a.x) + b.x) + c.x) + d.x;
                        acc.y = (((acc.y + a.y) + b.y) + c.y) + d.y;
                        acc.z = (((acc.z + a.z) + b.z) + c.z) + d.z;
                        acc.w = (((acc.w + a.w) + b.w) + c.w) + d.w;
                    }
                    for (; sl < p.splits; ++sl) {
                        const float4 a = __ldcg(src + sl * sq);
                        acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
                    }
                    const int64_t o = static_cast<int64_t>(tok_s[pos]) * p.N + n0 + 4 * c4;
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
                    const int pos = idx / rows, rr = idx % rows;
                    float acc = 0.f;
                    for (int sl = 0; sl < p.splits; ++sl)
                        acc += __ldcg(p.part + (static_cast<int64_t>(sl) * p.M + pos) * p.N + n0 + rr);
                    const int64_t o = static_cast<int64_t>(tok_s[pos]) * p.N + n0 + rr;
                    if (p.y_bf16) static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(acc);
                    else static_cast<float*>(p.y)[o] = acc;
                }
            }
            if (threadIdx.x == 0) p.tickets[tile] = 0u;
        }
    }
    if (warp == 0) {
        // every MMA this CTA issued has completed before its tensor memory is freed
        if (plan_ok) mbar_wait_sleep(&drain, 0, kWaitLimit, p.status, 30, p.diag);
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Staging for one linear (one block per staged row), written as K / 64 stage
// images of Mb + Rmax rows x 128 bytes, one per 64-column block, each laid
// out as the kernel's shared-memory stage (row q at 128 q, its 16-byte chunk
// c at chunk position c ^ (q & 7): the 128-byte swizzle):
//   X_c rows [0, Mb) bf16: grouped order, row p = x[t] * 2^s_t (zero rows
//       past the valid tokens);
//   X_p rows Mb + [0, R) bytes: entry rows of the plan; row j of entry e
//       holds, if grouped position e_col + j is a token of the entry's
//       variant v, x[t] 2^s_t as e4m3 hi and lo, per block 64 bytes of hi
//       then 64 of lo, byte 32w + 4j + b of a half holding column
//       32w + j + 8b; otherwise zeros;
//   s_t = 7 - floor(log2(max_k |x[t,k]|)) (0 for zero rows), clamped to
//       [-120, 120];
//   the split-K tickets zeroed.
// ---------------------------------------------------------------------------
// Largest |x| of a bf16 row (bf16 bit patterns without the sign order like
// magnitudes), reduced over the block.
__device__ float row_absmax(const uint4* __restrict__ src, int64_t vec_per_row) {
    __shared__ uint32_t red[8];
    uint32_t mx = 0;
    for (int64_t i = threadIdx.x; i < vec_per_row; i += blockDim.x) {
        const uint4 v = __ldg(src + i);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) mx = max(mx, max(w4[k] & 0x7FFFu, (w4[k] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    uint32_t all = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) all = max(all, red[i]);
    return __uint_as_float(all << 16);
}

// s with 2^s xmax in [128, 256) (0 for a zero or non-finite maximum),
// clamped to [-120, 120] like the per-variant kernel's: every token whose
// largest |x| lies in [2^-113, 2^128) gets the full range; 2^s and 2^-s stay
// normal floats.
__device__ __forceinline__ int scale_exponent(float xmax) {
    if (!(xmax > 0.f) || !(xmax < 3.0e38f)) return 0;
    const int biased = static_cast<int>((__float_as_uint(xmax) >> 23) & 0xFF);
    const int e = biased > 0 ? biased - 127 : -126;
    return max(-120, min(120, 7 - e));
}

// 16-byte unit `chunk` of staged row q's 2K bytes in the stage images: block
// kb = chunk / 8 holds the row at bytes (kb img_rows + q) 128, its chunk
// c = chunk % 8 at chunk position c ^ (q & 7) (the 128-byte swizzle of a
// 1024-byte aligned stage).
__device__ __forceinline__ uint4* image_chunk(uint8_t* ximg, int img_rows, int q, int64_t chunk) {
    const int64_t kb = chunk >> 3;
    const int c = static_cast<int>(chunk & 7);
    return reinterpret_cast<uint4*>(ximg + (kb * img_rows + q) * 128 + ((c ^ (q & 7)) << 4));
}

__global__ void __launch_bounds__(256) fold_prep_kernel(const uint4* __restrict__ x, int K, int M, int Mb,
                                                        const SegPlan* __restrict__ plan,
                                                        const FoldPlan* __restrict__ fold,
                                                        const int32_t* __restrict__ pos2tok,
                                                        const int32_t* __restrict__ pos_var,
                                                        int32_t* __restrict__ sexp, uint8_t* __restrict__ ximg,
                                                        int img_rows, unsigned* tickets, int n_tickets) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int rr = blockIdx.x;
    const int64_t vec_per_row = K / 8;
    if (rr == 0)
        for (int i = threadIdx.x; i < n_tickets; i += blockDim.x) tickets[i] = 0u;
    const int n_valid = M - plan->n_invalid;
    if (rr < Mb) {
        const int pos = rr;
        const int tok = pos < n_valid ? pos2tok[pos] : -1;
        if (tok < 0) {
            for (int64_t i = threadIdx.x; i < vec_per_row; i += blockDim.x)
                *image_chunk(ximg, img_rows, pos, i) = make_uint4(0, 0, 0, 0);
            if (threadIdx.x == 0) sexp[pos] = 0;
            return;
        }
        const uint4* src = x + static_cast<int64_t>(tok) * vec_per_row;
        const int s = scale_exponent(row_absmax(src, vec_per_row));
        if (threadIdx.x == 0) sexp[pos] = s;
        const float sc = pow2i(s);
        for (int64_t i = threadIdx.x; i < vec_per_row; i += blockDim.x) {
            const uint4 v = __ldg(src + i);
            uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            if (s != 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(bf16_lo(w4[k]) * sc, bf16_hi(w4[k]) * sc);
                    w4[k] = *reinterpret_cast<const uint32_t*>(&pr);
                }
            }
            *image_chunk(ximg, img_rows, pos, i) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        return;
    }
    const int r = rr - Mb;
    if (r >= fold->R) return;
    int tok = -1;
    for (int e = 0; e < fold->n_entries; ++e) {
        const int row0 = fold->e_row[e];
        if (r >= row0 && r < row0 + fold->e_n[e]) {
            const int pos = fold->e_col[e] + (r - row0);
            const int d = fold->e_slot[e];
            if (pos >= plan->off[d] && pos < plan->off[d] + plan->cnt[d]) tok = pos2tok[pos];
            break;
        }
    }
    const int q = Mb + r;                                        // 2K bytes: hi and lo per block
    if (tok < 0) {
        for (int64_t i = threadIdx.x; i < vec_per_row; i += blockDim.x)
            *image_chunk(ximg, img_rows, q, i) = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4* src = x + static_cast<int64_t>(tok) * vec_per_row;
    const int s = scale_exponent(row_absmax(src, vec_per_row));
    const float sc = pow2i(s);
    // one thread per 32-column group: 64 source bytes in, 32 bytes of hi and
    // 32 of lo out; output word jj holds columns jj, jj + 8, jj + 16, jj + 24
    // (converted two at a time)
    for (int grp = threadIdx.x; grp < K / 32; grp += blockDim.x) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 q = __ldg(src + 4 * grp + i);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[8 * i + 2 * k] = bf16_lo(w4[k]) * sc;
                v[8 * i + 2 * k + 1] = bf16_hi(w4[k]) * sc;
            }
        }
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            uint32_t hw = 0, lw = 0;
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {               // columns jj + 16 pr and jj + 16 pr + 8
                const float a0 = v[jj + 16 * pr], a1 = v[jj + 16 * pr + 8];
                const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
                const float2 hb = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
                const __nv_fp8x2_storage_t l2 =
                    __nv_cvt_float2_to_fp8x2(make_float2(a0 - hb.x, a1 - hb.y), __NV_SATFINITE, __NV_E4M3);
                hw |= static_cast<uint32_t>(h2) << (16 * pr);
                lw |= static_cast<uint32_t>(l2) << (16 * pr);
            }
            hi[jj] = hw;
            lo[jj] = lw;
        }
        // block grp / 2: hi at bytes 32 (grp & 1) .. +32, lo at 64 + the same
        const int64_t c0 = 8 * static_cast<int64_t>(grp >> 1) + 2 * (grp & 1);
        *image_chunk(ximg, img_rows, q, c0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *image_chunk(ximg, img_rows, q, c0 + 1) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        *image_chunk(ximg, img_rows, q, c0 + 4) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *image_chunk(ximg, img_rows, q, c0 + 5) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    }
}

int fold_dmax(int64_t M, int32_t V) {
    int64_t d = V < M ? V : M;
    return static_cast<int>(d < kFoldMaxSlots ? d : kFoldMaxSlots);
}

// Sign-operand rows: the entries' chunks, at most (chunks + variants - 1)
// of 16 rows (variant runs meet other runs only at their end chunks).
int fold_rmax(int64_t M, int32_t V) {
    const int r = 16 * (pad16(static_cast<int>(M)) / 16 + fold_dmax(M, V) - 1);
    return r > 16 ? r : 16;
}

constexpr int kMaxClusterSplits = 16;          // cluster size (above 8: non-portable, where the device allows it)

// Clusters of `s` CTAs of the kernel (one per SM at `smem` bytes) that run at
// once -- the GPCs' SM counts need not be multiples of s.  Cached per device;
// 0 if the query fails.
int fold_cluster_capacity(int s, int smem) {
    static int cache[64][kMaxClusterSplits + 1] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev][s] > 0) return cache[dev][s];
    if (!set_smem_attr(reinterpret_cast<const void*>(fold_decode_kernel), smem, 2)) return 0;
    if (s > 8 && cudaFuncSetAttribute(reinterpret_cast<const void*>(fold_decode_kernel),
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
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
    if (cudaOccupancyMaxActiveClusters(&n, fold_decode_kernel, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 0;
    }
    return cache[dev][s] = n;
}

// K slices per row tile (in pairs of 64-column blocks) and how they are
// summed: minimise waves x (fixed per-CTA cost + blocks per slice x time per
// block) + the split-K reduction.  Up to 16 slices may form one cluster and
// be summed in shared memory (waves counted in the clusters that fit at
// once, the reduction nearly free); otherwise the CTA that finishes the tile
// last sums the slices' partials from HBM, with waves counted in single CTAs
// (measured with the reduction switched off: ~2.5 us + ~0.6 us per slice at
// 128 tokens, in proportion to the tokens).  The time per block is the
// larger of its HBM time (W tile + one bits tile per variant at ~45 GB/s per
// SM) and its MMA issue time (~55 cycles per MMA per issuer warp at ~2 GHz).
struct FoldSplit {
    int splits;
    bool cluster;
};
FoldSplit fold_splits(int64_t n_tiles, int kb_total, int sms, int dmax, int64_t M, int smem) {
    const double hbm_us = (16.0 + dmax) * 1024.0 / 45.0e3;
    const int entries = (dmax + kIss - 1) / kIss + 1;
    const double issue_us = 2.0 * (2 * entries) * 55.0 / 2000.0;
    const double kb_us = hbm_us > issue_us ? hbm_us : issue_us;
    const double fixed_us = 4.0;
    const double tok = static_cast<double>(M) / 128.0;
    const int npairs = (kb_total + 1) / 2;
    FoldSplit best{1, false};
    double best_t = 1e30;
    auto consider = [&](int s, bool cluster, int64_t waves, double reduce) {
        const double t = static_cast<double>(waves) * (fixed_us + 2 * ((npairs + s - 1) / s) * kb_us) + reduce;
        if (t < best_t * 0.98) { best_t = t; best = FoldSplit{s, cluster}; }
    };
    for (int s = 1; s <= 32 && s <= npairs; ++s) {
        consider(s, false, (n_tiles * s + sms - 1) / sms, s > 1 ? tok * (2.5 + 0.6 * s) : 0.0);
        if (s > 1 && s <= kMaxClusterSplits) {
            const int cap = fold_cluster_capacity(s, smem);
            if (cap > 0) consider(s, true, (n_tiles + cap - 1) / cap, 0.5);
        }
    }
    return best;
}

// Shared-memory plan of one launch: ring depths that fit next to the static
// shared memory (about 4 KB) under the 227 KB limit.
struct FoldSmem {
    int wstages, xstages, bslots, bytes;
};
FoldSmem fold_smem(int Mb, int rmax, int dmax) {
    FoldSmem f;
    f.bslots = dmax > 0 ? dmax : 1;
    const int budget = 227 * 1024 - 4096;
    const int bits = kBStages * f.bslots * 2048;
    const int xs = (Mb + rmax) * 128;
    for (f.xstages = kXMax; f.xstages >= 1; --f.xstages)
        for (f.wstages = kWMax; f.wstages >= 3; --f.wstages) {
            f.bytes = f.wstages * static_cast<int>(kWTile) + bits + f.xstages * xs + 1024;
            if (f.bytes <= budget) return f;
        }
    f.wstages = 0;                               // does not fit
    return f;
}

struct FoldScratch {
    uint8_t* ximg;
    int32_t* sexp;
    float* part;
    unsigned* tickets;
    size_t bytes;
};

FoldScratch fold_scratch(void* base, int64_t M, int64_t N, int64_t K, int32_t V, FoldSplit sp) {
    FoldScratch d{};
    char* p = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* r = p ? p + off : nullptr;
        off += round_up(bytes, kAlign);
        return r;
    };
    const int Mb = pad16(static_cast<int>(M));
    // (K / 64) stage images of (Mb + Rmax) rows x 128 bytes
    d.ximg = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(Mb + fold_rmax(M, V)) * K * 2));
    d.sexp = reinterpret_cast<int32_t*>(take(static_cast<size_t>(Mb) * 4));
    const int64_t n_tiles = (N + kBN - 1) / kBN;
    // HBM partials only for the ticket reduction
    d.part = (sp.splits > 1 && !sp.cluster) ? reinterpret_cast<float*>(take(static_cast<size_t>(sp.splits) * M * N * 4))
                                            : nullptr;
    d.tickets = reinterpret_cast<unsigned*>(take(static_cast<size_t>(n_tiles) * 4));
    d.bytes = off;
    return d;
}

FoldSplit splits_for(int64_t M, int64_t N, int64_t K, int32_t V) {
    const int64_t n_tiles = (N + kBN - 1) / kBN;
    const int dmax = fold_dmax(M, V);
    const int smem = fold_smem(pad16(static_cast<int>(M)), fold_rmax(M, V), dmax).bytes;
    return fold_splits(n_tiles, static_cast<int>(K / kBK), sm_count(), dmax, M, smem);
}

}  // namespace

bool decode_fold_supported(const LinearArgs& a) {
    return a.M >= 1 && pad16(static_cast<int>(a.M > 4096 ? 4096 : a.M)) <= kFoldMaxCols &&
           (a.V < a.M ? a.V : a.M) <= kFoldMaxSlots && a.K % kBK == 0 && a.K >= kBK && a.N >= 1 &&
           a.N < (int64_t(1) << 31) && a.K < (int64_t(1) << 31);
}

size_t decode_fold_scratch_bytes(int64_t M, int64_t N, int64_t K, int32_t V) {
    if (M < 1 || pad16(static_cast<int>(M > 4096 ? 4096 : M)) > kFoldMaxCols || K % kBK != 0) return 0;
    return fold_scratch(nullptr, M, N, K, V, splits_for(M, N, K, V)).bytes;
}

bd_status launch_decode_fold(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s) {
    const int M = static_cast<int>(a.M), N = static_cast<int>(a.N), K = static_cast<int>(a.K);
    const int Mb = pad16(M);
    const int64_t n_tiles = (a.N + kBN - 1) / kBN;
    const FoldSplit sp = splits_for(a.M, a.N, a.K, a.V);
    const int splits = sp.splits;
    FoldScratch sc = fold_scratch(w.tc_scratch, a.M, a.N, a.K, a.V, sp);
    if (sc.bytes > w.tc_bytes) return BD_ERR_WORKSPACE;
    const int rmax = fold_rmax(a.M, a.V);

    fold_prep_kernel<<<Mb + rmax, 256, 0, s>>>(static_cast<const uint4*>(a.x), K, M, Mb, w.g.plan,
                                              w.g.fold, w.g.pos2tok, w.g.pos_var, sc.sexp, sc.ximg, Mb + rmax,
                                              sc.tickets, splits > 1 ? static_cast<int>(n_tiles) : 0);
    if (launch_status() != BD_OK) return BD_ERR_CUDA;

    FoldParams p;
    memset(&p, 0, sizeof p);
    if (!make_tmap_bf16_sw128(&p.tm_w, a.w_base, a.N, a.K, kBN)) return BD_ERR_CUDA;
    p.ximg = sc.ximg;
    for (int v = 0; v < a.V; ++v)
        if (!make_tmap_bits(&p.tm_bits[v], a.bits.p[v], a.N, a.K / 32, kBN)) return BD_ERR_CUDA;
    p.plan = w.g.plan;
    p.fold = w.g.fold;
    p.pos2tok = w.g.pos2tok;
    p.pos_var = w.g.pos_var;
    p.alphas = a.alphas;
    p.alpha_rows = a.alpha_rows;
    p.sexp = sc.sexp;
    p.y = a.y;
    p.part = sc.part;
    p.tickets = sc.tickets;
    p.status = w.status;
    p.diag = w.status + 2;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Mb = Mb;
    p.Rmax = rmax;
    p.splits = splits;
    p.cluster_reduce = (splits > 1 && sp.cluster) ? 1 : 0;
    p.y_bf16 = (a.y_dtype == BD_BF16);
    const FoldSmem fs = fold_smem(Mb, rmax, fold_dmax(a.M, a.V));
    if (fs.wstages == 0) return BD_ERR_UNSUPPORTED;
    p.wstages = fs.wstages;
    p.xstages = fs.xstages;
    p.bslots = fs.bslots;
    const int smem = fs.bytes;
    if (!set_smem_attr(reinterpret_cast<const void*>(fold_decode_kernel), smem, 2)) return BD_ERR_CUDA;
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
    if (cudaLaunchKernelEx(&cfg, fold_decode_kernel, p) != cudaSuccess) return BD_ERR_CUDA;
    return launch_status();
}

}  // namespace bd
