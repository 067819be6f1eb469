// bd_linear.cu -- the multi-variant fused linear: token grouping, the CUDA-core
// kernel, and the dispatcher behind bitdelta_linear.
//
// Page: "BitDelta: serving 14 Zen models from one GPU cluster", section
// "Serving architecture": variants share one resident base; a request's
// effective weight W_eff = W_base + alpha_v * sign(delta_v) is rebuilt on the
// fly inside the matmul kernel from the base weights and the packed delta
// bits, and never written to HBM.  A batch here mixes tokens of different
// variants; they are grouped by variant id so that each variant's bits are
// read once per weight tile.
//
// Every path computes, per token t of variant v and output row n,
//   y[t, n] = sum_k x[t,k] W_base[n,k]  +  alpha_v * sum_k x[t,k] s_v[n,k]
// with fp32 accumulation, i.e. the base product and the sign product are kept
// apart and combined with the f32 alpha in the epilogue.
#include "bd_internal.cuh"
#include "bd_paths.cuh"

namespace bd {

LinearWorkspace linear_workspace_layout(void* base, int64_t M, int64_t N, int64_t K, int32_t V) {
    LinearWorkspace w{};
    char* p = static_cast<char*>(base);
    size_t off = 0;
    w.status = reinterpret_cast<unsigned*>(p);
    off += kHeaderBytes;
    auto take = [&](size_t bytes) {
        char* r = p ? p + off : nullptr;
        off += round_up(bytes, kAlign);
        return r;
    };
    const size_t m = static_cast<size_t>(M > 0 ? M : 0);
    w.g.counts = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (V + 2)));
    w.g.offsets = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (V + 3)));
    w.g.pos2tok = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (m ? m : 1)));
    w.g.pos_var = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (m ? m : 1)));
    w.g.plan = reinterpret_cast<SegPlan*>(take(sizeof(SegPlan)));
    w.g.fold = reinterpret_cast<FoldPlan*>(take(sizeof(FoldPlan)));
    w.group_end = off;
    w.tc_bytes = tc_scratch_bytes(M, N, K, V);
    w.tc_scratch = w.tc_bytes ? take(w.tc_bytes) : nullptr;
    w.total = off;
    return w;
}

namespace {

// ---------------------------------------------------------------------------
// Token grouping: a stable counting sort of the tokens by variant id.
// Bucket 0 holds id -1 (the base model), bucket 1 + v holds variant v, and the
// last bucket collects ids outside [-1, V) (reported, output rows zeroed).
// One block; tokens are placed 1024 at a time with warp match + ballots so the
// order inside every bucket is the token order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int bucket_of(int32_t id, int V) {
    return (id >= -1 && id < V) ? id + 1 : V + 1;
}

// Issue plan of the folded decode kernel.  Each present variant's run of
// grouped positions is one "entry": its +-1 tile, two sign MMAs (hi, lo) per
// K step over the 16-column chunks the run touches, and those chunks' rows
// of the sign operand.  The entries are dealt to the kFoldIssuers issuer
// groups round-robin (entry e to group e % kFoldIssuers), so no group has
// more than one entry above another whatever the run lengths; the chunks
// are split into kFoldIssuers near-equal contiguous ranges only for zeroing
// the sign accumulator and for the epilogue.
constexpr int kFoldChunks = kFoldMaxCols / 16;

// Bit d of mask[c]: run d (first position off[d], cnt[d] tokens) has a token
// in chunk c.
__device__ void fold_masks(const int32_t* off, const int32_t* cnt, int D, uint32_t* mask) {
    for (int c = 0; c < kFoldChunks; ++c) mask[c] = 0;
    for (int d = 0; d < D; ++d) {
        const int c0 = off[d] / 16, c1 = (off[d] + cnt[d] - 1) / 16;
        for (int c = c0; c <= c1; ++c) mask[c] |= 1u << d;
    }
}

__device__ void fold_plan(const SegPlan& pl, int M, FoldPlan* fp) {
    constexpr int I = kFoldIssuers;
    const int C = pad16(M) / 16;
    fp->ok = 0;
    fp->C = C;
    fp->R = 0;
    fp->n_entries = 0;
    for (int i = 0; i < I; ++i) { fp->iss_col[i] = 0; fp->iss_n[i] = 0; fp->iss_e0[i] = 0; fp->iss_ne[i] = 0; }
    if (C > kFoldChunks || pl.D > kFoldMaxSlots) return;
    int row = 0;
    for (int d = 0; d < pl.D; ++d) {
        const int c0 = pl.off[d] / 16, c1 = (pl.off[d] + pl.cnt[d] - 1) / 16;
        fp->e_col[d] = 16 * c0;
        fp->e_n[d] = 16 * (c1 - c0 + 1);
        fp->e_slot[d] = d;
        fp->e_row[d] = row;
        row += 16 * (c1 - c0 + 1);
    }
    for (int i = 0; i < I; ++i) {
        const int a = C * i / I, b = C * (i + 1) / I;
        fp->iss_col[i] = 16 * a;
        fp->iss_n[i] = 16 * (b - a);
        fp->iss_e0[i] = i;                              // entries i, i + I, i + 2 I, ...
        fp->iss_ne[i] = pl.D > i ? (pl.D - i + I - 1) / I : 0;
    }
    fp->n_entries = pl.D;
    fp->R = row;
    fp->ok = 1;
}

// Order of the variant runs in the grouped layout.  Candidate 0 is the id
// order; candidate c > 0 is a seeded shuffle of it (Fisher-Yates, indices
// drawn with the "lowbias32" integer hash of c and the step).
constexpr int kOrderTries = 1;                   // candidates per thread
__device__ __forceinline__ uint32_t lowbias32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}
__device__ void run_order(int cand, const int* present, int D, int* ord) {
    for (int d = 0; d < D; ++d) ord[d] = present[d];
    if (cand == 0) return;
    for (int i = D - 1; i > 0; --i) {
        const int j = static_cast<int>(lowbias32(static_cast<uint32_t>(cand) * 0x9E3779B9u + static_cast<uint32_t>(i)) %
                                       static_cast<uint32_t>(i + 1));
        const int t = ord[i];
        ord[i] = ord[j];
        ord[j] = t;
    }
}

// Score of an order for the folded kernel: the sign-operand rows (in
// chunks) -- runs that share a chunk each need its rows.
__device__ int order_score(const int* ord, int D, const int* total, int n_base) {
    int32_t off[kFoldMaxSlots], cnt[kFoldMaxSlots];
    int run = n_base;
    for (int d = 0; d < D; ++d) {
        off[d] = run;
        cnt[d] = total[ord[d] + 1];
        run += cnt[d];
    }
    uint32_t mask[kFoldChunks];
    fold_masks(off, cnt, D, mask);
    int rows = 0;
    for (int c = 0; c < kFoldChunks; ++c) rows += __popc(mask[c]);
    return rows;
}

__global__ void __launch_bounds__(1024) group_kernel(const int32_t* __restrict__ ids, int M, int V,
                                                     int group_budget, int order_search, GroupView g,
                                                     unsigned* status) {
    extern __shared__ int sm[];
    const int nb = V + 2;
    int* hist = sm;                    // [32][nb] per-warp counts of the current slice
    int* total = hist + 32 * nb;       // [nb]
    int* start = total + nb;           // [nb]
    int* placed = start + nb;          // [nb]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < nb; i += blockDim.x) { total[i] = 0; placed[i] = 0; }
    __syncthreads();
    bool bad = false;
    for (int t = threadIdx.x; t < M; t += blockDim.x) {
        const int b = bucket_of(ids[t], V);
        bad |= (b == V + 1);
        atomicAdd(&total[b], 1);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) report(status, BD_ERR_VARIANT);
    // Order of the variant runs: for a batch the folded decode kernel may
    // take (the caller says whether it can), the best of blockDim.x * kOrderTries candidate orders (ties go to the
    // lowest candidate, so the result does not depend on timing); otherwise
    // the id order.
    __shared__ unsigned long long red[32];
    __shared__ int best_cand;
    int present[kFoldMaxSlots];
    int D = 0;
    for (int v = 0; v < V && D <= kFoldMaxSlots; ++v)
        if (total[v + 1] > 0) {
            if (D < kFoldMaxSlots) present[D] = v;
            ++D;
        }
    const int C = pad16(M) / 16;
    const bool search = order_search && D >= 2 && D <= kFoldMaxSlots && C <= kFoldChunks;
    unsigned long long key = ~0ull;
    if (search)
        for (int k = 0; k < kOrderTries; ++k) {
            const int cand = threadIdx.x * kOrderTries + k;
            int ord[kFoldMaxSlots];
            run_order(cand, present, D, ord);
            const unsigned long long kk = (static_cast<unsigned long long>(order_score(ord, D, total, total[0])) << 32) |
                                          static_cast<unsigned>(cand);
            key = kk < key ? kk : key;
        }
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
        key = other < key ? other : key;
    }
    if (lane == 0) red[warp] = key;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long b = ~0ull;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) b = red[w] < b ? red[w] : b;
        best_cand = search ? static_cast<int>(b & 0xffffffffu) : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // bucket order: base tokens, the variant runs, invalid ids
        int ord[BITDELTA_MAX_VARIANTS];
        int n = 0;
        if (search) {
            run_order(best_cand, present, D, ord);
            n = D;
        } else {
            for (int v = 0; v < V; ++v)
                if (total[v + 1] > 0) ord[n++] = v;
        }
        int run = total[0];
        start[0] = 0;
        for (int k = 0; k < n; ++k) {
            start[ord[k] + 1] = run;
            run += total[ord[k] + 1];
        }
        for (int v = 0; v < V; ++v)
            if (total[v + 1] == 0) start[v + 1] = run;
        start[V + 1] = run;
        for (int b = 0; b < nb; ++b) {
            g.offsets[b] = start[b];
            g.counts[b] = total[b];
        }
        g.offsets[nb] = run + total[V + 1];
        // segment plan: present variants in layout order, padded segments, passes
        SegPlan* pl = g.plan;
        pl->M = M;
        pl->n_base = total[0];
        pl->n_invalid = total[V + 1];
        int d = 0, rows = 0, groups = 0, group_rows = 0, group_vars = 0;
        pl->group_first[0] = 0;
        for (int k = 0; k < n; ++k) {
            const int v = ord[k];
            const int c = total[v + 1];
            const int pr = pad16(c);
            if (group_rows > 0 && (group_rows + pr > group_budget || group_vars == kMaxPassVariants)) {
                pl->group_first[++groups] = d;
                group_rows = 0;
                group_vars = 0;
            }
            pl->var[d] = v;
            pl->cnt[d] = c;
            pl->off[d] = start[v + 1];
            pl->seg[d] = rows;
            rows += pr;
            group_rows += pr;
            ++group_vars;
            ++d;
        }
        pl->D = d;
        pl->P = rows;
        pl->n_groups = groups + 1;
        pl->group_first[groups + 1] = d;
        fold_plan(*pl, M, g.fold);
    }
    __syncthreads();
    for (int s0 = 0; s0 < M; s0 += blockDim.x) {
        const int t = s0 + threadIdx.x;
        const int b = (t < M) ? bucket_of(ids[t], V) : -1;
        for (int i = threadIdx.x; i < 32 * nb; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const unsigned peers = __match_any_sync(0xffffffffu, b);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (b >= 0 && rank == 0) hist[warp * nb + b] = __popc(peers);
        __syncthreads();
        if (b >= 0) {
            int before = 0;
            for (int w = 0; w < warp; ++w) before += hist[w * nb + b];
            const int pos = start[b] + placed[b] + before + rank;
            g.pos2tok[pos] = t;
            g.pos_var[pos] = (b == V + 1) ? -2 : b - 1;
        }
        __syncthreads();
        for (int bb = threadIdx.x; bb < nb; bb += blockDim.x) {
            int sum = 0;
            for (int w = 0; w < 32; ++w) sum += hist[w * nb + bb];
            placed[bb] += sum;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// CUDA-core path.  One warp per output row; lanes stride over 8-column chunks
// of K (16-byte loads of W_base and x, one byte of bits per variant); tokens
// are walked in grouped order, 8 at a time, with separate fp32 accumulators
// for the base and sign products.
// ---------------------------------------------------------------------------
constexpr int kSimtWarps = 8;
constexpr int kSimtTok = 8;

__global__ void __launch_bounds__(kSimtWarps * 32)
simt_linear_kernel(const uint4* __restrict__ x, const uint4* __restrict__ w_base,
                   const float* __restrict__ alphas, int alpha_rows, BitsTable bt, int64_t M, int64_t N,
                   int64_t K, GroupView g, void* y, int y_bf16) {
    const int lane = threadIdx.x & 31;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kSimtWarps + (threadIdx.x >> 5);
    if (n >= N) return;
    const int64_t kc = K / 8;                              // 8-column chunks per row
    const uint4* wrow = w_base + n * kc;
    for (int64_t p0 = 0; p0 < M; p0 += kSimtTok) {
        int tok[kSimtTok], var[kSimtTok];
#pragma unroll
        for (int j = 0; j < kSimtTok; ++j) {
            const int64_t p = p0 + j;
            tok[j] = (p < M) ? g.pos2tok[p] : -1;
            var[j] = (p < M) ? g.pos_var[p] : -2;
        }
        float accb[kSimtTok], accs[kSimtTok];
#pragma unroll
        for (int j = 0; j < kSimtTok; ++j) { accb[j] = 0.f; accs[j] = 0.f; }
        for (int64_t c = lane; c < kc; c += 32) {
            const uint4 wv = __ldg(wrow + c);
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
            float wf[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) { wf[2 * i] = bf16_lo(ww[i]); wf[2 * i + 1] = bf16_hi(ww[i]); }
#pragma unroll
            for (int j = 0; j < kSimtTok; ++j) {
                if (tok[j] < 0 || var[j] == -2) continue;
                const uint4 xv = __ldg(x + static_cast<int64_t>(tok[j]) * kc + c);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                float xf[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) { xf[2 * i] = bf16_lo(xw[i]); xf[2 * i + 1] = bf16_hi(xw[i]); }
                float db = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) db = fmaf(xf[i], wf[i], db);
                accb[j] += db;
                if (var[j] >= 0) {
                    const uint32_t byte = __ldg(bt.p[var[j]] + n * kc + c);
                    float ds = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) ds += ((byte >> i) & 1u) ? xf[i] : -xf[i];
                    accs[j] += ds;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kSimtTok; ++j) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                accb[j] += __shfl_xor_sync(0xffffffffu, accb[j], o);
                accs[j] += __shfl_xor_sync(0xffffffffu, accs[j], o);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < kSimtTok; ++j) {
                if (tok[j] < 0) continue;
                float out = 0.f;
                if (var[j] >= 0) out = fmaf(alpha_rows ? alphas[var[j] * N + n] : alphas[var[j]], accs[j], accb[j]);
                else if (var[j] == -1) out = accb[j];
                const int64_t o = static_cast<int64_t>(tok[j]) * N + n;
                if (y_bf16) static_cast<__nv_bfloat16*>(y)[o] = __float2bfloat16_rn(out);
                else static_cast<float*>(y)[o] = out;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Small-batch CUDA-core path (M <= 4): a GEMV per output row.  `split` warps
// (1, 2, 4 or 8) share a row, each taking a contiguous 1/split of its
// 8-column chunks; each lane issues U 16-byte weight loads (plus the matching
// activation vectors and bits bytes) before doing any arithmetic, so enough
// bytes are in flight per SM to stream W_base at full HBM bandwidth.  Narrow
// matrices use split > 1 so that every SM holds enough warps and each warp
// makes fewer dependent round trips; the parts of a row are added in a fixed
// order.
// ---------------------------------------------------------------------------
template <int MT, int U, int SPLIT>
__global__ void __launch_bounds__(kSimtWarps * 32)
gemv_kernel(const uint4* __restrict__ x, const uint4* __restrict__ w_base,
            const float* __restrict__ alphas, int alpha_rows, BitsTable bt, int M, int64_t N, int64_t K,
            GroupView g, void* y, int y_bf16) {
    __shared__ float part_sum[SPLIT > 1 ? kSimtWarps : 1][2 * MT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int part = warp % SPLIT;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * (kSimtWarps / SPLIT) + warp / SPLIT;
    const bool row_ok = n < N;
    if (SPLIT == 1 && !row_ok) return;                      // no block-wide barrier below
    const int64_t kc = K / 8;
    const int64_t c_lo = SPLIT == 1 ? 0 : kc * part / SPLIT, c_hi = SPLIT == 1 ? kc : kc * (part + 1) / SPLIT;
    int tok[MT], var[MT];
    const uint8_t* bp[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
        tok[j] = (j < M) ? g.pos2tok[j] : -1;
        var[j] = (j < M) ? g.pos_var[j] : -2;
        if (var[j] == -2) tok[j] = -1;                      // invalid id: zero row
        bp[j] = (var[j] >= 0 && (SPLIT == 1 || row_ok)) ? bt.p[var[j]] + n * kc : nullptr;
    }
    float accb[MT], accs[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) { accb[j] = 0.f; accs[j] = 0.f; }
    const uint4* wrow = w_base + (SPLIT == 1 || row_ok ? n : 0) * kc;
    auto chunk = [&](const uint4& wv, const uint4 (&xv)[MT], const uint32_t (&bb)[MT]) {
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
        float wf[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) { wf[2 * i] = bf16_lo(ww[i]); wf[2 * i + 1] = bf16_hi(ww[i]); }
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            if (tok[j] < 0) continue;
            const uint32_t xw[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
            float xf[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) { xf[2 * i] = bf16_lo(xw[i]); xf[2 * i + 1] = bf16_hi(xw[i]); }
            float db = 0.f, ds = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                db = fmaf(xf[i], wf[i], db);
                ds += ((bb[j] >> i) & 1u) ? xf[i] : -xf[i];
            }
            accb[j] += db;
            accs[j] += ds;
        }
    };
    int64_t c = c_lo + lane;
    const int64_t c_end = (SPLIT == 1 || row_ok) ? c_hi : c_lo;   // a row past N does no work
    for (; c + 32 * (U - 1) < c_end; c += 32 * U) {
        uint4 wv[U];
        uint4 xv[U][MT];
        uint32_t bb[U][MT];
#pragma unroll
        for (int u = 0; u < U; ++u) wv[u] = ld_stream(wrow + c + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                xv[u][j] = tok[j] >= 0 ? __ldg(x + static_cast<int64_t>(tok[j]) * kc + c + 32 * u) : make_uint4(0, 0, 0, 0);
                bb[u][j] = bp[j] ? static_cast<uint32_t>(__ldg(bp[j] + c + 32 * u)) : 0u;
            }
#pragma unroll
        for (int u = 0; u < U; ++u) chunk(wv[u], xv[u], bb[u]);
    }
    for (; c < c_end; c += 32) {
        uint4 xv[MT];
        uint32_t bb[MT];
        const uint4 wv = ld_stream(wrow + c);
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            xv[j] = tok[j] >= 0 ? __ldg(x + static_cast<int64_t>(tok[j]) * kc + c) : make_uint4(0, 0, 0, 0);
            bb[j] = bp[j] ? static_cast<uint32_t>(__ldg(bp[j] + c)) : 0u;
        }
        chunk(wv, xv, bb);
    }
#pragma unroll
    for (int j = 0; j < MT; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            accb[j] += __shfl_xor_sync(0xffffffffu, accb[j], o);
            accs[j] += __shfl_xor_sync(0xffffffffu, accs[j], o);
        }
    }
    if (SPLIT > 1) {
        // the parts of a row, added in order 0, 1, ... by the row's first warp
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                part_sum[warp][j] = accb[j];
                part_sum[warp][MT + j] = accs[j];
            }
        __syncthreads();
        if (part != 0 || !row_ok) return;
        if (lane == 0)
            for (int q = 1; q < SPLIT; ++q)
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    accb[j] += part_sum[warp + q][j];
                    accs[j] += part_sum[warp + q][MT + j];
                }
    }
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < MT; ++j) {
            if (j >= M) continue;
            const int t = g.pos2tok[j];
            float out = 0.f;
            if (var[j] >= 0) out = fmaf(alpha_rows ? alphas[var[j] * N + n] : alphas[var[j]], accs[j], accb[j]);
            else if (var[j] == -1) out = accb[j];
            const int64_t o = static_cast<int64_t>(t) * N + n;
            if (y_bf16) static_cast<__nv_bfloat16*>(y)[o] = __float2bfloat16_rn(out);
            else static_cast<float*>(y)[o] = out;
        }
    }
}

bd_status launch_group(const int32_t* ids, int64_t M, int32_t V, const LinearWorkspace& w,
                       cudaStream_t s, bool order_search) {
    int threads = static_cast<int>(round_up(static_cast<size_t>(M), 32));
    if (threads > 1024) threads = 1024;
    if (order_search && threads < 256) threads = 256;        // at least 256 candidate orders
    const size_t smem = sizeof(int) * (32 * (V + 2) + 3 * (V + 2));
    group_kernel<<<1, threads, smem, s>>>(ids, static_cast<int>(M), V, decode_group_budget(M),
                                          order_search ? 1 : 0, w.g, w.status);
    return launch_status();
}

// Warps of gemv_kernel<MT, U> that run at once on the device (cached per
// device and instantiation).
template <int MT, int U>
int64_t gemv_resident_warps() {
    // every SPLIT uses the same registers within a few; the unsplit kernel decides
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, gemv_kernel<MT, U, 2>, kSimtWarps * 32, 0) != cudaSuccess ||
            nb < 1) {
            cudaGetLastError();
            nb = 1;
        }
        cache[dev] = nb;
    }
    return static_cast<int64_t>(cache[dev]) * kSimtWarps * sm_count();
}

// Warps per GEMV row: the most (1 to 8) that keep every warp of the launch
// resident at once and give each at least one full round of U 16-byte loads
// per lane.
int gemv_split(int64_t N, int64_t K, int U, int64_t resident) {
    int split = 1;
    while (split < kSimtWarps && N * split * 2 <= resident && (K / 8) / (split * 2) >= 32 * U) split *= 2;
    return split;
}

bd_status launch_simt(const LinearArgs& a, const LinearWorkspace& w, cudaStream_t s) {
    const int64_t blocks = (a.N + kSimtWarps - 1) / kSimtWarps;
    if (a.M <= 4) {
        const uint4* xx = static_cast<const uint4*>(a.x);
        const uint4* wb = static_cast<const uint4*>(a.w_base);
        const int M = static_cast<int>(a.M);
        const int yb = a.y_dtype == BD_BF16;
        const int U = a.M <= 2 ? 4 : 2;
        const int64_t resident = a.M == 1   ? gemv_resident_warps<1, 4>()
                                 : a.M == 2 ? gemv_resident_warps<2, 4>()
                                            : gemv_resident_warps<4, 2>();
        const int split = gemv_split(a.N, a.K, U, resident);
        const int rows_per_block = kSimtWarps / split;
        const unsigned grid = static_cast<unsigned>((a.N + rows_per_block - 1) / rows_per_block);
        auto go = [&](auto kern) {
            kern<<<grid, kSimtWarps * 32, 0, s>>>(xx, wb, a.alphas, a.alpha_rows, a.bits, M, a.N, a.K, w.g, a.y, yb);
        };
        if (a.M == 1) {
            if (split == 1) go(gemv_kernel<1, 4, 1>);
            else if (split == 2) go(gemv_kernel<1, 4, 2>);
            else if (split == 4) go(gemv_kernel<1, 4, 4>);
            else go(gemv_kernel<1, 4, 8>);
        } else if (a.M == 2) {
            if (split == 1) go(gemv_kernel<2, 4, 1>);
            else if (split == 2) go(gemv_kernel<2, 4, 2>);
            else if (split == 4) go(gemv_kernel<2, 4, 4>);
            else go(gemv_kernel<2, 4, 8>);
        } else {
            if (split == 1) go(gemv_kernel<4, 2, 1>);
            else if (split == 2) go(gemv_kernel<4, 2, 2>);
            else if (split == 4) go(gemv_kernel<4, 2, 4>);
            else go(gemv_kernel<4, 2, 8>);
        }
        return launch_status();
    }
    simt_linear_kernel<<<static_cast<unsigned>(blocks), kSimtWarps * 32, 0, s>>>(
        static_cast<const uint4*>(a.x), static_cast<const uint4*>(a.w_base), a.alphas, a.alpha_rows, a.bits,
        a.M, a.N, a.K, w.g, a.y, a.y_dtype == BD_BF16);
    return launch_status();
}

bd_status check_linear_args(const void* x, const int32_t* ids, int64_t M, int64_t N, int64_t K,
                            const void* w_base, const float* alphas,
                            const uint32_t* const* bits, int32_t V, const void* y,
                            bd_dtype y_dtype) {
    if (M < 0 || N < 1 || K < 32 || K % 32 != 0) return BD_ERR_SHAPE;
    if (V < 0 || V > BITDELTA_MAX_VARIANTS) return BD_ERR_SHAPE;
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return BD_ERR_SHAPE;
    if (y_dtype != BD_F32 && y_dtype != BD_BF16) return BD_ERR_DTYPE;
    if (M == 0) return BD_OK;
    if (!x || !ids || !w_base || !y) return BD_ERR_NULL;
    if (V > 0 && (!alphas || !bits)) return BD_ERR_NULL;
    for (int v = 0; v < V; ++v)
        if (!bits[v]) return BD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(w_base, 16) || !aligned(y, 16) || !aligned(ids, 4))
        return BD_ERR_ALIGN;
    if (V > 0 && !aligned(alphas, 4)) return BD_ERR_ALIGN;
    for (int v = 0; v < V; ++v)
        if (!aligned(bits[v], 16)) return BD_ERR_ALIGN;
    return BD_OK;
}

}  // namespace
}  // namespace bd

using namespace bd;

extern "C" size_t bitdelta_linear_workspace(int64_t M, int64_t N, int64_t K, int32_t V) {
    if (M < 0 || N < 1 || K < 32 || K % 32 != 0 || V < 0 || V > BITDELTA_MAX_VARIANTS) return 0;
    return linear_workspace_layout(nullptr, M, N, K, V).total;
}

namespace {

bd_status prepare(const void* x, int64_t M, int64_t N, int64_t K, const void* w_base,
                  const float* alphas, int alpha_rows, const uint32_t* const* bits, int32_t V, void* y,
                  bd_dtype y_dtype, void* workspace, size_t ws_bytes, bd_path& path,
                  LinearArgs& a, LinearWorkspace& w) {
    if (!workspace) return BD_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return BD_ERR_ALIGN;
    w = linear_workspace_layout(workspace, M, N, K, V);
    if (ws_bytes < w.total) return BD_ERR_WORKSPACE;
    a.x = x;
    a.M = M;
    a.N = N;
    a.K = K;
    a.w_base = w_base;
    a.alphas = alphas;
    a.alpha_rows = alpha_rows;
    a.V = V;
    for (int v = 0; v < BITDELTA_MAX_VARIANTS; ++v)
        a.bits.p[v] = (v < V) ? reinterpret_cast<const uint8_t*>(bits[v]) : nullptr;
    a.bits_host = bits;
    a.y = y;
    a.y_dtype = y_dtype;
    if (path == BD_PATH_AUTO) path = choose_path(a);
    if (path != BD_PATH_SIMT && path != BD_PATH_DECODE_TC && path != BD_PATH_PREFILL_TC &&
        path != BD_PATH_DECODE_FOLD && path != BD_PATH_DECODE_WEFF)
        return BD_ERR_UNSUPPORTED;
    if (path == BD_PATH_DECODE_WEFF && !decode_weff_supported(a)) return BD_ERR_UNSUPPORTED;
    if (path == BD_PATH_DECODE_TC && !decode_tc_supported(a)) return BD_ERR_UNSUPPORTED;
    if (path == BD_PATH_DECODE_FOLD && !decode_fold_supported(a)) return BD_ERR_UNSUPPORTED;
    if (path == BD_PATH_PREFILL_TC && !prefill_tc_supported(a)) return BD_ERR_UNSUPPORTED;
    return BD_OK;
}

}  // namespace

namespace bd {
bd_path choose_path(const LinearArgs& a) {
    // GEMV (CUDA cores) for 1-2 tokens; from 3 tokens the tensor-core decode
    // kernel is faster (4096 x 4096: 11.9 / 14.5 / 24.6 / 26.6 us for 1-4
    // tokens on CUDA cores against 22.5 us on tensor cores)
    if (a.M <= 2) return BD_PATH_SIMT;
    // One variant (V == 1): bf16 W_eff tiles built in shared memory and the
    // activations used as they are -- no staging kernel; faster than the
    // per-variant kernel on every shape measured (4096 x 4096 at 8 to 128
    // tokens: 19.6 to 23.8 us against 20.9 to 26.7 us, graph-replayed; the
    // 1024 x 8192, 8192 x 8192 and 28672 x 8192 shapes at 64 tokens by 7 to
    // 27%)
    if (a.V == 1 && decode_weff_supported(a)) return BD_PATH_DECODE_WEFF;
    // Measured on GB300 (q, k/v, gate and 4096 x 4096 shapes, 2 to 14 Zipf
    // variants, 16 to 128 tokens): the per-variant sign kernel wins for few
    // variants or few tokens; the folded kernel, whose cost hardly grows with
    // the number of variants, wins from 32 tokens on once there are 8 or more
    // variants, and from 32 tokens on for narrow outputs (N <= 2048) whatever
    // the variant count.
    if (a.V >= 2 && a.M >= 32 && (a.V >= 8 || a.N <= 2048) && decode_fold_supported(a))
        return BD_PATH_DECODE_FOLD;
    if (decode_tc_supported(a)) return BD_PATH_DECODE_TC;
    if (prefill_tc_supported(a)) return BD_PATH_PREFILL_TC;
    return BD_PATH_SIMT;
}

}  // namespace bd

namespace {

bd_status launch_path(bd_path path, const LinearArgs& a, const LinearWorkspace& w,
                      cudaStream_t s) {
    switch (path) {
        case BD_PATH_DECODE_TC: return launch_decode_tc(a, w, s);
        case BD_PATH_DECODE_FOLD: return launch_decode_fold(a, w, s);
        case BD_PATH_PREFILL_TC: return launch_prefill_tc(a, w, s);
        case BD_PATH_DECODE_WEFF: return launch_decode_weff(a, w, s);
        default: return launch_simt(a, w, s);
    }
}

}  // namespace

extern "C" bd_status bitdelta_group(const int32_t* variant_ids, int64_t M, int32_t V,
                                    void* workspace, size_t ws_bytes, void* stream) {
    if (M < 0 || M > (int64_t(1) << 30) || V < 0 || V > BITDELTA_MAX_VARIANTS) return BD_ERR_SHAPE;
    if (M == 0) return BD_OK;
    if (!variant_ids) return BD_ERR_NULL;
    if (!aligned(variant_ids, 4)) return BD_ERR_ALIGN;
    if (!workspace) return BD_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return BD_ERR_ALIGN;
    LinearWorkspace w = linear_workspace_layout(workspace, M, 1, 32, V);
    if (ws_bytes < w.group_end) return BD_ERR_WORKSPACE;
    return launch_group(variant_ids, M, V, w, static_cast<cudaStream_t>(stream), true);
}

extern "C" bd_status bitdelta_linear_grouped(const void* x, int64_t M, int64_t N, int64_t K,
                                             const void* w_base, const float* alphas,
                                             const uint32_t* const* bits, int32_t V, void* y,
                                             bd_dtype y_dtype, void* workspace, size_t ws_bytes,
                                             void* stream, bd_path path) {
    const int32_t one = 0;
    bd_status st = check_linear_args(x, &one, M, N, K, w_base, alphas, bits, V, y, y_dtype);
    if (st != BD_OK) return st;
    if (M == 0) return BD_OK;
    LinearArgs a;
    LinearWorkspace w;
    a.ids = nullptr;
    st = prepare(x, M, N, K, w_base, alphas, 0, bits, V, y, y_dtype, workspace, ws_bytes, path, a, w);
    if (st != BD_OK) return st;
    return launch_path(path, a, w, static_cast<cudaStream_t>(stream));
}

extern "C" bd_status bitdelta_linear_ex(const void* x, const int32_t* variant_ids, int64_t M,
                                        int64_t N, int64_t K, const void* w_base,
                                        const float* alphas, const uint32_t* const* bits,
                                        int32_t V, void* y, bd_dtype y_dtype, void* workspace,
                                        size_t ws_bytes, void* stream, bd_path path) {
    bd_status st = check_linear_args(x, variant_ids, M, N, K, w_base, alphas, bits, V, y, y_dtype);
    if (st != BD_OK) return st;
    if (M == 0) return BD_OK;
    LinearArgs a;
    LinearWorkspace w;
    a.ids = variant_ids;
    st = prepare(x, M, N, K, w_base, alphas, 0, bits, V, y, y_dtype, workspace, ws_bytes, path, a, w);
    if (st != BD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = launch_group(variant_ids, M, V, w, s, path == BD_PATH_DECODE_FOLD);
    if (st != BD_OK) return st;
    return launch_path(path, a, w, s);
}

extern "C" bd_status bitdelta_linear_rows(const void* x, const int32_t* variant_ids, int64_t M,
                                          int64_t N, int64_t K, const void* w_base,
                                          const float* alpha_rows, const uint32_t* const* bits,
                                          int32_t V, void* y, bd_dtype y_dtype, void* workspace,
                                          size_t ws_bytes, void* stream, bd_path path) {
    bd_status st = check_linear_args(x, variant_ids, M, N, K, w_base, alpha_rows, bits, V, y, y_dtype);
    if (st != BD_OK) return st;
    if (M == 0) return BD_OK;
    LinearArgs a;
    LinearWorkspace w;
    a.ids = variant_ids;
    st = prepare(x, M, N, K, w_base, alpha_rows, 1, bits, V, y, y_dtype, workspace, ws_bytes, path, a, w);
    if (st != BD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = launch_group(variant_ids, M, V, w, s, path == BD_PATH_DECODE_FOLD);
    if (st != BD_OK) return st;
    return launch_path(path, a, w, s);
}

extern "C" bd_status bitdelta_linear(const void* x, const int32_t* variant_ids, int64_t M,
                                     int64_t N, int64_t K, const void* w_base,
                                     const float* alphas, const uint32_t* const* bits, int32_t V,
                                     void* y, bd_dtype y_dtype, void* workspace, size_t ws_bytes,
                                     void* stream) {
    return bitdelta_linear_ex(x, variant_ids, M, N, K, w_base, alphas, bits, V, y, y_dtype,
                              workspace, ws_bytes, stream, BD_PATH_AUTO);
}
