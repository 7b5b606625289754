// Tensor-core (tcgen05 / TMEM) kernels of the bf16 MiTA forward pass.
//
// Steps of "MiTA Attention: Efficient Fast-Weight Scaling via a Mixture of
// Top-k Activations" (gist.science summaries) and where they run:
//   shared expert Vt = softmax(scale Qt K^T) V and the raw scores Qt K^T that
//   rank the top-k sets (Arabic edition, section 2)        -> k_landmark_tc
//   routing of each query to s landmarks                    -> k_route_tc
//   grouping (query, slot) pairs by routed expert           -> k_bucket_*
//   one softmax per query over K* = [Qt, K_(e1), ..]
//   and V* = [Vt, V_(e1), ..] (Dutch edition,
//   "Wiskundige Formulering")                               -> k_expert_tc
//
// Tiles are 128 rows (TMEM lanes) by 128 keys. One thread per row: thread r
// owns TMEM lane r, reads its score row, keeps the running max / sum of the
// online softmax and writes its probabilities (bf16) into the swizzled P tile
// that the second MMA (O += P V) reads. Thread 0 issues the MMAs; completion
// is signalled through an mbarrier with a bounded wait.
#include "internal.h"
#include "tc.cuh"

namespace mita {
using namespace tc;

namespace {

constexpr int kT = 128;                     // rows per tile = keys per chunk
constexpr int kPTile = kT * kT * 2;         // P tile bytes (128 x 128 bf16)
// K buffer that the P tile reuses: large enough for either.
template <int D> constexpr int kp_bytes() { return kT * D * 2 > kPTile ? kT * D * 2 : kPTile; }
constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 0);  // S[128 x 128] = A[128 x d] B[128 x d]^T

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem) { return tmem + ((threadIdx.x & ~31u) << 16); }

// Thread 0 waits on the MMA barrier; everyone then syncs. Returns false (for
// all threads) if the wait ran out.
__device__ __forceinline__ bool sync_on_mma(uint64_t* bar, uint32_t& phase, int* status) {
    int bad = 0;
    if (threadIdx.x == 0) bad = !mbar_wait(bar, phase, status);
    phase ^= 1u;
    bad = __syncthreads_or(bad);
    fence_after_sync();
    return !bad;
}

// Issues S = A * B^T over the head dim D (K-major A and B tiles of 128 rows).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tS, uint32_t sA, uint32_t sB, bool accumulate_first) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kT * 128 + (kk & 3) * 32;
        mma_bf16(tS, sdesc(sA + off, 16, 1024), sdesc(sB + off, 16, 1024), kIdS,
                 (kk > 0 || accumulate_first) ? 1u : 0u);
    }
}

// Issues O (+)= P * V: P is a K-major 128 x 128 tile, V an MN-major
// 128 keys x D tile (D contiguous).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t sP, uint32_t sV, bool accumulate) {
    constexpr uint32_t id = idesc_bf16(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk) {
        const uint32_t offp = (kk >> 2) * kT * 128 + (kk & 3) * 32;
        mma_bf16(tO, sdesc(sP + offp, 16, 1024), sdesc(sV + kk * 2048, kT * 128, 1024), id,
                 (kk > 0 || accumulate) ? 1u : 0u);
    }
}

// Where the landmark pass sends the raw scores of a row that pass the
// row's threshold: (score, key index) records appended at cand[n++].
struct CandOut {
    int2* cand;  // nullptr: no emission
    float thr;
    int j0;      // key index of column 0 of the chunk
    int n;
};

// Online softmax of this thread's row of one chunk of scores held in TMEM.
// nk keys are valid; sl = scale * log2(e). The reference max moves only when
// the chunk max exceeds it by more than 8 (probabilities stay <= 2^8), and
// then O (TMEM) is rescaled. Raw scores >= co.thr are emitted when co.cand.
template <int D>
__device__ __forceinline__ void chunk_softmax(uint32_t tS, uint32_t tO, uint8_t* sP, int nk, bool row_ok, float sl,
                                              bool first, float& mref, float& l, CandOut& co) {
    const int r = threadIdx.x;
    float mx = -INFINITY;
#pragma unroll 1
    for (int c0 = 0; c0 < kT; c0 += 32) {
        float v[32];
        tmem_ld32(tS + c0, v);
        tmem_wait_ld();
        if (co.cand && row_ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < nk && v[j] >= co.thr) co.cand[co.n++] = make_int2(__float_as_int(v[j]), co.j0 + c0 + j);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (row_ok && c0 + j < nk) mx = fmaxf(mx, v[j] * sl);
    }
    float mnew = mref, alpha = 1.0f;
    if (mx > mref + 8.0f) {
        mnew = mx;
        alpha = ex2(mref - mnew);
    }
    float sum = 0.0f;
#pragma unroll 1
    for (int c0 = 0; c0 < kT; c0 += 32) {
        float v[32];
        tmem_ld32(tS + c0, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const float p0 = (row_ok && c0 + j < nk) ? ex2(fmaf(v[j], sl, -mnew)) : 0.0f;
            const float p1 = (row_ok && c0 + j + 1 < nk) ? ex2(fmaf(v[j + 1], sl, -mnew)) : 0.0f;
            sum += p0 + p1;
            pk[j >> 1] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(sP + sw_off(r, (c0 >> 3) + q, kT)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
    l = l * alpha + sum;
    mref = mnew;
    const bool resc = !first && alpha != 1.0f;
    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            float o[32];
            tmem_ld32(tO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] *= alpha;
            tmem_st32(tO + c0, o);
        }
        tmem_wait_st();
    }
}

// Copies an R-row operand tile (R a multiple of 8): row t comes from
// src_row(t) (nullptr -> zero row), D bf16 per row, into the swizzled layout
// at sbase. src_row(-1) must return any valid global address.
template <int D, typename RowPtr>
__device__ __forceinline__ void load_rows(uint32_t sbase, int R, RowPtr src_row) {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
#pragma unroll 4
    for (int i = threadIdx.x; i < R * CPR; i += blockDim.x) {
        const int row = i / CPR, c = i % CPR;
        const __nv_bfloat16* p = src_row(row);
        cp_async16(sbase + sw_off(row, c, R), p ? (const void*)(p + c * 8) : (const void*)src_row(-1), p != nullptr);
    }
}

template <int D, typename RowPtr>
__device__ __forceinline__ void load_tile(uint32_t sbase, RowPtr src_row) {
    load_rows<D>(sbase, kT, src_row);
}

// Keeps the SMAX largest keys seen so far, descending; a key equal to one
// already held stays behind it, so with increasing indices ties go to the
// lower index.
template <int SMAX>
__device__ __forceinline__ void top_insert(uint32_t (&bu)[SMAX], int (&bi)[SMAX], uint32_t u, int i) {
#pragma unroll
    for (int t = 0; t < SMAX; ++t) {
        const bool gt = u > bu[t];
        const uint32_t tu = bu[t];
        const int ti = bi[t];
        bu[t] = gt ? u : tu;
        bi[t] = gt ? i : ti;
        u = gt ? tu : u;
        i = gt ? ti : i;
    }
}

}  // namespace

// ------------------------------------------------------------------------
// Landmark pass: per (landmark tile, key split, head). S = Qhi K^T + Qlo K^T
// (the bf16 split of fp32 Qt keeps the ranking scores at fp32 accuracy);
// every score at or above its row's threshold is recorded as a top-k
// candidate, and an online-softmax partial of Vt over the split is written.
template <int D>
__global__ void __launch_bounds__(128, 1)
    k_landmark_tc(const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
                  const __nv_bfloat16* __restrict__ Qhi, const __nv_bfloat16* __restrict__ Qlo,
                  const float* __restrict__ thr, int2* __restrict__ cand, int* __restrict__ ccount,
                  float* __restrict__ Opart, float2* __restrict__ ML, int N, int m, int m_pad,
                  int splits, int chunks_per_split, float sl, int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    constexpr int TILE = kT * D * 2;
    constexpr int kKP = kp_bytes<D>();
    uint8_t* sHi = sm;
    uint8_t* sLo = sm + TILE;
    uint8_t* sK = sm + 2 * TILE;  // also the P tile (128 x 128 bf16) once S is in TMEM
    uint8_t* sV = sK + kKP;
    const int mt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z, r = threadIdx.x;

    if (r < 32) tmem_alloc(&tmem_slot, 256);
    if (r == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tS = lane_base(tmem), tO = lane_base(tmem) + 128;
    uint32_t phase = 0;

    const size_t qrow0 = (size_t)bh * m_pad + (size_t)mt * kT;
    load_tile<D>(smem_u32(sHi), [&](int t) { return Qhi + (qrow0 + (t < 0 ? 0 : t)) * D; });
    load_tile<D>(smem_u32(sLo), [&](int t) { return Qlo + (qrow0 + (t < 0 ? 0 : t)) * D; });

    const int row = mt * kT + r;
    const bool row_ok = row < m;
    const int j_begin = sp * chunks_per_split * kT;
    const int j_end = min(N, j_begin + chunks_per_split * kT);
    const __nv_bfloat16* Kb = K + (size_t)bh * N * D;
    const __nv_bfloat16* Vb = V + (size_t)bh * N * D;
    float mref = -INFINITY, l = 0.0f;
    bool ok = true;
    int c = 0;
    const size_t crow = ((size_t)bh * m_pad + row) * splits + sp;  // this row's record region of this split
    CandOut co;
    co.cand = row_ok ? cand + crow * (size_t)chunks_per_split * kT : nullptr;
    co.thr = row_ok ? thr[(size_t)bh * m + row] : 0.0f;
    co.n = 0;
    for (int j0 = j_begin; j0 < j_end; j0 += kT, ++c) {
        const int nk = min(kT, j_end - j0);
        load_tile<D>(smem_u32(sK), [&](int t) { return (t >= 0 && t < nk) ? Kb + (size_t)(j0 + t) * D : (t < 0 ? Kb : nullptr); });
        load_tile<D>(smem_u32(sV), [&](int t) { return (t >= 0 && t < nk) ? Vb + (size_t)(j0 + t) * D : (t < 0 ? Vb : nullptr); });
        cp_async_wait_all();
        fence_proxy_async();
        __syncthreads();
        if (r == 0) {
            fence_after_sync();
            issue_qk<D>(tS, smem_u32(sHi), smem_u32(sK), false);
            issue_qk<D>(tS, smem_u32(sLo), smem_u32(sK), true);
            mma_commit(&bar);
        }
        if (!(ok = sync_on_mma(&bar, phase, status))) break;
        co.j0 = j0;
        chunk_softmax<D>(tS, tO, sK, nk, row_ok, sl, c == 0, mref, l, co);
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        if (r == 0) {
            fence_after_sync();
            issue_pv<D>(tO, smem_u32(sK), smem_u32(sV), c > 0);
            mma_commit(&bar);
        }
        if (!(ok = sync_on_mma(&bar, phase, status))) break;
    }
    if (ok) {
        const size_t orow = ((size_t)bh * splits + sp) * m_pad + row;
        if (c == 0) {  // empty split (cannot happen with the host's split sizing)
            for (int c0 = 0; c0 < D; ++c0) Opart[orow * D + c0] = 0.0f;
        } else {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                float o[32];
                tmem_ld32(tO + c0, o);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(Opart + orow * D + c0 + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
            }
        }
        ML[orow] = make_float2(mref, l);
        ccount[crow] = co.n;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (r < 32) tmem_dealloc(tmem, 256);
}

// Sample pass of the top-k selection: raw scores of each landmark row against
// every R-th key (n_samp keys), same MMA sequence as the landmark pass.
template <int D>
__global__ void __launch_bounds__(128)
    k_sample_tc(const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ Qhi,
                const __nv_bfloat16* __restrict__ Qlo, float* __restrict__ Ssamp, int N, int m, int m_pad, int R,
                int n_samp, int chunks_per_cta, int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    constexpr int TILE = kT * D * 2;
    uint8_t* sHi = sm;
    uint8_t* sLo = sm + TILE;
    uint8_t* sK = sm + 2 * TILE;
    const int mt = blockIdx.x, cg = blockIdx.y, bh = blockIdx.z, r = threadIdx.x;
    if (r < 32) tmem_alloc(&tmem_slot, 128);
    if (r == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tS = lane_base(tmem);
    uint32_t phase = 0;
    const size_t qrow0 = (size_t)bh * m_pad + (size_t)mt * kT;
    load_tile<D>(smem_u32(sHi), [&](int t) { return Qhi + (qrow0 + (t < 0 ? 0 : t)) * D; });
    load_tile<D>(smem_u32(sLo), [&](int t) { return Qlo + (qrow0 + (t < 0 ? 0 : t)) * D; });
    const __nv_bfloat16* Kb = K + (size_t)bh * N * D;
    const int row = mt * kT + r;
    for (int c = cg * chunks_per_cta; c < (cg + 1) * chunks_per_cta && c * kT < n_samp; ++c) {
        const int t0 = c * kT, nk = min(kT, n_samp - t0);
        load_tile<D>(smem_u32(sK), [&](int t) {
            return (t >= 0 && t < nk) ? Kb + (size_t)(t0 + t) * R * D : (t < 0 ? Kb : nullptr);
        });
        cp_async_wait_all();
        fence_proxy_async();
        __syncthreads();
        if (r == 0) {
            fence_after_sync();
            issue_qk<D>(tS, smem_u32(sHi), smem_u32(sK), false);
            issue_qk<D>(tS, smem_u32(sLo), smem_u32(sK), true);
            mma_commit(&bar);
        }
        if (!sync_on_mma(&bar, phase, status)) break;
        float* dst = Ssamp + ((size_t)bh * m + (row < m ? row : 0)) * n_samp + t0;
#pragma unroll 1
        for (int c0 = 0; c0 < kT; c0 += 32) {
            float v[32];
            tmem_ld32(tS + c0, v);
            tmem_wait_ld();
            if (row < m)
                for (int j = 0; j < 32 && c0 + j < nk; ++j) dst[c0 + j] = v[j];
        }
        fence_before_sync();
        __syncthreads();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (r < 32) tmem_dealloc(tmem, 128);
}

// Merges the per-split partials: Vt = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// Writes Vt fp32 [BH][m][D] and the bf16 copy [BH][m_pad][D] (padding rows 0).
__global__ void k_vt_combine(const float* __restrict__ Opart, const float2* __restrict__ ML, int splits, int m,
                             int m_pad, int D, float* __restrict__ Vt, __nv_bfloat16* __restrict__ Vtb) {
    const int i = blockIdx.x, bh = blockIdx.y;
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float out = 0.0f;
        if (i < m) {
            float M = -INFINITY;
            for (int s = 0; s < splits; ++s) M = fmaxf(M, ML[((size_t)bh * splits + s) * m_pad + i].x);
            float num = 0.0f, den = 0.0f;
            for (int s = 0; s < splits; ++s) {
                const size_t o = ((size_t)bh * splits + s) * m_pad + i;
                const float2 ml = ML[o];
                if (ml.y == 0.0f) continue;
                const float w = exp2f(ml.x - M);
                num += w * Opart[o * D + c];
                den += w * ml.y;
            }
            out = num / den;
            Vt[((size_t)bh * m + i) * D + c] = out;
        }
        Vtb[((size_t)bh * m_pad + i) * D + c] = __float2bfloat16_rn(out);
    }
}

// ------------------------------------------------------------------------
// Routing: R = Q Qhi^T + Q Qlo^T (the bf16 split of fp32 Qt keeps routing
// scores at fp32 accuracy), then each thread keeps the s best landmarks of
// its query row (ties to the lower landmark index). Also clears the
// per-query merge counters.

template <int SMAX>
__device__ __forceinline__ void route_epilogue(uint32_t tR, int m, int s, int q, bool q_ok, int32_t* __restrict__ Erow,
                                               int* __restrict__ cnt_q) {
    uint32_t bu[SMAX];
    int bi[SMAX];
#pragma unroll
    for (int t = 0; t < SMAX; ++t) { bu[t] = 0u; bi[t] = -1; }
#pragma unroll 1
    for (int c0 = 0; c0 < m; c0 += 32) {
        float v[32];
        tmem_ld32(tR + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (c0 + j < m) top_insert<SMAX>(bu, bi, order_key(v[j]), c0 + j);
    }
    if (q_ok) {
#pragma unroll
        for (int t = 0; t < SMAX; ++t)
            if (t < s) Erow[t] = bi[t];
        *cnt_q = 0;
    }
}

// Persistent variant for m_pad <= 256: each CTA walks a contiguous range of
// 128-query tiles; Qt (hi, lo) of the current head stays in shared memory and
// the next query tile is loaded and multiplied while this tile's routes are
// picked (two TMEM accumulators).
template <int D, int SMAX>
__global__ void __launch_bounds__(128, 1)
    k_route_tc(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Qhi,
               const __nv_bfloat16* __restrict__ Qlo, int N, int m, int m_pad, int s, int tiles_per_head,
               int total_tiles, uint32_t tmem_cols, int32_t* __restrict__ E, int* __restrict__ cnt,
               int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int QT = m_pad * D * 2;
    uint8_t* sHi = sm;
    uint8_t* sLo = sm + QT;
    uint8_t* sQb[2] = {sm + 2 * QT, sm + 2 * QT + kT * D * 2};
    const int r = threadIdx.x;
    const int per = (total_tiles + gridDim.x - 1) / gridDim.x;
    const int t_begin = blockIdx.x * per, t_end = min(total_tiles, t_begin + per);
    if (t_begin >= t_end) return;
    if (r < 32) tmem_alloc(&tmem_slot, tmem_cols);
    if (r == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    uint32_t phase = 0;
    const uint32_t idR = idesc_bf16(128, m_pad, 0, 0);

    auto load_q = [&](int t, int b) {
        const int bh = t / tiles_per_head, q0 = (t % tiles_per_head) * kT;
        const __nv_bfloat16* Qb = Q + (size_t)bh * N * D;
        load_tile<D>(smem_u32(sQb[b]), [&](int i) {
            return i < 0 ? Qb : (q0 + i < N ? Qb + (size_t)(q0 + i) * D : nullptr);
        });
    };
    auto load_landmarks = [&](int bh) {
        const __nv_bfloat16* h = Qhi + (size_t)bh * m_pad * D;
        const __nv_bfloat16* lo = Qlo + (size_t)bh * m_pad * D;
        load_rows<D>(smem_u32(sHi), m_pad, [&](int i) { return h + (size_t)(i < 0 ? 0 : i) * D; });
        load_rows<D>(smem_u32(sLo), m_pad, [&](int i) { return lo + (size_t)(i < 0 ? 0 : i) * D; });
    };
    auto issue = [&](int b) {
        const uint32_t tR = tmem + b * m_pad;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t offa = (kk >> 2) * kT * 128 + (kk & 3) * 32;
            const uint32_t offb = (kk >> 2) * m_pad * 128 + (kk & 3) * 32;
            mma_bf16(tR, sdesc(smem_u32(sQb[b]) + offa, 16, 1024), sdesc(smem_u32(sHi) + offb, 16, 1024), idR,
                     kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t offa = (kk >> 2) * kT * 128 + (kk & 3) * 32;
            const uint32_t offb = (kk >> 2) * m_pad * 128 + (kk & 3) * 32;
            mma_bf16(tR, sdesc(smem_u32(sQb[b]) + offa, 16, 1024), sdesc(smem_u32(sLo) + offb, 16, 1024), idR, 1u);
        }
        mma_commit(&bar);
    };

    int t = t_begin, b = 0;
    load_landmarks(t / tiles_per_head);
    load_q(t, 0);
    cp_async_wait_all();
    fence_proxy_async();
    __syncthreads();
    if (r == 0) {
        fence_after_sync();
        issue(0);
    }
    for (; t < t_end; ++t, b ^= 1) {
        const int tn = t + 1;
        const bool has_next = tn < t_end;
        const bool new_head = has_next && (tn / tiles_per_head != t / tiles_per_head);
        if (has_next && !new_head) load_q(tn, b ^ 1);
        if (!sync_on_mma(&bar, phase, status)) break;  // MMA(t) done: its Q tile and the landmarks are free
        if (has_next) {
            if (new_head) {
                load_landmarks(tn / tiles_per_head);
                load_q(tn, b ^ 1);
            }
            cp_async_wait_all();
            fence_proxy_async();
            __syncthreads();
            if (r == 0) {
                fence_after_sync();
                issue(b ^ 1);
            }
        }
        const int bh = t / tiles_per_head, q = (t % tiles_per_head) * kT + r;
        const bool q_ok = q < N;
        route_epilogue<SMAX>(lane_base(tmem) + b * m_pad, m, s, q, q_ok, E + ((size_t)bh * N + (q_ok ? q : 0)) * s,
                             cnt + (size_t)bh * N + (q_ok ? q : 0));
        fence_before_sync();
    }
    // drain an MMA still in flight if the loop left early
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (r < 32) tmem_dealloc(tmem, tmem_cols);
}

// Variant for m_pad > 256: one CTA per 128-query tile, landmarks streamed in
// 128-row chunks into consecutive TMEM column blocks.
template <int D, int SMAX>
__global__ void __launch_bounds__(128)
    k_route_chunked_tc(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Qhi,
                       const __nv_bfloat16* __restrict__ Qlo, int N, int m, int m_pad, int s, uint32_t tmem_cols,
                       int32_t* __restrict__ E, int* __restrict__ cnt, int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    constexpr int TILE = kT * D * 2;
    uint8_t* sQ = sm;
    uint8_t* sHi = sm + TILE;
    uint8_t* sLo = sm + 2 * TILE;
    const int qt = blockIdx.x, bh = blockIdx.y, r = threadIdx.x;
    if (r < 32) tmem_alloc(&tmem_slot, tmem_cols);
    if (r == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tR = lane_base(tmem);
    uint32_t phase = 0;
    const int q0 = qt * kT;
    const __nv_bfloat16* Qb = Q + (size_t)bh * N * D;
    load_tile<D>(smem_u32(sQ), [&](int t) { return (t >= 0 && q0 + t < N) ? Qb + (size_t)(q0 + t) * D : (t < 0 ? Qb : nullptr); });
    bool ok = true;
    for (int lc = 0; lc * kT < m_pad; ++lc) {
        const size_t base = (size_t)bh * m_pad + (size_t)lc * kT;
        load_tile<D>(smem_u32(sHi), [&](int t) { return Qhi + (base + (t < 0 ? 0 : t)) * D; });
        load_tile<D>(smem_u32(sLo), [&](int t) { return Qlo + (base + (t < 0 ? 0 : t)) * D; });
        cp_async_wait_all();
        fence_proxy_async();
        __syncthreads();
        if (r == 0) {
            fence_after_sync();
            issue_qk<D>(tR + lc * kT, smem_u32(sQ), smem_u32(sHi), false);
            issue_qk<D>(tR + lc * kT, smem_u32(sQ), smem_u32(sLo), true);
            mma_commit(&bar);
        }
        if (!(ok = sync_on_mma(&bar, phase, status))) break;
    }
    if (ok) {
        const int q = q0 + r;
        const bool q_ok = q < N;
        route_epilogue<SMAX>(tR, m, s, q, q_ok, E + ((size_t)bh * N + (q_ok ? q : 0)) * s,
                             cnt + (size_t)bh * N + (q_ok ? q : 0));
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (r < 32) tmem_dealloc(tmem, tmem_cols);
}

// ------------------------------------------------------------------------
// Bucketing of (query, slot) pairs by routed expert. Within an expert's
// bucket the slot-0 pairs come first (they also attend to the shared slots),
// then the others; each bucket is cut into 128-row work tiles.

// counts[bh][e][cls], cls = 0 for slot 0, 1 for slots >= 1.
__global__ void k_bucket_count(const int32_t* __restrict__ E, int N, int m, int s, int* __restrict__ counts,
                               int use_smem, int* __restrict__ status) {
    extern __shared__ int hist[];
    const int bh = blockIdx.y;
    if (use_smem) {
        for (int i = threadIdx.x; i < 2 * m; i += blockDim.x) hist[i] = 0;
        __syncthreads();
    }
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q < N) {
        for (int t = 0; t < s; ++t) {
            const int e = E[((size_t)bh * N + q) * s + t];
            if (e < 0 || e >= m) {
                set_status(status, kStBounds);
                continue;
            }
            const int idx = 2 * e + (t > 0);
            if (use_smem) atomicAdd(&hist[idx], 1);
            else atomicAdd(&counts[(size_t)bh * 2 * m + idx], 1);
        }
    }
    if (use_smem) {
        __syncthreads();
        for (int i = threadIdx.x; i < 2 * m; i += blockDim.x)
            if (hist[i]) atomicAdd(&counts[(size_t)bh * 2 * m + i], hist[i]);
    }
}

// Per head: bucket offsets, scatter cursors and the head's work tiles
// (x = head, y = expert, z = first bucket row, w = rows | shared_rows << 8).
__global__ void __launch_bounds__(512) k_bucket_scan(const int* __restrict__ counts, int m, int Ns,
                                                     int* __restrict__ cursors, int* __restrict__ toff,
                                                     int* __restrict__ tile_ctr, int4* __restrict__ tiles) {
    __shared__ int tmp[33];
    __shared__ int sh_base;
    const int bh = blockIdx.x;
    const int* c = counts + (size_t)bh * 2 * m;
    int run_off = 0, run_t = 0;
    for (int e0 = 0; e0 < m; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int c0 = e < m ? c[2 * e] : 0, c1 = e < m ? c[2 * e + 1] : 0;
        const int n = c0 + c1, nt = (n + kT - 1) / kT;
        int tot_n, tot_t;
        const int off = block_excl_scan(n, tmp, &tot_n);
        const int to = block_excl_scan(nt, tmp, &tot_t);
        if (e < m) {
            cursors[((size_t)bh * m + e) * 2] = run_off + off;
            cursors[((size_t)bh * m + e) * 2 + 1] = run_off + off + c0;
            toff[(size_t)bh * m + e] = run_t + to;
        }
        run_off += tot_n;
        run_t += tot_t;
    }
    if (threadIdx.x == 0) sh_base = atomicAdd(tile_ctr, run_t);
    __syncthreads();
    const int base = sh_base;
    for (int e = threadIdx.x; e < m; e += blockDim.x) {
        const int c0 = c[2 * e], n = c0 + c[2 * e + 1];
        const int start = cursors[((size_t)bh * m + e) * 2];
        const int t0 = base + toff[(size_t)bh * m + e];
        for (int i = 0; i * kT < n; ++i) {
            const int rows = min(kT, n - i * kT);
            const int shr = max(0, min(rows, c0 - i * kT));
            tiles[t0 + i] = make_int4(bh, e, start + i * kT, rows | (shr << 8));
        }
    }
    (void)Ns;
}

// perm[bh][pos] = q << 3 | slot, at the pair's place in its expert's bucket.
__global__ void k_bucket_scatter(const int32_t* __restrict__ E, int N, int m, int s, int* __restrict__ cursors,
                                 int32_t* __restrict__ perm) {
    const int bh = blockIdx.y;
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= N) return;
    for (int t = 0; t < s; ++t) {
        const int e = E[((size_t)bh * N + q) * s + t];
        if (e < 0 || e >= m) continue;
        const int pos = atomicAdd(&cursors[((size_t)bh * m + e) * 2 + (t > 0)], 1);
        perm[(size_t)bh * N * s + pos] = (q << 3) | t;
    }
}

// ------------------------------------------------------------------------
// Expert attention, persistent over the work tiles. A tile is up to 128
// (query, slot) pairs routed to one expert e: their queries are gathered into
// the A tile; the keys are the shared slots (landmark keys Qt, values Vt;
// only for slot-0 rows) followed by the k keys of I_e, 128 per chunk. Each
// row ends with a partial (normalized bf16 output, log2-sum-exp) for its
// (query, slot); the last of a query's s partials to finish merges them and
// writes the output row.
template <int D>
__global__ void __launch_bounds__(128)
    k_expert_tc(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                const __nv_bfloat16* __restrict__ V, const __nv_bfloat16* __restrict__ Qhi,
                const __nv_bfloat16* __restrict__ Vtb, const int32_t* __restrict__ I, const int32_t* __restrict__ perm,
                const int4* __restrict__ tiles, const int* __restrict__ tile_ctr, int* __restrict__ tile_next,
                __nv_bfloat16* __restrict__ O, __nv_bfloat16* __restrict__ part, float* __restrict__ lse,
                int* __restrict__ cnt, int N, int m, int m_pad, int k, int s, int shared_on, float sl,
                int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int sh_tile;
    __shared__ int rowq[kT];   // gathered query of each row (or -1)
    __shared__ int keyj[kT];   // key row index of the current chunk (or -1)
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    constexpr int TILE = kT * D * 2;
    constexpr int kKP = kp_bytes<D>();
    uint8_t* sQ = sm;
    uint8_t* sK = sm + TILE;  // K tile, then the P tile (128 x 128 bf16)
    uint8_t* sV = sK + kKP;
    const int r = threadIdx.x;
    if (r < 32) tmem_alloc(&tmem_slot, 256);
    if (r == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tS = lane_base(tmem), tO = lane_base(tmem) + 128;
    uint32_t phase = 0;
    const int ntiles = *(volatile const int*)tile_ctr;
    bool ok = true;
    for (;;) {
        if (r == 0) sh_tile = atomicAdd(tile_next, 1);
        __syncthreads();
        const int t = sh_tile;
        if (t >= ntiles) break;
        const int4 td = tiles[t];
        const int bh = td.x, e = td.y, start = td.z, rows = td.w & 255, shrows = td.w >> 8;
        const int Ns = N * s;
        int q = -1, slot = 0;
        if (r < rows) {
            const int pk = perm[(size_t)bh * Ns + start + r];
            q = pk >> 3;
            slot = pk & 7;
        }
        rowq[r] = q;
        const __nv_bfloat16* Qb = Q + (size_t)bh * N * D;
        const __nv_bfloat16* Kb = K + (size_t)bh * N * D;
        const __nv_bfloat16* Vb = V + (size_t)bh * N * D;
        __syncthreads();
        load_tile<D>(smem_u32(sQ), [&](int i) { return i < 0 ? Qb : (rowq[i] >= 0 ? Qb + (size_t)rowq[i] * D : nullptr); });
        const int nsh = (shared_on && shrows > 0) ? (m + kT - 1) / kT : 0;
        const int nex = (k + kT - 1) / kT;
        float mref = -INFINITY, l = 0.0f;
        for (int c = 0; c < nsh + nex; ++c) {
            const bool shc = c < nsh;
            int nk;
            const __nv_bfloat16 *kbase, *vbase;
            if (shc) {
                nk = min(kT, m - c * kT);
                keyj[r] = r < nk ? c * kT + r : -1;
                kbase = Qhi + (size_t)bh * m_pad * D;
                vbase = Vtb + (size_t)bh * m_pad * D;
            } else {
                const int cc = c - nsh;
                nk = min(kT, k - cc * kT);
                int j = -1;
                if (r < nk) {
                    j = I[((size_t)bh * m + e) * k + cc * kT + r];
                    if (j < 0 || j >= N) {
                        set_status(status, kStBounds);
                        j = -1;
                    }
                }
                keyj[r] = j;
                kbase = Kb;
                vbase = Vb;
            }
            __syncthreads();
            load_tile<D>(smem_u32(sK), [&](int i) { return i < 0 ? kbase : (keyj[i] >= 0 ? kbase + (size_t)keyj[i] * D : nullptr); });
            load_tile<D>(smem_u32(sV), [&](int i) { return i < 0 ? vbase : (keyj[i] >= 0 ? vbase + (size_t)keyj[i] * D : nullptr); });
            cp_async_wait_all();
            fence_proxy_async();
            __syncthreads();
            if (r == 0) {
                fence_after_sync();
                issue_qk<D>(tS, smem_u32(sQ), smem_u32(sK), false);
                mma_commit(&bar);
            }
            if (!(ok = sync_on_mma(&bar, phase, status))) break;
            const bool row_ok = q >= 0 && (!shc || r < shrows);
            CandOut none;
            none.cand = nullptr;
            chunk_softmax<D>(tS, tO, sK, nk, row_ok, sl, c == 0, mref, l, none);
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            if (r == 0) {
                fence_after_sync();
                issue_pv<D>(tO, smem_u32(sK), smem_u32(sV), c > 0);
                mma_commit(&bar);
            }
            if (!(ok = sync_on_mma(&bar, phase, status))) break;
        }
        if (!ok) break;
        // epilogue: every thread reads its TMEM lane (warp-collective), valid rows store
        const bool valid = q >= 0;
        const float inv = valid ? 1.0f / l : 0.0f;
        const size_t pr = valid ? ((size_t)bh * N + q) * s + slot : 0;
        __nv_bfloat16* dst = !valid ? nullptr : (s == 1) ? O + ((size_t)bh * N + q) * D : part + pr * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            float o[32];
            tmem_ld32(tO + c0, o);
            tmem_wait_ld();
            if (valid) {
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) pk[j >> 1] = pack_bf16(o[j] * inv, o[j + 1] * inv);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4*>(dst + c0 + 8 * u) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
        }
        if (valid && s > 1) {
            lse[pr] = mref + __log2f(l);
            __threadfence();
            const int old = atomicAdd(&cnt[(size_t)bh * N + q], 1);
            if (old == s - 1) {
                __threadfence();
                const size_t p0 = ((size_t)bh * N + q) * s;
                float L = -INFINITY;
                for (int j = 0; j < s; ++j) L = fmaxf(L, __ldcg(lse + p0 + j));
                float w[kMaxS], wsum = 0.0f;
                for (int j = 0; j < s; ++j) {
                    w[j] = exp2f(__ldcg(lse + p0 + j) - L);
                    wsum += w[j];
                }
                const float winv = 1.0f / wsum;
                __nv_bfloat16* od = O + ((size_t)bh * N + q) * D;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 8) {
                    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    for (int j = 0; j < s; ++j) {
                        const uint4 raw = __ldcg(reinterpret_cast<const uint4*>(part + (p0 + j) * D + c0));
                        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 f = __bfloat1622float2(h[u]);
                            acc[2 * u] = fmaf(w[j], f.x, acc[2 * u]);
                            acc[2 * u + 1] = fmaf(w[j], f.y, acc[2 * u + 1]);
                        }
                    }
                    *reinterpret_cast<uint4*>(od + c0) =
                        make_uint4(pack_bf16(acc[0] * winv, acc[1] * winv), pack_bf16(acc[2] * winv, acc[3] * winv),
                                   pack_bf16(acc[4] * winv, acc[5] * winv), pack_bf16(acc[6] * winv, acc[7] * winv));
                }
            }
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (r < 32) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ host

static int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

TcPlan tc_plan(const Dims& D) {
    TcPlan p;
    p.m_pad = (D.m + kT - 1) / kT * kT;
    p.m_tiles = p.m_pad / kT;
    const int nchunks = (D.N + kT - 1) / kT;
    const long long target = 4LL * 148;
    long long sp = (target + (long long)D.BH * p.m_tiles - 1) / ((long long)D.BH * p.m_tiles);
    if (sp < 1) sp = 1;
    if (sp > nchunks) sp = nchunks;
    p.chunks_per_split = (int)((nchunks + sp - 1) / sp);
    p.splits = (nchunks + p.chunks_per_split - 1) / p.chunks_per_split;
    p.max_tiles = (long long)D.BH * ((long long)D.N * D.s / kT + D.m + 1);
    int cols = 32;
    const int want = p.m_pad <= 256 ? 2 * p.m_pad : p.m_pad;
    while (cols < want) cols <<= 1;
    p.route_cols = cols;
    // sample stride ~ sqrt(N / 2k) balances the sample pass against the
    // candidates it lets through (about R * k per row); n_samp >= k always
    int R = (int)sqrt((double)D.N / (2.0 * D.k));
    if (R > D.N / D.k) R = D.N / D.k;
    if (R > 32) R = 32;
    if (R < 1) R = 1;
    p.R = R;
    p.n_samp = (D.N + R - 1) / R;
    p.cand_cap = (long long)p.chunks_per_split * kT;
    return p;
}

bool tc_supported(const Dims& D) {
    return D.dtype == 1 && (D.d == 64 || D.d == 128) && D.m <= 512 && D.N <= (1 << 20);
}

template <typename F>
static cudaError_t set_smem(F* f, int bytes) {
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DD, int SMAX>
static cudaError_t launch_route_s(const Dims& D, const TcPlan& P, const TcWork& W, const __nv_bfloat16* q,
                                  int32_t* E, int* status, cudaStream_t st) {
    cudaError_t e;
    const int tile = kT * DD * 2;
    if (P.m_pad <= 256) {
        const int smem = 2 * P.m_pad * DD * 2 + 2 * tile + 1024;
        if ((e = set_smem(k_route_tc<DD, SMAX>, smem))) return e;
        const int tph = (D.N + kT - 1) / kT;
        const int total = tph * D.BH;
        const int grid = std::min(total, num_sms());
        k_route_tc<DD, SMAX><<<grid, 128, smem, st>>>(q, W.Qhi, W.Qlo, D.N, D.m, P.m_pad, D.s, tph, total,
                                                      (uint32_t)P.route_cols, E, W.cnt, status);
    } else {
        const int smem = std::max(3 * tile, 100 * 1024) + 1024;
        if ((e = set_smem(k_route_chunked_tc<DD, SMAX>, smem))) return e;
        dim3 grid((D.N + kT - 1) / kT, D.BH);
        k_route_chunked_tc<DD, SMAX><<<grid, 128, smem, st>>>(q, W.Qhi, W.Qlo, D.N, D.m, P.m_pad, D.s,
                                                              (uint32_t)P.route_cols, E, W.cnt, status);
    }
    if ((e = cudaGetLastError())) return e;
    count_launch();
    return cudaSuccess;
}

template <int DD>
static cudaError_t launch_route(const Dims& D, const TcPlan& P, const TcWork& W, const __nv_bfloat16* q, int32_t* E,
                                int* status, cudaStream_t st) {
    if (D.s <= 1) return launch_route_s<DD, 1>(D, P, W, q, E, status, st);
    if (D.s <= 2) return launch_route_s<DD, 2>(D, P, W, q, E, status, st);
    if (D.s <= 4) return launch_route_s<DD, 4>(D, P, W, q, E, status, st);
    return launch_route_s<DD, 8>(D, P, W, q, E, status, st);
}

template <int DD>
static cudaError_t forward_tc_t(const Dims& D, const TcPlan& P, const TcWork& W, const void* Q, const void* K,
                                const void* V, void* O, float* Vt, int32_t* I, int32_t* E, int* status, int upto,
                                cudaStream_t st) {
    const __nv_bfloat16* q = (const __nv_bfloat16*)Q;
    const __nv_bfloat16* kk = (const __nv_bfloat16*)K;
    const __nv_bfloat16* v = (const __nv_bfloat16*)V;
    const float sl = D.scale * 1.4426950408889634f;
    const int tile = kT * DD * 2;
    cudaError_t e;
    // top-k threshold from a strided sample of the keys
    prof_mark(st, "topk_sample");
    {
        const int smem = std::max(3 * tile, 100 * 1024) + 1024;
        if ((e = set_smem(k_sample_tc<DD>, smem))) return e;
        const int cpc = 4;
        const int groups = (P.n_samp + cpc * kT - 1) / (cpc * kT);
        k_sample_tc<DD><<<dim3(P.m_tiles, groups, D.BH), 128, smem, st>>>(kk, W.Qhi, W.Qlo, W.Ssamp, D.N, D.m,
                                                                         P.m_pad, P.R, P.n_samp, cpc, status);
        if ((e = cudaGetLastError())) return e;
        count_launch();
        if ((e = launch_sample_threshold(W.Ssamp, (long long)D.BH * D.m, P.n_samp, D.k, W.thr, st))) return e;
    }
    // landmark pass: top-k candidates and the shared-expert partials
    prof_mark(st, "landmark");
    {
        const int smem = std::max(3 * tile + kp_bytes<DD>(), 100 * 1024) + 1024;
        if ((e = set_smem(k_landmark_tc<DD>, smem))) return e;
        dim3 grid(P.m_tiles, P.splits, D.BH);
        k_landmark_tc<DD><<<grid, 128, smem, st>>>(kk, v, W.Qhi, W.Qlo, W.thr, W.cand, W.ccount, W.Opart, W.ML, D.N,
                                                  D.m, P.m_pad, P.splits, P.chunks_per_split, sl, status);
        if ((e = cudaGetLastError())) return e;
        count_launch();
    }
    prof_mark(st, "topk_select");
    if ((e = launch_topk_cand(W.cand, W.ccount, P.splits, P.cand_cap, D.BH, D.m, P.m_pad, D.N, D.k, I, status, st)))
        return e;
    if (upto >= 2) {
        prof_mark(st, "vt_combine");
        count_launch();
        k_vt_combine<<<dim3(P.m_pad, D.BH), DD, 0, st>>>(W.Opart, W.ML, P.splits, D.m, P.m_pad, DD, Vt, W.Vtb);
        if ((e = cudaGetLastError())) return e;
    }
    if (!E) return cudaSuccess;
    // routing
    prof_mark(st, "route");
    if ((e = launch_route<DD>(D, P, W, q, E, status, st))) return e;
    if (upto < 2) return cudaSuccess;
    // bucketing
    prof_mark(st, "bucket");
    if ((e = cudaMemsetAsync(W.zero_begin, 0, W.zero_bytes, st))) return e;
    {
        const int use_smem = D.m <= 4096;
        dim3 grid((D.N + 255) / 256, D.BH);
        k_bucket_count<<<grid, 256, use_smem ? 8 * D.m : 0, st>>>(E, D.N, D.m, D.s, W.counts, use_smem, status);
        k_bucket_scan<<<D.BH, 512, 0, st>>>(W.counts, D.m, D.N * D.s, W.cursors, W.toff, W.tile_ctr, W.tiles);
        k_bucket_scatter<<<grid, 256, 0, st>>>(E, D.N, D.m, D.s, W.cursors, W.perm);
        if ((e = cudaGetLastError())) return e;
        count_launch(3);
    }
    // expert attention + merge
    prof_mark(st, "expert");
    {
        const int smem = std::max(2 * tile + kp_bytes<DD>(), 100 * 1024) + 1024;
        if ((e = set_smem(k_expert_tc<DD>, smem))) return e;
        k_expert_tc<DD><<<2 * num_sms(), 128, smem, st>>>(q, kk, v, W.Qhi, W.Vtb, I, W.perm, W.tiles, W.tile_ctr,
                                                          W.tile_ctr + 1, (__nv_bfloat16*)O, W.part, W.lse, W.cnt,
                                                          D.N, D.m, P.m_pad, D.k, D.s, D.shared ? 1 : 0, sl, status);
        if ((e = cudaGetLastError())) return e;
        count_launch();
    }
    return cudaSuccess;
}

cudaError_t launch_forward_tc(const Dims& D, const TcPlan& P, const TcWork& W, const void* Q, const void* K,
                              const void* V, void* O, float* Vt, int32_t* I, int32_t* E, int* status, int upto,
                              cudaStream_t st) {
    return D.d == 64 ? forward_tc_t<64>(D, P, W, Q, K, V, O, Vt, I, E, status, upto, st)
                     : forward_tc_t<128>(D, P, W, Q, K, V, O, Vt, I, E, status, upto, st);
}

}  // namespace mita
