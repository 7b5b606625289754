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
#include <cuda.h>

#include "internal.h"
#include "tc.cuh"

namespace mita {
using namespace tc;


namespace {

constexpr int kT = 128;                     // rows per tile = keys per chunk
constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 0);  // S[128 x 128] = A[128 x d] B[128 x d]^T

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem) { return tmem + ((threadIdx.x & 96u) << 16); }

// One warp's epilogue staging area: 16 rows of PPR 16-byte pieces
// (a warpgroup's half of a partial row, PPR = 8 at d = 128, 4 at d = 64);
// piece u of row r sits at u ^ ((r / (8 / PPR)) % PPR), which keeps both the
// row-wise writes and the piece-wise reads free of bank conflicts.
constexpr int kStageWarp = 16 * 128;
template <int PPR>
__device__ __forceinline__ uint32_t stage_off(int r, int u) {
    return (r * PPR + (u ^ ((r / (8 / PPR)) & (PPR - 1)))) << 4;
}



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

// Wait budgets in SM clock cycles: about one second normally; about one
// millisecond for a launch that injects a stall (the fault tests).
constexpr long long kSpin = 2LL << 30, kSpinTest = 1LL << 21;

// Bounded wait used by the warp-specialized kernels: gives up when another
// role has set the abort flag, or after `lim` cycles (then sets the device
// status and the abort flag itself).
__device__ __forceinline__ bool ws_wait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort_flag,
                                        long long lim = kSpin) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > lim) {
            set_status(status, kStTimeout);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// Waits (bounded, ignoring the abort flag) for work this CTA has already
// issued to the asynchronous units (MMAs, TMA loads) to land, so that the
// CTA never frees TMEM or exits under them, also after an abort.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* status) {
    (void)mbar_wait(bar, parity, status);
}

// Named barrier over `nthreads` threads (a multiple of 32) of the CTA; the
// calling warp reconverges first.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    __syncwarp();
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
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

// Issues O (+)= P * V with P (128 x 128 bf16) in TMEM at column tP (eight
// columns per 16 keys) and V an MN-major 128 keys x D tile in shared memory.
template <int D>
__device__ __forceinline__ void issue_pv_ts(uint32_t tO, uint32_t tP, uint32_t sV, bool accumulate) {
    constexpr uint32_t id = idesc_bf16(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
        mma_bf16_ts(tO, tP + kk * 8, sdesc(sV + kk * 2048, kT * 128, 1024), id, (kk > 0 || accumulate) ? 1u : 0u);
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

// Keeps the SMAX largest keys seen so far, ordered by key descending and, for
// equal keys, index ascending (ties to the lower index). The comparison holds
// for the entry being inserted and for every entry it displaces down the list
// (a displaced entry can have a lower index than an equal key behind it).
// Empty slots are key 0, index -1 (every real key is > 0).
template <int SMAX>
__device__ __forceinline__ void top_insert(uint32_t (&bu)[SMAX], int (&bi)[SMAX], uint32_t u, int i) {
#pragma unroll
    for (int t = 0; t < SMAX; ++t) {
        const bool gt = u > bu[t] || (u == bu[t] && (uint32_t)i < (uint32_t)bi[t]);
        const uint32_t tu = bu[t];
        const int ti = bi[t];
        bu[t] = gt ? u : tu;
        bi[t] = gt ? i : ti;
        u = gt ? tu : u;
        i = gt ? ti : i;
    }
}

// Stores (score bits, key) at base[n] if pass, and counts it: a predicated
// store, so that a sparse stream of passing scores costs no branches.
__device__ __forceinline__ void emit_cand(int2* base, int& n, float score, int key, bool pass) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %3, 0;\n\t"
        "@p st.global.v2.b32 [%0], {%1, %2};\n\t}" ::"l"(base + n),
        "r"(__float_as_int(score)), "r"(key), "r"((uint32_t)pass)
        : "memory");
    n += pass ? 1 : 0;
}

// Largest of three (the three-input max.f32 of sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Largest of 64 values: a tree of three-input maxima (four levels).
__device__ __forceinline__ float max64(const float (&v)[64]) {
    float t[22];
#pragma unroll
    for (int j = 0; j < 21; ++j) t[j] = fmax3(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
    t[21] = v[63];
    float u[8];
#pragma unroll
    for (int j = 0; j < 7; ++j) u[j] = fmax3(t[3 * j], t[3 * j + 1], t[3 * j + 2]);
    u[7] = t[21];
    return fmax3(fmax3(u[0], u[1], u[2]), fmax3(u[3], u[4], u[5]), fmaxf(u[6], u[7]));
}

// Lowest j with v[j] == x, 64 if there is none (a tree of minima).
__device__ __forceinline__ int first_eq64(const float (&v)[64], float x) {
    int c[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) c[j] = v[2 * j] == x ? 2 * j : (v[2 * j + 1] == x ? 2 * j + 1 : 64);
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
        for (int j = 0; j < h; ++j) c[j] = min(c[j], c[j + h]);
    return c[0];
}

}  // namespace

// Sample pass of the top-k selection: raw scores of each landmark row against
// a sample of the keys (runs of 16 consecutive keys, one run every 16R keys;
// n_samp slots, those past the last key scored -inf), same MMA sequence as
// the landmark pass.
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
        // sample t is key (t / 16) * 16R + t % 16: runs of 16 consecutive keys
        load_tile<D>(smem_u32(sK), [&](int t) {
            if (t < 0) return Kb;
            const int u = t0 + t;
            const long long j = (long long)(u >> 4) * 16 * R + (u & 15);
            return (t < nk && j < N) ? Kb + (size_t)j * D : (const __nv_bfloat16*)nullptr;
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
            if (row < m) {
                const int u0 = t0 + c0;
                const long long last = (long long)((u0 + 31) >> 4) * 16 * R + ((u0 + 31) & 15);
                if (c0 + 32 <= nk && last < N) {  // all 32 slots real keys: eight 16-byte stores
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                } else {
                    for (int j = 0; j < 32 && c0 + j < nk; ++j) {
                        const int u = u0 + j;
                        const long long key = (long long)(u >> 4) * 16 * R + (u & 15);
                        dst[c0 + j] = key < N ? v[j] : -INFINITY;  // slots past the last key rank last
                    }
                }
            }
        }
        fence_before_sync();
        __syncthreads();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (r < 32) tmem_dealloc(tmem, 128);
}

// Landmark pass, warp-specialized: per (landmark tile, key split, head).
//   warps 0-7  two softmax warpgroups, one per half of each 128-key chunk
//              (thread <-> TMEM lane = landmark row); they emit the top-k
//              candidates of their columns and share the row max / sum
//   warp 8     producer: the landmark tile (hi, lo) once, then TMA bulk
//              loads of consecutive K and V chunks into an NS-stage ring
//   warp 9     MMA issuer: S = Qhi K^T + Qlo K^T (bf16 split of fp32 Qt) into
//              one of two TMEM buffers, O += P V with P written over S in TMEM
// Candidate records of column half w go to region (row, split, w), whose
// capacity is that half's key count (chunks_per_split * 64).
template <int D, int NS>
__global__ void __launch_bounds__(320, 1)
    k_landmark_ws(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __nv_bfloat16* __restrict__ Qhi, const __nv_bfloat16* __restrict__ Qlo,
                  const float* __restrict__ thr, int2* __restrict__ cand, int* __restrict__ ccount,
                  float* __restrict__ Opart, float2* __restrict__ ML, int N, int m, int m_pad, int splits,
                  int chunks_per_split, float sl, int causal, int stall, int* __restrict__ status) {
    constexpr int TILE = kT * D * 2;
    constexpr int DH = D / 2;
    constexpr uint32_t kS0 = 0, kO = 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sHi = sm;
    uint8_t* sLo = sm + TILE;
    uint8_t* sK = sm + 2 * TILE;   // NS stages
    uint8_t* sV = sK + NS * TILE;  // NS stages
    // a stage's keys and values are released separately: K(c) once S(c) is
    // done, V(c) once O += P V of c is, so the next keys load while the
    // softmax of c still runs
    __shared__ uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full[2], xbar[2];
    __shared__ uint64_t pv_done, o_full, q_bar, ebar, drain;
    __shared__ float xmax[2][2][kT], xl[2][kT];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;
    const long long lim = stall ? kSpinTest : kSpin;
    const int mt = blockIdx.x, sp = blockIdx.y, bh = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j_begin = sp * chunks_per_split * kT;
    const int j_end = min(N, j_begin + chunks_per_split * kT);
    const int nc = (j_end - j_begin + kT - 1) / kT;  // >= 1 by the host's split sizing
    if (warp == 9) tmem_alloc(&tmem_slot, 512);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 8);
            mbar_init(&xbar[i], 8);
        }
        mbar_init(&pv_done, 1);
        mbar_init(&o_full, 1);
        mbar_init(&q_bar, 32);
        mbar_init(&ebar, 8);
        mbar_init(&drain, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    if (warp == 8) {
        // ------------------------------------------------------- producer
        // fault test: the first CTA never loads its first chunk, so the MMA
        // warp's bounded wait for it runs out
        const int skip = (stall && mt == 0 && sp == 0 && bh == 0) ? 0 : -1;
        if (lane == 0 && skip != 0) {
            // the first keys go out before the landmark tiles: their HBM latency
            // overlaps the tiles' copies (the stage is free: its first use)
            mbar_expect_tx(&k_full[0], TILE);
#pragma unroll
            for (int cb = 0; cb < D / 64; ++cb)
                tma_load_2d(smem_u32(sK) + cb * kT * 128, &tmK, cb * 64, bh * N + j_begin, &k_full[0]);
        }
        {
            constexpr int CPR = D / 8, RPI = 32 / CPR;
            const int cc = lane % CPR;
            const size_t y0 = (size_t)bh * m_pad + (size_t)mt * kT;
            for (int r0 = 0; r0 < kT; r0 += RPI) {
                const int r = r0 + lane / CPR;
                cp_async16(smem_u32(sHi) + sw_off(r, cc, kT), Qhi + (y0 + r) * D + cc * 8, true);
                cp_async16(smem_u32(sLo) + sw_off(r, cc, kT), Qlo + (y0 + r) * D + cc * 8, true);
            }
            cp_async_arrive(&q_bar);
        }
        if (lane == 0) {
            // keys of chunk c go out before values of chunk c - 1: the keys' stage
            // frees first (S of c - NS completes before O += P V of c - 1 - NS)
            int issued_k = 1, issued_v = 0;  // keys of chunk 0: above
            for (int c = 0; c <= nc; ++c) {
                if (c > 0 && c < nc) {
                    const int st = c % NS, use = c / NS;
                    const int y = bh * N + j_begin + c * kT;  // rows past the split are masked, past the end read 0
                    if (!ws_wait(&k_empty[st], (use & 1) ^ 1, status, abort_v, lim)) break;
                    issued_k = c + 1;
                    if (c != skip) {
                        mbar_expect_tx(&k_full[st], TILE);
#pragma unroll
                        for (int cb = 0; cb < D / 64; ++cb)
                            tma_load_2d(smem_u32(sK + st * TILE) + cb * kT * 128, &tmK, cb * 64, y, &k_full[st]);
                    }
                }
                if (c > 0) {
                    const int cv = c - 1, st = cv % NS, use = cv / NS;
                    const int y = bh * N + j_begin + cv * kT;
                    if (!ws_wait(&v_empty[st], (use & 1) ^ 1, status, abort_v, lim)) break;
                    issued_v = cv + 1;
                    if (cv != skip) {
                        mbar_expect_tx(&v_full[st], TILE);
#pragma unroll
                        for (int cb = 0; cb < D / 64; ++cb)
                            tma_load_2d(smem_u32(sV + st * TILE) + cb * kT * 128, &tmV, cb * 64, y, &v_full[st]);
                    }
                }
            }
            // the loads still in flight (at most the last NS issued of each kind)
            // land before the CTA may exit
            for (int c = max(0, issued_k - NS); c < issued_k; ++c)
                if (c != skip) drain_wait(&k_full[c % NS], (c / NS) & 1, status);
            for (int c = max(0, issued_v - NS); c < issued_v; ++c)
                if (c != skip) drain_wait(&v_full[c % NS], (c / NS) & 1, status);
        }
        __syncwarp();
        cp_async_wait_all();
    } else if (warp == 9) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = ws_wait(&q_bar, 0, status, abort_v, lim);
            fence_proxy_async();  // the landmark tiles came through cp.async (generic proxy)
            auto flush_pv = [&](int h) -> bool {
                if (!ws_wait(&p_full[h & 1], (h >> 1) & 1, status, abort_v, lim)) return false;
                if (!ws_wait(&v_full[h % NS], (h / NS) & 1, status, abort_v, lim)) return false;
                fence_after_sync();
                issue_pv_ts<D>(tmem + kO, tmem + kS0 + (h & 1) * 128, smem_u32(sV + (h % NS) * TILE), h > 0);
                mma_commit(&pv_done);
                mma_commit(&v_empty[h % NS]);
                if (h == nc - 1) mma_commit(&o_full);
                return true;
            };
            for (int c = 0; c < nc && ok; ++c) {
                const int st = c % NS, sb = c & 1;
                if (!(ok = ws_wait(&k_full[st], (c / NS) & 1, status, abort_v, lim))) break;
                fence_after_sync();
                issue_qk<D>(tmem + kS0 + sb * 128, smem_u32(sHi), smem_u32(sK + st * TILE), false);
                issue_qk<D>(tmem + kS0 + sb * 128, smem_u32(sLo), smem_u32(sK + st * TILE), true);
                mma_commit(&s_full[sb]);
                mma_commit(&k_empty[st]);
                if (c > 0 && !(ok = flush_pv(c - 1))) break;
            }
            if (ok) flush_pv(nc - 1);
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&drain);
            drain_wait(&drain, 0, status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax + epilogue
        const int wg = warp >> 2, r = threadIdx.x & 127;
        const int row = mt * kT + r;
        const bool row_ok = row < m;
        const float th = row_ok ? thr[(size_t)bh * m + row] : 0.0f;
        // causal variant: the shared expert of landmark `row` attends to the keys
        // of its prefix, j < hi (the top-k candidates still come from every key)
        int lo_row, hi_row = N;
        if (causal && row_ok) pool_bin(row, N, m, &lo_row, &hi_row);
        const long long capw = (long long)chunks_per_split * 64;
        const size_t region = (((size_t)bh * m_pad + row) * splits + sp) * 2 + wg;
        int2* cw = cand + region * capw;
        int ncand = 0;
        float mref = -INFINITY, l = 0.0f;
        bool ok = true;
        const uint32_t tO = lane_base(tmem) + kO + wg * DH;
        const bool warp_rows = __any_sync(0xffffffffu, row_ok);  // this warp holds a real landmark row
        for (int c = 0; c < nc; ++c) {
            const int sb = c & 1, j0 = j_begin + c * kT;
            if (!__all_sync(0xffffffffu, ws_wait(&s_full[sb], (c >> 1) & 1, status, abort_v, lim))) { ok = false; break; }
            fence_after_sync();
            const uint32_t tS = lane_base(tmem) + kS0 + sb * 128;
            const int nval = row_ok ? min(kT, j_end - j0) - 64 * wg : 0;   // real keys of this half
            const int nsm = min(nval, hi_row - j0 - 64 * wg);               // ... inside the softmax
            float v[64];
            tmem_ld32(tS + 64 * wg, v);
            tmem_ld32(tS + 64 * wg + 32, v + 32);
            tmem_wait_ld();
            float mx = -INFINITY;
            if (!warp_rows) {
                // padding rows only (m not a multiple of 128): nothing to emit or weigh
            } else if (nsm >= 64 && sl > 0.0f) {  // every column real: one tree maximum
#pragma unroll
                for (int j = 0; j < 64; ++j) emit_cand(cw, ncand, v[j], j0 + 64 * wg + j, v[j] >= th);
                mx = max64(v) * sl;
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    emit_cand(cw, ncand, v[j], j0 + 64 * wg + j, j < nval && v[j] >= th);
                    mx = fmaxf(mx, j < nsm ? v[j] * sl : -INFINITY);
                }
            }
            xmax[c & 1][wg][r] = mx;
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&xbar[c & 1]);
            if (!__all_sync(0xffffffffu, ws_wait(&xbar[c & 1], (c >> 1) & 1, status, abort_v, lim))) { ok = false; break; }
            fence_after_sync();
            mx = fmaxf(mx, xmax[c & 1][wg ^ 1][r]);
            float mnew = mref, alpha = 1.0f;
            if (mx > mref + 8.0f) {
                mnew = mx;
                alpha = ex2(mref - mnew);
            }
            float sum = 0.0f;
            uint32_t pkd[32];
            if (warp_rows) {
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    const float e0 = ex2(fmaf(v[j], sl, -mnew)), e1 = ex2(fmaf(v[j + 1], sl, -mnew));
                    const float p0 = j < nsm ? e0 : 0.0f, p1 = j + 1 < nsm ? e1 : 0.0f;
                    sum += p0 + p1;
                    pkd[j >> 1] = pack_bf16(p0, p1);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) pkd[j] = 0u;
            }
            tmem_st32(tS + 32 * wg, reinterpret_cast<const float*>(pkd));
            tmem_wait_st();
            l = l * alpha + sum;
            mref = mnew;
            if (__any_sync(0xffffffffu, c > 0 && alpha != 1.0f)) {
                // S(c) done implies PV(c-2) done: this wait can only see PV(c-1)'s phase
                if (!__all_sync(0xffffffffu, ws_wait(&pv_done, (c - 1) & 1, status, abort_v, lim))) { ok = false; break; }
                fence_after_sync();
                const float a = (c > 0) ? alpha : 1.0f;
#pragma unroll 1
                for (int c0 = 0; c0 < DH; c0 += 32) {
                    float o[32];
                    tmem_ld32(tO + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= a;
                    tmem_st32(tO + c0, o);
                }
                tmem_wait_st();
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[c & 1]);
        }
        if (ok && __all_sync(0xffffffffu, ws_wait(&o_full, 0, status, abort_v, lim))) {
            fence_after_sync();
            float o[DH];
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 32) tmem_ld32(tO + c0, o + c0);
            tmem_wait_ld();
            xl[wg][r] = l;
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ebar);
            if (__all_sync(0xffffffffu, ws_wait(&ebar, 0, status, abort_v, lim))) {
                const float lt = l + xl[wg ^ 1][r];
                const size_t orow = ((size_t)bh * splits + sp) * m_pad + row;
                // this warp's 32 half rows go through the key/value stages (idle
                // once O is complete), so that each store writes whole 128-byte
                // lines: two (d = 128) or four (d = 64) half rows per instruction
                constexpr int PD = DH + 4;  // padded pitch (floats): conflict-free both ways
                constexpr int PPR = DH / 4, RPI = 32 / PPR;
                static_assert(8 * 32 * PD * 4 <= 2 * NS * TILE, "staging fits in the key/value stages");
                fence_proxy_async();  // the stages were last read by MMAs (async proxy)
                float* stg = reinterpret_cast<float*>(sK) + (size_t)warp * 32 * PD;
#pragma unroll
                for (int j = 0; j < DH; j += 4)
                    *reinterpret_cast<float4*>(stg + lane * PD + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
                __syncwarp();
                float* od = Opart + (orow - lane) * D + wg * DH;  // this warp's first row
#pragma unroll
                for (int i = 0; i < 32 / RPI; ++i) {
                    const int rl = i * RPI + lane / PPR, u = lane % PPR;
                    *reinterpret_cast<float4*>(od + (size_t)rl * D + 4 * u) =
                        *reinterpret_cast<const float4*>(stg + rl * PD + 4 * u);
                }
                if (wg == 0) ML[orow] = make_float2(mref, row_ok ? lt : 0.0f);
                ccount[region] = ncand;
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

// Merges the per-split partials: Vt = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// Writes Vt fp32 [BH][m][D] and the bf16 copy [BH][m_pad][D] (padding rows 0).
// One block per (landmark row, head): D/4 lanes of four columns times
// blockDim / (D/4) split lanes (a power of two, about the split count, so a
// few splits take a small block), each split lane summing every such split,
// then a sum over the split lanes in shared memory. The splits run in
// parallel, so a head split many ways, as few heads are, costs no longer than
// one split few ways.
template <int D>
__global__ void __launch_bounds__(256) k_vt_combine(const float* __restrict__ Opart, const float2* __restrict__ ML,
                                                    int splits, int m, int m_pad, float* __restrict__ Vt,
                                                    __nv_bfloat16* __restrict__ Vtb) {
    constexpr int CG = D / 4, SLMAX = 256 / CG;
    __shared__ float4 red[SLMAX][CG];
    __shared__ float rden[SLMAX], wmax[8];
    const int i = blockIdx.x, bh = blockIdx.y;
    const int cg = threadIdx.x % CG, sl = threadIdx.x / CG, nsl = blockDim.x / CG, nw = blockDim.x >> 5;
    __nv_bfloat162* vb = reinterpret_cast<__nv_bfloat162*>(Vtb + ((size_t)bh * m_pad + i) * D + 4 * cg);
    if (i >= m) {  // a padding row: zeros in the bf16 copy only
        if (sl == 0) vb[0] = vb[1] = __floats2bfloat162_rn(0.0f, 0.0f);
        return;
    }
    const size_t o0 = (size_t)bh * splits * m_pad + i;  // ML index of split 0; split s adds s * m_pad
    float M = -INFINITY;
    for (int s = threadIdx.x; s < splits; s += blockDim.x) M = fmaxf(M, ML[o0 + (size_t)s * m_pad].x);
#pragma unroll
    for (int x = 16; x >= 1; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = M;
    __syncthreads();
    for (int w = 0; w < nw; ++w) M = fmaxf(M, wmax[w]);
    float4 num = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float den = 0.0f;
    for (int s = sl; s < splits; s += nsl) {
        const size_t o = o0 + (size_t)s * m_pad;
        const float2 ml = ML[o];
        if (ml.y == 0.0f) continue;
        const float w = exp2f(ml.x - M);
        const float4 v = reinterpret_cast<const float4*>(Opart + o * D)[cg];
        num.x += w * v.x;
        num.y += w * v.y;
        num.z += w * v.z;
        num.w += w * v.w;
        den += w * ml.y;
    }
    red[sl][cg] = num;
    if (cg == 0) rden[sl] = den;
    __syncthreads();
    if (sl == 0) {
        float4 a = red[0][cg];
        float dd = rden[0];
        for (int j = 1; j < nsl; ++j) {
            const float4 b = red[j][cg];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
            dd += rden[j];
        }
        const float4 out = make_float4(a.x / dd, a.y / dd, a.z / dd, a.w / dd);
        float* vt = Vt + ((size_t)bh * m + i) * D + 4 * cg;  // a caller's buffer: 4-byte alignment only
        vt[0] = out.x;
        vt[1] = out.y;
        vt[2] = out.z;
        vt[3] = out.w;
        vb[0] = __floats2bfloat162_rn(out.x, out.y);
        vb[1] = __floats2bfloat162_rn(out.z, out.w);
    }
}

// ------------------------------------------------------------------------
// Routing: R = Q Qhi^T + Q Qlo^T (the bf16 split of fp32 Qt keeps routing
// scores at fp32 accuracy), then each thread keeps the s best landmarks of
// its query row (ties to the lower landmark index).

// The SMAX best landmarks of columns [c_begin, c_end) (c_begin a multiple of
// 64), descending, ties to the lower index; blocks of 64 are visited in
// increasing index order, and a block only contributes while its largest
// remaining score beats the SMAX-th best (an equal score has a higher index
// and ranks behind). Empty entries: key 0, index -1.
template <int SMAX>
__device__ __forceinline__ void route_top(uint32_t tR, int c_begin, int c_end, uint32_t (&bu)[SMAX], int (&bi)[SMAX]) {
#pragma unroll
    for (int t = 0; t < SMAX; ++t) { bu[t] = 0u; bi[t] = -1; }
    const int m = c_end;
#pragma unroll 1
    for (int c0 = c_begin; c0 < c_end; c0 += 64) {
        float v[64];
        tmem_ld32(tR + c0, v);
        tmem_ld32(tR + c0 + 32, v + 32);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = c0 + j < m ? v[j] : -INFINITY;
        float mx = max64(v);
#pragma unroll 1
        for (int u = 0; u < SMAX; ++u) {
            if (!(mx > -INFINITY) || order_key(mx) <= bu[SMAX - 1]) break;
            const int i = first_eq64(v, mx);
            top_insert<SMAX>(bu, bi, order_key(mx), c0 + i);
#pragma unroll
            for (int j = 0; j < 64; ++j) v[j] = j == i ? -INFINITY : v[j];
            mx = max64(v);
        }
    }
}

template <int SMAX>
__device__ __forceinline__ void route_epilogue(uint32_t tR, int m, int s, int q, bool q_ok, int32_t* __restrict__ Erow) {
    uint32_t bu[SMAX];
    int bi[SMAX];
    route_top<SMAX>(tR, 0, m, bu, bi);
    if (q_ok) {
#pragma unroll
        for (int t = 0; t < SMAX; ++t)
            if (t < s) Erow[t] = bi[t];
    }
}

// Persistent variant for m_pad <= 256: each CTA walks a contiguous range of
// 128-query tiles; Qt (hi, lo) of the current head stays in shared memory and
// the next query tile is loaded and multiplied while this tile's routes are
// picked (two TMEM accumulators). Two warpgroups: each thread of warpgroup h
// picks its query's best landmarks among the column blocks of half h, and
// warpgroup 0 merges the two lists.
template <int D, int SMAX>
__global__ void __launch_bounds__(256, 1)
    k_route_tc(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Qhi,
               const __nv_bfloat16* __restrict__ Qlo, int N, int m, int m_pad, int s, int tiles_per_head,
               int total_tiles, uint32_t tmem_cols, int32_t* __restrict__ E,
               int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    __shared__ uint32_t xkey[kT][SMAX];  // the second half's best, handed to the first
    __shared__ int xidx[kT][SMAX];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int QT = m_pad * D * 2;
    uint8_t* sHi = sm;
    uint8_t* sLo = sm + QT;
    uint8_t* sQb[2] = {sm + 2 * QT, sm + 2 * QT + kT * D * 2};
    const int r = threadIdx.x & (kT - 1), half = threadIdx.x >> 7;
    const int per = (total_tiles + gridDim.x - 1) / gridDim.x;
    const int t_begin = blockIdx.x * per, t_end = min(total_tiles, t_begin + per);
    if (t_begin >= t_end) return;
    if (threadIdx.x < 32) tmem_alloc(&tmem_slot, tmem_cols);
    if (threadIdx.x == 0) {
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
    if (threadIdx.x == 0) {
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
            if (threadIdx.x == 0) {
                fence_after_sync();
                issue(b ^ 1);
            }
        }
        const int bh = t / tiles_per_head, q = (t % tiles_per_head) * kT + r;
        const bool q_ok = q < N;
        // column blocks of 64 split between the halves (the second half's blocks
        // have the higher indices, so on equal scores the first half's win)
        const int nblk = (m + 63) / 64, split = ((nblk + 1) / 2) * 64;
        uint32_t bu[SMAX];
        int bi[SMAX];
        route_top<SMAX>(lane_base(tmem) + b * m_pad, half ? split : 0, half ? m : min(m, split), bu, bi);
        if (half) {
#pragma unroll
            for (int u = 0; u < SMAX; ++u) {
                xkey[r][u] = bu[u];
                xidx[r][u] = bi[u];
            }
        }
        fence_before_sync();
        __syncthreads();
        if (!half && q_ok) {
#pragma unroll
            for (int u = 0; u < SMAX; ++u)
                if (xidx[r][u] >= 0) top_insert<SMAX>(bu, bi, xkey[r][u], xidx[r][u]);
            int32_t* Erow = E + ((size_t)bh * N + q) * s;
#pragma unroll
            for (int u = 0; u < SMAX; ++u)
                if (u < s) Erow[u] = bi[u];
        }
    }
    // drain an MMA still in flight if the loop left early
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (threadIdx.x < 32) tmem_dealloc(tmem, tmem_cols);
}

// Routing + shared slots with two query tiles in flight (m_pad == 128): each
// softmax warpgroup owns every other tile of the CTA and holds whole rows (one
// query per thread), so its routing choice and its softmax over the shared
// logits need no exchange with the other warpgroup, and the two run out of
// phase: one's exponentials overlap the other's routing, epilogue stores and
// MMAs. Warpgroup w: TMEM columns 128 w (R, then P over it) and 256 + 128 w
// (the shared-slot output). The producer warp loads consecutive 128-query
// tiles by TMA (NSQ-stage ring) and the head's Qt (hi, lo) and Vt by cp.async
// when the head changes; the old landmarks are released once every older tile
// (the other warpgroup's last one) has its P Vt issued.
template <int D, int SMAX, int NSQ>
__global__ void __launch_bounds__(320, 1)
    k_route_pp(const __grid_constant__ CUtensorMap tmQ, const __nv_bfloat16* __restrict__ Qhi,
               const __nv_bfloat16* __restrict__ Qlo, const __nv_bfloat16* __restrict__ Vtb, int N, int m, int s,
               int tiles_per_head, int total_tiles, float sl, int causal, int32_t* __restrict__ E,
               __nv_bfloat16* __restrict__ sh_part, float* __restrict__ sh_lse, int* __restrict__ counts,
               int* __restrict__ status) {
    constexpr int TILE = kT * D * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sHi = sm;
    uint8_t* sLo = sm + TILE;
    uint8_t* sVt = sm + 2 * TILE;
    uint8_t* sQ = sm + 3 * TILE;        // NSQ stages
    uint8_t* sStage = sQ + NSQ * TILE;  // 8 x kStageWarp epilogue staging
    __shared__ uint64_t q_full[NSQ], q_empty[NSQ], r_full[2], p_full[2], o_full[2], o_free[2];
    __shared__ uint64_t lm_full, lm_free, drain;
    __shared__ int qgen[NSQ];  // landmark load each query tile uses (1-based)
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = (total_tiles + gridDim.x - 1) / gridDim.x;
    const int t_begin = blockIdx.x * per, t_end = min(total_tiles, t_begin + per);
    const int nloc = max(0, t_end - t_begin);
    if (nloc == 0) return;
    if (warp == 9) tmem_alloc(&tmem_slot, 512);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSQ; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&r_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_free[i], 4);
        }
        mbar_init(&lm_full, 32);
        mbar_init(&lm_free, 1);
        mbar_init(&drain, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    auto head = [&](int tl) { return (t_begin + tl) / tiles_per_head; };
    if (warp == 8) {
        // ------------------------------------------------------- producer
        constexpr int CPR = D / 8, RPI = 32 / CPR;
        const int cc = lane % CPR;
        int cur = -1, gen = 0;
        for (int tl = 0; tl < nloc; ++tl) {
            const int bh = head(tl);
            const bool reload = bh != cur;
            const int st = tl % NSQ;
            int okw = 1;
            if (lane == 0) okw = ws_wait(&q_empty[st], ((tl / NSQ) & 1) ^ 1, status, abort_v);
            if (!__shfl_sync(0xffffffffu, okw, 0)) break;
            if (lane == 0) {
                qgen[st] = gen + (reload ? 1 : 0);
                mbar_expect_tx(&q_full[st], TILE);  // also publishes qgen
                const int y = bh * N + ((t_begin + tl) % tiles_per_head) * kT;  // rows past the head: masked
#pragma unroll
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_2d(smem_u32(sQ + st * TILE) + cb * kT * 128, &tmQ, cb * 64, y, &q_full[st]);
            }
            __syncwarp();
            if (reload) {
                // every MMA on the previous head's landmarks must be done: the MMA
                // warp commits lm_free once per head it leaves (gen - 1 so far)
                if (gen > 0) {
                    okw = 1;
                    if (lane == 0) okw = ws_wait(&lm_free, (gen - 1) & 1, status, abort_v);
                    if (!__shfl_sync(0xffffffffu, okw, 0)) break;
                }
                const size_t y0 = (size_t)bh * kT;
                for (int r0 = 0; r0 < kT; r0 += RPI) {
                    const int r = r0 + lane / CPR;
                    const size_t off = (y0 + r) * D + cc * 8;
                    cp_async16(smem_u32(sHi) + sw_off(r, cc, kT), Qhi + off, true);
                    cp_async16(smem_u32(sLo) + sw_off(r, cc, kT), Qlo + off, true);
                    cp_async16(smem_u32(sVt) + sw_off(r, cc, kT), Vtb + off, true);
                }
                cp_async_arrive(&lm_full);
                ++gen;
                cur = bh;
            }
        }
        cp_async_wait_all();
    } else if (warp == 9) {
        // ------------------------------------------------------ MMA issuer
        // One thread polls without blocking. Per warpgroup w (tiles tl = 2 j + w):
        // R of tile j once its R buffer is free (P Vt of tile j - 1 issued), its
        // query tile is in and its landmarks are loaded; P Vt of tile j once its
        // probabilities are in and the epilogue of tile j - 1 has read O.
        if (lane == 0) {
            int nR[2] = {0, 0}, nP[2] = {0, 0};
            const int G[2] = {(nloc + 1) / 2, nloc / 2};
            int cur_gen = 0, rel = 0;
            long long idle0 = clock64();
            while (nP[0] < G[0] || nP[1] < G[1]) {
                bool prog = false;
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    if (nR[w] < G[w] && nR[w] == nP[w]) {
                        const int j = nR[w], tl = 2 * j + w, st = tl % NSQ;
                        if (mbar_test_wait(&q_full[st], (tl / NSQ) & 1)) {
                            const int gen = qgen[st];
                            bool ready = true;
                            if (gen == cur_gen + 1) {
                                if (cur_gen > 0 && rel < cur_gen) {
                                    // release the old landmarks once the other warpgroup's last
                                    // older tile has its P Vt issued, or waits for the new
                                    // landmarks itself (then its older tiles are all done)
                                    const int wo = w ^ 1, jo = (tl - 1) >> 1;
                                    const bool done_o = nP[wo] > jo ||
                                                        (nR[wo] == jo && nP[wo] == jo && qgen[(tl - 1) % NSQ] == gen);
                                    if (done_o) {
                                        mma_commit(&lm_free);
                                        ++rel;
                                        prog = true;
                                    } else {
                                        ready = false;
                                    }
                                }
                                if (ready) {
                                    if (mbar_test_wait(&lm_full, (gen - 1) & 1)) {
                                        cur_gen = gen;
                                        fence_proxy_async();  // landmarks came through cp.async (generic proxy)
                                        prog = true;
                                    } else {
                                        ready = false;
                                    }
                                }
                            } else if (gen != cur_gen) {
                                ready = false;  // the other warpgroup's older tile moves the landmarks first
                            }
                            if (ready) {
                                fence_after_sync();
                                issue_qk<D>(tmem + w * 128, smem_u32(sQ + st * TILE), smem_u32(sHi), false);
                                issue_qk<D>(tmem + w * 128, smem_u32(sQ + st * TILE), smem_u32(sLo), true);
                                mma_commit(&r_full[w]);
                                mma_commit(&q_empty[st]);
                                ++nR[w];
                                prog = true;
                            }
                        }
                    }
                    if (nP[w] < nR[w]) {
                        const int j = nP[w];
                        if (mbar_test_wait(&p_full[w], j & 1) && mbar_test_wait(&o_free[w], (j & 1) ^ 1)) {
                            fence_after_sync();
                            issue_pv_ts<D>(tmem + 256 + w * 128, tmem + w * 128, smem_u32(sVt), false);
                            mma_commit(&o_full[w]);
                            ++nP[w];
                            prog = true;
                        }
                    }
                }
                if (prog) {
                    idle0 = clock64();
                } else {
                    if (*abort_v) break;
                    if (clock64() - idle0 > kSpin) {
                        set_status(status, kStTimeout);
                        *abort_v = 1;
                        break;
                    }
                }
            }
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&drain);
            drain_wait(&drain, 0, status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax + epilogue
        const int w = warp >> 2, r = threadIdx.x & 127;
        uint8_t* stage = sStage + warp * kStageWarp;
        const uint32_t tR = lane_base(tmem) + w * 128, tO = lane_base(tmem) + 256 + w * 128;
        for (int j = 0;; ++j) {
            const int tl = 2 * j + w;
            if (tl >= nloc) break;
            const int bh = head(tl), q0 = ((t_begin + tl) % tiles_per_head) * kT, q = q0 + r;
            const bool q_ok = q < N;
            if (!__all_sync(0xffffffffu, ws_wait(&r_full[w], j & 1, status, abort_v))) break;
            fence_after_sync();
            // causal variant: the shared slots are the landmarks whose bin is
            // complete at query q (a prefix of the landmarks); routing still
            // ranks all of them
            const int nsm = causal ? min(m, landmarks_complete(q_ok ? q : N - 1, N, m)) : m;
            // pass 1, 64 columns at a time: the s best landmarks (ties to the lower
            // index) and the largest shared-slot logit
            uint32_t bu[SMAX];
            int bi[SMAX];
#pragma unroll
            for (int u = 0; u < SMAX; ++u) {
                bu[u] = 0u;
                bi[u] = -1;
            }
            float mx = -INFINITY;
            [[maybe_unused]] float bv[SMAX];  // SMAX <= 2: the best scores so far, with bi
            if constexpr (SMAX <= 2) {
#pragma unroll
                for (int u = 0; u < SMAX; ++u) bv[u] = -INFINITY;
            }
#pragma unroll 1
            for (int c0 = 0; c0 < m; c0 += 64) {  // blocks past the last landmark hold nothing
                float v[64];
                tmem_ld32(tR + c0, v);
                tmem_ld32(tR + c0 + 32, v + 32);
                tmem_wait_ld();
                if (m < c0 + 64) {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj) v[jj] = c0 + jj < m ? v[jj] : -INFINITY;
                }
                float bmx = max64(v);
                if (sl > 0.0f && nsm >= min(m, c0 + 64)) {
                    mx = fmaxf(mx, bmx * sl);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj) mx = fmaxf(mx, c0 + jj < nsm ? v[jj] * sl : -INFINITY);
                }
                if constexpr (SMAX <= 2) {
                    // one pass over the block keeping its SMAX best in column order
                    // (a strict comparison keeps the lower column among equal
                    // scores), then merged into the row's best by (score, lower
                    // column); one chain measured faster than interleaved ones
                    constexpr int NCH = 1;  // chains
                    float a[NCH][SMAX];
                    int ai[NCH][SMAX];
#pragma unroll
                    for (int h = 0; h < NCH; ++h)
#pragma unroll
                        for (int u = 0; u < SMAX; ++u) {
                            a[h][u] = -INFINITY;
                            ai[h][u] = -1;
                        }
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj) {
                        const int h = jj % NCH;
                        const float x = v[jj];
                        const bool p1 = x > a[h][0];
                        if constexpr (SMAX == 2) {
                            const bool p2 = x > a[h][1];
                            a[h][1] = p1 ? a[h][0] : (p2 ? x : a[h][1]);
                            ai[h][1] = p1 ? ai[h][0] : (p2 ? jj : ai[h][1]);
                        }
                        a[h][0] = p1 ? x : a[h][0];
                        ai[h][0] = p1 ? jj : ai[h][0];  // the block's column; c0 added below
                    }
#pragma unroll
                    for (int h = 0; h < NCH; ++h)
#pragma unroll
                        for (int u = 0; u < SMAX; ++u) {
                            float x = a[h][u];
                            int xi = ai[h][u] >= 0 ? c0 + ai[h][u] : -1;
#pragma unroll
                            for (int t = 0; t < SMAX; ++t) {
                                const bool gt = xi >= 0 && (x > bv[t] || (x == bv[t] && (uint32_t)xi < (uint32_t)bi[t]));
                                const float tv = bv[t];
                                const int ti = bi[t];
                                bv[t] = gt ? x : tv;
                                bi[t] = gt ? xi : ti;
                                x = gt ? tv : x;
                                xi = gt ? ti : xi;
                            }
                        }
                } else {
#pragma unroll 1
                    for (int u = 0; u < SMAX; ++u) {
                        if (!(bmx > -INFINITY) || order_key(bmx) <= bu[SMAX - 1]) break;
                        const int i = first_eq64(v, bmx);
                        top_insert<SMAX>(bu, bi, order_key(bmx), c0 + i);
#pragma unroll
                        for (int jj = 0; jj < 64; ++jj) v[jj] = jj == i ? -INFINITY : v[jj];
                        bmx = max64(v);
                    }
                }
            }
            // pass 2: the probabilities, P of keys 0..63 over columns 0..31 (scores
            // read), then of keys 64..127 over columns 32..63
            float l = 0.0f;
#pragma unroll 1
            for (int c0 = 0; c0 < kT; c0 += 64) {
                float v[64];
                tmem_ld32(tR + c0, v);
                tmem_ld32(tR + c0 + 32, v + 32);
                tmem_wait_ld();
                float s0 = 0.0f, s1 = 0.0f;
                uint32_t pkd[32];
#pragma unroll
                for (int jj = 0; jj < 64; jj += 2) {
                    const float e0 = ex2(fmaf(v[jj], sl, -mx)), e1 = ex2(fmaf(v[jj + 1], sl, -mx));
                    const float p0 = c0 + jj < nsm ? e0 : 0.0f, p1 = c0 + jj + 1 < nsm ? e1 : 0.0f;
                    if (jj & 2) s1 += p0 + p1;
                    else s0 += p0 + p1;
                    pkd[jj >> 1] = pack_bf16(p0, p1);
                }
                l += s0 + s1;
                tmem_st32(tR + (c0 >> 1), reinterpret_cast<const float*>(pkd));
            }
            tmem_wait_st();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[w]);
            if (q_ok) {
                int32_t* Erow = E + ((size_t)bh * N + q) * s;
#pragma unroll
                for (int u = 0; u < SMAX; ++u)
                    if (u < s) {
                        Erow[u] = bi[u];
                        // the bucketing's per-(head, expert, slot 0 / later) counts
                        if (bi[u] < 0 || bi[u] >= m) set_status(status, kStBounds);
                        else atomicAdd(counts + ((size_t)bh * m + bi[u]) * 2 + (u > 0), 1);
                    }
            }
            // epilogue: the normalized shared-slot partial row and its log2-sum-exp
            if (!__all_sync(0xffffffffu, ws_wait(&o_full[w], j & 1, status, abort_v))) break;
            fence_after_sync();
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;  // no slot (causal only): zero partial
            const size_t row0 = (size_t)bh * N + q0 + (r & ~31);  // this warp's first row
            constexpr int PPR = 8, RPS = 32 / PPR;  // 16-byte pieces per 64-column half row, rows per store
            // O in halves of 64 columns (registers); the next P Vt of this warpgroup
            // waits for o_free, but it also needs this warpgroup's next P, which
            // comes after this epilogue anyway
#pragma unroll 1
            for (int hh = 0; hh < D / 64; ++hh) {
                float o[64];
                tmem_ld32(tO + 64 * hh, o);
                tmem_ld32(tO + 64 * hh + 32, o + 32);
                tmem_wait_ld();
                if (hh == D / 64 - 1) {
                    fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&o_free[w]);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // lanes 16h .. 16h + 15 stage their rows
                    if ((lane >> 4) == h) {
#pragma unroll
                        for (int u = 0; u < PPR; ++u) {
                            const float* x = o + 8 * u;
                            *reinterpret_cast<uint4*>(stage + stage_off<PPR>(lane & 15, u)) =
                                make_uint4(pack_bf16(x[0] * inv, x[1] * inv), pack_bf16(x[2] * inv, x[3] * inv),
                                           pack_bf16(x[4] * inv, x[5] * inv), pack_bf16(x[6] * inv, x[7] * inv));
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 16 / RPS; ++i) {
                        const int rl = 16 * h + i * RPS + lane / PPR, u = lane % PPR;
                        const uint4 w4 = *reinterpret_cast<const uint4*>(stage + stage_off<PPR>(rl - 16 * h, u));
                        if (q0 + (r & ~31) + rl < N)
                            *reinterpret_cast<uint4*>(sh_part + (row0 + rl) * D + 64 * hh + 8 * u) = w4;
                    }
                    __syncwarp();
                }
            }
            if (q_ok) sh_lse[(size_t)bh * N + q] = l > 0.0f ? mx + __log2f(l) : -INFINITY;
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

// Variant for m_pad > 256: one CTA per 128-query tile, landmarks streamed in
// 128-row chunks into consecutive TMEM column blocks.
template <int D, int SMAX>
__global__ void __launch_bounds__(128)
    k_route_chunked_tc(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Qhi,
                       const __nv_bfloat16* __restrict__ Qlo, int N, int m, int m_pad, int s, uint32_t tmem_cols,
                       int32_t* __restrict__ E, int* __restrict__ status) {
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
        route_epilogue<SMAX>(tR, m, s, q, q_ok, E + ((size_t)bh * N + (q_ok ? q : 0)) * s);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (r < 32) tmem_dealloc(tmem, tmem_cols);
}

// ------------------------------------------------------------------------
// Bucketing of (query, slot) pairs by routed expert. Within an expert's
// bucket the slot-0 pairs come first, then the others (a fixed order, so the
// work tiles are the same from run to run); each bucket is cut into 128-row
// work tiles.

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
// (x = head, y = expert, z = first bucket row, w = rows | slot_0_rows << 8).
// xtl[bh * m + e] = (first tile, tile count) of each expert's bucket.
__global__ void __launch_bounds__(512) k_bucket_scan(const int* __restrict__ counts, int m, int Ns,
                                                     int* __restrict__ cursors, int* __restrict__ toff,
                                                     int* __restrict__ tile_ctr, int4* __restrict__ tiles,
                                                     int2* __restrict__ xtl) {
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
        xtl[(size_t)bh * m + e] = make_int2(t0, (n + kT - 1) / kT);
        for (int i = 0; i * kT < n; ++i) {
            const int rows = min(kT, n - i * kT);
            const int shr = max(0, min(rows, c0 - i * kT));
            tiles[t0 + i] = make_int4(bh, e, start + i * kT, rows | (shr << 8));
        }
    }
    (void)Ns;
}

// perm[bh][pos] = q << 3 | slot, at the pair's place in its expert's bucket.
// With use_smem, a block first ranks its pairs per (expert, class) bin in
// shared memory, then reserves each non-empty bin's range with one global
// atomic, instead of one contended global atomic per pair.
__global__ void k_bucket_scatter(const int32_t* __restrict__ E, int N, int m, int s, int* __restrict__ cursors,
                                 int32_t* __restrict__ perm, int use_smem) {
    extern __shared__ int bins[];  // 2m local counts, then the bins' global bases
    const int bh = blockIdx.y;
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    int* cur = cursors + (size_t)bh * m * 2;
    if (!use_smem) {
        if (q >= N) return;
        for (int t = 0; t < s; ++t) {
            const int e = E[((size_t)bh * N + q) * s + t];
            if (e < 0 || e >= m) continue;
            const int pos = atomicAdd(&cur[e * 2 + (t > 0)], 1);
            perm[(size_t)bh * N * s + pos] = (q << 3) | t;
        }
        return;
    }
    for (int i = threadIdx.x; i < 2 * m; i += blockDim.x) bins[i] = 0;
    __syncthreads();
    int bin[kMaxS], rank[kMaxS];
#pragma unroll
    for (int t = 0; t < kMaxS; ++t) {
        bin[t] = -1;
        if (t < s && q < N) {
            const int e = E[((size_t)bh * N + q) * s + t];
            if (e >= 0 && e < m) {
                bin[t] = e * 2 + (t > 0);
                rank[t] = atomicAdd(&bins[bin[t]], 1);
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 2 * m; i += blockDim.x) {
        const int c = bins[i];
        bins[i] = c ? atomicAdd(&cur[i], c) : 0;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kMaxS; ++t)
        if (bin[t] >= 0) perm[(size_t)bh * N * s + bins[bin[t]] + rank[t]] = (q << 3) | t;
}

// Output rows from the partials: each query's ne expert partials (normalized
// bf16 rows with their log2-sum-exp; the s routed slots times their
// sub-experts) and its ns shared-slot partials, weighted by 2^(lse - max): the
// softmax over the union of the partials' keys. One thread per 8 columns of a
// query; the partials come in groups of four, all loads of a group in flight
// at once, with an online rescale when a later group raises the maximum.
template <int D>
__global__ void __launch_bounds__(256) k_merge(const __nv_bfloat16* __restrict__ part, const float* __restrict__ lse,
                                               int ne, const __nv_bfloat16* __restrict__ sh_part,
                                               const float* __restrict__ sh_lse, int ns, __nv_bfloat16* __restrict__ O,
                                               long long nq) {
    constexpr int G = D / 8;   // threads per query
    constexpr int kGrp = 4;    // partials per group
    const long long qi = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / G;
    const int gcol = (threadIdx.x % G) * 8;
    if (qi >= nq) return;
    float L = -INFINITY, wsum = 0.0f;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j0 = 0; j0 < ne + ns; j0 += kGrp) {
        uint4 raw[kGrp];
        float lj[kGrp];
#pragma unroll
        for (int j = 0; j < kGrp; ++j) {
            const int t = j0 + j;
            lj[j] = -INFINITY;
            if (t < ne) {
                lj[j] = lse[qi * ne + t];
                raw[j] = *reinterpret_cast<const uint4*>(part + (qi * ne + t) * D + gcol);
            } else if (t < ne + ns) {
                lj[j] = sh_lse[qi * ns + (t - ne)];
                raw[j] = *reinterpret_cast<const uint4*>(sh_part + (qi * ns + (t - ne)) * D + gcol);
            }
        }
        float gm = lj[0];
#pragma unroll
        for (int j = 1; j < kGrp; ++j) gm = fmaxf(gm, lj[j]);
        if (gm > L) {  // rescale what earlier groups added (nothing before the first real partial)
            const float a = L > -INFINITY ? exp2f(L - gm) : 0.0f;
            wsum *= a;
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] *= a;
            L = gm;
        }
#pragma unroll
        for (int j = 0; j < kGrp; ++j) {
            if (!(lj[j] > -INFINITY)) continue;  // absent, or empty (causal only): weighs 0
            const float w = exp2f(lj[j] - L);
            wsum += w;
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float2 f = __bfloat1622float2(h[v]);
                acc[2 * v] = fmaf(w, f.x, acc[2 * v]);
                acc[2 * v + 1] = fmaf(w, f.y, acc[2 * v + 1]);
            }
        }
    }
    const float winv = wsum > 0.0f ? 1.0f / wsum : 0.0f;  // no slot at all (causal only): a zero row
    *reinterpret_cast<uint4*>(O + qi * D + gcol) =
        make_uint4(pack_bf16(acc[0] * winv, acc[1] * winv), pack_bf16(acc[2] * winv, acc[3] * winv),
                   pack_bf16(acc[4] * winv, acc[5] * winv), pack_bf16(acc[6] * winv, acc[7] * winv));
}

// The common case of the merge above (S <= kMaxS expert partials, at most
// one shared partial): every load of a query in flight at once, and no
// registers held for partials that are not there.
template <int D, int S>
__global__ void __launch_bounds__(256) k_merge_few(const __nv_bfloat16* __restrict__ part, const float* __restrict__ lse,
                                               const __nv_bfloat16* __restrict__ sh_part,
                                               const float* __restrict__ sh_lse, __nv_bfloat16* __restrict__ O,
                                               long long nq) {
    constexpr int G = D / 8;  // threads per query
    const long long qi = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / G;
    const int gcol = (threadIdx.x % G) * 8;
    if (qi >= nq) return;
    float lj[S + 1];
    float L = -INFINITY;
#pragma unroll
    for (int j = 0; j < S; ++j) {
        lj[j] = lse[qi * S + j];
        L = fmaxf(L, lj[j]);
    }
    lj[S] = sh_part ? sh_lse[qi] : -INFINITY;
    L = fmaxf(L, lj[S]);
    uint4 raw[S + 1];
#pragma unroll
    for (int j = 0; j < S; ++j) raw[j] = *reinterpret_cast<const uint4*>(part + (qi * S + j) * D + gcol);
    if (sh_part) raw[S] = *reinterpret_cast<const uint4*>(sh_part + qi * D + gcol);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, wsum = 0.0f;
#pragma unroll
    for (int j = 0; j <= S; ++j) {
        if (j == S && !sh_part) continue;
        const float w = lj[j] > -INFINITY ? exp2f(lj[j] - L) : 0.0f;  // an empty partial (causal only) weighs 0
        wsum += w;
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float2 f = __bfloat1622float2(h[v]);
            acc[2 * v] = fmaf(w, f.x, acc[2 * v]);
            acc[2 * v + 1] = fmaf(w, f.y, acc[2 * v + 1]);
        }
    }
    const float winv = wsum > 0.0f ? 1.0f / wsum : 0.0f;  // no slot at all (causal only): a zero row
    *reinterpret_cast<uint4*>(O + qi * D + gcol) =
        make_uint4(pack_bf16(acc[0] * winv, acc[1] * winv), pack_bf16(acc[2] * winv, acc[3] * winv),
                   pack_bf16(acc[4] * winv, acc[5] * winv), pack_bf16(acc[6] * winv, acc[7] * winv));
}

template <int D, int S>
static void launch_merge_few(const TcWork& W, bool shared, void* O, long long nq, unsigned blocks, int ns,
                             cudaStream_t st) {
    if constexpr (S < kMaxS) {
        if (ns > S) return launch_merge_few<D, S + 1>(W, shared, O, nq, blocks, ns, st);
    }
    k_merge_few<D, S><<<blocks, 256, 0, st>>>(W.part, W.lse, shared ? W.sh_part : nullptr, W.sh_lse,
                                              (__nv_bfloat16*)O, nq);
}

// Producer warps of the expert kernel.
constexpr int kNPW = 3;

// ------------------------------------------------------------------------
// Expert attention with the expert's keys and values resident in shared
// memory. Persistent, one CTA per SM. The CTAs claim whole experts (all
// tiles of one (head, expert) bucket) from a counter, in head order: the load
// stays balanced, an expert's keys and values are gathered once for all its
// tiles, and at any moment all SMs work on about one head. An expert of more
// than 256 keys is cut into sub-experts of ksub <= 256 consecutive keys of its
// (ascending) set, each its own work unit with its own partial output; the
// merge kernel combines every partial of a query by log-sum-exp, which is the
// softmax over the union of their keys. The probabilities are written over
// the scores in TMEM and O += P V reads them from there.
//
// Shared mode (I == nullptr): the same kernel computes the shared slots of
// every query (keys Qt, values Vt: the bf16 rows K, V of each head, kv_head_rows
// apart) over tiles of 128 consecutive queries, in claims of sh_grp tiles,
// and with more than 256 landmarks in sub-experts as above.
//
// Chunk stream: chunk g is key chunk c = g % nex of the CTA's tile g / nex.
// The MMA warp keeps S of chunks g and g + 1 in flight while the softmax
// works on g (S of g + 2 goes right after O += P V of g, into the buffer P
// of g held), except across a change of resident keys, where the old keys'
// last O += P V goes first. The softmax warps defer a tile's epilogue until
// they have done the next tile's first chunk, so the last O += P V of a tile
// is never waited for. Each warp stages 16 rows at a time in shared memory,
// so that a store instruction writes whole 128-byte halves of four partial
// rows.
struct ResTile {
    int bh, e, start, rows, gen;  // gen: loads of the resident keys so far (this tile uses load gen - 1); rows < 0: end
    int sub, kk;                  // sub-expert and its key count
};

// expert attention with resident keys: warps 0-7 softmax + epilogue,
// 8 .. 8 + kNPW - 1 producers, then the MMA warp
constexpr int kResThreads = 32 * (8 + kNPW + 1);
// The launch gives every thread 168 registers; the producer and MMA warpgroup
// hands some down (kResRegsLo) and the two softmax warpgroups take them up
// (kResRegsHi): 4 * 32 * Lo + 8 * 32 * Hi = 384 * 168.
constexpr int kResRegsLo = 120, kResRegsHi = 192;
static_assert(kResThreads == 384 && 4 * kResRegsLo + 8 * kResRegsHi == 12 * 168, "register split must match the launch");

template <int D>
__global__ void __launch_bounds__(kResThreads, 1)
    k_expert_res(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                 const __nv_bfloat16* __restrict__ V, long long kv_head_rows, const int32_t* __restrict__ I,
                 const int32_t* __restrict__ perm, const int4* __restrict__ tiles, const int2* __restrict__ xtl,
                 int nx, int* __restrict__ work_ctr, __nv_bfloat16* __restrict__ part, float* __restrict__ lse, int N,
                 int m, int k, int s, int ksub, int nsub, int npc, int sh_tph, int sh_grp, float sl, int causal,
                 int stall, int* __restrict__ status) {
    constexpr int TILE = kT * D * 2;
    constexpr uint32_t kS0 = 0, kO0 = 256;  // TMEM: S/P buffers 0 / 128, O buffers 256 / 384
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = sm;             // 2 query tiles
    uint8_t* sK = sm + 2 * TILE;  // resident key chunks (up to 2)
    uint8_t* sV = sm + 4 * TILE;  // resident value chunks
    uint8_t* sStage = sm + 6 * TILE;  // 8 x kStageWarp epilogue staging

    __shared__ uint64_t q_full[2], q_empty[2], kv_full[2], kv_rel[2], s_full[2], p_full[2], o_full[2], o_free[2];
    __shared__ uint64_t pv_done, drain;
    __shared__ ResTile tinfo[2];
    __shared__ int4 pnext[2];    // producer warp 0 -> all producer warps: the tile to load (w < 0: none)
    __shared__ int pstop;        // producer warp 0 -> all producer warps: stop (a wait failed)
    __shared__ int rowq[2][kT];  // q << 3 | slot of each tile row, -1 past the tile's rows
    __shared__ int rowok[2][kT]; // causal variant: keys of the row's expert at or before its query
    __shared__ int keyrow[kT];
    __shared__ int keyall[2 * kT];  // causal variant: the current expert's key indices (ascending)
    __shared__ float xmax[2][2][kT], xl[2][2][kT];  // [parity][half][row] exchange of the two softmax halves
    __shared__ uint64_t xbar[2], ebar[2];          // exchange barriers (per chunk / per tile), one arrival per warp
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;
    const long long lim = stall ? kSpinTest : kSpin;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nex = (ksub + kT - 1) / kT;  // <= 2
    if (warp == 8 + kNPW) tmem_alloc(&tmem_slot, 512);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 33 * kNPW);
            mbar_init(&q_empty[i], 1 + 8);
            mbar_init(&kv_full[i], 32 * kNPW);
            mbar_init(&kv_rel[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 8);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_free[i], 8);
        }
        mbar_init(&pv_done, 1);
        mbar_init(&drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&xbar[i], 8);
            mbar_init(&ebar[i], 8);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;
    constexpr int CPR = D / 8, RPI = 32 / CPR;  // 16-byte chunks per row, rows per warp instruction

    if (warp >= 8 && warp < 8 + kNPW) {
        // ------------------------------------------------------- producers
        regs_dec<kResRegsLo>();
        // Warp 0 claims the work and hands each tile to all producer warps
        // (named barrier 1); all kNPW warps gather the tile's query rows and
        // the resident keys / values (row pairs dealt round-robin). The index
        // loads of the next tile (its bucket rows, and the expert's key
        // indices when the expert changes) are issued one tile ahead, so that
        // no gather waits on a dependent global load.
        const int pw = warp - 8;
        int cur_bh = -1, cur_e = -1, cur_u = -1, gen = 0;
        int x_t = 0, x_end = 0;         // warp 0, lane 0: tiles left of the claimed expert
        int x_u = 0, x_bh = 0;          // warp 0, lane 0: its sub-expert (and head, shared mode)
        bool stall_pending = false;     // fault test: this CTA's first tile goes unpublished
        const int cc = lane % CPR;
        // warp 0, lane 0: the next tile of the claimed work (w < 0: none left);
        // w = rows | (sub-expert << 16)
        auto next_tile = [&]() -> int4 {
            int4 td = make_int4(0, 0, 0, -1);
            if (*abort_v) return td;
            while (x_t >= x_end) {
                const int x = atomicAdd(work_ctr, 1);
                if (x >= nx) return td;
                if (x == 0 && stall) stall_pending = true;
                if (I) {  // piece x % npc of sub-expert xu % nsub of expert xu / nsub, xu = x / npc
                    const int xu = x / npc, pc = x % npc;
                    const int2 r = xtl[xu / nsub];
                    const int per = (r.y + npc - 1) / npc;  // tiles per piece (a piece may be empty)
                    x_t = r.x + pc * per;
                    x_end = min(r.x + r.y, x_t + per);
                    x_u = xu % nsub;
                } else {  // head, sub-expert, group of sh_grp query tiles
                    const int ngrp = (sh_tph + sh_grp - 1) / sh_grp;
                    x_bh = x / (nsub * ngrp);
                    x_u = (x / ngrp) % nsub;
                    x_t = (x % ngrp) * sh_grp;
                    x_end = min(sh_tph, x_t + sh_grp);
                }
            }
            if (I) {
                int4 t = tiles[x_t++];
                t.w = (t.w & 255) | (x_u << 16);
                return t;
            }
            const int start = (x_t++) * kT;
            return make_int4(x_bh, 0, start, min(kT, N - start) | (x_u << 16));
        };
        // keys of sub-expert u
        auto keys_of = [&](int u) { return min(ksub, k - u * ksub); };
        // this lane's rows of a tile: r = lane + 32 i, the ones dealt to this warp
        auto own = [&](int r) { return ((r / RPI) % kNPW) == pw; };
        int pkv[kT / 32];        // bucket entries (q << 3 | slot) of the next tile's rows, -1 for none
        int krv[2][kT / 32];     // key indices of the next expert's rows (when it changes)
        auto prefetch = [&](const int4& td) {
            const int rows = td.w & 255, u = td.w >> 16;
            const int32_t* pb = I ? perm + (size_t)td.x * N * s + td.z : nullptr;
#pragma unroll
            for (int i = 0; i < kT / 32; ++i) {
                const int r = lane + 32 * i;
                pkv[i] = (td.w >= 0 && own(r) && r < rows) ? (I ? pb[r] : (td.z + r) << 3) : -1;
            }
            if (td.w >= 0 && (td.x != cur_bh || td.y != cur_e || u != cur_u)) {
                const int kk = keys_of(u);
                const int32_t* Ie = I ? I + ((size_t)td.x * m + td.y) * k + (size_t)u * ksub : nullptr;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < kT / 32; ++i) {
                        const int t2 = c * kT + lane + 32 * i;
                        krv[c][i] = (c < nex && own(lane + 32 * i) && t2 < kk) ? (I ? Ie[t2] : u * ksub + t2) : 0;
                    }
            }
        };
        if (pw == 0 && lane == 0) pnext[0] = next_tile();
        named_sync(1, 32 * kNPW);
        int4 td = pnext[0];
        prefetch(td);
        for (int tl = 0;; ++tl) {
            const int qs = tl & 1;
            // the slot is free (warp 0 waits, then tells the others)
            if (pw == 0 && lane == 0)
                pstop = !ws_wait(&q_empty[qs], ((tl >> 1) & 1) ^ 1, status, abort_v, lim) || *abort_v;
            named_sync(1, 32 * kNPW);
            if (pstop) break;
            if (td.w < 0) {
                // no more work: an end marker for the consumers, in the free slot
                if (pw == 0 && lane == 0) tinfo[qs] = ResTile{0, 0, 0, -1, 0, 0, 0};
                cp_async_arrive(&q_full[qs]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_full[qs]);
                break;
            }
            const int bh = td.x, e = td.y, start = td.z, rows = td.w & 255, u = td.w >> 16, kk = keys_of(u);
            const bool reload = bh != cur_bh || e != cur_e || u != cur_u;
            (void)start;
#pragma unroll
            for (int i = 0; i < kT / 32; ++i) {
                const int r = lane + 32 * i;
                if (!own(r)) continue;
                int pk = pkv[i];
                if (pk >= 0 && (pk >> 3) >= N) {
                    set_status(status, kStBounds);
                    pk = -1;
                }
                rowq[qs][r] = r < rows ? pk : -1;
            }
            if (causal) {
                // each row's count of expert keys at or before its query: the
                // expert's indices are ascending, so a binary search per row
                if (reload) {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int i = 0; i < kT / 32; ++i)
                            if (own(lane + 32 * i) && c * kT + lane + 32 * i < kk)
                                keyall[c * kT + lane + 32 * i] = krv[c][i];
                    named_sync(1, 32 * kNPW);
                }
#pragma unroll
                for (int i = 0; i < kT / 32; ++i) {
                    const int r = lane + 32 * i;
                    if (!own(r)) continue;
                    const int pk = rowq[qs][r];
                    int lo = 0, hi = kk;  // first index with key > q
                    if (pk >= 0) {
                        const int q = pk >> 3;
                        while (lo < hi) {
                            const int mid = (lo + hi) >> 1;
                            if (keyall[mid] <= q) lo = mid + 1;
                            else hi = mid;
                        }
                    }
                    rowok[qs][r] = lo;
                }
            }
            if (pw == 0 && lane == 0) tinfo[qs] = ResTile{bh, e, start, rows, gen + (reload ? 1 : 0), u, kk};
            __syncwarp();
            {
                const __nv_bfloat16* Qb = Q + (size_t)bh * N * D;
                const uint32_t dq = smem_u32(sQ + qs * TILE);
#pragma unroll 4
                for (int r0 = pw * RPI; r0 < kT; r0 += kNPW * RPI) {
                    const int r = r0 + lane / CPR, pk = rowq[qs][r];
                    cp_async16(dq + sw_off(r, cc, kT), Qb + (size_t)(pk >= 0 ? pk >> 3 : 0) * D + cc * 8, pk >= 0);
                }
                cp_async_arrive(&q_full[qs]);  // counts once this thread's copies have landed
                __syncwarp();
                // publishes this warp's rowq rows (and tinfo); the fault test
                // leaves one arrival out, so the consumers' bounded waits run out
                const bool skip = stall_pending && pw == 0;
                stall_pending = false;
                if (lane == 0 && !skip) mbar_arrive(&q_full[qs]);
            }
            if (reload) {
                const __nv_bfloat16* Kb = K + (size_t)bh * kv_head_rows * D;
                const __nv_bfloat16* Vb = V + (size_t)bh * kv_head_rows * D;
                bool okc = true;
#pragma unroll
                for (int c = 0; c < 2; ++c) {  // nex <= 2 chunks (unrolled: krv stays in registers)
                    if (c >= nex) break;
                    // every MMA on the previous keys of this chunk is done: the MMA
                    // warp commits kv_rel[c] once per change of keys (gen - 1 so far)
                    if (gen > 0) {
                        int okw = 1;
                        if (lane == 0) okw = ws_wait(&kv_rel[c], (gen - 1) & 1, status, abort_v, lim);
                        if (!__shfl_sync(0xffffffffu, okw, 0)) { okc = false; break; }
                    }
#pragma unroll
                    for (int i = 0; i < kT / 32; ++i) {
                        const int r = lane + 32 * i;
                        if (!own(r)) continue;
                        int j = krv[c][i];
                        if (j < 0 || j >= kv_head_rows) {
                            set_status(status, kStBounds);
                            j = 0;
                        }
                        keyrow[r] = j;
                    }
                    __syncwarp();
                    const uint32_t dk = smem_u32(sK + c * TILE), dv = smem_u32(sV + c * TILE);
#pragma unroll 4
                    for (int r0 = pw * RPI; r0 < kT; r0 += kNPW * RPI) {
                        const int r = r0 + lane / CPR;
                        const size_t off = (size_t)keyrow[r] * D + cc * 8;
                        cp_async16(dk + sw_off(r, cc, kT), Kb + off, true);
                        cp_async16(dv + sw_off(r, cc, kT), Vb + off, true);
                    }
                    cp_async_arrive(&kv_full[c]);
                    __syncwarp();
                }
                // after a failed wait the abort flag is up: the next tile's
                // slot wait hands every producer warp the stop
                if (okc) {
                    ++gen;
                    cur_bh = bh;
                    cur_e = e;
                    cur_u = u;
                }
            }
            // the next tile, and its index loads in flight while this one is consumed
            if (pw == 0 && lane == 0) pnext[(tl + 1) & 1] = next_tile();
            named_sync(1, 32 * kNPW);
            td = pnext[(tl + 1) & 1];
            prefetch(td);
        }
        cp_async_wait_all();  // nothing of ours may still be in flight when the CTA exits
    } else if (warp == 8 + kNPW) {
        // ------------------------------------------------------ MMA issuer
        regs_dec<kResRegsLo>();
        // One thread polls the barriers without blocking: O += P V of chunk g
        // goes out as soon as its probabilities are in, and S of the next
        // chunk as soon as its query tile and keys are; neither waits behind
        // the other. S runs at most one chunk ahead of the last O += P V.
        if (lane == 0) {
            int G = 0x7fffffff;    // chunks in all, known once the end marker is seen
            int g = 0;             // next chunk whose O += P V is to be issued
            int ns = 0;            // next chunk whose S is to be issued
            int seen_tl = -1;      // last tile whose query tile was seen
            int s_gen = 0, cur_gen = 0;  // keys of chunk ns's tile / of the S issued last
            bool rel_early = false;      // old keys' other chunks released, the last one pending
            long long idle0 = clock64();
            while (g < G) {
                bool prog = false;
                // ---- S of chunk ns
                if (ns < G && ns <= g + 1) {
                    const int tl = ns / nex, c = ns - tl * nex, qs = tl & 1;
                    bool ready = true;
                    if (tl != seen_tl) {
                        if (mbar_test_wait(&q_full[qs], (tl >> 1) & 1)) {
                            seen_tl = tl;
                            const ResTile ti = tinfo[qs];
                            prog = true;
                            if (ti.rows < 0) {
                                G = ns;
                                ready = false;
                            } else {
                                s_gen = ti.gen;
                            }
                        } else {
                            ready = false;
                        }
                    }
                    if (ready && s_gen != cur_gen) {
                        if (cur_gen > 0) {
                            // the old keys' other chunks are done with once their last
                            // O += P V is issued (S runs at most one chunk ahead)
                            if (!rel_early) {
                                for (int c2 = 0; c2 < nex - 1; ++c2) mma_commit(&kv_rel[c2]);
                                rel_early = true;
                                prog = true;
                            }
                            if (g < ns) {
                                ready = false;  // the old keys' last O += P V goes first
                            } else {
                                mma_commit(&kv_rel[nex - 1]);
                                rel_early = false;
                                cur_gen = s_gen;
                            }
                        } else {
                            cur_gen = s_gen;
                        }
                    }
                    if (ready && mbar_test_wait(&kv_full[c], (s_gen - 1) & 1)) {
                        fence_proxy_async();  // copied tiles (generic proxy) -> the MMA's async-proxy reads
                        fence_after_sync();
                        issue_qk<D>(tmem + kS0 + (ns & 1) * 128, smem_u32(sQ + qs * TILE), smem_u32(sK + c * TILE),
                                    false);
                        mma_commit(&s_full[ns & 1]);
                        if (c == nex - 1) mma_commit(&q_empty[qs]);
                        ++ns;
                        prog = true;
                    }
                }
                // ---- O += P V of chunk g
                if (g < ns && g < G) {
                    const int tl = g / nex, c = g - tl * nex, ob = tl & 1;
                    if (mbar_test_wait(&p_full[g & 1], (g >> 1) & 1) &&
                        (c != 0 || mbar_test_wait(&o_free[ob], ((tl >> 1) & 1) ^ 1))) {
                        fence_after_sync();
                        issue_pv_ts<D>(tmem + kO0 + ob * 128, tmem + kS0 + (g & 1) * 128, smem_u32(sV + c * TILE),
                                       c > 0);
                        mma_commit(&pv_done);
                        if (c == nex - 1) mma_commit(&o_full[ob]);
                        ++g;
                        prog = true;
                    }
                }
                if (prog) {
                    idle0 = clock64();
                } else {
                    if (*abort_v) break;
                    if (clock64() - idle0 > lim) {
                        set_status(status, kStTimeout);
                        *abort_v = 1;
                        break;
                    }
                }
            }
            // every MMA this thread issued has completed before TMEM is freed
            mma_commit(&drain);
            drain_wait(&drain, 0, status);
        }
        __syncwarp();
    } else {
        // -------------------------------------------- softmax + epilogue
        regs_inc<kResRegsHi>();
        // two warpgroups share each row: wg 0 takes keys 0..63 of a chunk and
        // output columns 0..D/2-1, wg 1 the other halves; the row max and the
        // row sum are exchanged through shared memory (bounded mbarrier waits)
        constexpr int DH = D / 2;
        const int wg = warp >> 2, r = threadIdx.x & 127;
        const bool fast = sl > 0.0f;  // the row max of the scaled scores is the scaled max
        uint8_t* stage = sStage + warp * kStageWarp;
        // epilogue of tile pt: normalized bf16 partial rows (row pk >> 3, slot
        // pk & 7 of head pti.bh) and their log2-sum-exp, then the count and,
        // for the queries whose last half row this is, the merge
        // plt: the whole row sum when the two halves already exchanged it (with the
        // next tile's first row maxima); last: the CTA's last tile, whose
        // epilogue exchanges the row sum itself
        auto epilogue = [&](int pt, const ResTile& pti, int pk, float pl, float pm, float plt, bool last) -> bool {
            constexpr int PPR = DH / 8, RPI = 32 / PPR;  // pieces per half row, rows per store instruction
            const int ob = pt & 1;
            if (!__all_sync(0xffffffffu, ws_wait(&o_full[ob], (pt >> 1) & 1, status, abort_v, lim))) return false;
            fence_after_sync();
            const uint32_t tO = lane_base(tmem) + kO0 + ob * 128 + wg * DH;
            float o[DH];
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 32) tmem_ld32(tO + c0, o + c0);
            tmem_wait_ld();
            float lt = plt;
            if (last) {  // the CTA's last tile: one exchange of its own (ebar's only use)
                xl[pt & 1][wg][r] = pl;
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ebar[0]);
                if (!__all_sync(0xffffffffu, ws_wait(&ebar[0], 0, status, abort_v, lim))) return false;
                lt = pl + xl[pt & 1][wg ^ 1][r];
            } else {
                fence_before_sync();
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(&o_free[ob]);
            const float inv = (pk >= 0 && lt > 0.0f) ? 1.0f / lt : 0.0f;  // no key (causal only): zero partial
            const size_t pr = pk >= 0 ? (((size_t)pti.bh * N + (pk >> 3)) * s + (pk & 7)) * nsub + pti.sub : 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // lanes 16h .. 16h + 15 stage their rows
                if ((lane >> 4) == h) {
#pragma unroll
                    for (int u = 0; u < PPR; ++u) {
                        const float* x = o + 8 * u;
                        *reinterpret_cast<uint4*>(stage + stage_off<PPR>(lane & 15, u)) =
                            make_uint4(pack_bf16(x[0] * inv, x[1] * inv), pack_bf16(x[2] * inv, x[3] * inv),
                                       pack_bf16(x[4] * inv, x[5] * inv), pack_bf16(x[6] * inv, x[7] * inv));
                    }
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 16 / RPI; ++i) {
                    const int rl = i * RPI + lane / PPR, u = lane % PPR;
                    const uint4 w4 = *reinterpret_cast<const uint4*>(stage + stage_off<PPR>(rl, u));
                    const size_t prr = __shfl_sync(0xffffffffu, pr, 16 * h + rl);
                    const int pkr = __shfl_sync(0xffffffffu, pk, 16 * h + rl);
                    if (pkr >= 0) *reinterpret_cast<uint4*>(part + prr * D + wg * DH + 8 * u) = w4;
                }
                __syncwarp();
            }
            if (wg == 0 && pk >= 0) lse[pr] = lt > 0.0f ? pm + __log2f(lt) : -INFINITY;
            return true;
        };
        int g = 0;
        bool have_prev = false, ok = true;
        ResTile pti{};
        int ppk = -1;
        float pl = 0.0f, pm = 0.0f;
        int tl = 0;
        for (;; ++tl) {
            const int qs = tl & 1, ob = tl & 1;
            if (!__all_sync(0xffffffffu, ws_wait(&q_full[qs], (tl >> 1) & 1, status, abort_v, lim))) {
                ok = false;
                break;
            }
            const ResTile ti = tinfo[qs];
            if (ti.rows < 0) break;  // end of the work
            const int pk = rowq[qs][r];
            const int kok = causal ? rowok[qs][r] : ti.kk;  // the row's keys (a prefix of the sub-expert's)
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[qs]);  // tinfo / rowq read; the MMA releases the tile itself
            const bool valid = pk >= 0;
            float mref = -INFINITY, l = 0.0f;  // l: this half's share of the row sum
            const uint32_t tO = lane_base(tmem) + kO0 + ob * 128 + wg * DH;
            for (int c = 0; c < nex; ++c, ++g) {
                const int sb = g & 1;
                if (!__all_sync(0xffffffffu, ws_wait(&s_full[sb], (g >> 1) & 1, status, abort_v, lim))) { ok = false; break; }
                fence_after_sync();
                const uint32_t tS = lane_base(tmem) + kS0 + sb * 128;
                const int nval = valid ? min(kT, kok - c * kT) - 64 * wg : 0;  // valid columns of this half
                const bool full = __all_sync(0xffffffffu, nval >= 64) && fast;
                float v[64];
                tmem_ld32(tS + 64 * wg, v);
                tmem_ld32(tS + 64 * wg + 32, v + 32);
                tmem_wait_ld();
                float mx = -INFINITY;
                if (full) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) mx = fmaxf(mx, v[j]);
                    mx *= sl;
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) mx = fmaxf(mx, j < nval ? v[j] * sl : -INFINITY);
                }
                xmax[g & 1][wg][r] = mx;
                if (c == 0 && have_prev) xl[(tl - 1) & 1][wg][r] = pl;  // the previous tile's row-sum half
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&xbar[g & 1]);
                // both halves have read S(g) and posted their max (bounded wait)
                if (!__all_sync(0xffffffffu, ws_wait(&xbar[g & 1], (g >> 1) & 1, status, abort_v, lim))) { ok = false; break; }
                fence_after_sync();
                mx = fmaxf(mx, xmax[g & 1][wg ^ 1][r]);
                float mnew = mref, alpha = 1.0f;
                if (mx > mref + 8.0f) {
                    mnew = mx;
                    alpha = ex2(mref - mnew);
                }
                float sum = 0.0f;
                uint32_t pkd[32];
                if (full) {
#pragma unroll
                    for (int j = 0; j < 64; j += 2) {
                        const float p0 = ex2(fmaf(v[j], sl, -mnew)), p1 = ex2(fmaf(v[j + 1], sl, -mnew));
                        sum += p0 + p1;
                        pkd[j >> 1] = pack_bf16(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 64; j += 2) {
                        const float e0 = ex2(fmaf(v[j], sl, -mnew)), e1 = ex2(fmaf(v[j + 1], sl, -mnew));
                        const float p0 = j < nval ? e0 : 0.0f, p1 = j + 1 < nval ? e1 : 0.0f;
                        sum += p0 + p1;
                        pkd[j >> 1] = pack_bf16(p0, p1);
                    }
                }
                // P (bf16, two keys per column) over the scores: keys 64wg.. -> columns 32wg..
                tmem_st32(tS + 32 * wg, reinterpret_cast<const float*>(pkd));
                tmem_wait_st();
                l = l * alpha + sum;
                mref = mnew;
                if (__any_sync(0xffffffffu, c > 0 && alpha != 1.0f)) {
                    // S(g) done implies O += P V of chunk g - 2 done: this wait can only
                    // see chunk g - 1's phase
                    if (!__all_sync(0xffffffffu, ws_wait(&pv_done, (g - 1) & 1, status, abort_v, lim))) { ok = false; break; }
                    fence_after_sync();
                    const float a = (c > 0) ? alpha : 1.0f;
#pragma unroll 1
                    for (int c0 = 0; c0 < DH; c0 += 32) {
                        float o[32];
                        tmem_ld32(tO + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] *= a;
                        tmem_st32(tO + c0, o);
                    }
                    tmem_wait_st();
                }
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[g & 1]);
                // the previous tile's epilogue, now that its last O += P V has had a chunk's time
                if (c == 0 && have_prev) {
                    // the other half posted its share before this chunk's exchange
                    if (!(ok = epilogue(tl - 1, pti, ppk, pl, pm, pl + xl[(tl - 1) & 1][wg ^ 1][r], false))) break;
                    have_prev = false;
                }
            }
            if (!ok) break;
            have_prev = true;
            pti = ti;
            ppk = pk;
            pl = l;
            pm = mref;
        }
        if (ok && have_prev) epilogue(tl - 1, pti, ppk, pl, pm, 0.0f, true);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 8 + kNPW) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ host

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 152;
    }
    return n;
}

TcPlan tc_plan(const Dims& D) {
    TcPlan p;
    p.m_pad = (D.m + kT - 1) / kT * kT;
    p.m_tiles = p.m_pad / kT;
    const int nchunks = (D.N + kT - 1) / kT;
    // key splits of the landmark pass: one CTA per (landmark tile, split, head),
    // one CTA per SM, so a launch runs in waves; the split count minimizes
    // waves x (chunks per split + 3), three chunks' time being about what a
    // CTA spends outside its chunk loop (start, first loads, epilogue). At most
    // 128 splits: <= 256 candidate regions per row (two column halves per
    // split) stay stageable in the selection.
    long long sp = 1;
    {
        long long best_cost = -1;
        for (long long c = 1; c <= 128 && c <= nchunks; ++c) {
            const long long cps = (nchunks + c - 1) / c, spl = (nchunks + cps - 1) / cps;
            const long long waves = ((long long)D.BH * p.m_tiles * spl + num_sms() - 1) / num_sms();
            const long long cost = waves * (cps + 3);
            if (best_cost < 0 || cost <= best_cost) {
                best_cost = cost;
                sp = c;
            }
        }
    }
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
    if (R > 32) R = 32;
    if (R < 1) R = 1;
    // the sample must hold at least k real keys: runs of 16 every 16R keys
    auto n_valid = [&](int r) {
        const long long span = 16LL * r, full = D.N / span, rest = D.N - full * span;
        return full * 16 + std::min<long long>(16, rest);
    };
    while (R > 1 && n_valid(R) < D.k) --R;
    p.R = R;
    p.n_samp = (int)(((long long)D.N + 16LL * R - 1) / (16LL * R) * 16);
    p.cand_cap = (long long)p.chunks_per_split * kT;
    p.resident = D.shared && p.m_pad == kT && D.k <= 2 * kT;
    p.route_shared = D.shared && p.m_pad == kT;
    p.ksub = std::min(D.k, 2 * kT);
    p.nsub = (D.k + p.ksub - 1) / p.ksub;
    p.ksub_sh = std::min(D.m, 2 * kT);
    p.nsub_sh = (D.m + p.ksub_sh - 1) / p.ksub_sh;
    p.nsh = !D.shared ? 0 : p.route_shared ? 1 : p.nsub_sh;
    return p;
}

bool tc_supported(const Dims& D) {
    return D.dtype == 1 && (D.d == 64 || D.d == 128) && D.m <= 512 && D.N <= (1 << 20);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

// Tensor map over `rows` rows of D bf16 (row-major) read in boxes of 64
// columns x 128 rows with the 128-byte swizzle (the operand tile layout).
static cudaError_t tile_map(CUtensorMap* map, const void* base, long long rows, int D) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kT};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
    if (P.route_shared) {  // routes + the shared-slot partial in one pass
        alignas(64) CUtensorMap mq;
        if ((e = tile_map(&mq, q, (long long)D.BH * D.N, DD))) return e;
        constexpr int NSQ = 3;
        const int smem = (3 + NSQ) * tile + 8 * kStageWarp + 1024;
        if ((e = set_smem(k_route_pp<DD, SMAX, NSQ>, smem))) return e;
        const int tph = (D.N + kT - 1) / kT;
        const int total = tph * D.BH;
        const int grid = std::min(total, num_sms());
        k_route_pp<DD, SMAX, NSQ><<<grid, 320, smem, st>>>(mq, W.Qhi, W.Qlo, W.Vtb, D.N, D.m, D.s, tph, total,
                                                           D.scale * 1.4426950408889634f, D.causal ? 1 : 0, E,
                                                           W.sh_part, W.sh_lse, W.counts, status);
    } else if (P.m_pad <= 256) {
        const int smem = 2 * P.m_pad * DD * 2 + 2 * tile + 1024;
        if ((e = set_smem(k_route_tc<DD, SMAX>, smem))) return e;
        const int tph = (D.N + kT - 1) / kT;
        const int total = tph * D.BH;
        const int grid = std::min(total, num_sms());
        k_route_tc<DD, SMAX><<<grid, 256, smem, st>>>(q, W.Qhi, W.Qlo, D.N, D.m, P.m_pad, D.s, tph, total,
                                                      (uint32_t)P.route_cols, E, status);
    } else {
        const int smem = std::max(3 * tile, 100 * 1024) + 1024;
        if ((e = set_smem(k_route_chunked_tc<DD, SMAX>, smem))) return e;
        dim3 grid((D.N + kT - 1) / kT, D.BH);
        k_route_chunked_tc<DD, SMAX><<<grid, 128, smem, st>>>(q, W.Qhi, W.Qlo, D.N, D.m, P.m_pad, D.s,
                                                              (uint32_t)P.route_cols, E, status);
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
    // mita_select passes no V: the landmark pass still runs its P V MMAs (their
    // result, the shared expert, is not used then) and reads K in V's place
    const __nv_bfloat16* v = (const __nv_bfloat16*)(V ? V : K);
    const float sl = D.scale * 1.4426950408889634f;
    const int tile = kT * DD * 2;
    cudaError_t e;
    // top-k threshold from a strided sample of the keys
    prof_mark(st, "topk_sample");
    {
        const int smem = std::max(3 * tile, 100 * 1024) + 1024;
        if ((e = set_smem(k_sample_tc<DD>, smem))) return e;
        // sample chunks per CTA: the fewest (of one to four) that keep the grid
        // within one wave of two CTAs per SM, else four; a few heads then
        // spread over more SMs, and many heads do not spill into a second wave
        const int nch = (P.n_samp + kT - 1) / kT;
        int cpc = 1;
        while (cpc < 4 && (long long)P.m_tiles * ((nch + cpc - 1) / cpc) * D.BH > 2LL * num_sms()) ++cpc;
        const int groups = (nch + cpc - 1) / cpc;
        k_sample_tc<DD><<<dim3(P.m_tiles, groups, D.BH), 128, smem, st>>>(kk, W.Qhi, W.Qlo, W.Ssamp, D.N, D.m,
                                                                         P.m_pad, P.R, P.n_samp, cpc, status);
        if ((e = cudaGetLastError())) return e;
        count_launch();
        prof_mark(st, "topk_threshold");
        if ((e = launch_sample_threshold(W.Ssamp, (long long)D.BH * D.m, P.n_samp, D.k, W.thr, st))) return e;
    }
    // landmark pass: top-k candidates and the shared-expert partials
    prof_mark(st, "landmark");
    {
        alignas(64) CUtensorMap mk, mv;
        const long long rows = (long long)D.BH * D.N;
        if ((e = tile_map(&mk, kk, rows, DD)) || (e = tile_map(&mv, v, rows, DD))) return e;
        constexpr int NS = DD == 64 ? 4 : 2;
        const int smem = (2 + 2 * NS) * tile + 1024;
        if ((e = set_smem(k_landmark_ws<DD, NS>, smem))) return e;
        dim3 grid(P.m_tiles, P.splits, D.BH);
        k_landmark_ws<DD, NS><<<grid, 320, smem, st>>>(mk, mv, W.Qhi, W.Qlo, W.thr, W.cand, W.ccount, W.Opart, W.ML,
                                                      D.N, D.m, P.m_pad, P.splits, P.chunks_per_split, sl,
                                                      D.causal ? 1 : 0,
                                                      (D.flags & MITA_TESTFLAG_STALL_PRODUCER) ? 1 : 0, status);
        if ((e = cudaGetLastError())) return e;
        count_launch();
    }
    prof_mark(st, "topk_select");
    // two record regions (column halves) per (row, split)
    if ((e = launch_topk_cand(W.cand, W.ccount, 2 * P.splits, P.cand_cap / 2, D.BH, D.m, P.m_pad, D.N, D.k,
                              (long long)P.R * D.k, I, status, st)))
        return e;
    if (upto >= 2) {
        prof_mark(st, "vt_combine");
        count_launch();
        // split lanes: a power of two covering the splits, a warp at least, 256 threads at most
        int vt_threads = DD / 4;
        while (vt_threads < 256 && (vt_threads < 32 || vt_threads / (DD / 4) < P.splits)) vt_threads *= 2;
        k_vt_combine<DD><<<dim3(P.m_pad, D.BH), vt_threads, 0, st>>>(W.Opart, W.ML, P.splits, D.m, P.m_pad, Vt,
                                                                    W.Vtb);
        if ((e = cudaGetLastError())) return e;
    }
    if (!E) return cudaSuccess;
    // routing (the routing pass with the shared slots also counts the routes
    // per expert for the bucketing, into counts cleared here)
    prof_mark(st, "route");
    if ((e = cudaMemsetAsync(W.zero_begin, 0, W.zero_bytes, st))) return e;
    if ((e = launch_route<DD>(D, P, W, q, E, status, st))) return e;
    if (upto < 2) return cudaSuccess;
    // bucketing
    prof_mark(st, "bucket");
    {
        const int use_smem = D.m <= 4096;
        dim3 grid((D.N + 255) / 256, D.BH);
        if (!P.route_shared) {
            k_bucket_count<<<grid, 256, use_smem ? 8 * D.m : 0, st>>>(E, D.N, D.m, D.s, W.counts, use_smem, status);
            count_launch();
        }
        k_bucket_scan<<<D.BH, 512, 0, st>>>(W.counts, D.m, D.N * D.s, W.cursors, W.toff, W.tile_ctr, W.tiles,
                                            W.xtl);
        k_bucket_scatter<<<grid, 256, use_smem ? 8 * D.m : 0, st>>>(E, D.N, D.m, D.s, W.cursors, W.perm, use_smem);
        if ((e = cudaGetLastError())) return e;
        count_launch(2);
    }
    // expert attention (and, with more than 128 landmarks, the shared slots) + merge
    {
        const int smem = 6 * tile + 8 * kStageWarp + 1024;
        const int stall = (D.flags & MITA_TESTFLAG_STALL_PRODUCER) ? 1 : 0;
        if ((e = set_smem(k_expert_res<DD>, smem))) return e;
        if (P.nsh && !P.route_shared) {
            prof_mark(st, "shared");
            const int tph = (D.N + kT - 1) / kT;
            const long long want = (long long)D.BH * P.nsub_sh * tph / (8LL * num_sms());
            const int grp = (int)std::max(1LL, std::min((long long)tph, want));
            const int ngrp = (tph + grp - 1) / grp;
            k_expert_res<DD><<<num_sms(), kResThreads, smem, st>>>(
                q, W.Qhi, W.Vtb, P.m_pad, nullptr, nullptr, nullptr, nullptr, D.BH * P.nsub_sh * ngrp, W.tile_ctr + 2,
                W.sh_part, W.sh_lse, D.N, D.m, D.m, 1, P.ksub_sh, P.nsub_sh, 1, tph, grp, sl, 0, stall, status);
            if ((e = cudaGetLastError())) return e;
            count_launch();
        }
        prof_mark(st, "expert_res");
        // with few (sub-)experts per SM (a few heads), each is cut into up to
        // eight pieces of consecutive tiles, so that the largest ones do not
        // set the kernel's length (a piece reloads its expert's keys)
        const long long units = (long long)D.BH * D.m * P.nsub, want = 4LL * num_sms();
        const int npc = (int)std::max(1LL, std::min(8LL, (want + units - 1) / units));
        k_expert_res<DD><<<num_sms(), kResThreads, smem, st>>>(
            q, kk, v, D.N, I, W.perm, W.tiles, W.xtl, (int)(units * npc), W.tile_ctr + 1, W.part, W.lse, D.N, D.m,
            D.k, D.s, P.ksub, P.nsub, npc, 0, 1, sl, D.causal ? 1 : 0, stall, status);
        if ((e = cudaGetLastError())) return e;
        count_launch();
        prof_mark(st, "merge");
        const long long nq = (long long)D.BH * D.N;
        const unsigned mblocks = (unsigned)((nq * (DD / 8) + 255) / 256);
        if (D.s * P.nsub <= kMaxS && P.nsh <= 1)
            launch_merge_few<DD, 1>(W, P.nsh > 0, O, nq, mblocks, D.s * P.nsub, st);
        else
            k_merge<DD><<<mblocks, 256, 0, st>>>(W.part, W.lse, D.s * P.nsub, W.sh_part, W.sh_lse, P.nsh,
                                                 (__nv_bfloat16*)O, nq);
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

