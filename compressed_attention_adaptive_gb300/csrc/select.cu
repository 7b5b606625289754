// Exact top-k selection per landmark row: the expert index sets I_i of
// "MiTA Attention: Efficient Fast-Weight Scaling via a Mixture of Top-k
// Activations" (gist.science summaries, Arabic edition section 2: the top-k
// indices of K^T qt_i form expert i). Ties go to the lower key index and each
// set is written in ascending index order.
//
// Method: MSD radix select on the 32-bit order-preserving key of each score
// (four 8-bit digit histograms) finds the k-th largest key v and how many of
// the keys equal to v are still needed; one ordered pass then keeps every
// score above v and the first needed ones equal to v, so the output comes out
// ascending without a sort.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mita {

// Digit search of one radix pass, by warp 0: the largest bin b such that the
// bins b..255 hold at least `rem` keys (bin 0 if none does), the count in the
// bins above b (*above) and in b itself (*in_b). Lane L holds bins
// 255 - 8L .. 248 - 8L; a shuffle prefix sum over lanes finds the lane where
// the running count from the top reaches rem, which then scans its 8 bins.
// Returns true on the one lane that found it.
__device__ __forceinline__ bool radix_digit(const unsigned* hist, int rem, int* b_out, int* above, int* in_b) {
    const int lane = threadIdx.x & 31;
    int c[8], lsum = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        c[t] = (int)hist[255 - 8 * lane - t];
        lsum += c[t];
    }
    int incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned ball = __ballot_sync(0xffffffffu, incl >= rem);
    const int L = ball ? __ffs(ball) - 1 : 31;
    if (lane != L) return false;
    int acc = incl - lsum;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        if (t == 7 || acc + c[t] >= rem) {
            *b_out = 255 - 8 * lane - t;
            *above = acc;
            *in_b = c[t];
            return true;
        }
        acc += c[t];
    }
    return true;
}

// Shared part of both selectors: finds (v, rem) over n keys produced by
// key_of(j). All threads of the block return the same values.
template <typename KeyOf>
__device__ __forceinline__ void radix_kth(int n, int k, KeyOf key_of, unsigned* hist, uint32_t* v_out,
                                          int* rem_out) {
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_rem;
    uint32_t prefix = 0u, mask = 0u;
    int rem = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += blockDim.x) {
            const uint32_t u = key_of(j);
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            int b, acc, in_b;
            if (radix_digit(hist, rem, &b, &acc, &in_b)) {
                sh_prefix = prefix | ((uint32_t)b << shift);
                sh_rem = rem - acc;
            }
        }
        __syncthreads();
        prefix = sh_prefix;
        rem = sh_rem;
        mask |= 0xFFu << shift;
    }
    *v_out = prefix;
    *rem_out = rem;
}

// One block per row of a dense score matrix S [rows][N].
__global__ void __launch_bounds__(512) k_topk_dense(const float* __restrict__ S, int N, int k,
                                                    int32_t* __restrict__ I) {
    __shared__ unsigned hist[256];
    __shared__ int tmp[33];
    const size_t row = blockIdx.x;
    const float* s = S + row * N;
    uint32_t v;
    int rem;
    radix_kth(N, k, [&](int j) { return order_key(s[j]); }, hist, &v, &rem);
    int out = 0, eq_seen = 0;
    int32_t* dst = I + row * k;
    for (int base = 0; base < N; base += blockDim.x) {
        const int j = base + threadIdx.x;
        const uint32_t u = (j < N) ? order_key(s[j]) : 0u;
        const int is_eq = (j < N && u == v);
        int eq_tot;
        const int eq_before = block_excl_scan(is_eq, tmp, &eq_tot);
        const int take = (j < N) && (u > v || (is_eq && eq_seen + eq_before < rem));
        int tot;
        const int pos = block_excl_scan(take, tmp, &tot);
        if (take) dst[out + pos] = j;
        out += tot;
        eq_seen += eq_tot;
    }
}

// Inverse of order_key.
__device__ __forceinline__ float key_float(uint32_t v) {
    return __uint_as_float((v & 0x80000000u) ? (v & 0x7FFFFFFFu) : ~v);
}

// Per landmark row of sample scores (n_samp >= k of them): the k-th largest,
// lowered by a small margin, is a threshold that at least k keys of the full
// row reach, so every top-k key of the row scores at or above it.
__global__ void __launch_bounds__(512) k_sample_threshold(const float* __restrict__ Ssamp, int n_samp, int k,
                                                          float* __restrict__ thr, int staged) {
    extern __shared__ uint32_t skeys[];  // the row's order keys when staged
    __shared__ unsigned hist[256];
    const size_t row = blockIdx.x;
    const float* s = Ssamp + row * n_samp;
    uint32_t v;
    int rem;
    if (staged) {  // one coalesced read of the row; the radix passes run in shared memory
        for (int j = threadIdx.x; j < n_samp; j += blockDim.x) skeys[j] = order_key(s[j]);
        __syncthreads();
        radix_kth(n_samp, k, [&](int j) { return skeys[j]; }, hist, &v, &rem);
    } else {
        radix_kth(n_samp, k, [&](int j) { return order_key(s[j]); }, hist, &v, &rem);
    }
    if (threadIdx.x == 0) {
        const float t = key_float(v);
        thr[row] = t - 1e-3f * fmaxf(1.0f, fabsf(t));
    }
}

// Rows of the warp-per-row selects handled by one block (at most).
constexpr int kRowsPerBlock = 8;

// Warp-level MSD radix select: the largest key v such that at least `rem` of
// the keys key_of accepts are >= v (four 8-bit digit passes over the keys that
// each(f) hands the warp's lanes, f(u, j) per key, with the warp's own 256-bin
// histogram). Returns v; *rem_out = how many keys equal to v are still needed,
// *eq_out = how many accepted keys equal v.
template <typename Each, typename KeyOf>
__device__ __forceinline__ uint32_t warp_radix_select(Each each, KeyOf key_of, int rem, unsigned* hist, int* rem_out,
                                                      int* eq_out) {
    const int lane = threadIdx.x & 31;
    uint32_t prefix = 0u, mask = 0u;
    int eq = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = lane; b < 256; b += 32) hist[b] = 0u;
        __syncwarp();
        each([&](uint32_t u0, int j) {
            bool ok;
            const uint32_t u = key_of(u0, j, &ok);
            if (ok && (u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
        });
        __syncwarp();
        int b = 0, above = 0, in_b = 0;
        const bool found = radix_digit(hist, rem, &b, &above, &in_b);
        const int src = __ffs(__ballot_sync(0xffffffffu, found)) - 1;
        b = __shfl_sync(0xffffffffu, b, src);
        above = __shfl_sync(0xffffffffu, above, src);
        in_b = __shfl_sync(0xffffffffu, in_b, src);
        prefix |= (uint32_t)b << shift;
        rem -= above;
        eq = in_b;
        mask |= 0xFFu << shift;
        __syncwarp();  // every lane has read the histogram before the next pass clears it
    }
    *rem_out = rem;
    *eq_out = eq;
    return prefix;
}

// The same threshold with one warp per row and no block-wide barrier, for rows
// of at most 4096 samples (where it measured faster than a block per row); the
// row is read once per digit pass (16 KB at n_samp = 4096, from L1/L2).
__global__ void __launch_bounds__(32 * kRowsPerBlock) k_sample_threshold_w(const float* __restrict__ Ssamp,
                                                                         long long rows, int n_samp, int k,
                                                                         float* __restrict__ thr) {
    __shared__ unsigned hist_all[kRowsPerBlock][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kRowsPerBlock + warp;
    if (row >= rows) return;  // the whole warp: nothing below syncs the block
    const float* s = Ssamp + row * n_samp;
    auto each = [&](auto f) {
        for (int j = lane; j < n_samp; j += 32) f(order_key(s[j]), j);
    };
    int rem, eq;
    const uint32_t v = warp_radix_select(each, [](uint32_t u, int, bool* ok) { *ok = true; return u; }, k,
                                         hist_all[warp], &rem, &eq);
    if (lane == 0) {
        const float t = key_float(v);
        thr[row] = t - 1e-3f * fmaxf(1.0f, fabsf(t));
    }
}

// Candidates of one row as (order key, key index) pairs: either staged in
// shared memory (n of them) or read from the `splits` record regions in
// global memory (region sp holding counts[sp] records at base + sp * cap).
struct CandSrc {
    const uint32_t* skey;
    const int* sidx;
    int n;
    const int2* base;
    const int* counts;
    int splits;
    long long cap;
    template <typename F> __device__ __forceinline__ void each(F f) const {
        if (skey) {
            for (int t = threadIdx.x; t < n; t += blockDim.x) f(skey[t], sidx[t]);
        } else {
            for (int sp = 0; sp < splits; ++sp) {
                const int c = (int)min((long long)max(counts[sp], 0), cap);
                const int2* b = base + sp * cap;
                for (int t = threadIdx.x; t < c; t += blockDim.x) {
                    const int2 r = b[t];
                    f(order_key(__int_as_float(r.x)), r.y);
                }
            }
        }
    }
};

// MSD radix select over the candidates: the largest key v such that at least
// `rem` candidates (those key_of accepts) are >= v, as 4 passes of 8-bit
// digits. Returns v, the count of that key still needed (*rem_out) and how
// many candidates have it (*eq_out).
template <typename KeyOf>
__device__ __forceinline__ uint32_t radix_select(const CandSrc& cs, int rem, KeyOf key_of, unsigned* hist,
                                                 int* rem_out, int* eq_out) {
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_rem, sh_eq;
    uint32_t prefix = 0u, mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        cs.each([&](uint32_t u0, int j) {
            bool ok;
            const uint32_t u = key_of(u0, j, &ok);
            if (ok && (u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
        });
        __syncthreads();
        if (threadIdx.x < 32) {
            int b, acc, in_b;
            if (radix_digit(hist, rem, &b, &acc, &in_b)) {
                sh_prefix = prefix | ((uint32_t)b << shift);
                sh_rem = rem - acc;
                sh_eq = in_b;
            }
        }
        __syncthreads();
        prefix = sh_prefix;
        rem = sh_rem;
        mask |= 0xFFu << shift;
    }
    *rem_out = rem;
    *eq_out = sh_eq;
    return prefix;
}

// Candidate regions (key split x column half) a row can have and still be
// staged in shared memory.
constexpr int kMaxRegions = 256;

// Exact top-k of one landmark row from its candidates: the k-th largest score
// key v, the lowest key indices among scores equal to v, then the chosen keys
// marked in a bitmap and written out in ascending order. Dynamic shared
// memory: ceil(N / 32) bitmap words, then room for `stage_cap` staged
// candidates (key and index arrays); rows with more candidates are read from
// global memory on every pass instead.
template <int TB>
__global__ void __launch_bounds__(TB) k_topk_cand(const int2* __restrict__ cand, const int* __restrict__ ccount,
                                                   int splits, long long cap, int m, int m_pad, int N, int k,
                                                   int stage_cap, int32_t* __restrict__ I, int* __restrict__ status) {
    extern __shared__ uint32_t dyn[];
    __shared__ unsigned hist[256];
    __shared__ int tmp[33];
    __shared__ int sh_off[kMaxRegions + 1];
    __shared__ int sh_total;
    const int bh = blockIdx.y, i = blockIdx.x;
    const size_t rrow = (size_t)bh * m_pad + i;
    const int nwords = (N + 31) >> 5;
    uint32_t* bits = dyn;
    uint32_t* skey = dyn + nwords;
    int* sidx = reinterpret_cast<int*>(skey + stage_cap);
    const int* cnts = ccount + rrow * splits;
    const int2* base = cand + rrow * splits * cap;
    for (int w = threadIdx.x; w < nwords; w += blockDim.x) bits[w] = 0u;
    // region counts: read in parallel (up to kMaxRegions staged), then prefix offsets
    __shared__ int sh_cnt[kMaxRegions];
    // a region never holds more than cap records; the clamp keeps every read in
    // bounds even when a landmark pass gave up before writing its counts
    auto region_count = [&](int sp) { return (int)min((long long)max(cnts[sp], 0), cap); };
    for (int sp = threadIdx.x; sp < kMaxRegions; sp += blockDim.x) sh_cnt[sp] = sp < splits ? region_count(sp) : 0;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0;
        for (int sp = 0; sp < splits; ++sp) {
            const int c = sp < kMaxRegions ? sh_cnt[sp] : region_count(sp);
            if (sp < kMaxRegions) sh_off[sp] = tot;
            tot += c;
        }
        sh_total = tot;
    }
    __syncthreads();
    const int total = sh_total;
    int32_t* dst = I + ((size_t)bh * m + i) * k;
    if (total < k) {  // cannot happen when the threshold holds; flag it
        if (threadIdx.x == 0) set_status(status, kStBounds);
        for (int t = threadIdx.x; t < k; t += blockDim.x) dst[t] = t;
        return;
    }
    CandSrc cs{nullptr, nullptr, 0, base, cnts, splits, cap};
    if (total <= stage_cap && splits <= kMaxRegions) {  // one read of the records, the passes run in shared memory
        // flat over all records (independent loads): record gi sits in the last
        // region whose offset is <= gi (empty regions share the next offset)
        for (int gi = threadIdx.x; gi < total; gi += blockDim.x) {
            int lo = 0, hi = splits - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sh_off[mid] <= gi) lo = mid;
                else hi = mid - 1;
            }
            const int2 r = base[lo * cap + (gi - sh_off[lo])];
            skey[gi] = order_key(__int_as_float(r.x));
            sidx[gi] = r.y;
        }
        __syncthreads();
        cs.skey = skey;
        cs.sidx = sidx;
        cs.n = total;
    }
    int rem, n_eq;
    const uint32_t v = radix_select(cs, k, [](uint32_t u, int, bool* ok) { *ok = true; return u; }, hist, &rem, &n_eq);
    // among keys equal to v keep the rem lowest indices: the rem-th largest of ~index
    uint32_t idx_cut = 0u;  // take every key equal to v
    if (rem < n_eq) {
        int r2, e2;
        idx_cut = radix_select(cs, rem, [v](uint32_t u, int j, bool* ok) { *ok = (u == v); return ~(uint32_t)j; },
                               hist, &r2, &e2);
    }
    cs.each([&](uint32_t u, int j) {
        const bool take = u > v || (u == v && ~(uint32_t)j >= idx_cut);
        if (take && j >= 0 && j < N) atomicOr(&bits[j >> 5], 1u << (j & 31));
    });
    __syncthreads();
    // ascending write-out
    int out = 0;
    for (int w0 = 0; w0 < nwords; w0 += blockDim.x) {
        const int w = w0 + threadIdx.x;
        const uint32_t word = w < nwords ? bits[w] : 0u;
        int tot;
        const int pos = block_excl_scan(__popc(word), tmp, &tot);
        uint32_t x = word;
        int o = out + pos;
        while (x) {
            const int b = __ffs(x) - 1;
            x &= x - 1;
            if (o < k) dst[o] = (w << 5) + b;
            ++o;
        }
        out += tot;
    }
    if (threadIdx.x == 0 && out != k) set_status(status, kStBounds);
}

cudaError_t launch_sample_threshold(const float* Ssamp, long long rows, int n_samp, int k, float* thr,
                                    cudaStream_t st) {
    // a warp per row is faster for many rows of at most 4096 samples, a block
    // per row for fewer rows (under ~16 per SM: a few heads) or longer ones
    if (n_samp <= 4096 && rows >= 16LL * num_sms()) {
        k_sample_threshold_w<<<(unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock), 32 * kRowsPerBlock, 0, st>>>(
            Ssamp, rows, n_samp, k, thr);
        count_launch();
        return cudaGetLastError();
    }
    const int bytes = n_samp * 4;
    const int staged = bytes <= 96 * 1024;
    if (staged) {
        cudaError_t e0 = cudaFuncSetAttribute(k_sample_threshold, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e0 != cudaSuccess) return e0;
    }
    k_sample_threshold<<<(unsigned)rows, 512, staged ? bytes : 0, st>>>(Ssamp, n_samp, k, thr, staged);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_topk_cand(const int2* cand, const int* ccount, int splits, long long cap, int BH, int m, int m_pad,
                             int N, int k, long long expect, int32_t* I, int* status, cudaStream_t st) {
    const int bitmap = ((N + 31) / 32) * 4;
    // stage about three times the expected candidate count (12k at most) so
    // that several rows fit on an SM; larger rows read from global memory
    const long long want = std::min<long long>(12288, std::max<long long>(1024, 3 * expect));
    const int stage_cap = (int)std::max<long long>(0, std::min<long long>(want, (160 * 1024 - bitmap) / 8));
    const int smem = bitmap + stage_cap * 8;
    // rows of 2^17 keys or more (4096 bitmap words, several times more candidates
    // per row) run faster with 1024 threads, smaller ones with 512 (measured)
    auto run = [&](auto kern, int tb) -> cudaError_t {
        cudaError_t e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e0 != cudaSuccess) return e0;
        kern<<<dim3(m, BH), tb, smem, st>>>(cand, ccount, splits, cap, m, m_pad, N, k, stage_cap, I, status);
        return cudaSuccess;
    };
    cudaError_t e0 = N >= (1 << 17) ? run(k_topk_cand<1024>, 1024) : run(k_topk_cand<512>, 512);
    if (e0 != cudaSuccess) return e0;
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_topk_dense(const float* S, long long rows, int N, int k, int32_t* I, cudaStream_t st) {
    k_topk_dense<<<(unsigned)rows, 512, 0, st>>>(S, N, k, I);
    count_launch();
    return cudaGetLastError();
}

}  // namespace mita
