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
#include "common.cuh"
#include "internal.h"

namespace mita {

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
        if (threadIdx.x == 0) {
            int acc = 0, b = 255;
            for (; b > 0; --b) {
                if (acc + (int)hist[b] >= rem) break;
                acc += (int)hist[b];
            }
            sh_prefix = prefix | ((uint32_t)b << shift);
            sh_rem = rem - acc;
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
                                                          float* __restrict__ thr) {
    __shared__ unsigned hist[256];
    const size_t row = blockIdx.x;
    const float* s = Ssamp + row * n_samp;
    uint32_t v;
    int rem;
    radix_kth(n_samp, k, [&](int j) { return order_key(s[j]); }, hist, &v, &rem);
    if (threadIdx.x == 0) {
        const float t = key_float(v);
        thr[row] = t - 1e-3f * fmaxf(1.0f, fabsf(t));
    }
}

// Candidates of one row: `splits` regions of (score, key) records, region sp
// holding counts[sp] records at base + sp * cap.
struct CandRow {
    const int2* base;
    const int* counts;
    int splits;
    long long cap;
    template <typename F> __device__ __forceinline__ void each(F f) const {
        for (int sp = 0; sp < splits; ++sp) {
            const int c = counts[sp];
            const int2* b = base + sp * cap;
            for (int t = threadIdx.x; t < c; t += blockDim.x) f(b[t]);
        }
    }
};

// Exact top-k of one landmark row from its candidates: radix select of the
// k-th largest score, the lowest key indices among scores equal to it, then
// the chosen keys marked in a bitmap and written out in ascending order.
// Dynamic shared memory: ceil(N / 32) words.
__global__ void __launch_bounds__(512) k_topk_cand(const int2* __restrict__ cand, const int* __restrict__ ccount,
                                                   int splits, long long cap, int m, int m_pad, int N, int k,
                                                   int32_t* __restrict__ I, int* __restrict__ status) {
    extern __shared__ uint32_t bits[];
    __shared__ unsigned hist[256];
    __shared__ int tmp[33];
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_rem, sh_total, sh_eq;
    const int bh = blockIdx.y, i = blockIdx.x;
    const size_t rrow = (size_t)bh * m_pad + i;
    CandRow cr{cand + rrow * splits * cap, ccount + rrow * splits, splits, cap};
    const int nwords = (N + 31) >> 5;
    for (int w = threadIdx.x; w < nwords; w += blockDim.x) bits[w] = 0u;
    if (threadIdx.x == 0) {
        int tot = 0;
        for (int sp = 0; sp < splits; ++sp) tot += ccount[rrow * splits + sp];
        sh_total = tot;
    }
    __syncthreads();
    int32_t* dst = I + ((size_t)bh * m + i) * k;
    if (sh_total < k) {  // cannot happen when the threshold holds; flag it
        if (threadIdx.x == 0) set_status(status, kStBounds);
        for (int t = threadIdx.x; t < k; t += blockDim.x) dst[t] = t;
        return;
    }
    // k-th largest score key v, and how many keys equal to v are needed (rem)
    uint32_t prefix = 0u, mask = 0u;
    int rem = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
        __syncthreads();
        cr.each([&](int2 c) {
            const uint32_t u = order_key(__int_as_float(c.x));
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
        });
        __syncthreads();
        if (threadIdx.x == 0) {
            int acc = 0, b = 255;
            for (; b > 0; --b) {
                if (acc + (int)hist[b] >= rem) break;
                acc += (int)hist[b];
            }
            sh_prefix = prefix | ((uint32_t)b << shift);
            sh_rem = rem - acc;
            sh_eq = (int)hist[b];
        }
        __syncthreads();
        prefix = sh_prefix;
        rem = sh_rem;
        mask |= 0xFFu << shift;
    }
    const uint32_t v = prefix;
    const int n_eq = sh_eq;  // keys equal to v among the candidates
    // among keys equal to v keep the rem lowest indices: the rem-th largest of ~index
    uint32_t idx_cut = 0xFFFFFFFFu;  // ~index >= idx_cut  <=> index <= ~idx_cut
    if (rem < n_eq) {
        uint32_t p2 = 0u, m2 = 0u;
        int r2 = rem;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
            __syncthreads();
            cr.each([&](int2 c) {
                if (order_key(__int_as_float(c.x)) != v) return;
                const uint32_t u = ~(uint32_t)c.y;
                if ((u & m2) == p2) atomicAdd(&hist[(u >> shift) & 255u], 1u);
            });
            __syncthreads();
            if (threadIdx.x == 0) {
                int acc = 0, b = 255;
                for (; b > 0; --b) {
                    if (acc + (int)hist[b] >= r2) break;
                    acc += (int)hist[b];
                }
                sh_prefix = p2 | ((uint32_t)b << shift);
                sh_rem = r2 - acc;
            }
            __syncthreads();
            p2 = sh_prefix;
            r2 = sh_rem;
            m2 |= 0xFFu << shift;
        }
        idx_cut = p2;
    } else {
        idx_cut = 0u;  // take every key equal to v
    }
    cr.each([&](int2 c) {
        const uint32_t u = order_key(__int_as_float(c.x));
        const bool take = u > v || (u == v && ~(uint32_t)c.y >= idx_cut);
        if (take && c.y >= 0 && c.y < N) atomicOr(&bits[c.y >> 5], 1u << (c.y & 31));
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
    k_sample_threshold<<<(unsigned)rows, 512, 0, st>>>(Ssamp, n_samp, k, thr);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_topk_cand(const int2* cand, const int* ccount, int splits, long long cap, int BH, int m, int m_pad,
                             int N, int k, int32_t* I, int* status, cudaStream_t st) {
    const int smem = ((N + 31) / 32) * 4;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_topk_cand, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    k_topk_cand<<<dim3(m, BH), 512, smem, st>>>(cand, ccount, splits, cap, m, m_pad, N, k, I, status);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_topk_dense(const float* S, long long rows, int N, int k, int32_t* I, cudaStream_t st) {
    k_topk_dense<<<(unsigned)rows, 512, 0, st>>>(S, N, k, I);
    count_launch();
    return cudaGetLastError();
}

}  // namespace mita
