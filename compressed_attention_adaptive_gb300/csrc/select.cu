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

cudaError_t launch_topk_dense(const float* S, long long rows, int N, int k, int32_t* I, cudaStream_t st) {
    k_topk_dense<<<(unsigned)rows, 512, 0, st>>>(S, N, k, I);
    return cudaGetLastError();
}

}  // namespace mita
