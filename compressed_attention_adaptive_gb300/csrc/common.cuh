// Shared device helpers of libmita: element access, ordered keys, block scans
// and the device status word. No method arithmetic lives here.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mita {

// Device status codes (mirror mita_status).
enum : int { kStOk = 0, kStTimeout = 5, kStBounds = 6 };

// Internal flag bit in Dims::flags (never a public MITA_FLAG_*): the call is
// one part of a larger one, so its first kernel keeps the device status word.
constexpr unsigned kFlagKeepStatus = 1u << 30;

// Problem dimensions after validation (1-D pooling is a 1 x N grid).
struct Dims {
    int B, H, BH, N, d, m, k, s;
    int gh, gw, lh, lw;
    float scale;       // softmax scale (resolved, never 0)
    unsigned flags;
    int dtype;         // 0 f32, 1 bf16
    bool shared;       // shared slots present
    bool causal;       // causal variant (1-D pooling only)
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Record the first device-side error of a call (later ones are dropped).
__device__ __forceinline__ void set_status(int* st, int code) { atomicCAS(st, 0, code); }

// Monotone map float -> uint32 (larger float -> larger key). -0.0 is folded
// onto +0.0 first so that equal scores compare equal and tie on the index.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide reductions; `red` needs blockDim.x / 32 floats of shared memory.
__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = -INFINITY;
    for (int i = 0; i < nw; ++i) r = fmaxf(r, red[i]);
    return r;
}
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = 0.0f;
    for (int i = 0; i < nw; ++i) r += red[i];
    return r;
}

// Exclusive prefix sum of one int per thread across the block; returns the
// thread's offset and writes the block total to *total. `tmp` needs
// blockDim.x / 32 + 1 ints of shared memory.
__device__ __forceinline__ int block_excl_scan(int v, int* tmp, int* total) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (l >= o) x += y;
    }
    __syncthreads();
    if (l == 31) tmp[w] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int i = 0; i < nw; ++i) { int t = tmp[i]; tmp[i] = acc; acc += t; }
        tmp[nw] = acc;
    }
    __syncthreads();
    *total = tmp[nw];
    return tmp[w] + x - v;
}

// Causal variant (1-D pooling): landmark i's bin is complete for query t once
// its end hi_i = ceil((i + 1) N / m) <= t + 1; the number of such landmarks.
__host__ __device__ __forceinline__ int landmarks_complete(int t, int N, int m) {
    // largest i + 1 with (i + 1) N <= (t + 1) m, i.e. floor((t + 1) m / N)
    return (int)(((long long)(t + 1) * m) / N);
}

// Adaptive-average-pooling bin [lo, hi) of bin i when L cells pool to P bins.
__host__ __device__ __forceinline__ void pool_bin(int i, int L, int P, int* lo, int* hi) {
    *lo = (int)(((long long)i * L) / P);
    *hi = (int)((((long long)(i + 1) * L) + P - 1) / P);
}

}  // namespace mita
