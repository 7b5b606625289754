// CUDA-core kernels of the MiTA forward pass: landmark pooling (used by every
// path), and an fp32 implementation of the remaining steps used for float32
// inputs, for head dims the tensor-core path does not take, and as a second
// GPU implementation for cross-checks.
//
// Steps follow "MiTA Attention: Efficient Fast-Weight Scaling via a Mixture of
// Top-k Activations" (gist.science summaries): landmark queries by adaptive
// average pooling, the shared expert Vt = Atten(Qt, K, V) and the top-k sets
// I_i (Arabic edition, section 2), and the per-query softmax over
// K* = [Qt, K_(e1), ..., K_(es)], V* = [Vt, V_(e1), ..., V_(es)] (Dutch
// edition, "Wiskundige Formulering").
#include "common.cuh"
#include "internal.h"

namespace mita {

// ------------------------------------------------------------------ pooling

// Qt[bh][i] = mean of Q over the adaptive bin of landmark i (1-D bins are the
// 1 x N grid case). One block per (landmark, head); 256 threads split into
// d/8 channel groups x token lanes, 8 channels per thread. Also writes the
// bf16 split Qt = hi + lo (rows m..m_pad-1 zeroed) when hi/lo are given.
template <typename T>
__global__ void __launch_bounds__(256) k_pool(const T* __restrict__ Q, float* __restrict__ Qt,
                                              __nv_bfloat16* __restrict__ hi, __nv_bfloat16* __restrict__ lo,
                                              int m_pad, Dims D, int* __restrict__ status) {
    __shared__ float red[256 * 8];
    const int i = blockIdx.x, bh = blockIdx.y, d = D.d;
    // the first kernel of every call resets the device status word (not in the
    // later parts of a call split into several)
    if (status && !(D.flags & kFlagKeepStatus) && i == 0 && bh == 0 && threadIdx.x == 0) *status = kStOk;
    const int ncg = d >> 3, nlanes = 256 / ncg;
    const int cg = threadIdx.x % ncg, tl = threadIdx.x / ncg;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    int cnt = 1;
    if (i < D.m) {
        int r0, r1, c0, c1;
        pool_bin(i / D.lw, D.gh, D.lh, &r0, &r1);
        pool_bin(i % D.lw, D.gw, D.lw, &c0, &c1);
        const int nc = c1 - c0;
        cnt = (r1 - r0) * nc;
        if (tl < nlanes) {
            const T* base = Q + (size_t)bh * D.N * d + cg * 8;
            // token t of the bin is (row r0 + t / nc, column c0 + t % nc); the
            // lane walks t = tl, tl + nlanes, ... keeping (row, column) by steps,
            // four tokens' loads in flight before their sums
            int r = tl / nc, c = tl % nc;
            for (int t = tl; t < cnt; t += 4 * nlanes) {
                uint4 v[4][sizeof(T) / 2];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (t + u * nlanes < cnt) {
                        const T* p = base + ((size_t)(r0 + r) * D.gw + (c0 + c)) * d;
#pragma unroll
                        for (int w = 0; w < (int)(sizeof(T) / 2); ++w) v[u][w] = reinterpret_cast<const uint4*>(p)[w];
                    }
                    c += nlanes;
                    while (c >= nc) {
                        c -= nc;
                        ++r;
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (t + u * nlanes >= cnt) break;
                    if constexpr (sizeof(T) == 2) {
                        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v[u][0]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 f = __bfloat1622float2(b2[j]);
                            acc[2 * j] += f.x;
                            acc[2 * j + 1] += f.y;
                        }
                    } else {
                        const float* f = reinterpret_cast<const float*>(&v[u][0]);
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[j] += f[j];
                    }
                }
            }
        }
    }
    if (tl < nlanes)
#pragma unroll
        for (int j = 0; j < 8; ++j) red[tl * d + cg * 8 + j] = acc[j];
    __syncthreads();
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float v = 0.0f;
        if (i < D.m) {
            for (int t = 0; t < nlanes; ++t) v += red[t * d + c];
            v /= (float)cnt;
            Qt[((size_t)bh * D.m + i) * d + c] = v;
        }
        if (hi) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v);
            hi[((size_t)bh * m_pad + i) * d + c] = h;
            lo[((size_t)bh * m_pad + i) * d + c] = __float2bfloat16_rn(v - __bfloat162float(h));
        }
    }
}

// ---------------------------------------------------------- fp32 NT GEMM

// C[b][i][j] = sum_c A[b][i][c] * B[b][j][c] (both operands row-major with
// the reduction dim contiguous), 64 x 64 tiles, 4 x 4 outputs per thread.
template <typename TA, typename TB>
__global__ void __launch_bounds__(256) k_gemm_nt(const TA* __restrict__ A, long long sA, const TB* __restrict__ B,
                                                 long long sB, float* __restrict__ C, long long sC, int M, int Nn,
                                                 int K) {
    __shared__ __align__(16) float As[16][68];
    __shared__ __align__(16) float Bs[16][68];
    const int b = blockIdx.z, m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const TA* Ab = A + b * sA;
    const TB* Bb = B + b * sB;
    const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = t + 256 * r, row = e >> 4, kk = e & 15;
            const int gk = k0 + kk;
            As[kk][row] = (m0 + row < M && gk < K) ? to_f(Ab[(size_t)(m0 + row) * K + gk]) : 0.0f;
            Bs[kk][row] = (n0 + row < Nn && gk < K) ? to_f(Bb[(size_t)(n0 + row) * K + gk]) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bw[j], acc[i][j]);
        }
        __syncthreads();
    }
    float* Cb = C + b * sC;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = m0 + ty * 4 + i, c = n0 + tx * 4 + j;
            if (r < M && c < Nn) Cb[(size_t)r * Nn + c] = acc[i][j];
        }
}

// --------------------------------------------------------- shared expert

// Per landmark row of raw scores S (length N): stats = (max of scale*s,
// 1 / sum exp(scale*s - max)); over the keys of the landmark's prefix
// j < hi_i only in the causal variant.
__global__ void __launch_bounds__(256) k_row_softmax_stats(const float* __restrict__ S, int N, int m, int causal,
                                                           float scale, float2* __restrict__ stats) {
    __shared__ float red[32];
    const float* s = S + (size_t)blockIdx.x * N;
    int lo, hi = N;
    if (causal) pool_bin(blockIdx.x % m, N, m, &lo, &hi);
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < hi; j += blockDim.x) mx = fmaxf(mx, scale * s[j]);
    mx = block_max(mx, red);
    float sum = 0.0f;
    for (int j = threadIdx.x; j < hi; j += blockDim.x) sum += expf(scale * s[j] - mx);
    sum = block_sum(sum, red);
    if (threadIdx.x == 0) stats[blockIdx.x] = make_float2(mx, 1.0f / sum);
}

// Vt[b][i][c] = sum_j softmax_j(scale * S[b][i][j]) V[b][j][c]; 64 x 64 output
// tiles, the probabilities formed on the fly from S and the row stats.
template <typename T>
__global__ void __launch_bounds__(256) k_pv_simt(const float* __restrict__ S, const float2* __restrict__ stats,
                                                 const T* __restrict__ V, float* __restrict__ Vt, int m, int N,
                                                 int d, float scale, int causal) {
    __shared__ __align__(16) float As[16][68];
    __shared__ __align__(16) float Bs[16][68];
    const int b = blockIdx.z, m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const float* Sb = S + (size_t)b * m * N;
    const float2* st = stats + (size_t)b * m;
    const T* Vb = V + (size_t)b * N * d;
    const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < N; k0 += 16) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = t + 256 * r;
            {
                const int row = e >> 4, kk = e & 15, gi = m0 + row, gk = k0 + kk;
                float p = 0.0f;
                int lo, hi = N;
                if (causal && gi < m) pool_bin(gi, N, m, &lo, &hi);
                if (gi < m && gk < hi) {
                    const float2 sx = st[gi];
                    p = expf(scale * Sb[(size_t)gi * N + gk] - sx.x) * sx.y;
                }
                As[kk][row] = p;
            }
            {
                const int kk = e >> 6, col = e & 63, gk = k0 + kk, gc = n0 + col;
                Bs[kk][col] = (gk < N && gc < d) ? to_f(Vb[(size_t)gk * d + gc]) : 0.0f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bw[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = m0 + ty * 4 + i, c = n0 + tx * 4 + j;
            if (r < m && c < d) Vt[((size_t)b * m + r) * d + c] = acc[i][j];
        }
}

// ---------------------------------------------------------------- routing

// One thread per query: the s largest routing scores of its row R[q][0..m)
// (ties to the lower landmark index), written by descending score.
__global__ void k_route_dense(const float* __restrict__ R, long long nq, int m, int s, int32_t* __restrict__ E) {
    const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= nq) return;
    const float* r = R + q * m;
    uint32_t bu[kMaxS];
    int bi[kMaxS];
    for (int t = 0; t < s; ++t) { bu[t] = 0u; bi[t] = -1; }
    for (int i = 0; i < m; ++i) {
        const uint32_t u = order_key(r[i]);
        if (u <= bu[s - 1] && bi[s - 1] >= 0) continue;
        int pos = s - 1;
        while (pos > 0 && (bi[pos - 1] < 0 || u > bu[pos - 1])) {
            bu[pos] = bu[pos - 1];
            bi[pos] = bi[pos - 1];
            --pos;
        }
        bu[pos] = u;
        bi[pos] = i;
    }
    for (int t = 0; t < s; ++t) E[q * s + t] = bi[t];
}

// ----------------------------------------------------------------- output

// One block per query: one softmax over the m shared slots (keys Qt, values
// Vt) and the s*k routed slots (keys/values of the routed experts' sets,
// duplicates kept), fp32 throughout.
template <typename T>
__global__ void __launch_bounds__(128) k_out_simt(const T* __restrict__ Q, const T* __restrict__ K,
                                                  const T* __restrict__ V, const float* __restrict__ Qt,
                                                  const float* __restrict__ Vt, const int32_t* __restrict__ I,
                                                  const int32_t* __restrict__ E, T* __restrict__ O, Dims D,
                                                  int* __restrict__ status) {
    extern __shared__ float sm[];
    __shared__ float red[32];
    const int d = D.d, m_sh = D.shared ? D.m : 0, nslot = m_sh + D.s * D.k;
    float* qv = sm;
    float* lg = sm + d;
    int* src = reinterpret_cast<int*>(lg + nslot);
    const long long qg = blockIdx.x;
    const int bh = (int)(qg / D.N);
    const int tq = (int)(qg % D.N);  // the query's position
    // causal variant: the shared slots of complete bins, routed keys up to tq
    const int m_ok = D.causal ? landmarks_complete(tq, D.N, D.m) : D.m;
    const T* Kb = K + (size_t)bh * D.N * d;
    const T* Vb = V + (size_t)bh * D.N * d;
    const float* Qtb = Qt + (size_t)bh * D.m * d;
    const float* Vtb = Vt + (size_t)bh * D.m * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) qv[c] = to_f(Q[qg * d + c]);
    __syncthreads();
    float mx = -INFINITY;
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) {
        float dot = 0.0f;
        int j;
        if (u < m_sh) {
            if (u >= m_ok) {
                src[u] = INT_MIN;
                lg[u] = -INFINITY;
                continue;
            }
            j = -1 - u;
            const float* kr = Qtb + (size_t)u * d;
            for (int c = 0; c < d; ++c) dot = fmaf(qv[c], kr[c], dot);
        } else {
            const int v = u - m_sh, slot = v / D.k, t = v % D.k;
            const int e = E[qg * D.s + slot];
            j = (e >= 0 && e < D.m) ? I[((size_t)bh * D.m + e) * D.k + t] : -1;
            if (e < 0 || e >= D.m || j < 0 || j >= D.N) {
                set_status(status, kStBounds);
                src[u] = INT_MIN;
                lg[u] = -INFINITY;
                continue;
            }
            if (D.causal && j > tq) {
                src[u] = INT_MIN;
                lg[u] = -INFINITY;
                continue;
            }
            const T* kr = Kb + (size_t)j * d;
            for (int c = 0; c < d; ++c) dot = fmaf(qv[c], to_f(kr[c]), dot);
        }
        src[u] = j;
        lg[u] = D.scale * dot;
        mx = fmaxf(mx, lg[u]);
    }
    mx = block_max(mx, red);
    float sum = 0.0f;
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) {
        const float p = (src[u] == INT_MIN) ? 0.0f : expf(lg[u] - mx);
        lg[u] = p;
        sum += p;
    }
    sum = block_sum(sum, red);
    const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;  // no slot (causal only): a zero row
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float acc = 0.0f;
        for (int u = 0; u < nslot; ++u) {
            const int j = src[u];
            if (j == INT_MIN) continue;
            const float v = (j < 0) ? Vtb[(size_t)(-1 - j) * d + c] : to_f(Vb[(size_t)j * d + c]);
            acc = fmaf(lg[u], v, acc);
        }
        O[qg * d + c] = from_f<T>(acc * inv);
    }
}

// ----------------------------------------------------------------- launch

template <typename T>
static cudaError_t pool_t(const Dims& D, const void* Q, float* Qt, __nv_bfloat16* hi, __nv_bfloat16* lo, int m_pad,
                          int* status, cudaStream_t st) {
    dim3 grid(hi ? m_pad : D.m, D.BH);
    k_pool<T><<<grid, 256, 0, st>>>((const T*)Q, Qt, hi, lo, m_pad, D, status);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pool(const Dims& D, const void* Q, float* Qt, __nv_bfloat16* hi, __nv_bfloat16* lo, int m_pad,
                        int* status, cudaStream_t st) {
    return D.dtype == 0 ? pool_t<float>(D, Q, Qt, hi, lo, m_pad, status, st)
                        : pool_t<__nv_bfloat16>(D, Q, Qt, hi, lo, m_pad, status, st);
}

template <typename T>
static cudaError_t select_simt_t(const Dims& D, const void* Q, const void* K, const float* Qt, float* S, float* R,
                                 int32_t* I, int32_t* E, cudaStream_t st) {
    // landmark scores S = Qt K^T (raw), then the top-k sets
    {
        dim3 grid((D.N + 63) / 64, (D.m + 63) / 64, D.BH);
        k_gemm_nt<float, T><<<grid, 256, 0, st>>>(Qt, (long long)D.m * D.d, (const T*)K, (long long)D.N * D.d, S,
                                                  (long long)D.m * D.N, D.m, D.N, D.d);
    }
    count_launch();
    cudaError_t e = launch_topk_dense(S, (long long)D.BH * D.m, D.N, D.k, I, st);
    if (e != cudaSuccess) return e;
    // routing scores R = Q Qt^T, then the top-s routes per query
    if (E) {
        dim3 grid((D.m + 63) / 64, (D.N + 63) / 64, D.BH);
        k_gemm_nt<T, float><<<grid, 256, 0, st>>>((const T*)Q, (long long)D.N * D.d, Qt, (long long)D.m * D.d, R,
                                                  (long long)D.N * D.m, D.N, D.m, D.d);
        const long long nq = (long long)D.BH * D.N;
        k_route_dense<<<(unsigned)((nq + 255) / 256), 256, 0, st>>>(R, nq, D.m, D.s, E);
        count_launch(2);
    }
    return cudaGetLastError();
}

cudaError_t launch_select_simt(const Dims& D, const void* Q, const void* K, const float* Qt, float* S, float* R,
                               int32_t* I, int32_t* E, cudaStream_t st) {
    return D.dtype == 0 ? select_simt_t<float>(D, Q, K, Qt, S, R, I, E, st)
                        : select_simt_t<__nv_bfloat16>(D, Q, K, Qt, S, R, I, E, st);
}

template <typename T>
static cudaError_t shared_simt_t(const Dims& D, const void* V, const float* S, float2* stats, float* Vt,
                                 cudaStream_t st) {
    k_row_softmax_stats<<<D.BH * D.m, 256, 0, st>>>(S, D.N, D.m, D.causal ? 1 : 0, D.scale, stats);
    dim3 grid((D.d + 63) / 64, (D.m + 63) / 64, D.BH);
    k_pv_simt<T><<<grid, 256, 0, st>>>(S, stats, (const T*)V, Vt, D.m, D.N, D.d, D.scale, D.causal ? 1 : 0);
    count_launch(2);
    return cudaGetLastError();
}

cudaError_t launch_row_stats(const Dims& D, const float* S, float2* stats, cudaStream_t st) {
    k_row_softmax_stats<<<D.BH * D.m, 256, 0, st>>>(S, D.N, D.m, D.causal ? 1 : 0, D.scale, stats);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_shared_simt(const Dims& D, const void* V, const float* S, float2* stats, float* Vt,
                               cudaStream_t st) {
    return D.dtype == 0 ? shared_simt_t<float>(D, V, S, stats, Vt, st)
                        : shared_simt_t<__nv_bfloat16>(D, V, S, stats, Vt, st);
}

size_t out_simt_smem(const Dims& D) {
    const size_t nslot = (size_t)(D.shared ? D.m : 0) + (size_t)D.s * D.k;
    return (size_t)D.d * 4 + nslot * 8;
}

template <typename T>
static cudaError_t out_simt_t(const Dims& D, const void* Q, const void* K, const void* V, const float* Qt,
                              const float* Vt, const int32_t* I, const int32_t* E, void* O, int* status,
                              cudaStream_t st) {
    const size_t smem = out_simt_smem(D);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_out_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    k_out_simt<T><<<(unsigned)((long long)D.BH * D.N), 128, smem, st>>>((const T*)Q, (const T*)K, (const T*)V, Qt,
                                                                         Vt, I, E, (T*)O, D, status);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_out_simt(const Dims& D, const void* Q, const void* K, const void* V, const float* Qt,
                            const float* Vt, const int32_t* I, const int32_t* E, void* O, int* status,
                            cudaStream_t st) {
    return D.dtype == 0 ? out_simt_t<float>(D, Q, K, V, Qt, Vt, I, E, O, status, st)
                        : out_simt_t<__nv_bfloat16>(D, Q, K, V, Qt, Vt, I, E, O, status, st);
}

}  // namespace mita
