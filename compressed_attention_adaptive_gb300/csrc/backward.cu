// Backward pass of the MiTA forward, on CUDA cores in fp32.
//
// The pages ("MiTA Attention: Efficient Fast-Weight Scaling via a Mixture of
// Top-k Activations", gist.science summaries) describe the forward pass and
// report training speed, but print no backward pass. This is the chain rule
// through the forward's steps with the expert sets I and the routes E held
// fixed (a top-k choice is piecewise constant):
//   per query t over its slots u (the m shared slots, then the k keys of each
//   routed expert): P_t = softmax(tau q_t . key_u), dP_tu = dO_t . val_u,
//   D_t = sum_u P_tu dP_tu, dZ_tu = P_tu (dP_tu - D_t);
//   dq_t = tau sum_u dZ_tu key_u; a routed key j gets dk_j += tau dZ_tu q_t,
//   dv_j += P_tu dO_t; a shared slot i gets dQt_i += tau dZ_ti q_t,
//   dVt_i += P_ti dO_t;
//   the shared expert Vt = A V, A = softmax(tau Qt K^T):
//   dS = A o (dVt V^T - rowdot(dVt, Vt)), dQt += tau dS K, dK += tau dS^T Qt,
//   dV += A^T dVt;
//   the landmarks: dq_t += dQt_i / |bin_i| for the bins i that hold t.
// Per-query work runs one block per query; the reductions over queries and
// keys are fp32 GEMMs on CUDA cores; routed keys accumulate with atomics.
#include "internal.h"

namespace mita {
namespace {

// C[b] (+)= alpha * sum_kk A(i, kk) B(kk, j): A(i, kk) at A[i * a_i + kk * a_k],
// B(kk, j) at B[kk * b_k + j * b_j]; C row-major M x Nn. 64 x 64 tiles,
// 4 x 4 outputs per thread, operands widened to fp32 as they are staged. With
// ksplit > 1 (a long reduction and few output tiles) blockIdx.z also picks a
// range of the reduction and the results are added into C atomically.
template <typename TA, typename TB>
__global__ void __launch_bounds__(256) k_gemm_strided(const TA* __restrict__ A, long long sA, long long a_i,
                                                      long long a_k, const TB* __restrict__ B, long long sB,
                                                      long long b_k, long long b_j, float* __restrict__ C,
                                                      long long sC, int M, int Nn, int K, float alpha,
                                                      int accumulate, int ksplit) {
    __shared__ __align__(16) float As[16][68];
    __shared__ __align__(16) float Bs[16][68];
    const int b = blockIdx.z / ksplit, ks = blockIdx.z % ksplit;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int kc = (K + ksplit - 1) / ksplit, kb = ks * kc, ke = min(K, kb + kc);
    const TA* Ab = A + b * sA;
    const TB* Bb = B + b * sB;
    const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
    float acc[4][4] = {};
    for (int k0 = kb; k0 < ke; k0 += 16) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = t + 256 * r, row = e >> 4, kk = e & 15, gk = k0 + kk;
            As[kk][row] = (m0 + row < M && gk < ke) ? to_f(Ab[(m0 + row) * a_i + gk * a_k]) : 0.0f;
            Bs[kk][row] = (n0 + row < Nn && gk < ke) ? to_f(Bb[gk * b_k + (n0 + row) * b_j]) : 0.0f;
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
            if (r < M && c < Nn) {
                float* dst = Cb + (size_t)r * Nn + c;
                if (ksplit > 1) atomicAdd(dst, alpha * acc[i][j]);
                else *dst = accumulate ? *dst + alpha * acc[i][j] : alpha * acc[i][j];
            }
        }
}

template <typename TA, typename TB>
cudaError_t gemm(const TA* A, long long sA, long long a_i, long long a_k, const TB* B, long long sB, long long b_k,
                 long long b_j, float* C, long long sC, int M, int Nn, int K, float alpha, bool accumulate, int batch,
                 cudaStream_t st) {
    const long long tiles = (long long)((Nn + 63) / 64) * ((M + 63) / 64) * batch;
    int ksplit = 1;
    while (tiles * ksplit < 2 * 152 && (K + 2 * ksplit - 1) / (2 * ksplit) >= 256) ksplit *= 2;
    cudaError_t e;
    if (ksplit > 1 && !accumulate) {  // the split results add up into a cleared C
        for (int b = 0; b < batch; ++b)
            if ((e = cudaMemsetAsync(C + b * sC, 0, sizeof(float) * (size_t)M * Nn, st))) return e;
    }
    dim3 grid((Nn + 63) / 64, (M + 63) / 64, batch * ksplit);
    k_gemm_strided<TA, TB><<<grid, 256, 0, st>>>(A, sA, a_i, a_k, B, sB, b_k, b_j, C, sC, M, Nn, K, alpha,
                                                 accumulate ? 1 : 0, ksplit);
    count_launch();
    return cudaGetLastError();
}

// The shared expert's attention A = softmax(scale Qt K^T) from the raw scores
// S and the row statistics (max of scale * s, 1 / sum), in place.
__global__ void k_bwd_shared_attn(float* __restrict__ S, const float2* __restrict__ stats, long long rows, int N,
                                  float scale) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= rows * N) return;
    const float2 st = stats[e / N];
    S[e] = expf(scale * S[e] - st.x) * st.y;
}

// One block of 4 warps per query: its slots' logits and probabilities again
// (as in the forward), dP = dO . val, D = sum P dP, dZ = P (dP - D); dq of the
// query; the shared slots' P and dZ (for the reductions over queries) and the
// routed slots' P and dZ (for the per-expert reductions into dK, dV). A warp
// takes one slot at a time: its key and value rows are read whole by the
// warp (DD / 32 elements per lane) and the dot products reduced across it.
template <typename T, int DD>
__device__ __forceinline__ void load_row(const T* __restrict__ src, float (&x)[DD / 32], int lane) {
    constexpr int CPL = DD / 32;
    if constexpr (sizeof(T) == 2) {
        if constexpr (CPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * CPL);
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(src + lane * CPL);
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw));
            x[0] = a.x; x[1] = a.y;
        }
    } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) x[c] = to_f(src[lane * CPL + c]);
    }
}

template <typename T, int DD>
__global__ void __launch_bounds__(128) k_bwd_query(const T* __restrict__ Q, const T* __restrict__ K,
                                                   const T* __restrict__ V, const T* __restrict__ dO,
                                                   const float* __restrict__ Qt, const float* __restrict__ Vt,
                                                   const int32_t* __restrict__ I, const int32_t* __restrict__ E,
                                                   float* __restrict__ dQacc, float* __restrict__ Psh,
                                                   float* __restrict__ dZsh, float* __restrict__ Pr,
                                                   float* __restrict__ dZr, Dims D, int* __restrict__ status) {
    constexpr int CPL = DD / 32;
    extern __shared__ float sm[];
    __shared__ float red[32];
    __shared__ float wacc[4][DD];
    const int m_sh = D.shared ? D.m : 0, nslot = m_sh + D.s * D.k;
    float* lg = sm;               // logits, then P
    float* dp = lg + nslot;       // dP, then dZ
    int* src = reinterpret_cast<int*>(dp + nslot);  // shared slot i: -1 - i; routed key j: j; bad: INT_MIN
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long qg = blockIdx.x;
    const int bh = (int)(qg / D.N);
    // every slot's key index first (the routed experts' index rows are read whole)
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) {
        int j;
        if (u < m_sh) {
            j = -1 - u;
        } else {
            const int v = u - m_sh, slot = v / D.k, t = v % D.k;
            const int e = E[qg * D.s + slot];
            j = (e >= 0 && e < D.m) ? I[((size_t)bh * D.m + e) * D.k + t] : -1;
            if (e < 0 || e >= D.m || j < 0 || j >= D.N) j = INT_MIN;
        }
        src[u] = j;
    }
    __syncthreads();
    const T* Kb = K + (size_t)bh * D.N * DD;
    const T* Vb = V + (size_t)bh * D.N * DD;
    const float* Qtb = Qt + (size_t)bh * D.m * DD;
    const float* Vtb = Vt + (size_t)bh * D.m * DD;
    float qv[CPL], gv[CPL];
    load_row<T, DD>(Q + qg * DD, qv, lane);
    load_row<T, DD>(dO + qg * DD, gv, lane);
#pragma unroll 4
    for (int u = warp; u < nslot; u += 4) {
        const int j = src[u];
        float kr[CPL], vr[CPL];
        if (j == INT_MIN) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) kr[c] = vr[c] = 0.0f;
        } else if (j < 0) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                kr[c] = Qtb[(size_t)(-1 - j) * DD + lane * CPL + c];
                vr[c] = Vtb[(size_t)(-1 - j) * DD + lane * CPL + c];
            }
        } else {
            load_row<T, DD>(Kb + (size_t)j * DD, kr, lane);
            load_row<T, DD>(Vb + (size_t)j * DD, vr, lane);
        }
        float dot = 0.0f, dpu = 0.0f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            dot = fmaf(qv[c], kr[c], dot);
            dpu = fmaf(gv[c], vr[c], dpu);
        }
        dot = warp_sum(dot);
        dpu = warp_sum(dpu);
        if (lane == 0) {
            if (j == INT_MIN) set_status(status, kStBounds);
            lg[u] = j == INT_MIN ? -INFINITY : D.scale * dot;
            dp[u] = j == INT_MIN ? 0.0f : dpu;
        }
    }
    __syncthreads();
    float mx = -INFINITY;
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) mx = fmaxf(mx, lg[u]);
    mx = block_max(mx, red);
    float sum = 0.0f;
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) {
        const float p = (src[u] == INT_MIN) ? 0.0f : expf(lg[u] - mx);
        lg[u] = p;
        sum += p;
    }
    sum = block_sum(sum, red);
    const float inv = sum > 0.0f ? 1.0f / sum : 0.0f;
    float dsum = 0.0f;
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) {
        lg[u] *= inv;
        dsum += lg[u] * dp[u];
    }
    const float Dt = block_sum(dsum, red);
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) {
        const float dz = lg[u] * (dp[u] - Dt);
        dp[u] = dz;
        if (u < m_sh) {
            Psh[qg * D.m + u] = lg[u];
            dZsh[qg * D.m + u] = dz;
        } else {  // a routed slot: P and dZ for the per-expert reduction into dK, dV
            Pr[qg * (size_t)D.s * D.k + (u - m_sh)] = lg[u];
            dZr[qg * (size_t)D.s * D.k + (u - m_sh)] = dz;
        }
    }
    __syncthreads();
    // dq = scale sum_u dZ_u key_u: each warp over its slots, then the 4 warps summed
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.0f;
#pragma unroll 4
    for (int u = warp; u < nslot; u += 4) {
        const int j = src[u];
        if (j == INT_MIN) continue;
        float kr[CPL];
        if (j < 0) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) kr[c] = Qtb[(size_t)(-1 - j) * DD + lane * CPL + c];
        } else {
            load_row<T, DD>(Kb + (size_t)j * DD, kr, lane);
        }
        const float dz = dp[u];
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] = fmaf(dz, kr[c], acc[c]);
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) wacc[warp][lane * CPL + c] = acc[c];
    __syncthreads();
    for (int c = threadIdx.x; c < DD; c += blockDim.x)
        dQacc[qg * DD + c] = D.scale * (wacc[0][c] + wacc[1][c] + wacc[2][c] + wacc[3][c]);
}

// Bucketing of the (query, slot) pairs by routed expert for the reductions
// into dK, dV: counts per expert, offsets per head, then the pairs' places
// (the order inside a bucket does not matter to a sum). A block (256 queries
// of one head) counts and ranks its pairs per expert in shared memory and
// touches each expert's global counter once.
__global__ void k_bwd_bucket_count(const int32_t* __restrict__ E, int N, int m, int s, int* __restrict__ counts) {
    extern __shared__ int hist[];
    const int bh = blockIdx.y;
    for (int i = threadIdx.x; i < m; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q < N)
        for (int t = 0; t < s; ++t) {
            const int e = E[((size_t)bh * N + q) * s + t];
            if (e >= 0 && e < m) atomicAdd(&hist[e], 1);
        }
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += blockDim.x)
        if (hist[i]) atomicAdd(&counts[(size_t)bh * m + i], hist[i]);
}

__global__ void __launch_bounds__(512) k_bwd_bucket_scan(const int* __restrict__ counts, int m,
                                                         int* __restrict__ offs, int* __restrict__ cursors) {
    __shared__ int tmp[33];
    const int bh = blockIdx.x;
    int run = 0;
    for (int e0 = 0; e0 < m; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int c = e < m ? counts[(size_t)bh * m + e] : 0;
        int tot;
        const int o = block_excl_scan(c, tmp, &tot);
        if (e < m) {
            offs[(size_t)bh * (m + 1) + e] = run + o;
            cursors[(size_t)bh * m + e] = run + o;
        }
        run += tot;
    }
    if (threadIdx.x == 0) offs[(size_t)bh * (m + 1) + m] = run;
}

__global__ void k_bwd_bucket_scatter(const int32_t* __restrict__ E, int N, int m, int s, int* __restrict__ cursors,
                                     int* __restrict__ rows) {
    extern __shared__ int bins[];  // m local counts, then the bins' global bases
    const int bh = blockIdx.y;
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    for (int i = threadIdx.x; i < m; i += blockDim.x) bins[i] = 0;
    __syncthreads();
    int bin[kMaxS], rank[kMaxS];
#pragma unroll
    for (int t = 0; t < kMaxS; ++t) {
        bin[t] = -1;
        if (t < s && q < N) {
            const int e = E[((size_t)bh * N + q) * s + t];
            if (e >= 0 && e < m) {
                bin[t] = e;
                rank[t] = atomicAdd(&bins[e], 1);
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
        const int c = bins[i];
        bins[i] = c ? atomicAdd(&cursors[(size_t)bh * m + i], c) : 0;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kMaxS; ++t)
        if (bin[t] >= 0) rows[(size_t)bh * N * s + bins[bin[t]] + rank[t]] = (q << 3) | t;
}

// dK, dV of one expert's keys, 64 keys per block: thread (key jl, dim group
// cg) sums over the expert's (query, slot) pairs dk_j += scale dZ q and
// dv_j += P dO for its D / 4 dims in registers, the pairs' query and dO rows
// staged 32 at a time in shared memory; then one atomic add per element (a
// key in several experts' sets adds up).
constexpr int kRowSplits = 16;

template <typename T, int DD>
__global__ void __launch_bounds__(256) k_bwd_expert_kv(const T* __restrict__ Q, const T* __restrict__ dO,
                                                       const int32_t* __restrict__ I, const int* __restrict__ offs,
                                                       const int* __restrict__ rows, const float* __restrict__ Pr,
                                                       const float* __restrict__ dZr, float* __restrict__ dKacc,
                                                       float* __restrict__ dVacc, int N, int m, int k, int s,
                                                       float scale) {
    constexpr int CG = DD / 4;  // dims per thread
    constexpr int RB = 16;      // pairs staged at a time
    __shared__ __align__(16) float sq[RB][DD], sg[RB][DD];
    __shared__ float sdz[RB][64], sp[RB][64];
    __shared__ int srow[RB];
    const int e = blockIdx.y, bh = blockIdx.z / kRowSplits, part = blockIdx.z % kRowSplits;
    const int jl = threadIdx.x >> 2, cg = threadIdx.x & 3;
    const int jpos = blockIdx.x * 64 + jl;
    const bool kok = jpos < k;
    // this block's share of the expert's pairs: the experts' sizes differ a
    // lot (routing follows the data), so a large one is split over up to
    // kRowSplits blocks of at least 256 pairs
    const int e0 = offs[(size_t)bh * (m + 1) + e], e1 = offs[(size_t)bh * (m + 1) + e + 1];
    const int chunk = max(256, (e1 - e0 + kRowSplits - 1) / kRowSplits);
    const int b0 = min(e1, e0 + part * chunk), b1 = min(e1, b0 + chunk);
    if (b0 >= b1) return;
    const int* rb = rows + (size_t)bh * N * s;
    float ak[CG], av[CG];
#pragma unroll
    for (int c = 0; c < CG; ++c) ak[c] = av[c] = 0.0f;
    for (int r0 = b0; r0 < b1; r0 += RB) {
        const int nr = min(RB, b1 - r0);
        __syncthreads();
        if (threadIdx.x < RB) srow[threadIdx.x] = threadIdx.x < nr ? rb[r0 + threadIdx.x] : 0;
        __syncthreads();
        // the pairs' query and dO rows, and their P and dZ on this block's 64 keys
        for (int i = threadIdx.x; i < nr * DD; i += blockDim.x) {
            const int rr = i / DD, c = i % DD;
            const size_t qg = (size_t)bh * N + (srow[rr] >> 3);
            sq[rr][c] = to_f(Q[qg * DD + c]);
            sg[rr][c] = to_f(dO[qg * DD + c]);
        }
        for (int i = threadIdx.x; i < nr * 64; i += blockDim.x) {
            const int rr = i >> 6, jj = i & 63, jp = blockIdx.x * 64 + jj;
            const int pk = srow[rr];
            const size_t slot = ((size_t)bh * N + (pk >> 3)) * s + (pk & 7);
            sdz[rr][jj] = jp < k ? dZr[slot * k + jp] : 0.0f;
            sp[rr][jj] = jp < k ? Pr[slot * k + jp] : 0.0f;
        }
        __syncthreads();
        for (int rr = 0; rr < nr; ++rr) {
            const float dz = scale * sdz[rr][jl], p = sp[rr][jl];
            const float4* q4 = reinterpret_cast<const float4*>(&sq[rr][cg * CG]);
            const float4* g4 = reinterpret_cast<const float4*>(&sg[rr][cg * CG]);
#pragma unroll
            for (int c4 = 0; c4 < CG / 4; ++c4) {
                const float4 a = q4[c4], b = g4[c4];
                ak[4 * c4] = fmaf(dz, a.x, ak[4 * c4]);
                ak[4 * c4 + 1] = fmaf(dz, a.y, ak[4 * c4 + 1]);
                ak[4 * c4 + 2] = fmaf(dz, a.z, ak[4 * c4 + 2]);
                ak[4 * c4 + 3] = fmaf(dz, a.w, ak[4 * c4 + 3]);
                av[4 * c4] = fmaf(p, b.x, av[4 * c4]);
                av[4 * c4 + 1] = fmaf(p, b.y, av[4 * c4 + 1]);
                av[4 * c4 + 2] = fmaf(p, b.z, av[4 * c4 + 2]);
                av[4 * c4 + 3] = fmaf(p, b.w, av[4 * c4 + 3]);
            }
        }
    }
    if (!kok) return;
    const int j = I[((size_t)bh * m + e) * k + jpos];
    if (j < 0 || j >= N) return;
    float* dk = dKacc + ((size_t)bh * N + j) * DD + cg * CG;
    float* dv = dVacc + ((size_t)bh * N + j) * DD + cg * CG;
#pragma unroll
    for (int c = 0; c < CG; ++c) {
        atomicAdd(dk + c, ak[c]);
        atomicAdd(dv + c, av[c]);
    }
}

// dS = A o (dA - delta), in place over dA.
__global__ void k_bwd_shared_ds(const float* __restrict__ A, float* __restrict__ dA, const float* __restrict__ delta,
                                long long rows, int N) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= rows * N) return;
    dA[e] = A[e] * (dA[e] - delta[e / N]);
}

// delta_i = dVt_i . Vt_i, one warp per landmark row.
__global__ void k_rowdot(const float* __restrict__ X, const float* __restrict__ Y, float* __restrict__ out,
                         long long rows, int d) {
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float acc = 0.0f;
    for (int c = lane; c < d; c += 32) acc = fmaf(X[row * d + c], Y[row * d + c], acc);
    acc = warp_sum(acc);
    if (lane == 0) out[row] = acc;
}

// dq_t += dQt_i / |bin_i| for every 1-D pooling bin i that holds t (at most
// two when N % m != 0), then every gradient to the storage type.
template <typename T>
__global__ void k_bwd_finish(const float* __restrict__ dQacc, const float* __restrict__ dKacc,
                             const float* __restrict__ dVacc, const float* __restrict__ dQt, T* __restrict__ dQ,
                             T* __restrict__ dK, T* __restrict__ dV, long long BH, int N, int m, int d, int pool) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= BH * N * d) return;
    const int c = (int)(e % d);
    const long long row = e / d;
    const int t = (int)(row % N);
    const long long bh = row / N;
    float g = dQacc[e];
    if (pool) {
        const int i0 = (int)(((long long)t * m) / N);
        for (int i = max(0, i0 - 1); i <= min(m - 1, i0 + 1); ++i) {
            int lo, hi;
            pool_bin(i, N, m, &lo, &hi);
            if (t >= lo && t < hi) g += dQt[(bh * m + i) * d + c] / (float)(hi - lo);
        }
    }
    dQ[e] = from_f<T>(g);
    dK[e] = from_f<T>(dKacc[e]);
    dV[e] = from_f<T>(dVacc[e]);
}

template <typename T>
cudaError_t backward_t(const Dims& D, const BwdWork& W, const void* Qv, const void* Kv, const void* Vv,
                       const void* dOv, const int32_t* I, const int32_t* E, void* dQv, void* dKv, void* dVv,
                       int* status, cudaStream_t st) {
    const T *Q = (const T*)Qv, *K = (const T*)Kv, *V = (const T*)Vv, *dO = (const T*)dOv;
    const long long BH = D.BH, N = D.N, d = D.d, m = D.m;
    const long long Nd = N * d, md = m * d, mN = m * N;
    cudaError_t e;
    prof_mark(st, "bwd_shared_fwd");
    // forward quantities: Qt, the raw landmark scores S = Qt K^T, Vt and the row statistics
    if ((e = launch_pool(D, Q, W.Qt, nullptr, nullptr, 0, status, st))) return e;
    if (D.shared) {
        // S = Qt K^T, its row statistics, A = softmax(scale S) in place, Vt = A V
        if ((e = gemm(W.Qt, md, d, 1, K, Nd, 1, d, W.S, mN, (int)m, (int)N, (int)d, 1.0f, false, (int)BH, st)))
            return e;
        if ((e = launch_row_stats(D, W.S, W.stats, st))) return e;
        k_bwd_shared_attn<<<(unsigned)((BH * mN + 255) / 256), 256, 0, st>>>(W.S, W.stats, BH * m, (int)N, D.scale);
        count_launch();
        if ((e = cudaGetLastError())) return e;
        if ((e = gemm(W.S, mN, N, 1, V, Nd, d, 1, W.Vt, md, (int)m, (int)d, (int)N, 1.0f, false, (int)BH, st)))
            return e;
    }
    prof_mark(st, "bwd_query");
    if ((e = cudaMemsetAsync(W.dKacc, 0, sizeof(float) * BH * Nd, st))) return e;
    if ((e = cudaMemsetAsync(W.dVacc, 0, sizeof(float) * BH * Nd, st))) return e;
    {
        const int m_sh = D.shared ? D.m : 0;
        const size_t smem = sizeof(float) * 2 * (m_sh + D.s * (size_t)D.k) + sizeof(int) * (m_sh + D.s * (size_t)D.k);
        if (d == 128) {
            if (smem > 40 * 1024 &&
                (e = cudaFuncSetAttribute(k_bwd_query<T, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
                return e;
            k_bwd_query<T, 128><<<(unsigned)(BH * N), 128, smem, st>>>(Q, K, V, dO, W.Qt, W.Vt, I, E, W.dQacc,
                                                                      W.Psh, W.dZsh, W.Pr, W.dZr, D, status);
        } else {
            if (smem > 40 * 1024 &&
                (e = cudaFuncSetAttribute(k_bwd_query<T, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
                return e;
            k_bwd_query<T, 64><<<(unsigned)(BH * N), 128, smem, st>>>(Q, K, V, dO, W.Qt, W.Vt, I, E, W.dQacc,
                                                                     W.Psh, W.dZsh, W.Pr, W.dZr, D, status);
        }
        count_launch();
        if ((e = cudaGetLastError())) return e;
    }
    prof_mark(st, "bwd_routed_kv");
    {
        const long long nq = BH * N;
        if ((e = cudaMemsetAsync(W.counts, 0, sizeof(int) * BH * m, st))) return e;
        (void)nq;
        const dim3 qgrid((unsigned)((N + 255) / 256), (unsigned)BH);
        const size_t hsm = sizeof(int) * m;
        k_bwd_bucket_count<<<qgrid, 256, hsm, st>>>(E, (int)N, (int)m, D.s, W.counts);
        k_bwd_bucket_scan<<<(unsigned)BH, 512, 0, st>>>(W.counts, (int)m, W.offs, W.cursors);
        k_bwd_bucket_scatter<<<qgrid, 256, hsm, st>>>(E, (int)N, (int)m, D.s, W.cursors, W.rows);
        dim3 grid((D.k + 63) / 64, (unsigned)m, (unsigned)(BH * kRowSplits));
        if (d == 128)
            k_bwd_expert_kv<T, 128><<<grid, 256, 0, st>>>(Q, dO, I, W.offs, W.rows, W.Pr, W.dZr, W.dKacc, W.dVacc,
                                                          (int)N, (int)m, D.k, D.s, D.scale);
        else
            k_bwd_expert_kv<T, 64><<<grid, 256, 0, st>>>(Q, dO, I, W.offs, W.rows, W.Pr, W.dZr, W.dKacc, W.dVacc,
                                                         (int)N, (int)m, D.k, D.s, D.scale);
        count_launch(4);
        if ((e = cudaGetLastError())) return e;
    }
    if (D.shared) {
        prof_mark(st, "bwd_shared");
        // dVt = Psh^T dO, dQt = scale dZsh^T Q (reductions over the queries)
        if ((e = gemm(W.Psh, N * m, 1, m, dO, Nd, d, 1, W.dVt, md, (int)m, (int)d, (int)N, 1.0f, false, (int)BH, st)))
            return e;
        if ((e = gemm(W.dZsh, N * m, 1, m, Q, Nd, d, 1, W.dQt, md, (int)m, (int)d, (int)N, D.scale, false, (int)BH,
                      st)))
            return e;
        // shared expert: dA = dVt V^T, delta = rowdot(dVt, Vt), dS = A o (dA - delta)
        if ((e = gemm(W.dVt, md, d, 1, V, Nd, 1, d, W.dA, mN, (int)m, (int)N, (int)d, 1.0f, false, (int)BH, st)))
            return e;
        k_rowdot<<<(unsigned)((BH * m * 32 + 255) / 256), 256, 0, st>>>(W.dVt, W.Vt, W.delta, BH * m, (int)d);
        k_bwd_shared_ds<<<(unsigned)((BH * mN + 255) / 256), 256, 0, st>>>(W.S, W.dA, W.delta, BH * m, (int)N);
        count_launch(2);
        if ((e = cudaGetLastError())) return e;
        // dQt += scale dS K, dK += scale dS^T Qt, dV += A^T dVt
        if ((e = gemm(W.dA, mN, N, 1, K, Nd, d, 1, W.dQt, md, (int)m, (int)d, (int)N, D.scale, true, (int)BH, st)))
            return e;
        if ((e = gemm(W.dA, mN, 1, N, W.Qt, md, d, 1, W.dKacc, Nd, (int)N, (int)d, (int)m, D.scale, true, (int)BH,
                      st)))
            return e;
        if ((e = gemm(W.S, mN, 1, N, W.dVt, md, d, 1, W.dVacc, Nd, (int)N, (int)d, (int)m, 1.0f, true, (int)BH, st)))
            return e;
    }
    prof_mark(st, "bwd_finish");
    k_bwd_finish<T><<<(unsigned)((BH * Nd + 255) / 256), 256, 0, st>>>(W.dQacc, W.dKacc, W.dVacc, W.dQt, (T*)dQv,
                                                                       (T*)dKv, (T*)dVv, BH, (int)N, (int)m,
                                                                       (int)d, D.shared ? 1 : 0);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

size_t bwd_query_smem(const Dims& D) {
    const size_t nslot = (size_t)(D.shared ? D.m : 0) + (size_t)D.s * D.k;
    return sizeof(float) * 2 * nslot + sizeof(int) * nslot + sizeof(float) * 4 * 128;
}

cudaError_t launch_backward(const Dims& D, const BwdWork& W, const void* Q, const void* K, const void* V,
                            const void* dO, const int32_t* I, const int32_t* E, void* dQ, void* dK, void* dV,
                            int* status, cudaStream_t st) {
    return D.dtype == 0 ? backward_t<float>(D, W, Q, K, V, dO, I, E, dQ, dK, dV, status, st)
                        : backward_t<__nv_bfloat16>(D, W, Q, K, V, dO, I, E, dQ, dK, dV, status, st);
}

}  // namespace mita
