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
// 4 x 4 outputs per thread, operands widened to fp32 as they are staged.
template <typename TA, typename TB>
__global__ void __launch_bounds__(256) k_gemm_strided(const TA* __restrict__ A, long long sA, long long a_i,
                                                      long long a_k, const TB* __restrict__ B, long long sB,
                                                      long long b_k, long long b_j, float* __restrict__ C,
                                                      long long sC, int M, int Nn, int K, float alpha,
                                                      int accumulate) {
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
            const int e = t + 256 * r, row = e >> 4, kk = e & 15, gk = k0 + kk;
            As[kk][row] = (m0 + row < M && gk < K) ? to_f(Ab[(m0 + row) * a_i + gk * a_k]) : 0.0f;
            Bs[kk][row] = (n0 + row < Nn && gk < K) ? to_f(Bb[gk * b_k + (n0 + row) * b_j]) : 0.0f;
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
                *dst = accumulate ? *dst + alpha * acc[i][j] : alpha * acc[i][j];
            }
        }
}

template <typename TA, typename TB>
cudaError_t gemm(const TA* A, long long sA, long long a_i, long long a_k, const TB* B, long long sB, long long b_k,
                 long long b_j, float* C, long long sC, int M, int Nn, int K, float alpha, bool accumulate, int batch,
                 cudaStream_t st) {
    dim3 grid((Nn + 63) / 64, (M + 63) / 64, batch);
    k_gemm_strided<TA, TB><<<grid, 256, 0, st>>>(A, sA, a_i, a_k, B, sB, b_k, b_j, C, sC, M, Nn, K, alpha,
                                                 accumulate ? 1 : 0);
    count_launch();
    return cudaGetLastError();
}

// One block per query: its slots' logits and probabilities again (as in the
// forward), dP = dO . val, D = sum P dP, dZ = P (dP - D); dq of the query;
// the shared slots' P and dZ rows (for the reductions over queries); the
// routed keys' contributions added into dK, dV with atomics.
template <typename T>
__global__ void __launch_bounds__(128) k_bwd_query(const T* __restrict__ Q, const T* __restrict__ K,
                                                   const T* __restrict__ V, const T* __restrict__ dO,
                                                   const float* __restrict__ Qt, const float* __restrict__ Vt,
                                                   const int32_t* __restrict__ I, const int32_t* __restrict__ E,
                                                   float* __restrict__ dQacc, float* __restrict__ dKacc,
                                                   float* __restrict__ dVacc, float* __restrict__ Psh,
                                                   float* __restrict__ dZsh, Dims D, int* __restrict__ status) {
    extern __shared__ float sm[];
    __shared__ float red[32];
    const int d = D.d, m_sh = D.shared ? D.m : 0, nslot = m_sh + D.s * D.k;
    float* qv = sm;
    float* gv = sm + d;            // dO of the query
    float* lg = gv + d;            // logits, then P
    float* dp = lg + nslot;        // dP, then dZ
    int* src = reinterpret_cast<int*>(dp + nslot);  // shared slot i: -1 - i; routed key j: j; bad: INT_MIN
    const long long qg = blockIdx.x;
    const int bh = (int)(qg / D.N);
    const T* Kb = K + (size_t)bh * D.N * d;
    const T* Vb = V + (size_t)bh * D.N * d;
    const float* Qtb = Qt + (size_t)bh * D.m * d;
    const float* Vtb = Vt + (size_t)bh * D.m * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        qv[c] = to_f(Q[qg * d + c]);
        gv[c] = to_f(dO[qg * d + c]);
    }
    __syncthreads();
    float mx = -INFINITY;
    for (int u = threadIdx.x; u < nslot; u += blockDim.x) {
        float dot = 0.0f, dpu = 0.0f;
        int j;
        if (u < m_sh) {
            j = -1 - u;
            const float* kr = Qtb + (size_t)u * d;
            const float* vr = Vtb + (size_t)u * d;
            for (int c = 0; c < d; ++c) {
                dot = fmaf(qv[c], kr[c], dot);
                dpu = fmaf(gv[c], vr[c], dpu);
            }
        } else {
            const int v = u - m_sh, slot = v / D.k, t = v % D.k;
            const int e = E[qg * D.s + slot];
            j = (e >= 0 && e < D.m) ? I[((size_t)bh * D.m + e) * D.k + t] : -1;
            if (e < 0 || e >= D.m || j < 0 || j >= D.N) {
                set_status(status, kStBounds);
                src[u] = INT_MIN;
                lg[u] = -INFINITY;
                dp[u] = 0.0f;
                continue;
            }
            const T* kr = Kb + (size_t)j * d;
            const T* vr = Vb + (size_t)j * d;
            for (int c = 0; c < d; ++c) {
                dot = fmaf(qv[c], to_f(kr[c]), dot);
                dpu = fmaf(gv[c], to_f(vr[c]), dpu);
            }
        }
        src[u] = j;
        lg[u] = D.scale * dot;
        dp[u] = dpu;
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
        }
    }
    __syncthreads();
    const size_t head0 = (size_t)bh * D.N * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float acc = 0.0f;
        for (int u = 0; u < nslot; ++u) {
            const int j = src[u];
            if (j == INT_MIN) continue;
            const float kc = (j < 0) ? Qtb[(size_t)(-1 - j) * d + c] : to_f(Kb[(size_t)j * d + c]);
            acc = fmaf(dp[u], kc, acc);
            if (j >= 0) {  // a routed key: its dk and dv (a key in several routed experts adds up)
                atomicAdd(dKacc + head0 + (size_t)j * d + c, D.scale * dp[u] * qv[c]);
                atomicAdd(dVacc + head0 + (size_t)j * d + c, lg[u] * gv[c]);
            }
        }
        dQacc[qg * d + c] = D.scale * acc;
    }
}

// The shared expert's attention A = softmax(scale Qt K^T) again from the raw
// scores S and the row statistics (max of scale * s, 1 / sum), and
// dS = A o (dA - delta): S is overwritten by A, dA by dS.
__global__ void k_bwd_shared_ds(float* __restrict__ S, float* __restrict__ dA, const float2* __restrict__ stats,
                                const float* __restrict__ delta, long long rows, int N, float scale) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= rows * N) return;
    const long long row = e / N;
    const float2 st = stats[row];
    const float a = expf(scale * S[e] - st.x) * st.y;
    S[e] = a;
    dA[e] = a * (dA[e] - delta[row]);
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
        if ((e = gemm(W.Qt, md, d, 1, K, Nd, 1, d, W.S, mN, (int)m, (int)N, (int)d, 1.0f, false, (int)BH, st)))
            return e;
        if ((e = launch_shared_simt(D, V, W.S, W.stats, W.Vt, st))) return e;
    }
    prof_mark(st, "bwd_query");
    if ((e = cudaMemsetAsync(W.dKacc, 0, sizeof(float) * BH * Nd, st))) return e;
    if ((e = cudaMemsetAsync(W.dVacc, 0, sizeof(float) * BH * Nd, st))) return e;
    {
        const int m_sh = D.shared ? D.m : 0;
        const size_t smem = sizeof(float) * (2 * d + 2 * (m_sh + D.s * (size_t)D.k)) +
                            sizeof(int) * (m_sh + D.s * (size_t)D.k);
        if (smem > 48 * 1024 &&
            (e = cudaFuncSetAttribute(k_bwd_query<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
            return e;
        k_bwd_query<T><<<(unsigned)(BH * N), 128, smem, st>>>(Q, K, V, dO, W.Qt, W.Vt, I, E, W.dQacc, W.dKacc,
                                                             W.dVacc, W.Psh, W.dZsh, D, status);
        count_launch();
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
        k_bwd_shared_ds<<<(unsigned)((BH * mN + 255) / 256), 256, 0, st>>>(W.S, W.dA, W.stats, W.delta, BH * m,
                                                                           (int)N, D.scale);
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
    return sizeof(float) * (2 * (size_t)D.d + 2 * nslot) + sizeof(int) * nslot;
}

cudaError_t launch_backward(const Dims& D, const BwdWork& W, const void* Q, const void* K, const void* V,
                            const void* dO, const int32_t* I, const int32_t* E, void* dQ, void* dK, void* dV,
                            int* status, cudaStream_t st) {
    return D.dtype == 0 ? backward_t<float>(D, W, Q, K, V, dO, I, E, dQ, dK, dV, status, st)
                        : backward_t<__nv_bfloat16>(D, W, Q, K, V, dO, I, E, dQ, dK, dV, status, st);
}

}  // namespace mita
