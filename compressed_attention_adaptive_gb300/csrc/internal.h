// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mita {

constexpr int kMaxS = 8;  // routed experts per query the kernels support

// api.cu: phase markers (CUDA events while profiling is on) and the count of
// kernels launched by this library.
void prof_mark(cudaStream_t st, const char* phase);
void count_launch(int n = 1);

// api.cu (for the static-workspace entry point)
}  // namespace mita
#include "../../include/mita.h"
namespace mita {
mita_status validate(const mita_params* p);
mita_status report_error(mita_status st, const char* msg);
void clear_error();  // empties the calling thread's mita_last_error() detail
mita_status forward_on_workspace(const mita_params* p, const void* Q, const void* K, const void* V, void* O,
                                 void* ws, size_t ws_bytes, void* stream);

// simt.cu
cudaError_t launch_pool(const Dims& D, const void* Q, float* Qt, __nv_bfloat16* hi, __nv_bfloat16* lo, int m_pad,
                        int* status, cudaStream_t st);
cudaError_t launch_select_simt(const Dims& D, const void* Q, const void* K, const float* Qt, float* S, float* R,
                               int32_t* I, int32_t* E, cudaStream_t st);
cudaError_t launch_shared_simt(const Dims& D, const void* V, const float* S, float2* stats, float* Vt,
                               cudaStream_t st);
// per landmark row of raw scores S: (max of scale * s, 1 / sum exp(scale * s - max))
cudaError_t launch_row_stats(const Dims& D, const float* S, float2* stats, cudaStream_t st);
size_t out_simt_smem(const Dims& D);
cudaError_t launch_out_simt(const Dims& D, const void* Q, const void* K, const void* V, const float* Qt,
                            const float* Vt, const int32_t* I, const int32_t* E, void* O, int* status,
                            cudaStream_t st);

// select.cu
cudaError_t launch_topk_dense(const float* S, long long rows, int N, int k, int32_t* I, cudaStream_t st);
cudaError_t launch_sample_threshold(const float* Ssamp, long long rows, int n_samp, int k, float* thr,
                                    cudaStream_t st);
cudaError_t launch_topk_cand(const int2* cand, const int* ccount, int splits, long long cap, int BH, int m, int m_pad,
                             int N, int k, long long expect, int32_t* I, int* status, cudaStream_t st);

}  // namespace mita

namespace mita {

// tc.cu: sizes of the tensor-core path for one problem.
struct TcPlan {
    int m_pad;             // landmarks rounded up to 128
    int m_tiles;           // m_pad / 128
    int splits;            // key splits of the landmark pass
    int chunks_per_split;  // 128-key chunks per split
    long long max_tiles;   // upper bound on expert work tiles
    int route_cols;        // TMEM columns of the routing kernel
    int R;                 // top-k sample stride (every R-th key)
    int n_samp;            // sampled keys per row (>= k)
    long long cand_cap;    // candidate records per (row, split)
    bool resident;         // the causal variant's tensor-core path: m <= 128, k <= 256, shared slots on
    bool route_shared;     // the routing pass also computes the shared slots (m <= 128, shared slots on)
    int ksub, nsub;        // keys per sub-expert (<= 256) and sub-experts per expert
    int ksub_sh, nsub_sh;  // the same for the shared slots when they run as their own pass (m > 128)
    int nsh;               // shared-slot partials per query (0 with the shared slots off)
};

// Workspace buffers of the tensor-core path.
struct TcWork {
    __nv_bfloat16 *Qhi, *Qlo, *Vtb;  // [BH][m_pad][d]
    float* Opart;                    // [BH][splits][m_pad][d]
    float2* ML;                      // [BH][splits][m_pad]
    float* Ssamp;                    // [BH][m][n_samp] sample scores
    float* thr;                      // [BH][m] candidate thresholds
    int2* cand;                      // [BH][m_pad][splits][2][cand_cap / 2] (score, key) records
    int* ccount;                     // [BH][m_pad][splits][2]
    int* counts;                     // [BH][m][2]
    int* tile_ctr;                   // [3]: tiles written, expert and shared-pass claims of the expert attention
    void* zero_begin;                // counts .. tile_ctr, cleared each call
    size_t zero_bytes;
    int* cursors;                    // [BH][m][2]
    int* toff;                       // [BH][m]
    int4* tiles;                     // [max_tiles]
    int2* xtl;                       // [BH][m] (first tile, tile count) of each expert
    int32_t* perm;                   // [BH][N*s]
    __nv_bfloat16* part;             // [BH][N][s][nsub][d]
    float* lse;                      // [BH][N][s][nsub]
    __nv_bfloat16* sh_part;          // [BH][N][nsh][d] shared-slot partials
    float* sh_lse;                   // [BH][N][nsh]
};

bool tc_supported(const Dims& D);
TcPlan tc_plan(const Dims& D);
// SMs of the current device, queried once (152, a GB300's, if the query fails)
int num_sms();
cudaError_t launch_forward_tc(const Dims& D, const TcPlan& P, const TcWork& W, const void* Q, const void* K,
                              const void* V, void* O, float* Vt, int32_t* I, int32_t* E, int* status, int upto,
                              cudaStream_t st);

}  // namespace mita

namespace mita {

// backward.cu: workspace of the backward pass (fp32 throughout).
struct BwdWork {
    float *Qt, *Vt;             // [BH][m][d] landmarks and shared expert again
    float2* stats;              // [BH][m] row max of scale * s and 1 / row sum of the shared expert
    float *S, *dA;              // [BH][m][N] raw landmark scores (then A) and dA (then dS)
    float *Psh, *dZsh;          // [BH][N][m] the shared slots' P and dZ per query
    float *dQt, *dVt, *delta;   // [BH][m][d], [BH][m][d], [BH][m]
    float *dQacc, *dKacc, *dVacc;  // [BH][N][d] fp32 accumulators
    float *Pr, *dZr;            // [BH][N][s][k] the routed slots' P and dZ per query
    int *counts, *cursors;      // [BH][m] bucket sizes and scatter cursors
    int *offs, *rows;           // [BH][m + 1] bucket offsets, [BH][N * s] pairs in bucket order
};
size_t bwd_query_smem(const Dims& D);
cudaError_t launch_backward(const Dims& D, const BwdWork& W, const void* Q, const void* K, const void* V,
                            const void* dO, const int32_t* I, const int32_t* E, void* dQ, void* dK, void* dV,
                            int* status, cudaStream_t st);

}  // namespace mita
