/*
 * mita.h -- C ABI of libmita.so, the GB300 (sm_103a) MiTA attention forward.
 *
 * The operation is the forward pass of "MiTA Attention: Efficient Fast-Weight
 * Scaling via a Mixture of Top-k Activations" as summarized on gist.science:
 *
 *   landmarks    Qt = adaptive average pooling of Q, m rows      (Arabic ed. s2, "mechanism details";
 *                                                                  Dutch ed. "Kernconcepten" 1)
 *   shared       Vt = softmax(scale * Qt K^T) V                  (Arabic ed. s2: Vt = Atten(Qt, K, V))
 *   expert sets  I_i = indices of the k largest k_j . qt_i       (Arabic ed. s2; Dutch ed. "Kernconcepten" 3)
 *   routing      e_1(q) .. e_s(q)                                (Dutch ed. "Wiskundige Formulering")
 *   output       O_q = softmax attention of q over
 *                K* = [Qt, K_(e1), .., K_(es)], V* = [Vt, V_(e1), .., V_(es)]
 *                                                                (Dutch ed. "Wiskundige Formulering")
 *
 * The summaries leave four points open; this library fixes them as follows:
 *   - the shared expert's keys are Qt (its values are Vt);
 *   - a query is routed to the s landmarks with the largest q . qt_i, ties to
 *     the lower landmark index, listed by descending score;
 *   - top-k ranks raw (unscaled) scores, ties to the lower key index, and each
 *     I_i is returned in ascending key order;
 *   - expert sets that overlap are concatenated (a key picked by two routed
 *     experts fills two slots), and one softmax runs over all m + s*k slots.
 *
 * Conventions for every entry point:
 *   - Tensors are DEVICE pointers, contiguous, row-major [B, H, rows, d]
 *     (d fastest). Q, K, V, O use `dtype`; Qt / Vt outputs are float32;
 *     index outputs are int32.
 *   - The caller owns all memory, including the workspace (device memory of at
 *     least mita_workspace_size() bytes, 256-byte aligned). The library never
 *     allocates, frees or synchronizes inside these calls.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). Outputs are valid once the stream reaches them.
 *   - Argument errors are returned synchronously before anything is enqueued.
 *     A failed launch returns MITA_ERR_CUDA. Errors detected on the device
 *     (an index out of range, a bounded wait that ran out) are written to a
 *     status word inside the workspace and read with mita_device_status().
 *     The first kernel of every call resets that word, so it holds the first
 *     device-side error of the most recent call on the workspace: read it
 *     after each call whose device status matters.
 *   - Calls are reentrant; concurrent calls must use distinct workspaces.
 */
#ifndef MITA_H
#define MITA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MITA_OK = 0,
    MITA_ERR_INVALID_ARG = 1, /* bad shape, pointer, flag or dtype             */
    MITA_ERR_UNSUPPORTED = 2, /* valid MiTA parameters this library cannot run */
    MITA_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or too small       */
    MITA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed          */
    MITA_ERR_TIMEOUT = 5,     /* device: a bounded wait gave up                */
    MITA_ERR_BOUNDS = 6       /* device: an index was out of range             */
} mita_status;

typedef enum { MITA_DTYPE_F32 = 0, MITA_DTYPE_BF16 = 1 } mita_dtype;

enum {
    /* Leave the m shared slots out of the output softmax (only the routed
     * experts remain). With k = N and s = 1 the output is plain softmax
     * attention, which tests use as an identity. */
    MITA_FLAG_NO_SHARED = 1u << 0,
    /* Run every step on CUDA cores in fp32 even where the tensor-core path
     * applies (a second GPU implementation for cross-checks). */
    MITA_FLAG_SIMT = 1u << 1,
    /* The causal variant (the summaries describe none; these rules are this
     * library's reading, for 1-D pooling only): the shared expert of landmark
     * i attends to the keys of its prefix, j < hi_i, where [lo_i, hi_i) is
     * its pooling bin; query t has landmark i's shared slot only once that bin
     * is complete (hi_i <= t + 1); expert sets and routes are selected as in
     * the non-causal pass, and of a routed expert's keys query t attends to
     * those with j <= t; a query left with no slot gets a zero output row.
     * Runs on the tensor-core path when m <= 128, k <= 256 and the shared
     * slots are on, and on the CUDA-core path (float32, or MITA_FLAG_SIMT);
     * other shapes return MITA_ERR_UNSUPPORTED. With 2-D pooling it is
     * MITA_ERR_INVALID_ARG. */
    MITA_FLAG_CAUSAL = 1u << 2
};

/* Fault test of the device-side failure detection, not for production: in
 * one CTA of the landmark pass and one of the expert attention, a producer
 * leaves out one of the signals its consumers wait for, and every bounded
 * wait of those two kernels gives up after about a millisecond instead of a
 * second. The call then records MITA_ERR_TIMEOUT in the device status word
 * (read with mita_device_status()); every role of the stalled CTAs leaves its
 * loop, lets its copies and MMAs in flight land and frees its tensor memory,
 * so the next call on the same workspace runs normally. Outputs of the
 * flagged call are undefined. Only the tensor-core path has these waits: on
 * the CUDA-core path the flag has no effect. (A macro, since the bit is
 * outside the int range of a C enum constant.) */
#define MITA_TESTFLAG_STALL_PRODUCER (1u << 31)

typedef struct {
    int B, H, N, d;   /* batch, heads, tokens, head dim (8 <= d <= 256, d % 8 == 0) */
    int m, k, s;      /* landmarks (1..N), top-k width (1..N), routed experts (1..min(m, 8)) */
    int grid_h, grid_w; /* token grid for 2-D pooling (grid_h * grid_w == N);
                           grid_h == 0 means 1-D pooling over N tokens           */
    int lm_h, lm_w;   /* landmark grid (lm_h * lm_w == m); ignored for 1-D      */
    float scale;      /* softmax scale; 0 means 1/sqrt(d)                        */
    unsigned flags;   /* MITA_FLAG_*                                             */
    int dtype;        /* mita_dtype of Q, K, V and O                             */
} mita_params;

/* Bytes of device workspace needed for `p`; 0 if `p` is invalid. On the
 * tensor-core path it holds one bf16 partial output row per (query, routed
 * slot, 256-key sub-expert), so it grows with s * ceil(k / 256): about
 * 2 * B * H * N * d * s * ceil(k / 256) bytes for those rows (2.0 GB in all at
 * B2 H16 N32768 d128, m128, k256, s2). */
size_t mita_workspace_size(const mita_params* p);

/* Landmark queries only. Qt: float32 [B, H, m, d], caller-owned device memory. */
mita_status mita_landmarks(const mita_params* p, const void* Q, float* Qt, void* ws, size_t ws_bytes,
                           void* stream);

/* Landmarks, expert index sets and routes, without the attention outputs.
 * idx: int32 [B, H, m, k], each row ascending; route: int32 [B, H, N, s],
 * descending routing score. Either output may be NULL. */
mita_status mita_select(const mita_params* p, const void* Q, const void* K, int32_t* idx, int32_t* route,
                        void* ws, size_t ws_bytes, void* stream);

/* The whole forward pass. O: [B, H, N, d] in `dtype`. idx_out ([B, H, m, k]),
 * route_out ([B, H, N, s]) and Vt_out (float32 [B, H, m, d]) are optional
 * (NULL to skip) copies of the intermediate index sets, routes and shared
 * expert values. */
mita_status mita_forward(const mita_params* p, const void* Q, const void* K, const void* V, void* O,
                         int32_t* idx_out, int32_t* route_out, float* Vt_out, void* ws, size_t ws_bytes,
                         void* stream);

/* Bytes of DEVICE memory mita_forward_host() needs: room for Q, K, V and O
 * plus the workspace. */
size_t mita_host_buffer_size(const mita_params* p);

/* The forward pass on HOST buffers: Q, K, V, O are host pointers (pinned
 * memory gives full copy speed), `dev` is caller-owned device memory of at
 * least mita_host_buffer_size() bytes. Copies Q, K, V to the device, runs the
 * forward pass, copies O back. The heads are processed in a few groups so that
 * one group's copies overlap another's compute: the copies run on two streams
 * the library keeps per device, ordered after earlier work on `stream` and
 * joined back into it, so all of the call's work is ordered on `stream`
 * (concurrent calls from several host threads enqueue one after another). The
 * call returns without waiting; the host buffers must stay valid until
 * `stream` has passed it. The device status word is the workspace's, at
 * offset 4 * align_up(B*H*N*d*element size, 1024) bytes of `dev`. */
mita_status mita_forward_host(const mita_params* p, const void* Q, const void* K, const void* V, void* O,
                              void* dev, size_t dev_bytes, void* stream);

/* Synchronizes `stream`, returns the device status word of workspace `ws`
 * (MITA_OK if no device-side error was recorded by the most recent call on
 * `ws`) and clears it. */
mita_status mita_device_status(void* ws, void* stream);

/* Static description of a status code. */
const char* mita_status_string(mita_status s);

/* Detail of the last error returned on the calling thread ("" if none). */
const char* mita_last_error(void);

/* ---- backward pass ---------------------------------------------------------
 * The summaries describe the forward pass and report training speed, but print
 * no backward pass; this one is the chain rule through the forward's steps with
 * the expert sets and routes held fixed (a top-k choice is piecewise constant
 * and has no gradient): through each query's softmax over its shared and
 * routed slots, through the shared expert Vt = softmax(scale Qt K^T) V, and
 * through the pooling of the landmarks. Runs on CUDA cores in fp32 (the inputs
 * widened from `dtype`). Non-causal, 1-D pooling only (other settings return
 * MITA_ERR_UNSUPPORTED).
 *
 * Bytes of device workspace mita_backward() needs for `p`; 0 if `p` is invalid
 * or unsupported there. */
size_t mita_backward_workspace_size(const mita_params* p);

/* Gradients of sum(O * dO) with respect to Q, K, V. Q, K, V, dO and the
 * outputs dQ, dK, dV: device [B, H, N, d] in `dtype`; idx [B, H, m, k] and
 * route [B, H, N, s]: the expert sets and routes of the forward pass whose
 * gradient is wanted (mita_forward's idx_out / route_out, or mita_select's).
 * Every output row is written. Asynchronous on `stream`; argument errors are
 * returned before anything is enqueued; an index out of range in idx or route
 * is recorded in the workspace's status word (mita_device_status on `ws`). */
mita_status mita_backward(const mita_params* p, const void* Q, const void* K, const void* V, const void* dO,
                          const int32_t* idx, const int32_t* route, void* dQ, void* dK, void* dV, void* ws,
                          size_t ws_bytes, void* stream);

/* 1 if `p` runs on the tcgen05 tensor-core path, 0 if on CUDA cores, -1 if invalid. */
int mita_uses_tensor_cores(const mita_params* p);

/* ---- forward pass without device allocation --------------------------------
 * Not part of the method (the summaries have no counterpart): an interface
 * for callers that cannot allocate device memory. Some code may not call
 * cudaMalloc at all: it can synchronize the whole device, another framework
 * may own all device memory through its own pool, or the caller is a plugin
 * that only receives the tensors it works on. mita_forward_static() is
 * mita_forward() with its workspace in a library-owned static device array of
 * MITA_STATIC_WORKSPACE_BYTES, so the caller passes only Q, K, V and O.
 *   - Problems whose mita_workspace_size() exceeds the static area are
 *     rejected with MITA_ERR_UNSUPPORTED; nothing is enqueued.
 *   - The call allocates nothing (no cudaMalloc, no allocating library call).
 *     Every GPU on which the library is loaded holds the static area until the
 *     process exits.
 *   - The first call on a device looks up the area's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. `stream` must belong to the current device.
 *   - All calls share the one area, which keeps the last call's contents; the
 *     pass clears what must start at zero itself. Calls whose work overlaps on
 *     the GPU (different streams, or concurrent host threads) race on the area
 *     and must be serialized by the caller.
 *   - status_out (optional, device int32) receives the call's device status
 *     word (MITA_OK or MITA_ERR_TIMEOUT / MITA_ERR_BOUNDS) once the stream
 *     reaches it. */
#define MITA_STATIC_WORKSPACE_BYTES (64u << 20)
mita_status mita_forward_static(const mita_params* p, const void* Q, const void* K, const void* V, void* O,
                                int32_t* status_out, void* stream);

/* ---- measurement hooks (not part of the method) ---------------------------
 * Number of kernels this library has launched in the process so far. */
long long mita_launch_count(void);

/* Opens a phase profile: until mita_profile_end(), every call records a CUDA
 * event on its stream at the start of each phase (landmark pooling, top-k
 * sample and threshold, landmark pass, top-k selection, shared-expert combine,
 * routing, bucketing, the shared slots' own pass when there are more than 128
 * landmarks, expert attention, merge) and at its end; up to max_marks events
 * in total (created here, kept for reuse). Process-wide; not for concurrent
 * calls. */
mita_status mita_profile_begin(int max_marks);

/* Closes the profile: waits for the last event, sums the milliseconds of each
 * phase over all profiled calls into ms[i] and writes the phase names,
 * newline-separated, into `names`. Returns the number of phases (<= max_phases)
 * or -1 on a CUDA error. */
int mita_profile_end(char* names, size_t names_bytes, double* ms, int max_phases);

#ifdef __cplusplus
}
#endif

#endif /* MITA_H */
