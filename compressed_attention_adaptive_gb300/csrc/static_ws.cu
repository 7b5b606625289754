// The forward pass on a workspace the library owns, for callers that cannot
// allocate device memory themselves: code that must not call cudaMalloc
// (which can synchronize the whole device, or is forbidden where another
// framework owns all device memory through its own pool), plugins that only
// receive the tensors they work on, and real-time or capture-sensitive code
// that may enqueue work but never allocate.
//
// The workspace is one file-scope device array of MITA_STATIC_WORKSPACE_BYTES.
// Every GPU on which the library is loaded holds it until the process exits.
// In host code the array's name is only a stand-in for the symbol: its device
// address comes from cudaGetSymbolAddress, once per device, on the first call
// made with that device current.
#include <stdio.h>

#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[MITA_STATIC_WORKSPACE_BYTES];

std::mutex g_static_mu;
constexpr int kMaxDevices = 256;
void* g_static_addr[kMaxDevices] = {};  // device address of g_static_ws per device ordinal

}  // namespace

extern "C" mita_status mita_forward_static(const mita_params* p, const void* Q, const void* K, const void* V,
                                           void* O, int32_t* status_out, void* stream) {
    using namespace mita;
    clear_error();
    mita_status st = validate(p);
    if (st) return st;
    const size_t need = mita_workspace_size(p);
    if (need > MITA_STATIC_WORKSPACE_BYTES) {
        char msg[160];
        snprintf(msg, sizeof msg, "problem needs %zu bytes of workspace; the static area holds %zu", need,
                 (size_t)MITA_STATIC_WORKSPACE_BYTES);
        return report_error(MITA_ERR_UNSUPPORTED, msg);
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return report_error(MITA_ERR_CUDA, "no usable current device");
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        if (!g_static_addr[dev]) {
            void* addr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&addr, g_static_ws);
            if (e != cudaSuccess || !addr) {
                char msg[160];
                snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static workspace: %s", cudaGetErrorString(e));
                return report_error(MITA_ERR_CUDA, msg);
            }
            g_static_addr[dev] = addr;
        }
        ws = g_static_addr[dev];
    }
    st = forward_on_workspace(p, Q, K, V, O, ws, MITA_STATIC_WORKSPACE_BYTES, stream);
    if (st) return st;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, (cudaStream_t)stream) != cudaSuccess)
        return report_error(MITA_ERR_CUDA, "copy of the device status word failed");
    return MITA_OK;
}
