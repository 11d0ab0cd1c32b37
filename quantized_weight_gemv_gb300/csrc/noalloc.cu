// qgemv_grouped_noalloc: the grouped GEMV for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain a workspace: code that runs where the CUDA
// allocator must not be touched (inside a host callback or a real-time decode loop
// that forbids allocation), plug-ins whose host application owns every device
// allocation, or C callers that link only this library and have no allocator of
// their own.  For them this entry point keeps the grouped GEMV's scratch - the
// quantised activations - in a fixed array that is part of the library's device
// image, so the call itself needs no memory beyond the caller's inputs and outputs.
//
// The array is QG_NOALLOC_WS_BYTES (2 MiB).  Every GPU on which the library is
// loaded holds it until the process exits.  All calls share it:
//  * calls whose work could overlap on the GPU (on different streams, or on one
//    stream with programmatic dependent launch across unrelated work that uses this
//    entry point too) race on it and must be ordered by the caller;
//  * it keeps the contents of the last call; nothing in it has to start at zero,
//    because each call writes every byte it reads before reading it.
#include <mutex>

#include "qg_internal.h"

namespace {

// The scratch itself.  In host code this name is only a stand-in for the device
// array: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_ws[QG_NOALLOC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices];  // device address of g_noalloc_ws, per device (nullptr: not set up)

// Device address of the scratch on the current device; looked up once per device,
// with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return QG_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ws_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return QG_ERR_CUDA;
        }
        g_ws_addr[dev] = p;
    }
    *out = g_ws_addr[dev];
    return QG_OK;
}

}  // namespace

extern "C" int qgemv_grouped_noalloc(int bits, const qg_gemv_desc* descs, int count, unsigned flags, void* stream) {
    // the descriptors first, exactly as qgemv_grouped checks them (so a bad k or n gives
    // the same status as there), then the size of the group's quantised activations
    int active = 0;
    int rc = qg::check_grouped(bits, descs, count, &active);
    if (rc != QG_OK || active == 0) return rc;
    if (qg_grouped_workspace_bytes(descs, count) > (size_t)QG_NOALLOC_WS_BYTES) return QG_ERR_WORKSPACE;
    void* ws = nullptr;
    rc = scratch_address(&ws);
    if (rc != QG_OK) return rc;
    // the work is launched by the allocating entry point, on the fixed scratch
    return qgemv_grouped(bits, descs, count, ws, (size_t)QG_NOALLOC_WS_BYTES, flags, stream);
}
