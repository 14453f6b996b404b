// qgemm_noalloc.cu -- qgemm_q4k for callers that cannot allocate device memory.
//
// Some callers cannot obtain device memory at the point where they call the
// GEMM: a plugin running inside a host framework that owns all device memory
// through its own pool and hands the plugin no allocator, or code on a path
// where cudaMalloc is not allowed or not acceptable (inside a host callback,
// or a latency-critical path that must not pay for an allocation and the
// device synchronisation it can imply).  Such a caller cannot provide the
// workspace qgemm_q4k needs for the fp16 copy of the activations.
//
// qgemm_q4k_noalloc gives them the same computation with the scratch held in
// a fixed array in device memory that this library defines at file scope
// (QGEMM_NOALLOC_SCRATCH_BYTES, 16 MiB).  Every GPU that loads the library
// holds that array until the process exits.  The entry point itself calls no
// cudaMalloc, cudaFree or allocating library routine.
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "qgemm.h"

namespace {

// The shared scratch: one per device, in the module's global memory.  Host
// code must not use this name as an address (on the host it is only a
// stand-in); the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[QGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mtx;
void* g_scratch_ptr[kMaxDevices];   // set once the lookup has succeeded on that device

// The device address of this device's copy of the scratch array, looked up
// with that device current.  A failed lookup is not remembered: the next call
// tries again.  Its error is also taken off the runtime's last-error slot, so
// that it is not reported later by an unrelated launch check.
cudaError_t scratch_of(int dev, void** out) {
    std::lock_guard<std::mutex> lk(g_setup_mtx);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int qgemm_q4k_noalloc(const void* w, int64_t N, int64_t K, int64_t ldw, const int8_t* xqs,
                                 const float* xd, const int16_t* xbsums, int64_t M, float* y, int64_t ldy,
                                 qgemm_stream_t stream) {
    const size_t need = qgemm_workspace_bytes(M, N, K);
    if (need > QGEMM_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "qgemm_q4k_noalloc: M=%lld, K=%lld needs %zu bytes of scratch; the built-in scratch holds %zu "
                 "(use qgemm_q4k with a workspace)",
                 static_cast<long long>(M), static_cast<long long>(K), need,
                 static_cast<size_t>(QGEMM_NOALLOC_SCRATCH_BYTES));
        return qg::set_last_error(QGEMM_EUNSUPPORTED, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return qg::set_last_error(QGEMM_ECUDA, "qgemm_q4k_noalloc: no usable current device");
    // Set-up, once per device (retried until it succeeds), with that device
    // current: look up the device address of this device's scratch array.
    void* scratch = nullptr;
    e = scratch_of(dev, &scratch);
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof(msg), "qgemm_q4k_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return qg::set_last_error(QGEMM_ECUDA, msg);
    }
    // Everything the GEMM reads from the scratch is first written by the
    // operand-preparation kernel of the same call, so nothing has to be
    // cleared between calls.
    return qgemm_q4k(w, N, K, ldw, xqs, xd, xbsums, M, y, ldy, scratch, QGEMM_NOALLOC_SCRATCH_BYTES,
                     stream);
}
