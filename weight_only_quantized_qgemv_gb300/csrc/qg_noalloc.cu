// qg_noalloc.cu -- qexpert_group for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: a plugin running inside a
// host application that owns all of the GPU's memory through its own allocator
// and hands plugins none, or a decode loop that must never allocate.  This
// entry point gives them the routed-expert group with its scratch in a fixed
// array compiled into the library: every GPU that loads the library holds
// QEXPERT_NOALLOC_SCRATCH_BYTES of it until the process exits.  The caller
// still passes the inputs and the output.
#include <atomic>

#include <cuda_runtime.h>

#include "qg_internal.h"

// The scratch itself.  In host code this name is only a stand-in for the
// device array, never a device address: the address is looked up per device.
static __device__ __align__(256) unsigned char g_expert_scratch[QEXPERT_NOALLOC_SCRATCH_BYTES];

// Device address of g_expert_scratch on each device, looked up at the first
// call made with that device current.  Atomic, so host threads making their
// first call on a device at the same time do not race (they store the same
// address).  A cudaDeviceReset invalidates it: reload the library after one.
static std::atomic<void*> g_scratch_addr[64];

extern "C" int qexpert_group_noalloc(int fmt, int gs, const void* gate, const float* gate_s, const void* up,
                                     const float* up_s, const void* down, const float* down_s, int E, int D, int F,
                                     const float* x, int s, int k, const int32_t* ids, const float* wts, float* out,
                                     int32_t* status_dev, void* stream)
{
    const size_t need = qexpert_group_workspace(E, D, F, s, k);
    if (need > (size_t)QEXPERT_NOALLOC_SCRATCH_BYTES) return QSTATUS_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QSTATUS_LAUNCH;
    void* scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (scratch == nullptr) {
        if (cudaGetSymbolAddress(&scratch, g_expert_scratch) != cudaSuccess || scratch == nullptr)
            return QSTATUS_LAUNCH;
        g_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
    return qexpert_group(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts, out, scratch,
                         (size_t)QEXPERT_NOALLOC_SCRATCH_BYTES, status_dev, stream);
}
