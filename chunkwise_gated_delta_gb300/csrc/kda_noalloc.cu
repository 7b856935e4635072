// kda_chunk_fwd_noalloc: the forward for callers that cannot allocate device
// memory at the point of the call.
//
// kda_chunk_fwd needs a workspace besides its inputs and outputs: its first
// word is where the kernels report a device-side error, and on the bf16 path
// the rest, when given, holds the chunk records of the two-kernel form.
// Callers that cannot provide one -- frameworks whose caching allocator owns
// all device memory, plugins and embedded hosts that only hand over the input
// and output tensors, latency-critical paths that cannot afford a cudaMalloc
// (which may synchronise the device) -- use this entry point instead.  The status word then lives in a small array owned by
// the library, defined below (every GPU that loads the library holds it until
// the process exits), and the forward runs its single-kernel form, which
// builds each chunk's Z inside the scan kernel and needs no records.
#include <cuda_runtime.h>

#include "kda.h"

namespace {

// Library-owned replacement for the caller's workspace: the status word,
// padded to an aligned block -- all the single-kernel forward needs, at any
// problem size, so no size is rejected for want of scratch.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// In host code `g_noalloc_scratch` names a host-side stand-in, not the device
// array.  Its device address belongs to the CUDA context that is current, not
// to the device number: after cudaDeviceReset, or under a driver-API context
// other than the primary one, an address kept from an earlier call would point
// at freed memory.  So every call looks it up again, with the caller's device
// current; the lookup allocates nothing.
cudaError_t scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(const kda_fwd_args *args, kda_stream_t stream) {
    if (!args) return KDA_ERR_INVALID_ARG;
    kda_fwd_args a = *args;
    a.workspace = nullptr;          // the caller's workspace fields are ignored
    a.workspace_bytes = 0;
    if (kda_chunk_fwd_workspace(&a) == 0) return kda_chunk_fwd(&a, stream);   // reports the argument error
    const size_t need = kNoAllocScratchBytes;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (s != nullptr) {
        // the array of the current device is cleared and used on `stream`: both must be on it
        int sdev = -1;
        if (cudaStreamGetDevice(s, &sdev) != cudaSuccess) return KDA_ERR_CUDA;
        if (sdev != dev) return KDA_ERR_INVALID_ARG;
    }
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    // The array keeps the previous call's contents: the status word must start at zero.
    if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    a.workspace = scratch;
    a.workspace_bytes = kNoAllocScratchBytes;
    return kda_chunk_fwd(&a, stream);
}
