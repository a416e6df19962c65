// ulysses_dist_attn_fwd_noalloc: the unfused forward with its scratch memory in a
// fixed, library-owned device array instead of a caller-supplied workspace.
//
// Some callers cannot call cudaMalloc (or any allocating routine): an application whose
// memory pool has already reserved all the device memory it is allowed to use, or a
// plugin loaded into a host runtime that gives it no allocator and forbids allocation
// (and the device synchronisation cudaMalloc may cause) on its hot path.  For them this
// entry point needs only the inputs and outputs they already own.
//
// The scratch is the file-scope array below: kNoAllocScratchBytes of device memory that
// every GPU which loads this library holds until the process exits.  All calls share it
// and it keeps the last call's contents; the unfused forward writes every scratch byte it
// later reads (the exchange writes the head-layout copies before attention reads them,
// attention writes the head-layout output before the second exchange reads it), so
// nothing has to start at zero.  Calls whose work overlaps on the GPU (for instance on
// two streams) race on the array and give wrong results: serialise them.
//
// In host code `g_noalloc_scratch` is only a host-side stand-in for the device array, not
// a device address; passing it to a kernel would fault or, where the GPU can reach host
// memory, silently use the wrong memory.  The real address comes from
// cudaGetSymbolAddress, taken once per device with that device current, on the first call
// made on that device; make that first call before any stream capture begins.
#include <mutex>

#include "../../include/ulysses.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = ULYSSES_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (dev >= 0 && dev < kMaxDevices && g_scratch_addr[dev]) {
        *out = g_scratch_addr[dev];
        return cudaSuccess;
    }
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) g_scratch_addr[dev] = ptr;
    *out = ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" uly_status ulysses_dist_attn_fwd_noalloc(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                                    int causal, const void* const* q_seq, const void* const* k_seq,
                                                    const void* const* v_seq, void* const* o_seq,
                                                    cudaStream_t stream) {
    const size_t need = ulysses_dist_attn_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, 0);
    if (need == 0)  // invalid arguments: let the regular entry point name the error
        return ulysses_dist_attn_fwd(P, b, s, h_q, h_kv, d, dtype, causal, q_seq, k_seq, v_seq, o_seq, nullptr, 0,
                                     0, stream);
    if (need > kNoAllocScratchBytes) return ULY_ERR_INVALID_ARG;  // beyond the fixed scratch
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return ULY_ERR_CUDA;
    return ulysses_dist_attn_fwd(P, b, s, h_q, h_kv, d, dtype, causal, q_seq, k_seq, v_seq, o_seq, scratch,
                                 kNoAllocScratchBytes, 0, stream);
}
