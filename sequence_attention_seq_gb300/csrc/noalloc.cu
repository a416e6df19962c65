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
// cudaGetSymbolAddress, taken once per device (once per CUDA context of that device) with
// that device current, on the first call made there; make that first call before any
// stream capture begins.  The address is cached together with the identifier of the
// context it belongs to: after cudaDeviceReset the device gets a new primary context (with
// a new copy of the array), and the next call looks the address up again.  With CUDA's
// lazy module loading (the default) the first lookup is also when the module holding the
// array is loaded and its memory reserved, so that first call fails with ULY_ERR_CUDA if
// the device has less than kNoAllocScratchBytes free.
//
// Nothing on this path allocates: no cudaMalloc or cudaFree, and no host heap allocation
// in this library's code (the argument records and overlap checks live on the stack).
#include <cuda.h>

#include <mutex>

#include "../../include/ulysses.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = ULYSSES_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(f);
}

// Identifier of the calling thread's current context (0 if there is none yet).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    return !ctx || get_id(ctx, id) == CUDA_SUCCESS;
}

struct CachedAddress {
    unsigned long long ctx_id;  // context the address belongs to (0: none cached)
    void* addr;
};

std::mutex g_scratch_mu;
CachedAddress g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array in the current device's context (set-up on first
// use in each context).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = 0;
    if (!current_context_id(&id)) return cudaErrorNotSupported;
    CachedAddress& c = g_scratch_addr[dev];
    if (id != 0 && c.ctx_id == id && c.addr) {
        *out = c.addr;
        return cudaSuccess;
    }
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);  // initialises the context if needed
    if (e != cudaSuccess) return e;
    if (!current_context_id(&id) || id == 0) return cudaErrorNotSupported;
    c.ctx_id = id;
    c.addr = ptr;
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
