// Host-side interfaces between the C ABI layer (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace uly {

constexpr int kMaxRanks = 64;  // largest P any entry point accepts

// ----------------------------------------------------------------------- permutes
// One tensor of an all-to-all exchange.  `contig[r]` are the head-layout buffers (written
// or read as contiguous slabs), `strided[j]` the seq-layout buffers (rows of h*d elements).
struct PermuteTensor {
    const void* src[kMaxRanks];
    void* dst[kMaxRanks];
    int h;  // heads of this tensor in seq layout (h_q for Q/O, h_kv for K/V)
};

// direction: 0 = seq -> head (all-to-all #1), 1 = head -> seq (all-to-all #2).
cudaError_t launch_permute(int direction, int P, int b, int s, int d, int elem_bytes, const PermuteTensor* tensors,
                           int ntensors, cudaStream_t stream);

// ----------------------------------------------------------------- fp32 attention
struct AttnPtrs {
    const void* q[kMaxRanks];
    const void* k[kMaxRanks];
    const void* v[kMaxRanks];
    void* o[kMaxRanks];
};

// Head-layout local attention, fp32 in/out, all P ranks in one grid.
cudaError_t launch_attention_fp32(int P, int b, int s, int h_q, int h_kv, int d, int causal, const AttnPtrs& ptrs,
                                  cudaStream_t stream);

// ------------------------------------------------------ bf16 tensor-core attention
// fused == 0: head-layout buffers per rank (the ptrs arrays hold head-layout pointers).
// fused != 0: seq-layout buffers per rank; the kernel gathers/scatters itself.
int tc_attention_supported(int d);
cudaError_t launch_attention_tc(int P, int b, int s, int h_q, int h_kv, int d, int causal, int fused,
                                const AttnPtrs& ptrs, cudaStream_t stream, int* unsupported);

// Device error word of the tensor-core kernels (bounded waits that gave up).
cudaError_t read_device_error(unsigned int* value, int clear);

}  // namespace uly
