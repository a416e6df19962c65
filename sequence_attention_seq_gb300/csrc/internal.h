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
    int h;     // heads of this tensor in seq layout (h_q for Q/O, h_kv for K/V)
    int hsub;  // heads per rank moved by this call (0: all h/P); the head-layout side holds hsub heads
    int hoff;  // first moved head within each rank's group of h/P heads
    int rep;   // > 1: K/V heads replicated (h < P, P % h == 0): rank r receives head r / rep only
               // (direction 0 only)
};

// K/V heads per rank, and how many ranks share each K/V head.  With fewer K/V heads than
// ranks (P a multiple of h_kv), each K/V head is replicated on P / h_kv consecutive ranks,
// one head per rank: rank r's query heads are exactly the ones that use K/V head r / rep.
inline int kv_heads_per_rank(int P, int h_kv) { return h_kv >= P ? h_kv / P : 1; }
inline int kv_replication(int P, int h_kv) { return h_kv >= P ? 1 : P / h_kv; }

// direction: 0 = seq -> head (all-to-all #1), 1 = head -> seq (all-to-all #2); 1 to 4 tensors.
cudaError_t launch_permute(int direction, int P, int b, int s, int d, int elem_bytes, const PermuteTensor* tensors,
                           int ntensors, cudaStream_t stream);

// out[c][a] = in[a][c] for A x C runs of run_bytes each: the local halves of one rank's
// all-to-all with other GPUs (the send blocks before the collective, the layout after it).
// block_transpose_fits: false when a slab (A runs) would exceed the kernel's 32-bit vector
// index (2^31 - 1 vectors of up to 16 bytes); launch_block_transpose then refuses the copy.
bool block_transpose_fits(uint64_t A, uint64_t C, uint64_t run_bytes, const void* in, const void* out);
cudaError_t launch_block_transpose(uint64_t A, uint64_t C, uint64_t run_bytes, const void* in, void* out,
                                   cudaStream_t stream);

// The backward of the replicating exchange: gradients of K/V heads replicated on `rep` ranks.
// src[r]: rank r's fp32 head-layout partial gradient [b][s][1][d] (from its own query heads);
// dst[j]: bf16 seq layout [b][s/P][h_kv][d] = the sum over the rep replicas, rounded once.
cudaError_t launch_kv_grad_sum(int P, int rep, int b, int s, int h_kv, int d, const void* const* src,
                               void* const* dst, cudaStream_t stream);

// ----------------------------------------------------------------- fp32 attention
struct AttnPtrs {
    const void* q[kMaxRanks];
    const void* k[kMaxRanks];
    const void* v[kMaxRanks];
    void* o[kMaxRanks];
    float* lse[kMaxRanks];  // optional (all null = none): per-row log-sum-exp, [b][h_q/P][s] fp32
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

// Two-level (Ulysses x Ring) attention: P = Pu*Pr head-layout buffers, buffer g*Pu + u
// holding ring group g's s/Pr tokens of heads [u*h/Pu, (u+1)*h/Pu); every query attends
// over the whole sequence, reading the K/V blocks of the other groups from their buffers.
// Needs P <= 16 and (s/Pr) % 128 == 0 (else *unsupported = 1).
cudaError_t launch_attention_tc_usp(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, int causal,
                                    const AttnPtrs& head, cudaStream_t stream, int* unsupported);

// Backward of the bf16 tensor-core attention.  fused == 0: q/k/v/dout/dq/dk/dv are the
// head-layout buffers of every head rank.  fused != 0: they are the seq-layout buffers of
// every seq rank, and the kernels gather/scatter through their tile addressing (needs
// P <= 16 and (s/P) % 128 == 0, else *unsupported = 1).  O and dO for the row sums D are
// read from `o_rows` / `do_rows` in head layout, or in seq layout when od_seq_layout != 0
// (then indexed by seq rank j, not by head rank r).  The statistics (lse, lse2, dsum)
// are always per head rank.
struct BwdPtrs {
    int od_seq_layout;
    const void* q[kMaxRanks];
    const void* k[kMaxRanks];
    const void* v[kMaxRanks];
    const void* dout[kMaxRanks];
    const void* o_rows[kMaxRanks];
    const void* do_rows[kMaxRanks];
    const float* lse[kMaxRanks];  // [b][h_q/P][s], natural log, from the forward
    void* dq[kMaxRanks];
    void* dk[kMaxRanks];
    void* dv[kMaxRanks];
    float* lse2[kMaxRanks];       // scratch [b][h_q/P][s_pad], s_pad = ceil(s/128)*128
    float* dsum[kMaxRanks];       // scratch, same shape
    int kv_grad_f32;              // unfused only: dk/dv receive fp32 partial sums (replicated K/V heads)
};
cudaError_t launch_attention_bwd_tc(int P, int b, int s, int h_q, int h_kv, int d, int causal, int fused,
                                    const BwdPtrs& ptrs, cudaStream_t stream, int* unsupported);
// Backward of the two-level forward: q/k/v/dout/dq/dk/dv are the P = Pu*Pr ranks' buffers in
// the group head layout [b][s/Pr][h/Pu][d]; o_rows/do_rows the seq-layout O and dO
// (od_seq_layout must be 1); lse/lse2/dsum one array per Ulysses unit u < Pu over all s rows.
cudaError_t launch_attention_bwd_tc_usp(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, int causal,
                                        const BwdPtrs& ptrs, cudaStream_t stream, int* unsupported);

// Device error word of the tensor-core kernels (bounded waits that gave up).
// One CTA whose bounded wait on a barrier that never completes gives up after limit_ns and
// sets the timeout bit of the device error word (the failure path, exercised without a fault).
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);
cudaError_t read_device_error(unsigned int* value, int clear);

}  // namespace uly
