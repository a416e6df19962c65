/*
 * ulysses.h -- C ABI of the GB300 (sm_103a) Ulysses DistributedAttention forward and backward.
 *
 * The method ("DeepSpeed-Ulysses 深度解析：用 All-to-All 序列并行撑起百万 Token 超长序列训练",
 * section "核心设计：沿序列切分 + 两次 All-to-All", steps 1-5): each of P sequence-parallel
 * ranks holds a contiguous block of s/P tokens of Q, K and V with all heads; all-to-all #1
 * turns that into all s tokens of h/P heads; every rank runs ordinary attention
 * softmax(Q K^T / sqrt(d)) V on its heads; all-to-all #2 restores the sequence split.
 *
 * On one GPU the P ranks are P disjoint device buffers, so each all-to-all is a transpose
 * in device memory.  Layouts (row-major, batch first, element type `uly_dtype`):
 *     seq layout  (rank j):  [b][s/P][h][d]   tokens j*s/P .. (j+1)*s/P-1, all heads
 *     head layout (rank r):  [b][s][h/P][d]   all tokens, heads r*h/P .. (r+1)*h/P-1
 * Token blocks and head groups are contiguous and ordered by rank ("02 · DeepSpeed-Ulysses",
 * section 2 "all-to-all 的转置与重分布": split the head axis, part j to rank j, concatenate
 * what arrives along the sequence axis).
 *
 * Common rules for every entry point:
 *  - Pointer arrays (`const void* const* x`) are HOST arrays of P DEVICE pointers, one per
 *    rank, read only during the call.  Every device pointer must be 16-byte aligned.
 *  - The caller owns all device memory and the stream.  The library allocates no device
 *    memory, keeps no per-call state, and may be called from several host threads.
 *  - Calls only enqueue work on `stream` and return; a kernel fault surfaces through the
 *    usual CUDA error checks on that stream.  Argument errors are reported before any
 *    work is enqueued, and nothing is written in that case.
 *  - Outputs must not overlap inputs (out-of-place only); this is checked.
 *  - Return value: ULY_OK, or the first error found (see uly_status).
 */
#ifndef ULYSSES_GB300_H
#define ULYSSES_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ULY_OK = 0,
    ULY_ERR_INVALID_ARG = 1, /* bad sizes or divisibility, null/misaligned/overlapping pointers, small workspace */
    ULY_ERR_UNSUPPORTED = 2, /* valid arguments for which no kernel exists (dtype/d combination, fused shape) */
    ULY_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a kernel launch failed */
    ULY_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (reported by ulysses_device_status) */
} uly_status;

typedef enum {
    ULY_FP32 = 0, /* IEEE binary32 inputs and outputs, fp32 arithmetic throughout (no TF32) */
    ULY_BF16 = 1  /* bfloat16 inputs and outputs, fp32 accumulation and softmax */
} uly_dtype;

/*
 * All-to-all #1, sequence -> head ("02 · DeepSpeed-Ulysses", section 2, send/receive
 * listing; "DeepSpeed-Ulysses 深度解析", step 3).
 *   out_head[r][bb][j*s/P + t][hh][:] = in_seq[j][bb][t][r*h/P + hh][:]
 * for every rank r, source rank j, batch bb < b, token t < s/P, head hh < h/P.
 * Sizes: 1 <= P <= 64, b >= 1, s >= 1, h >= 1, d >= 1, s % P == 0, h % P == 0.
 * in_seq: P pointers to [b][s/P][h][d]; out_head: P pointers to [b][s][h/P][d].
 * A pure bit copy (dtype only fixes the element size), so the result is bit-exact.
 */
uly_status ulysses_a2a_seq2head(int P, int b, int s, int h, int d, uly_dtype dtype,
                                const void* const* in_seq, void* const* out_head,
                                cudaStream_t stream);

/*
 * All-to-all #2, head -> sequence: the inverse of ulysses_a2a_seq2head ("02 ·
 * DeepSpeed-Ulysses", section 2, last paragraph; section 1 figure caption).
 *   out_seq[j][bb][t][r*h/P + hh][:] = in_head[r][bb][j*s/P + t][hh][:]
 * in_head: P pointers to [b][s][h/P][d]; out_seq: P pointers to [b][s/P][h][d].
 * Same size rules as ulysses_a2a_seq2head; bit-exact.
 */
uly_status ulysses_a2a_head2seq(int P, int b, int s, int h, int d, uly_dtype dtype,
                                const void* const* in_head, void* const* out_seq,
                                cudaStream_t stream);

/*
 * The local halves of one rank's all-to-all when the P ranks are P processes on P GPUs
 * (one rank per process, the exchange itself a collective between them): "DeepSpeed-Ulysses
 * 深度解析", section "构建序列并行通信组" (DistributedAttention over a sequence-parallel
 * process group) and "大模型分布式训练通信原语及其应用", section 5 "AllToAll（全交换）"
 * (every rank cuts its input into P parts, sends part i to rank i, and lays the parts it
 * receives out in sending-rank order).  With S = s/P and H = h/P, every send and receive
 * buffer is P contiguous blocks [P][b][S][H][d] -- block i of the send buffer goes to rank i,
 * block j of the receive buffer came from rank j -- so an equal-split all-to-all (NCCL
 * ncclSend/ncclRecv pairs, or torch.distributed.all_to_all_single) moves them:
 *   ulysses_a2a_pack(0, ...):   local = this rank's seq shard [b][S][h][d];
 *                               send block r = heads [r*H, (r+1)*H) of every token.
 *   ulysses_a2a_unpack(0, ...): recv block j = tokens [j*S, (j+1)*S) of this rank's heads;
 *                               local = this rank's head shard [b][s][H][d].
 *   ulysses_a2a_pack(1, ...):   local = this rank's head shard [b][s][H][d];
 *                               send block j = tokens [j*S, (j+1)*S).
 *   ulysses_a2a_unpack(1, ...): recv block r = heads [r*H, (r+1)*H) of this rank's tokens;
 *                               local = this rank's seq shard [b][S][h][d].
 * pack(0), the collective and unpack(0) together give this rank's part of
 * ulysses_a2a_seq2head; pack(1), the collective and unpack(1) its part of
 * ulysses_a2a_head2seq.  Both sides hold b*S*h*d elements.  Sizes as the exchanges above;
 * besides, the largest contiguous piece a call writes (b*S*H*d elements for pack(0),
 * s*H*d for unpack(0), b*S*H*d for pack(1)) must fit in 2^31 - 1 copy vectors (16 bytes each
 * when the rows and pointers are 16-byte aligned, else 8, 4, 2 or 1).  A larger piece,
 * direction not 0 or 1, a null or misaligned pointer, or overlapping in/out buffers give
 * ULY_ERR_INVALID_ARG.  Bit copies.  Device pointers, owned by the caller; enqueued on stream.
 */
uly_status ulysses_a2a_pack(int direction, int P, int b, int s, int h, int d, uly_dtype dtype,
                            const void* local, void* send, cudaStream_t stream);
uly_status ulysses_a2a_unpack(int direction, int P, int b, int s, int h, int d, uly_dtype dtype,
                              const void* recv, void* local, cudaStream_t stream);


/*
 * Local attention of every rank, head layout in and out ("DeepSpeed-Ulysses 深度解析",
 * step 4: softmax(Q K^T / sqrt(d)) V per local head over the full sequence).
 *   o_head[r][bb][i][hh][:] = sum_j softmax_j(q.k_j / sqrt(d)) v_j
 * with q = q_head[r][bb][i][hh], k_j / v_j = k_head / v_head[r][bb][j][hh / (h_q/h_kv)].
 * causal != 0 masks keys j > i (global positions: after all-to-all #1 the local token
 * index is the global one -- "长上下文训练中的 SP 与 CP", section on Ring Attention,
 * causal paragraph).  The scale is fixed at 1/sqrt(d).
 * Sizes: P, b, s >= 1; h_q % P == 0, h_q % h_kv == 0 (grouped K/V heads: rank r's query
 * heads read only the K/V heads it holds -- "02 · DeepSpeed-Ulysses", section 3), and
 * either h_kv % P == 0 (every rank holds h_kv/P K/V heads) or P % h_kv == 0 (fewer K/V
 * heads than ranks: each K/V head is replicated on the rep = P/h_kv ranks whose query
 * heads use it, rank r holding head r/rep -- "DeepSpeed-Ulysses 深度解析", sections
 * "两行代码替换注意力" (num_kv_heads) and "构建序列并行通信组" (head counts and the
 * degree divide each other, one way or the other); "长上下文训练中的 SP 与 CP", section on
 * Ulysses (replicating K/V lifts the divisibility rule at the cost of memory and traffic)).
 * Else ULY_ERR_INVALID_ARG.  Below, Hk = h_kv/P, or 1 when replicated.
 * q_head / o_head: P pointers to [b][s][h_q/P][d]; k_head / v_head: P pointers to
 * [b][s][Hk][d].
 * Kernels: ULY_BF16 with d in {64, 128} (tcgen05 tensor cores, fp32 accumulation, the
 * softmax weights rounded to bf16 before the P.V product, output rounded to nearest even);
 * ULY_FP32 with d % 4 == 0 and d <= 256 (fp32 FMA, no tensor cores).  Other combinations
 * return ULY_ERR_UNSUPPORTED.  Any s is accepted (ragged tiles are masked).
 */
uly_status ulysses_local_attention(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                   int causal,
                                   const void* const* q_head, const void* const* k_head,
                                   const void* const* v_head, void* const* o_head,
                                   cudaStream_t stream);

/*
 * Bytes of device workspace ulysses_dist_attn_fwd needs for these arguments: the
 * head-layout copies of Q, K, V and O of every rank (each 256-byte aligned) when
 * fused == 0, and 0 when fused != 0.  Returns 0 for arguments that are invalid.
 */
size_t ulysses_dist_attn_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d,
                                         uly_dtype dtype, int fused);

/*
 * The whole DistributedAttention forward ("DeepSpeed-Ulysses 深度解析", steps 3-5):
 * all-to-all #1 on Q, K and V, local attention on every rank, all-to-all #2 on the output.
 *   q_seq / o_seq: P pointers to [b][s/P][h_q][d]; k_seq / v_seq: P pointers to
 *   [b][s/P][h_kv][d].  Size rules as ulysses_local_attention.  With replicated K/V
 *   heads all-to-all #1 sends K/V head r/rep to rank r (a broadcast of every head to its
 *   rep ranks).
 * fused == 0: three launches (one for the Q, K and V exchanges, one attention, one
 *   output exchange) through `workspace` (device memory, 256-byte aligned, at least
 *   ulysses_dist_attn_workspace_bytes(...) bytes, owned by the caller).
 * fused != 0: one launch; the attention kernel reads its Q/K/V tiles straight from the
 *   seq-layout buffers and stores its output tiles straight into o_seq, so no
 *   head-layout copy exists.  Needs ULY_BF16, d in {64, 128} and (s/P) % 128 == 0, else
 *   ULY_ERR_UNSUPPORTED (any P up to 64).  workspace may be NULL.
 * Both paths give the same bits for the same inputs.
 */
uly_status ulysses_dist_attn_fwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                 int causal,
                                 const void* const* q_seq, const void* const* k_seq,
                                 const void* const* v_seq, void* const* o_seq,
                                 void* workspace, size_t workspace_bytes, int fused,
                                 cudaStream_t stream);

/*
 * The unfused forward with its exchanges overlapped with attention ("DeepSpeed-Ulysses
 * 深度解析", section "怎么用：极简接入与通信组初始化", subsection "两行代码替换注意力":
 * passing `sp_stream` to DistributedAttention overlaps the Q/K/V all-to-all with the
 * computation).  The local heads of every rank are split into n_chunks equal groups
 * (chunk c = local query heads [c*h_q/P/n, (c+1)*h_q/P/n) and the matching K/V heads).
 * On `side_stream` run, in order: all-to-all #1 of chunks 0 and 1, then for every chunk c
 * all-to-all #2 of c (after c's attention) and all-to-all #1 of c+2; on `stream` the
 * attention of chunk c runs once c's inputs are there.  So while chunk c is computed the
 * side stream moves chunk c-1's output and chunk c+1's inputs.  `stream` waits for
 * everything before the call returns control of the results to it; `side_stream` first
 * waits for the work already on `stream`.  side_stream may equal stream (no overlap).
 * Arguments and results as ulysses_dist_attn_fwd with fused == 0 -- the same bits --
 * plus: 1 <= n_chunks <= 64 and (h_q/P) % n_chunks == 0, and either (h_kv/P) % n_chunks
 * == 0 (every chunk has its own K/V heads) or n_chunks % (h_kv/P) == 0 (grouped heads:
 * n_chunks/(h_kv/P) consecutive chunks share one K/V head, exchanged with the first of
 * them), else ULY_ERR_INVALID_ARG.  Replicated K/V heads (P % h_kv == 0) leave every rank
 * one K/V head, which all chunks share (exchanged, as a broadcast, with chunk 0);
 * workspace: 256-byte aligned, at least ulysses_dist_attn_overlap_workspace_bytes(...)
 * bytes (the chunks' head-layout Q, K, V, O).  The call creates and destroys CUDA events
 * (host objects) for the cross-stream ordering; it allocates no device memory.
 */
size_t ulysses_dist_attn_overlap_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d,
                                                 uly_dtype dtype, int n_chunks);
uly_status ulysses_dist_attn_fwd_overlap(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                         int causal,
                                         const void* const* q_seq, const void* const* k_seq,
                                         const void* const* v_seq, void* const* o_seq,
                                         void* workspace, size_t workspace_bytes, int n_chunks,
                                         cudaStream_t stream, cudaStream_t side_stream);

/*
 * The two-level forward, Ulysses inside groups and a ring across them ("长上下文训练中的
 * SP 与 CP", section "组合与配置：区分算法组合和并行维度", subsection "Ulysses + Ring：组合两种
 * Attention 路线": 256K tokens on 8 devices as Ulysses degree 4 x Ring degree 2;
 * "02 · DeepSpeed-Ulysses", section 4 "a2a+p2p 分层 CP").  P = Pu * Pr ranks; rank
 * j = g*Pu + u holds tokens [j*s/P, (j+1)*s/P) of every head, so ring group g (ranks
 * g*Pu .. g*Pu+Pu-1) holds the contiguous segment g of s/Pr tokens.
 *  1. all-to-all #1 inside every group: rank (g, u) gets segment g's tokens of heads
 *     [u*h/Pu, (u+1)*h/Pu) (query and K/V heads alike);
 *  2. every rank's queries attend over the whole sequence, taking the K/V of segment g'
 *     from rank (g', u) -- the blocks a ring across the groups would pass to it
 *     ("Ring Attention：Q 留在本地，KV 沿环传递") -- merged by the online softmax of the
 *     attention kernel, with the causal mask on global positions;
 *  3. all-to-all #2 inside every group.
 * On one GPU the ring's transfers are reads of the other ranks' buffers (no copy).
 *   q_seq / o_seq: P pointers to [b][s/P][h_q][d]; k_seq / v_seq: [b][s/P][h_kv][d].
 * Sizes: Pu, Pr >= 1, Pu*Pr <= 64, s % (Pu*Pr) == 0, h_q % Pu == 0, h_q % h_kv == 0, and
 * h_kv % Pu == 0 or Pu % h_kv == 0 (fewer K/V heads than Ulysses ranks: each K/V head is
 * replicated on the Pu/h_kv ranks of every group whose query heads use it, as in
 * ulysses_local_attention with P = Pu), else ULY_ERR_INVALID_ARG.  Kernel: ULY_BF16, d in {64, 128},
 * and (s/Pr) % 128 == 0, else ULY_ERR_UNSUPPORTED.  The result equals
 * ulysses_dist_attn_fwd over the same P ranks bit for bit.  workspace: 256-byte aligned,
 * at least ulysses_usp_workspace_bytes(...) bytes (every rank's group head-layout Q, K,
 * V, O).  Five kinds of launches: Pr exchanges in, one attention, Pr exchanges out.
 */
size_t ulysses_usp_workspace_bytes(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype);
uly_status ulysses_usp_attn_fwd(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                int causal,
                                const void* const* q_seq, const void* const* k_seq,
                                const void* const* v_seq, void* const* o_seq,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Training on the two-level layout (the backward of the pipeline above: each exchange's
 * backward is the opposite exchange, "DeepSpeed-Ulysses 深度解析", section "核心设计", and
 * the attention's backward is the ordinary one, "02 · DeepSpeed-Ulysses", section 5).
 *
 * ulysses_usp_attn_fwd_lse: ulysses_usp_attn_fwd that also saves the softmax statistics:
 *   lse: Pu pointers, lse[u] = fp32 [b][h_q/Pu][s], the natural-log log-sum-exp of the
 *   scaled scores of every query row of heads [u*h_q/Pu, (u+1)*h_q/Pu), all s positions
 *   (the rows of every ring group's rank u).  Needs ULY_BF16 (else ULY_ERR_UNSUPPORTED) and
 *   lse non-null, not overlapping any other argument (else ULY_ERR_INVALID_ARG).
 * ulysses_usp_attn_bwd: dQ, dK, dV in the seq layout of the inputs, from Q, K, V, the
 *   forward's O, the gradient dO (all seq layout, P = Pu*Pr pointers each) and the lse of
 *   ulysses_usp_attn_fwd_lse:
 *     1. all-to-all #1 on Q, K, V and dO inside every ring group;
 *     2. the attention backward of every Ulysses unit over the whole sequence, reading and
 *        writing each tile in the buffer of the ring group that holds its tokens;
 *     3. all-to-all #2 on dQ, dK, dV inside every ring group.
 *   Same sizes and kernel limits as ulysses_usp_attn_fwd, bf16 only, and Pu*Pr <= 48 (else
 *   ULY_ERR_UNSUPPORTED).  dq/dk/dv must not
 *   overlap each other or any input.  The results equal ulysses_dist_attn_bwd over the same
 *   P ranks bit for bit where h_kv % P == 0 (with replicated K/V heads the plain call's
 *   dK/dV come from another summation order).  workspace:
 *   256-byte aligned, at least ulysses_usp_bwd_workspace_bytes(...) bytes (every rank's group
 *   head-layout Q, K, V, dO, dQ, dK, dV and, per Ulysses unit, two fp32 row arrays); it
 *   returns 0 for shapes the call rejects.
 */
uly_status ulysses_usp_attn_fwd_lse(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                    int causal, const void* const* q_seq, const void* const* k_seq,
                                    const void* const* v_seq, void* const* o_seq, float* const* lse,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t ulysses_usp_bwd_workspace_bytes(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype);
uly_status ulysses_usp_attn_bwd(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                int causal, const void* const* q_seq, const void* const* k_seq,
                                const void* const* v_seq, const void* const* o_seq, const void* const* do_seq,
                                const float* const* lse, void* const* dq_seq, void* const* dk_seq,
                                void* const* dv_seq, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The unfused forward without any allocation by the caller or the library.  DeepSpeed-Ulysses
 * itself has no such call: this exists for callers that cannot call cudaMalloc -- for example an
 * application whose memory pool already holds all the device memory it may use, or a
 * plugin whose host runtime gives it no allocator on its hot path.
 * Same arguments, layouts, results and errors as ulysses_dist_attn_fwd with fused == 0,
 * except that the workspace is a fixed array of ULYSSES_NOALLOC_SCRATCH_BYTES bytes of
 * device memory inside the library, which every GPU that loads the library holds until
 * the process exits.  Calls needing more scratch than that
 * (ulysses_dist_attn_workspace_bytes(..., fused = 0) > ULYSSES_NOALLOC_SCRATCH_BYTES)
 * return ULY_ERR_INVALID_ARG without enqueuing work.
 * Set-up: the first call in each CUDA context of a device looks up the array's device
 * address (make it before any stream capture begins).  Under CUDA's lazy module loading
 * (the default) that lookup also loads the module holding the array and reserves its
 * memory, so the first call returns ULY_ERR_CUDA if the device has less than
 * ULYSSES_NOALLOC_SCRATCH_BYTES free; make it early.  The address is cached per context,
 * so a cudaDeviceReset (which gives the device a new context and a new array) is handled
 * by a fresh lookup on the next call.
 * Every call shares the array and finds the previous call's contents there; the forward
 * writes each scratch byte before reading it, so nothing needs clearing.  Calls whose work
 * overlaps on the GPU (e.g. on two streams) race on it and must be serialised by the caller.
 * No cudaMalloc, cudaFree or other allocating routine is called, and the library's own code
 * makes no host heap allocation on this path (the CUDA runtime's internal bookkeeping is
 * outside its control).
 */
#define ULYSSES_NOALLOC_SCRATCH_BYTES (64ull << 20)
uly_status ulysses_dist_attn_fwd_noalloc(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                         int causal,
                                         const void* const* q_seq, const void* const* k_seq,
                                         const void* const* v_seq, void* const* o_seq,
                                         cudaStream_t stream);

/*
 * ------------------------------------------------------------------------------------
 * Training: forward with the saved softmax statistics, and the backward.
 *
 * "02 · DeepSpeed-Ulysses", section 5 (backward): the gradient of all-to-all #2 is
 * all-to-all #1 applied to dO, the local attention's gradient is the ordinary attention
 * backward, and the gradient of all-to-all #1 is all-to-all #2 applied to dQ, dK and dV.
 * The attention backward uses, for every query row i of every local head,
 *   L_i = log sum_{visible j} exp(q_i.k_j / sqrt(d))        (natural log, fp32)
 *   P_ij = exp(q_i.k_j / sqrt(d) - L_i),  D_i = sum_c dO_ic O_ic,
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i.v_j - D_i),
 *   dQ_i = sum_j dS_ij k_j / sqrt(d),  dK_j = sum_i dS_ij q_i / sqrt(d)
 * (grouped heads: dK/dV of a K/V head sum over all query heads that read it).
 * lse arrays: P pointers, rank r's is [b][h_q/P][s] fp32 (row (bb, hh, i) = L_i of local
 * head hh, i.e. global head r*h_q/P + hh), 16-byte aligned like every device pointer.
 * Only ULY_BF16 with d in {64, 128} has these kernels (else ULY_ERR_UNSUPPORTED).
 * dP, P and dS are formed in fp32; P and dS are rounded to bf16 before their tile
 * products (as P is in the forward); gradients are accumulated in fp32 and rounded to
 * nearest even at the end.  Each gradient element is written exactly once (no atomics),
 * so repeated calls give the same bits.
 * ------------------------------------------------------------------------------------
 */

/*
 * ulysses_local_attention plus the per-row log-sum-exp: same arguments, layouts and
 * output, and lse[r][bb][hh][i] = L_i as defined above.  lse must not overlap any other
 * argument.
 */
uly_status ulysses_local_attention_fwd_lse(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                           int causal,
                                           const void* const* q_head, const void* const* k_head,
                                           const void* const* v_head, void* const* o_head,
                                           float* const* lse, cudaStream_t stream);

/*
 * ulysses_dist_attn_fwd (same workspace, same fused / unfused rules and bits) plus the
 * log-sum-exp of every head rank's rows: lse[r] is indexed in head layout ([b][h_q/P][s],
 * all s tokens of rank r's heads), which is what ulysses_dist_attn_bwd takes back.
 */
uly_status ulysses_dist_attn_fwd_lse(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                     int causal,
                                     const void* const* q_seq, const void* const* k_seq,
                                     const void* const* v_seq, void* const* o_seq, float* const* lse,
                                     void* workspace, size_t workspace_bytes, int fused,
                                     cudaStream_t stream);

/*
 * Bytes of workspace the backward needs: for every rank two fp32 row arrays
 * [b][h_q/P][ceil(s/128)*128] (L in base 2 and D), and, when dist != 0 and fused == 0,
 * the head-layout copies of Q, K, V, dO, dQ, dK and dV; each array 256-byte aligned.
 * 0 for arguments that are invalid or unsupported.
 */
size_t ulysses_attn_bwd_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                        int dist, int fused);

/*
 * Backward of ulysses_local_attention, head layout in and out.
 *   q_head, o_head, do_head, dq_head: P pointers to [b][s][h_q/P][d];
 *   k_head, v_head, dk_head, dv_head: P pointers to [b][s][Hk][d] (Hk as in
 *   ulysses_local_attention; with replicated K/V heads dk_head / dv_head hold each
 *   rank's share only, the gradient of its own query heads);
 *   lse: from ulysses_local_attention_fwd_lse on the same q, k (and causal flag).
 * Four launches: row statistics, dK/dV, dQ (one pair per 16 ranks).  Outputs must not
 * overlap each other, any input or the workspace (256-byte aligned, at least
 * ulysses_attn_bwd_workspace_bytes(..., dist = 0, fused = 0) bytes, owned by the caller).
 */
uly_status ulysses_local_attention_bwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                       int causal,
                                       const void* const* q_head, const void* const* k_head,
                                       const void* const* v_head, const void* const* o_head,
                                       const void* const* do_head, const float* const* lse,
                                       void* const* dq_head, void* const* dk_head, void* const* dv_head,
                                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The whole DistributedAttention backward, seq layout in and out.
 * fused == 0: all-to-all #1 on Q, K, V and dO (one launch), D from the seq-layout O and
 *   dO, the local backward of every rank, all-to-all #2 on dQ, dK and dV (one launch).
 * fused != 0: D and the statistics, then the dK/dV and dQ kernels read their Q/K/V/dO
 *   tiles straight from the seq-layout buffers and write dQ/dK/dV rows straight into the
 *   seq-layout outputs, so no head-layout copy exists (the backward of the fused
 *   forward).  Needs P <= 48 and (s/P) % 128 == 0, else ULY_ERR_UNSUPPORTED.  Both paths
 *   give the same bits where h_kv % P == 0 (for replicated K/V heads, see below).
 *   q_seq, o_seq, do_seq, dq_seq: P pointers to [b][s/P][h_q][d];
 *   k_seq, v_seq, dk_seq, dv_seq: P pointers to [b][s/P][h_kv][d];
 *   lse: from ulysses_dist_attn_fwd_lse (head-layout indexed).
 * Replicated K/V heads (P % h_kv == 0, h_kv < P): dK and dV of head h are the sum of
 *   the shares of its rep ranks.  fused == 0 writes the shares in fp32 and adds them in
 *   a fixed order before one rounding to bf16 (the reverse of the broadcast); fused != 0
 *   needs no sum, since its dK/dV kernel owns every global K/V head and reads all of that
 *   head's query heads.  The two orders of summation round differently, so there dK and
 *   dV of the two paths may differ in the last bits (dQ and the forward do not).
 * workspace: 256-byte aligned, at least ulysses_attn_bwd_workspace_bytes(..., dist = 1,
 * fused) bytes.  Size and overlap rules as ulysses_local_attention_bwd plus the exchange rules.
 */
uly_status ulysses_dist_attn_bwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                 const void* const* q_seq, const void* const* k_seq,
                                 const void* const* v_seq, const void* const* o_seq,
                                 const void* const* do_seq, const float* const* lse,
                                 void* const* dq_seq, void* const* dk_seq, void* const* dv_seq,
                                 void* workspace, size_t workspace_bytes, int fused, cudaStream_t stream);

/*
 * Self-test of the failure path: enqueues one CTA that waits, with the same bounded wait the
 * kernels use, on a barrier that nothing completes; after limit_ns nanoseconds
 * (1e3 .. 1e10, else ULY_ERR_INVALID_ARG) it gives up, sets the timeout bit of the device
 * error word and returns, leaving the context usable.  ulysses_device_status then reports
 * ULY_ERR_TIMEOUT.  Until that status is read with clear != 0, every kernel of this library
 * that starts sees the error word and exits at once.
 */
uly_status ulysses_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

/*
 * Reads (and, if clear != 0, resets) the library's device-side error word after
 * synchronising the current device.  Returns ULY_ERR_TIMEOUT if a kernel's bounded wait
 * gave up since the last reset (that kernel then wrote no output), ULY_ERR_CUDA if the
 * device could not be queried, ULY_OK otherwise.
 */
uly_status ulysses_device_status(int clear);

/* Static, human-readable name of a status code. */
const char* ulysses_status_string(uly_status status);

#ifdef __cplusplus
}
#endif
#endif /* ULYSSES_GB300_H */
