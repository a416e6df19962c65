// C ABI of the Ulysses forward (declared in include/ulysses.h): argument validation, the
// composition of the three stages, and dispatch to the kernels.  Nothing here allocates
// device memory, and nothing allocates on the host heap either: argument records live on
// the stack and the overlap checks use fixed-capacity range sets.  Every argument error is
// reported before any work is enqueued.
#include <cstdint>
#include <cstring>
#include <initializer_list>

#include "../../include/ulysses.h"
#include "internal.h"

namespace {

using uly::kMaxRanks;

constexpr uint64_t kMaxSlabVecs = (1ull << 31) - 1;  // 32-bit index space of the permute kernel
constexpr int kMaxChunks = 64;                        // head groups of the overlapped forward

int elem_bytes(uly_dtype dt) { return dt == ULY_FP32 ? 4 : (dt == ULY_BF16 ? 2 : 0); }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

// A fixed-capacity set of byte ranges (at most six per-rank buffer lists of kMaxRanks).
struct RangeSet {
    static constexpr int kCap = 6 * kMaxRanks;
    Range v[kCap];
    int n = 0;
    bool push(Range r) {
        if (n >= kCap) return false;
        v[n++] = r;
        return true;
    }
    bool append(const RangeSet& o) {
        for (int i = 0; i < o.n; ++i)
            if (!push(o.v[i])) return false;
        return true;
    }
};

RangeSet one_range(const void* p, uint64_t bytes) {
    RangeSet r;
    r.push({reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + (uintptr_t)bytes});
    return r;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Non-null, 16-byte aligned pointers; collects their byte ranges.
bool collect(const void* const* ptrs, int P, uint64_t bytes, RangeSet& out) {
    if (!ptrs) return false;
    for (int i = 0; i < P; ++i) {
        if (!ptrs[i] || !aligned16(ptrs[i])) return false;
        const uintptr_t lo = reinterpret_cast<uintptr_t>(ptrs[i]);
        if (!out.push({lo, lo + (uintptr_t)bytes})) return false;
    }
    return true;
}

bool overlaps(const RangeSet& a, const RangeSet& b) {
    for (int i = 0; i < a.n; ++i)
        for (int k = 0; k < b.n; ++k) {
            const Range& x = a.v[i];
            const Range& y = b.v[k];
            if (x.lo < y.hi && y.lo < x.hi && x.hi > x.lo && y.hi > y.lo) return true;
        }
    return false;
}

bool self_overlap(const RangeSet& a) {
    for (int i = 0; i < a.n; ++i)
        for (int k = i + 1; k < a.n; ++k)
            if (a.v[i].lo < a.v[k].hi && a.v[k].lo < a.v[i].hi && a.v[i].hi > a.v[i].lo && a.v[k].hi > a.v[k].lo)
                return true;
    return false;
}

// Shape rules shared by the exchanges: 1 <= P <= 64, positive sizes, s % P, h % P, and
// index ranges the kernels can address.
uly_status check_exchange_shape(int P, int b, int s, int h, int d, uly_dtype dt) {
    if (P < 1 || P > kMaxRanks || b < 1 || s < 1 || h < 1 || d < 1) return ULY_ERR_INVALID_ARG;
    if (s % P || h % P) return ULY_ERR_INVALID_ARG;
    const int e = elem_bytes(dt);
    if (!e) return ULY_ERR_INVALID_ARG;
    const uint64_t run = (uint64_t)(h / P) * d * e;
    if ((uint64_t)(s / P) * run > kMaxSlabVecs) return ULY_ERR_INVALID_ARG;  // even at 1-byte vectors
    if ((uint64_t)P * P * b > (1ull << 31)) return ULY_ERR_INVALID_ARG;
    return ULY_OK;
}

// The K/V exchange of the attention pipeline: split (P | h_kv) or replicated (h_kv | P, one
// head per rank).
uly_status check_kv_exchange_shape(int P, int b, int s, int h_kv, int d, uly_dtype dt) {
    if (h_kv < 1 || h_kv >= P || P % h_kv) return check_exchange_shape(P, b, s, h_kv, d, dt);
    return check_exchange_shape(P, b, s, P, d, dt);  // one head per rank, like P heads split P ways
}

// K/V heads either split over the ranks (P | h_kv) or, with fewer K/V heads than ranks,
// replicated on P / h_kv ranks each (h_kv | P): the head counts must be multiples of one
// another ("DeepSpeed-Ulysses 深度解析", API section, num_kv_heads; "02 · DeepSpeed-Ulysses",
// section 3: replicating K/V lifts the divisibility limit at a cost in memory and traffic).
uly_status check_kv_exchange_shape(int P, int b, int s, int h_kv, int d, uly_dtype dt);

uly_status check_attention_shape(int P, int b, int s, int hq, int hkv, int d, uly_dtype dt) {
    if (P < 1 || P > kMaxRanks || b < 1 || s < 1 || hq < 1 || hkv < 1 || d < 1) return ULY_ERR_INVALID_ARG;
    if (hq % P || hq % hkv || (hkv % P && P % hkv)) return ULY_ERR_INVALID_ARG;
    if (!elem_bytes(dt)) return ULY_ERR_INVALID_ARG;
    if ((long long)b * P > 65535 || hq / P > 65535) return ULY_ERR_INVALID_ARG;
    if ((long long)b * hq * ((s + 127) / 128) > 0x7fffffffLL) return ULY_ERR_INVALID_ARG;
    if (dt == ULY_FP32 && (d % 4 != 0 || d > 256)) return ULY_ERR_UNSUPPORTED;
    if (dt == ULY_BF16 && !uly::tc_attention_supported(d)) return ULY_ERR_UNSUPPORTED;
    return ULY_OK;
}

uint64_t round256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

// The backward and the log-sum-exp forward exist for the bf16 tensor-core path only.
uly_status check_train_shape(int P, int b, int s, int hq, int hkv, int d, uly_dtype dt) {
    uly_status st = check_attention_shape(P, b, s, hq, hkv, d, dt);
    if (st != ULY_OK) return st;
    if (dt != ULY_BF16) return ULY_ERR_UNSUPPORTED;
    return ULY_OK;
}

// Per-rank bytes of one [b][h_q/P][s_pad] fp32 row array (s_pad = s rounded up to 128).
uint64_t row_array_bytes(int P, int b, int s, int hq) {
    return round256((uint64_t)b * (hq / P) * (((uint64_t)s + 127) / 128 * 128) * 4);
}

bool collect_f(const float* const* ptrs, int P, uint64_t bytes, RangeSet& out) {
    return collect(reinterpret_cast<const void* const*>(ptrs), P, bytes, out);
}

bool workspace_ok(const void* ws, size_t have, size_t need) {
    return ws && !(reinterpret_cast<uintptr_t>(ws) & 255u) && have >= need;
}

uly_status exchange(int direction, int P, int b, int s, int h, int d, uly_dtype dt, const void* const* in,
                    void* const* out, cudaStream_t stream) {
    uly_status st = check_exchange_shape(P, b, s, h, d, dt);
    if (st != ULY_OK) return st;
    const uint64_t bytes = (uint64_t)b * (s / P) * h * d * elem_bytes(dt);  // equal on both sides
    RangeSet ri, ro;
    if (!collect(in, P, bytes, ri) || !collect(reinterpret_cast<const void* const*>(out), P, bytes, ro))
        return ULY_ERR_INVALID_ARG;
    if (overlaps(ri, ro) || self_overlap(ro)) return ULY_ERR_INVALID_ARG;
    uly::PermuteTensor t;
    memset(&t, 0, sizeof(t));
    for (int r = 0; r < P; ++r) {
        t.src[r] = in[r];
        t.dst[r] = out[r];
    }
    t.h = h;
    return uly::launch_permute(direction, P, b, s, d, elem_bytes(dt), &t, 1, stream) == cudaSuccess ? ULY_OK
                                                                                                  : ULY_ERR_CUDA;
}

uly_status run_attention(int P, int b, int s, int hq, int hkv, int d, uly_dtype dt, int causal, int fused,
                         const uly::AttnPtrs& ptrs, cudaStream_t stream) {
    if (dt == ULY_FP32) {
        if (fused || ptrs.lse[0]) return ULY_ERR_UNSUPPORTED;
        return uly::launch_attention_fp32(P, b, s, hq, hkv, d, causal, ptrs, stream) == cudaSuccess ? ULY_OK
                                                                                                    : ULY_ERR_CUDA;
    }
    int unsupported = 0;
    cudaError_t e = uly::launch_attention_tc(P, b, s, hq, hkv, d, causal, fused, ptrs, stream, &unsupported);
    if (unsupported) return ULY_ERR_UNSUPPORTED;
    return e == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

// Head-layout attention of every rank; lse (optional, bf16 path only) receives the
// per-row log-sum-exp.
uly_status local_attention(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                           const void* const* q_head, const void* const* k_head, const void* const* v_head,
                           void* const* o_head, float* const* lse, cudaStream_t stream) {
    uly_status st = check_attention_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    const int e = elem_bytes(dtype);
    const uint64_t qb = (uint64_t)b * s * (h_q / P) * d * e,
                   kb = (uint64_t)b * s * uly::kv_heads_per_rank(P, h_kv) * d * e;
    RangeSet rq, rk, rv, ro, rl;
    if (!collect(q_head, P, qb, rq) || !collect(k_head, P, kb, rk) || !collect(v_head, P, kb, rv) ||
        !collect(reinterpret_cast<const void* const*>(o_head), P, qb, ro))
        return ULY_ERR_INVALID_ARG;
    if (overlaps(ro, rq) || overlaps(ro, rk) || overlaps(ro, rv) || self_overlap(ro)) return ULY_ERR_INVALID_ARG;
    if (lse) {
        if (!collect_f(lse, P, (uint64_t)b * (h_q / P) * s * 4, rl)) return ULY_ERR_INVALID_ARG;
        if (self_overlap(rl) || overlaps(rl, rq) || overlaps(rl, rk) || overlaps(rl, rv) || overlaps(rl, ro))
            return ULY_ERR_INVALID_ARG;
    }
    uly::AttnPtrs ptrs;
    memset(&ptrs, 0, sizeof(ptrs));
    for (int r = 0; r < P; ++r) {
        ptrs.q[r] = q_head[r];
        ptrs.k[r] = k_head[r];
        ptrs.v[r] = v_head[r];
        ptrs.o[r] = o_head[r];
        ptrs.lse[r] = lse ? lse[r] : nullptr;
    }
    return run_attention(P, b, s, h_q, h_kv, d, dtype, causal, 0, ptrs, stream);
}

// Pointers of one head-layout scratch set inside a workspace: per rank, in this order,
// the arrays whose per-rank sizes are listed in `sizes` (each 256-byte aligned).
struct SizeList {
    static constexpr int kCap = 16;
    uint64_t v[kCap];
    int n = 0;
    SizeList() = default;
    SizeList(std::initializer_list<uint64_t> xs) {
        for (uint64_t x : xs) push(x);
    }
    void push(uint64_t x) {
        if (n < kCap) v[n++] = x;
    }
};

struct Carve {
    uint8_t* base;
    uint64_t per_rank;
    uint64_t offs[SizeList::kCap];
    Carve(void* ws, const SizeList& sizes) : base(static_cast<uint8_t*>(ws)), per_rank(0) {
        for (int i = 0; i < sizes.n; ++i) {
            offs[i] = per_rank;
            per_rank += round256(sizes.v[i]);
        }
    }
    void* at(int r, int k) const { return base + (uint64_t)r * per_rank + offs[k]; }
};

// Workspace of the backward: per rank the two fp32 row arrays (lse2, D), and for the
// unfused distributed backward the head-layout Q, K, V, dO, dQ, dK, dV.
SizeList bwd_sizes(int P, int b, int s, int hq, int hkv, int d, int dist) {
    const uint64_t ra = row_array_bytes(P, b, s, hq);
    SizeList v{ra, ra};
    if (dist == 1) {
        const uint64_t qb = (uint64_t)b * s * (hq / P) * d * 2,
                       kb = (uint64_t)b * s * uly::kv_heads_per_rank(P, hkv) * d * 2;
        // replicated K/V heads: each rank's dK/dV is an fp32 partial sum
        const uint64_t gb = uly::kv_replication(P, hkv) > 1 ? 2 * kb : kb;
        for (uint64_t x : {qb, kb, kb, qb, qb, gb, gb}) v.push(x);
    }
    return v;
}

uly_status run_backward(int P, int b, int s, int hq, int hkv, int d, int causal, int fused,
                        const uly::BwdPtrs& ptrs, cudaStream_t stream) {
    int unsupported = 0;
    cudaError_t e = uly::launch_attention_bwd_tc(P, b, s, hq, hkv, d, causal, fused, ptrs, stream, &unsupported);
    if (unsupported) return ULY_ERR_UNSUPPORTED;
    return e == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

size_t dist_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int fused) {
    if (check_attention_shape(P, b, s, h_q, h_kv, d, dtype) == ULY_ERR_INVALID_ARG) return 0;
    if (s % P) return 0;
    if (fused) return 0;
    const int e = elem_bytes(dtype);
    const uint64_t qb = round256((uint64_t)b * s * (h_q / P) * d * e);
    const uint64_t kb = round256((uint64_t)b * s * uly::kv_heads_per_rank(P, h_kv) * d * e);
    return (size_t)((uint64_t)P * (2 * qb + 2 * kb));
}

// The forward pipeline; lse (optional) receives the per-row log-sum-exp of every rank.
uly_status dist_attn_fwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                         const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                         void* const* o_seq, float* const* lse, void* workspace, size_t workspace_bytes, int fused,
                         cudaStream_t stream) {
    uly_status st = check_attention_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    st = check_exchange_shape(P, b, s, h_q, d, dtype);
    if (st != ULY_OK) return st;
    st = check_kv_exchange_shape(P, b, s, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    const int e = elem_bytes(dtype);
    const int S = s / P;
    const uint64_t qsb = (uint64_t)b * S * h_q * d * e, ksb = (uint64_t)b * S * h_kv * d * e;
    RangeSet rq, rk, rv, ro;
    if (!collect(q_seq, P, qsb, rq) || !collect(k_seq, P, ksb, rk) || !collect(v_seq, P, ksb, rv) ||
        !collect(reinterpret_cast<const void* const*>(o_seq), P, qsb, ro))
        return ULY_ERR_INVALID_ARG;
    if (overlaps(ro, rq) || overlaps(ro, rk) || overlaps(ro, rv) || self_overlap(ro)) return ULY_ERR_INVALID_ARG;
    RangeSet rl;
    if (lse) {
        if (!collect_f(lse, P, (uint64_t)b * (h_q / P) * s * 4, rl)) return ULY_ERR_INVALID_ARG;
        if (self_overlap(rl) || overlaps(rl, rq) || overlaps(rl, rk) || overlaps(rl, rv) || overlaps(rl, ro))
            return ULY_ERR_INVALID_ARG;
    }

    if (fused) {
        if (dtype != ULY_BF16) return ULY_ERR_UNSUPPORTED;
        uly::AttnPtrs ptrs;
        memset(&ptrs, 0, sizeof(ptrs));
        for (int r = 0; r < P; ++r) {
            ptrs.q[r] = q_seq[r];
            ptrs.k[r] = k_seq[r];
            ptrs.v[r] = v_seq[r];
            ptrs.o[r] = o_seq[r];
            ptrs.lse[r] = lse ? lse[r] : nullptr;
        }
        return run_attention(P, b, s, h_q, h_kv, d, dtype, causal, 1, ptrs, stream);
    }

    const size_t need = dist_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, 0);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return ULY_ERR_INVALID_ARG;
    const RangeSet rw = one_range(workspace, need);
    if (overlaps(rw, rq) || overlaps(rw, rk) || overlaps(rw, rv) || overlaps(rw, ro) || overlaps(rw, rl))
        return ULY_ERR_INVALID_ARG;

    // workspace: per rank [Q_head | K_head | V_head | O_head], each 256-byte aligned
    const uint64_t qhb = round256((uint64_t)b * s * (h_q / P) * d * e);
    const uint64_t khb = round256((uint64_t)b * s * uly::kv_heads_per_rank(P, h_kv) * d * e);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uly::AttnPtrs head;
    memset(&head, 0, sizeof(head));
    for (int r = 0; r < P; ++r) {
        uint8_t* base = ws + (uint64_t)r * (2 * qhb + 2 * khb);
        head.q[r] = base;
        head.k[r] = base + qhb;
        head.v[r] = base + qhb + khb;
        head.o[r] = base + qhb + 2 * khb;
        head.lse[r] = lse ? lse[r] : nullptr;
    }
    // (1) all-to-all #1 for Q, K and V in one launch
    uly::PermuteTensor t[3];
    memset(t, 0, sizeof(t));
    for (int r = 0; r < P; ++r) {
        t[0].src[r] = q_seq[r];
        t[0].dst[r] = const_cast<void*>(head.q[r]);
        t[1].src[r] = k_seq[r];
        t[1].dst[r] = const_cast<void*>(head.k[r]);
        t[2].src[r] = v_seq[r];
        t[2].dst[r] = const_cast<void*>(head.v[r]);
    }
    t[0].h = h_q;
    t[1].h = h_kv;
    t[2].h = h_kv;
    t[1].rep = t[2].rep = uly::kv_replication(P, h_kv);  // fewer K/V heads than ranks: copies
    if (uly::launch_permute(0, P, b, s, d, e, t, 3, stream) != cudaSuccess) return ULY_ERR_CUDA;
    // (2) local attention of every rank
    st = run_attention(P, b, s, h_q, h_kv, d, dtype, causal, 0, head, stream);
    if (st != ULY_OK) return st;
    // (3) all-to-all #2 for the output
    uly::PermuteTensor to;
    memset(&to, 0, sizeof(to));
    for (int r = 0; r < P; ++r) {
        to.src[r] = head.o[r];
        to.dst[r] = o_seq[r];
    }
    to.h = h_q;
    return uly::launch_permute(1, P, b, s, d, e, &to, 1, stream) == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

}  // namespace

extern "C" {

uly_status ulysses_a2a_seq2head(int P, int b, int s, int h, int d, uly_dtype dtype, const void* const* in_seq,
                                void* const* out_head, cudaStream_t stream) {
    return exchange(0, P, b, s, h, d, dtype, in_seq, out_head, stream);
}

uly_status ulysses_a2a_head2seq(int P, int b, int s, int h, int d, uly_dtype dtype, const void* const* in_head,
                                void* const* out_seq, cudaStream_t stream) {
    return exchange(1, P, b, s, h, d, dtype, in_head, out_seq, stream);
}

// The local halves of one rank's exchange with other GPUs: the send blocks before the
// collective and the layout after it, each one block transpose.
static uly_status a2a_local(int pack, int direction, int P, int b, int s, int h, int d, uly_dtype dtype,
                            const void* in, void* out, cudaStream_t stream) {
    uly_status st = check_exchange_shape(P, b, s, h, d, dtype);
    if (st != ULY_OK) return st;
    if (direction != 0 && direction != 1) return ULY_ERR_INVALID_ARG;
    const uint64_t e = (uint64_t)elem_bytes(dtype), S = (uint64_t)(s / P), H = (uint64_t)(h / P);
    const uint64_t bytes = (uint64_t)b * S * h * d * e;  // one rank's share, on either side
    RangeSet ri, ro;
    if (!collect(&in, 1, bytes, ri) || !collect(const_cast<const void* const*>(&out), 1, bytes, ro) || overlaps(ri, ro))
        return ULY_ERR_INVALID_ARG;
    const uint64_t head_run = H * d * e, block_run = S * H * d * e;
    uint64_t A, C, run;
    if (direction == 0 && pack) {         // seq shard [b*S][P][H*d] -> blocks [P][b*S][H*d]
        A = (uint64_t)b * S, C = P, run = head_run;
    } else if (direction == 0) {          // received blocks [P][b][S*H*d] -> head shard [b][P][S*H*d]
        A = P, C = b, run = block_run;
    } else if (pack) {                    // head shard [b][P][S*H*d] -> blocks [P][b][S*H*d]
        A = b, C = P, run = block_run;
    } else {                              // received blocks [P][b*S][H*d] -> seq shard [b*S][P][H*d]
        A = P, C = (uint64_t)b * S, run = head_run;
    }
    if (!uly::block_transpose_fits(A, C, run, in, out)) return ULY_ERR_INVALID_ARG;
    return uly::launch_block_transpose(A, C, run, in, out, stream) == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

uly_status ulysses_a2a_pack(int direction, int P, int b, int s, int h, int d, uly_dtype dtype, const void* local,
                            void* send, cudaStream_t stream) {
    return a2a_local(1, direction, P, b, s, h, d, dtype, local, send, stream);
}

uly_status ulysses_a2a_unpack(int direction, int P, int b, int s, int h, int d, uly_dtype dtype, const void* recv,
                              void* local, cudaStream_t stream) {
    return a2a_local(0, direction, P, b, s, h, d, dtype, recv, local, stream);
}

uly_status ulysses_local_attention(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                   const void* const* q_head, const void* const* k_head, const void* const* v_head,
                                   void* const* o_head, cudaStream_t stream) {
    return local_attention(P, b, s, h_q, h_kv, d, dtype, causal, q_head, k_head, v_head, o_head, nullptr, stream);
}

uly_status ulysses_local_attention_fwd_lse(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                           int causal, const void* const* q_head, const void* const* k_head,
                                           const void* const* v_head, void* const* o_head, float* const* lse,
                                           cudaStream_t stream) {
    uly_status st = check_train_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    if (!lse) return ULY_ERR_INVALID_ARG;
    return local_attention(P, b, s, h_q, h_kv, d, dtype, causal, q_head, k_head, v_head, o_head, lse, stream);
}

size_t ulysses_dist_attn_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int fused) {
    return dist_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, fused);
}

uly_status ulysses_dist_attn_fwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                 const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                                 void* const* o_seq, void* workspace, size_t workspace_bytes, int fused,
                                 cudaStream_t stream) {
    return dist_attn_fwd(P, b, s, h_q, h_kv, d, dtype, causal, q_seq, k_seq, v_seq, o_seq, nullptr, workspace,
                         workspace_bytes, fused, stream);
}

uly_status ulysses_dist_attn_fwd_lse(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                     const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                                     void* const* o_seq, float* const* lse, void* workspace, size_t workspace_bytes,
                                     int fused, cudaStream_t stream) {
    uly_status st = check_train_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    if (!lse) return ULY_ERR_INVALID_ARG;
    return dist_attn_fwd(P, b, s, h_q, h_kv, d, dtype, causal, q_seq, k_seq, v_seq, o_seq, lse, workspace,
                         workspace_bytes, fused, stream);
}

size_t ulysses_attn_bwd_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int dist,
                                        int fused) {
    if (check_train_shape(P, b, s, h_q, h_kv, d, dtype) != ULY_OK) return 0;
    if (dist && (check_exchange_shape(P, b, s, h_q, d, dtype) != ULY_OK ||
                 check_kv_exchange_shape(P, b, s, h_kv, d, dtype) != ULY_OK))
        return 0;
    uint64_t per_rank = 0;
    const SizeList sizes = bwd_sizes(P, b, s, h_q, h_kv, d, dist && !fused ? 1 : 0);
    for (int i = 0; i < sizes.n; ++i) per_rank += round256(sizes.v[i]);
    return (size_t)(per_rank * P);
}

uly_status ulysses_local_attention_bwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                       const void* const* q_head, const void* const* k_head,
                                       const void* const* v_head, const void* const* o_head,
                                       const void* const* do_head, const float* const* lse, void* const* dq_head,
                                       void* const* dk_head, void* const* dv_head, void* workspace,
                                       size_t workspace_bytes, cudaStream_t stream) {
    uly_status st = check_train_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    const uint64_t qb = (uint64_t)b * s * (h_q / P) * d * 2,
                   kb = (uint64_t)b * s * uly::kv_heads_per_rank(P, h_kv) * d * 2;
    RangeSet in, rdq, rdk, rdv;
    if (!collect(q_head, P, qb, in) || !collect(k_head, P, kb, in) || !collect(v_head, P, kb, in) ||
        !collect(o_head, P, qb, in) || !collect(do_head, P, qb, in) ||
        !collect_f(lse, P, (uint64_t)b * (h_q / P) * s * 4, in) ||
        !collect(reinterpret_cast<const void* const*>(dq_head), P, qb, rdq) ||
        !collect(reinterpret_cast<const void* const*>(dk_head), P, kb, rdk) ||
        !collect(reinterpret_cast<const void* const*>(dv_head), P, kb, rdv))
        return ULY_ERR_INVALID_ARG;
    RangeSet outs;
    if (!outs.append(rdq) || !outs.append(rdk) || !outs.append(rdv)) return ULY_ERR_INVALID_ARG;
    if (self_overlap(outs) || overlaps(outs, in)) return ULY_ERR_INVALID_ARG;
    const size_t need = ulysses_attn_bwd_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, 0, 0);
    if (!workspace_ok(workspace, workspace_bytes, need)) return ULY_ERR_INVALID_ARG;
    const RangeSet rw = one_range(workspace, need);
    if (overlaps(rw, in) || overlaps(rw, outs)) return ULY_ERR_INVALID_ARG;
    const Carve ws(workspace, bwd_sizes(P, b, s, h_q, h_kv, d, 0));
    uly::BwdPtrs p_rec;
    uly::BwdPtrs* p = &p_rec;
    memset(p, 0, sizeof(uly::BwdPtrs));
    for (int r = 0; r < P; ++r) {
        p->q[r] = q_head[r];
        p->k[r] = k_head[r];
        p->v[r] = v_head[r];
        p->dout[r] = do_head[r];
        p->o_rows[r] = o_head[r];
        p->do_rows[r] = do_head[r];
        p->lse[r] = lse[r];
        p->dq[r] = dq_head[r];
        p->dk[r] = dk_head[r];
        p->dv[r] = dv_head[r];
        p->lse2[r] = static_cast<float*>(ws.at(r, 0));
        p->dsum[r] = static_cast<float*>(ws.at(r, 1));
    }
    p->od_seq_layout = 0;
    st = run_backward(P, b, s, h_q, h_kv, d, causal, 0, *p, stream);
    return st;
}

uly_status ulysses_dist_attn_bwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                 const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                                 const void* const* o_seq, const void* const* do_seq, const float* const* lse,
                                 void* const* dq_seq, void* const* dk_seq, void* const* dv_seq, void* workspace,
                                 size_t workspace_bytes, int fused, cudaStream_t stream) {
    uly_status st = check_train_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    st = check_exchange_shape(P, b, s, h_q, d, dtype);
    if (st != ULY_OK) return st;
    st = check_kv_exchange_shape(P, b, s, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    const int S = s / P;
    const uint64_t qsb = (uint64_t)b * S * h_q * d * 2, ksb = (uint64_t)b * S * h_kv * d * 2;
    RangeSet in, rdq, rdk, rdv;
    if (!collect(q_seq, P, qsb, in) || !collect(k_seq, P, ksb, in) || !collect(v_seq, P, ksb, in) ||
        !collect(o_seq, P, qsb, in) || !collect(do_seq, P, qsb, in) ||
        !collect_f(lse, P, (uint64_t)b * (h_q / P) * s * 4, in) ||
        !collect(reinterpret_cast<const void* const*>(dq_seq), P, qsb, rdq) ||
        !collect(reinterpret_cast<const void* const*>(dk_seq), P, ksb, rdk) ||
        !collect(reinterpret_cast<const void* const*>(dv_seq), P, ksb, rdv))
        return ULY_ERR_INVALID_ARG;
    RangeSet outs;
    if (!outs.append(rdq) || !outs.append(rdk) || !outs.append(rdv)) return ULY_ERR_INVALID_ARG;
    if (self_overlap(outs) || overlaps(outs, in)) return ULY_ERR_INVALID_ARG;
    if (fused && (P > 48 || S % 128 != 0)) return ULY_ERR_UNSUPPORTED;
    const size_t need = ulysses_attn_bwd_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, 1, fused);
    if (!workspace_ok(workspace, workspace_bytes, need)) return ULY_ERR_INVALID_ARG;
    const RangeSet rw = one_range(workspace, need);
    if (overlaps(rw, in) || overlaps(rw, outs)) return ULY_ERR_INVALID_ARG;
    if (fused) {
        // one launch chain: statistics, then the two kernels read Q/K/V/dO from the seq-layout
        // buffers and write dQ/dK/dV into them through their tile addressing
        const Carve ws(workspace, bwd_sizes(P, b, s, h_q, h_kv, d, 0));
        uly::BwdPtrs p_rec;
    uly::BwdPtrs* p = &p_rec;
        memset(p, 0, sizeof(uly::BwdPtrs));
        for (int r = 0; r < P; ++r) {
            p->q[r] = q_seq[r];
            p->k[r] = k_seq[r];
            p->v[r] = v_seq[r];
            p->dout[r] = do_seq[r];
            p->o_rows[r] = o_seq[r];
            p->do_rows[r] = do_seq[r];
            p->lse[r] = lse[r];
            p->dq[r] = dq_seq[r];
            p->dk[r] = dk_seq[r];
            p->dv[r] = dv_seq[r];
            p->lse2[r] = static_cast<float*>(ws.at(r, 0));
            p->dsum[r] = static_cast<float*>(ws.at(r, 1));
        }
        p->od_seq_layout = 1;
        st = run_backward(P, b, s, h_q, h_kv, d, causal, 1, *p, stream);
        return st;
    }
    const Carve ws(workspace, bwd_sizes(P, b, s, h_q, h_kv, d, 1));
    enum { LSE2, DSUM, QH, KH, VH, DOH, DQH, DKH, DVH };
    // (1) all-to-all #1 on Q, K, V and dO (the backward of all-to-all #2 is all-to-all #1)
    uly::PermuteTensor t_rec[4];
    uly::PermuteTensor* t = t_rec;
    memset(t, 0, 4 * sizeof(uly::PermuteTensor));
    const void* const* srcs[4] = {q_seq, k_seq, v_seq, do_seq};
    const int dsts[4] = {QH, KH, VH, DOH};
    for (int k = 0; k < 4; ++k) {
        for (int r = 0; r < P; ++r) {
            t[k].src[r] = srcs[k][r];
            t[k].dst[r] = ws.at(r, dsts[k]);
        }
        t[k].h = (k == 1 || k == 2) ? h_kv : h_q;
        if (k == 1 || k == 2) t[k].rep = uly::kv_replication(P, h_kv);
    }
    cudaError_t ce = uly::launch_permute(0, P, b, s, d, 2, t, 4, stream);
    if (ce != cudaSuccess) return ULY_ERR_CUDA;
    // (2) local backward of every rank; D straight from the seq-layout O and dO
    uly::BwdPtrs p_rec;
    uly::BwdPtrs* p = &p_rec;
    memset(p, 0, sizeof(uly::BwdPtrs));
    for (int r = 0; r < P; ++r) {
        p->q[r] = ws.at(r, QH);
        p->k[r] = ws.at(r, KH);
        p->v[r] = ws.at(r, VH);
        p->dout[r] = ws.at(r, DOH);
        p->o_rows[r] = o_seq[r];
        p->do_rows[r] = do_seq[r];
        p->lse[r] = lse[r];
        p->dq[r] = ws.at(r, DQH);
        p->dk[r] = ws.at(r, DKH);
        p->dv[r] = ws.at(r, DVH);
        p->lse2[r] = static_cast<float*>(ws.at(r, LSE2));
        p->dsum[r] = static_cast<float*>(ws.at(r, DSUM));
    }
    p->od_seq_layout = 1;
    p->kv_grad_f32 = uly::kv_replication(P, h_kv) > 1 ? 1 : 0;
    st = run_backward(P, b, s, h_q, h_kv, d, causal, 0, *p, stream);
    if (st != ULY_OK) return st;
    // (3) all-to-all #2 on dQ, dK, dV (the backward of all-to-all #1).  Replicated K/V heads:
    //     every replica holds the gradient from its own query heads, and the backward of the
    //     copy is their sum
    const int kv_rep = uly::kv_replication(P, h_kv);
    const int n_plain = kv_rep > 1 ? 1 : 3;
    memset(t, 0, 3 * sizeof(uly::PermuteTensor));
    void* const* dsts2[3] = {dq_seq, dk_seq, dv_seq};
    const int srcs2[3] = {DQH, DKH, DVH};
    for (int k = 0; k < 3; ++k) {
        for (int r = 0; r < P; ++r) {
            t[k].src[r] = ws.at(r, srcs2[k]);
            t[k].dst[r] = dsts2[k][r];
        }
        t[k].h = k == 0 ? h_q : h_kv;
    }
    ce = uly::launch_permute(1, P, b, s, d, 2, t, n_plain, stream);
    for (int k = 1; k < 3 && kv_rep > 1 && ce == cudaSuccess; ++k)
        ce = uly::launch_kv_grad_sum(P, kv_rep, b, s, h_kv, d, t[k].src, t[k].dst, stream);
    return ce == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

// Head groups of the overlapped forward.  Chunk c holds local query heads
// [c*Hc, (c+1)*Hc).  When n_chunks divides the local K/V heads, chunk c has its own K/V
// heads [c*Hkc, (c+1)*Hkc).  When n_chunks is a multiple of them instead (grouped heads with
// few K/V heads per rank), n_chunks/Hk consecutive chunks share one K/V head, exchanged
// with the first of them.
struct OverlapPlan {
    int nc, Hc, Hkc, kv_groups, chunks_per_kv;
    bool valid;
    int kv_of(int c) const { return c / chunks_per_kv; }
    bool new_kv(int c) const { return c % chunks_per_kv == 0; }
};

OverlapPlan overlap_plan(int P, int h_q, int h_kv, int n_chunks) {
    OverlapPlan pl{n_chunks, 0, 0, 0, 1, false};
    // replicated K/V heads (P a multiple of h_kv): one K/V head per rank, shared by every chunk
    const int Hq = h_q / P, Hk = uly::kv_heads_per_rank(P, h_kv);
    if (n_chunks < 1 || n_chunks > kMaxChunks || Hq % n_chunks) return pl;
    pl.Hc = Hq / n_chunks;
    if (Hk % n_chunks == 0) {
        pl.Hkc = Hk / n_chunks;
        pl.kv_groups = n_chunks;
    } else if (n_chunks % Hk == 0) {
        pl.Hkc = 1;
        pl.kv_groups = Hk;
        pl.chunks_per_kv = n_chunks / Hk;
    } else {
        return pl;
    }
    pl.valid = true;
    return pl;
}

size_t ulysses_dist_attn_overlap_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                                 int n_chunks) {
    if (check_attention_shape(P, b, s, h_q, h_kv, d, dtype) == ULY_ERR_INVALID_ARG) return 0;
    const OverlapPlan pl = overlap_plan(P, h_q, h_kv, n_chunks);
    if (s % P || !pl.valid) return 0;
    const int e = elem_bytes(dtype);
    const uint64_t qb = round256((uint64_t)b * s * pl.Hc * d * e);
    const uint64_t kb = round256((uint64_t)b * s * pl.Hkc * d * e);
    return (size_t)((uint64_t)P * (2 * qb * pl.nc + 2 * kb * pl.kv_groups));
}

uly_status ulysses_dist_attn_fwd_overlap(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                         const void* const* q_seq, const void* const* k_seq,
                                         const void* const* v_seq, void* const* o_seq, void* workspace,
                                         size_t workspace_bytes, int n_chunks, cudaStream_t stream,
                                         cudaStream_t side_stream) {
    uly_status st = check_attention_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    st = check_exchange_shape(P, b, s, h_q, d, dtype);
    if (st != ULY_OK) return st;
    st = check_kv_exchange_shape(P, b, s, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    const OverlapPlan pl = overlap_plan(P, h_q, h_kv, n_chunks);
    if (!pl.valid) return ULY_ERR_INVALID_ARG;
    const int e = elem_bytes(dtype);
    const int S = s / P;
    const uint64_t qsb = (uint64_t)b * S * h_q * d * e, ksb = (uint64_t)b * S * h_kv * d * e;
    RangeSet rq, rk, rv, ro;
    if (!collect(q_seq, P, qsb, rq) || !collect(k_seq, P, ksb, rk) || !collect(v_seq, P, ksb, rv) ||
        !collect(reinterpret_cast<const void* const*>(o_seq), P, qsb, ro))
        return ULY_ERR_INVALID_ARG;
    if (overlaps(ro, rq) || overlaps(ro, rk) || overlaps(ro, rv) || self_overlap(ro)) return ULY_ERR_INVALID_ARG;
    const size_t need = ulysses_dist_attn_overlap_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, n_chunks);
    if (!workspace_ok(workspace, workspace_bytes, need)) return ULY_ERR_INVALID_ARG;
    const RangeSet rw = one_range(workspace, need);
    if (overlaps(rw, rq) || overlaps(rw, rk) || overlaps(rw, rv) || overlaps(rw, ro)) return ULY_ERR_INVALID_ARG;

    // workspace: [chunk][rank] head-layout Q and O of the chunk's query heads, then
    // [K/V group][rank] head-layout K and V
    const int nc = pl.nc, Hc = pl.Hc, Hkc = pl.Hkc;
    const Carve wq(workspace, {(uint64_t)b * s * Hc * d * e, (uint64_t)b * s * Hc * d * e});
    const Carve wkv(static_cast<uint8_t*>(workspace) + wq.per_rank * nc * P,
                    {(uint64_t)b * s * Hkc * d * e, (uint64_t)b * s * Hkc * d * e});
    auto buf = [&](int c, int r, int k) {  // k: 0 Q, 1 K, 2 V, 3 O
        return k == 0 || k == 3 ? wq.at(c * P + r, k == 0 ? 0 : 1) : wkv.at(pl.kv_of(c) * P + r, k - 1);
    };

    cudaEvent_t ev[2 * kMaxChunks + 2];
    int n_ev = 0;
    auto cleanup = [&]() {
        for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
    };
    for (int i = 0; i < 2 * nc + 2; ++i) {
        if (cudaEventCreateWithFlags(&ev[n_ev], cudaEventDisableTiming) != cudaSuccess) {
            cleanup();
            return ULY_ERR_CUDA;
        }
        ++n_ev;
    }
    cudaEvent_t ev_start = ev[0], ev_done = ev[1];
    auto ev_in = [&](int c) { return ev[2 + c]; };
    auto ev_attn = [&](int c) { return ev[2 + nc + c]; };

    uly::PermuteTensor t_rec[3];
    uly::PermuteTensor* t = t_rec;
    auto exchange_in = [&](int c) {  // all-to-all #1 for chunk c's query heads, and its K/V heads
        memset(t, 0, 3 * sizeof(uly::PermuteTensor));  // unless an earlier chunk exchanged them
        const void* const* src[3] = {q_seq, k_seq, v_seq};
        const int nt = pl.new_kv(c) ? 3 : 1;
        for (int k = 0; k < nt; ++k) {
            for (int r = 0; r < P; ++r) {
                t[k].src[r] = src[k][r];
                t[k].dst[r] = buf(c, r, k);
            }
            t[k].h = k == 0 ? h_q : h_kv;
            t[k].hsub = k == 0 ? Hc : Hkc;
            t[k].hoff = k == 0 ? c * Hc : pl.kv_of(c) * Hkc;
            if (k > 0) t[k].rep = uly::kv_replication(P, h_kv);
        }
        return uly::launch_permute(0, P, b, s, d, e, t, nt, side_stream);
    };
    auto exchange_out = [&](int c) {  // all-to-all #2 for chunk c's output heads (side stream)
        memset(t, 0, sizeof(uly::PermuteTensor));
        for (int r = 0; r < P; ++r) {
            t[0].src[r] = buf(c, r, 3);
            t[0].dst[r] = o_seq[r];
        }
        t[0].h = h_q;
        t[0].hsub = Hc;
        t[0].hoff = c * Hc;
        return uly::launch_permute(1, P, b, s, d, e, t, 1, side_stream);
    };
    uly::AttnPtrs head_rec;
    uly::AttnPtrs* head = &head_rec;
    bool ok = cudaEventRecord(ev_start, stream) == cudaSuccess &&
              cudaStreamWaitEvent(side_stream, ev_start, 0) == cudaSuccess;
    for (int c = 0; c < 2 && c < nc && ok; ++c)
        ok = exchange_in(c) == cudaSuccess && cudaEventRecord(ev_in(c), side_stream) == cudaSuccess;
    for (int c = 0; c < nc && ok; ++c) {
        // main stream: attention of chunk c once its inputs are exchanged
        memset(head, 0, sizeof(uly::AttnPtrs));
        for (int r = 0; r < P; ++r) {
            head->q[r] = buf(c, r, 0);
            head->k[r] = buf(c, r, 1);
            head->v[r] = buf(c, r, 2);
            head->o[r] = buf(c, r, 3);
        }
        ok = cudaStreamWaitEvent(stream, ev_in(c), 0) == cudaSuccess;
        if (ok) {
            st = run_attention(P, b, s, Hc * P, Hkc * P, d, dtype, causal, 0, *head, stream);
            ok = st == ULY_OK;
        }
        ok = ok && cudaEventRecord(ev_attn(c), stream) == cudaSuccess;
        // side stream: chunk c's output exchange, then chunk c+2's input exchange, both
        // running while the main stream computes chunk c+1
        ok = ok && cudaStreamWaitEvent(side_stream, ev_attn(c), 0) == cudaSuccess && exchange_out(c) == cudaSuccess;
        if (ok && c + 2 < nc)
            ok = exchange_in(c + 2) == cudaSuccess && cudaEventRecord(ev_in(c + 2), side_stream) == cudaSuccess;
    }
    ok = ok && cudaEventRecord(ev_done, side_stream) == cudaSuccess &&
         cudaStreamWaitEvent(stream, ev_done, 0) == cudaSuccess;
    cleanup();  // destroying a recorded event is legal: its resources go once the work completes
    if (!ok) return st != ULY_OK ? st : ULY_ERR_CUDA;
    return ULY_OK;
}

size_t ulysses_usp_workspace_bytes(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype) {
    if (Pu < 1 || Pr < 1 || Pu * Pr > kMaxRanks || s % (Pu * Pr) || h_kv < 1) return 0;
    if (check_attention_shape(Pu, b, s / Pr, h_q, h_kv, d, dtype) == ULY_ERR_INVALID_ARG) return 0;
    const int e = elem_bytes(dtype), L = s / Pr;
    const uint64_t qb = round256((uint64_t)b * L * (h_q / Pu) * d * e);
    const uint64_t kb = round256((uint64_t)b * L * uly::kv_heads_per_rank(Pu, h_kv) * d * e);
    return (size_t)((uint64_t)Pu * Pr * (2 * qb + 2 * kb));
}

}  // extern "C"

namespace {

// The two-level forward; lse (optional) receives, per Ulysses unit u < Pu, the log-sum-exp
// of its heads' rows over the whole sequence.
uly_status usp_attn_fwd(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                        const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                        void* const* o_seq, float* const* lse, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
    if (Pu < 1 || Pr < 1 || Pu * Pr > kMaxRanks || s < 1 || s % (Pu * Pr)) return ULY_ERR_INVALID_ARG;
    const int P = Pu * Pr, L = s / Pr, S = s / P;
    // heads split over the Ulysses degree only; the exchanges run inside each group of Pu ranks
    uly_status st = check_attention_shape(Pu, b, L, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    st = check_exchange_shape(Pu, b, L, h_q, d, dtype);
    if (st != ULY_OK) return st;
    st = check_kv_exchange_shape(Pu, b, L, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    if ((long long)b * h_q * ((s + 127) / 128) > 0x7fffffffLL) return ULY_ERR_INVALID_ARG;
    if (dtype != ULY_BF16 || L % 128 != 0) return ULY_ERR_UNSUPPORTED;
    const int Hk = uly::kv_heads_per_rank(Pu, h_kv), kv_rep = uly::kv_replication(Pu, h_kv);
    const uint64_t qsb = (uint64_t)b * S * h_q * d * 2, ksb = (uint64_t)b * S * h_kv * d * 2;
    RangeSet rq, rk, rv, ro;
    if (!collect(q_seq, P, qsb, rq) || !collect(k_seq, P, ksb, rk) || !collect(v_seq, P, ksb, rv) ||
        !collect(reinterpret_cast<const void* const*>(o_seq), P, qsb, ro))
        return ULY_ERR_INVALID_ARG;
    if (overlaps(ro, rq) || overlaps(ro, rk) || overlaps(ro, rv) || self_overlap(ro)) return ULY_ERR_INVALID_ARG;
    RangeSet rl;
    if (lse) {
        if (!collect_f(lse, Pu, (uint64_t)b * (h_q / Pu) * s * 4, rl)) return ULY_ERR_INVALID_ARG;
        if (self_overlap(rl) || overlaps(rl, rq) || overlaps(rl, rk) || overlaps(rl, rv) || overlaps(rl, ro))
            return ULY_ERR_INVALID_ARG;
    }
    const size_t need = ulysses_usp_workspace_bytes(Pu, Pr, b, s, h_q, h_kv, d, dtype);
    if (!workspace_ok(workspace, workspace_bytes, need)) return ULY_ERR_INVALID_ARG;
    const RangeSet rw = one_range(workspace, need);
    if (overlaps(rw, rq) || overlaps(rw, rk) || overlaps(rw, rv) || overlaps(rw, ro) || overlaps(rw, rl))
        return ULY_ERR_INVALID_ARG;

    // workspace: per rank [Q | K | V | O] in head layout of its group: [b][s/Pr][h/Pu][d]
    const Carve ws(workspace, {(uint64_t)b * L * (h_q / Pu) * d * 2, (uint64_t)b * L * Hk * d * 2,
                               (uint64_t)b * L * Hk * d * 2, (uint64_t)b * L * (h_q / Pu) * d * 2});
    uly::PermuteTensor t_rec[3];
    uly::PermuteTensor* t = t_rec;
    cudaError_t ce = cudaSuccess;
    // (1) all-to-all #1 inside every ring group of Pu consecutive ranks
    for (int g = 0; g < Pr && ce == cudaSuccess; ++g) {
        memset(t, 0, 3 * sizeof(uly::PermuteTensor));
        const void* const* src[3] = {q_seq, k_seq, v_seq};
        for (int k = 0; k < 3; ++k) {
            for (int u = 0; u < Pu; ++u) {
                t[k].src[u] = src[k][g * Pu + u];
                t[k].dst[u] = ws.at(g * Pu + u, k);
            }
            t[k].h = k == 0 ? h_q : h_kv;
            if (k > 0) t[k].rep = kv_rep;  // replicated K/V heads: a broadcast inside the group
        }
        ce = uly::launch_permute(0, Pu, b, L, d, 2, t, 3, stream);
    }
    // (2) attention over the whole sequence: the ring's K/V blocks are read from the buffers
    //     of the ranks that hold them
    uly::AttnPtrs head_rec;
    uly::AttnPtrs* head = &head_rec;
    memset(head, 0, sizeof(uly::AttnPtrs));
    for (int j = 0; j < P; ++j) {
        head->q[j] = ws.at(j, 0);
        head->k[j] = ws.at(j, 1);
        head->v[j] = ws.at(j, 2);
        head->o[j] = ws.at(j, 3);
    }
    for (int u = 0; u < Pu && lse; ++u) head->lse[u] = lse[u];
    int unsupported = 0;
    if (ce == cudaSuccess) ce = uly::launch_attention_tc_usp(Pu, Pr, b, s, h_q, h_kv, d, causal, *head, stream,
                                                             &unsupported);
    // (3) all-to-all #2 inside every ring group
    for (int g = 0; g < Pr && ce == cudaSuccess && !unsupported; ++g) {
        memset(t, 0, sizeof(uly::PermuteTensor));
        for (int u = 0; u < Pu; ++u) {
            t[0].src[u] = ws.at(g * Pu + u, 3);
            t[0].dst[u] = o_seq[g * Pu + u];
        }
        t[0].h = h_q;
        ce = uly::launch_permute(1, Pu, b, L, d, 2, t, 1, stream);
    }
    if (unsupported) return ULY_ERR_UNSUPPORTED;
    return ce == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

}  // namespace

extern "C" {

uly_status ulysses_usp_attn_fwd(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                                void* const* o_seq, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return usp_attn_fwd(Pu, Pr, b, s, h_q, h_kv, d, dtype, causal, q_seq, k_seq, v_seq, o_seq, nullptr, workspace,
                        workspace_bytes, stream);
}

uly_status ulysses_usp_attn_fwd_lse(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype,
                                    int causal, const void* const* q_seq, const void* const* k_seq,
                                    const void* const* v_seq, void* const* o_seq, float* const* lse,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!lse) return ULY_ERR_INVALID_ARG;
    if (dtype != ULY_BF16) return ULY_ERR_UNSUPPORTED;
    return usp_attn_fwd(Pu, Pr, b, s, h_q, h_kv, d, dtype, causal, q_seq, k_seq, v_seq, o_seq, lse, workspace,
                        workspace_bytes, stream);
}

// Workspace of the two-level backward: per rank the group head-layout Q, K, V, dO, dQ, dK, dV
// ([b][s/Pr][h/Pu][d]), then per Ulysses unit the two fp32 row arrays over all s rows.
size_t ulysses_usp_bwd_workspace_bytes(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype) {
    if (ulysses_usp_workspace_bytes(Pu, Pr, b, s, h_q, h_kv, d, dtype) == 0 || dtype != ULY_BF16) return 0;
    const int L = s / Pr;
    const uint64_t qb = round256((uint64_t)b * L * (h_q / Pu) * d * 2);
    const uint64_t kb = round256((uint64_t)b * L * uly::kv_heads_per_rank(Pu, h_kv) * d * 2);
    // replicated K/V heads: the dK/dV slots hold every replica's fp32 share until they are summed
    const uint64_t gb = uly::kv_replication(Pu, h_kv) > 1 ? 2 * kb : kb;
    const uint64_t ra = row_array_bytes(Pu, b, s, h_q);
    return (size_t)((uint64_t)Pu * Pr * (4 * qb + kb + 2 * gb) + (uint64_t)Pu * 2 * ra);
}

uly_status ulysses_usp_attn_bwd(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                                const void* const* o_seq, const void* const* do_seq, const float* const* lse,
                                void* const* dq_seq, void* const* dk_seq, void* const* dv_seq, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
    if (Pu < 1 || Pr < 1 || Pu * Pr > kMaxRanks || s < 1 || s % (Pu * Pr)) return ULY_ERR_INVALID_ARG;
    const int P = Pu * Pr, L = s / Pr, S = s / P;
    uly_status st = check_train_shape(Pu, b, L, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    st = check_exchange_shape(Pu, b, L, h_q, d, dtype);
    if (st != ULY_OK) return st;
    st = check_kv_exchange_shape(Pu, b, L, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    if ((long long)b * h_q * ((s + 127) / 128) > 0x7fffffffLL) return ULY_ERR_INVALID_ARG;
    if (P > 48 || L % 128 != 0) return ULY_ERR_UNSUPPORTED;
    const int Hk = uly::kv_heads_per_rank(Pu, h_kv), kv_rep = uly::kv_replication(Pu, h_kv);
    const uint64_t qsb = (uint64_t)b * S * h_q * d * 2, ksb = (uint64_t)b * S * h_kv * d * 2;
    RangeSet in, rdq, rdk, rdv;
    if (!collect(q_seq, P, qsb, in) || !collect(k_seq, P, ksb, in) || !collect(v_seq, P, ksb, in) ||
        !collect(o_seq, P, qsb, in) || !collect(do_seq, P, qsb, in) ||
        !collect_f(lse, Pu, (uint64_t)b * (h_q / Pu) * s * 4, in) ||
        !collect(reinterpret_cast<const void* const*>(dq_seq), P, qsb, rdq) ||
        !collect(reinterpret_cast<const void* const*>(dk_seq), P, ksb, rdk) ||
        !collect(reinterpret_cast<const void* const*>(dv_seq), P, ksb, rdv))
        return ULY_ERR_INVALID_ARG;
    RangeSet outs;
    if (!outs.append(rdq) || !outs.append(rdk) || !outs.append(rdv)) return ULY_ERR_INVALID_ARG;
    if (self_overlap(outs) || overlaps(outs, in)) return ULY_ERR_INVALID_ARG;
    const size_t need = ulysses_usp_bwd_workspace_bytes(Pu, Pr, b, s, h_q, h_kv, d, dtype);
    if (!workspace_ok(workspace, workspace_bytes, need)) return ULY_ERR_INVALID_ARG;
    const RangeSet rw = one_range(workspace, need);
    if (overlaps(rw, in) || overlaps(rw, outs)) return ULY_ERR_INVALID_ARG;

    const uint64_t qb = (uint64_t)b * L * (h_q / Pu) * d * 2, kb = (uint64_t)b * L * Hk * d * 2;
    const uint64_t gb = kv_rep > 1 ? 2 * kb : kb;  // fp32 shares of replicated K/V heads
    enum { QH, KH, VH, DOH, DQH, DKH, DVH };
    const Carve ws(workspace, {qb, kb, kb, qb, qb, gb, gb});
    const uint64_t ra = row_array_bytes(Pu, b, s, h_q);
    const Carve wr(static_cast<uint8_t*>(workspace) + ws.per_rank * P, {ra, ra});
    // (1) all-to-all #1 on Q, K, V and dO inside every ring group
    uly::PermuteTensor t_rec[4];
    uly::PermuteTensor* t = t_rec;
    cudaError_t ce = cudaSuccess;
    const void* const* srcs[4] = {q_seq, k_seq, v_seq, do_seq};
    const int dsts[4] = {QH, KH, VH, DOH};
    for (int g = 0; g < Pr && ce == cudaSuccess; ++g) {
        memset(t, 0, 4 * sizeof(uly::PermuteTensor));
        for (int k = 0; k < 4; ++k) {
            for (int u = 0; u < Pu; ++u) {
                t[k].src[u] = srcs[k][g * Pu + u];
                t[k].dst[u] = ws.at(g * Pu + u, dsts[k]);
            }
            t[k].h = (k == 1 || k == 2) ? h_kv : h_q;
            if (k == 1 || k == 2) t[k].rep = kv_rep;
        }
        ce = uly::launch_permute(0, Pu, b, L, d, 2, t, 4, stream);
    }
    if (ce != cudaSuccess) return ULY_ERR_CUDA;
    // (2) the attention backward over the whole sequence (statistics from the seq-layout O, dO)
    uly::BwdPtrs p_rec;
    uly::BwdPtrs* p = &p_rec;
    memset(p, 0, sizeof(uly::BwdPtrs));
    for (int j = 0; j < P; ++j) {
        p->q[j] = ws.at(j, QH);
        p->k[j] = ws.at(j, KH);
        p->v[j] = ws.at(j, VH);
        p->dout[j] = ws.at(j, DOH);
        p->o_rows[j] = o_seq[j];
        p->do_rows[j] = do_seq[j];
        p->dq[j] = ws.at(j, DQH);
        p->dk[j] = ws.at(j, DKH);
        p->dv[j] = ws.at(j, DVH);
    }
    for (int u = 0; u < Pu; ++u) {
        p->lse[u] = lse[u];
        p->lse2[u] = static_cast<float*>(wr.at(u, 0));
        p->dsum[u] = static_cast<float*>(wr.at(u, 1));
    }
    p->od_seq_layout = 1;
    p->kv_grad_f32 = kv_rep > 1 ? 1 : 0;
    int unsupported = 0;
    ce = uly::launch_attention_bwd_tc_usp(Pu, Pr, b, s, h_q, h_kv, d, causal, *p, stream, &unsupported);
    if (unsupported) return ULY_ERR_UNSUPPORTED;
    if (ce != cudaSuccess) return ULY_ERR_CUDA;
    // (3) all-to-all #2 on dQ, dK, dV inside every ring group.  Replicated K/V heads: the
    //     group's replicas of a head hold the gradients from their own query heads, and the
    //     backward of the broadcast is their sum
    const int n_plain = kv_rep > 1 ? 1 : 3;
    void* const* dsts2[3] = {dq_seq, dk_seq, dv_seq};
    const int srcs2[3] = {DQH, DKH, DVH};
    for (int g = 0; g < Pr && ce == cudaSuccess; ++g) {
        memset(t, 0, 3 * sizeof(uly::PermuteTensor));
        for (int k = 0; k < 3; ++k) {
            for (int u = 0; u < Pu; ++u) {
                t[k].src[u] = ws.at(g * Pu + u, srcs2[k]);
                t[k].dst[u] = dsts2[k][g * Pu + u];
            }
            t[k].h = k == 0 ? h_q : h_kv;
        }
        ce = uly::launch_permute(1, Pu, b, L, d, 2, t, n_plain, stream);
        for (int k = 1; k < 3 && kv_rep > 1 && ce == cudaSuccess; ++k)
            ce = uly::launch_kv_grad_sum(Pu, kv_rep, b, L, h_kv, d, t[k].src, t[k].dst, stream);
    }
    return ce == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

uly_status ulysses_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    if (limit_ns < 1000ull || limit_ns > 10000000000ull) return ULY_ERR_INVALID_ARG;
    return uly::launch_wait_selftest(limit_ns, stream) == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
}

uly_status ulysses_device_status(int clear) {
    unsigned int v = 0;
    if (uly::read_device_error(&v, clear) != cudaSuccess) return ULY_ERR_CUDA;
    return v ? ULY_ERR_TIMEOUT : ULY_OK;
}

const char* ulysses_status_string(uly_status status) {
    switch (status) {
        case ULY_OK: return "ULY_OK";
        case ULY_ERR_INVALID_ARG: return "ULY_ERR_INVALID_ARG";
        case ULY_ERR_UNSUPPORTED: return "ULY_ERR_UNSUPPORTED";
        case ULY_ERR_CUDA: return "ULY_ERR_CUDA";
        case ULY_ERR_TIMEOUT: return "ULY_ERR_TIMEOUT";
    }
    return "ULY_UNKNOWN_STATUS";
}

}  // extern "C"
