// C ABI of the Ulysses forward (declared in include/ulysses.h): argument validation, the
// composition of the three stages, and dispatch to the kernels.  Nothing here allocates
// device memory; every argument error is reported before any work is enqueued.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <utility>
#include <vector>

#include "../../include/ulysses.h"
#include "internal.h"

namespace {

using uly::kMaxRanks;

constexpr uint64_t kMaxSlabVecs = (1ull << 31) - 1;  // 32-bit index space of the permute kernel

int elem_bytes(uly_dtype dt) { return dt == ULY_FP32 ? 4 : (dt == ULY_BF16 ? 2 : 0); }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Non-null, 16-byte aligned pointers; collects their byte ranges.
bool collect(const void* const* ptrs, int P, uint64_t bytes, std::vector<Range>& out) {
    if (!ptrs) return false;
    for (int i = 0; i < P; ++i) {
        if (!ptrs[i] || !aligned16(ptrs[i])) return false;
        const uintptr_t lo = reinterpret_cast<uintptr_t>(ptrs[i]);
        out.push_back({lo, lo + (uintptr_t)bytes});
    }
    return true;
}

bool overlaps(const std::vector<Range>& a, const std::vector<Range>& b) {
    for (const Range& x : a)
        for (const Range& y : b)
            if (x.lo < y.hi && y.lo < x.hi && x.hi > x.lo && y.hi > y.lo) return true;
    return false;
}

bool self_overlap(const std::vector<Range>& a) {
    for (size_t i = 0; i < a.size(); ++i)
        for (size_t k = i + 1; k < a.size(); ++k)
            if (a[i].lo < a[k].hi && a[k].lo < a[i].hi && a[i].hi > a[i].lo && a[k].hi > a[k].lo) return true;
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

uly_status check_attention_shape(int P, int b, int s, int hq, int hkv, int d, uly_dtype dt) {
    if (P < 1 || P > kMaxRanks || b < 1 || s < 1 || hq < 1 || hkv < 1 || d < 1) return ULY_ERR_INVALID_ARG;
    if (hq % P || hkv % P || hq % hkv) return ULY_ERR_INVALID_ARG;
    if (!elem_bytes(dt)) return ULY_ERR_INVALID_ARG;
    if ((long long)b * P > 65535 || hq / P > 65535) return ULY_ERR_INVALID_ARG;
    if ((long long)b * hq * ((s + 127) / 128) > 0x7fffffffLL) return ULY_ERR_INVALID_ARG;
    if (dt == ULY_FP32 && (d % 4 != 0 || d > 256)) return ULY_ERR_UNSUPPORTED;
    if (dt == ULY_BF16 && !uly::tc_attention_supported(d)) return ULY_ERR_UNSUPPORTED;
    return ULY_OK;
}

uint64_t round256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

uly_status exchange(int direction, int P, int b, int s, int h, int d, uly_dtype dt, const void* const* in,
                    void* const* out, cudaStream_t stream) {
    uly_status st = check_exchange_shape(P, b, s, h, d, dt);
    if (st != ULY_OK) return st;
    const uint64_t bytes = (uint64_t)b * (s / P) * h * d * elem_bytes(dt);  // equal on both sides
    std::vector<Range> ri, ro;
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
        if (fused) return ULY_ERR_UNSUPPORTED;
        return uly::launch_attention_fp32(P, b, s, hq, hkv, d, causal, ptrs, stream) == cudaSuccess ? ULY_OK
                                                                                                    : ULY_ERR_CUDA;
    }
    int unsupported = 0;
    cudaError_t e = uly::launch_attention_tc(P, b, s, hq, hkv, d, causal, fused, ptrs, stream, &unsupported);
    if (unsupported) return ULY_ERR_UNSUPPORTED;
    return e == cudaSuccess ? ULY_OK : ULY_ERR_CUDA;
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

uly_status ulysses_local_attention(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                   const void* const* q_head, const void* const* k_head, const void* const* v_head,
                                   void* const* o_head, cudaStream_t stream) {
    uly_status st = check_attention_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    const int e = elem_bytes(dtype);
    const uint64_t qb = (uint64_t)b * s * (h_q / P) * d * e, kb = (uint64_t)b * s * (h_kv / P) * d * e;
    std::vector<Range> rq, rk, rv, ro;
    if (!collect(q_head, P, qb, rq) || !collect(k_head, P, kb, rk) || !collect(v_head, P, kb, rv) ||
        !collect(reinterpret_cast<const void* const*>(o_head), P, qb, ro))
        return ULY_ERR_INVALID_ARG;
    if (overlaps(ro, rq) || overlaps(ro, rk) || overlaps(ro, rv) || self_overlap(ro)) return ULY_ERR_INVALID_ARG;
    uly::AttnPtrs ptrs;
    memset(&ptrs, 0, sizeof(ptrs));
    for (int r = 0; r < P; ++r) {
        ptrs.q[r] = q_head[r];
        ptrs.k[r] = k_head[r];
        ptrs.v[r] = v_head[r];
        ptrs.o[r] = o_head[r];
    }
    return run_attention(P, b, s, h_q, h_kv, d, dtype, causal, 0, ptrs, stream);
}

size_t ulysses_dist_attn_workspace_bytes(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int fused) {
    if (check_attention_shape(P, b, s, h_q, h_kv, d, dtype) == ULY_ERR_INVALID_ARG) return 0;
    if (s % P) return 0;
    if (fused) return 0;
    const int e = elem_bytes(dtype);
    const uint64_t qb = round256((uint64_t)b * s * (h_q / P) * d * e);
    const uint64_t kb = round256((uint64_t)b * s * (h_kv / P) * d * e);
    return (size_t)((uint64_t)P * (2 * qb + 2 * kb));
}

uly_status ulysses_dist_attn_fwd(int P, int b, int s, int h_q, int h_kv, int d, uly_dtype dtype, int causal,
                                 const void* const* q_seq, const void* const* k_seq, const void* const* v_seq,
                                 void* const* o_seq, void* workspace, size_t workspace_bytes, int fused,
                                 cudaStream_t stream) {
    uly_status st = check_attention_shape(P, b, s, h_q, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    st = check_exchange_shape(P, b, s, h_q, d, dtype);
    if (st != ULY_OK) return st;
    st = check_exchange_shape(P, b, s, h_kv, d, dtype);
    if (st != ULY_OK) return st;
    const int e = elem_bytes(dtype);
    const int S = s / P;
    const uint64_t qsb = (uint64_t)b * S * h_q * d * e, ksb = (uint64_t)b * S * h_kv * d * e;
    std::vector<Range> rq, rk, rv, ro;
    if (!collect(q_seq, P, qsb, rq) || !collect(k_seq, P, ksb, rk) || !collect(v_seq, P, ksb, rv) ||
        !collect(reinterpret_cast<const void* const*>(o_seq), P, qsb, ro))
        return ULY_ERR_INVALID_ARG;
    if (overlaps(ro, rq) || overlaps(ro, rk) || overlaps(ro, rv) || self_overlap(ro)) return ULY_ERR_INVALID_ARG;

    if (fused) {
        if (dtype != ULY_BF16) return ULY_ERR_UNSUPPORTED;
        uly::AttnPtrs ptrs;
        memset(&ptrs, 0, sizeof(ptrs));
        for (int r = 0; r < P; ++r) {
            ptrs.q[r] = q_seq[r];
            ptrs.k[r] = k_seq[r];
            ptrs.v[r] = v_seq[r];
            ptrs.o[r] = o_seq[r];
        }
        return run_attention(P, b, s, h_q, h_kv, d, dtype, causal, 1, ptrs, stream);
    }

    const size_t need = ulysses_dist_attn_workspace_bytes(P, b, s, h_q, h_kv, d, dtype, 0);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
        return ULY_ERR_INVALID_ARG;
    std::vector<Range> rw{{reinterpret_cast<uintptr_t>(workspace), reinterpret_cast<uintptr_t>(workspace) + need}};
    if (overlaps(rw, rq) || overlaps(rw, rk) || overlaps(rw, rv) || overlaps(rw, ro)) return ULY_ERR_INVALID_ARG;

    // workspace: per rank [Q_head | K_head | V_head | O_head], each 256-byte aligned
    const uint64_t qhb = round256((uint64_t)b * s * (h_q / P) * d * e);
    const uint64_t khb = round256((uint64_t)b * s * (h_kv / P) * d * e);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uly::AttnPtrs head;
    memset(&head, 0, sizeof(head));
    for (int r = 0; r < P; ++r) {
        uint8_t* base = ws + (uint64_t)r * (2 * qhb + 2 * khb);
        head.q[r] = base;
        head.k[r] = base + qhb;
        head.v[r] = base + qhb + khb;
        head.o[r] = base + qhb + 2 * khb;
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
