// All-to-all #1 (seq -> head) and #2 (head -> seq) of the Ulysses forward as transposes
// between P per-rank buffers in one device's memory.
//
// "02 · DeepSpeed-Ulysses", section 2 "all-to-all 的转置与重分布": rank j splits its
// [s/P, h, d] block along heads, part r goes to rank r, and rank r concatenates the parts
// along the sequence axis in source-rank order.  With batch first:
//     head[r][bb][j*S + t][hh][:] == seq[j][bb][t][r*H + hh][:]     (S = s/P, H = h/P)
// For every (rank r, source rank j, batch bb) the head-layout side is one contiguous slab
// of S rows of H*d elements, and the seq-layout side is S runs of H*d elements with a
// pitch of h*d elements.  A call may also move only heads [hoff, hoff+hsub) of every
// rank's group (the head-layout side then holds hsub heads): the chunked, overlapped
// forward exchanges one head group at a time.  The kernel streams those slabs with 16-byte
// (or narrower) vector loads and stores: the contiguous side is fully coalesced, the
// strided side moves whole runs.  On GB300 it runs at the device's copy bandwidth; a
// version that moved whole runs as TMA tensor-map boxes measured 1.5-7% slower on every
// shape of the exchange sweep and is not used.
#include <cstring>
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "internal.h"

namespace uly {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct PermuteJob {
    const uint8_t* src[kMaxRanks];
    uint8_t* dst[kMaxRanks];
    uint64_t run_bytes;   // hsub*d*e: one contiguous run on the seq-layout side (H*d*e for a whole group)
    uint64_t rank_bytes;  // H*d*e: distance between consecutive ranks' head groups in a seq-layout row
    uint64_t head_off;    // hoff*d*e: first moved head inside a rank's group
    uint64_t row_pitch;   // h*d*e: seq-layout row pitch
    uint32_t rep;         // ranks sharing one head group (replicated K/V heads), else 1
    uint32_t slab_vecs;   // S*run_bytes / VEC
    FastDiv run_vecs;     // run_bytes / VEC
};

struct PermuteParams {
    PermuteJob job[4];
    uint32_t ntensors;
    uint32_t units;  // P*P*b slabs per tensor
    uint32_t P, S, s;
};

template <int VEC>
struct VecT;
template <>
struct VecT<16> { using T = uint4; };
template <>
struct VecT<8> { using T = uint2; };
template <>
struct VecT<4> { using T = uint32_t; };
template <>
struct VecT<2> { using T = uint16_t; };
template <>
struct VecT<1> { using T = uint8_t; };

template <typename T>
__device__ __forceinline__ T load_stream(const uint8_t* p) {
    return __ldcs(reinterpret_cast<const T*>(p));
}
template <>
__device__ __forceinline__ uint8_t load_stream<uint8_t>(const uint8_t* p) {
    return *reinterpret_cast<const volatile uint8_t*>(p);
}

// DIR 0: seq -> head (read strided, write contiguous); DIR 1: head -> seq (the reverse).
template <int VEC, int DIR>
__global__ void __launch_bounds__(kThreads) permute_kernel(const __grid_constant__ PermuteParams p) {
    using V = typename VecT<VEC>::T;
    const uint32_t P = p.P;
    for (uint32_t yu = blockIdx.y; yu < p.ntensors * p.units; yu += gridDim.y) {
        const uint32_t t = yu / p.units;
        const uint32_t u = yu - t * p.units;
        const uint32_t j = u % P;  // seq-layout rank (token block j)
        const uint32_t rest = u / P;
        const uint32_t r = rest % P;  // head-layout rank (head group r)
        const uint32_t bb = rest / P;
        const PermuteJob& J = p.job[t];
        const uint64_t off_contig = ((uint64_t)bb * p.s + (uint64_t)j * p.S) * J.run_bytes;
        const uint64_t off_strided =
            (uint64_t)bb * p.S * J.row_pitch + (uint64_t)(r / J.rep) * J.rank_bytes + J.head_off;
        const uint8_t* src = DIR == 0 ? J.src[j] + off_strided : J.src[r] + off_contig;
        uint8_t* dst = DIR == 0 ? J.dst[r] + off_contig : J.dst[j] + off_strided;
        const uint32_t n = J.slab_vecs;
        for (uint32_t i0 = blockIdx.x * (kThreads * kUnroll) + threadIdx.x; i0 < n;
             i0 += gridDim.x * (kThreads * kUnroll)) {
            V val[kUnroll];
            uint64_t so[kUnroll], co[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const uint32_t i = i0 + k * kThreads;
                const uint32_t row = fdiv(i, J.run_vecs);
                const uint32_t col = i - row * J.run_vecs.d;
                so[k] = (uint64_t)row * J.row_pitch + (uint64_t)col * VEC;
                co[k] = (uint64_t)i * VEC;
                if (i < n) val[k] = load_stream<V>(DIR == 0 ? src + so[k] : src + co[k]);
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const uint32_t i = i0 + k * kThreads;
                if (i < n) *reinterpret_cast<V*>(DIR == 0 ? dst + co[k] : dst + so[k]) = val[k];
            }
        }
    }
}

template <int VEC>
cudaError_t launch_vec(int direction, const PermuteParams& prm, uint32_t max_slab, cudaStream_t stream) {
    const uint32_t ys = prm.ntensors * prm.units;
    const uint32_t grid_y = ys < 65535u ? ys : 65535u;
    const uint64_t per_unit = (max_slab + (uint64_t)kThreads * kUnroll - 1) / ((uint64_t)kThreads * kUnroll);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // one full wave of 8 resident 256-thread blocks per SM, spread over the slabs
    const uint64_t target = (uint64_t)sms * 8;
    uint64_t gx = (target + grid_y - 1) / grid_y;
    if (gx > per_unit) gx = per_unit;
    if (gx < 1) gx = 1;
    if (gx > 65535) gx = 65535;
    dim3 grid((unsigned)gx, grid_y, 1);
    if (direction == 0)
        permute_kernel<VEC, 0><<<grid, kThreads, 0, stream>>>(prm);
    else
        permute_kernel<VEC, 1><<<grid, kThreads, 0, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_permute(int direction, int P, int b, int s, int d, int elem_bytes, const PermuteTensor* tensors,
                           int ntensors, cudaStream_t stream) {
    if (ntensors < 1 || ntensors > 4) return cudaErrorInvalidValue;
    for (int t = 0; t < ntensors; ++t)  // replication only broadcasts (the reverse sums: launch_kv_grad_sum)
        if (tensors[t].rep > 1 && (direction != 0 || tensors[t].h * tensors[t].rep != P)) return cudaErrorInvalidValue;
    if ((uint64_t)ntensors * P * P * b > 0xffffffffull) {  // one launch per tensor keeps the slab index in 32 bits
        for (int t = 0; t < ntensors; ++t) {
            const cudaError_t e = launch_permute(direction, P, b, s, d, elem_bytes, tensors + t, 1, stream);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    PermuteParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.ntensors = (uint32_t)ntensors;
    prm.P = (uint32_t)P;
    prm.S = (uint32_t)(s / P);
    prm.s = (uint32_t)s;
    prm.units = (uint32_t)P * (uint32_t)P * (uint32_t)b;
    // widest vector that divides every run and offset (all pointers are 16-byte aligned by contract)
    auto per_rank = [&](int t) { return tensors[t].rep > 1 ? 1 : tensors[t].h / P; };  // heads of a rank's group
    auto hsub = [&](int t) { return tensors[t].hsub > 0 ? tensors[t].hsub : per_rank(t); };
    int vec = 16;
    for (int t = 0; t < ntensors; ++t) {
        const uint64_t unit = (uint64_t)d * elem_bytes;
        const uint64_t sizes[3] = {hsub(t) * unit, (uint64_t)per_rank(t) * unit, (uint64_t)tensors[t].hoff * unit};
        for (uint64_t x : sizes)
            while (vec > 1 && x % vec) vec >>= 1;
    }
    uint32_t max_slab = 0;
    for (int t = 0; t < ntensors; ++t) {
        PermuteJob& J = prm.job[t];
        for (int r = 0; r < P; ++r) {
            J.src[r] = static_cast<const uint8_t*>(tensors[t].src[r]);
            J.dst[r] = static_cast<uint8_t*>(tensors[t].dst[r]);
        }
        J.run_bytes = (uint64_t)hsub(t) * d * elem_bytes;
        J.rank_bytes = (uint64_t)per_rank(t) * d * elem_bytes;
        J.rep = tensors[t].rep > 1 ? (uint32_t)tensors[t].rep : 1u;
        J.head_off = (uint64_t)tensors[t].hoff * d * elem_bytes;
        J.row_pitch = (uint64_t)tensors[t].h * d * elem_bytes;
        J.slab_vecs = (uint32_t)((uint64_t)prm.S * J.run_bytes / vec);
        J.run_vecs = make_fastdiv((uint32_t)(J.run_bytes / vec));
        if (J.slab_vecs > max_slab) max_slab = J.slab_vecs;
    }
    if (max_slab == 0) return cudaSuccess;
    switch (vec) {
        case 16: return launch_vec<16>(direction, prm, max_slab, stream);
        case 8: return launch_vec<8>(direction, prm, max_slab, stream);
        case 4: return launch_vec<4>(direction, prm, max_slab, stream);
        case 2: return launch_vec<2>(direction, prm, max_slab, stream);
        default: return launch_vec<1>(direction, prm, max_slab, stream);
    }
}

namespace {

struct KvGradSumParams {
    const uint8_t* src[kMaxRanks];
    uint8_t* dst[kMaxRanks];
    uint64_t n_vec;  // P * b * (s/P) * h_kv * (d/8) output vectors of 8 bf16
    uint32_t rep, b, s, S, hkv, dvec;
};

// One thread per 8 output elements: the rep replicas' fp32 partial gradients, summed.
__global__ void __launch_bounds__(256) kv_grad_sum_kernel(const __grid_constant__ KvGradSumParams p) {
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n_vec;
         i += (uint64_t)gridDim.x * blockDim.x) {
        uint64_t r = i;
        const uint32_t v = (uint32_t)(r % p.dvec);
        r /= p.dvec;
        const uint32_t h = (uint32_t)(r % p.hkv);
        r /= p.hkv;
        const uint32_t t = (uint32_t)(r % p.S);
        r /= p.S;
        const uint32_t bb = (uint32_t)(r % p.b);
        const uint32_t j = (uint32_t)(r / p.b);
        // fp32 head layout of replica rank h*rep + k: [b][s][1][d]; token j*S + t
        const uint64_t src_off = (((uint64_t)bb * p.s + (uint64_t)j * p.S + t) * p.dvec + v) * 32;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (uint32_t k = 0; k < p.rep; ++k) {
            const float4* x = reinterpret_cast<const float4*>(p.src[h * p.rep + k] + src_off);
            const float4 a = __ldcs(x), c = __ldcs(x + 1);
            acc[0] += a.x;
            acc[1] += a.y;
            acc[2] += a.z;
            acc[3] += a.w;
            acc[4] += c.x;
            acc[5] += c.y;
            acc[6] += c.z;
            acc[7] += c.w;
        }
        uint4 out;
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
        // seq layout of rank j: [b][s/P][h_kv][d]
        const uint64_t dst_off = ((((uint64_t)bb * p.S + t) * p.hkv + h) * p.dvec + v) * 16;
        *reinterpret_cast<uint4*>(p.dst[j] + dst_off) = out;
    }
}

}  // namespace

cudaError_t launch_kv_grad_sum(int P, int rep, int b, int s, int h_kv, int d, const void* const* src,
                               void* const* dst, cudaStream_t stream) {
    if (rep < 1 || h_kv * rep != P || d % 8 || s % P) return cudaErrorInvalidValue;
    KvGradSumParams prm;
    memset(&prm, 0, sizeof(prm));
    for (int r = 0; r < P; ++r) {
        prm.src[r] = static_cast<const uint8_t*>(src[r]);
        prm.dst[r] = static_cast<uint8_t*>(dst[r]);
    }
    prm.rep = (uint32_t)rep;
    prm.b = (uint32_t)b;
    prm.s = (uint32_t)s;
    prm.S = (uint32_t)(s / P);
    prm.hkv = (uint32_t)h_kv;
    prm.dvec = (uint32_t)(d / 8);
    prm.n_vec = (uint64_t)P * b * prm.S * h_kv * prm.dvec;
    if (prm.n_vec == 0) return cudaSuccess;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    uint64_t blocks = (prm.n_vec + 255) / 256;
    const uint64_t cap = (uint64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    kv_grad_sum_kernel<<<(unsigned)blocks, 256, 0, stream>>>(prm);
    return cudaGetLastError();
}

namespace {

// out[c][a] = in[a][c] for runs of run_bytes (a < A, c < C): the local halves of one rank's
// all-to-all with other GPUs (see launch_block_transpose).  Slab c = the A runs that land
// contiguously at out[c][0..A); they lie C runs apart in `in`.  grid.y walks the slabs,
// grid.x the vectors of a slab (read strided, written contiguously), as permute_kernel
// does, so small runs (a few KB) still give every thread four vectors in flight.
struct BlockTransposeParams {
    const uint8_t* in;
    uint8_t* out;
    uint64_t run_bytes;   // bytes of one run
    uint64_t in_pitch;    // C * run_bytes: from in[a][c] to in[a+1][c]
    uint64_t slab_bytes;  // A * run_bytes
    uint32_t C;
    uint32_t slab_vecs;   // A * run_bytes / VEC
    FastDiv run_vecs;     // run_bytes / VEC
};

template <int VEC>
__global__ void __launch_bounds__(kThreads) block_transpose_kernel(const __grid_constant__ BlockTransposeParams p) {
    using V = typename VecT<VEC>::T;
    for (uint32_t c = blockIdx.y; c < p.C; c += gridDim.y) {
        const uint8_t* src = p.in + (uint64_t)c * p.run_bytes;  // in[0][c]
        uint8_t* dst = p.out + (uint64_t)c * p.slab_bytes;      // out[c][0]
        const uint32_t n = p.slab_vecs;
        for (uint32_t i0 = blockIdx.x * (kThreads * kUnroll) + threadIdx.x; i0 < n;
             i0 += gridDim.x * (kThreads * kUnroll)) {
            V val[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const uint32_t i = i0 + k * kThreads;
                const uint32_t a = fdiv(i, p.run_vecs);
                const uint32_t col = i - a * p.run_vecs.d;
                if (i < n) val[k] = load_stream<V>(src + (uint64_t)a * p.in_pitch + (uint64_t)col * VEC);
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const uint32_t i = i0 + k * kThreads;
                if (i < n) *reinterpret_cast<V*>(dst + (uint64_t)i * VEC) = val[k];
            }
        }
    }
}

template <int VEC>
cudaError_t launch_bt(const BlockTransposeParams& prm, cudaStream_t stream) {
    const uint32_t grid_y = prm.C < 65535u ? prm.C : 65535u;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const uint64_t per_slab = (prm.slab_vecs + (uint64_t)kThreads * kUnroll - 1) / ((uint64_t)kThreads * kUnroll);
    uint64_t gx = ((uint64_t)sms * 8 + grid_y - 1) / grid_y;  // one wave of 8 blocks per SM
    if (gx > per_slab) gx = per_slab;
    if (gx < 1) gx = 1;
    if (gx > 65535) gx = 65535;
    block_transpose_kernel<VEC><<<dim3((unsigned)gx, grid_y, 1), kThreads, 0, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace

static int block_transpose_vec(uint64_t run_bytes, const void* in, const void* out) {
    int vec = 16;
    while (vec > 1 && (run_bytes % vec || (reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % vec))
        vec >>= 1;
    return vec;
}

// A slab's vector index is 32-bit: at most 2^31 - 1 vectors, so that the grid-stride steps
// past the end never wrap.
bool block_transpose_fits(uint64_t A, uint64_t C, uint64_t run_bytes, const void* in, const void* out) {
    if (A == 0 || C == 0 || run_bytes == 0) return true;
    const uint64_t rv = run_bytes / block_transpose_vec(run_bytes, in, out);
    return C <= 0xffffffffull && rv <= 0x7fffffffull && A <= 0x7fffffffull / rv;
}

cudaError_t launch_block_transpose(uint64_t A, uint64_t C, uint64_t run_bytes, const void* in, void* out,
                                   cudaStream_t stream) {
    if (A == 0 || C == 0 || run_bytes == 0) return cudaSuccess;
    if (!block_transpose_fits(A, C, run_bytes, in, out)) return cudaErrorInvalidValue;
    const int vec = block_transpose_vec(run_bytes, in, out);
    BlockTransposeParams prm;
    prm.in = static_cast<const uint8_t*>(in);
    prm.out = static_cast<uint8_t*>(out);
    prm.run_bytes = run_bytes;
    prm.in_pitch = C * run_bytes;
    prm.slab_bytes = A * run_bytes;
    prm.C = (uint32_t)C;
    prm.slab_vecs = (uint32_t)(A * (run_bytes / vec));
    prm.run_vecs = make_fastdiv((uint32_t)(run_bytes / vec));
    switch (vec) {
        case 16: return launch_bt<16>(prm, stream);
        case 8: return launch_bt<8>(prm, stream);
        case 4: return launch_bt<4>(prm, stream);
        case 2: return launch_bt<2>(prm, stream);
        default: return launch_bt<1>(prm, stream);
    }
}

}  // namespace uly
