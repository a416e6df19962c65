// fp32 local attention (head layout), fp32 FMA arithmetic throughout -- no tensor cores,
// no TF32 -- for the fp32 I/O path of the Ulysses forward.
//
// "DeepSpeed-Ulysses 深度解析", step 4: every rank computes softmax(Q K^T / sqrt(d)) V for its
// local heads over the whole sequence.  The softmax is evaluated blockwise with a running
// row maximum m, a running sum l and an unnormalised accumulator A, initialised to
// (-inf, 0, 0) and finished as A / l ("长上下文训练中的 SP 与 CP", section on Ring
// Attention, online-softmax paragraph); the causal mask compares global positions.
//
// Work split: a block of 128 threads owns 32 query rows of one (rank, batch, head); four
// threads share a row and each keeps every fourth element of q and of the accumulator in
// registers.  Key/value tiles of kBK rows are staged in shared memory and shared by the
// 32 rows.
#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace uly {
namespace {

constexpr int kRows = 32;
constexpr int kThreads = kRows * 4;
constexpr int kBK = 32;

struct F32Params {
    AttnPtrs ptrs;
    int b, s, Hq, Hk, g, d, causal;
    float scale;
};

template <int DMAX>
__global__ void __launch_bounds__(kThreads) attn_fp32_kernel(const __grid_constant__ F32Params p) {
    constexpr int DS = DMAX / 4;
    extern __shared__ float4 smem_f4[];
    float* Ks = reinterpret_cast<float*>(smem_f4);
    const int d = p.d;
    float* Vs = Ks + kBK * d;
    float* sS = Vs + kBK * d;  // [kRows][kBK] scores of the current tile

    const int rank = blockIdx.z / p.b;
    const int bb = blockIdx.z % p.b;
    const int hh = blockIdx.y;
    const int kh = hh / p.g;
    const int q0 = blockIdx.x * kRows;
    const int row = threadIdx.x >> 2;
    const int ql = threadIdx.x & 3;
    const int qi = q0 + row;

    const float* Q = static_cast<const float*>(p.ptrs.q[rank]);
    const float* K = static_cast<const float*>(p.ptrs.k[rank]);
    const float* V = static_cast<const float*>(p.ptrs.v[rank]);
    float* O = static_cast<float*>(p.ptrs.o[rank]);

    float q[DS], acc[DS];
#pragma unroll
    for (int i = 0; i < DS; ++i) {
        const int c = ql + 4 * i;
        q[i] = (c < d && qi < p.s) ? Q[(((size_t)bb * p.s + qi) * p.Hq + hh) * d + c] : 0.f;
        acc[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    const int q_last = min(q0 + kRows, p.s) - 1;
    const int kv_end = p.causal ? q_last + 1 : p.s;
    const int d4 = d >> 2;
    for (int k0 = 0; k0 < kv_end; k0 += kBK) {
        __syncthreads();
        for (int e = threadIdx.x; e < kBK * d4; e += kThreads) {
            const int kr = e / d4, c4 = e - kr * d4;
            const int key = k0 + kr;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (key < p.s) {
                const size_t off = (((size_t)bb * p.s + key) * p.Hk + kh) * d + 4 * c4;
                kv = *reinterpret_cast<const float4*>(K + off);
                vv = *reinterpret_cast<const float4*>(V + off);
            }
            reinterpret_cast<float4*>(Ks)[e] = kv;
            reinterpret_cast<float4*>(Vs)[e] = vv;
        }
        __syncthreads();

        // scores of this tile -> sS[row][kk] (written by the first thread of each quad)
        float* srow = sS + row * kBK;
        float tmax = -INFINITY;
#pragma unroll 2
        for (int kk = 0; kk < kBK; ++kk) {
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < DS; ++i) {
                const int c = ql + 4 * i;
                if (c < d) part = fmaf(q[i], Ks[kk * d + c], part);
            }
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            const int key = k0 + kk;
            const bool visible = key < p.s && (!p.causal || key <= qi);
            const float sc = visible ? part * p.scale : -INFINITY;
            if (ql == 0) srow[kk] = sc;
            tmax = fmaxf(tmax, sc);
        }
        __syncwarp();
        const float m_new = fmaxf(m, tmax);
        if (m_new != -INFINITY) {  // else nothing visible yet for this row
            const float alpha = expf(m - m_new);
            l *= alpha;
#pragma unroll
            for (int i = 0; i < DS; ++i) acc[i] *= alpha;
#pragma unroll 2
            for (int kk = 0; kk < kBK; ++kk) {
                const float pk = expf(srow[kk] - m_new);
                l += pk;
#pragma unroll
                for (int i = 0; i < DS; ++i) {
                    const int c = ql + 4 * i;
                    if (c < d) acc[i] = fmaf(pk, Vs[kk * d + c], acc[i]);
                }
            }
            m = m_new;
        }
        __syncwarp();
    }
    if (qi < p.s) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int i = 0; i < DS; ++i) {
            const int c = ql + 4 * i;
            if (c < d) O[(((size_t)bb * p.s + qi) * p.Hq + hh) * d + c] = acc[i] * inv;
        }
    }
}

template <int DMAX>
cudaError_t launch_dmax(const F32Params& prm, int P, cudaStream_t stream) {
    const size_t smem = ((size_t)2 * kBK * prm.d + (size_t)kRows * kBK) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(attn_fp32_kernel<DMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((prm.s + kRows - 1) / kRows, prm.Hq, prm.b * P);
    attn_fp32_kernel<DMAX><<<grid, kThreads, smem, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_fp32(int P, int b, int s, int h_q, int h_kv, int d, int causal, const AttnPtrs& ptrs,
                                  cudaStream_t stream) {
    F32Params prm;
    memset(&prm, 0, sizeof(prm));
    prm.ptrs = ptrs;
    prm.b = b;
    prm.s = s;
    prm.Hq = h_q / P;
    prm.Hk = kv_heads_per_rank(P, h_kv);
    prm.g = prm.Hq / prm.Hk;  // within a rank (its K/V heads may be replicas shared with other ranks)
    prm.d = d;
    prm.causal = causal ? 1 : 0;
    prm.scale = 1.0f / sqrtf((float)d);
    if (d <= 32) return launch_dmax<32>(prm, P, stream);
    if (d <= 64) return launch_dmax<64>(prm, P, stream);
    if (d <= 128) return launch_dmax<128>(prm, P, stream);
    return launch_dmax<256>(prm, P, stream);
}

}  // namespace uly
