// bf16 local attention on the sm_103a tensor cores (tcgen05.mma, fp32 accumulators in
// tensor memory, operands staged by TMA), with an optional fused mode that folds both
// Ulysses all-to-alls into the tile addressing.
//
// What it computes ("DeepSpeed-Ulysses 深度解析", step 4): for every query row i of every
// local head, O_i = softmax_j(q_i . k_j / sqrt(d)) v_j over the whole sequence, keys j > i
// masked when causal (global positions, "长上下文训练中的 SP 与 CP", Ring Attention
// section, causal paragraph), query head hh reading K/V head hh / g for grouped heads.
// The softmax runs blockwise with the running maximum / running sum / unnormalised
// accumulator recurrence of the same page's online-softmax paragraph, in base 2: scores
// are scaled by log2(e)/sqrt(d) and exponentiated with the hardware ex2.
//
// Tiles: 128 query rows x 128 keys; head dim d in {64, 128}.  One CTA per (rank, batch,
// head, query tile), 6 warps with fixed roles:
//   warp 0      TMA producer: Q once, then K_j and V_j into 2-stage rings
//   warp 1      allocates tensor memory and issues tcgen05.mma from one thread:
//                 S_j = Q K_j^T into one of two S buffers (tensor memory),
//                 O  += P_j V_j  into the O accumulator (tensor memory)
//   warps 2..5  softmax: one thread per query row reads its S row from tensor memory,
//               masks, updates (m, l), writes P_j = exp2(S - m) as bf16 into shared
//               memory, rescales O when the reference maximum moved; finally O / l is
//               written through shared memory with TMA stores.
// The MMA for S_{j+1} runs while the softmax works on S_j.  The reference maximum is
// only raised when a row maximum exceeds it by more than 8 (a factor 256), so O is
// rarely rescaled; P entries stay below 256, exact enough in bf16, and the final O / l
// is unchanged mathematically.
//
// Fused mode ("DeepSpeed-Ulysses 深度解析", steps 3 and 5; the all-to-alls of "02 ·
// DeepSpeed-Ulysses" section 3 "可合并"): the Q/K/V tiles of tokens [t0, t0+128) come
// straight from source rank t0 / (s/P)'s seq-layout buffer at head column gh, and the
// output tile goes straight to that rank's seq-layout output, so the head-layout copies
// never exist.  Requires (s/P) % 128 == 0 so no tile straddles two ranks.
//
// Every wait is bounded in time.  A wait that gives up sets a bit in a device error word
// and the CTA drains its copies and MMAs, frees tensor memory and exits; every later
// CTA sees the word and exits at once (ulysses_device_status reads and clears it).
#include <cstring>
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "internal.h"

namespace uly {

__device__ unsigned int g_uly_error_word = 0;

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 192;
constexpr int kMaxMaps = 16;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr unsigned int kErrTimeout = 1u;

struct TcParams {
    CUtensorMap mq[kMaxMaps];
    CUtensorMap mk[kMaxMaps];
    CUtensorMap mv[kMaxMaps];
    CUtensorMap mo[kMaxMaps];
    int s;             // sequence length
    int rows_per_map;  // tokens held by one map: s/P when fused, s otherwise
    int n_qtiles;      // ceil(s / BM)
    int heads;         // query heads per map group: h_q (fused) or h_q/P (per rank)
    int g;             // query heads per K/V head
    int b;
    int nranks;        // rank groups in this launch (fused: 1)
    int causal;
    float scale_log2;  // log2(e) / sqrt(d)
};

template <int D>
struct Smem {
    static constexpr uint32_t kTileQ = BM * D * 2;  // bytes of a Q (or K, V) tile
    static constexpr uint32_t kTileKV = BN * D * 2;
    static constexpr uint32_t kTileP = BM * BN * 2;
    static constexpr uint32_t offQ = 0;
    static constexpr uint32_t offK = offQ + kTileQ;
    static constexpr uint32_t offV = offK + 2 * kTileKV;
    static constexpr uint32_t offP = offV + 2 * kTileKV;
    static constexpr uint32_t offBar = offP + kTileP;
    static constexpr uint32_t kBarBytes = 256;
    static constexpr uint32_t kUsed = offBar + kBarBytes;
    // 1 KB slack to align the base to 1024 bytes; d=64 pads to keep one CTA per SM
    // (each CTA takes all 512 tensor-memory columns).
    static constexpr uint32_t kAlloc = (kUsed + 1024) > 120u * 1024u ? (kUsed + 1024) : 120u * 1024u;
};

enum BarIdx {
    B_Q_FULL = 0,
    B_K_FULL = 1,   // +stage
    B_K_EMPTY = 3,  // +stage
    B_V_FULL = 5,   // +stage
    B_V_EMPTY = 7,  // +stage
    B_S_FULL = 9,   // +buffer
    B_S_EMPTY = 11, // +buffer
    B_P_FULL = 13,
    B_O_DONE = 14,
    B_MMA_DONE = 15,
    B_COUNT = 16
};

struct Shared {
    volatile int abort;
    uint32_t tmem_base;
};

__device__ __forceinline__ bool error_word_set() {
    return *reinterpret_cast<volatile unsigned int*>(&g_uly_error_word) != 0u;
}

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA abort flag) when
// the time limit passes, the CTA is aborting, or another CTA reported an error.
__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Shared* sh) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (sh->abort) return false;
        if ((it & 63u) == 0u) {
            if (error_word_set()) {
                sh->abort = 1;
                return false;
            }
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicOr(&g_uly_error_word, kErrTimeout);
                sh->abort = 1;
                return false;
            }
        }
    }
}

// Warp-uniform version for warps whose next step is a .sync.aligned tcgen05 collective.
__device__ __forceinline__ bool wait_phase_warp(uint64_t* bar, uint32_t parity, Shared* sh) {
    const bool ok = wait_phase(bar, parity, sh);
    return __all_sync(0xffffffffu, ok);
}

struct TileCoord {
    int map;  // index into the map arrays
    int row;  // token coordinate inside that map
};

__device__ __forceinline__ TileCoord tile_coord(const TcParams& p, int rank, int t0) {
    TileCoord c;
    c.map = rank + t0 / p.rows_per_map;
    c.row = t0 % p.rows_per_map;
    return c;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
    using L = Smem<D>;
    constexpr int KSTEPS_QK = D / 16;  // MMA K-steps for S = Q K^T
    constexpr int KSTEPS_PV = BN / 16; // MMA K-steps for O += P V
    constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, D, true);
    constexpr uint32_t kHalfQ = BM * 128;  // bytes of one 64-column slab of a 128-row tile
    constexpr uint32_t kHalfKV = BN * 128;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
    Shared* sh = reinterpret_cast<Shared*>(smem + L::offBar + B_COUNT * sizeof(uint64_t));
    const uint32_t sbase = smem_addr(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- block -> (rank, batch, kv head, query tile, head within group); heavy tiles first
    int bid = blockIdx.x;
    const int hg = bid % p.g;
    bid /= p.g;
    const int qt = p.n_qtiles - 1 - (bid % p.n_qtiles);
    bid /= p.n_qtiles;
    const int kv_heads = p.heads / p.g;
    const int kvh = bid % kv_heads;
    bid /= kv_heads;
    const int bb = bid % p.b;
    const int rank = bid / p.b;
    const int head = kvh * p.g + hg;
    const int q0 = qt * BM;
    const int n_kv = p.causal ? (qt + 1) : (p.s + BN - 1) / BN;

    if (threadIdx.x == 0) {
        sh->abort = error_word_set() ? 1 : 0;
        for (int i = 0; i < B_COUNT; ++i) {
            // the four softmax warps arrive once each on S_EMPTY and P_FULL
            const bool per_warp = i == B_S_EMPTY || i == B_S_EMPTY + 1 || i == B_P_FULL;
            mbar_init(&bars[i], per_warp ? 4u : 1u);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    if (sh->abort) return;  // an earlier CTA failed: nothing allocated yet, leave at once

    if (warp == 1) {
        tmem_alloc(&sh->tmem_base, kTmemCols);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    const uint32_t tS[2] = {tmem, tmem + 128u};
    const uint32_t tO = tmem + 256u;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const TileCoord qc = tile_coord(p, rank, q0);
            tma_prefetch_desc(&p.mq[qc.map]);
            mbar_arrive_expect_tx(&bars[B_Q_FULL], L::kTileQ);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(sbase + L::offQ + c * kHalfQ, &p.mq[qc.map], &bars[B_Q_FULL], c * 64, head, qc.row, bb);
            int issued_k[2] = {0, 0}, issued_v[2] = {0, 0};
            bool ok = true;
            for (int j = 0; j < n_kv && ok; ++j) {
                const int st = j & 1;
                const uint32_t ph = ((j >> 1) & 1) ^ 1;
                const TileCoord kc = tile_coord(p, rank, j * BN);
                ok = wait_phase(&bars[B_K_EMPTY + st], ph, sh);
                if (!ok) break;
                mbar_arrive_expect_tx(&bars[B_K_FULL + st], L::kTileKV);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(sbase + L::offK + st * L::kTileKV + c * kHalfKV, &p.mk[kc.map], &bars[B_K_FULL + st],
                                c * 64, kvh, kc.row, bb);
                ++issued_k[st];
                ok = wait_phase(&bars[B_V_EMPTY + st], ph, sh);
                if (!ok) break;
                mbar_arrive_expect_tx(&bars[B_V_FULL + st], L::kTileKV);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(sbase + L::offV + st * L::kTileKV + c * kHalfKV, &p.mv[kc.map], &bars[B_V_FULL + st],
                                c * 64, kvh, kc.row, bb);
                ++issued_v[st];
            }
            if (!ok) {
                // drain: every copy issued must land before shared memory goes away
                const uint64_t t0 = global_timer_ns();
                for (int st = 0; st < 2; ++st) {
                    if (issued_k[st])
                        while (!mbar_try_wait(&bars[B_K_FULL + st], ((issued_k[st] - 1) & 1)) &&
                               global_timer_ns() - t0 < kWaitLimitNs) {
                        }
                    if (issued_v[st])
                        while (!mbar_try_wait(&bars[B_V_FULL + st], ((issued_v[st] - 1) & 1)) &&
                               global_timer_ns() - t0 < kWaitLimitNs) {
                        }
                }
                const uint64_t t1 = global_timer_ns();
                while (!mbar_try_wait(&bars[B_Q_FULL], 0) && global_timer_ns() - t1 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = wait_phase(&bars[B_Q_FULL], 0, sh);
            tc_fence_after();
            for (int j = 0; j <= n_kv && ok; ++j) {
                if (j < n_kv) {
                    const int st = j & 1;
                    ok = wait_phase(&bars[B_K_FULL + st], (j >> 1) & 1, sh);
                    if (ok) ok = wait_phase(&bars[B_S_EMPTY + st], ((j >> 1) & 1) ^ 1, sh);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < KSTEPS_QK; ++kk) {
                        const uint64_t da = smem_desc_sw128(sbase + L::offQ + (kk >> 2) * kHalfQ + (kk & 3) * 32, 16, 1024);
                        const uint64_t db = smem_desc_sw128(
                            sbase + L::offK + st * L::kTileKV + (kk >> 2) * kHalfKV + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ss(tS[st], da, db, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars[B_S_FULL + st]);
                    mma_commit(&bars[B_K_EMPTY + st]);
                }
                if (j >= 1) {
                    const int jp = j - 1;
                    const int st = jp & 1;
                    ok = wait_phase(&bars[B_P_FULL], jp & 1, sh);
                    if (ok) ok = wait_phase(&bars[B_V_FULL + st], (jp >> 1) & 1, sh);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < KSTEPS_PV; ++kk) {
                        const uint64_t da = smem_desc_sw128(sbase + L::offP + (kk >> 2) * kHalfQ + (kk & 3) * 32, 16, 1024);
                        // V is [keys][d] with d contiguous: MN-major B operand; 64-column slabs
                        // kHalfKV apart (leading offset), 8-key groups 1024 bytes apart (stride).
                        const uint64_t db = smem_desc_sw128(sbase + L::offV + st * L::kTileKV + kk * 16 * 128, kHalfKV, 1024);
                        mma_bf16_ss(tO, da, db, kIdescPV, (jp > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&bars[B_O_DONE]);
                    mma_commit(&bars[B_V_EMPTY + st]);
                }
            }
            // every MMA issued above completes before tensor memory is released
            mma_commit(&bars[B_MMA_DONE]);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&bars[B_MMA_DONE], 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int sub = warp & 3;          // tensor-memory lane quarter this warp may access
        const int row = sub * 32 + lane;   // query row within the tile
        const int qrow = q0 + row;         // global query position
        const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
        uint8_t* sP = smem + L::offP;
        float m_ref = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            ok = wait_phase_warp(&bars[B_S_FULL + sb], (j >> 1) & 1, sh);
            if (!ok) break;
            tc_fence_after();
            // pass 1: row maximum of the (masked) scores, 32 columns at a time
            const int k0 = j * BN;
            const bool need_mask = (p.causal && k0 + BN - 1 > q0) || k0 + BN > p.s;
            const int lim = need_mask ? min(p.s - k0, p.causal ? qrow - k0 + 1 : BN) : BN;  // visible columns
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tS[sb] + lane_off + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (c * 32 + e < lim) mx = fmaxf(mx, __uint_as_float(r[e]));
            }
            const float mx2 = mx * p.scale_log2;
            float m_new = m_ref;
            if (j == 0 || mx2 > m_ref + 8.0f) m_new = mx2;
            if (m_new == -INFINITY) m_new = 0.f;  // row with nothing visible yet (padding rows only)
            const float alpha = (j == 0) ? 0.f : ex2_approx(m_ref - m_new);
            // pass 2: P = exp2(S * log2(e)/sqrt(d) - m), row sum, packed to bf16 pairs
            float rsum = 0.f;
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tS[sb] + lane_off + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float x0 = (c * 32 + e < lim) ? __uint_as_float(r[e]) : -INFINITY;
                    const float x1 = (c * 32 + e + 1 < lim) ? __uint_as_float(r[e + 1]) : -INFINITY;
                    const float e0 = ex2_approx(fmaf(x0, p.scale_log2, -m_new));
                    const float e1 = ex2_approx(fmaf(x1, p.scale_log2, -m_new));
                    rsum += e0 + e1;
                    pk[(c * 32 + e) / 2] = pack_bf16x2(e0, e1);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_S_EMPTY + sb]);
            if (j >= 1) {
                // P_{j-1} V_{j-1} done: the P buffer is free and O holds the sum through j-1
                ok = wait_phase_warp(&bars[B_O_DONE], (j - 1) & 1, sh);
                if (!ok) break;
                tc_fence_after();
                const bool rescale = m_new != m_ref;
                if (__any_sync(0xffffffffu, rescale)) {
                    const float f = rescale ? alpha : 1.0f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tO + lane_off + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                        tmem_st32(tO + lane_off + c * 32, r);
                    }
                    tmem_wait_st();
                }
            }
            // P row -> shared memory, K-major 128B-swizzled layout (two 64-key slabs)
#pragma unroll
            for (int c16 = 0; c16 < BN / 8; ++c16) {
                const uint4 w = make_uint4(pk[c16 * 4 + 0], pk[c16 * 4 + 1], pk[c16 * 4 + 2], pk[c16 * 4 + 3]);
                const uint32_t off = (c16 >> 3) * kHalfQ + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
                *reinterpret_cast<uint4*>(sP + off) = w;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_P_FULL]);
            l_sum = (j == 0) ? rsum : l_sum * alpha + rsum;
            m_ref = m_new;
        }
        if (ok) ok = wait_phase_warp(&bars[B_O_DONE], (n_kv - 1) & 1, sh);
        if (ok) {
            tc_fence_after();
            // epilogue: O / l -> bf16 -> this warp's 32 rows of the staging tile (Q's slot,
            // free since the last S MMA completed) -> TMA store of a 32-row box per slab
            const float inv = l_sum > 0.f ? 1.0f / l_sum : 0.f;
            uint8_t* stage = smem + L::offQ;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + lane_off + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * inv, __uint_as_float(r[q4 * 8 + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * inv, __uint_as_float(r[q4 * 8 + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * inv, __uint_as_float(r[q4 * 8 + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * inv, __uint_as_float(r[q4 * 8 + 7]) * inv);
                    const int col = c * 32 + q4 * 8;  // first of 8 output columns
                    const uint32_t off = (col >> 6) * kHalfQ + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4);
                    *reinterpret_cast<uint4*>(stage + off) = w;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && q0 + sub * 32 < p.s) {  // boxes wholly past the end are skipped
                const TileCoord oc = tile_coord(p, rank, q0);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_store_4d(&p.mo[oc.map], sbase + L::offQ + c * kHalfQ + sub * 32 * 128, c * 64, head,
                                 oc.row + sub * 32, bb);
                tma_store_commit_and_drain();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// 4-D map over a [b][rows][heads][d] bf16 buffer; box = 64 columns x 1 head x box_rows.
bool make_map(CUtensorMap* m, const void* base, int b, int rows, int heads, int d, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows, (cuuint64_t)b};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2, (cuuint64_t)rows * heads * d * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const TcParams& prm, long long nblocks, cudaStream_t stream) {
    const uint32_t smem = Smem<D>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attn_tc_kernel<D><<<(unsigned)nblocks, kThreads, smem, stream>>>(prm);
    return cudaGetLastError();
}

}  // namespace

int tc_attention_supported(int d) { return d == 64 || d == 128; }

cudaError_t launch_attention_tc(int P, int b, int s, int h_q, int h_kv, int d, int causal, int fused,
                                const AttnPtrs& ptrs, cudaStream_t stream, int* unsupported) {
    *unsupported = 0;
    if (!tc_attention_supported(d) || (fused && (P > kMaxMaps || (s / P) % BM != 0))) {
        *unsupported = 1;
        return cudaSuccess;
    }
    TcParams* prm = new TcParams;
    memset(prm, 0, sizeof(TcParams));
    prm->s = s;
    prm->n_qtiles = (s + BM - 1) / BM;
    prm->g = h_q / h_kv;
    prm->b = b;
    prm->causal = causal ? 1 : 0;
    prm->scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    cudaError_t err = cudaSuccess;
    if (fused) {
        const int S = s / P;
        prm->rows_per_map = S;
        prm->heads = h_q;
        prm->nranks = 1;
        for (int j = 0; j < P && err == cudaSuccess; ++j) {
            if (!make_map(&prm->mq[j], ptrs.q[j], b, S, h_q, d, BM) ||
                !make_map(&prm->mk[j], ptrs.k[j], b, S, h_kv, d, BN) ||
                !make_map(&prm->mv[j], ptrs.v[j], b, S, h_kv, d, BN) ||
                !make_map(&prm->mo[j], ptrs.o[j], b, S, h_q, d, 32))
                err = cudaErrorInvalidValue;
        }
        if (err == cudaSuccess) {
            const long long nblocks = (long long)b * h_q * prm->n_qtiles;
            err = d == 64 ? launch_d<64>(*prm, nblocks, stream) : launch_d<128>(*prm, nblocks, stream);
        }
    } else {
        const int Hq = h_q / P, Hk = h_kv / P;
        prm->rows_per_map = s;
        prm->heads = Hq;
        for (int r0 = 0; r0 < P && err == cudaSuccess; r0 += kMaxMaps) {
            const int nr = (P - r0) < kMaxMaps ? (P - r0) : kMaxMaps;
            prm->nranks = nr;
            for (int i = 0; i < nr && err == cudaSuccess; ++i) {
                const int r = r0 + i;
                if (!make_map(&prm->mq[i], ptrs.q[r], b, s, Hq, d, BM) ||
                    !make_map(&prm->mk[i], ptrs.k[r], b, s, Hk, d, BN) ||
                    !make_map(&prm->mv[i], ptrs.v[r], b, s, Hk, d, BN) ||
                    !make_map(&prm->mo[i], ptrs.o[r], b, s, Hq, d, 32))
                    err = cudaErrorInvalidValue;
            }
            if (err != cudaSuccess) break;
            const long long nblocks = (long long)nr * b * Hq * prm->n_qtiles;
            err = d == 64 ? launch_d<64>(*prm, nblocks, stream) : launch_d<128>(*prm, nblocks, stream);
        }
    }
    delete prm;
    return err;
}

cudaError_t read_device_error(unsigned int* value, int clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_uly_error_word, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_uly_error_word, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace uly
