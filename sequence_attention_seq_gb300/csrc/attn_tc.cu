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
// Work unit: one CTA owns two consecutive 128-row query tiles (Q0, Q1) of one (rank,
// batch, head) and streams 128-key K/V tiles through a 4-slot shared-memory ring; each
// K/V tile serves both query tiles.  Head dim d in {64, 128}.  10 warps:
//   warps 0-3   softmax for Q0, warps 4-7 softmax for Q1: one thread per query row
//               (warp w may access tensor-memory lanes 32*(w%4)..+31)
//   warp 8      TMA producer: Q0, Q1 once, then K_j, V_j into the ring
//   warp 9      allocates tensor memory; one thread issues every tcgen05.mma
// Tensor memory (512 columns): S0 | S1 | O0 | O1, 128 columns each.  The softmax writes
// P_k = exp2(S_k*c - m) as bf16 pairs back over the first 64 columns of S_k, and
// O_k += P_k V_j reads P_k straight from tensor memory.
// MMA order per key tile j: PV0(j), S0(j+1), PV1(j), S1(j+1).  The tensor pipe executes
// MMAs in issue order and a commit covers every earlier MMA, so when a softmax group sees
// S_k(j+1) complete, PV_k(j) is complete too: O_k can be rescaled right away, and S_k(j+1)
// never overwrites P_k(j) early.  While one softmax group works on its tile, the tensor
// pipe runs the other group's PV and S (measured faster than PV0 PV1 S0 S1, whose shorter
// overlap window costs more than the pipe drain between PV_k(j) and S_k(j+1) it avoids).
// The reference maximum m is only raised when a row maximum exceeds it by more than 8
// (a factor 256), so O is rarely rescaled; P entries stay below 256, exact enough in
// bf16, and the final O / l is unchanged mathematically.  After a row's first key tile
// the maximum itself is rarely needed: the row's terms are formed against m first, and a
// sum of at most 256 shows that none exceeds 2^8.
//
// Fused mode ("DeepSpeed-Ulysses 深度解析", steps 3 and 5; "02 · DeepSpeed-Ulysses",
// section 3, whose comparison table notes that the two exchanges lend themselves to being
// combined): the tiles of tokens [t0, t0+128) come
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

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per tile
constexpr int kSlots = 4; // K/V ring slots
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kMaxMaps = 16;      // maps per launch: unfused rank groups, the backward
constexpr int kMaxMapsWide = 64;  // fused and two-level forwards over more than kMaxMaps ranks
constexpr int kMaxMapsBwdWide = 48;  // fused and two-level backwards (four maps per rank)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr unsigned int kErrTimeout = 1u;

// NM maps of each kind: kMaxMaps, or kMaxMapsWide for more ranks (about 25 KB of kernel
// parameters, so the common launches keep the small block).
template <int NM>
struct TcParamsT {
    static constexpr int kMaps = NM;
    CUtensorMap mq[NM];
    CUtensorMap mk[NM];
    CUtensorMap mv[NM];
    uint8_t* optr[NM];  // output buffers (same indexing as the maps): [b][rows][heads][d] bf16
    float* lse[NM];     // optional per-row log-sum-exp (natural log), per head rank [b][lse_heads][s]
    int lse_heads;            // query heads per head rank: the heads of one lse array
    int s;             // sequence length
    int rows_per_map;  // tokens held by one map: s/P when fused, s/Pr for the two-level forward, s otherwise
    int map_stride;    // map index step from one token block to the next (Pu for the two-level forward, else 1)
    int n_qtiles;      // ceil(s / BM)
    int n_pairs;       // ceil(n_qtiles / 2)
    int heads;         // query heads per map group: h_q (fused) or h_q/P (per rank)
    int g;             // query heads per K/V head
    int b;
    int nranks;        // rank groups in this launch (fused: 1)
    int n_items;       // query-tile pairs in this launch: nranks * b * heads * n_pairs
    int band_units;    // causal: (rank, batch, K/V head) units per band (see decode_item)
    int causal;
    float scale_log2;  // log2(e) / sqrt(d)
};
using TcParams = TcParamsT<kMaxMaps>;

template <int D>
struct Smem {
    static constexpr uint32_t kTile = BM * D * 2;  // bytes of one Q, K or V tile
    static constexpr uint32_t offQ = 0;            // Q0, Q1
    static constexpr uint32_t offKV = 2 * kTile;   // ring of kSlots tiles
    static constexpr uint32_t offBar = offKV + kSlots * kTile;
    static constexpr uint32_t kBarBytes = 256;
    static constexpr uint32_t kUsed = offBar + kBarBytes;
    // 1 KB slack to align the base to 1024 bytes; d=64 pads so that one CTA (which takes
    // all 512 tensor-memory columns) fills an SM.
    static constexpr uint32_t kAlloc = (kUsed + 1024) > 120u * 1024u ? (kUsed + 1024) : 120u * 1024u;
};

enum BarIdx {
    B_Q_FULL = 0,                       // +tile (2)
    B_KV_FULL = 2,                      // +slot (4)
    B_KV_EMPTY = B_KV_FULL + kSlots,    // +slot (4)
    B_S_FULL = B_KV_EMPTY + kSlots,     // +tile (2)
    B_P_FULL = B_S_FULL + 2,            // +tile (2), 4 arrivals each
    B_O_FINAL = B_P_FULL + 2,           // +tile (2)
    B_Q_EMPTY = B_O_FINAL + 2,          // +tile (2): the last S MMA of an item has read Q_t
    B_O_EMPTY = B_Q_EMPTY + 2,          // +tile (2), 4 arrivals each: the epilogue has read O_t
    B_MMA_DONE = B_O_EMPTY + 2,
    B_COUNT = B_MMA_DONE + 1
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
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Shared* sh,
                                           uint64_t limit_ns = kWaitLimitNs) {
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
            if (global_timer_ns() - t0 > limit_ns) {
                atomicOr(&g_uly_error_word, kErrTimeout);
                sh->abort = 1;
                return false;
            }
        }
    }
}

// Self-test of the wait above: one warp waits on a barrier that nothing ever completes, with
// the given limit, exactly as the attention kernels' waits do; the wait gives up, raises the
// timeout bit of the device error word and the kernel returns.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ Shared sh;
    if (threadIdx.x == 0) {
        sh.abort = 0;
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    wait_phase(&bar, 0, &sh, limit_ns);  // no arrival: phase 0 never completes
    __syncthreads();
}

// Warp-uniform version for warps whose next step is a .sync.aligned tcgen05 collective.
__device__ __forceinline__ bool wait_phase_warp(uint64_t* bar, uint32_t parity, Shared* sh) {
    const bool ok = wait_phase(bar, parity, sh);
    return __all_sync(0xffffffffu, ok);
}

// Bounded drain wait used on the way out (no abort check: the copies/MMAs must land).
__device__ __forceinline__ void drain_phase(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < kWaitLimitNs) {
    }
}

struct TileCoord {
    int map;  // index into the map arrays
    int row;  // token coordinate inside that map
};

// Token t0 of the global sequence, for the unit `rank` of a work item: the map (buffer)
// holding it and its row there.  Unfused: map = rank, row = t0.  Fused: rank = 0 and the
// map is the seq-layout rank t0 / (s/P).  Two-level (Ulysses x Ring): rank = u and the map
// is ring group t0 / (s/Pr)'s rank u, i.e. the K/V blocks of the other ring groups are read
// where those ranks hold them.
template <class PR>
__device__ __forceinline__ TileCoord tile_coord(const PR& p, int rank, int t0) {
    TileCoord c;
    c.map = rank + (t0 / p.rows_per_map) * p.map_stride;
    c.row = t0 % p.rows_per_map;
    return c;
}

// Work item w (a query-tile pair) -> coordinates.  Every role of a CTA walks the same
// sequence.  Causal: the (rank, batch, K/V head) units form bands of band_units units whose
// K and V fit in L2 together; bands run one after another, and inside a band the pair
// index is slowest and descending, so the band's items are sorted heaviest first and the
// snake assignment balances the CTAs while all of them stream the same few heads' K/V.
// Non-causal (all items equal): the pairs of one head are adjacent, so concurrent CTAs
// share K/V in L2.  In both, the query heads that share a K/V head are adjacent.
struct Item {
    int rank, bb, kvh, head, qt0, n0, n1;
};

template <class PR>
__device__ __forceinline__ Item decode_item(const PR& p, int w) {
    Item it;
    const int kv_heads = p.heads / p.g;
    const int hg = w % p.g;
    w /= p.g;
    int pair;
    if (p.causal) {
        const int units = p.nranks * p.b * kv_heads;
        const int per_band = p.band_units * p.n_pairs;
        const int band = w / per_band;
        const int base = band * p.band_units;
        const int in_band = units - base < p.band_units ? units - base : p.band_units;
        const int r = w - band * per_band;
        int u = base + r % in_band;
        pair = p.n_pairs - 1 - r / in_band;
        it.kvh = u % kv_heads;
        u /= kv_heads;
        it.bb = u % p.b;
        it.rank = u / p.b;
    } else {
        pair = w % p.n_pairs;
        w /= p.n_pairs;
        it.kvh = w % kv_heads;
        w /= kv_heads;
        it.bb = w % p.b;
        it.rank = w / p.b;
    }
    it.head = it.kvh * p.g + hg;
    it.qt0 = 2 * pair;
    const bool has_q1 = it.qt0 + 1 < p.n_qtiles;
    const int n_kv_all = (p.s + BN - 1) / BN;
    it.n0 = p.causal ? it.qt0 + 1 : n_kv_all;  // key tiles query tile 0 needs
    it.n1 = has_q1 ? (p.causal ? it.qt0 + 2 : n_kv_all) : 0;
    return it;
}

// The k-th item of CTA c: rounds of gridDim.x items, alternating direction (snake), so
// the heavy-first order spreads evenly; -1 when the CTA has no k-th item.
template <class PR>
__device__ __forceinline__ int item_index(const PR& p, int k) {
    const int G = gridDim.x, c = blockIdx.x;
    const int w = k * G + ((k & 1) ? G - 1 - c : c);
    return w < p.n_items ? w : -1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Columns >= lim of a score row -> -inf (diagonal and ragged tiles only).
__device__ __forceinline__ void mask_row(uint32_t (&r)[BN], int lim) {
#pragma unroll
    for (int e = 0; e < BN; ++e)
        if (e >= lim) r[e] = 0xff800000u;
}

// Row maximum of the 128 score columns.
__device__ __forceinline__ float row_max(const uint32_t (&r)[BN]) {
    float acc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int e = 0; e < BN; e += 8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = __uint_as_float(r[e + u]);
        acc[(e >> 3) & 3] = fmax3(acc[(e >> 3) & 3], fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], fmax3(x[5], x[6], x[7])));
    }
    return fmax3(acc[0], acc[1], fmax3(acc[2], acc[3], -INFINITY));
}

// P = exp2(S*scale - m) for columns [32c, 32c+32), packed into 16 bf16 pairs at pk[0..15];
// returns their sum.
__device__ __forceinline__ float chunk_exp(const uint32_t (&r)[BN], int c, float scale, float neg_m, uint32_t* pk) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const int col = c * 32 + e;
        const float x0 = __uint_as_float(r[col]), x1 = __uint_as_float(r[col + 1]);
        float a0, a1;
        ffma2(a0, a1, x0, x1, scale, scale, neg_m, neg_m);  // S*scale - m for two columns at once
        const float e0 = ex2_approx(a0);
        const float e1 = ex2_approx(a1);
        fadd2(s0, s1, s0, s1, e0, e1);
        pk[e >> 1] = pack_bf16x2(e0, e1);
    }
    return s0 + s1;
}

template <int D, int NM>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcParamsT<NM> p) {
    using L = Smem<D>;
    constexpr int KSTEPS_QK = D / 16;  // MMA K-steps for S = Q K^T
    constexpr int KSTEPS_PV = BN / 16; // MMA K-steps for O += P V
    constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, D, true);
    constexpr uint32_t kSlab = BM * 128;  // bytes of one 64-column slab of a 128-row tile

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
    Shared* sh = reinterpret_cast<Shared*>(smem + L::offBar + B_COUNT * sizeof(uint64_t));
    const uint32_t sbase = smem_addr(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        sh->abort = error_word_set() ? 1 : 0;
        for (int i = 0; i < B_COUNT; ++i) {
            const bool per_warp = i == B_P_FULL || i == B_P_FULL + 1 || i == B_O_EMPTY || i == B_O_EMPTY + 1;
            mbar_init(&bars[i], per_warp ? 4u : 1u);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    if (sh->abort) return;  // an earlier CTA failed: nothing allocated yet, leave at once

    if (warp == kMmaWarp) tmem_alloc(&sh->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        // Whole warp, warp-uniform operands, one elected lane issues.  Q_t of the next item
        // is loaded as soon as the last S MMA of the current item has read Q_t.
        int n = 0;                   // ring loads issued so far (slot n % kSlots)
        int quse[2] = {0, 0};        // Q_t loads issued so far
        bool ok = true;
        // K/V tiles are read by every item of their head: kept in L2 ahead of the Q tiles,
        // which one item reads once
        const uint64_t keep = l2_policy_evict_last(), once = l2_policy_evict_first();
        for (int k = 0; ok; ++k) {
            const int w = item_index(p, k);
            if (w < 0) break;
            const Item it = decode_item(p, w);
            for (int t = 0; t < 2 && ok; ++t) {
                if ((t ? it.n1 : it.n0) == 0) continue;
                if (quse[t] > 0) ok = wait_phase_warp(&bars[B_Q_EMPTY + t], (quse[t] - 1) & 1, sh);
                if (!ok) break;
                const TileCoord qc = tile_coord(p, it.rank, (it.qt0 + t) * BM);
                mbar_arrive_expect_tx_warp(&bars[B_Q_FULL + t], L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_warp_hint(sbase + L::offQ + t * L::kTile + c * kSlab, &p.mq[qc.map],
                                          &bars[B_Q_FULL + t], c * 64, it.head, qc.row, it.bb, once);
                ++quse[t];
            }
            const int n_max = it.n0 > it.n1 ? it.n0 : it.n1;
            for (int e = 0; e < 2 * n_max && ok; ++e, ++n) {
                const int j = e >> 1, slot = n % kSlots;
                ok = wait_phase_warp(&bars[B_KV_EMPTY + slot], ((n / kSlots) & 1) ^ 1, sh);
                if (!ok) break;
                const TileCoord kc = tile_coord(p, it.rank, j * BN);
                const CUtensorMap* map = (e & 1) ? &p.mv[kc.map] : &p.mk[kc.map];
                mbar_arrive_expect_tx_warp(&bars[B_KV_FULL + slot], L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_warp_hint(sbase + L::offKV + slot * L::kTile + c * kSlab, map,
                                          &bars[B_KV_FULL + slot], c * 64, it.kvh, kc.row, it.bb, keep);
            }
        }
        if (!ok) {  // every copy issued must land before shared memory goes away
            for (int slot = 0; slot < kSlots; ++slot) {
                const int cnt = (n - slot + kSlots - 1) / kSlots;  // loads that went to this slot
                if (cnt > 0) drain_phase(&bars[B_KV_FULL + slot], (cnt - 1) & 1);
            }
            for (int t = 0; t < 2; ++t)
                if (quse[t] > 0) drain_phase(&bars[B_Q_FULL + t], (quse[t] - 1) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Whole warp, warp-uniform operands; one elected lane issues every tcgen05.mma and
        // tcgen05.commit (so all commits track that lane's MMAs).
        auto kv_slot = [](int n) { return n % kSlots; };
        auto kv_par = [](int n) { return (uint32_t)((n / kSlots) & 1); };
        const uint64_t dq0 = smem_desc_sw128(sbase + L::offQ, 16, 1024);
        const uint64_t dkv0 = smem_desc_sw128(sbase + L::offKV, 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(sbase + L::offKV, kSlab, 1024);
        int n = 0;                 // ring position of the current item's K_0
        int use[2] = {0, 0};       // items so far in which query tile t took part
        int sn[2] = {0, 0};        // S_t tiles computed so far (S_FULL / P_FULL phases)
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int w = item_index(p, k);
            if (w < 0) break;
            const Item it = decode_item(p, w);
            const int nt0 = it.n0, nt1 = it.n1;
            const int n_max = nt0 > nt1 ? nt0 : nt1;
            auto nt = [&](int t) { return t ? nt1 : nt0; };
            auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T
                const uint64_t qd = dq0 + ((t * L::kTile) >> 4);
                const uint64_t kd = dkv0 + ((kv_slot(n + 2 * j) * L::kTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < KSTEPS_QK; ++kk) {
                    const uint32_t off = ((kk >> 2) * kSlab + (kk & 3) * 32) >> 4;
                    mma_bf16_ss_warp(tmem + 128u * t, qd + off, kd + off, kIdescQK, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int j) {  // O_t += P_t V_j, P_t from tensor memory
                // V is [keys][d], d contiguous: MN-major B; 64-column slabs kSlab apart (leading
                // offset), 8-key groups 1024 bytes apart (stride offset)
                const uint64_t vd = dv0 + ((kv_slot(n + 2 * j + 1) * L::kTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < KSTEPS_PV; ++kk)
                    mma_bf16_ts_warp(tmem + 256u + 128u * t, tmem + 128u * t + kk * 8, vd + ((kk * 16 * 128) >> 4),
                                     kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
            };
            for (int t = 0; t < 2 && ok; ++t)
                if (nt(t) > 0) ok = wait_phase_warp(&bars[B_Q_FULL + t], use[t] & 1, sh);
            if (ok) ok = wait_phase_warp(&bars[B_KV_FULL + kv_slot(n)], kv_par(n), sh);
            if (!ok) break;
            tc_fence_after();
            for (int t = 0; t < 2; ++t)
                if (nt(t) > 0) {
                    issue_s(t, 0);
                    mma_commit_warp(&bars[B_S_FULL + t]);
                    if (nt(t) == 1) mma_commit_warp(&bars[B_Q_EMPTY + t]);
                }
            mma_commit_warp(&bars[B_KV_EMPTY + kv_slot(n)]);
            for (int j = 0; j < n_max && ok; ++j) {
                ok = wait_phase_warp(&bars[B_KV_FULL + kv_slot(n + 2 * j + 1)], kv_par(n + 2 * j + 1), sh);
                const bool next = j + 1 < n_max;
                bool k_next_ready = false;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= nt(t)) continue;
                    // PV_t(0) overwrites O_t: the previous item's epilogue must have read it
                    if (j == 0 && use[t] > 0) ok = wait_phase_warp(&bars[B_O_EMPTY + t], (use[t] - 1) & 1, sh);
                    if (ok) ok = wait_phase_warp(&bars[B_P_FULL + t], (sn[t] + j) & 1, sh);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(t, j);
                    if (j + 1 < nt(t)) {
                        if (!k_next_ready) {  // K_{j+1} is only needed from here on
                            ok = wait_phase_warp(&bars[B_KV_FULL + kv_slot(n + 2 * j + 2)], kv_par(n + 2 * j + 2), sh);
                            if (!ok) break;
                            k_next_ready = true;
                        }
                        tc_fence_after();
                        issue_s(t, j + 1);
                        mma_commit_warp(&bars[B_S_FULL + t]);
                        if (j + 2 == nt(t)) mma_commit_warp(&bars[B_Q_EMPTY + t]);  // last read of Q_t
                    } else {
                        mma_commit_warp(&bars[B_O_FINAL + t]);
                    }
                }
                if (!ok) break;
                mma_commit_warp(&bars[B_KV_EMPTY + kv_slot(n + 2 * j + 1)]);
                if (next) mma_commit_warp(&bars[B_KV_EMPTY + kv_slot(n + 2 * j + 2)]);
            }
            for (int t = 0; t < 2; ++t)
                if (nt(t) > 0) {
                    sn[t] += nt(t);
                    ++use[t];
                }
            n += 2 * n_max;
        }
        // every MMA issued above completes before tensor memory is released
        mma_commit_warp(&bars[B_MMA_DONE]);
        drain_phase(&bars[B_MMA_DONE], 0);
    } else {
        // ------------------------------------------------------------ softmax warps
        const int t = warp >> 2;           // query tile of this group
        const int sub = warp & 3;          // tensor-memory lane quarter this warp may access
        const int row = sub * 32 + lane;   // query row within the tile
        const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
        const uint32_t tS = tmem + 128u * t + lane_off;
        const uint32_t tO = tmem + 256u + 128u * t + lane_off;
        const float scale = p.scale_log2;
        int use = 0, sn = 0;               // items and S tiles this group has processed
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int w = item_index(p, k);
            if (w < 0) break;
            const Item it = decode_item(p, w);
            const int nkv = t == 0 ? it.n0 : it.n1;
            if (nkv == 0) continue;        // this item has no second query tile
            const int q0 = (it.qt0 + t) * BM;
            const int qrow = q0 + row;     // global query position
            float m_ref = -INFINITY, l_sum = 0.f;
            for (int j = 0; j < nkv; ++j) {
                ok = wait_phase_warp(&bars[B_S_FULL + t], (sn + j) & 1, sh);
                if (!ok) break;
                tc_fence_after();
                const int k0 = j * BN;
                const bool need_mask = (p.causal && k0 + BN - 1 > q0) || k0 + BN > p.s;
                const int lim = min(p.s - k0, p.causal ? qrow - k0 + 1 : BN);  // visible columns of this row
                // The whole S row in one tensor-memory load, then the exponentials.  The first key
                // tile of a row sets the reference m from the row maximum.  Later tiles first form
                // their terms against the current reference, in registers: a row whose terms sum
                // to at most 256 has no term above 2^8, so its maximum exceeds m by at most 8 and
                // m stands (the rule above).  Only when some row's sum is larger does the warp
                // reload S (nothing has been stored over it yet) and take the maximum; rows whose
                // maximum exceeds m by more than 8 raise m, and the terms are formed again.
                uint32_t sr[BN];
                tmem_ld128(tS, sr);
                tmem_wait_ld();
                if (need_mask) mask_row(sr, lim);
                float m_new = m_ref, rsum = 0.f;
                do {
                    if (j > 0) {
                        uint32_t pk[BN / 2];
#pragma unroll
                        for (int c = 0; c < BN / 32; ++c) rsum += chunk_exp(sr, c, scale, -m_ref, pk + 16 * c);
                        const bool big = !(rsum <= 256.0f);  // also for an infinite sum
                        if (!__any_sync(0xffffffffu, big)) {
#pragma unroll
                            for (int c = 0; c < BN / 32; ++c)
                                tmem_st16(tS + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16 * c));
                            break;
                        }
                        tmem_ld128(tS, sr);
                        tmem_wait_ld();
                        if (need_mask) mask_row(sr, lim);
                        const float mx2 = row_max(sr) * scale;
                        if (big && mx2 > m_ref + 8.0f) m_new = mx2;
                    } else {
                        m_new = row_max(sr) * scale;
                        if (m_new == -INFINITY) m_new = 0.f;  // a row with nothing visible yet (padding rows only)
                    }
                    rsum = 0.f;
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t pk[16];
                        rsum += chunk_exp(sr, c, scale, -m_new, pk);
                        tmem_st16(tS + c * 16, pk);
                    }
                } while (0);
                const float alpha = (j == 0) ? 0.f : ex2_approx(m_ref - m_new);
                // O_t already holds P_t(j-1) V_{j-1} (S_t(j) was issued after it): rescale in place
                if (j > 0 && __any_sync(0xffffffffu, m_new != m_ref)) {
                    const float f = m_new != m_ref ? alpha : 1.0f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                        tmem_st32(tO + c * 32, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_P_FULL + t]);
                l_sum = (j == 0) ? rsum : l_sum * alpha + rsum;
                m_ref = m_new;
            }
            if (ok) ok = wait_phase_warp(&bars[B_O_FINAL + t], use & 1, sh);
            if (!ok) break;
            tc_fence_after();
            // epilogue: O / l -> bf16, each thread stores its own row (16-byte stores), then
            // O_t is handed back to the MMA warp for the next item
            const float inv = l_sum > 0.f ? 1.0f / l_sum : 0.f;
            const TileCoord oc = tile_coord(p, it.rank, q0);
            const bool row_ok = qrow < p.s;
            uint8_t* orow = p.optr[oc.map] +
                            ((((size_t)it.bb * p.rows_per_map + oc.row + row) * p.heads + it.head) * D) * 2;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * inv, __uint_as_float(r[q4 * 8 + 1]) * inv);
                    v.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * inv, __uint_as_float(r[q4 * 8 + 3]) * inv);
                    v.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * inv, __uint_as_float(r[q4 * 8 + 5]) * inv);
                    v.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * inv, __uint_as_float(r[q4 * 8 + 7]) * inv);
                    if (row_ok) *reinterpret_cast<uint4*>(orow + (c * 32 + q4 * 8) * 2) = v;
                }
            }
            // log-sum-exp of the scaled scores, natural log, in the head rank's [b][h/P][s] array:
            // unfused, the item's rank is the head rank; fused, the head is global
            const int lr = it.rank + it.head / p.lse_heads, lh = it.head % p.lse_heads;
            if (p.lse[lr] && row_ok)
                p.lse[lr][((size_t)it.bb * p.lse_heads + lh) * p.s + qrow] =
                    (m_ref + log2f(l_sum)) * 0.6931471805599453f;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_O_EMPTY + t]);
            sn += nkv;
            ++use;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
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

// Causal band size.  When the K and V of every (rank, batch, K/V head) unit of the launch
// fit in L2 together, one band: the global heaviest-first order balances best.  Otherwise
// as many units as keep their K and V within about a third of the 129 MB L2 (at least one),
// so that all CTAs stream the same few heads' K/V and L2 serves the re-reads.
constexpr double kL2Bytes = 129.0 * 1024 * 1024;
constexpr double kBandBytes = 48.0 * 1024 * 1024;

int band_units_for(int s, int d, int units) {
    const double kv_bytes = 2.0 * s * d * 2;  // K and V of one unit, bf16
    if (kv_bytes * units <= kL2Bytes) return units;
    int bu = (int)(kBandBytes / kv_bytes);
    if (bu < 1) bu = 1;
    if (bu > units) bu = units;
    return bu;
}

template <int D, int NM>
cudaError_t launch_d(TcParamsT<NM>& prm, long long n_items, cudaStream_t stream) {
    const uint32_t smem = Smem<D>::kAlloc;
    cudaError_t e =
        cudaFuncSetAttribute(attn_tc_kernel<D, NM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM walks the items (each CTA fills an SM: smem and all TMEM)
    prm.n_items = (int)n_items;
    const long long grid = n_items < sms ? n_items : sms;
    attn_tc_kernel<D, NM><<<(unsigned)grid, kThreads, smem, stream>>>(prm);
    return cudaGetLastError();
}

#include "attn_bwd.cuh"

}  // namespace

int tc_attention_supported(int d) { return d == 64 || d == 128; }

namespace {

template <class PR>
void fill_common(PR* prm, int s, int b, int g, int causal, int d) {
    memset(prm, 0, sizeof(PR));
    prm->s = s;
    prm->map_stride = 1;
    prm->n_qtiles = (s + BM - 1) / BM;
    prm->n_pairs = (prm->n_qtiles + 1) / 2;
    prm->g = g;
    prm->b = b;
    prm->causal = causal ? 1 : 0;
    prm->scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
}

template <class PR>
cudaError_t launch_any_d(PR& prm, int d, long long n_items, cudaStream_t stream) {
    return d == 64 ? launch_d<64>(prm, n_items, stream) : launch_d<128>(prm, n_items, stream);
}

// The fused forward: one map per seq-layout rank buffer (NM >= P).
template <int NM>
cudaError_t launch_fused_fwd(int P, int b, int s, int h_q, int h_kv, int d, int causal, const AttnPtrs& ptrs,
                             bool want_lse, cudaStream_t stream) {
    TcParamsT<NM> prm_rec;
    TcParamsT<NM>* prm = &prm_rec;
    fill_common(prm, s, b, h_q / h_kv, causal, d);
    const int S = s / P;
    prm->rows_per_map = S;
    prm->heads = h_q;
    prm->lse_heads = h_q / P;  // the statistics go to the head ranks' arrays
    prm->nranks = 1;
    for (int j = 0; j < P; ++j) {
        if (!make_map(&prm->mq[j], ptrs.q[j], b, S, h_q, d, BM) || !make_map(&prm->mk[j], ptrs.k[j], b, S, h_kv, d, BN) ||
            !make_map(&prm->mv[j], ptrs.v[j], b, S, h_kv, d, BN))
            return cudaErrorInvalidValue;
        prm->optr[j] = static_cast<uint8_t*>(ptrs.o[j]);
        prm->lse[j] = want_lse ? ptrs.lse[j] : nullptr;
    }
    const long long n_items = (long long)b * h_q * prm->n_pairs;
    prm->band_units = band_units_for(s, d, b * h_kv);
    return launch_any_d(*prm, d, n_items, stream);
}

// The two-level forward: one map per rank's group head-layout buffer (NM >= Pu * Pr).
template <int NM>
cudaError_t launch_usp_fwd(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, int causal, const AttnPtrs& head,
                           cudaStream_t stream) {
    const int P = Pu * Pr, L = s / Pr;
    const int Hq = h_q / Pu, Hk = kv_heads_per_rank(Pu, h_kv);  // 1: a replicated K/V head
    TcParamsT<NM> prm_rec;
    TcParamsT<NM>* prm = &prm_rec;
    fill_common(prm, s, b, Hq / Hk, causal, d);
    prm->rows_per_map = L;
    prm->map_stride = Pu;
    prm->heads = Hq;
    prm->lse_heads = Hq;  // statistics (if asked for) per Ulysses unit over all s rows
    prm->nranks = Pu;
    for (int j = 0; j < P; ++j) {
        if (!make_map(&prm->mq[j], head.q[j], b, L, Hq, d, BM) || !make_map(&prm->mk[j], head.k[j], b, L, Hk, d, BN) ||
            !make_map(&prm->mv[j], head.v[j], b, L, Hk, d, BN))
            return cudaErrorInvalidValue;
        prm->optr[j] = static_cast<uint8_t*>(head.o[j]);
    }
    for (int u = 0; u < Pu; ++u) prm->lse[u] = head.lse[u];  // unit u's rows of every ring group
    const long long n_items = (long long)Pu * b * Hq * prm->n_pairs;
    prm->band_units = band_units_for(s, d, Pu * b * Hk);
    return launch_any_d(*prm, d, n_items, stream);
}

}  // namespace

cudaError_t launch_attention_tc(int P, int b, int s, int h_q, int h_kv, int d, int causal, int fused,
                                const AttnPtrs& ptrs, cudaStream_t stream, int* unsupported) {
    *unsupported = 0;
    const bool want_lse = ptrs.lse[0] != nullptr;
    if (!tc_attention_supported(d) || (fused && (P > kMaxMapsWide || (s / P) % BM != 0))) {
        *unsupported = 1;
        return cudaSuccess;
    }
    if (fused)
        return P <= kMaxMaps ? launch_fused_fwd<kMaxMaps>(P, b, s, h_q, h_kv, d, causal, ptrs, want_lse, stream)
                             : launch_fused_fwd<kMaxMapsWide>(P, b, s, h_q, h_kv, d, causal, ptrs, want_lse, stream);
    // unfused: the head ranks in groups of up to kMaxMaps per launch
    TcParams prm_rec;
    TcParams* prm = &prm_rec;
    const int Hq = h_q / P, Hk = kv_heads_per_rank(P, h_kv);
    fill_common(prm, s, b, Hq / Hk, causal, d);  // g within a rank (its K/V heads may be shared replicas)
    prm->rows_per_map = s;
    prm->heads = Hq;
    prm->lse_heads = Hq;
    cudaError_t err = cudaSuccess;
    for (int r0 = 0; r0 < P && err == cudaSuccess; r0 += kMaxMaps) {
        const int nr = (P - r0) < kMaxMaps ? (P - r0) : kMaxMaps;
        prm->nranks = nr;
        for (int i = 0; i < nr; ++i) {
            const int r = r0 + i;
            if (!make_map(&prm->mq[i], ptrs.q[r], b, s, Hq, d, BM) || !make_map(&prm->mk[i], ptrs.k[r], b, s, Hk, d, BN) ||
                !make_map(&prm->mv[i], ptrs.v[r], b, s, Hk, d, BN))
                return cudaErrorInvalidValue;
            prm->optr[i] = static_cast<uint8_t*>(ptrs.o[r]);
            prm->lse[i] = want_lse ? ptrs.lse[r] : nullptr;
        }
        const long long n_items = (long long)nr * b * Hq * prm->n_pairs;
        prm->band_units = band_units_for(s, d, nr * b * Hk);
        err = launch_any_d(*prm, d, n_items, stream);
    }
    return err;
}

cudaError_t launch_attention_tc_usp(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, int causal,
                                    const AttnPtrs& head, cudaStream_t stream, int* unsupported) {
    *unsupported = 0;
    const int P = Pu * Pr, L = s / Pr;
    if (!tc_attention_supported(d) || P > kMaxMapsWide || L % BM != 0) {
        *unsupported = 1;
        return cudaSuccess;
    }
    return P <= kMaxMaps ? launch_usp_fwd<kMaxMaps>(Pu, Pr, b, s, h_q, h_kv, d, causal, head, stream)
                         : launch_usp_fwd<kMaxMapsWide>(Pu, Pr, b, s, h_q, h_kv, d, causal, head, stream);
}

namespace {

// Row statistics for the backward: D and the base-2 log-sum-exp of every query row, into
// per-head-rank arrays (n_head_ranks of them, h_q / n_head_ranks heads each), all in one grid.
// O and dO are read in head layout (one buffer per head rank) or in seq layout (n_seq_ranks
// buffers of s / n_seq_ranks tokens, all heads).
cudaError_t launch_bwd_prep(int n_head_ranks, int n_seq_ranks, int b, int s, int h_q, int d, const BwdPtrs& ptrs,
                            cudaStream_t stream) {
    const int n_tiles = (s + 127) / 128;
    PrepParams pp_rec;
    PrepParams* pp = &pp_rec;
    memset(pp, 0, sizeof(PrepParams));
    const int nb = ptrs.od_seq_layout ? n_seq_ranks : n_head_ranks;
    for (int r = 0; r < nb; ++r) {
        pp->o[r] = static_cast<const uint8_t*>(ptrs.o_rows[r]);
        pp->dout[r] = static_cast<const uint8_t*>(ptrs.do_rows[r]);
    }
    for (int r = 0; r < n_head_ranks; ++r) {
        pp->lse[r] = ptrs.lse[r];
        pp->lse2[r] = ptrs.lse2[r];
        pp->dsum[r] = ptrs.dsum[r];
    }
    pp->b = b;
    pp->s = s;
    pp->s_pad = n_tiles * 128;
    pp->Hq = h_q / n_head_ranks;
    pp->d = d;
    pp->S = s / n_seq_ranks;
    pp->hq_total = h_q;
    pp->seq_layout = ptrs.od_seq_layout ? 1 : 0;
    pp->lanes_log2 = d == 64 ? 3 : 4;
    pp->units = n_head_ranks * b * pp->Hq;
    // x: the s_pad rows of a unit, kPrepRows per lane group; y: the units
    const int per_block = 256 >> pp->lanes_log2;
    const int gx = (pp->s_pad + per_block * kPrepRows - 1) / (per_block * kPrepRows);
    const int gy = pp->units < 65535 ? pp->units : 65535;
    bwd_prep_kernel<<<dim3((unsigned)gx, (unsigned)gy, 1), 256, 0, stream>>>(*pp);
    return cudaGetLastError();
}

}  // namespace

namespace {

template <class PR>
void fill_bwd_common(PR* prm, int s, int b, int causal, int d) {
    memset(prm, 0, sizeof(PR));
    const int n_tiles = (s + 127) / 128;
    prm->s = s;
    prm->s_pad = n_tiles * 128;
    prm->n_tiles = n_tiles;
    prm->b = b;
    prm->causal = causal ? 1 : 0;
    prm->map_stride = 1;
    prm->scale = (float)(1.0 / std::sqrt((double)d));
    prm->scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
}

template <class PR>
cudaError_t launch_bwd_any_d(const PR& prm, int d, int nranks, cudaStream_t stream) {
    return d == 64 ? launch_bwd_d<64>(prm, nranks, stream) : launch_bwd_d<128>(prm, nranks, stream);
}

// dK/dV and dQ over the seq-layout buffers: one map per rank buffer and kind (NM >= P).
template <int NM>
cudaError_t launch_fused_bwd(int P, int b, int s, int h_q, int h_kv, int d, int causal, const BwdPtrs& ptrs,
                             cudaStream_t stream) {
    BwdParamsT<NM> prm_rec;
    BwdParamsT<NM>* prm = &prm_rec;
    fill_bwd_common(prm, s, b, causal, d);
    const int S = s / P;
    prm->g = h_q / h_kv;
    prm->hq_rank = h_q / P;
    prm->rows_per_map = S;
    prm->hq = h_q;
    prm->hkv = h_kv;
    for (int j = 0; j < P; ++j) {
        if (!make_map(&prm->mq[j], ptrs.q[j], b, S, h_q, d, 128) || !make_map(&prm->mk[j], ptrs.k[j], b, S, h_kv, d, 128) ||
            !make_map(&prm->mv[j], ptrs.v[j], b, S, h_kv, d, 128) ||
            !make_map(&prm->mdo[j], ptrs.dout[j], b, S, h_q, d, 128))
            return cudaErrorInvalidValue;
        prm->dq[j] = static_cast<uint8_t*>(ptrs.dq[j]);
        prm->dk[j] = static_cast<uint8_t*>(ptrs.dk[j]);
        prm->dv[j] = static_cast<uint8_t*>(ptrs.dv[j]);
        prm->lse2[j] = ptrs.lse2[j];  // head rank j's statistics
        prm->dsum[j] = ptrs.dsum[j];
    }
    return launch_bwd_any_d(*prm, d, 1, stream);
}

// The two-level backward's dK/dV and dQ over the Pu units: one map per rank buffer and kind.
template <int NM>
cudaError_t launch_usp_bwd(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, int causal, const BwdPtrs& ptrs,
                           cudaStream_t stream) {
    const int P = Pu * Pr, L = s / Pr;
    const int Hq = h_q / Pu, Hk = kv_heads_per_rank(Pu, h_kv);  // 1: a replicated K/V head
    BwdParamsT<NM> prm_rec;
    BwdParamsT<NM>* prm = &prm_rec;
    fill_bwd_common(prm, s, b, causal, d);
    prm->g = Hq / Hk;  // within a unit
    prm->hq_rank = Hq;
    prm->hq = Hq;
    prm->hkv = Hk;
    prm->rows_per_map = L;
    prm->map_stride = Pu;
    prm->kv_grad_f32 = ptrs.kv_grad_f32;
    for (int j = 0; j < P; ++j) {
        if (!make_map(&prm->mq[j], ptrs.q[j], b, L, Hq, d, 128) || !make_map(&prm->mk[j], ptrs.k[j], b, L, Hk, d, 128) ||
            !make_map(&prm->mv[j], ptrs.v[j], b, L, Hk, d, 128) ||
            !make_map(&prm->mdo[j], ptrs.dout[j], b, L, Hq, d, 128))
            return cudaErrorInvalidValue;
        prm->dq[j] = static_cast<uint8_t*>(ptrs.dq[j]);
        prm->dk[j] = static_cast<uint8_t*>(ptrs.dk[j]);
        prm->dv[j] = static_cast<uint8_t*>(ptrs.dv[j]);
    }
    for (int u = 0; u < Pu; ++u) {
        prm->lse2[u] = ptrs.lse2[u];
        prm->dsum[u] = ptrs.dsum[u];
    }
    return launch_bwd_any_d(*prm, d, Pu, stream);
}

}  // namespace

cudaError_t launch_attention_bwd_tc(int P, int b, int s, int h_q, int h_kv, int d, int causal, int fused,
                                    const BwdPtrs& ptrs, cudaStream_t stream, int* unsupported) {
    *unsupported = 0;
    if (!tc_attention_supported(d) || (fused && (P > kMaxMapsBwdWide || (s / P) % 128 != 0))) {
        *unsupported = 1;
        return cudaSuccess;
    }
    // (1) row sums D and base-2 log-sum-exp, all ranks in one grid
    cudaError_t err = launch_bwd_prep(P, P, b, s, h_q, d, ptrs, stream);
    if (err != cudaSuccess) return err;
    // (2) dK/dV and dQ: one launch pair over seq-layout buffers (fused), else up to kMaxMaps
    //     head ranks per launch pair
    if (fused)
        return P <= kMaxMaps ? launch_fused_bwd<kMaxMaps>(P, b, s, h_q, h_kv, d, causal, ptrs, stream)
                             : launch_fused_bwd<kMaxMapsBwdWide>(P, b, s, h_q, h_kv, d, causal, ptrs, stream);
    const int Hq = h_q / P, Hk = kv_heads_per_rank(P, h_kv);
    BwdParams prm_rec;
    BwdParams* prm = &prm_rec;
    fill_bwd_common(prm, s, b, causal, d);
    prm->hq_rank = Hq;
    prm->rows_per_map = s;
    prm->hq = Hq;
    prm->hkv = Hk;
    prm->g = Hq / Hk;  // within a rank (its K/V heads may be replicas shared with other ranks)
    prm->kv_grad_f32 = ptrs.kv_grad_f32;
    for (int r0 = 0; r0 < P && err == cudaSuccess; r0 += kMaxMaps) {
        const int nr = (P - r0) < kMaxMaps ? (P - r0) : kMaxMaps;
        for (int i = 0; i < nr; ++i) {
            const int r = r0 + i;
            if (!make_map(&prm->mq[i], ptrs.q[r], b, s, Hq, d, 128) || !make_map(&prm->mk[i], ptrs.k[r], b, s, Hk, d, 128) ||
                !make_map(&prm->mv[i], ptrs.v[r], b, s, Hk, d, 128) ||
                !make_map(&prm->mdo[i], ptrs.dout[r], b, s, Hq, d, 128))
                return cudaErrorInvalidValue;
            prm->dq[i] = static_cast<uint8_t*>(ptrs.dq[r]);
            prm->dk[i] = static_cast<uint8_t*>(ptrs.dk[r]);
            prm->dv[i] = static_cast<uint8_t*>(ptrs.dv[r]);
            prm->lse2[i] = ptrs.lse2[r];
            prm->dsum[i] = ptrs.dsum[r];
        }
        err = launch_bwd_any_d(*prm, d, nr, stream);
    }
    return err;
}

cudaError_t launch_attention_bwd_tc_usp(int Pu, int Pr, int b, int s, int h_q, int h_kv, int d, int causal,
                                        const BwdPtrs& ptrs, cudaStream_t stream, int* unsupported) {
    *unsupported = 0;
    const int P = Pu * Pr, L = s / Pr;
    if (!tc_attention_supported(d) || P > kMaxMapsBwdWide || L % 128 != 0) {
        *unsupported = 1;
        return cudaSuccess;
    }
    // (1) statistics per Ulysses unit (Pu head ranks over all s rows), O and dO in seq layout
    cudaError_t err = launch_bwd_prep(Pu, P, b, s, h_q, d, ptrs, stream);
    if (err != cudaSuccess) return err;
    // (2) dK/dV and dQ over the Pu units, every tile read from (written to) the buffer of the
    //     ring group that holds its tokens: the forward's two-level tile addressing
    return P <= kMaxMaps ? launch_usp_bwd<kMaxMaps>(Pu, Pr, b, s, h_q, h_kv, d, causal, ptrs, stream)
                         : launch_usp_bwd<kMaxMapsBwdWide>(Pu, Pr, b, s, h_q, h_kv, d, causal, ptrs, stream);
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
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
