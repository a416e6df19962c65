// Backward of the bf16 local attention on the sm_103a tensor cores.  Included by attn_tc.cu
// inside its anonymous namespace: it shares the bounded waits, the device error word, the
// bf16 packing and the tensor-map encoder.
//
// What it computes ("02 · DeepSpeed-Ulysses", section 5: the local attention's backward is
// the ordinary one).  With the per-row log-sum-exp L_i of the scaled scores saved by the
// forward, P_ij = exp(q_i.k_j/sqrt(d) - L_i) (0 for masked keys) and D_i = sum_c dO_ic O_ic:
//   dV_j = sum_i P_ij dO_i          dP_ij = dO_i . v_j         dS_ij = P_ij (dP_ij - D_i)
//   dK_j = sum_i dS_ij q_i / sqrt(d)                           dQ_i = sum_j dS_ij k_j / sqrt(d)
// Three launches, no atomics, every output element written once:
//   bwd_prep_kernel  D_i from O and dO, and L_i in base-2 units, into padded per-row arrays
//   bwd_dkdv_kernel  one CTA per (rank, batch, K/V head, 128-key tile).  S^T = K Q^T and
//                    dP^T = V dO^T land in tensor memory; sixteen row warps (four per tensor
//                    memory lane quarter, each owning 32 of the 128 query columns; the dQ
//                    kernel uses eight, two per quarter, 64 columns each) form P^T
//                    (bf16, written back over S^T) and dS^T (bf16, written back over dP^T);
//                    dV += P^T dO and dK += dS^T Q both take their A operand straight from
//                    tensor memory, so shared memory holds only K, V and the Q/dO stream.
//                    The loop runs over every query head of the K/V head's group and every
//                    query tile that sees the key tile.
//   bwd_dq_kernel    one CTA per (rank, batch, query head, 128-query tile).  S = Q K^T (two
//                    tensor-memory buffers, so S of tile n+2 can be computed while tile n+1
//                    is being worked on) and dP = dO V^T; the row warps write dS as bf16 over
//                    S and dQ += dS K takes it from tensor memory.
// Recomputing S and dP in both kernels costs 7 tile products instead of 5 but needs neither
// atomics nor a second pass over dQ, and gives the same bits on every run.
//
// Tile orders.  All CTAs of one head stream the same sequence of Q/dO (or K/V) tiles at
// the same time, so each tile is read from DRAM about once and served from L2 after that:
// the dK/dV kernel walks query tiles from the last one down (causal: down to the diagonal
// tile, which comes last and is the only masked one), the dQ kernel walks key tiles from 0
// up (causal: up to the diagonal).  Within a head, the CTAs with the most tiles come first.
// Rows past the sequence end read zeros (TMA fill) and get L = +inf, so their P is 0.
//
// Every wait is bounded like the forward's: a wait that gives up sets the device error
// word, and the CTA drains its copies and MMAs, frees tensor memory and returns.

// Warp roles of both kernels: RW row warps (RW/4 per tensor-memory lane quarter, each
// owning 128/(RW/4) tile columns), then the TMA producer warp, then the MMA warp.
template <int RW>
struct RowCfg {
    static constexpr int kRows = RW;
    static constexpr int kProducer = RW;
    static constexpr int kMma = RW + 1;
    static constexpr int kThreads = (RW + 2) * 32;
    static constexpr int kColGroups = RW / 4;       // row warps sharing one lane quarter
    static constexpr int kColW = 128 / kColGroups;  // tile columns each row warp owns
    static constexpr int kChunks = kColW / 32;      // 32-column tensor-memory loads per warp
};
constexpr int kRowsKV = 16;  // dK/dV kernel: faster than 8 on the DiT workload
constexpr int kRowsQ = 8;    // dQ kernel: 8 and 16 measure the same; 8 needs fewer threads
constexpr int kRingKV = 5;   // dK/dV kernel: Q/dO ring slots
constexpr int kRingQ = 5;    // dQ kernel: K/V ring slots

// Maps and gradient buffers are indexed like the forward's: token t of the sequence, for
// the unit `rank` of a CTA, lives in buffer rank + (t / rows_per_map) * map_stride at row
// t % rows_per_map.  Two-level (Ulysses x Ring): unit u of a Ulysses group, buffers of ring
// group t / (s/Pr)'s rank u (rows_per_map = s/Pr, map_stride = Pu).
// Unfused: one buffer per head rank (rows_per_map = s, hq/hkv = that rank's heads).  Fused:
// one buffer per seq rank (rows_per_map = s/P, hq/hkv = all heads, rank = 0), so the
// exchanges happen in the tile addressing.  The row statistics always live per head rank:
// head h of a CTA belongs to head rank rank + h / hq_rank, local head h % hq_rank.
// NM maps of each kind: kMaxMaps, or kMaxMapsBwdWide for fused or two-level calls over
// more rank buffers (four maps per rank: at most 48 ranks fit the 32 KB parameter limit).
template <int NM>
struct BwdParamsT {
    static constexpr int kMaps = NM;
    CUtensorMap mq[NM], mk[NM], mv[NM], mdo[NM];
    uint8_t* dq[NM];        // [b][rows][hq][d] bf16
    uint8_t* dk[NM];        // [b][rows][hkv][d] bf16 (fp32 with kv_grad_f32)
    uint8_t* dv[NM];
    const float* lse2[NM];  // per head rank [b][hq_rank][s_pad]: log-sum-exp, base-2 units (+inf on padding)
    const float* dsum[NM];  // per head rank [b][hq_rank][s_pad]: D (0 on padding)
    int s, s_pad, n_tiles, hq, hkv, g, b, causal;
    int rows_per_map;             // s (unfused), s/P (fused) or s/Pr (two-level)
    int map_stride;               // map step from one token block to the next (Pu two-level, else 1)
    int hq_rank;                  // query heads per head rank
    float scale_log2;             // log2(e)/sqrt(d)
    float scale;                  // 1/sqrt(d)
    int kv_grad_f32;              // host: launch the dK/dV kernel that stores fp32 partial sums
    int n_units;                  // dK/dV work: (rank, batch, K/V head) units of the launch
    int kv_items;                 // n_units * n_tiles
    int band_units;               // causal: units per band (see kv_item)
    int n_units_q;                // dQ work: (rank, batch, query head) units of the launch
    int q_items;                  // n_units_q * n_tiles
    int band_units_q;             // causal: units per band (see q_item)
};
using BwdParams = BwdParamsT<kMaxMaps>;

struct BwdTok {
    int map, row;
};
template <class PR>
__device__ __forceinline__ BwdTok bwd_tok(const PR& p, int rank, int t0) {
    return BwdTok{rank + (t0 / p.rows_per_map) * p.map_stride, t0 % p.rows_per_map};
}

// Row statistics of (batch bb, query head h of the CTA's unit `rank`), from query q0 on.
template <class PR>
__device__ __forceinline__ size_t bwd_stat_off(const PR& p, int bb, int h, int q0) {
    return ((size_t)bb * p.hq_rank + h % p.hq_rank) * p.s_pad + q0;
}
template <class PR>
__device__ __forceinline__ int bwd_stat_rank(const PR& p, int rank, int h) { return rank + h / p.hq_rank; }

// ------------------------------------------------------------------------- prep
struct PrepParams {
    const uint8_t* o[kMaxRanks];
    const uint8_t* dout[kMaxRanks];
    const float* lse[kMaxRanks];  // [b][Hq][s], natural log
    float* lse2[kMaxRanks];
    float* dsum[kMaxRanks];
    int units;                    // P * b * Hq (rank, batch, head) units
    int b, s, s_pad, Hq, d, S, hq_total, seq_layout;
    int lanes_log2;               // log2(d / 8): lanes per row
};

// d/8 lanes per (rank, batch, head, token) row, 16 bytes each.  O and dO are read in the
// layout the caller holds them in: head layout of rank r, or (seq_layout) the seq layout,
// where head-layout row (r, hh, t) is row t % S of rank t / S at head r*Hq + hh.
constexpr int kPrepRows = 4;  // rows per lane group: their loads are all in flight at once

// grid.y walks the (rank, batch, head) units, so their coordinates are decoded once per
// block; grid.x covers the token rows of a unit, kPrepRows per lane group (rows t, t + G, ...).
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __grid_constant__ PrepParams p) {
    const int lanes_log2 = p.lanes_log2;
    const int sub = (int)(threadIdx.x & ((1u << lanes_log2) - 1));
    const int per_block = 256 >> lanes_log2;  // lane groups per block
    const int G = (int)gridDim.x * per_block;
    const int grp = (int)blockIdx.x * per_block + (int)(threadIdx.x >> lanes_log2);
    for (int u = blockIdx.y; u < p.units; u += gridDim.y) {  // block-uniform: every shuffle has the whole warp
        const int hh = u % p.Hq, r1 = u / p.Hq;
        const int bb = r1 % p.b, r = r1 / p.b;
        uint4 a[kPrepRows], c[kPrepRows];
#pragma unroll
        for (int k = 0; k < kPrepRows; ++k) {
            const int t = grp + k * G;
            a[k] = make_uint4(0, 0, 0, 0);
            c[k] = make_uint4(0, 0, 0, 0);
            if (t < p.s) {
                size_t off;
                const uint8_t *o, *gp;
                if (p.seq_layout) {
                    const int j = t / p.S;
                    off = (((size_t)bb * p.S + (t - j * p.S)) * p.hq_total + (size_t)r * p.Hq + hh) * (size_t)p.d * 2;
                    o = p.o[j];
                    gp = p.dout[j];
                } else {
                    off = (((size_t)bb * p.s + t) * p.Hq + hh) * (size_t)p.d * 2;
                    o = p.o[r];
                    gp = p.dout[r];
                }
                a[k] = *reinterpret_cast<const uint4*>(o + off + sub * 16);
                c[k] = *reinterpret_cast<const uint4*>(gp + off + sub * 16);
            }
        }
        const size_t vbase = ((size_t)bb * p.Hq + hh) * p.s_pad;
        const size_t lbase = ((size_t)bb * p.Hq + hh) * p.s;
#pragma unroll
        for (int k = 0; k < kPrepRows; ++k) {
            const int t = grp + k * G;
            const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
            const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c[k]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = __bfloat1622float2(a2[e]), fc = __bfloat1622float2(c2[e]);
                acc = fmaf(fa.x, fc.x, fmaf(fa.y, fc.y, acc));
            }
            for (int o = 1 << (lanes_log2 - 1); o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (t < p.s_pad && sub == 0) {
                if (t < p.s) {
                    p.dsum[r][vbase + t] = acc;
                    p.lse2[r][vbase + t] = p.lse[r][lbase + t] * 1.4426950408889634f;
                } else {
                    p.dsum[r][vbase + t] = 0.f;
                    p.lse2[r][vbase + t] = INFINITY;
                }
            }
        }
    }
}

// --------------------------------------------------------------- shared pieces
template <int D, int RING>
struct BwdSmem {
    static constexpr uint32_t kTile = 128 * D * 2;
    static constexpr uint32_t offFixA = 0;          // K (dK/dV kernel) or Q (dQ kernel)
    static constexpr uint32_t offFixB = kTile;      // V or dO
    static constexpr uint32_t offRing = 2 * kTile;  // RING streamed tiles
    static constexpr uint32_t offBar = offRing + RING * kTile;
    static constexpr uint32_t kBarSlots = 24;
    static constexpr uint32_t kUsed = offBar + kBarSlots * 8 + 64;
    static constexpr uint32_t kAlloc = kUsed + 1024;  // slack to align the base to 1024 bytes
};

// Stores NC accumulator columns of this thread's tensor-memory lane as bf16 (times mul).
template <int NC>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, uint8_t* dst, float mul, bool ok) {
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * mul, __uint_as_float(r[q4 * 8 + 1]) * mul);
            v.y = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * mul, __uint_as_float(r[q4 * 8 + 3]) * mul);
            v.z = pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * mul, __uint_as_float(r[q4 * 8 + 5]) * mul);
            v.w = pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * mul, __uint_as_float(r[q4 * 8 + 7]) * mul);
            if (ok) *reinterpret_cast<uint4*>(dst + (c * 32 + q4 * 8) * 2) = v;
        }
    }
}

// As store_row_bf16, in fp32 (a partial sum that is added to others before rounding).
template <int NC>
__device__ __forceinline__ void store_row_f32(uint32_t taddr, uint8_t* dst, float mul, bool ok) {
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(taddr + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
            float4 v;
            v.x = __uint_as_float(r[q4 * 4 + 0]) * mul;
            v.y = __uint_as_float(r[q4 * 4 + 1]) * mul;
            v.z = __uint_as_float(r[q4 * 4 + 2]) * mul;
            v.w = __uint_as_float(r[q4 * 4 + 3]) * mul;
            if (ok) *reinterpret_cast<float4*>(dst + (c * 32 + q4 * 4) * 4) = v;
        }
    }
}

// Initialises the barriers (those in [rows_from, rows_to) count one arrival per row warp)
// and allocates tensor memory; false when the CTA must leave at once.
__device__ __forceinline__ bool bwd_setup(uint64_t* bars, int nbars, int rows_from, int rows_to, int row_warps,
                                          int mma_warp, Shared* sh) {
    if (threadIdx.x == 0) {
        sh->abort = error_word_set() ? 1 : 0;
        for (int i = 0; i < nbars; ++i)
            mbar_init(&bars[i], (i >= rows_from && i < rows_to) ? (uint32_t)row_warps : 1u);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (sh->abort) return false;
    if ((threadIdx.x >> 5) == mma_warp) tmem_alloc(&sh->tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return true;
}

// d (128 x 128, fp32 in tensor memory) = A B^T, A and B 128 x D K-major tiles in shared memory.
template <int D>
__device__ __forceinline__ void mma_kmajor(uint32_t d, uint64_t a, uint64_t b) {
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, false);
    constexpr uint32_t kSlab = 128 * 128;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kSlab + (kk & 3) * 32) >> 4;
        mma_bf16_ss_warp(d, a + off, b + off, kIdesc, kk > 0 ? 1u : 0u);
    }
}

// acc (128 x D) += A (128 x 128 bf16 pairs in tensor memory at a_tmem) * B (128 x D tile in
// shared memory, D contiguous: MN-major).  Each row warp packs its kColW columns of A into
// the first kColW/2 tensor-memory columns of its own kColW-column group, so columns
// 16k..16k+15 of A sit at a_tmem + kColW*(16k / kColW) + (16k % kColW)/2.
template <int D, int kColW>
__device__ __forceinline__ void mma_acc_tmemA(uint32_t acc, uint32_t a_tmem, uint64_t b_mn, bool accumulate) {
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, D, true);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_bf16_ts_warp(acc, a_tmem + (kk * 16 / kColW) * kColW + ((kk * 16) % kColW) / 2,
                         b_mn + ((kk * 16 * 128) >> 4), kIdesc, (accumulate || kk > 0) ? 1u : 0u);
}

// ------------------------------------------------------------------ dK / dV
// Work item = (rank, batch, K/V head, 128-key tile); a unit = (rank, batch, K/V head).
// Non-causal (all items equal): the key tiles of a unit are adjacent, so the CTAs working
// at the same time stream the same Q/dO tiles and L2 serves the re-reads.  Causal (key tile
// kt has g*(n_tiles-kt) steps): the units form bands of band_units units, and inside a band
// the key tile is slowest and ascending, so the items run heaviest first.  band_units = 1
// gives the unit-major order, key tile ascending.
struct KvItem {
    int rank, bb, kvh, kt;
};

template <class PR>
__device__ __forceinline__ KvItem kv_item(const PR& p, int w) {
    int u, kt;
    if (p.causal) {
        const int per_band = p.band_units * p.n_tiles;
        const int band = w / per_band, base = band * p.band_units;
        const int in_band = p.n_units - base < p.band_units ? p.n_units - base : p.band_units;
        const int r = w - band * per_band;
        u = base + r % in_band;
        kt = r / in_band;
    } else {
        u = w / p.n_tiles;
        kt = w % p.n_tiles;
    }
    KvItem it;
    it.kvh = u % p.hkv;
    u /= p.hkv;
    it.bb = u % p.b;
    it.rank = u / p.b;
    it.kt = kt;
    return it;
}

// The k-th item of this CTA.  PERSIST: rounds of gridDim.x items, alternating direction
// (snake), so a heaviest-first order spreads evenly over the CTAs.  Else one item per CTA
// (the loops that call this run once, and their running counters fold to constants).
// -1 when the CTA has no k-th item.
template <bool PERSIST>
__device__ __forceinline__ int bwd_item_index(int n_items, int k) {
    const int G = gridDim.x, c = blockIdx.x;
    const int w = PERSIST ? k * G + ((k & 1) ? G - 1 - c : c) : (k == 0 ? c : n_items);
    return w < n_items ? w : -1;
}

// Persistent (grid below the item count): each CTA walks its items; every role walks the
// same sequence, and the barrier phases run on across items.  With one CTA per item the
// loop runs once.  At an item boundary the producer loads the next K/V
// as soon as the last S^T and dP^T products have read the current ones, and the MMA warp
// issues the next item's first S^T and dP^T right after the last dK product, so both run
// while the row warps store dK and dV.  The next item's first dV product (which overwrites
// the accumulator) waits for P-ready, which every row warp signals only after its epilogue.
// Tensor memory: S^T (then P^T) 0..127 | dP^T (then dS^T) 128..255 | dK 256.. | dV 384..
// F32: dk/dv receive fp32 partial sums (a replicated K/V head's share from this rank).
template <int D, int RW, bool F32, bool PERSIST, int NM>
__global__ void __launch_bounds__(RowCfg<RW>::kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParamsT<NM> p) {
    using C = RowCfg<RW>;
    constexpr int kBwdRowWarps = C::kRows, kBwdProducer = C::kProducer, kBwdMma = C::kMma;
    constexpr int kColGroups = C::kColGroups, kColW = C::kColW, kChunks = C::kChunks;
    using L = BwdSmem<D, kRingKV>;
    constexpr uint32_t kSlab = 128 * 128;
    enum {
        FIX = 0, FIX_EMPTY, FULL, EMPTY = FULL + kRingKV, S_FULL = EMPTY + kRingKV, DP_FULL, P_READY, DS_READY, FINAL,
        MMA_DONE, NBARS
    };
    static_assert(NBARS <= (int)L::kBarSlots, "barrier slots");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
    Shared* sh = reinterpret_cast<Shared*>(smem + L::offBar + L::kBarSlots * 8);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // step n of an item: query tile n_tiles-1 - n/g of query head kvh*g + n%g
    const int g = p.g, n_tiles = p.n_tiles;
    auto item_steps = [&p, g, n_tiles](const KvItem& it) { return g * (n_tiles - (p.causal ? it.kt : 0)); };
    auto step_qt = [n_tiles, g](int n) { return n_tiles - 1 - n / g; };

    if (!bwd_setup(bars, NBARS, P_READY, DS_READY + 1, kBwdRowWarps, kBwdMma, sh)) return;
    const uint32_t tmem = sh->tmem_base;

    if (warp == kBwdProducer) {
        // per item: the fixed tiles K (A) and V (B) of its key tile, then Q and dO per step
        int issued = 0, fix_loads = 0;  // ring loads and fixed-tile loads issued so far
        bool ok = true;
        for (int k = 0; ok && (PERSIST || k == 0); ++k) {
            const int w = bwd_item_index<PERSIST>(p.kv_items, k);
            if (w < 0) break;
            const KvItem it = kv_item(p, w);
            const int n_steps = item_steps(it);
            if (k > 0) {  // the previous item's last S^T and dP^T have read K and V
                ok = wait_phase_warp(&bars[FIX_EMPTY], (k - 1) & 1, sh);
                if (!ok) break;
            }
            const BwdTok kp = bwd_tok(p, it.rank, it.kt * 128);
            mbar_arrive_expect_tx_warp(&bars[FIX], 2 * L::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                tma_load_4d_warp(sbase + L::offFixA + c * kSlab, &p.mk[kp.map], &bars[FIX], c * 64, it.kvh, kp.row,
                                 it.bb);
                tma_load_4d_warp(sbase + L::offFixB + c * kSlab, &p.mv[kp.map], &bars[FIX], c * 64, it.kvh, kp.row,
                                 it.bb);
            }
            ++fix_loads;
            for (int m = 0; m < 2 * n_steps; ++m) {
                const int slot = issued % kRingKV;
                ok = wait_phase_warp(&bars[EMPTY + slot], ((issued / kRingKV) & 1) ^ 1, sh);
                if (!ok) break;
                const int n = m >> 1;
                const BwdTok qp = bwd_tok(p, it.rank, step_qt(n) * 128);
                mbar_arrive_expect_tx_warp(&bars[FULL + slot], L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_warp(sbase + L::offRing + slot * L::kTile + c * kSlab,
                                     (m & 1) ? &p.mdo[qp.map] : &p.mq[qp.map], &bars[FULL + slot], c * 64,
                                     it.kvh * g + n % g, qp.row, it.bb);
                ++issued;
            }
        }
        if (!ok) {  // let the copies in flight land before the CTA leaves
            for (int slot = 0; slot < kRingKV; ++slot) {
                const int cnt = (issued - slot + kRingKV - 1) / kRingKV;
                if (cnt > 0) drain_phase(&bars[FULL + slot], (cnt - 1) & 1);
            }
            if (fix_loads > 0) drain_phase(&bars[FIX], (fix_loads - 1) & 1);
        }
    } else if (warp == kBwdMma) {
        const uint64_t dk_a = smem_desc_sw128(sbase + L::offFixA, 16, 1024);        // K
        const uint64_t dv_a = smem_desc_sw128(sbase + L::offFixB, 16, 1024);        // V
        const uint64_t ring_k = smem_desc_sw128(sbase + L::offRing, 16, 1024);      // Q / dO, K-major
        const uint64_t ring_mn = smem_desc_sw128(sbase + L::offRing, kSlab, 1024);  // Q / dO, MN-major
        int m0 = 0;  // ring position of the current item's first Q tile
        int gs = 0;  // steps of the earlier items (the per-step barriers' phases run on)
        bool ok = true;
        for (int k = 0; ok && (PERSIST || k == 0); ++k) {
            const int w = bwd_item_index<PERSIST>(p.kv_items, k);
            if (w < 0) break;
            const int n_steps = item_steps(kv_item(p, w));
            auto so = [m0](int m) { return (uint64_t)((((m0 + m) % kRingKV) * L::kTile) >> 4); };
            auto full = [&](int m) {
                return wait_phase_warp(&bars[FULL + (m0 + m) % kRingKV], ((m0 + m) / kRingKV) & 1, sh);
            };
            auto release = [&](int m) { mma_commit_warp(&bars[EMPTY + (m0 + m) % kRingKV]); };
            ok = wait_phase_warp(&bars[FIX], k & 1, sh) && full(0);
            if (ok) {
                tc_fence_after();
                mma_kmajor<D>(tmem, dk_a, ring_k + so(0));  // S^T(0)
                mma_commit_warp(&bars[S_FULL]);
                ok = full(1);
            }
            if (ok) {
                tc_fence_after();
                mma_kmajor<D>(tmem + 128u, dv_a, ring_k + so(1));  // dP^T(0)
                mma_commit_warp(&bars[DP_FULL]);
                if (n_steps == 1) mma_commit_warp(&bars[FIX_EMPTY]);  // K and V read for the last time
            }
            for (int n = 0; n < n_steps && ok; ++n) {
                const int mq = 2 * n, mo = 2 * n + 1;
                ok = wait_phase_warp(&bars[P_READY], (gs + n) & 1, sh);
                if (!ok) break;
                tc_fence_after();
                mma_acc_tmemA<D, kColW>(tmem + 384u, tmem, ring_mn + so(mo), n > 0);  // dV += P^T dO
                release(mo);
                if (n + 1 < n_steps) {  // S^T(n+1) over P^T(n): issued after the product that reads it
                    ok = full(mq + 2);
                    if (!ok) break;
                    tc_fence_after();
                    mma_kmajor<D>(tmem, dk_a, ring_k + so(mq + 2));
                    mma_commit_warp(&bars[S_FULL]);
                }
                ok = wait_phase_warp(&bars[DS_READY], (gs + n) & 1, sh);
                if (!ok) break;
                tc_fence_after();
                mma_acc_tmemA<D, kColW>(tmem + 256u, tmem + 128u, ring_mn + so(mq), n > 0);  // dK += dS^T Q
                release(mq);
                if (n + 1 < n_steps) {  // dP^T(n+1) over dS^T(n): issued after the product that reads it
                    ok = full(mo + 2);
                    if (!ok) break;
                    tc_fence_after();
                    mma_kmajor<D>(tmem + 128u, dv_a, ring_k + so(mo + 2));
                    mma_commit_warp(&bars[DP_FULL]);
                    if (n + 2 == n_steps) mma_commit_warp(&bars[FIX_EMPTY]);
                }
            }
            if (!ok) break;
            mma_commit_warp(&bars[FINAL]);  // dK and dV of this item are complete
            gs += n_steps;
            m0 += 2 * n_steps;
        }
        // every MMA issued above completes before tensor memory is released
        mma_commit_warp(&bars[MMA_DONE]);
        drain_phase(&bars[MMA_DONE], 0);
    } else {
        // row warps: thread = key row; warp group cg owns query columns [cg*kColW, +kColW)
        const int sub = warp & 3, cg = warp >> 2;
        const int row = sub * 32 + lane;
        const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
        const uint32_t tS = tmem + lane_off + cg * kColW, tdP = tmem + 128u + lane_off + cg * kColW;
        const float sc = p.scale_log2;
        int gs = 0;
        bool ok = true;
        for (int k = 0; ok && (PERSIST || k == 0); ++k) {
            const int w = bwd_item_index<PERSIST>(p.kv_items, k);
            if (w < 0) break;
            const KvItem it = kv_item(p, w);
            const int n_steps = item_steps(it);
            const int kt = it.kt;
            const int k0 = kt * 128, key = k0 + row;
            const int head0 = it.kvh * g;                  // first query head of the step sequence
            const int bh0 = it.bb * p.hq_rank;             // batch offset of the statistic rows
            auto step_head = [head0, g](int n) { return head0 + n % g; };
            auto stat_off = [&](int n) {  // offset of step n's first row statistic of this warp
                return ((size_t)bh0 + step_head(n) % p.hq_rank) * p.s_pad + step_qt(n) * 128 + cg * kColW;
            };
            const int rank = it.rank;
            for (int n = 0; n < n_steps; ++n) {
                const int qt = step_qt(n);
                const int qb = qt * 128 + cg * kColW;  // first query column of this warp
                const size_t vbase = stat_off(n);
                const int sr = bwd_stat_rank(p, rank, step_head(n));
                const float4* l4 = reinterpret_cast<const float4*>(p.lse2[sr] + vbase);
                const float4* d4 = reinterpret_cast<const float4*>(p.dsum[sr] + vbase);
                if (n + 1 < n_steps && lane < 2 * kChunks) {  // next step's statistics: one 128-byte line per lane
                    const size_t nb = stat_off(n + 1) + (lane % kChunks) * 32;
                    const int nr = bwd_stat_rank(p, rank, step_head(n + 1));
                    prefetch_l1(lane < kChunks ? p.lse2[nr] + nb : p.dsum[nr] + nb);
                }
                const bool diag = p.causal && qt == kt;
                float pf[kColW];
                ok = wait_phase_warp(&bars[S_FULL], (gs + n) & 1, sh);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t sv[32];
                    float lv[32];
                    tmem_ld32(tS + c * 32, sv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 x = __ldg(l4 + c * 8 + i);
                        lv[4 * i] = x.x;
                        lv[4 * i + 1] = x.y;
                        lv[4 * i + 2] = x.z;
                        lv[4 * i + 3] = x.w;
                    }
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float a0, a1;
                        ffma2(a0, a1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), sc, sc, -lv[e], -lv[e + 1]);
                        float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
                        if (diag) {
                            const int q = qb + c * 32 + e;
                            p0 = key <= q ? p0 : 0.f;
                            p1 = key <= q + 1 ? p1 : 0.f;
                        }
                        pf[c * 32 + e] = p0;
                        pf[c * 32 + e + 1] = p1;
                        pk[e >> 1] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + c * 16, pk);  // P^T over S^T columns this warp has already read
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[P_READY]);

                ok = wait_phase_warp(&bars[DP_FULL], (gs + n) & 1, sh);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t dv[32];
                    float dl[32];
                    tmem_ld32(tdP + c * 32, dv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 x = __ldg(d4 + c * 8 + i);
                        dl[4 * i] = x.x;
                        dl[4 * i + 1] = x.y;
                        dl[4 * i + 2] = x.z;
                        dl[4 * i + 3] = x.w;
                    }
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float t0, t1;
                        fadd2(t0, t1, __uint_as_float(dv[e]), __uint_as_float(dv[e + 1]), -dl[e], -dl[e + 1]);
                        fmul2(t0, t1, pf[c * 32 + e], pf[c * 32 + e + 1], t0, t1);
                        pk[e >> 1] = pack_bf16x2(t0, t1);
                    }
                    tmem_st16(tdP + c * 16, pk);  // dS^T over dP^T columns this warp has already read
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[DS_READY]);
            }
            if (ok) ok = wait_phase_warp(&bars[FINAL], k & 1, sh);
            if (!ok) break;
            constexpr int kEpi = D / kColGroups >= 32 ? D / kColGroups : 32;  // accumulator columns per warp
            if (cg * kEpi < D) {
                tc_fence_after();
                const bool kok = key < p.s;
                const BwdTok kt_ = bwd_tok(p, rank, kok ? key : k0);
                constexpr size_t kEl = F32 ? 4 : 2;  // bytes per stored element
                const KvItem e_it = kv_item(p, w);
                const size_t off = (((size_t)e_it.bb * p.rows_per_map + kt_.row) * p.hkv + e_it.kvh) * (size_t)D * kEl +
                                   cg * kEpi * kEl;
                if constexpr (F32) {
                    store_row_f32<kEpi>(tmem + 256u + lane_off + cg * kEpi, p.dk[kt_.map] + off, p.scale, kok);
                    store_row_f32<kEpi>(tmem + 384u + lane_off + cg * kEpi, p.dv[kt_.map] + off, 1.0f, kok);
                } else {
                    store_row_bf16<kEpi>(tmem + 256u + lane_off + cg * kEpi, p.dk[kt_.map] + off, p.scale, kok);
                    store_row_bf16<kEpi>(tmem + 384u + lane_off + cg * kEpi, p.dv[kt_.map] + off, 1.0f, kok);
                }
            }
            gs += n_steps;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ----------------------------------------------------------------------- dQ
// Work item = (rank, batch, query head, 128-query tile); a unit = (rank, batch, query head).
// The query tiles of a unit run last tile first (the heaviest first under the causal mask).
// Non-causal: a unit's tiles are adjacent.  Causal: bands of band_units_q units with the
// query tile slowest inside a band (band_units_q = 1: unit-major).  Query heads sharing a
// K/V head are adjacent units.
struct QItem {
    int rank, bb, hh, qt;
};

template <class PR>
__device__ __forceinline__ QItem q_item(const PR& p, int w) {
    int u, r;
    if (p.causal) {
        const int per_band = p.band_units_q * p.n_tiles;
        const int band = w / per_band, base = band * p.band_units_q;
        const int in_band = p.n_units_q - base < p.band_units_q ? p.n_units_q - base : p.band_units_q;
        const int i = w - band * per_band;
        u = base + i % in_band;
        r = i / in_band;
    } else {
        u = w / p.n_tiles;
        r = w % p.n_tiles;
    }
    QItem it;
    it.qt = p.n_tiles - 1 - r;
    it.hh = u % p.hq;
    u /= p.hq;
    it.bb = u % p.b;
    it.rank = u / p.b;
    return it;
}

// Persistent as the dK/dV kernel: each CTA walks its items (once when the grid has one CTA
// per item) with the barrier phases running on across items.  The producer loads the next
// Q and dO as soon as the item's last S and dP have read the current ones; the next item's
// first S, dP and second S follow the last dQ product and run while the row warps store
// dQ; the next item's first dQ product (which overwrites the accumulator) waits for
// dS-ready, which every row warp signals only after its epilogue.
// Tensor memory: S/dS buffer 0 0..127 | dP 128..255 | dQ 256.. | S/dS buffer 1 384..511.
template <int D, int RW, bool PERSIST, int NM>
__global__ void __launch_bounds__(RowCfg<RW>::kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParamsT<NM> p) {
    using C = RowCfg<RW>;
    constexpr int kBwdRowWarps = C::kRows, kBwdProducer = C::kProducer, kBwdMma = C::kMma;
    constexpr int kColGroups = C::kColGroups, kColW = C::kColW, kChunks = C::kChunks;
    using L = BwdSmem<D, kRingQ>;
    constexpr uint32_t kSlab = 128 * 128;
    enum {
        FIX = 0, FIX_EMPTY, FULL, EMPTY = FULL + kRingQ, S_FULL = EMPTY + kRingQ, DP_FULL = S_FULL + 2, DS_READY,
        FINAL, MMA_DONE, NBARS
    };
    static_assert(NBARS <= (int)L::kBarSlots, "barrier slots");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
    Shared* sh = reinterpret_cast<Shared*>(smem + L::offBar + L::kBarSlots * 8);
    const uint32_t sbase = smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto item_steps = [&p](const QItem& it) { return p.causal ? it.qt + 1 : p.n_tiles; };  // key tiles

    if (!bwd_setup(bars, NBARS, DS_READY, DS_READY + 1, kBwdRowWarps, kBwdMma, sh)) return;
    const uint32_t tmem = sh->tmem_base;
    auto sbuf = [tmem](int gn) { return tmem + ((gn & 1) ? 384u : 0u); };  // by global step

    if (warp == kBwdProducer) {
        // per item: the fixed tiles Q (A) and dO (B) of its query tile, then K_n and V_n
        int issued = 0, fix_loads = 0;
        bool ok = true;
        for (int k = 0; ok && (PERSIST || k == 0); ++k) {
            const int w = bwd_item_index<PERSIST>(p.q_items, k);
            if (w < 0) break;
            const QItem it = q_item(p, w);
            const int n_steps = item_steps(it), kvh = it.hh / p.g;
            if (k > 0) {  // the previous item's last S and dP have read Q and dO
                ok = wait_phase_warp(&bars[FIX_EMPTY], (k - 1) & 1, sh);
                if (!ok) break;
            }
            const BwdTok qp = bwd_tok(p, it.rank, it.qt * 128);
            mbar_arrive_expect_tx_warp(&bars[FIX], 2 * L::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                tma_load_4d_warp(sbase + L::offFixA + c * kSlab, &p.mq[qp.map], &bars[FIX], c * 64, it.hh, qp.row,
                                 it.bb);
                tma_load_4d_warp(sbase + L::offFixB + c * kSlab, &p.mdo[qp.map], &bars[FIX], c * 64, it.hh, qp.row,
                                 it.bb);
            }
            ++fix_loads;
            for (int m = 0; m < 2 * n_steps; ++m) {  // K_n, then V_n
                const int slot = issued % kRingQ;
                ok = wait_phase_warp(&bars[EMPTY + slot], ((issued / kRingQ) & 1) ^ 1, sh);
                if (!ok) break;
                const BwdTok kp = bwd_tok(p, it.rank, (m >> 1) * 128);
                mbar_arrive_expect_tx_warp(&bars[FULL + slot], L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d_warp(sbase + L::offRing + slot * L::kTile + c * kSlab,
                                     (m & 1) ? &p.mv[kp.map] : &p.mk[kp.map], &bars[FULL + slot], c * 64, kvh, kp.row,
                                     it.bb);
                ++issued;
            }
        }
        if (!ok) {  // let the copies in flight land before the CTA leaves
            for (int slot = 0; slot < kRingQ; ++slot) {
                const int cnt = (issued - slot + kRingQ - 1) / kRingQ;
                if (cnt > 0) drain_phase(&bars[FULL + slot], (cnt - 1) & 1);
            }
            if (fix_loads > 0) drain_phase(&bars[FIX], (fix_loads - 1) & 1);
        }
    } else if (warp == kBwdMma) {
        const uint64_t q_a = smem_desc_sw128(sbase + L::offFixA, 16, 1024);         // Q
        const uint64_t do_a = smem_desc_sw128(sbase + L::offFixB, 16, 1024);        // dO
        const uint64_t ring_k = smem_desc_sw128(sbase + L::offRing, 16, 1024);      // K / V, K-major
        const uint64_t ring_mn = smem_desc_sw128(sbase + L::offRing, kSlab, 1024);  // K, MN-major
        int m0 = 0;  // ring position of the current item's K_0
        int gs = 0;  // steps of the earlier items (buffers and per-step phases run on)
        bool ok = true;
        for (int k = 0; ok && (PERSIST || k == 0); ++k) {
            const int w = bwd_item_index<PERSIST>(p.q_items, k);
            if (w < 0) break;
            const int n_steps = item_steps(q_item(p, w));
            auto so = [m0](int m) { return (uint64_t)((((m0 + m) % kRingQ) * L::kTile) >> 4); };
            auto full = [&](int m) {
                return wait_phase_warp(&bars[FULL + (m0 + m) % kRingQ], ((m0 + m) / kRingQ) & 1, sh);
            };
            auto issue_s = [&](int n) {  // S(n) = Q K_n^T into the buffer of global step gs+n
                mma_kmajor<D>(sbuf(gs + n), q_a, ring_k + so(2 * n));
                mma_commit_warp(&bars[S_FULL + ((gs + n) & 1)]);
            };
            auto issue_dp = [&](int n) {  // dP(n) = dO V_n^T; V_n is not read after this
                mma_kmajor<D>(tmem + 128u, do_a, ring_k + so(2 * n + 1));
                mma_commit_warp(&bars[DP_FULL]);
                mma_commit_warp(&bars[EMPTY + (m0 + 2 * n + 1) % kRingQ]);
                if (n + 1 == n_steps) mma_commit_warp(&bars[FIX_EMPTY]);  // Q and dO read for the last time
            };
            ok = wait_phase_warp(&bars[FIX], k & 1, sh) && full(0);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                ok = full(1);
            }
            if (ok) {
                tc_fence_after();
                issue_dp(0);
                if (n_steps > 1) {
                    ok = full(2);
                    if (ok) {
                        tc_fence_after();
                        issue_s(1);
                    }
                }
            }
            for (int n = 0; n < n_steps && ok; ++n) {
                ok = wait_phase_warp(&bars[DS_READY], (gs + n) & 1, sh);
                if (!ok) break;
                tc_fence_after();
                mma_acc_tmemA<D, kColW>(tmem + 256u, sbuf(gs + n), ring_mn + so(2 * n), n > 0);  // dQ += dS K
                mma_commit_warp(&bars[EMPTY + (m0 + 2 * n) % kRingQ]);
                if (n + 1 < n_steps) {  // the row warps have read dP(n)
                    ok = full(2 * n + 3);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dp(n + 1);
                }
                if (n + 2 < n_steps) {  // dS(n)'s buffer: dS(n) is read by the product issued above
                    ok = full(2 * n + 4);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(n + 2);
                }
            }
            if (!ok) break;
            mma_commit_warp(&bars[FINAL]);  // dQ of this item is complete
            gs += n_steps;
            m0 += 2 * n_steps;
        }
        // every MMA issued above completes before tensor memory is released
        mma_commit_warp(&bars[MMA_DONE]);
        drain_phase(&bars[MMA_DONE], 0);
    } else {
        // row warps: thread = query row; warp group cg owns key columns [cg*kColW, +kColW)
        const int sub = warp & 3, cg = warp >> 2;
        const int row = sub * 32 + lane;
        const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
        const float sc = p.scale_log2;
        const uint32_t tdP = tmem + 128u + lane_off + cg * kColW;
        int gs = 0;
        bool ok = true;
        for (int k = 0; ok && (PERSIST || k == 0); ++k) {
            const int w = bwd_item_index<PERSIST>(p.q_items, k);
            if (w < 0) break;
            const QItem it = q_item(p, w);
            const int n_steps = item_steps(it);
            const int qt = it.qt, q0 = qt * 128, qrow = q0 + row;
            const size_t vi = bwd_stat_off(p, it.bb, it.hh, qrow);  // qrow < s_pad always
            const int sr = bwd_stat_rank(p, it.rank, it.hh);
            const float neg_l = -p.lse2[sr][vi];
            const float neg_d = -p.dsum[sr][vi];
            const int lim = p.causal ? min(p.s, qrow + 1) : p.s;  // keys < lim are visible
            for (int n = 0; n < n_steps; ++n) {
                const int gn = gs + n;
                const uint32_t tS = sbuf(gn) + lane_off + cg * kColW;
                const int kb = n * 128 + cg * kColW;  // first key column of this warp
                // masked: the causal diagonal tile, and keys past the end (zero rows; kept out of
                // the product so that no inf/nan can reach it)
                const bool mask = (p.causal && n == qt) || kb + kColW > p.s;
                float pf[kColW];
                ok = wait_phase_warp(&bars[S_FULL + (gn & 1)], (gn >> 1) & 1, sh);
                if (!ok) break;
                tc_fence_after();
                uint32_t sv[kChunks][32];  // every chunk's load in flight before one wait
#pragma unroll
                for (int c = 0; c < kChunks; ++c) tmem_ld32(tS + c * 32, sv[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float a0, a1;
                        ffma2(a0, a1, __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]), sc, sc, neg_l, neg_l);
                        float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
                        if (mask) {
                            const int key = kb + c * 32 + e;
                            p0 = key < lim ? p0 : 0.f;
                            p1 = key + 1 < lim ? p1 : 0.f;
                        }
                        pf[c * 32 + e] = p0;
                        pf[c * 32 + e + 1] = p1;
                    }
                }
                ok = wait_phase_warp(&bars[DP_FULL], gn & 1, sh);
                if (!ok) break;
                tc_fence_after();
                uint32_t dv[kChunks][32];
#pragma unroll
                for (int c = 0; c < kChunks; ++c) tmem_ld32(tdP + c * 32, dv[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float t0, t1;
                        fadd2(t0, t1, __uint_as_float(dv[c][e]), __uint_as_float(dv[c][e + 1]), neg_d, neg_d);
                        fmul2(t0, t1, pf[c * 32 + e], pf[c * 32 + e + 1], t0, t1);
                        pk[e >> 1] = pack_bf16x2(t0, t1);
                    }
                    tmem_st16(tS + c * 16, pk);  // dS over S columns this warp has already read
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[DS_READY]);
            }
            if (ok) ok = wait_phase_warp(&bars[FINAL], k & 1, sh);
            if (!ok) break;
            constexpr int kEpi = D / kColGroups >= 32 ? D / kColGroups : 32;  // accumulator columns per warp
            if (cg * kEpi < D) {
                tc_fence_after();
                const bool qok = qrow < p.s;
                const BwdTok qt_ = bwd_tok(p, it.rank, qok ? qrow : q0);
                const size_t off =
                    (((size_t)it.bb * p.rows_per_map + qt_.row) * p.hq + it.hh) * (size_t)D * 2 + cg * kEpi * 2;
                store_row_bf16<kEpi>(tmem + 256u + lane_off + cg * kEpi, p.dq[qt_.map] + off, p.scale, qok);
            }
            gs += n_steps;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kBwdMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
// Causal band of the dK/dV items: all units when their Q and dO fit in L2 together, else as
// many as keep them within the band budget (at least one).
inline int bwd_band_units(int s_pad, int d, int g, int units) {
    const double qdo_bytes = 2.0 * g * s_pad * d * 2;  // Q and dO of one unit's query heads, bf16
    if (qdo_bytes * units <= kL2Bytes) return units;
    int bu = (int)(kBandBytes / qdo_bytes);
    if (bu < 1) bu = 1;
    if (bu > units) bu = units;
    return bu;
}

// Causal band of the dQ items, by the K and V they stream: the query heads of a band share
// the K/V heads whose tiles fit in L2 together (all units when everything fits).
inline int bwd_band_units_q(int s_pad, int d, int g, int units) {
    const double kv_bytes = 2.0 * s_pad * d * 2;  // K and V of one K/V head, bf16
    if (kv_bytes * units / g <= kL2Bytes) return units;
    int bu = (int)(kBandBytes / kv_bytes) * g;
    if (bu < 1) bu = 1;
    if (bu > units) bu = units;
    return bu;
}

template <int D, int NM>
cudaError_t launch_bwd_d(const BwdParamsT<NM>& prm_in, int nranks, cudaStream_t stream) {
    using LK = BwdSmem<D, kRingKV>;
    using LQ = BwdSmem<D, kRingQ>;
    BwdParamsT<NM> prm = prm_in;
    prm.n_units = nranks * prm.b * prm.hkv;
    prm.kv_items = prm.n_units * prm.n_tiles;
    prm.band_units = bwd_band_units(prm.s_pad, D, prm.g, prm.n_units);
    // Persistent when the static order balances the CTAs and the items are short enough for
    // their fixed cost (about 8k cycles of set-up and epilogue against 2-3k per step) to
    // matter: items all equal (non-causal), or causal in one band heaviest first with at most
    // 64 tiles (33 steps per item on average).  Other causal work runs one item per CTA in
    // unit-major order (band_units = 1): the hardware's block scheduler balances the unequal
    // items as they finish, and the CTAs running at once share the same heads' tiles in L2.
    const bool short_causal = prm.n_tiles <= 64;
    const bool persistent = !prm.causal || (short_causal && prm.band_units == prm.n_units);
    if (!persistent) prm.band_units = 1;
    prm.n_units_q = nranks * prm.b * prm.hq;
    prm.q_items = prm.n_units_q * prm.n_tiles;
    prm.band_units_q = bwd_band_units_q(prm.s_pad, D, prm.g, prm.n_units_q);
    const bool persistent_q = !prm.causal || (short_causal && prm.band_units_q == prm.n_units_q);
    if (!persistent_q) prm.band_units_q = 1;
    auto* dkdv = prm.kv_grad_f32 ? (persistent ? bwd_dkdv_kernel<D, kRowsKV, true, true, NM>
                                               : bwd_dkdv_kernel<D, kRowsKV, true, false, NM>)
                                 : (persistent ? bwd_dkdv_kernel<D, kRowsKV, false, true, NM>
                                               : bwd_dkdv_kernel<D, kRowsKV, false, false, NM>);
    auto* dq = persistent_q ? bwd_dq_kernel<D, kRowsQ, true, NM> : bwd_dq_kernel<D, kRowsQ, false, NM>;
    cudaError_t e = cudaFuncSetAttribute(dkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LK::kAlloc);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(dq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LQ::kAlloc);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // dK/dV: one CTA per SM when persistent (each CTA fills an SM: shared memory and all TMEM)
    const long long gk = persistent && prm.kv_items > sms ? sms : prm.kv_items;
    const long long gq = persistent_q && prm.q_items > sms ? sms : prm.q_items;
    dkdv<<<(unsigned)gk, RowCfg<kRowsKV>::kThreads, LK::kAlloc, stream>>>(prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dq<<<(unsigned)gq, RowCfg<kRowsQ>::kThreads, LQ::kAlloc, stream>>>(prm);
    return cudaGetLastError();
}
