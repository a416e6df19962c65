// The all-to-all exchanges with the strided side moved by TMA tensor copies.
//
// "02 · DeepSpeed-Ulysses", section 2 "all-to-all 的转置与重分布": with batch first,
//     head[r][bb][j*S + t][hh][:] == seq[j][bb][t][r*H + hh][:]      (S = s/P, H = h/P)
// For every (head rank r, seq rank j, batch bb) the head-layout side is one contiguous slab
// of S rows of `run` bytes, and the seq-layout side is the same S rows at a pitch of h*d
// elements.  Each seq-layout buffer is described to the TMA unit as a 4-D tensor
//     [b][S][cols][inner]     (inner: a divisor of the run, at most 1 KB; cols = row / inner)
// so one tensor copy moves a box of R whole runs (R rows x run bytes, up to 32 KB) between
// that buffer and shared memory, where it lies exactly as the R contiguous head-layout rows;
// the head-layout side then moves with one plain bulk copy.  seq -> head: tensor load, bulk
// store; head -> seq: bulk load, tensor store (rows past the slab's end fall outside the
// tensor and are neither read into nor written from the slab).
//
// One warp per CTA, one CTA per SM, lane 0 issues everything: a ring of kPermStages boxes,
// loads running kPermStages - 1 chunks ahead of the stores.  Chunks are dealt out round
// robin with the head rank fastest, so the CTAs working at one time cover whole seq-layout
// rows.  Every wait is bounded like the attention kernels' waits; a wait that gives up sets
// the device error word, lets the copies it issued land, and the CTA returns.

constexpr int kPermMaxMaps = 192;            // tensor maps per launch (24 KB of parameters)
constexpr uint32_t kPermStageBytes = 32768;  // one box
constexpr int kPermStages = 6;
constexpr int kPermCtasPerSm = 1;

struct TmaPermJob {
    uint64_t chunk_end;   // one past this tensor's last chunk in the launch's numbering
    uint32_t map0;        // entry of rank 0 in maps[] / contig[]
    uint32_t run;         // bytes of one head-layout row
    uint32_t col0;        // column block (of `inner` bytes) where rank 0's moved heads start
    uint32_t rank_cols;   // column blocks between consecutive ranks' head groups
    uint32_t rep;         // ranks sharing one head group (replicated K/V heads), else 1
    uint32_t R;           // rows per box
    uint32_t n_rb;        // boxes per (head rank, seq rank, batch) slab
    uint32_t box_bytes;   // R * run
};

struct TmaPermParams {
    CUtensorMap maps[kPermMaxMaps];  // seq-layout buffers, 4-D [b][S][cols][inner] of 32-bit words
    uint8_t* contig[kPermMaxMaps];   // head-layout buffers
    TmaPermJob job[4];
    uint32_t ntensors, P, S;
    uint64_t s;
    uint64_t n_chunks;
};

// Bounded single-thread wait (the permute CTA has no abort flag: one thread issues and waits).
__device__ __forceinline__ bool perm_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (error_word_set()) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicOr(&g_uly_error_word, kErrTimeout);
                return false;
            }
        }
    }
}

struct PermChunk {
    const CUtensorMap* map;  // seq-layout buffer of rank j
    uint8_t* contig;         // first head-layout byte of the box
    int col, row, bb;        // tensor coordinates of the box (inner coordinate 0)
    uint32_t box_bytes, rows_bytes;
};

__device__ __forceinline__ PermChunk perm_chunk(const TmaPermParams& p, uint64_t c) {
    uint32_t t = 0;
    while (t + 1 < p.ntensors && c >= p.job[t].chunk_end) ++t;
    const TmaPermJob& J = p.job[t];
    uint64_t x = c - (t ? p.job[t - 1].chunk_end : 0);
    const uint32_t r = (uint32_t)(x % p.P);
    x /= p.P;
    const uint32_t rb = (uint32_t)(x % J.n_rb);
    x /= J.n_rb;
    const uint32_t j = (uint32_t)(x % p.P);
    const uint32_t bb = (uint32_t)(x / p.P);
    const uint32_t row0 = rb * J.R;
    const uint32_t rows = min(J.R, p.S - row0);
    PermChunk k;
    k.map = &p.maps[J.map0 + j];
    k.contig = p.contig[J.map0 + r] + ((uint64_t)bb * p.s + (uint64_t)j * p.S + row0) * J.run;
    k.col = (int)((r / J.rep) * J.rank_cols + J.col0);
    k.row = (int)row0;
    k.bb = (int)bb;
    k.box_bytes = J.box_bytes;
    k.rows_bytes = rows * J.run;
    return k;
}

// DIR 0: seq -> head (tensor load, bulk store); DIR 1: head -> seq (bulk load, tensor store).
template <int DIR>
__global__ void __launch_bounds__(32, 1) permute_tma_kernel(const __grid_constant__ TmaPermParams p) {
    extern __shared__ __align__(1024) uint8_t perm_smem_raw[];
    __shared__ __align__(8) uint64_t bars[kPermStages];
    if (threadIdx.x != 0) return;
    const uint32_t base = (smem_addr(perm_smem_raw) + 1023u) & ~1023u;
    if (error_word_set()) return;  // an earlier kernel failed: nothing issued yet
    for (int i = 0; i < kPermStages; ++i) mbar_init(&bars[i], 1);
    fence_mbarrier_init();

    const uint64_t G = gridDim.x;
    const uint64_t n_mine = p.n_chunks > blockIdx.x ? (p.n_chunks - blockIdx.x + G - 1) / G : 0;
    auto chunk_of = [&](uint64_t i) { return perm_chunk(p, blockIdx.x + i * G); };
    auto issue_load = [&](uint64_t i) {
        const PermChunk k = chunk_of(i);
        const int st = (int)(i % kPermStages);
        const uint32_t dst = base + st * kPermStageBytes;
        if (DIR == 0) {
            mbar_arrive_expect_tx(&bars[st], k.box_bytes);
            tma_load_4d(dst, k.map, &bars[st], 0, k.col, k.row, k.bb);
        } else {
            mbar_arrive_expect_tx(&bars[st], k.rows_bytes);
            bulk_load(dst, k.contig, k.rows_bytes, &bars[st]);
        }
    };
    uint64_t loaded = 0;
    for (; loaded < n_mine && loaded < (uint64_t)kPermStages; ++loaded) issue_load(loaded);
    uint64_t i = 0;
    for (; i < n_mine; ++i) {
        const int st = (int)(i % kPermStages);
        if (!perm_wait(&bars[st], (uint32_t)((i / kPermStages) & 1))) break;
        const PermChunk k = chunk_of(i);
        const uint32_t src = base + st * kPermStageBytes;
        if (DIR == 0)
            bulk_store(k.contig, src, k.rows_bytes);
        else
            tma_store_4d(k.map, src, 0, k.col, k.row, k.bb);
        bulk_commit();
        // the previous box's store has read its stage: refill that stage
        if (i >= 1 && loaded < n_mine) {
            bulk_wait_read<1>();
            issue_load(loaded++);
        }
    }
    if (i < n_mine) {  // a wait gave up: let every load issued land before shared memory goes away
        for (uint64_t k = i; k < loaded; ++k) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&bars[k % kPermStages], (uint32_t)((k / kPermStages) & 1)) &&
                   global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
    bulk_wait<0>();  // every store has completed
}
