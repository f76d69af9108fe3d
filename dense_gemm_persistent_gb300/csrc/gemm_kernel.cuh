// gemm_kernel.cuh -- the persistent, warp-specialised tcgen05 GEMM kernel.
//
// One CTA per SM loops over output tiles in a swizzled (grouped) raster order.
// With PAIR, two CTAs of a cluster (two SMs) share one 256-row tile: each loads
// its own 128 rows of A and half of the B tile, the even CTA issues
// tcgen05.mma.cta_group::2 over both, and each CTA's Tensor Memory holds its
// 128 rows of the accumulator. Per SM this halves the B traffic from L2 and
// leaves room for more pipeline stages. The warps of a CTA split the work:
//   warp 0     TMA producer: streams 128-byte-wide K slices of A and B into an
//              S-stage shared-memory ring (128B swizzle), one mbarrier pair
//              (full / empty) per stage.
//   warp 1     MMA issuer: one thread issues tcgen05.mma for each K slice into
//              one of two FP32 accumulators in Tensor Memory and commits the
//              stage back to the producer; owns the TMEM allocation.
//   epilogue   warps 2-9 (2-5 for the small-M form and 64-wide tiles): read the
//              finished accumulator with tcgen05.ld (each warp a 32-lane quarter
//              and part of the columns, one output row per thread), apply
//              scales, alpha/beta, bias and activation in FP32, convert once,
//              and write through swizzled shared memory with TMA stores (or,
//              for the transposed small-M form, with coalesced direct stores),
//              while the MMA warp fills the other accumulator.
// Per-K-group-scale tile kernels (GS) use warp 2 as a scale producer, leave
// warp 3 idle and run the epilogue on warps 4-11; their epilogue folds every
// group's product into an FP32 running sum in registers.
//
// Work items are whole tiles or K segments of split tiles (the last partial
// wave, or every tile of a grid that does not fill the GPU); each segment
// finishes its share of the tile's 32-column units, reading the other
// segments' partials from the workspace or, when the segments form one
// cluster, from the peers' shared memory. The requantising form (MODE_ROWQ)
// turns the BF16 stash into E4M3 codes with per-row scales band by band: once
// every work item of a row band has been counted in, epilogue warps convert
// its rows between their own tiles, and the last band after their last tile.
//
// The method is the one the pages describe -- tiles of C per block, K walked in
// slices through a multi-buffered shared-memory pipeline, FP32 accumulation,
// fused epilogue (DeepGEMM write-up, czchanglian.com/news/51329, §2-§3, §6;
// "DeepGEMM: FP8 Tensor Core GEMM", bjdmk.com.cn/news/6078902, §2.2, §3.1-3.2) --
// rebuilt for sm_103a: TMA replaces cp.async, mbarriers replace
// __syncthreads/wait_prior, the hardware 128B swizzle replaces the hand XOR,
// Tensor Memory replaces register accumulators, and a persistent tile loop
// replaces the one-block-per-tile grid.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace dg {

enum Mode : int {
    MODE_TILE = 0,  // D tile stored as is (TMA store)
    MODE_SWAP = 1,  // the MMA computed D^T: store transposed with direct stores
    MODE_ROWQ = 2,  // stash y, per-row amax, E4M3 requantisation of finished row bands
};

enum ErrBits : unsigned {
    ERR_TIMEOUT_PRODUCER = 1u,
    ERR_TIMEOUT_MMA = 2u,
    ERR_TIMEOUT_EPILOGUE = 4u,
    ERR_TIMEOUT_ROW_BAND = 8u,
    ERR_TIMEOUT_DRAIN = 16u,
    ERR_ARRIVAL = 32u,   // a split tile's arrival counter could not be updated
};

struct Params {
    // Problem in the MMA's orientation: rows M, columns N, reduction K.
    int M, N, K;
    int tiles_m, tiles_n, num_tiles, k_blocks, group_m;
    int stages;      // depth of the shared-memory ring (at most the variant's STAGES)
    int tmem_cols;   // Tensor Memory columns each CTA allocates
    // K-group promotion: the K slices of a tile are split into acc_groups
    // contiguous groups, each accumulated by the tensor core into its own TMEM
    // accumulator (BN columns apart) and summed in FP32 by the epilogue.
    // acc_stride = TMEM columns between the two accumulator buffers.
    int acc_groups, acc_stride;
    float alpha, beta;
    const void* C;  // beta != 0: C in the output's orientation
    int64_t ldc;
    int c_f32;      // 1: C is FP32, 0: BF16
    void* D;        // direct-store modes: output pointer
    int64_t ldd;
    int d_f32;      // 1: D is FP32, 0: BF16 (MODE_TILE / MODE_SWAP)
    const float* row_scale;  // per MMA row, or null
    const float* col_scale;  // per MMA column, or null
    // Per-K-group scales (GS kernels): in K group j (group_kb K slices), MMA
    // row r and column c are scaled by row_gscale[j * gs_ld_row + r] *
    // col_gscale[j * gs_ld_col + c] before the groups are summed.
    const float* row_gscale;
    const float* col_gscale;
    int64_t gs_ld_row, gs_ld_col;
    // Block-scaled weights: one scale per (K group, block of 2^shift MMA rows /
    // columns) instead of one per row / column (0 = per row / column). Entry
    // of row m in group j: row_gscale[j * gs_ld_row + (m >> gs_row_shift)].
    int gs_row_shift, gs_col_shift;
    int group_kb;
    const float* bias;       // per output channel, or null
    int act;                 // 0 none, 1 ReLU, 2 GELU (erf), 3 SiLU
    // MODE_ROWQ
    unsigned* amax;          // [M] |y| maxima as float bits; zero before launch
    unsigned long long* rq_next;   // requantisation chunks claimed so far; zero before launch
    unsigned* band_count;    // [row bands] epilogue-warp arrivals per band; zero before launch
    int rq_gpc;              // raster groups per row band
    const uint16_t* stash;   // [M,N] BF16 y values (what tmD writes)
    uint8_t* q_out;          // [M,N] E4M3 codes
    float* out_row_scale;    // [M]
    unsigned* status;        // sticky device error word (calls without a workspace status word)
    // The call's status word in the caller's workspace, or null: (epoch << 8) |
    // error bits, tagged with this launch's epoch so that a word left by an
    // earlier launch (or any other data) is replaced instead of merged.
    unsigned long long* ws_status;
    uint64_t wait_ns;        // limit of every bounded device-side wait
    // Testing of the bounded waits: < 0 off; otherwise the TMA producer of
    // every CTA stops after issuing this many stage loads, so that the MMA's
    // wait for the next stage runs out and the kernel drains and returns.
    long long stall_after;
    // Split tiles (all modes): tiles [0, dp_tiles) run whole; each of the
    // remaining tiles is split along K into `split` segments (tail_items in
    // all), every unit taking at most one (before its whole tiles, if any;
    // with seg_first the split tiles are the first num_tiles - dp_tiles of the
    // raster instead of the last).
    // 32-column unit u of each epilogue warp's region belongs to segment
    // u % split: a segment parks the units others own as FP32 partials in
    // `partials`, counts its arrival in tail_count, waits (bounded) for every
    // segment of the region, and finishes its own units from its accumulator
    // plus the others' partials.
    int dp_tiles, split, tail_items;
    int seg_first;           // 1: a unit runs its split item before its whole tiles
    float* partials;         // [tail_items][CTAS][EPI_WARPS][units][UNIT/4][32 lanes] float4
    // Split-K through distributed shared memory (single-CTA kernels, under-
    // filled grids): the split K segments of a tile are the CTAs of one
    // cluster of `split` CTAs (rank = segment); partials go through the idle
    // pipeline buffers and the peers' shared memory instead of the workspace.
    int cluster_split;
    // Tail tiles split along N instead (CTA-pair 256-wide kernels): each of
    // the tiles from dp_tiles on is run as two 256 x 128 halves (tail_items =
    // 2 x those tiles), each a whole K range with an N = 128 MMA; no partials.
    int tail_halves;
    // [split tile][CTAS][EPI_WARPS]: (epoch << 8) | (parked << 4) | arrivals
    unsigned long long* tail_count;
    unsigned long long epoch;        // unique per launch (56 bits): stale counters need no clearing
    // Exchange of a split tile's partial sums through the workspace.
    // 1 (the launch is cooperative, so every segment is resident): every
    //   segment parks the units others own, waits for all, and finishes its own.
    // 0 (no residency guarantee): no segment waits for one that may not have
    //   started. A segment counts its arrival first; all but the last to arrive
    //   park every unit and leave, and the last waits only for those (already
    //   running) segments' parking, then finishes every unit.
    int split_sym;
};

// One unit of work: a whole tile (item < 0) or one K segment of a split tile.
struct Work {
    int tile, kb0, kb1, item;
    int half;   // -1: the whole tile; 0 / 1: that 128-column half (tail_halves)
};

// The iter-th work item of a unit (a CTA, or a CTA pair): its whole tiles
// unit, unit + units, ... (dp_tiles of them in all), then its tail item (a K
// segment or an N half of a split tile), or with seg_first its K segment first.
__device__ __forceinline__ bool next_work(const Params& p, int unit, int units, int iter, Work& w) {
    // With seg_first, a unit's K segment of a split tile runs before its whole
    // tiles, so that the segments' exchange of partial sums (a chain of L2 round
    // trips) overlaps the next tile's mainloop instead of ending the kernel.
    // Every segment of a split tile is then its unit's first item, all running
    // at once, and the split tiles are the raster's first ones (tiles [0, S),
    // whole tiles from S on), next to the whole tiles started alongside them.
    const bool front = p.seg_first && p.split > 1 && !p.tail_halves && p.dp_tiles > 0;
    const bool seg_first = front && unit < p.tail_items;
    const int dp0 = front ? p.num_tiles - p.dp_tiles : 0;   // first whole tile
    if (seg_first) {
        if (iter == 0) {
            const int seg = unit % p.split;
            w.half = -1;
            w.tile = unit / p.split;
            w.kb0 = (seg * p.k_blocks) / p.split;
            w.kb1 = ((seg + 1) * p.k_blocks) / p.split;
            w.item = unit;
            return true;
        }
        --iter;
    }
    const int dp_count = p.dp_tiles > unit ? (p.dp_tiles - unit + units - 1) / units : 0;
    w.half = -1;
    if (iter < dp_count) {
        w.tile = dp0 + unit + iter * units;
        w.kb0 = 0;
        w.kb1 = p.k_blocks;
        w.item = -1;
        return true;
    }
    if (seg_first) return false;   // its split item ran first
    const int j = unit + (iter - dp_count) * units;
    if (j >= p.tail_items) return false;
    if (p.tail_halves) {
        w.tile = p.dp_tiles + j / 2;
        w.half = j % 2;
        w.kb0 = 0;
        w.kb1 = p.k_blocks;
        w.item = -1;
        return true;
    }
    const int seg = j % p.split;
    w.tile = p.dp_tiles + j / p.split;
    w.kb0 = (seg * p.k_blocks) / p.split;
    w.kb1 = ((seg + 1) * p.k_blocks) / p.split;
    w.item = j;
    return true;
}



template <int BN_, bool FP8_, bool A_MN_, bool B_MN_, int MODE_, bool PAIR_ = false, bool GS_ = false, int KS_ = 1>
struct Cfg {
    static constexpr int BM = 128;                // accumulator rows per CTA
    static constexpr bool PAIR = PAIR_;
    static constexpr int CTAS = PAIR ? 2 : 1;     // CTAs sharing one tile
    static constexpr int TILE_M = BM * CTAS;      // output rows per tile
    static constexpr int BN = BN_;
    static constexpr bool FP8 = FP8_;
    static constexpr bool A_MN = A_MN_;
    static constexpr bool B_MN = B_MN_;
    static constexpr int MODE = MODE_;
    // Per-K-group scales: each group's product goes to one of two TMEM
    // buffers and the epilogue warps fold it, scaled, into FP32 registers.
    static constexpr bool GS = GS_;
    static constexpr int ESZ = FP8 ? 1 : 2;       // operand bytes
    static constexpr int BK = 128 / ESZ;          // K elements per stage (128 bytes)
    static constexpr int UMMA_K = 32 / ESZ;       // K elements per MMA (32 bytes)
    static constexpr int MN_ATOM = 128 / ESZ;     // MN elements per 128-byte row (MN-major)
    // K slices (128 bytes of K each) per pipeline stage. With 2, each operand
    // of a stage arrives in one 3-D TMA copy of two consecutive slices (the
    // TMA unit fills a CTA's shared memory ~16 % faster in 32 KB copies than
    // in 16 KB ones); the slices land one after the other, each an ordinary
    // 128B-swizzled slice (K-major), or the N atoms hold 2 x BK rows of K each
    // (MN-major B).
    static constexpr int KS = KS_;
    static constexpr int SLICE_A = BM * 128;      // bytes of one K slice of A
    static constexpr int A_BYTES = KS * BM * 128;
    static constexpr int BN_CTA = BN / CTAS;      // B rows (N) each CTA loads
    static constexpr int SLICE_B = BN_CTA * 128;  // bytes of one K slice of B (K-major)
    static constexpr int B_BYTES = KS * BN_CTA * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // Epilogue warps: two per TMEM lane quarter (each takes half of the tile's
    // columns) for tiles of 128 columns or more, whose FP8 mainloop per tile can
    // be shorter than one warp-quarter's epilogue, and for the 16-wide small-M
    // form, whose epilogue sums up to 32 K-group accumulators at the end of the
    // call (a warp reads TMEM at a fixed rate, so two warps a quarter halve
    // that; its 320 threads still fit twice in an SM's registers for the
    // compact footprint); one per quarter otherwise.
    static constexpr int EPI_WARPS = (MODE == MODE_SWAP) ? ((GS || BN != 16) ? 4 : 8) : (BN < 128 ? 4 : 8);
    static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);   // columns per epilogue warp
    static constexpr int STAGING_BYTES = (MODE == MODE_SWAP) ? 0 : EPI_WARPS * 4096;  // one 4 KB box each
    // Per-K-group scales (tile modes): a scale-producer warp copies each
    // group's BN column scales and this CTA's 128 row scales into a ring of
    // SC_SLOTS shared-memory slots ahead of the epilogue (the small-M form
    // reads its few scales directly).
    static constexpr bool GS_SMEM = GS && MODE != MODE_SWAP;
    static constexpr int SC_SLOTS = GS_SMEM ? 4 : 0;
    static constexpr int SLOT_FLOATS = BN + BM;
    static constexpr int GS_BYTES = SC_SLOTS * SLOT_FLOATS * 4;
    static constexpr int BAR_BYTES = GS_SMEM ? 384 : 256;
    static constexpr int SMEM_LIMIT = 232448;  // 227 KB opt-in maximum per CTA
    static constexpr int SMEM_FIXED = 1024 + STAGING_BYTES + GS_BYTES + BAR_BYTES;   // all but the ring
    static constexpr int STAGES_FIT = (SMEM_LIMIT - SMEM_FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
    // The small-M (transposed) form also runs in a compact footprint, chosen
    // per call for short calls: at most half of an SM's 228 KB of shared
    // memory (less the 1 KB the hardware reserves per CTA) and half of its
    // Tensor Memory, so that the next call's CTAs become resident and run their
    // prologue while this call's finish (programmatic dependent launch).
    static constexpr int STAGES_HALF_FIT = (115712 - SMEM_FIXED) / STAGE_BYTES;
    static constexpr int STAGES_COMPACT =
        (MODE == MODE_SWAP && STAGES_HALF_FIT < STAGES) ? STAGES_HALF_FIT : STAGES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + GS_BYTES + BAR_BYTES;
    static constexpr int TMEM_COLS = (MODE == MODE_SWAP && !GS) ? 512
                                   : (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
    static constexpr uint32_t IDESC = make_idesc(FP8 ? 0u : 1u, A_MN, B_MN, TILE_M, BN);
    // tail halves (PAIR, BN = 256): N = 128 per pair, 64 B rows per CTA
    // Tail tiles as two N halves: each CTA loads 64 rows of B (K-major), or
    // whole 128-byte atoms of it (MN-major; one for BF16, none fits for E4M3).
    static constexpr bool HALVES = PAIR && BN == 256 && !GS && (!B_MN || (BN_CTA / 2) % MN_ATOM == 0);
    static constexpr uint32_t IDESC_HALF = make_idesc(FP8 ? 0u : 1u, A_MN, B_MN, TILE_M, BN / 2);
    static constexpr int B_BYTES_HALF = KS * (BN_CTA / 2) * 128;
    // Per-K-group scales keep each epilogue thread's share of the running sum
    // (EPI_COLS FP32 values) in registers. With 8 epilogue warps that needs more
    // than the 168 registers a thread of a 10-warp block can have, so those
    // kernels run 12 warps as three warpgroups -- producer, MMA issuer and two
    // idle warps, then the 8 epilogue warps -- and move registers from the
    // first warpgroup to the others (setmaxnreg).
    static constexpr bool REG_SPLIT = GS && EPI_WARPS == 8;
    // first epilogue warp: the per-group tile kernels use warp 2 as the scale
    // producer (warp 3 idles), the split kernels need whole warpgroups
    static constexpr int EPI_WARP0 = (REG_SPLIT || GS_SMEM) ? 4 : 2;
    static constexpr int NUM_THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    static constexpr int LAUNCH_REGS = 168;   // per thread at launch (12 warps: 3 per SM sub-partition)
    static constexpr int REGS_LOW = 56, REGS_HIGH = 224;
    static_assert(!REG_SPLIT || 128 * REGS_LOW + 32 * EPI_WARPS * REGS_HIGH <= NUM_THREADS * LAUNCH_REGS,
                  "register split exceeds the launch allocation");

    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128");
    static_assert(KS == 1 || (KS == 2 && !GS && !A_MN && MODE != MODE_SWAP && (PAIR || MODE == MODE_TILE)),
                  "two-slice stages: tile forms");
    static_assert(!B_MN || BN_CTA % MN_ATOM == 0, "MN-major B needs whole 128-byte atoms");
    static_assert(!PAIR || (MODE != MODE_SWAP && !A_MN && BN == 256), "CTA pairs: 256 x 256 tiles");
    static_assert(MODE == MODE_SWAP || EPI_COLS % 64 == 0, "tile epilogue works in 64-column boxes");
    static_assert(STAGES >= 2 && STAGES_COMPACT >= 2, "pipeline depth");
    static_assert(!GS || (FP8 && MODE != MODE_ROWQ), "per-K-group scales: FP8, tile or small-M form");
    // block-scaled weights: a warp's columns lie inside one 128-column block
    static_assert(!GS_SMEM || 128 % EPI_COLS == 0, "warp columns within a weight block");
    static_assert(BN < 32 || BN % 32 == 0, "epilogue reads 32-column units");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
    // full/empty per stage, 2 + 2 accumulator, drain, scale slots; TMEM address + abort flag
    static_assert((2 * STAGES + 5 + 2 * SC_SLOTS) * 8 + 8 <= BAR_BYTES, "barriers fit");
    // split-K through the cluster parks a whole accumulator in the pipeline buffers
    static_assert(EPI_WARPS * BN / (EPI_WARPS / 4) * 32 * 4 <= STAGES_COMPACT * STAGE_BYTES, "parked partials fit");
};

__device__ __forceinline__ void tile_coords(int t, const Params& p, int& mb, int& nb) {
    // Grouped raster: bands of group_m tile-rows; inside a band, walk down the
    // rows first, then across the columns, so CTAs resident at the same time
    // share A row-strips and B column-strips in L2.
    const int group_tiles = p.group_m * p.tiles_n;
    const int g = t / group_tiles;
    const int first_m = g * p.group_m;
    const int rows = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * group_tiles;
    mb = first_m + r % rows;
    nb = r / rows;
}

// Row bands of the requantising form: rq_gpc raster groups (group_m tile rows
// with all their tile columns, consecutive in the raster) each, so that the
// band counters fit the workspace header. A band's rows are final once every
// epilogue warp of every CTA has counted in every work item of its tiles.
constexpr int kMaxBands = 62;
constexpr int RQ_CHUNK = 4096;   // values of one row converted per claim (16 x 16 bytes per lane)

__device__ __forceinline__ int band_of_tile(const Params& p, int t) {
    return t / (p.group_m * p.tiles_n) / p.rq_gpc;
}

template <class CF>
__device__ __forceinline__ unsigned band_expected(const Params& p, int b) {
    const int t0 = b * p.rq_gpc * p.group_m * p.tiles_n;
    const int t1 = min((b + 1) * p.rq_gpc * p.group_m, p.tiles_m) * p.tiles_n;
    const int tail = max(0, t1 - max(t0, p.dp_tiles));   // split tiles: several items each
    const int extra = p.tail_halves ? 1 : p.split - 1;
    return static_cast<unsigned>(t1 - t0 + tail * extra) * CF::CTAS * CF::EPI_WARPS;
}

// Activations applied to 32 values at once; the switch is taken once per
// 32-column unit so the per-element code is straight-line and interleaves.
// SiLU uses the fast exponential and division: their relative error (a few
// units of 2^-22) is far below the BF16 / E4M3 output rounding.
__device__ __forceinline__ void activation32(float (&v)[32], int act) {
    switch (act) {
        case 1:
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.0f);
            break;
        case 2:
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.5f * v[j] * (1.0f + erff(v[j] * 0.70710678118654752f));
            break;
        case 3:
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __fdividef(v[j], 1.0f + __expf(-v[j]));
            break;
        default:
            break;
    }
}

// Records error bits: in the call's workspace status word when it has one
// (tagged with the launch epoch), else in the per-device word.
__device__ __forceinline__ void record_error(const Params& p, unsigned bit) {
    if (p.ws_status != nullptr) {
        unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(p.ws_status);
        for (int tries = 0; tries < 4096; ++tries) {
            const bool mine = (old >> 8) == p.epoch;
            if (mine && (old & bit) == bit) return;
            const unsigned long long next = mine ? (old | bit) : ((p.epoch << 8) | bit);
            const unsigned long long seen = atomicCAS(p.ws_status, old, next);
            if (seen == old) return;
            old = seen;
        }
    }
    atomicOr(p.status, bit);   // no workspace word (or it could not be updated)
}

__device__ __forceinline__ void raise_error(const Params& p, unsigned bit, volatile int* abort) {
    record_error(p, bit);
    *abort = 1;
}

// Loads base[idx .. idx+3] (every lane of the warp reads the same address);
// entries at or beyond n read as 0. base must be 16-byte aligned, idx % 4 == 0.
__device__ __forceinline__ float4 ld_bcast4(const float* base, int idx, int n) {
    if (idx + 3 < n) return __ldg(reinterpret_cast<const float4*>(base + idx));
    float4 r;
    r.x = idx < n ? __ldg(base + idx) : 0.0f;
    r.y = idx + 1 < n ? __ldg(base + idx + 1) : 0.0f;
    r.z = idx + 2 < n ? __ldg(base + idx + 2) : 0.0f;
    r.w = 0.0f;
    return r;
}

// Per-K-group scales: sum[c] += P[c] * rs * s[c] for the UNIT columns of one
// Tensor Memory load, in packed FP32 pairs.
__device__ __forceinline__ void gs_fold4(float* sum, const uint32_t* r, float rs, float4 s) {
    float w0, w1, w2, w3;
    fmul2(w0, w1, s.x, s.y, rs, rs);
    fmul2(w2, w3, s.z, s.w, rs, rs);
    ffma2(sum[0], sum[1], __uint_as_float(r[0]), __uint_as_float(r[1]), w0, w1);
    ffma2(sum[2], sum[3], __uint_as_float(r[2]), __uint_as_float(r[3]), w2, w3);
}

// Column scales from a shared-memory copy of this warp's columns (broadcast reads).
template <int UNIT>
__device__ __forceinline__ void gs_fold_smem(float* sum, const uint32_t (&r)[UNIT], float rs, const float* cs) {
#pragma unroll
    for (int c = 0; c < UNIT; c += 4) gs_fold4(sum + c, r + c, rs, *reinterpret_cast<const float4*>(cs + c));
}

// One scale for all of this warp's columns (block-scaled weights: the warp's
// columns lie in one block), so one fused multiply-add per output per group.
template <int UNIT>
__device__ __forceinline__ void gs_fold_uniform(float* sum, const uint32_t (&r)[UNIT], float s) {
#pragma unroll
    for (int c = 0; c < UNIT; c += 2) ffma2(sum[c], sum[c + 1], __uint_as_float(r[c]), __uint_as_float(r[c + 1]), s, s);
}

// Column scales read from global memory one by one (the small-M form, whose
// column scale table has any row length); columns at or beyond ncols get 0.
template <int UNIT>
__device__ __forceinline__ void gs_fold(float* sum, const uint32_t (&r)[UNIT], float rs, const float* cs, int col,
                                        int ncols) {
#pragma unroll
    for (int c = 0; c < UNIT; c += 4) {
        float4 s;
        s.x = col + c < ncols ? __ldg(cs + col + c) : 0.0f;
        s.y = col + c + 1 < ncols ? __ldg(cs + col + c + 1) : 0.0f;
        s.z = col + c + 2 < ncols ? __ldg(cs + col + c + 2) : 0.0f;
        s.w = col + c + 3 < ncols ? __ldg(cs + col + c + 3) : 0.0f;
        gs_fold4(sum + c, r + c, rs, s);
    }
}

// Column j of a warp's columns from the per-lane float4 vectors that hold
// them (lane l holds columns 4l .. 4l + 3): a warp shuffle, no memory access.
__device__ __forceinline__ float4 lane_f4(const float4& x, int src_lane) {
    return make_float4(__shfl_sync(0xffffffffu, x.x, src_lane), __shfl_sync(0xffffffffu, x.y, src_lane),
                       __shfl_sync(0xffffffffu, x.z, src_lane), __shfl_sync(0xffffffffu, x.w, src_lane));
}

// The FP32 epilogue arithmetic shared by all modes for 32 consecutive columns
// of one row: v = alpha * (rs * cs[j] * acc) + beta * c[j] + bias[j], then act.
// Tile modes take the column scales and bias from per-lane float4 vectors
// loaded before the accumulator was ready (cs_l, bias_l: lane l holds the
// warp's columns 4l .. 4l + 3; this unit starts at lane lane0); the
// transposed small-M form reads its column scales directly.
template <bool SWAP>
__device__ __forceinline__ void epilogue_math(float (&v)[32], const Params& p, int row, int col0,
                                              int ncols, float rs, float bias_row, const float4& cs_l,
                                              const float4& bias_l, int lane0, const float4* cs_sw) {
    const bool row_ok = row < p.M;
    // column-indexed scale (per MMA column)
    if (p.col_scale) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            if (j < ncols) {
                float4 s;
                if constexpr (SWAP)
                    s = cs_sw[j / 4];
                else
                    s = lane_f4(cs_l, lane0 + j / 4);
                v[j] *= s.x; v[j + 1] *= s.y; v[j + 2] *= s.z; v[j + 3] *= s.w;
            }
        }
    }
    const float a = p.alpha * rs;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= a;
    if (p.beta != 0.0f && row_ok) {
        if constexpr (!SWAP) {
            // C row segment, in the output's orientation: row-major, this thread's row.
            if (p.c_f32) {
                const float* c = static_cast<const float*>(p.C) + row * p.ldc + col0;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    if (j < ncols && col0 + j < p.N) {
                        const float4 cv = *reinterpret_cast<const float4*>(c + j);
                        v[j] += p.beta * cv.x; v[j + 1] += p.beta * cv.y;
                        v[j + 2] += p.beta * cv.z; v[j + 3] += p.beta * cv.w;
                    }
            } else {
                const uint16_t* c = static_cast<const uint16_t*>(p.C) + row * p.ldc + col0;
#pragma unroll
                for (int j = 0; j < 32; j += 8)
                    if (j < ncols && col0 + j < p.N) {
                        const uint4 cv = *reinterpret_cast<const uint4*>(c + j);
                        const uint32_t w[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            v[j + 2 * h] += p.beta * bf16_lo(w[h]);
                            v[j + 2 * h + 1] += p.beta * bf16_hi(w[h]);
                        }
                    }
            }
        } else {
            // Transposed: MMA column j is output row j, MMA row is output column.
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < ncols && col0 + j < p.N) {
                    const int64_t off = static_cast<int64_t>(col0 + j) * p.ldc + row;
                    const float cv = p.c_f32 ? static_cast<const float*>(p.C)[off]
                                             : __uint_as_float(static_cast<uint32_t>(
                                                   static_cast<const uint16_t*>(p.C)[off]) << 16);
                    v[j] += p.beta * cv;
                }
        }
    }
    if constexpr (SWAP) {
        if (p.bias) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += bias_row;
        }
    } else {
        if (p.bias) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                if (j < ncols) {
                    const float4 b = lane_f4(bias_l, lane0 + j / 4);
                    v[j] += b.x; v[j + 1] += b.y; v[j + 2] += b.z; v[j + 3] += b.w;
                }
        }
    }
    activation32(v, p.act);
}

// Converts 32 finished values of this thread's row and stages them; every
// 128-byte box row (32 FP32 or 64 BF16 columns) is sent with one TMA store per
// warp (32 rows). One 4 KB staging box per warp: before refilling it, the
// previous box's store must have finished reading it.
template <class CF>
__device__ __forceinline__ void tile_store_unit(const float (&v)[32], const Params& p, int u, int col0, int row_base,
                                                int lane, uint8_t* box, int& stores, const CUtensorMap* tmD) {
    const bool f32_out = (CF::MODE == MODE_TILE) && p.d_f32;
    const int half = f32_out ? 0 : (u & 1);
    if (half == 0) {
        if (stores >= 1 && lane == 0) bulk_wait_read<0>();
        __syncwarp();
    }
    uint8_t* rowp = box + lane * 128;
    const int sw = lane & 7;
    if (f32_out) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 wv = make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                                        __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
            *reinterpret_cast<uint4*>(rowp + ((c ^ sw) << 4)) = wv;
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 wv = make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                        pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                                        pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
            *reinterpret_cast<uint4*>(rowp + (((half * 4 + c) ^ sw) << 4)) = wv;
        }
    }
    if (f32_out || half == 1) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            // outputs (and the requantising stash) are not read again before
            // they leave L2: let them go first, ahead of the evict-last operands
            tma_store_2d_hint(tmD, box, f32_out ? col0 : col0 - 32, row_base, policy_evict_first());
            bulk_commit();
        }
        ++stores;
    }
}

template <class CF>
__global__ void __launch_bounds__(CF::NUM_THREADS, 1)
    gemm_persistent(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBh,
                    const __grid_constant__ CUtensorMap tmD, const Params p) {
    // ring depth: chosen per launch for the small-M form (compact or full),
    // fixed for the others
    const int S = CF::MODE == MODE_SWAP ? p.stages : CF::STAGES;
    const uint32_t tmem_cols = CF::MODE == MODE_SWAP ? static_cast<uint32_t>(p.tmem_cols) : CF::TMEM_COLS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint8_t* staging = smem + S * CF::STAGE_BYTES;
    float* gs_area = reinterpret_cast<float*>(staging + CF::STAGING_BYTES);   // GS scale slots
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + CF::STAGING_BYTES + CF::GS_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* acc_full = bars + 2 * S;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint64_t* sc_full = drain + 1;                 // GS scale slots: filled / free
    uint64_t* sc_empty = sc_full + CF::SC_SLOTS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sc_empty + CF::SC_SLOTS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pairs: rank 0 is the leader that issues the MMAs; a tile is shared by
    // the pair, so the tile loop runs over pairs.
    const uint32_t rank = CF::PAIR ? cluster_ctarank() : 0u;
    const int unit0 = static_cast<int>(blockIdx.x) / CF::CTAS;
    const int units = static_cast<int>(gridDim.x) / CF::CTAS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], CF::EPI_WARPS * CF::CTAS);  // every epilogue warp of the pair
        }
        mbar_init(drain, 1);
        for (int sl = 0; sl < CF::SC_SLOTS; ++sl) {
            mbar_init(&sc_full[sl], 32);               // every lane of the scale producer
            mbar_init(&sc_empty[sl], CF::EPI_WARPS);   // every epilogue warp of this CTA
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        if (p.k_blocks > 0) {  // with K == 0 the operand maps are not encoded
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
        }
        if (CF::MODE != MODE_SWAP) tma_prefetch_desc(&tmD);
    }
    if constexpr (CF::PAIR) {
        // the peer's barriers must be initialised before any cross-CTA signal
        __syncthreads();
        cluster_sync();
        if (warp == 1) {
            tmem_alloc_pair(tmem_slot, tmem_cols);
            tmem_relinquish_pair();
        }
        tc_fence_before();
        __syncthreads();
        cluster_sync();
    } else {
        if (warp == 1) {
            tmem_alloc(tmem_slot, tmem_cols);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
    }
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above (barriers, TMEM, descriptor prefetch) may overlap the
    // previous kernel in the stream; global memory is touched only from here.
    grid_dependency_wait();
    if (threadIdx.x == 0) grid_launch_dependents();

    if (warp < CF::EPI_WARP0) {
        // Register reallocation happens once per warpgroup, at one point in
        // each role's branch (the code after it is compiled to that count).
        if constexpr (CF::REG_SPLIT) regs_dec<CF::REGS_LOW>();
        if (warp == 0) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                const uint64_t pol = policy_evict_last();
                uint32_t stage = 0, phase = 0;
                int64_t issued = 0;
                bool ok = true, stalled = false;
                Work w;
                for (int it = 0; ok && !stalled && next_work(p, unit0, units, it, w); ++it) {
                    int mb, nb;
                    tile_coords(w.tile, p, mb, nb);
                    const int row0 = mb * CF::TILE_M + static_cast<int>(rank) * CF::BM;   // this CTA's A rows
                    // this CTA's B rows (of a tail half: its 64 of the half's 128)
                    const bool half = CF::HALVES && w.half >= 0;
                    const int col0 = half ? nb * CF::BN + w.half * (CF::BN / 2) + static_cast<int>(rank) * (CF::BN_CTA / 2)
                                          : nb * CF::BN + static_cast<int>(rank) * CF::BN_CTA;
                    for (int kb = w.kb0; kb < w.kb1; ++kb) {
                        if (issued == p.stall_after) {   // testing the bounded waits: stop here
                            stalled = true;
                            break;
                        }
                        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        uint8_t* sa = stages + stage * CF::STAGE_BYTES;
                        uint8_t* sb = sa + CF::A_BYTES;
                        const int k0 = kb * CF::KS * CF::BK;   // first K element of the stage
                        if constexpr (CF::PAIR && CF::KS == 2) {
                            // one 3-D copy per operand: slices kb * 2 and kb * 2 + 1
                            if (rank == 0)
                                mbar_arrive_expect_tx(&full[stage],
                                                      CF::CTAS * (half ? CF::A_BYTES + CF::B_BYTES_HALF : CF::STAGE_BYTES));
                            const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                            tma_load_3d_pair(sa, &tmA, fb, 0, row0, kb * 2, pol);
                            if constexpr (CF::B_MN)   // atoms of MN_ATOM columns, 2 x BK rows of K each
                                tma_load_3d_pair(sb, half ? &tmBh : &tmB, fb, 0, k0, col0 / CF::MN_ATOM, pol);
                            else
                                tma_load_3d_pair(sb, half ? &tmBh : &tmB, fb, 0, col0, kb * 2, pol);
                        } else if constexpr (CF::PAIR) {
                            // both CTAs' copies complete on the leader's full barrier
                            if (rank == 0)
                                mbar_arrive_expect_tx(&full[stage],
                                                      CF::CTAS * (half ? CF::A_BYTES + CF::B_BYTES_HALF : CF::STAGE_BYTES));
                            const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                            tma_load_2d_pair(sa, &tmA, fb, k0, row0, pol);
                            if constexpr (CF::B_MN) {
                                // 128-byte atoms of MN_ATOM columns each (a half loads the first ones only)
                                const int atoms = (half ? CF::BN_CTA / 2 : CF::BN_CTA) / CF::MN_ATOM;
    #pragma unroll
                                for (int i = 0; i < CF::BN_CTA / CF::MN_ATOM; ++i)
                                    if (i < atoms)
                                        tma_load_2d_pair(sb + i * CF::BK * 128, &tmB, fb, col0 + i * CF::MN_ATOM, k0, pol);
                            } else {
                                tma_load_2d_pair(sb, half ? &tmBh : &tmB, fb, k0, col0, pol);
                            }
                        } else if constexpr (CF::KS == 2) {
                            // one 3-D copy per operand: slices kb * 2 and kb * 2 + 1
                            mbar_arrive_expect_tx(&full[stage], CF::STAGE_BYTES);
                            tma_load_3d(sa, &tmA, &full[stage], 0, row0, kb * 2, pol);
                            if constexpr (CF::B_MN)   // atoms of MN_ATOM columns, 2 x BK rows of K each
                                tma_load_3d(sb, &tmB, &full[stage], 0, k0, col0 / CF::MN_ATOM, pol);
                            else
                                tma_load_3d(sb, &tmB, &full[stage], 0, col0, kb * 2, pol);
                        } else {
                            mbar_arrive_expect_tx(&full[stage], CF::STAGE_BYTES);
                            if constexpr (CF::A_MN) {
    #pragma unroll
                                for (int i = 0; i < CF::BM / CF::MN_ATOM; ++i)
                                    tma_load_2d(sa + i * CF::BK * 128, &tmA, &full[stage], row0 + i * CF::MN_ATOM, k0,
                                                pol);
                            } else {
                                tma_load_2d(sa, &tmA, &full[stage], k0, row0, pol);
                            }
                            if constexpr (CF::B_MN) {
    #pragma unroll
                                for (int i = 0; i < CF::BN_CTA / CF::MN_ATOM; ++i)
                                    tma_load_2d(sb + i * CF::BK * 128, &tmB, &full[stage], col0 + i * CF::MN_ATOM, k0,
                                                pol);
                            } else {
                                tma_load_2d(sb, &tmB, &full[stage], k0, col0, pol);
                            }
                        }
                        ++issued;
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
                if (!ok) raise_error(p, ERR_TIMEOUT_PRODUCER, abort_flag);
                // Drain: every copy this thread issued must have landed before the
                // CTA can exit (normally these waits return at once). The peer of a
                // pair signals the leader's full barriers, so it waits instead for
                // the MMA's release of its last use of each stage.
                for (int s = 0; s < S; ++s) {
                    const int64_t cnt = issued > s ? (issued - s + S - 1) / S : 0;
                    uint64_t* bar = (CF::PAIR && rank != 0) ? &empty[s] : &full[s];
                    if (cnt > 0 && !mbar_wait(bar, static_cast<uint32_t>((cnt - 1) & 1), nullptr, p.wait_ns))
                        raise_error(p, ERR_TIMEOUT_DRAIN, abort_flag);
                }
            }
            __syncwarp();
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0 && rank == 0) {
                // The tensor core's instruction queue is shallow (issue time equals
                // execution time), so this loop must spend almost nothing between
                // MMAs: descriptors are built once and advanced by additions, and
                // K-group boundaries are tracked incrementally (a division per K
                // slice here measurably starves the tensor pipe).
                const uint32_t s0 = smem_u32(stages);
                const uint64_t a_desc0 = smem_desc_sw128(s0, CF::A_MN ? CF::BK * 128 : 16, 1024);
                // (MN-major B: N atoms KS x BK rows of K apart)
                const uint64_t b_desc0 =
                    smem_desc_sw128(s0 + CF::A_BYTES, CF::B_MN ? CF::KS * CF::BK * 128 : 16, 1024);
                constexpr uint32_t A_KSTEP = (CF::A_MN ? CF::UMMA_K * 128 : 32) >> 4;
                constexpr uint32_t B_KSTEP = (CF::B_MN ? CF::UMMA_K * 128 : 32) >> 4;
                constexpr uint32_t STAGE_STEP = CF::STAGE_BYTES >> 4;
                const int kblocks = p.k_blocks, ngroups = p.acc_groups;
                uint32_t stage = 0, phase = 0;
                bool ok = true;
                int local = 0;
                Work w;
                // The MMAs of one pipeline stage (KS K slices of NK1 MMAs each) into
                // accumulator d_tmem; `first` starts a fresh accumulation. b_slice:
                // descriptor step between the stage's K slices of K-major B (a tail
                // half's B slices are half as tall).
                constexpr int NK1 = CF::BK / CF::UMMA_K;
                constexpr uint32_t A_SLICE = CF::SLICE_A >> 4;
                auto issue_stage = [&](uint32_t d_tmem, uint32_t st, bool first, uint32_t idesc, uint32_t b_slice) {
                    const uint64_t ad = a_desc0 + st * STAGE_STEP;
                    const uint64_t bd = b_desc0 + st * STAGE_STEP;
    #pragma unroll
                    for (int k = 0; k < CF::KS * NK1; ++k) {
                        const uint32_t acc = (!first || k > 0) ? 1u : 0u;
                        const uint32_t ao = (k / NK1) * A_SLICE + (k % NK1) * A_KSTEP;
                        const uint32_t bo = CF::B_MN ? k * B_KSTEP : (k / NK1) * b_slice + (k % NK1) * B_KSTEP;
                        if constexpr (CF::PAIR) {
                            if constexpr (CF::FP8)
                                mma_f8_pair(d_tmem, ad + ao, bd + bo, idesc, acc);
                            else
                                mma_bf16_pair(d_tmem, ad + ao, bd + bo, idesc, acc);
                        } else {
                            if constexpr (CF::FP8)
                                mma_f8(d_tmem, ad + ao, bd + bo, idesc, acc);
                            else
                                mma_bf16(d_tmem, ad + ao, bd + bo, idesc, acc);
                        }
                    }
                    // the stage is free (in both CTAs of a pair) once these MMAs have read it
                    if constexpr (CF::PAIR)
                        mma_commit_pair(&empty[st], 3);
                    else
                        mma_commit(&empty[st]);
                };
                if constexpr (CF::GS) {
                    // Per-K-group scales: every scale group of every work item gets
                    // its own accumulator, alternating between the two TMEM buffers
                    // (gcount counts groups over the whole loop, so the epilogue can
                    // fold one group while the next is computed).
                    int gcount = 0;
                    for (int it = 0; ok && next_work(p, unit0, units, it, w); ++it) {
                        int kin = w.kb1 > w.kb0 ? w.kb0 % p.group_kb : 0;   // position inside the group
                        uint32_t d_tmem = tmem_base;
                        int gb = 0;
                        for (int kb = w.kb0; kb < w.kb1; ++kb) {
                            const bool first = (kb == w.kb0) || kin == 0;
                            if (first) {
                                gb = gcount & 1;
                                if (!mbar_wait(&acc_empty[gb], ((gcount >> 1) & 1) ^ 1, abort_flag, p.wait_ns)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                d_tmem = tmem_base + static_cast<uint32_t>(gb * p.acc_stride);
                            }
                            if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_stage(d_tmem, stage, first, CF::IDESC, CF::SLICE_B >> 4);
                            if (++stage == S) {
                                stage = 0;
                                phase ^= 1;
                            }
                            if (++kin == p.group_kb || kb + 1 == w.kb1) {
                                // the group's product is ready for the epilogue
                                if constexpr (CF::PAIR)
                                    mma_commit_pair(&acc_full[gb], 3);
                                else
                                    mma_commit(&acc_full[gb]);
                                ++gcount;
                                kin = 0;
                            }
                        }
                    }
                } else
                for (int it = 0; ok && next_work(p, unit0, units, it, w); ++it, ++local) {
                    const int buf = local & 1;
                    const uint32_t acc_phase = (local >> 1) & 1;
                    if (!mbar_wait(&acc_empty[buf], acc_phase ^ 1, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc_base = tmem_base + static_cast<uint32_t>(buf * p.acc_stride);
                    // group g covers K slices [ceil(g*KB/G), ceil((g+1)*KB/G))
                    int group = 0;
                    int next_group_start = w.kb1;
                    if (ngroups > 1) {   // a K segment may start inside the groups
                        group = (w.kb0 * ngroups) / kblocks;
                        next_group_start = ((group + 1) * kblocks + ngroups - 1) / ngroups;
                    }
                    uint32_t d_tmem = acc_base + static_cast<uint32_t>(group * CF::BN);
                    // a tail half is one MMA of half the width
                    const bool half_item = CF::HALVES && w.half >= 0;
                    const uint32_t idesc_item = half_item ? CF::IDESC_HALF : CF::IDESC;
                    const uint32_t b_slice = (half_item ? CF::SLICE_B / 2 : CF::SLICE_B) >> 4;
                    for (int kb = w.kb0; kb < w.kb1; ++kb) {
                        if (!mbar_wait(&full[stage], phase, abort_flag, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        bool first_in_group = (kb == w.kb0);
                        if (kb == next_group_start) {
                            ++group;
                            first_in_group = true;
                            next_group_start = ((group + 1) * kblocks + ngroups - 1) / ngroups;
                            d_tmem = acc_base + static_cast<uint32_t>(group * CF::BN);
                        }
                        issue_stage(d_tmem, stage, first_in_group, idesc_item, b_slice);
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    // accumulator ready for the epilogue (of both CTAs of a pair)
                    if constexpr (CF::PAIR)
                        mma_commit_pair(&acc_full[buf], 3);
                    else
                        mma_commit(&acc_full[buf]);
                }
                if (!ok) raise_error(p, ERR_TIMEOUT_MMA, abort_flag);
                // Drain: all issued MMAs complete before TMEM is released.
                if constexpr (CF::PAIR)
                    mma_commit_pair(drain, 1);
                else
                    mma_commit(drain);
                if (!mbar_wait(drain, 0, nullptr, p.wait_ns)) raise_error(p, ERR_TIMEOUT_DRAIN, abort_flag);
            }
            __syncwarp();
        } else if (CF::GS_SMEM && warp == 2) {
            // ------------------------------------------------------------ scale producer
            // For every scale group of every work item, in the epilogue's order:
            // the tile's BN column scales (16 bytes per copy; N % 4 == 0) and this
            // CTA's 128 row scales (4 bytes per copy; any M) into the next slot,
            // zero past the edges; each lane's copies arrive on the slot's full
            // barrier when they land.
            int gcount = 0;
            bool ok = true;
            Work w;
            for (int it = 0; ok && next_work(p, unit0, units, it, w); ++it) {
                if (w.kb1 <= w.kb0) continue;
                int mb, nb;
                tile_coords(w.tile, p, mb, nb);
                const int row0 = mb * CF::TILE_M + static_cast<int>(rank) * CF::BM;
                const int col0 = nb * CF::BN;
                const int j0 = w.kb0 / p.group_kb, j1 = (w.kb1 - 1) / p.group_kb + 1;
                for (int j = j0; j < j1; ++j, ++gcount) {
                    const int slot = gcount % (CF::SC_SLOTS > 0 ? CF::SC_SLOTS : 1);
                    const uint32_t ph = static_cast<uint32_t>(gcount / (CF::SC_SLOTS > 0 ? CF::SC_SLOTS : 1)) & 1u;
                    if (!mbar_wait(&sc_empty[slot], ph ^ 1u, abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    float* dst = gs_area + slot * CF::SLOT_FLOATS;
                    const float* cs = p.col_gscale + j * p.gs_ld_col;
                    const float* rs = p.row_gscale + j * p.gs_ld_row;
                    if (p.gs_col_shift == 0) {
#pragma unroll
                        for (int c = lane * 4; c < CF::BN; c += 128) {
                            const int n = col0 + c;
                            cp_async_16(dst + c, cs + (n < p.N ? n : 0), n < p.N ? 16u : 0u);
                        }
                    } else {   // each column gets its block's scale
#pragma unroll
                        for (int c = lane; c < CF::BN; c += 32) {
                            const int n = col0 + c;
                            cp_async_4(dst + c, cs + ((n < p.N ? n : 0) >> p.gs_col_shift), n < p.N ? 4u : 0u);
                        }
                    }
#pragma unroll
                    for (int r = lane; r < CF::BM; r += 32) {
                        const int m = row0 + r;
                        cp_async_4(dst + CF::BN + r, rs + (m < p.M ? m : 0), m < p.M ? 4u : 0u);
                    }
                    cp_async_mbar_arrive(&sc_full[slot]);
                }
            }
            if (!ok) raise_error(p, ERR_TIMEOUT_PRODUCER, abort_flag);
            cp_async_wait<0>();   // no copy into this CTA's shared memory outlives it
        }
        if (!CF::PAIR && p.cluster_split) {   // the split-K cluster barrier, once per thread
            __syncwarp();
            cluster_sync();
        }
    } else {
        if constexpr (CF::REG_SPLIT) regs_inc<CF::REGS_HIGH>();
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                        // TMEM lane quarter this warp may access
        const int ew = warp - CF::EPI_WARP0;           // epilogue warp index
        const int cbase = (ew >> 2) * CF::EPI_COLS;    // first tile column this warp handles
        uint8_t* stg = staging + ew * 4096;            // this warp's 4 KB staging box (tile modes)
        constexpr int UNIT = CF::EPI_COLS < 32 ? CF::EPI_COLS : 32;
        constexpr int NUNITS = CF::EPI_COLS / UNIT;
        constexpr int UNIT_F4 = UNIT / 4;              // float4 per lane per unit in a partial
        // partial layout: [item][cta][epilogue warp][unit][UNIT_F4][32 lanes] float4
        constexpr int64_t ITEM_F4 = static_cast<int64_t>(CF::CTAS) * CF::EPI_WARPS * NUNITS * UNIT_F4 * 32;
        // GS: the u loops index the register-resident group sum, so they unroll
        constexpr int U_UNROLL = CF::GS ? NUNITS : 1;
        int stores = 0;
        int local = 0;
        int gcount = 0;   // GS: scale groups folded so far (both buffers alternate)
        bool cluster_done = false;   // passed the split-K cluster barrier
        bool ok = true;

        // Requantisation (MODE_ROWQ): s[m] = amax[m] / 448; q = RN_E4M3(y * (1 / s[m])),
        // saturating. The stash is cut into chunks of RQ_CHUNK values of one row,
        // in row order (so in band order), claimed one at a time by epilogue
        // warps through a global counter; the warp converting a row's first
        // chunk writes the row scale. Lane l reads 8 x 16 bytes at once.
        const int64_t rq_cpr = (p.N + RQ_CHUNK - 1) / RQ_CHUNK;   // chunks per row
        const int64_t rq_chunks = static_cast<int64_t>(p.M) * rq_cpr;
        auto band_of_chunk = [&](int64_t j) {
            return static_cast<int>(j / rq_cpr) / CF::TILE_M / p.group_m / p.rq_gpc;
        };
        auto rq_convert = [&](int64_t j) {
            const int64_t m = j / rq_cpr;
            const int c0 = static_cast<int>(j % rq_cpr) * RQ_CHUNK;
            const int len8 = min(RQ_CHUNK, p.N - c0) / 8;   // N is a multiple of 16
            const float amax = __uint_as_float(__ldcg(p.amax + m));
            const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
            const float inv = amax > 0.0f ? 1.0f / s : 0.0f;
            if (lane == 0 && c0 == 0) p.out_row_scale[m] = s;
            const uint4* src = reinterpret_cast<const uint4*>(p.stash + m * p.N + c0);
            uint2* dst = reinterpret_cast<uint2*>(p.q_out + m * p.N + c0);
            uint4 y[RQ_CHUNK / 256];
#pragma unroll
            for (int i = 0; i < RQ_CHUNK / 256; ++i) {
                const int g = lane + 32 * i;
                y[i] = g < len8 ? __ldcs(src + g) : make_uint4(0u, 0u, 0u, 0u);   // last use
            }
#pragma unroll
            for (int i = 0; i < RQ_CHUNK / 256; ++i) {
                const int g = lane + 32 * i;
                if (g < len8) {
                    const uint32_t w0 = pack_e4m3x2(bf16_lo(y[i].x) * inv, bf16_hi(y[i].x) * inv);
                    const uint32_t w1 = pack_e4m3x2(bf16_lo(y[i].y) * inv, bf16_hi(y[i].y) * inv);
                    const uint32_t w2 = pack_e4m3x2(bf16_lo(y[i].z) * inv, bf16_hi(y[i].z) * inv);
                    const uint32_t w3 = pack_e4m3x2(bf16_lo(y[i].w) * inv, bf16_hi(y[i].w) * inv);
                    __stcs(dst + g, make_uint2(w0 | (w1 << 16), w2 | (w3 << 16)));
                }
            }
        };
        // Chunks are claimed in order with one atomic add each (a compare-and-
        // swap that claimed only ready chunks failed under the contention of a
        // thousand warps). A claimed chunk whose band is not complete yet stays
        // this warp's pending chunk until it is. rq_work converts chunks while
        // their bands are complete and stop() is false; it returns with
        // rq_pending >= 0 if it stopped at an incomplete band.
        long long rq_pending = -1;
        bool rq_done = false;   // every chunk has been claimed
        int rq_ready_band = -1;   // a band this warp has seen complete (acquired)
        auto rq_band_ready = [&](long long j) {
            const int b = band_of_chunk(j);
            if (b == rq_ready_band) return true;
            unsigned ready = 0;
            if (lane == 0) ready = ld_acquire_u32(p.band_count + b) >= band_expected<CF>(p, b) ? 1u : 0u;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            __syncwarp();
            if (ready) {
                __threadfence();   // the band's stash and maxima after its count
                rq_ready_band = b;
            }
            return ready != 0;
        };
        // lane 0: the next ticket, requested while the current chunk converts
        auto rq_claim = [&]() -> long long {
            long long j = 0;
            if (lane == 0) j = static_cast<long long>(atomicAdd(p.rq_next, 1ull));
            return j;
        };
        auto rq_work = [&](auto stop, int max_chunks) {
            for (int c = 0; c < max_chunks && !rq_done && !stop(); ++c) {
                if (rq_pending < 0) rq_pending = __shfl_sync(0xffffffffu, rq_claim(), 0);
                if (rq_pending >= rq_chunks) {
                    rq_done = true;
                    break;
                }
                if (!rq_band_ready(rq_pending)) break;
                const long long next = rq_claim();
                rq_convert(rq_pending);
                rq_pending = __shfl_sync(0xffffffffu, next, 0);
            }
        };

        Work w;
        for (int it = 0; next_work(p, unit0, units, it, w); ++it, ++local) {
            int mb, nb;
            tile_coords(w.tile, p, mb, nb);
            const int buf = local & 1;
            const int row_base = mb * CF::TILE_M + static_cast<int>(rank) * CF::BM + q * 32;
            const int row = row_base + lane;
            // A tail half has 128 accumulator columns, 64 per warp.
            const bool hw = CF::HALVES && w.half >= 0;
            const int cb = hw ? cbase / 2 : cbase;   // this warp's first accumulator column
            const int ocol = nb * CF::BN + (hw ? w.half * (CF::BN / 2) : 0) + cb;   // ... and its output column
            const int nunits = hw ? NUNITS / 2 : NUNITS;
            // The item's scales and bias do not depend on the MMA: fetch them
            // before waiting for the accumulator. Tile modes: lane l takes the
            // warp's columns 4l .. 4l + 3 (0 past N), shared by shuffles later.
            const float rs = (p.row_scale && row < p.M) ? p.row_scale[row] : 1.0f;
            float bias_row = 0.0f;
            if constexpr (CF::MODE == MODE_SWAP)
                if (p.bias && row < p.M) bias_row = p.bias[row];
            float4 cs_l = make_float4(1.f, 1.f, 1.f, 1.f), bias_l = make_float4(0.f, 0.f, 0.f, 0.f);
            // (per-K-group-scale kernels have no column scale here, and fetch
            // their bias after the group loop, whose running sum fills the registers)
            auto load_cols = [&]() {
                const int cl = ocol + 4 * lane;
                if (4 * lane < (hw ? CF::EPI_COLS / 2 : CF::EPI_COLS) && cl < p.N) {
                    if (!CF::GS && p.col_scale) cs_l = ld_bcast4(p.col_scale, cl, p.N);
                    if (p.bias) bias_l = ld_bcast4(p.bias, cl, p.N);
                }
            };
            if constexpr (CF::MODE != MODE_SWAP && !CF::GS) load_cols();
            // Small-M form: the MMA columns' (tokens') scales of this warp, 0
            // past N, likewise fetched before the accumulator is ready.
            constexpr bool SW_PRE = CF::MODE == MODE_SWAP && !CF::GS;   // (K-group scales: per group)
            constexpr int SW4 = SW_PRE ? (CF::EPI_COLS + 3) / 4 : 1;
            float4 cs_sw[SW4];
            cs_sw[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (SW_PRE) {
#pragma unroll
                for (int i = 0; i < SW4; ++i)
                    cs_sw[i] = (p.col_scale && ocol + 4 * i < p.N) ? ld_bcast4(p.col_scale, ocol + 4 * i, p.N)
                                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if constexpr (!CF::GS) {
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(&acc_full[buf], acc_phase, abort_flag, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(buf * p.acc_stride);
            // the K groups this item accumulated (a K segment touches only its own)
            int g0 = 0, g1 = 1;
            if (p.k_blocks > 0 && p.acc_groups > 1) {
                g0 = (w.kb0 * p.acc_groups) / p.k_blocks;
                g1 = ((w.kb1 - 1) * p.acc_groups) / p.k_blocks + 1;
            }
            float rowmax = 0.0f;
            const bool part = w.item >= 0;   // a K segment of a split tile

            // Per-K-group scales: fold each scale group's product into gsum as
            // soon as the MMA warp has finished it, then hand its buffer back.
            float gsum[CF::GS ? CF::EPI_COLS : 1];
            if constexpr (CF::GS) {
#pragma unroll
                for (int c = 0; c < CF::EPI_COLS; ++c) gsum[c] = 0.0f;
                if (w.kb1 > w.kb0) {
                    const int j0 = w.kb0 / p.group_kb, j1 = (w.kb1 - 1) / p.group_kb + 1;
                    const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(cbase);
                    const int colw = nb * CF::BN + cbase;   // this warp's first MMA column
                    const bool blk_cols = p.gs_col_shift != 0;
                    // Tile modes: scales from the scale producer's slot gcount % SC_SLOTS.
                    // Small-M form: row scale one per lane into a register, fetched
                    // two groups ahead (after the hand-back arrive, which is relaxed
                    // so it does not wait for them); column scales read directly.
                    auto load_rs = [&](int j) {
                        return (j < j1 && row < p.M) ? __ldg(p.row_gscale + j * p.gs_ld_row + (row >> p.gs_row_shift))
                                                     : 0.0f;
                    };
                    float rs_cur = 0.0f, rs_nxt = 0.0f;
                    if constexpr (!CF::GS_SMEM) {
                        rs_cur = load_rs(j0);
                        rs_nxt = load_rs(j0 + 1);
                    }
                    for (int j = j0; j < j1; ++j, ++gcount) {
                        const int gb = gcount & 1;
                        const int slot = gcount % (CF::SC_SLOTS > 0 ? CF::SC_SLOTS : 1);
                        const float* csj;
                        float rsj;
                        if constexpr (CF::GS_SMEM) {
                            const uint32_t ph = static_cast<uint32_t>(gcount / CF::SC_SLOTS) & 1u;
                            if (!mbar_wait(&sc_full[slot], ph, abort_flag, p.wait_ns)) {
                                ok = false;
                                break;
                            }
                            const float* sl = gs_area + slot * CF::SLOT_FLOATS;
                            csj = sl + cbase;
                            rsj = sl[CF::BN + q * 32 + lane];
                        } else {
                            csj = p.col_gscale + j * p.gs_ld_col;
                            rsj = rs_cur;
                        }
                        if (!mbar_wait(&acc_full[gb], (gcount >> 1) & 1, abort_flag, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // two Tensor Memory loads in flight per wait
#pragma unroll
                        for (int u = 0; u < NUNITS; u += 2) {
                            constexpr int PAIRED = NUNITS >= 2 ? 2 : 1;
                            uint32_t r[PAIRED][UNIT];
#pragma unroll
                            for (int h = 0; h < PAIRED; ++h) {
                                const uint32_t ta = tq + static_cast<uint32_t>(gb * p.acc_stride + (u + h) * UNIT);
                                if constexpr (UNIT == 32)
                                    tmem_ld32(ta, r[h]);
                                else
                                    tmem_ld16(ta, r[h]);
                            }
                            tmem_ld_wait();
#pragma unroll
                            for (int h = 0; h < PAIRED; ++h) {
                                if constexpr (CF::GS_SMEM) {
                                    if (blk_cols)
                                        gs_fold_uniform<UNIT>(gsum + (u + h) * UNIT, r[h], rsj * csj[0]);
                                    else
                                        gs_fold_smem<UNIT>(gsum + (u + h) * UNIT, r[h], rsj, csj + (u + h) * UNIT);
                                } else
                                    gs_fold<UNIT>(gsum + (u + h) * UNIT, r[h], rsj, csj, colw + (u + h) * UNIT, p.N);
                            }
                        }
                        tc_fence_before();
                        __syncwarp();   // every lane is done with TMEM buffer gb and scale slot
                        // The buffer's and slot's reads have completed (tcgen05.wait::ld;
                        // shared loads consumed), so the hand-backs need no memory
                        // ordering: relaxed arrives, which do not wait for loads in flight.
                        if (lane == 0) {
                            if (CF::PAIR && rank != 0)
                                mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&acc_empty[gb]), 0));
                            else
                                mbar_arrive_relaxed(&acc_empty[gb]);
                            if constexpr (CF::GS_SMEM) mbar_arrive_relaxed(&sc_empty[slot]);
                        }
                        if constexpr (!CF::GS_SMEM) {
                            rs_cur = rs_nxt;
                            rs_nxt = load_rs(j + 2);
                        }
                    }
                }
                if (!ok) break;
            }

            if constexpr (CF::MODE != MODE_SWAP && CF::GS) load_cols();

            // The accumulator of 32 (or 16) columns, FP32 sum of its K groups.
            auto load_acc = [&](int u, float (&v)[32]) {
                if constexpr (CF::GS) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = j < UNIT ? gsum[u * UNIT + j] : 0.0f;
                } else {
                const int tcol = cb + u * UNIT;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                // K groups (the small-M form only): GB loads in flight per wait
                // (64 registers), then the rest
                constexpr int GB = CF::MODE == MODE_SWAP ? (UNIT == 32 ? 2 : 4) : 1;
                int g = g0;
#pragma unroll 1
                for (; GB > 1 && g + GB <= g1; g += GB) {
                    uint32_t r[GB][UNIT];
#pragma unroll
                    for (int h = 0; h < GB; ++h)
                        tmem_ld_unit<UNIT>(taddr + static_cast<uint32_t>((g + h) * CF::BN + tcol), r[h]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < GB; ++h)
#pragma unroll
                        for (int j = 0; j < UNIT; ++j) v[j] += __uint_as_float(r[h][j]);
                }
#pragma unroll 1
                for (; g < g1; ++g) {
                    uint32_t r[UNIT];
                    tmem_ld_unit<UNIT>(taddr + static_cast<uint32_t>(g * CF::BN + tcol), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < UNIT; ++j) v[j] += __uint_as_float(r[j]);
                }
                if (p.k_blocks == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                }
                }
            };
            // Epilogue arithmetic and output of finished values. `direct`: store
            // this unit with plain global stores instead of a TMA box (the K
            // segments of a split tile each finish single units).
            auto finish = [&](int u, float (&v)[32], bool direct) {
                const int col0 = ocol + u * UNIT;
                // this unit's token scales, picked with constant indices (registers)
                float4 cu[SW_PRE ? (UNIT + 3) / 4 : 1];
#pragma unroll
                for (int i = 0; i < (SW_PRE ? (UNIT + 3) / 4 : 1); ++i) {
                    cu[i] = cs_sw[SW_PRE ? i : 0];
#pragma unroll
                    for (int uu = 1; uu < NUNITS; ++uu)
                        if (SW_PRE && u == uu) cu[i] = cs_sw[(uu * UNIT / 4 + i) % SW4];
                }
                epilogue_math<CF::MODE == MODE_SWAP>(v, p, row, col0, UNIT, rs, bias_row, cs_l, bias_l,
                                                     u * UNIT / 4, cu);
                if constexpr (CF::MODE == MODE_ROWQ) {
                    if (row < p.M) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < p.N) rowmax = fmaxf(rowmax, fabsf(v[j]));
                    }
                }
                if constexpr (CF::MODE == MODE_TILE || CF::MODE == MODE_ROWQ) {
                    if (direct) {
                        // row-major D (the BF16 stash for requantisation), this
                        // thread's row: 16-byte chunks, each wholly inside or outside
                        // N (N is a multiple of 8 for BF16, 4 for FP32)
                        if (row < p.M) {
                            if (CF::MODE == MODE_TILE && p.d_f32) {
                                float* d = static_cast<float*>(p.D) + static_cast<int64_t>(row) * p.ldd + col0;
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    if (col0 + 4 * c < p.N)
                                        *reinterpret_cast<float4*>(d + 4 * c) =
                                            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                            } else {
                                uint16_t* d = (CF::MODE == MODE_ROWQ ? const_cast<uint16_t*>(p.stash)
                                                                     : static_cast<uint16_t*>(p.D)) +
                                              static_cast<int64_t>(row) * p.ldd + col0;
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    if (col0 + 8 * c < p.N)
                                        *reinterpret_cast<uint4*>(d + 8 * c) =
                                            make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]),
                                                       pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                                       pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                                                       pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
                            }
                        }
                        return;
                    }
                }
                if constexpr (CF::MODE == MODE_SWAP) {
                    // MMA column = output row; MMA row = output column.
                    if (row < p.M) {
#pragma unroll
                        for (int j = 0; j < UNIT; ++j)
                            if (col0 + j < p.N) {
                                const int64_t off = static_cast<int64_t>(col0 + j) * p.ldd + row;
                                if (p.d_f32)
                                    static_cast<float*>(p.D)[off] = v[j];
                                else
                                    static_cast<uint16_t*>(p.D)[off] =
                                        static_cast<uint16_t>(pack_bf16x2(v[j], 0.0f) & 0xFFFFu);
                            }
                    }
                } else {
                    tile_store_unit<CF>(v, p, u, col0, row_base, lane, stg, stores, &tmD);
                }
            };

            // A split tile is finished by all of its K segments together: unit u
            // (32 columns) of this warp's region belongs to segment u % split.
            // When every segment is resident (a cluster, or a cooperative
            // launch), each parks the units other segments own as FP32 partials,
            // counts its arrival, waits until every segment has arrived, then
            // adds the others' partials of its own units to its accumulator and
            // stores them directly: about one round trip through L2 per segment
            // instead of a single warp reading every partial unit by unit.
            // Otherwise the last segment to arrive finishes the region (below).
            const int item0 = part ? (w.item / p.split) * p.split : 0;
            const int seg = part ? w.item - item0 : 0;
            auto owner = [&](int u) { return u % p.split; };
            // generic writes to buffers the TMA (async proxy) filled
            if (part && p.cluster_split) fence_proxy_async_smem();
            const bool unit_pass = !part || p.cluster_split || p.split_sym;
            if (unit_pass) {
#pragma unroll U_UNROLL
                for (int u = 0; u < nunits; ++u) {
                    float v[32];
                    load_acc(u, v);
                    if (part && owner(u) != seg) {
                        // a unit another segment finishes: park the raw FP32
                        // accumulator; each warp-wide store writes 512 contiguous bytes
                        if (p.cluster_split) {
                            // into this CTA's idle pipeline buffers (every stage has been
                            // consumed: this is the unit's last item), for the peers
                            float4* dst = reinterpret_cast<float4*>(stages) + (ew * NUNITS + u) * (UNIT_F4 * 32) + lane;
#pragma unroll
                            for (int j = 0; j < UNIT_F4; ++j)
                                dst[32 * j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        } else {
                            float4* dst = reinterpret_cast<float4*>(p.partials) + w.item * ITEM_F4 +
                                          ((static_cast<int64_t>(rank) * CF::EPI_WARPS + ew) * NUNITS + u) *
                                              (UNIT_F4 * 32) +
                                          lane;
#pragma unroll
                            for (int j = 0; j < UNIT_F4; ++j)
                                __stcg(dst + 32 * j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                        }
                    }
                    if (!CF::GS && u == nunits - 1 && !part) {
                        // Last read of this accumulator: hand it back to the MMA warp
                        // (a K segment's, after its units are finished: it reads its own
                        // units again then).
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (CF::PAIR && rank != 0)
                                mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[buf]), 0));
                            else
                                mbar_arrive(&acc_empty[buf]);
                        }
                    }
                    if (!part) finish(u, v, false);
                }
            }
            if constexpr (CF::MODE == MODE_ROWQ) {
                if (row < p.M) atomicMax(&p.amax[row], __float_as_uint(rowmax));
            }
            if constexpr (CF::MODE != MODE_ROWQ && !CF::PAIR) {
                if (part && p.cluster_split) {
                    // Every segment of the tile is a CTA of this cluster (rank =
                    // segment). One cluster barrier publishes the parked units;
                    // each thread of each CTA arrives at it exactly once.
                    __syncwarp();
                    cluster_sync();
                    cluster_done = true;
                    if (seg < NUNITS) {
#pragma unroll U_UNROLL
                        for (int u = 0; u < NUNITS; ++u) {
                            if (owner(u) != seg) continue;
                            float v[32];
                            load_acc(u, v);
                            const uint32_t mine =
                                smem_u32(reinterpret_cast<float4*>(stages) + (ew * NUNITS + u) * (UNIT_F4 * 32) + lane);
                            float4 f[3][UNIT_F4];
#pragma unroll
                            for (int o = 0; o < 3; ++o) {
                                const int peer = o + (o >= seg ? 1 : 0);
                                const uint32_t base = peer < p.split ? mapa_shared(mine, static_cast<uint32_t>(peer)) : 0u;
#pragma unroll
                                for (int j = 0; j < UNIT_F4; ++j)
                                    f[o][j] = peer < p.split ? ld_shared_cluster_f4(base + 16u * 32u * j)
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int o = 0; o < 3; ++o)
#pragma unroll
                                for (int j = 0; j < UNIT_F4; ++j) {
                                    v[4 * j] += f[o][j].x;
                                    v[4 * j + 1] += f[o][j].y;
                                    v[4 * j + 2] += f[o][j].z;
                                    v[4 * j + 3] += f[o][j].w;
                                }
                            finish(u, v, true);
                        }
                    }
                }
            }
            {
                if (part && !p.cluster_split) {
                    // The split tile's counter word for this warp's region:
                    // (launch epoch << 8) | (segments parked << 4) | arrivals; a word
                    // left by any earlier launch counts as zero of each.
                    unsigned long long* cnt =
                        p.tail_count + ((w.item / p.split) * CF::CTAS + rank) * CF::EPI_WARPS + ew;
                    // lane 0: counts this segment in; returns how many had arrived
                    // before it, or -1 if the word could not be updated.
                    auto arrive = [&]() -> int {
                        unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(cnt);
                        for (int tries = 0; tries < 4096; ++tries) {
                            const bool cur = (old >> 8) == p.epoch;
                            const unsigned long long next = cur ? old + 1 : ((p.epoch << 8) | 1ull);
                            const unsigned long long seen = atomicCAS(cnt, old, next);
                            if (seen == old) return cur ? static_cast<int>(old & 0xFull) : 0;
                            old = seen;
                        }
                        return -1;
                    };
                    // lane 0: bounded wait until the word satisfies done(word)
                    auto await = [&](auto done) -> unsigned {
                        unsigned long long seen = ld_acquire_u64(cnt);
                        const uint64_t t0 = globaltimer();
                        while (!done(seen)) {
                            if (*abort_flag || globaltimer() - t0 > p.wait_ns) return 0u;
                            __nanosleep(32);
                            seen = ld_acquire_u64(cnt);
                        }
                        return 1u;
                    };
                    // v += the other segments' partials of unit u, all loads in flight together
                    auto add_partials = [&](int u, float (&v)[32]) {
                        const float4* src = reinterpret_cast<const float4*>(p.partials) + item0 * ITEM_F4 +
                                            ((static_cast<int64_t>(rank) * CF::EPI_WARPS + ew) * NUNITS + u) *
                                                (UNIT_F4 * 32) +
                                            lane;
                        float4 f[3][UNIT_F4];
#pragma unroll
                        for (int o = 0; o < 3; ++o) {
                            const int sgi = o + (o >= seg ? 1 : 0);
#pragma unroll
                            for (int j = 0; j < UNIT_F4; ++j)
                                f[o][j] = sgi < p.split ? __ldcg(src + sgi * ITEM_F4 + 32 * j)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int o = 0; o < 3; ++o)
#pragma unroll
                            for (int j = 0; j < UNIT_F4; ++j) {
                                v[4 * j] += f[o][j].x;
                                v[4 * j + 1] += f[o][j].y;
                                v[4 * j + 2] += f[o][j].z;
                                v[4 * j + 3] += f[o][j].w;
                            }
                    };
                    if (p.split_sym) {
                        // Every segment of the tile is resident (cooperative launch):
                        // count this warp's parked units in, then (if this segment
                        // owns units of the region) wait for all segments and finish
                        // them: own accumulator from Tensor Memory (handed back to
                        // the MMA only after this), the others from the workspace.
                        __threadfence();   // this lane's partial stores before the count
                        __syncwarp();
                        const bool owns = seg < NUNITS;
                        unsigned ready = 0;
                        if (lane == 0) {
                            __threadfence();
                            const int before = arrive();
                            if (before < 0) {
                                record_error(p, ERR_ARRIVAL);
                            } else if (owns) {
                                const unsigned long long want = (p.epoch << 8) | static_cast<unsigned long long>(p.split);
                                ready = await([&](unsigned long long x) { return x == want; });
                                __threadfence();
                            } else {
                                ready = 1u;
                            }
                        }
                        ready = __shfl_sync(0xffffffffu, ready, 0);
                        __threadfence();   // the other segments' partials after their count
                        if (!ready) {
                            ok = false;
                        } else if (owns) {
#pragma unroll U_UNROLL
                            for (int u = 0; u < NUNITS; ++u) {
                                if (owner(u) != seg) continue;
                                float v[32];
                                load_acc(u, v);
                                add_partials(u, v);
                                finish(u, v, true);
                            }
                            if constexpr (CF::MODE == MODE_ROWQ) {   // the row maxima of the units finished here
                                if (row < p.M) atomicMax(&p.amax[row], __float_as_uint(rowmax));
                            }
                        }
                    } else {
                        // No residency guarantee: never wait for a segment that may
                        // not have started. Arrive first; all but the last arrival
                        // park every unit and leave; the last waits only for the
                        // earlier arrivals (running, and waiting on nothing) to
                        // finish parking, then finishes every unit of the region.
                        int before = 0;
                        if (lane == 0) before = arrive();
                        before = __shfl_sync(0xffffffffu, before, 0);
                        if (before < 0) {
                            if (lane == 0) record_error(p, ERR_ARRIVAL);
                            ok = false;
                        } else if (before < p.split - 1) {
#pragma unroll U_UNROLL
                            for (int u = 0; u < NUNITS; ++u) {
                                float v[32];
                                load_acc(u, v);
                                float4* dst = reinterpret_cast<float4*>(p.partials) + w.item * ITEM_F4 +
                                              ((static_cast<int64_t>(rank) * CF::EPI_WARPS + ew) * NUNITS + u) *
                                                  (UNIT_F4 * 32) +
                                              lane;
#pragma unroll
                                for (int j = 0; j < UNIT_F4; ++j)
                                    __stcg(dst + 32 * j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                            }
                            __threadfence();   // this lane's partial stores before the count
                            __syncwarp();
                            if (lane == 0) red_release_add_u64(cnt, 1ull << 4);
                        } else {
                            unsigned ready = 0;
                            if (lane == 0) {
                                const unsigned long long want = static_cast<unsigned long long>(p.split - 1);
                                ready = await([&](unsigned long long x) {
                                    return (x >> 8) == p.epoch && ((x >> 4) & 0xFull) == want;
                                });
                                __threadfence();
                            }
                            ready = __shfl_sync(0xffffffffu, ready, 0);
                            __threadfence();   // the other segments' partials after their count
                            if (!ready) {
                                ok = false;
                            } else {
#pragma unroll U_UNROLL
                                for (int u = 0; u < NUNITS; ++u) {
                                    float v[32];
                                    load_acc(u, v);
                                    add_partials(u, v);
                                    finish(u, v, true);
                                }
                                if constexpr (CF::MODE == MODE_ROWQ) {
                                    if (row < p.M) atomicMax(&p.amax[row], __float_as_uint(rowmax));
                                }
                            }
                        }
                    }
                }
            }
            if (!ok) break;
            if (!CF::GS && part) {
                // the K segment's last read of this accumulator is done
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CF::PAIR && rank != 0)
                        mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[buf]), 0));
                    else
                        mbar_arrive(&acc_empty[buf]);
                }
            }
            if constexpr (CF::MODE == MODE_ROWQ) {
                // This warp's share of the item is done: once its TMA stores have
                // completed (and, like its plain stores and row maxima, are
                // visible), count it into the item's row band.
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    bulk_wait_all();
                    fence_proxy_async_global();
                    __threadfence();
                    red_release_add_u32(p.band_count + band_of_tile(p, w.tile), 1u);
                }
                __syncwarp();
                // Until the next accumulator is ready, convert chunks of complete
                // bands (never waiting for one: the MMA may need this warp soon).
                Work wn;
                if (next_work(p, unit0, units, it + 1, wn)) {
                    const int nl = local + 1;
                    rq_work([&]() { return mbar_test(&acc_full[nl & 1], static_cast<uint32_t>(nl >> 1) & 1u); }, 16);
                }
            }
        }
        if (!ok) raise_error(p, ERR_TIMEOUT_EPILOGUE, abort_flag);
        if constexpr (CF::MODE == MODE_ROWQ) {
            // The rest of the chunks, waiting (bounded) for their bands.
            while (ok && !*abort_flag) {
                rq_work([]() { return false; }, 1 << 30);
                if (rq_done) break;
                unsigned ready = 1;   // the pending chunk's band is not complete yet
                if (lane == 0) {
                    const int b = band_of_chunk(rq_pending);
                    const unsigned want = band_expected<CF>(p, b);
                    const uint64_t t0 = globaltimer();
                    while (ld_acquire_u32(p.band_count + b) < want) {
                        if (*abort_flag || globaltimer() - t0 > p.wait_ns) {
                            ready = 0;
                            break;
                        }
                        __nanosleep(500);
                    }
                }
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (!ready) {
                    if (lane == 0) raise_error(p, ERR_TIMEOUT_ROW_BAND, abort_flag);
                    break;
                }
            }
        }
        if (!CF::PAIR && p.cluster_split && !cluster_done) {   // the split-K barrier, once per thread
            __syncwarp();
            cluster_sync();
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (CF::PAIR) {
        // neither CTA may leave while the pair's MMAs can still read its shared memory
        cluster_sync();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc_pair(tmem_base, tmem_cols);
        }
    } else {
        // with split-K through the cluster, no CTA leaves while a peer may
        // still read its parked partials
        if (p.cluster_split) cluster_sync();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem_base, tmem_cols);
        }
    }
}

}  // namespace dg
