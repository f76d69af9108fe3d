// api.cu -- the C ABI: argument validation, planning, TMA tensor maps, launch,
// the device-side status words, and the planner overrides. Interface as on the FP8 page
// ("DeepGEMM: FP8 Tensor Core GEMM", bjdmk.com.cn/news/6078902, §5.1): pointers,
// M/N/K, scale descriptor, a workspace whose size is queried beforehand, and a
// stream; nothing is allocated per call.
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "dgemm.h"
#include "kernels.h"

namespace {

__device__ unsigned int g_status = 0;  // sticky device-side error bits, one word per device

constexpr int kMaxDevices = 64;
constexpr int kWeightBlock = 128;       // output channels per weight scale (block-scaled entry)
constexpr int kWeightBlockShift = 7;
constexpr size_t kWsStatus = DGEMM_WS_STATUS_BYTES;  // every workspace: the call's status word first
constexpr size_t kWsHeader = 256;  // requantisation: chunk claim counter + row-band counters
static_assert(8 + 4 * dg::kMaxBands <= kWsHeader, "row-band counters fit the header");
static_assert(kWsStatus % 256 == 0 && kWsStatus >= 8, "status header keeps the layout 256-byte aligned");
constexpr int64_t kMinTailSlices = 48;  // shortest tile (K slices) worth splitting
constexpr int64_t kCompactSlices = 16;  // longest work item (K slices) of a compact small-M call

struct DeviceState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int cc_major = 0, cc_minor = 0, num_sms = 0;
    unsigned* status = nullptr;
};
DeviceState g_dev[kMaxDevices];

// ---- planner overrides (tuning sweeps, tests): process-wide, defaults = the
// planner's own choices. The DGEMM_* environment variables are read once, at
// the first call, and only when DGEMM_ENV_OVERRIDES=1.
void overrides_defaults(dgemm_overrides_t* o) {
    o->tile_n = 0;
    o->cta_pair = -1;
    o->tail_split = -1;
    o->tail_halves = -1;
    o->cluster_split = -1;
    o->seg_first = -1;
    o->raster_group = 0;
    o->cooperative = -1;
    o->kslices = -1;
    o->wait_limit_ns = 0;
    o->stall_after_loads = -1;
}

std::mutex g_ovr_mutex;
dgemm_overrides_t g_ovr;                   // guarded by g_ovr_mutex
std::atomic<bool> g_ovr_set{false};        // g_ovr differs from the defaults
std::once_flag g_ovr_once;

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    if (v[0] == 'f') return 1;             // "force" (DGEMM_TAIL_SPLIT)
    return std::atoi(v);
}

void init_overrides() {
    dgemm_overrides_t o;
    overrides_defaults(&o);
    const char* opt_in = std::getenv("DGEMM_ENV_OVERRIDES");
    if (opt_in && opt_in[0] == '1') {
        o.tile_n = env_int("DGEMM_TILE_N", 0);
        o.cta_pair = env_int("DGEMM_CTA_PAIR", -1);
        o.tail_split = env_int("DGEMM_TAIL_SPLIT", -1);
        o.tail_halves = env_int("DGEMM_TAIL_HALVES", -1);
        o.cluster_split = env_int("DGEMM_CLUSTER_SPLIT", -1);
        o.seg_first = env_int("DGEMM_SEG_FIRST", -1);
        o.raster_group = env_int("DGEMM_RASTER_GROUP", 0);
        o.cooperative = env_int("DGEMM_COOPERATIVE", -1);
        o.kslices = env_int("DGEMM_KSLICES", -1);
        if (const char* w = std::getenv("DGEMM_WAIT_LIMIT_NS")) o.wait_limit_ns = std::atoll(w);
    }
    std::lock_guard<std::mutex> lk(g_ovr_mutex);
    g_ovr = o;
    dgemm_overrides_t d;
    overrides_defaults(&d);
    g_ovr_set.store(std::memcmp(&o, &d, sizeof o) != 0, std::memory_order_release);
}

// The overrides in force for one call (the defaults unless some were set).
dgemm_overrides_t overrides_now() {
    std::call_once(g_ovr_once, init_overrides);
    dgemm_overrides_t o;
    if (!g_ovr_set.load(std::memory_order_acquire)) {
        overrides_defaults(&o);
        return o;
    }
    std::lock_guard<std::mutex> lk(g_ovr_mutex);
    return g_ovr;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int g_nk = 0;
constexpr int kMaxKernels = 96;
const dg::KernelInfo* g_kernels[kMaxKernels];
std::atomic<unsigned char> g_attr_set[64][kMaxDevices];
std::once_flag g_kernels_once;

void collect_kernels() {
    int n[4] = {0, 0, 0, 0};
    const dg::KernelInfo* t[4] = {dg::kernels_bf16(&n[0]), dg::kernels_fp8(&n[1]), dg::kernels_fp8_grouped(&n[2]),
                                  dg::kernels_two_slice(&n[3])};
    for (int j = 0; j < 4; ++j)
        for (int i = 0; i < n[j] && g_nk < kMaxKernels; ++i) g_kernels[g_nk++] = &t[j][i];
}

int find_kernel(int bn, int fp8, int a_mn, int b_mn, int mode, int pair, int gs, int ks = 1) {
    std::call_once(g_kernels_once, collect_kernels);
    for (int i = 0; i < g_nk; ++i) {
        const dg::KernelInfo* k = g_kernels[i];
        if (k->bn == bn && k->fp8 == fp8 && k->a_mn == a_mn && k->b_mn == b_mn && k->mode == mode &&
            k->pair == pair && k->gs == gs && k->ks == ks)
            return i;
    }
    return -1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t dtype_bytes(dgemm_dtype_t t) { return t == DGEMM_F32 ? 4 : t == DGEMM_BF16 ? 2 : 1; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int pair_ctas(int pair) { return pair ? 2 : 1; }

// Split-K for grids that do not fill the GPU: K segments per tile so that
// tiles x segments <= units, each segment at least 8 K slices, at most 4 (the
// last-arriving warp sums the others' partials with all loads in flight).
int64_t underfill_split(int64_t tiles, int64_t units, int64_t k_blocks) {
    if (tiles <= 0 || tiles >= units) return 1;
    int64_t s = units / tiles;
    if (s > k_blocks / 8) s = k_blocks / 8;
    if (s > 4) s = 4;
    return s < 1 ? 1 : s;
}

// Launch epochs for the tail-split arrival counters: 56-bit values, unique per
// launch within a process and started from a per-process pseudo-random point,
// so counter words left in a reused workspace (by any earlier call, or by other
// data) are not mistaken for this launch's arrivals.
// Every launch gets one; the workspace status word is tagged with it too.
constexpr unsigned long long kEpochMask = (1ull << 56) - 1;
std::atomic<unsigned long long> g_epoch{0};
unsigned long long g_epoch_first = 0;   // the first epoch this process issues
std::once_flag g_epoch_once;

void init_epoch() {
    std::call_once(g_epoch_once, []() {
        unsigned long long x = static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count());
        x ^= reinterpret_cast<uintptr_t>(&g_epoch) * 0x9E3779B97F4A7C15ull;
        x ^= x >> 31;
        x *= 0xBF58476D1CE4E5B9ull;
        x ^= x >> 29;
        g_epoch_first = (x + 1) & kEpochMask;
        g_epoch.store(x, std::memory_order_relaxed);
    });
}

unsigned long long next_epoch() {
    init_epoch();
    unsigned long long e;
    do {   // 0 tags a cleared status word: never issued
        e = (g_epoch.fetch_add(1, std::memory_order_relaxed) + 1) & kEpochMask;
    } while (e == 0);
    return e;
}

// Whether epoch e was issued by this process (so a status word tagged with it
// was written by one of its launches, not left by other data).
bool issued_epoch(unsigned long long e) {
    init_epoch();
    if (e == 0) return false;
    const unsigned long long last = g_epoch.load(std::memory_order_relaxed) & kEpochMask;
    return ((e - g_epoch_first) & kEpochMask) <= ((last - g_epoch_first) & kEpochMask);
}

struct Plan {
    dgemm_plan_t pub;
    int kernel;        // index into g_kernels
    int mode;
    int a_mn, b_mn;
    int64_t Mm, Nm;    // problem in the MMA's orientation
    int bk;            // K elements per stage
    int ks;            // K slices (128 bytes of K) per stage: 2 = operands in 3-D TMA copies
    int slice_k;       // K elements per slice
    int acc_stride;    // TMEM columns between the two accumulator buffers
    int gs;            // per-K-group scales (group_kb K slices per group)
    int group_kb;
    int dp_tiles, split, tail_items;   // tail splitting (MODE_TILE)
    int cluster_split;                 // split K segments of a tile form a cluster of `split` CTAs
    int tail_halves;                   // tail tiles run as two N halves (tail_items = 2 x tail tiles)
    int seg_first;                     // split K segments run before the whole tiles
    size_t split_offset;               // workspace offset of the split area (after the requant stash)
    size_t tail_count_bytes;           // workspace: per-warp arrival counters
    int stages;                        // ring depth of the launch
    int tmem_cols;                     // Tensor Memory columns per CTA
    size_t smem;                       // dynamic shared memory of the launch
};

// Validates the sizes, enums and epilogue; picks the kernel variant and grid.
// Pure host logic: needs no GPU.
// max_pairs: co-resident 2-CTA clusters; max_quads: co-resident 4-CTA clusters.
dgemm_status_t make_plan(int fp8, int64_t M, int64_t N, int64_t K, dgemm_b_layout_t bl, dgemm_dtype_t d_dtype,
                         const dgemm_epilogue_t* epi, int num_sms, int max_pairs, int max_quads, bool allow_split,
                         Plan* out, int k_group = 0) {
    const dgemm_overrides_t ov = overrides_now();
    if (M < 0 || N < 0 || K < 0 || num_sms <= 0 || k_group < 0) return DGEMM_ERR_INVALID_VALUE;
    if (bl != DGEMM_B_KN && bl != DGEMM_B_NK) return DGEMM_ERR_INVALID_VALUE;
    if (d_dtype != DGEMM_F32 && d_dtype != DGEMM_BF16 && d_dtype != DGEMM_E4M3) return DGEMM_ERR_INVALID_VALUE;
    const int act = epi ? epi->act : DGEMM_ACT_NONE;
    const int oq = epi ? epi->out_quant : DGEMM_QUANT_NONE;
    if (act < DGEMM_ACT_NONE || act > DGEMM_ACT_SILU) return DGEMM_ERR_INVALID_VALUE;
    if (oq != DGEMM_QUANT_NONE && oq != DGEMM_QUANT_E4M3_ROW_AMAX) return DGEMM_ERR_INVALID_VALUE;
    if ((oq == DGEMM_QUANT_E4M3_ROW_AMAX) != (d_dtype == DGEMM_E4M3)) return DGEMM_ERR_INVALID_VALUE;
    // Index arithmetic in the kernels is 32-bit per dimension.
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return DGEMM_ERR_NOT_SUPPORTED;
    const size_t esz = fp8 ? 1 : 2;
    // TMA: every row pitch a multiple of 16 bytes.
    if ((static_cast<size_t>(K) * esz) % 16 != 0) return DGEMM_ERR_MISALIGNED;
    if (bl == DGEMM_B_KN && (static_cast<size_t>(N) * esz) % 16 != 0) return DGEMM_ERR_MISALIGNED;
    if ((static_cast<size_t>(N) * dtype_bytes(d_dtype)) % 16 != 0) return DGEMM_ERR_MISALIGNED;

    // Per-K-group scales: groups of whole K slices (128 E4M3 values), no
    // requantising epilogue.
    const int gs = k_group > 0 ? 1 : 0;
    if (gs && (!fp8 || k_group % 128 != 0 || oq != DGEMM_QUANT_NONE)) return DGEMM_ERR_NOT_SUPPORTED;

    Plan p{};
    p.bk = static_cast<int>(128 / esz);
    p.gs = gs;
    p.group_kb = gs ? k_group / p.bk : 0;
    const bool swap = (oq == DGEMM_QUANT_NONE) && M <= 64;
    const bool pairs_ok = max_pairs > 0 && ov.cta_pair != 0;
    const bool force_split = ov.tail_split == 1;
    // (the requantising epilogue takes the tail split, not split-K of under-filled grids)
    const bool split_ok = allow_split && ov.tail_split != 0;
    if (ov.cluster_split == 0) max_quads = 0;   // split-K through the workspace only
    const bool cluster_ok = ov.cluster_split != 0;
    const int64_t kb_all = (K + (128 / static_cast<int64_t>(esz)) - 1) / (128 / static_cast<int64_t>(esz));
    int bn;
    int pair = 0;
    if (swap) {
        p.mode = dg::MODE_SWAP;
        p.Mm = N;
        p.Nm = M;
        p.a_mn = (bl == DGEMM_B_KN);  // the MMA's A operand is op(B)^T
        p.b_mn = 0;
        bn = M <= 16 ? 16 : M <= 32 ? 32 : 64;
    } else {
        p.mode = oq ? dg::MODE_ROWQ : dg::MODE_TILE;
        p.Mm = M;
        p.Nm = N;
        p.a_mn = 0;
        p.b_mn = (bl == DGEMM_B_KN);
        // Wave-cost model: cost = waves x (tile area per SM) x inefficiency.
        // A CTA pair's 256 x 256 tile is the most efficient per FLOP (least L2
        // traffic per SM, deepest pipeline); narrower single-CTA tiles need
        // more operand bandwidth per FLOP but quantise into waves more finely.
        struct Cand { int bn, pair; double penalty; };
        // Penalties from measurement: 128 x 128 tiles ran at 0.55x the per-SM
        // rate of 128 x 256 tiles (8192^3 FP8), being shared-memory-bound.
        const Cand cands[4] = {{256, 1, 1.0}, {256, 0, 1.15}, {128, 0, 2.1}, {64, 0, 3.0}};
        double best = 1e300;
        bn = 256;
        for (const Cand& c : cands) {
            if (p.mode == dg::MODE_ROWQ && c.bn != 256) continue;
            if (c.pair && (!pairs_ok || M <= 128)) continue;
            // Per-K-group scales in groups of one or two K slices: the fold,
            // not the operand feed, sets the pace, and a pair's TMEM buffer
            // takes its next group only when all 16 epilogue warps of both
            // CTAs have folded the last one, so single CTAs (8 warps a
            // buffer) run faster despite more operand copies per FLOP.
            // 4096 x 11008 x 4096 E4M3, TFLOP/s, single vs pair: g = 128
            // 1310 vs 1199 per channel, 1866 vs 1752 with weight blocks;
            // g = 256 1998 vs 1918, 2145 vs 2167; g = 512 2296 vs 2367,
            // 2395 vs 2540.
            if (c.pair && gs && p.group_kb <= 2) continue;
            if (fp8 && p.b_mn && c.bn < 128) continue;
            const int64_t tm = c.pair ? 256 : 128;
            const int64_t units = c.pair ? max_pairs : num_sms;
            const int64_t tiles = ((M + tm - 1) / tm) * ((N + c.bn - 1) / c.bn);
            const int64_t waves = (tiles + units - 1) / units;
            double cost = static_cast<double>(waves) * (128.0 * c.bn) * c.penalty;
            // under one wave, split-K divides each unit's work (reduction ~15 % of a tile)
            // (the reduction ~15 % of a tile through the workspace, ~5 % when the
            // segments of a single-CTA tile share a cluster)
            const int64_t sk = (split_ok && !oq) ? underfill_split(tiles, units, kb_all) : 1;
            const bool cl = cluster_ok && !c.pair && (sk == 2 || sk == 4) && tiles <= (sk == 2 ? max_pairs : max_quads);
            if (sk > 1) cost = (128.0 * c.bn) * c.penalty * (1.0 / static_cast<double>(sk) + (cl ? 0.05 : 0.15));
            if (cost < best) {
                best = cost;
                bn = c.bn;
                pair = c.pair;
            }
        }
        // At most one wave of single-CTA tiles: the time is set by each CTA's
        // TMA copies -- a fixed ~90 ns per copy plus the bytes at ~213 GB/s
        // per SM, i.e. ~19.2 KB of streaming per copy: one copy of A and one of
        // B (or one per 128-byte atom of MN-major B) per K slice, or one of each
        // per two slices where the tile takes two-slice stages -- plus the
        // partial sums its K segments exchange, ~13x slower per byte through
        // distributed shared memory (~27x through the workspace). Fitted to
        // 1024 x 1024 x 4096 BF16 with one slice per stage (128 x 256 in 4
        // segments 16.5 us = 128 x 128 in 2 segments 16.4 us); with two-slice
        // stages the second took 15.95 us against 18.5, and FP8 11.9 against
        // 14.1, the order the model gives.
        const int64_t tiles_w = ((M + 127) / 128) * ((N + bn - 1) / bn);
        if (!pair && p.mode == dg::MODE_TILE && tiles_w <= num_sms) {
            const int64_t slice_k = static_cast<int64_t>(128 / esz);
            auto two_slice = [&](int w) {
                return !gs && ov.kslices != 1 && K % slice_k == 0 && (!p.b_mn || N % slice_k == 0) &&
                       find_kernel(w, fp8, p.a_mn, p.b_mn, p.mode, 0, gs, 2) >= 0;
            };
            constexpr double kCopyBytes = 19170.0;   // ~90 ns at ~213 GB/s
            double best_t = 1e300;
            for (const Cand& c : cands) {
                if (c.pair || (fp8 && p.b_mn && c.bn < 128)) continue;
                const int64_t tiles = ((M + 127) / 128) * ((N + c.bn - 1) / c.bn);
                if (tiles > num_sms) continue;
                const int64_t sk = split_ok ? underfill_split(tiles, num_sms, kb_all) : 1;
                const bool cl = cluster_ok && (sk == 2 || sk == 4) && tiles <= (sk == 2 ? max_pairs : max_quads);
                const double copies = two_slice(c.bn) ? 1.0 : 1.0 + (p.b_mn ? c.bn / static_cast<double>(slice_k) : 1.0);
                const double stream = (static_cast<double>(128 + c.bn) * 128.0 + copies * kCopyBytes) *
                                      static_cast<double>((kb_all + sk - 1) / sk);
                const double xchg = sk > 1 ? 128.0 * c.bn * 4.0 * static_cast<double>(sk - 1) / static_cast<double>(sk) *
                                                 (cl ? 13.4 : 26.8)
                                           : 0.0;
                if (stream + xchg < best_t) {
                    best_t = stream + xchg;
                    bn = c.bn;
                }
            }
        }
    }
    // The tile width override applies when such a variant exists (tests reach
    // every variant with it; tuning sweeps).
    if (ov.tile_n > 0) {
        const int v = ov.tile_n;
        if (v != bn && find_kernel(v, fp8, p.a_mn, p.b_mn, p.mode, 0, gs) >= 0) {
            bn = v;
            pair = 0;
        }
    }
    // cta_pair = 1 forces the CTA-pair variant when one exists for this tile.
    if (ov.cta_pair == 1 && !swap && M > 128 && max_pairs > 0 &&
        find_kernel(bn, fp8, p.a_mn, p.b_mn, p.mode, 1, gs) >= 0)
        pair = 1;
    p.kernel = find_kernel(bn, fp8, p.a_mn, p.b_mn, p.mode, pair, gs);
    if (p.kernel < 0) return DGEMM_ERR_NOT_SUPPORTED;
    // Two K slices per stage for tile kernels (CTA pairs and single CTAs; not
    // per-K-group scales) whose operands can be viewed as stacks of whole
    // 128-byte K slices (K a multiple of the slice; N a multiple of the 128-byte
    // atom for B stored K x N): each operand of a stage is then one 3-D TMA copy
    // of twice the bytes, and the TMA unit, which spends a fixed time on every
    // copy, fills the stages faster. The kslices = 1 override keeps one slice.
    p.ks = 1;
    p.slice_k = p.bk;
    if ((pair || p.mode == dg::MODE_TILE) && !gs && (p.mode == dg::MODE_TILE || p.mode == dg::MODE_ROWQ) && K > 0 &&
        K % p.bk == 0 &&
        (!p.b_mn || N % (128 / static_cast<int64_t>(esz)) == 0) && ov.kslices != 1) {
        const int k2 = find_kernel(bn, fp8, p.a_mn, p.b_mn, p.mode, pair, gs, 2);
        if (k2 >= 0) {
            p.kernel = k2;
            p.ks = 2;
            p.bk = 2 * p.slice_k;
        }
    }
    const dg::KernelInfo* k = g_kernels[p.kernel];
    const int tile_m = pair ? 256 : 128;
    const int64_t tiles_m = (p.Mm + tile_m - 1) / tile_m, tiles_n = (p.Nm + bn - 1) / bn;
    if (tiles_m * tiles_n > INT32_MAX) return DGEMM_ERR_NOT_SUPPORTED;
    p.pub.swap_ab = swap ? 1 : 0;
    p.pub.tile_m = tile_m;
    p.pub.tile_n = bn;
    p.pub.cta_group = pair ? 2 : 1;
    p.pub.stages = k->stages;
    p.pub.num_tiles = static_cast<int>(tiles_m * tiles_n);
    const int units = pair ? max_pairs : num_sms;
    p.pub.grid = (pair ? 2 : 1) * static_cast<int>(p.pub.num_tiles < units ? p.pub.num_tiles : units);
    p.pub.raster_group = static_cast<int>(tiles_m < 8 ? (tiles_m > 0 ? tiles_m : 1) : 8);
    if (ov.raster_group >= 1 && ov.raster_group <= tiles_m) p.pub.raster_group = ov.raster_group;
    p.pub.smem_bytes = static_cast<size_t>(k->smem_bytes);

    // Tail splitting: when the tiles do not fill the last wave, run the full
    // waves whole and split each leftover tile along K into as many segments
    // as there are idle units (at most 2), so the wave ends after half a tile
    // instead of a whole one. Needs workspace for FP32 partials, bounded by
    // one tile-sized partial per unit. The partials' round trip through L2
    // costs a few microseconds, so only long tiles (>= kMinTailSlices K
    // slices) are split, and problems with no full wave are left alone.
    // DGEMM_TAIL_SPLIT=0 disables splitting, =force drops the length rule.
    const int64_t k_blocks = (K + p.bk - 1) / p.bk;   // pipeline stages along K
    p.dp_tiles = p.pub.num_tiles;
    p.split = 1;
    p.tail_items = 0;
    p.tail_count_bytes = 0;
    // workspace: status header, per-warp arrival counters, one FP32 partial
    // tile per unit
    size_t split_bytes = 0;
    auto use_split = [&](int dp_tiles, int split, int items) {
        p.dp_tiles = dp_tiles;
        p.split = split;
        p.tail_items = items;
        p.pub.grid = pair_ctas(pair) * (items > units ? units : (dp_tiles > 0 ? units : items));
        p.tail_count_bytes = round_up(static_cast<size_t>(units) * pair_ctas(pair) * k->epi_warps * 8, 256);
        split_bytes = p.tail_count_bytes + static_cast<size_t>(units) * pair_ctas(pair) * 128 * static_cast<size_t>(bn) * 4;
        p.split_offset = kWsStatus;
        p.pub.workspace_bytes = kWsStatus + split_bytes;
    };
    // Split-K when the tiles do not fill one wave (decode shapes, small M x N
    // with long K): every tile is split into K segments run on the idle units.
    // When the segments can form clusters (single-CTA kernels, 2 or 4
    // segments, every cluster resident at once) they are summed through
    // distributed shared memory instead, and no workspace is needed.
    const int64_t sk = (split_ok && k_blocks > 0) ? underfill_split(p.pub.num_tiles, units, k_blocks * p.ks) : 1;
    p.cluster_split = 0;
    if (sk > 1 && (p.mode == dg::MODE_TILE || p.mode == dg::MODE_SWAP)) {
        if (cluster_ok && !pair && (sk == 2 || sk == 4) && p.pub.num_tiles <= (sk == 2 ? max_pairs : max_quads)) {
            p.cluster_split = 1;
            p.dp_tiles = 0;
            p.split = static_cast<int>(sk);
            p.tail_items = p.pub.num_tiles * static_cast<int>(sk);
            p.pub.grid = p.tail_items;
            p.tail_count_bytes = 0;
            p.pub.workspace_bytes = 0;
        } else {
            use_split(0, static_cast<int>(sk), p.pub.num_tiles * static_cast<int>(sk));
        }
    } else if ((p.mode == dg::MODE_TILE || p.mode == dg::MODE_ROWQ) && split_ok && k_blocks > 0) {
        const int rem = p.pub.num_tiles % units;
        if (rem > 0 && p.pub.num_tiles >= units && (force_split || k_blocks * p.ks >= kMinTailSlices)) {
            int64_t split64 = units / rem;
            if (split64 > k_blocks * p.ks / 8) split64 = k_blocks * p.ks / 8;   // >= 8 K slices each
            if (split64 > 2) split64 = 2;   // a third or fourth partial costs more than it saves
            const int split = static_cast<int>(split64);
            if (split >= 2) use_split(p.pub.num_tiles - rem, split, rem * split);
        }
        // N halves (CTA-pair 256-wide kernels) where the K split does not
        // apply: when twice the leftover tiles fit in the last wave, each runs
        // as two 256 x 128 halves over the whole K range, with no partials,
        // reduction or workspace. A half does half the MMA work but reads
        // three quarters of the tile's operand bytes, so on long tiles the K
        // split (half of both) finishes the wave sooner despite its reduction:
        // 4096^3 BF16 ran at 1654 TFLOP/s split along K, 1590 in halves;
        // FP8 4096 x 11008 x 4096 (too short to split) at 3197 in halves,
        // 3165 with whole tiles. The tail_halves = 0 override disables it.
        if (p.split == 1 && rem > 0 && k->halves && 2 * rem <= units && ov.tail_halves != 0) {
            p.tail_halves = 1;
            p.dp_tiles = p.pub.num_tiles - rem;
            p.tail_items = 2 * rem;
            p.pub.grid = pair_ctas(pair) * (p.dp_tiles > 0 ? units : p.tail_items);
        }
    }
    // Footprint. Short small-M calls (every CTA one work item of at most
    // kCompactSlices K slices) run compact -- at most half of the SM's shared
    // memory and Tensor Memory -- so that the next call's CTAs can be resident
    // while these finish (with the 16-wide kernel's registers, two CTAs fit):
    // 1 x 4096 x 4096 and 16 x 4096 x 4096 took 11.9-12.3 us instead of
    // 12.7-13.1, and 32 x 4096 x 4096 (32 wide) 14.0 instead of 14.5. Longer
    // streams keep the full ring, which the compact one slows: 16 x 18432 x
    // 7168 47.0 vs 46.3 us, 64 x 8192^2 32.5 vs 30.0, FP8 64 x 8192^2 (32
    // slices a segment) 20.2 vs 19.6 (200-step runs and CUDA graphs, one GPU).
    const bool compact = p.mode == dg::MODE_SWAP && p.pub.num_tiles <= units && k_blocks > 0 &&
                         (k_blocks * p.ks + p.split - 1) / p.split <= kCompactSlices;
    p.stages = compact ? k->stages_compact : k->stages;
    p.smem = static_cast<size_t>(compact ? k->smem_compact : k->smem_bytes);
    p.tmem_cols = compact && k->tmem_cols > 256 ? 256 : k->tmem_cols;
    p.pub.stages = p.stages;
    p.pub.smem_bytes = p.smem;

    // K-group promotion. The transposed small-M kernel owns all of its Tensor
    // Memory (512 columns, 256 compact) but needs only BN per accumulator: it
    // splits K into as many groups as fit (two buffers of half of it when a CTA
    // runs several tiles, one of all of it when it runs one) and sums them in
    // FP32, which cuts the tensor core's round-toward-zero accumulation error
    // by about that factor.
    int groups = 1;
    p.acc_stride = bn;
    if (gs) {
        groups = static_cast<int>((K + k_group - 1) / k_group);  // scale groups (two buffers alternate)
    } else if (p.mode == dg::MODE_SWAP) {
        const bool one_tile = p.pub.num_tiles <= p.pub.grid;  // (no pairs in this mode)
        const int max_groups = (one_tile ? p.tmem_cols : p.tmem_cols / 2) / bn;
        groups = static_cast<int>(k_blocks < max_groups ? (k_blocks > 0 ? k_blocks : 1) : max_groups);
        p.acc_stride = groups * bn;
    }
    p.pub.k_groups = groups;
    p.pub.tail_tiles = p.pub.num_tiles - p.dp_tiles;
    p.pub.tail_split = p.split;
    p.pub.tail_units = p.split > 1 ? p.tail_items : (p.tail_halves ? p.tail_items : 0);
    p.pub.k_slices = p.ks;
    p.pub.cluster_split = p.cluster_split;
    p.pub.tail_halves = p.tail_halves;
    // Requantisation: status header, barrier header, row maxima, BF16 stash,
    // then (tail split) the split area.
    if (oq) {
        const size_t base =
            kWsStatus + kWsHeader + round_up(static_cast<size_t>(M) * 4, 256) + static_cast<size_t>(M) * N * 2;
        if (p.split > 1) {
            p.split_offset = round_up(base, 256);
            p.pub.workspace_bytes = p.split_offset + split_bytes;
        } else {
            p.pub.workspace_bytes = base;
        }
    }
    // Cross-CTA waits. The requantising kernel's last waits (for the row bands
    // other CTAs are still finishing) need every CTA resident: it is launched
    // cooperatively (the grid is sized from the measured occupancy too). Split
    // tiles that exchange partial sums through the workspace either run in a
    // cooperative launch, where every segment waits for all (under-filled
    // grids: the exchange ends the kernel, so its shortest form pays), or in a
    // plain launch, where no segment waits for one that may not have started
    // (the last to arrive finishes the tile: the tail split, whose exchange
    // overlaps whole tiles and which keeps programmatic dependent launch).
    // The cooperative = 0 override drops the attribute (profilers that cannot
    // launch cooperative cluster grids); the requantising form's band waits
    // then rely on an otherwise idle GPU, and every wait stays bounded.
    const bool ws_exchange = p.split > 1 && !p.cluster_split;
    int coop = (p.mode == dg::MODE_ROWQ || (ws_exchange && p.dp_tiles == 0)) ? 1 : 0;
    if (ov.cooperative == 0) coop = 0;
    if (ov.cooperative == 1 && ws_exchange) coop = 1;
    p.pub.cooperative = coop;
    // The K segments of split tiles run first in the plain tile form, as the
    // raster's first tiles, so their exchange of partial sums overlaps whole
    // tiles (+5 % at 4096^3 BF16); the requantising form keeps them last (its
    // row bands count the split tiles at the end of the raster).
    p.seg_first = (p.mode == dg::MODE_TILE && ov.seg_first != 0) ? 1 : 0;
    *out = p;
    return DGEMM_OK;
}

void init_encode() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// 2-D row-major tensor: `inner` contiguous elements per row, `outer` rows,
// rows `pitch` bytes apart; box of box_inner x box_outer; 128-byte swizzle;
// out-of-range elements load as zero and are not stored.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t pitch, uint32_t box_inner, uint32_t box_outer) {
    std::call_once(g_encode_once, init_encode);
    if (!g_encode) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a row-major matrix as a stack of 128-byte slices: dims
// (inner elements of one slice, rows, slices), strides (row pitch, slice
// pitch) in bytes; box of box_inner x box_rows x box_slices; 128-byte swizzle;
// out-of-range rows and slices load as zero.
bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t rows,
               uint64_t slices, uint64_t row_pitch, uint64_t slice_pitch, uint32_t box_inner, uint32_t box_rows,
               uint32_t box_slices) {
    std::call_once(g_encode_once, init_encode);
    if (!g_encode) return false;
    const cuuint64_t dims[3] = {inner, rows, slices};
    const cuuint64_t strides[2] = {row_pitch, slice_pitch};
    const cuuint32_t box[3] = {box_inner, box_rows, box_slices};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

dgemm_status_t device_state(DeviceState** out, int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DGEMM_ERR_NOT_SUPPORTED;
    DeviceState& d = g_dev[dev];
    std::call_once(d.once, [&d, dev]() {
        cudaError_t e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess && d.cc_major == 10 && d.cc_minor == 3)
            e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status);
        d.err = e;
    });
    if (d.err != cudaSuccess) return DGEMM_ERR_CUDA;
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return DGEMM_ERR_ARCH;
    *out = &d;
    *dev_out = dev;
    return DGEMM_OK;
}

// Dynamic shared memory opt-in, once per kernel variant and device.
cudaError_t configure_kernel(int kernel, int devid) {
    std::atomic<unsigned char>& flag = g_attr_set[kernel][devid];
    if (flag.load(std::memory_order_acquire)) return cudaSuccess;
    const dg::KernelInfo* k = g_kernels[kernel];
    cudaError_t e = cudaFuncSetAttribute(k->func, cudaFuncAttributeMaxDynamicSharedMemorySize, k->smem_bytes);
    if (e == cudaSuccess && k->launch_regs > 0) {
        // A kernel that moves registers between warpgroups must be launched
        // with at least the registers its split adds up to, or the raising
        // warpgroups would wait forever: refuse to launch it otherwise.
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, k->func);
        if (e == cudaSuccess && fa.numRegs < k->launch_regs) e = cudaErrorInvalidConfiguration;
    }
    if (e == cudaSuccess) flag.store(1, std::memory_order_release);
    return e;
}

// How many clusters of `size` CTAs (2: the CTA-pair kernels; 4: single-CTA
// kernels whose split K segments share a cluster) fit on the device at once,
// measured once per device with the occupancy API on a representative kernel
// (every variant runs one CTA per SM). 0: none.
int g_max_clusters[kMaxDevices][2][2];
std::once_flag g_clusters_once[kMaxDevices][2][2];

int max_clusters(DeviceState* dev, int devid, int fp8, int size) {
    const int si = size == 2 ? 0 : 1;
    std::call_once(g_clusters_once[devid][fp8][si], [&]() {
        int best = 0;
        std::call_once(g_kernels_once, collect_kernels);
        for (int i = 0; i < g_nk; ++i) {
            const dg::KernelInfo* k = g_kernels[i];
            if (k->pair != (size == 2 ? 1 : 0) || k->fp8 != fp8 || k->mode != dg::MODE_TILE || k->gs) continue;
            if (configure_kernel(i, devid) != cudaSuccess) continue;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(size * dev->num_sms));
            cfg.blockDim = dim3(static_cast<unsigned>(k->threads));
            cfg.dynamicSmemBytes = static_cast<size_t>(k->smem_bytes);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(size);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k->func, &cfg) == cudaSuccess) best = n;
            else (void)cudaGetLastError();
            break;
        }
        g_max_clusters[devid][fp8][si] = best > dev->num_sms / size ? dev->num_sms / size : best;
    });
    return g_max_clusters[devid][fp8][si];
}

int max_pairs(DeviceState* dev, int devid, int fp8) { return max_clusters(dev, devid, fp8, 2); }
int max_quads(DeviceState* dev, int devid, int fp8) { return max_clusters(dev, devid, fp8, 4); }

// Without a device: a GB300's measured 36 four-CTA clusters on 152 SMs, scaled.
int quads_estimate(int num_sms) { return num_sms * 36 / 152; }

CUtensorMapDataType tm_type(dgemm_dtype_t t) {
    return t == DGEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                          : t == DGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
}

// status_in_ws: device-side errors of the call go to the status word at the
// start of ws (when ws holds at least kWsStatus bytes) instead of the
// per-device word.
dgemm_status_t run(int fp8, const void* A, const void* B, dgemm_b_layout_t bl, const float* a_scale,
                   const float* b_scale, const void* C, dgemm_dtype_t c_dtype, void* D, dgemm_dtype_t d_dtype,
                   int64_t M, int64_t N, int64_t K, float alpha, float beta, const dgemm_epilogue_t* epi, void* ws,
                   size_t ws_bytes, cudaStream_t stream, int k_group = 0, int b_block = 1,
                   bool status_in_ws = true) {
    // ---- arguments that need no device
    if (b_block != 1 && (b_block != kWeightBlock || k_group <= 0)) return DGEMM_ERR_INVALID_VALUE;
    Plan plan;
    dgemm_status_t st = make_plan(fp8, M, N, K, bl, d_dtype, epi, 2, 1, 0, false, &plan, k_group);
    if (st != DGEMM_OK) return st;
    if (M == 0 || N == 0) return DGEMM_OK;
    if (!D || (K > 0 && (!A || !B))) return DGEMM_ERR_INVALID_VALUE;
    if (fp8 && (!a_scale || !b_scale)) return DGEMM_ERR_INVALID_VALUE;
    if (beta != 0.0f) {
        if (!C) return DGEMM_ERR_INVALID_VALUE;
        if (c_dtype != DGEMM_F32 && c_dtype != DGEMM_BF16) return DGEMM_ERR_INVALID_VALUE;
        if ((static_cast<size_t>(N) * dtype_bytes(c_dtype)) % 16 != 0) return DGEMM_ERR_MISALIGNED;
        if (!aligned16(C)) return DGEMM_ERR_MISALIGNED;
    }
    const int oq = epi ? epi->out_quant : DGEMM_QUANT_NONE;
    const float* bias = epi ? epi->bias : nullptr;
    if (oq && !epi->out_row_scale) return DGEMM_ERR_INVALID_VALUE;
    if ((K > 0 && (!aligned16(A) || !aligned16(B))) || !aligned16(D)) return DGEMM_ERR_MISALIGNED;
    if ((a_scale && !aligned16(a_scale)) || (b_scale && !aligned16(b_scale)) || (bias && !aligned16(bias)) ||
        (oq && !aligned16(epi->out_row_scale)) || (ws && !aligned16(ws)))
        return DGEMM_ERR_MISALIGNED;
    if (plan.pub.workspace_bytes > 0 && (!ws || ws_bytes < plan.pub.workspace_bytes))
        return DGEMM_ERR_WORKSPACE_TOO_SMALL;

    // ---- device
    DeviceState* dev = nullptr;
    int devid = 0;
    st = device_state(&dev, &devid);
    if (st != DGEMM_OK) return st;
    const int pairs = max_pairs(dev, devid, fp8);
    const int quads = max_quads(dev, devid, fp8);
    st = make_plan(fp8, M, N, K, bl, d_dtype, epi, dev->num_sms, pairs, quads, true, &plan, k_group);
    if (st != DGEMM_OK) return st;
    if (plan.split > 1 && plan.pub.workspace_bytes > 0 && (!ws || ws_bytes < plan.pub.workspace_bytes)) {
        st = make_plan(fp8, M, N, K, bl, d_dtype, epi, dev->num_sms, pairs, quads, false, &plan,
                       k_group);  // no room: whole tiles
        if (st != DGEMM_OK) return st;
    }
    const dg::KernelInfo* k = g_kernels[plan.kernel];
    if (configure_kernel(plan.kernel, devid) != cudaSuccess) return DGEMM_ERR_CUDA;

    // ---- tensor maps
    const dgemm_dtype_t in_t = fp8 ? DGEMM_E4M3 : DGEMM_BF16;
    const size_t esz = fp8 ? 1 : 2;
    const int mn_atom = static_cast<int>(128 / esz);
    alignas(64) CUtensorMap tmA, tmB, tmBh, tmD;
    std::memset(&tmA, 0, sizeof tmA);
    std::memset(&tmB, 0, sizeof tmB);
    std::memset(&tmBh, 0, sizeof tmBh);
    std::memset(&tmD, 0, sizeof tmD);
    // The MMA's operands: X (rows of the MMA's M) and Y (rows of its N).
    const void* X = plan.pub.swap_ab ? B : A;
    const void* Y = plan.pub.swap_ab ? A : B;
    if (K > 0 && plan.ks == 2) {
        // two K slices per stage: each operand of a stage in one 3-D copy
        const uint64_t sk = plan.slice_k;   // elements per 128-byte slice
        const uint64_t nslices = static_cast<uint64_t>(K) / sk;
        const uint32_t bn_cta = static_cast<uint32_t>(plan.pub.tile_n / plan.pub.cta_group);
        bool ok = encode_3d(&tmA, tm_type(in_t), X, sk, plan.Mm, nslices, K * esz, 128, sk, 128, 2);
        if (!ok) return DGEMM_ERR_CUDA;
        if (plan.b_mn) {   // B stored K x N: N atoms of 128 bytes, 2 slices of K rows each
            const uint64_t atoms = static_cast<uint64_t>(N) / mn_atom;
            ok = encode_3d(&tmB, tm_type(in_t), Y, mn_atom, K, atoms, N * esz, 128, mn_atom, 2 * sk,
                           bn_cta / mn_atom);
            if (ok && plan.tail_halves)
                ok = encode_3d(&tmBh, tm_type(in_t), Y, mn_atom, K, atoms, N * esz, 128, mn_atom, 2 * sk,
                               bn_cta / 2 / mn_atom);
        } else {           // B stored N x K: K-major like A
            ok = encode_3d(&tmB, tm_type(in_t), Y, sk, plan.Nm, nslices, K * esz, 128, sk, bn_cta, 2);
            if (ok && plan.tail_halves)
                ok = encode_3d(&tmBh, tm_type(in_t), Y, sk, plan.Nm, nslices, K * esz, 128, sk, bn_cta / 2, 2);
        }
        if (!ok) return DGEMM_ERR_CUDA;
    } else if (K > 0) {
        bool ok;
        if (plan.a_mn)  // X = op(B)^T with B stored K x N: MN-major
            ok = encode_2d(&tmA, tm_type(in_t), X, N, K, N * esz, mn_atom, plan.bk);
        else            // X stored Mm x K: K-major
            ok = encode_2d(&tmA, tm_type(in_t), X, K, plan.Mm, K * esz, plan.bk, 128);
        if (!ok) return DGEMM_ERR_CUDA;
        if (plan.b_mn)  // Y = B stored K x N: MN-major
            ok = encode_2d(&tmB, tm_type(in_t), Y, N, K, N * esz, mn_atom, plan.bk);
        else            // Y stored Nm x K: K-major
            ok = encode_2d(&tmB, tm_type(in_t), Y, K, plan.Nm, K * esz, plan.bk,
                           static_cast<uint32_t>(plan.pub.tile_n / plan.pub.cta_group));
        if (!ok) return DGEMM_ERR_CUDA;
        // a tail half's B rows: half the box of K-major B (MN-major B loads
        // whole atoms through tmB)
        if (plan.tail_halves && !plan.b_mn &&
            !encode_2d(&tmBh, tm_type(in_t), Y, K, plan.Nm, K * esz, plan.bk,
                       static_cast<uint32_t>(plan.pub.tile_n / plan.pub.cta_group / 2)))
            return DGEMM_ERR_CUDA;
    }
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const size_t amax_bytes = round_up(static_cast<size_t>(M) * 4, 256);
    if (plan.mode == dg::MODE_TILE) {
        const size_t dsz = dtype_bytes(d_dtype);
        if (!encode_2d(&tmD, tm_type(d_dtype), D, N, M, N * dsz, static_cast<uint32_t>(128 / dsz), 32))
            return DGEMM_ERR_CUDA;
    } else if (plan.mode == dg::MODE_ROWQ) {
        if (!encode_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, wsb + kWsStatus + kWsHeader + amax_bytes, N, M, N * 2,
                       64, 32))
            return DGEMM_ERR_CUDA;
    }

    // ---- parameters
    dg::Params p{};
    p.M = static_cast<int>(plan.Mm);
    p.N = static_cast<int>(plan.Nm);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((plan.Mm + plan.pub.tile_m - 1) / plan.pub.tile_m);
    p.tiles_n = static_cast<int>((plan.Nm + plan.pub.tile_n - 1) / plan.pub.tile_n);
    p.num_tiles = plan.pub.num_tiles;
    p.k_blocks = static_cast<int>((K + plan.bk - 1) / plan.bk);
    p.group_m = plan.pub.raster_group;
    p.acc_groups = plan.gs ? 1 : plan.pub.k_groups;
    p.acc_stride = plan.acc_stride;
    p.stages = plan.stages;
    p.tmem_cols = plan.tmem_cols;
    p.alpha = alpha;
    p.beta = beta;
    p.C = beta != 0.0f ? C : nullptr;
    p.ldc = N;
    p.c_f32 = c_dtype == DGEMM_F32;
    p.D = D;
    p.ldd = N;
    p.d_f32 = d_dtype == DGEMM_F32;
    if (plan.gs) {
        // group-major tables: a_scale [G][M], b_scale [G][N] (block-scaled
        // weights: [G][ceil(N / 128)])
        const int64_t nb_cols = b_block > 1 ? (N + b_block - 1) / b_block : N;
        const int shift = b_block > 1 ? kWeightBlockShift : 0;
        p.row_gscale = plan.pub.swap_ab ? b_scale : a_scale;
        p.col_gscale = plan.pub.swap_ab ? a_scale : b_scale;
        p.gs_ld_row = plan.pub.swap_ab ? nb_cols : M;
        p.gs_ld_col = plan.pub.swap_ab ? M : nb_cols;
        p.gs_row_shift = plan.pub.swap_ab ? shift : 0;
        p.gs_col_shift = plan.pub.swap_ab ? 0 : shift;
        p.group_kb = plan.group_kb;
    } else {
        p.row_scale = plan.pub.swap_ab ? b_scale : a_scale;
        p.col_scale = plan.pub.swap_ab ? a_scale : b_scale;
    }
    p.bias = bias;
    p.act = epi ? epi->act : 0;
    const dgemm_overrides_t ov = overrides_now();
    p.status = dev->status;
    p.epoch = next_epoch();
    p.ws_status = (status_in_ws && ws && ws_bytes >= kWsStatus) ? static_cast<unsigned long long*>(ws) : nullptr;
    p.wait_ns = ov.wait_limit_ns > 0 ? static_cast<uint64_t>(ov.wait_limit_ns) : dg::kWaitLimitNs;
    p.stall_after = ov.stall_after_loads;
    p.dp_tiles = plan.dp_tiles;
    p.split = plan.split;
    p.tail_items = plan.tail_items;
    p.seg_first = plan.seg_first;
    p.split_sym = plan.pub.cooperative;
    if (plan.split > 1) {
        p.tail_count = reinterpret_cast<unsigned long long*>(wsb + plan.split_offset);
        p.partials = reinterpret_cast<float*>(wsb + plan.split_offset + plan.tail_count_bytes);
    }
    if (plan.mode == dg::MODE_ROWQ) {
        // after the status header: the chunk claim counter, then one arrival
        // counter per row band (a band of rq_gpc raster groups, so that at
        // most kMaxBands of them)
        uint8_t* hdr = wsb + kWsStatus;
        p.rq_next = reinterpret_cast<unsigned long long*>(hdr);
        p.band_count = reinterpret_cast<unsigned*>(hdr + 8);
        const int64_t groups = (p.tiles_m + p.group_m - 1) / p.group_m;
        p.rq_gpc = static_cast<int>(groups > 0 ? (groups + dg::kMaxBands - 1) / dg::kMaxBands : 1);
        p.amax = reinterpret_cast<unsigned*>(hdr + kWsHeader);
        p.stash = reinterpret_cast<const uint16_t*>(hdr + kWsHeader + amax_bytes);
        p.q_out = static_cast<uint8_t*>(D);
        p.out_row_scale = epi->out_row_scale;
        if (cudaMemsetAsync(hdr, 0, kWsHeader + amax_bytes, stream) != cudaSuccess) return DGEMM_ERR_CUDA;
    }
    p.cluster_split = plan.cluster_split;
    p.tail_halves = plan.tail_halves;
    if (plan.tail_halves && !k->halves) return DGEMM_ERR_NOT_SUPPORTED;
    if (k->launch(tmA, tmB, tmBh, tmD, p, plan.pub.grid, stream, plan.pub.cooperative != 0,
                  plan.cluster_split ? plan.split : 1, plan.smem) != cudaSuccess)
        return DGEMM_ERR_CUDA;
    return DGEMM_OK;
}

}  // namespace

extern "C" {

dgemm_status_t dgemm_bf16(const void* A, const void* B, dgemm_b_layout_t b_layout, const void* C,
                          dgemm_dtype_t c_dtype, void* D, dgemm_dtype_t d_dtype, int64_t M, int64_t N, int64_t K,
                          float alpha, float beta, const dgemm_epilogue_t* epi, void* ws, size_t ws_bytes,
                          dgemm_stream_t stream) {
    return run(0, A, B, b_layout, nullptr, nullptr, C, c_dtype, D, d_dtype, M, N, K, alpha, beta, epi, ws, ws_bytes,
               reinterpret_cast<cudaStream_t>(stream));
}

dgemm_status_t dgemm_fp8_scaled(const void* Aq, const void* Bq, dgemm_b_layout_t b_layout, const float* a_scale,
                                const float* b_scale, int k_group, const void* C, dgemm_dtype_t c_dtype, void* D,
                                dgemm_dtype_t d_dtype, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                const dgemm_epilogue_t* epi, void* ws, size_t ws_bytes, dgemm_stream_t stream) {
    return run(1, Aq, Bq, b_layout, a_scale, b_scale, C, c_dtype, D, d_dtype, M, N, K, alpha, beta, epi, ws,
               ws_bytes, reinterpret_cast<cudaStream_t>(stream), k_group);
}

dgemm_status_t dgemm_fp8_blockscaled(const void* Aq, const void* Bq, dgemm_b_layout_t b_layout,
                                     const float* a_scale, const float* b_scale, int k_group, const void* C,
                                     dgemm_dtype_t c_dtype, void* D, dgemm_dtype_t d_dtype, int64_t M, int64_t N,
                                     int64_t K, float alpha, float beta, const dgemm_epilogue_t* epi, void* ws,
                                     size_t ws_bytes, dgemm_stream_t stream) {
    if (k_group <= 0) return DGEMM_ERR_INVALID_VALUE;
    return run(1, Aq, Bq, b_layout, a_scale, b_scale, C, c_dtype, D, d_dtype, M, N, K, alpha, beta, epi, ws,
               ws_bytes, reinterpret_cast<cudaStream_t>(stream), k_group, kWeightBlock);
}

size_t dgemm_workspace_size(int is_fp8, int64_t M, int64_t N, int64_t K, dgemm_b_layout_t b_layout,
                            const dgemm_epilogue_t* epi) {
    // SM count of the current device if there is one, else a GB300's 152.
    int sms = 152, pairs = 76, quads = quads_estimate(152);
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        DeviceState* ds = nullptr;
        int devid = 0;
        if (device_state(&ds, &devid) == DGEMM_OK) {
            sms = ds->num_sms;
            pairs = max_pairs(ds, devid, is_fp8 ? 1 : 0);
            quads = max_quads(ds, devid, is_fp8 ? 1 : 0);
        }
    } else {
        (void)cudaGetLastError();
    }
    Plan plan;
    const dgemm_dtype_t d = (epi && epi->out_quant) ? DGEMM_E4M3 : DGEMM_BF16;
    if (make_plan(is_fp8 ? 1 : 0, M, N, K, b_layout, d, epi, sms, pairs, quads, true, &plan) != DGEMM_OK) {
        // the output dtype is not an argument here: retry with FP32 output
        if (make_plan(is_fp8 ? 1 : 0, M, N, K, b_layout, DGEMM_F32, epi, sms, pairs, quads, true, &plan) !=
            DGEMM_OK)
            return 0;
    }
    return plan.pub.workspace_bytes;
}

dgemm_status_t dgemm_plan(int is_fp8, int64_t M, int64_t N, int64_t K, dgemm_b_layout_t b_layout,
                          dgemm_dtype_t d_dtype, const dgemm_epilogue_t* epi, int k_group, int num_sms,
                          dgemm_plan_t* plan) {
    if (!plan) return DGEMM_ERR_INVALID_VALUE;
    int pairs = num_sms / 2, quads = quads_estimate(num_sms);
    if (num_sms <= 0) {  // the current device: its SM count and measured cluster occupancy
        DeviceState* ds = nullptr;
        int devid = 0;
        const dgemm_status_t dst = device_state(&ds, &devid);
        if (dst != DGEMM_OK) return dst;
        num_sms = ds->num_sms;
        pairs = max_pairs(ds, devid, is_fp8 ? 1 : 0);
        quads = max_quads(ds, devid, is_fp8 ? 1 : 0);
    }
    Plan p;
    const dgemm_status_t st =
        make_plan(is_fp8 ? 1 : 0, M, N, K, b_layout, d_dtype, epi, num_sms, pairs, quads, true, &p, k_group);
    if (st == DGEMM_OK) *plan = p.pub;
    return st;
}

const char* dgemm_status_string(dgemm_status_t s) {
    switch (s) {
        case DGEMM_OK: return "success";
        case DGEMM_ERR_INVALID_VALUE: return "invalid argument (NULL pointer, negative size or bad enum)";
        case DGEMM_ERR_NOT_SUPPORTED: return "request not supported by this build";
        case DGEMM_ERR_MISALIGNED: return "pointer or leading dimension not 16-byte aligned";
        case DGEMM_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than dgemm_workspace_size()";
        case DGEMM_ERR_CUDA: return "a CUDA runtime or driver call failed";
        case DGEMM_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait gave up";
        case DGEMM_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    }
    return "unknown status";
}

dgemm_status_t dgemm_query_device_status(const void* ws, dgemm_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return DGEMM_ERR_CUDA;
    DeviceState* dev = nullptr;
    int devid = 0;
    const dgemm_status_t st = device_state(&dev, &devid);
    if (st != DGEMM_OK) return st;
    if (ws != nullptr) {
        // the workspace's status word: errors of calls that used this workspace,
        // tagged with their launch epoch (any other content reads as no error)
        if (!aligned16(ws)) return DGEMM_ERR_MISALIGNED;
        unsigned long long w = 0;
        if (cudaMemcpy(&w, ws, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) return DGEMM_ERR_CUDA;
        if ((w & 0xFFull) == 0 || !issued_epoch(w >> 8)) return DGEMM_OK;
        const unsigned long long zero = 0;
        if (cudaMemcpy(const_cast<void*>(ws), &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return DGEMM_ERR_CUDA;
        return DGEMM_ERR_DEVICE_TIMEOUT;
    }
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return DGEMM_ERR_CUDA;
    if (v == 0) return DGEMM_OK;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess) return DGEMM_ERR_CUDA;
    return DGEMM_ERR_DEVICE_TIMEOUT;
}

void dgemm_overrides_init(dgemm_overrides_t* o) {
    if (o) overrides_defaults(o);
}

dgemm_status_t dgemm_set_overrides(const dgemm_overrides_t* o) {
    std::call_once(g_ovr_once, init_overrides);
    dgemm_overrides_t v;
    overrides_defaults(&v);
    if (o) {
        if (o->tile_n < 0 || o->cta_pair < -1 || o->cta_pair > 1 || o->tail_split < -1 || o->tail_split > 1 ||
            o->tail_halves < -1 || o->tail_halves > 0 || o->cluster_split < -1 || o->cluster_split > 0 ||
            o->seg_first < -1 || o->seg_first > 1 ||
            o->raster_group < 0 || o->cooperative < -1 || o->cooperative > 1 ||
            !(o->kslices == -1 || o->kslices == 1 || o->kslices == 2) || o->wait_limit_ns < 0 ||
            o->stall_after_loads < -1)
            return DGEMM_ERR_INVALID_VALUE;
        v = *o;
    }
    dgemm_overrides_t d;
    overrides_defaults(&d);
    std::lock_guard<std::mutex> lk(g_ovr_mutex);
    g_ovr = v;
    g_ovr_set.store(std::memcmp(&v, &d, sizeof v) != 0, std::memory_order_release);
    return DGEMM_OK;
}

dgemm_status_t dgemm_get_overrides(dgemm_overrides_t* o) {
    if (!o) return DGEMM_ERR_INVALID_VALUE;
    *o = overrides_now();
    return DGEMM_OK;
}

}  // extern "C"

// ---- Allocation-free variant of the requantising FP8 GEMM -------------------
// For callers that cannot allocate device memory when they run the GEMM (see
// dgemm.h): the scratch the requantising kernel needs comes from this
// file-scope device array instead of a caller workspace. In host code the name
// g_noalloc_scratch is only a host-side stand-in, never a device address; the
// device address is looked up once per device with cudaGetSymbolAddress and
// passed to the kernel through the workspace argument of run().
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DGEMM_NOALLOC_SCRATCH_BYTES];

struct NoAllocScratch {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void* ptr = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocScratch g_noalloc[kMaxDevices];

}  // namespace

extern "C" dgemm_status_t dgemm_fp8_rowquant_noalloc(const void* Aq, const void* Bq, dgemm_b_layout_t b_layout,
                                                     const float* a_scale, const float* b_scale, const void* C,
                                                     dgemm_dtype_t c_dtype, void* Dq, int64_t M, int64_t N,
                                                     int64_t K, float alpha, float beta,
                                                     const dgemm_epilogue_t* epi, dgemm_stream_t stream) {
    if (!epi || epi->out_quant != DGEMM_QUANT_E4M3_ROW_AMAX) return DGEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return DGEMM_ERR_INVALID_VALUE;
    // the requantising scratch without a split area (with too little room for
    // one, run() keeps whole tiles)
    const size_t need =
        kWsStatus + kWsHeader + round_up(static_cast<size_t>(M) * 4, 256) + static_cast<size_t>(M) * N * 2;
    if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || need > DGEMM_NOALLOC_SCRATCH_BYTES)
        return DGEMM_ERR_WORKSPACE_TOO_SMALL;
    DeviceState* dev = nullptr;
    int devid = 0;
    const dgemm_status_t st = device_state(&dev, &devid);  // also rejects devices other than sm_103
    if (st != DGEMM_OK) return st;
    NoAllocScratch& s = g_noalloc[devid];
    std::call_once(s.once, [&s]() {
        s.err = cudaGetSymbolAddress(&s.ptr, g_noalloc_scratch);
    });
    if (s.err != cudaSuccess || s.ptr == nullptr) return DGEMM_ERR_CUDA;
    // (device-side errors go to the per-device word: the caller cannot name the array)
    return run(1, Aq, Bq, b_layout, a_scale, b_scale, C, c_dtype, Dq, DGEMM_E4M3, M, N, K, alpha, beta, epi, s.ptr,
               DGEMM_NOALLOC_SCRATCH_BYTES, reinterpret_cast<cudaStream_t>(stream), 0, 1, false);
}
