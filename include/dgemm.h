/*
 * dgemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * The library computes, on one GPU,
 *
 *     D = epilogue( alpha * op(A) . op(B) + beta * C )
 *
 * in two forms: BF16 operands with FP32 accumulation (dgemm_bf16), and FP8
 * E4M3 operands with one FP32 scale per row of A (per token) and one per
 * output channel of B applied to the FP32 accumulator inside the kernel
 * (dgemm_fp8_scaled). The epilogue (bias, activation, output conversion or
 * per-row E4M3 requantisation) runs inside the same kernel, so no second
 * kernel reads the product.
 *
 * Sources, cited by page title and section:
 *   [W1] DeepGEMM write-up, czchanglian.com/news/51329: C = alpha*A*B + beta*C,
 *        A is M x K, B is K x N (§1.1); FP32 accumulation of 16-bit inputs
 *        (§3.1); fused bias + activation (§6.1); per-token output
 *        quantisation in the epilogue (§6.2).
 *   [W3] "DeepGEMM: FP8 Tensor Core GEMM", bjdmk.com.cn/news/6078902:
 *        E4M3 operands with per-token x per-channel scales applied to the
 *        accumulated result (§1.2, §3.2); the call takes pointers, M/N/K, a
 *        scale descriptor, a workspace whose size is queried first so nothing
 *        is allocated at run time, and a CUDA stream (§5.1).
 *
 * Conventions shared by every entry point
 *   - All matrices are row-major and contiguous: A is M x K (leading
 *     dimension K); B is K x N (DGEMM_B_KN, leading dimension N) or N x K
 *     (DGEMM_B_NK, leading dimension K: the weight layout of a linear layer,
 *     D = A . B^T); C and D are M x N (leading dimension N).
 *   - Every pointer argument except `stream` is a DEVICE pointer, except the
 *     `epi` and `plan` structs, which live in host memory and are read or
 *     written before the call returns. The caller owns all memory; the library
 *     allocates none, per call or otherwise (it only caches small host-side
 *     state such as device properties).
 *   - Device pointers must be 16-byte aligned and every leading dimension in
 *     bytes a multiple of 16 (the tensor-memory-accelerator rule); otherwise
 *     the call returns DGEMM_ERR_MISALIGNED before launching anything.
 *   - M == 0 or N == 0: nothing to do, DGEMM_OK. K == 0 is valid: the product
 *     is zero and D = epilogue(beta * C).
 *   - beta == 0: C is not read and may be NULL (BLAS convention). C may equal
 *     D (in-place update) when c_dtype == d_dtype.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream). Argument errors return synchronously, before launch.
 *     A failed launch returns DGEMM_ERR_CUDA. Every device-side wait is
 *     bounded (about one second); one that gives up is recorded in the call's
 *     status word -- the first DGEMM_WS_STATUS_BYTES bytes of its workspace
 *     when it was given one at least that large, else a per-device word --
 *     and the kernel drains and returns. dgemm_query_device_status reports it.
 *   - The device must be compute capability 10.3 (GB300, sm_103a); any other
 *     device gives DGEMM_ERR_ARCH.
 *   - The library caches per-device state on first use (properties, kernel
 *     attributes, the device addresses of its own __device__ words). Do not
 *     keep using it on a device after cudaDeviceReset: a reset frees those
 *     addresses, and later calls would launch with stale ones.
 */
#ifndef DGEMM_H
#define DGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* The same type as cudaStream_t. */
typedef struct CUstream_st* dgemm_stream_t;

typedef enum {
    DGEMM_OK = 0,
    DGEMM_ERR_INVALID_VALUE = 1,       /* NULL pointer, negative size, bad enum  */
    DGEMM_ERR_NOT_SUPPORTED = 2,       /* valid request this build cannot serve  */
    DGEMM_ERR_MISALIGNED = 3,          /* pointer or leading dimension alignment */
    DGEMM_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes < dgemm_workspace_size(...)   */
    DGEMM_ERR_CUDA = 5,                /* a CUDA runtime/driver call failed      */
    DGEMM_ERR_DEVICE_TIMEOUT = 6,      /* a bounded device-side wait gave up     */
    DGEMM_ERR_ARCH = 7                 /* device is not sm_103                   */
} dgemm_status_t;

typedef enum { DGEMM_F32 = 0, DGEMM_BF16 = 1, DGEMM_E4M3 = 2 } dgemm_dtype_t;

/* Bytes at the start of a workspace that hold the call's status word (an
 * epoch-tagged word: its contents on entry do not matter). */
#define DGEMM_WS_STATUS_BYTES 256

typedef enum {
    DGEMM_B_KN = 0, /* B stored K x N row-major                      */
    DGEMM_B_NK = 1  /* B stored N x K row-major (D = A . B^T)         */
} dgemm_b_layout_t;

typedef enum {
    DGEMM_ACT_NONE = 0,
    DGEMM_ACT_RELU = 1,
    DGEMM_ACT_GELU = 2, /* erf form: y/2 (1 + erf(y / sqrt 2))          */
    DGEMM_ACT_SILU = 3  /* y / (1 + exp(-y))                             */
} dgemm_act_t;

typedef enum {
    DGEMM_QUANT_NONE = 0,
    /* D is E4M3 with one FP32 scale per row: s[m] = max_n |y[m,n]| / 448 and
     * D[m,n] = RN_E4M3(y[m,n] / s[m]), saturating; a row of zeros gets s = 1.
     * [W1] §6.2 (per-token output quantisation fused in the epilogue). */
    DGEMM_QUANT_E4M3_ROW_AMAX = 1
} dgemm_out_quant_t;

/* Fused epilogue, applied in this order after alpha*acc + beta*C:
 * + bias[n] -> activation -> output conversion or requantisation.
 * [W1] §6.1-6.2. A NULL dgemm_epilogue_t* means: no bias, no activation, no
 * requantisation. */
typedef struct {
    const float* bias;    /* [N] FP32 device pointer, or NULL                   */
    int act;              /* dgemm_act_t                                        */
    int out_quant;        /* dgemm_out_quant_t; E4M3_ROW_AMAX needs d_dtype E4M3 */
    float* out_row_scale; /* [M] FP32 device pointer, written when out_quant != 0 */
} dgemm_epilogue_t;

/* What the planner chose for a problem (filled by dgemm_plan). */
typedef struct {
    int swap_ab;           /* 1: computes D^T = op(B)^T . A^T so the 128-row MMA
                              dimension runs over N (small-M, decode shapes)     */
    int tile_m, tile_n;    /* output tile of one CTA, in the MMA's orientation  */
    int cta_group;         /* CTAs that share one MMA (1 or 2)                  */
    int stages;            /* shared-memory pipeline depth (the small-M form's
                              short calls run a compact ring of at most half an
                              SM's shared memory and 256 TMEM columns)          */
    int num_tiles;         /* output tiles                                      */
    int grid;              /* CTAs launched (persistent: <= SM count)           */
    int cooperative;       /* 1: launched cooperatively, so every CTA is
                              resident: CTAs wait on row bands other CTAs
                              finish (requantisation) or on every K segment of
                              a split tile (partials through the workspace)   */
    int raster_group;      /* tile rows per band of the swizzled raster         */
    int k_groups;          /* K-group promotion: K is split into this many
                              contiguous groups, each accumulated by the tensor
                              core separately and summed in FP32 (1 = off)      */
    int tail_tiles;        /* tiles beyond the last whole wave that are split
                              (along K, or along N with tail_halves) so the
                              partial wave finishes sooner (0 = none). In the
                              plain (not requantising) form their K segments
                              run first, as the raster's first tiles, and their
                              partial sums are exchanged while whole tiles
                              run; otherwise they run last                    */
    int tail_split;        /* K segments per tail tile (1 = no splitting)       */
    int cluster_split;     /* 1: the K segments of each split tile run as one
                              thread-block cluster and are summed through
                              distributed shared memory (no workspace needed) */
    int tail_halves;       /* 1: the tail_tiles run instead as two halves of
                              tile_n / 2 columns each, every half over the
                              whole K range (no workspace needed)            */
    int tail_units;        /* units (CTAs or CTA pairs) that run the tail's
                              K segments or halves, one each (0 = none)        */
    int k_slices;          /* 128-byte K slices per pipeline stage (2: each
                              operand of a stage arrives in one 3-D TMA copy) */
    size_t smem_bytes;     /* dynamic shared memory per CTA                     */
    size_t workspace_bytes;/* what dgemm_workspace_size returns for this call   */
} dgemm_plan_t;

/* BF16 GEMM: D = epi(alpha * A . op(B) + beta * C), FP32 accumulation.
 *   A        [M,K] BF16.          B [K,N] or [N,K] BF16 per b_layout.
 *   C        [M,N] of c_dtype (F32 or BF16); read only when beta != 0.
 *   D        [M,N] of d_dtype: F32 or BF16, or E4M3 with
 *            epi->out_quant == DGEMM_QUANT_E4M3_ROW_AMAX.
 *   ws       device workspace of ws_bytes bytes, its contents arbitrary on
 *            entry. Its first DGEMM_WS_STATUS_BYTES bytes hold the call's
 *            status word (when ws_bytes is at least that; read it with
 *            dgemm_query_device_status(ws, stream)). With the requantising
 *            epilogue it is required: at least
 *            256 + 256 + 4 * ceil(M / 64) * 64 + 2 * M * N bytes (status
 *            header, progress counters, row maxima, BF16 stash);
 *            dgemm_workspace_size(...) also counts room for splitting the last
 *            partial wave of tiles along K, which is made only when ws_bytes
 *            covers it. Otherwise optional: with at least
 *            dgemm_workspace_size(...) bytes, tiles may be split along K (the
 *            last partial wave, or every tile when the tiles do not fill the
 *            GPU) with FP32 partials in the workspace; with less, only splits
 *            that need no workspace are made (the K segments of a tile running
 *            as one thread-block cluster).
 * [W1] §1.1, §3.1, §6. */
dgemm_status_t dgemm_bf16(const void* A, const void* B, dgemm_b_layout_t b_layout,
                          const void* C, dgemm_dtype_t c_dtype,
                          void* D, dgemm_dtype_t d_dtype,
                          int64_t M, int64_t N, int64_t K, float alpha, float beta,
                          const dgemm_epilogue_t* epi, void* ws, size_t ws_bytes,
                          dgemm_stream_t stream);

/* FP8 E4M3 scaled GEMM:
 *   D = epi(alpha * diag(a_scale) . (Aq . op(Bq)) . diag(b_scale) + beta * C)
 *   Aq       [M,K] E4M3 codes (1 byte each).   Bq [K,N] or [N,K] E4M3 codes.
 *   k_group  0: one scale per row and per channel, constant along K, applied
 *            once to the FP32 accumulator (exact):
 *              a_scale [M] FP32, one per row of A (per token), stride 1;
 *              b_scale [N] FP32, one per output channel n, stride 1.
 *            g > 0, a multiple of 128: per-K-group scales ([W3] §3.2 asks to
 *            confirm per-GEMM or per-group granularity). K is cut into
 *            G = ceil(K / g) groups of g (the last may be shorter) and
 *              D = epi(alpha * sum_j diag(a_scale[j]) (Aq_j . op(Bq_j)) diag(b_scale[j]) + beta * C)
 *            with Aq_j, Bq_j the group's K slice. Tables are group-major:
 *              a_scale [G][M] (a_scale[j*M + m]), b_scale [G][N] (b_scale[j*N + n]).
 *            Each group's product is accumulated by the tensor core and folded
 *            into the FP32 sum, scaled, by the epilogue warps (2 FP32 operations
 *            per output element per group, so small groups cost throughput).
 *            Not combinable with DGEMM_QUANT_E4M3_ROW_AMAX; g not a multiple of
 *            128: DGEMM_ERR_NOT_SUPPORTED; g < 0: DGEMM_ERR_INVALID_VALUE.
 *   C, D, epi, ws as for dgemm_bf16.
 * [W3] §1.2, §3.2, §5.1. */
dgemm_status_t dgemm_fp8_scaled(const void* Aq, const void* Bq, dgemm_b_layout_t b_layout,
                                const float* a_scale, const float* b_scale, int k_group,
                                const void* C, dgemm_dtype_t c_dtype,
                                void* D, dgemm_dtype_t d_dtype,
                                int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                const dgemm_epilogue_t* epi, void* ws, size_t ws_bytes,
                                dgemm_stream_t stream);

/* FP8 E4M3 GEMM with block-scaled weights: dgemm_fp8_scaled with k_group = g
 * > 0, except that one weight scale covers a block of 128 output channels
 * by g K elements (the last block of each group may be narrower in N):
 *   a_scale  [G][M] FP32, one per (row of A, K group), as for dgemm_fp8_scaled;
 *   b_scale  [G][ceil(N / 128)] FP32: b_scale[j * ceil(N / 128) + n / 128]
 *            scales code Bq[k][n] (or Bq[n][k]) of group j = k / g.
 * Every 128 columns of a tile then share one scale per group, so the epilogue
 * folds each group with one fused multiply-add per output instead of two.
 * Errors: k_group <= 0 gives DGEMM_ERR_INVALID_VALUE; otherwise as for
 * dgemm_fp8_scaled. [W3] §3.2 (per-group scale granularity). */
dgemm_status_t dgemm_fp8_blockscaled(const void* Aq, const void* Bq, dgemm_b_layout_t b_layout,
                                     const float* a_scale, const float* b_scale, int k_group,
                                     const void* C, dgemm_dtype_t c_dtype,
                                     void* D, dgemm_dtype_t d_dtype,
                                     int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                     const dgemm_epilogue_t* epi, void* ws, size_t ws_bytes,
                                     dgemm_stream_t stream);

/* Workspace bytes a call with these arguments can use (0 when none). Query it
 * once and pass a buffer at least this large ([W3] §5.1). Uses the current
 * device's SM count when a device is present (else 152, a GB300); no kernel
 * runs. Returns 0 for invalid arguments. */
size_t dgemm_workspace_size(int is_fp8, int64_t M, int64_t N, int64_t K,
                            dgemm_b_layout_t b_layout, const dgemm_epilogue_t* epi);

/* The plan a call with these arguments would use on a GPU with num_sms SMs
 * (host-only, no GPU needed; CTA pairs assumed to fill half the SMs), or, with
 * num_sms <= 0, on the current device (its SM count and measured CTA-pair
 * occupancy). k_group as for dgemm_fp8_scaled (0 for BF16 and per-row scales;
 * the block-scaled entry plans like its k_group). Assumes a workspace of at
 * least dgemm_workspace_size bytes. Returns DGEMM_OK and fills *plan, or the
 * same argument error the GEMM call would return for these sizes. */
dgemm_status_t dgemm_plan(int is_fp8, int64_t M, int64_t N, int64_t K,
                          dgemm_b_layout_t b_layout, dgemm_dtype_t d_dtype,
                          const dgemm_epilogue_t* epi, int k_group, int num_sms, dgemm_plan_t* plan);

/* Static English description of a status code; never NULL. */
const char* dgemm_status_string(dgemm_status_t status);

/* Synchronises `stream`, then returns and clears a status word:
 *   ws != NULL: the status word at the start of that workspace, written by
 *            the calls that were given it (with at least DGEMM_WS_STATUS_BYTES
 *            bytes) since the last query of it;
 *   ws == NULL: the per-device word of the current device, written by the
 *            calls on this device that had no such workspace (and by the
 *            allocation-free entry point below).
 * Returns DGEMM_OK, DGEMM_ERR_DEVICE_TIMEOUT if one of those kernels gave up a
 * bounded wait, or DGEMM_ERR_CUDA if the stream itself reports an error.
 * Two calls with different workspaces report their timeouts separately.
 * [W3] §5.1 (the call returns a status; device errors are read afterwards). */
dgemm_status_t dgemm_query_device_status(const void* ws, dgemm_stream_t stream);

/* ---- Planner overrides (tuning sweeps and tests) ----------------------------
 *
 * By default the planner makes every choice below. These overrides replace
 * some of its choices for every later call in the process (tests use them to
 * reach each kernel variant and split path; tuning sweeps to compare them).
 * A field at its default (dgemm_overrides_init) keeps the planner's choice.
 * The DGEMM_* environment variables named beside the fields are read once, at
 * the first call, and only when DGEMM_ENV_OVERRIDES=1 is set too: a stray
 * variable alone changes nothing. dgemm_plan honours the overrides as well. */
typedef struct {
    int tile_n;          /* 0; or 64, 128, 256: single-CTA tiles of this width where
                            that variant exists (DGEMM_TILE_N)                     */
    int cta_pair;        /* -1; 0: no CTA pairs; 1: CTA pairs where a pair variant
                            exists (DGEMM_CTA_PAIR)                                 */
    int tail_split;      /* -1; 0: never split tiles along K; 1: split the last
                            partial wave's tiles whatever their length
                            (DGEMM_TAIL_SPLIT, "force" = 1)                         */
    int tail_halves;     /* -1; 0: never run tail tiles as N halves (DGEMM_TAIL_HALVES) */
    int cluster_split;   /* -1; 0: split-K partials always through the workspace
                            (DGEMM_CLUSTER_SPLIT)                                   */
    int seg_first;       /* -1; 0: split segments after the whole tiles
                            (DGEMM_SEG_FIRST)                                       */
    int raster_group;    /* 0; else tile rows per band of the raster (DGEMM_RASTER_GROUP) */
    int cooperative;     /* -1; 0: launch nothing cooperatively (for profilers that
                            cannot launch cooperative cluster grids: the
                            requantising form's row-band waits then rely on an
                            otherwise idle GPU); 1: launch every plan whose split
                            tiles exchange partials through the workspace
                            cooperatively (DGEMM_COOPERATIVE)                       */
    int kslices;         /* -1; 1: one 128-byte K slice per pipeline stage (the
                            planner takes two, fetched in 3-D copies, for CTA-pair
                            tiles and 128- or 64-wide single-CTA tiles whose K,
                            and N when B is stored K x N, are whole multiples of
                            128 bytes) (DGEMM_KSLICES)                              */
    int64_t wait_limit_ns;     /* 0: about one second; else the limit of every
                                  bounded device-side wait (DGEMM_WAIT_LIMIT_NS)    */
    int64_t stall_after_loads; /* -1; testing the bounded waits: every CTA's operand
                                  producer stops after this many stage loads, so the
                                  tensor-core issuer's wait for the next stage runs
                                  out (DGEMM_ERR_DEVICE_TIMEOUT); no environment
                                  variable                                          */
} dgemm_overrides_t;

/* Fills *o with the defaults (every choice left to the planner). */
void dgemm_overrides_init(dgemm_overrides_t* o);
/* Sets the overrides for later calls (NULL: the defaults). Out-of-range
 * fields give DGEMM_ERR_INVALID_VALUE and change nothing. Calls already
 * launched are not affected. */
dgemm_status_t dgemm_set_overrides(const dgemm_overrides_t* o);
/* The overrides in force. */
dgemm_status_t dgemm_get_overrides(dgemm_overrides_t* o);

/* ---- Allocation-free variant (no counterpart in the paper) ----------------
 *
 * Some callers cannot allocate device memory at the point where they run a
 * GEMM: code inside a custom memory pool or allocator callback, a real-time
 * path that must not block on cudaMalloc's device-wide synchronisation, or an
 * embedded runtime whose memory is carved out once at start-up. The per-row
 * E4M3 requantisation epilogue needs scratch memory (progress counters, the
 * row maxima and a BF16 copy of the pre-quantisation tile values), which
 * dgemm_fp8_scaled takes from a caller-provided workspace. This entry point
 * takes it instead from one statically sized device array inside the library,
 * so the caller passes only inputs and outputs and nothing is allocated.
 *
 *   - The array is DGEMM_NOALLOC_SCRATCH_BYTES (32 MiB) per device and is held
 *     by every GPU that loads the library until the process exits.
 *   - A call needs 512 + 4 * ceil(M / 64) * 64 + 2 * M * N bytes of it (the
 *     requantising workspace without the split area); larger problems return
 *     DGEMM_ERR_WORKSPACE_TOO_SMALL before anything is launched. M*N up to
 *     about 16.7 million elements fits (e.g. 2048 x 8192). The last partial
 *     wave of tiles is split along K only when the split area fits as well
 *     (dgemm_workspace_size(1, M, N, K, b_layout, epi) <= the array); otherwise
 *     it runs as whole tiles, with the same results.
 *   - Device-side errors of these calls go to the per-device status word:
 *     read them with dgemm_query_device_status(NULL, stream).
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     CUDA stream capture begins.
 *   - All calls share the one array, which keeps the last call's contents; the
 *     call clears the parts that must start at zero. Calls whose kernels
 *     overlap on the GPU (different streams, or different host threads) race
 *     on the array and give wrong results: serialise them.
 *   - Arguments and results are those of dgemm_fp8_scaled with k_group = 0,
 *     d_dtype E4M3 and epi->out_quant == DGEMM_QUANT_E4M3_ROW_AMAX (required,
 *     with epi->out_row_scale). */
#define DGEMM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

dgemm_status_t dgemm_fp8_rowquant_noalloc(const void* Aq, const void* Bq, dgemm_b_layout_t b_layout,
                                          const float* a_scale, const float* b_scale,
                                          const void* C, dgemm_dtype_t c_dtype, void* Dq,
                                          int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                          const dgemm_epilogue_t* epi, dgemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DGEMM_H */
