/*
 * skgemm -- stream-K GEMM, implicit-GEMM convolution backward-weight and fp8 row/col-scaled
 * GEMM on one NVIDIA GB300 (sm_103a). C ABI.
 *
 * Sources of the operations (web pages, cited by title and section):
 *  [P1] "feat(ck-tile): stream-K GEMM TE to dispatcher bridge" (ROCm composable_kernel commit
 *       58c1bcbe2e), Design note and Changes: a single-problem GEMM call with the same C ABI as the
 *       regular GEMM, returning 0 on success, -1 on a launch error, -2 for unsupported arguments;
 *       the launch owns the reduction workspace.
 *  [P2] rocm-libraries PR #13151 "feat(rocke): stream-K for implicit-GEMM conv wgrad", PR body
 *       (Technical Details: Partitioner, Wgrad kernel, Constraints) and commits: the stream-K
 *       partition (data-parallel tiles + a pool of stream-K CTAs with contiguous balanced
 *       iteration ranges), launch modes dp_sk / persistent, reductions linear / tree / atomic /
 *       workspace, CTA pool -1 = arch default, conv groups folded into GEMM-M.
 *  [P3] rocm-libraries PR #9979 (RowColQuant GEMM bridge), Scope: fp8 rcr GEMM with a per-row
 *       scale of A and a per-column scale of B applied in the epilogue to an fp32 accumulator.
 *
 * Conventions for every compute call:
 *  - Pointers A, B, x, dy, C, dw, sa, sb, ws are DEVICE pointers owned by the caller. The library
 *    neither frees nor retains them. `stream` is a cudaStream_t passed as void* (NULL = the
 *    legacy default stream). Calls are asynchronous: 0 means "enqueued".
 *  - Return value: 0 ok; -1 a CUDA call or kernel launch failed (message in sk_last_error());
 *    -2 the arguments are unsupported (nothing was enqueued, no memory was touched).
 *  - `streamk`: SK_OFF (one CTA per output tile over the whole reduction), SK_DP_SK (grid = DP
 *    tiles + stream-K CTAs), SK_PERSISTENT (grid = pool; each CTA runs its DP tiles, then its
 *    stream-K range), or SK_SPLITK (comparator: every tile cut into s = max(1, pool/tiles) equal
 *    K slices, combined by the same reductions).
 *    SK_AUTO picks between SK_DP_SK and SK_SPLITK ([P2] commits "ConvGroupedRequest.streamk now
 *    defaults to auto" and the review fix "auto builds the launch partition, requires sk_ctas > 0";
 *    this selection was later reverted from the pages' dispatcher): stream-K when the tiles do not
 *    fill the pool (T < P) and the reduction is long (T * I >= 1024), and only if the plan the
 *    launch would use has stream-K CTAs; split-K otherwise (plain data-parallel when T >= P),
 *    except that the shifted-row forward convolution (whose CTAs keep the filter resident) with
 *    more tiles than CTAs runs SK_PERSISTENT. The resolved mode is what sk_plan reports.
 *    SK_HYBRID is SK_DP_SK with one full wave more in the stream-K region whenever the pool does
 *    not divide the tiles and the tiles fill at least one wave: P + T mod P stream-K tiles, so
 *    that every stream-K CTA runs between one and two tiles' worth of iterations (a variant of
 *    [P2]'s remainder-only rule; otherwise the same plan as SK_DP_SK).
 *  - `reduction`: SK_LINEAR and SK_TREE are deterministic (bit-identical across launches with the
 *    same plan); SK_ATOMIC needs an fp32 output; SK_WORKSPACE adds into fp32 scratch and runs a
 *    second (Stage-2) kernel that writes the output. SK_REDUCTION_AUTO resolves to SK_WORKSPACE
 *    ([P2] "streamk_reduction defaults to auto, which resolves to the workspace reduction").
 *  - `ctas`: the CTA pool; -1 = default (one CTA per SM for linear/tree; SMs x min(4, CTAs that
 *    fit on one SM) for atomic/workspace). 0 and values below -1 are rejected with -2.
 *  - `ws`, `ws_bytes`: workspace of at least sk_workspace_bytes() bytes, 256-byte aligned. With
 *    ws == NULL the library allocates it on `stream` (cudaMallocAsync) and frees it after the
 *    launch (cudaFreeAsync). The workspace holds the per-CTA flag table, a control block, and
 *    the partial tiles (linear/tree) or the fp32 scratch (workspace). The library zeroes the flags,
 *    the control block and the scratch (and, for SK_ATOMIC, the output) on `stream` before every
 *    launch; partial tiles are never zeroed.
 *  - Concurrent calls that share one workspace must be ordered on one stream.
 *  - Tiles are 128 x 128 (M x N), or 256 x 128 / 256 x 256 for a CTA pair (sk_set_tile); the
 *    reduction step is 64 elements for 16-bit inputs and 128 for fp8.
 */
#ifndef SKGEMM_H
#define SKGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { SK_F16 = 0, SK_BF16 = 1, SK_F32 = 2, SK_E4M3 = 3 };                  /* element types */
enum { SK_OFF = 0, SK_DP_SK = 1, SK_PERSISTENT = 2, SK_SPLITK = 3, SK_AUTO = 4,
       SK_HYBRID = 5 };                                                      /* streamk */
enum { SK_LINEAR = 0, SK_TREE = 1, SK_ATOMIC = 2, SK_WORKSPACE = 3, SK_REDUCTION_AUTO = 4 };
                                                                             /* reduction    */
enum { SK_OP_GEMM = 0, SK_OP_FP8_ROWCOL = 1, SK_OP_WGRAD = 2, SK_OP_FPROP = 3, SK_OP_DGRAD = 4,
       SK_OP_FP8_BLOCK = 5 };
                                                                             /* operation    */
enum { SK_SEG_FULL = 0, SK_SEG_OWNER = 1, SK_SEG_PEER = 2 };                /* segment kind */

#define SK_OK 0
#define SK_ERR_LAUNCH (-1)
#define SK_ERR_UNSUPPORTED (-2)

/* Problem description for the host-only planning calls. Fields not used by `op` are ignored. */
typedef struct sk_problem {
    int32_t op;        /* SK_OP_*                                                     */
    int32_t ab_dtype;  /* input type: SK_F16 / SK_BF16 (GEMM, wgrad), SK_E4M3 (fp8)   */
    int32_t c_dtype;   /* output type                                                 */
    int32_t groups;    /* wgrad conv groups (>= 1)                                    */
    int64_t M, N, K;   /* GEMM / fp8 GEMM: C[M][N] = A[M][K] * B[N][K]^T              */
    int64_t n, h, w, c, k, r, s;          /* convolutions: x[n][h][w][c], dy / y [n][ho][wo][k],
                                             filter [k][r][s][c/groups]                           */
    int32_t stride_h, stride_w, pad_h, pad_w;
} sk_problem;

/* The resolved partition ("plan"), computed once on the host and passed to the kernel by value.
 * [P2] commit "Add StreamKIterPartition": the plan is returned by value so that no derived
 * quantity can be recomputed with different rounding. All fields are int64 for a fixed layout. */
typedef struct sk_plan_t {
    int64_t op, mode, reduction;
    int64_t tm, tn, tk;              /* tile M, tile N, reduction step                        */
    int64_t gemm_m, gemm_n, kred;    /* GEMM view per group: rows, columns, reduction length  */
    int64_t groups;
    int64_t tiles_m, tiles_n;        /* per group                                              */
    int64_t tiles;                   /* T = groups * tiles_m * tiles_n                         */
    int64_t iters_per_tile;          /* I = ceil(kred / tk)                                    */
    int64_t pool;                    /* P (resolved)                                           */
    int64_t sk_tiles, dp_tiles;      /* SK tiles are ids [0, sk_tiles), DP tiles the rest      */
    int64_t sk_ctas;                 /* CTAs with a stream-K range (0 = all data-parallel)     */
    int64_t sk_iters;                /* sk_tiles * I                                            */
    int64_t iters_per_sk_cta;        /* >= 1, also when sk_ctas == 0                           */
    int64_t extra_iters;             /* the first extra_iters SK CTAs take one more iteration  */
    int64_t splits;                  /* SK_SPLITK only: K slices per tile                      */
    int64_t grid;                    /* CTAs launched                                           */
    int64_t publishers;              /* CTAs owning a flag (it counts the partials they hand on) */
    int64_t max_contributors;        /* most CTAs sharing one tile                              */
    int64_t tree_rounds;             /* ceil(log2(max_contributors))                            */
    int64_t shared_tiles;            /* tiles with more than one contributor                   */
    int64_t flag_bytes;              /* round_up(4 * publishers * tm / 128, 256)                */
    int64_t control_offset;          /* = flag_bytes; 256-byte control block: ticket and       */
                                     /* spread-fold arrival counters                          */
    int64_t partial_offset, partial_bytes;   /* linear/tree: partial_slots * tm * tn * 4       */
    int64_t scratch_offset, scratch_bytes;   /* workspace: (SK tiles) * tm * tn * 4            */
    int64_t ws_bytes;                /* total workspace bytes                                   */
    int64_t partial_slots;           /* one per contributor of a shared tile: slot first+t+j for
                                        contributor j of stream-K tile t (sk_ctas + sk_tiles in
                                        all), t*splits+j for split-K                            */
} sk_plan_t;

/* One piece of a CTA's work: iterations [k_begin, k_end) of tile `tile`. */
typedef struct sk_segment_t {
    int64_t tile;
    int64_t k_begin, k_end;
    int64_t kind;          /* SK_SEG_FULL: sole writer; SK_SEG_OWNER: first of several; SK_SEG_PEER */
    int64_t index;         /* position among the tile's contributors (0 = owner)                    */
    int64_t n_contrib;     /* contributors of the tile (1 for SK_SEG_FULL)                          */
    int64_t first_cta;     /* logical id of the tile's owner (-1 for SK_SEG_FULL)                   */
} sk_segment_t;

/*
 * C[M][N] = A[M][K] * B[N][K]^T ("rcr": A row-major, B column-major K x N, C row-major) with
 * fp32 accumulation. [P1] Summary (fp16/rcr stream-K GEMM) and [P2] Technical Details.
 *   ab_dtype: SK_F16 or SK_BF16. c_dtype: the same 16-bit type, or SK_F32.
 *   lda, ldb: row strides in elements of A and B (>= K; lda*2 and ldb*2 multiples of 16 bytes;
 *   K a multiple of 8). ldc: row stride of C in elements (>= N, 16-byte aligned rows).
 *   SK_ATOMIC requires c_dtype == SK_F32.
 */
int sk_gemm_rcr(int ab_dtype, int c_dtype, int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                int streamk, int reduction, int ctas, void* ws, size_t ws_bytes, void* stream);

/*
 * C[m][n] = bf16( (sum_k e4m3(A8[m][k]) * e4m3(B8[n][k])) * sa[m] * sb[n] ). [P3] Scope: fp8
 * rcr, per-row A scale and per-column B scale (one scale each, no quant groups), fp32
 * accumulator narrowed only in the epilogue. A8: [M][K] row-major OCP E4M3 bytes (K a multiple
 * of 16); B8: [N][K]; sa: M floats; sb: N floats; C_bf16: [M][ldc]. SK_ATOMIC is rejected (the
 * output is 16-bit).
 */
int sk_gemm_rowcol_fp8(int64_t M, int64_t N, int64_t K, const void* A8, const void* B8,
                       const float* sa, const float* sb, void* C_bf16, int64_t ldc,
                       int streamk, int reduction, int ctas, void* ws, size_t ws_bytes,
                       void* stream);

/*
 * C[m][n] = bf16( (sum_k e4m3(A8[m][k]) * e4m3(B8[n][k])) * scale_a * scale_b ). PR #10439 (the
 * five block-scale quant GEMM bridges), Summary, "tensor_quant": one scalar scale for the whole A
 * matrix and one for the whole B matrix, applied in the epilogue. Same operands, layouts and
 * limits as sk_gemm_rowcol_fp8; the scales are passed by value.
 */
int sk_gemm_tensorquant_fp8(int64_t M, int64_t N, int64_t K, const void* A8, const void* B8,
                            float scale_a, float scale_b, void* C_bf16, int64_t ldc, int streamk,
                            int reduction, int ctas, void* ws, size_t ws_bytes, void* stream);

/*
 * Block-scaled fp8 GEMM. PR #10439 (the five block-scale quant GEMM bridges), Summary: "aquant"
 * (A scaled in blocks along K), "bquant" (B scaled in 2-D blocks along N and K) and "abquant"
 * (both). With ka = k / a_group_k and kb = k / b_group_k (integer division),
 *   C[m][n] = bf16( sum_k e4m3(A8[m][k]) * e4m3(B8[n][k]) * sa[m][ka] * sb[n / b_group_n][kb] ),
 * summed in fp32: the tensor cores form the exact-product partial of each 128-wide K step, and
 * the epilogue scales it by that step's block scales and adds it to the running fp32 sum.
 *   sa: [M][ceil(K / a_group_k)] fp32, row-major, or NULL (aquant off: scale 1);
 *   sb: [ceil(N / b_group_n)][ceil(K / b_group_k)] fp32, row-major, or NULL (bquant off).
 *   a_group_k, b_group_k: multiples of 128 (one K step never straddles two blocks);
 *   b_group_n: a multiple of 128 (one 128-column tile never straddles two blocks). Group sizes
 *   of a NULL scale are ignored. Operands, layouts and limits otherwise as sk_gemm_rowcol_fp8
 *   (SK_ATOMIC rejected). Tile: 128 x 128; sk_set_tile(SK_TILE_256_PAIR) selects a 256 x 128
 *   CTA-pair tile instead (SK_TILE_256x256_PAIR is rejected).
 */
int sk_gemm_blockscale_fp8(int64_t M, int64_t N, int64_t K, const void* A8, const void* B8,
                           const float* sa, int64_t a_group_k, const float* sb, int64_t b_group_n,
                           int64_t b_group_k, void* C_bf16, int64_t ldc, int streamk,
                           int reduction, int ctas, void* ws, size_t ws_bytes, void* stream);

/*
 * Backward-weight 2-D convolution as an implicit GEMM. [P2] PR body "Wgrad kernel" and commit
 * "Port CK Tile's stream-K to the backward-weight convolution": the output is filter-sized, the
 * reduction runs over N*Ho*Wo, and conv groups fold into GEMM-M per group.
 *   dw[g*Kg+k][r][s][c] = sum_{n,ho,wo} dy[n][ho][wo][g*Kg+k] * x[n][ho*sh-ph+r][wo*sw-pw+s][g*Cg+c]
 *   x: [N][H][W][C] (NHWC), dy: [N][Ho][Wo][K], dw: [K][R][S][C/groups] dense,
 *   Ho = (H + 2*pad_h - R)/stride_h + 1, Wo likewise; x outside the image reads as zero.
 *   in_dtype: SK_F16 or SK_BF16; dw_dtype: SK_F32 or in_dtype.
 *   Supported: (C/groups) a multiple of 64, K a multiple of 8, dilation 1, R, S <= 16, padding
 *   < filter size.
 */
int sk_conv2d_wgrad_nhwc(int in_dtype, int dw_dtype, int64_t N, int64_t H, int64_t W, int64_t C,
                         int64_t K, int64_t R, int64_t S, int stride_h, int stride_w, int pad_h,
                         int pad_w, int groups, const void* x, const void* dy, void* dw,
                         int streamk, int reduction, int ctas, void* ws, size_t ws_bytes,
                         void* stream);

/*
 * Forward convolution as an implicit GEMM on the same stream-K machinery. [P2] lists the forward
 * convolution as future work of the wgrad port; this call is that extension (no page gives its
 * kernel).
 *   y[n][ho][wo][g*Kg+k] = sum_{r,s,c} x[n][ho*sh-ph+r][wo*sw-pw+s][g*Cg+c] * w[g*Kg+k][r][s][c]
 *   x: [N][H][W][C] (NHWC), w: [K][R][S][C/groups] (KRSC), y: [N][Ho][Wo][K] (NHWC),
 *   Ho = (H + 2*pad_h - R)/stride_h + 1, Wo likewise; x outside the image reads as zero.
 *   GEMM view per group: M = N*Ho*Wo output pixels, N = K/groups filters, reduction R*S*C/groups.
 *   in_dtype: SK_F16 or SK_BF16; y_dtype: in_dtype or SK_F32 (SK_ATOMIC needs SK_F32).
 *   Supported: (C/groups) a multiple of 64, K a multiple of 8, dilation 1, R, S <= 16, padding
 *   < filter size. The 128 x 128 tile (sk_set_tile's pair tiles return -2). Under SK_TILE_AUTO a
 *   layer of one group of 64 channels into 64 filters, stride 1, R, S <= 3 and Wo + S - 1 <= 64
 *   takes the shifted-row view instead (see sk_set_tile): the same sums, M = output positions in
 *   pairs of output rows of 64, N = 64, one reduction step per tap.
 */
int sk_conv2d_fprop_nhwc(int in_dtype, int y_dtype, int64_t N, int64_t H, int64_t W, int64_t C,
                         int64_t K, int64_t R, int64_t S, int stride_h, int stride_w, int pad_h,
                         int pad_w, int groups, const void* x, const void* w, void* y,
                         int streamk, int reduction, int ctas, void* ws, size_t ws_bytes,
                         void* stream);

/*
 * Data gradient of the convolution (the backward pass to the input) as an implicit GEMM, with the
 * same conventions as sk_conv2d_fprop_nhwc. Same source as above: future work of the wgrad port.
 *   dx[n][h][w][g*Cg+c] = sum_{r,s,k} dy[n][ho][wo][g*Kg+k] * w[g*Kg+k][r][s][c]
 *                         over the (ho, wo) with ho*sh-ph+r = h, wo*sw-pw+s = w
 *   dy: [N][Ho][Wo][K], w: [K][R][S][C/groups], dx: [N][H][W][C] (written whole).
 *   GEMM view per group: M = N*H*W input pixels, N = C/groups channels, reduction R*S*K/groups,
 *   computed as a stride-1 convolution of dy with the flipped filter. With a stride above 1 it
 *   runs one such convolution per output phase (the dx pixels h = sh*i + a, w = sw*j + b): only
 *   the taps r = (a + ph) mod sh + sh*t reach them (likewise s), over an H/sh x W/sw grid;
 *   phases that no tap reaches are zero. sk_workspace_bytes gives the phases' workspaces side
 *   by side (each rounded up to 256 bytes): with that much (or ws == NULL, the library then
 *   allocating it) the phases may run at the same time; a workspace that holds only the largest
 *   phase also works, and the phases whose plans share tiles then run one after another. sk_plan
 *   has no single plan for a strided call and returns -2.
 *   Supported: strides 1..8, (K/groups) a multiple of 64, C/groups a multiple of 8, dilation 1,
 *   R, S <= 16, padding < filter size. The 128 x 128 tile; under SK_TILE_AUTO a stride-1 layer of
 *   one group of 64 filters into 64 channels with R, S <= 3 and W + S - 1 <= 64 takes the
 *   shifted-row view (see sk_set_tile). A strided call's phases always take the 128 x 128 tile.
 */
int sk_conv2d_dgrad_nhwc(int in_dtype, int dx_dtype, int64_t N, int64_t H, int64_t W, int64_t C,
                         int64_t K, int64_t R, int64_t S, int stride_h, int stride_w, int pad_h,
                         int pad_w, int groups, const void* dy, const void* w, void* dx,
                         int streamk, int reduction, int ctas, void* ws, size_t ws_bytes,
                         void* stream);

/*
 * sk_gemm_rcr without any device allocation. (The pages have no counterpart; this call exists
 * for users of this library.)
 *
 * Some callers cannot allocate device memory at call time: code whose GPU memory is owned by
 * another allocator (a framework's caching allocator or an inference server that reserved the
 * device and hands out only pre-sized buffers), and latency-bound callers that cannot absorb
 * the device-wide synchronisation cudaMalloc/cudaFree can cause. This variant takes the same
 * arguments as sk_gemm_rcr except the workspace: it uses a fixed scratch area compiled into the
 * library as a static device array of SK_STATIC_WS_BYTES bytes (16 MiB), which every GPU that
 * loads the library keeps until the process exits. It calls no cudaMalloc/cudaFree and no
 * allocating library routine.
 *  - The first call on a device looks up that device's copy of the array (cudaGetSymbolAddress,
 *    which can load the library's GPU module); make that first call before any stream capture.
 *    The address is kept per device and CUDA context: the first call after the device's context
 *    was created again (e.g. after cudaDeviceReset) looks it up again.
 *  - A problem whose plan needs more than SK_STATIC_WS_BYTES of workspace is rejected with -2
 *    and a message giving both sizes (linear/tree need one fp32 tile per stream-K CTA, workspace
 *    one per shared tile: 64 KiB with the 128 x 128 tile, 256 KiB with the 256 x 256 pair tile,
 *    which the automatic tile choice takes for GEMMs with M > 128 and at least 64 tiles of
 *    256 x 256; atomic and off need only the flag/control header).
 *  - All calls share the one array and it keeps the previous call's contents: each call clears
 *    the flags, the control block and the scratch it reads before use, on `stream`. Calls that
 *    can overlap on the GPU (different streams, or several host threads) race on the array and
 *    give wrong results; order them on one stream.
 */
#define SK_STATIC_WS_BYTES (16u << 20)
int sk_gemm_rcr_static_ws(int ab_dtype, int c_dtype, int64_t M, int64_t N, int64_t K,
                          const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                          int64_t ldc, int streamk, int reduction, int ctas, void* stream);

/* Workspace bytes the call described by `p` needs (device query for ctas == -1). 0 / -2. */
int sk_workspace_bytes(const sk_problem* p, int streamk, int reduction, int ctas, size_t* out);

/*
 * Host-only: resolve the partition for problem `p`. `num_sms` > 0 gives the SM count used for
 * ctas == -1 (num_sms <= 0 queries the current device). Does not touch the GPU otherwise.
 * Returns 0, or -2 (message in sk_last_error()).
 */
int sk_plan(const sk_problem* p, int streamk, int reduction, int ctas, int num_sms,
            sk_plan_t* out);

/* Host-only: the work of logical CTA `cta` under `plan`, in execution order (the same walk the
 * kernel makes). Writes up to max_out segments, the total count to *n_out. 0 / -2. */
int sk_plan_cta_work(const sk_plan_t* plan, int64_t cta, sk_segment_t* out, int max_out,
                     int* n_out);

/* Host-only: default CTA pool for `reduction` given the SM count and the CTAs of the kernel that
 * fit on one SM. [P2] commit "Resolve streamk_ctas=-1 from the reduction". 0 / -2. */
int sk_default_pool(int reduction, int num_sms, int ctas_per_sm, int* out);

/* Synchronise `stream`, then report whether a bounded wait in a kernel gave up since the last
 * call: 0 = no, -1 = yes (details in sk_last_error()); clears the record. */
int sk_device_status(void* stream);

/*
 * Failure-detection self-test (no counterpart on the pages). Enqueues on `stream` one thread that
 * waits, with the linear/tree receivers' own bounded routine, on a device flag that nothing ever
 * sets; after `timeout_ms` (1..1000) it gives up and records the hand-off timeout exactly as a lost
 * hand-off would (cta -1, tile -1, sender -1). The next sk_device_status on the stream then returns
 * -1 with that message and clears it. Nothing faults or hangs, and the context stays usable.
 * Returns 0 (enqueued), -1 (launch error) or -2 (bad timeout, or no sm_103a device).
 */
int sk_probe_flag_timeout(int timeout_ms, void* stream);

/* Reason for the last -1 / -2 returned on this thread (never NULL). */
const char* sk_last_error(void);

/* Library version: major*10000 + minor*100 + patch. */
int sk_version(void);

/*
 * Tile shape for the later calls of the calling thread, planning calls included. (No counterpart on
 * the pages, whose tiles are one workgroup's; this is a GB300 kernel choice.)
 *  SK_TILE_AUTO (the default): SK_TILE_256x256_PAIR for the GEMM and fp8 GEMM when M > 128 and
 *    the output has at least 64 tiles of 256 x 256; SK_TILE_128 otherwise. Few large tiles over a
 *    long reduction would be shared by many CTAs each; the 128 x 128 tile keeps those fixups
 *    smaller. Wgrad with 64-channel, 64-filter groups, at most 3 column taps and a column stride
 *    of 1 or 2 (and output rows of at most 64 positions with the taps' shifts) takes the
 *    shifted-row view: M = (tap row, channel), N = (column tap, filter), reduction over the
 *    output rows padded to 64 positions per K step; a 128 x 192 tile on one CTA, or, for three or
 *    four tap rows over a long reduction (about 128 K steps per SM or more), a 256 x 192 tile on a
 *    CTA pair. Other wgrad shapes use the 128 x 128 tile of the pages' view. The forward
 *    convolution and the stride-1 data gradient of one group of 64 channels into 64 with at most
 *    3 x 3 taps and output rows of at most 64 positions with the column taps take the shifted-row
 *    convolution view: a 128 x 64 tile of two output rows, one reduction step per tap, computed
 *    from one box of R + 1 input rows read at each tap's row shift, the filter kept in shared
 *    memory for all of a CTA's tiles (with SK_AUTO and more tiles than CTAs, SK_PERSISTENT with
 *    every tile data-parallel).
 *  SK_TILE_128: one CTA computes each 128 x 128 output tile.
 *  SK_TILE_256_PAIR: a cluster of two CTAs on neighbouring SMs computes each 256 x 128 tile with the
 *    two-SM tensor-core instruction; each CTA stages its 128 rows of A and 64 of the 128 rows of B,
 *    which cuts the operand bytes each SM takes in per MMA by a quarter.
 *  SK_TILE_256x256_PAIR: the same with 256 x 256 tiles; each CTA stages 128 rows of A and 128 of B,
 *    half the bytes per MMA of the 128 x 128 tile.
 *  For the pair tiles the stream-K partition is the same algorithm over the pair tiles, and its CTA
 *  pool `ctas` counts pairs (the default pool is resolved over SMs / 2). SK_TILE_256_PAIR also
 *  selects the shifted-row wgrad's 256 x 192 pair tile for the shapes it takes (whatever their
 *  size); the other wgrad shapes, fprop and dgrad return -2 under the pair tiles.
 * Returns the previous setting, or -2 for an unknown value.
 */
enum { SK_TILE_AUTO = 0, SK_TILE_128 = 1, SK_TILE_256_PAIR = 2, SK_TILE_256x256_PAIR = 3 };
int sk_set_tile(int tile);

/*
 * Instrumentation (no counterpart on the pages; used by the benchmark to time the main kernel
 * alone). sk_timing_enable(1) makes the calling thread's later compute calls record a pair of CUDA
 * events on their stream around the main stream-K kernel, and count every kernel the library
 * launches; sk_timing_enable(0) stops recording. Both clear earlier records.
 * sk_timing_read waits for the recorded events, returns the summed main-kernel time in ms, the
 * number of main-kernel launches and of all library kernel launches, and clears the records.
 */
int sk_timing_enable(int on);
int sk_timing_read(double* main_ms, int64_t* main_launches, int64_t* all_launches);

#ifdef __cplusplus
}
#endif

#endif /* SKGEMM_H */
