// Kernel parameter blocks and launch entry points of the CUDA path (internal to libskgemm).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "skgemm.h"

namespace sk {

enum OpKind : int {
    kOpGemm16 = 0, kOpFp8 = 1, kOpWgrad16 = 2, kOpFprop16 = 3, kOpDgrad16 = 4,
    kOpFp8Block = 5,   // fp8 with block scales: each K step's partial promoted by the epilogue
    // Wgrad of 64-channel, 64-filter groups on shifted rows (one x row serves every column tap):
    // W stride 1 (one phase of x columns) or 2 (even and odd columns).
    kOpWgradRow1 = 6, kOpWgradRow2 = 7,
    // Forward convolution (stride 1, 64 channels, 64 filters, at most 3 x 3 taps) on shifted rows:
    // a tile is two output rows of 64 positions, the x rows for all taps come in one box and the
    // filter stays in shared memory.
    kOpFpropRow = 8
};

__host__ __device__ constexpr bool is_wgrad_row(int op) {
    return op == kOpWgradRow1 || op == kOpWgradRow2;
}

// Forward convolution and data gradient fold conv groups into the output's columns (the output
// is [pixels][channels]); wgrad folds them into its rows.
__host__ __device__ constexpr bool folds_groups_into_columns(int op) {
    return op == kOpFprop16 || op == kOpDgrad16 || op == kOpFpropRow;
}

constexpr int kTileM = 128;
constexpr int kTileN = 128;

// Instruction descriptor: fp32 accumulator, dense, M x N, A/B formats and majorness.
//  kind::f16    : fmt 0 = f16, 1 = bf16.   kind::f8f6f4 : fmt 0 = e4m3, 1 = e5m2.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, bool a_mn_major,
                                                  bool b_mn_major, uint32_t M, uint32_t N) {
    return (1u << 4)                     // D format: f32
           | (a_fmt << 7) | (b_fmt << 10)  //
           | (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
           ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Output rows of one phase of a strided data gradient: traversal pixel m = (n, i, j) of an
// HoWo = Hp*Wp grid (width Wo = Wp) is dx pixel (n, dsh*i + ah, dsw*j + aw) of an Hd x Wd image.
// `on` = 0: the rows are the traversal pixels themselves.
// `vh` > 0: only grid positions i < vh, j < vw are output pixels (the shifted-row fprop pads rows
// to 64 positions and images to an even row count); map_row gives -1 for the others.
struct RowMap {
    int64_t HoWo;
    int32_t on, Wo, Hd, Wd, dsh, dsw, ah, aw;
    int32_t vh, vw;
};

__host__ __device__ __forceinline__ int64_t map_row(const RowMap& rm, int64_t m) {
    if (!rm.on) return m;
    const int64_t n = m / rm.HoWo;
    const int64_t rem = m - n * rm.HoWo;
    const int64_t i = rem / rm.Wo;
    const int64_t j = rem - i * rm.Wo;
    if (rm.vh > 0 && (i >= rm.vh || j >= rm.vw)) return -1;
    return (n * rm.Hd + rm.dsh * i + rm.ah) * rm.Wd + rm.dsw * j + rm.aw;
}

// Geometry the convolution producers need to turn an iteration into im2col coordinates. The im2col
// traversal runs over the pixels of one image grid: wgrad and fprop the output grid (Ho x Wo), dgrad
// the input grid (H x W, stride 1, padding R-1-ph / S-1-pw with the taps flipped) or, for a strided
// dgrad, the grid of one output phase.
struct ConvGeom {
    int64_t HoWo;          // pixels per image of the traversal grid
    int32_t Wo;            // width of the traversal grid
    int32_t sh, sw, ph, pw;   // traversal stride and padding
    int32_t R, S;          // taps of the traversal window
    // dgrad: traversal tap (r, s) reads filter tap (r0 + dsh*(R-1-r), s0 + dsw*(S-1-s)) of a
    // filter Sf taps wide (stride 1: r0 = s0 = 0, dsh = dsw = 1, Sf = S: the flipped filter)
    int32_t r0, s0, dsh, dsw, Sf;
    RowMap rows;           // output rows (dgrad phases of a strided convolution)
    int32_t Cg, Kg;        // wgrad: channels and filters per group; fprop / dgrad: channels per
                           // group of the im2col'd tensor (x: C/G, dy: K/G) and filter rows per group
    int32_t Cw;            // fprop / dgrad: channels per group of the filter (C/G)
    // Shifted-row wgrad (kOpWgradRow*): a K step is `rows_per_step` output rows of `wseg`
    // positions (rows_per_step * wseg = 64) of image n, rows counted per image over ho_pad (Ho
    // rounded up to rows_per_step). Column tap s = sw * q + phase reads the dy row shifted by q
    // positions (q <= qmax); phase p holds nq[p] taps.
    int32_t ho, ho_pad, rows_per_step, wseg, qmax;
    int32_t nq[2];
    // Shifted-row wgrad: CTAs the 64 filters are split over (1, or 2 for a CTA pair, each holding
    // 32 of them). A phase's D columns are fsplit halves, each nq blocks of 64/fsplit filters, one
    // block per shift q = nq - 1 - block.
    int32_t fsplit;
    // Shifted-row wgrad ring stage: up to stage_steps consecutive K steps of one image. Per column
    // phase (x_phase_bytes apart) the x rows of the CTA's tap rows for all of them: with
    // x_shared_box one box of stage_steps * rows_per_step + 1 rows (sh = 1: the lower tap row is
    // the next row, x_lbo = wseg * 128 bytes on), else one box per tap row (x_lbo = stage_steps *
    // 8 KB apart); then the dy rows of all of them at dy_off.
    int32_t stage_steps, x_lbo, x_phase_bytes, dy_off, x_shared_box;
    // Shifted-row fprop: the filter's taps arrive as one 3-D box (64 channels x 64 filters x R*S
    // taps, tap-major in shared memory) instead of one 2-D box per tap.
    int32_t filter_box;
    // Shifted-row kernel run as a data gradient: the filter's taps flipped (traversal tap t reads
    // filter tap R*S - 1 - t) and B MN-major (the output channels are the filter's contiguous ones).
    int32_t row_flip;
};

// Shifted-row wgrad ring: stage capacity (bytes) and stage count of each instance (one x column
// phase, or two). One CTA: deep rings of one-step stages (8 x 26 KB, 5 x 42 KB), for reductions
// short per CTA, where the ramp and the tail dominate; a CTA pair: several steps per stage
// (4 x 48 KB, 3 x 73 KB: fewer, larger copies and x rows shared by the steps), for long ones.
constexpr int wgrow_stage_bytes(int op, int cg) {
    return cg == 1 ? (op == kOpWgradRow1 ? 26 * 1024 : 42 * 1024)
                   : (op == kOpWgradRow1 ? 48 * 1024 : 73 * 1024);
}
constexpr int wgrow_stages(int op, int cg) {
    return cg == 1 ? (op == kOpWgradRow1 ? 8 : 5) : (op == kOpWgradRow1 ? 4 : 3);
}

struct KernelParams {
    CUtensorMap tmap_a;    // GEMM: A [M][K]; fp8: A8 [M][K]; wgrad: dy as [N*Ho*Wo][K];
                           // shifted-row wgrad: x [N][H][W][C], strided rows of 64 channels
    CUtensorMap tmap_b;    // GEMM: B [N][K]; fp8: B8 [N][K]; wgrad: im2col view of x;
                           // shifted-row wgrad: dy [N][Ho][Wo][K], rows of 64 filters (128-byte
                           // swizzle), or of 32 for a CTA pair (64-byte swizzle)
    CUtensorMap tmap_c;    // when c_tma: C [M][N] 16-bit, 64 x 32 boxes, 128-byte swizzle
    sk_plan_t plan;
    void* c;               // output
    int64_t ldc;           // output row stride (elements)
    const float* sa;       // fp8 row scales; null for the per-tensor scaling below
    const float* sb;       // fp8 column scales; null for the per-tensor scaling below
    float scale;           // fp8 with sa == sb == null: the product of the two tensor scales
    uint32_t* flags;       // per-publisher flags (linear/tree)
    uint32_t* control;     // [0] ticket counter; [1 + tile * CG + half] spread-fold arrival counters
    float* partials;       // linear/tree partial tiles, one slot per publisher
    float* scratch;        // workspace reduction scratch, one tile per shared-tile candidate
    ConvGeom conv;
    uint64_t flag_timeout_ns;
    uint64_t mbar_timeout_ns;
    uint32_t idesc;
    int32_t c_dtype;
    int32_t c_tma;         // 1: a CTA's last complete tile is written with TMA stores (tmap_c)
    // linear / tree: 1 = every contributor of a shared tile publishes its partial, counts it in the
    // tile's arrival counter (control block word 1 + tile * CG + half) and adds a share of the tile
    // once the counter has reached the tile's contributors (all publishing CTAs are resident at
    // once); 0 = the owner (and each tree receiver) adds its senders' partials. The same sums
    // either way.
    int32_t spread;
    // 1: logical CTA ids come from a ticket counter in the control block, taken in start order
    // (linear/tree with more CTAs than can be resident at once, where a CTA may wait on a later
    // one); 0: the block (cluster) index, and the wait for the zeroing kernel's writes moves from
    // the prologue to the first access of the zeroed words.
    int32_t ticket;
    // Launches of one call that do not read each other's results (the phases of a strided data
    // gradient, each writing its own pixels, with no shared tile): bit 0 = this kernel was
    // launched to overlap the previous one and waits for nothing of it; bit 1 = it lets the next
    // one start as soon as all its CTAs have started.
    int32_t pdl_chain;
    // kOpFp8Block: sa [M][nka] (A blocks of gka along K) and sb [ceil(N/gnb)][nkb] (B blocks of
    // gnb x gkb), either may be null; gka, gkb and gnb multiples of 128.
    const float* bsa;
    const float* bsb;
    int64_t nka, nkb;
    int32_t gka, gnb, gkb;
};

struct Stage2Params {
    sk_plan_t plan;
    int32_t op_kind;       // OpKind: where the group of a tile goes in the output
    RowMap rows;           // output rows of the tile rows (identity unless a dgrad phase)
    void* c;
    int64_t ldc;
    const float* sa;
    const float* sb;
    float scale;           // fp8 per-tensor scaling (sa == sb == null)
    int32_t tensor_scaled; // 1: multiply by `scale`
    const float* scratch;
    int32_t c_dtype;
    ConvGeom conv;         // shifted-row wgrad: where a tile row and column go in dW
    // 1: launched to overlap the main kernel's tail (programmatic dependent launch); every thread
    // waits for the main kernel's completion before its first access
    int32_t after_main;
};

// Ranges a zeroing kernel clears ahead of a main kernel: up to three 16-byte aligned 1-D ranges
// (sizes multiples of 16 bytes) and one 2-D range of `rows` rows of `row_bytes` (a multiple of 4)
// at `pitch` bytes apart.
struct ZeroParams {
    void* ptr[3];
    int64_t bytes[3];
    int32_t nranges;
    void* out;
    int64_t pitch, row_bytes, rows;
};

// cg: 1 = one CTA per tile; 2 = a cluster of two CTAs per 256 x tn tile (GEMMs: tn 128 with 4
// stages, tn 256 with 3; shifted-row wgrad: tn 192). st: stages of the operand ring.
// Dynamic shared memory of one CTA of the main kernel.
size_t main_smem_bytes(int op, int cg, int tn, int st);
// How many CTAs of the main kernel fit on one SM (0 if the device query fails).
int main_ctas_per_sm(int op, int cg, int tn, int st);
// Launch the main kernel: p.plan.grid logical CTAs, each one CTA (cg 1) or one cluster of two
// (cg 2). `after_zero`: the launch directly follows launch_zero on `stream` and may overlap its
// tail. Returns a cudaError_t value.
int launch_main(const KernelParams& p, int op, int cg, int tn, int st, bool after_zero,
                cudaStream_t stream);
// Launch the zeroing kernel (nothing when every range is empty). Returns a cudaError_t value.
int launch_zero(const ZeroParams& z, cudaStream_t stream);
// Launch the Stage-2 reduce over the shared tiles of a workspace plan.
int launch_stage2(const Stage2Params& p, cudaStream_t stream);
// Read and clear the device error record: returns the code (0 = none) and fills info[3].
int take_device_error(cudaStream_t stream, long long info[3]);
// Launch the failure-detection probe: a bounded flag wait that runs out after limit_ns and records
// the hand-off timeout. Returns a cudaError_t value.
int launch_flag_timeout_probe(uint64_t limit_ns, cudaStream_t stream);

}  // namespace sk
