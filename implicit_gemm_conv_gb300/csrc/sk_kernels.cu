// Stream-K mainloop, fixups and Stage-2 reduce for sm_103a.
//
// One kernel serves the three operations (rcr GEMM, implicit-GEMM wgrad, fp8 row/col GEMM). The
// CTA walks the work the plan gives its logical id (sk_plan.h): data-parallel tiles and/or one
// contiguous range of MAC iterations that may straddle tiles ("one bounded loop", rocm-libraries
// PR #13151, commit "Port CK Tile's stream-K to the backward-weight convolution").
//
// Warp roles (192 threads):
//   warp 0     TMA producer: stages A and B tiles into a ring of shared-memory stages.
//   warp 1     MMA issuer: one thread issues tcgen05.mma into a double-buffered TMEM accumulator
//              and commits it at every segment (tile) boundary; the warp owns the TMEM allocation.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, then per segment one of
//                - complete tile: scale (fp8), convert, store;
//                - linear / tree: receive the partials of later CTAs (acquire a per-CTA flag,
//                  add in a fixed order), then either store the tile or publish this CTA's
//                  partial and release its flag;
//                - atomic: red.add.f32 into the fp32 output;
//                - workspace: red.add.f32 into fp32 scratch (Stage-2 writes the output).
//   (PR #13151, PR body "Wgrad kernel": linear and tree are deterministic hand-offs through
//   per-CTA flags, atomic is fp32-only, workspace is fp32 scratch plus a Stage-2 reduce.)
//
// Logical CTA ids come from a ticket counter, so a CTA only ever waits on CTAs with larger ids,
// which started after it; every wait is bounded and records an error instead of hanging.
//
// CG = 2 runs each logical CTA as a cluster of two CTAs on neighbouring SMs (a "pair") that
// computes a 256 x TN tile with the two-SM tensor-core instruction (tcgen05 cta_group::2): each CTA
// stages its 128 rows of A and TN/2 of the TN rows of B, so one SM takes in fewer operand bytes
// per MMA cycle than with a 128 x 128 tile (24 KB per 256 cycles for TN = 128, 32 KB per 512
// cycles for TN = 256, against 32 KB per 256). The even CTA issues the MMAs and its commits arrive
// on the barriers of both CTAs; both CTAs' producers count their bytes on the even CTA's stage
// barrier. Each CTA's epilogue owns its 128 accumulator rows, and for the fixups each half of a
// pair acts as a CTA of its own: partial slot and flag (pair * 2 + rank), scratch half
// (tile * 2 + rank).
#include <stddef.h>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sk_kernels.h"
#include "sk_plan.h"
#include "sk_ptx.cuh"

namespace sk {

__device__ unsigned long long g_sk_error[4];   // code, cta, tile, detail (first error wins)

enum : unsigned long long {
    kErrFlagWait = 1,   // a linear/tree receive gave up waiting for a flag
    kErrPipeline = 2,   // an mbarrier wait inside the CTA gave up
    kErrBounds = 3,     // a self-check found an index outside its buffer (access skipped)
};

__device__ __noinline__ void record_error(unsigned long long code, long long cta, long long tile,
                                          long long detail) {
    if (atomicCAS(&g_sk_error[0], 0ull, code) == 0ull) {
        g_sk_error[1] = static_cast<unsigned long long>(cta);
        g_sk_error[2] = static_cast<unsigned long long>(tile);
        g_sk_error[3] = static_cast<unsigned long long>(detail);
    }
}

// Bounded wait of a linear/tree receiver until a hand-off flag reaches `need` (acquire at gpu
// scope; a flag counts the partials its CTA has published). `t0` is the caller's deadline origin
// (0 = not started; set on the first miss), so that several receives can share one deadline.
// False once `limit_ns` has passed since t0 without the flag.
__device__ __forceinline__ bool wait_flag(const uint32_t* f, uint32_t need, uint64_t& t0,
                                          uint64_t limit_ns) {
    while (ld_acquire_gpu(f) < need) {
        if (t0 == 0) t0 = globaltimer_ns();
        if (globaltimer_ns() - t0 > limit_ns) return false;
        __nanosleep(128);
    }
    return true;
}

constexpr int kEpiThreadsWait = 128;       // the epilogue warps (warps 2-5)
constexpr uint32_t kEpiBarrierWait = 2;    // their named barrier for the flag waits

// All 128 epilogue threads wait together until the flags of `count` CTAs have reached their
// values: thread i polls the flags of items i, i + 128, ... (acquire at gpu scope), and a barrier
// reduction tells every thread when all are set, so the round trips to L2 overlap instead of
// following one another. `item(k, cta_of_k, need_of_k)` names item k's CTA and flag value. One
// deadline for all (`limit_ns`), decided collectively. Returns the CTA of a missing flag, or -1.
template <typename Item>
__device__ int64_t wait_flags_all(const uint32_t* flags, int cg, int64_t half, int64_t count,
                                  int ethread, uint64_t limit_ns, Item&& item) {
    uint64_t t0 = 0;
    int64_t missing = -1;
    while (true) {
        bool mine = true;
        for (int64_t k = ethread; k < count; k += kEpiThreadsWait) {
            int64_t c;
            uint32_t need;
            item(k, c, need);
            if (ld_acquire_gpu(flags + c * cg + half) < need) {
                mine = false;
                missing = c;
            }
        }
        if (named_bar_and(kEpiBarrierWait, kEpiThreadsWait, mine)) {
            __threadfence();   // every thread's later reads come after the flags polled above
            return -1;
        }
        if (t0 == 0) t0 = globaltimer_ns();
        const bool late = globaltimer_ns() - t0 > limit_ns;
        if (named_bar_or(kEpiBarrierWait, kEpiThreadsWait, late)) return missing < 0 ? -2 : missing;
        __nanosleep(64);
    }
}

// A flag that nothing ever sets, for sk_probe_flag_timeout.
__device__ uint32_t g_sk_unset_flag;

// Failure-detection probe: one thread waits on g_sk_unset_flag with the receivers' own routine,
// gives up after limit_ns and records the receivers' error (cta -1, tile -1, sender -1), exactly as
// a lost hand-off would; the host reads it with take_device_error. Nothing faults or hangs.
__global__ void sk_flag_timeout_probe_kernel(uint64_t limit_ns) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    uint64_t t0 = 0;
    if (!wait_flag(&g_sk_unset_flag, 1u, t0, limit_ns)) record_error(kErrFlagWait, -1, -1, -1);
}

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kEpiBarrier = 1;
// The prologue of a one-CTA launch without a ticket, whose producer does not wait for it: the
// barrier initialisation published to the other warps, and those warps' own prologue.
constexpr uint32_t kPrologueBar = 3, kPrologueBar2 = 4;

template <int OP, int TN, int CG, int ST>
struct Cfg {
    static_assert(CG == 1 || OP == kOpGemm16 || OP == kOpFp8 || OP == kOpFp8Block ||
                      is_wgrad_row(OP),
                  "CTA pairs serve the GEMMs and the shifted-row wgrad");
    static_assert(CG == 2 || TN == 128 || (is_wgrad_row(OP) && TN == 192) ||
                      (OP == kOpFpropRow && TN == 64),
                  "one CTA computes 128 x 128 tiles (shifted-row wgrad: 128 x 192; shifted-row "
                  "fprop: 128 x 64)");
    static constexpr bool kFpRow = OP == kOpFpropRow;
    static constexpr bool kFp8 = OP == kOpFp8 || OP == kOpFp8Block;
    static constexpr bool kWgRow = is_wgrad_row(OP);
    static constexpr int kPhases = OP == kOpWgradRow2 ? 2 : 1;   // x column phases (W stride)
    static constexpr int kElem = kFp8 ? 1 : 2;
    static constexpr int TK = 128 / kElem;                 // one 128-byte swizzle row per K step
    static constexpr int kTileMAll = kTileM * CG;          // tile rows of the CTA (pair)
    static constexpr int kBRows = TN / CG;                 // B rows this CTA stages
    // Shifted-row wgrad stage: a fixed capacity laid out at run time (ConvGeom stage_steps,
    // x_phase_bytes, x_lbo, dy_off): per x column phase the CTA's x rows of up to stage_steps K
    // steps (8 KB of 64 positions x 64 channels per step and tap row), then their dy rows (64
    // positions x the CTA's filters per step: 128-byte rows, or 64-byte rows of 32 filters in each
    // CTA of a pair) and 16 zero rows for the shifts' overrun.
    static constexpr int kDyRowBytes = 128 / CG;
    static constexpr int kDyPadRows = 16;
    // Shifted-row fprop stage: the x box of a tile's two output rows for every tap row (at most
    // four rows of 64 positions x 64 channels, 32 KB) and 1 KB for the column taps' overrun; its
    // filter (at most 9 taps of 64 x 64) stays in its own 72 KB region for the whole kernel.
    static constexpr int kABytes = kWgRow ? wgrow_stage_bytes(OP, CG)
                                   : kFpRow ? 33 * 1024 : kTileM * 128;   // 16 KB
    static constexpr int kBBytes = (kWgRow || kFpRow) ? 0 : kBRows * 128;
    static constexpr int kResBytes = kFpRow ? 9 * 8192 : 0;
    static constexpr int kStageBytes = kABytes + kBBytes;
    // ST stages in the ring; two CTAs share an SM when the ring is at most 96 KB.
    static constexpr int kStages = ST;
    static constexpr int kMinBlocks = ST * kStageBytes <= 96 * 1024 ? 2 : 1;
    // fp32 accumulator buffers in TMEM: two (the epilogue of one segment overlaps the MMAs of the
    // next), except for the 256-column accumulator of a 256 x 256 pair, which keeps one, and the
    // shifted-row fprop, whose tiles take about as long to store as to compute: four of 64
    // columns, so that the MMAs never wait for an epilogue.
    // Block-scaled fp8: the two buffers take one K step's partial each (the MMAs run up to two steps
    // ahead of the epilogue's promotion); the last step's buffer then holds the segment's sum.
    static constexpr int kAccBufs = (TN == 256 || kWgRow) ? 1 : kFpRow ? 4 : 2;
    static constexpr int kTmemCols = kAccBufs * TN;
    // The allocation is a power of two of at least 32 columns.
    static constexpr int kTmemAlloc = kTmemCols <= 32 ? 32 : kTmemCols <= 64 ? 64
                                      : kTmemCols <= 128 ? 128 : kTmemCols <= 256 ? 256 : 512;
    // Barrier slots: [full x ST][empty x ST][acc full x kAccBars][acc empty x kAccBars][fold].
    static constexpr int kAccBars = kAccBufs < 2 ? 2 : kAccBufs;
    static constexpr int kBarTfull = 2 * kStages;
    static constexpr int kBarTempty = 2 * kStages + kAccBars;
    static constexpr int kBarFold = 2 * kStages + 2 * kAccBars;
    static constexpr int kMmaK = kFp8 ? 32 : 16;
    static constexpr int kMmasPerStage = TK / kMmaK;
    // The owner's fold stages partial tiles through the (then idle) operand ring in units of
    // 128 rows x (32 x kFoldUnitChunks) fp32 columns, contiguous in the fragment-major layout:
    // 64 KB with one CTA per SM, 32 KB in the smaller ring of a pair.
    static constexpr int kFoldUnitChunks =
        (CG == 1 && (TN / 32) % 4 == 0 && ST * kStageBytes >= 128 * 1024) ? 4 : 2;   // 32-column chunks per unit
    static constexpr int kFoldUnitBytes = kTileM * 32 * 4 * kFoldUnitChunks;
    static constexpr int kFoldBufs = kStages * kStageBytes / kFoldUnitBytes;
    static_assert(kFoldBufs >= 2, "the fold needs two staging buffers");
    static_assert((TN / 32) % kFoldUnitChunks == 0, "tile N must be a multiple of the fold unit");
    static constexpr int kRingBytes = kStages * kStageBytes;   // a multiple of 1024
    // One CTA per SM with a 16-bit output (every op but wgrad): a dedicated 32 KB buffer where the
    // epilogue stages each complete 128 x 128 tile for its TMA stores, so that every tile, not only
    // a CTA's last, leaves that way while the producer already fills the ring for the next one.
    // The block-scaled fp8 pair keeps one too (its ring is deep enough without the space).
    // A 3-stage one-CTA ring (two CTAs per SM) has none: its last tile leaves through the ring.
    // The shifted-row fprop stages its 128 x 64 tiles (16 KB) the same way.
    static constexpr int kEpiStageBytes =
        ((CG == 1 && OP != kOpWgrad16 && !kWgRow && ST > 3) || OP == kOpFp8Block)
            ? kTileM * TN * 2
            : 0;
    static constexpr int kCtlBytes = 64;                         // SmemCtl, 1024-aligned
    static constexpr int kBarRes = kBarFold + kFoldBufs;   // shifted-row fprop: filter loaded
    static constexpr int kBarBytes = (kBarRes + 1) * 8;
    // Block-scaled fp8: each epilogue thread's ring of block scales (A and B) copied kScaleAhead
    // K steps ahead of their use, so that their global-memory latency stays off the per-step path.
    static constexpr int kScaleAhead = OP == kOpFp8Block ? 8 : 0;
    static constexpr int kScaleBytes = kScaleAhead * kEpiThreads * 2 * 4;
    static constexpr size_t kSmem =
        1024 + size_t(kRingBytes) + kEpiStageBytes + kScaleBytes + kResBytes + kCtlBytes +
        kBarBytes;
};

// Per-CTA control words. The block starts right after the operand ring, so tmem_base (written by
// tcgen05.alloc) sits at a 1024-byte aligned address.
struct SmemCtl {
    uint32_t tmem_base;
    uint32_t abort;
    long long cta;
    uint32_t epi_ok[2];   // epilogue: accumulator-ready verdict, one slot per alternate segment
    uint32_t warp_ok[2][4];   // block-scaled fp8: each epilogue warp's verdict on a segment's steps
};
static_assert(sizeof(SmemCtl) <= 64, "SmemCtl must fit its 64-byte slot");
constexpr uint32_t kTmemSentinel = 0xFFFFFFFFu;   // not a TMEM address: lane and column out of range

// ---------------------------------------------------------------------------------------------
// operand producer
// ---------------------------------------------------------------------------------------------

// Per-tile constants of the wgrad B operand: for each 64-column slab of the tile, its channel
// coordinate and filter-tap offsets. Computed once per segment, so the per-iteration work of the
// single producer thread is one pixel decomposition (32-bit divisions) and the TMA issues.
template <int TN>
struct WgradSlabs {
    int32_t c[TN / 64];
    uint16_t off_w[TN / 64], off_h[TN / 64];
};

template <int TN>
__device__ __forceinline__ void wgrad_slabs(const ConvGeom& cg, int64_t g, int64_t nt,
                                            WgradSlabs<TN>& sl) {
    const int32_t RS = cg.R * cg.S;
#pragma unroll
    for (int j = 0; j < TN / 64; ++j) {
        const int32_t n0 = static_cast<int32_t>(nt * TN + 64 * j);
        int32_t tap = n0 / cg.Cg;
        const int32_t c0 = n0 - tap * cg.Cg;
        if (tap >= RS) tap = RS - 1;   // slab past the last tap: any valid data, masked later
        const int32_t r = tap / cg.S;
        sl.c[j] = static_cast<int32_t>(g) * cg.Cg + c0;
        sl.off_w[j] = static_cast<uint16_t>(tap - r * cg.S);
        sl.off_h[j] = static_cast<uint16_t>(r);
    }
}

// fprop / dgrad: the first pixel of an M tile in the im2col traversal, decomposed once per segment.
struct PixelStart {
    int32_t w, h, n;   // traversal start (w, h) with the padding applied, image n
};

__device__ __forceinline__ void pixel_start(const ConvGeom& cg, int64_t mt, PixelStart& ps) {
    const uint32_t p0 = static_cast<uint32_t>(mt * kTileM);   // < 2^31 (checked on the host)
    const uint32_t howo = static_cast<uint32_t>(cg.HoWo), wo_n = static_cast<uint32_t>(cg.Wo);
    const uint32_t n_img = p0 / howo;
    const uint32_t rem = p0 - n_img * howo;
    const uint32_t ho = rem / wo_n;
    const uint32_t wo = rem - ho * wo_n;
    ps.w = static_cast<int32_t>(wo) * cg.sw - cg.pw;
    ps.h = static_cast<int32_t>(ho) * cg.sh - cg.ph;
    ps.n = static_cast<int32_t>(n_img);
}

// Shifted-row wgrad stage layout: the one-CTA kernel's is fixed (one step: per phase the two tap
// rows' x boxes, 8 KB apart, then the dy rows); the pair's comes from the host (ConvGeom).
template <int CG, int PHASES>
struct RowLayout {
    uint32_t x_lbo, x_phase, dy_off;
    bool shared_box;
    __device__ __forceinline__ explicit RowLayout(const ConvGeom& cg) {
        if constexpr (CG == 1) {
            x_lbo = 8192u;
            x_phase = 16384u;
            dy_off = PHASES * 16384u;
            shared_box = false;
        } else {
            x_lbo = static_cast<uint32_t>(cg.x_lbo);
            x_phase = static_cast<uint32_t>(cg.x_phase_bytes);
            dy_off = static_cast<uint32_t>(cg.dy_off);
            shared_box = cg.x_shared_box != 0;
        }
    }
};

template <int OP, int TN, int CG, int ST>
__device__ __forceinline__ void issue_loads(const KernelParams& P, int64_t g, int64_t mt,
                                            int64_t nt, int64_t k, uint32_t a_dst, uint32_t b_dst,
                                            uint32_t bar, const WgradSlabs<TN>& sl, uint32_t rank,
                                            const PixelStart& ps) {
    using C = Cfg<OP, TN, CG, ST>;
    if constexpr (OP == kOpFpropRow) {
        // Tile mt: output rows 2*mt and 2*mt+1 of the images' rows counted over ho_pad (even), 64
        // positions each from column 0. One box: the x rows ho0 - ph ... ho0 - ph + R of image n,
        // 64 positions from column -pw (outside the image reads zeros), 64 channels.
        const ConvGeom& cg = P.conv;
        const uint32_t t0 = 2u * static_cast<uint32_t>(mt);
        const uint32_t hp = static_cast<uint32_t>(cg.ho_pad);
        const uint32_t n_img = t0 / hp;
        const int32_t ho0 = static_cast<int32_t>(t0 - n_img * hp);
        tma_load_4d(a_dst, &P.tmap_a, bar, static_cast<int32_t>(g) * cg.Cg, -cg.pw, ho0 - cg.ph,
                    static_cast<int32_t>(n_img));
        (void)k;
        (void)b_dst;
    } else if constexpr (folds_groups_into_columns(OP)) {
        // Reduction index k*64 = (tap, channel block) with the channels fastest.
        const ConvGeom& cg = P.conv;
        const int32_t kk = static_cast<int32_t>(k) * C::TK;
        const int32_t tap = kk / cg.Cg;
        const int32_t c0 = kk - tap * cg.Cg;
        const int32_t r = tap / cg.S;
        const int32_t s = tap - r * cg.S;
        // A: 128 pixels x 64 channels of the im2col'd tensor at tap (r, s) (K-major).
        tma_load_im2col_4d(a_dst, &P.tmap_a, bar, static_cast<int32_t>(g) * cg.Cg + c0, ps.w, ps.h,
                           ps.n, static_cast<uint16_t>(s), static_cast<uint16_t>(r));
        if constexpr (OP == kOpFprop16) {
            // B: 128 filters x 64 of their (r, s, c) entries, w viewed as [K][R*S*C/G] (K-major).
            tma_load_2d(b_dst, &P.tmap_b, bar, kk,
                        static_cast<int32_t>(g * cg.Kg + nt * TN));
        } else {
            // B: the filter at the flipped tap, 64 output-gradient channels (rows of w) x 128 input
            // channels as two 64-channel slabs (MN-major).
            const int32_t fr = cg.r0 + cg.dsh * (cg.R - 1 - r);
            const int32_t fs = cg.s0 + cg.dsw * (cg.S - 1 - s);
            const int32_t col = (fr * cg.Sf + fs) * cg.Cw + static_cast<int32_t>(nt * TN);
#pragma unroll
            for (int j = 0; j < TN / 64; ++j)
                tma_load_2d(b_dst + j * (C::TK * 128), &P.tmap_b, bar, col + 64 * j,
                            static_cast<int32_t>(g) * cg.Kg + c0);
        }
    } else if constexpr (is_wgrad_row(OP)) {
        // A stage from K step k on: rows_per_step output rows of image n per step (rows counted
        // per image over ho_pad), each a segment of wseg positions. B = dy from position -qmax, so
        // that each segment starts with the zero halo that the shifted reads of its first
        // positions take (and the last step's overrun reads the next row's); A = per column phase
        // the x rows of the CTA's two tap rows, at traversal strides (sw, sh) from the tensor map.
        // A CTA pair splits the filters: this CTA's 32 of them; its tap rows are the pair tile's
        // 128-row half of (tap row, channel): rows 2 * (mt * CG + rank) and the next.
        const ConvGeom& cg = P.conv;
        const uint32_t rr0 = static_cast<uint32_t>(k) * static_cast<uint32_t>(cg.rows_per_step);
        const uint32_t hp = static_cast<uint32_t>(cg.ho_pad);
        const uint32_t n_img = rr0 / hp;   // < 2^31 (checked on the host)
        const int32_t ho0 = static_cast<int32_t>(rr0 - n_img * hp);
        auto load4 = [&](uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y, int32_t z) {
            if constexpr (CG == 2)
                tma_load_4d_pair(dst, m, bar, x, y, z, static_cast<int32_t>(n_img));
            else
                tma_load_4d(dst, m, bar, x, y, z, static_cast<int32_t>(n_img));
        };
        const RowLayout<CG, C::kPhases> lay(cg);
        load4(a_dst + lay.dy_off, &P.tmap_b,
              static_cast<int32_t>(g) * cg.Kg + static_cast<int32_t>(rank) * (64 / CG), -cg.qmax,
              ho0);
        const int32_t r0 = 2 * (static_cast<int32_t>(mt) * CG + static_cast<int32_t>(rank));
#pragma unroll
        for (int phs = 0; phs < C::kPhases; ++phs) {
            const uint32_t xd = a_dst + phs * lay.x_phase;
            if (lay.shared_box) {   // both tap rows in one box of stage_steps * rows_per_step + 1 rows
                if (r0 < cg.R)
                    load4(xd, &P.tmap_a, static_cast<int32_t>(g) * cg.Cg, phs - cg.pw,
                          ho0 + r0 - cg.ph);
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (r0 + j < cg.R)
                        load4(xd + j * lay.x_lbo, &P.tmap_a,
                              static_cast<int32_t>(g) * cg.Cg, phs - cg.pw,
                              cg.sh * ho0 + r0 + j - cg.ph);
            }
        }
    } else if constexpr (CG == 2) {
        // This CTA's rows of the pair tile: A rows [128*rank, +128), B rows [TN/2*rank, +TN/2).
        const int32_t kx = static_cast<int32_t>(k * C::TK);
        tma_load_2d_pair(a_dst, &P.tmap_a, bar, kx,
                         static_cast<int32_t>(mt * C::kTileMAll + rank * kTileM));
        tma_load_2d_pair(b_dst, &P.tmap_b, bar, kx,
                         static_cast<int32_t>(nt * TN + rank * C::kBRows));
    } else if constexpr (OP != kOpWgrad16) {
        const int32_t kx = static_cast<int32_t>(k * C::TK);
        tma_load_2d(a_dst, &P.tmap_a, bar, kx, static_cast<int32_t>(mt * kTileM));
        tma_load_2d(b_dst, &P.tmap_b, bar, kx, static_cast<int32_t>(nt * TN));
    } else {
        // A = dy viewed as [pixels][K]: two 64-filter slabs of TK pixel rows (MN-major).
        const ConvGeom& cg = P.conv;
        const uint32_t p0 = static_cast<uint32_t>(k) * C::TK;   // < 2^31 (checked on the host)
        const int32_t k0 = static_cast<int32_t>(g * cg.Kg + mt * kTileM);
#pragma unroll
        for (int j = 0; j < kTileM / 64; ++j)
            tma_load_2d(a_dst + j * (C::TK * 128), &P.tmap_a, bar, k0 + 64 * j,
                        static_cast<int32_t>(p0));
        // B = im2col(x): per 64-column slab one filter tap (r, s) and 64 channels, TK pixels
        // starting at output pixel p0 = (n, ho, wo).
        const uint32_t howo = static_cast<uint32_t>(cg.HoWo), wo_n = static_cast<uint32_t>(cg.Wo);
        const uint32_t n_img = p0 / howo;
        const uint32_t rem = p0 - n_img * howo;
        const uint32_t ho = rem / wo_n;
        const uint32_t wo = rem - ho * wo_n;
        const int32_t w = static_cast<int32_t>(wo) * cg.sw - cg.pw;
        const int32_t h = static_cast<int32_t>(ho) * cg.sh - cg.ph;
#pragma unroll
        for (int j = 0; j < TN / 64; ++j)
            tma_load_im2col_4d(b_dst + j * (C::TK * 128), &P.tmap_b, bar, sl.c[j], w, h,
                               static_cast<int32_t>(n_img), sl.off_w[j], sl.off_h[j]);
    }
}

// Start offset of a segment's iteration order: rotated for stream-K segments (see
// sk_segment_rotation), natural order for data-parallel tiles and the off / split-K modes. Advances
// `tau`, the stream-K iterations this CTA has run.
__device__ __forceinline__ int64_t segment_rotation(const sk_plan_t& plan, bool dp,
                                                    const sk_segment_t& seg, int64_t& tau) {
    if (dp || plan.mode == SK_OFF || plan.mode == SK_SPLITK) return 0;
    const int64_t len = seg.k_end - seg.k_begin;
    const int64_t rot = sk_segment_rotation(plan.iters_per_sk_cta, seg.k_begin, len, tau);
    tau += len;
    return rot;
}

// K steps in the ring stage at position j of a segment's rotated order: one, or for the
// shifted-row wgrad up to stage_steps consecutive steps of one image before the order wraps or the
// segment ends. The producer and the MMA issuer walk the same stages.
template <int OP, int CG>
__device__ __forceinline__ int64_t stage_step_count(const ConvGeom& cg, const sk_segment_t& seg,
                                                    int64_t rot, int64_t j) {
    if constexpr (OP == kOpFpropRow) {
        // every tap of the segment reads the tile's one x box
        (void)cg;
        (void)rot;
        return (seg.k_end - seg.k_begin) - j;
    } else if constexpr (!is_wgrad_row(OP) || CG == 1) {   // one-CTA row wgrad: one step per stage
        return 1;
    } else {
        const int64_t len = seg.k_end - seg.k_begin;
        int64_t k = seg.k_begin + rot + j;
        int64_t run;
        if (k >= seg.k_end) {
            k -= len;
            run = seg.k_begin + rot - k;   // up to the wrap point
        } else {
            run = seg.k_end - k;
        }
        const uint32_t rr0 = static_cast<uint32_t>(k) * static_cast<uint32_t>(cg.rows_per_step);
        const uint32_t hp = static_cast<uint32_t>(cg.ho_pad);
        const uint32_t ho0 = rr0 - (rr0 / hp) * hp;
        const int64_t img = static_cast<int64_t>((hp - ho0) / static_cast<uint32_t>(cg.rows_per_step));
        return imin(imin(static_cast<int64_t>(cg.stage_steps), run), img);
    }
}

template <int OP, int TN, int CG, int ST>
__device__ void run_producer(const KernelParams& P, int64_t cta, uint32_t ring, uint32_t bars,
                             volatile SmemCtl* ctl, uint32_t rank) {
    using C = Cfg<OP, TN, CG, ST>;
    const sk_plan_t& plan = P.plan;
    SegCursor cur;
    seg_init(plan, cta, cur);
    sk_segment_t seg;
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0, tau = 0;
    bool ok = true;
    bool res_pending = false;   // shifted-row fprop: filter copies in flight (drained at the end)
    if constexpr (C::kFpRow) {
        // The filter, tap (r, s) = w[0..63][r][s][0..63] (64 filters x 64 channels, K-major), 8 KB
        // apart in the resident region, once for the CTA's whole work.
        const uint32_t res = ring + C::kRingBytes + C::kEpiStageBytes + C::kScaleBytes;
        const uint32_t bar = bars + C::kBarRes * 8;
        const int taps = P.conv.R * P.conv.S;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(taps) * 8192u);
        if (P.conv.filter_box)
            tma_load_3d(res, &P.tmap_b, bar, 0, 0, 0);
        else
            for (int t = 0; t < taps; ++t) tma_load_2d(res + t * 8192, &P.tmap_b, bar, t * 64, 0);
        res_pending = true;
    }
    while (true) {
        const bool dp = cur.dp_next >= 0;
        if (!ok || !seg_next(plan, cta, cur, seg)) break;
        int64_t g, mt, nt;
        tile_coords(plan, seg.tile, g, mt, nt);
        // Bytes one stage receives (of both CTAs of a pair). A shifted-row wgrad stage is whole
        // boxes whatever its steps: each CTA's dy box (64 positions of its filters per step) and
        // per phase its x box(es): a shared box of stage_steps * rows_per_step + 1 rows when its
        // upper tap row is inside the filter, else one box of stage_steps * 8 KB per tap row
        // inside it.
        uint32_t stage_tx = CG * C::kStageBytes;
        if constexpr (C::kFpRow) stage_tx = static_cast<uint32_t>(P.conv.R + 1) * 8192u;
        if constexpr (C::kWgRow) {
            const ConvGeom& cg = P.conv;
            const uint32_t T = CG == 1 ? 1u : static_cast<uint32_t>(cg.stage_steps);
            const RowLayout<CG, C::kPhases> lay(cg);
            uint32_t x = 0;
            for (int c = 0; c < CG; ++c) {
                const int64_t r0 = 2 * (mt * CG + c);
                if (lay.shared_box)
                    x += r0 < cg.R ? (T * static_cast<uint32_t>(cg.rows_per_step) + 1u) *
                                         static_cast<uint32_t>(cg.wseg) * 128u
                                   : 0u;
                else
                    x += (r0 + 1 < cg.R ? 2u : (r0 < cg.R ? 1u : 0u)) * T * 8192u;
            }
            stage_tx = static_cast<uint32_t>(CG) * T * 64u * static_cast<uint32_t>(C::kDyRowBytes) +
                       static_cast<uint32_t>(C::kPhases) * x;
        }
        WgradSlabs<TN> slabs;
        if constexpr (OP == kOpWgrad16) wgrad_slabs<TN>(P.conv, g, nt, slabs);
        PixelStart ps{0, 0, 0};
        if constexpr (folds_groups_into_columns(OP) && !C::kFpRow) pixel_start(P.conv, mt, ps);
        const int64_t len = seg.k_end - seg.k_begin;
        const int64_t rot = segment_rotation(plan, dp, seg, tau);
        if constexpr (C::kWgRow && CG == 1) {
            // One K step per stage. The copies' coordinates advance step by step (image n, output
            // row ho0), with no division and no per-step setup, so that the thread's own work
            // between a stage's last copy and the next stage's first stays short against the
            // copy engine's time per box (a copy instruction waits for the previous box).
            const ConvGeom& cg = P.conv;
            const uint32_t rps = static_cast<uint32_t>(cg.rows_per_step);
            const uint32_t hp = static_cast<uint32_t>(cg.ho_pad);
            const int32_t r0 = 2 * static_cast<int32_t>(mt);
            const int32_t dy_c = static_cast<int32_t>(g) * cg.Kg, x_c = static_cast<int32_t>(g) * cg.Cg;
            const RowLayout<CG, C::kPhases> lay(cg);
            // k * rows_per_step < 2^31 (checked on the host)
            const uint32_t kb = static_cast<uint32_t>(seg.k_begin);
            const uint32_t ke = static_cast<uint32_t>(seg.k_end);
            uint32_t kk = static_cast<uint32_t>(seg.k_begin + rot);
            uint32_t n_img = (kk * rps) / hp;
            uint32_t ho0 = kk * rps - n_img * hp;
            for (int64_t j = 0; j < len; ++j) {
                const uint32_t full = bars + stage * 8, empty = bars + (C::kStages + stage) * 8;
                if (!mbar_wait(empty, phase ^ 1, P.mbar_timeout_ns) || ctl->abort) {
                    record_error(kErrPipeline, cta, seg.tile, 0);
                    ctl->abort = 1;
                    ok = false;
                    break;
                }
                const uint32_t a_dst = ring + stage * C::kStageBytes;
                mbar_arrive_expect_tx(full, stage_tx);
                const int32_t h0 = static_cast<int32_t>(ho0), ni = static_cast<int32_t>(n_img);
                tma_load_4d(a_dst + lay.dy_off, &P.tmap_b, full, dy_c, -cg.qmax, h0, ni);
#pragma unroll
                for (int phs = 0; phs < C::kPhases; ++phs)
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj)
                        if (r0 + jj < cg.R)
                            tma_load_4d(a_dst + phs * lay.x_phase + jj * lay.x_lbo, &P.tmap_a, full,
                                        x_c, phs - cg.pw, cg.sh * h0 + r0 + jj - cg.ph, ni);
                ++issued;
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1;
                }
                if (++kk == ke) {   // the rotation wraps to the segment's start
                    kk = kb;
                    n_img = (kk * rps) / hp;
                    ho0 = kk * rps - n_img * hp;
                } else if ((ho0 += rps) == hp) {   // ho_pad is a multiple of rows_per_step
                    ho0 = 0;
                    ++n_img;
                }
            }
            continue;
        }
        for (int64_t j = 0; j < len; j += stage_step_count<OP, CG>(P.conv, seg, rot, j)) {
            int64_t k = seg.k_begin + rot + j;
            if (k >= seg.k_end) k -= len;
            const uint32_t full = bars + stage * 8, empty = bars + (C::kStages + stage) * 8;
            if (!mbar_wait(empty, phase ^ 1, P.mbar_timeout_ns) || ctl->abort) {
                record_error(kErrPipeline, cta, seg.tile, 0);
                ctl->abort = 1;
                ok = false;
                break;
            }
            const uint32_t a_dst = ring + stage * C::kStageBytes;
            if constexpr (CG == 2) {
                // Both CTAs' bytes are counted on the even CTA's barrier, which expects them all.
                if (rank == 0) mbar_arrive_expect_tx(full, stage_tx);
                issue_loads<OP, TN, CG, ST>(P, g, mt, nt, k, a_dst, a_dst + C::kABytes,
                                            mapa_shared(full, 0), slabs, rank, ps);
            } else {
                mbar_arrive_expect_tx(full, stage_tx);
                issue_loads<OP, TN, CG, ST>(P, g, mt, nt, k, a_dst, a_dst + C::kABytes, full, slabs,
                                            rank, ps);
            }
            ++issued;
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
    // The filter's copies land before the CTA can exit, even if it had no work.
    if (res_pending) mbar_wait(bars + C::kBarRes * 8, 0u, 10000000ull);
    if constexpr (CG == 2) {
        // The copies of a pair complete on the even CTA's barriers, so this CTA waits until the
        // MMAs have consumed its last stages (their commits arrive here too): then nothing is
        // still in flight into this CTA's shared memory, nor any commit on its way to it.
        for (int i = 0; i < C::kStages && i < issued; ++i) {
            if (stage == 0) {
                stage = C::kStages;
                phase ^= 1;
            }
            --stage;
            mbar_wait(bars + (C::kStages + stage) * 8, phase, 10000000ull);
        }
    } else if (!ok) {
        // Let the copies already in flight land before the CTA can exit.
        for (int i = 0; i < C::kStages && i < issued; ++i) {
            if (stage == 0) {
                stage = C::kStages;
                phase ^= 1;
            }
            --stage;
            mbar_wait(bars + stage * 8, phase, 10000000ull);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// MMA issuer
// ---------------------------------------------------------------------------------------------

// Waits for one ring stage and issues its MMAs into d_tmem (accumulating onto what is there when
// `accumulate`), then commits the stage back to the producer. False if the wait gave up.
template <int OP, int TN, int CG, int ST>
__device__ __forceinline__ bool mma_stage(const KernelParams& P, int64_t cta,
                                          const sk_segment_t& seg, uint32_t ring, uint32_t bars,
                                          volatile SmemCtl* ctl, uint32_t d_tmem, bool accumulate,
                                          uint32_t& stage, uint32_t& phase, int64_t steps,
                                          int64_t k0) {
    using C = Cfg<OP, TN, CG, ST>;
    static_assert(C::kMmasPerStage == 4, "a K step is four MMAs");
    const uint32_t full = bars + stage * 8, empty = bars + (C::kStages + stage) * 8;
    const uint32_t a_addr = ring + stage * C::kStageBytes;
    const uint32_t b_addr = a_addr + C::kABytes;
    // The stage's descriptors go into registers before its data is awaited, and its MMAs then
    // leave back to back (mma_x4): the issuing thread stalls while the tensor pipe runs the
    // previous MMA, so work between two MMAs would leave the pipe idle.
    uint64_t ad[C::kPhases][4], bd[C::kPhases][4];
    uint32_t idesc[C::kPhases], col0[C::kPhases];
    bool live[C::kPhases];
    if constexpr (C::kWgRow) {
        // Per K step and column phase: D[(tap row, channel)][(shift, filter)] over the step's 64
        // positions. A = the CTA's upper and lower tap-row x rows of the step (8 KB per step
        // along the box, the lower one x_lbo bytes after the upper); B = the step's dy rows read
        // at the phase's nq shifts, one block of the CTA's filters per shift, each block one row
        // after the previous (LBO = one dy row): block b holds shift q = nq - 1 - b, its rows
        // start at qmax - q. The phase's taps fill D columns [col0, col0 + 64 * nq); a CTA pair
        // (M = 256: four tap rows) takes the first half of them from the even CTA's 32 filters
        // and the second half from the odd CTA's, in 64-byte swizzled rows. The descriptors here
        // are the stage's first step; step t adds t * 8 KB (A) and t * 64 dy rows (B).
        const ConvGeom& cg = P.conv;
        const RowLayout<CG, C::kPhases> lay(cg);
        uint32_t c0 = 0;
#pragma unroll
        for (int phs = 0; phs < C::kPhases; ++phs) {
            const uint32_t nq = static_cast<uint32_t>(cg.nq[phs]);
            idesc[phs] = (P.idesc & ~(0x3Fu << 17)) | ((nq * 64u >> 3) << 17);
            col0[phs] = c0;
            live[phs] = nq > 0;
            const uint32_t xa = a_addr + phs * lay.x_phase;
            const uint32_t b0 = a_addr + lay.dy_off +
                                static_cast<uint32_t>(cg.qmax + 1 - static_cast<int>(nq)) *
                                    static_cast<uint32_t>(C::kDyRowBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                ad[phs][kk] = smem_desc_sw128(xa + kk * 2048, lay.x_lbo, 1024);
                bd[phs][kk] = CG == 1 ? smem_desc_sw128(b0 + kk * 2048, 128, 1024)
                                      : smem_desc_sw64(b0 + kk * 16 * C::kDyRowBytes,
                                                       C::kDyRowBytes, 8 * C::kDyRowBytes);
            }
            c0 += nq * 64u;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            // MN-major: 16 K-rows of 128 B per MMA; 64-element slabs TK*128 B apart.
            // K-major: advance 32 B (one MMA's K) inside the 128-byte swizzle row.
            if constexpr (OP == kOpWgrad16)
                ad[0][kk] = smem_desc_sw128(a_addr + kk * 2048, C::TK * 128, 1024);
            else
                ad[0][kk] = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            if constexpr (OP == kOpWgrad16 || OP == kOpDgrad16)
                bd[0][kk] = smem_desc_sw128(b_addr + kk * 2048, C::TK * 128, 1024);
            else
                bd[0][kk] = smem_desc_sw128(b_addr + kk * 32, 16, 1024);
        }
        idesc[0] = P.idesc;
        col0[0] = 0;
        live[0] = true;
    }
    // The abort flag is read here only for the block-scaled op: elsewhere the read on every step
    // measured slower (128x128 tile: 1012 against 1064 TFLOP/s), and a stalled producer still ends
    // the wait at its time limit.
    if (!mbar_wait(full, phase, P.mbar_timeout_ns) || (OP == kOpFp8Block && ctl->abort)) {
        record_error(kErrPipeline, cta, seg.tile, 2);
        ctl->abort = 1;
        return false;
    }
    tc_fence_after();
    const uint32_t acc = accumulate ? 1u : 0u;
    if constexpr (C::kFpRow) {
        // Step k = tap (r, s) of the reduction (64 channels each). D[(output row, position)][filter]
        // += x[row + r][position + s][c] * w[filter][r][s][c]: A = the box's rows from row r,
        // position s on (128 consecutive 128-byte rows, K-major: any row may start the 128-byte
        // swizzle pattern); B = the resident filter tap (K-major). Steps in the segment's order,
        // which wraps at k_end.
        // Descriptors: the base ones plus the tap's offset in 16-byte units (addresses stay
        // below 2^18, so the sums never leave the 14-bit address field); (r, s) advance with the
        // tap, no division per step.
        // As a data gradient (row_flip) B is the flipped tap, MN-major: 16 of its 128-byte rows
        // (filters) per MMA, 8-row atoms 1024 bytes apart.
        const uint32_t res = ring + C::kRingBytes + C::kEpiStageBytes + C::kScaleBytes;
        const bool flip = P.conv.row_flip != 0;
        const uint64_t a_base = smem_desc_sw128(a_addr, 16, 1024);
        const uint64_t b_base = smem_desc_sw128(res, flip ? 8192 : 16, 1024);
        const uint64_t b_kstep = flip ? 128 : 2;
        const int S = P.conv.S, taps_1 = P.conv.R * P.conv.S - 1;
        int tap = static_cast<int>(k0);
        int r = tap / S, s_ = tap - r * S;
        for (int64_t t = 0; t < steps; ++t) {
            const uint64_t ao = static_cast<uint64_t>((r * 64 + s_) * 8);
            const uint64_t bo = static_cast<uint64_t>((flip ? taps_1 - tap : tap) * 512);
            uint64_t a[4], b[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                a[kk] = a_base + ao + 2 * kk;
                b[kk] = b_base + bo + b_kstep * kk;
            }
            mma_x4<CG, false>(d_tmem, a, b, P.idesc, t > 0 ? 1u : acc);
            // next tap in the segment's order, which wraps from k_end - 1 to k_begin
            if (++tap == seg.k_end) {
                tap = static_cast<int>(seg.k_begin);
                r = tap / S;
                s_ = tap - r * S;
            } else if (++s_ == S) {
                s_ = 0;
                ++r;
            }
        }
    } else if constexpr (C::kWgRow) {
        // Descriptor address fields count 16-byte units.
        constexpr uint64_t kStepA = 8192 >> 4, kStepB = (64 * C::kDyRowBytes) >> 4;
        const int64_t nsteps = CG == 1 ? 1 : steps;
        for (int64_t t = 0; t < nsteps; ++t) {
#pragma unroll
            for (int phs = 0; phs < C::kPhases; ++phs) {
                if (!live[phs]) continue;
                uint64_t a[4], b[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    a[kk] = ad[phs][kk] + static_cast<uint64_t>(t) * kStepA;
                    b[kk] = bd[phs][kk] + static_cast<uint64_t>(t) * kStepB;
                }
                mma_x4<CG, false>(d_tmem + col0[phs], a, b, idesc[phs], t > 0 ? 1u : acc);
            }
        }
    } else {
        (void)steps;
        (void)k0;
        mma_x4<CG, C::kFp8>(d_tmem + col0[0], ad[0], bd[0], idesc[0], acc);
    }
    tc_commit<CG>(empty);
    if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1;
    }
    return true;
}

template <int OP, int TN, int CG, int ST>
__device__ void run_mma(const KernelParams& P, int64_t cta, uint32_t ring, uint32_t bars,
                        uint32_t tmem_base, volatile SmemCtl* ctl) {
    using C = Cfg<OP, TN, CG, ST>;
    const sk_plan_t& plan = P.plan;
    SegCursor cur;
    seg_init(plan, cta, cur);
    sk_segment_t seg;
    uint32_t stage = 0, phase = 0;
    int64_t nseg = 0, tau = 0;
    int64_t total_commits = 0;
    bool any = false, ok = true;
    if constexpr (C::kFpRow) {   // the resident filter, loaded once by the producer
        if (!mbar_wait(bars + C::kBarRes * 8, 0u, P.mbar_timeout_ns)) {
            record_error(kErrPipeline, cta, -1, 6);
            ctl->abort = 1;
            ok = false;
        }
        tc_fence_after();
    }
    while (true) {
        const bool dp = cur.dp_next >= 0;
        if (!ok || !seg_next(plan, cta, cur, seg)) break;
        const int64_t len = seg.k_end - seg.k_begin;
        const uint32_t acc = static_cast<uint32_t>(nseg % C::kAccBufs);
        const uint32_t acc_phase = static_cast<uint32_t>((nseg / C::kAccBufs) & 1);
        const uint32_t tfull = bars + (C::kBarTfull + acc) * 8;
        const uint32_t tempty = bars + (C::kBarTempty + acc) * 8;
        // A pair's accumulator is free once the epilogues of both CTAs have released it.
        const bool free_acc = CG == 2 ? mbar_wait_cluster(tempty, acc_phase ^ 1, P.mbar_timeout_ns)
                                      : mbar_wait(tempty, acc_phase ^ 1, P.mbar_timeout_ns);
        if (!free_acc || ctl->abort) {
            record_error(kErrPipeline, cta, seg.tile, 1);
            ctl->abort = 1;
            break;
        }
        tc_fence_after();
        uint32_t d_tmem = tmem_base + acc * TN;
        // The shifted-row kernels group K steps into stages as the producer does (same rotation).
        const int64_t rot = (is_wgrad_row(OP) || OP == kOpFpropRow)
                                ? segment_rotation(plan, dp, seg, tau) : 0;
        for (int64_t j = 0, steps = 1; j < len; j += steps) {
            steps = stage_step_count<OP, CG>(P.conv, seg, rot, j);
            int64_t k0 = seg.k_begin + rot + j;
            if (k0 >= seg.k_end) k0 -= len;
            // Block scales: every K step starts a fresh partial.
            const bool accumulate = OP == kOpFp8Block ? false : j > 0;
            if (!mma_stage<OP, TN, CG, ST>(P, cta, seg, ring, bars, ctl, d_tmem, accumulate, stage,
                                           phase, steps, k0)) {
                ok = false;
                break;
            }
            ++total_commits;
            any = true;
            if constexpr (OP == kOpFp8Block) {
                // One partial per K step: the epilogue scales it with that step's block scales. Its
                // completion is the ring stage's commit (mma_stage), which the epilogue waits on.
                ++nseg;
                if (j + 1 < len) {
                    const uint32_t a2 = static_cast<uint32_t>(nseg % C::kAccBufs);
                    const uint32_t ph2 = static_cast<uint32_t>((nseg / C::kAccBufs) & 1);
                    const uint32_t te2 = bars + (C::kBarTempty + a2) * 8;
                    const bool free2 = CG == 2 ? mbar_wait_cluster(te2, ph2 ^ 1, P.mbar_timeout_ns)
                                               : mbar_wait(te2, ph2 ^ 1, P.mbar_timeout_ns);
                    if (!free2 || ctl->abort) {
                        record_error(kErrPipeline, cta, seg.tile, 1);
                        ctl->abort = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    d_tmem = tmem_base + a2 * TN;
                }
            }
        }
        if (!ok) break;
        if constexpr (OP != kOpFp8Block) {
            tc_commit<CG>(tfull);
            ++nseg;
        }
    }
    // Before the CTA may exit, every commit it issued must have landed: the last commit of each
    // stage of the ring is awaited, so that no arrival can reach this SM's shared memory after the
    // CTA is gone (the next CTA there may lay it out differently).
    if (any) {
        int64_t n = total_commits < C::kStages ? total_commits : C::kStages;
        uint32_t st = stage, ph = phase;
        for (int64_t i = 0; i < n; ++i) {
            if (st == 0) {
                st = C::kStages;
                ph ^= 1;
            }
            --st;
            mbar_wait(bars + (C::kStages + st) * 8, ph, 10000000ull);
        }
    }
    if (OP != kOpFp8Block && nseg > 0) {   // and the last accumulator commit
        const int64_t last = nseg - 1;
        mbar_wait(bars + (C::kBarTfull + last % C::kAccBufs) * 8,
                  static_cast<uint32_t>((last / C::kAccBufs) & 1), 10000000ull);
    }
}

// ---------------------------------------------------------------------------------------------
// epilogue
// ---------------------------------------------------------------------------------------------

struct EpiCtx {
    int64_t out_row;       // output row of this thread (g*gemm_m + m)
    bool row_ok;           // m < gemm_m
    int64_t n_base;        // first output column of the tile
    int64_t n_end;         // output columns of this tile's group end here (exclusive)
    int row;               // accumulator row 0..127
    int64_t half;          // CG = 2: rank of this CTA in its pair (which 128 rows of the tile); else 0
    int64_t mt;            // the tile's row block (shifted-row fprop: output rows 2*mt, 2*mt + 1)
    float row_scale;       // fp8: sa[out_row] (per-tensor: the scale product); else 1
};

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// Shifted-row wgrad: the dW offset, relative to the thread's (group, tap row, channel) base, of
// the first filter of the 32 D columns starting at `col` (a multiple of 32), or -1 past the tile's
// taps. A phase's columns are cg.fsplit halves (one per CTA of the filter split), each nq blocks of
// 64 / fsplit consecutive filters (`ldc` = R*S*C/G elements apart), block b for shift
// q = nq - 1 - b.
__device__ __forceinline__ int64_t wgrow_col_offset(const ConvGeom& cg, int64_t ldc, int col) {
    const int fw = 64 / cg.fsplit;   // filters per block
    int cb = 0;
#pragma unroll
    for (int phs = 0; phs < 2; ++phs) {
        const int nq = cg.nq[phs];
        if (col < cb + nq * 64) {
            const int local = col - cb;
            const int h = local / (nq * fw), rem = local - h * nq * fw;
            const int b = rem / fw, k0 = h * fw + (rem - b * fw);
            const int s = cg.sw * (nq - 1 - b) + phs;
            return static_cast<int64_t>(k0) * ldc + static_cast<int64_t>(s) * cg.Cg;
        }
        cb += nq * 64;
    }
    return -1;
}

// Where an element of the tile goes: the output, its type and the op (which decides how tile rows
// and columns map to output rows and columns), the fp8 scales (scale_mode 0: none; 1: sa[row] *
// sb[column]; 2: the per-tensor product `scale`) and the convolution geometry.
struct OutSpec {
    void* c;
    int64_t ldc;
    int32_t c_dtype, op_kind;
    const float* sa;
    const float* sb;
    float scale;
    int32_t scale_mode;
    const ConvGeom* conv;
};

// Scale, convert and store four consecutive GEMM-view columns n0..n0+3 of row m of group g
// (columns past gemm_n are dropped; rows and columns outside the view are the caller's to skip).
__device__ __forceinline__ void store4_out(const sk_plan_t& plan, const OutSpec& o, int64_t g,
                                           int64_t m, int64_t n0, float (&v)[4]) {
    const bool fold_cols = folds_groups_into_columns(o.op_kind);
    const int64_t out_row = fold_cols ? map_row(o.conv->rows, m) : g * plan.gemm_m + m;
    if (out_row < 0) return;   // a padded position (shifted-row fprop)
    if (o.scale_mode == 1) {
        const float rs = o.sa[out_row];
        for (int j = 0; j < 4; ++j) v[j] *= rs * (n0 + j < plan.gemm_n ? o.sb[n0 + j] : 0.0f);
    } else if (o.scale_mode == 2) {
        for (int j = 0; j < 4; ++j) v[j] *= o.scale;
    }
    if (is_wgrad_row(o.op_kind)) {   // four consecutive filters of one (tap, channel)
        const ConvGeom& cg = *o.conv;
        const int64_t r = m >> 6, c = m & 63;
        const int64_t coff = wgrow_col_offset(cg, o.ldc, static_cast<int>(n0 & ~int64_t(31)));
        if (coff < 0) return;
        const int64_t base = (g * cg.Kg) * o.ldc + r * cg.S * cg.Cg + c + coff + (n0 & 31) * o.ldc;
        for (int j = 0; j < 4; ++j) {
            if (o.c_dtype == SK_F32)
                static_cast<float*>(o.c)[base + j * o.ldc] = v[j];
            else if (o.c_dtype == SK_BF16)
                static_cast<__nv_bfloat16*>(o.c)[base + j * o.ldc] = __float2bfloat16_rn(v[j]);
            else
                static_cast<__half*>(o.c)[base + j * o.ldc] = __float2half_rn(v[j]);
        }
        return;
    }
    const int64_t col = fold_cols ? g * plan.gemm_n + n0 : n0;
    const int64_t off = out_row * o.ldc + col;
    const bool full = n0 + 4 <= plan.gemm_n;
    if (o.c_dtype == SK_F32) {
        float* dst = static_cast<float*>(o.c) + off;
        if (full) *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        else for (int j = 0; j < 4 && n0 + j < plan.gemm_n; ++j) dst[j] = v[j];
    } else if (o.c_dtype == SK_BF16) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(o.c) + off;
        if (full) {
            __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t*>(&a);
            w.y = *reinterpret_cast<uint32_t*>(&b);
            *reinterpret_cast<uint2*>(dst) = w;
        } else {
            for (int j = 0; j < 4 && n0 + j < plan.gemm_n; ++j) dst[j] = __float2bfloat16_rn(v[j]);
        }
    } else {
        __half* dst = static_cast<__half*>(o.c) + off;
        if (full) {
            __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t*>(&a);
            w.y = *reinterpret_cast<uint32_t*>(&b);
            *reinterpret_cast<uint2*>(dst) = w;
        } else {
            for (int j = 0; j < 4 && n0 + j < plan.gemm_n; ++j) dst[j] = __float2half_rn(v[j]);
        }
    }
}

// Store 32 consecutive columns (n_base + col0 ...) of this thread's row.
template <int OP>
__device__ __forceinline__ void store_out(const KernelParams& P, const EpiCtx& e, int col0,
                                          float (&v)[32]) {
    if (!e.row_ok) return;
    if constexpr (is_wgrad_row(OP)) {
        // 32 filters of one (tap, channel): a warp's lanes hold consecutive channels, so each
        // filter's 32 values form one contiguous 128-byte (fp32) or 64-byte line.
        const int64_t off = wgrow_col_offset(P.conv, P.ldc, col0);
        if (off < 0) return;
        const int64_t base = e.out_row + off;
        if (P.c_dtype == SK_F32) {
            float* dst = static_cast<float*>(P.c) + base;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[i * P.ldc] = v[i];
        } else if (P.c_dtype == SK_BF16) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(P.c) + base;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[i * P.ldc] = __float2bfloat16_rn(v[i]);
        } else {
            __half* dst = static_cast<__half*>(P.c) + base;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[i * P.ldc] = __float2half_rn(v[i]);
        }
        return;
    }
    const int64_t n0 = e.n_base + col0;
    const int64_t ncols = e.n_end;
    if (n0 >= ncols) return;
    if constexpr (OP == kOpFp8) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int64_t n = n0 + i;
            v[i] *= e.row_scale * (n < ncols ? (P.sb ? __ldg(P.sb + n) : 1.0f) : 0.0f);
        }
    }
    const bool full = n0 + 32 <= ncols;
    if (P.c_dtype == SK_F32) {
        float* dst = static_cast<float*>(P.c) + e.out_row * P.ldc + n0;
        if (full) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
            for (int i = 0; i < 32 && n0 + i < ncols; ++i) dst[i] = v[i];
        }
    } else if (P.c_dtype == SK_BF16) {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(P.c) + e.out_row * P.ldc + n0;
        if (full) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                uint4 w;
                __nv_bfloat162 h0 = __floats2bfloat162_rn(v[i], v[i + 1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(v[i + 2], v[i + 3]);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(v[i + 4], v[i + 5]);
                __nv_bfloat162 h3 = __floats2bfloat162_rn(v[i + 6], v[i + 7]);
                w.x = *reinterpret_cast<uint32_t*>(&h0);
                w.y = *reinterpret_cast<uint32_t*>(&h1);
                w.z = *reinterpret_cast<uint32_t*>(&h2);
                w.w = *reinterpret_cast<uint32_t*>(&h3);
                *reinterpret_cast<uint4*>(dst + i) = w;
            }
        } else {
            for (int i = 0; i < 32 && n0 + i < ncols; ++i) dst[i] = __float2bfloat16_rn(v[i]);
        }
    } else {
        __half* dst = static_cast<__half*>(P.c) + e.out_row * P.ldc + n0;
        if (full) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
                uint4 w;
                __half2 h0 = __floats2half2_rn(v[i], v[i + 1]);
                __half2 h1 = __floats2half2_rn(v[i + 2], v[i + 3]);
                __half2 h2 = __floats2half2_rn(v[i + 4], v[i + 5]);
                __half2 h3 = __floats2half2_rn(v[i + 6], v[i + 7]);
                w.x = *reinterpret_cast<uint32_t*>(&h0);
                w.y = *reinterpret_cast<uint32_t*>(&h1);
                w.z = *reinterpret_cast<uint32_t*>(&h2);
                w.w = *reinterpret_cast<uint32_t*>(&h3);
                *reinterpret_cast<uint4*>(dst + i) = w;
            }
        } else {
            for (int i = 0; i < 32 && n0 + i < ncols; ++i) dst[i] = __float2half_rn(v[i]);
        }
    }
}

// Partial tiles are fragment-major: float4 index (col/4) * 128 + row, so that a warp's 32 rows
// touch 512 contiguous bytes.
template <int TN>
__device__ __forceinline__ float* frag_ptr(float* tile_base, int col0, int i, int row) {
    return tile_base + ((static_cast<int64_t>((col0 + i) >> 2) * kTileM) + row) * 4;
}

// Calls f(chunk, v) for every 32-column chunk of this thread's accumulator row, in order. Two
// chunks are read per TMEM round trip (two loads, one wait): the epilogue is bound by these round
// trips, not by the arithmetic between them.
template <int kChunks, typename F>
__device__ __forceinline__ void for_each_chunk(uint32_t t_acc, F&& f, int first_pair = 0) {
    static_assert(kChunks % 2 == 0, "chunks are read in pairs");
    constexpr int kPairs = kChunks / 2;
#pragma unroll 1
    for (int i = 0; i < kPairs; ++i) {
        const int ch = 2 * (first_pair + i < kPairs ? first_pair + i : first_pair + i - kPairs);
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(t_acc + ch * 32, r0);
        tmem_ld_32x32b_x32(t_acc + (ch + 1) * 32, r1);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = as_f(r0[i]);
        f(ch, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = as_f(r1[i]);
        f(ch + 1, v);
    }
}

// Writes this thread's accumulator row of a complete tile (16-bit output, one group in the output)
// with TMA tile stores: each epilogue warp stages its 32 rows x 64 columns in `ring` (128-byte rows,
// 128-byte swizzled, so that the 16-byte writes of a warp hit distinct banks) and one lane stores
// the box. Full-line writes replace the per-row 16-byte writes of store_out, whose 32 rows per warp
// instruction cost one L2 request each. The tensor map clips rows and columns outside C. `ring`
// is the dedicated epilogue buffer of a one-CTA kernel, or for a CTA pair the operand ring, which
// is idle only during a CTA's last segment. The warp waits until its boxes have been read out of
// shared memory, so the buffer is free again on return.
template <int OP, int TN>
__device__ void store_tile_tma(const KernelParams& P, const EpiCtx& e, uint32_t t_acc,
                               uint32_t ring, int quarter, int lane) {
    constexpr int kSlabs = TN / 64;
    const int64_t ncols = P.plan.gemm_n;
    const bool bf16 = P.c_dtype == SK_BF16;
    const int32_t y0 = static_cast<int32_t>(e.out_row - lane);   // the warp's first row
    if constexpr (OP == kOpFpropRow) {
        // The shifted-row fprop's staging buffer is its own: the previous tile's store has to be
        // out of it before it is written again (waited here, not after each store).
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
    }
#pragma unroll 1
    for (int sl = 0; sl < kSlabs; ++sl) {
        uint32_t r[2][32];
        tmem_ld_32x32b_x32(t_acc + sl * 64, r[0]);
        tmem_ld_32x32b_x32(t_acc + sl * 64 + 32, r[1]);
        tmem_ld_wait();
        uint32_t packed[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float a = as_f(r[h][i]), b = as_f(r[h][i + 1]);
                if constexpr (OP == kOpFp8) {
                    const int64_t n = e.n_base + sl * 64 + h * 32 + i;
                    a *= e.row_scale * (n < ncols ? (P.sb ? __ldg(P.sb + n) : 1.0f) : 0.0f);
                    b *= e.row_scale * (n + 1 < ncols ? (P.sb ? __ldg(P.sb + n + 1) : 1.0f) : 0.0f);
                }
                uint32_t w;
                if (bf16) {
                    __nv_bfloat162 x = __floats2bfloat162_rn(a, b);
                    w = *reinterpret_cast<uint32_t*>(&x);
                } else {
                    __half2 x = __floats2half2_rn(a, b);
                    w = *reinterpret_cast<uint32_t*>(&x);
                }
                packed[h * 16 + i / 2] = w;
            }
        }
        const uint32_t buf = ring + static_cast<uint32_t>((quarter * kSlabs + sl) * 4096);
        const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u)) << 4),
                         packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if constexpr (OP == kOpFpropRow) {
            // The warp's 32 rows: positions (quarter & 1) * 32 ... of output row 2*mt + quarter / 2
            // (rows counted per image over ho_pad); C is [N][Ho][Wo][64] and the map clips
            // positions past Wo. A padding row (past Ho) or a box wholly past Wo is not stored.
            const uint32_t hp = static_cast<uint32_t>(P.conv.ho_pad);
            const uint32_t t0 = 2u * static_cast<uint32_t>(e.mt);
            const uint32_t n_img = t0 / hp;
            const int32_t ho = static_cast<int32_t>(t0 - n_img * hp) + (quarter >> 1);
            const int32_t wo0 = (quarter & 1) * 32;
            if (lane == 0 && ho < P.conv.ho && wo0 < P.conv.rows.vw)
                tma_store_4d(&P.tmap_c, buf, 0, wo0, ho, static_cast<int32_t>(n_img));
        } else {
            if (lane == 0)
                tma_store_2d(&P.tmap_c, buf, static_cast<int32_t>(e.n_base + sl * 64), y0);
        }
    }
    if (lane == 0) {
        bulk_commit_group();
        if constexpr (OP != kOpFpropRow) bulk_wait_group_read0();
    }
    __syncwarp();
}

// Owner's fold of its senders' partial tiles (linear, or the last tree round), staged through the
// operand ring with bulk copies of 64 KB units, kFoldBufs of them in flight; the running sum stays
// in the owner's TMEM accumulator. Per element the additions run in sender order, so the result
// does not depend on timing. Only the owner segment, always a CTA's last, takes this path: by then
// every stage of the ring has been consumed.
template <int OP, int TN, int CG, int ST, typename SenderFn>
__device__ void staged_fold(const KernelParams& P, int64_t cta, const sk_segment_t& seg,
                            const EpiCtx& e, uint32_t t_acc, int ethread, int64_t ns,
                            SenderFn sender, uint32_t ring, uint32_t fold_bars) {
    using C = Cfg<OP, TN, CG, ST>;
    constexpr int kChunks = TN / 32;
    constexpr int kUnitsPerSender = kChunks / C::kFoldUnitChunks;
    const int64_t units = ns * kUnitsPerSender;   // sender-major
    auto issue = [&](int64_t u) {
        const int64_t i = u / kUnitsPerSender, h = u - i * kUnitsPerSender;
        const int64_t slot = partial_slot(P.plan, seg.tile, seg.first_cta, sender(i));
        const uint32_t buf = static_cast<uint32_t>(u % C::kFoldBufs);
        const uint32_t bar = fold_bars + buf * 8;
        if (slot < 0 || slot >= P.plan.partial_slots) {   // never expected: record and skip
            record_error(kErrBounds, cta, seg.tile, slot);
            return;
        }
        const float* src = P.partials + (slot * CG + e.half) * static_cast<int64_t>(kTileM * TN) +
                           h * (kTileM * 32 * C::kFoldUnitChunks);
        mbar_arrive_expect_tx(bar, C::kFoldUnitBytes);
        bulk_copy_g2s(ring + buf * C::kFoldUnitBytes, src, C::kFoldUnitBytes, bar);
    };
    if (ethread == 0) {
        fence_proxy_async_global();   // the acquired partials are read by the async proxy
        for (int64_t u = 0; u < units && u < C::kFoldBufs; ++u) issue(u);
    }
    const uint8_t* ring_ptr = nullptr;
    asm volatile("cvta.shared.u64 %0, %1;" : "=l"(ring_ptr) : "l"(static_cast<uint64_t>(ring)));
    bool ok = true;
    for (int64_t u = 0; u < units; ++u) {
        const int64_t h = u % kUnitsPerSender;
        const uint32_t buf = static_cast<uint32_t>(u % C::kFoldBufs);
        const uint32_t parity = static_cast<uint32_t>((u / C::kFoldBufs) & 1);
        if (ok && !mbar_wait(fold_bars + buf * 8, parity, P.mbar_timeout_ns)) {
            record_error(kErrPipeline, cta, seg.tile, 4);
            ok = false;
        }
        const float4* src = reinterpret_cast<const float4*>(ring_ptr + buf * C::kFoldUnitBytes);
#pragma unroll 1
        for (int c = 0; c < C::kFoldUnitChunks; ++c) {
            const int ch = static_cast<int>(h) * C::kFoldUnitChunks + c;
            uint32_t r[32];
            tmem_ld_32x32b_x32(t_acc + ch * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = src[(c * 8 + q) * kTileM + e.row];
                r[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) + x.x);
                r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + x.y);
                r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + x.z);
                r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + x.w);
            }
            tmem_st_32x32b_x32(t_acc + ch * 32, r);
        }
        tmem_st_wait();
        named_bar_sync(kEpiBarrier, kEpiThreads);   // buffer `buf` may be refilled
        if (ethread == 0 && ok && u + C::kFoldBufs < units) issue(u + C::kFoldBufs);
    }
    if (P.c_tma) {   // the owner segment is its CTA's last, and the fold has left the ring
        store_tile_tma<OP, TN>(P, e, t_acc, C::kEpiStageBytes ? ring + C::kRingBytes : ring,
                               e.row >> 5, e.row & 31);
        return;
    }
    for_each_chunk<kChunks>(t_acc, [&](int ch, float (&v)[32]) { store_out<OP>(P, e, ch * 32, v); });
}

template <int OP, int TN, int CG, int ST>
__device__ void epilogue_segment(const KernelParams& P, int64_t cta, const sk_segment_t& seg,
                                 const EpiCtx& e, uint32_t t_acc, int ethread, uint32_t ring,
                                 uint32_t fold_bars, bool last) {
    const sk_plan_t& plan = P.plan;
    constexpr int kChunks = TN / 32;
    const int red = static_cast<int>(plan.reduction);

    if (seg.kind == SK_SEG_FULL) {
        using C = Cfg<OP, TN, CG, ST>;
        if (P.c_tma && (C::kEpiStageBytes > 0 || last)) {
            store_tile_tma<OP, TN>(P, e, t_acc, C::kEpiStageBytes ? ring + C::kRingBytes : ring,
                                   e.row >> 5, e.row & 31);
            return;
        }
        for_each_chunk<kChunks>(t_acc,
                                [&](int ch, float (&v)[32]) { store_out<OP>(P, e, ch * 32, v); });
        return;
    }
    // The contributors of a tile add into the same words at about the same time; each starts at
    // its own pair of 32-column chunks (by CTA id), so that at any moment they spread over the
    // tile's columns instead of queueing on the same L2 lines.
    const int first_pair = static_cast<int>(cta % (kChunks / 2));
    if (red == SK_ATOMIC) {
        // tcgen05.ld is warp-collective (.sync.aligned): every lane loads, and only the lanes of
        // rows inside the output add.
        if constexpr (is_wgrad_row(OP)) {
            for_each_chunk<kChunks>(t_acc, [&](int ch, float (&v)[32]) {
                if (!e.row_ok) return;
                const int64_t off = wgrow_col_offset(P.conv, P.ldc, ch * 32);
                if (off < 0) return;
                float* dst = static_cast<float*>(P.c) + e.out_row + off;
#pragma unroll
                for (int i = 0; i < 32; ++i) red_add_f32(dst + i * P.ldc, v[i]);
            }, first_pair);
            return;
        }
        for_each_chunk<kChunks>(t_acc, [&](int ch, float (&v)[32]) {
            if (!e.row_ok) return;
            const int64_t n0 = e.n_base + ch * 32;
            float* dst = static_cast<float*>(P.c) + e.out_row * P.ldc + n0;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                if (n0 + i + 4 <= e.n_end) {
                    red_add_v4(dst + i, v[i], v[i + 1], v[i + 2], v[i + 3]);
                } else {
                    for (int j = 0; j < 4; ++j)
                        if (n0 + i + j < e.n_end) red_add_f32(dst + i + j, v[i + j]);
                }
            }
        }, first_pair);
        return;
    }
    if (red == SK_WORKSPACE) {
        float* base = P.scratch + (seg.tile * CG + e.half) * static_cast<int64_t>(kTileM * TN);
        for_each_chunk<kChunks>(t_acc, [&](int ch, float (&v)[32]) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                red_add_v4(frag_ptr<TN>(base, ch * 32, i, e.row), v[i], v[i + 1], v[i + 2],
                           v[i + 3]);
        }, first_pair);
        return;
    }

    // linear / tree. Every contributor's partial has its own slot; this CTA's flag counts the
    // partials it has published.
    const int64_t my_slot = partial_slot(plan, seg.tile, seg.first_cta, seg.index);
    const bool slot_ok = my_slot >= 0 && my_slot < plan.partial_slots;
    float* own = P.partials + (my_slot * CG + e.half) * static_cast<int64_t>(kTileM * TN);
    if (P.spread) {
        // Spread fold: hand the partial on now; the additions, a share of the tile for every
        // contributor, follow in spread_fold once the CTA's last segment is out.
        if (!slot_ok) {   // never expected: record and skip the stores
            if (ethread == 0) record_error(kErrBounds, cta, seg.tile, my_slot);
            return;
        }
        // Rows outside the output (a tile's padding rows) are not stored: the folders add
        // whatever their slots hold there, and those sums are never written out.
        for_each_chunk<kChunks>(t_acc, [&](int ch, float (&v)[32]) {
            if (!e.row_ok) return;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                __stcg(reinterpret_cast<float4*>(frag_ptr<TN>(own, ch * 32, i, e.row)),
                       make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        });
        // The barrier orders every epilogue thread's stores before the releases below, which make
        // them visible (cumulatively) to a CTA that acquires the flag or the tile's arrival
        // counter (control block word 1 + tile * CG + half), which the folders poll; the folders
        // read the partials with bulk copies (the async proxy).
        fence_proxy_async_global();
        named_bar_sync(kEpiBarrier, kEpiThreads);
        if (ethread == 0) {
            st_release_gpu(P.flags + cta * CG + e.half, publication(plan, cta, seg.tile));
            red_release_gpu_add(P.control + 1 + seg.tile * CG + e.half, 1u);
        }
        return;
    }

    // Owner fold: the contributor indices this one receives from, in fold order. Linear: the
    // owner takes 1, 2, ..., n-1. Tree: at most one sender per round.
    int32_t tree[32];
    int64_t ns = 0;
    const bool lin = red == SK_LINEAR;
    if (lin) {
        ns = seg.index == 0 ? seg.n_contrib - 1 : 0;
    } else {
        for_each_tree_sender(seg.index, seg.n_contrib, plan.tree_rounds, [&](int64_t j) {
            if (ns < 32) tree[ns++] = static_cast<int32_t>(j);
        });
    }
    auto sender = [&](int64_t i) -> int64_t { return lin ? i + 1 : tree[i]; };
    if (ns > 0) {
        // All senders' flags polled at once by the epilogue threads, one deadline for all: a lost
        // hand-off costs at most flag_timeout_ns, however many senders the segment has.
        const int64_t miss = wait_flags_all(P.flags, CG, e.half, ns, ethread, P.flag_timeout_ns,
                                            [&](int64_t k, int64_t& c2, uint32_t& need) {
                                                c2 = seg.first_cta + sender(k);
                                                need = publication(plan, c2, seg.tile);
                                            });
        if (miss != -1 && ethread == 0) record_error(kErrFlagWait, cta, seg.tile, miss);
    }

    if (seg.kind == SK_SEG_OWNER && ns > 0) {
        staged_fold<OP, TN, CG, ST>(P, cta, seg, e, t_acc, ethread, ns, sender, ring, fold_bars);
        return;
    }

    bool publish = seg.kind == SK_SEG_PEER;
    if (publish && !slot_ok) {   // never expected: record and skip the stores
        if (ethread == 0) record_error(kErrBounds, cta, seg.tile, -2);
        publish = false;
    }
    for_each_chunk<kChunks>(t_acc, [&](int ch, float (&v)[32]) {
        for (int64_t s = 0; s < ns; ++s) {
            const float* src =
                P.partials + (partial_slot(plan, seg.tile, seg.first_cta, sender(s)) * CG + e.half) *
                                 static_cast<int64_t>(kTileM * TN);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 q = __ldcg(reinterpret_cast<const float4*>(
                    frag_ptr<TN>(const_cast<float*>(src), ch * 32, i, e.row)));
                v[i] += q.x;
                v[i + 1] += q.y;
                v[i + 2] += q.z;
                v[i + 3] += q.w;
            }
        }
        if (publish) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                __stcg(reinterpret_cast<float4*>(frag_ptr<TN>(own, ch * 32, i, e.row)),
                       make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        } else {
            store_out<OP>(P, e, ch * 32, v);
        }
    });
    if (publish) {
        fence_proxy_async_global();   // a receiver may read this partial with bulk copies
        __threadfence();
        named_bar_sync(kEpiBarrier, kEpiThreads);
        if (ethread == 0)
            st_release_gpu(P.flags + cta * CG + e.half, publication(plan, cta, seg.tile));
    }
}

// A shared tile whose additions this CTA takes part in under the spread fold.
struct PendingFold {
    int64_t tile, first, n, index;
};

// Spread fold of a shared tile (linear or tree): wait until every contributor has handed its partial
// on, then add up this CTA's share of the tile's elements from all the partials, in the
// reduction's own order (linear: contributor 0, then 1, 2, ...; tree: the index-based pairwise
// rounds, kept as a binary counter of partial sums), and store them. The sums are the owner fold's,
// bit for bit. The tile's F = 128 * TN / 4 float4s (fragment-major, per 128-row half) are split
// evenly among its "folders": the contributors whose range lies in this one shared tile, or all of
// them when none does (two contributors that each share a second tile); a contributor that shares
// two tiles then folds none of the first. A share is contiguous in every slot, and a tile's slots
// are consecutive (partial_slot(tile, first, j) = slot 0 + j): all threads copy the share's slices
// of the n partials into the idle operand ring with coalesced loads (several in flight each), in
// chunks that fit half of it, then every thread adds up its elements there.
template <int OP, int TN, int CG, int ST>
__device__ void spread_fold(const KernelParams& P, int64_t cta, const PendingFold& pd, int ethread,
                            int64_t half, uint32_t ring, uint32_t fold_bar, uint32_t& fold_phase) {
    using C = Cfg<OP, TN, CG, ST>;
    const sk_plan_t& plan = P.plan;
    constexpr int kF4 = kTileM * TN / 4;
    constexpr uint32_t kBufBytes = (C::kRingBytes / 2) & ~15u;
    const int64_t n = pd.n;
    // Folders: the contributors with a single shared tile. Only the first contributor (if this is
    // its second shared tile) and the last (if its range runs on into a later shared tile) can
    // share another; the others lie inside this tile.
    auto shares_two = [&](int64_t j) {
        if (plan.mode == SK_SPLITK) return false;
        const int64_t c2 = pd.first + j;
        if (j == 0) return publication(plan, c2, pd.tile) == 2;
        if (j + 1 < n) return false;
        const int64_t end = sk_end(plan, c2);
        if (end - udiv31(end, plan.iters_per_tile) * plan.iters_per_tile == 0) return false;
        int64_t f2, n2;
        tile_contributors(plan, udiv31(end - 1, plan.iters_per_tile), f2, n2);
        return udiv31(end - 1, plan.iters_per_tile) != pd.tile && n2 > 1;
    };
    const bool skip0 = shares_two(0), skip1 = n > 1 && shares_two(n - 1);
    int64_t nfold = n - (skip0 ? 1 : 0) - (skip1 ? 1 : 0), me = pd.index - (skip0 ? 1 : 0);
    if ((pd.index == 0 && skip0) || (pd.index == n - 1 && skip1)) me = -1;
    if (nfold <= 0) {   // everyone folds
        nfold = n;
        me = pd.index;
    }
    if (me < 0) return;   // this CTA's part of the tile is its partial only
    const int64_t stride = static_cast<int64_t>(CG) * kTileM * TN;   // floats between slots
    const float* base = P.partials + (partial_slot(plan, pd.tile, pd.first, 0) * CG + half) *
                                         static_cast<int64_t>(kTileM * TN);
    const int64_t b = me * kF4 / nfold, e = (me + 1) * kF4 / nfold;
    const int64_t cap = imax(1, static_cast<int64_t>(kBufBytes) / (16 * n));   // float4s per chunk
    // A share that fits one chunk is gathered in arrival order: the lanes of the first epilogue
    // warp poll the contributors' flags (each contributor's flag counts the partials it has
    // published) and copy a contributor's slice as soon as its partial is out, so the copies
    // overlap the wait for the last ones; the additions below still run in contributor order.
    // Otherwise one thread polls the tile's arrival counter until all n contributors have counted
    // their partials, and the slices follow chunk by chunk. Either way the verdict goes to all
    // epilogue threads through a barrier reduction.
    const bool early = e - b <= cap;
    bool arrived = true;
    if (early) {
        if (ethread < 32) {
            const uint32_t bytes = static_cast<uint32_t>((e - b) * 16);
            if (ethread == 0) mbar_arrive_expect_tx(fold_bar, static_cast<uint32_t>(n) * bytes);
            __syncwarp();
            // this lane's contributors: j = lane, lane + 32, ... (a bit per pending one)
            uint32_t pending = 0;
            for (int64_t j = ethread, q = 0; j < n; j += 32, ++q) pending |= 1u << q;
            uint64_t t0 = 0;
            while (pending != 0) {
                // The flags of this lane's pending contributors, read together (relaxed loads, not
                // one acquire after another); one acquire fence then orders every partial seen out
                // before the copies that read it.
                uint32_t ready = 0;
                for (int64_t j = ethread, q = 0; j < n; j += 32, ++q) {
                    if (!(pending & (1u << q))) continue;
                    const int64_t c2 = pd.first + j;
                    if (ld_relaxed_gpu(P.flags + c2 * CG + half) >= publication(plan, c2, pd.tile))
                        ready |= 1u << q;
                }
                if (ready != 0) {
                    fence_acq_rel_gpu();
                    fence_proxy_async_global();   // the acquired partials are read by the async proxy
                    for (int64_t j = ethread, q = 0; j < n; j += 32, ++q)
                        if (ready & (1u << q))
                            bulk_copy_g2s(ring + static_cast<uint32_t>(j) * bytes,
                                          base + j * stride + b * 4, bytes, fold_bar);
                    pending &= ~ready;
                }
                if (pending == 0) break;
                if (t0 == 0) t0 = globaltimer_ns();
                if (globaltimer_ns() - t0 > P.flag_timeout_ns) {
                    arrived = false;
                    break;
                }
                __nanosleep(64);
            }
        }
    } else if (ethread == 0) {
        uint64_t t0 = 0;
        arrived = wait_flag(P.control + 1 + pd.tile * CG + half, static_cast<uint32_t>(n), t0,
                            P.flag_timeout_ns);
    }
    if (!named_bar_and(kEpiBarrierWait, kEpiThreadsWait, arrived)) {
        if (ethread == 0) record_error(kErrFlagWait, cta, pd.tile, -3);
        return;
    }
    __threadfence();
    int64_t g, mt, nt;
    tile_coords(plan, pd.tile, g, mt, nt);
    const OutSpec o{P.c, P.ldc, P.c_dtype, OP, P.sa, P.sb, P.scale,
                    OP == kOpFp8 ? (P.sa != nullptr ? 1 : 2) : 0, &P.conv};
    const bool lin = plan.reduction == SK_LINEAR;
    uint8_t* ring_ptr = nullptr;
    asm volatile("cvta.shared.u64 %0, %1;" : "=l"(ring_ptr) : "l"(static_cast<uint64_t>(ring)));
    float4* sbuf = reinterpret_cast<float4*>(ring_ptr);
    auto add4 = [](const float4& x, const float4& y) {
        return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
    };
    for (int64_t c0 = b; c0 < e; c0 += cap) {
        const int64_t len = imin(cap, e - c0);
        const uint32_t bytes = static_cast<uint32_t>(len * 16);
        // The chunk's slices of all n partials, slot-major, each one contiguous run of `bytes`:
        // one bulk copy per partial, issued by the lanes of the first epilogue warp and counted on
        // the fold barrier, whose single arrival (lane 0) expects them all.
        if (ethread < 32 && !early) {
            fence_proxy_async_global();   // the acquired partials are read by the async proxy
            if (ethread == 0) mbar_arrive_expect_tx(fold_bar, static_cast<uint32_t>(n) * bytes);
            __syncwarp();
            for (int64_t j = ethread; j < n; j += 32)
                bulk_copy_g2s(ring + static_cast<uint32_t>(j) * bytes, base + j * stride + c0 * 4,
                              bytes, fold_bar);
        }
        const bool landed = mbar_wait(fold_bar, fold_phase, P.mbar_timeout_ns);
        fold_phase ^= 1u;
        if (!named_bar_and(kEpiBarrierWait, kEpiThreadsWait, landed)) {
            // Never expected (a copy outstanding for the barrier's whole time limit): the error is
            // recorded for the host and the CTA stops folding.
            if (ethread == 0) record_error(kErrPipeline, cta, pd.tile, 5);
            return;
        }
        for (int64_t i = ethread; i < len; i += kEpiThreads) {
            auto part = [&](int64_t j) { return sbuf[j * len + i]; };
            float4 v;
            if (lin) {
                // The same additions in the same order; four slices are read ahead so that the
                // shared-memory latency is not paid on every one.
                v = part(0);
                int64_t j = 1;
                for (; j + 4 <= n; j += 4) {
                    const float4 x0 = part(j), x1 = part(j + 1), x2 = part(j + 2), x3 = part(j + 3);
                    v = add4(v, x0);
                    v = add4(v, x1);
                    v = add4(v, x2);
                    v = add4(v, x3);
                }
                for (; j < n; ++j) v = add4(v, part(j));
            } else {
                // Tree: the pending block sums of the rounds form a binary counter. Contributor
                // j's partial is added (on the right) to the block held at every level where j
                // has a set bit, lowest first, and the result is held at the first clear bit; at
                // the end the blocks of n's set bits are added right (low level) to left. acc[L]
                // is a block of 2^L partials; n < 256 (the host takes the owner fold otherwise).
                float4 acc[8];
                for (int64_t j = 0; j < n; ++j) {
                    float4 x = part(j);
#pragma unroll
                    for (int L = 0; L < 8; ++L) {
                        if ((j >> L) & 1) {
                            x = add4(acc[L], x);
                        } else {
                            acc[L] = x;
                            break;
                        }
                    }
                }
                bool have = false;
#pragma unroll
                for (int L = 0; L < 8; ++L) {
                    if ((n >> L) & 1) {
                        v = have ? add4(acc[L], v) : acc[L];
                        have = true;
                    }
                }
            }
            const int64_t idx = c0 + i;
            const int row = static_cast<int>(idx % kTileM), q4 = static_cast<int>(idx / kTileM);
            const int64_t m = mt * (kTileM * CG) + half * kTileM + row;
            const int64_t n0 = nt * TN + q4 * 4;
            if (m >= plan.gemm_m || n0 >= plan.gemm_n) continue;
            float w[4] = {v.x, v.y, v.z, v.w};
            store4_out(plan, o, g, m, n0, w);
        }
        named_bar_sync(kEpiBarrier, kEpiThreads);   // the buffer is free again
    }
}

// Block-scaled fp8, one segment: for each K step (in the order the MMAs ran it) wait for its fresh
// partial in TMEM, load it and free its buffer, scale every row by sa[m][kb] * sb[n-block][kb] and
// add it to the running sum, which each thread keeps for its row in registers; at the segment's
// end the sum is written to the TMEM columns after the partial buffers and goes through the usual
// fixups. False if a wait gave up.
template <int TN, int CG, int ST>
__device__ bool promote_segment(const KernelParams& P, int64_t cta, const sk_segment_t& seg, bool dp,
                                int64_t& tau, int64_t& nstep, int64_t seg_count, uint32_t tmem_base,
                                uint32_t bars,
                                volatile SmemCtl* ctl, uint32_t ring, int warp, int ethread,
                                bool last, uint32_t rank) {
    constexpr int OP = kOpFp8Block;
    using C = Cfg<OP, TN, CG, ST>;
    const sk_plan_t& plan = P.plan;
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int64_t g, mt, nt;
    tile_coords(plan, seg.tile, g, mt, nt);
    EpiCtx e;
    e.row = row;
    e.half = static_cast<int64_t>(rank);   // a pair's CTA holds rows rank*128 .. of the tile
    e.mt = mt;
    const int64_t m = mt * C::kTileMAll + static_cast<int64_t>(rank) * kTileM + row;
    e.row_ok = m < plan.gemm_m;
    e.out_row = m;
    e.n_base = nt * TN;
    e.n_end = plan.gemm_n;
    e.row_scale = 1.0f;
    const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
    const int64_t len = seg.k_end - seg.k_begin;
    const int64_t rot = segment_rotation(plan, dp, seg, tau);
    const float* sa_row = (P.bsa != nullptr && e.row_ok) ? P.bsa + m * P.nka : nullptr;
    const float* sb_blk = P.bsb != nullptr ? P.bsb + (e.n_base / P.gnb) * P.nkb : nullptr;
    // Scale ring: slot d of this thread holds the (A, B) block scales of step j = d (mod D).
    constexpr int D = C::kScaleAhead;
    static_assert((D & (D - 1)) == 0, "the scale ring's depth is a power of two");
    const uint32_t scl = ring + C::kRingBytes + C::kEpiStageBytes + static_cast<uint32_t>(ethread) * 8u;
    // Fetch cursor: the K step kf of the next step to fetch (the MMAs' rotated order) and its A / B
    // block index and offset inside the block, advanced by one step at a time (the block sizes are
    // whole K steps), so that no division is on the per-step path.
    const int32_t ga = P.gka / C::TK, gb = P.gkb / C::TK;
    int64_t kf = seg.k_begin + rot, qa = kf / ga, qb = kf / gb;
    int32_t ra = static_cast<int32_t>(kf - qa * ga), rb = static_cast<int32_t>(kf - qb * gb);
    int64_t jf = 0;
    auto fetch = [&]() {   // one commit group per step, empty past the segment's end
        if (jf < len) {
            const uint32_t slot = scl + static_cast<uint32_t>(jf & (D - 1)) * (kEpiThreads * 8u);
            if (sa_row) cp_async_4(slot, sa_row + qa);
            if (sb_blk) cp_async_4(slot + 4, sb_blk + qb);
            if (++kf == seg.k_end) {   // the rotation wraps to the segment's start
                kf = seg.k_begin;
                qa = kf / ga;
                qb = kf / gb;
                ra = static_cast<int32_t>(kf - qa * ga);
                rb = static_cast<int32_t>(kf - qb * gb);
            } else {
                if (++ra == ga) { ra = 0; ++qa; }
                if (++rb == gb) { rb = 0; ++qb; }
            }
        }
        ++jf;
        cp_async_commit();
    };
    for (int d = 0; d < D; ++d) fetch();
    // Partial buffer for this CTA's nstep-th K step, and the ring stage whose MMA commit marks that
    // step's partial complete (and the phase of that commit), advanced by counting. The commit of
    // a stage cannot complete a second phase before the epilogue has seen the first: the MMAs of
    // the stage's next use wait for a partial buffer that the epilogue frees only after this step.
    uint32_t acc = static_cast<uint32_t>(nstep % C::kAccBufs);
    uint32_t rs = static_cast<uint32_t>(nstep % C::kStages);
    uint32_t rs_phase = static_cast<uint32_t>((nstep / C::kStages) & 1);
    float run[TN];   // this thread's row of the running sum
#pragma unroll
    for (int i = 0; i < TN; ++i) run[i] = 0.0f;
    // A pair's partial-buffer barriers live in the even CTA, whose thread issues the MMAs.
    auto release = [&](uint32_t bar) {
        if (CG == 2 && rank != 0)
            mbar_arrive_cluster(mapa_shared(bar, 0));
        else
            mbar_arrive(bar);
    };
    // Each warp waits for the partials on its own (lane 0, bounded; the verdict is shuffled to the
    // warp), so that no barrier of all four warps is on the per-step path; after a failed wait a
    // warp only runs the loop out. The four verdicts meet at one barrier after the loop, so every
    // warp takes the same path into the fixups.
    uint32_t ok = 1;
    for (int64_t j = 0; j < len; ++j) {
        const uint32_t done = bars + (C::kStages + rs) * 8;   // the stage's MMA commit
        const uint32_t tempty = bars + (C::kBarTempty + acc) * 8;
        if (ok) {
            uint32_t v = 0;
            if (lane == 0) {
                v = (mbar_wait(done, rs_phase, P.mbar_timeout_ns) && !ctl->abort) ? 1u : 0u;
                if (!v) {
                    record_error(kErrPipeline, cta, seg.tile, 3);
                    ctl->abort = 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, v, 0);
        }
        if (!ok) {
            fetch();
            continue;
        }
        tc_fence_after();
        cp_async_wait<D - 1>();   // this step's group (the oldest in flight) has landed
        const uint32_t slot = scl + static_cast<uint32_t>(j & (D - 1)) * (kEpiThreads * 8u);
        float s = e.row_ok ? 1.0f : 0.0f;
        if (sa_row) s *= ld_shared_f32(slot);
        if (sb_blk) s *= ld_shared_f32(slot + 4);
        const uint32_t t_part = tmem_base + lanes + acc * TN;
        // Two 32-column chunks per TMEM round trip, each scaled into the running sum.
#pragma unroll
        for (int c = 0; c < TN / 32; c += 2) {
            uint32_t p0[32], p1[32];
            tmem_ld_32x32b_x32(t_part + c * 32, p0);
            tmem_ld_32x32b_x32(t_part + (c + 1) * 32, p1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                run[c * 32 + i] = fmaf(s, as_f(p0[i]), run[c * 32 + i]);
                run[(c + 1) * 32 + i] = fmaf(s, as_f(p1[i]), run[(c + 1) * 32 + i]);
            }
        }
        fetch();   // step j + D, into the slot just read (its value is consumed above)
        if (j + 1 < len) {   // the last step's buffer is kept: it takes the segment's sum below
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release(tempty);
            ++nstep;
            if (++acc == C::kAccBufs) acc = 0;
            if (++rs == C::kStages) {
                rs = 0;
                rs_phase ^= 1u;
            }
        }
    }
    cp_async_wait_all();
    const int par = static_cast<int>(seg_count & 1);
    if (lane == 0) ctl->warp_ok[par][quarter] = ok;
    named_bar_sync(kEpiBarrier, kEpiThreads);
    // A slot of this parity is written again only after every warp has passed the next segment's
    // barrier, i.e. after all four have read it here.
    if (!(ctl->warp_ok[par][0] & ctl->warp_ok[par][1] & ctl->warp_ok[par][2] & ctl->warp_ok[par][3]))
        return false;
    // The segment's sum goes to the buffer of its last step, where the fixups and the stores read
    // it; then that buffer is released like the others.
    const uint32_t t_sum = tmem_base + lanes + acc * TN;
#pragma unroll
    for (int c = 0; c < TN / 32; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(run[c * 32 + i]);
        tmem_st_32x32b_x32(t_sum + c * 32, r);
    }
    tmem_st_wait();
    tc_fence_after();
    epilogue_segment<OP, TN, CG, ST>(P, cta, seg, e, t_sum, ethread, ring,
                                     bars + C::kBarFold * 8, last);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) release(bars + (C::kBarTempty + acc) * 8);
    ++nstep;
    return true;
}

template <int OP, int TN, int CG, int ST>
__device__ void run_epilogue(const KernelParams& P, int64_t cta, uint32_t ring, uint32_t bars,
                             uint32_t tmem_base, int warp, volatile SmemCtl* ctl, uint32_t rank) {
    using C = Cfg<OP, TN, CG, ST>;
    const sk_plan_t& plan = P.plan;
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int quarter = warp & 3;                 // TMEM lanes this warp may access
    const int row = quarter * 32 + lane;
    const int ethread = static_cast<int>(threadIdx.x) - 64;
    SegCursor cur;
    seg_init(plan, cta, cur);
    sk_segment_t seg;
    int64_t nseg = 0, tau = 0, nblk = 0;
    // Without a ticket the zeroing kernel may still be running: the epilogue's first write (output,
    // scratch, partials, flags or counters) comes after its writes. A chained launch has no such
    // predecessor (its previous kernel writes other pixels and no word it reads).
    if (!P.ticket && !(P.pdl_chain & 1)) grid_dependency_wait();
    // Spread fold: the shared tiles of this CTA (at most two), folded once all its segments are out.
    const bool spread = P.spread && (plan.reduction == SK_LINEAR || plan.reduction == SK_TREE);
    PendingFold pend[2];
    int npend = 0;
    bool aborted = false;
    auto note_shared = [&](const sk_segment_t& sg) {
        if (spread && sg.kind != SK_SEG_FULL && npend < 2)
            pend[npend++] = PendingFold{sg.tile, sg.first_cta, sg.n_contrib, sg.index};
    };
    while (true) {
        const bool dp = cur.dp_next >= 0;
        if (!seg_next(plan, cta, cur, seg)) break;
        if constexpr (OP == kOpFp8Block) {
            SegCursor ahead = cur;
            sk_segment_t next;
            const bool last = !seg_next(plan, cta, ahead, next);
            if (!promote_segment<TN, CG, ST>(P, cta, seg, dp, tau, nseg, nblk, tmem_base, bars, ctl,
                                             ring, warp, ethread, last, rank)) {
                aborted = true;
                break;
            }
            note_shared(seg);
            ++nblk;
            continue;
        }
        const uint32_t acc = static_cast<uint32_t>(nseg % C::kAccBufs);
        const uint32_t acc_phase = static_cast<uint32_t>((nseg / C::kAccBufs) & 1);
        const uint32_t tfull = bars + (C::kBarTfull + acc) * 8;
        const uint32_t tempty = bars + (C::kBarTempty + acc) * 8;
        // One thread waits (bounded) and the verdict goes to all 128 epilogue threads through a
        // named barrier, so that every epilogue warp takes the same path and no barrier below
        // can be left short of arrivals.
        if (ethread == 0) {
            const bool ready = mbar_wait(tfull, acc_phase, P.mbar_timeout_ns) && !ctl->abort;
            if (!ready) {
                record_error(kErrPipeline, cta, seg.tile, 3);
                ctl->abort = 1;
            }
            ctl->epi_ok[nseg & 1] = ready ? 1u : 0u;
        }
        named_bar_sync(kEpiBarrier, kEpiThreads);
        if (!ctl->epi_ok[nseg & 1]) {
            aborted = true;
            break;
        }
        tc_fence_after();
        int64_t g, mt, nt;
        tile_coords(plan, seg.tile, g, mt, nt);
        EpiCtx e;
        e.row = row;
        e.half = static_cast<int64_t>(rank);
        e.mt = mt;
        const int64_t m = mt * C::kTileMAll + static_cast<int64_t>(rank) * kTileM + row;
        e.row_ok = m < plan.gemm_m;
        if constexpr (OP == kOpFpropRow) {
            // Row (output row 2*mt + row / 64, position row % 64) of the image's rows counted over
            // ho_pad: an output pixel when the row is below Ho and the position below Wo (what
            // map_row gives, in 32-bit arithmetic: n * ho_pad * 64 < 2^31).
            const uint32_t hp = static_cast<uint32_t>(P.conv.ho_pad);
            const uint32_t t0 = 2u * static_cast<uint32_t>(mt);
            const uint32_t n_img = t0 / hp;
            const int32_t ho = static_cast<int32_t>(t0 - n_img * hp) + (row >> 6);
            const int32_t wo = row & 63;
            const int32_t Wo = P.conv.rows.vw;
            e.row_ok = ho < P.conv.ho && wo < Wo;
            e.out_row = e.row_ok ? (static_cast<int64_t>(n_img) * P.conv.ho + ho) * Wo + wo : 0;
            e.n_base = 0;
            e.n_end = plan.gemm_n;
        } else if constexpr (folds_groups_into_columns(OP)) {
            e.out_row = map_row(P.conv.rows, m);
            e.n_base = g * plan.gemm_n + nt * TN;
            e.n_end = (g + 1) * plan.gemm_n;
        } else if constexpr (is_wgrad_row(OP)) {
            // Row m = (tap row r, channel c) of group g: dW[(g*Kg + k)][r][s][c] at
            // out_row + k * ldc + s * Cg.
            const int64_t r = m >> 6, c = m & 63;
            e.out_row = e.row_ok ? (g * P.conv.Kg) * P.ldc + r * P.conv.S * P.conv.Cg + c : 0;
            e.n_base = 0;
            e.n_end = plan.gemm_n;
        } else {
            e.out_row = g * plan.gemm_m + m;
            e.n_base = nt * TN;
            e.n_end = plan.gemm_n;
        }
        e.row_scale = 1.0f;
        if constexpr (OP == kOpFp8)
            e.row_scale = e.row_ok ? (P.sa ? __ldg(P.sa + e.out_row) : P.scale) : 0.0f;
        const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * TN;
        SegCursor ahead = cur;
        sk_segment_t next;
        const bool last = !seg_next(plan, cta, ahead, next);
        if constexpr (C::kWgRow && CG == 1) {
            if (seg.kind != SK_SEG_FULL && plan.reduction == SK_ATOMIC && !last) {
                // A CTA whose range reaches into the next tile: the single accumulator goes to
                // registers at once (192 columns a thread) and is released before this segment's
                // additions, so that the next segment's MMAs start while they issue. (A CTA's last
                // segment keeps the chunked additions of epilogue_segment, whose starting chunk
                // differs from CTA to CTA: the contributors of a tile end together there. The
                // same early release before a spread fold's publication gained nothing: that
                // fold waits for the later segment's partial anyway.)
                uint32_t r[TN / 32][32];
#pragma unroll
                for (int c = 0; c < TN / 32; ++c) tmem_ld_32x32b_x32(t_acc + c * 32, r[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty);
                if (e.row_ok) {
#pragma unroll
                    for (int c = 0; c < TN / 32; ++c) {
                        const int64_t off = wgrow_col_offset(P.conv, P.ldc, c * 32);
                        if (off < 0) continue;
                        float* dst = static_cast<float*>(P.c) + e.out_row + off;
#pragma unroll
                        for (int i = 0; i < 32; ++i) red_add_f32(dst + i * P.ldc, as_f(r[c][i]));
                    }
                }
                ++nseg;
                continue;
            }
        }
        epilogue_segment<OP, TN, CG, ST>(P, cta, seg, e, t_acc, ethread, ring,
                                         bars + C::kBarFold * 8, last);
        note_shared(seg);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            // A pair's accumulator-empty barrier lives in the even CTA, whose thread issues the MMAs.
            if (CG == 2 && rank != 0)
                mbar_arrive_cluster(mapa_shared(tempty, 0));
            else
                mbar_arrive(tempty);
        }
        ++nseg;
    }
    // The fold barrier is free here: the owner fold, its other user, never runs in a spread plan.
    uint32_t fold_phase = 0;
    if (!aborted)
        for (int i = 0; i < npend; ++i)
            spread_fold<OP, TN, CG, ST>(P, cta, pend[i], ethread, static_cast<int64_t>(rank), ring,
                                        bars + C::kBarFold * 8, fold_phase);
    if constexpr (OP == kOpFpropRow) {   // the last tile store has read its staging buffer
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------------------------

template <int OP, int TN, int CG, int ST>
__global__ void __launch_bounds__(kThreads, Cfg<OP, TN, CG, ST>::kMinBlocks)
    sk_main_kernel(const __grid_constant__ KernelParams P) {
    using C = Cfg<OP, TN, CG, ST>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    static_assert(sizeof(SmemCtl) <= C::kCtlBytes, "control block");
    const uint32_t ring = smem_u32(smem);
    volatile SmemCtl* ctl =
        reinterpret_cast<volatile SmemCtl*>(smem + C::kRingBytes + C::kEpiStageBytes +
                                            C::kScaleBytes + C::kResBytes);
    const uint32_t bars = ring + C::kRingBytes + C::kEpiStageBytes + C::kScaleBytes +
                          C::kResBytes + C::kCtlBytes;
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const uint32_t ctl_addr = smem_u32(const_cast<SmemCtl*>(ctl));
    if (threadIdx.x == 96) {
        // Every role's first reads of the parameters miss this SM's constant cache, one after
        // another (the ticket flag before the prologue's barrier, the plan at each role's start):
        // one word of every 64-byte line of them, read here at once with fixed offsets, brings
        // them in while the prologue runs.
        constexpr int kLines = static_cast<int>((sizeof(KernelParams) + 63) / 64);
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(&P);
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < kLines; ++i) v ^= pw[i * 16];
        asm volatile("" ::"r"(v));
    }

    // One CTA without a ticket: the producer needs nothing of the prologue after the barriers'
    // initialisation (not the TMEM allocation, the pad rows of the shifted-row wgrad or a ticket;
    // its CTA id is the block index), so it starts its copies while the other warps finish it.
    const bool early = CG == 1 && !P.ticket;
    uint32_t ticket = 0;
    if (threadIdx.x == 0) {
        if (P.pdl_chain & 2) grid_launch_dependents();   // the next launch of the call may start
        tma_prefetch_desc(&P.tmap_a);
        tma_prefetch_desc(&P.tmap_b);
        // The allocation below overwrites this; whatever a previous kernel left in shared memory
        // can never be taken for a TMEM address.
        ctl->tmem_base = kTmemSentinel;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bars + s * 8, 1);                    // full: producer arrive + tx bytes
            mbar_init(bars + (C::kStages + s) * 8, 1);     // empty: MMA commit
        }
        for (int a = 0; a < C::kAccBars; ++a) {
            mbar_init(bars + (C::kBarTfull + a) * 8, 1);                          // accumulator full
            mbar_init(bars + (C::kBarTempty + a) * 8, CG * kEpiThreads / 32);     // ... empty
        }
        for (int f = 0; f < C::kFoldBufs; ++f)
            mbar_init(bars + (C::kBarFold + f) * 8, 1);   // owner's fold buffers
        mbar_init(bars + C::kBarRes * 8, 1);              // shifted-row fprop: filter loaded
        fence_mbarrier_init();
        ctl->abort = 0;
    }
    if (early && warp == 0) {
        // The arrival publishes the barriers and the sentinel to the other warps. The producer
        // drains its own copies if it stops early (run_producer), and meets the others only at
        // the CTA's last barrier.
        named_bar_arrive(kPrologueBar, kThreads);
        if (elect_one()) run_producer<OP, TN, CG, ST>(P, static_cast<int64_t>(blockIdx.x), ring, bars,
                                                      ctl, 0u);
        __syncwarp();
        tc_fence_before();
        __syncthreads();
        return;
    }
    // Barriers and the sentinel are in place (and, for a pair, both CTAs have started) before the
    // allocation writes the slot.
    if (early) {
        named_bar_sync(kPrologueBar, kThreads);
    } else {
        if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    }
    if (warp == 1) {
        tmem_alloc<CG>(ctl_addr + static_cast<uint32_t>(offsetof(SmemCtl, tmem_base)),
                       C::kTmemAlloc);
        tmem_relinquish<CG>();
    }
    if constexpr (C::kWgRow) {
        // The 16 rows after the dy rows of every stage, which the shifted reads of a stage's last
        // positions reach, hold zeros. No copy ever writes them (the fold, which reuses the ring,
        // comes after the CTA's last MMA), so every thread clears a part of them once; the fence
        // makes the stores visible to the tensor cores, and the barrier below orders them before
        // the first MMA.
        const uint32_t pad0 = RowLayout<CG, C::kPhases>(P.conv).dy_off +
                              (CG == 1 ? 1u : static_cast<uint32_t>(P.conv.stage_steps)) * 64u *
                                  C::kDyRowBytes;
        constexpr int kPadBytes = C::kDyPadRows * C::kDyRowBytes;
        const int first = early ? 32 : 0;   // the producer warp is already copying
        for (int i = static_cast<int>(threadIdx.x) - first; i < C::kStages * kPadBytes / 16;
             i += kThreads - first) {
            const int st = i / (kPadBytes / 16), b = i - st * (kPadBytes / 16);
            st_shared_v4(ring + st * C::kStageBytes + pad0 + b * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    // The launch may overlap the tail of the kernel that zeroes the flags, the control block (the
    // ticket and arrival counters), the scratch and, for the atomic reduction, the output (a
    // programmatic dependent launch): everything above touches only this CTA's shared memory, its
    // TMEM and the tensor maps. A launch without that dependency passes straight through the waits.
    if (P.ticket) {
        // Logical ids in start order: every thread waits for the zeroed counter first. A pair
        // takes one ticket, in its even CTA, and hands it to both (the barrier below publishes
        // the stores).
        grid_dependency_wait();
        if (threadIdx.x == 0 && rank == 0) {
            ticket = atomicAdd(P.control, 1u);
            if constexpr (CG == 2) {
                const uint32_t cta_off = ctl_addr + static_cast<uint32_t>(offsetof(SmemCtl, cta));
                st_shared_cluster_u64(mapa_shared(cta_off, 0), ticket);
                st_shared_cluster_u64(mapa_shared(cta_off, 1), ticket);
            } else {
                ctl->cta = static_cast<long long>(ticket);
            }
        }
    } else if (threadIdx.x == 0) {
        // No CTA waits on one that may not have started (no waits at all, or every CTA of the
        // grid resident at once): the block index, one per CTA pair (clusters of two consecutive
        // blocks). Only the epilogue writes zeroed words; its threads wait for them there.
        ctl->cta = static_cast<long long>(CG == 2 ? (blockIdx.x >> 1) : blockIdx.x);
    }
    tc_fence_before();
    if (early) {
        named_bar_sync(kPrologueBar2, kThreads - 32);
    } else {
        if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    }
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int64_t cta = early ? static_cast<int64_t>(blockIdx.x) : static_cast<int64_t>(ctl->cta);
    // Every thread reads the same slot, so the whole CTA takes this exit together. It is never
    // expected; it keeps a bad slot from ever reaching a TMEM access. A pair takes the verdict
    // of both its slots, so that both CTAs leave together.
    auto bad_slot = [](uint32_t t) {
        return t == kTmemSentinel || (t >> 16) != 0 || (t & 0xFFFFu) + C::kTmemAlloc > 512u;
    };
    // `freeable`: the columns this CTA was granted can be handed back on the way out. A pair frees
    // only when both slots are TMEM addresses, since its deallocation is issued by both CTAs.
    bool bad = bad_slot(tmem_base);
    bool freeable = !bad;
    if constexpr (CG == 2) {
        const uint32_t peer = ld_shared_cluster_u32(
            mapa_shared(ctl_addr + static_cast<uint32_t>(offsetof(SmemCtl, tmem_base)), rank ^ 1u));
        freeable = freeable && !bad_slot(peer);
        bad = bad || bad_slot(peer) || peer != tmem_base;
        cluster_sync();   // the peer's slot has been read before either CTA can leave
    }
    if (bad) {
        // Never expected. Nothing has touched TMEM yet; the columns are still released before the
        // CTA leaves, so that a later CTA's allocation on this SM is not left waiting for them.
        if (threadIdx.x == 32) {
            record_error(kErrBounds, cta, -1, static_cast<long long>(tmem_base));
            ctl->abort = 1;   // an early producer stops at its next wait and drains its copies
        }
        tc_fence_before();
        if constexpr (CG == 2) cluster_sync(); else __syncthreads();
        if (warp == 1 && freeable) {
            tc_fence_after();
            tmem_dealloc<CG>(tmem_base, C::kTmemAlloc);
        }
        return;
    }

    if (warp == 0) {   // not an early producer: that warp has left above
        if (elect_one()) run_producer<OP, TN, CG, ST>(P, cta, ring, bars, ctl, rank);
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 0 && elect_one()) run_mma<OP, TN, CG, ST>(P, cta, ring, bars, tmem_base, ctl);
        __syncwarp();
    } else {
        run_epilogue<OP, TN, CG, ST>(P, cta, ring, bars, tmem_base, warp, ctl, rank);
    }

    tc_fence_before();
    // A pair leaves together: no arrival or shared-memory access of one CTA can reach the other
    // after it has gone.
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, C::kTmemAlloc);
    }
}

// ---------------------------------------------------------------------------------------------
// Stage-2: fp32 scratch of the shared tiles -> output (scaled for fp8)
// ---------------------------------------------------------------------------------------------

constexpr int kStage2Threads = 256;

// Grid (shared-tile candidates, tile float4s / 256): one float4 of fp32 scratch per thread, read in
// the fragment-major order the fixup wrote it. A pair tile (CG = 2) is two such 128-row halves.
template <int TN, int CG>
__global__ void __launch_bounds__(kStage2Threads) sk_stage2_kernel(const __grid_constant__ Stage2Params P) {
    if (P.after_main) grid_dependency_wait();   // the scratch is complete once the main kernel is
    const sk_plan_t& plan = P.plan;
    const int64_t t = blockIdx.x;
    int64_t first, n;
    tile_contributors(plan, t, first, n);
    if (n <= 1) return;   // written directly by its only contributor
    int64_t g, mt, nt;
    tile_coords(plan, t, g, mt, nt);
    const int idx = static_cast<int>(blockIdx.y) * kStage2Threads + static_cast<int>(threadIdx.x);
    constexpr int kHalf = kTileM * TN / 4;   // float4s of one 128-row half
    const int half = idx / kHalf, r = idx - half * kHalf;
    const int q4 = r / kTileM, row = r - q4 * kTileM;
    const int64_t m = mt * (kTileM * CG) + half * kTileM + row;
    const int64_t n0 = nt * TN + q4 * 4;
    if (m >= plan.gemm_m || n0 >= plan.gemm_n) return;
    const float* base = P.scratch + t * static_cast<int64_t>(kTileM * CG * TN);
    const float4 q = __ldcs(reinterpret_cast<const float4*>(base + static_cast<int64_t>(idx) * 4));
    float v[4] = {q.x, q.y, q.z, q.w};
    const OutSpec o{P.c, P.ldc, P.c_dtype, P.op_kind, P.sa, P.sb, P.scale,
                    P.sa != nullptr ? 1 : (P.tensor_scaled ? 2 : 0), &P.conv};
    store4_out(plan, o, g, m, n0, v);
}

// ---------------------------------------------------------------------------------------------
// host-side launch helpers
// ---------------------------------------------------------------------------------------------

template <int OP, int TN, int CG, int ST>
static int launch_main_t(const KernelParams& p, bool after_zero, cudaStream_t stream) {
    using C = Cfg<OP, TN, CG, ST>;
    auto kern = sk_main_kernel<OP, TN, CG, ST>;
    // Set once per device (the attribute belongs to the function in that device's context).
    static unsigned long long smem_set = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
    if (dev < 0 || !(smem_set & (1ull << dev))) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::kSmem));
        if (e != cudaSuccess) return static_cast<int>(e);
        if (dev >= 0) smem_set |= 1ull << dev;
    }
    if (p.plan.grid <= 0) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.plan.grid * CG));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (CG == 2) {   // one cluster of two CTAs per logical CTA
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = CG;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (after_zero) {   // start while the zeroing kernel just before it finishes
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, kern, p));
}

template <int OP, int TN, int CG, int ST>
static int ctas_per_sm_t() {
    using C = Cfg<OP, TN, CG, ST>;
    auto kern = sk_main_kernel<OP, TN, CG, ST>;
    // Queried once per device.
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
    if (dev >= 0 && cached[dev] > 0) return cached[dev];
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmem)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, C::kSmem) != cudaSuccess)
        return 0;
    if (dev >= 0) cached[dev] = n;
    return n;
}

template <int OP, int TN, int CG, int ST>
static size_t smem_bytes_t() {
    return Cfg<OP, TN, CG, ST>::kSmem;
}

// (op, cg, tn, stages) -> the kernel instantiation (the stages follow from cg and tn); the
// im2col wgrad has no pair form (the host rejects it first); the shifted-row wgrad has a one-CTA
// 128 x 192 form with one-step stages (8 of 26 KB, or 5 of 42 KB with two x column phases) and a
// 256 x 192 pair form with several steps per stage (4 of 48 KB, or 3 of 73 KB); the block-scaled
// fp8 GEMM has a 128 x 128 form (5 stages beside its 32 KB store staging
// and its scale ring) and a 256 x 128 pair form (7 stages).
#define SK_DISPATCH(op, cg, tn, st, fn, ...)                                                \
    ((cg) == 2                                                                              \
         ? ((op) == kOpWgradRow1 ? fn<kOpWgradRow1, 192, 2, 4>(__VA_ARGS__)                  \
            : (op) == kOpWgradRow2 ? fn<kOpWgradRow2, 192, 2, 3>(__VA_ARGS__)                \
            : (tn) == 256 ? ((op) == kOpFp8 ? fn<kOpFp8, 256, 2, 3>(__VA_ARGS__)             \
                             : (st) == 7 ? fn<kOpGemm16, 256, 2, 7>(__VA_ARGS__)               \
                                          : fn<kOpGemm16, 256, 2, 3>(__VA_ARGS__))            \
                        : ((op) == kOpFp8 ? fn<kOpFp8, 128, 2, 4>(__VA_ARGS__)                \
                           : (op) == kOpFp8Block ? fn<kOpFp8Block, 128, 2, 7>(__VA_ARGS__)    \
                                          : fn<kOpGemm16, 128, 2, 4>(__VA_ARGS__)))           \
     : (op) == kOpGemm16 ? fn<kOpGemm16, 128, 1, 6>(__VA_ARGS__)                              \
     : (op) == kOpFp8    ? fn<kOpFp8, 128, 1, 6>(__VA_ARGS__)                                 \
     : (op) == kOpFprop16 ? fn<kOpFprop16, 128, 1, 3>(__VA_ARGS__)                            \
     : (op) == kOpFpropRow ? fn<kOpFpropRow, 64, 1, 4>(__VA_ARGS__)                           \
     : (op) == kOpDgrad16 ? fn<kOpDgrad16, 128, 1, 3>(__VA_ARGS__)                            \
     : (op) == kOpFp8Block ? fn<kOpFp8Block, 128, 1, 5>(__VA_ARGS__)                          \
     : (op) == kOpWgradRow1 ? fn<kOpWgradRow1, 192, 1, 8>(__VA_ARGS__)                        \
     : (op) == kOpWgradRow2 ? fn<kOpWgradRow2, 192, 1, 5>(__VA_ARGS__)                        \
                         : fn<kOpWgrad16, 128, 1, 7>(__VA_ARGS__))

size_t main_smem_bytes(int op, int cg, int tn, int st) {
    return SK_DISPATCH(op, cg, tn, st, smem_bytes_t);
}

int main_ctas_per_sm(int op, int cg, int tn, int st) {
    return SK_DISPATCH(op, cg, tn, st, ctas_per_sm_t);
}

int launch_main(const KernelParams& p, int op, int cg, int tn, int st, bool after_zero,
                cudaStream_t stream) {
    if (cg == 2 && op != kOpGemm16 && op != kOpFp8 && op != kOpFp8Block && !is_wgrad_row(op))
        return static_cast<int>(cudaErrorInvalidValue);
    return SK_DISPATCH(op, cg, tn, st, launch_main_t, p, after_zero, stream);
}

template <int TN, int CG>
static int launch_stage2_t(const Stage2Params& p, dim3 grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kStage2Threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.after_main ? 1 : 0;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, sk_stage2_kernel<TN, CG>, p));
}

int launch_stage2(const Stage2Params& p, cudaStream_t stream) {
    const int64_t tiles = n_shared_candidates(p.plan);
    if (tiles <= 0) return 0;
    const int cg = p.plan.tm == 2 * kTileM ? 2 : 1;
    const int tn = p.plan.tn == 256 ? 256 : p.plan.tn == 64 ? 64 : p.plan.tn == 192 ? 192 : 128;
    const unsigned slices = static_cast<unsigned>(cg * kTileM * tn / 4 / kStage2Threads);
    const dim3 grid(static_cast<unsigned>(tiles), slices);
    if (tn == 64) return launch_stage2_t<64, 1>(p, grid, stream);
    if (tn == 192) return cg == 2 ? launch_stage2_t<192, 2>(p, grid, stream)
                                  : launch_stage2_t<192, 1>(p, grid, stream);
    if (tn == 256) return launch_stage2_t<256, 2>(p, grid, stream);
    return cg == 2 ? launch_stage2_t<128, 2>(p, grid, stream) : launch_stage2_t<128, 1>(p, grid, stream);
}

// Zeroes up to three 16-byte aligned ranges (flags + control block, scratch) and one strided
// 2-D range of 4-byte words (the fp32 output of the atomic reduction) ahead of a main kernel.
// Every CTA first lets the main kernel's launch begin, so that its start-up overlaps this kernel.
__global__ void __launch_bounds__(256) sk_zero_kernel(const __grid_constant__ ZeroParams z) {
    grid_launch_dependents();
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int r = 0; r < z.nranges; ++r) {
        uint4* p = static_cast<uint4*>(z.ptr[r]);
        const int64_t n = z.bytes[r] / 16;
        for (int64_t i = tid; i < n; i += nthr) p[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (z.rows > 0) {
        const int64_t words = z.row_bytes / 4;
        const int64_t n = words * z.rows;
        for (int64_t i = tid; i < n; i += nthr) {
            const int64_t row = i / words, w = i - row * words;
            reinterpret_cast<uint32_t*>(static_cast<char*>(z.out) + row * z.pitch)[w] = 0u;
        }
    }
}

int launch_zero(const ZeroParams& z, cudaStream_t stream) {
    int64_t work = z.rows * (z.row_bytes / 4);
    for (int r = 0; r < z.nranges; ++r) work += z.bytes[r] / 16;
    if (work <= 0) return 0;
    const int64_t blocks = imin(imax(ceil_div(work, 256 * 8), 1), 1184);
    sk_zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(z);
    return static_cast<int>(cudaGetLastError());
}

int launch_flag_timeout_probe(uint64_t limit_ns, cudaStream_t stream) {
    sk_flag_timeout_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return static_cast<int>(cudaGetLastError());
}

int take_device_error(cudaStream_t stream, long long info[3]) {
    unsigned long long h[4] = {0, 0, 0, 0};
    if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(h, g_sk_error, sizeof(h)) != cudaSuccess) return -1;
    if (h[0] != 0) {
        const unsigned long long z[4] = {0, 0, 0, 0};
        if (cudaMemcpyToSymbol(g_sk_error, z, sizeof(z)) != cudaSuccess) return -1;
    }
    info[0] = static_cast<long long>(h[1]);
    info[1] = static_cast<long long>(h[2]);
    info[2] = static_cast<long long>(h[3]);
    return static_cast<int>(h[0]);
}

}  // namespace sk
