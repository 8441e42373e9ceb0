// C ABI of libskgemm: argument validation (-2), the host planner, workspace layout, TMA
// descriptors and the launch sequence on the caller's stream.
//
// The single-problem call shape and its return codes follow "feat(ck-tile): stream-K GEMM TE to
// dispatcher bridge" (Design note / Changes: returns 0, -1 on a launch error, -2 for
// unsupported arguments; the launch owns the reduction workspace). The knobs streamk /
// reduction / ctas, the CTA-pool default and the validator's rejections follow rocm-libraries
// PR #13151 (PR body: Technical Details, Constraints; commits "Resolve streamk_ctas=-1 from the
// reduction" and "Address review feedback").
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <utility>
#include <vector>

#include "sk_kernels.h"
#include "sk_plan.h"
#include "skgemm.h"

namespace {

thread_local char g_err[512] = "";
thread_local int g_tile = SK_TILE_AUTO;   // sk_set_tile

// Sets the calling thread's tile setting for a scope.
struct TileGuard {
    int prev;
    explicit TileGuard(int tile) : prev(g_tile) { g_tile = tile; }
    ~TileGuard() { g_tile = prev; }
};

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(SK_ERR_LAUNCH, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

const char* mode_name(int m) {
    switch (m) {
        case SK_OFF: return "off";
        case SK_DP_SK: return "dp_sk";
        case SK_PERSISTENT: return "persistent";
        case SK_SPLITK: return "splitk";
        case SK_HYBRID: return "hybrid";
        default: return "?";
    }
}
const char* red_name(int r) {
    switch (r) {
        case SK_LINEAR: return "linear";
        case SK_TREE: return "tree";
        case SK_ATOMIC: return "atomic";
        case SK_WORKSPACE: return "workspace";
        default: return "?";
    }
}
const char* dtype_name(int d) {
    switch (d) {
        case SK_F16: return "f16";
        case SK_BF16: return "bf16";
        case SK_F32: return "f32";
        case SK_E4M3: return "e4m3";
        default: return "?";
    }
}
int dtype_size(int d) { return d == SK_F32 ? 4 : d == SK_E4M3 ? 1 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- device facts ---------------------------------------------------------------------------

struct DevInfo {
    bool ok = false;
    int sms = 0, major = 0, minor = 0;
};

std::mutex g_dev_mu;
DevInfo g_dev[64];

int current_device_info(DevInfo& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SK_ERR_UNSUPPORTED, "no CUDA device: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SK_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].ok) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess)
            return fail(SK_ERR_UNSUPPORTED, "cannot query device %d: %s", dev, cudaGetErrorString(e));
        g_dev[dev].sms = prop.multiProcessorCount;
        g_dev[dev].major = prop.major;
        g_dev[dev].minor = prop.minor;
        g_dev[dev].ok = true;
    }
    out = g_dev[dev];
    return SK_OK;
}

// Make the device that owns `p` current (pointers from another runtime instance carry their
// device in their attributes).
int select_device_of(const void* p) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SK_ERR_UNSUPPORTED, "cannot query the output pointer: %s", cudaGetErrorString(e));
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
        return fail(SK_ERR_UNSUPPORTED, "output pointer is not device memory");
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != a.device) {
        e = cudaSetDevice(a.device);
        if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    }
    return SK_OK;
}

int check_arch(DevInfo& d) {
    int rc = current_device_info(d);
    if (rc != SK_OK) return rc;
    if (!(d.major == 10 && d.minor == 3))
        return fail(SK_ERR_UNSUPPORTED,
                    "device is sm_%d%d; this library is built for sm_103a (GB300) only", d.major,
                    d.minor);
    return SK_OK;
}

// ---- planner --------------------------------------------------------------------------------

int resolve_pool(int reduction, int ctas, int num_sms, int ctas_per_sm, int64_t& pool) {
    if (ctas == 0 || ctas < -1)
        return fail(SK_ERR_UNSUPPORTED, "streamk_ctas must be -1 (default) or >= 1, got %d", ctas);
    if (ctas > 0) {
        pool = ctas;
        return SK_OK;
    }
    if (num_sms <= 0) return fail(SK_ERR_UNSUPPORTED, "default CTA pool needs the SM count");
    if (reduction == SK_LINEAR || reduction == SK_TREE) {
        pool = num_sms;   // every CTA may wait on a later one: one per SM
    } else {
        int per = ctas_per_sm < 1 ? 1 : ctas_per_sm;
        pool = static_cast<int64_t>(num_sms) * (per < 4 ? per : 4);
    }
    return SK_OK;
}

struct View {          // GEMM view of a problem
    int64_t gemm_m, gemm_n, kred, groups;
    int op_kind;       // sk::OpKind
};

// Geometry of the shifted-row wgrad (see wgrad_row_geom).
struct RowGeom {
    int64_t ho, wo, ho_pad;
    int wseg, rows_per_step, qmax, sw;
    int nq[2];
};

// The shifted-row wgrad serves groups of 64 channels and 64 filters with at most 3 column taps,
// a column stride of 1 or 2, and output rows short enough that a row and the shifts' halo fit one
// 64-position K step: wseg = the power of two >= Wo + qmax (at most 64), rows_per_step = 64/wseg
// output rows per step, rows counted per image over Ho rounded up to rows_per_step. Column tap
// s = sw*q + p (phase p < sw) reads x column sw*(wo + q) + p - pad, i.e. the x row of phase p read
// at position wo + q: q <= qmax = ceil(S/sw) - 1. False when the problem does not fit.
bool wgrad_row_geom(const sk_problem& p, RowGeom& g) {
    if (p.op != SK_OP_WGRAD || p.groups < 1 || p.c % p.groups || p.k % p.groups) return false;
    if (p.c / p.groups != 64 || p.k / p.groups != 64) return false;
    if (p.s < 1 || p.s > 3 || p.r < 1 || p.stride_w < 1 || p.stride_w > 2 || p.stride_h < 1 ||
        p.stride_h > 8)
        return false;
    g.sw = p.stride_w;
    g.ho = (p.h + 2 * p.pad_h - p.r) / p.stride_h + 1;
    g.wo = (p.w + 2 * p.pad_w - p.s) / p.stride_w + 1;
    if (g.ho < 1 || g.wo < 1) return false;
    g.nq[0] = static_cast<int>((p.s + g.sw - 1) / g.sw);
    g.nq[1] = g.sw == 2 ? static_cast<int>(p.s / 2) : 0;
    g.qmax = g.nq[0] - 1;
    g.wseg = 1;
    while (g.wseg < g.wo + g.qmax) g.wseg *= 2;
    if (g.wseg > 64) return false;
    g.rows_per_step = 64 / g.wseg;
    if (static_cast<int64_t>(g.rows_per_step) * p.stride_h > 256) return false;   // TMA box rows
    g.ho_pad = sk::round_up(g.ho, g.rows_per_step);
    if (p.n * g.ho_pad >= (int64_t(1) << 31)) return false;   // 32-bit row index in the kernel
    return true;
}

int problem_view_pages(const sk_problem& p, View& v);

// The shifted-row kernel serves stride-1 convolutions of one group of 64 channels into 64, at
// most 3 x 3 taps and output rows of at most 64 positions with the column taps' overrun
// (width + S - 1 <= 64): the forward convolution (x -> y, Ho x Wo), and the data gradient as the
// stride-1 convolution of dy with the flipped filter, padding R - 1 - p (dy -> dx, H x W). A tile is
// two output rows of 64 positions (rows counted per image over the height rounded up to even),
// its reduction the taps (64 channels each). th x tw: the output grid of that traversal.
bool conv_row_geom(const sk_problem& p, int64_t& th, int64_t& tw, int64_t& th_pad) {
    if ((p.op != SK_OP_FPROP && p.op != SK_OP_DGRAD) || p.groups != 1 || p.c != 64 || p.k != 64)
        return false;
    if (p.stride_h != 1 || p.stride_w != 1 || p.r < 1 || p.r > 3 || p.s < 1 || p.s > 3) return false;
    if (p.pad_h < 0 || p.pad_w < 0 || p.pad_h >= p.r || p.pad_w >= p.s) return false;
    const int64_t ho = p.h + 2 * p.pad_h - p.r + 1, wo = p.w + 2 * p.pad_w - p.s + 1;
    if (ho < 1 || wo < 1) return false;
    th = p.op == SK_OP_FPROP ? ho : p.h;
    tw = p.op == SK_OP_FPROP ? wo : p.w;
    if (tw + p.s - 1 > 64) return false;
    th_pad = sk::round_up(th, 2);
    return p.n * th_pad * 64 < (int64_t(1) << 31);
}

// The GEMM view of a problem under the calling thread's tile setting. Wgrad: the pages' view
// (M = K/G filters, N = R*S*C/G, reduction over N*Ho*Wo output pixels), or with the automatic
// tile, where it fits, the shifted-row view: M = (tap row r, channel) = R*64 in 128-row tiles (two
// tap rows), N = (column tap s, filter) = S*64 in one 192-column tile, reduction over the padded
// positions N*ho_pad*wseg.
int problem_view(const sk_problem& p, View& v) {
    int rc = problem_view_pages(p, v);
    if (rc) return rc;
    int64_t fho, fwo, fho_pad;
    if ((v.op_kind == sk::kOpFprop16 || v.op_kind == sk::kOpDgrad16) && g_tile == SK_TILE_AUTO &&
        conv_row_geom(p, fho, fwo, fho_pad)) {
        v.gemm_m = p.n * fho_pad * 64;
        v.gemm_n = 64;
        v.kred = p.r * p.s * 64;
        v.op_kind = sk::kOpFpropRow;
        return SK_OK;
    }
    RowGeom g;
    if (v.op_kind == sk::kOpWgrad16 && (g_tile == SK_TILE_AUTO || g_tile == SK_TILE_256_PAIR) &&
        wgrad_row_geom(p, g)) {
        v.gemm_m = p.r * 64;
        v.gemm_n = p.s * 64;
        v.kred = p.n * g.ho_pad * g.wseg;
        v.op_kind = g.sw == 1 ? sk::kOpWgradRow1 : sk::kOpWgradRow2;
    }
    return SK_OK;
}

int problem_view_pages(const sk_problem& p, View& v) {
    switch (p.op) {
        case SK_OP_GEMM:
        case SK_OP_FP8_ROWCOL:
        case SK_OP_FP8_BLOCK:
            v.gemm_m = p.M;
            v.gemm_n = p.N;
            v.kred = p.K;
            v.groups = 1;
            v.op_kind = p.op == SK_OP_GEMM       ? sk::kOpGemm16
                        : p.op == SK_OP_FP8_BLOCK ? sk::kOpFp8Block
                                                  : sk::kOpFp8;
            return SK_OK;
        case SK_OP_FPROP:
        case SK_OP_DGRAD: {
            if (p.groups < 1) return fail(SK_ERR_UNSUPPORTED, "groups must be >= 1");
            if (p.stride_h < 1 || p.stride_w < 1) return fail(SK_ERR_UNSUPPORTED, "stride must be >= 1");
            const int64_t Ho = (p.h + 2 * p.pad_h - p.r) / p.stride_h + 1;
            const int64_t Wo = (p.w + 2 * p.pad_w - p.s) / p.stride_w + 1;
            if (p.h + 2 * p.pad_h < p.r || p.w + 2 * p.pad_w < p.s || Ho < 1 || Wo < 1)
                return fail(SK_ERR_UNSUPPORTED, "filter larger than the padded image");
            v.groups = p.groups;
            if (p.op == SK_OP_FPROP) {   // output pixels x filters, reduction over (r, s, c)
                v.gemm_m = p.n * Ho * Wo;
                v.gemm_n = p.k / p.groups;
                v.kred = p.r * p.s * (p.c / p.groups);
                v.op_kind = sk::kOpFprop16;
            } else {                     // input pixels x channels, reduction over (r, s, k)
                v.gemm_m = p.n * p.h * p.w;
                v.gemm_n = p.c / p.groups;
                v.kred = p.r * p.s * (p.k / p.groups);
                v.op_kind = sk::kOpDgrad16;
            }
            return SK_OK;
        }
        case SK_OP_WGRAD: {
            if (p.groups < 1) return fail(SK_ERR_UNSUPPORTED, "groups must be >= 1");
            if (p.stride_h < 1 || p.stride_w < 1) return fail(SK_ERR_UNSUPPORTED, "stride must be >= 1");
            const int64_t Ho = (p.h + 2 * p.pad_h - p.r) / p.stride_h + 1;
            const int64_t Wo = (p.w + 2 * p.pad_w - p.s) / p.stride_w + 1;
            if (p.h + 2 * p.pad_h < p.r || p.w + 2 * p.pad_w < p.s || Ho < 1 || Wo < 1)
                return fail(SK_ERR_UNSUPPORTED, "filter larger than the padded image");
            v.groups = p.groups;
            v.gemm_m = p.k / p.groups;
            v.gemm_n = p.r * p.s * (p.c / p.groups);
            v.kred = p.n * Ho * Wo;
            v.op_kind = sk::kOpWgrad16;
            return SK_OK;
        }
        default:
            return fail(SK_ERR_UNSUPPORTED, "unknown op %d", p.op);
    }
}

int build_plan_resolved(const sk_problem& prob, int mode, int reduction, int ctas, int num_sms,
                        int ctas_per_sm, sk_plan_t& p, bool all_dp = false);

constexpr int64_t kAutoPairMinTiles = 64;   // SK_TILE_AUTO: pair tiles needed for the pair kernel
constexpr int64_t kSpreadMinContributors = 8;   // linear / tree: contributors for the spread fold
constexpr int64_t kRowPairMinSteps = 128 * 148;  // shifted-row wgrad: K steps for the pair kernel
constexpr int64_t kAutoLongReductionSteps = 512;  // SK_TILE_AUTO: K steps for the deep-ring pair

// The kernel shape for a problem under the calling thread's tile setting: cg CTAs per logical CTA
// (1, or 2 for a CTA pair) and the tile's N; the tile's M is 128 * cg.
struct TileCfg {
    int cg, tn, st;   // CTAs per logical CTA, tile N, operand-ring stages
};
int tile_cfg(const View& v, TileCfg& t) {
    if (v.op_kind == sk::kOpFpropRow) {   // 128 x 64 tile, 4 stages of 33 KB + the 72 KB filter
        t = TileCfg{1, 64, 4};
        return SK_OK;
    }
    if (sk::is_wgrad_row(v.op_kind)) {
        // Three or four tap rows (M = 192 or 256) over a long reduction (at least
        // kRowPairMinSteps K steps of 128-row tiles in all, about 128 per SM): a 256 x 192 tile
        // on a CTA pair, each CTA holding two tap rows and half the filters, with several K steps
        // per ring stage. Otherwise a 128 x 192 tile on one CTA with one-step stages: with a
        // few dozen steps per CTA its deeper ring ramps up faster (measured on the 32x56x56 and
        // grouped 64x28x28 wgrad, 20.1 against 21.2-24.3 us).
        // SK_TILE_256_PAIR asks for the pair kernel whatever the size.
        const int64_t steps = v.groups * sk::ceil_div(v.gemm_m, sk::kTileM) * (v.kred / 64);
        const bool pair = g_tile == SK_TILE_256_PAIR ||
                          ((v.gemm_m == 3 * 64 || v.gemm_m == 4 * 64) && steps >= kRowPairMinSteps);
        t = TileCfg{pair ? 2 : 1, 192, sk::wgrow_stages(v.op_kind, pair ? 2 : 1)};
        return SK_OK;
    }
    if (v.op_kind == sk::kOpFp8Block) {
        // Two 128-column partial buffers fill 256 TMEM columns (the running sum stays in the
        // epilogue's registers), so the tile is 128 columns wide: 128 x 128 on one CTA (5 ring
        // stages beside the store staging and the scale ring, the default), or 256 x 128 on a CTA
        // pair (7 stages) on request. The pair's per-step hand-off of each partial between the two
        // CTAs measured twice as slow as the one-CTA tile's, so it is not chosen by itself.
        if (g_tile == SK_TILE_256x256_PAIR)
            return fail(SK_ERR_UNSUPPORTED, "the block-scaled fp8 GEMM has no 256 x 256 tile");
        t = g_tile == SK_TILE_256_PAIR ? TileCfg{2, 128, 7} : TileCfg{1, 128, 5};
        return SK_OK;
    }
    // fprop / dgrad: 3 stages and no store staging, so that two CTAs share an SM (their reductions
    // are short, and the other CTA's mainloop covers one's prologue and epilogue).
    const bool conv_fwd = v.op_kind == sk::kOpFprop16 || v.op_kind == sk::kOpDgrad16;
    t = {1, sk::kTileN, v.op_kind == sk::kOpWgrad16 ? 7 : conv_fwd ? 3 : 6};
    switch (g_tile) {
        case SK_TILE_128: return SK_OK;
        case SK_TILE_256_PAIR:
        case SK_TILE_256x256_PAIR:
            if (v.op_kind != sk::kOpGemm16 && v.op_kind != sk::kOpFp8)
                return fail(SK_ERR_UNSUPPORTED, "the CTA-pair tiles serve the GEMMs and the shifted-row wgrad only");
            // Rings of about 96 KB, so that two CTAs share an SM and one's epilogue overlaps the
            // other's mainloop (measured faster than one CTA per SM with twice the stages).
            t = g_tile == SK_TILE_256_PAIR ? TileCfg{2, 128, 4} : TileCfg{2, 256, 3};
            return SK_OK;
        default: {   // SK_TILE_AUTO
            // The 256 x 256 pair where the problem has rows for it and enough pair tiles that the
            // data-parallel part carries the work. With few tiles over a long reduction, the
            // smaller tile splits the reduction among fewer CTAs per tile (cheaper fixups).
            const int64_t pair_tiles = sk::ceil_div(v.gemm_m, 2 * sk::kTileM) * sk::ceil_div(v.gemm_n, 256);
            if ((v.op_kind == sk::kOpGemm16 || v.op_kind == sk::kOpFp8) && v.gemm_m > sk::kTileM &&
                pair_tiles >= kAutoPairMinTiles)
                t = TileCfg{2, 256, 3};
            // Few tiles over a long 16-bit reduction (the 512 x 512 x 65536 GEMM): each SM takes in
            // the operands of its share of the MMAs through its copy engine, at about 115 GB/s, so
            // the 256 x 256 pair tile's half bytes per FLOP matter most; one CTA per SM with a
            // 7-stage ring (224 KB) keeps its copies in flight.
            else if (v.op_kind == sk::kOpGemm16 && v.gemm_m > sk::kTileM && v.gemm_n > 128 &&
                     v.kred / 64 >= kAutoLongReductionSteps)
                t = TileCfg{2, 256, 7};
            return SK_OK;
        }
    }
}
int problem_tile(const sk_problem& prob, TileCfg& t) {
    View v;
    int rc = problem_view(prob, v);
    if (rc) return rc;
    return tile_cfg(v, t);
}

// SK_AUTO: stream-K for few tiles over a long reduction, and only when the partition the launch
// would use has stream-K CTAs; split-K everywhere else.
constexpr int64_t kAutoMinIterations = 1024;   // T * I at which the reduction counts as long

int build_plan(const sk_problem& prob, int mode, int reduction, int ctas, int num_sms,
               int ctas_per_sm, sk_plan_t& p) {
    if (reduction == SK_REDUCTION_AUTO) reduction = SK_WORKSPACE;
    if (mode != SK_AUTO) return build_plan_resolved(prob, mode, reduction, ctas, num_sms, ctas_per_sm, p);
    int rc = build_plan_resolved(prob, SK_DP_SK, reduction, ctas, num_sms, ctas_per_sm, p);
    if (rc) return rc;
    if (p.tiles < p.pool && p.tiles * p.iters_per_tile >= kAutoMinIterations && p.sk_ctas > 0)
        return SK_OK;
    // The shifted-row fprop keeps its filter resident: with more tiles than CTAs each CTA loads
    // it once and runs its tiles in turn (persistent) instead of one CTA per tile. Its tiles are
    // short (one K step per tap), so a stream-K wave's fixups cost more than the last wave's idle
    // CTAs: every tile stays data-parallel.
    View v;
    if (p.tiles > p.pool && problem_view(prob, v) == SK_OK && v.op_kind == sk::kOpFpropRow)
        return build_plan_resolved(prob, SK_PERSISTENT, reduction, ctas, num_sms, ctas_per_sm, p,
                                   true);
    return build_plan_resolved(prob, SK_SPLITK, reduction, ctas, num_sms, ctas_per_sm, p);
}

// all_dp: no stream-K region whatever the tile count (SK_PERSISTENT: every CTA runs tiles
// cta, cta + pool, ...).
int build_plan_resolved(const sk_problem& prob, int mode, int reduction, int ctas, int num_sms,
                        int ctas_per_sm, sk_plan_t& p, bool all_dp) {
    if (mode < SK_OFF || mode > SK_HYBRID || mode == SK_AUTO)
        return fail(SK_ERR_UNSUPPORTED, "unknown streamk mode %d", mode);
    if (reduction < SK_LINEAR || reduction > SK_WORKSPACE)
        return fail(SK_ERR_UNSUPPORTED, "unknown streamk reduction %d", reduction);
    View v;
    int rc = problem_view(prob, v);
    if (rc) return rc;
    if (v.gemm_m < 1 || v.gemm_n < 1 || v.kred < 1 || v.groups < 1)
        return fail(SK_ERR_UNSUPPORTED, "empty problem (M=%lld N=%lld K=%lld)", (long long)v.gemm_m,
                    (long long)v.gemm_n, (long long)v.kred);
    TileCfg tc;
    rc = tile_cfg(v, tc);
    if (rc) return rc;
    const int cg = tc.cg;
    // A pair kernel's pool counts pairs: its default is resolved over SM pairs.
    int64_t P = 0;
    rc = resolve_pool(reduction, ctas, num_sms / cg, ctas_per_sm, P);
    if (rc) return rc;
    memset(&p, 0, sizeof(p));
    p.op = prob.op;
    p.mode = mode;
    p.reduction = reduction;
    p.tm = sk::kTileM * cg;
    p.tn = tc.tn;
    p.tk = (prob.op == SK_OP_FP8_ROWCOL || prob.op == SK_OP_FP8_BLOCK) ? 128 : 64;
    p.gemm_m = v.gemm_m;
    p.gemm_n = v.gemm_n;
    p.kred = v.kred;
    p.groups = v.groups;
    p.tiles_m = sk::ceil_div(v.gemm_m, p.tm);
    p.tiles_n = sk::ceil_div(v.gemm_n, p.tn);
    p.tiles = v.groups * p.tiles_m * p.tiles_n;
    p.iters_per_tile = sk::ceil_div(v.kred, p.tk);
    p.pool = P;
    p.iters_per_sk_cta = 1;
    const int64_t T = p.tiles, I = p.iters_per_tile;
    if (mode == SK_OFF) {
        p.dp_tiles = T;
        p.grid = T;
    } else if (mode == SK_SPLITK) {
        int64_t s = P / T;
        if (s < 1) s = 1;
        if (s > I) s = I;
        p.splits = s;
        p.dp_tiles = s == 1 ? T : 0;
        p.grid = T * s;
        p.publishers = s > 1 ? T * s : 0;
    } else {
        p.sk_tiles = T % P;
        if (mode == SK_HYBRID && T >= P && p.sk_tiles > 0) p.sk_tiles += P;   // one wave more
        p.dp_tiles = T - p.sk_tiles;
        p.sk_iters = p.sk_tiles * I;
        if (all_dp || p.sk_tiles == 0 || p.sk_iters < P) {   // too few iterations for the pool: all-DP
            p.sk_tiles = 0;
            p.dp_tiles = T;
            p.sk_iters = 0;
            p.sk_ctas = 0;
        } else {
            p.sk_ctas = P;
            p.iters_per_sk_cta = sk::imax(1, p.sk_iters / p.sk_ctas);
            p.extra_iters = p.sk_iters % p.sk_ctas;
        }
        p.grid = (mode == SK_DP_SK || mode == SK_HYBRID) ? p.sk_ctas + p.dp_tiles : P;
        p.publishers = p.sk_ctas;
    }
    if (p.grid > 0x7fffffffLL) return fail(SK_ERR_UNSUPPORTED, "grid too large");
    // The kernels walk iterations, tiles and CTA ids with 32-bit arithmetic.
    if (p.tiles * p.iters_per_tile > 0x7fffffffLL)
        return fail(SK_ERR_UNSUPPORTED, "too many MAC iterations (tiles x iterations per tile >= 2^31)");
    int64_t maxc = 1, shared = 0;
    for (int64_t t = 0; t < sk::n_shared_candidates(p); ++t) {
        int64_t first, n;
        sk::tile_contributors(p, t, first, n);
        if (n > maxc) maxc = n;
        shared += n > 1;
    }
    p.max_contributors = maxc;
    p.shared_tiles = shared;
    while ((int64_t(1) << p.tree_rounds) < maxc) ++p.tree_rounds;
    if (reduction == SK_TREE && p.tree_rounds > 32)
        return fail(SK_ERR_UNSUPPORTED, "tree reduction supports at most 2^32 contributors");
    const int64_t tile_bytes = p.tm * p.tn * 4;
    // One flag per 128-row half: each CTA of a pair publishes and receives its half on its own.
    p.flag_bytes = sk::round_up(4 * p.publishers * cg, 256);
    p.control_offset = p.flag_bytes;
    p.partial_offset = p.control_offset + sk::kControlBytes;
    p.partial_slots = mode == SK_SPLITK ? p.publishers : (p.sk_ctas > 0 ? p.sk_ctas + p.sk_tiles : 0);
    p.partial_bytes = (reduction == SK_LINEAR || reduction == SK_TREE) ? p.partial_slots * tile_bytes : 0;
    p.scratch_offset = p.partial_offset + p.partial_bytes;
    p.scratch_bytes = reduction == SK_WORKSPACE ? sk::n_shared_candidates(p) * tile_bytes : 0;
    p.ws_bytes = p.scratch_offset + p.scratch_bytes;
    return SK_OK;
}

// ---- TMA descriptors ------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const int*, const int*,
                                   cuuint32_t, cuuint32_t, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

std::once_flag g_enc_once;
EncodeTiledFn g_encode_tiled = nullptr;
EncodeIm2colFn g_encode_im2col = nullptr;

int load_encoders() {
    std::call_once(g_enc_once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<EncodeTiledFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(f);
    });
    if (!g_encode_tiled || !g_encode_im2col)
        return fail(SK_ERR_LAUNCH, "cuTensorMapEncode* entry points unavailable");
    return SK_OK;
}

// 2-D K-major (inner dimension first) tile map with 128-byte swizzle; box = {box_inner, box_outer}.
int encode_2d(CUtensorMap* m, const void* base, int elem, uint64_t inner, uint64_t outer,
              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(m, elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                                2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SK_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return SK_OK;
}

uint64_t flag_timeout_ns() {
    const char* s = getenv("SKGEMM_FLAG_TIMEOUT_MS");
    long long ms = s ? atoll(s) : 1000;
    if (ms < 1) ms = 1;
    return static_cast<uint64_t>(ms) * 1000000ull;
}

// ---- instrumentation ------------------------------------------------------------------------

struct Timing {
    bool on = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> used, pool;
    int64_t main_launches = 0, all_launches = 0;
    ~Timing() {
        for (auto& p : used) { cudaEventDestroy(p.first); cudaEventDestroy(p.second); }
        for (auto& p : pool) { cudaEventDestroy(p.first); cudaEventDestroy(p.second); }
    }
    void recycle() {
        pool.insert(pool.end(), used.begin(), used.end());
        used.clear();
        main_launches = all_launches = 0;
    }
};
thread_local Timing g_timing;

// Record the start event of one main-kernel launch; returns the pair index or -1.
int timing_start(cudaStream_t s) {
    if (!g_timing.on) return -1;
    std::pair<cudaEvent_t, cudaEvent_t> ev;
    if (!g_timing.pool.empty()) {
        ev = g_timing.pool.back();
        g_timing.pool.pop_back();
    } else if (cudaEventCreate(&ev.first) != cudaSuccess || cudaEventCreate(&ev.second) != cudaSuccess) {
        return -1;
    }
    cudaEventRecord(ev.first, s);
    g_timing.used.push_back(ev);
    return static_cast<int>(g_timing.used.size()) - 1;
}

// ---- launch sequence ------------------------------------------------------------------------

// part: 0 = the zeroing kernel (where the plan needs one), the main kernel and Stage-2; 1 = the
// zeroing kernel alone; 2 = the main kernel and Stage-2 alone, the workspace's words having been
// zeroed by an earlier part-1 call on the same stream.
int run(const sk_problem& prob, int mode, int reduction, int ctas, sk::KernelParams& kp,
        void* out, size_t out_pitch_bytes, size_t out_rows, size_t out_row_bytes, void* ws,
        size_t ws_bytes, cudaStream_t stream, int part = 0) {
    DevInfo dev;
    int rc = check_arch(dev);
    if (rc) return rc;
    View v;
    problem_view(prob, v);
    TileCfg tc;
    rc = tile_cfg(v, tc);
    if (rc) return rc;
    const int per_sm = sk::main_ctas_per_sm(v.op_kind, tc.cg, tc.tn, tc.st);
    sk_plan_t plan;
    rc = build_plan(prob, mode, reduction, ctas, dev.sms, per_sm, plan);
    if (rc) return rc;
    if (ws != nullptr) {
        if (ws_bytes < static_cast<size_t>(plan.ws_bytes))
            return fail(SK_ERR_UNSUPPORTED, "workspace too small: %zu < %lld bytes", ws_bytes,
                        (long long)plan.ws_bytes);
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
            return fail(SK_ERR_UNSUPPORTED, "workspace must be 256-byte aligned");
    }
    bool own_ws = false;
    cudaError_t e;
    if (ws == nullptr) {
        e = cudaMallocAsync(&ws, static_cast<size_t>(plan.ws_bytes), stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
        own_ws = true;
    }
    uint8_t* w = static_cast<uint8_t*>(ws);
    kp.plan = plan;
    kp.flags = reinterpret_cast<uint32_t*>(w);
    kp.control = reinterpret_cast<uint32_t*>(w + plan.control_offset);
    kp.partials = reinterpret_cast<float*>(w + plan.partial_offset);
    kp.scratch = reinterpret_cast<float*>(w + plan.scratch_offset);
    kp.flag_timeout_ns = flag_timeout_ns();
    kp.mbar_timeout_ns = 2000000000ull;
    // linear / tree: spread the additions over the contributors of a shared tile when a tile has
    // many of them (the owner's fold grows with their count, a folder's share shrinks), all the
    // CTAs that publish can be resident at once (each waits for all of its tiles' contributors),
    // and a tree's binary counter of partial sums (8 levels) holds its contributors; otherwise
    // the owner fold of the pages, whose waits target only later CTAs. Measured on GB300: with
    // 4-5 contributors per tile (the 3840x4096x4096 GEMM on 74 CTA pairs) the owner fold is faster,
    // with 19-74 (the wgrad workloads) the spread fold by 1.4-3x.
    // The spread fold's arrival counters (one per shared-tile candidate and CTA of a pair) fill the
    // control block's words after the ticket.
    const int64_t resident = static_cast<int64_t>(dev.sms / tc.cg) * (per_sm > 0 ? per_sm : 1);
    const int64_t candidates = plan.mode == SK_SPLITK ? (plan.splits > 1 ? plan.tiles : 0)
                                                      : plan.sk_tiles;
    kp.spread = 0;
    if ((plan.reduction == SK_LINEAR || plan.reduction == SK_TREE) && plan.shared_tiles > 0) {
        kp.spread = plan.max_contributors >= kSpreadMinContributors &&
                    plan.publishers <= resident &&
                    candidates * tc.cg <= sk::kControlBytes / 4 - 1 &&
                    (plan.reduction == SK_LINEAR || plan.max_contributors < 256);
    }
    // A ticket orders the logical ids by start time where a CTA may wait on a later one that is
    // not yet resident; with no waits (atomic, workspace, data-parallel) or the whole grid
    // resident at once, the block index serves.
    kp.ticket = (plan.reduction == SK_LINEAR || plan.reduction == SK_TREE) &&
                plan.shared_tiles > 0 && plan.grid > resident;

    rc = SK_OK;
    do {
        // One kernel zeroes the flags and the control block, the workspace reduction's scratch and,
        // for the atomic reduction, the output; the main kernel is launched to overlap its tail and
        // waits for its writes before it touches any of those words. With the library's timing
        // on, an event sits between the two, so they run one after the other.
        sk::ZeroParams z;
        memset(&z, 0, sizeof(z));
        const int64_t head = plan.flag_bytes + sk::kControlBytes;
        if (plan.partial_bytes == 0) {   // flags, control and scratch are contiguous
            z.ptr[z.nranges] = w;
            z.bytes[z.nranges++] = head + plan.scratch_bytes;
        } else {
            z.ptr[z.nranges] = w;
            z.bytes[z.nranges++] = head;
            if (plan.scratch_bytes > 0) {
                z.ptr[z.nranges] = w + plan.scratch_offset;
                z.bytes[z.nranges++] = plan.scratch_bytes;
            }
        }
        if (plan.reduction == SK_ATOMIC && plan.shared_tiles > 0 && out_rows > 0) {
            z.out = out;
            z.pitch = static_cast<int64_t>(out_pitch_bytes);
            z.row_bytes = static_cast<int64_t>(out_row_bytes);
            z.rows = static_cast<int64_t>(out_rows);
        }
        // Nothing to zero when no tile is shared and no ticket is drawn (the data-parallel plans):
        // the main kernel then runs alone, without overlapping what came before it.
        const bool need_zero = plan.shared_tiles > 0 || kp.ticket || z.out != nullptr;
        const bool zero = need_zero && part == 0;
        int le = 0;
        if (need_zero && part != 2) {
            le = sk::launch_zero(z, stream);
            if (le != 0) { rc = cuda_fail(static_cast<cudaError_t>(le), "zeroing kernel launch"); break; }
            if (g_timing.on) ++g_timing.all_launches;
        }
        if (part == 1) break;
        const int tslot = timing_start(stream);
        // A chained launch (kp.pdl_chain bit 0, set by the caller) overlaps the previous kernel
        // only when nothing is zeroed just before it, no ticket is drawn (its prologue waits for
        // the previous kernel) and no timing event sits between the two.
        if (zero || kp.ticket || tslot >= 0) kp.pdl_chain &= ~1;
        // Stage-2 follows: it starts while the main kernel ends and waits for it on the device.
        const bool stage2 = plan.reduction == SK_WORKSPACE && plan.shared_tiles > 0;
        if (stage2 && tslot < 0) kp.pdl_chain |= 2;
        le = sk::launch_main(kp, v.op_kind, tc.cg, tc.tn, tc.st,
                             (zero && tslot < 0) || (kp.pdl_chain & 1) != 0, stream);
        if (tslot >= 0) cudaEventRecord(g_timing.used[tslot].second, stream);
        if (le != 0) { rc = cuda_fail(static_cast<cudaError_t>(le), "main kernel launch"); break; }
        if (g_timing.on) { ++g_timing.main_launches; ++g_timing.all_launches; }
        if (plan.reduction == SK_WORKSPACE && plan.shared_tiles > 0) {
            sk::Stage2Params s2;
            s2.plan = plan;
            s2.c = kp.c;
            s2.ldc = kp.ldc;
            s2.sa = kp.sa;
            s2.sb = kp.sb;
            s2.scale = kp.scale;
            s2.tensor_scaled = (v.op_kind == sk::kOpFp8 && kp.sa == nullptr) ? 1 : 0;
            s2.scratch = kp.scratch;
            s2.c_dtype = kp.c_dtype;
            s2.op_kind = v.op_kind;
            s2.rows = kp.conv.rows;
            s2.conv = kp.conv;
            s2.after_main = tslot < 0 ? 1 : 0;
            le = sk::launch_stage2(s2, stream);
            if (le != 0) { rc = cuda_fail(static_cast<cudaError_t>(le), "stage-2 launch"); break; }
            if (g_timing.on) ++g_timing.all_launches;
        }
    } while (false);
    if (own_ws) {
        e = cudaFreeAsync(ws, stream);
        if (e != cudaSuccess && rc == SK_OK) rc = cuda_fail(e, "cudaFreeAsync(workspace)");
    }
    return rc;
}

int check_common(int mode, int reduction, int ctas, int c_dtype) {
    if (mode < SK_OFF || mode > SK_HYBRID) return fail(SK_ERR_UNSUPPORTED, "unknown streamk mode %d", mode);
    if (reduction < SK_LINEAR || reduction > SK_REDUCTION_AUTO)
        return fail(SK_ERR_UNSUPPORTED, "unknown streamk reduction %d", reduction);
    if (ctas == 0 || ctas < -1)
        return fail(SK_ERR_UNSUPPORTED, "streamk_ctas must be -1 (default) or >= 1, got %d", ctas);
    if (reduction == SK_ATOMIC && c_dtype != SK_F32)
        return fail(SK_ERR_UNSUPPORTED, "reduction 'atomic' needs an fp32 output, got %s",
                    dtype_name(c_dtype));
    return SK_OK;
}

// One output phase (a, b) of a data gradient with strides (sh, sw): the dx pixels
// (sh*i + a, sw*j + b). Only the filter taps r = r0 + sh*t (t < Rt) reach them, with
// dx[sh*i + a] = sum_t dy[i + q - t] * w[r0 + sh*t], q = (a + pad - r0) / sh: a stride-1
// convolution of dy over an Hp x Wp grid with Rt x St taps and low padding Rt - 1 - q.
struct DgradPhase {
    int64_t Hp, Wp;   // phase pixels per image
    int Rt, St;       // taps of the phase
    int r0, s0;       // first filter tap of the phase
    int padh, padw;   // traversal low padding
    int a, b;         // offset of the phase in dx
    bool live() const { return Hp > 0 && Wp > 0 && Rt > 0 && St > 0; }
};

void dgrad_phase_1d(int64_t X, int64_t R, int sigma, int pad, int a, int64_t& Xp, int& Rt, int& r0,
                    int& padl) {
    r0 = (a + pad) % sigma;
    Rt = r0 < R ? static_cast<int>((R - 1 - r0) / sigma + 1) : 0;
    const int q = (a + pad - r0) / sigma;
    padl = Rt - 1 - q;
    Xp = a < X ? (X - 1 - a) / sigma + 1 : 0;
}

// The plan-level problem of one phase: its pixel grid and taps as a stride-1 data gradient
// (padding taps-1 only keeps the view's image-size check satisfied; the view uses n*h*w, c/groups
// and r*s*k/groups).
void set_phase_problem(sk_problem& prob, int64_t Hp, int64_t Wp, int Rt, int St) {
    prob.h = Hp; prob.w = Wp; prob.r = Rt; prob.s = St;
    prob.stride_h = 1; prob.stride_w = 1; prob.pad_h = Rt - 1; prob.pad_w = St - 1;
}

void dgrad_phases(int64_t H, int64_t W, int64_t R, int64_t S, int sh, int sw, int ph, int pw,
                  std::vector<DgradPhase>& out) {
    out.clear();
    for (int a = 0; a < sh; ++a)
        for (int b = 0; b < sw; ++b) {
            DgradPhase p;
            p.a = a;
            p.b = b;
            dgrad_phase_1d(H, R, sh, ph, a, p.Hp, p.Rt, p.r0, p.padh);
            dgrad_phase_1d(W, S, sw, pw, b, p.Wp, p.St, p.s0, p.padw);
            out.push_back(p);
        }
}

}  // namespace

// =============================================================================================
// C ABI
// =============================================================================================

extern "C" {

const char* sk_last_error(void) { return g_err; }

int sk_version(void) { return 100; }

int sk_set_tile(int tile) {
    if (tile != SK_TILE_AUTO && tile != SK_TILE_128 && tile != SK_TILE_256_PAIR &&
        tile != SK_TILE_256x256_PAIR)
        return fail(SK_ERR_UNSUPPORTED, "unknown tile setting %d", tile);
    const int prev = g_tile;
    g_tile = tile;
    return prev;
}

int sk_default_pool(int reduction, int num_sms, int ctas_per_sm, int* out) {
    if (!out) return fail(SK_ERR_UNSUPPORTED, "out is NULL");
    if (reduction == SK_REDUCTION_AUTO) reduction = SK_WORKSPACE;
    if (reduction < SK_LINEAR || reduction > SK_WORKSPACE)
        return fail(SK_ERR_UNSUPPORTED, "unknown streamk reduction %d", reduction);
    int64_t pool = 0;
    int rc = resolve_pool(reduction, -1, num_sms, ctas_per_sm, pool);
    if (rc) return rc;
    *out = static_cast<int>(pool);
    return SK_OK;
}

int sk_plan(const sk_problem* p, int streamk, int reduction, int ctas, int num_sms, sk_plan_t* out) {
    if (!p || !out) return fail(SK_ERR_UNSUPPORTED, "NULL argument");
    if (p->op == SK_OP_DGRAD && (p->stride_h > 1 || p->stride_w > 1))
        return fail(SK_ERR_UNSUPPORTED, "a strided dgrad runs one plan per output phase; "
                                        "sk_workspace_bytes covers them all");
    int per_sm = 1;
    if (ctas == -1 && num_sms <= 0) {
        DevInfo d;
        int rc = current_device_info(d);
        if (rc) return rc;
        num_sms = d.sms;
        View v;
        if (problem_view(*p, v) == SK_OK) {
            TileCfg tc;
            rc = tile_cfg(v, tc);
            if (rc) return rc;
            per_sm = sk::main_ctas_per_sm(v.op_kind, tc.cg, tc.tn, tc.st);
        }
    }
    return build_plan(*p, streamk, reduction, ctas, num_sms, per_sm, *out);
}

int sk_plan_cta_work(const sk_plan_t* plan, int64_t cta, sk_segment_t* out, int max_out, int* n_out) {
    if (!plan || !n_out || (max_out > 0 && !out)) return fail(SK_ERR_UNSUPPORTED, "NULL argument");
    if (cta < 0 || cta >= plan->grid) return fail(SK_ERR_UNSUPPORTED, "cta %lld outside the grid", (long long)cta);
    sk::SegCursor c;
    sk::seg_init(*plan, cta, c);
    sk_segment_t s;
    int n = 0;
    while (sk::seg_next(*plan, cta, c, s)) {
        if (n < max_out) out[n] = s;
        ++n;
    }
    *n_out = n;
    return SK_OK;
}

int sk_workspace_bytes(const sk_problem* p, int streamk, int reduction, int ctas, size_t* out) {
    if (!p || !out) return fail(SK_ERR_UNSUPPORTED, "NULL argument");
    if (p->op == SK_OP_DGRAD && (p->stride_h > 1 || p->stride_w > 1)) {
        // The phases' workspaces side by side (the phases may run at the same time), in the
        // pages' view as their launches take it.
        const TileGuard pages_view(g_tile == SK_TILE_AUTO ? SK_TILE_128 : g_tile);
        if (p->stride_h < 1 || p->stride_w < 1 || p->stride_h > 8 || p->stride_w > 8)
            return fail(SK_ERR_UNSUPPORTED, "stride must be in [1, 8]");
        std::vector<DgradPhase> phases;
        dgrad_phases(p->h, p->w, p->r, p->s, p->stride_h, p->stride_w, p->pad_h, p->pad_w, phases);
        size_t sum = 0;
        for (const DgradPhase& ph : phases) {
            if (!ph.live()) continue;
            sk_problem q = *p;
            set_phase_problem(q, ph.Hp, ph.Wp, ph.Rt, ph.St);
            sk_plan_t plan;
            const int rc = sk_plan(&q, streamk, reduction, ctas, 0, &plan);
            if (rc) return rc;
            sum += static_cast<size_t>(sk::round_up(plan.ws_bytes, 256));
        }
        *out = sum;
        return SK_OK;
    }
    sk_plan_t plan;
    int rc = sk_plan(p, streamk, reduction, ctas, 0, &plan);
    if (rc) return rc;
    *out = static_cast<size_t>(plan.ws_bytes);
    return SK_OK;
}

int sk_gemm_rcr(int ab_dtype, int c_dtype, int64_t M, int64_t N, int64_t K, const void* A,
                int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, int streamk,
                int reduction, int ctas, void* ws, size_t ws_bytes, void* stream) {
    if (ab_dtype != SK_F16 && ab_dtype != SK_BF16)
        return fail(SK_ERR_UNSUPPORTED, "GEMM inputs must be f16 or bf16, got %s", dtype_name(ab_dtype));
    if (c_dtype != ab_dtype && c_dtype != SK_F32)
        return fail(SK_ERR_UNSUPPORTED, "GEMM output must be %s or f32, got %s", dtype_name(ab_dtype),
                    dtype_name(c_dtype));
    int rc = check_common(streamk, reduction, ctas, c_dtype);
    if (rc) return rc;
    if (M < 0 || N < 0 || K < 0) return fail(SK_ERR_UNSUPPORTED, "negative size");
    if (M == 0 || N == 0) return SK_OK;   // nothing to write
    if (!C || (K > 0 && (!A || !B))) return fail(SK_ERR_UNSUPPORTED, "NULL pointer");
    const int cs = dtype_size(c_dtype);
    if (K % 8 != 0) return fail(SK_ERR_UNSUPPORTED, "K must be a multiple of 8 (16-byte rows), got %lld", (long long)K);
    if (ldc < N || (K > 0 && (lda < K || ldb < K)))
        return fail(SK_ERR_UNSUPPORTED, "leading dimension smaller than the row");
    if ((ldc * cs) % 16 || (K > 0 && ((lda * 2) % 16 || (ldb * 2) % 16)))
        return fail(SK_ERR_UNSUPPORTED, "lda, ldb and ldc rows must be multiples of 16 bytes");
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B))))
        return fail(SK_ERR_UNSUPPORTED, "A, B and C must be 16-byte aligned");
    rc = select_device_of(C);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {   // empty reduction: C = 0
        cudaError_t e = cudaMemset2DAsync(C, static_cast<size_t>(ldc * cs), 0,
                                          static_cast<size_t>(N * cs), static_cast<size_t>(M), st);
        return e == cudaSuccess ? SK_OK : cuda_fail(e, "cudaMemset2DAsync(C)");
    }
    rc = load_encoders();
    if (rc) return rc;
    sk_problem prob;
    memset(&prob, 0, sizeof(prob));
    prob.op = SK_OP_GEMM;
    prob.ab_dtype = ab_dtype;
    prob.c_dtype = c_dtype;
    prob.M = M;
    prob.N = N;
    prob.K = K;
    prob.groups = 1;
    TileCfg tc;
    rc = problem_tile(prob, tc);
    if (rc) return rc;
    sk::KernelParams kp;
    memset(&kp, 0, sizeof(kp));
    // Each CTA stages 128 rows of A and tile_n / cg rows of B per step.
    rc = encode_2d(&kp.tmap_a, A, 2, K, M, lda * 2, 64, 128);
    if (rc) return rc;
    rc = encode_2d(&kp.tmap_b, B, 2, K, N, ldb * 2, 64, static_cast<uint32_t>(tc.tn / tc.cg));
    if (rc) return rc;
    kp.c = C;
    kp.ldc = ldc;
    kp.c_dtype = c_dtype;
    if (c_dtype != SK_F32) {   // 16-bit C: complete tiles leave through TMA tile stores
        rc = encode_2d(&kp.tmap_c, C, 2, N, M, ldc * 2, 64, 32);
        if (rc) return rc;
        kp.c_tma = 1;
    }
    const uint32_t fmt = ab_dtype == SK_BF16 ? 1u : 0u;
    kp.idesc = sk::make_idesc(fmt, fmt, false, false, static_cast<uint32_t>(sk::kTileM * tc.cg),
                              static_cast<uint32_t>(tc.tn));
    return run(prob, streamk, reduction, ctas, kp, C, ldc * cs, M, N * cs, ws, ws_bytes, st);
}

namespace {

struct BlockScales {   // the block-scaled form; blocked == false for the other two
    bool blocked = false;
    const float* sa = nullptr;
    const float* sb = nullptr;
    int64_t gka = 0, gnb = 0, gkb = 0;
};

// The fp8 GEMM with per-row / per-column scales (sa, sb), per-tensor scales (sa == sb == null,
// `scale` = scale_a * scale_b), or block scales (`bs.blocked`; sa == sb == null here, the block
// scales travel in `bs`).
int fp8_gemm(int64_t M, int64_t N, int64_t K, const void* A8, const void* B8, const float* sa,
             const float* sb, float scale, void* C_bf16, int64_t ldc, int streamk, int reduction,
             int ctas, void* ws, size_t ws_bytes, void* stream, const BlockScales& bs = BlockScales()) {
    int rc = check_common(streamk, reduction, ctas, SK_BF16);
    if (rc) return rc;
    if (M < 0 || N < 0 || K < 0) return fail(SK_ERR_UNSUPPORTED, "negative size");
    if (M == 0 || N == 0) return SK_OK;
    if (!A8 || !B8 || !C_bf16 || (sa == nullptr) != (sb == nullptr))
        return fail(SK_ERR_UNSUPPORTED, "NULL pointer");
    if (K < 16 || K % 16 != 0) return fail(SK_ERR_UNSUPPORTED, "K must be a positive multiple of 16, got %lld", (long long)K);
    if (ldc < N || (ldc * 2) % 16) return fail(SK_ERR_UNSUPPORTED, "ldc must be >= N with 16-byte rows");
    if (!aligned16(A8) || !aligned16(B8) || !aligned16(C_bf16))
        return fail(SK_ERR_UNSUPPORTED, "A8, B8 and C must be 16-byte aligned");
    rc = select_device_of(C_bf16);
    if (rc) return rc;
    rc = load_encoders();
    if (rc) return rc;
    sk_problem prob;
    memset(&prob, 0, sizeof(prob));
    prob.op = bs.blocked ? SK_OP_FP8_BLOCK : SK_OP_FP8_ROWCOL;
    prob.ab_dtype = SK_E4M3;
    prob.c_dtype = SK_BF16;
    prob.M = M;
    prob.N = N;
    prob.K = K;
    prob.groups = 1;
    TileCfg tc;
    rc = problem_tile(prob, tc);
    if (rc) return rc;
    sk::KernelParams kp;
    memset(&kp, 0, sizeof(kp));
    rc = encode_2d(&kp.tmap_a, A8, 1, K, M, K, 128, 128);
    if (rc) return rc;
    rc = encode_2d(&kp.tmap_b, B8, 1, K, N, K, 128, static_cast<uint32_t>(tc.tn / tc.cg));
    if (rc) return rc;
    kp.c = C_bf16;
    kp.ldc = ldc;
    kp.c_dtype = SK_BF16;
    rc = encode_2d(&kp.tmap_c, C_bf16, 2, N, M, ldc * 2, 64, 32);
    if (rc) return rc;
    kp.c_tma = 1;
    kp.sa = sa;
    kp.sb = sb;
    kp.scale = scale;
    if (bs.blocked) {
        kp.bsa = bs.sa;
        kp.bsb = bs.sb;
        kp.nka = bs.sa ? sk::ceil_div(K, bs.gka) : 0;
        kp.nkb = bs.sb ? sk::ceil_div(K, bs.gkb) : 0;
        kp.gka = static_cast<int32_t>(bs.sa ? bs.gka : 128);
        kp.gnb = static_cast<int32_t>(bs.sb ? bs.gnb : 128);
        kp.gkb = static_cast<int32_t>(bs.sb ? bs.gkb : 128);
    }
    kp.idesc = sk::make_idesc(0, 0, false, false, static_cast<uint32_t>(sk::kTileM * tc.cg),
                              static_cast<uint32_t>(tc.tn));
    return run(prob, streamk, reduction, ctas, kp, C_bf16, ldc * 2, M, N * 2, ws, ws_bytes,
               static_cast<cudaStream_t>(stream));
}

}  // namespace

int sk_gemm_rowcol_fp8(int64_t M, int64_t N, int64_t K, const void* A8, const void* B8,
                       const float* sa, const float* sb, void* C_bf16, int64_t ldc, int streamk,
                       int reduction, int ctas, void* ws, size_t ws_bytes, void* stream) {
    if (M > 0 && N > 0 && (!sa || !sb)) return fail(SK_ERR_UNSUPPORTED, "NULL pointer");
    return fp8_gemm(M, N, K, A8, B8, sa, sb, 1.0f, C_bf16, ldc, streamk, reduction, ctas, ws,
                    ws_bytes, stream);
}

int sk_gemm_tensorquant_fp8(int64_t M, int64_t N, int64_t K, const void* A8, const void* B8,
                            float scale_a, float scale_b, void* C_bf16, int64_t ldc, int streamk,
                            int reduction, int ctas, void* ws, size_t ws_bytes, void* stream) {
    return fp8_gemm(M, N, K, A8, B8, nullptr, nullptr, scale_a * scale_b, C_bf16, ldc, streamk,
                    reduction, ctas, ws, ws_bytes, stream);
}

int sk_gemm_blockscale_fp8(int64_t M, int64_t N, int64_t K, const void* A8, const void* B8,
                           const float* sa, int64_t a_group_k, const float* sb, int64_t b_group_n,
                           int64_t b_group_k, void* C_bf16, int64_t ldc, int streamk,
                           int reduction, int ctas, void* ws, size_t ws_bytes, void* stream) {
    if (sa && (a_group_k < 128 || a_group_k % 128 != 0 || a_group_k > 0x40000000LL))
        return fail(SK_ERR_UNSUPPORTED, "a_group_k must be a positive multiple of 128, got %lld",
                    (long long)a_group_k);
    if (sb && (b_group_k < 128 || b_group_k % 128 != 0 || b_group_k > 0x40000000LL))
        return fail(SK_ERR_UNSUPPORTED, "b_group_k must be a positive multiple of 128, got %lld",
                    (long long)b_group_k);
    if (sb && (b_group_n < 128 || b_group_n % 128 != 0 || b_group_n > 0x40000000LL))
        return fail(SK_ERR_UNSUPPORTED, "b_group_n must be a positive multiple of 128, got %lld",
                    (long long)b_group_n);
    BlockScales bs;
    bs.blocked = true;
    bs.sa = sa;
    bs.sb = sb;
    bs.gka = a_group_k;
    bs.gnb = b_group_n;
    bs.gkb = b_group_k;
    return fp8_gemm(M, N, K, A8, B8, nullptr, nullptr, 1.0f, C_bf16, ldc, streamk, reduction, ctas,
                    ws, ws_bytes, stream, bs);
}

int sk_conv2d_wgrad_nhwc(int in_dtype, int dw_dtype, int64_t N, int64_t H, int64_t W, int64_t C,
                         int64_t K, int64_t R, int64_t S, int stride_h, int stride_w, int pad_h,
                         int pad_w, int groups, const void* x, const void* dy, void* dw,
                         int streamk, int reduction, int ctas, void* ws, size_t ws_bytes,
                         void* stream) {
    if (in_dtype != SK_F16 && in_dtype != SK_BF16)
        return fail(SK_ERR_UNSUPPORTED, "wgrad inputs must be f16 or bf16, got %s", dtype_name(in_dtype));
    if (dw_dtype != SK_F32 && dw_dtype != in_dtype)
        return fail(SK_ERR_UNSUPPORTED, "dW must be f32 or %s, got %s", dtype_name(in_dtype),
                    dtype_name(dw_dtype));
    int rc = check_common(streamk, reduction, ctas, dw_dtype);
    if (rc) return rc;
    if (N < 0 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1)
        return fail(SK_ERR_UNSUPPORTED, "sizes must be positive");
    if (groups < 1 || C % groups || K % groups)
        return fail(SK_ERR_UNSUPPORTED, "groups must divide C and K");
    if (stride_h < 1 || stride_w < 1 || stride_h > 8 || stride_w > 8)
        return fail(SK_ERR_UNSUPPORTED, "stride must be in [1, 8]");
    if (pad_h < 0 || pad_w < 0 || pad_h >= R || pad_w >= S)
        return fail(SK_ERR_UNSUPPORTED, "padding must be in [0, filter size)");
    if (R > 16 || S > 16) return fail(SK_ERR_UNSUPPORTED, "filter taps beyond 16 are not supported");
    const int64_t Cg = C / groups, Kg = K / groups;
    if (Cg % 64) return fail(SK_ERR_UNSUPPORTED, "channels per group must be a multiple of 64, got %lld", (long long)Cg);
    if (Kg % 8) return fail(SK_ERR_UNSUPPORTED, "filters per group must be a multiple of 8, got %lld", (long long)Kg);
    const int64_t Ho = (H + 2 * pad_h - R) / stride_h + 1;
    const int64_t Wo = (W + 2 * pad_w - S) / stride_w + 1;
    if (H + 2 * pad_h < R || W + 2 * pad_w < S || Ho < 1 || Wo < 1)
        return fail(SK_ERR_UNSUPPORTED, "filter larger than the padded image");
    const int64_t up_w = (Wo - 1) * stride_w - pad_w - (W - 1);
    const int64_t up_h = (Ho - 1) * stride_h - pad_h - (H - 1);
    if (up_w < -128 || up_h < -128 || up_w > 127 || up_h > 127 || -pad_w < -128 || -pad_h < -128)
        return fail(SK_ERR_UNSUPPORTED, "im2col bounding box outside the 4-D TMA range");
    if (N * Ho * Wo + 64 >= (int64_t(1) << 31) || N >= (int64_t(1) << 31))
        return fail(SK_ERR_UNSUPPORTED, "too many output pixels (N*Ho*Wo must stay below 2^31 - 64)");
    if (!x || !dy || !dw) return fail(SK_ERR_UNSUPPORTED, "NULL pointer");
    if (!aligned16(x) || !aligned16(dy) || !aligned16(dw))
        return fail(SK_ERR_UNSUPPORTED, "x, dy and dw must be 16-byte aligned");
    const int64_t RSC = R * S * Cg;
    const int cs = dtype_size(dw_dtype);
    if (N == 0) {   // empty reduction: dW = 0
        rc = select_device_of(dw);
        if (rc) return rc;
        cudaError_t e = cudaMemsetAsync(dw, 0, static_cast<size_t>(K * RSC * cs), static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? SK_OK : cuda_fail(e, "cudaMemsetAsync(dw)");
    }
    rc = select_device_of(dw);
    if (rc) return rc;
    rc = load_encoders();
    if (rc) return rc;
    sk_problem prob;
    memset(&prob, 0, sizeof(prob));
    prob.op = SK_OP_WGRAD;
    prob.ab_dtype = in_dtype;
    prob.c_dtype = dw_dtype;
    prob.n = N; prob.h = H; prob.w = W; prob.c = C; prob.k = K; prob.r = R; prob.s = S;
    prob.stride_h = stride_h; prob.stride_w = stride_w; prob.pad_h = pad_h; prob.pad_w = pad_w;
    prob.groups = groups;
    sk::KernelParams kp;
    memset(&kp, 0, sizeof(kp));
    const uint32_t fmt = in_dtype == SK_BF16 ? 1u : 0u;
    View view;
    rc = problem_view(prob, view);
    if (rc) return rc;
    RowGeom rg;
    if (sk::is_wgrad_row(view.op_kind) && wgrad_row_geom(prob, rg)) {
        // Shifted-row wgrad. A: x rows of 64 channels, `wseg` positions at column stride sw and
        // `rows_per_step` rows at row stride sh (the traversal strides of the map), from any
        // (column, row) start: outside the image reads zeros. B: dy rows of 64 filters.
        TileCfg tc;
        rc = tile_cfg(view, tc);
        if (rc) return rc;
        // Ring stage: the most K steps (at most 8, at most one image's) whose boxes fit the stage:
        // per column phase the x rows (a CTA pair with sh = 1: one box of T * rows_per_step + 1
        // rows holding both tap rows; else one box of T * rows_per_step rows per tap row), then
        // the dy rows with 16 zero rows after them; every box 1024-byte aligned.
        const int64_t dy_row = 128 / tc.cg;
        const int64_t cap = sk::wgrow_stage_bytes(view.op_kind, tc.cg);
        const int64_t steps_per_image = rg.ho_pad / rg.rows_per_step;
        int64_t T = 0, x_phase = 0;
        // The one-CTA kernel keeps a box per tap row (measured faster there than one box of
        // both: 0.27 against 0.44 us per step on the 32x56x56 wgrad).
        const bool shared_box = stride_h == 1 && tc.cg == 2;
        for (int64_t t = sk::imin(8, steps_per_image); t >= 1 && T == 0; --t) {
            const int64_t rows = t * rg.rows_per_step;
            if (rows + 1 > 256 || rows * stride_h > 256) continue;   // TMA box dimensions
            const int64_t xp = shared_box ? sk::round_up((rows + 1) * rg.wseg * 128, 1024)
                                          : 2 * t * 8192;
            const int64_t dy = sk::round_up((t * 64 + 16) * dy_row, 1024);
            if (stride_w * xp + dy <= cap) {
                T = t;
                x_phase = xp;
            }
        }
        if (T == 0) return fail(SK_ERR_UNSUPPORTED, "shifted-row wgrad stage does not fit");
        kp.conv.stage_steps = static_cast<int32_t>(T);
        kp.conv.x_lbo = static_cast<int32_t>(shared_box ? rg.wseg * 128 : T * 8192);
        kp.conv.x_shared_box = shared_box ? 1 : 0;
        kp.conv.x_phase_bytes = static_cast<int32_t>(x_phase);
        kp.conv.dy_off = static_cast<int32_t>(stride_w * x_phase);
        {
            const cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
            const cuuint64_t strides[3] = {(cuuint64_t)(C * 2), (cuuint64_t)(W * C * 2),
                                           (cuuint64_t)(H * W * C * 2)};
            // The box spans sh image rows per loaded row (the traversal stride takes every sh-th).
            const cuuint32_t box[4] = {64, (cuuint32_t)(rg.wseg * stride_w),
                                       (cuuint32_t)(shared_box ? T * rg.rows_per_step + 1
                                                               : T * rg.rows_per_step * stride_h),
                                       1};
            const cuuint32_t estr[4] = {1, (cuuint32_t)stride_w, (cuuint32_t)stride_h, 1};
            CUresult r = g_encode_tiled(&kp.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                                        const_cast<void*>(x), dims, strides, box, estr,
                                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return fail(SK_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(x) failed (%d)", (int)r);
        }
        {
            // A CTA pair splits the filters: each CTA reads rows of 32 (64 bytes, 64-byte swizzle).
            const cuuint64_t dims[4] = {(cuuint64_t)K, (cuuint64_t)Wo, (cuuint64_t)Ho, (cuuint64_t)N};
            const cuuint64_t strides[3] = {(cuuint64_t)(K * 2), (cuuint64_t)(Wo * K * 2),
                                           (cuuint64_t)(Ho * Wo * K * 2)};
            const cuuint32_t box[4] = {(cuuint32_t)(64 / tc.cg), (cuuint32_t)rg.wseg,
                                       (cuuint32_t)(T * rg.rows_per_step), 1};
            const cuuint32_t estr[4] = {1, 1, 1, 1};
            CUresult r = g_encode_tiled(&kp.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                                        const_cast<void*>(dy), dims, strides, box, estr,
                                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                                        tc.cg == 2 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return fail(SK_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(dy) failed (%d)", (int)r);
        }
        kp.c = dw;
        kp.ldc = RSC;
        kp.c_dtype = dw_dtype;
        // M = 128 per CTA (two tap rows x 64 channels; 256 for a pair), both operands MN-major; the
        // kernel sets N per column phase.
        kp.idesc = sk::make_idesc(fmt, fmt, true, true, static_cast<uint32_t>(128 * tc.cg),
                                  static_cast<uint32_t>(64 * rg.nq[0]));
        kp.conv.fsplit = tc.cg;
        kp.conv.sh = stride_h;
        kp.conv.sw = stride_w;
        kp.conv.ph = pad_h;
        kp.conv.pw = pad_w;
        kp.conv.R = static_cast<int32_t>(R);
        kp.conv.S = static_cast<int32_t>(S);
        kp.conv.Cg = static_cast<int32_t>(Cg);
        kp.conv.Kg = static_cast<int32_t>(Kg);
        kp.conv.ho = static_cast<int32_t>(rg.ho);
        kp.conv.ho_pad = static_cast<int32_t>(rg.ho_pad);
        kp.conv.rows_per_step = rg.rows_per_step;
        kp.conv.wseg = rg.wseg;
        kp.conv.qmax = rg.qmax;
        kp.conv.nq[0] = rg.nq[0];
        kp.conv.nq[1] = rg.nq[1];
        return run(prob, streamk, reduction, ctas, kp, dw, RSC * cs, K, RSC * cs, ws, ws_bytes,
                   static_cast<cudaStream_t>(stream));
    }
    // dy as a [N*Ho*Wo][K] matrix: 64-filter x 64-pixel boxes (MN-major operand)
    rc = encode_2d(&kp.tmap_a, dy, 2, K, N * Ho * Wo, K * 2, 64, 64);
    if (rc) return rc;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
        const cuuint64_t strides[3] = {(cuuint64_t)(C * 2), (cuuint64_t)(W * C * 2),
                                       (cuuint64_t)(H * W * C * 2)};
        const int lower[2] = {-pad_w, -pad_h};
        const int upper[2] = {static_cast<int>(up_w), static_cast<int>(up_h)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)stride_w, (cuuint32_t)stride_h, 1};
        CUresult r = g_encode_im2col(&kp.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                                     const_cast<void*>(x), dims, strides, lower, upper, 64, 64, estr,
                                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(SK_ERR_UNSUPPORTED, "cuTensorMapEncodeIm2col failed (%d)", (int)r);
    }
    kp.c = dw;
    kp.ldc = RSC;
    kp.c_dtype = dw_dtype;
    kp.idesc = sk::make_idesc(fmt, fmt, true, true, 128, static_cast<uint32_t>(sk::kTileN));
    kp.conv.HoWo = Ho * Wo;
    kp.conv.Wo = static_cast<int32_t>(Wo);
    kp.conv.sh = stride_h;
    kp.conv.sw = stride_w;
    kp.conv.ph = pad_h;
    kp.conv.pw = pad_w;
    kp.conv.R = static_cast<int32_t>(R);
    kp.conv.S = static_cast<int32_t>(S);
    kp.conv.Cg = static_cast<int32_t>(Cg);
    kp.conv.Kg = static_cast<int32_t>(Kg);
    return run(prob, streamk, reduction, ctas, kp, dw, RSC * cs, K, RSC * cs, ws, ws_bytes,
               static_cast<cudaStream_t>(stream));
}

namespace {

// Shared checks and set-up of the forward-convolution and data-gradient calls. `act` is the
// im2col'd activation (x for fprop, dy for dgrad) of shape [N][AH][AW][AC]; the traversal runs
// over a TH x TW grid with stride (tsh, tsw) and padding (tph, tpw).
int conv_fwd_like(int op, int in_dtype, int out_dtype, int64_t N, int64_t H, int64_t W, int64_t C,
                  int64_t K, int64_t R, int64_t S, int stride_h, int stride_w, int pad_h, int pad_w,
                  int groups, const void* act, const void* wt, void* out, int streamk,
                  int reduction, int ctas, void* ws, size_t ws_bytes, void* stream) {
    const bool fprop = op == SK_OP_FPROP;
    const char* name = fprop ? "fprop" : "dgrad";
    if (in_dtype != SK_F16 && in_dtype != SK_BF16)
        return fail(SK_ERR_UNSUPPORTED, "%s inputs must be f16 or bf16, got %s", name, dtype_name(in_dtype));
    if (out_dtype != SK_F32 && out_dtype != in_dtype)
        return fail(SK_ERR_UNSUPPORTED, "%s output must be f32 or %s, got %s", name,
                    dtype_name(in_dtype), dtype_name(out_dtype));
    int rc = check_common(streamk, reduction, ctas, out_dtype);
    if (rc) return rc;
    if (N < 0 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1)
        return fail(SK_ERR_UNSUPPORTED, "sizes must be positive");
    if (groups < 1 || C % groups || K % groups)
        return fail(SK_ERR_UNSUPPORTED, "groups must divide C and K");
    if (stride_h < 1 || stride_w < 1 || stride_h > 8 || stride_w > 8)
        return fail(SK_ERR_UNSUPPORTED, "stride must be in [1, 8]");
    if (pad_h < 0 || pad_w < 0 || pad_h >= R || pad_w >= S)
        return fail(SK_ERR_UNSUPPORTED, "padding must be in [0, filter size)");
    if (R > 16 || S > 16) return fail(SK_ERR_UNSUPPORTED, "filter taps beyond 16 are not supported");
    const int64_t Cg = C / groups, Kg = K / groups;
    const int64_t red_ch = fprop ? Cg : Kg;   // channels per group the reduction walks
    if (red_ch % 64)
        return fail(SK_ERR_UNSUPPORTED, "%s per group must be a multiple of 64, got %lld",
                    fprop ? "channels" : "filters", (long long)red_ch);
    if (C % 8 || K % 8 || Cg % 8)
        return fail(SK_ERR_UNSUPPORTED, "C, K and C/groups must be multiples of 8 (16-byte rows)");
    const int64_t Ho = (H + 2 * pad_h - R) / stride_h + 1;
    const int64_t Wo = (W + 2 * pad_w - S) / stride_w + 1;
    if (H + 2 * pad_h < R || W + 2 * pad_w < S || Ho < 1 || Wo < 1)
        return fail(SK_ERR_UNSUPPORTED, "filter larger than the padded image");
    const bool phased = !fprop && (stride_h > 1 || stride_w > 1);
    std::vector<DgradPhase> phases;
    if (phased) dgrad_phases(H, W, R, S, stride_h, stride_w, pad_h, pad_w, phases);
    // Every launch's im2col bounding box and pixel count must fit the TMA and the 32-bit pixel
    // index, checked before anything is enqueued.
    auto box_ok = [&](int64_t AH, int64_t AW, int64_t TH, int64_t TW, int tsh, int tsw, int tph,
                      int tpw) {
        const int64_t up_w = (TW - 1) * tsw - tpw - (AW - 1);
        const int64_t up_h = (TH - 1) * tsh - tph - (AH - 1);
        return !(up_w < -128 || up_h < -128 || up_w > 127 || up_h > 127 || -tpw < -128 ||
                 -tph < -128 || -tpw > 127 || -tph > 127) &&
               N * TH * TW + 128 < (int64_t(1) << 31);
    };
    if (N >= (int64_t(1) << 31)) return fail(SK_ERR_UNSUPPORTED, "too many images");
    if (!phased) {
        const bool ok = fprop ? box_ok(H, W, Ho, Wo, stride_h, stride_w, pad_h, pad_w)
                              : box_ok(Ho, Wo, H, W, 1, 1, static_cast<int>(R - 1 - pad_h),
                                       static_cast<int>(S - 1 - pad_w));
        if (!ok) return fail(SK_ERR_UNSUPPORTED, "im2col bounding box or pixel count outside the TMA range");
    } else {
        for (const DgradPhase& ph : phases)
            if (ph.live() && !box_ok(Ho, Wo, ph.Hp, ph.Wp, 1, 1, ph.padh, ph.padw))
                return fail(SK_ERR_UNSUPPORTED, "im2col bounding box or pixel count outside the TMA range");
    }
    if (!act || !wt || !out) return fail(SK_ERR_UNSUPPORTED, "NULL pointer");
    if (!aligned16(act) || !aligned16(wt) || !aligned16(out))
        return fail(SK_ERR_UNSUPPORTED, "activations, filter and output must be 16-byte aligned");
    rc = select_device_of(out);
    if (rc) return rc;
    if (N == 0) return SK_OK;   // no pixels: nothing to write
    rc = load_encoders();
    if (rc) return rc;
    const int cs = dtype_size(out_dtype);
    const int64_t ldc = fprop ? K : C;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // One implicit GEMM over a traversal grid TH x TW of the activation AH x AW (channels AC).
    auto launch = [&](int64_t AH, int64_t AW, int64_t TH, int64_t TW, int tsh, int tsw, int tph,
                      int tpw, int Rt, int St, int r0, int s0, const sk::RowMap& rows,
                      bool zeroed, int chain = 0, void* lws = nullptr, size_t lws_bytes = 0,
                      int part = 0, bool own_slice = false) -> int {
        // The im2col kernel serves the pages' view: a dgrad phase problem that fits the shifted-row
        // view keeps the 128 x 128 tile (the automatic tile's choice for the pages' view).
        const TileGuard pages_view(g_tile == SK_TILE_AUTO ? SK_TILE_128 : g_tile);
        const int64_t AC = fprop ? C : K;
        sk_problem prob;
        memset(&prob, 0, sizeof(prob));
        prob.op = op;
        prob.ab_dtype = in_dtype;
        prob.c_dtype = out_dtype;
        prob.n = N; prob.c = C; prob.k = K; prob.groups = groups;
        if (rows.on) {   // a dgrad phase: its traversal grid and taps, as a stride-1 problem
            set_phase_problem(prob, TH, TW, Rt, St);
        } else {
            prob.h = H; prob.w = W; prob.r = R; prob.s = S;
            prob.stride_h = stride_h; prob.stride_w = stride_w; prob.pad_h = pad_h; prob.pad_w = pad_w;
        }
        sk::KernelParams kp;
        memset(&kp, 0, sizeof(kp));
        {   // A: im2col of the activation, 128 pixels x 64 channels per load (K-major)
            const cuuint64_t dims[4] = {(cuuint64_t)AC, (cuuint64_t)AW, (cuuint64_t)AH, (cuuint64_t)N};
            const cuuint64_t strides[3] = {(cuuint64_t)(AC * 2), (cuuint64_t)(AW * AC * 2),
                                           (cuuint64_t)(AH * AW * AC * 2)};
            const int lower[2] = {-tpw, -tph};
            const int upper[2] = {static_cast<int>((TW - 1) * tsw - tpw - (AW - 1)),
                                  static_cast<int>((TH - 1) * tsh - tph - (AH - 1))};
            const cuuint32_t estr[4] = {1, (cuuint32_t)tsw, (cuuint32_t)tsh, 1};
            CUresult r = g_encode_im2col(&kp.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                                         const_cast<void*>(act), dims, strides, lower, upper, 64,
                                         128, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                         CU_TENSOR_MAP_SWIZZLE_128B,
                                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS)
                return fail(SK_ERR_UNSUPPORTED, "cuTensorMapEncodeIm2col failed (%d)", (int)r);
        }
        // B: the filter as [K][R*S*C/G]; fprop 64 x 128-row boxes (K-major), dgrad 64 x 64 boxes
        // (two per step, MN-major).
        const int64_t Cg = C / groups;
        const int64_t RSC = R * S * Cg;
        int rc2 = encode_2d(&kp.tmap_b, wt, 2, RSC, K, RSC * 2, 64, fprop ? 128 : 64);
        if (rc2) return rc2;
        const int64_t pixels = N * TH * TW;
        kp.c = out;
        kp.ldc = ldc;
        kp.c_dtype = out_dtype;
        // One group and contiguous rows: complete tiles leave through TMA tile stores.
        if (out_dtype != SK_F32 && groups == 1 && !rows.on) {
            rc2 = encode_2d(&kp.tmap_c, out, 2, ldc, pixels, ldc * 2, 64, 32);
            if (rc2) return rc2;
            kp.c_tma = 1;
        }
        const uint32_t fmt = in_dtype == SK_BF16 ? 1u : 0u;
        kp.idesc = sk::make_idesc(fmt, fmt, false, !fprop, 128, static_cast<uint32_t>(sk::kTileN));
        kp.conv.HoWo = TH * TW;
        kp.conv.Wo = static_cast<int32_t>(TW);
        kp.conv.sh = tsh;
        kp.conv.sw = tsw;
        kp.conv.ph = tph;
        kp.conv.pw = tpw;
        kp.conv.R = Rt;
        kp.conv.S = St;
        kp.conv.r0 = r0;
        kp.conv.s0 = s0;
        kp.conv.dsh = rows.on ? stride_h : 1;
        kp.conv.dsw = rows.on ? stride_w : 1;
        kp.conv.Sf = static_cast<int32_t>(S);
        kp.conv.Cg = static_cast<int32_t>(red_ch);
        kp.conv.Kg = static_cast<int32_t>(Kg);
        kp.conv.Cw = static_cast<int32_t>(Cg);
        kp.conv.rows = rows;
        kp.pdl_chain = chain;
        // A dgrad phase writes scattered rows of dx, zeroed beforehand when needed: no per-launch
        // zeroing of a row range (out_rows 0).
        return run(prob, streamk, reduction, ctas, kp, out, ldc * cs, zeroed ? 0 : pixels, ldc * cs,
                   own_slice ? lws : ws, own_slice ? lws_bytes : ws_bytes, st, part);
    };

    // The shifted-row kernel over the activation (AH x AW, 64 channels) into the TH x TW output
    // (64 channels) with padding (tph, tpw). A: boxes of 64 channels x 64 positions (from column
    // -tpw) x R + 1 rows (from row ho0 - tph); outside the activation reads zeros. B: the filter's
    // taps [tap][filter][channel] of w[K][R][S][C]: for fprop (output channel = filter) K-major,
    // for dgrad (output channel = channel, the taps flipped) MN-major.
    auto row_launch = [&](const sk_problem& prob, int64_t AH, int64_t AW, int64_t TH, int64_t TW,
                          int tph, int tpw, bool flip) -> int {
        sk::KernelParams kp;
        memset(&kp, 0, sizeof(kp));
        {
            const cuuint64_t dims[4] = {64, (cuuint64_t)AW, (cuuint64_t)AH, (cuuint64_t)N};
            const cuuint64_t strides[3] = {128, (cuuint64_t)(AW * 128), (cuuint64_t)(AH * AW * 128)};
            const cuuint32_t box[4] = {64, 64, (cuuint32_t)(R + 1), 1};
            const cuuint32_t estr[4] = {1, 1, 1, 1};
            CUresult r = g_encode_tiled(&kp.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4,
                                        const_cast<void*>(act), dims, strides, box, estr,
                                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS)
                return fail(SK_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(activation) failed (%d)", (int)r);
        }
        // The filter as one box (strides: a filter R*S*64 * 2 bytes, a tap 128 bytes), else one
        // [K][R*S*64] box per tap.
        const int64_t RSC = R * S * 64;
        {
            const cuuint64_t dims[3] = {64, 64, (cuuint64_t)(R * S)};
            const cuuint64_t strides[2] = {(cuuint64_t)(RSC * 2), 128};
            const cuuint32_t box[3] = {64, 64, (cuuint32_t)(R * S)};
            const cuuint32_t estr[3] = {1, 1, 1};
            kp.conv.filter_box =
                g_encode_tiled(&kp.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(wt),
                               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
        if (!kp.conv.filter_box) {
            int rc2 = encode_2d(&kp.tmap_b, wt, 2, RSC, 64, RSC * 2, 64, 64);
            if (rc2) return rc2;
        }
        kp.c = out;
        kp.ldc = 64;
        kp.c_dtype = out_dtype;
        // A 16-bit output leaves through TMA tile stores: [N][TH][TW][64], boxes of 32 positions x
        // 64 channels; the map clips the positions past TW.
        if (out_dtype != SK_F32) {
            const cuuint64_t dims[4] = {64, (cuuint64_t)TW, (cuuint64_t)TH, (cuuint64_t)N};
            const cuuint64_t strides[3] = {128, (cuuint64_t)(TW * 128), (cuuint64_t)(TH * TW * 128)};
            const cuuint32_t box[4] = {64, 32, 1, 1};
            const cuuint32_t estr[4] = {1, 1, 1, 1};
            CUresult r = g_encode_tiled(&kp.tmap_c, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, out, dims,
                                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                        CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS)
                return fail(SK_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(output) failed (%d)", (int)r);
            kp.c_tma = 1;
        }
        const uint32_t fmt = in_dtype == SK_BF16 ? 1u : 0u;
        kp.idesc = sk::make_idesc(fmt, fmt, false, flip, 128, 64);
        kp.conv.row_flip = flip ? 1 : 0;
        kp.conv.ph = tph;
        kp.conv.pw = tpw;
        kp.conv.sh = 1;
        kp.conv.sw = 1;
        kp.conv.R = static_cast<int32_t>(R);
        kp.conv.S = static_cast<int32_t>(S);
        kp.conv.Cg = 64;
        kp.conv.Kg = 64;
        kp.conv.Cw = 64;
        const int64_t th_pad = sk::round_up(TH, 2);
        kp.conv.ho = static_cast<int32_t>(TH);
        kp.conv.ho_pad = static_cast<int32_t>(th_pad);
        // Tile rows are (image, row over th_pad, position over 64): an output pixel when the row
        // is below TH and the position below TW.
        kp.conv.rows.on = 1;
        kp.conv.rows.HoWo = th_pad * 64;
        kp.conv.rows.Wo = 64;
        kp.conv.rows.Hd = static_cast<int32_t>(TH);
        kp.conv.rows.Wd = static_cast<int32_t>(TW);
        kp.conv.rows.dsh = 1;
        kp.conv.rows.dsw = 1;
        kp.conv.rows.vh = static_cast<int32_t>(TH);
        kp.conv.rows.vw = static_cast<int32_t>(TW);
        return run(prob, streamk, reduction, ctas, kp, out, 64 * cs, N * TH * TW, 64 * cs, ws,
                   ws_bytes, st);
    };

    sk::RowMap identity;
    memset(&identity, 0, sizeof(identity));
    {
        sk_problem whole;
        memset(&whole, 0, sizeof(whole));
        whole.op = op;
        whole.ab_dtype = in_dtype;
        whole.c_dtype = out_dtype;
        whole.n = N; whole.h = H; whole.w = W; whole.c = C; whole.k = K; whole.r = R; whole.s = S;
        whole.stride_h = stride_h; whole.stride_w = stride_w; whole.pad_h = pad_h; whole.pad_w = pad_w;
        whole.groups = groups;
        int64_t th, tw, th_pad;
        if (g_tile == SK_TILE_AUTO && conv_row_geom(whole, th, tw, th_pad))
            return fprop ? row_launch(whole, H, W, Ho, Wo, pad_h, pad_w, false)
                         : row_launch(whole, Ho, Wo, H, W, static_cast<int>(R - 1 - pad_h),
                                      static_cast<int>(S - 1 - pad_w), true);
    }
    if (fprop)
        return launch(H, W, Ho, Wo, stride_h, stride_w, pad_h, pad_w, static_cast<int>(R),
                      static_cast<int>(S), 0, 0, identity, false);
    if (!phased)   // stride 1: a stride-1 convolution of dy with the flipped filter, padding R-1-p
        return launch(Ho, Wo, H, W, 1, 1, static_cast<int>(R - 1 - pad_h),
                      static_cast<int>(S - 1 - pad_w), static_cast<int>(R), static_cast<int>(S), 0,
                      0, identity, false);
    // Strided: one launch per output phase. dx is zeroed first when a phase has no taps (its
    // pixels receive nothing) or when the atomic reduction adds into it.
    bool zero_first = reduction == SK_ATOMIC;
    for (const DgradPhase& ph : phases) zero_first = zero_first || !ph.live();
    if (zero_first) {
        cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(N * H * W * ldc * cs), st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(dx)");
    }
    // The phases write disjoint pixels of dx and read only dy and w. With a workspace of its own
    // for every phase (side by side; the library allocates them when the caller passes none, and
    // sk_workspace_bytes reports their sum), the zeroing kernels of all phases run first and then
    // every phase's main kernel starts while the previous one runs (a programmatic dependent
    // launch that waits for nothing of it). With one shared workspace (a caller's, holding the
    // largest phase only) a phase whose plan shares no tile still overlaps the previous phase; the
    // others follow it in order.
    std::vector<const DgradPhase*> live;
    for (const DgradPhase& ph : phases)
        if (ph.live()) live.push_back(&ph);
    std::vector<char> solo(live.size(), 0);
    std::vector<size_t> wsz(live.size(), 0);
    size_t total = 0;
    {
        const TileGuard pages_view(g_tile == SK_TILE_AUTO ? SK_TILE_128 : g_tile);
        for (size_t i = 0; i < live.size(); ++i) {
            sk_problem q;
            memset(&q, 0, sizeof(q));
            q.op = op; q.ab_dtype = in_dtype; q.c_dtype = out_dtype;
            q.n = N; q.c = C; q.k = K; q.groups = groups;
            set_phase_problem(q, live[i]->Hp, live[i]->Wp, live[i]->Rt, live[i]->St);
            sk_plan_t pl;
            rc = sk_plan(&q, streamk, reduction, ctas, 0, &pl);
            if (rc) return rc;
            solo[i] = pl.shared_tiles == 0 ? 1 : 0;
            wsz[i] = static_cast<size_t>(sk::round_up(pl.ws_bytes, 256));
            total += wsz[i];
        }
    }
    auto phase_rows = [&](const DgradPhase& ph) {
        sk::RowMap rm;
        memset(&rm, 0, sizeof(rm));
        rm.on = 1;
        rm.HoWo = ph.Hp * ph.Wp;
        rm.Wo = static_cast<int32_t>(ph.Wp);
        rm.Hd = static_cast<int32_t>(H);
        rm.Wd = static_cast<int32_t>(W);
        rm.dsh = stride_h;
        rm.dsw = stride_w;
        rm.ah = ph.a;
        rm.aw = ph.b;
        return rm;
    };
    const bool side = ws == nullptr || ws_bytes >= total;
    if (side) {
        uint8_t* wbase = static_cast<uint8_t*>(ws);
        if (ws == nullptr) {
            cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&wbase), total, st);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
        }
        size_t off = 0;
        for (size_t i = 0; i < live.size() && rc == SK_OK; off += wsz[i], ++i) {
            if (solo[i]) continue;
            const DgradPhase& ph = *live[i];
            rc = launch(Ho, Wo, ph.Hp, ph.Wp, 1, 1, ph.padh, ph.padw, ph.Rt, ph.St, ph.r0, ph.s0,
                        phase_rows(ph), true, 0, wbase + off, wsz[i], 1, true);
        }
        off = 0;
        for (size_t i = 0; i < live.size() && rc == SK_OK; off += wsz[i], ++i) {
            const DgradPhase& ph = *live[i];
            const int chain = (i > 0 ? 1 : 0) | (i + 1 < live.size() ? 2 : 0);
            rc = launch(Ho, Wo, ph.Hp, ph.Wp, 1, 1, ph.padh, ph.padw, ph.Rt, ph.St, ph.r0, ph.s0,
                        phase_rows(ph), true, chain, wbase + off, wsz[i], 2, true);
        }
        if (ws == nullptr) {
            cudaError_t e = cudaFreeAsync(wbase, st);
            if (e != cudaSuccess && rc == SK_OK) rc = cuda_fail(e, "cudaFreeAsync(workspace)");
        }
        return rc;
    }
    for (size_t i = 0; i < live.size(); ++i) {
        const DgradPhase& ph = *live[i];
        const int chain = (i > 0 && solo[i] ? 1 : 0) | (i + 1 < live.size() && solo[i + 1] ? 2 : 0);
        rc = launch(Ho, Wo, ph.Hp, ph.Wp, 1, 1, ph.padh, ph.padw, ph.Rt, ph.St, ph.r0, ph.s0,
                    phase_rows(ph), true, chain);
        if (rc) return rc;
    }
    return SK_OK;
}

}  // namespace

int sk_conv2d_fprop_nhwc(int in_dtype, int y_dtype, int64_t N, int64_t H, int64_t W, int64_t C,
                         int64_t K, int64_t R, int64_t S, int stride_h, int stride_w, int pad_h,
                         int pad_w, int groups, const void* x, const void* w, void* y,
                         int streamk, int reduction, int ctas, void* ws, size_t ws_bytes,
                         void* stream) {
    return conv_fwd_like(SK_OP_FPROP, in_dtype, y_dtype, N, H, W, C, K, R, S, stride_h, stride_w,
                         pad_h, pad_w, groups, x, w, y, streamk, reduction, ctas, ws, ws_bytes,
                         stream);
}

int sk_conv2d_dgrad_nhwc(int in_dtype, int dx_dtype, int64_t N, int64_t H, int64_t W, int64_t C,
                         int64_t K, int64_t R, int64_t S, int stride_h, int stride_w, int pad_h,
                         int pad_w, int groups, const void* dy, const void* w, void* dx,
                         int streamk, int reduction, int ctas, void* ws, size_t ws_bytes,
                         void* stream) {
    return conv_fwd_like(SK_OP_DGRAD, in_dtype, dx_dtype, N, H, W, C, K, R, S, stride_h, stride_w,
                         pad_h, pad_w, groups, dy, w, dx, streamk, reduction, ctas, ws, ws_bytes,
                         stream);
}

int sk_timing_enable(int on) {
    g_timing.recycle();
    g_timing.on = on != 0;
    return SK_OK;
}

int sk_timing_read(double* main_ms, int64_t* main_launches, int64_t* all_launches) {
    double total = 0.0;
    for (auto& p : g_timing.used) {
        cudaError_t e = cudaEventSynchronize(p.second);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, p.first, p.second);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
        total += ms;
    }
    if (main_ms) *main_ms = total;
    if (main_launches) *main_launches = g_timing.main_launches;
    if (all_launches) *all_launches = g_timing.all_launches;
    g_timing.recycle();
    return SK_OK;
}

int sk_device_status(void* stream) {
    long long info[3] = {0, 0, 0};
    int code = sk::take_device_error(static_cast<cudaStream_t>(stream), info);
    if (code < 0) return fail(SK_ERR_LAUNCH, "cannot read the device status");
    if (code == 0) return SK_OK;
    if (code == 1)
        return fail(SK_ERR_LAUNCH, "linear/tree hand-off timed out: cta %lld tile %lld waiting on cta %lld",
                    info[0], info[1], info[2]);
    return fail(SK_ERR_LAUNCH, "pipeline wait timed out: cta %lld tile %lld (role %lld)", info[0],
                info[1], info[2]);
}

int sk_probe_flag_timeout(int timeout_ms, void* stream) {
    if (timeout_ms < 1 || timeout_ms > 1000)
        return fail(SK_ERR_UNSUPPORTED, "timeout_ms must be in [1, 1000], got %d", timeout_ms);
    DevInfo dev;
    int rc = check_arch(dev);
    if (rc) return rc;
    const int e = sk::launch_flag_timeout_probe(static_cast<uint64_t>(timeout_ms) * 1000000ull,
                                                static_cast<cudaStream_t>(stream));
    if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "probe launch");
    return SK_OK;
}

// ---- fixed-scratch variant (no device allocation) --------------------------------------------
//
// Workspace for callers that cannot allocate device memory at call time. The array lives in the
// library's device image; host code only ever passes its per-device address, looked up below.
static __device__ __align__(256) unsigned char g_sk_static_ws[SK_STATIC_WS_BYTES];

static std::mutex g_static_ws_mu;

// The array's address on each device, looked up once per device and CUDA context: a context that
// was torn down and created again (cudaDeviceReset) loads the module again, so the address is
// looked up again when the current context's id changes. Without the driver's context-id entry
// points the address is looked up on every call.
struct StaticWsAddr {
    bool valid = false;
    unsigned long long ctx_id = 0;
    void* ptr = nullptr;
};
static StaticWsAddr g_static_ws_addr[64];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
static std::once_flag g_ctx_fn_once;
static CtxGetCurrentFn g_ctx_get_current = nullptr;
static CtxGetIdFn g_ctx_get_id = nullptr;

static bool current_context_id(unsigned long long& id) {
    std::call_once(g_ctx_fn_once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    CUcontext ctx = nullptr;
    return g_ctx_get_current && g_ctx_get_id && g_ctx_get_current(&ctx) == CUDA_SUCCESS &&
           ctx != nullptr && g_ctx_get_id(ctx, &id) == CUDA_SUCCESS;
}

int sk_gemm_rcr_static_ws(int ab_dtype, int c_dtype, int64_t M, int64_t N, int64_t K,
                          const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                          int64_t ldc, int streamk, int reduction, int ctas, void* stream) {
    if (M == 0 || N == 0 || K == 0)   // nothing that needs a workspace
        return sk_gemm_rcr(ab_dtype, c_dtype, M, N, K, A, lda, B, ldb, C, ldc, streamk, reduction,
                           ctas, nullptr, 0, stream);
    if (!C) return fail(SK_ERR_UNSUPPORTED, "NULL pointer");
    int rc = select_device_of(C);
    if (rc) return rc;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(SK_ERR_UNSUPPORTED, "device index %d out of range", dev);
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_static_ws_mu);
        StaticWsAddr& a = g_static_ws_addr[dev];
        unsigned long long id = 0;
        const bool have_id = current_context_id(id);
        if (!have_id || !a.valid || a.ctx_id != id) {   // set-up, with this device current
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_sk_static_ws);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
            unsigned long long id2 = 0;
            a.valid = current_context_id(id2);   // the lookup may have created the context
            a.ctx_id = id2;
            a.ptr = p;
        }
        ws = a.ptr;
    }
    // Size the plan the call will use and refuse it up front if it does not fit.
    sk_problem prob;
    memset(&prob, 0, sizeof(prob));
    prob.op = SK_OP_GEMM;
    prob.ab_dtype = ab_dtype;
    prob.c_dtype = c_dtype;
    prob.M = M;
    prob.N = N;
    prob.K = K;
    prob.groups = 1;
    sk_plan_t plan;
    rc = sk_plan(&prob, streamk, reduction, ctas, 0, &plan);
    if (rc) return rc;
    if (plan.ws_bytes > static_cast<int64_t>(SK_STATIC_WS_BYTES))
        return fail(SK_ERR_UNSUPPORTED,
                    "this problem needs %lld bytes of workspace; the fixed scratch holds %u bytes "
                    "(use sk_gemm_rcr with a caller workspace, a smaller pool, or atomic)",
                    (long long)plan.ws_bytes, (unsigned)SK_STATIC_WS_BYTES);
    return sk_gemm_rcr(ab_dtype, c_dtype, M, N, K, A, lda, B, ldb, C, ldc, streamk, reduction, ctas,
                       ws, SK_STATIC_WS_BYTES, stream);
}

}  // extern "C"
