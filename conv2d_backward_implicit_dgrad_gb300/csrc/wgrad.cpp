// C ABI of the weight gradient (declared in include/wgrad.h): plan geometry,
// workspace, tensor maps and the three launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <new>

#include "wgrad.h"
#include "wgrad_internal.h"

struct wgrad_plan_s {
    int device;
    dgrad::WgradGeometry g;
    dgrad::WgradMainParams mp;
    dgrad::WgradRunParams wp;   // run mode
    dgrad::WgradPlaneParams np;   // plane mode
    const void *map_x, *map_g;    // the tensors the per-call tensor maps were last encoded on (plane, direct)
    dgrad::WgradPackParams pp;
    dgrad::WgradReduceParams rp;
    uint32_t *err;
    float *gf, *xc, *part;
    size_t workspace_bytes;
};

namespace dgrad {

namespace {

constexpr int kWgSplitChunks = 12;      // longest K range of one split-precision unit, in 32-position chunks
constexpr int kWgBarrierBytes = 2048;   // barrier block + alignment slack of the stage ring
constexpr long long kWgTimeoutNs = 1000000000LL;

int ceil_div(int a, int b) { return (a + b - 1) / b; }
int round_up(int a, int b) { return ceil_div(a, b) * b; }
int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
int pow2_at_least(int v) {
    int p = 32;
    while (p < v) p *= 2;
    return p;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

// Run mode (see WgradRunParams).  Taps are grouped by (kernel row, input
// copy); within a group consecutive taps read consecutive positions, so a
// tile of spt of them is a contiguous run of position blocks.  The stage
// length L and the tiles per unit come from a cost model: a tensor copy
// takes about kWgCopyCycles on an SM whatever its size (up to 32 KB), a
// 128 x bn x 8 TF32 MMA about kWgMmaCycles(bn); both overlap, the slower
// bounds a stage.  Returns false where the segment mode stays.
constexpr int kWgCopyCycles = 550;
static int mma_cycles(int bn) { return bn <= 32 ? 66 : (bn <= 64 ? 72 : (bn <= 128 ? 84 : 128)); }

static bool plan_run(WgradGeometry &g, int sm_count) {
    if (!g.blocked) return false;
    const int halves = g.split ? 2 : 1;   // split precision: hi and lo copies, three MMA passes
    int sr = 8;   // rows per position block: the input channels rounded up to a power of two, 8 .. 128
    while (sr < g.Ci && sr < 128) sr *= 2;
    const int spt = 128 / sr;
    g.n_groups = 0;
    int ntap = 0;
    for (int kh = 0; kh < g.kH; ++kh) {
        for (int kw = 0; kw < g.kW; ++kw) {
            const int t = kh * g.kW + kw;
            bool seen = false;   // a group of this row and copy already holds the tap
            for (int k2 = 0; k2 < kw; ++k2)
                if (g.tap_copy[kh * g.kW + k2] == g.tap_copy[t]) seen = true;
            if (seen) continue;
            if (g.n_groups == kWgMaxGroups) return false;
            const int gi = g.n_groups++;
            g.grp_copy[gi] = g.tap_copy[t];
            g.grp_base[gi] = g.tap_off[t] / 32;
            g.grp_tap0[gi] = ntap;
            g.grp_nt[gi] = 0;
            for (int k2 = kw; k2 < g.kW; ++k2) {
                const int t2 = kh * g.kW + k2;
                if (g.tap_copy[t2] != g.tap_copy[t]) continue;
                if (g.tap_off[t2] != g.tap_off[t] + 32 * g.grp_nt[gi]) return false;   // not consecutive positions
                g.grp_taps[ntap++] = t2;
                ++g.grp_nt[gi];
            }
        }
    }
    g.n_tiles = 0;
    for (int gi = 0; gi < g.n_groups; ++gi) {
        g.grp_nmt[gi] = ceil_div(g.grp_nt[gi], spt);
        for (int m = 0; m < g.grp_nmt[gi]; ++m) {
            if (g.n_tiles == kWgMaxTiles) return false;
            g.tile_grp[g.n_tiles] = gi;
            g.tile_m0[g.n_tiles++] = m * spt;
        }
    }
    // Stage length L (a copy of L + spt - 1 position blocks of sr rows and
    // one of L grad_out blocks of bn rows, at most 256 rows each) and tiles per
    // unit: the least time per (tile, chunk) with at least two stages in
    // shared memory and the unit's accumulators in tensor memory.
    const int l_max = std::min(8, std::min(256 / sr - spt + 1, 256 / g.bn));
    double best = -1.0;
    int bl = 0, bt = 0, bd = 0;
    for (int L = 1; L <= l_max; ++L)
        for (int tpu = 1; tpu <= std::min(g.n_tiles, 512 / g.bn); ++tpu) {
            if (g.split && L > kWgSplitChunks) continue;
            const long long stage =
                halves * ((long long)tpu * (L + spt - 1) * sr * 128 + (long long)L * g.bn * 128);
            const int d = (int)std::min<long long>(kWgMaxStages, (kMaxSmem - kWgBarrierBytes) / stage);
            if (d < 2) continue;
            const int sets = ceil_div(g.n_tiles, tpu);
            const double per_stage = std::max((double)halves * (tpu + 1) * kWgCopyCycles,
                                              (double)L * tpu * 4 * (2 * halves - 1) * mma_cycles(g.bn));
            const double cost = per_stage / L * sets;   // per chunk, all tiles
            if (best < 0 || cost < best * 0.999) {
                best = cost;
                bl = L; bt = tpu; bd = d;
            }
        }
    // With one position per copy and one tap per tile nothing is shared: the
    // segment mode does the same copies.
    if (!bl || (bl == 1 && spt == 1)) return false;
    g.seg_rows = sr;
    g.spt = spt;
    g.cpt = ceil_div(g.Ci, sr);
    g.run_len = bl;
    g.tpu = bt;
    g.n_sets = ceil_div(g.n_tiles, bt);
    g.stages = bd;
    g.xbox_bytes = (bl + spt - 1) * sr * 128;
    g.bbox_bytes = bl * g.bn * 128;
    g.smem_bytes = kWgBarrierBytes + bd * halves * (bt * g.xbox_bytes + g.bbox_bytes);
    g.acc_sets = 2 * bt * g.bn <= 512 ? 2 : 1;
    g.tmem_cols = pow2_at_least(std::max(32, g.acc_sets * bt * g.bn));
    // K splits within each image group, units of whole stages: minimise
    // ceil(units / sm) * (stages + about two stages of fill and partial-tile
    // stores) per unit.
    const int per = g.n_sets * g.cpt * g.n_nt * g.Q;
    const int stages_total = ceil_div(g.cpi, bl);
    // Split precision: at most kWgSplitChunks chunks accumulate in one unit
    // (see the segment mode's K splits).
    const int ks_lo = g.split ? ceil_div(stages_total, std::max(1, kWgSplitChunks / bl)) : 1;
    const int ks_hi = std::max(ks_lo, std::min(stages_total / 2, ceil_div(8 * sm_count, per)));
    long long bestk = -1;
    int nk = ks_lo;
    for (int k = ks_lo; k <= ks_hi; ++k) {
        const int sps = ceil_div(stages_total, k);
        if (ceil_div(stages_total, sps) != k) continue;
        const long long cost = (long long)ceil_div(per * k, sm_count) * (sps + 2);
        if (bestk < 0 || cost < bestk) {
            bestk = cost;
            nk = k;
        }
    }
    g.cps = ceil_div(stages_total, nk) * bl;
    g.nksq = ceil_div(g.cpi, g.cps);
    g.n_ks = g.Q * g.nksq;
    g.n_mt = g.n_tiles;
    const long long units = (long long)per * g.nksq;
    if (units > INT_MAX / 2) return false;
    g.n_units = (int)units;
    g.grid = std::min(g.n_units, sm_count);
    g.part_elems = (size_t)g.Q * g.nksq * g.cpt * g.n_nt * g.n_tiles * g.bn * 128;
    g.run_mode = 1;
    return true;
}

// Plane mode (see WgradPlaneParams): stride 1, oH = H and oW = W, rows of a
// multiple of 4 positions (whole-row shifts of grad_out are then 16-byte
// tensor-copy coordinates), more than one tap (a 1x1 kernel takes the
// direct mode), TF32 (the MMA reads the caller's values, so there is no
// hi/lo split).  A's kW * ci_rows rows fill n_mt tiles of 128, B's kH *
// co_rows rows one MMA N; all n_mt * nb accumulator columns must fit tensor
// memory.  One CTA per SM, each over a contiguous range of chunks.
static void plan_plane(WgradGeometry &g, int sm_count) {
    if (g.split || g.s != 1 || g.oH != g.H || g.oW != g.W || g.kH * g.kW < 2 || g.W % 4 != 0) return;
    if (g.kW > 7) return;   // column shifts |kw - pw| <= 3: within one 16-byte piece
    const long long hw = (long long)g.H * g.W;
    const int ci_rows = round_up(g.Ci, 8), co_rows = round_up(g.Co, 8);
    const int nb = round_up(g.kH * co_rows, 16);
    const int n_mt = ceil_div(g.kW * ci_rows, 128);
    if (ci_rows > 256 || co_rows > 256 || nb > 256 || n_mt * nb > 512) return;
    if ((g.kW - 1) * ci_rows > 4 * 128) return;   // shifted rows: at most four per shifting thread
    const long long cpi = (hw + 31) / 32, chunks = cpi * g.N;
    if (hw > INT_MAX / 2 || chunks > INT_MAX / 2) return;
    const int stage_bytes = n_mt * 128 * 128 + nb * 128;
    const int stages = std::min(kWgMaxStages, (kMaxSmem - kWgBarrierBytes) / stage_bytes);
    if (stages < 2) return;
    g.plane = 1;
    g.run_mode = 0;
    g.f = 1;   // K = image, position: no images interleaved
    g.lf = 0;
    g.Q = g.N;
    g.ci_rows = ci_rows;
    g.co_rows = co_rows;
    g.seg_rows = ci_rows;
    g.bn = nb;
    g.n_mt = n_mt;
    g.n_nt = 1;
    g.cpi = (int)cpi;
    g.total_chunks = (int)chunks;
    g.grid = (int)std::min<long long>(sm_count, chunks);
    g.n_ks = g.grid;
    g.n_units = g.grid;
    g.cps = ceil_div(g.total_chunks, g.grid);
    g.stages = stages;
    g.smem_bytes = kWgBarrierBytes + stages * stage_bytes;
    g.tmem_cols = pow2_at_least(n_mt * nb);
    g.g_elems = g.x_elems = 0;
    g.part_elems = (size_t)g.grid * g.kW * ci_rows * nb;
}

dgrad_status_t make_wgrad_geometry(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int precision, int sm_count, WgradGeometry *out, bool allow_plane) {
    if (N < 1 || Ci < 1 || H < 1 || W < 1 || Co < 1 || kH < 1 || kW < 1 || stride < 1 || pad_h < 0 || pad_w < 0)
        return DGRAD_ERR_INVALID_ARG;
    if (precision != DGRAD_PREC_FP32 && precision != DGRAD_PREC_TF32 && precision != DGRAD_PREC_TF32X3)
        return DGRAD_ERR_INVALID_ARG;
    const long long nh = (long long)H + 2LL * pad_h - kH, nw = (long long)W + 2LL * pad_w - kW;
    if (nh < 0 || nw < 0) return DGRAD_ERR_INVALID_ARG;
    if (precision == DGRAD_PREC_FP32) return DGRAD_ERR_UNSUPPORTED;
    if (stride > kWgMaxRowPhases || (long long)kH * kW > kMaxTaps) return DGRAD_ERR_UNSUPPORTED;
    if (sm_count < 1) sm_count = 152;
    WgradGeometry g;
    std::memset(&g, 0, sizeof(g));
    g.N = N; g.Ci = Ci; g.H = H; g.W = W; g.Co = Co; g.kH = kH; g.kW = kW;
    g.s = stride; g.ph = pad_h; g.pw = pad_w;
    g.split = precision == DGRAD_PREC_TF32X3 ? 1 : 0;
    const int halves = g.split ? 2 : 1;
    g.oH = (int)(nh / stride) + 1;
    g.oW = (int)(nw / stride) + 1;
    // Direct mode: a 1x1 kernel with stride 1 and no padding reads the input at
    // the grad_out position itself, so both operands are K-major in NCHW as
    // given (K = image, position): no frames; the tensor copies read the
    // caller's tensors (per-image planes of H*W positions, a multiple of 4 for
    // the 16-byte stride rule; the last chunk of a plane is zero-filled past its
    // end) and the MMA takes the TF32 part of the fp32 values.
    g.direct = !g.split && kH == 1 && kW == 1 && stride == 1 && pad_h == 0 && pad_w == 0 &&
               ((long long)H * W) % 4 == 0 && (long long)H * W <= INT_MAX / 2;
    if (g.direct) {
        g.f = 1; g.lf = 0; g.m = 4; g.Q = N; g.blocked = 0;
        g.Ty = g.Tu = 0;
        g.Wf = g.oW;
        g.Kimg = g.oH * g.oW;
        g.cpi = ceil_div(g.Kimg, 32);
        g.Lx = g.Kimg;
        g.n_copies = 1;
        g.copy_rh[0] = g.copy_rw[0] = g.copy_r[0] = 0;
        g.taps = 1;
        g.tap_copy[0] = 0;
        g.tap_off[0] = 0;
    }
    // Images interleaved along K.  Batch-blocked frames (f = 32, batches of
    // 32 or more with at most 1/8 of padding images): a 32-element K chunk is
    // one frame position of 32 images and a (position, channel block) tile is
    // one contiguous run of memory.  Otherwise f = 4 (2, 1 for smaller
    // batches): a tap offset of whole columns is then a multiple of 4
    // positions (16 bytes, the tensor-copy alignment) once the copies absorb
    // column shifts mod m = 4/f.
    if (!g.direct) {
        g.blocked = N >= 32 && (round_up(N, 32) - N) * 8 <= N;
        g.f = g.blocked ? 32 : (N >= 4 ? 4 : (N >= 2 ? 2 : 1));
        g.lf = g.f == 32 ? 5 : (g.f == 4 ? 2 : (g.f == 2 ? 1 : 0));
        g.m = g.f >= 4 ? 1 : 4 / g.f;
        g.Q = ceil_div(N, g.f);
        // Decomposition of the taps: kh - ph = s*dh + rh, kw - pw = s*dw + rw.
        int dh_of[kMaxTaps], rh_of[kMaxTaps], dw_of[kMaxTaps], rw_of[kMaxTaps];
        int dh_min = INT_MAX, dh_max = INT_MIN, dw_min = INT_MAX, dw_max = INT_MIN;
        for (int kh = 0; kh < kH; ++kh) {
            dh_of[kh] = floor_div(kh - pad_h, stride);
            rh_of[kh] = kh - pad_h - dh_of[kh] * stride;
            dh_min = std::min(dh_min, dh_of[kh]);
            dh_max = std::max(dh_max, dh_of[kh]);
        }
        for (int kw = 0; kw < kW; ++kw) {
            dw_of[kw] = floor_div(kw - pad_w, stride);
            rw_of[kw] = kw - pad_w - dw_of[kw] * stride;
            dw_min = std::min(dw_min, dw_of[kw]);
            dw_max = std::max(dw_max, dw_of[kw]);
        }
        g.Ty = std::max(0, -dh_min);
        g.Tu = std::max(0, -dw_min);
        // Frame rows hold grad_out columns 0..oW-1 and every column a tap reads
        // for them (u = ow + dw + Tu - r <= oW - 1 + dw_max + Tu), a multiple of m.
        const long long wf = round_up(g.oW + std::max(0, dw_max) + g.Tu, g.m);
        if (wf * g.oH * g.f > INT_MAX / 4) return DGRAD_ERR_UNSUPPORTED;
        g.Wf = (int)wf;
        g.Kimg = round_up(g.oH * g.Wf * g.f, 32);
        g.cpi = g.Kimg / 32;
        // Copies: one per (row phase, column phase, column shift r) some tap reads.
        g.n_copies = 0;
        g.taps = kH * kW;
        int max_off = 0;
        for (int kh = 0; kh < kH; ++kh)
            for (int kw = 0; kw < kW; ++kw) {
                const int t = kh * kW + kw;
                const int r = (dw_of[kw] + g.Tu) % g.m;
                int c = -1;
                for (int i = 0; i < g.n_copies; ++i)
                    if (g.copy_rh[i] == rh_of[kh] && g.copy_rw[i] == rw_of[kw] && g.copy_r[i] == r) c = i;
                if (c < 0) {
                    if (g.n_copies == kWgMaxCopies) return DGRAD_ERR_UNSUPPORTED;
                    c = g.n_copies++;
                    g.copy_rh[c] = rh_of[kh];
                    g.copy_rw[c] = rw_of[kw];
                    g.copy_r[c] = r;
                }
                g.tap_copy[t] = c;
                g.tap_off[t] = ((dh_of[kh] + g.Ty) * g.Wf + (dw_of[kw] + g.Tu - r)) * g.f;
                max_off = std::max(max_off, g.tap_off[t]);
            }
        const long long lx = (long long)g.Kimg + max_off;
        if (lx > INT_MAX / 2) return DGRAD_ERR_UNSUPPORTED;
        g.Lx = (int)lx;   // a multiple of 4 (of 32 when blocked): Kimg of 32, every offset of 4 (32)
    }
    // Row tiles: (tap, input-channel block) segments of seg_rows rows.
    g.seg_rows = std::min(128, round_up(Ci, 8));
    g.cpt = ceil_div(Ci, g.seg_rows);
    g.n_segs = g.taps * g.cpt;
    if (g.n_segs > kWgMaxSegs) return DGRAD_ERR_UNSUPPORTED;
    g.spt = 128 / g.seg_rows;
    g.n_mt = ceil_div(g.n_segs, g.spt);
    // Column tiles of output channels (MMA N <= 256).
    g.n_nt = ceil_div(Co, 256);
    g.bn = round_up(ceil_div(Co, g.n_nt), 16);
    // K splits.  A CTA runs units w = blockIdx.x, + grid, ...; the slowest CTA
    // runs ceil(units / grid) units of up to cps chunks each, plus about two
    // chunks' worth of time per unit for its partial tile, so the split count
    // minimises ceil(tiles * n_ks / sm) * (cps + 2) (ties: fewer splits), with
    // units of at least 8 chunks and at most eight waves of them.
    const long long total_chunks = (long long)g.Q * g.cpi;
    if (total_chunks > INT_MAX / 2) return DGRAD_ERR_UNSUPPORTED;
    g.total_chunks = (int)total_chunks;
    const int tiles = g.n_mt * g.n_nt;
    // Split precision: the tensor cores' fp32 accumulation loses accuracy about
    // in proportion to the number of MMAs accumulated into one accumulator
    // (measured near 2e-8 relative error per MMA on random data), so a unit
    // takes at most kWgSplitChunks chunks (12 MMAs each) and the rest of the
    // sum goes to the fp32 reduction of the partial tiles.
    const int ks_lo = g.split ? ceil_div(g.total_chunks, kWgSplitChunks) : 1;
    const int ks_hi = std::max(ks_lo, std::min(std::max(1, g.total_chunks / 8), ceil_div(8 * sm_count, tiles)));
    long long best_cost = -1;
    int n_ks = ks_lo;
    for (int k = ks_lo; k <= ks_hi; ++k) {
        const int cps = ceil_div(g.total_chunks, k);
        if (ceil_div(g.total_chunks, cps) != k) continue;   // the same split as a smaller count
        const long long cost = (long long)ceil_div(tiles * k, sm_count) * (cps + 2);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            n_ks = k;
        }
    }
    g.cps = ceil_div(g.total_chunks, n_ks);
    g.n_ks = ceil_div(g.total_chunks, g.cps);
    const long long units = (long long)tiles * g.n_ks;
    if (units > INT_MAX / 2) return DGRAD_ERR_UNSUPPORTED;
    g.n_units = (int)units;
    g.grid = std::min(g.n_units, sm_count);
    const int stage_bytes = halves * (128 * 128 + g.bn * 128);
    g.stages = std::min(kWgMaxStages, (kMaxSmem - kWgBarrierBytes) / stage_bytes);
    if (g.stages < 2) return DGRAD_ERR_UNSUPPORTED;
    g.smem_bytes = kWgBarrierBytes + g.stages * stage_bytes;
    g.tmem_cols = pow2_at_least(2 * g.bn);
    g.g_elems = g.direct ? 0 : (size_t)halves * g.Q * Co * g.Kimg;
    g.x_elems = g.direct ? 0 : (size_t)halves * g.n_copies * g.Q * Ci * g.Lx;
    if ((g.g_elems + g.x_elems) / 4 > (size_t)INT_MAX) return DGRAD_ERR_UNSUPPORTED;   // 32-bit pack indices
    g.part_elems = (size_t)g.n_units * g.bn * 128;
    plan_run(g, sm_count);
    if (allow_plane) plan_plane(g, sm_count);
    *out = g;
    return DGRAD_OK;
}

}  // namespace dgrad

namespace {

using dgrad::WgradGeometry;

void fill_wgrad_info(const WgradGeometry &g, size_t ws, wgrad_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->N = g.N; info->Ci = g.Ci; info->H = g.H; info->W = g.W; info->Co = g.Co;
    info->kH = g.kH; info->kW = g.kW; info->stride = g.s; info->pad_h = g.ph; info->pad_w = g.pw;
    info->oH = g.oH; info->oW = g.oW;
    info->precision = g.split ? DGRAD_PREC_TF32X3 : DGRAD_PREC_TF32;
    info->interleave = g.f;
    info->mode = g.plane ? 3 : (g.run_mode ? 1 : (g.direct ? 2 : 0));
    info->Wf = g.Wf; info->Kimg = g.Kimg; info->Lx = g.Lx; info->n_copies = g.n_copies;
    info->seg_rows = g.seg_rows; info->n_mt = g.n_mt; info->n_nt = g.n_nt; info->n_ks = g.n_ks;
    info->slice_n = g.bn; info->n_units = g.n_units; info->grid = g.grid; info->stages = g.stages;
    info->smem_bytes = g.smem_bytes; info->tmem_cols = g.tmem_cols;
    info->workspace_bytes = ws;
    info->useful_flops = 2.0 * g.N * g.Co * g.oH * g.oW * (double)g.Ci * g.kH * g.kW;
    info->algorithmic_bytes =
        4.0 * ((double)g.N * g.Co * g.oH * g.oW + (double)g.N * g.Ci * g.H * g.W + (double)g.Co * g.Ci * g.kH * g.kW);
}

size_t workspace_of(const WgradGeometry &g) {
    return 256 + dgrad::align256(g.g_elems * 4) + dgrad::align256(g.x_elems * 4) + dgrad::align256(g.part_elems * 4);
}

dgrad_status_t wcuda(cudaError_t e) { return dgrad::cuda_status(e); }

bool wal16(const void *p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }
bool woverlap(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t a0 = (uintptr_t)a, a1 = a0 + an, b0 = (uintptr_t)b, b1 = b0 + bn;
    return a0 < b1 && b0 < a1;
}

// Tensor maps of the input copies (xc) and grad_out frame (gf); in direct mode
// the caller's input and grad_out themselves.
dgrad_status_t encode_maps(wgrad_plan_s *pl, const float *xsrc, const float *gsrc) {
    auto fn = dgrad::tensor_map_encoder();
    if (!fn) return DGRAD_ERR_CUDA;
    const WgradGeometry &g = pl->g;
    const cuuint32_t es4[4] = {1u, 1u, 1u, 1u};
    const cuuint64_t halves = g.split ? 2 : 1;
    cuuint64_t xd[4], xs[3], gd[3], gs[2];
    if (g.blocked) {   // [copy][q * Px + position][ci][32 images], [q * Pg + position][co][32 images]
        const cuuint64_t px = (cuuint64_t)g.Lx / 32, pg = (cuuint64_t)g.cpi;
        xd[0] = 32; xd[1] = (cuuint64_t)g.Ci; xd[2] = (cuuint64_t)g.Q * px; xd[3] = (cuuint64_t)g.n_copies * halves;
        xs[0] = 128; xs[1] = 128 * (cuuint64_t)g.Ci; xs[2] = xs[1] * g.Q * px;
        gd[0] = 32; gd[1] = (cuuint64_t)g.Co; gd[2] = (cuuint64_t)g.Q * pg * halves;
        gs[0] = 128; gs[1] = 128 * (cuuint64_t)g.Co;
    } else {           // [copy][q][ci][Lx], [q][co][Kimg]
        xd[0] = (cuuint64_t)g.Lx; xd[1] = (cuuint64_t)g.Ci; xd[2] = (cuuint64_t)g.Q;
        xd[3] = (cuuint64_t)g.n_copies * halves;
        xs[0] = (cuuint64_t)g.Lx * 4; xs[1] = xs[0] * g.Ci; xs[2] = xs[1] * g.Q;
        gd[0] = (cuuint64_t)g.Kimg; gd[1] = (cuuint64_t)g.Co; gd[2] = (cuuint64_t)g.Q * halves;
        gs[0] = (cuuint64_t)g.Kimg * 4; gs[1] = gs[0] * g.Co;
    }
    const cuuint32_t xbox[4] = {32u, (cuuint32_t)g.seg_rows, g.run_mode ? (cuuint32_t)(g.run_len + g.spt - 1) : 1u, 1u};
    if (fn(&pl->mp.x_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(xsrc), xd, xs, xbox, es4,
           CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DGRAD_ERR_CUDA;
    const cuuint32_t gbox[3] = {32u, (cuuint32_t)g.bn, g.run_mode ? (cuuint32_t)g.run_len : 1u};
    if (fn(&pl->mp.g_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(gsrc), gd, gs, gbox, es4,
           CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DGRAD_ERR_CUDA;
    return DGRAD_OK;
}

// Plane mode: the caller's input and grad_out as {H*W, channels, N} with
// boxes of 32 positions x all channels (rows past the channel count read as
// zeros).
dgrad_status_t encode_plane_maps(wgrad_plan_s *pl, const float *x, const float *go) {
    auto fn = dgrad::tensor_map_encoder();
    if (!fn) return DGRAD_ERR_CUDA;
    const WgradGeometry &g = pl->g;
    const cuuint32_t es[3] = {1u, 1u, 1u};
    const cuuint64_t hw = (cuuint64_t)g.H * g.W;
    const cuuint64_t xd[3] = {hw, (cuuint64_t)g.Ci, (cuuint64_t)g.N}, xs[2] = {hw * 4, hw * 4 * g.Ci};
    const cuuint64_t gd[3] = {hw, (cuuint64_t)g.Co, (cuuint64_t)g.N}, gs[2] = {hw * 4, hw * 4 * g.Co};
    const cuuint32_t xb[3] = {32u, (cuuint32_t)g.ci_rows, 1u}, gb[3] = {32u, (cuuint32_t)g.co_rows, 1u};
    if (fn(&pl->np.x_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(x), xd, xs, xb, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DGRAD_ERR_CUDA;
    if (fn(&pl->np.g_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(go), gd, gs, gb, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return DGRAD_ERR_CUDA;
    return DGRAD_OK;
}

void fill_wgrad_params(wgrad_plan_s *pl) {
    const WgradGeometry &g = pl->g;
    dgrad::WgradMainParams &m = pl->mp;
    m.part = pl->part;
    m.err = pl->err;
    m.n_mt = g.n_mt; m.n_nt = g.n_nt; m.n_ks = g.n_ks; m.n_units = g.n_units; m.bn = g.bn;
    m.seg_rows = g.seg_rows; m.spt = g.spt; m.n_segs = g.n_segs; m.cpi = g.cpi;
    m.total_chunks = g.total_chunks; m.cps = g.cps; m.stages = g.stages; m.tmem_cols = g.tmem_cols;
    m.idesc = dgrad::tf32_idesc(128, g.bn);
    m.split = g.split; m.Q = g.Q; m.n_copies = g.n_copies;
    m.blocked = g.blocked; m.Px = g.Lx / 32;
    m.timeout_ns = dgrad::kWgTimeoutNs;
    for (int sidx = 0; sidx < g.n_segs; ++sidx) {
        const int t = sidx / g.cpt;
        m.seg[sidx] = make_int4(g.tap_copy[t], (sidx - t * g.cpt) * g.seg_rows, g.tap_off[t], 0);
    }
    dgrad::WgradPackParams &q = pl->pp;
    q.gf = pl->gf; q.xc = pl->xc;
    q.N = g.N; q.Ci = g.Ci; q.H = g.H; q.W = g.W; q.Co = g.Co; q.oH = g.oH; q.oW = g.oW;
    q.s = g.s; q.Wf = g.Wf; q.Kimg = g.Kimg; q.Lx = g.Lx; q.Ty = g.Ty; q.Tu = g.Tu;
    q.Q = g.Q; q.lf = g.lf; q.blocked = g.blocked; q.Px = g.Lx / 32; q.Pg = g.cpi;
    const long long co_blocks = (g.Co + dgrad::kWgPackCh - 1) / dgrad::kWgPackCh;
    const long long ci_blocks = (g.Ci + dgrad::kWgPackCh - 1) / dgrad::kWgPackCh;
    q.g_tiles = (long long)g.Q * co_blocks * ((g.cpi + dgrad::kWgPackTile - 1) / dgrad::kWgPackTile);
    q.x_tiles = (long long)g.n_copies * g.Q * ci_blocks * ((g.Lx / 32 + dgrad::kWgPackTile - 1) / dgrad::kWgPackTile);
    for (int c = 0; c < g.n_copies; ++c) q.copy[c] = make_int4(g.copy_rh[c], g.copy_rw[c], g.copy_r[c], 0);
    q.split = g.split;
    q.g4 = (long long)(g.g_elems / 4 / (g.split ? 2 : 1));
    q.x4 = (long long)(g.x_elems / 4 / (g.split ? 2 : 1));
    dgrad::WgradReduceParams &r = pl->rp;
    r.part = pl->part;
    r.Co = g.Co; r.Ci = g.Ci; r.taps = g.taps; r.bn = g.bn; r.n_mt = g.n_mt; r.n_nt = g.n_nt; r.n_ks = g.n_ks;
    r.seg_rows = g.seg_rows; r.cpt = g.cpt; r.spt = g.spt; r.n_segs = g.n_segs;
    r.total = (long long)g.n_mt * g.n_nt * g.bn * 128;
    r.run_mode = g.run_mode;
    if (g.plane) {
        r.plane = 1;
        r.ci_rows = g.ci_rows; r.co_rows = g.co_rows; r.kH = g.kH; r.kW = g.kW; r.a_rows = g.kW * g.ci_rows;
        r.total = (long long)r.a_rows * g.bn;
        dgrad::WgradPlaneParams &n = pl->np;
        n.part = pl->part;
        n.err = pl->err;
        n.N = g.N; n.Ci = g.Ci; n.HW = g.H * g.W; n.W = g.W; n.kH = g.kH; n.kW = g.kW; n.ph = g.ph; n.pw = g.pw;
        n.ci_rows = g.ci_rows; n.co_rows = g.co_rows; n.nb = g.bn; n.n_mt = g.n_mt; n.cpi = g.cpi;
        n.total_chunks = g.total_chunks; n.stages = g.stages; n.tmem_cols = g.tmem_cols;
        n.a_bytes = (uint32_t)g.n_mt * 128u * 128u;
        n.stage_bytes = n.a_bytes + (uint32_t)g.bn * 128u;
        n.idesc = dgrad::tf32_idesc(128, g.bn);
        n.timeout_ns = dgrad::kWgTimeoutNs;
    }
    r.red_warps = 1;
    while (r.red_warps < 8 && r.red_warps * 8 < g.n_ks) r.red_warps *= 2;
    if (g.run_mode) {
        r.n_tiles = g.n_tiles;
        r.total = (long long)g.cpt * g.n_nt * g.n_tiles * g.bn * 128;
        for (int t = 0; t < g.n_tiles; ++t) r.tile[t] = make_int2(g.tile_grp[t], g.tile_m0[t]);
        for (int gi = 0; gi < g.n_groups; ++gi) r.grp[gi] = make_int2(g.grp_tap0[gi], g.grp_nt[gi]);
        for (int t = 0; t < g.taps; ++t) r.taps_of[t] = g.grp_taps[t];
        dgrad::WgradRunParams &w = pl->wp;
        w.part = pl->part;
        w.err = pl->err;
        w.n_units = g.n_units; w.n_sets = g.n_sets; w.tpu = g.tpu; w.n_tiles = g.n_tiles;
        w.cpt = g.cpt; w.n_nt = g.n_nt; w.nksq = g.nksq; w.cps = g.cps;
        w.Pg = g.cpi; w.Px = g.Lx / 32; w.seg_rows = g.seg_rows; w.L = g.run_len; w.bn = g.bn;
        w.stages = g.stages; w.acc_sets = g.acc_sets; w.tmem_cols = g.tmem_cols;
        w.xbox_bytes = g.xbox_bytes; w.bbox_bytes = g.bbox_bytes;
        w.split = g.split; w.n_copies = g.n_copies; w.Q = g.Q;
        w.idesc = dgrad::tf32_idesc(128, g.bn);
        w.timeout_ns = dgrad::kWgTimeoutNs;
        for (int t = 0; t < g.n_tiles; ++t) {
            const int gi = g.tile_grp[t];
            w.tile[t] = make_int2(g.grp_copy[gi], g.grp_base[gi] + g.tile_m0[t]);
        }
    }
}

}  // namespace

extern "C" {

dgrad_status_t wgrad_describe(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                              int pad_w, dgrad_precision_t precision, int sm_count, wgrad_plan_info_t *info) {
    if (!info) return DGRAD_ERR_INVALID_ARG;
    WgradGeometry g;
    dgrad_status_t st =
        dgrad::make_wgrad_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision, sm_count, &g);
    if (st != DGRAD_OK) return st;
    fill_wgrad_info(g, workspace_of(g), info);
    return DGRAD_OK;
}

dgrad_status_t wgrad_describe_taps(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                   int pad_w, int cap, int *copy, int *offset, int *copy_rh, int *copy_rw,
                                   int *copy_shift, int *n_copies, int *ty, int *tu, int *interleave) {
    if (!copy || !offset || !copy_rh || !copy_rw || !copy_shift || !n_copies || !ty || !tu || !interleave)
        return DGRAD_ERR_INVALID_ARG;
    WgradGeometry g;
    dgrad_status_t st =
        dgrad::make_wgrad_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, DGRAD_PREC_TF32, 0, &g, false);
    if (st != DGRAD_OK) return st;
    if (g.taps > cap || g.n_copies > cap) return DGRAD_ERR_INVALID_ARG;
    for (int t = 0; t < g.taps; ++t) {
        copy[t] = g.tap_copy[t];
        offset[t] = g.tap_off[t];
    }
    for (int c = 0; c < g.n_copies; ++c) {
        copy_rh[c] = g.copy_rh[c];
        copy_rw[c] = g.copy_rw[c];
        copy_shift[c] = g.copy_r[c];
    }
    *n_copies = g.n_copies;
    *ty = g.Ty;
    *tu = g.Tu;
    *interleave = g.f;
    return DGRAD_OK;
}

dgrad_status_t wgrad_describe_run(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                                     int pad_w, int sm_count, int cap, int *hdr, int *groups, int *taps, int *tiles) {
    if (!hdr || !groups || !taps || !tiles) return DGRAD_ERR_INVALID_ARG;
    WgradGeometry g;
    dgrad_status_t st = dgrad::make_wgrad_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, DGRAD_PREC_TF32,
                                                   sm_count, &g, false);
    if (st != DGRAD_OK) return st;
    if (!g.run_mode) return DGRAD_ERR_UNSUPPORTED;
    if (g.taps > cap || g.n_groups > cap || g.n_tiles > cap) return DGRAD_ERR_INVALID_ARG;
    const int h[15] = {g.n_groups, g.n_tiles, g.spt, g.seg_rows, g.stages, g.cpi, g.Lx / 32, g.cps,
                       g.nksq, g.cpt, g.n_nt, g.Q, g.run_len, g.tpu, g.n_sets};
    for (int i = 0; i < 15; ++i) hdr[i] = h[i];
    for (int gi = 0; gi < g.n_groups; ++gi) {
        int *e = groups + 6 * gi;
        e[0] = g.grp_copy[gi]; e[1] = g.grp_base[gi]; e[2] = g.grp_nt[gi];
        e[3] = g.grp_nmt[gi]; e[4] = 0; e[5] = g.grp_tap0[gi];
    }
    for (int t = 0; t < g.taps; ++t) taps[t] = g.grp_taps[t];
    for (int t = 0; t < g.n_tiles; ++t) {
        tiles[2 * t] = g.tile_grp[t];
        tiles[2 * t + 1] = g.tile_m0[t];
    }
    return DGRAD_OK;
}

dgrad_status_t wgrad_plan(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h, int pad_w,
                          dgrad_precision_t precision, wgrad_plan_t *plan_out) {
    return wgrad_plan_ex(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision, nullptr, plan_out);
}

dgrad_status_t wgrad_plan_ex(int N, int Ci, int H, int W, int Co, int kH, int kW, int stride, int pad_h,
                             int pad_w, dgrad_precision_t precision, const wgrad_options_t *opts,
                             wgrad_plan_t *plan_out) {
    if (!plan_out) return DGRAD_ERR_INVALID_ARG;
    *plan_out = nullptr;
    if (opts && (opts->timeout_us < 0 || opts->wait_test < 0 || opts->wait_test > 1)) return DGRAD_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_NO_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DGRAD_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return DGRAD_ERR_NO_DEVICE;
    wgrad_plan_s *pl = new (std::nothrow) wgrad_plan_s;
    if (!pl) return DGRAD_ERR_OOM;
    std::memset(pl, 0, sizeof(*pl));
    pl->device = dev;
    dgrad_status_t st = dgrad::make_wgrad_geometry(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision,
                                                   prop.multiProcessorCount, &pl->g);
    if (st != DGRAD_OK) {
        delete pl;
        return st;
    }
    const size_t ws = workspace_of(pl->g);
    void *mem = nullptr;
    if (cudaMalloc(&mem, ws) != cudaSuccess) {
        cudaGetLastError();
        delete pl;
        return DGRAD_ERR_OOM;
    }
    if (cudaMemset(mem, 0, 256) != cudaSuccess || cudaStreamSynchronize(nullptr) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(mem);
        delete pl;
        return DGRAD_ERR_CUDA;
    }
    uint8_t *b = static_cast<uint8_t *>(mem);
    pl->err = reinterpret_cast<uint32_t *>(b);
    pl->gf = reinterpret_cast<float *>(b + 256);
    pl->xc = reinterpret_cast<float *>(b + 256 + dgrad::align256(pl->g.g_elems * 4));
    pl->part = reinterpret_cast<float *>(b + 256 + dgrad::align256(pl->g.g_elems * 4) +
                                         dgrad::align256(pl->g.x_elems * 4));
    pl->workspace_bytes = ws;
    fill_wgrad_params(pl);
    if (opts) {
        const long long tmo = opts->timeout_us > 0 ? 1000LL * opts->timeout_us : dgrad::kWgTimeoutNs;
        pl->mp.timeout_ns = pl->wp.timeout_ns = pl->np.timeout_ns = tmo;
        pl->mp.wait_test = pl->wp.wait_test = pl->np.wait_test = opts->wait_test;
    }
    // Direct and plane modes encode their maps at run time, on the caller's tensors.
    if (!pl->g.direct && !pl->g.plane && (st = encode_maps(pl, pl->xc, pl->gf)) != DGRAD_OK) {
        cudaFree(mem);
        delete pl;
        return st;
    }
    pl->wp.x_map = pl->mp.x_map;
    pl->wp.g_map = pl->mp.g_map;
    *plan_out = pl;
    return DGRAD_OK;
}

dgrad_status_t wgrad_plan_info(wgrad_plan_t plan, wgrad_plan_info_t *info) {
    if (!plan || !info) return DGRAD_ERR_INVALID_ARG;
    fill_wgrad_info(plan->g, plan->workspace_bytes, info);
    return DGRAD_OK;
}

dgrad_status_t wgrad_run(wgrad_plan_t plan, const float *grad_out, const float *input, float *grad_weight,
                         void *stream) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    if (!wal16(grad_out) || !wal16(input) || !wal16(grad_weight)) return DGRAD_ERR_MISALIGNED;
    const WgradGeometry &g = plan->g;
    const size_t go_b = (size_t)g.N * g.Co * g.oH * g.oW * 4, x_b = (size_t)g.N * g.Ci * g.H * g.W * 4;
    const size_t w_b = (size_t)g.Co * g.Ci * g.kH * g.kW * 4;
    if (woverlap(grad_weight, w_b, grad_out, go_b) || woverlap(grad_weight, w_b, input, x_b)) return DGRAD_ERR_ALIAS;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (dev != plan->device) return DGRAD_ERR_WRONG_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    plan->pp.go = grad_out;
    plan->pp.x = input;
    plan->rp.dw = grad_weight;
    dgrad_status_t st = DGRAD_OK;
    // Direct and plane modes: no frames, the tensor copies read the caller's
    // tensors (maps re-encoded only when the pointers change).
    const bool remap = plan->map_x != input || plan->map_g != grad_out;
    if (g.plane) {
        if (remap && (st = encode_plane_maps(plan, input, grad_out)) != DGRAD_OK) return st;
        plan->np.x = input;
        st = wcuda(dgrad::launch_wgrad_plane(plan->np, g.grid, g.smem_bytes, s));
    } else {
        if (g.direct) {
            if (remap && (st = encode_maps(plan, input, grad_out)) != DGRAD_OK) return st;
        } else if ((st = wcuda(dgrad::launch_wgrad_pack(plan->pp, s))) != DGRAD_OK) {
            return st;
        }
        st = wcuda(g.run_mode ? dgrad::launch_wgrad_run(plan->wp, g.grid, g.smem_bytes, s)
                         : dgrad::launch_wgrad_main(plan->mp, g.grid, g.smem_bytes, s));
    }
    if (st != DGRAD_OK) return st;
    if (g.plane || g.direct) {
        plan->map_x = input;
        plan->map_g = grad_out;
    }
    return wcuda(dgrad::launch_wgrad_reduce(plan->rp, s));
}

dgrad_status_t wgrad_plan_check(wgrad_plan_t plan) {
    if (!plan) return DGRAD_ERR_INVALID_ARG;
    uint32_t word = 0;
    if (cudaMemcpy(&word, plan->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (word == 0) return DGRAD_OK;
    if (cudaMemset(plan->err, 0, sizeof(word)) != cudaSuccess) return DGRAD_ERR_CUDA;
    return DGRAD_ERR_DEVICE_TIMEOUT;
}

void wgrad_plan_destroy(wgrad_plan_t plan) {
    if (!plan) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    cudaDeviceSynchronize();
    cudaFree(plan->err);
    if (cur >= 0 && cur != plan->device) cudaSetDevice(cur);
    delete plan;
}

}  // extern "C"
