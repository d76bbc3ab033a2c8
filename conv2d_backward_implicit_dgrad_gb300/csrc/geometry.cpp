// Host-side planning: the sub-pixel phase split, the zero-padded grad_out
// frame, and the tiling of the main kernels.  No CUDA calls here, so
// dgrad_describe() works without a device.
#include <algorithm>
#include <climits>
#include <cstring>

#include "dgrad_internal.h"

namespace dgrad {

namespace {

int out_extent(int in, int k, int s, int p) {
    long long num = (long long)in + 2LL * p - k;
    if (num < 0) return 0;
    return (int)(num / s + 1);
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }
int round_up(int a, int b) { return ceil_div(a, b) * b; }

// Row (or column) taps of phase a along one axis.
//
// Input row ih = s*q + a receives kernel row kh exactly when
// (a + pad - kh) is a multiple of s (meganeura's divisibility test, general-
// stride branch of its B-tile load; doppler's "(py - ky) % stride" skip).
// Those rows are kh = r + s*j with r = (a + pad) mod s, and they read
// grad_out row oh = q + c - j with c = floor((a + pad)/s).  A tap whose
// grad_out rows lie outside [0, o) for every output row q < nq only ever
// meets padding; it contributes nothing and is dropped.
struct AxisTaps {
    int r, c, nq;
    int count;
    int j[64];
};

AxisTaps axis_taps(int a, int pad, int s, int k, int in, int o) {
    AxisTaps t{};
    t.r = (a + pad) % s;
    t.c = (a + pad) / s;
    t.nq = a < in ? ceil_div(in - a, s) : 0;
    t.count = 0;
    for (int j = 0; t.r + s * j < k; ++j) {
        int lo = t.c - j, hi = t.c - j + t.nq - 1;   // grad_out rows read by q = 0 .. nq-1
        if (t.nq > 0 && hi >= 0 && lo <= o - 1) t.j[t.count++] = j;
    }
    return t;
}

}  // namespace

dgrad_status_t make_geometry(int N, int Ci, int H, int W, int Co, int kH, int kW,
                             int stride, int pad_h, int pad_w, Geometry *g) {
    if (N < 1 || Ci < 1 || H < 1 || W < 1 || Co < 1 || kH < 1 || kW < 1 || stride < 1 ||
        pad_h < 0 || pad_w < 0)
        return DGRAD_ERR_INVALID_ARG;
    int oH = out_extent(H, kH, stride, pad_h), oW = out_extent(W, kW, stride, pad_w);
    if (oH < 1 || oW < 1) return DGRAD_ERR_INVALID_ARG;
    if (stride > kMaxStride || kH > 64 || kW > 64 || kH * kW > kMaxTaps) return DGRAD_ERR_UNSUPPORTED;
    const long long lim = INT_MAX;
    if ((long long)N * Co * oH * oW > lim || (long long)N * Ci * H * W > lim ||
        (long long)Co * Ci * kH * kW > lim)
        return DGRAD_ERR_UNSUPPORTED;

    std::memset(g, 0, sizeof(*g));
    g->N = N; g->Ci = Ci; g->H = H; g->W = W; g->Co = Co; g->kH = kH; g->kW = kW;
    g->s = stride; g->ph = pad_h; g->pw = pad_w; g->oH = oH; g->oW = oW;

    AxisTaps rows[kMaxStride], cols[kMaxStride];
    for (int a = 0; a < stride; ++a) rows[a] = axis_taps(a, pad_h, stride, kH, H, oH);
    for (int b = 0; b < stride; ++b) cols[b] = axis_taps(b, pad_w, stride, kW, W, oW);

    // Leading zero rows/cols so that every kept tap has a non-negative offset.
    int Ph = 0, Pw = 0;
    for (int a = 0; a < stride; ++a)
        for (int i = 0; i < rows[a].count; ++i) Ph = std::max(Ph, rows[a].j[i] - rows[a].c);
    for (int b = 0; b < stride; ++b)
        for (int i = 0; i < cols[b].count; ++i) Pw = std::max(Pw, cols[b].j[i] - cols[b].c);

    int max_dr = 0, max_dc = 0, nq_max = 0, nu_max = 0;
    int tap_dr[kMaxTaps], tap_dc[kMaxTaps];
    g->n_phases = 0;
    g->n_taps = 0;
    for (int a = 0; a < stride; ++a) {
        for (int b = 0; b < stride; ++b) {
            const AxisTaps &R = rows[a], &C = cols[b];
            if (R.nq == 0 || C.nq == 0) continue;   // no input element in this phase
            PhaseDesc &p = g->phase[g->n_phases++];
            p.a = a; p.b = b; p.Hq = R.nq; p.Wq = C.nq;
            p.tap_begin = g->n_taps;
            p.tap_count = R.count * C.count;
            p.row_len = C.count;
            p.sub = 1;
            p.col = 0;
            nq_max = std::max(nq_max, R.nq);
            nu_max = std::max(nu_max, C.nq);
            for (int x = 0; x < R.count; ++x)
                for (int y = 0; y < C.count; ++y) {
                    int j = R.j[x], i = C.j[y];
                    TapDesc &t = g->tap[g->n_taps++];
                    t.kh = R.r + stride * j;
                    t.kw = C.r + stride * i;
                    t.phase = g->n_phases - 1;
                    int dr = R.c - j + Ph, dc = C.c - i + Pw;
                    max_dr = std::max(max_dr, dr);
                    max_dc = std::max(max_dc, dc);
                    tap_dr[g->n_taps - 1] = dr;
                    tap_dc[g->n_taps - 1] = dc;
                    t.dr = dr;
                    t.dc = dc;
                    t.shift = 0;   // set below once Wp is known
                }
        }
    }
    // Frame size: hold every grad_out row (oH + Ph) and every output row
    // (nq_max), and let the deepest read of the last valid output row wrap
    // only into the next image's leading zero rows (nq_max + max_dr - Ph).
    // Same for columns, where a wrap lands in the next row's leading zeros.
    int Hv = std::max(nq_max, std::max(oH + Ph, nq_max + max_dr - Ph));
    int Wp = std::max(nu_max, std::max(oW + Pw, nu_max + max_dc - Pw));
    g->Ph = Ph; g->Pw = Pw; g->Hv = Hv; g->Wp = Wp;
    g->max_shift = 0;
    for (int t = 0; t < g->n_taps; ++t) {
        g->tap[t].shift = tap_dr[t] * Wp + tap_dc[t];
        g->max_shift = std::max(g->max_shift, g->tap[t].shift);
    }
    g->positions = (long long)N * Hv * Wp;
    if (g->positions + g->max_shift + 4LL * kBlockM > lim) return DGRAD_ERR_UNSUPPORTED;
    return DGRAD_OK;
}

int build_mgroups(const Geometry &g, const Tiling &t, MGroup *out, int *perm, int *phase_units) {
    int n = 0;
    if (!t.pgroup) {
        int units = 0;
        for (int ph = 0; ph < g.n_phases; ++ph) {
            const PhaseDesc &pd = g.phase[ph];
            phase_units[ph] = units;
            const int step = t.grouped ? std::max(1, pd.row_len) : 1;
            units += t.grouped ? pd.row_len : 1;
            for (int tp = pd.tap_begin; tp < pd.tap_begin + pd.tap_count; tp += step) {
                MGroup &m = out[n++];
                m.col = phase_units[ph];
                m.tap0 = tp;
                m.ntaps = step;
                m.a_shift = g.tap[tp + step - 1].shift;   // a row's last tap has the smallest column offset
                m.first = tp == pd.tap_begin ? 1 : 0;
            }
        }
        for (int i = 0; i < g.n_taps; ++i) perm[i] = i;
        return n;
    }
    // Shared-shift groups.  Phases with taps, and for every shift the set of
    // phases that have a tap with it (a phase has at most one tap per shift).
    int q[kMaxPhases], nq = 0;
    for (int ph = 0; ph < g.n_phases; ++ph)
        if (g.phase[ph].tap_count > 0) q[nq++] = ph;
    if (nq < 2 || nq > 4) return -1;
    int shifts[kMaxTaps], nsh = 0;
    unsigned masks[kMaxTaps];
    for (int i = 0; i < g.n_taps; ++i) {
        int k = 0;
        while (k < nsh && shifts[k] != g.tap[i].shift) ++k;
        if (k == nsh) {
            shifts[nsh] = g.tap[i].shift;
            masks[nsh++] = 0;
        }
        masks[k] |= 1u << g.tap[i].phase;
    }
    unsigned all = 0;
    for (int i = 0; i < nq; ++i) all |= 1u << q[i];
    int lead = -1;   // a shift that every phase has: the first group
    for (int k = 0; k < nsh && lead < 0; ++k)
        if (masks[k] == all) lead = k;
    if (lead < 0) return -1;
    // An order of the phases in tensor memory that makes every group contiguous.
    int order[4] = {0, 1, 2, 3};
    bool found = false;
    do {
        int pos[kMaxPhases];
        for (int i = 0; i < nq; ++i) pos[q[order[i]]] = i;
        bool ok = true;
        for (int k = 0; k < nsh && ok; ++k) {
            int lo = nq, hi = -1, cnt = 0;
            for (int i = 0; i < nq; ++i)
                if (masks[k] & (1u << q[i])) {
                    lo = std::min(lo, pos[q[i]]);
                    hi = std::max(hi, pos[q[i]]);
                    ++cnt;
                }
            ok = hi - lo + 1 == cnt;
        }
        found = ok;
    } while (!found && std::next_permutation(order, order + nq));
    if (!found) return -1;
    for (int ph = 0; ph < g.n_phases; ++ph) phase_units[ph] = 0;   // phases without taps: never read
    for (int i = 0; i < nq; ++i) phase_units[q[order[i]]] = i;
    // Groups: the lead shift first, then the others by falling size; taps of
    // a group in tensor-memory order of their phases.
    int gorder[kMaxTaps], ng = 0;
    gorder[ng++] = lead;
    for (int c = nq; c >= 1; --c)
        for (int k = 0; k < nsh; ++k)
            if (k != lead && __builtin_popcount(masks[k]) == c) gorder[ng++] = k;
    int np = 0;
    for (int gi = 0; gi < ng; ++gi) {
        const int k = gorder[gi];
        MGroup &m = out[n++];
        m.tap0 = np;
        m.a_shift = shifts[k];
        m.first = gi == 0 ? 1 : 0;
        m.col = nq;
        for (int i = 0; i < nq; ++i) {   // phases in tensor-memory order
            const int ph = q[order[i]];
            if (!(masks[k] & (1u << ph))) continue;
            m.col = std::min(m.col, i);
            for (int tp = g.phase[ph].tap_begin; tp < g.phase[ph].tap_begin + g.phase[ph].tap_count; ++tp)
                if (g.tap[tp].shift == shifts[k]) perm[np++] = tp;
        }
        m.ntaps = np - m.tap0;
    }
    return n;
}

namespace {

int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p *= 2;
    return p;
}

constexpr int kBarrierBytes = 4096;   // mbarriers + TMEM slot (1 KB), MMA group table (2 KB), 1024-byte alignment slack
constexpr int kMaxResidentChunks = 32;
constexpr int kMaxTmemAStages = 6;   // tensor-memory A source with image-aligned tiles (kernel arrays hold 8)
constexpr int kMaxTcRows = 1024;   // frame rows one tcgen05 A stage may hold (16 per producer thread)
// Packed frames up to 2 GiB.  The frame path beats producer warps even when
// the frame does not stay in L2 (7x7 stem, 114 MB frame: 145 us per call
// against 212 us with producers).
constexpr size_t kMaxFrameBytes = size_t(2) << 30;

// Split the MMA groups of one channel chunk into B stages of at most `cap`
// taps each, balanced; false when one MMA group alone exceeds `cap`.
bool split_b_stages(const MGroup *mg, int n_mg, int total_taps, int cap, Tiling &t) {
    if (cap < 1) return false;
    for (int i = 0; i < n_mg; ++i)
        if (mg[i].ntaps > cap) return false;
    int stages = (total_taps + cap - 1) / cap;
    for (;; ++stages) {
        const int target = (total_taps + stages - 1) / stages;
        int n = 0, taps = 0, largest = 0;
        t.bg_first[0] = 0;
        for (int i = 0; i < n_mg; ++i) {
            if (taps > 0 && taps + mg[i].ntaps > target) {
                largest = std::max(largest, taps);
                t.bg_first[++n] = i;
                taps = 0;
            }
            taps += mg[i].ntaps;
        }
        largest = std::max(largest, taps);
        t.bg_first[++n] = n_mg;
        if (largest <= cap) {
            t.n_tgroups = n;
            t.tap_group = largest;
            return true;
        }
        if (stages > n_mg) return false;
    }
}

// Fill the sizes that follow from (tm, bn, grouped) for the tcgen05 path
// (kc = 32); returns false when no pipeline depth fits in shared memory or
// the accumulators do not fit in tensor memory.  The packed weights of one
// channel chunk are streamed in B stages of whole MMA groups; when all of
// them fit next to two A stages they stay resident instead.
bool size_tc(const Geometry &g, Tiling &t, int want_resident) {
    t.n_slices = ceil_div(g.Ci, t.bn);
    // Split precision runs three K passes (hi*lo, lo*hi, hi*hi) per channel chunk.
    t.n_chunks = ceil_div(g.Co, t.kc) * (t.split ? 3 : 1);
    MGroup mg[kMaxTaps];
    int perm[kMaxTaps], units[kMaxPhases];
    t.n_mgroups = build_mgroups(g, t, mg, perm, units);
    if (t.n_mgroups < 0) return false;
    for (int i = 0; i < t.n_mgroups; ++i)
        if (mg[i].ntaps * t.bn > 256) return false;   // MMA N limit
    int max_sub = 1, sub_cols = 0;
    for (int p = 0; p < g.n_phases; ++p) {
        const int sub = t.grouped ? g.phase[p].row_len : 1;
        max_sub = std::max(max_sub, sub);
        sub_cols += sub * t.bn;
    }
    if (t.grouped && (t.tm != 1 || max_sub > kMaxSub)) return false;
    t.tile_step = t.tm * kBlockM - (max_sub - 1);
    // Cross-warp row exchange of grouped units: two buffers of 4 warps x slots
    // rows of 16 columns, or, for a single phase, of the slice's bn columns
    // (published once per unit).
    t.xchg_unit = max_sub > 1 && g.n_phases == 1 ? 1 : 0;
    // Grouped units' epilogues (sub-accumulators, combine) take about twice an
    // ungrouped one: with two accumulator sets a second epilogue warp group
    // takes every other unit (tensor-copy launches; 10 warps).
    t.epi_groups = (t.grouped && t.a_tma && max_sub > 1 && 2 * t.tm * sub_cols <= kTmemCols) ? 2 : 1;
    t.xchg_bytes = max_sub > 1 ? t.epi_groups * 2 * 4 * (max_sub * (max_sub - 1) / 2) * (t.xchg_unit ? t.bn : 16) * 4
                               : 0;
    const int raw_rows = t.tm * kBlockM + g.max_shift;
    t.band_rows = raw_rows;
    const int tmem_img_tiles = ceil_div(g.oH * g.oW, kBlockM);
    const bool tmem_aligned = t.a_tmem && t.img_align_sms > 0 &&
                              (long long)g.N * tmem_img_tiles * t.n_slices <= t.img_align_sms;
    if (t.a_tmem) {
        // Each shared-memory stage holds two tensor copies of 128 plane
        // elements x 32 channels (a tile of 128 positions spans at most two
        // images when the plane has >= 128 elements): 256 rows of 128 B.
        // When every unit fits one wave anyway, tiles are aligned to images
        // instead (ceil(plane / 128) per image, the last one partly empty):
        // one copy per stage, so twice the stages fit in the same memory
        // (measured: pointwise main kernel 33.4 -> 31.4 us, 128 units on 128
        // CTAs instead of 98 on 98).
        if (t.tm != 1 || t.grouped || t.pgroup || g.max_shift != 0) return false;
        t.stg_box = kBlockM;
        t.a_nbox = tmem_aligned ? 1 : 2;
        t.a_box_rows = 0;
        t.a_rows = t.a_nbox * kBlockM;
    } else if (t.a_staged) {
        // One tensor copy per A stage of the plane elements the band holds:
        // at most one per frame row, plus up to 3 before them (the copy
        // starts on a 16-byte boundary of the plane).  The copy lands in the
        // stage itself (stg_box elements x 32 channels = stg_box 128-byte
        // rows) and is transposed there.
        t.stg_box = round_up(raw_rows + 3, 4);
        if (t.tm != 1 || t.stg_box > 256) return false;
        t.a_nbox = 1;
        t.a_box_rows = 0;
        t.a_rows = round_up(std::max(raw_rows, t.stg_box), 8);
    } else if (t.a_tma) {   // tensor copies of at most 256 rows each
        t.a_nbox = ceil_div(raw_rows, 256);
        t.a_box_rows = round_up(ceil_div(raw_rows, t.a_nbox), 8);
        t.a_rows = t.a_nbox * t.a_box_rows;
    } else {
        t.a_nbox = t.a_box_rows = 0;
        t.a_rows = round_up(raw_rows, 8);
        if (t.a_rows > kMaxTcRows) return false;
    }
    const long long a_bytes = (long long)t.a_rows * t.kc * 4;
    const long long tap_bytes = (long long)t.bn * t.kc * 4;
    const long long budget = kMaxSmem - kBarrierBytes - t.xchg_bytes;
    const int taps = std::max(1, g.n_taps);
    t.b_resident = 0;
    if (want_resident && t.want_b_stages == 0 && t.n_slices == 1 && t.n_chunks <= kMaxResidentChunks) {
        long long b_all = (long long)t.n_chunks * taps * tap_bytes;
        if (b_all + 2 * a_bytes <= budget) {
            t.b_resident = 1;
            t.tap_group = taps;
            t.n_tgroups = 1;
            t.bg_first[0] = 0;
            t.bg_first[1] = t.n_mgroups;
            t.b_stages = t.n_chunks;
            t.chunk_bytes = (int)(taps * tap_bytes);
            t.a_stages = (int)std::min<long long>(4, (budget - b_all) / a_bytes);
        }
    }
    if (want_resident && !t.b_resident) return false;
    if (!t.b_resident) {
        // Largest B stage with nst B stages (two unless requested) and at
        // least two A stages (three when they fit without shrinking the
        // stage below half).
        // Automatic depth: when a whole chunk's taps fit one stage with four
        // (or three) stages and three A stages, take the deeper pipeline:
        // such plans (1x1 kernels) run short MMA bursts per chunk, and the
        // weight copies then need more chunks in flight (measured: pointwise
        // main kernel 31.4 -> 26.9 us with four stages).  Otherwise two large
        // stages (more stages measured slower for 3x3 and larger kernels).
        int nst = t.want_b_stages;
        for (int cand = 4; nst == 0 && cand >= 3; --cand)
            if ((budget - 3 * a_bytes) / (cand * tap_bytes) >= taps) nst = cand;
        if (nst == 0) nst = 2;
        long long cap = (budget - 2 * a_bytes) / (nst * tap_bytes);
        if (cap < 1) return false;
        cap = std::min<long long>(cap, taps);
        long long cap3 = (budget - 3 * a_bytes) / (nst * tap_bytes);
        if (cap3 >= std::min<long long>(taps, std::max<long long>(1, (cap + 1) / 2))) cap = std::min<long long>(cap3, taps);
        if (!split_b_stages(mg, t.n_mgroups, g.n_taps, (int)cap, t)) return false;
        t.chunk_bytes = (int)(t.tap_group * tap_bytes);
        t.b_stages = nst;
        long long left = budget - (long long)t.b_stages * t.chunk_bytes;
        t.a_stages = (int)std::min<long long>(tmem_aligned ? kMaxTmemAStages : 4, left / a_bytes);
    }
    if (t.a_stages < 2) return false;
    t.smem_bytes = (int)(kBarrierBytes + t.xchg_bytes + t.a_stages * a_bytes + (long long)t.b_stages * t.chunk_bytes);
    t.acc_cols = t.tm * sub_cols;
    // a_tmem: four 32-column A slots after the accumulators
    const int a_cols = t.a_tmem ? 4 * t.kc : 0;
    if (t.acc_cols + a_cols > kTmemCols) return false;
    t.acc_bufs = (2 * t.acc_cols + a_cols <= kTmemCols) ? 2 : 1;
    t.a_tslots = t.a_tmem ? 4 : 0;
    t.a_tcol = t.acc_bufs * t.acc_cols;
    t.tmem_cols = pow2_at_least(t.acc_bufs * t.acc_cols + a_cols);
    if (tmem_aligned) {
        t.img_tiles = tmem_img_tiles;
        t.n_tiles = g.N * t.img_tiles;
    } else if (t.a_staged) {
        // Tiles never cross an image (a band is one copy from one image):
        // each image's tiles cover its frame positions up to the last one
        // that is an output of some phase.
        int nq = 0, nu = 0;
        for (int p = 0; p < g.n_phases; ++p) nq = std::max(nq, g.phase[p].Hq), nu = std::max(nu, g.phase[p].Wq);
        const int out_span = (nq - 1) * g.Wp + nu;
        t.img_tiles = ceil_div(out_span, t.tile_step);
        t.n_tiles = g.N * t.img_tiles;
    } else {
        t.img_tiles = 0;
        t.n_tiles = (int)((g.positions + t.tile_step - 1) / t.tile_step);
    }
    t.n_work = (long long)t.n_tiles * t.n_slices;
    t.packed_bytes = (size_t)t.n_slices * t.n_chunks * (size_t)taps * (size_t)tap_bytes;
    return true;
}

// FFMA path.  Frame plans (a_tma): the band is a_nbox tensor copies of
// a_box_rows <= 256 rows per 4-channel group, a ring of as many stages as
// fit (at least two), one persistent CTA per SM.  Without a frame: one stage,
// one CTA per work unit.
bool size_simt(const Geometry &g, Tiling &t, int sm_count) {
    t.tm = 1;
    t.n_slices = ceil_div(g.Ci, t.bn);
    t.n_chunks = ceil_div(g.Co, t.kc);
    t.chunk_bytes = g.n_taps * t.kc * t.bn * 4;
    int max_phase_taps = 0;
    for (int p = 0; p < g.n_phases; ++p) max_phase_taps = std::max(max_phase_taps, g.phase[p].tap_count);
    t.tap_group = std::max(1, max_phase_taps);
    t.b_resident = 0;
    t.acc_bufs = t.acc_cols = t.tmem_cols = 0;
    t.tile_step = simt_unit_rows(t.bn);
    t.n_tiles = (int)((g.positions + t.tile_step - 1) / t.tile_step);
    t.n_work = (long long)t.n_tiles * t.n_slices * g.n_phases;
    t.packed_bytes = (size_t)t.n_slices * t.n_chunks * (size_t)t.chunk_bytes;
    const int raw = simt_unit_rows(t.bn) + g.max_shift;
    t.band_rows = raw;
    if (t.a_tma) {
        t.a_nbox = ceil_div(raw, 256);
        t.a_box_rows = round_up(ceil_div(raw, t.a_nbox), 8);
        t.a_rows = t.a_nbox * t.a_box_rows;
        const int stage = simt_stage_bytes(t.a_rows, t.kc, t.bn, t.tap_group);
        if (t.n_work > INT_MAX) return false;
        // 64-channel slices: 8 x 8 register tiles, two CTAs per SM, when two
        // stages each fit in half of the SM's shared memory (228 KB, 1 KB per
        // CTA reserved).  Measured steps (frame): resnet_stage 195 us vs 204
        // with 8 x 4 tiles, pointwise 219 vs 244 (few taps: launched without
        // the dependent launch -- its half-size CTAs, resident early, slowed
        // the pack: 259 us), strided_downsample 118 vs 131 (with the
        // tap-balanced schedule; round-robin, 203 us vs 170).
        const int half = (kSmemPerSm / 2 - 1024 - kSimtPipeHeader) / stage;
        t.simt_wide = t.bn == 64 && half >= 2 ? 1 : 0;
        const int stages = std::min(kSimtMaxStages, t.simt_wide ? half : (kMaxSmem - kSimtPipeHeader) / stage);
        if (stages < 2) return false;
        t.a_stages = t.b_stages = stages;
        t.smem_bytes = kSimtPipeHeader + stages * stage;
        t.grid = (int)std::min<long long>(t.n_work, (long long)(t.simt_wide ? 2 : 1) * sm_count);
        return true;
    }
    t.a_rows = round_up(raw, 8);
    const int a_bytes = t.a_rows * t.kc * 4;
    const int b_bytes = max_phase_taps * t.kc * t.bn * 4;
    t.a_stages = 1;
    t.b_stages = 1;
    t.smem_bytes = a_bytes + b_bytes;
    if (t.smem_bytes > kMaxSmem) return false;
    t.grid = 0;
    return true;
}

// col2im path: GEMM N = Ci*kH*kW columns (one 128-byte packed row each),
// K = Co in 32-channel chunks, M = 128 frame positions per tile; the packed
// weights stay resident; a band of R input rows (a multiple of the stride)
// collects the tiles of the positions that reach it.  R minimises the
// busiest CTA's tile count (bands are dealt round-robin), preferring larger
// bands on ties (fewer write-outs).
dgrad_status_t choose_c2i(const Geometry &g, int precision, int sm_count, Tiling *out) {
    if (precision != DGRAD_PREC_TF32) return DGRAD_ERR_UNSUPPORTED;
    const int ncols = g.Ci * g.kH * g.kW;
    if (ncols > kC2iMaxCols || g.Ci > 4) return DGRAD_ERR_UNSUPPORTED;   // stems: up to 4 input channels
    Tiling t{};
    t.path = DGRAD_PATH_COL2IM;
    t.tm = 1;
    t.bn = round_up(ncols, 16);
    t.n_slices = 1;
    t.kc = 32;
    t.n_chunks = ceil_div(g.Co, 32);
    if (t.n_chunks > 32) return DGRAD_ERR_UNSUPPORTED;   // one resident-weight barrier per chunk
    t.co_v = std::max(32, round_up(g.Co, 4));
    t.frame_bytes = (size_t)g.positions * t.co_v * 4;
    if ((long long)g.positions * t.co_v > INT_MAX) return DGRAD_ERR_UNSUPPORTED;
    t.a_tma = 1;
    t.a_box_rows = kBlockM;
    t.a_nbox = 1;
    t.a_rows = kBlockM;
    t.b_resident = 1;
    t.chunk_bytes = t.bn * 128;
    t.packed_bytes = (size_t)t.n_chunks * t.chunk_bytes;
    // band row: input columns iw at iw + pw; wide enough for every contribution
    // (iw + pw <= (oW - 1)*s + kW - 1) and for every column written out (< W + pw)
    t.c2i_pitch = std::max((g.oW - 1) * g.s + g.kW, g.W + g.pw);
    const long long b_all = (long long)t.packed_bytes;
    const int a_bytes = kBlockM * 128;
    long long best = LLONG_MAX;
    for (int R = g.s; R <= 64; R += g.s) {
        const long long acc = 4LL * 4 * g.Ci * R * t.c2i_pitch;   // one band copy per epilogue warp
        const long long left = kMaxSmem - kBarrierBytes - b_all - acc;
        const int stages = (int)std::min<long long>(4, left / a_bytes);
        if (stages < 2) break;
        // positions (frame rows) a band of R rows needs: oh with oh*s - ph + kh in [r0, r0 + R)
        const int rows = (R - 1 + g.kH - 1) / g.s + 1;
        const long long tiles = ((long long)rows * g.Wp + kBlockM - 1) / kBlockM;
        const long long bands = (long long)g.N * ceil_div(g.H, R);
        const long long grid = std::min<long long>(bands, sm_count);
        // a tile's chunks fill n_chunks stages: with fewer than two tiles'
        // worth the next tile's copies cannot start early (measured on the
        // 7x7 stem: 226 us with two stages of two chunks), so such a band
        // size costs three times its tiles
        const long long cost = (bands + grid - 1) / grid * tiles * (stages >= 2 * t.n_chunks ? 1 : 3);
        if (cost <= best) {
            best = cost;
            t.c2i_R = R;
            t.a_stages = stages;
            t.smem_bytes = (int)(kBarrierBytes + b_all + (long long)stages * a_bytes + acc);
        }
        if (R >= g.H) break;
    }
    if (best == LLONG_MAX) return DGRAD_ERR_UNSUPPORTED;
    t.c2i_bands = g.N * ceil_div(g.H, t.c2i_R);
    t.b_stages = t.n_chunks;
    t.n_tiles = t.c2i_bands;
    t.n_work = t.c2i_bands;
    t.grid = std::max(1, std::min(t.c2i_bands, sm_count));
    t.acc_bufs = 2;
    t.acc_cols = t.bn;
    t.tmem_cols = pow2_at_least(2 * t.bn);
    t.tile_step = kBlockM;
    *out = t;
    return DGRAD_OK;
}

}  // namespace

dgrad_status_t choose_tiling(const Geometry &g, int precision, const dgrad_options_t *opts,
                             int sm_count, Tiling *out) {
    dgrad_options_t o{};
    if (opts) o = *opts;
    if (sm_count < 1) sm_count = 152;
    int path = o.path;
    const bool split = precision == DGRAD_PREC_TF32X3;
    if (path == DGRAD_PATH_AUTO) path = (precision == DGRAD_PREC_FP32) ? DGRAD_PATH_SIMT : DGRAD_PATH_TCGEN05;
    if (path == DGRAD_PATH_COL2IM) return choose_c2i(g, precision, sm_count, out);
    if (path != DGRAD_PATH_SIMT && path != DGRAD_PATH_TCGEN05) return DGRAD_ERR_INVALID_ARG;
    if (path == DGRAD_PATH_TCGEN05 && precision == DGRAD_PREC_FP32) return DGRAD_ERR_UNSUPPORTED;
    if (path == DGRAD_PATH_SIMT && split) return DGRAD_ERR_UNSUPPORTED;
    if (o.slice_n && (o.slice_n % 16 || o.slice_n > 256)) return DGRAD_ERR_INVALID_ARG;
    if (o.chunk_k && (o.chunk_k % 8 || o.chunk_k > 64)) return DGRAD_ERR_INVALID_ARG;
    if (o.tile_blocks < 0 || o.tile_blocks > 4 || o.grid < 0) return DGRAD_ERR_INVALID_ARG;

    Tiling t{};
    t.path = path;
    t.split = split ? 1 : 0;
    const int passes = split ? 3 : 1;   // K passes per channel chunk
    if (path == DGRAD_PATH_SIMT) {
        int ci16 = round_up(g.Ci, 16);
        t.bn = o.slice_n ? o.slice_n : (ci16 <= 16 ? 16 : ci16 <= 32 ? 32 : 64);
        if (t.bn != 16 && t.bn != 32 && t.bn != 64) return DGRAD_ERR_INVALID_ARG;
        // At most 4 input channels: 4-channel slices in the gather kernel
        // (1024-position units), instead of 16-channel ones of which 12 or
        // more are padding, where the 1024-position units still fill a wave
        // of CTAs (smaller problems keep the 128-position units: more CTAs);
        // the frame pipeline keeps 16.  Measured: stem step 371 us vs 1267.
        const bool narrow = !o.slice_n && g.Ci <= 4 && o.a_source != 1 &&
                            g.positions * g.n_phases >= (long long)simt_unit_rows(4) * sm_count;
        t.kc = o.chunk_k ? o.chunk_k : 16;
        if (t.kc != 8 && t.kc != 16 && t.kc != 32) return DGRAD_ERR_INVALID_ARG;
        if (o.a_source < 0 || o.a_source > 4) return DGRAD_ERR_INVALID_ARG;
        if (o.a_source == 3 || o.a_source == 4) return DGRAD_ERR_UNSUPPORTED;
        // grad_out reaches the FFMA loop as tensor copies of the packed frame
        // (the pipelined kernel), or gathered by the CTA's own threads
        // (a_source 2, and plans without a frame buffer).  Automatic: the
        // frame where every phase has at most 4 taps, or where the frame
        // pipeline runs 8 x 8 register tiles; else the gather.  The frame
        // costs a pack pass, and with the same 8 x 4 tiles its FFMA loop runs
        // no faster than the gather's (both are bound by the shared-memory
        // reads of the register tiles): it wins where the band fill is a large
        // share of a chunk's work, i.e. few taps per chunk (measured steps:
        // pointwise 244 us vs 341, strided_downsample 175 vs 184), or with
        // the larger tiles (resnet_stage 195 vs 200; with 8 x 4 tiles 204);
        // the stem (16-channel slices) 1625 vs 1268.
        t.co_v = std::max(32, round_up(g.Co, 4));
        t.frame_bytes = (size_t)g.positions * t.co_v * 4;
        const bool frame_fits = t.frame_bytes <= kMaxFrameBytes && (long long)g.positions * t.co_v <= INT_MAX;
        if (o.a_source == 1 && (long long)g.positions * t.co_v > INT_MAX) return DGRAD_ERR_UNSUPPORTED;
        int max_phase_taps = 0;
        for (int p = 0; p < g.n_phases; ++p) max_phase_taps = std::max(max_phase_taps, g.phase[p].tap_count);
        t.a_tma = o.a_source == 2 ? 0 : o.a_source == 1 ? 1 : frame_fits ? 1 : 0;
        bool sized = size_simt(g, t, sm_count);
        if (narrow && (!t.a_tma || !sized || (max_phase_taps > 4 && !t.simt_wide))) {
            Tiling t4 = t;   // the gather kernel with 4-channel slices, where its band fits
            t4.bn = 4;
            t4.a_tma = 0;
            t4.simt_wide = 0;
            if (size_simt(g, t4, sm_count)) {
                t = t4;
                sized = true;
            }
        }
        if (!sized && (o.a_source != 0 || !t.a_tma)) return DGRAD_ERR_UNSUPPORTED;
        if (o.a_source == 0 && t.a_tma && (!sized || (max_phase_taps > 4 && !t.simt_wide))) {
            t.a_tma = 0;   // automatic: no ring of two stages, or 8 x 4 tiles on many taps; gather instead
            t.simt_wide = 0;
            if (!size_simt(g, t, sm_count)) return DGRAD_ERR_UNSUPPORTED;
        }
        if (!t.a_tma) t.frame_bytes = 0;
        *out = t;
        return DGRAD_OK;
    }

    // tcgen05: one MMA block is 128 positions x bn input channels; every
    // active phase has its own fp32 accumulator in tensor memory.
    int ci16 = round_up(g.Ci, 16);
    int bn_cap = std::min(256, (kTmemCols / g.n_phases) / 16 * 16);
    int bn = std::min(ci16, bn_cap);
    int tiles1 = (int)((g.positions + kBlockM - 1) / kBlockM);
    // Slice width: the fewest waves of work units times the cost of one unit,
    // counted in shared-memory cycles (the operand port moves 128 B/clk; an
    // MMA of N columns takes max(N/2, its operand bytes / 128) cycles per K
    // step of 8, and the tensor copies of A and streamed B add their bytes).
    if (!o.slice_n) {
        const int taps = std::max(1, g.n_taps);
        const double a_band = (double)(kBlockM + g.max_shift) * 128.0;
        double best = 1e300;
        int best_bn = bn;
        for (int cand = bn; cand >= 16 && cand % 16 == 0; cand /= 2) {
            const int slices = ceil_div(g.Ci, cand);
            const long long units = (long long)tiles1 * slices;
            const long long waves = (units + sm_count - 1) / sm_count;
            const double mma = taps * 4.0 * std::max(cand / 2.0, (4096.0 + cand * 32.0) / 128.0);
            const bool resident =
                slices == 1 && (double)ceil_div(g.Co, 32) * passes * taps * cand * 128.0 <= 150.0 * 1024;
            const double copies = (a_band + (resident ? 0.0 : taps * cand * 128.0)) / 128.0;
            const double cost = (double)waves * ceil_div(g.Co, 32) * passes * (mma + copies);
            if (cost < best * 0.98) {
                best = cost;
                best_bn = cand;
            }
        }
        bn = best_bn;
    }
    if (o.slice_n) bn = o.slice_n;
    if (g.n_phases * bn > kTmemCols) return DGRAD_ERR_UNSUPPORTED;

    int tm_pref[4] = {0, 0, 0, 0};
    int n_tm = 0;
    if (o.tile_blocks) {
        tm_pref[n_tm++] = o.tile_blocks;
    } else {
        long long units2 = (long long)ceil_div(tiles1, 2) * ceil_div(g.Ci, bn);
        if (units2 >= 2LL * sm_count) tm_pref[n_tm++] = 2;
        tm_pref[n_tm++] = 1;
    }
    // Operand rows are one 128-byte swizzle row: 32 output channels per chunk.
    if (o.chunk_k && o.chunk_k != 32) return DGRAD_ERR_INVALID_ARG;
    if (o.a_source < 0 || o.a_source > 4) return DGRAD_ERR_INVALID_ARG;
    // grad_out reaches the MMA either as tensor copies of a packed,
    // channels-last frame, or through producer warps.  Split precision takes
    // the frame at any size: its rows carry the hi and lo halves, each padded
    // to whole 32-channel chunks so that a chunk's copy never reads the other
    // half.
    t.co_h = split ? round_up(g.Co, 32) : 0;
    t.co_v = split ? 2 * t.co_h : std::max(32, round_up(g.Co, 4));
    t.frame_bytes = (size_t)g.positions * t.co_v * 4;
    if (split && o.a_source == 2) return DGRAD_ERR_UNSUPPORTED;
    if (o.a_source == 1 || split)
        t.a_tma = 1;
    else if (o.a_source == 2)
        t.a_tma = 0;
    else
        t.a_tma = t.frame_bytes <= kMaxFrameBytes ? 1 : 0;
    // Staged A source (no frame, no grad_out pack): each A stage is one
    // tensor copy of grad_out viewed as [N][Co][oH*oW] (the plane stride
    // must be a multiple of 16 bytes) holding the band's plane elements,
    // which needs a band of at most 253 rows (one 128-row block).  Opt-in:
    // measured slower than the frame on every workload (resnet_stage main
    // kernel 50 us vs 25), because the in-place transposition's shared-
    // memory reads and writes compete with the tensor core's operand reads
    // for the shared-memory port.
    const bool stg_ok = (long long)g.oH * g.oW % 4 == 0 && kBlockM + g.max_shift + 3 <= 256;
    t.a_staged = 0;
    if (o.a_source == 3) {
        if (!stg_ok || o.tile_blocks > 1) return DGRAD_ERR_UNSUPPORTED;
        t.a_tma = 1;
        t.a_staged = 1;
    }
    // 1x1 kernel, stride 1, no padding: the operand A of a tile is grad_out
    // itself, with no shifted windows, so it can sit in tensor memory
    // (tcgen05.mma reads A from there): the epilogue warps write each
    // 32-channel chunk of a tile there from a tensor copy of the NCHW planes
    // (no frame, no grad_out pass).  Needs planes of at least 128 elements
    // (a tile then spans at most two images) that start 16-byte aligned.
    // The automatic choice for such shapes (pointwise step 47.4 -> 36.6 us in
    // TF32, 88.6 -> 75.2 in split precision: the frame pass is gone).
    const long long plane = (long long)g.oH * g.oW;
    const bool tm_ok = g.kH == 1 && g.kW == 1 && g.s == 1 && g.ph == 0 && g.pw == 0 && plane % 4 == 0 &&
                       plane >= kBlockM && g.n_taps == 1;
    t.a_tmem = 0;
    if (o.a_source == 4) {
        if (!tm_ok || o.tile_blocks > 1 || o.group_taps == 1 || o.group_taps == 3) return DGRAD_ERR_UNSUPPORTED;
        t.a_tma = 1;
        t.a_tmem = 1;
    } else if (o.a_source == 0 && tm_ok && o.tile_blocks <= 1) {
        t.a_tma = 1;
        t.a_tmem = 1;
    }
    if (t.a_tmem) t.frame_bytes = 0;
    if (t.a_staged) t.frame_bytes = 0;
    if (t.a_tma && !t.a_staged && !t.a_tmem && (long long)g.positions * t.co_v > INT_MAX) return DGRAD_ERR_UNSUPPORTED;
    if (!t.a_tma) t.frame_bytes = 0;
    // Grouping the taps of a kernel row into one MMA (N = taps x bn) cuts the
    // MMA time when bn alone leaves the MMA bound by its fixed cost of
    // reading A (a 128 x 64 x 8 TF32 MMA takes ~72 cycles, 128 x 192 x 8 ~106),
    // but triples the epilogue's tensor-memory reads and adds its row
    // shifts.  With the boundary rows exchanged once per unit and a second
    // epilogue warp group (two accumulator sets), the grouped plan is the
    // faster one for one-phase TF32 shapes with bn < 128 (resnet_stage main
    // kernel 25.2 us vs 27.2): the automatic choice there, falling back to
    // ungrouped when it does not fit.  Split precision keeps two 128-row
    // blocks per unit ungrouped (61.9 us vs 64.1 grouped).  Taps of different phases with the
    // same frame shift share one MMA whenever the phases can be ordered in
    // tensor memory for it (stride-2 shapes): fewer, wider MMAs, each phase
    // still its own accumulator, so the epilogue is unchanged.  That is the
    // automatic choice for several phases.
    if (o.group_taps < 0 || o.group_taps > 3) return DGRAD_ERR_INVALID_ARG;
    if (o.b_stages != 0 && (o.b_stages < 2 || o.b_stages > 8)) return DGRAD_ERR_INVALID_ARG;
    t.want_b_stages = o.b_stages;
    int group_pref[2][2];   // (kernel-row groups, shared-shift groups) in order of preference
    int n_group = 0;
    if (o.group_taps == 1) {
        if (o.tile_blocks > 1) return DGRAD_ERR_UNSUPPORTED;   // grouped MMAs take one 128-row block per unit
        group_pref[n_group][0] = 1, group_pref[n_group++][1] = 0;
    } else if (o.group_taps == 3) {
        group_pref[n_group][0] = 0, group_pref[n_group++][1] = 1;
    } else {
        if (o.group_taps == 0 && g.n_phases > 1) group_pref[n_group][0] = 0, group_pref[n_group++][1] = 1;
        if (o.group_taps == 0 && g.n_phases == 1 && t.a_tma && !t.split && g.kW >= 2 && bn < 128 &&
            o.tile_blocks <= 1)
            group_pref[n_group][0] = 1, group_pref[n_group++][1] = 0;
        group_pref[n_group][0] = 0, group_pref[n_group++][1] = 0;
    }
    t.img_align_sms = sm_count;
    bool ok = false;
    for (int gi = 0; gi < n_group && !ok; ++gi) {
        for (int want_res = 1; want_res >= 0 && !ok; --want_res) {
            for (int i = 0; i < n_tm && !ok; ++i) {
                Tiling c = t;
                c.grouped = group_pref[gi][0];
                c.pgroup = group_pref[gi][1];
                c.tm = (c.grouped || c.a_staged || c.a_tmem) ? 1 : tm_pref[i];
                c.bn = bn;
                c.kc = 32;
                if (!size_tc(g, c, want_res)) continue;
                t = c;
                ok = true;
            }
        }
    }
    if (!ok) return DGRAD_ERR_UNSUPPORTED;
    long long grid = o.grid ? o.grid : std::min<long long>(t.n_work, sm_count);
    t.grid = (int)std::max<long long>(1, std::min<long long>(grid, t.n_work));
    *out = t;
    return DGRAD_OK;
}

void fill_main_params(const Geometry &g, const Tiling &t, int round_tf32, MainParams *mp) {
    MainParams &m = *mp;
    std::memset(&m, 0, sizeof(m));
    m.N = g.N; m.Ci = g.Ci; m.Co = g.Co; m.H = g.H; m.W = g.W; m.oH = g.oH; m.oW = g.oW; m.s = g.s;
    m.Ph = g.Ph; m.Pw = g.Pw; m.Hv = g.Hv; m.Wp = g.Wp; m.HvWp = g.Hv * g.Wp;
    m.positions = (int)g.positions;
    m.tm = t.tm; m.bn = t.bn; m.n_slices = t.n_slices; m.kc = t.kc; m.n_chunks = t.n_chunks;
    m.n_tiles = t.n_tiles; m.n_work = (int)t.n_work;
    m.a_rows = t.a_rows; m.a_stages = t.a_stages; m.b_stages = t.b_stages; m.b_resident = t.b_resident;
    m.chunk_bytes = t.chunk_bytes;
    m.tap_group = t.tap_group; m.n_tgroups = t.n_tgroups;
    m.vec_producer = use_vec_producer(g, t) ? 1 : 0;
    m.a_tma = t.a_tma; m.a_box_rows = t.a_box_rows; m.a_nbox = t.a_nbox;
    m.a_staged = t.a_staged; m.stg_box = t.stg_box; m.band_rows = t.band_rows; m.img_tiles = t.img_tiles;
    m.a_tmem = t.a_tmem; m.a_tslots = t.a_tslots; m.a_tcol = t.a_tcol;
    // staged: about 128 KB of grad_out boxes in flight to L2 per CTA, ahead
    // of the copies (HBM latency times a CTA's share of the bandwidth is
    // ~70 KB), at least two stages
    // (tensor-memory A: none -- the prefetches queue on the copy engine ahead
    // of the weight and grad_out copies the MMAs wait for; measured slower)
    m.prefetch_ahead = t.a_staged ? std::max(2, std::min(16, (128 * 1024) / (t.stg_box * 128))) : 0;
    m.acc_bufs = t.acc_bufs; m.acc_cols = t.acc_cols; m.tmem_cols = t.tmem_cols;
    m.round_tf32 = round_tf32;
    m.split_chunks = t.split ? t.n_chunks / 3 : 0;
    m.co_h = t.co_h;
    m.n_phases = g.n_phases;
    m.n_taps = g.n_taps;
    m.idesc = tf32_idesc(kBlockM, t.bn);
    m.tile_step = t.tile_step;
    m.grouped = t.grouped;
    m.xchg_bytes = t.xchg_bytes;
    m.xchg_unit = t.xchg_unit;
    m.epi_groups = t.epi_groups;
    MGroup mg[kMaxTaps];
    int perm[kMaxTaps], units[kMaxPhases];
    const int n_mg = t.path == DGRAD_PATH_TCGEN05 ? build_mgroups(g, t, mg, perm, units) : 0;
    m.max_sub = 1;
    for (int i = 0; i < g.n_phases; ++i) {
        m.phase[i] = g.phase[i];
        m.phase[i].sub = t.grouped ? g.phase[i].row_len : 1;
        m.phase[i].col = t.path == DGRAD_PATH_TCGEN05 ? units[i] * t.bn : i * t.bn;
        m.max_sub = std::max(m.max_sub, m.phase[i].sub);
    }
    // The epilogue stores the s column phases of a row phase together when
    // each row is whole (W % s == 0, every phase present) and the tensor-
    // memory loads of one batch of them fit in 64 registers.
    m.vec_w = (t.path == DGRAD_PATH_TCGEN05 && (g.s == 2 || g.s == 4) && g.W % g.s == 0 &&
               g.n_phases == g.s * g.s && g.s * m.max_sub <= 4) ? 1 : 0;
    for (int i = 0; i < g.n_taps; ++i) m.tap[i] = g.tap[i];
    if (t.path == DGRAD_PATH_TCGEN05) {
        m.n_mgroups = n_mg;
        const uint32_t tap_b = (uint32_t)t.bn * 128u;   // bytes of one tap of one chunk of B
        for (int i = 0; i < m.n_mgroups; ++i) {
            m.mgroup[i].x = (uint32_t)mg[i].a_shift * 128u;
            m.mgroup[i].y = (uint32_t)(mg[i].col * t.bn) | (mg[i].first ? 0x80000000u : 0u);
            m.mgroup[i].z = (uint32_t)mg[i].tap0 * tap_b;
            m.mgroup[i].w = tf32_idesc(kBlockM, mg[i].ntaps * t.bn);
        }
        for (int i = 0; i <= t.n_tgroups; ++i) {
            m.bg_first[i] = t.bg_first[i];
            m.bg_tap0[i] = t.bg_first[i] < m.n_mgroups ? mg[t.bg_first[i]].tap0 : g.n_taps;
        }
    }
}

void fill_prepack_params(const Geometry &g, const Tiling &t, int round_tf32, PrepackParams *qp) {
    PrepackParams &q = *qp;
    std::memset(&q, 0, sizeof(q));
    q.Co = g.Co; q.Ci = g.Ci; q.kH = g.kH; q.kW = g.kW;
    q.n_taps = g.n_taps; q.bn = t.bn; q.n_slices = t.n_slices; q.kc = t.kc; q.n_chunks = t.n_chunks;
    q.round_tf32 = round_tf32;
    q.split_chunks = t.split ? t.n_chunks / 3 : 0;
    q.layout = t.path == DGRAD_PATH_TCGEN05 ? 1 : (t.path == DGRAD_PATH_COL2IM ? 2 : 0);
    q.total = (long long)(t.packed_bytes / 4);
    // tcgen05 path: taps in the packing order of the plan's MMA groups
    MGroup mg[kMaxTaps];
    int perm[kMaxTaps], units[kMaxPhases];
    if (t.path != DGRAD_PATH_TCGEN05 || build_mgroups(g, t, mg, perm, units) < 0)
        for (int i = 0; i < g.n_taps; ++i) perm[i] = i;
    for (int i = 0; i < g.n_taps; ++i) {
        q.tap_kh[i] = g.tap[perm[i]].kh;
        q.tap_kw[i] = g.tap[perm[i]].kw;
    }
}

}  // namespace dgrad

namespace dgrad {

void fill_c2i_params(const Geometry &g, const Tiling &t, C2iParams *cp) {
    C2iParams &c = *cp;
    std::memset(&c, 0, sizeof(c));
    c.N = g.N; c.Ci = g.Ci; c.H = g.H; c.W = g.W; c.Co = g.Co; c.kH = g.kH; c.kW = g.kW;
    c.s = g.s; c.ph = g.ph; c.pw = g.pw; c.oH = g.oH; c.oW = g.oW;
    c.Ph = g.Ph; c.Pw = g.Pw; c.Hv = g.Hv; c.Wp = g.Wp;
    c.n_chunks = t.n_chunks; c.bn = t.bn; c.ncols = g.Ci * g.kH * g.kW;
    c.R = t.c2i_R; c.pitch = t.c2i_pitch;
    c.bands_per_img = (g.H + t.c2i_R - 1) / t.c2i_R;
    c.n_bands = t.c2i_bands;
    c.a_stages = t.a_stages; c.tmem_cols = t.tmem_cols; c.chunk_bytes = t.chunk_bytes;
    c.idesc = tf32_idesc(kBlockM, t.bn);
    for (int r = 0; r < c.ncols && r < kC2iMaxCols; ++r) {   // tap-major columns: r = (kh*kW + kw)*Ci + ci
        const int tap = r / g.Ci, ci = r % g.Ci, kh = tap / g.kW, kw = tap % g.kW;
        c.col_kh[r] = kh;
        c.col_off[r] = (ci * t.c2i_R + kh) * t.c2i_pitch + kw;
    }
}

}  // namespace dgrad
