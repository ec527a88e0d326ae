// Host side of libconvt3d: descriptor validation, the output-parity class
// decomposition, workspace layout and the C-ABI entry points.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "convt3d_internal.h"

using namespace convt3d;

namespace {

thread_local char g_last_error[512] = "";

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

convt3d_status_t fail(convt3d_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

convt3d_status_t cuda_fail(cudaError_t e, const char *what) {
    set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return CONVT3D_ERR_CUDA;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Output extent along one dimension: (in-1)*s - 2p + dil*(k-1) + op + 1.
int64_t out_extent(int64_t in, int k, int s, int p, int op, int dil) {
    return (in - 1) * s - 2 * p + (int64_t)dil * (k - 1) + op + 1;
}

// The per-dimension shape a descriptor describes (index 0 = d, 1 = h, 2 = w).
struct Shape {
    int kk[3], ss[3], pp[3], op[3], dil[3];
    int G;
};

Shape shape_of(const convt3d_desc_t &d) {
    Shape s;
    for (int a = 0; a < 3; ++a) {
        s.kk[a] = d.per_dim ? d.kdims[a] : d.k;
        s.ss[a] = d.per_dim ? d.strides[a] : d.stride;
        s.pp[a] = d.per_dim ? d.pads[a] : d.pad;
        s.op[a] = d.per_dim ? d.out_pads[a] : d.out_pad;
        s.dil[a] = d.dilation[a] == 0 ? 1 : d.dilation[a];
    }
    s.G = d.conv_groups == 0 ? 1 : d.conv_groups;
    return s;
}

// Output-parity decomposition.  For output index o = s*q + r along one
// dimension, the taps t that reach it satisfy (r + p - dil*t) = s*delta for an
// integer delta, and then read input index i = q + delta (the gather form
// of the index relation od = id*s - p + kd derived on page l2_p49, with the
// dilated tap position dil*kd).  For stride 1 there is one class holding all
// k taps with delta = p - dil*t.
struct DimTaps {
    int n;
    int t[8];
    int delta[8];
    int Q;
};

DimTaps dim_taps(int Dout, int k, int s, int p, int dil, int r) {
    DimTaps d{};
    for (int t = 0; t < k; ++t) {
        int num = r + p - dil * t;
        if (((num % s) + s) % s == 0) {
            d.t[d.n] = t;
            d.delta[d.n] = num / s;  // exact division
            ++d.n;
        }
    }
    d.Q = Dout > r ? (Dout - r + s - 1) / s : 0;
    return d;
}

bool build_geometry(const convt3d_desc_t &d, Geometry &g) {
    memset(&g, 0, sizeof(g));
    const Shape sh = shape_of(d);
    g.N = d.N; g.Cin = d.Cin; g.Cout = d.Cout; g.Din = d.Din; g.Hin = d.Hin; g.Win = d.Win;
    for (int a = 0; a < 3; ++a) {
        g.kk[a] = sh.kk[a]; g.ss[a] = sh.ss[a]; g.pp[a] = sh.pp[a]; g.op[a] = sh.op[a]; g.dil[a] = sh.dil[a];
    }
    g.kvol = g.kk[0] * g.kk[1] * g.kk[2];
    g.G = sh.G;
    const int in[3] = {d.Din, d.Hin, d.Win};
    int out[3];
    for (int a = 0; a < 3; ++a) out[a] = (int)out_extent(in[a], g.kk[a], g.ss[a], g.pp[a], g.op[a], g.dil[a]);
    g.Do = out[0]; g.Ho = out[1]; g.Wo = out[2];
    g.nclasses = g.ss[0] * g.ss[1] * g.ss[2];
    int tap = 0;
    for (int rd = 0; rd < g.ss[0]; ++rd)
        for (int rh = 0; rh < g.ss[1]; ++rh)
            for (int rw = 0; rw < g.ss[2]; ++rw) {
                const int c = (rd * g.ss[1] + rh) * g.ss[2] + rw;
                DimTaps td = dim_taps(g.Do, g.kk[0], g.ss[0], g.pp[0], g.dil[0], rd);
                DimTaps th = dim_taps(g.Ho, g.kk[1], g.ss[1], g.pp[1], g.dil[1], rh);
                DimTaps tw = dim_taps(g.Wo, g.kk[2], g.ss[2], g.pp[2], g.dil[2], rw);
                ClassDesc &cl = g.cls[c];
                cl.rd = rd; cl.rh = rh; cl.rw = rw;
                cl.Qd = td.Q; cl.Qh = th.Q; cl.Qw = tw.Q;
                cl.nt_d = td.n; cl.nt_h = th.n; cl.nt_w = tw.n;
                cl.ntaps = td.n * th.n * tw.n;
                cl.tap_begin = tap;
                cl.step_d = g.dil[0];
                cl.lo_d = cl.lo_h = cl.lo_w = 0;
                if (td.n) cl.lo_d = *std::min_element(td.delta, td.delta + td.n);
                if (th.n) cl.lo_h = *std::min_element(th.delta, th.delta + th.n);
                if (tw.n) cl.lo_w = *std::min_element(tw.delta, tw.delta + tw.n);
                for (int a = 0; a < td.n; ++a)
                    for (int b = 0; b < th.n; ++b)
                        for (int e = 0; e < tw.n; ++e) {
                            if (tap >= kMaxTaps) return false;
                            TapDesc &t = g.taps[tap++];
                            t.dd = (int8_t)td.delta[a];
                            t.dh = (int8_t)th.delta[b];
                            t.dw = (int8_t)tw.delta[e];
                            t.widx = (int16_t)((td.t[a] * g.kk[1] + th.t[b]) * g.kk[2] + tw.t[e]);
                        }
            }
    g.ntaps = tap;
    return tap == g.kvol;
}

// Arrange classes into GEMM groups and order groups heaviest first.
void build_groups(convt3d_plan_s &p) {
    const Geometry &g = p.g;
    const int kchunk = p.chunk;
    const int kc = (g.Cin + kchunk - 1) / kchunk;
    p.ngroups = 0;
    // the two w-parity classes of each (rd, rh) share a tile where both accumulators fit
    // tensor memory twice (double-buffered): 2 classes x Cout_pad x 2 <= 512 columns
    if (p.tc && g.ss[2] == 2 && p.cout_pad <= 128) {
        for (int rd = 0; rd < g.ss[0]; ++rd)
            for (int rh = 0; rh < g.ss[1]; ++rh) {
                GroupDesc &G = p.grp[p.ngroups++];
                G.ncls = 2;
                G.cls[0] = (rd * g.ss[1] + rh) * 2 + 0;
                G.cls[1] = (rd * g.ss[1] + rh) * 2 + 1;
                const ClassDesc &a = g.cls[G.cls[0]], &b = g.cls[G.cls[1]];
                G.Qd = a.Qd; G.Qh = a.Qh; G.Qw = std::max(a.Qw, b.Qw);
                G.ksteps = (a.ntaps + b.ntaps) * kc;
            }
    } else {
        for (int c = 0; c < g.nclasses; ++c) {
            GroupDesc &G = p.grp[p.ngroups++];
            G.ncls = 1;
            G.cls[0] = G.cls[1] = c;
            const ClassDesc &a = g.cls[c];
            G.Qd = a.Qd; G.Qh = a.Qh; G.Qw = a.Qw;
            G.ksteps = a.ntaps * kc;
        }
    }
    // Merged w-taps of each pair: the distinct w offsets of the two classes,
    // shared ones first.  A K step of a shared offset loads the activation
    // slice once and feeds both classes with one MMA of N = 2 * Cout_pad.
    for (int i = 0; i < p.ngroups; ++i) {
        GroupDesc &G = p.grp[i];
        G.nm = 0;
        if (G.ncls != 2) continue;
        const ClassDesc &c0 = g.cls[G.cls[0]], &c1 = g.cls[G.cls[1]];
        int dw[2][8], n[2] = {c0.nt_w, c1.nt_w};
        for (int e = 0; e < n[0]; ++e) dw[0][e] = g.taps[c0.tap_begin + e].dw;
        for (int e = 0; e < n[1]; ++e) dw[1][e] = g.taps[c1.tap_begin + e].dw;
        for (int pass = 0; pass < 2; ++pass)  // pass 0: shared offsets, pass 1: the rest
            for (int c = 0; c < 2; ++c)
                for (int e = 0; e < n[c]; ++e) {
                    int other = -1;
                    for (int f = 0; f < n[1 - c]; ++f)
                        if (dw[1 - c][f] == dw[c][e]) other = f;
                    const bool shared = other >= 0;
                    if ((pass == 0) != shared || (shared && c == 1)) continue;
                    const int m = G.nm++;
                    G.mdw[m] = (int8_t)dw[c][e];
                    G.mmask[m] = (uint8_t)(shared ? 3 : 1 << c);
                    G.me[m][c] = (int8_t)e;
                    G.me[m][1 - c] = (int8_t)other;
                }
    }
    std::stable_sort(p.grp, p.grp + p.ngroups,
                     [](const GroupDesc &a, const GroupDesc &b) { return a.ksteps > b.ksteps; });
    int prefix = 0;
    for (int i = 0; i < p.ngroups; ++i) {
        GroupDesc &G = p.grp[i];
        G.vol = G.Qd * G.Qh * G.Qw;
        G.tiles = (G.vol + p.tile_m - 1) / p.tile_m;
        G.div_qw = make_fastdiv((uint32_t)std::max(G.Qw, 1));
        G.div_qhw = make_fastdiv((uint32_t)std::max(G.Qh * G.Qw, 1));
        G.tile_prefix = prefix;
        prefix += G.tiles;
    }
    p.tiles_per_sample = prefix;
    p.tiles = (int64_t)prefix * g.N;
}

convt3d_status_t validate(const convt3d_desc_t &d) {
    if (d.N < 1 || d.Cin < 1 || d.Cout < 1 || d.Din < 1 || d.Hin < 1 || d.Win < 1)
        return fail(CONVT3D_ERR_INVALID_ARG, "sizes must be >= 1");
    for (int a = 0; a < 3; ++a)
        if (d.dilation[a] < 0) return fail(CONVT3D_ERR_INVALID_ARG, "dilation must be >= 1 (0 means 1)");
    if (d.conv_groups < 0) return fail(CONVT3D_ERR_INVALID_ARG, "conv_groups must be >= 1 (0 means 1)");
    const Shape sh = shape_of(d);
    const int in[3] = {d.Din, d.Hin, d.Win};
    int64_t out[3];
    for (int a = 0; a < 3; ++a) {
        if (sh.kk[a] < 1 || sh.ss[a] < 1 || sh.pp[a] < 0 || sh.op[a] < 0)
            return fail(CONVT3D_ERR_INVALID_ARG, "k, stride >= 1 and pad, out_pad >= 0 required");
        if (sh.op[a] >= std::max(sh.ss[a], sh.dil[a]))
            return fail(CONVT3D_ERR_INVALID_ARG, "out_pad must be smaller than stride or dilation");
        out[a] = out_extent(in[a], sh.kk[a], sh.ss[a], sh.pp[a], sh.op[a], sh.dil[a]);
        if (out[a] < 1) return fail(CONVT3D_ERR_INVALID_ARG, "output extent < 1");
    }
    if (d.Cin % sh.G || d.Cout % sh.G) return fail(CONVT3D_ERR_INVALID_ARG, "conv_groups must divide Cin and Cout");
    if (d.epilogue < CONVT3D_EPI_IDENTITY || d.epilogue > CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL)
        return fail(CONVT3D_ERR_INVALID_ARG, "unknown epilogue %d", d.epilogue);
    if (d.precision < CONVT3D_PREC_3XTF32 || d.precision > CONVT3D_PREC_FP16)
        return fail(CONVT3D_ERR_INVALID_ARG, "unknown precision %d", d.precision);
    if (d.epilogue == CONVT3D_EPI_RELU_GROUPNORM && (d.groups < 1 || d.Cout % d.groups != 0))
        return fail(CONVT3D_ERR_INVALID_ARG, "groups must divide Cout");
    const bool bn_any = d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL ||
                        d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL;
    if ((d.epilogue == CONVT3D_EPI_RELU_GROUPNORM || bn_any) && !(d.eps > 0.0f && isfinite(d.eps)))
        return fail(CONVT3D_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (bn_any && !isfinite(d.scale)) return fail(CONVT3D_ERR_INVALID_ARG, "scale must be finite");
    // Limits of this build (valid operations it does not run).
    if (d.io_bf16 && d.io_fp16) return fail(CONVT3D_ERR_INVALID_ARG, "io_bf16 and io_fp16 are exclusive");
    if (d.io_bf16 && d.precision != CONVT3D_PREC_BF16)
        return fail(CONVT3D_ERR_UNSUPPORTED, "bf16 tensors need precision CONVT3D_PREC_BF16");
    if (d.io_fp16 && d.precision != CONVT3D_PREC_FP16)
        return fail(CONVT3D_ERR_UNSUPPORTED, "fp16 tensors need precision CONVT3D_PREC_FP16");
    for (int a = 0; a < 3; ++a) {
        if (sh.ss[a] > 2) return fail(CONVT3D_ERR_UNSUPPORTED, "stride > 2");
        if (sh.kk[a] > 7) return fail(CONVT3D_ERR_UNSUPPORTED, "k > 7");
        if (sh.dil[a] * (sh.kk[a] - 1) > 30) return fail(CONVT3D_ERR_UNSUPPORTED, "dilation * (k - 1) > 30");
        if (sh.pp[a] > sh.dil[a] * (sh.kk[a] - 1)) return fail(CONVT3D_ERR_UNSUPPORTED, "pad > dilation * (k - 1)");
        if (sh.ss[a] == 2 && (sh.kk[a] < 2 || sh.dil[a] % 2 == 0))
            return fail(CONVT3D_ERR_UNSUPPORTED, "stride 2 needs k >= 2 and an odd dilation (parity classes without taps)");
    }
    if (d.Cout > kMaxCout) return fail(CONVT3D_ERR_UNSUPPORTED, "Cout > 512");
    const int64_t lim = (int64_t)1 << 31;
    if ((int64_t)d.N * d.Cout * out[0] * out[1] * out[2] >= lim || (int64_t)d.N * d.Cin * d.Din * d.Hin * d.Win >= lim / 2 ||
        (int64_t)d.N * 256 * d.Din * d.Hin * d.Win >= ((int64_t)1 << 40))
        return fail(CONVT3D_ERR_UNSUPPORTED, "tensor larger than 2^31 elements");
    return CONVT3D_OK;
}

// The tensor-core path loads activation tiles with TMA im2col, whose
// bounding-box corners must lie in [-16, 15] for 5-D tensors: per dimension
// the lower corner is the smallest tap offset and the upper corner makes the
// box span exactly the class's Q positions.
bool im2col_corners_ok(const convt3d_plan_s &p) {
    const Geometry &g = p.g;
    for (int i = 0; i < p.ngroups; ++i) {
        const GroupDesc &G = p.grp[i];
        for (int c = 0; c < G.ncls; ++c) {
            const ClassDesc &cl = g.cls[G.cls[c]];
            const int lo[3] = {cl.lo_d, cl.lo_h, cl.lo_w};
            const int Q[3] = {G.Qd, G.Qh, G.Qw};
            const int in[3] = {g.Din, g.Hin, g.Win};
            const int span[3] = {(cl.nt_d - 1) * g.dil[0], (cl.nt_h - 1) * g.dil[1], (cl.nt_w - 1) * g.dil[2]};
            for (int a = 0; a < 3; ++a) {
                const int upper = Q[a] - in[a] + lo[a];
                if (lo[a] < -16 || lo[a] > 15 || upper < -16 || upper > 15) return false;
                if (span[a] > 15) return false;  // per-load im2col offsets (delta - lo) kept within 0..15
            }
        }
    }
    return true;
}

}  // namespace

namespace convt3d {
// Record a failure detail for convt3d_last_error from another translation unit.
void report_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}
}  // namespace convt3d

extern "C" {

int convt3d_version(void) { return 100; }

const char *convt3d_last_error(void) { return g_last_error; }

const char *convt3d_status_string(convt3d_status_t st) {
    switch (st) {
        case CONVT3D_OK: return "ok";
        case CONVT3D_ERR_INVALID_ARG: return "invalid argument";
        case CONVT3D_ERR_UNSUPPORTED: return "unsupported by this build";
        case CONVT3D_ERR_WORKSPACE: return "workspace missing or too small";
        case CONVT3D_ERR_CUDA: return "CUDA error";
        case CONVT3D_ERR_TIMEOUT: return "device-side wait timed out";
        case CONVT3D_ERR_DEVICE_ASSERT: return "device-side check failed";
        case CONVT3D_ERR_NOT_PACKED: return "weights not packed into this workspace";
    }
    return "unknown status";
}

convt3d_status_t convt3d_plan_create(const convt3d_desc_t *desc, convt3d_plan_t *out) {
    g_last_error[0] = 0;
    if (!out) return fail(CONVT3D_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!desc) return fail(CONVT3D_ERR_INVALID_ARG, "desc is NULL");
    convt3d_status_t st = validate(*desc);
    if (st != CONVT3D_OK) return st;
    convt3d_plan_s *p = new (std::nothrow) convt3d_plan_s();
    if (!p) return fail(CONVT3D_ERR_INVALID_ARG, "out of host memory");
    memset(p, 0, sizeof(*p));
    p->d = *desc;
    if (!build_geometry(p->d, p->g)) {
        delete p;
        return fail(CONVT3D_ERR_UNSUPPORTED, "tap table overflow");
    }
    // The main kernel's configuration: tensor cores (tc) or the FFMA kernel.
    auto configure = [&](bool tc) {
        p->tc = tc;
        const bool split = desc->precision == CONVT3D_PREC_3XTF32 || desc->precision == CONVT3D_PREC_3XBF16;
        p->planes = tc ? (split ? 2 : 1) : 0;
        p->cl = desc->channels_last != 0;
        p->io16 = desc->io_bf16 ? kBF16 : (desc->io_fp16 ? kF16 : kF32);
        p->half = tc && desc->precision == CONVT3D_PREC_FP16;
        p->bf16 = tc && (desc->precision == CONVT3D_PREC_BF16 || desc->precision == CONVT3D_PREC_3XBF16 || p->half);
        p->elem_bytes = p->bf16 ? 2 : 4;
        p->chunk = tc ? kTcRowBytes / p->elem_bytes : 8;
        p->tile_m = tc ? kTcTileM : kFfmaTileM;
        p->cin_pad = round_up(desc->Cin, p->chunk);
        p->cout_pad = round_up(desc->Cout, 16);
        p->nslices = 1;
        if (!tc) {  // the FFMA kernel's register tiles need a power-of-two channel count
            while (p->cout_pad & (p->cout_pad - 1)) p->cout_pad += 16;
        } else if (p->cout_pad > kTcMaxSliceN) {
            // one MMA (and one TMA weight box) spans at most 256 columns: equal slices of
            // a multiple of 16 columns, walked one after another over the tile's K steps
            p->nslices = (p->cout_pad + kTcMaxSliceN - 1) / kTcMaxSliceN;
            p->cout_pad = round_up(desc->Cout, 16 * p->nslices);
        }
        // Pairs merge where the combined MMA fits (N = 2 * Cout_pad <= 128): there the
        // instruction count, not the tensor pipe, bounds the main loop.
        p->merged = tc && p->g.ss[2] == 2 && p->cout_pad <= 64;
        build_groups(*p);
    };
    configure(desc->precision != CONVT3D_PREC_FFMA);
    const bool eval_bn = desc->epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL;
    // Few input channels, stride 2 along w, NCDHW fp32 tensors, bf16 operands: the
    // kernel that reads x itself (per-slice TMA slabs, operands split on chip).
    p->direct = p->tc && !eval_bn && direct_supported(*p);
    if (p->tc && !p->direct && !eval_bn && !im2col_corners_ok(*p)) {
        // The tensor-core loads cannot address this shape (TMA im2col corners beyond
        // [-16, 15]): the FFMA kernel runs it instead, in fp32, at least as accurate as any
        // tensor-core precision; it has no 16-bit tensors at the boundary.
        if (desc->io_bf16 || desc->io_fp16) {
            delete p;
            return fail(CONVT3D_ERR_UNSUPPORTED, "shape outside the TMA im2col corner range (16-bit tensors)");
        }
        configure(false);
    }
    if (eval_bn && bn_eval_smem_bytes(*p) > 200 * 1024) {
        delete p;
        return fail(CONVT3D_ERR_UNSUPPORTED, "evaluation-mode BatchNorm needs kd*H*W + kd*kh*W <= 51200");
    }
    p->momentum = 0.1f;

    // Workspace layout.
    size_t off = kStatusBytes;
    p->wpk_elems = (size_t)p->g.ntaps * p->cin_pad * p->cout_pad;
    p->off_wpk_hi = off;
    if (p->direct) {  // the direct kernel's own packed layout (both planes, stage images per d-slice)
        off = align_up(off + direct_weight_bytes(*p), 256);
        p->off_wpk_lo = off;
    } else {
        off = align_up(off + p->wpk_elems * p->elem_bytes, 256);
        p->off_wpk_lo = off;
        if (p->planes == 2) off = align_up(off + p->wpk_elems * p->elem_bytes, 256);
    }
    p->xs_elems = (p->tc && !eval_bn && !p->direct) ? (size_t)desc->N * desc->Din * desc->Hin * desc->Win * p->cin_pad : 0;
    p->off_xs_hi = off;
    off = align_up(off + p->xs_elems * p->elem_bytes, 256);
    p->off_xs_lo = off;
    if (p->planes == 2) off = align_up(off + p->xs_elems * p->elem_bytes, 256);
    size_t per_tile = 0, stat = 0;
    // partial rows hold (count, sum, M2) per group / channel; GroupNorm's statistics are
    // (mean, rstd) per (n, g), BatchNorm's the (count, sum, M2) per (n, row split, c)
    if (desc->epilogue == CONVT3D_EPI_RELU_GROUPNORM) {
        per_tile = 3 * (size_t)desc->groups;
        stat = (size_t)desc->N * desc->groups * 2;
    }
    p->stat_rows_per_tile = p->tc ? kTcStatRows : 1;
    p->bn_splits = 1;
    if (desc->epilogue == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL) {
        // the first reduction splits each sample's rows so that its grid has about
        // 600 blocks of 32 channels (4 per SM), each range at least 8 rows long
        const int rows = p->tiles_per_sample * p->stat_rows_per_tile;
        const int blocks = ((desc->Cout + 31) / 32) * desc->N;
        p->bn_splits = std::max(1, std::min((600 + blocks - 1) / blocks, rows / 8));
        per_tile = 3 * (size_t)desc->Cout;
        stat = (size_t)desc->N * p->bn_splits * desc->Cout * 3;
    }
    p->partial_doubles = per_tile * (size_t)p->tiles * p->stat_rows_per_tile;
    p->stat_doubles = stat;
    p->off_partials = off;
    off = align_up(off + p->partial_doubles * 8, 256);
    p->off_stats = off;
    off = align_up(off + p->stat_doubles * 8, 256);
    p->off_box = off;
    if (eval_bn) off = align_up(off + (size_t)desc->N * desc->Cin * p->g.kvol * 4, 256);
    p->ev_ks = eval_bn ? bn_eval_ksplits(p->g.ntaps, desc->Cin) : 1;
    p->off_evpart = off;
    if (p->ev_ks > 1) off = align_up(off + (size_t)p->ev_ks * desc->N * desc->Cout * 8, 256);
    p->off_evcnt = off;
    if (p->ev_ks > 1) off = align_up(off + (size_t)desc->Cout * ((desc->N + 15) / 16) * 4, 256);
    p->ws_total = off;
    *out = p;
    return CONVT3D_OK;
}

void convt3d_plan_destroy(convt3d_plan_t p) {
    if (!p) return;
    if (p->tc_cache) tc_cache_free(p->tc_cache);
    if (p->direct_cache) direct_cache_free(p->direct_cache);
    if (p->ev_created) {
        cudaEventDestroy(p->ev0);
        cudaEventDestroy(p->ev1);
    }
    delete p;
}

convt3d_status_t convt3d_output_shape(convt3d_plan_t p, int64_t shape[5]) {
    if (!p || !shape) return fail(CONVT3D_ERR_INVALID_ARG, "NULL argument");
    const bool pooled = p->d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL ||
                        p->d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL;
    shape[0] = p->d.N;
    shape[1] = p->d.Cout;
    shape[2] = pooled ? 1 : p->g.Do;
    shape[3] = pooled ? 1 : p->g.Ho;
    shape[4] = pooled ? 1 : p->g.Wo;
    return CONVT3D_OK;
}

size_t convt3d_workspace_bytes(convt3d_plan_t p) { return p ? p->ws_total : 0; }

convt3d_status_t convt3d_plan_info(convt3d_plan_t p, convt3d_info_t *info) {
    if (!p || !info) return fail(CONVT3D_ERR_INVALID_ARG, "NULL argument");
    memset(info, 0, sizeof(*info));
    convt3d_output_shape(p, info->out_shape);
    const convt3d_desc_t &d = p->d;
    const Geometry &g = p->g;
    info->num_classes = g.nclasses;
    info->gemm_m = (int64_t)d.N * g.Do * g.Ho * g.Wo;
    info->gemm_n = d.Cout;
    int64_t ktot = 0;
    for (int c = 0; c < g.nclasses; ++c) ktot += (int64_t)d.Cin * g.cls[c].ntaps;
    info->gemm_k_total = ktot;
    info->tiles = p->tiles;
    info->main_kernel = p->direct ? 2 : (p->tc ? 0 : 1);
    info->tile_m = p->tile_m;
    const bool gn = d.epilogue == CONVT3D_EPI_RELU_GROUPNORM;
    const bool bn = d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL;
    const bool ev = d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL;
    info->launches_per_forward = ev ? 2 : (p->tc && !p->direct ? 2 : 1) + (gn ? 2 : 0) + (bn ? 2 : 0);
    info->launches_per_pack = 1;
    info->useful_flop = 2.0 * d.N * d.Cout * (double)(d.Cin / g.G) * g.kvol * d.Din * d.Hin * d.Win;
    // Issued: every tile runs its class(es)' taps over tile_m rows and cout_pad columns -- the
    // tensor-core path only the taps live for the tile, with three products per term.
    double issued = 0;
    for (int i = 0; i < p->ngroups; ++i) {
        const GroupDesc &G = p->grp[i];
        double taps = 0;
        for (int t = 0; t < G.tiles; ++t) {
            for (int c = 0; c < G.ncls; ++c) {
                const ClassDesc &C = g.cls[G.cls[c]];
                if (p->tc) {
                    const TapRange r = tile_taps(G, C, t, p->tile_m, g.Din);
                    taps += r.end - r.begin;
                } else {
                    taps += C.ntaps;
                }
            }
        }
        issued += 2.0 * (double)d.N * p->tile_m * p->cout_pad * (double)p->cin_pad * taps;
    }
    info->issued_mma_flop = issued * (p->planes == 2 ? 3.0 : 1.0);
    const double eb = p->io16 != kF32 ? 2.0 : 4.0;  // bytes per element of x, w and y at the boundary
    const double xbytes = eb * d.N * d.Cin * (double)d.Din * d.Hin * d.Win;
    const double wbytes = eb * d.Cin * (d.Cout / g.G) * (double)g.kvol;
    const double ybytes = eb * d.N * d.Cout * (double)g.Do * g.Ho * g.Wo;
    const double out_bytes = (bn || ev) ? eb * d.N * d.Cout : ybytes;
    // Main kernel: reads x (tensor-core path: the staged hi+lo copy; the direct kernel: x itself) and the packed weights once,
    // writes the output once (BN+pool: nothing but partials).
    const double planes = (p->planes == 2 ? 2.0 : 1.0) * p->elem_bytes / eb;  // staged operand bytes / boundary bytes
    info->gemm_min_bytes = (p->direct ? xbytes : planes * xbytes) + planes * wbytes + (bn ? 0.0 : ybytes);
    // Whole forward as the pages define it: x and w in, the output out, plus the second pass
    // over y that GroupNorm's global statistics force.
    info->forward_min_bytes = xbytes + wbytes + out_bytes + (gn ? 2.0 * ybytes : 0.0);
    if (ev) {  // no convolution runs: box sums over x, then a contraction with w
        info->issued_mma_flop = 2.0 * d.N * d.Cout * (double)d.Cin * g.kvol;
        info->gemm_min_bytes = xbytes;
    }
    return CONVT3D_OK;
}

static convt3d_status_t check_ws(convt3d_plan_t p, void *ws, size_t bytes) {
    if (!ws) return fail(CONVT3D_ERR_WORKSPACE, "workspace is NULL");
    if (bytes < p->ws_total)
        return fail(CONVT3D_ERR_WORKSPACE, "workspace %zu bytes < required %zu", bytes, p->ws_total);
    if ((uintptr_t)ws % 256) return fail(CONVT3D_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    return CONVT3D_OK;
}

convt3d_status_t convt3d_pack_weights(convt3d_plan_t p, const void *wv, void *ws, size_t ws_bytes,
                                      void *stream) {
    g_last_error[0] = 0;
    const float *w = static_cast<const float *>(wv);  // 16-bit data when io_bf16 / io_fp16: the kernels reinterpret it
    if (!p || !w) return fail(CONVT3D_ERR_INVALID_ARG, "NULL plan or weight");
    if ((uintptr_t)w % 16) return fail(CONVT3D_ERR_INVALID_ARG, "w must be 16-byte aligned");
    convt3d_status_t st = check_ws(p, ws, ws_bytes);
    if (st) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char *base = (char *)ws;
    cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing status word");
    if (p->ev_ks > 1) {  // the split contraction's arrival counters start at zero (each forward resets them)
        e = cudaMemsetAsync(base + p->off_evcnt, 0, p->ws_total - p->off_evcnt, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing arrival counters");
    }
    e = p->direct ? launch_direct_pack(*p, w, base + p->off_wpk_hi, s)
                  : launch_pack_weights(*p, w, (float *)(base + p->off_wpk_hi),
                                        p->planes == 2 ? (float *)(base + p->off_wpk_lo) : nullptr, p->tc, s);
    if (e != cudaSuccess) return cuda_fail(e, "pack_weights launch");
    p->packed_ws = ws;
    return CONVT3D_OK;
}

}  // extern "C"

namespace {

// Argument checks shared by the forward entry points; `affine`: gamma and beta are read.
convt3d_status_t forward_checks(convt3d_plan_t p, const void *x, const float *bias, const float *gamma,
                                const float *beta, const void *y, void *ws, size_t ws_bytes, bool affine) {
    if (!p || !y) return fail(CONVT3D_ERR_INVALID_ARG, "NULL plan or y");
    const convt3d_desc_t &d = p->d;
    if (d.has_bias && !bias) return fail(CONVT3D_ERR_INVALID_ARG, "has_bias set but bias is NULL");
    const bool norm = d.epilogue == CONVT3D_EPI_RELU_GROUPNORM || d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL ||
                      d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL;
    if (affine && norm && (!gamma || !beta)) return fail(CONVT3D_ERR_INVALID_ARG, "gamma and beta are required");
    for (const void *ptr : {x, y, (const void *)bias, (const void *)gamma, (const void *)beta})
        if ((uintptr_t)ptr % 16) return fail(CONVT3D_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
    if (x && x == y) return fail(CONVT3D_ERR_INVALID_ARG, "y must not alias x");
    convt3d_status_t st = check_ws(p, ws, ws_bytes);
    if (st) return st;
    if (p->packed_ws != ws) return fail(CONVT3D_ERR_NOT_PACKED, "call convt3d_pack_weights on this workspace first");
    return CONVT3D_OK;
}

// The per-sample part of the forward for samples [n0, n1): input staging and the main
// kernel with its fused epilogue (statistics partials land in per-tile slots).
convt3d_status_t forward_main(convt3d_plan_t p, const float *x, const float *b, float *y, char *base, int n0, int n1,
                              cudaStream_t s) {
    cudaError_t e;
    double *partials = (double *)(base + p->off_partials);
    if (p->prof_enabled) {
        if (!p->ev_created) {
            if ((e = cudaEventCreate(&p->ev0)) != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
            if ((e = cudaEventCreate(&p->ev1)) != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
            p->ev_created = 1;
        }
    }
    if (p->direct) {
        if (p->prof_enabled && (e = cudaEventRecord(p->ev0, s)) != cudaSuccess) return cuda_fail(e, "event");
        e = launch_direct(*p, x, base + p->off_wpk_hi, b, y, (uint32_t *)base, s);
        if (e != cudaSuccess) return cuda_fail(e, "direct tensor-core GEMM launch");
    } else if (p->tc) {
        const bool two = p->planes == 2;
        float *xs_hi = (float *)(base + p->off_xs_hi), *xs_lo = two ? (float *)(base + p->off_xs_lo) : nullptr;
        e = launch_stage_input(*p, x, xs_hi, xs_lo, n0, n1, s);
        if (e != cudaSuccess) return cuda_fail(e, "stage_input launch");
        if (p->prof_enabled && (e = cudaEventRecord(p->ev0, s)) != cudaSuccess) return cuda_fail(e, "event");
        e = launch_tc(*p, xs_hi, xs_lo, (const float *)(base + p->off_wpk_hi),
                      two ? (const float *)(base + p->off_wpk_lo) : nullptr, b, y, partials, (uint32_t *)base, n0, n1,
                      s);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core GEMM launch");
    } else {
        if (p->prof_enabled && (e = cudaEventRecord(p->ev0, s)) != cudaSuccess) return cuda_fail(e, "event");
        e = launch_ffma(*p, x, (const float *)(base + p->off_wpk_hi), b, y, partials, n0, n1, s);
        if (e != cudaSuccess) return cuda_fail(e, "FFMA GEMM launch");
    }
    if (p->prof_enabled) {
        if ((e = cudaEventRecord(p->ev1, s)) != cudaSuccess) return cuda_fail(e, "event");
        p->prof_valid = 1;
    }
    return CONVT3D_OK;
}

// The passes over the whole batch: GroupNorm's statistics and normalise pass, BatchNorm's
// statistics, pooled output and running statistics (nothing for the other epilogues).
convt3d_status_t forward_post(convt3d_plan_t p, const float *b, const float *gamma, const float *beta, float *y,
                              char *base, cudaStream_t s) {
    cudaError_t e;
    double *partials = (double *)(base + p->off_partials);
    double *stats = (double *)(base + p->off_stats);
    if (p->d.epilogue == CONVT3D_EPI_RELU_GROUPNORM) {
        e = launch_gn_finalize(*p, partials, stats, s);
        if (e != cudaSuccess) return cuda_fail(e, "groupnorm finalize launch");
        e = launch_gn_normalize(*p, stats, gamma, beta, b, y, s);
        if (e != cudaSuccess) return cuda_fail(e, "groupnorm normalize launch");
    } else if (p->d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL) {
        e = launch_bn_finalize(*p, partials, stats, gamma, beta, y, s);
        if (e != cudaSuccess) return cuda_fail(e, "batchnorm finalize launch");
    }
    return CONVT3D_OK;
}

}  // namespace

extern "C" {

convt3d_status_t convt3d_forward(convt3d_plan_t p, const void *xv, const float *bias, const float *gamma,
                                 const float *beta, void *yv, void *ws, size_t ws_bytes, void *stream) {
    g_last_error[0] = 0;
    // 16-bit data when io_bf16 / io_fp16: the kernels reinterpret these pointers
    const float *x = static_cast<const float *>(xv);
    float *y = static_cast<float *>(yv);
    if (!p || !x) return fail(CONVT3D_ERR_INVALID_ARG, "NULL plan or x");
    const convt3d_desc_t &d = p->d;
    if (d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL && (!p->run_mean || !p->run_var))
        return fail(CONVT3D_ERR_INVALID_ARG, "evaluation-mode BatchNorm needs convt3d_set_running_stats");
    convt3d_status_t st = forward_checks(p, x, bias, gamma, beta, y, ws, ws_bytes, true);
    if (st) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char *base = (char *)ws;
    const float *b = d.has_bias ? bias : nullptr;
    if (d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL) {
        // no convolution: input box sums and a contraction with the packed weight
        cudaError_t e = launch_bn_eval(*p, x, (const float *)(base + p->off_wpk_hi),
                                       p->planes == 2 ? (const float *)(base + p->off_wpk_lo) : nullptr, b, gamma, beta,
                                       (float *)(base + p->off_box), (double *)(base + p->off_evpart),
                                       (unsigned *)(base + p->off_evcnt), y, s);
        if (e != cudaSuccess) return cuda_fail(e, "evaluation-mode batchnorm launch");
        return CONVT3D_OK;
    }
    st = forward_main(p, x, b, y, base, 0, d.N, s);
    if (st) return st;
    return forward_post(p, b, gamma, beta, y, base, s);
}

convt3d_status_t convt3d_forward_samples(convt3d_plan_t p, const void *xv, const float *bias, void *yv, void *ws,
                                         size_t ws_bytes, int n0, int n1, void *stream) {
    g_last_error[0] = 0;
    const float *x = static_cast<const float *>(xv);
    float *y = static_cast<float *>(yv);
    if (!p || !x) return fail(CONVT3D_ERR_INVALID_ARG, "NULL plan or x");
    if (n0 < 0 || n1 > p->d.N || n0 >= n1) return fail(CONVT3D_ERR_INVALID_ARG, "need 0 <= n0 < n1 <= N");
    if (p->d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL)
        return fail(CONVT3D_ERR_UNSUPPORTED, "evaluation-mode BatchNorm runs as one convt3d_forward");
    if (p->direct && (n0 != 0 || n1 != p->d.N))
        return fail(CONVT3D_ERR_UNSUPPORTED, "this plan's main kernel (main_kernel 2) runs the whole batch at once");
    convt3d_status_t st = forward_checks(p, x, bias, nullptr, nullptr, y, ws, ws_bytes, false);
    if (st) return st;
    return forward_main(p, x, p->d.has_bias ? bias : nullptr, y, (char *)ws, n0, n1, (cudaStream_t)stream);
}

convt3d_status_t convt3d_forward_finish(convt3d_plan_t p, const float *bias, const float *gamma, const float *beta,
                                        void *yv, void *ws, size_t ws_bytes, void *stream) {
    g_last_error[0] = 0;
    float *y = static_cast<float *>(yv);
    if (p && p->d.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL)
        return fail(CONVT3D_ERR_UNSUPPORTED, "evaluation-mode BatchNorm runs as one convt3d_forward");
    convt3d_status_t st = forward_checks(p, nullptr, bias, gamma, beta, y, ws, ws_bytes, true);
    if (st) return st;
    return forward_post(p, p->d.has_bias ? bias : nullptr, gamma, beta, y, (char *)ws, (cudaStream_t)stream);
}

convt3d_status_t convt3d_check(convt3d_plan_t p, void *ws, void *stream) {
    if (!p) return fail(CONVT3D_ERR_INVALID_ARG, "NULL plan");
    if (!ws) {  // the built-in workspace of convt3d_forward_static_workspace on the current device
        ws = static_workspace_address();
        if (!ws) return CONVT3D_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t word[4] = {0, 0, 0, 0};
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    e = cudaMemcpy(word, ws, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading status word");
    if (word[0] == kErrNone) return CONVT3D_OK;
    e = cudaMemset(ws, 0, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e, "clearing status word");
    if (word[0] == kErrTimeout)
        return fail(CONVT3D_ERR_TIMEOUT, "device wait timed out (site %u, block %u)", word[1], word[2]);
    return fail(CONVT3D_ERR_DEVICE_ASSERT, "device check failed (code %u, site %u)", word[0], word[1]);
}

convt3d_status_t convt3d_set_running_stats(convt3d_plan_t p, float *running_mean, float *running_var,
                                           float momentum) {
    if (!p) return fail(CONVT3D_ERR_INVALID_ARG, "NULL plan");
    if ((running_mean == nullptr) != (running_var == nullptr))
        return fail(CONVT3D_ERR_INVALID_ARG, "running_mean and running_var are set together");
    if (!(momentum >= 0.0f && momentum <= 1.0f)) return fail(CONVT3D_ERR_INVALID_ARG, "momentum must be in [0, 1]");
    if (((uintptr_t)running_mean | (uintptr_t)running_var) % 4)
        return fail(CONVT3D_ERR_INVALID_ARG, "running statistics must be 4-byte aligned");
    p->run_mean = running_mean;
    p->run_var = running_var;
    p->momentum = momentum;
    return CONVT3D_OK;
}

convt3d_status_t convt3d_profile_enable(convt3d_plan_t p, int enable) {
    if (!p) return fail(CONVT3D_ERR_INVALID_ARG, "NULL plan");
    p->prof_enabled = enable ? 1 : 0;
    p->prof_valid = 0;
    return CONVT3D_OK;
}

convt3d_status_t convt3d_profile_read(convt3d_plan_t p, float *ms) {
    if (!p || !ms) return fail(CONVT3D_ERR_INVALID_ARG, "NULL argument");
    if (!p->prof_valid) return fail(CONVT3D_ERR_INVALID_ARG, "no profiled forward yet");
    cudaError_t e = cudaEventSynchronize(p->ev1);
    if (e != cudaSuccess) return cuda_fail(e, "event synchronize");
    e = cudaEventElapsedTime(ms, p->ev0, p->ev1);
    if (e != cudaSuccess) return cuda_fail(e, "event elapsed time");
    return CONVT3D_OK;
}

}  // extern "C"
