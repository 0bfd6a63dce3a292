// Conv2D forward / preceding-layer gradient / weight gradient as implicit GEMMs
// over NHWC activations and RSCK filters (ApproxTrain Sec. VI-B, Algorithms 3
// and 4, Fig. 8).  The page's IM2COL, IM2COL_PLG, IM2COL_Weight and
// TransposeAndReverse kernels become operand addressing inside the LUT-GEMM:
// no column buffer is materialised.
#include <algorithm>

#include "gemm_kernel.cuh"

namespace {

using amsim::OperandDesc;
using amsim::Problem;

struct Geo {
    int N, H, W, C, K, R, S, sh, sw, ph, pw, dh, dw, P, Q;
};

int geometry(const amsim_conv_desc *d, Geo *g)
{
    if (!d) return AMSIM_EINVAL;
    *g = {d->N, d->H, d->W, d->C, d->K, d->R, d->S, d->stride_h, d->stride_w, d->pad_h, d->pad_w,
          d->dil_h, d->dil_w, 0, 0};
    if (g->N < 0 || g->H < 1 || g->W < 1 || g->C < 1 || g->K < 1 || g->R < 1 || g->S < 1) return AMSIM_EINVAL;
    if (g->sh < 1 || g->sw < 1 || g->ph < 0 || g->pw < 0 || g->dh < 1 || g->dw < 1) return AMSIM_EINVAL;
    const long long hh = (long long)g->H + 2LL * g->ph - (long long)g->dh * (g->R - 1) - 1;
    const long long ww = (long long)g->W + 2LL * g->pw - (long long)g->dw * (g->S - 1) - 1;
    if (hh < 0 || ww < 0) return AMSIM_EINVAL;
    g->P = (int)(hh / g->sh + 1);
    g->Q = (int)(ww / g->sw + 1);
    // index arithmetic inside the kernels is 32-bit per coordinate, 64-bit per address
    const long long px = (long long)g->N * std::max(g->H * (long long)g->W, (long long)g->P * g->Q);
    if (px > 0x7FFFFFFFLL || (long long)g->R * g->S * std::max(g->C, g->K) > 0x7FFFFFFFLL) return AMSIM_EUNSUPPORTED;
    return AMSIM_OK;
}

OperandDesc blank(const float *ptr, int rows)
{
    OperandDesc d = {};
    d.ptr = ptr;
    d.rows = rows;
    d.kD0 = d.kD1 = d.rE0 = d.rE1 = 1;
    d.IH = d.IW = 1;
    d.sy = d.sx = 1;
    return d;
}

OperandDesc dense(const float *ptr, int rows, long long s_row, long long s_k)
{
    OperandDesc d = blank(ptr, rows);
    d.s_row = s_row;
    d.s_k = s_k;
    return d;
}

// x viewed as the im2col matrix of the forward pass: row = output pixel
// (n,p,q), k = (r,s,c); value x[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c].
OperandDesc x_im2col(const Geo &g, const float *x)
{
    OperandDesc d = blank(x, g.N * g.P * g.Q);
    d.gather = 1;
    d.rE0 = g.Q; d.rE1 = g.P;
    d.rcx[0] = g.sw; d.rcy[1] = g.sh; d.rcb[2] = (long long)g.H * g.W * g.C;
    d.ry0 = -g.ph; d.rx0 = -g.pw;
    d.kD0 = g.C; d.kD1 = g.S;
    d.kcb[0] = 1; d.kcx[1] = g.dw; d.kcy[2] = g.dh;
    d.IH = g.H; d.IW = g.W; d.Cs = g.C;
    d.extent = (long long)g.N * g.H * g.W * g.C;
    return d;
}

// x viewed for the weight gradient: row = (r,s,c), k = (n,p,q).
OperandDesc x_im2col_weight(const Geo &g, const float *x)
{
    OperandDesc d = blank(x, g.R * g.S * g.C);
    d.gather = 1;
    d.rE0 = g.C; d.rE1 = g.S;
    d.rcb[0] = 1; d.rcx[1] = g.dw; d.rcy[2] = g.dh;
    d.ry0 = -g.ph; d.rx0 = -g.pw;
    d.kD0 = g.Q; d.kD1 = g.P;
    d.kcx[0] = g.sw; d.kcy[1] = g.sh; d.kcb[2] = (long long)g.H * g.W * g.C;
    d.IH = g.H; d.IW = g.W; d.Cs = g.C;
    d.extent = (long long)g.N * g.H * g.W * g.C;
    return d;
}

// dy viewed as the padded-dilated error columns of the preceding-layer
// gradient: row = input pixel (n,h,w), k = (r,s,k); value dy[n,p,q,k] with
// p = (h + ph - r*dh)/sh, q = (w + pw - s*dw)/sw when integral and in range.
OperandDesc dy_im2col_plg(const Geo &g, const float *dy)
{
    OperandDesc d = blank(dy, g.N * g.H * g.W);
    d.gather = 1;
    d.rE0 = g.W; d.rE1 = g.H;
    d.rcx[0] = 1; d.rcy[1] = 1; d.rcb[2] = (long long)g.P * g.Q * g.K;
    d.ry0 = g.ph; d.rx0 = g.pw;
    d.kD0 = g.K; d.kD1 = g.S;
    d.kcb[0] = 1; d.kcx[1] = -g.dw; d.kcy[2] = -g.dh;
    d.IH = g.P; d.IW = g.Q; d.Cs = g.K;
    d.sy = g.sh; d.sx = g.sw;
    d.extent = (long long)g.N * g.P * g.Q * g.K;
    return d;
}

// Filter transposed (in/out channels swapped) for the preceding-layer
// gradient: row = c, k = (r,s,k); value w[r,s,c,k].  The spatial reversal of
// TransposeAndReverse is carried by the dy addressing above.
OperandDesc w_transposed(const Geo &g, const float *w)
{
    OperandDesc d = blank(w, g.C);
    d.gather = 1;
    d.rE0 = g.C; d.rE1 = 1;
    d.rcb[0] = g.K;
    d.kD0 = g.K; d.kD1 = g.S;
    d.kcb[0] = 1; d.kcb[1] = (long long)g.C * g.K; d.kcb[2] = (long long)g.S * g.C * g.K;
    d.IH = 1; d.IW = 1; d.Cs = 0;
    d.extent = (long long)g.R * g.S * g.C * g.K;
    return d;
}

// ------------------------------------------------------------------ tensor boxes
// With unit strides the raw-tile kernel reads a convolution's operands in
// place: for filter tap (r, s) the im2col rows of whole output rows are one
// box of the NHWC activation whose start row and column are the tap's
// offsets (out-of-range pixels arrive as zeros), and the weight gradient's
// rows are 64-channel runs of the activation at each tap's input position.

amsim::TmaRawMap raw_map(const float *base, int rank, const uint64_t *dims, const uint32_t *box, int swizzle64)
{
    amsim::TmaRawMap m = {};
    m.base = base;
    m.rank = rank;
    uint64_t stride = 4;
    for (int i = 0; i < rank; ++i) {
        m.dims[i] = dims[i];
        m.box[i] = box[i];
        stride *= dims[i];
        if (i + 1 < rank) m.strides[i] = stride;
    }
    m.swizzle64 = swizzle64;
    return m;
}

// Fills *cv and returns true when pass `which` of geometry g can use tensor boxes.
bool conv_raw(const Geo &g, int which, const float *t0, const float *t1, amsim::ConvRaw *cv)
{
    using amsim::kern::BK;
    using amsim::kern::BL;
    using amsim::kern::BU;
    if (g.sh != 1 || g.sw != 1) return false;
    *cv = {};
    cv->S = g.S;
    if (which == 0) {
        // y[n,p,q,k] = sum x[n, p - ph + r dh, q - pw + s dw, c] w[r,s,c,k]
        if (g.C % 16 || BL % g.Q || g.P % (BL / g.Q)) return false;
        cv->mode = 1;
        const uint64_t ud[3] = {(uint64_t)g.K, (uint64_t)g.R * g.S * g.C, 1};
        const uint32_t ub[3] = {(uint32_t)BU, (uint32_t)BK, 1};
        cv->umap = raw_map(t1, 3, ud, ub, 0);                  // w[(r,s,c)][k]: rows k innermost
        const uint64_t ld[4] = {(uint64_t)g.C, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.N};
        const uint32_t lb[4] = {(uint32_t)BK, (uint32_t)g.Q, (uint32_t)(BL / g.Q), 1};
        cv->lmap = raw_map(t0, 4, ld, lb, 1);                  // x NHWC, [row][channel] boxes
        cv->ch = g.C;
        cv->rows_tile = BL / g.Q;
        cv->tiles_img = g.P / cv->rows_tile;
        cv->ybase = -g.ph;
        cv->ystep = g.dh;
        cv->xbase = -g.pw;
        cv->xstep = g.dw;
    } else if (which == 1) {
        // dx[n,h,w,c] = sum dy[n, h + ph - r dh, w + pw - s dw, k] w[r,s,c,k]
        if (g.K % 16 || BL % g.W || g.H % (BL / g.W)) return false;
        cv->mode = 1;
        // the filter with its channel axes swapped: rows c, steps (r, s, k) -> boxes of
        // 16 k by 64 c of one tap, [c][k]
        const uint64_t ud[3] = {(uint64_t)g.K, (uint64_t)g.C, (uint64_t)g.R * g.S};
        const uint32_t ub[3] = {(uint32_t)BK, (uint32_t)BU, 1};
        cv->umap = raw_map(t1, 3, ud, ub, 1);
        cv->u_kfast = 1;
        cv->u_tap = 1;
        const uint64_t ld[4] = {(uint64_t)g.K, (uint64_t)g.Q, (uint64_t)g.P, (uint64_t)g.N};
        const uint32_t lb[4] = {(uint32_t)BK, (uint32_t)g.W, (uint32_t)(BL / g.W), 1};
        cv->lmap = raw_map(t0, 4, ld, lb, 1);                  // dy NHWC
        cv->ch = g.K;
        cv->rows_tile = BL / g.W;
        cv->tiles_img = g.H / cv->rows_tile;
        cv->ybase = g.ph;
        cv->ystep = -g.dh;
        cv->xbase = g.pw;
        cv->xstep = -g.dw;
    } else {
        // dw[r,s,c,k] = sum over (n,p,q) of x[n, p - ph + r dh, q - pw + s dw, c] dy[n,p,q,k]
        if (g.C % 64 || g.Q % 16) return false;
        cv->mode = 2;
        const uint64_t ud[3] = {(uint64_t)g.K, (uint64_t)g.N * g.P * g.Q, 1};
        const uint32_t ub[3] = {(uint32_t)BU, (uint32_t)BK, 1};
        cv->umap = raw_map(t1, 3, ud, ub, 0);                  // dy[(n,p,q)][k]: rows k innermost
        const uint64_t ld[4] = {(uint64_t)g.C, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.N};
        const uint32_t lb[4] = {64, (uint32_t)BK, 1, 1};
        cv->lmap = raw_map(t0, 4, ld, lb, 0);                  // x NHWC, [pixel][channel] = [k][row]
        cv->ch = g.C;
        cv->N = g.N;
        cv->P = g.P;
        cv->Q = g.Q;
        cv->rows = g.R * g.S * g.C;
        cv->ybase = -g.ph;
        cv->ystep = g.dh;
        cv->xbase = -g.pw;
        cv->xstep = g.dw;
    }
    return true;
}

void set_out(Problem *pr, float *out, long long c_su, long long c_sl)
{
    pr->c_ptr = out;
    pr->c_bs = 0;
    pr->c_su = c_su;
    pr->c_sl = c_sl;
    pr->alpha = 1.0f;
    pr->beta = 0.0f;
    pr->batch = 1;
}

int build(const amsim_conv_desc *desc, int which, const float *t0, const float *t1, float *out, Problem *pr)
{
    Geo g;
    int rc = geometry(desc, &g);
    if (rc) return rc;
    // A 1x1 filter at stride 1 without padding reads every operand as a plain
    // matrix (pixels x channels): dense operands, no gather.
    const bool pointwise = g.R == 1 && g.S == 1 && g.sh == 1 && g.sw == 1 && g.ph == 0 && g.pw == 0;
    if (pointwise) {
        const int pix = g.N * g.H * g.W;
        if (which == 0) {
            pr->U = dense(t1, g.K, 1, g.K);              // w[c][k]: row k, index c
            pr->L = dense(t0, pix, g.C, 1);              // x[pixel][c]
            pr->K = g.C;
            set_out(pr, out, 1, g.K);
        } else if (which == 1) {
            pr->U = dense(t1, g.C, g.K, 1);              // w[c][k]: row c, index k
            pr->L = dense(t0, pix, g.K, 1);              // dy[pixel][k]
            pr->K = g.K;
            set_out(pr, out, 1, g.C);
        } else {
            pr->U = dense(t1, g.K, 1, g.K);              // dy[pixel][k]: row k, index pixel
            pr->L = dense(t0, g.C, 1, g.C);              // x[pixel][c]: row c, index pixel
            pr->K = pix;
            set_out(pr, out, 1, g.K);
        }
        pr->u_is_first = false;
        const long long outs = (long long)pr->U.rows * pr->L.rows;
        if (outs > 0 && (!t0 || !t1 || !out)) return AMSIM_EINVAL;
        return AMSIM_OK;
    }
    if (which == 0) {            // y = conv(x, w): first operand x
        pr->U = dense(t1, g.K, 1, g.K);                  // w[(r,s,c)][k]: row k, index rsc
        pr->L = x_im2col(g, t0);
        pr->K = g.R * g.S * g.C;
        pr->u_is_first = false;
        set_out(pr, out, 1, g.K);                        // y[(n,p,q)][k]
    } else if (which == 1) {     // dx from (dy, w): first operand dy
        pr->U = w_transposed(g, t1);
        pr->L = dy_im2col_plg(g, t0);
        pr->K = g.R * g.S * g.K;
        pr->u_is_first = false;
        set_out(pr, out, 1, g.C);                        // dx[(n,h,w)][c]
    } else {                     // dw from (x, dy): first operand x
        pr->U = dense(t1, g.K, 1, g.K);                  // dy[(n,p,q)][k]: row k, index npq
        pr->L = x_im2col_weight(g, t0);
        pr->K = g.N * g.P * g.Q;
        pr->u_is_first = false;
        set_out(pr, out, 1, g.K);                        // dw[(r,s,c)][k]
    }
    const long long outs = (long long)pr->U.rows * pr->L.rows;
    if (outs > 0 && (!t0 || !t1 || !out)) return AMSIM_EINVAL;
    return AMSIM_OK;
}

int run(const amsim_conv_desc *desc, int which, const float *t0, const float *t1, float *out, amsim_lut_t lut,
        void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    Problem pr;
    rc = build(desc, which, t0, t1, out, &pr);
    if (rc) return rc;
    Geo g;
    geometry(desc, &g);
    amsim::ConvRaw cv;
    if (pr.U.gather || pr.L.gather)
        if (conv_raw(g, which, t0, t1, &cv)) pr.conv = &cv;
    return amsim::run_problem(pr, lut, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int amsim_conv2d_out_hw(const amsim_conv_desc *desc, int *P, int *Q)
{
    Geo g;
    int rc = geometry(desc, &g);
    if (rc) return rc;
    if (P) *P = g.P;
    if (Q) *Q = g.Q;
    return AMSIM_OK;
}

int amsim_conv2d_fwd(const amsim_conv_desc *desc, const float *x, const float *w, float *y, amsim_lut_t lut,
                     void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    return run(desc, 0, x, w, y, lut, ws, ws_bytes, stream);
}

int amsim_conv2d_bwd_data(const amsim_conv_desc *desc, const float *dy, const float *w, float *dx, amsim_lut_t lut,
                          void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    return run(desc, 1, dy, w, dx, lut, ws, ws_bytes, stream);
}

int amsim_conv2d_bwd_filter(const amsim_conv_desc *desc, const float *x, const float *dy, float *dw,
                            amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    return run(desc, 2, x, dy, dw, lut, ws, ws_bytes, stream);
}

size_t amsim_conv2d_workspace_size(const amsim_conv_desc *desc, int which, amsim_lut_t lut)
{
    if (!lut || which < 0 || which > 2) return 0;
    // distinct dummy addresses keep the operands' planes apart
    static const float dummy0 = 0.0f, dummy1 = 0.0f;
    static float dummy_out = 0.0f;
    Problem pr;
    if (build(desc, which, &dummy0, &dummy1, &dummy_out, &pr)) return 0;
    Geo g;
    geometry(desc, &g);
    amsim::ConvRaw cv;
    if (pr.U.gather || pr.L.gather)
        if (conv_raw(g, which, &dummy0, &dummy1, &cv)) pr.conv = &cv;
    return amsim::problem_workspace(pr, lut);
}

}  // extern "C"
