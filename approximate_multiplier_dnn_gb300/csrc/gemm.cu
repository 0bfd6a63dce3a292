// Host planning for the LUT-GEMM kernels (tile counts, split-K, LUT residency,
// operand roles), the deterministic split-K reduction, and the GEMM ABI
// (ApproxTrain Sec. VI-D GEMM kernel; Sec. VI-C AMDENSE forward and gradients).
#include <algorithm>
#include <cmath>
#include <vector>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "gemm_raw.cuh"
#include "predecode.h"

namespace amsim {

namespace {

using kern::BK;
using kern::BL;
using kern::BU;

constexpr int kMaxSmemLut = 160 * 1024;   // LUTs up to this size are staged in shared memory

// Paths taken by the calling thread's current (or last) GEMM / conv call.
thread_local int g_last_path = 0;

// Stream-K flag values: every launch gets a fresh one, so flags left in
// scratch by earlier launches never match.
std::atomic<unsigned long long> g_epoch{0x5EED0001ULL};

// Cooperative launches (amsim_set_cooperative_launches): on, stream-K launches
// finish cut tiles inside the kernel and phased calls run as one launch.
std::atomic<bool> g_coop{true};
bool coop_launches() { return g_coop.load(std::memory_order_relaxed); }

int device_sms(int dev)
{
    static std::atomic<int> cache[64];
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    if (dev >= 0 && dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Launch plan for a group of problems sharing one LUT.
struct Plan {
    int tiles_u[kern::kMaxProblems], tiles_l[kern::kMaxProblems], kt[kern::kMaxProblems];
    long long tiles[kern::kMaxProblems], iter0[kern::kMaxProblems];
    long long total_tiles, iters;
    bool streamk;
    int ctas;
    size_t ws_bytes;   // scratch the chosen plan uses
    size_t sk_bytes;   // scratch stream-K would use
};

// Launch plan for tiles of shape tc (the narrow shape unless given).
Plan make_plan(const Problem *p, int n, int sms, size_t ws_avail, const kern::TileCfg &tc = kern::kNarrowTiles)
{
    Plan pl = {};
    for (int i = 0; i < n; ++i) {
        const bool empty = p[i].U.rows == 0 || p[i].L.rows == 0 || p[i].batch == 0;
        pl.tiles_u[i] = std::max(1, ceil_div(p[i].U.rows, tc.bu));
        pl.tiles_l[i] = std::max(1, ceil_div(p[i].L.rows, tc.bl));
        pl.kt[i] = std::max(1, ceil_div(p[i].K, tc.bk));
        pl.tiles[i] = empty ? 0 : (long long)pl.tiles_u[i] * pl.tiles_l[i] * p[i].batch;
        pl.iter0[i] = pl.iters;
        pl.iters += pl.tiles[i] * pl.kt[i];
        pl.total_tiles += pl.tiles[i];
    }
    pl.ctas = (int)std::min<long long>(std::min(sms, kern::kMaxFixupParts), pl.iters);
    // two partial-sum slots and two flags per CTA
    pl.sk_bytes = (size_t)2 * pl.ctas * tc.bu * tc.bl * sizeof(float) + (size_t)2 * pl.ctas * sizeof(unsigned long long);
    // Stream-K over (tile, stage) iterations with one persistent CTA per SM,
    // unless the tiles fit in one wave that fills the SMs nearly whole (then
    // one CTA per tile).  Persistent CTAs stage the LUT once and keep the
    // copy ring full across tile boundaries, so a tile's epilogue overlaps the
    // next tile's first copies.
    const long long waves = (pl.total_tiles + sms - 1) / std::max(1, sms);
    const double dp_eff = pl.total_tiles > 0 ? (double)pl.total_tiles / (double)(waves * sms) : 1.0;
    pl.streamk = pl.ctas > 1 && (dp_eff < 0.9 || waves > 1) && pl.sk_bytes <= ws_avail;
    pl.ws_bytes = pl.streamk ? pl.sk_bytes : 0;
    return pl;
}

bool streamk_bounds_by_cost(const Problem *p, int n, const Plan &pl, kern::KParams &kp);

int launch_ws(int width, const kern::KParams &kp, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    switch (width) {
    case 8: return kern::launch_ws_w8(kp, gl, grid, smem, st);
    case 16: return kern::launch_ws_w16(kp, gl, grid, smem, st);
    default: return kern::launch_ws_w32(kp, gl, grid, smem, st);
    }
}

int launch_w(int width, const kern::KParams &kp, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    switch (width) {
    case 8: return kern::launch_w8(kp, gl, grid, smem, st);
    case 16: return kern::launch_w16(kp, gl, grid, smem, st);
    default: return kern::launch_w32(kp, gl, grid, smem, st);
    }
}

// ------------------------------------------------------------------ predecoded operands
// Every dense operand of a launch becomes a plane pair [batch][2][K][rows_pad]
// in scratch, after the stream-K region and a block of per-plane flags.

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encode_tiled()
{
    static std::once_flag once;
    static EncodeTiled fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
        cudaGetLastError();
    });
    return fn;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// two 8-byte flags per plane: "an element with |x| >= 2^64" at [j], "an
// element with 0 < |x| < 2^-63" at [kMaxDecodeJobs + j] (the block keeps its
// 512 bytes, part of the scratch size callers have been told)
constexpr size_t kFlagBlock = 512;
static_assert(kern::kMaxDecodeJobs * 16 <= (int)kFlagBlock, "plane flags fit the block");

struct PlaneKey {
    const float *src;
    long long bs, s_row, s_k;
    int rows, K, nb, offshift;
    bool operator==(const PlaneKey &o) const
    {
        return src == o.src && bs == o.bs && s_row == o.s_row && s_k == o.s_k && rows == o.rows && K == o.K &&
               nb == o.nb && offshift == o.offshift;
    }
};

PlaneKey plane_key(const OperandDesc &d, int K, int batch, int offshift)
{
    const int nb = (d.batch_stride == 0 || batch <= 1) ? 1 : batch;
    return PlaneKey{d.ptr, nb > 1 ? (long long)d.batch_stride : 0LL, d.s_row, d.s_k, d.rows, K, nb, offshift};
}

int rows_pad(int rows) { return (rows + 3) & ~3; }

// `planes` words per element: one packed word, or an offset and a scale.
size_t plane_bytes(const PlaneKey &k, int planes)
{
    return align256((size_t)k.nb * planes * k.K * rows_pad(k.rows) * 4);
}

// Distinct planes of problems [0, n) (operand order U0, L0, U1, L1, ...):
// slot[2i] / slot[2i+1] give the plane index of problem i's U / L operand.
struct PlaneSet {
    PlaneKey key[kern::kMaxDecodeJobs];
    size_t off[kern::kMaxDecodeJobs];    // from the start of the plane region
    int n;
    int nplanes[kern::kMaxDecodeJobs];   // 1: packed words, 2: offset and scale planes
    bool uniform[kern::kMaxDecodeJobs];  // the plane of a U operand (its zeros take the table's zero row)
    int slot[2 * kern::kMaxProblems];
    size_t bytes;
    double elems;    // operand elements decoded (padded rows), for the path decision
};

// False when some problem cannot take the predecoded path (gather operand,
// empty reduction).  planes: U operands' plane count + 4 x L operands'.
bool plan_planes(const Problem *p, int n, const Plan &pl, int M, int wlog, int planes, PlaneSet *ps)
{
    ps->n = 0;
    ps->bytes = 0;
    ps->elems = 0.0;
    for (int i = 0; i < n; ++i) {
        if (pl.tiles[i] == 0) continue;
        if (p[i].U.gather || p[i].L.gather || p[i].K <= 0) return false;
        for (int r = 0; r < 2; ++r) {
            const OperandDesc &d = r == 0 ? p[i].U : p[i].L;
            const PlaneKey k = plane_key(d, p[i].K, p[i].batch, r == 0 ? M + wlog : wlog);
            int j = 0;
            while (j < ps->n && !(ps->key[j] == k)) ++j;
            if (j == ps->n) {
                ps->key[j] = k;
                ps->off[j] = ps->bytes;
                // (U and L planes never coincide: their offset shifts differ)
                ps->nplanes[j] = r == 0 ? (planes & 3) : (planes >> 2);
                ps->uniform[j] = r == 0;
                ps->bytes += plane_bytes(k, ps->nplanes[j]);
                ps->elems += (double)k.nb * k.K * rows_pad(k.rows);
                ++ps->n;
            }
            ps->slot[2 * i + r] = j;
        }
    }
    return true;
}

// The planes pay for their extra memory traffic (written once, read at least
// once) when operand elements are reused by several tiles; a large operand
// read by a single tile row (attention's P in O = P V) is decoded as cheaply
// inside the GEMM.  Measured on GB300 with two-plane (8-byte) elements: 0.03
// plane bytes per MAC gains, 0.13 loses.  Below 64 MB of planes the pass
// costs microseconds either way.  The measure stays 8 bytes per decoded
// element, whatever the planes' layout, so the thresholds keep their meaning.
double launch_macs(const Problem *p, int n, const Plan &pl)
{
    double macs = 0.0;
    for (int i = 0; i < n; ++i)
        if (pl.tiles[i] > 0) macs += (double)p[i].U.rows * p[i].L.rows * (double)p[i].K * p[i].batch;
    return macs;
}

double planes_bytes_per_mac(const Problem *p, int n, const Plan &pl, const PlaneSet &ps)
{
    const double macs = launch_macs(p, n, pl);
    return macs > 0.0 ? 8.0 * ps.elems / macs : 1e30;
}

// Planes rather than raw tiles, for operands the raw-tile kernel could read
// in place.  Measured on GB300 (plane kernel with wide tiles and packed
// words, raw-tile kernel with 64 x 256 tiles), in plane bytes per MAC:
//  * 2048^3 (0.008): planes; 1024^3 (0.016): planes 4 % faster;
//  * batched 512 x 512 x 64 attention scores and a 1x1 conv's 200704 x 256 x
//    256 GEMM (0.031): planes 7 % faster;
//  * 256 x 256 x 16384 and 65536 x 128 x 512 (0.063): raw 2-6 % faster;
//  * an MLP layer's GEMMs (200 M MACs or fewer, 0.018 - 0.05) and 512^3: raw
//    9 - 20 % faster -- the predecode launch is not paid back.
bool planes_beat_raw(const Problem *p, int n, const Plan &pl, const PlaneSet &ps)
{
    const double bpm = planes_bytes_per_mac(p, n, pl, ps);
    return bpm < 0.01 || (bpm < 0.04 && launch_macs(p, n, pl) >= 1073741824.0);
}

bool planes_pay(const Problem *p, int n, const Plan &pl, const PlaneSet &ps)
{
    if (8.0 * ps.elems <= (double)((size_t)64 << 20)) return true;
    return planes_bytes_per_mac(p, n, pl, ps) <= 0.05;
}

// Every box dimension of a tiled tensor map must lie in [1, 256].  A launch
// built with a 512-row box was not refused by the encoder and its copies
// faulted the GPU (illegal address), so maps are checked here first.
bool boxes_ok(const cuuint32_t *box, int rank)
{
    for (int i = 0; i < rank; ++i)
        if (box[i] < 1 || box[i] > 256) return false;
    return true;
}

// Ring depth of the TMA kernel with tiles of shape tc beside a LUT region of
// lut_bytes (0 if none fits).
int tma_stages(size_t lut_bytes, const kern::TileCfg &tc, int planes)
{
    const long long room = (long long)kMaxSmemPerCta - kern::tma_cfg_smem_bytes(tc, planes, (int)lut_bytes, 0);
    long long s = room / kern::tma_stage_bytes(tc, planes);
    if (s > kern::kTmaMaxStages) s = kern::kTmaMaxStages;
    return s >= kern::tma_min_stages(tc, planes) ? (int)s : 0;
}

// Tile shape, LUT placement and plane layout of the predecoded (TMA) kernel:
// the wide shape with the table in shared memory when a ring of its minimum
// depth fits beside it, else the narrow shape with the table in shared
// memory, else the wide shape reading the table from global memory.  With
// the table in shared memory the planes hold packed operand words (offsets
// below 2^18); from global memory, whose offsets reach 2^23, two planes.
// Measured on GB300 (4096^3, Mitchell, two planes): M = 7 runs 6.5 % faster
// and M = 9 25 % faster on wide tiles; at M = 8 (a 128 KB table) the wide
// ring does not fit, and the narrow kernel beats the wide kernel reading the
// table from global memory.
struct TmaChoice {
    kern::TileCfg tc;
    bool wide, gl;
    int planes;    // U operands' planes + 4 x L operands' (1: packed words, 2: offset and scale)
    int stages;
    size_t lutb;   // LUT region in shared memory (0 when read from global)
};

TmaChoice tma_choice(amsim_lut_t lut)
{
    if (gemm_table_bytes(lut) <= (size_t)kMaxSmemLut) {
        const size_t lutb = kern::lut_region_bytes((int)gemm_table_bytes(lut));
        const int planes = kern::tma_planes(false);
        if (const int s = tma_stages(lutb, kern::kWideTiles, planes))
            return {kern::kWideTiles, true, false, planes, s, lutb};
        if (const int s = tma_stages(lutb, kern::kNarrowTiles, planes))
            return {kern::kNarrowTiles, false, false, planes, s, lutb};
    }
    const int planes = kern::tma_planes(true);
    return {kern::kWideTiles, true, true, planes, tma_stages(0, kern::kWideTiles, planes), 0};
}

int encode_plane_map(CUtensorMap *map, const PlaneKey &k, void *base, int box_rows, int box_k, int planes)
{
    EncodeTiled enc = encode_tiled();
    if (!enc) return AMSIM_EUNSUPPORTED;
    const cuuint64_t pitch = (cuuint64_t)rows_pad(k.rows) * 4;
    const cuuint64_t dims[4] = {(cuuint64_t)k.rows, (cuuint64_t)k.K, (cuuint64_t)planes, (cuuint64_t)k.nb};
    const cuuint64_t strides[3] = {pitch, pitch * (cuuint64_t)k.K, pitch * (cuuint64_t)k.K * planes};
    const cuuint32_t box[4] = {(cuuint32_t)box_rows, (cuuint32_t)box_k, (cuuint32_t)planes, 1};
    if (!boxes_ok(box, 4)) return AMSIM_EUNSUPPORTED;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, base, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? AMSIM_OK : AMSIM_EUNSUPPORTED;
}

// Access-pattern flags of a decode job (see DecodeJob).
void classify_job(kern::DecodeJob &d)
{
    const bool aligned = (reinterpret_cast<uintptr_t>(d.src) & 15) == 0 && (d.batch <= 1 || d.bs % 4 == 0);
    d.rowfast = d.s_row == 1 && d.rdiv >= d.rows && d.rlim >= d.rows && d.roff == 0 && d.kdiv >= d.K;
    if (d.rowfast)
        d.vec = aligned && (d.s_k % 4 == 0 || d.K == 1);
    else
        d.vec = aligned && d.s_k == 1 && (d.kdiv >= d.K || d.kdiv % 4 == 0) && d.s_row % 4 == 0 &&
                d.s_rhi % 4 == 0 && d.s_khi % 4 == 0;
}

int encode_raw_spec(CUtensorMap *map, const TmaRawMap &m)
{
    EncodeTiled enc = encode_tiled();
    if (!enc) return AMSIM_EUNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(m.base) & 15) return AMSIM_EUNSUPPORTED;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], estr[5];
    for (int i = 0; i < m.rank; ++i) {
        dims[i] = m.dims[i];
        box[i] = m.box[i];
        estr[i] = 1;
        if (i + 1 < m.rank) strides[i] = m.strides[i];
    }
    if (!boxes_ok(box, m.rank)) return AMSIM_EUNSUPPORTED;
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)m.rank, const_cast<float *>(m.base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           m.swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? AMSIM_OK : AMSIM_EUNSUPPORTED;
}

int launch_tma(int width, bool wide, const kern::KParams &kp, const kern::TmaMaps &maps, bool gl, dim3 grid,
               size_t smem, cudaStream_t st)
{
    if (wide) {
        switch (width) {
        case 8: return kern_wide::launch_tma_w8(kp, maps, gl, grid, smem, st);
        case 16: return kern_wide::launch_tma_w16(kp, maps, gl, grid, smem, st);
        default: return kern_wide::launch_tma_w32(kp, maps, gl, grid, smem, st);
        }
    }
    switch (width) {
    case 8: return kern::launch_tma_w8(kp, maps, gl, grid, smem, st);
    case 16: return kern::launch_tma_w16(kp, maps, gl, grid, smem, st);
    default: return kern::launch_tma_w32(kp, maps, gl, grid, smem, st);
    }
}

// The predecode pass, then the TMA LUT-GEMM over its planes: stream-K plans
// launch cooperatively and finish cut tiles inside the kernel, else (or
// without a cooperative launch) the separate fixup kernel does.
int run_tma(int width, bool wide, kern::KParams &tp, const kern::TmaMaps &maps, const kern::DecodeParams &dp,
            bool gl, long long blocks, size_t smem, int sms, bool streamk, cudaStream_t stream)
{
    const dim3 grid((unsigned)blocks);
    int rc = kern::launch_predecode(dp, sms, stream);
    if (rc) return rc;
    const int base = AMSIM_PATH_PLANES | (streamk ? AMSIM_PATH_STREAMK : 0) | (wide ? AMSIM_PATH_WIDE_TILES : 0);
    tp.fused = streamk && coop_launches() ? 1 : 0;
    rc = launch_tma(width, wide, tp, maps, gl, grid, smem, stream);
    if (rc == kern::AMSIM_ENOTCOOP) {
        tp.fused = 0;
        rc = launch_tma(width, wide, tp, maps, gl, grid, smem, stream);
    }
    if (rc) return rc;
    g_last_path |= base | (streamk && !tp.fused ? AMSIM_PATH_FIXUP : 0);
    if (!streamk || tp.fused) return AMSIM_OK;
    return wide ? kern_wide::launch_fixup(tp, tp.ctas - 1, stream) : kern::launch_fixup(tp, tp.ctas - 1, stream);
}

// ------------------------------------------------------------------ raw tiles
// A dense operand the copy engine reads in place: unit stride along rows or
// along k, the other strides multiples of 4 elements, and (when checked) a
// 16-byte aligned base.
bool raw_ok(const OperandDesc &d, int K, int batch, bool check_ptr)
{
    if (d.gather || d.rows <= 0 || K <= 0) return false;
    const bool rowfast = d.s_row == 1;
    if (!rowfast && d.s_k != 1) return false;
    const long long outer = rowfast ? d.s_k : d.s_row;
    if (outer <= 0 || outer % 4) return false;
    if (batch > 1 && d.batch_stride != 0 && d.batch_stride % 4) return false;
    if (check_ptr && (reinterpret_cast<uintptr_t>(d.ptr) & 15)) return false;
    return true;
}

// Elements of operands the raw-tile kernel would read with plain loads above
// which the launch prefers planes (plain loads serve small operands, such as
// a 10-wide layer's, without a predecode launch).
constexpr double kDirectElems = 256.0 * 1024;

// Every operand dense; each either copy-engine-strided or, in total, small
// enough for plain loads.
bool all_raw_ok(const Problem *p, int n, const Plan &pl, bool check_ptr)
{
    double direct = 0.0;
    for (int i = 0; i < n; ++i) {
        if (pl.tiles[i] == 0) continue;
        if (p[i].conv || p[i].U.gather || p[i].L.gather || p[i].K <= 0) return false;
        if (!raw_ok(p[i].U, p[i].K, p[i].batch, check_ptr))
            direct += (double)p[i].U.rows * p[i].K * (p[i].U.batch_stride ? p[i].batch : 1);
        if (!raw_ok(p[i].L, p[i].K, p[i].batch, check_ptr))
            direct += (double)p[i].L.rows * p[i].K * (p[i].L.batch_stride ? p[i].batch : 1);
    }
    return direct <= kDirectElems;
}

// 3-D map (rows or k innermost, then the other, then batch) over a raw operand.
int encode_raw_map(CUtensorMap *map, const OperandDesc &d, int K, int batch, int box_rows)
{
    EncodeTiled enc = encode_tiled();
    if (!enc) return AMSIM_EUNSUPPORTED;
    const bool rowfast = d.s_row == 1;
    const cuuint64_t outer = (cuuint64_t)(rowfast ? d.s_k : d.s_row);
    const cuuint64_t nb = (d.batch_stride == 0 || batch <= 1) ? 1 : (cuuint64_t)batch;
    const cuuint64_t inner_dim = rowfast ? (cuuint64_t)d.rows : (cuuint64_t)K;
    const cuuint64_t outer_dim = rowfast ? (cuuint64_t)K : (cuuint64_t)d.rows;
    const cuuint64_t dims[3] = {inner_dim, outer_dim, nb};
    // one batch only: any 16-byte multiple covering the operand serves as its stride
    const cuuint64_t bstride = nb > 1 ? (cuuint64_t)d.batch_stride * 4 : ((outer * outer_dim * 4 + 15) & ~15ULL);
    const cuuint64_t strides[2] = {outer * 4, bstride};
    const cuuint32_t box[3] = {rowfast ? (cuuint32_t)box_rows : (cuuint32_t)kern::BK,
                               rowfast ? (cuuint32_t)kern::BK : (cuuint32_t)box_rows, 1};
    if (!boxes_ok(box, 3)) return AMSIM_EUNSUPPORTED;
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(d.ptr), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           rowfast ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? AMSIM_OK : AMSIM_EUNSUPPORTED;
}

// Closed-form product code of the raw-tile kernel for a handle (0: the table).
int alu_code(amsim_lut_t lut)
{
    if (!lut || !lut->closed_form) return 0;
    return lut->kind == AMSIM_MITCHELL ? 1 : 2;
}

int launch_raw(int width, const kern::KParams &kp, const kern::TmaMaps &maps, bool gl, dim3 grid, size_t smem,
               cudaStream_t st, const kern::PhaseTable *pt = nullptr)
{
    if (kp.alu) return kern::launch_raw_alu(kp, maps, pt, grid, smem, st);
    switch (width) {
    case 8: return kern::launch_raw_w8(kp, maps, pt, gl, grid, smem, st);
    case 16: return kern::launch_raw_w16(kp, maps, pt, gl, grid, smem, st);
    default: return kern::launch_raw_w32(kp, maps, pt, gl, grid, smem, st);
    }
}

// Scratch the predecoded path adds after `base` bytes of stream-K scratch.
size_t tma_extra(size_t base, const PlaneSet &ps) { return align256(base) - base + kFlagBlock + ps.bytes; }

}  // namespace

size_t problems_workspace(const Problem *p, int n, amsim_lut_t lut)
{
    if (n <= 0 || n > kern::kMaxProblems) return 0;
    const int dev = lut ? lut->device : 0;
    const int sms = device_sms(dev);
    Plan pl = make_plan(p, n, sms, (size_t)-1);
    size_t need = pl.ws_bytes;
    PlaneSet rps;
    const int rwlog = lut ? (lut->width_bits == 8 ? 0 : lut->width_bits == 16 ? 1 : 2) : 0;
    if (lut && encode_tiled() && pl.iters < 0x7FFFFFFFLL && all_raw_ok(p, n, pl, false) &&
        (alu_code(lut) ||
         !(plan_planes(p, n, pl, lut->M, rwlog, 2 + 4 * 2, &rps) && rps.n > 0 && planes_beat_raw(p, n, pl, rps)))) {
        // operand tiles are copied in place and decoded inside the GEMM
    } else if (lut && encode_tiled() && n == 1 && p[0].conv) {
        // convolution tiles are copied in place as tensor boxes
    } else if (lut && encode_tiled()) {
        // the predecoded kernel's own plan (its tile shape's stream-K slots), then the planes
        const int wlog = lut->width_bits == 8 ? 0 : lut->width_bits == 16 ? 1 : 2;
        const TmaChoice tc = tma_choice(lut);
        const Plan tpl = make_plan(p, n, sms, (size_t)-1, tc.tc);
        PlaneSet ps;
        if (plan_planes(p, n, tpl, lut->M, wlog, tc.planes, &ps) && ps.n > 0 && planes_pay(p, n, tpl, ps))
            need = std::max(need, tpl.ws_bytes + tma_extra(tpl.ws_bytes, ps));
    }
    return need;
}

size_t problems_workspace_streamk(const Problem *p, int n, amsim_lut_t lut)
{
    if (n <= 0 || n > kern::kMaxProblems) return 0;
    const int dev = lut ? lut->device : 0;
    return make_plan(p, n, device_sms(dev), (size_t)-1).ws_bytes;
}

size_t problem_workspace(const Problem &p, amsim_lut_t lut) { return problems_workspace(&p, 1, lut); }

namespace {

// Launch parameters of the problems that have tiles (in launch order).
void fill_params(const Problem *p, int n, const Plan &pl, amsim_lut_t lut, kern::KParams &kp)
{
    int np = 0;
    long long tile0 = 0;
    for (int i = 0; i < n; ++i) {
        if (pl.tiles[i] == 0) continue;
        kern::ProbParams &q = kp.pr[np++];
        q.tile0 = tile0;
        tile0 += pl.tiles[i];
        q.U = p[i].U;
        q.L = p[i].L;
        q.K = p[i].K;
        q.batch = p[i].batch;
        q.tiles_u = pl.tiles_u[i];
        q.tiles_l = pl.tiles_l[i];
        q.kt_total = pl.kt[i];
        q.tiles = pl.tiles[i];
        q.iter0 = pl.iter0[i];
        q.table = p[i].u_is_first ? lut->d_narrow : lut->d_narrow_t;
        q.c_ptr = p[i].c_ptr;
        q.c_bs = p[i].c_bs;
        q.c_su = p[i].c_su;
        q.c_sl = p[i].c_sl;
        q.alpha = p[i].alpha;
        q.beta = p[i].beta;
        q.u_kfast = p[i].U.gather ? (p[i].U.kcb[0] == 1) : (p[i].U.s_k == 1 && p[i].U.s_row != 1);
        q.l_kfast = p[i].L.gather ? (p[i].L.kcb[0] == 1) : (p[i].L.s_k == 1 && p[i].L.s_row != 1);
    }
    kp.nprob = np;
    kp.streamk = pl.streamk ? 1 : 0;
    kp.iters = pl.iters;
    kp.ctas = pl.ctas;
    kp.M = lut->M;
    kp.wlog = lut->width_bits == 8 ? 0 : lut->width_bits == 16 ? 1 : 2;
    kp.fmt = exp_format(lut->exp_bits);
}

// Raw-tile operands of dense problems: a tensor map per copy-engine-strided
// operand, plain loads for the rest.
int encode_raw_problems(const Problem *p, int n, const Plan &pl, kern::KParams &tp, kern::TmaMaps &maps)
{
    int erc = AMSIM_OK;
    for (int i = 0, qi = 0; i < n && erc == AMSIM_OK; ++i) {
        if (pl.tiles[i] == 0) continue;
        kern::ProbParams &q = tp.pr[qi];
        q.u_direct = !raw_ok(p[i].U, p[i].K, p[i].batch, true);
        q.l_direct = !raw_ok(p[i].L, p[i].K, p[i].batch, true);
        if (q.u_direct || q.l_direct) tp.direct = 1;
        if (!q.u_direct) erc = encode_raw_map(&maps.u[qi], p[i].U, p[i].K, p[i].batch, BU);
        if (erc == AMSIM_OK && !q.l_direct) erc = encode_raw_map(&maps.l[qi], p[i].L, p[i].K, p[i].batch, BL);
        ++qi;
        q.u_kfast = p[i].U.s_row != 1;
        q.l_kfast = p[i].L.s_row != 1;
        q.u_bsel = (p[i].U.batch_stride != 0 && p[i].batch > 1) ? 1 : 0;
        q.l_bsel = (p[i].L.batch_stride != 0 && p[i].batch > 1) ? 1 : 0;
    }
    return erc;
}

// Shared memory of the raw-tile kernel and whether its LUT is read from global
// (closed-form launches stage no table).
size_t raw_smem(amsim_lut_t lut, bool *gl)
{
    if (alu_code(lut)) {
        *gl = false;
        return (size_t)kern::raw_smem_bytes(0);
    }
    bool raw_gl = gemm_table_bytes(lut) > (size_t)kMaxSmemLut;
    if (!raw_gl && kern::raw_smem_bytes((int)gemm_table_bytes(lut)) > kMaxSmemPerCta) raw_gl = true;
    *gl = raw_gl;
    return (size_t)kern::raw_smem_bytes(raw_gl ? 0 : (int)gemm_table_bytes(lut));
}

// One launch for problems that all read the same LUT orientation.
int run_same_table(const Problem *p, int n, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (n <= 0) return AMSIM_OK;
    if (n > kern::kMaxProblems) return AMSIM_EINVAL;
    const int sms = device_sms(lut->device);
    // scratch that breaks the 256-byte alignment rule is not used
    if (reinterpret_cast<uintptr_t>(ws) & 255) ws = nullptr;
    const Plan pl = make_plan(p, n, sms, ws ? ws_bytes : 0);
    if (pl.total_tiles == 0) return AMSIM_OK;

    // Shared-memory LUT when it fits beside the warp-specialised kernel's
    // rings; else beside the single-role kernel's stages; else read from global.
    const size_t lut_smem = kern::lut_region_bytes((int)gemm_table_bytes(lut));
    bool use_ws = true, gl = false;
    if (gemm_table_bytes(lut) > (size_t)kMaxSmemLut) gl = true;
    else if ((size_t)kern::kWsFixedSmem + lut_smem <= (size_t)kMaxSmemPerCta) gl = false;
    else if ((size_t)kern::kFixedSmem + lut_smem <= (size_t)kMaxSmemPerCta) use_ws = false;
    else gl = true;
    kern::KParams kp = {};
    fill_params(p, n, pl, lut, kp);
    kp.table_bytes = gl ? 0 : (int)gemm_table_bytes(lut);
    kp.ws = static_cast<float *>(ws);

    const long long blocks = pl.streamk ? pl.ctas : pl.total_tiles;
    if (blocks > 0x7FFFFFFFLL) return AMSIM_EUNSUPPORTED;

    // Raw operand tiles copied in place by TMA and decoded in shared memory,
    // when every operand is dense with copy-engine strides -- unless planes
    // fit the scratch and beat them (planes_beat_raw: large launches whose
    // operand elements are reused by many tiles).
    // The predecoded kernel's tile shape and its own plan, which it runs only
    // as planned with unlimited scratch (planes after its stream-K region).
    const TmaChoice tc = tma_choice(lut);
    const Plan tpl = make_plan(p, n, sms, (size_t)-1, tc.tc);
    PlaneSet ps;
    const bool planes_fit = ws && encode_tiled() && plan_planes(p, n, tpl, lut->M, kp.wlog, tc.planes, &ps) && ps.n > 0 &&
                            ws_bytes >= tpl.ws_bytes + tma_extra(tpl.ws_bytes, ps);
    // (the raw-tile kernel counts a launch's iterations in 32 bits)
    const bool raw_fits = pl.iters < 0x7FFFFFFFLL;
    const bool conv_raw = raw_fits && n == 1 && p[0].conv && pl.tiles[0] > 0 && encode_tiled();
    // Closed-form products exist only in the raw-tile kernel, which then takes
    // every problem it can read.  Formats with fewer than 8 exponent bits run
    // on the in-kernel-decode kernels only (their decoders apply the cast).
    const int alu = alu_code(lut);
    const bool fmt = kp.fmt.on != 0;
    if (!fmt && (conv_raw || (raw_fits && encode_tiled() && all_raw_ok(p, n, pl, true) &&
                              (alu || !(planes_fit && planes_beat_raw(p, n, pl, ps)))))) {
        bool raw_gl = false;
        const size_t smem = raw_smem(lut, &raw_gl);
        kern::TmaMaps maps = {};
        kern::KParams tp = kp;
        int erc = AMSIM_OK;
        if (conv_raw) {
            const ConvRaw &cv = *p[0].conv;
            erc = encode_raw_spec(&maps.u[0], cv.umap);
            if (erc == AMSIM_OK) erc = encode_raw_spec(&maps.l[0], cv.lmap);
            kern::ProbParams &q = tp.pr[0];
            q.u_kfast = cv.u_kfast;
            q.l_kfast = cv.mode == 1 ? 1 : 0;
            q.u_bsel = q.l_bsel = 0;
            tp.conv = cv.mode;
            tp.cv_u_tap = cv.u_tap;
            tp.cv_ch = cv.ch;
            tp.cv_S = cv.S;
            tp.cv_tiles_img = cv.tiles_img;
            tp.cv_rows_tile = cv.rows_tile;
            tp.cv_ybase = cv.ybase;
            tp.cv_ystep = cv.ystep;
            tp.cv_xbase = cv.xbase;
            tp.cv_xstep = cv.xstep;
            tp.cv_N = cv.N;
            tp.cv_P = cv.P;
            tp.cv_Q = cv.Q;
            tp.cv_rows = cv.rows;
        } else {
            erc = encode_raw_problems(p, n, pl, tp, maps);
        }
        if (erc == AMSIM_OK) {
            tp.alu = alu;
            tp.table_bytes = (raw_gl || alu) ? 0 : (int)gemm_table_bytes(lut);
            tp.epoch = g_epoch.fetch_add(1, std::memory_order_relaxed);
            tp.fused = pl.streamk && coop_launches() ? 1 : 0;
            streamk_bounds_by_cost(p, n, pl, tp);
            const dim3 grid((unsigned)blocks);
            int rc = launch_raw(lut->width_bits, tp, maps, raw_gl, grid, smem, stream);
            if (rc == kern::AMSIM_ENOTCOOP) {
                tp.fused = 0;
                rc = launch_raw(lut->width_bits, tp, maps, raw_gl, grid, smem, stream);
            }
            if (rc == AMSIM_OK) {
                const bool fix = pl.streamk && !tp.fused;
                g_last_path |= AMSIM_PATH_RAW_TILES | (pl.streamk ? AMSIM_PATH_STREAMK : 0) |
                               (fix ? AMSIM_PATH_FIXUP : 0) | (tp.conv ? AMSIM_PATH_CONV_BOXES : 0) |
                               (alu ? AMSIM_PATH_CLOSED_FORM : 0);
                return fix ? kern::launch_fixup(tp, pl.ctas - 1, stream) : AMSIM_OK;
            }
            if (rc != AMSIM_EUNSUPPORTED) return rc;
        }
    }

    // Predecoded operands copied by TMA, when every operand is dense (or a
    // convolution laid out for TMA) and the scratch holds the planes after the
    // stream-K region.
    const long long tblocks = tpl.streamk ? tpl.ctas : tpl.total_tiles;
    if (!fmt && planes_fit && planes_pay(p, n, tpl, ps) && tc.stages > 0 && tblocks <= 0x7FFFFFFFLL) {
        kern::KParams tp = {};
        fill_params(p, n, tpl, lut, tp);
        tp.ws = static_cast<float *>(ws);
        uint8_t *base = static_cast<uint8_t *>(ws);
        const size_t flags_off = align256(tpl.ws_bytes);
        unsigned long long *flags = reinterpret_cast<unsigned long long *>(base + flags_off);
        uint8_t *planes = base + flags_off + kFlagBlock;
        const unsigned long long epoch = g_epoch.fetch_add(1, std::memory_order_relaxed);
        kern::DecodeParams dp = {};
        dp.M = lut->M;
        dp.epoch = epoch;
        long long dtiles = 0;
        for (int j = 0; j < ps.n; ++j) {
            const PlaneKey &k = ps.key[j];
            kern::DecodeJob &d = dp.job[j];
            d.src = k.src;
            d.bs = k.bs;
            d.s_row = k.s_row;
            d.s_k = k.s_k;
            d.s_rhi = 0;
            d.s_khi = 0;
            d.rdiv = k.rows;
            d.roff = 0;
            d.rlim = k.rows;
            d.kdiv = k.K;
            d.rows = k.rows;
            d.K = k.K;
            d.batch = k.nb;
            d.rows_pad = rows_pad(k.rows);
            d.offshift = k.offshift;
            d.packed = ps.nplanes[j] == 1;
            d.plane = reinterpret_cast<uint32_t *>(planes + ps.off[j]);
            d.flag = flags + j;
            d.flag_small = flags + kern::kMaxDecodeJobs + j;
            d.zero_off = ps.uniform[j] ? kern::uniform_zero_row(lut->M, k.offshift) : 0u;
            d.tiles_r = ceil_div(k.rows, kern::kDecodeTileR);
            d.tiles_k = ceil_div(k.K, kern::kDecodeTileK);
            d.tile0 = dtiles;
            dtiles += (long long)k.nb * d.tiles_r * d.tiles_k;
            classify_job(d);
        }
        dp.njobs = ps.n;
        dp.tiles = dtiles;
        kern::TmaMaps maps = {};
        int erc = AMSIM_OK;
        for (int i = 0, qi = 0; i < n && erc == AMSIM_OK; ++i) {
            if (tpl.tiles[i] == 0) continue;
            const int ju = ps.slot[2 * i], jl = ps.slot[2 * i + 1];
            erc = encode_plane_map(&maps.u[qi], ps.key[ju], planes + ps.off[ju], tc.tc.bu, tc.tc.bk, ps.nplanes[ju]);
            if (erc == AMSIM_OK)
                erc = encode_plane_map(&maps.l[qi], ps.key[jl], planes + ps.off[jl], tc.tc.bl, tc.tc.bk, ps.nplanes[jl]);
            kern::ProbParams &q = tp.pr[qi++];
            q.u_big = flags + ju;
            q.l_big = flags + jl;
            q.u_small = flags + kern::kMaxDecodeJobs + ju;
            q.l_small = flags + kern::kMaxDecodeJobs + jl;
            q.u_bsel = ps.key[ju].nb > 1 ? 1 : 0;
            q.l_bsel = ps.key[jl].nb > 1 ? 1 : 0;
        }
        if (erc == AMSIM_OK) {
            tp.table_bytes = tc.gl ? 0 : (int)gemm_table_bytes(lut);
            tp.stages = tc.stages;
            tp.epoch = epoch;
            const size_t smem = (size_t)kern::tma_cfg_smem_bytes(tc.tc, tc.planes, (int)tc.lutb, tp.stages);
            const int rc = run_tma(lut->width_bits, tc.wide, tp, maps, dp, tc.gl, tblocks, smem, sms, tpl.streamk,
                                   stream);
            if (rc != AMSIM_EUNSUPPORTED) return rc;
        }
    }

    const size_t lutb = gl ? 0 : kern::lut_region_bytes(kp.table_bytes);
    // warp-specialised kernel next; the single-role kernel if its register
    // split cannot be honoured on this device
    int rc = AMSIM_EUNSUPPORTED;
    const int sk = pl.streamk ? AMSIM_PATH_STREAMK : 0;
    if (use_ws) {
        // stream-K: finish cut tiles inside the kernel when a cooperative
        // launch is possible, else run the separate fixup kernel afterwards
        kp.fused = pl.streamk && coop_launches() ? 1 : 0;
        kp.epoch = g_epoch.fetch_add(1, std::memory_order_relaxed);
        rc = launch_ws(lut->width_bits, kp, gl, dim3((unsigned)blocks), (size_t)kern::kWsFixedSmem + lutb, stream);
        if (rc == kern::AMSIM_ENOTCOOP) {
            kp.fused = 0;
            rc = launch_ws(lut->width_bits, kp, gl, dim3((unsigned)blocks), (size_t)kern::kWsFixedSmem + lutb, stream);
        }
        if (rc == AMSIM_OK) g_last_path |= AMSIM_PATH_INKERNEL_DECODE | sk;
        if (rc == AMSIM_OK && kp.fused) return AMSIM_OK;
    }
    if (rc == AMSIM_EUNSUPPORTED) {
        kp.fused = 0;
        rc = launch_w(lut->width_bits, kp, gl, dim3((unsigned)blocks), (size_t)kern::kFixedSmem + lutb, stream);
        if (rc == AMSIM_OK) g_last_path |= AMSIM_PATH_SINGLE_ROLE | sk;
    }
    if (rc || !pl.streamk) return rc;
    g_last_path |= AMSIM_PATH_FIXUP;
    return kern::launch_fixup(kp, pl.ctas - 1, stream);
}

}  // namespace

int run_problems(const Problem *p, int n, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    g_last_path = 0;
    if (n <= 0) return AMSIM_OK;
    if (n > kern::kMaxProblems) return AMSIM_EINVAL;
    if (lut->symmetric) return run_same_table(p, n, lut, ws, ws_bytes, stream);
    // an asymmetric LUT read in both orientations: one launch per orientation
    Problem part[kern::kMaxProblems];
    for (int orient = 0; orient < 2; ++orient) {
        int m = 0;
        for (int i = 0; i < n; ++i)
            if ((int)p[i].u_is_first == orient) part[m++] = p[i];
        int rc = run_same_table(part, m, lut, ws, ws_bytes, stream);
        if (rc) return rc;
    }
    return AMSIM_OK;
}

int run_problem(const Problem &p, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    return run_problems(&p, 1, lut, ws, ws_bytes, stream);
}

namespace {

// Scratch of a phased launch: a completion flag per phase and CTA, per tile
// an arrival ticket and a spare word, then (256-byte aligned) two partial-sum
// slots of a BU x BL tile per CTA and phase, from which the last part of a cut
// tile adds all parts in CTA order.
size_t phased_sk_bytes(int nphase, int G, long long tiles)
{
    const size_t words = ((size_t)nphase * G + 2 * (size_t)tiles) * sizeof(unsigned long long);
    return align256(words) + (size_t)nphase * G * 2 * BU * BL * sizeof(float);
}

// Problems [first[ph], first[ph + 1]) of phase ph (the last ends at n).
void phase_bounds(const int *first, int nphase, int n, int ph, int *lo, int *hi)
{
    *lo = first[ph];
    *hi = ph + 1 < nphase ? first[ph + 1] : n;
}

// One launch can run all phases: dense operands for the raw-tile kernel,
// one LUT orientation, at most kMaxPhases phases and kMaxProblems problems.
bool phased_ok(const Problem *p, int n, int nphase, const Plan &pl, amsim_lut_t lut, bool check_ptr)
{
    if (nphase < 2 || nphase > kern::kMaxPhases || n > kern::kMaxProblems || pl.ctas < 2) return false;
    if (lut->exp_bits != 8) return false;           // formats run on the in-kernel-decode kernels
    if (pl.ctas > kern::kMaxPhasedCtas) return false;
    if (pl.iters >= 0x7FFFFFFFLL) return false;     // the raw-tile kernel counts iterations in 32 bits
    if (!encode_tiled()) return false;
    bool gl = false;
    raw_smem(lut, &gl);
    if (gl) return false;                           // phased launches stage the LUT in shared memory
    for (int i = 1; i < n; ++i)
        if (!lut->symmetric && p[i].u_is_first != p[0].u_is_first) return false;
    return all_raw_ok(p, n, pl, check_ptr);
}

// Relative time of one stage of a tile: consumer warps whose rows or columns
// all lie past the operands' edges skip their lookups, and such stages run
// faster -- measured on GB300 from per-CTA timelines of phased launches, a
// stage with a fraction f of its warps busy takes about 0.47 + 0.53 f of a
// full stage (0.6 at f = 1/4) -- so shares are cut by this cost, not by count.
// A tail tile (all real lane columns in the first column block) runs in a
// tail layout, every warp on half (or, with at most 64 real columns, a
// quarter) of a warp's lookups, and its producer decodes only the columns
// that layout reads.  Measured on GB300 against a full stage: 0.58 (64 x 128
// GEMM tiles) and 0.43 (64 x 64) for one tile per SM; 0.51 and 0.45 for the
// 64-column tail of the 3x3 filter gradient with the 8-bit Mitchell and the
// 16-bit exact table.  A share that overestimates a stage's cost loses less
// than one that underestimates it, so the model takes 0.62 and 0.50.
// (Phased launches keep the regular layout on tail tiles: tail_layout false.)
double stage_cost(const Problem &p, int ut, int lt, bool tail_layout)
{
    constexpr int WUn = BU / kern::TM, WLn = BL / (32 * kern::TN);
    if (tail_layout && kern::narrow_tail_tile(lt * BL, p.L.rows)) return 0.50;
    if (tail_layout && kern::tail_tile(lt * BL, p.L.rows)) return 0.62;
    int busy = 0;
    for (int wu = 0; wu < WUn; ++wu)
        for (int wl = 0; wl < WLn; ++wl)
            busy += (ut * BU + wu * kern::TM < p.U.rows && lt * BL + wl * 32 * kern::TN < p.L.rows) ? 1 : 0;
    return 0.47 + 0.53 * busy / (WUn * WLn);
}

// Stream-K shares of an ordinary raw-tile launch cut by stage cost: CTA c
// starts where the running cost of the launch's tiles (in iteration order)
// reaches c / G of the total, rounded to a stage, every share at least one
// stage.  False (keep the even split) when every stage costs the same, when
// the launch has more than 16 tiles per CTA (each share then holds a mix of
// tiles close to the launch's own, and the walk over the tiles would cost
// host time), or when the table does not hold the CTAs or the iterations.
bool streamk_bounds_by_cost(const Problem *p, int n, const Plan &pl, kern::KParams &kp)
{
    kp.sk_n = 0;
    const int G = pl.ctas;
    if (!pl.streamk || G > kern::kMaxPhasedCtas || pl.iters >= 0x7FFFFFFFLL || pl.iters < G) return false;
    if (pl.total_tiles > 16LL * G) return false;
    struct Run { long long it0; int kt; double w; };
    std::vector<Run> runs;                  // tiles in iteration order
    double C = 0.0;
    bool uneven = false;
    for (int i = 0; i < n; ++i) {
        if (pl.tiles[i] == 0) continue;
        long long it = pl.iter0[i];
        for (int b = 0; b < p[i].batch; ++b)
            for (int ut = 0; ut < pl.tiles_u[i]; ++ut)
                for (int lt = 0; lt < pl.tiles_l[i]; ++lt) {
                    const double w = stage_cost(p[i], ut, lt, true);
                    uneven |= w != 1.0;
                    runs.push_back({it, pl.kt[i], w});
                    C += w * pl.kt[i];
                    it += pl.kt[i];
                }
    }
    if (!uneven) return false;
    int *bound = kp.sk_bound;
    bound[0] = 0;
    size_t r = 0;
    double before = 0.0;                    // cost of the runs before run r
    for (int c = 1; c < G; ++c) {
        const double target = C * c / G;
        while (r + 1 < runs.size() && before + runs[r].w * runs[r].kt <= target) {
            before += runs[r].w * runs[r].kt;
            ++r;
        }
        const long long s = std::llround((target - before) / runs[r].w);
        long long it = runs[r].it0 + std::min<long long>(std::max<long long>(s, 0), runs[r].kt);
        it = std::max<long long>(it, bound[c - 1] + 1);             // no empty share
        it = std::min<long long>(it, pl.iters - (G - c));           // room for the shares after it
        bound[c] = (int)it;
    }
    bound[G] = (int)pl.iters;
    kp.sk_n = G;
    return true;
}

// Share boundaries of every phase.  CTAs 0 .. c-1 together get, through
// phase ph, the cumulative stage cost c / G of phases 0 .. ph (rounded to a
// stage): each phase's boundary for CTA c is where the phase's running cost
// reaches that target minus what the earlier phases actually gave those
// CTAs, so the rounding of one phase is made up in the next and per-CTA
// totals stay within about a stage of each other however many phases there
// are.
void phased_bounds_by_cost(const Problem *p, const Plan &pl, const int *first, int nphase, int n, int G,
                           kern::PhaseTable *pt)
{
    std::vector<double> prev(G + 1, 0.0), target(G + 1), actual(G + 1);
    double V = 0.0;
    for (int ph = 0; ph < nphase; ++ph) {
        int lo, hi;
        phase_bounds(first, nphase, n, ph, &lo, &hi);
        struct Run { int kt; double w; };
        std::vector<Run> runs;                  // tiles in iteration order
        double C = 0.0;
        long long W = 0;
        for (int i = lo; i < hi; ++i) {
            if (pl.tiles[i] == 0) continue;
            for (int b = 0; b < p[i].batch; ++b)
                for (int ut = 0; ut < pl.tiles_u[i]; ++ut)
                    for (int lt = 0; lt < pl.tiles_l[i]; ++lt) {
                        const double w = stage_cost(p[i], ut, lt, false);
                        runs.push_back({pl.kt[i], w});
                        C += w * pl.kt[i];
                        W += pl.kt[i];
                    }
        }
        V += C;
        target[0] = 0.0;
        for (int c = 1; c < G; ++c)
            target[c] = std::min(std::max(V * c / G - prev[c], target[c - 1]), C);
        target[G] = C;
        int *bound = pt->bound[ph];
        bound[0] = 0;
        actual[0] = 0.0;
        int c = 1;
        long long it = 0;
        double cum = 0.0;
        for (const Run &r : runs) {
            const double tc = r.w * r.kt;
            while (c < G && cum + tc >= target[c]) {
                const long long k =
                    std::min<long long>(std::max<long long>(std::llround((target[c] - cum) / r.w), 0), r.kt);
                bound[c] = (int)(it + k);
                actual[c] = cum + k * r.w;
                ++c;
            }
            cum += tc;
            it += r.kt;
        }
        for (; c <= G; ++c) {
            bound[c] = (int)W;
            actual[c] = C;
        }
        for (int k = 1; k <= G; ++k) prev[k] += actual[k];
    }
}

}  // namespace

int run_phased(const Problem *p, int n, int nphase, const int *first, const int *after, amsim_lut_t lut, void *ws,
               size_t ws_bytes, cudaStream_t stream)
{
    g_last_path = 0;
    if (n <= 0) return AMSIM_OK;
    if (reinterpret_cast<uintptr_t>(ws) & 255) ws = nullptr;
    const int sms = device_sms(lut->device);
    Plan pl = make_plan(p, std::min(n, kern::kMaxProblems), sms, (size_t)-1);
    if (pl.total_tiles == 0 && n <= kern::kMaxProblems) return AMSIM_OK;
    if (ws && coop_launches() && phased_ok(p, n, nphase, pl, lut, true) &&
        ws_bytes >= phased_sk_bytes(nphase, pl.ctas, pl.total_tiles)) {
        pl.streamk = true;
        kern::KParams tp = {};
        fill_params(p, n, pl, lut, tp);
        bool gl = false;
        const size_t smem = raw_smem(lut, &gl);
        tp.alu = alu_code(lut);
        tp.table_bytes = (gl || tp.alu) ? 0 : (int)gemm_table_bytes(lut);
        tp.ws = static_cast<float *>(ws);
        tp.nphase = nphase;
        for (int ph = 0; ph < nphase; ++ph) {
            int lo, hi;
            phase_bounds(first, nphase, n, ph, &lo, &hi);
            tp.ph_iter0[ph] = lo < n ? pl.iter0[lo] : pl.iters;
            tp.ph_after[ph] = after[ph];
        }
        tp.ph_iter0[nphase] = pl.iters;
        kern::PhaseTable pt;
        phased_bounds_by_cost(p, pl, first, nphase, n, pl.ctas, &pt);
        kern::TmaMaps maps = {};
        int rc = encode_raw_problems(p, n, pl, tp, maps);
        if (rc == AMSIM_OK) {
            tp.epoch = g_epoch.fetch_add(1, std::memory_order_relaxed);
            tp.fused = 1;
            rc = launch_raw(lut->width_bits, tp, maps, gl, dim3((unsigned)pl.ctas), smem, stream, &pt);
            if (rc == AMSIM_OK) {
                g_last_path = AMSIM_PATH_RAW_TILES | AMSIM_PATH_STREAMK | AMSIM_PATH_PHASED |
                              (tp.alu ? AMSIM_PATH_CLOSED_FORM : 0);
                return AMSIM_OK;
            }
            if (rc != kern::AMSIM_ENOTCOOP && rc != AMSIM_EUNSUPPORTED) return rc;
        }
    }
    // one grouped launch (or more) per phase, in order on the stream
    int path = 0;
    for (int ph = 0; ph < nphase; ++ph) {
        int lo, hi;
        phase_bounds(first, nphase, n, ph, &lo, &hi);
        for (int base = lo; base < hi; base += kern::kMaxProblems) {
            const int rc = run_problems(p + base, std::min(hi - base, kern::kMaxProblems), lut, ws, ws_bytes, stream);
            path |= g_last_path;
            if (rc) return rc;
        }
    }
    g_last_path = path;
    return AMSIM_OK;
}

size_t phased_workspace(const Problem *p, int n, int nphase, const int *first, amsim_lut_t lut)
{
    size_t best = 0;
    for (int ph = 0; ph < nphase; ++ph) {
        int lo, hi;
        phase_bounds(first, nphase, n, ph, &lo, &hi);
        for (int base = lo; base < hi; base += kern::kMaxProblems)
            best = std::max(best, problems_workspace(p + base, std::min(hi - base, kern::kMaxProblems), lut));
    }
    if (n <= kern::kMaxProblems) {
        const Plan pl = make_plan(p, n, device_sms(lut->device), (size_t)-1);
        if (phased_ok(p, n, nphase, pl, lut, false))
            best = std::max(best, phased_sk_bytes(nphase, pl.ctas, pl.total_tiles));
    }
    return best;
}

}  // namespace amsim

// ------------------------------------------------------------------ GEMM ABI
namespace {

using amsim::OperandDesc;
using amsim::Problem;
using amsim::kern::BL;
using amsim::kern::BU;

OperandDesc dense(const float *ptr, int rows, long long s_row, long long s_k, long long batch_stride)
{
    OperandDesc d = {};
    d.ptr = ptr;
    d.rows = rows;
    d.gather = 0;
    d.s_row = s_row;
    d.s_k = s_k;
    d.batch_stride = batch_stride;
    d.kD0 = d.kD1 = d.rE0 = d.rE1 = 1;
    d.IH = d.IW = 1;
    d.sy = d.sx = 1;
    return d;
}

bool trans_flag(char t, bool *out)
{
    if (t == 'N' || t == 'n') { *out = false; return true; }
    if (t == 'T' || t == 't') { *out = true; return true; }
    return false;
}

// Padded tile area if U = first operand's rows (a) and L = second's (b).
long long padded_area(int u_rows, int l_rows)
{
    return (long long)((u_rows + BU - 1) / BU) * BU * ((long long)((l_rows + BL - 1) / BL) * BL);
}

int build_gemm(char transA, char transB, int m, int n, int k, float alpha, const float *A, int lda,
               long long strideA, const float *B, int ldb, long long strideB, float beta, float *C, int ldc,
               long long strideC, int batch, Problem *pr)
{
    bool ta, tb;
    if (!trans_flag(transA, &ta) || !trans_flag(transB, &tb)) return AMSIM_EINVAL;
    if (m < 0 || n < 0 || k < 0 || batch < 0) return AMSIM_EINVAL;
    if (strideA < 0 || strideB < 0 || strideC < 0) return AMSIM_EINVAL;
    if (lda < std::max(1, ta ? m : k) || ldb < std::max(1, tb ? k : n) || ldc < std::max(1, n)) return AMSIM_EINVAL;
    if (batch > 0 && m > 0 && n > 0) {
        if (!C) return AMSIM_EINVAL;
        if (k > 0 && (!A || !B)) return AMSIM_EINVAL;
    }
    const OperandDesc a = dense(A, m, ta ? 1 : lda, ta ? lda : 1, strideA);
    const OperandDesc b = dense(B, n, tb ? ldb : 1, tb ? 1 : ldb, strideB);
    const bool swap = padded_area(n, m) < padded_area(m, n);
    pr->U = swap ? b : a;
    pr->L = swap ? a : b;
    pr->u_is_first = !swap;
    pr->K = k;
    pr->batch = batch;
    pr->c_ptr = C;
    pr->c_bs = strideC;
    pr->c_su = swap ? 1 : ldc;
    pr->c_sl = swap ? ldc : 1;
    pr->alpha = alpha;
    pr->beta = beta;
    return AMSIM_OK;
}

}  // namespace

namespace amsim {

size_t gemm_workspace(char transA, char transB, int m, int n, int k, int batch, amsim_lut_t lut, bool streamk_only)
{
    if (!lut) return 0;
    Problem pr;
    static const float dummy = 0.0f;
    float *dc = const_cast<float *>(&dummy);
    bool ta, tb;
    if (!trans_flag(transA, &ta) || !trans_flag(transB, &tb) || m < 0 || n < 0 || k < 0 || batch < 1) return 0;
    // A distinct dummy address per operand keeps the two planes apart, and a
    // nonzero batch stride sizes one plane per batch (the most a call can need).
    static const float dummy2 = 0.0f;
    if (build_gemm(transA, transB, m, n, k, 1.0f, &dummy, std::max(1, ta ? m : k), 1, &dummy2,
                   std::max(1, tb ? k : n), 1, 0.0f, dc, std::max(1, n), 0, batch, &pr))
        return 0;
    return streamk_only ? problems_workspace_streamk(&pr, 1, lut) : problem_workspace(pr, lut);
}

void set_last_path(int bits) { g_last_path = bits; }

int encode_tensor_map(CUtensorMap_st *map, const TmaRawMap &m) { return encode_raw_spec(map, m); }

}  // namespace amsim

extern "C" {

int amsim_last_path(void) { return amsim::g_last_path; }

int amsim_gemm_strided_batched(char transA, char transB, int m, int n, int k, float alpha, const float *A, int lda,
                               int64_t strideA, const float *B, int ldb, int64_t strideB, float beta, float *C,
                               int ldc, int64_t strideC, int batch, amsim_lut_t lut, void *ws, size_t ws_bytes,
                               amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    Problem pr;
    rc = build_gemm(transA, transB, m, n, k, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC, batch,
                    &pr);
    if (rc) return rc;
    return amsim::run_problem(pr, lut, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

int amsim_gemm(char transA, char transB, int m, int n, int k, float alpha, const float *A, int lda, const float *B,
               int ldb, float beta, float *C, int ldc, amsim_lut_t lut, void *ws, size_t ws_bytes,
               amsim_stream_t stream)
{
    return amsim_gemm_strided_batched(transA, transB, m, n, k, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1, lut,
                                      ws, ws_bytes, stream);
}

static int grouped_build(const amsim_gemm_problem *g, Problem *pr)
{
    return build_gemm(g->transA, g->transB, g->m, g->n, g->k, g->alpha, g->A, g->lda, g->strideA, g->B, g->ldb,
                      g->strideB, g->beta, g->C, g->ldc, g->strideC, g->batch, pr);
}

int amsim_gemm_grouped(int count, const amsim_gemm_problem *problems, amsim_lut_t lut, void *ws, size_t ws_bytes,
                       amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    if (count < 0 || (count > 0 && !problems)) return AMSIM_EINVAL;
    Problem pr[amsim::kern::kMaxProblems];
    for (int i = 0; i < count; ++i) {           // validate everything before enqueuing anything
        rc = grouped_build(&problems[i], &pr[0]);
        if (rc) return rc;
    }
    for (int base = 0; base < count; base += amsim::kern::kMaxProblems) {
        const int n = std::min(count - base, amsim::kern::kMaxProblems);
        for (int i = 0; i < n; ++i) grouped_build(&problems[base + i], &pr[i]);
        rc = amsim::run_problems(pr, n, lut, ws, ws_bytes, static_cast<cudaStream_t>(stream));
        if (rc) return rc;
    }
    return AMSIM_OK;
}

namespace {

// Phases of a phased call: phase_first[0] == 0, non-decreasing, within
// [0, count]; phase_after[ph] in [0, ph].
bool phases_valid(int count, int nphase, const int *phase_first, const int *phase_after)
{
    if (nphase < 1 || !phase_first || !phase_after || phase_first[0] != 0) return false;
    for (int ph = 0; ph < nphase; ++ph) {
        if (phase_first[ph] < 0 || phase_first[ph] > count) return false;
        if (ph > 0 && phase_first[ph] < phase_first[ph - 1]) return false;
        if (phase_after[ph] < 0 || phase_after[ph] > ph) return false;
    }
    return true;
}

}  // namespace

int amsim_gemm_phased(int count, const amsim_gemm_problem *problems, int nphase, const int *phase_first,
                      const int *phase_after, amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    if (count < 0 || (count > 0 && !problems)) return AMSIM_EINVAL;
    if (!phases_valid(count, nphase, phase_first, phase_after)) return AMSIM_EINVAL;
    Problem pr[amsim::kern::kMaxProblems];
    for (int i = 0; i < count; ++i) {           // validate everything before enqueuing anything
        rc = grouped_build(&problems[i], &pr[0]);
        if (rc) return rc;
    }
    if (count <= amsim::kern::kMaxProblems) {
        for (int i = 0; i < count; ++i) grouped_build(&problems[i], &pr[i]);
        return amsim::run_phased(pr, count, nphase, phase_first, phase_after, lut, ws, ws_bytes,
                                 static_cast<cudaStream_t>(stream));
    }
    // more problems than one launch holds: the phases one after another
    for (int ph = 0; ph < nphase; ++ph) {
        const int lo = phase_first[ph], hi = ph + 1 < nphase ? phase_first[ph + 1] : count;
        rc = amsim_gemm_grouped(hi - lo, problems + lo, lut, ws, ws_bytes, stream);
        if (rc) return rc;
    }
    return AMSIM_OK;
}

size_t amsim_gemm_phased_workspace_size(int count, const amsim_gemm_problem *problems, int nphase,
                                        const int *phase_first, const int *phase_after, amsim_lut_t lut)
{
    if (!lut || count <= 0 || !problems || !phases_valid(count, nphase, phase_first, phase_after)) return 0;
    if (count > amsim::kern::kMaxProblems) {
        size_t best = 0;
        for (int ph = 0; ph < nphase; ++ph) {
            const int lo = phase_first[ph], hi = ph + 1 < nphase ? phase_first[ph + 1] : count;
            if (hi > lo) best = std::max(best, amsim_gemm_grouped_workspace_size(hi - lo, problems + lo, lut));
        }
        return best;
    }
    Problem pr[amsim::kern::kMaxProblems];
    for (int i = 0; i < count; ++i)
        if (grouped_build(&problems[i], &pr[i])) return 0;
    return amsim::phased_workspace(pr, count, nphase, phase_first, lut);
}

size_t amsim_gemm_grouped_workspace_size(int count, const amsim_gemm_problem *problems, amsim_lut_t lut)
{
    if (!lut || count <= 0 || !problems) return 0;
    Problem pr[amsim::kern::kMaxProblems];
    size_t best = 0;
    for (int base = 0; base < count; base += amsim::kern::kMaxProblems) {
        const int n = std::min(count - base, amsim::kern::kMaxProblems);
        for (int i = 0; i < n; ++i)
            if (grouped_build(&problems[base + i], &pr[i])) return 0;
        best = std::max(best, amsim::problems_workspace(pr, n, lut));
    }
    return best;
}

size_t amsim_gemm_workspace_size(char transA, char transB, int m, int n, int k, int batch, amsim_lut_t lut)
{
    return amsim::gemm_workspace(transA, transB, m, n, k, batch, lut, false);
}

}  // extern "C"

extern "C" int amsim_set_cooperative_launches(int on)
{
    if (on != 0 && on != 1) return AMSIM_EINVAL;
    amsim::g_coop.store(on != 0, std::memory_order_relaxed);
    return AMSIM_OK;
}
