// Host side of libmoeblock: plan, workspace layout, argument validation, TMA
// tensor maps and the launch sequence of each C-ABI call.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "kernels.cuh"

using namespace moe;

struct moe_plan {
    moe_dims d;
    int device;
    int num_sms;
    const void *wr, *wg, *wu, *wd, *sg, *su, *sd;
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_sg, tm_su, tm_sd;
    CUtensorMap tm_wr;    // router weights for the tensor-core screening (E <= 256)
    bool tc_route;        // the large-batch router applies to this shape
    cudaEvent_t fwd_events[5];
    int n_fwd_events;
    uint64_t wait_ns;     // limit of the kernels' pipeline waits (0: built in)
    // quantised experts (qbits 8 or 4; 0: bf16): tm_wg .. tm_sd map the codes,
    // these the scales
    int qbits;
    CUtensorMap tm_cg, tm_cu, tm_cd, tm_csg, tm_csu, tm_csd;
};

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
moe_status fail(moe_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

moe_status ok() {
    g_last_error.clear();
    return MOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 tensor map, row-major [d2][d1][d0] (rank 2 if d2 == 0), box (64, box1[, 1]),
// 128-byte swizzle, out-of-bounds elements read as zero.
bool encode_bf16(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint32_t box1, CUtensorMapL2promotion l2) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint32_t rank = d2 ? 3 : 2;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {64, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A tensor map without swizzle: dims[0] innermost (elements), box[i] elements;
// rank 2 or 3; out-of-bounds elements read as zero.
bool encode_plain(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* ptr,
                  uint32_t rank, const uint64_t* dims, const uint32_t* box,
                  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[3], strides[2];
    cuuint32_t b[3], estr[3] = {1, 1, 1};
    for (uint32_t i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
    strides[0] = dims[0] * esize;
    strides[1] = dims[0] * dims[1] * esize;
    CUresult r = fn(m, dt, rank, const_cast<void*>(ptr), d, strides, b, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

moe_status check_dims(const moe_dims* d) {
    if (!d) return fail(MOE_ERR_INVALID_ARG, "dims is NULL");
    if (d->H <= 0 || d->H % 256)
        return fail(MOE_ERR_UNSUPPORTED, "H=%d must be a positive multiple of 256", d->H);
    if (d->E < 1 || d->E > 1024) return fail(MOE_ERR_UNSUPPORTED, "E=%d must be in [1, 1024]", d->E);
    if (d->k < 1 || d->k > 32 || d->k > d->E)
        return fail(MOE_ERR_UNSUPPORTED, "k=%d must be in [1, min(32, E)]", d->k);
    if (d->I <= 0 || d->I % 64) return fail(MOE_ERR_UNSUPPORTED, "I=%d must be a positive multiple of 64", d->I);
    if (d->Is <= 0 || d->Is % 64)
        return fail(MOE_ERR_UNSUPPORTED, "Is=%d must be a positive multiple of 64", d->Is);
    if (d->max_rows < 1 || d->max_blocks < 1)
        return fail(MOE_ERR_INVALID_ARG, "max_rows=%d and max_blocks=%d must be >= 1", d->max_rows,
                    d->max_blocks);
    if (d->max_rows > (1 << 21) || (int64_t)d->max_rows * d->k > (1 << 30) ||
        (int64_t)d->max_rows * d->H > (int64_t)1 << 34)
        return fail(MOE_ERR_UNSUPPORTED, "max_rows=%d too large (at most 2^21)", d->max_rows);
    return MOE_OK;
}

moe_status check_call(const moe_plan* p, int32_t R, const int32_t* off, int32_t nb, void* ws,
                      size_t ws_bytes) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    if (R < 0 || R > p->d.max_rows)
        return fail(MOE_ERR_INVALID_ARG, "R=%d outside [0, max_rows=%d]", R, p->d.max_rows);
    if (nb < 1 || nb > p->d.max_blocks)
        return fail(MOE_ERR_INVALID_ARG, "nb=%d outside [1, max_blocks=%d]", nb, p->d.max_blocks);
    if (!off || !aligned(off, 4)) return fail(MOE_ERR_INVALID_ARG, "block_offsets NULL or misaligned");
    if (!ws || !aligned(ws, 256)) return fail(MOE_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
    const size_t need = make_layout(p->d).total;
    if (ws_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device)
        return fail(MOE_ERR_INVALID_ARG, "current device %d is not the plan's device %d", dev,
                    p->device);
    return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

moe_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

bool moe::plan_view(const moe_plan* p, PlanView* out) {
    if (!p || !out) return false;
    out->d = p->d;
    out->device = p->device;
    out->num_sms = p->num_sms;
    out->w_router = p->wr;
    return true;
}

moe_status moe::set_error(moe_status s, const char* msg) {
    g_last_error = msg ? msg : "";
    return s;
}

namespace {

// Record forward event i of the plan on `st`, if the plan has events.  Under
// stream capture an event record must be an external node to be recorded at
// every graph launch (a plain record only orders the capture).
cudaError_t mark_event(const moe_plan* p, int i, cudaStream_t st) {
    if (p->n_fwd_events != 5) return cudaSuccess;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cap);
    if (e != cudaSuccess) return e;
    return cudaEventRecordWithFlags(
        p->fwd_events[i], st,
        cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

// The forward's launches after validation: the scatter, the two grouped GEMMs
// and the combine.  `marked`: event 0 of the plan's forward events was already
// recorded by the caller.
moe_status enqueue_forward(const moe_plan* p, const void* x, int32_t R,
                           const int32_t* block_offsets, int32_t nb, const int32_t* topk_idx,
                           const float* w_renorm, const uint32_t* keep, const uint8_t* live,
                           void* y, float* y_f32, void* workspace, cudaStream_t st,
                           bool marked) {
    const moe_dims& d = p->d;
    const Layout L = make_layout(d);
    const bool small = R <= kSmallRows;
    // units of the streaming shape (32 rows, two CTAs per SM): small calls, and
    // quantised weights at any size; the down GEMM also up to kStreamDownRows
    // rows (few pairs per expert: its CTA-pair units would be mostly empty)
    const bool su = small || p->qbits != 0;
    const bool sd = su || R <= kStreamDownRows;
    const int nt_gu = su ? kSmallN : kLargeNGU;
    const int nt_dn = sd ? kSmallN : kLargeNDown;

    ScatterArgs sa{block_offsets, topk_idx, w_renorm, keep, R, d.H, d.E, d.k, d.I, d.Is, nb, nt_gu, nt_dn,
                   su ? 64 : 128, sd ? 128 : 256,
                   at<int32_t>(workspace, L.prank), at<int32_t>(workspace, L.hist),
                   at<int32_t>(workspace, L.count),
                   at<int32_t>(workspace, L.expert_off), at<int32_t>(workspace, L.misc),
                   at<int4>(workspace, L.units_gu), at<int4>(workspace, L.units_dn),
                   at<int32_t>(workspace, L.pair_row), at<float>(workspace, L.pair_w),
                   at<int32_t>(workspace, L.inv),
                   at<uint32_t>(workspace, L.status),
                   live, at<int32_t>(workspace, L.shared_rows), at<int32_t>(workspace, L.shared_inv),
                   at<int32_t>(workspace, L.live_base)};
    GemmMaps gu{}, dn{};
    const auto L2A = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    gu.a0 = p->tm_wg; gu.a1 = p->tm_wu; gu.a2 = p->tm_sg; gu.a3 = p->tm_su;
    dn.a0 = p->tm_wd; dn.a1 = p->tm_wd; dn.a2 = p->tm_sd; dn.a3 = p->tm_sd;
    if (p->qbits) {
        gu.s0 = p->tm_cg; gu.s1 = p->tm_cu; gu.s2 = p->tm_csg; gu.s3 = p->tm_csu;
        dn.s0 = p->tm_cd; dn.s1 = p->tm_cd; dn.s2 = p->tm_csd; dn.s3 = p->tm_csd;
    } else {
        gu.s0 = gu.s1 = gu.s2 = gu.s3 = p->tm_wg;   // unused by the bf16 kernels
        dn.s0 = dn.s1 = dn.s2 = dn.s3 = p->tm_wd;
    }
    // B rows per TMA box: k_gemm's streaming shape 32 (gate/up: x) and 16 (down:
    // h); k_down_pair a rank's 128
    const uint32_t box_gu = su ? 32 : 128, box_dn = sd ? 16 : 128;
    bool good = encode_bf16(&gu.b1, x, d.H, (uint64_t)R, 0, box_gu, L2A) &&
                encode_bf16(&gu.bg, x, d.H, (uint64_t)R, 0, 1, L2A) &&
                encode_bf16(&dn.b0, at<void>(workspace, L.h), (uint64_t)d.I, (uint64_t)L.max_pairs, 0,
                            box_dn, L2A) &&
                encode_bf16(&dn.b1, at<void>(workspace, L.hs), 2 * (uint64_t)d.Is,
                            (uint64_t)d.max_rows, 0, box_dn, L2A);
    if (!good) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation tensor");
    GemmArgs ga{at<int4>(workspace, L.units_gu), at<int32_t>(workspace, L.misc) + 1, d.E, d.H, d.I,
                d.Is, R, static_cast<const __nv_bfloat16*>(x), at<__nv_bfloat16>(workspace, L.h),
                at<__nv_bfloat16>(workspace, L.hs),
                at<int32_t>(workspace, L.pair_row), at<float>(workspace, L.pair_w),
                at<__half>(workspace, L.ys), at<uint8_t>(workspace, L.ysx),
                (int)(L.max_pairs + d.max_rows), at<int32_t>(workspace, L.misc) + 4,
                (int)L.max_pairs, at<uint32_t>(workspace, L.status),
                live ? at<int32_t>(workspace, L.shared_rows) : nullptr, p->wait_ns};
    auto mark = [&](int i) { return mark_event(p, i, st); };
    cudaError_t e = marked ? cudaSuccess : mark(0);
    if (e == cudaSuccess) e = launch_scatter(sa, small, p->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "scatter launch");
    if ((e = mark(1)) == cudaSuccess) e = launch_gemm(kGateUp, su, p->qbits, gu, ga, p->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "gate/up GEMM launch");
    GemmArgs gd = ga;
    gd.units = at<int4>(workspace, L.units_dn);
    gd.n_units = at<int32_t>(workspace, L.misc) + 2;
    if ((e = mark(2)) == cudaSuccess) e = launch_gemm(kDown, sd, p->qbits, dn, gd, p->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "down GEMM launch");
    CombineArgs ca{at<__half>(workspace, L.ys), at<uint8_t>(workspace, L.ysx),
                   (int)(L.max_pairs + d.max_rows), at<int32_t>(workspace, L.misc) + 4,
                   at<int32_t>(workspace, L.inv), R, d.H, d.k,
                   (int)L.max_pairs, static_cast<__nv_bfloat16*>(y), y_f32,
                   at<uint32_t>(workspace, L.status), live, at<int32_t>(workspace, L.shared_inv)};
    if ((e = mark(3)) == cudaSuccess) e = launch_combine(ca, p->num_sms, !sd, st);
    if (e == cudaSuccess) e = mark(4);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return ok();
}

}  // namespace

extern "C" {

int32_t moe_version(void) { return 100; }

const char* moe_last_error(void) { return g_last_error.c_str(); }

size_t moe_workspace_bytes(const moe_dims* dims) {
    if (check_dims(dims) != MOE_OK) return 0;
    return make_layout(*dims).total;
}

moe_status moe_plan_create(const moe_dims* dims, const void* w_router, const void* w_gate,
                           const void* w_up, const void* w_down, const void* ws_gate,
                           const void* ws_up, const void* ws_down, moe_plan** out) {
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    moe_status s = check_dims(dims);
    if (s != MOE_OK) return s;
    const void* ws[7] = {w_router, w_gate, w_up, w_down, ws_gate, ws_up, ws_down};
    const char* names[7] = {"w_router", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"};
    for (int i = 0; i < 7; ++i)
        if (!ws[i] || !aligned(ws[i], 16))
            return fail(MOE_ERR_INVALID_ARG, "%s is NULL or not 16-byte aligned", names[i]);
    moe_plan* p = new moe_plan();
    p->d = *dims;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess) e = gemm_set_attributes();
    if (e == cudaSuccess) e = gateup_pair_set_attributes(p->num_sms);
    if (e == cudaSuccess) e = down_pair_set_attributes(p->num_sms);
    if (e == cudaSuccess) e = route_tc_set_attributes();
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "device query");
    }
    p->wr = w_router; p->wg = w_gate; p->wu = w_up; p->wd = w_down;
    p->sg = ws_gate; p->su = ws_up; p->sd = ws_down;
    const moe_dims& d = *dims;
    const auto L2W = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    bool good = encode_bf16(&p->tm_wg, w_gate, d.H, d.I, d.E, 64, L2W) &&
                encode_bf16(&p->tm_wu, w_up, d.H, d.I, d.E, 64, L2W) &&
                encode_bf16(&p->tm_wd, w_down, d.I, d.H, d.E, 128, L2W) &&
                encode_bf16(&p->tm_sg, ws_gate, d.H, d.Is, 0, 64, L2W) &&
                encode_bf16(&p->tm_su, ws_up, d.H, d.Is, 0, 64, L2W) &&
                encode_bf16(&p->tm_sd, ws_down, d.Is, d.H, 0, 128, L2W);
    p->tc_route = d.E <= 256 && d.E % 16 == 0 && d.k <= 16 && d.H <= 8192;
    if (good && p->tc_route)
        good = encode_bf16(&p->tm_wr, w_router, d.H, d.E, 0,
                           (uint32_t)((d.E > 128 && d.E % 32 == 0) ? d.E / 2 : d.E),
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (!good) {
        delete p;
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight tensor");
    }
    *out = p;
    return ok();
}

moe_status moe_plan_create_quantized(const moe_dims* dims, const void* w_router,
                                     const moe_quant_weights* qw, moe_plan** out) {
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    moe_status s = check_dims(dims);
    if (s != MOE_OK) return s;
    if (!qw) return fail(MOE_ERR_INVALID_ARG, "quantised weights are NULL");
    if (qw->bits != 8 && qw->bits != 4)
        return fail(MOE_ERR_UNSUPPORTED, "bits=%d: quantised experts are 8 or 4 bits", qw->bits);
    const void* ws[9] = {w_router, qw->gate_up, qw->down, qw->gate_up_scale, qw->down_scale,
                         qw->shared_gate_up, qw->shared_down, qw->shared_gate_up_scale,
                         qw->shared_down_scale};
    const char* names[9] = {"w_router", "gate_up", "down", "gate_up_scale", "down_scale",
                            "shared_gate_up", "shared_down", "shared_gate_up_scale",
                            "shared_down_scale"};
    for (int i = 0; i < 9; ++i)
        if (!ws[i] || !aligned(ws[i], 16))
            return fail(MOE_ERR_INVALID_ARG, "%s is NULL or not 16-byte aligned", names[i]);
    moe_plan* p = new moe_plan();
    p->d = *dims;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess) e = gemm_set_attributes();
    if (e == cudaSuccess) e = gateup_pair_set_attributes(p->num_sms);
    if (e == cudaSuccess) e = down_pair_set_attributes(p->num_sms);
    if (e == cudaSuccess) e = route_tc_set_attributes();
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "device query");
    }
    const moe_dims& d = *dims;
    p->qbits = qw->bits;
    p->wr = w_router;
    p->wg = qw->gate_up; p->wu = qw->gate_up; p->wd = qw->down;
    p->sg = qw->shared_gate_up; p->su = qw->shared_gate_up; p->sd = qw->shared_down;
    // codes: uint8, K in bytes (halved for 4 bits), boxes of 64 K x 128 rows
    // (gate/up: 64 gate rows and their 64 up rows, interleaved), swizzled over
    // the box's row width (64 or 32 bytes) for the converters' row reads; scales: bf16
    // [blocks][rows], boxes of 128 rows x 2 blocks.  The up maps (tm_wu, tm_su,
    // tm_cu, tm_csu) repeat the gate/up ones: the interleaved tensor holds both.
    const uint64_t kb = qw->bits == 8 ? 1 : 2;
    const uint32_t cbox = (uint32_t)(64 / kb);
    const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const auto B16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t dg[3] = {d.H / kb, 2 * (uint64_t)d.I, (uint64_t)d.E}, dd[3] = {d.I / kb, (uint64_t)d.H, (uint64_t)d.E};
    const uint64_t dsg[2] = {d.H / kb, 2 * (uint64_t)d.Is}, dsd[2] = {d.Is / kb, (uint64_t)d.H};
    const uint32_t bt[3] = {cbox, 128, 1};
    const CUtensorMapSwizzle csw = qw->bits == 8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    const uint64_t cg[3] = {2 * (uint64_t)d.I, (uint64_t)(d.H / 32), (uint64_t)d.E};
    const uint64_t cd[3] = {(uint64_t)d.H, (uint64_t)(d.I / 32), (uint64_t)d.E};
    const uint64_t csg[2] = {2 * (uint64_t)d.Is, (uint64_t)(d.H / 32)}, csd[2] = {(uint64_t)d.H, (uint64_t)(d.Is / 32)};
    const uint32_t sb[3] = {128, 2, 1};
    bool good = encode_plain(&p->tm_wg, U8, 1, qw->gate_up, 3, dg, bt, csw) &&
                encode_plain(&p->tm_wd, U8, 1, qw->down, 3, dd, bt, csw) &&
                encode_plain(&p->tm_sg, U8, 1, qw->shared_gate_up, 2, dsg, bt, csw) &&
                encode_plain(&p->tm_sd, U8, 1, qw->shared_down, 2, dsd, bt, csw) &&
                encode_plain(&p->tm_cg, B16, 2, qw->gate_up_scale, 3, cg, sb) &&
                encode_plain(&p->tm_cd, B16, 2, qw->down_scale, 3, cd, sb) &&
                encode_plain(&p->tm_csg, B16, 2, qw->shared_gate_up_scale, 2, csg, sb) &&
                encode_plain(&p->tm_csd, B16, 2, qw->shared_down_scale, 2, csd, sb);
    p->tm_wu = p->tm_wg; p->tm_su = p->tm_sg; p->tm_cu = p->tm_cg; p->tm_csu = p->tm_csg;
    p->tc_route = d.E <= 256 && d.E % 16 == 0 && d.k <= 16 && d.H <= 8192;
    if (good && p->tc_route)
        good = encode_bf16(&p->tm_wr, w_router, d.H, d.E, 0,
                           (uint32_t)((d.E > 128 && d.E % 32 == 0) ? d.E / 2 : d.E),
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (!good) {
        delete p;
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for a quantised weight tensor");
    }
    *out = p;
    return ok();
}

void moe_plan_destroy(moe_plan* plan) { delete plan; }

moe_status moe_block_route(const moe_plan* p, const void* x, int32_t R,
                           const int32_t* block_offsets, int32_t nb, const float* logit_bias,
                           int32_t* topk_idx, float* topk_w, void* workspace,
                           size_t workspace_bytes, moe_stream_t stream) {
    return moe_block_route_probs(p, x, R, block_offsets, nb, logit_bias, topk_idx, topk_w, nullptr,
                                 workspace, workspace_bytes, stream);
}

moe_status moe_block_route_probs(const moe_plan* p, const void* x, int32_t R,
                                 const int32_t* block_offsets, int32_t nb, const float* logit_bias,
                                 int32_t* topk_idx, float* topk_w, float* topk_p, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream) {
    moe_status s = check_call(p, R, block_offsets, nb, workspace, workspace_bytes);
    if (s != MOE_OK) return s;
    if (!x || !aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x is NULL or not 16-byte aligned");
    if (!topk_idx || !topk_w || !aligned(topk_idx, 4) || !aligned(topk_w, 4))
        return fail(MOE_ERR_INVALID_ARG, "topk_idx/topk_w NULL or misaligned");
    if (topk_p && !aligned(topk_p, 4)) return fail(MOE_ERR_INVALID_ARG, "topk_p misaligned");
    if (logit_bias && !aligned(logit_bias, 4)) return fail(MOE_ERR_INVALID_ARG, "logit_bias misaligned");
    if (R == 0) return ok();
    const Layout L = make_layout(p->d);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the probabilities need the exact logit of every expert: the fixed-order
    // router computes them all; the tensor-core screen only the candidates'
    if (p->tc_route && R >= kTcRouteMinRows && !topk_p) {
        CUtensorMap tm_x;
        if (!encode_bf16(&tm_x, x, p->d.H, (uint64_t)R, 0, 128, CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for x");
        RouteTcArgs ta{static_cast<const __nv_bfloat16*>(x),
                       static_cast<const __nv_bfloat16*>(p->wr), logit_bias, block_offsets, R,
                       p->d.H, p->d.E, p->d.k, nb,
                       at<float>(workspace, L.wnorm), at<float>(workspace, L.logits), topk_idx, topk_w,
                       at<uint32_t>(workspace, L.status), p->wait_ns,
                       route_tc_parts(R, p->d.E, p->d.H, logit_rows(p->d.max_rows), p->num_sms)};
        cudaError_t e = launch_route_tc(ta, tm_x, p->tm_wr, p->num_sms, st);
        if (e != cudaSuccess) return cuda_fail(e, "route launch");
        return ok();
    }
    cudaError_t e = cudaMemsetAsync(at<uint8_t>(workspace, L.route_cnt), 0,
                                    sizeof(uint32_t) * (size_t)R, st);
    if (e != cudaSuccess) return cuda_fail(e, "route counters");
    RouteArgs a{static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(p->wr),
                logit_bias, block_offsets, R, p->d.H, p->d.E, p->d.k, nb,
                at<float>(workspace, L.logits), at<uint32_t>(workspace, L.route_cnt), topk_idx,
                topk_w, at<uint32_t>(workspace, L.status), topk_p};
    e = launch_route(a, p->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    return ok();
}

moe_status moe_block_coreset(const moe_plan* p, int32_t R, const int32_t* block_offsets,
                             int32_t nb, const int32_t* topk_idx, const float* topk_w, float tau,
                             uint32_t* keep, int32_t* core_size, float* w_renorm,
                             int32_t* n_empty, void* workspace, size_t workspace_bytes,
                             moe_stream_t stream) {
    return moe_block_coreset_budget(p, R, block_offsets, nb, topk_idx, topk_w, tau, 0, keep,
                                    core_size, w_renorm, n_empty, workspace, workspace_bytes, stream);
}

moe_status moe_block_coreset_budget(const moe_plan* p, int32_t R, const int32_t* block_offsets,
                                    int32_t nb, const int32_t* topk_idx, const float* topk_w,
                                    float tau, int32_t max_experts, uint32_t* keep,
                                    int32_t* core_size, float* w_renorm, int32_t* n_empty,
                                    void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return moe_block_coreset_mass(p, R, block_offsets, nb, topk_idx, topk_w, nullptr, tau,
                                  max_experts, keep, core_size, w_renorm, n_empty, workspace,
                                  workspace_bytes, stream);
}

moe_status moe_block_coreset_mass(const moe_plan* p, int32_t R, const int32_t* block_offsets,
                                  int32_t nb, const int32_t* topk_idx, const float* topk_w,
                                  const float* topk_mass, float tau, int32_t max_experts,
                                  uint32_t* keep, int32_t* core_size, float* w_renorm,
                                  int32_t* n_empty, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream) {
    moe_status s = check_call(p, R, block_offsets, nb, workspace, workspace_bytes);
    if (s != MOE_OK) return s;
    if (!(tau > 0.0f)) return fail(MOE_ERR_INVALID_ARG, "tau=%g must be > 0 (and not NaN)", (double)tau);
    if (max_experts < 0) return fail(MOE_ERR_INVALID_ARG, "max_experts=%d must be >= 0", max_experts);
    if (!topk_idx || !topk_w || !keep || !core_size || !w_renorm)
        return fail(MOE_ERR_INVALID_ARG, "a required coreset pointer is NULL");
    const void* ps[7] = {topk_idx, topk_w, keep, core_size, w_renorm, n_empty, topk_mass};
    for (const void* q : ps)
        if (q && !aligned(q, 4)) return fail(MOE_ERR_INVALID_ARG, "coreset pointer misaligned");
    const Layout L = make_layout(p->d);
    CoresetArgs a{block_offsets, topk_idx, topk_w, topk_mass, R, p->d.E, p->d.k, nb, tau,
                  max_experts, keep, core_size, w_renorm, n_empty, at<uint32_t>(workspace, L.status)};
    cudaError_t e = launch_coreset(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "coreset launch");
    return ok();
}

moe_status moe_block_forward(const moe_plan* p, const void* x, int32_t R,
                             const int32_t* block_offsets, int32_t nb, const int32_t* topk_idx,
                             const float* w_renorm, const uint32_t* keep, void* y, float* y_f32,
                             void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return moe_block_forward_live(p, x, R, block_offsets, nb, topk_idx, w_renorm, keep, nullptr, y,
                                  y_f32, workspace, workspace_bytes, stream);
}

moe_status moe_block_forward_live(const moe_plan* p, const void* x, int32_t R,
                                  const int32_t* block_offsets, int32_t nb, const int32_t* topk_idx,
                                  const float* w_renorm, const uint32_t* keep, const uint8_t* live,
                                  void* y, float* y_f32, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream) {
    moe_status s = check_call(p, R, block_offsets, nb, workspace, workspace_bytes);
    if (s != MOE_OK) return s;
    if (!x || !aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x is NULL or not 16-byte aligned");
    if (!y || !aligned(y, 16)) return fail(MOE_ERR_INVALID_ARG, "y is NULL or not 16-byte aligned");
    if (y_f32 && !aligned(y_f32, 16)) return fail(MOE_ERR_INVALID_ARG, "y_f32 not 16-byte aligned");
    if (!topk_idx || !w_renorm || !keep || !aligned(topk_idx, 4) || !aligned(w_renorm, 4) ||
        !aligned(keep, 4))
        return fail(MOE_ERR_INVALID_ARG, "topk_idx/w_renorm/keep NULL or misaligned");
    if (R == 0) return ok();
    return enqueue_forward(p, x, R, block_offsets, nb, topk_idx, w_renorm, keep, live, y, y_f32,
                           workspace, reinterpret_cast<cudaStream_t>(stream), false);
}

moe_status moe_block_pass(const moe_plan* p, const void* x, int32_t R, const int32_t* block_offsets,
                          int32_t nb, const float* logit_bias, float tau, int32_t max_experts,
                          int32_t* topk_idx, float* topk_w, float* topk_p, uint32_t* keep,
                          int32_t* core_size, float* w_renorm, int32_t* n_empty, void* y,
                          float* y_f32, void* workspace, size_t workspace_bytes,
                          moe_stream_t stream) {
    moe_status s = check_call(p, R, block_offsets, nb, workspace, workspace_bytes);
    if (s != MOE_OK) return s;
    if (!x || !aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x is NULL or not 16-byte aligned");
    if (!y || !aligned(y, 16)) return fail(MOE_ERR_INVALID_ARG, "y is NULL or not 16-byte aligned");
    if (y_f32 && !aligned(y_f32, 16)) return fail(MOE_ERR_INVALID_ARG, "y_f32 not 16-byte aligned");
    if (!topk_idx || !topk_w || !keep || !core_size || !w_renorm)
        return fail(MOE_ERR_INVALID_ARG, "a required pass output is NULL");
    const void* ps[8] = {topk_idx, topk_w, keep, core_size, w_renorm, n_empty, topk_p, logit_bias};
    for (const void* q : ps)
        if (q && !aligned(q, 4)) return fail(MOE_ERR_INVALID_ARG, "pass pointer misaligned");
    if (!(tau > 0.0f)) return fail(MOE_ERR_INVALID_ARG, "tau=%g must be > 0 (and not NaN)", (double)tau);
    if (max_experts < 0) return fail(MOE_ERR_INVALID_ARG, "max_experts=%d must be >= 0", max_experts);
    if (R == 0) return ok();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the router, coreset and forward kernels of the three calls, back to back with
    // programmatic dependent launch between them (no host synchronisation)
    cudaError_t e = mark_event(p, 0, st);
    if (e != cudaSuccess) return cuda_fail(e, "event record");
    s = moe_block_route_probs(p, x, R, block_offsets, nb, logit_bias, topk_idx, topk_w, topk_p,
                              workspace, workspace_bytes, stream);
    if (s != MOE_OK) return s;
    s = moe_block_coreset_mass(p, R, block_offsets, nb, topk_idx, topk_w, topk_p, tau, max_experts,
                               keep, core_size, w_renorm, n_empty, workspace, workspace_bytes, stream);
    if (s != MOE_OK) return s;
    return enqueue_forward(p, x, R, block_offsets, nb, topk_idx, w_renorm, keep, nullptr, y, y_f32,
                           workspace, st, true);
}

moe_status moe_plan_set_forward_events(moe_plan* p, moe_event_t const* events,
                                       int32_t n_events) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    if (n_events == 0) {
        p->n_fwd_events = 0;
        return ok();
    }
    if (n_events != 5 || !events) return fail(MOE_ERR_INVALID_ARG, "need exactly 5 events");
    for (int i = 0; i < 5; ++i) {
        if (!events[i]) return fail(MOE_ERR_INVALID_ARG, "event %d is NULL", i);
        p->fwd_events[i] = reinterpret_cast<cudaEvent_t>(events[i]);
    }
    p->n_fwd_events = 5;
    return ok();
}

moe_status moe_plan_set_wait_limit(moe_plan* p, uint64_t limit_ns) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
    p->wait_ns = limit_ns;
    return ok();
}

moe_status moe_read_device_status(const void* workspace, moe_stream_t stream, uint32_t* out) {
    if (!workspace || !aligned(workspace, 256) || !out)
        return fail(MOE_ERR_INVALID_ARG, "workspace or out invalid");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(out, workspace, sizeof(uint32_t) * MOE_STATUS_WORDS,
                                    cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    return ok();
}

moe_status moe_clear_device_status(void* workspace, moe_stream_t stream) {
    if (!workspace || !aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace invalid");
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t) * MOE_STATUS_WORDS,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return ok();
}

}  // extern "C"
