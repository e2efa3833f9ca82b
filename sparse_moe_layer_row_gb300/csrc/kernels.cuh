// Argument blocks and launchers of the kernels of libmoeblock (router.cu,
// coreset.cu, scatter.cu, gemm.cu); the host code in api.cu fills them in.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

struct RouteArgs {
    const __nv_bfloat16* x;
    const __nv_bfloat16* wr;
    const float* bias;
    const int32_t* off;
    int R, H, E, k, nb;
    float* logits;
    uint32_t* cnt;
    int32_t* topk_idx;
    float* topk_w;
    uint32_t* status;
    float* topk_p;        // [R, k] probabilities under the full softmax, or NULL
};
// Large-batch router (tensor-core screening + exact recompute of candidates).
constexpr int kCandCap = 32;      // candidates kept per row before falling back
struct RouteTcArgs {
    const __nv_bfloat16* x;
    const __nv_bfloat16* wr;
    const float* bias;
    const int32_t* off;
    int R, H, E, k, nb;
    float* wnorm;         // [E]
    float* logits;        // [nk][R, E] approximate logits (tensor cores), one slice per K part
    int32_t* topk_idx;
    float* topk_w;
    uint32_t* status;
    uint64_t wait_ns;     // limit of a pipeline wait (0: the built-in limit)
    int nk;               // parts the screen's K range is split into (summed in order by the exact pass)
};
struct CoresetArgs {
    const int32_t* off;
    const int32_t* topk_idx;
    const float* topk_w;
    const float* mass;    // [R, k] masses of the slots, or NULL: the masses are topk_w
    int R, E, k, nb;
    float tau;
    int max_experts;      // expert budget per block (<= 0: none)
    uint32_t* keep;
    int32_t* core_size;
    float* w_renorm;
    int32_t* n_empty;
    uint32_t* status;
};
struct ScatterArgs {
    const int32_t* off;
    const int32_t* topk_idx;
    const float* w_renorm;
    const uint32_t* keep;
    int R, H, E, k, I, Is, nb;
    int nt_gu, nt_dn;   // rows per unit of the gate/up and of the down GEMM
    int gu_rows;        // intermediate rows per gate/up unit (64 or 128)
    int dn_cols;        // hidden outputs per down unit (128, or 256 on CTA pairs)
    int32_t* prank;       // [R * k] rank of a pair among its block's pairs of its expert, or -1
    int32_t* hist;        // [nb, E] pairs per (block, expert), then bases within the expert
    int32_t* count;       // [E] surviving pairs per expert
    int32_t* expert_off;
    int32_t* misc;
    int4* units_gu;
    int4* units_dn;
    int32_t* pair_row;
    float* pair_w;
    int32_t* inv;         // [R * k] staging row of (row, slot), or -1
    uint32_t* status;
    // live-row reuse: only rows with live[r] != 0 are evaluated (NULL: all rows)
    const uint8_t* live;
    int32_t* shared_rows; // [R] the live rows in order: the shared expert's rows
    int32_t* shared_inv;  // [R] position of a row in shared_rows, or -1 (dead)
    int32_t* live_base;   // [nb] live rows per block, then live rows before the block
};
// y[r] = shared output + sum over surviving slots (rank order) of staged outputs
struct CombineArgs {
    const __half* ys;     // [max_pairs + max_rows, H] staged per-pair / shared outputs
    const uint8_t* ysx;   // [H / 32, max_pairs + max_rows] exponent of each staged quarter row
    int ld_x;             // max_pairs + max_rows (the staging rows)
    const int32_t* scaled;   // nonzero: some exponent is not 0 (else ysx need not be read)
    const int32_t* inv;   // [R * k]
    int R, H, k, shared_row0;
    __nv_bfloat16* y;
    float* y_f32;
    uint32_t* status;
    const uint8_t* live;         // rows with live[r] == 0 are left as they are (NULL: all live)
    const int32_t* shared_inv;   // [R] staging index of a row's shared output (NULL: r)
};
struct GemmArgs {
    const int4* units;
    const int32_t* n_units;
    int E, H, I, Is;
    int R;                // rows of x (gathered row indices >= R read as zero)
    const __nv_bfloat16* x;  // [R, H] (rows gathered by the large gate/up loaders)
    __nv_bfloat16* h;     // [pairs, I] routed activations (bf16)
    __nv_bfloat16* hs;    // [rows, 2Is] shared activations: bf16 hi part | bf16 lo part
    const int32_t* pair_row;
    const float* pair_w;
    __half* ys;           // [max_pairs + max_rows, H] staged outputs (down GEMM)
    uint8_t* ysx;         // [H / 32, max_pairs + max_rows] their quarter-row exponents
    int ld_x;             // max_pairs + max_rows
    int32_t* scaled;      // set to 1 when some exponent is not 0 (zeroed by the scatter)
    int shared_row0;      // staging row of the shared expert's row 0
    uint32_t* status;
    const int32_t* shared_rows;  // row of x of the shared expert's i-th row (NULL: i)
    uint64_t wait_ns;     // limit of a pipeline wait (0: the built-in limit)
};
// A unit (expert g, weight tile m, first row `start`, n rows) as the scatter
// writes it: g in [0, E] (E: the shared expert), 1 <= n <= nmax, rows inside
// h / hs and the staging buffer, m inside the weights.  Every role of a GEMM
// checks each unit it reads and skips one that fails (it can only fail if the
// workspace was overwritten while the call ran), so such a unit never drives a
// zero-width MMA or a store past a buffer; one role counts it.
// dn_cols: hidden outputs per down unit (128, or 256 on CTA pairs).
__device__ __forceinline__ bool unit_valid(const int4 un, const GemmArgs& a, int nmax, bool down,
                                           int gu_rows, int dn_cols = 128) {
    const int g = un.x, m = un.y, start = un.z, n = un.w;
    if (g < 0 || g > a.E || n < 1 || n > nmax || start < 0) return false;
    const int cap = g == a.E ? a.ld_x - a.shared_row0 : a.shared_row0;
    if (start > cap - n) return false;
    const int mt = down ? a.H / dn_cols : ((g == a.E ? a.Is : a.I) + gu_rows - 1) / gu_rows;
    return m >= 0 && m < mt;
}
struct GemmMaps {
    CUtensorMap a0, a1, a2, a3, b0, b1;
    CUtensorMap bg;   // x with a one-row box: TMA gather4 of routed rows (small batches)
    // quantised weights: a0..a3 are the codes, s0..s3 their scales (unused for bf16)
    CUtensorMap s0, s1, s2, s3;
};
// Small batches (R <= kSmallRows): one-CTA bookkeeping and gathered x rows.
constexpr int kSmallRows = 32;
constexpr int kMaxExperts = 1024;
cudaError_t launch_route(const RouteArgs&, int num_sms, cudaStream_t);
cudaError_t route_tc_set_attributes();
cudaError_t launch_route_tc(const RouteTcArgs&, const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                            int num_sms, cudaStream_t);
int route_tc_parts(int R, int E, int H, int64_t cap_rows, int num_sms);
cudaError_t launch_coreset(const CoresetArgs&, cudaStream_t);
cudaError_t launch_scatter(const ScatterArgs&, bool small, int num_sms, cudaStream_t);
// after_pair_down: the down GEMM before it ran on CTA pairs (k_down_pair)
cudaError_t launch_combine(const CombineArgs&, int num_sms, bool after_pair_down, cudaStream_t);
cudaError_t gemm_set_attributes();
cudaError_t launch_gemm(int mode, bool small, int qbits, const GemmMaps&, const GemmArgs&,
                        int grid, cudaStream_t);
// Gate/up of units of up to kLargeNGU rows on CTA pairs (gemm_pair.cu).
cudaError_t gateup_pair_set_attributes(int num_sms);
cudaError_t launch_gateup_pair(const GemmMaps&, const GemmArgs&, cudaStream_t);
// Down GEMM of units of up to kLargeNDown pairs x 256 hidden outputs on CTA
// pairs (gemm_pair.cu).
cudaError_t down_pair_set_attributes(int num_sms);
cudaError_t launch_down_pair(const GemmMaps&, const GemmArgs&, cudaStream_t);

enum { kGateUp = 0, kDown = 1 };

// Read-only view of a plan for entry points outside api.cu, and the setter of
// the thread's last-error message (both implemented in api.cu).
struct PlanView {
    moe_dims d;
    int device;
    int num_sms;
    const void* w_router;
};
bool plan_view(const moe_plan* plan, PlanView* out);
moe_status set_error(moe_status s, const char* msg);

}  // namespace moe
