// The front end of a small call (R <= 32 rows) in one launch: router logits,
// top-k and weights, the block coreset and the forward's bookkeeping.
//
// Model card "Clover-35B-A3B-Preview -- CMF", Hardware: every denoising pass
// runs as one GPU submission.  For a 32-row block the three steps before the
// expert GEMMs move about 1.2 MB (the router and the block's rows): their time
// is latency, and as three kernels it was three launches' worth of it, each
// waiting for the one before to finish.  Here:
//
//   1. every CTA computes logits of one row for four experts per warp (the
//      1 MiB router GEMV spread over the SMs, as in the small-batch router);
//   2. a CTA ticket elects the last CTA to finish; it alone carries on, with
//      every CTA's logits in L2: top-k and weights of each row (a warp per
//      row), the coreset of each block, then the pair lists and the GEMMs'
//      unit lists -- the same device code as the standalone kernels, so the
//      outputs are the same bits.
//
// Nothing waits on another CTA: the ticket is a counter that only the last
// arrival acts on.  The ticket must be zero at launch (the host clears it on
// the stream first).
#include "coreset_dev.cuh"
#include "route_common.cuh"
#include "scatter_dev.cuh"

namespace moe {

constexpr int kFrontThreads = kSmallThreads;   // the scatter's CTA size

__global__ void __launch_bounds__(kFrontThreads, 1) k_front(FrontArgs f) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    union FrontSmem {
        CoresetSmem c;
        ScatterSmallSmem s;
    };
    __shared__ FrontSmem sm;
    __shared__ int s_last;
    const RouteArgs& ra = f.r;
    const int lane = threadIdx.x & 31;
    // ---- 1. logits: one warp per (row, four experts)
    {
        const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
        const int nwarps = (gridDim.x * blockDim.x) >> 5;
        const int n_eg = (ra.E + kSmET - 1) / kSmET;
        const int ntasks = ra.R * n_eg;
        for (int t = warp; t < ntasks; t += nwarps) {
            const int row = t / n_eg;
            route_logits_1x4(ra, row, t - row * n_eg, lane);
        }
    }
    __threadfence();   // this thread's logits are visible before the CTA's ticket
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(f.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // ---- 2. the last CTA: top-k and weights, warp w taking rows w, w + 16, ...
    for (int r = threadIdx.x >> 5; r < ra.R; r += blockDim.x >> 5) route_topk(ra, r, r + 1, lane);
    __syncthreads();   // the CTA's topk_idx / topk_w (/ topk_p) writes are visible to it
    for (int b = 0; b < f.c.nb; ++b) coreset_block(f.c, b, sm.c, false);
    __syncthreads();   // keep / w_renorm written; the shared memory is reused below
    scatter_small(f.s, sm.s);
}

cudaError_t launch_front(const FrontArgs& f, int num_sms, cudaStream_t st) {
    const long tasks = (long)f.r.R * ((f.r.E + kSmET - 1) / kSmET);
    long grid = (tasks + kFrontThreads / 32 - 1) / (kFrontThreads / 32);
    if (grid > num_sms) grid = num_sms;
    if (grid < 1) grid = 1;
    return launch_kernel(k_front, dim3((unsigned)grid), dim3(kFrontThreads), 0, st, f);
}

}  // namespace moe
