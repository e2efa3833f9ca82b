// Router, SIMT path (small batches): logits in the fixed lane/stripe order,
// then top-k and softmax weights for every row.  The arithmetic is described
// in route_common.cuh (model card "Clover-35B-A3B-Preview -- CMF", intro:
// top-8 of 256 experts).
//
// Medium batches: one warp computes a 4-row x 8-expert tile of logits: 32 accumulators per
// lane, the stripes' loads double-buffered in registers.  The 32 lane sums of
// the 32 accumulators are reduced with a transposed butterfly (each step keeps
// half of the accumulators and trades the other half with the partner lane),
// which adds exactly the same pairs as the plain butterfly, so lane i ends
// with the finished sum of accumulator i.  The warp that finishes the last
// expert tile of a row group (ticket counter) runs top-k and softmax for
// those rows.  CTAs are one to eight warps, so that small batches spread over
// every SM.
#include "route_common.cuh"

namespace moe {

constexpr int kRT = 4;   // rows per warp tile
constexpr int kET = 8;   // experts per warp tile

struct Stripe {
    uint4 x[kRT];
    uint4 w[kET];
};

__device__ __forceinline__ void load_stripe(Stripe& s, const RouteArgs& a, int rg, int eg, int col) {
#pragma unroll
    for (int r = 0; r < kRT; ++r) {
        const int row = rg * kRT + r;
        s.x[r] = row < a.R ? __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)row * a.H + col))
                           : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int e = 0; e < kET; ++e) {
        const int ex = eg * kET + e;
        s.w[e] = ex < a.E ? __ldg(reinterpret_cast<const uint4*>(a.wr + (size_t)ex * a.H + col))
                          : make_uint4(0, 0, 0, 0);
    }
}

__global__ void __launch_bounds__(256, 1) k_route(RouteArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int n_rg = (a.R + kRT - 1) / kRT;
    const int n_eg = (a.E + kET - 1) / kET;
    const int ntasks = n_rg * n_eg;
    for (int t = warp; t < ntasks; t += nwarps) {
        const int rg = t / n_eg, eg = t - rg * n_eg;
        float acc[kRT * kET];
#pragma unroll
        for (int i = 0; i < kRT * kET; ++i) acc[i] = 0.0f;
        Stripe cur;
        load_stripe(cur, a, rg, eg, lane * 8);
        for (int s = 0; s < a.H; s += 256) {
            Stripe nxt = cur;
            if (s + 256 < a.H) load_stripe(nxt, a, rg, eg, s + 256 + lane * 8);
#pragma unroll
            for (int e = 0; e < kET; ++e)
#pragma unroll
                for (int r = 0; r < kRT; ++r) acc[r * kET + e] = dot8_bf16(cur.x[r], cur.w[e], acc[r * kET + e]);
            cur = nxt;
        }
        // transposed butterfly: after the step with partner distance o, lane
        // keeps the half of its accumulators whose index bit (o) equals its own.
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < o; ++i) {
                const float send = upper ? acc[i] : acc[i + o];
                const float keep = upper ? acc[i + o] : acc[i];
                const float recv = __shfl_xor_sync(0xffffffffu, send, o);
                acc[i] = __fadd_rn(keep, recv);
            }
        }
        {
            const int row = rg * kRT + (lane >> 3);
            const int ex = eg * kET + (lane & 7);
            if (row < a.R && ex < a.E) a.logits[(size_t)row * a.E + ex] = acc[0];
        }
        __syncwarp();
        __threadfence();
        uint32_t old = 0;
        if (lane == 0) old = atomicAdd(a.cnt + rg, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == (uint32_t)(n_eg - 1)) {
            __threadfence();
            if (lane == 0) a.cnt[rg] = 0u;  // ready for the next call
            const int r0 = rg * kRT;
            route_topk(a, r0, min(a.R, r0 + kRT), lane);
        }
    }
}

// Small batches: one warp computes 1 row x 4 experts.  Its stripes' loads are
// issued four stripes at a time (registers), and every later stripe of the
// row is prefetched into L1 first, so the warp pays about one memory round
// trip; two CTAs per SM put a 32-row call in one wave.  The four accumulators
// are reduced by two transposed halving steps and three plain butterfly steps
// (the same pairs as the contract's butterfly); a ticket per row lets the
// warp finishing a row run its top-k.
constexpr int kSmallRouteRows = 64;

__global__ void __launch_bounds__(256, 2) k_route_small(RouteArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int n_eg = (a.E + kSmET - 1) / kSmET;
    const int ntasks = a.R * n_eg;
    for (int t = warp; t < ntasks; t += nwarps) {
        const int row = t / n_eg, eg = t - row * n_eg;
        route_logits_1x4(a, row, eg, lane);
        __syncwarp();
        __threadfence();
        uint32_t old = 0;
        if (lane == 0) old = atomicAdd(a.cnt + row, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == (uint32_t)(n_eg - 1)) {
            __threadfence();
            if (lane == 0) a.cnt[row] = 0u;  // ready for the next call
            route_topk(a, row, row + 1, lane);
        }
    }
}

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st) {
    if (a.R <= kSmallRouteRows) {
        const long tasks = (long)a.R * ((a.E + kSmET - 1) / kSmET);
        long blocks = (tasks + 7) / 8;  // 8 warps per CTA
        if (blocks < 1) blocks = 1;
        return launch_kernel(k_route_small, dim3((unsigned)blocks), dim3(256), 0, st, a);
    }
    const int n_rg = (a.R + kRT - 1) / kRT;
    const int n_eg = (a.E + kET - 1) / kET;
    const long tasks = (long)n_rg * n_eg;
    // warps per CTA: enough CTAs to reach every SM first, then up to 8 warps
    long wpc = tasks / num_sms;
    wpc = wpc < 1 ? 1 : (wpc > 8 ? 8 : wpc);
    long blocks = (tasks + wpc - 1) / wpc;
    const long cap = (long)num_sms * (32 / wpc);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_kernel(k_route, dim3((unsigned)blocks), dim3((unsigned)(32 * wpc)), 0, st, a);
}

}  // namespace moe
