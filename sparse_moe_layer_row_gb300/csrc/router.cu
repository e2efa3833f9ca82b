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

template <int NE>
__device__ void route_topk_rows(const RouteArgs& a, int r0, int r1, int lane) {
    for (int r = r0; r < r1; ++r) {
        const float* brow = a.bias ? a.bias + (size_t)find_block(a.off, a.nb, r) * a.E : nullptr;
        uint32_t key[NE], id[NE];
        uint32_t valid = 0, nonfinite = 0;
#pragma unroll
        for (int i = 0; i < NE; ++i) {
            const int e = lane + 32 * i;
            id[i] = (uint32_t)e;
            key[i] = 0;
            if (e < a.E) {
                const float z = finish_logit(__ldcg(a.logits + (size_t)r * a.E + e), brow, e);
                if (!isfinite(z)) ++nonfinite;
                key[i] = order_key(z);
                valid |= 1u << i;
            }
        }
        nonfinite = __reduce_add_sync(0xffffffffu, nonfinite);
        if (lane == 0) status_add(a.status, MOE_STATUS_NONFINITE_LOGITS, nonfinite);
        uint32_t my_id, my_key;
        warp_topk<NE>(key, id, valid, a.k, lane, my_id, my_key);
        write_topk(a.topk_idx + (size_t)r * a.k, a.topk_w + (size_t)r * a.k, a.k, lane, my_id,
                   my_key);
        if (a.topk_p) write_topk_probs<NE>(a.topk_p + (size_t)r * a.k, a.k, lane, key, valid, my_key);
    }
}

__device__ void route_topk(const RouteArgs& a, int r0, int r1, int lane) {
    const int ne = (a.E + 31) >> 5;
    if (ne <= 1) route_topk_rows<1>(a, r0, r1, lane);
    else if (ne <= 2) route_topk_rows<2>(a, r0, r1, lane);
    else if (ne <= 4) route_topk_rows<4>(a, r0, r1, lane);
    else if (ne <= 8) route_topk_rows<8>(a, r0, r1, lane);
    else if (ne <= 16) route_topk_rows<16>(a, r0, r1, lane);
    else route_topk_rows<32>(a, r0, r1, lane);
}

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
constexpr int kSmET = 4;
constexpr int kSmPD = 4;   // stripes held in registers at a time

__device__ __forceinline__ void prefetch_l1_line(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

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
        const __nv_bfloat16* xr = a.x + (size_t)row * a.H;
        // L1 prefetch of stripes kSmPD.. of x and the four router rows: one
        // 128-byte line per lane and step (a stripe of a row is 4 lines)
        for (int l = lane; (kSmPD + l / 20) * 256 < a.H; l += 32) {
            const int st = kSmPD + l / 20, r5 = (l % 20) >> 2, q = l & 3;
            const int ex = eg * kSmET + r5 - 1;
            const __nv_bfloat16* base = r5 == 0 ? xr : a.wr + (size_t)(ex < a.E ? ex : 0) * a.H;
            prefetch_l1_line(base + st * 256 + q * 64);
        }
        float acc[kSmET];
#pragma unroll
        for (int i = 0; i < kSmET; ++i) acc[i] = 0.0f;
        for (int s0 = 0; s0 < a.H; s0 += kSmPD * 256) {
            uint4 xv[kSmPD], wv[kSmPD][kSmET];
#pragma unroll
            for (int si = 0; si < kSmPD; ++si) {
                const int col = s0 + si * 256 + lane * 8;
                const bool in = col < a.H;
                xv[si] = in ? __ldg(reinterpret_cast<const uint4*>(xr + col)) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int e = 0; e < kSmET; ++e) {
                    const int ex = eg * kSmET + e;
                    wv[si][e] = (in && ex < a.E)
                        ? __ldg(reinterpret_cast<const uint4*>(a.wr + (size_t)ex * a.H + col))
                        : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int si = 0; si < kSmPD; ++si) {
                if (s0 + si * 256 >= a.H) break;
#pragma unroll
                for (int e = 0; e < kSmET; ++e) acc[e] = dot8_bf16(xv[si], wv[si][e], acc[e]);
            }
        }
        // halving at partner distances 16 and 8 (4 -> 1 accumulators), then
        // plain butterfly steps at 4, 2, 1; lane holds expert (lane >> 3) & 3
#pragma unroll
        for (int o = 16, h = 2; o >= 8; o >>= 1, h >>= 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < h; ++i) {
                const float send = upper ? acc[i] : acc[i + h];
                const float keep = upper ? acc[i + h] : acc[i];
                acc[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
            }
        }
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) acc[0] = __fadd_rn(acc[0], __shfl_xor_sync(0xffffffffu, acc[0], o));
        {
            const int ex = eg * kSmET + ((lane >> 3) & 3);
            if ((lane & 7) == 0 && ex < a.E) a.logits[(size_t)row * a.E + ex] = acc[0];
        }
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
