// Router: logits, top-k and softmax weights for every row.
//
// Model card "Clover-35B-A3B-Preview -- CMF", intro: each row is routed to the
// top 8 of 256 experts.  The arithmetic is fixed so that top-k ids are
// reproducible bit for bit on any device:
//   * z[r,e] = sum_h x[r,h] W[e,h] in fp32.  Each bf16*bf16 product is exact in
//     fp32, so an fma adding it equals the add of the rounded product.  h is
//     cut into stripes of 256; lane p of a warp owns elements 8p..8p+7 of every
//     stripe and accumulates them in ascending h; the 32 lane sums are combined
//     in the xor-butterfly pattern (partner distance 16, 8, 4, 2, 1).
//   * z += bias[b,e] (optional), then z += 0 (turns -0 into +0).
//   * top-k by (z descending, id ascending), NaN below every number.
//   * w_j = a_j / (a_0 + ... + a_{k-1}) with a_j = exp_c(z_j - z_0), summed in
//     rank order; exp_c is a Cody-Waite range reduction (ln 2 split into a
//     12-significant-bit head 2839/4096 and an fp32 tail) followed by the
//     degree-7 Taylor polynomial of e^r in Horner form with fused multiply-adds
//     and a final scaling by 2^n through the exponent field.
//
// One warp computes a 4-row x 8-expert tile of logits: 32 accumulators per
// lane.  The 32 lane sums of the 32 accumulators are reduced with a
// transposed butterfly (each step keeps half of the accumulators and trades
// the other half with the partner lane), which adds exactly the same pairs as
// the plain butterfly, so lane i ends with the finished sum of accumulator i.
// The warp that finishes the last expert tile of a row group (ticket counter)
// runs the top-k and softmax for those rows.
#include "kernels.cuh"

namespace moe {

constexpr int kRT = 4;   // rows per warp tile
constexpr int kET = 8;   // experts per warp tile

// e^t for t <= 0 (see the file comment).
__device__ __forceinline__ float exp_c(float t) {
    const float kLog2e = 1.44269504088896341f;
    const float kLn2Hi = 0.693115234375f;                                   // 2839 / 4096
    const float kLn2Lo = (float)(0.69314718055994530942 - 0.693115234375);  // ln 2 - head
    if (t != t) return 0.0f;
    if (t < -87.0f) return 0.0f;
    const float n = rintf(__fmul_rn(t, kLog2e));
    float r = __fmaf_rn(-n, kLn2Hi, t);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = (float)(1.0 / 5040.0);
    p = __fmaf_rn(p, r, (float)(1.0 / 720.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 120.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 24.0));
    p = __fmaf_rn(p, r, (float)(1.0 / 6.0));
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ni = (int)n;
    return __fmul_rn(p, __uint_as_float((uint32_t)(ni + 127) << 23));
}

// Order-preserving key: larger float -> larger key; NaN -> 0.
__device__ __forceinline__ uint32_t order_key(float f) {
    if (f != f) return 0u;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ void bf16x8(uint4 v, float* f) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
    uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, o);
    uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), o);
    return ((uint64_t)hi << 32) | lo;
}

// Top-k and weights of rows [r0, r1) by one warp.
__device__ void route_topk(const RouteArgs& a, int r0, int r1, int lane) {
    const int ne = (a.E + 31) >> 5;
    for (int r = r0; r < r1; ++r) {
        const int b = a.bias ? find_block(a.off, a.nb, r) : 0;
        uint32_t key[32];
        uint32_t taken = 0;
        uint32_t nonfinite = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            key[i] = 0;
            const int e = lane + 32 * i;
            if (i < ne && e < a.E) {
                float z = __ldcg(a.logits + (size_t)r * a.E + e);
                if (a.bias) z = __fadd_rn(z, __ldg(a.bias + (size_t)b * a.E + e));
                z = __fadd_rn(z, 0.0f);
                if (!isfinite(z)) ++nonfinite;
                key[i] = order_key(z);
            } else {
                taken |= 1u << i;
            }
        }
        int my_e = 0;
        uint32_t my_key = 0;
        for (int j = 0; j < a.k; ++j) {
            uint64_t best = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (!((taken >> i) & 1u)) {
                    const uint64_t p = ((uint64_t)key[i] << 32) | (uint32_t)(~(uint32_t)(lane + 32 * i));
                    best = p > best ? p : best;
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const uint64_t other = shfl_xor_u64(best, o);
                best = other > best ? other : best;
            }
            const uint32_t e_win = ~(uint32_t)best;
            if (lane == (int)(e_win & 31u)) taken |= 1u << (e_win >> 5);
            if (lane == j) { my_e = (int)e_win; my_key = (uint32_t)(best >> 32); }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) nonfinite += __shfl_xor_sync(0xffffffffu, nonfinite, o);
        if (lane == 0) status_add(a.status, MOE_STATUS_NONFINITE_LOGITS, nonfinite);
        const float zj = key_value(my_key);
        const float m = __shfl_sync(0xffffffffu, zj, 0);
        const float aj = lane < a.k ? exp_c(__fsub_rn(zj, m)) : 0.0f;
        float S = 0.0f;
        for (int j = 0; j < a.k; ++j) S = __fadd_rn(S, __shfl_sync(0xffffffffu, aj, j));
        if (lane < a.k) {
            a.topk_idx[(size_t)r * a.k + lane] = my_e;
            a.topk_w[(size_t)r * a.k + lane] = __fdiv_rn(aj, S);
        }
    }
}

__global__ void __launch_bounds__(256) k_route(RouteArgs a) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int n_rg = (a.R + kRT - 1) / kRT;
    const int n_eg = (a.E + kET - 1) / kET;
    const int ntasks = n_rg * n_eg;
    const int H = a.H;
    for (int t = warp; t < ntasks; t += nwarps) {
        const int rg = t / n_eg, eg = t - rg * n_eg;
        float acc[kRT * kET];
#pragma unroll
        for (int i = 0; i < kRT * kET; ++i) acc[i] = 0.0f;
        for (int s = 0; s < H; s += 256) {
            const int col = s + lane * 8;
            float xf[kRT][8];
#pragma unroll
            for (int r = 0; r < kRT; ++r) {
                const int row = rg * kRT + r;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (row < a.R) v = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)row * H + col));
                bf16x8(v, xf[r]);
            }
#pragma unroll
            for (int e = 0; e < kET; ++e) {
                const int ex = eg * kET + e;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (ex < a.E) v = __ldg(reinterpret_cast<const uint4*>(a.wr + (size_t)ex * H + col));
                float wf[8];
                bf16x8(v, wf);
#pragma unroll
                for (int r = 0; r < kRT; ++r)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        acc[r * kET + e] = __fmaf_rn(xf[r][q], wf[q], acc[r * kET + e]);
            }
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
            const int r1 = min(a.R, r0 + kRT);
            route_topk(a, r0, r1, lane);
        }
    }
}

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st) {
    const int n_rg = (a.R + kRT - 1) / kRT;
    const int n_eg = (a.E + kET - 1) / kET;
    const long tasks = (long)n_rg * n_eg;
    long blocks = (tasks + 7) / 8;
    const long cap = (long)num_sms * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_route<<<(unsigned)blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
