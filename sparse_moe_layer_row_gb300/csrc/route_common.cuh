// Pieces of the routing arithmetic shared by the two router paths (router.cu:
// fixed-order SIMT logits for small batches; router_tc.cu: tensor-core
// screening + exact recompute of the candidates for large batches).  Both
// paths produce bit-identical logits, top-k ids and weights.
//
// Model card "Clover-35B-A3B-Preview -- CMF", intro: each row is routed to the
// top 8 of 256 experts.  The arithmetic (fixed so that ids are reproducible):
//   * z[r,e] = sum_h x[r,h] W[e,h] in fp32.  Each bf16*bf16 product is exact in
//     fp32, so an fma adding it equals the add of the rounded product (and the
//     mixed-precision fma.rn.f32.bf16, which takes the bf16 operands as they
//     are, gives the same bits as an fp32 fma of the widened operands).  h is
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
//   * on request, p_j = a_j / D, the selected experts' probabilities under the
//     softmax over all E experts (the probability-mass reading of "90% of its
//     routing", InfiniLM PR #604, Summary): D = sum over every expert e of
//     exp_c(z_e - z_0), lane p adding the experts p, p + 32, ... in ascending
//     e, the 32 lane sums combined by the same xor butterfly as the logits.
#pragma once

#include "kernels.cuh"

namespace moe {

// e^t for t <= 0 (see above).
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

// acc = fma(x_j, w_j, acc) for the eight bf16 pairs of (x, w), j ascending
// (element 2i is the low half of word i).
__device__ __forceinline__ float fma_bf16x2(uint32_t x, uint32_t w, float acc) {
    asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %1;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
        "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
        : "+f"(acc)
        : "r"(x), "r"(w));
    return acc;
}

__device__ __forceinline__ float dot8_bf16(uint4 x, uint4 w, float acc) {
    acc = fma_bf16x2(x.x, w.x, acc);
    acc = fma_bf16x2(x.y, w.y, acc);
    acc = fma_bf16x2(x.z, w.z, acc);
    return fma_bf16x2(x.w, w.w, acc);
}

// z -> z + bias, + 0, as the contract states (the bias value already loaded).
__device__ __forceinline__ float finish_logit_v(float dot, bool has_bias, float bias) {
    float z = dot;
    if (has_bias) z = __fadd_rn(z, bias);
    return __fadd_rn(z, 0.0f);
}

__device__ __forceinline__ float finish_logit(float dot, const float* bias_row, int e) {
    return finish_logit_v(dot, bias_row != nullptr, bias_row ? __ldg(bias_row + e) : 0.0f);
}

// In-lane bitonic sort of NI (a power of two) 64-bit values, descending.
template <int NI>
__device__ __forceinline__ void lane_sort_desc(unsigned long long (&c)[NI]) {
#pragma unroll
    for (int size = 2; size <= NI; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool desc = (i & size) == 0;
                    const unsigned long long a = c[i], b = c[j];
                    const bool sw = desc ? a < b : a > b;
                    c[i] = sw ? b : a;
                    c[j] = sw ? a : b;
                }
            }
}

// Warp top-k over entries spread across lanes: lane entry i holds (key[i],
// id[i]) when bit i of `valid` is set.  Order: key descending, id ascending.
// Lane j < k receives the j-th entry in my_id / my_key.  k must not exceed
// the number of valid entries in the warp.  Each entry becomes one 64-bit
// value (key, ~id) -- larger means earlier in the order, 0 for an invalid
// entry (a valid one is never 0: ids are below 2^31) -- each lane sorts its
// own values, and every round the warp takes the largest lane head (the key
// by one reduction, the id among the lanes holding that key by another) and
// that lane drops its head.  No divergent branch.
template <int NI>
__device__ __forceinline__ void warp_topk(const uint32_t (&key)[NI], const uint32_t (&id)[NI],
                                          uint32_t valid, int k, int lane, uint32_t& my_id,
                                          uint32_t& my_key) {
    unsigned long long c[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i)
        c[i] = ((valid >> i) & 1u) ? ((unsigned long long)key[i] << 32 | (uint32_t)~id[i]) : 0ull;
    lane_sort_desc<NI>(c);
    my_id = 0;
    my_key = 0;
    for (int j = 0; j < k; ++j) {
        const uint32_t hk = (uint32_t)(c[0] >> 32), hl = (uint32_t)c[0];
        const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t ml = __reduce_max_sync(0xffffffffu, hk == mk ? hl : 0u);
        const bool win = c[0] != 0ull && hk == mk && hl == ml;
#pragma unroll
        for (int i = 0; i + 1 < NI; ++i) c[i] = win ? c[i + 1] : c[i];
        c[NI - 1] = win ? 0ull : c[NI - 1];
        if (lane == j) {
            my_id = ~ml;
            my_key = mk;
        }
    }
}

// Softmax over the k selected logits (lane j < k holds rank j) and the store.
__device__ __forceinline__ void write_topk(int32_t* idx_out, float* w_out, int k, int lane,
                                           uint32_t my_id, uint32_t my_key) {
    const float zj = key_value(my_key);
    const float m = __shfl_sync(0xffffffffu, zj, 0);
    const float aj = lane < k ? exp_c(__fsub_rn(zj, m)) : 0.0f;
    float S = 0.0f;
    for (int j = 0; j < k; ++j) S = __fadd_rn(S, __shfl_sync(0xffffffffu, aj, j));
    if (lane < k) {
        idx_out[lane] = (int32_t)my_id;
        w_out[lane] = __fdiv_rn(aj, S);
    }
}

// The probability mass of the selected experts (lane j < k holds rank j):
// p_j = exp_c(z_j - z_0) / D, with D over every expert of the row.  key[i] of
// lane p is the key of expert p + 32 i (bit i of `valid`: the expert exists).
template <int NI>
__device__ __forceinline__ void write_topk_probs(float* p_out, int k, int lane,
                                                 const uint32_t (&key)[NI], uint32_t valid,
                                                 uint32_t my_key) {
    const float m = __shfl_sync(0xffffffffu, key_value(my_key), 0);
    float d = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i)
        if ((valid >> i) & 1u) d = __fadd_rn(d, exp_c(__fsub_rn(key_value(key[i]), m)));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d = __fadd_rn(d, __shfl_xor_sync(0xffffffffu, d, o));
    if (lane < k) p_out[lane] = __fdiv_rn(exp_c(__fsub_rn(key_value(my_key), m)), d);
}

// Top-k and softmax weights (and, on request, probabilities) of rows r0..r1-1
// from their finished logits in a.logits (before the bias); one warp.
template <int NE>
__device__ __forceinline__ void route_topk_rows(const RouteArgs& a, int r0, int r1, int lane) {
    for (int r = r0; r < r1; ++r) {
        const float* brow = a.bias ? a.bias + (size_t)find_block(a.off, a.nb, r) * a.E : nullptr;
        uint32_t key[NE], id[NE];
        uint32_t valid = 0, nonfinite = 0;
        // every load first (one memory round trip), then the keys
        float z[NE], bz[NE];
#pragma unroll
        for (int i = 0; i < NE; ++i) {
            const int e = lane + 32 * i;
            const int ec = e < a.E ? e : 0;
            z[i] = __ldcg(a.logits + (size_t)r * a.E + ec);
            bz[i] = brow ? __ldg(brow + ec) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < NE; ++i) {
            const int e = lane + 32 * i;
            id[i] = (uint32_t)e;
            key[i] = 0;
            if (e < a.E) {
                const float zi = finish_logit_v(z[i], brow != nullptr, bz[i]);
                if (!isfinite(zi)) ++nonfinite;
                key[i] = order_key(zi);
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

__device__ __forceinline__ void route_topk(const RouteArgs& a, int r0, int r1, int lane) {
    const int ne = (a.E + 31) >> 5;
    if (ne <= 1) route_topk_rows<1>(a, r0, r1, lane);
    else if (ne <= 2) route_topk_rows<2>(a, r0, r1, lane);
    else if (ne <= 4) route_topk_rows<4>(a, r0, r1, lane);
    else if (ne <= 8) route_topk_rows<8>(a, r0, r1, lane);
    else if (ne <= 16) route_topk_rows<16>(a, r0, r1, lane);
    else route_topk_rows<32>(a, r0, r1, lane);
}


// Logits of one row for four experts (eg * 4 .. eg * 4 + 3), one warp: its
// stripes' loads are issued four stripes at a time (registers), and every
// later stripe of the row is prefetched into L1 first, so the warp pays about
// one memory round trip.  The four accumulators are reduced by two transposed
// halving steps and three plain butterfly steps (the same pairs as the
// contract's butterfly); the logits go to a.logits (before the bias).
constexpr int kSmET = 4;   // experts per warp task
constexpr int kSmPD = 4;   // stripes held in registers at a time

__device__ __forceinline__ void prefetch_l1_line(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ void route_logits_1x4(const RouteArgs& a, int row, int eg, int lane) {
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
    }}

}  // namespace moe
