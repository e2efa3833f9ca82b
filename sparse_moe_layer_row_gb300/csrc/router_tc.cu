// Router, large-batch path: tensor-core screening, then the exact logits of
// the few experts that can still be in a row's top-k.
//
// The result is bit-identical to the SIMT path (route_common.cuh states the
// arithmetic).  The approximate logits only decide which experts are worth
// computing exactly:
//
//   z~[r,e] = tcgen05 bf16 MMA with fp32 accumulation (+ bias), and
//   |z~ - z| <= beta(r,e) = (H * 2^-21) * |x_r|_2 * |w_e|_2 (+ a rounding slack)
//
// where z is the exact-order contract logit.  The bound is a conservative
// assumption about the tensor core (products exact, fp32-class accumulation:
// the worst case of K/16 accumulation steps, each off by a few units in the
// last place of a partial sum no larger than sum|x w| <= |x| |w|, is below it
// by a wide margin); the parity tests against the CPU oracle check it.
// With T the k-th largest z~ of the row and bmax = max_e beta(r,e), every
// expert of the exact top-k satisfies z~ + beta >= T - bmax, and every expert
// failing that test has z < the k-th largest z, so the exact top-k is the
// top-k of the candidates.  Rows with more than kCandCap candidates (or with
// fewer than k comparable logits) are recomputed over all experts.
//
// Kernels: k_route_norms (|x_r| and |w_e|), k_route_tc (persistent; TMA ->
// tcgen05 -> TMEM, one 128-row tile per unit, all E <= 256 experts as the MMA
// N extent; epilogue thread = one row: k-th value and candidate list) and
// k_route_exact (one warp per row: candidates 16 at a time in the contract
// order, top-k, softmax).
#include "route_common.cuh"

namespace moe {

namespace {

constexpr int kTcStages = 4;
constexpr int kTcKMax = 16;
constexpr uint64_t kTcWaitNs = 2000000000ull;
constexpr uint64_t kTcDrainNs = 200000000ull;

struct TcCfg {
    static constexpr int kABytes = 128 * 128;
    static constexpr int kBBytes = 256 * 128;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kWnOff = kTcStages * kStageBytes;   // fp32 |w_e| (256)
    static constexpr int kBarOff = kWnOff + 256 * 4;
    static constexpr int kSmem = kBarOff + 256 + 1024;
};

__device__ __forceinline__ float slack(float z) { return fabsf(z) * 0x1p-20f + 0x1p-100f; }

}  // namespace

__global__ void __launch_bounds__(256) k_route_norms(RouteTcArgs a) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int v = warp; v < a.R + a.E; v += nwarps) {
        const __nv_bfloat16* p = v < a.R ? a.x + (size_t)v * a.H : a.wr + (size_t)(v - a.R) * a.H;
        float s = 0.0f;
        for (int c = lane * 8; c < a.H; c += 256) {
            float f[8];
            bf16x8(__ldg(reinterpret_cast<const uint4*>(p + c)), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) s = fmaf(f[i], f[i], s);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
            const float nrm = sqrtf(s) * 1.001f;  // covers the rounding of the sum
            if (v < a.R) a.xnorm[v] = nrm; else a.wnorm[v - a.R] = nrm;
        }
    }
}

__global__ void __launch_bounds__(192, 1)
k_route_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
           RouteTcArgs a) {
    using C = TcCfg;
    extern __shared__ uint8_t smem_raw[];
    const int ntiles = (a.R + 127) / 128;
    if ((int)blockIdx.x >= ntiles) return;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw);
    float* sw = reinterpret_cast<float*>(base + C::kWnOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kBarOff);
    uint64_t* empty = full + kTcStages;
    uint64_t* tfull = empty + kTcStages;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;

    for (int e = threadIdx.x; e < E; e += blockDim.x) sw[e] = __ldg(a.wnorm + e);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(tfull + i, 1); mbar_init(tempty + i, 128); }
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto give_up = [&]() {
        if (!*abort_flag) { *abort_flag = 1; status_add(a.status, MOE_STATUS_WAIT_TIMEOUT, 1); }
    };
    const int nkb = a.H >> 6;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t bytes = (uint32_t)(C::kABytes + E * 128);
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, abort_flag, kTcWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full + stage, bytes);
                    const uint32_t sA = sbase + stage * C::kStageBytes;
                    tma_load_2d(sA, &tm_x, kb * 64, t * 128, full + stage);
                    tma_load_2d(sA + C::kABytes, &tm_w, kb * 64, 0, full + stage);
                    if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
                }
            }
            for (int i = 0; i < kTcStages; ++i) {
                const uint64_t lim = *abort_flag ? kTcDrainNs : kTcWaitNs;
                if (!mbar_wait_bounded(empty + stage, phase ^ 1u, never, lim)) { give_up(); break; }
                if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16_f32(128, E);
            for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
                if (!mbar_wait_bounded(tempty + acc, acc_phase ^ 1u, abort_flag, kTcWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * 256);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(full + stage, phase, abort_flag, kTcWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = sbase + stage * C::kStageBytes;
                    const uint32_t sB = sA + C::kABytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(d, smem_desc_sw128(sA + kk * 32), smem_desc_sw128(sB + kk * 32),
                                    idesc, (kb | kk) != 0);
                    tc_commit(empty + stage);
                    if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(tfull + acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else {
        // epilogue: thread = row
        const int q = warp & 3;
        float wmax = 0.0f;
        for (int e = 0; e < E; ++e) wmax = fmaxf(wmax, sw[e]);
        const float G = (float)a.H * 0x1p-21f;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const bool okw = mbar_wait_bounded(tfull + acc, acc_phase, abort_flag, kTcWaitNs);
            if (__any_sync(0xffffffffu, !okw)) { give_up(); break; }
            __syncwarp();
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256);
            const int row = t * 128 + q * 32 + lane;
            const bool valid = row < a.R;
            const float* brow =
                (valid && a.bias) ? a.bias + (size_t)find_block(a.off, a.nb, row) * E : nullptr;
            const float xn = valid ? __ldg(a.xnorm + row) : 0.0f;
            const float gx = G * xn;
            // pass 1: the k-th largest approximate logit (NaN never enters)
            float top[kTcKMax];
#pragma unroll
            for (int i = 0; i < kTcKMax; ++i) top[i] = -INFINITY;
            float kth = -INFINITY;
            uint32_t nonfinite = 0;
            for (int c = 0; c < E; c += 16) {
                float v[16];
                __syncwarp();
                tmem_ld16(tb + (uint32_t)c, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float z = v[i];
                    if (brow) z = __fadd_rn(z, __ldg(brow + c + i));
                    nonfinite += !isfinite(z);
                    if (z > kth) {
                        // insert into the descending list top[0..k-1]
#pragma unroll
                        for (int j = kTcKMax - 1; j >= 0; --j) {
                            const float above = j > 0 ? top[j > 0 ? j - 1 : 0] : INFINITY;
                            if (j < a.k && z > top[j]) top[j] = z > above ? above : z;
                        }
#pragma unroll
                        for (int j = 0; j < kTcKMax; ++j)
                            if (j == a.k - 1) kth = top[j];
                    }
                }
            }
            const float T = kth;
            const float thr = T - (gx * wmax + slack(T));
            // pass 2: candidates in increasing expert order
            int cnt = 0;
            int32_t* cl = a.cand + (size_t)(valid ? row : 0) * kCandCap;
            for (int c = 0; c < E; c += 16) {
                float v[16];
                __syncwarp();
                tmem_ld16(tb + (uint32_t)c, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float z = v[i];
                    if (brow) z = __fadd_rn(z, __ldg(brow + c + i));
                    if (z + (gx * sw[c + i] + slack(z)) >= thr) {
                        if (valid && cnt < kCandCap) cl[cnt] = c + i;
                        ++cnt;
                    }
                }
            }
            if (valid) {
                const bool full_row = !(T > -INFINITY) || cnt > kCandCap || cnt < a.k;
                a.cand_cnt[row] = full_row ? -1 : cnt;
            }
            nonfinite = __reduce_add_sync(0xffffffffu, valid ? nonfinite : 0u);
            if (lane == 0) status_add(a.status, MOE_STATUS_NONFINITE_LOGITS, nonfinite);
            tc_fence_before();
            mbar_arrive(tempty + acc);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// One warp per row: exact logits of the candidates, 16 at a time, in the
// contract order; then top-k and softmax.
__global__ void __launch_bounds__(256) k_route_exact(RouteTcArgs a) {
    constexpr int NG = 16;  // groups of 16 candidates: up to 256 experts
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int r = warp; r < a.R; r += nwarps) {
        const int cc = __ldg(a.cand_cnt + r);
        const bool full_row = cc < 0;
        const int n = full_row ? a.E : cc;
        const int32_t* cl = a.cand + (size_t)r * kCandCap;
        const float* brow = a.bias ? a.bias + (size_t)find_block(a.off, a.nb, r) * a.E : nullptr;
        const __nv_bfloat16* xr = a.x + (size_t)r * a.H;
        uint32_t key[NG], id[NG];
        uint32_t valid = 0;
#pragma unroll
        for (int g = 0; g < NG; ++g) { key[g] = 0; id[g] = 0xFFFFFFFFu; }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            if (g * 16 >= n) break;
            int ex[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int ci = g * 16 + i;
                ex[i] = ci < n ? (full_row ? ci : __ldg(cl + ci)) : -1;
            }
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
            for (int s = 0; s < a.H; s += 256) {
                const int col = s + lane * 8;
                float xf[8];
                bf16x8(__ldg(reinterpret_cast<const uint4*>(xr + col)), xf);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float wf[8];
                    const uint4 wv = ex[i] >= 0
                        ? __ldg(reinterpret_cast<const uint4*>(a.wr + (size_t)ex[i] * a.H + col))
                        : make_uint4(0, 0, 0, 0);
                    bf16x8(wv, wf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i] = __fmaf_rn(xf[j], wf[j], acc[i]);
                }
            }
            // transposed halving over partner distances 16, 8, 4, 2 (16 -> 1
            // accumulators), then a plain butterfly step at distance 1: the
            // same pairs as the contract's butterfly.
#pragma unroll
            for (int o = 16, h = 8; o >= 2; o >>= 1, h >>= 1) {
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < h; ++i) {
                    const float send = upper ? acc[i] : acc[i + h];
                    const float keep = upper ? acc[i + h] : acc[i];
                    acc[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
                }
            }
            const float other = __shfl_xor_sync(0xffffffffu, acc[0], 1);
            const float dot = __fadd_rn(acc[0], other);
            // lane 2i (and 2i+1) now hold candidate g*16 + i
            const int ci = lane >> 1;
            int e = -1;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i == ci) e = ex[i];
            if ((lane & 1) == 0 && e >= 0) {
                key[g] = order_key(finish_logit(dot, brow, e));
                id[g] = (uint32_t)e;
                valid |= 1u << g;
            }
        }
        uint32_t my_id, my_key;
        warp_topk<NG>(key, id, valid, a.k, lane, my_id, my_key);
        write_topk(a.topk_idx + (size_t)r * a.k, a.topk_w + (size_t)r * a.k, a.k, lane, my_id,
                   my_key);
    }
}

cudaError_t route_tc_set_attributes() {
    return cudaFuncSetAttribute(k_route_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcCfg::kSmem);
}

cudaError_t launch_route_tc(const RouteTcArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                            int num_sms, cudaStream_t st) {
    long nb = (long)(a.R + a.E + 7) / 8;
    if (nb > (long)num_sms * 8) nb = (long)num_sms * 8;
    k_route_norms<<<(unsigned)(nb < 1 ? 1 : nb), 256, 0, st>>>(a);
    const int ntiles = (a.R + 127) / 128;
    const int grid = ntiles < num_sms ? ntiles : num_sms;
    k_route_tc<<<grid, 192, TcCfg::kSmem, st>>>(tm_x, tm_w, a);
    long eb = (long)(a.R + 7) / 8;
    if (eb > (long)num_sms * 16) eb = (long)num_sms * 16;
    k_route_exact<<<(unsigned)(eb < 1 ? 1 : eb), 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
