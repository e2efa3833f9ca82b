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
// where z is the exact-order contract logit.  The accumulation model the bound
// assumes: each tcgen05.mma (K = 16) adds its 16 products, exact in fp32
// (bf16 x bf16), to the fp32 accumulator with an error of at most four units
// of 2^-23 relative to |accumulator| + sum|products of the slice|, whatever
// its internal order, alignment or truncation.  Both terms are at most
// sum_h |x_h w_h| <= |x| |w| (Cauchy-Schwarz), so H/16 steps err by at most
// (H/16) 2^-21 2 |x||w| = H 2^-24 |x||w|.  When few rows leave SMs idle, the
// screen splits H into nk parts (one CTA each); part p's accumulator errs by
// at most (H/nk) 2^-24 |x_p||w_p|, the parts by (H/nk) 2^-24 |x||w| together
// (Cauchy-Schwarz over the parts), and the nk - 1 fp32 additions of the part
// sums in part order by (nk - 1) 2^-24 |x||w|: H 2^-24 |x||w| still bounds
// it.  The contract's fixed-order fp32 sum is within (H/32 + 5) 2^-24
// sum|x w| of the exact dot product (recursive summation over H/32 terms per
// lane, then five butterfly additions).  So
// |z~ - z| <= (H + H/32 + 5) 2^-24 |x||w| < beta = 8 H 2^-24 |x||w| for every
// H >= 256: beta covers that model about seven times over.  The norms are
// fp32 sums times 1.001, which covers their own rounding.  The model is not
// a documented property of the hardware; the parity tests against the CPU
// oracle, including rows built to put twin experts on the k-th place at gaps
// from 1/100 to 10 times beta, check it.
// With T the k-th largest z~ of the row and bmax = max_e beta(r,e), every
// expert of the exact top-k satisfies z~ + beta >= T - bmax, and every expert
// failing that test has z < the k-th largest z, so the exact top-k is the
// top-k of the candidates.  Rows with more than kCandCap candidates (or with
// fewer than k comparable logits) are recomputed over all experts.
//
// Kernels: k_route_norms (|x_r| and |w_e|), k_route_tc (persistent; TMA ->
// tcgen05 -> TMEM; a unit is a 128-row tile times one part of H times one
// half (or all) of the experts; the epilogue stores the approximate logits,
// one slice per part) and k_route_exact (one warp per row: the parts added,
// the k-th approximate value by warp reductions, the candidate
// list by ballots, then the candidates 16 at a time in the contract order,
// top-k and softmax).
#include "route_common.cuh"

namespace moe {

namespace {

constexpr int kTcStages = 4;
constexpr uint64_t kTcWaitNs = 2000000000ull;
constexpr uint64_t kTcDrainNs = 200000000ull;

struct TcCfg {
    static constexpr int kABytes = 128 * 128;
    static constexpr int kBBytes = 256 * 128;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kBarOff = kTcStages * kStageBytes;
    static constexpr int kSmem = kBarOff + 256 + 1024;
};

__device__ __forceinline__ float slack(float z) { return fabsf(z) * 0x1p-20f + 0x1p-100f; }

__device__ __forceinline__ void prefetch_l1(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

}  // namespace

// |w_e|_2 of every router row (times 1.001, which covers the rounding of the sum).
__global__ void __launch_bounds__(256) k_route_norms(RouteTcArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int e = warp; e < a.E; e += nwarps) {
        const __nv_bfloat16* p = a.wr + (size_t)e * a.H;
        float s = 0.0f;
        for (int c = lane * 8; c < a.H; c += 256) {
            float f[8];
            bf16x8(__ldg(reinterpret_cast<const uint4*>(p + c)), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) s = fmaf(f[i], f[i], s);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) a.wnorm[e] = sqrtf(s) * 1.001f;
    }
}

__global__ void __launch_bounds__(192, 1)
k_route_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
           RouteTcArgs a, int nsplit) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    using C = TcCfg;
    extern __shared__ uint8_t smem_raw[];
    const int ntiles = (a.R + 127) / 128;
    // a unit: (128-row tile t, K part kp, expert slice sp); the K parts of a
    // tile write their partial logits to slices kp of a.logits
    const int nk = a.nk;
    const int nunits = ntiles * nk * nsplit;
    const int NH = a.E / nsplit;  // experts per unit (MMA N)
    if ((int)blockIdx.x >= nunits) return;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kBarOff);
    uint64_t* empty = full + kTcStages;
    uint64_t* tfull = empty + kTcStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* dbar = tempty + 2;   // MMA drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dbar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(tfull + i, 1); mbar_init(tempty + i, 128); }
        mbar_init(dbar, 1);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
    }
    auto give_up = [&]() {
        if (!*abort_flag) { *abort_flag = 1; status_add(a.status, MOE_STATUS_WAIT_TIMEOUT, 1); }
    };
    const int nkb = (a.H >> 6) / nk;   // 64-wide K steps of a part
    const uint64_t kWaitNs = a.wait_ns ? a.wait_ns : kTcWaitNs;   // pipeline waits

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0, nfills = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t bytes = (uint32_t)(C::kABytes + NH * 128);
            for (int u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
                const int t = u / (nk * nsplit), kp = (u / nsplit) % nk, sp = u % nsplit;
                for (int kb = kp * nkb; kb < (kp + 1) * nkb; ++kb) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full + stage, bytes);
                    const uint32_t sA = sbase + stage * C::kStageBytes;
                    tma_load_2d(sA, &tm_x, kb * 64, t * 128, full + stage);
                    tma_load_2d(sA + C::kABytes, &tm_w, kb * 64, sp * NH, full + stage);
                    ++nfills;
                    if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
                }
            }
            // drain: the last fill of every stage has landed (consumed or not),
            // so no copy into this CTA's shared memory is in flight at exit
            for (int s = 0; s < kTcStages; ++s) {
                if (nfills < kTcStages && s >= nfills) break;
                const uint32_t par = s < stage ? phase : (phase ^ 1u);
                if (!mbar_wait_bounded(full + s, par, never, kTcDrainNs)) give_up();
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16_f32(128, NH);
            for (int u = blockIdx.x; ok && u < nunits; u += gridDim.x) {
                if (!mbar_wait_bounded(tempty + acc, acc_phase ^ 1u, abort_flag, kWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * 256);
                for (int kb = 0; kb < nkb; ++kb) {   // the part's K steps, from its start
                    if (!mbar_wait_bounded(full + stage, phase, abort_flag, kWaitNs)) {
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
            // drain: arrives once every MMA issued above has completed
            tc_commit(dbar);
            if (!mbar_wait_bounded(dbar, 0, never, kTcDrainNs)) give_up();
        }
    } else {
        // epilogue: thread = row; store the approximate logits
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
            const int t = u / (nk * nsplit), kp = (u / nsplit) % nk, sp = u % nsplit;
            const bool okw = mbar_wait_bounded(tfull + acc, acc_phase, abort_flag, kWaitNs);
            if (__any_sync(0xffffffffu, !okw)) { give_up(); break; }
            __syncwarp();
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256);
            const int row = t * 128 + q * 32 + lane;
            float* out = a.logits + ((size_t)kp * a.R + row) * a.E + sp * NH;
            for (int c = 0; c < NH; c += 16) {
                float v[16];
                __syncwarp();
                tmem_ld16(tb + (uint32_t)c, v);
                if (row < a.R) {
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4*>(out + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                }
            }
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

// Exact logits of every expert of row r (the fallback for rows whose
// screening is inconclusive), 16 at a time in the contract order; then top-k
// and softmax.  One warp.
__device__ __noinline__ void exact_full_row(const RouteTcArgs& a, int r, const float* brow, int lane) {
    constexpr int NG = 16;  // groups of 16 experts: up to 256
    const __nv_bfloat16* xr = a.x + (size_t)r * a.H;
    uint32_t key[NG], id[NG];
    uint32_t valid = 0;
#pragma unroll
    for (int g = 0; g < NG; ++g) { key[g] = 0; id[g] = 0xFFFFFFFFu; }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        if (g * 16 >= a.E) break;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        for (int s = 0; s < a.H; s += 256) {
            const int col = s + lane * 8;
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + col));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = g * 16 + i;
                const uint4 wv = e < a.E
                    ? __ldg(reinterpret_cast<const uint4*>(a.wr + (size_t)e * a.H + col))
                    : make_uint4(0, 0, 0, 0);
                acc[i] = dot8_bf16(xv, wv, acc[i]);
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
        const float dot = __fadd_rn(acc[0], __shfl_xor_sync(0xffffffffu, acc[0], 1));
        const int e = g * 16 + (lane >> 1);  // lanes 2i and 2i+1 hold expert g*16 + i
        if ((lane & 1) == 0 && e < a.E) {
            key[g] = order_key(finish_logit(dot, brow, e));
            id[g] = (uint32_t)e;
            valid |= 1u << g;
        }
    }
    uint32_t my_id, my_key;
    warp_topk<NG>(key, id, valid, a.k, lane, my_id, my_key);
    write_topk(a.topk_idx + (size_t)r * a.k, a.topk_w + (size_t)r * a.k, a.k, lane, my_id, my_key);
}

// A CTA takes tiles of kExRows rows.
//   1. warp w screens row w of the tile: copies x_r to shared memory, forms
//      |x_r|, finds the k-th approximate logit T and lists the candidates;
//   2. the tile's (row, candidate) pairs are shared out over the 8 warps, two
//      per pass: each lane accumulates its elements of both dot products in
//      the contract order, one halving step at partner distance 16 leaves
//      candidate 0 in lanes 0-15 and candidate 1 in lanes 16-31, and the
//      plain butterfly at 8, 4, 2, 1 finishes both;
//   3. warp w takes top-k and softmax of row w over its candidates.
// The loads are latency bound (L2 round trips of a few thousand cycles), so
// step 2 prefetches the next tile's x row and logits into L1.  Prefetching
// the next pair's router rows too measured slower (the 8192-row router 77
// against 83 us without it: the 16 warps' prefetched rows crowd L1).
constexpr int kExRows = 8;
constexpr int kExMaxH = 8192;  // x tile in shared memory: kExRows * H bf16

__global__ void __launch_bounds__(256, 2) k_route_exact(RouteTcArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t ex_smem[];
    __nv_bfloat16* s_x = reinterpret_cast<__nv_bfloat16*>(ex_smem);  // [kExRows][H]
    __shared__ int32_t s_ce[kExRows * kCandCap];  // candidate expert of each slot
    __shared__ float s_cz[kExRows * kCandCap];    // its exact logit (bias added)
    __shared__ int s_cnt[kExRows];                // candidates of the row; -1: all experts
    __shared__ int s_blk[kExRows];                // block of the row (bias row)
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nstripes = a.H >> 8;
    const float G = (float)a.H * 0x1p-21f;
    // max_e |w_e| (every warp computes the same value)
    float wmax = 0.0f;
    for (int e = lane; e < a.E; e += 32) wmax = fmaxf(wmax, __ldg(a.wnorm + e));
    wmax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(wmax)));
    const int ntiles = (a.R + kExRows - 1) / kExRows;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int r = tile * kExRows + w;
        // ------------------------------------------------ 1. screening of row r
        if (r < a.R) {
            const __nv_bfloat16* xr = a.x + (size_t)r * a.H;
            __nv_bfloat16* sx = s_x + (size_t)w * a.H;
            const int blk = a.bias ? find_block(a.off, a.nb, r) : 0;
            const float* brow = a.bias ? a.bias + (size_t)blk * a.E : nullptr;
            // the screen's K parts, added in part order (all eight loads of a
            // part are issued before they are used)
            float az[8];
            for (int s2 = 0; s2 < a.nk; ++s2) {
                const float* lp = a.logits + ((size_t)s2 * a.R + r) * a.E;
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = lane + 32 * i;
                    v[i] = e < a.E ? __ldg(lp + e) : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) az[i] = s2 == 0 ? v[i] : __fadd_rn(az[i], v[i]);
            }
            float ss = 0.0f;
            for (int c0 = 0; c0 < a.H; c0 += 8 * 256) {
                uint4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = c0 + i * 256 + lane * 8;
                    if (c < a.H) v[i] = __ldg(reinterpret_cast<const uint4*>(xr + c));
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = c0 + i * 256 + lane * 8;
                    if (c < a.H) {
                        *reinterpret_cast<uint4*>(sx + c) = v[i];
                        ss = dot8_bf16(v[i], v[i], ss);
                    }
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float gx = G * (sqrtf(ss) * 1.001f);  // 1.001 covers the rounding of the sum
            uint32_t sk[8];
            uint32_t nonfinite = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                sk[i] = 0;
                if (e < a.E) {
                    float z = az[i];
                    if (brow) z = __fadd_rn(z, __ldg(brow + e));
                    nonfinite += !isfinite(z);
                    az[i] = z;
                    sk[i] = order_key(z);
                }
            }
            nonfinite = __reduce_add_sync(0xffffffffu, nonfinite);
            if (lane == 0) status_add(a.status, MOE_STATUS_NONFINITE_LOGITS, nonfinite);
            // T = the k-th largest approximate logit: each lane sorts its eight
            // keys (descending), then k rounds pop the warp's largest head
#pragma unroll
            for (int rnd = 0; rnd < 8; ++rnd)
#pragma unroll
                for (int i = rnd & 1; i + 1 < 8; i += 2) {
                    const uint32_t hi = max(sk[i], sk[i + 1]), lo = min(sk[i], sk[i + 1]);
                    sk[i] = hi;
                    sk[i + 1] = lo;
                }
            uint32_t tkey = 0;
            for (int j = 0; j < a.k; ++j) {
                tkey = __reduce_max_sync(0xffffffffu, sk[0]);
                const uint32_t win = __reduce_min_sync(0xffffffffu, sk[0] == tkey ? (uint32_t)lane : 32u);
                if ((uint32_t)lane == win) {
#pragma unroll
                    for (int i = 0; i < 7; ++i) sk[i] = sk[i + 1];
                    sk[7] = 0;
                }
            }
            const float T = key_value(tkey);
            const float thr = T - (gx * wmax + slack(T));
            int cnt = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                const bool c = e < a.E && az[i] + (gx * __ldg(a.wnorm + (e < a.E ? e : 0)) + slack(az[i])) >= thr;
                const uint32_t m = __ballot_sync(0xffffffffu, c);
                const int pos = cnt + __popc(m & ((1u << lane) - 1u));
                if (c && pos < kCandCap) s_ce[w * kCandCap + pos] = e;
                cnt += __popc(m);
            }
            const bool full_row = !(T > -INFINITY) || cnt > kCandCap || cnt < a.k;
            if (lane == 0) {
                s_cnt[w] = full_row ? -1 : cnt;
                s_blk[w] = blk;
            }
        } else if (lane == 0) {
            s_cnt[w] = 0;
        }
        __syncthreads();
        // ------------------------------------- 2. exact logits of the candidates
        {
            const int cr = lane < kExRows ? max(s_cnt[lane], 0) : 0;
            int incl = cr;
#pragma unroll
            for (int o = 1; o < kExRows; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const int total = __shfl_sync(0xffffffffu, incl, kExRows - 1);
            const int excl = incl - cr;  // lane i < kExRows: first slot of row i
            {   // the next tile's row of this warp: x and approximate logits
                const int rn = (tile + gridDim.x) * kExRows + w;
                if (rn < a.R) {
                    const __nv_bfloat16* xn = a.x + (size_t)rn * a.H;
                    for (int c = lane * 64; c < a.H; c += 32 * 64) prefetch_l1(xn + c);
                    if (lane * 32 < a.E) prefetch_l1(a.logits + (size_t)rn * a.E + lane * 32);
                }
            }
            // expert of slot t (or -1 past the end) and its row in the tile
            auto slot = [&](int t, int& rr) {
                const uint32_t m = __ballot_sync(0xffffffffu, lane < kExRows && excl <= t);
                rr = __popc(m) - 1;
                const int first = __shfl_sync(0xffffffffu, excl, rr & 31);
                return t < total ? s_ce[rr * kCandCap + (t - first)] : -1;
            };
            for (int t0 = 2 * w; t0 < total; t0 += 2 * kExRows) {
                int row[2], e[2];
                e[0] = slot(t0, row[0]);
                e[1] = slot(t0 + 1, row[1]);
                float acc0 = 0.0f, acc1 = 0.0f;
                const __nv_bfloat16* x0 = s_x + (size_t)row[0] * a.H + lane * 8;
                const __nv_bfloat16* x1 = s_x + (size_t)row[1] * a.H + lane * 8;
                for (int s0 = 0; s0 < nstripes; s0 += 8) {
                    uint4 w0[8], w1[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int col = (s0 + i) * 256 + lane * 8;
                        const bool in = s0 + i < nstripes;
                        w0[i] = in ? __ldg(reinterpret_cast<const uint4*>(a.wr + (size_t)e[0] * a.H + col))
                                   : make_uint4(0, 0, 0, 0);
                        w1[i] = (in && e[1] >= 0)
                                    ? __ldg(reinterpret_cast<const uint4*>(a.wr + (size_t)e[1] * a.H + col))
                                    : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (s0 + i >= nstripes) break;
                        const int off = (s0 + i) * 256;
                        acc0 = dot8_bf16(*reinterpret_cast<const uint4*>(x0 + off), w0[i], acc0);
                        acc1 = dot8_bf16(*reinterpret_cast<const uint4*>(x1 + off), w1[i], acc1);
                    }
                }
                // halving at distance 16: lanes 0-15 keep candidate 0, 16-31 candidate 1
                const bool upper = (lane & 16) != 0;
                float v = __fadd_rn(upper ? acc1 : acc0,
                                    __shfl_xor_sync(0xffffffffu, upper ? acc0 : acc1, 16));
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
                const int h = lane >> 4;
                if ((lane & 15) == 0 && e[h] >= 0) {
                    const float* brow = a.bias ? a.bias + (size_t)s_blk[row[h]] * a.E : nullptr;
                    s_cz[t0 + h] = finish_logit(v, brow, e[h]);
                }
            }
        }
        __syncthreads();
        // ------------------------------------------------- 3. top-k of row r
        if (r < a.R) {
            const int c = s_cnt[w];
            const float* brow = a.bias ? a.bias + (size_t)s_blk[w] * a.E : nullptr;
            if (c >= 0) {
                // slots of row w start after the candidates of rows 0..w-1
                int first = 0;
                for (int i = 0; i < w; ++i) first += max(s_cnt[i], 0);
                uint32_t key[1] = {0u}, id[1] = {0xFFFFFFFFu};
                if (lane < c) {
                    key[0] = order_key(s_cz[first + lane]);
                    id[0] = (uint32_t)s_ce[w * kCandCap + lane];
                }
                uint32_t my_id, my_key;
                warp_topk<1>(key, id, lane < c ? 1u : 0u, a.k, lane, my_id, my_key);
                write_topk(a.topk_idx + (size_t)r * a.k, a.topk_w + (size_t)r * a.k, a.k, lane,
                           my_id, my_key);
            } else {
                exact_full_row(a, r, brow, lane);
            }
        }
        __syncthreads();  // the tile's shared memory is rewritten by the next tile
    }
}

cudaError_t route_tc_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(k_route_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcCfg::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_route_exact, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kExRows * kExMaxH * 2);
}

// Parts of H for the screen: the most (up to 8) that still leave every unit
// on its own SM, divide the 64-wide K steps evenly and fit the partial
// logits in the workspace (cap_rows rows of E logits).
int route_tc_parts(int R, int E, int H, int64_t cap_rows, int num_sms) {
    const int ntiles = (R + 127) / 128;
    const int nsplit = (E > 128 && E % 32 == 0) ? 2 : 1;
    int nk = 8;
    while (nk > 1 && ((H / 64) % nk != 0 || (int64_t)ntiles * nsplit * nk > num_sms ||
                      (int64_t)nk * R > cap_rows))
        nk >>= 1;
    return nk;
}

cudaError_t launch_route_tc(const RouteTcArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                            int num_sms, cudaStream_t st) {
    cudaError_t e = launch_kernel(k_route_norms, dim3((unsigned)((a.E + 7) / 8)), dim3(256), 0, st, a);
    const int ntiles = (a.R + 127) / 128;
    const int nsplit = (a.E > 128 && a.E % 32 == 0) ? 2 : 1;
    const int nunits = ntiles * a.nk * nsplit;
    const int grid = nunits < num_sms ? nunits : num_sms;
    if (e == cudaSuccess)
        e = launch_kernel(k_route_tc, dim3(grid), dim3(192), TcCfg::kSmem, st, tm_x, tm_w, a, nsplit);
    const long ntiles_ex = (a.R + kExRows - 1) / kExRows;
    const long eb = ntiles_ex < (long)num_sms * 2 ? ntiles_ex : (long)num_sms * 2;
    if (e == cudaSuccess)
        e = launch_kernel(k_route_exact, dim3((unsigned)eb), dim3(256),
                          (size_t)kExRows * a.H * 2, st, a);
    return e;
}

}  // namespace moe
