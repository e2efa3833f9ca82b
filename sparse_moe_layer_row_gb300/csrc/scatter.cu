// Forward bookkeeping: group the surviving (row, slot) pairs by expert so each
// touched expert's weights stream once per call, build the device-side work
// lists of the grouped GEMMs, and the final bf16 store.
//
// Model card "Clover-35B-A3B-Preview -- CMF", Hardware: "the experts a block
// uses are bound as they are routed" -- here: only experts with at least one
// surviving pair appear in the work lists.
//
// Pair order inside an expert is (row ascending, slot ascending), so the work
// lists and the GEMM tiles are the same on every run.  Nothing here waits on
// another CTA: the per-expert totals are combined by the last CTA to finish
// (ticket counter), which then writes the offsets and the unit lists for the
// GEMM launches that follow on the same stream.
#include "scatter_dev.cuh"

namespace moe {

constexpr int kScatThreads = 256;

// Large batches: a counting sort of the surviving (row, slot) pairs by expert,
// in three kernels, all parallel over blocks of rows:
//   k_scatter_hist   per block: pairs per expert (hist[b][e]) and each pair's
//                    rank among the block's pairs of its expert, rows in order
//                    (rows are taken 32 at a time, so any block size works)
//   k_scatter_scan   one warp per expert: base[b][e] = pairs of e in earlier
//                    blocks (in place over hist) and the expert's total; the
//                    last CTA to finish forms the expert offsets and the unit
//                    lists of both GEMMs
//   k_scatter_place  per block: each surviving pair's position, the pair
//                    lists (row, weight) and the inverse map (row, slot) -> pair
// No copy of x is made: the gate/up GEMM gathers its rows of x itself.
// A row that names the same expert twice contributes its first slot only
// (later duplicates are counted as bad ids).
constexpr int kHistRows = 32;

__global__ void __launch_bounds__(kScatThreads) k_scatter_hist(ScatterArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    __shared__ uint8_t s_slot[kHistRows][kMaxExperts];
    __shared__ int s_run[kMaxExperts];
    __shared__ int s_dup, s_live;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int E = a.E, k = a.k;
    const int words = (E + 31) >> 5;
    int r0 = a.off[b], r1 = a.off[b + 1];
    if (!(0 <= r0 && r0 <= r1 && r1 <= a.R)) r1 = r0 = 0;  // counted by the coreset call
    for (int e = tid; e < E; e += blockDim.x) s_run[e] = 0;
    if (tid == 0) { s_dup = 0; s_live = 0; }
    if (b == 0 && tid == 0) {
        a.misc[0] = 0;  // ticket of k_scatter_scan (next launch)
        a.misc[4] = 0;  // no staged output scaled yet (the down GEMM sets it)
    }
    for (int c0 = r0; c0 < r1; c0 += kHistRows) {
        const int nr = min(kHistRows, r1 - c0);
        __syncthreads();
        for (int i = tid; i < nr * E; i += blockDim.x) s_slot[i / E][i % E] = 0xFF;
        __syncthreads();
        for (int rr = tid; rr < nr; rr += blockDim.x) {
            const int r = c0 + rr;
            const bool lv = !a.live || a.live[r] != 0;  // dead rows: no pairs
            if (lv) atomicAdd(&s_live, 1);
            int dup = 0;
            for (int j = 0; j < k; ++j) {
                const int e = a.topk_idx[(size_t)r * k + j];
                a.prank[(size_t)r * k + j] = -1;
                if (!lv || e < 0 || e >= E) continue;
                if (!((a.keep[(size_t)b * words + (e >> 5)] >> (e & 31)) & 1u)) continue;
                if (s_slot[rr][e] != 0xFF) { ++dup; continue; }
                s_slot[rr][e] = (uint8_t)j;
            }
            if (dup) atomicAdd(&s_dup, dup);
        }
        __syncthreads();
        for (int e = tid; e < E; e += blockDim.x) {
            int run = s_run[e];
            for (int rr = 0; rr < nr; ++rr) {
                const int j = s_slot[rr][e];
                if (j == 0xFF) continue;
                a.prank[(size_t)(c0 + rr) * k + j] = run++;
            }
            s_run[e] = run;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) a.hist[(size_t)b * E + e] = s_run[e];
    if (tid == 0) {
        a.live_base[b] = s_live;
        status_add(a.status, MOE_STATUS_BAD_EXPERT_ID, (uint32_t)s_dup);
    }
}

constexpr int kScanThreads = 256;

constexpr int kDownGroup = 32;

__global__ void __launch_bounds__(kScanThreads) k_scatter_scan(ScatterArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    __shared__ int warp_sums[32];
    __shared__ int s_tot[kMaxExperts];
    __shared__ int s_cd[kMaxExperts + 1];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, E = a.E, nb = a.nb;
    // ---- one warp per expert: exclusive scan of its column of hist over blocks
    {
        const int e = blockIdx.x * (kScanThreads / 32) + (tid >> 5);
        if (e < E) {
            int run = 0;
            // 8 x 32 blocks per pass; all loads of a pass are issued before its
            // stores (a load after a store to the same array would wait for it)
            for (int b00 = 0; b00 < nb; b00 += 256) {
                int hv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int b = b00 + 32 * j + lane;
                    hv[j] = b < nb ? a.hist[(size_t)b * E + e] : 0;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int b = b00 + 32 * j + lane;
                    int incl = hv[j];
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int t = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += t;
                    }
                    if (b < nb) a.hist[(size_t)b * E + e] = run + incl - hv[j];
                    run += __shfl_sync(0xffffffffu, incl, 31);
                }
            }
            if (lane == 0) a.count[e] = run;
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(a.misc, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // ---- last CTA: live rows before each block, expert offsets and the unit lists
    for (int f = tid; f < E; f += blockDim.x) s_tot[f] = __ldcg(a.count + f);
    int nl;  // live rows: the shared expert's rows
    {
        const int per_b = (nb + blockDim.x - 1) / blockDim.x;
        const int b0 = min(nb, tid * per_b), b1 = min(nb, b0 + per_b);
        int cnt = 0;
        for (int b = b0; b < b1; ++b) cnt += __ldcg(a.live_base + b);
        int run = block_excl_scan_i32(cnt, warp_sums, &nl);
        for (int b = b0; b < b1; ++b) {
            const int c = __ldcg(a.live_base + b);
            a.live_base[b] = run;
            run += c;
        }
        if (!a.live) nl = a.R;  // every row: the shared expert's rows are 0 .. R-1
    }
    __syncthreads();
    const int mt_gu = (a.I + a.gu_rows - 1) / a.gu_rows, mt_gs = (a.Is + a.gu_rows - 1) / a.gu_rows;
    const int mt_dn = a.H / a.dn_cols;
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int sum = 0, ch_gu = 0, ch_dn = 0;
    for (int f = e0; f < e1; ++f) {
        sum += s_tot[f];
        ch_gu += (s_tot[f] + a.nt_gu - 1) / a.nt_gu;
        ch_dn += (s_tot[f] + a.nt_dn - 1) / a.nt_dn;
    }
    int tot_pairs, tot_gu, tot_dn;
    int p = block_excl_scan_i32(sum, warp_sums, &tot_pairs);
    int cg = block_excl_scan_i32(ch_gu, warp_sums, &tot_gu);
    int cd = block_excl_scan_i32(ch_dn, warp_sums, &tot_dn);
    const int sch_gu = (nl + a.nt_gu - 1) / a.nt_gu, sch_dn = (nl + a.nt_dn - 1) / a.nt_dn;
    const int base_gu = sch_gu * mt_gs;
    const int base_dn = sch_dn * mt_dn;
    // shared-expert units (group E, all rows): gate/up chunk-major, down tile-major
    for (int u = tid; u < base_gu; u += blockDim.x) {
        const int c = u / mt_gs, m = u - c * mt_gs;
        a.units_gu[u] = make_int4(E, m, c * a.nt_gu, min(a.nt_gu, nl - c * a.nt_gu));
    }
    for (int u = tid; u < base_dn; u += blockDim.x) {
        const int m = u / sch_dn, c = u - m * sch_dn;
        a.units_dn[u] = make_int4(E, m, c * a.nt_dn, min(a.nt_dn, nl - c * a.nt_dn));
    }
    // down units: expert groups of kDownGroup, each group ordered weight-tile
    // major, so the CTAs (or CTA pairs) running at one time write one slab of
    // dn_cols columns for the group's pairs and each group's activations are
    // reused from L2 across its weight tiles.
    {  // chunk prefix of each expert
        int q = cd;
        for (int f = e0; f < e1; ++f) {
            s_cd[f] = q;
            q += (s_tot[f] + a.nt_dn - 1) / a.nt_dn;
        }
    }
    if (tid == 0) s_cd[E] = tot_dn;
    __syncthreads();
    for (int f = e0; f < e1; ++f) {
        const int n = s_tot[f];
        a.expert_off[f] = p;
        write_units(a.units_gu, base_gu + cg * mt_gu, f, p, n, a.nt_gu, mt_gu);
        {
            const int g0 = f / kDownGroup * kDownGroup, g1 = min(E, g0 + kDownGroup);
            const int gbase = s_cd[g0], gchunks = s_cd[g1] - gbase;
            for (int m = 0; m < mt_dn; ++m) {
                int u = base_dn + gbase * mt_dn + m * gchunks + (s_cd[f] - gbase);
                for (int c0 = 0; c0 < n; c0 += a.nt_dn)
                    a.units_dn[u++] = make_int4(f, m, p + c0, min(a.nt_dn, n - c0));
            }
        }
        p += n;
        cg += (n + a.nt_gu - 1) / a.nt_gu;
    }
    if (tid == 0) {
        a.expert_off[E] = tot_pairs;
        a.misc[1] = base_gu + tot_gu * mt_gu;
        a.misc[2] = base_dn + tot_dn * mt_dn;
        a.misc[3] = tot_pairs;
    }
}

// One CTA per block: a thread per (row, slot) of the block.
__global__ void __launch_bounds__(kScatThreads) k_scatter_place(ScatterArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    __shared__ int warp_sums[32];
    const int b = blockIdx.x;
    const int E = a.E, k = a.k;
    int r0 = a.off[b], r1 = a.off[b + 1];
    if (!(0 <= r0 && r0 <= r1 && r1 <= a.R)) r1 = r0 = 0;
    // the block's live rows, in order, after the live rows of earlier blocks
    // (a.live is the same for the whole block, so the scans are block-uniform)
    int run = a.live ? a.live_base[b] : 0;
    for (int c0 = r0; a.live && c0 < r1; c0 += blockDim.x) {
        const int r = c0 + threadIdx.x;
        const int lv = (r < r1 && (!a.live || a.live[r] != 0)) ? 1 : 0;
        int n;
        const int pos = run + block_excl_scan_i32(lv, warp_sums, &n);
        if (r < r1) {
            a.shared_inv[r] = lv ? pos : -1;
            if (lv) a.shared_rows[pos] = r;
        }
        run += n;
    }
    for (int p = r0 * k + threadIdx.x; p < r1 * k; p += blockDim.x) {
        const int rk = a.prank[p];
        if (rk < 0) {
            a.inv[p] = -1;
            continue;
        }
        const int e = a.topk_idx[p];
        const int pos = a.expert_off[e] + a.hist[(size_t)b * E + e] + rk;
        a.pair_row[pos] = p / k;
        a.pair_w[pos] = a.w_renorm[p];
        a.inv[p] = pos;
    }
}

__global__ void __launch_bounds__(kSmallThreads) k_scatter_small(ScatterArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    __shared__ ScatterSmallSmem sm;
    scatter_small(a, sm);
}

// One warp per (row, 256 columns): y = staged shared output + the row's staged
// expert outputs, added in fp32 in rank order (shared first, then the slots;
// dead rows of a live-row call are skipped);
// lane owns 8 consecutive columns.  All of a task's contributions are loaded
// before they are added, eight at a time, so the loads overlap.  A staged
// value is v * 2^-s with s the exponent of its 32-column quarter (0 unless the
// down GEMM met a magnitude of 2^15 or more there); the product by 2^s is exact.
__device__ __forceinline__ float pow2_u8(uint32_t s) { return __uint_as_float((127u + s) << 23); }

// The combine of one call; kScaled: some staged quarter carries an exponent
// (the down GEMM's flag), so each contribution's exponent is read too.
template <bool kScaled>
__device__ __forceinline__ void combine_rows(const CombineArgs& a) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nchunk = a.H / 256;
    const int ntasks = a.R * nchunk;
    for (int t = warp; t < ntasks; t += nwarps) {
        const int r = t / nchunk;
        if (a.live && a.live[r] == 0) continue;  // dead row: its y stays as it is
        const int c = (t - r * nchunk) * 256 + lane * 8;
        const int pos = lane < a.k ? a.inv[(size_t)r * a.k + lane] : -1;
        const int srow = a.live ? a.shared_inv[r] : r;  // staging row of the shared output
        const uint8_t* xq = a.ysx + (size_t)(c >> 5) * a.ld_x;  // exponents of this quarter
        float acc[8];
        {
            const size_t sr = (size_t)(a.shared_row0 + srow);
            const uint4 v = *reinterpret_cast<const uint4*>(a.ys + sr * a.H + c);
            const float sc = kScaled ? pow2_u8(xq[sr]) : 1.0f;
            const __half2* hv = reinterpret_cast<const __half2*>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(hv[i]);
                acc[2 * i] = kScaled ? f.x * sc : f.x;
                acc[2 * i + 1] = kScaled ? f.y * sc : f.y;
            }
        }
        for (int j0 = 0; j0 < a.k; j0 += 8) {
            uint4 v[8];
            uint32_t sx[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int p = __shfl_sync(0xffffffffu, pos, (j0 + j) & 31);
                const bool on = j0 + j < a.k && p >= 0;
                v[j] = on ? *reinterpret_cast<const uint4*>(a.ys + (size_t)p * a.H + c)
                          : make_uint4(0, 0, 0, 0);
                sx[j] = kScaled && on ? xq[p] : 0u;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int p = __shfl_sync(0xffffffffu, pos, (j0 + j) & 31);
                if (j0 + j >= a.k || p < 0) continue;
                const float sc = pow2_u8(sx[j]);
                const __half2* hv = reinterpret_cast<const __half2*>(&v[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __half22float2(hv[i]);
                    acc[2 * i] += kScaled ? f.x * sc : f.x;
                    acc[2 * i + 1] += kScaled ? f.y * sc : f.y;
                }
            }
        }
        bool finite = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) finite = finite && isfinite(acc[i]);
        uint4 o;
        __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) ob[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        *reinterpret_cast<uint4*>(a.y + (size_t)r * a.H + c) = o;
        if (a.y_f32) {
            float4* yf = reinterpret_cast<float4*>(a.y_f32 + (size_t)r * a.H + c);
            yf[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            yf[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        // counted per (row, 256-column chunk) that holds a non-finite value
        if (__any_sync(0xffffffffu, !finite) && lane == 0)
            status_add(a.status, MOE_STATUS_NONFINITE_OUTPUT, 1);
    }
}

// kMinCtas CTAs per SM: after the CTA-pair down GEMM four, registers capped at 64, 32 warps per SM to keep
// more loads in flight (8192 rows: 69.6 -> 62.7 us); that down GEMM lets the
// combine launch only when it ends (common.cuh).  Otherwise one: launched
// early, four CTAs per SM waiting beside the streaming down GEMM slowed the
// step.
template <int kMinCtas>
__global__ void __launch_bounds__(256, kMinCtas) k_combine(CombineArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    if (*a.scaled) combine_rows<true>(a);
    else combine_rows<false>(a);
}

cudaError_t launch_scatter(const ScatterArgs& a, bool small, int num_sms, cudaStream_t st) {
    (void)num_sms;
    if (small) return launch_kernel(k_scatter_small, dim3(1), dim3(kSmallThreads), 0, st, a);
    cudaError_t e = launch_kernel(k_scatter_hist, dim3(a.nb), dim3(kScatThreads), 0, st, a);
    const int scan_ctas = (a.E + kScanThreads / 32 - 1) / (kScanThreads / 32);
    if (e == cudaSuccess)
        e = launch_kernel(k_scatter_scan, dim3(scan_ctas), dim3(kScanThreads), 0, st, a);
    if (e == cudaSuccess) e = launch_kernel(k_scatter_place, dim3(a.nb), dim3(kScatThreads), 0, st, a);
    return e;
}

cudaError_t launch_combine(const CombineArgs& a, int num_sms, bool after_pair_down, cudaStream_t st) {
    long blocks = ((long)a.R * (a.H / 256) + 7) / 8;
    if (blocks > (long)num_sms * 16) blocks = (long)num_sms * 16;
    if (blocks < 1) blocks = 1;
    if (after_pair_down)
        return launch_kernel(k_combine<4>, dim3((unsigned)blocks), dim3(256), 0, st, a);
    return launch_kernel(k_combine<1>, dim3((unsigned)blocks), dim3(256), 0, st, a);
}

}  // namespace moe
