// Device code of the block coreset (k_coreset: one CTA per block).  The
// method and its arithmetic are described in coreset.cu.
#pragma once

#include "kernels.cuh"

namespace moe {

constexpr int kCoreThreads = 1024;      // E > 256, few blocks: more threads rank each expert
constexpr int kCoreThreadsSort = 256;   // E > 256, many blocks (the sorting path)
constexpr int kCoreThreadsSmallE = 256; // E <= 256: a thread per expert
constexpr int kMaxE = 1024;
constexpr int kSortBlocks = 64;   // blocks from which the ranks come from a sort
constexpr int kPairCache = 2048;  // slots of a block kept in shared memory for the renormalisation

__device__ __forceinline__ uint64_t mass_threshold(float tau, uint64_t T) {
    const uint32_t u = __float_as_uint(tau);
    const uint32_t ex = (u >> 23) & 0xFFu;
    const uint64_t M = ex ? ((u & 0x7FFFFFu) | 0x800000u) : (u & 0x7FFFFFu);
    const int s = ex ? 150 - (int)ex : 149;
    const unsigned __int128 prod = (unsigned __int128)M * T;
    if (prod == 0) return 0;
    if (s >= 128) return 1;
    unsigned __int128 q = prod >> s;
    if ((q << s) != prod) q += 1;
    return (uint64_t)q;
}

// Exclusive block-wide scan of one uint64 per thread; returns the block total in *total.
__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, uint64_t* warp_sums, uint64_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        uint64_t ws = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t t = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += t;
        }
        if (lane < nw) warp_sums[lane] = ws;  // inclusive warp prefix
    }
    __syncthreads();
    const uint64_t before = warp ? warp_sums[warp - 1] : 0;
    *total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before + incl - v;
}

// Shared memory of one block's coreset.
struct CoresetSmem {
    unsigned long long Q[kMaxE];
    uint32_t touched[kMaxE / 32];
    uint32_t incore[kMaxE / 32];
    __align__(16) unsigned long long keys[kMaxE];
    uint64_t warp_sums[32];
    int warp_cnt[32];
    int32_t pe[kPairCache];   // the block's slots (expert, weight) when they fit
    float pw[kPairCache];
    uint8_t in_flag[256];     // E <= 256: the expert is in the coreset
    int s_bad, s_empty;
};

// The coreset of block b and its rows' renormalised weights, by the whole CTA
// (every thread calls it).  With E <= 256 and kCoreThreadsSmallE threads a
// thread ranks each expert; otherwise sort_ranks picks a bitonic sort (many
// CTAs share the SMs) rather than lanes counting the keys above each expert
// (few CTAs: latency counts); all give the same ranks.  The shared memory may
// be reused after the call returns.
__device__ __forceinline__ void coreset_block(const CoresetArgs& a, int b, CoresetSmem& sm,
                                              bool sort_ranks) {
    unsigned long long* Q = sm.Q;
    uint32_t* touched = sm.touched;
    uint32_t* incore = sm.incore;
    unsigned long long* keys = sm.keys;
    uint64_t* warp_sums = sm.warp_sums;
    int* warp_cnt = sm.warp_cnt;
    uint8_t* in_flag = sm.in_flag;
    int& s_bad = sm.s_bad;
    int& s_empty = sm.s_empty;
    const int tid = threadIdx.x;
    const int E = a.E, k = a.k;
    const int words = (E + 31) >> 5;
    const int r0 = a.off[b], r1 = a.off[b + 1];
    const bool valid = 0 <= r0 && r0 <= r1 && r1 <= a.R;
    if (!valid) {
        if (tid == 0) {
            status_add(a.status, MOE_STATUS_BAD_OFFSETS, 1);
            a.core_size[b] = 0;
            if (a.n_empty) a.n_empty[b] = 0;
        }
        for (int w = tid; w < words; w += blockDim.x) a.keep[(size_t)b * words + w] = 0;
        return;
    }
    for (int e = tid; e < E; e += blockDim.x) Q[e] = 0;
    for (int w = tid; w < kMaxE / 32; w += blockDim.x) { touched[w] = 0; incore[w] = 0; }
    if (tid == 0) { s_bad = 0; s_empty = 0; }
    __syncthreads();
    const int npairs = (r1 - r0) * k;
    const bool cached = npairs <= kPairCache;
    int bad = 0;
    for (int p = tid; p < npairs; p += blockDim.x) {
        const size_t i = (size_t)r0 * k + p;
        const int e = a.topk_idx[i];
        const float wt = a.topk_w[i];
        if (cached) {
            sm.pe[p] = e;
            sm.pw[p] = wt;
        }
        if (e < 0 || e >= E) { ++bad; continue; }
        const float w = a.mass ? a.mass[i] : wt;   // the slot's mass
        const unsigned long long q =
            (w >= 0.0f && w <= 1.0f) ? __float2ull_rz(__fmul_rn(w, 4294967296.0f)) : 0ull;
        atomicAdd(&Q[e], q);
        atomicOr(&touched[e >> 5], 1u << (e & 31));
    }
    if (bad) atomicAdd(&s_bad, bad);
    __syncthreads();
    bool renorm;   // else the rows keep their weights bit for bit
    if (E <= 256 && (int)blockDim.x == kCoreThreadsSmallE) {
        // A thread per expert.  Each warp sorts its 32 keys (one per lane,
        // a shuffle bitonic network) and keeps the run with its exclusive
        // prefix masses; an expert's rank is its place in its own run plus,
        // for every other run, the number of keys above its own there (a
        // binary search), and the mass above it the matching prefix masses.
        const int lane = tid & 31, warp = tid >> 5;
        constexpr int kRuns = kCoreThreadsSmallE / 32;
        unsigned long long* runk = keys;         // [kRuns][32] sorted keys
        unsigned long long* runp = keys + 256;   // [kRuns][32] mass before each
        const int e = tid;
        const bool tch = e < E && ((touched[e >> 5] >> (e & 31)) & 1u);
        // (Q desc, id asc) as one 64-bit key, as below; 0 for an untouched expert
        unsigned long long x =
            tch ? ((unsigned long long)Q[e] << 10 | (unsigned long long)(1023 - e)) + 1ull : 0ull;
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, x, stride);
                const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
                x = keep_max ? (x > o ? x : o) : (x < o ? x : o);
            }
        const unsigned long long qx = x ? (x - 1ull) >> 10 : 0ull;
        unsigned long long incl = qx;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        runk[warp * 32 + lane] = x;
        runp[warp * 32 + lane] = incl - qx;
        const uint32_t tm = __ballot_sync(0xffffffffu, x != 0ull);
        if (lane == 31) {
            warp_cnt[warp] = __popc(tm);
            warp_sums[warp] = incl;
        }
        in_flag[e] = 0;
        __syncthreads();
        uint64_t T = 0;
        int nt = 0;
#pragma unroll
        for (int w = 0; w < kRuns; ++w) {
            T += warp_sums[w];
            nt += warp_cnt[w];
        }
        const bool disabled = !(a.tau < 1.0f);
        const int cap = (a.max_experts > 0 && a.max_experts < nt) ? a.max_experts : nt;
        renorm = !disabled || cap < nt;
        if (renorm && x) {
            const uint64_t theta = disabled ? ~0ull : mass_threshold(a.tau, T);
            // runs are descending: cnt[w] = number of keys of run w above x
            // (32 when its last one is; else a binary search over 0 .. 31)
            int cnt[kRuns];
#pragma unroll
            for (int w = 0; w < kRuns; ++w) cnt[w] = (w != warp && runk[w * 32 + 31] > x) ? 32 : 0;
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1)
#pragma unroll
                for (int w = 0; w < kRuns; ++w)
                    if (w != warp && cnt[w] < 32 && runk[w * 32 + cnt[w] + step - 1] > x) cnt[w] += step;
            int rank = lane;
            unsigned long long above = runp[warp * 32 + lane];
#pragma unroll
            for (int w = 0; w < kRuns; ++w) {
                if (w == warp) continue;
                rank += cnt[w];
                above += cnt[w] < 32 ? runp[w * 32 + cnt[w]] : warp_sums[w];
            }
            // kept iff the mass ranked above is still below theta (the greedy
            // prefix) and, under the budget, the rank is below the cap
            const int ex = 1023 - (int)((x - 1ull) & 1023ull);
            in_flag[ex] = (disabled || above < theta) && rank < cap;
        }
        __syncthreads();
        const bool in = renorm ? (e < E && in_flag[e]) : tch;
        const uint32_t word = __ballot_sync(0xffffffffu, in);
        if (lane == 0 && warp < words) incore[warp] = word;
    } else {
    // block total T and touched count
    uint64_t part = 0;
    for (int e = tid; e < E; e += blockDim.x) part += Q[e];
    uint64_t T;
    (void)block_excl_scan_u64(part, warp_sums, &T);
    int nt = 0;
    for (int w = 0; w < words; ++w) nt += __popc(touched[w]);

    const bool disabled = !(a.tau < 1.0f);
    const int cap = (a.max_experts > 0 && a.max_experts < nt) ? a.max_experts : nt;
    renorm = !disabled || cap < nt;
    if (!renorm) {
        for (int w = tid; w < words; w += blockDim.x) incore[w] = touched[w];
    } else {
        const uint64_t theta = disabled ? ~0ull : mass_threshold(a.tau, T);
        // Order (Q desc, id asc) as one 64-bit key per expert: (Q << 10 | (1023 - e)) + 1
        // for touched experts, 0 otherwise (Q < 2^53: a block has fewer than 2^21 rows);
        // keys are unique, and Q and e can be read back from a key.
        int n = 32;
        while (n < E) n <<= 1;
        for (int e = tid; e < n; e += blockDim.x)
            keys[e] = (e < E && ((touched[e >> 5] >> (e & 31)) & 1u))
                          ? ((unsigned long long)Q[e] << 10 | (unsigned long long)(1023 - e)) + 1ull
                          : 0ull;
        __syncthreads();
        if (sort_ranks) {
            // bitonic sort, descending
            for (int kk = 2; kk <= n; kk <<= 1) {
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    for (int i = tid; i < n; i += blockDim.x) {
                        const int ixj = i ^ j;
                        if (ixj > i) {
                            const unsigned long long x = keys[i], y = keys[ixj];
                            if ((i & kk) == 0 ? x < y : x > y) { keys[i] = y; keys[ixj] = x; }
                        }
                    }
                    __syncthreads();
                }
            }
            // rank i is kept iff the mass ranked above it is still below theta (the
            // greedy prefix stops at the first expert whose inclusion reaches it)
            // and, under the budget, i < cap
            const int per = (n + blockDim.x - 1) / blockDim.x;
            const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
            uint64_t part2 = 0;
            for (int i = i0; i < i1; ++i) part2 += keys[i] ? (keys[i] - 1ull) >> 10 : 0ull;
            uint64_t tot2;
            uint64_t above = block_excl_scan_u64(part2, warp_sums, &tot2);
            for (int i = i0; i < i1; ++i) {
                const unsigned long long key = keys[i];
                if (!key) break;   // untouched experts sort last
                if ((disabled || above < theta) && i < cap) {
                    const int e = 1023 - (int)((key - 1ull) & 1023ull);
                    atomicOr(&incore[e >> 5], 1u << (e & 31));
                }
                above += (key - 1ull) >> 10;
            }
        } else {
            // tpe threads (consecutive lanes) rank an expert together: each
            // counts the keys above it in every tpe-th slot and their mass,
            // and the lanes add their counts
            int tpe = 1;
            while (tpe < 32 && tpe * 2 * E <= (int)blockDim.x) tpe <<= 1;
            const int q = tid & (tpe - 1), per_round = blockDim.x / tpe;
            for (int base = 0; base < E; base += per_round) {   // the same trip count for all
                const int e = base + tid / tpe;
                const unsigned long long ke = e < E ? keys[e] : 0ull;
                unsigned long long above = 0;
                int rank = 0;
                if (ke) {
                    for (int f = q; f < E; f += tpe) {
                        const bool gt = keys[f] > ke;
                        above += gt ? Q[f] : 0ull;
                        rank += gt;
                    }
                }
                for (int o = tpe >> 1; o > 0; o >>= 1) {
                    above += __shfl_xor_sync(0xffffffffu, above, o);
                    rank += __shfl_xor_sync(0xffffffffu, rank, o);
                }
                if (ke && q == 0 && (disabled || above < theta) && rank < cap)
                    atomicOr(&incore[e >> 5], 1u << (e & 31));
            }
        }
    }
    }
    __syncthreads();
    int c = 0;
    for (int w = 0; w < words; ++w) c += __popc(incore[w]);
    for (int w = tid; w < words; w += blockDim.x) a.keep[(size_t)b * words + w] = incore[w];
    if (tid == 0) a.core_size[b] = c;
    // renormalise rows: lanes in groups of kp (the power of two >= k), a row
    // per group and 32 / kp rows per warp at a time, lane j of a group holding
    // slot j; the sum of the surviving weights is taken in rank order, one
    // fp32 add at a time
    int empty = 0;
    {
        const int lane = tid & 31, nw = blockDim.x >> 5;
        int kp = 1;
        while (kp < k) kp <<= 1;
        const int gpw = 32 / kp, grp = lane / kp, j = lane - grp * kp;
        const uint32_t gmask = kp == 32 ? 0xFFFFFFFFu : ((1u << kp) - 1u);
        for (int rb = r0 + (tid >> 5) * gpw; rb < r1; rb += nw * gpw) {
            const int r = rb + grp;
            const bool act = r < r1 && j < k;
            const int p = (r - r0) * k + j;
            const int e = act ? (cached ? sm.pe[p] : a.topk_idx[(size_t)r * k + j]) : -1;
            const float wj = act ? (cached ? sm.pw[p] : a.topk_w[(size_t)r * k + j]) : 0.0f;
            float* wo = a.w_renorm + (size_t)r * k;
            if (!renorm) {
                if (act) wo[j] = wj;
                continue;
            }
            const bool in = e >= 0 && e < E && ((incore[e >> 5] >> (e & 31)) & 1u);
            const uint32_t inm = (__ballot_sync(0xffffffffu, in) >> (grp * kp)) & gmask;
            float s = 0.0f;
            for (int jj = 0; jj < k; ++jj) {
                const float v = __shfl_sync(0xffffffffu, wj, grp * kp + jj);
                if ((inm >> jj) & 1u) s = __fadd_rn(s, v);
            }
            if (act) {
                if (s == 0.0f) {
                    wo[j] = 0.0f;
                    if (j == 0) ++empty;
                } else {
                    wo[j] = in ? __fdiv_rn(wj, s) : 0.0f;
                }
            }
        }
    }
    if (empty) atomicAdd(&s_empty, empty);
    __syncthreads();
    if (tid == 0) {
        if (a.n_empty) a.n_empty[b] = s_empty;
        status_add(a.status, MOE_STATUS_EMPTY_ROWS, (uint32_t)s_empty);
        status_add(a.status, MOE_STATUS_BAD_EXPERT_ID, (uint32_t)s_bad);
    }
}

}  // namespace moe
