// Device code of the block coreset, shared by k_coreset (one CTA per block)
// and the fused front end of small calls (one CTA for every block).  The
// method and its arithmetic are described in coreset.cu.
#pragma once

#include "kernels.cuh"

namespace moe {

constexpr int kCoreThreads = 1024;      // few blocks: more threads rank each expert
constexpr int kCoreThreadsSort = 256;   // many blocks (the sorting path)
constexpr int kMaxE = 1024;
constexpr int kSortBlocks = 64;   // blocks from which the ranks come from a sort

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

// Sort 256 64-bit keys held eight per lane (slot i = 8 * lane + r) into
// descending order across the warp: a bitonic network whose strides below 8
// compare registers of one lane and whose strides of 8 and more trade a
// register with lane ^ (stride / 8).  36 steps, no shared memory, no barrier.
__device__ __forceinline__ void warp_sort256_desc(unsigned long long (&k)[8], int lane) {
#pragma unroll
    for (int size = 2; size <= 256; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 8) {
                const int lm = stride >> 3;                       // lane distance
                const bool lower = (lane & lm) == 0;              // the lower slot of the pair
                const bool desc = ((8 * lane) & size) == 0;       // this run sorts descending
                const bool keep_max = lower == desc;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, k[r], lm);
                    k[r] = keep_max ? (k[r] > o ? k[r] : o) : (k[r] < o ? k[r] : o);
                }
            } else {
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int pr = r ^ stride;
                    if (pr > r) {
                        const bool desc = ((8 * lane + r) & size) == 0;
                        const unsigned long long a = k[r], b = k[pr];
                        if (desc ? a < b : a > b) { k[r] = b; k[pr] = a; }
                    }
                }
            }
        }
    }
}

// Shared memory of one block's coreset.
struct CoresetSmem {
    unsigned long long Q[kMaxE];
    uint32_t touched[kMaxE / 32];
    uint32_t incore[kMaxE / 32];
    unsigned long long keys[kMaxE];
    uint64_t warp_sums[32];
    int s_bad, s_empty;
};

// The coreset of block b and its rows' renormalised weights, by the whole CTA
// (every thread calls it).  sort_ranks: rank the experts by a bitonic sort
// (many CTAs share the SMs) rather than by lanes counting the keys above each
// expert (few CTAs: latency counts); both give the same ranks.  The shared
// memory may be reused after the call returns.
__device__ __forceinline__ void coreset_block(const CoresetArgs& a, int b, CoresetSmem& sm,
                                              bool sort_ranks) {
    unsigned long long* Q = sm.Q;
    uint32_t* touched = sm.touched;
    uint32_t* incore = sm.incore;
    unsigned long long* keys = sm.keys;
    uint64_t* warp_sums = sm.warp_sums;
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
    int bad = 0;
    for (int p = tid; p < npairs; p += blockDim.x) {
        const size_t i = (size_t)r0 * k + p;
        const int e = a.topk_idx[i];
        if (e < 0 || e >= E) { ++bad; continue; }
        const float w = (a.mass ? a.mass : a.topk_w)[i];   // the slot's mass
        const unsigned long long q =
            (w >= 0.0f && w <= 1.0f) ? __float2ull_rz(__fmul_rn(w, 4294967296.0f)) : 0ull;
        atomicAdd(&Q[e], q);
        atomicOr(&touched[e >> 5], 1u << (e & 31));
    }
    if (bad) atomicAdd(&s_bad, bad);
    __syncthreads();
    // block total T and touched count
    uint64_t part = 0;
    for (int e = tid; e < E; e += blockDim.x) part += Q[e];
    uint64_t T;
    (void)block_excl_scan_u64(part, warp_sums, &T);
    int nt = 0;
    for (int w = 0; w < words; ++w) nt += __popc(touched[w]);

    const bool disabled = !(a.tau < 1.0f);
    const int cap = (a.max_experts > 0 && a.max_experts < nt) ? a.max_experts : nt;
    const bool renorm = !disabled || cap < nt;  // else the rows keep their weights bit for bit
    if (!renorm) {
        for (int w = tid; w < words; w += blockDim.x) incore[w] = touched[w];
    } else {
        const uint64_t theta = disabled ? ~0ull : mass_threshold(a.tau, T);
        // Order (Q desc, id asc) as one 64-bit key per expert: (Q << 10 | (1023 - e)) + 1
        // for touched experts, 0 otherwise (Q < 2^53: a block has fewer than 2^21 rows);
        // keys are unique, and Q and e can be read back from a key.
        const bool warp_sort = E <= 256;   // one warp sorts every key in registers
        int n = 32;
        while (n < E) n <<= 1;
        if (warp_sort) n = 256;
        for (int e = tid; e < n; e += blockDim.x)
            keys[e] = (e < E && ((touched[e >> 5] >> (e & 31)) & 1u))
                          ? ((unsigned long long)Q[e] << 10 | (unsigned long long)(1023 - e)) + 1ull
                          : 0ull;
        __syncthreads();
        if (warp_sort) {
            // warp 0: sort, then the exclusive prefix of the masses in that order;
            // slot i is kept iff the mass ranked above it is still below theta
            // (the greedy prefix) and, under the budget, i < cap
            if (tid < 32) {
                unsigned long long kk[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) kk[r] = keys[8 * tid + r];
                warp_sort256_desc(kk, tid);
                unsigned long long pre[8], run = 0;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    pre[r] = run;
                    run += kk[r] ? (kk[r] - 1ull) >> 10 : 0ull;
                }
                unsigned long long incl = run;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += t;
                }
                const unsigned long long lane_excl = incl - run;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const unsigned long long key = kk[r];
                    if (key && (disabled || lane_excl + pre[r] < theta) && 8 * tid + r < cap) {
                        const int e = 1023 - (int)((key - 1ull) & 1023ull);
                        atomicOr(&incore[e >> 5], 1u << (e & 31));
                    }
                }
            }
        } else if (sort_ranks) {
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
    __syncthreads();
    int c = 0;
    for (int w = 0; w < words; ++w) c += __popc(incore[w]);
    __syncthreads();
    for (int w = tid; w < words; w += blockDim.x) a.keep[(size_t)b * words + w] = incore[w];
    if (tid == 0) a.core_size[b] = c;
    // renormalise rows: a warp per row, lane j holding slot j (k <= 32); the sum
    // of the surviving weights is taken in rank order, one fp32 add at a time
    int empty = 0;
    {
        const int lane = tid & 31, nw = blockDim.x >> 5;
        for (int r = r0 + (tid >> 5); r < r1; r += nw) {
            const int e = lane < k ? a.topk_idx[(size_t)r * k + lane] : -1;
            const float wj = lane < k ? a.topk_w[(size_t)r * k + lane] : 0.0f;
            float* wo = a.w_renorm + (size_t)r * k;
            if (!renorm) {
                if (lane < k) wo[lane] = wj;
                continue;
            }
            const bool in = e >= 0 && e < E && ((incore[e >> 5] >> (e & 31)) & 1u);
            const uint32_t inm = __ballot_sync(0xffffffffu, in);
            float s = 0.0f;
            for (int j = 0; j < k; ++j) {
                const float v = __shfl_sync(0xffffffffu, wj, j);
                if ((inm >> j) & 1u) s = __fadd_rn(s, v);
            }
            if (s == 0.0f) {
                if (lane < k) wo[lane] = 0.0f;
                if (lane == 0) ++empty;
                continue;
            }
            if (lane < k) wo[lane] = in ? __fdiv_rn(wj, s) : 0.0f;
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
