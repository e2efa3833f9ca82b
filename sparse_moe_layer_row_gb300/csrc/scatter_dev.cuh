// Device code of the forward bookkeeping of the scatter kernels (scatter.cu):
// block scans, the GEMM unit lists, and the whole small-call scatter in one
// CTA.
#pragma once

#include "kernels.cuh"

namespace moe {

// Exclusive scan of one int per thread over the block; *total gets the sum.
__device__ __forceinline__ int block_excl_scan_i32(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int ws = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += t;
        }
        if (lane < nw) warp_sums[lane] = ws;
    }
    __syncthreads();
    const int before = warp ? warp_sums[warp - 1] : 0;
    *total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before + incl - v;
}

// Units of one group: chunks of nt pairs x weight tiles; chunk-major so the
// CTAs that run neighbouring units share the same rows of x (L2 reuse).
__device__ __forceinline__ void write_units(int4* out, int base, int g, int start, int n, int nt, int mtiles) {
    int u = base;
    for (int c0 = 0; c0 < n; c0 += nt) {
        const int cn = min(nt, n - c0);
        for (int m = 0; m < mtiles; ++m) out[u++] = make_int4(g, m, start + c0, cn);
    }
}

// Small batches (R <= kSmallRows): the whole bookkeeping in one CTA.
// Same outputs as the three-kernel path: pair lists in row order per expert,
// expert offsets and unit lists.  A row that names the same expert twice
// contributes its first slot only (later duplicates are counted as bad ids),
// so the counts and the lists always agree.  Every expert has at most one
// pair per row, so at most kSmallRows <= kSmallN pairs: one chunk (one unit
// per weight tile) per expert.  The rows holding an expert's pairs are one
// 32-bit mask; a pair's place in its expert's list is the number of rows
// below its own in that mask.
constexpr int kSmallThreads = 512;
static_assert(kSmallRows <= 32 && kSmallRows <= kSmallN, "a row per mask bit, one chunk per expert");

// Shared memory of the small-call scatter.
struct ScatterSmallSmem {
    uint32_t mask[kMaxExperts];                    // rows with a surviving pair of e
    int off[kMaxExperts];                          // e's first place in the pair list
    int chunk_exp[kMaxExperts];                    // expert of each non-empty chunk
    uint32_t keepw[kSmallRows][kMaxExperts / 32];  // keep words of each row's block
    int32_t ids[kSmallRows * 32];
    float w[kSmallRows * 32];
    uint8_t ok[kSmallRows * 32];                   // the pair survives (and is its row's first of e)
    uint8_t live[kSmallRows];
    int warp_sums[32];
    int s_dup, s_nl;
};

// The small-call scatter by the whole CTA (every thread calls it; written for
// kSmallThreads threads, correct for any multiple of 32).
__device__ __forceinline__ void scatter_small(const ScatterArgs& a, ScatterSmallSmem& sm) {
    const int tid = threadIdx.x;
    const int E = a.E, k = a.k, R = a.R;
    const int words = (E + 31) >> 5;
    // 1. inputs: slot lists, liveness, the keep words of each row's block
    for (int i = tid; i < R * k; i += blockDim.x) {
        sm.ids[i] = a.topk_idx[i];
        sm.w[i] = a.w_renorm[i];
    }
    for (int i = tid; i < R * words; i += blockDim.x) {
        const int r = i / words, wd = i - r * words;
        sm.keepw[r][wd] = a.keep[(size_t)find_block(a.off, a.nb, r) * words + wd];
    }
    if (tid < R) sm.live[tid] = !a.live || a.live[tid] != 0;
    for (int e = tid; e < E; e += blockDim.x) sm.mask[e] = 0u;
    if (tid == 0) sm.s_dup = 0;
    __syncthreads();
    // 2. a thread per (row, slot): the pair survives if its row is live, its
    // expert valid and kept for the row's block, and no earlier slot of the
    // row names the same expert; warp 0 lists the live rows (the shared
    // expert's rows) in order
    for (int i = tid; i < R * k; i += blockDim.x) {
        const int r = i / k, j = i - r * k;
        const int e = sm.ids[i];
        const bool kept = sm.live[r] && e >= 0 && e < E && ((sm.keepw[r][e >> 5] >> (e & 31)) & 1u);
        bool dup = false;
        if (kept)
            for (int jj = 0; jj < j; ++jj) dup |= sm.ids[r * k + jj] == e;
        const bool ok = kept && !dup;
        sm.ok[i] = ok;
        if (ok) atomicOr(&sm.mask[e], 1u << r);
        else a.inv[i] = -1;
        if (dup) atomicAdd(&sm.s_dup, 1);
    }
    if (tid < 32) {
        const bool lv = tid < R && sm.live[tid];
        const uint32_t m = __ballot_sync(0xffffffffu, lv);
        const int pos = __popc(m & ((1u << tid) - 1u));
        if (tid < R) a.shared_inv[tid] = lv ? pos : -1;
        if (lv) a.shared_rows[pos] = tid;
        if (tid == 0) sm.s_nl = __popc(m);
    }
    __syncthreads();
    // 3. per expert: its pair count, and (one scan of count << 16 | non-empty)
    // its place in the pair list and its chunk index
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int packed = 0;
    for (int e = e0; e < e1; ++e) {
        const int n = __popc(sm.mask[e]);
        packed += n << 16 | (n > 0);
    }
    int tot;
    int before = block_excl_scan_i32(packed, sm.warp_sums, &tot);
    for (int e = e0; e < e1; ++e) {
        const int n = __popc(sm.mask[e]);
        const int pp = before >> 16, ch = before & 0xFFFF;
        sm.off[e] = pp;
        if (n) sm.chunk_exp[ch] = e;
        a.expert_off[e] = pp;
        a.count[e] = n;
        before += n << 16 | (n > 0);
    }
    const int tot_pairs = tot >> 16, nch = tot & 0xFFFF;
    __syncthreads();
    // 4. the pair lists, then the unit lists (consecutive threads write
    // consecutive entries): the shared expert's chunk first, then one chunk
    // per non-empty expert, each as its weight tiles in order
    for (int i = tid; i < R * k; i += blockDim.x) {
        if (!sm.ok[i]) continue;
        const int r = i / k, e = sm.ids[i];
        const int pos = sm.off[e] + __popc(sm.mask[e] & ((1u << r) - 1u));
        a.pair_row[pos] = r;
        a.pair_w[pos] = sm.w[i];
        a.inv[i] = pos;
    }
    const int nl = sm.s_nl;
    const int s_chunks = nl > 0 ? 1 : 0;   // nl <= kSmallRows <= nt
    const int mt_gu = (a.I + a.gu_rows - 1) / a.gu_rows, mt_gs = (a.Is + a.gu_rows - 1) / a.gu_rows;
    const int mt_dn = a.H / a.dn_cols;
    const int base_gu = s_chunks * mt_gs, base_dn = s_chunks * mt_dn;
    const int n_gu = base_gu + nch * mt_gu, n_dn = base_dn + nch * mt_dn;
    for (int u = tid; u < n_gu + n_dn; u += blockDim.x) {
        const bool gu = u < n_gu;
        const int v = gu ? u : u - n_gu;
        const int base = gu ? base_gu : base_dn, mt = gu ? mt_gu : mt_dn;
        int4 un;
        if (v < base) {
            un = make_int4(E, v, 0, nl);
        } else {
            const int c = (v - base) / mt, m = (v - base) - c * mt;
            const int g = sm.chunk_exp[c];
            un = make_int4(g, m, sm.off[g], __popc(sm.mask[g]));
        }
        if (gu) a.units_gu[v] = un;
        else a.units_dn[v] = un;
    }
    if (tid == 0) {
        a.expert_off[E] = tot_pairs;
        a.misc[1] = n_gu;
        a.misc[2] = n_dn;
        a.misc[3] = tot_pairs;
        a.misc[4] = 0;  // no staged output scaled yet (the down GEMM sets it)
        status_add(a.status, MOE_STATUS_BAD_EXPERT_ID, (uint32_t)sm.s_dup);
    }
}

}  // namespace moe
