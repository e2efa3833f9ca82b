// Device code of the forward bookkeeping shared by the scatter kernels
// (scatter.cu) and the fused front end of small calls: block scans, the GEMM
// unit lists, and the whole small-call scatter in one CTA.
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
// so the counts and the lists always agree.
constexpr int kSmallThreads = 512;

// Shared memory of the small-call scatter.
struct ScatterSmallSmem {
    uint8_t s_slot[kSmallRows][kMaxExperts];
    int s_cnt[kMaxExperts];
    int warp_sums[32];
    // the inputs, read before anything is written: a load issued after a store
    // to memory that may alias waits for it, and the per-expert loops below
    // would pay one round trip per pair
    int32_t s_ids[kSmallRows * 32];
    float s_w[kSmallRows * 32];
    int s_blk[kSmallRows];
    uint8_t s_live[kSmallRows];
    int s_dup, s_nl;
};

// The small-call scatter by the whole CTA (every thread calls it; written for
// kSmallThreads threads, correct for any multiple of 32).
__device__ __forceinline__ void scatter_small(const ScatterArgs& a, ScatterSmallSmem& sm) {
    // slot of expert e in row r (< 32), kFree (kept for r's block, no slot yet)
    // or kDropped (not kept)
    constexpr uint8_t kFree = 0xFF, kDropped = 0xFE;
    auto& s_slot = sm.s_slot;
    int* s_cnt = sm.s_cnt;
    int* warp_sums = sm.warp_sums;
    int32_t* s_ids = sm.s_ids;
    float* s_w = sm.s_w;
    int* s_blk = sm.s_blk;
    uint8_t* s_live = sm.s_live;
    int& s_dup = sm.s_dup;
    int& s_nl = sm.s_nl;
    const int tid = threadIdx.x;
    const int E = a.E, k = a.k, R = a.R;
    const int words = (E + 31) >> 5;
    if (tid < R) {
        s_blk[tid] = find_block(a.off, a.nb, tid);
        s_live[tid] = !a.live || a.live[tid] != 0;
    }
    for (int i = tid; i < R * k; i += blockDim.x) {
        s_ids[i] = a.topk_idx[i];
        s_w[i] = a.w_renorm[i];
    }
    if (tid == 0) s_dup = 0;
    __syncthreads();
    for (int i = tid; i < R * words; i += blockDim.x) {   // one keep word per thread
        const int r = i / words, wd = i - r * words;
        const uint32_t kw = a.keep[(size_t)s_blk[r] * words + wd];
        for (int bit = 0; bit < 32 && wd * 32 + bit < E; ++bit)
            s_slot[r][wd * 32 + bit] = ((kw >> bit) & 1u) ? kFree : kDropped;
    }
    if (tid < 32) {  // live rows in order (R <= 32): the shared expert's rows
        const bool lv = tid < R && s_live[tid];
        const uint32_t m = __ballot_sync(0xffffffffu, lv);
        if (tid == 0) s_nl = __popc(m);
    }
    __syncthreads();
    if (tid < R) {
        int pos = 0;
        for (int r = 0; r < tid; ++r) pos += s_live[r];
        a.shared_inv[tid] = s_live[tid] ? pos : -1;
        if (s_live[tid]) a.shared_rows[pos] = tid;
    }
    const int nl = s_nl;
    // one thread per row: mark its surviving slots (first slot wins); dead rows none
    for (int r = tid; r < R; r += blockDim.x) {
        const bool lv = s_live[r];
        int dup = 0;
        for (int j = 0; j < k; ++j) {
            a.inv[(size_t)r * k + j] = -1;
            const int e = s_ids[r * k + j];
            if (!lv || e < 0 || e >= E) continue;
            const uint8_t st = s_slot[r][e];
            if (st == kDropped) continue;
            if (st != kFree) { ++dup; continue; }
            s_slot[r][e] = (uint8_t)j;
        }
        if (dup) atomicAdd(&s_dup, dup);
    }
    __syncthreads();
    // per expert: its rows (walk the rows in order)
    for (int e = tid; e < E; e += blockDim.x) {
        int n = 0;
        for (int r = 0; r < R; ++r) n += s_slot[r][e] < 32;
        s_cnt[e] = n;
    }
    __syncthreads();
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int sum = 0, ch = 0;
    for (int f = e0; f < e1; ++f) {
        sum += s_cnt[f];
        ch += (s_cnt[f] + a.nt_gu - 1) / a.nt_gu;
    }
    int tot_pairs, tot_ch;
    int pp = block_excl_scan_i32(sum, warp_sums, &tot_pairs);
    int cc = block_excl_scan_i32(ch, warp_sums, &tot_ch);
    const int mt_gu = (a.I + a.gu_rows - 1) / a.gu_rows, mt_gs = (a.Is + a.gu_rows - 1) / a.gu_rows;
    const int mt_dn = a.H / 128;
    const int s_chunks = (nl + a.nt_gu - 1) / a.nt_gu;   // nt_gu == nt_dn here
    const int base_gu = s_chunks * mt_gs, base_dn = s_chunks * mt_dn;
    if (tid == 0) {
        write_units(a.units_gu, 0, E, 0, nl, a.nt_gu, mt_gs);
        write_units(a.units_dn, 0, E, 0, nl, a.nt_dn, mt_dn);
    }
    for (int f = e0; f < e1; ++f) {
        const int n = s_cnt[f];
        a.expert_off[f] = pp;
        a.count[f] = n;
        write_units(a.units_gu, base_gu + cc * mt_gu, f, pp, n, a.nt_gu, mt_gu);
        write_units(a.units_dn, base_dn + cc * mt_dn, f, pp, n, a.nt_dn, mt_dn);
        int pos = pp;
        for (int r = 0; r < R && pos < pp + n; ++r) {
            const int j = s_slot[r][f];
            if (j >= 32) continue;
            a.pair_row[pos] = r;
            a.pair_w[pos] = s_w[r * k + j];
            a.inv[(size_t)r * k + j] = pos;
            ++pos;
        }
        pp += n;
        cc += (n + a.nt_gu - 1) / a.nt_gu;
    }
    if (tid == 0) {
        a.expert_off[E] = tot_pairs;
        a.misc[1] = base_gu + tot_ch * mt_gu;
        a.misc[2] = base_dn + tot_ch * mt_dn;
        a.misc[3] = tot_pairs;
        a.misc[4] = 0;  // no staged output scaled yet (the down GEMM sets it)
        status_add(a.status, MOE_STATUS_BAD_EXPERT_ID, (uint32_t)s_dup);
    }
}

}  // namespace moe
