// Forward bookkeeping: group the surviving (row, slot) pairs by expert so each
// touched expert's weights stream once per call, build the device-side work
// lists of the grouped GEMMs, and the final bf16 store.
//
// Model card "Clover-35B-A3B-Preview -- CMF", Hardware: "the experts a block
// uses are bound as they are routed" -- here: only experts with at least one
// surviving pair appear in the work lists.
//
// Pair order inside an expert is (row ascending, slot ascending), so the work
// list, the staging copy of x and the GEMM tiles are the same on every run.
// Nothing here waits on another CTA: the per-expert counts are combined by the
// last CTA to finish (ticket counter), which then writes the offsets and the
// unit lists for the GEMM launches that follow on the same stream.
#include "kernels.cuh"

namespace moe {

constexpr int kScatThreads = 256;

// Exclusive scan of one int per thread over the block; *total gets the sum.
__device__ int block_excl_scan_i32(int v, int* warp_sums, int* total) {
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

// Row -> block map, zeroed combine accumulator, reset ticket.
__global__ void k_fwd_prep(ScatterArgs a) {
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t nth = (size_t)gridDim.x * blockDim.x;
    for (size_t r = tid; r < (size_t)a.R; r += nth) a.row_block[r] = find_block(a.off, a.nb, (int)r);
    const size_t n4 = (size_t)a.R * a.H / 4;
    float4* y4 = reinterpret_cast<float4*>(a.y32);
    for (size_t i = tid; i < n4; i += nth) y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0) a.misc[0] = 0;
}

__device__ __forceinline__ int slots_for(const ScatterArgs& a, int r, int e) {
    const int b = a.row_block[r];
    const int words = (a.E + 31) >> 5;
    if (!((__ldg(a.keep + (size_t)b * words + (e >> 5)) >> (e & 31)) & 1u)) return 0;
    int c = 0;
    for (int j = 0; j < a.k; ++j) c += __ldg(a.topk_idx + (size_t)r * a.k + j) == e;
    return c;
}

// Units of one group: chunks of nt pairs x weight tiles; chunk-major so the
// CTAs that run neighbouring units share the same rows of x (L2 reuse).
__device__ void write_units(int4* out, int base, int g, int start, int n, int nt, int mtiles) {
    int u = base;
    for (int c0 = 0; c0 < n; c0 += nt) {
        const int cn = min(nt, n - c0);
        for (int m = 0; m < mtiles; ++m) out[u++] = make_int4(g, m, start + c0, cn);
    }
}

// One CTA per expert: count its surviving pairs; the last CTA builds offsets and units.
__global__ void __launch_bounds__(kScatThreads) k_scatter_count(ScatterArgs a) {
    __shared__ int warp_sums[32];
    __shared__ int s_last;
    const int e = blockIdx.x;
    int c = 0;
    for (int r = threadIdx.x; r < a.R; r += blockDim.x) c += slots_for(a, r, e);
    int total;
    (void)block_excl_scan_i32(c, warp_sums, &total);
    if (threadIdx.x == 0) {
        a.count[e] = total;
        __threadfence();
        s_last = atomicAdd(a.misc, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // --- last CTA: offsets over experts, then the unit lists ---
    const int E = a.E;
    const int mt_gu = a.I / 64, mt_gs = a.Is / 64, mt_dn = a.H / 128;
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, (int)threadIdx.x * per), e1 = min(E, e0 + per);
    int sum = 0, ch_gu = 0, ch_dn = 0;
    for (int f = e0; f < e1; ++f) {
        const int n = __ldcg(a.count + f);
        sum += n;
        ch_gu += (n + a.nt_gu - 1) / a.nt_gu;
        ch_dn += (n + a.nt_dn - 1) / a.nt_dn;
    }
    int tot_pairs, tot_gu, tot_dn;
    int p = block_excl_scan_i32(sum, warp_sums, &tot_pairs);
    int cg = block_excl_scan_i32(ch_gu, warp_sums, &tot_gu);
    int cd = block_excl_scan_i32(ch_dn, warp_sums, &tot_dn);
    // shared expert (group E) first: it has the most rows
    const int base_gu = (a.R + a.nt_gu - 1) / a.nt_gu * mt_gs;
    const int base_dn = (a.R + a.nt_dn - 1) / a.nt_dn * mt_dn;
    if (threadIdx.x == 0) {
        write_units(a.units_gu, 0, E, 0, a.R, a.nt_gu, mt_gs);
        write_units(a.units_dn, 0, E, 0, a.R, a.nt_dn, mt_dn);
    }
    for (int f = e0; f < e1; ++f) {
        const int n = __ldcg(a.count + f);
        a.expert_off[f] = p;
        write_units(a.units_gu, base_gu + cg * mt_gu, f, p, n, a.nt_gu, mt_gu);
        write_units(a.units_dn, base_dn + cd * mt_dn, f, p, n, a.nt_dn, mt_dn);
        p += n;
        cg += (n + a.nt_gu - 1) / a.nt_gu;
        cd += (n + a.nt_dn - 1) / a.nt_dn;
    }
    if (threadIdx.x == 0) {
        a.expert_off[E] = tot_pairs;
        a.misc[1] = base_gu + tot_gu * mt_gu;
        a.misc[2] = base_dn + tot_dn * mt_dn;
        a.misc[3] = tot_pairs;
        a.misc[0] = 0;
    }
}

// One CTA per expert: pair lists in (row, slot) order and the staged rows of x.
__global__ void __launch_bounds__(kScatThreads) k_scatter_fill(ScatterArgs a) {
    __shared__ int warp_sums[32];
    __shared__ int list_row[kScatThreads * 4];
    __shared__ int list_pos[kScatThreads * 4];
    const int e = blockIdx.x;
    const int n_e = a.count[e];
    if (n_e == 0) return;
    int pos0 = a.expert_off[e];
    const int hv = a.H / 8;  // uint4 per row of x
    for (int r0 = 0; r0 < a.R; r0 += blockDim.x) {
        const int r = r0 + threadIdx.x;
        const int c = r < a.R ? slots_for(a, r, e) : 0;
        int total;
        int pos = pos0 + block_excl_scan_i32(c, warp_sums, &total);
        if (c) {
            int li = pos - pos0;
            for (int j = 0; j < a.k; ++j) {
                if (a.topk_idx[(size_t)r * a.k + j] != e) continue;
                a.pair_row[pos] = r;
                a.pair_w[pos] = a.w_renorm[(size_t)r * a.k + j];
                if (li < kScatThreads * 4) { list_row[li] = r; list_pos[li] = pos; }
                ++pos;
                ++li;
            }
        }
        __syncthreads();
        // copy the listed rows of x (total may exceed the list only with duplicate ids)
        const int listed = min(total, kScatThreads * 4);
        for (int i = threadIdx.x; i < listed * hv; i += blockDim.x) {
            const int l = i / hv, v = i - l * hv;
            const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)list_row[l] * a.H);
            uint4* dst = reinterpret_cast<uint4*>(a.xp + (size_t)list_pos[l] * a.H);
            dst[v] = __ldg(src + v);
        }
        if (total > kScatThreads * 4) {
            // rare: more pairs than the list holds; copy the rest straight from the pair list
            for (int i = threadIdx.x + listed * hv; i < total * hv; i += blockDim.x) {
                const int l = i / hv, v = i - l * hv;
                const int pp = pos0 + l;
                const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)a.pair_row[pp] * a.H);
                reinterpret_cast<uint4*>(a.xp + (size_t)pp * a.H)[v] = __ldg(src + v);
            }
        }
        pos0 += total;
        __syncthreads();
    }
}

__global__ void k_finalize(FinalArgs a) {
    const size_t n4 = a.n / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.y32) + i);
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(a.y)[i] = packed;
        if (a.y_f32) reinterpret_cast<float4*>(a.y_f32)[i] = v;
    }
}

cudaError_t launch_scatter(const ScatterArgs& a, int num_sms, cudaStream_t st) {
    const size_t work = (size_t)a.R * a.H / 4;
    long blocks = (long)((work + 255) / 256);
    if (blocks > (long)num_sms * 8) blocks = (long)num_sms * 8;
    if (blocks < 1) blocks = 1;
    k_fwd_prep<<<(unsigned)blocks, 256, 0, st>>>(a);
    k_scatter_count<<<a.E, kScatThreads, 0, st>>>(a);
    k_scatter_fill<<<a.E, kScatThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalArgs& a, int num_sms, cudaStream_t st) {
    long blocks = (long)((a.n / 4 + 255) / 256);
    if (blocks > (long)num_sms * 8) blocks = (long)num_sms * 8;
    if (blocks < 1) blocks = 1;
    k_finalize<<<(unsigned)blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
