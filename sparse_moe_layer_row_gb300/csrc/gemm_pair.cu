// Gate/up GEMM (k_gateup_pair) and down GEMM (k_down_pair, below) for many
// rows per expert on CTA pairs (tcgen05 cta_group::2).
//
// The same SwiGLU first half as k_gemm<kGateUp> (model card "Clover-35B-A3B-
// Preview -- CMF", intro: 256 routed experts plus a shared expert), for units
// of up to 256 rows of x.  Two CTAs on neighbouring SMs form a cluster and
// run one MMA of M = 256, N = 256 per K = 16:
//
//   A (M = 256): rows of x, 128 in each CTA's shared memory (rank r holds
//                rows 128 r .. 128 r + 127 of the unit), gathered by 16-byte
//                cp.async from the loader warps;
//   B (N = 256): the tile's 128 gate rows in rank 0 and its 128 up rows in
//                rank 1, loaded by TMA;
//   D:           each CTA's TMEM holds its own 128 rows of x: columns 0..127
//                are g, 128..255 are u of the tile's 128 intermediate indices.
//
// An M = 128 MMA on one SM reads 16 KB of x and 32 KB of weights per 64-wide
// K step; here each SM reads 16 KB + 16 KB for the same work, so the pair
// needs two thirds of the operand bandwidth from L2 per flop.
//
// Roles (352 threads per CTA):
//   warp 0 lane 0   TMA producer of the CTA's weight half, completing on the
//                   CTA's own `full` barrier
//   warp 1          TMEM allocation (both ranks); lane 0 of rank 0 issues the
//                   MMAs and the commits, which arrive on the barriers of both
//                   ranks (stage `empty`, accumulator `tfull`)
//   warps 2..5      epilogue: TMEM -> silu(g) * u -> h (bf16; hi + lo bf16 for
//                   the shared expert) in 16-byte stores; release the
//                   accumulator on rank 0's `tempty`
//   warps 6..9      loaders: the CTA's rows of x into its x slot; each
//                   thread's copies arrive on its own CTA's `bfull` when they
//                   land (cp.async.mbarrier.arrive), so a loader never waits
//                   for its own copies and the ring depth is the only limit on
//                   the copies in flight
//   warp 10 lane 0  forwarder: waits for the CTA's `bfull` and `full` of a
//                   stage, fences the CTA's x tile for the async proxy and
//                   arrives on rank 0's `pfull` (two arrivals per stage, one
//                   per rank); the MMA thread waits for `pfull` alone, so no
//                   fence and only one wait sit between its stages.
// Each stage holds a weight half and an x tile (32 KB); both are freed by the
// same commit.  Every wait is bounded; a role that gives up raises the CTA's
// abort flag and the device status counter, and both CTAs leave their loops.
// Before the final cluster barrier, aborted or not, each CTA's producer waits
// for the `full` phase of the last fill of every stage (each CTA's weight
// copies complete on its own barrier, so it can see that they landed), the
// loaders wait for their own copies, and rank 0's MMA thread commits once more
// to a drain barrier and waits for it; only then is the TMEM released.
#include "kernels.cuh"

namespace moe {

namespace {

constexpr uint64_t kPairWaitNs = 2000000000ull;   // 2 s: far beyond any legal wait
constexpr uint64_t kPairDrainNs = 200000000ull;   // 0.2 s when draining after an abort

constexpr int kPStages = 7;
constexpr int kPThreads = 352;
constexpr int kPTile = 128 * 128;        // 128 rows x 64 bf16 (one SW128 tile)
constexpr int kPStageBytes = 2 * kPTile; // weight half, then x
constexpr int kPBarOff = kPStages * kPStageBytes;
constexpr int kPSmem = kPBarOff + 512 + 1024;
constexpr int kPAccCols = 256;
constexpr int kPTmemCols = 512;
static_assert(kPSmem <= 227 * 1024, "shared memory budget");
static_assert(8 * (4 * kPStages + 5) + 12 <= 512, "barrier region");

// ---- cluster / CTA-pair PTX -----------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// All threads of both CTAs.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of either CTA of the pair (cluster address), with the
// instruction's default semantics (release at CTA scope).  A cluster-scope
// release here measured about 1,500 cycles per arrival under load (it waits
// for the SM's memory operations in flight) and serialised the stage ring.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait with cluster-scope acquire (arrivals from the peer CTA); short
// limits poll without suspending, as in mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          volatile int* abort, uint64_t limit_ns) {
    const uint32_t addr = smem_u32(bar);
    if (limit_ns < kShortWaitNs) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_test_wait_cluster(addr, parity)) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
        return true;
    }
    if (mbar_try_wait_cluster(addr, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(addr, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at `bar`'s offset in both CTAs of the pair once every
// MMA issued so far by this thread completes.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

// Arrive on `bar` of this CTA only, once every MMA issued so far by this
// thread completes.
__device__ __forceinline__ void tc_commit_pair_local(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Arrive on `bar` once all cp.async copies issued so far by this thread have
// landed; the arrival counts toward the barrier's expected count.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// L2 eviction policies for cache-hinted copies: the weight stream of the
// CTA-pair gate/up GEMM (the routed experts' tiles, each read once) goes first,
// so the gathered rows of x (each read by k experts' units at different times)
// and the shared expert's tiles (read by every chunk of rows) stay in L2.
// Without the hint about 150 MB of x were read again from DRAM at 8192 rows.
__device__ __forceinline__ uint64_t l2_policy_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void tma_load_3d_h(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                              int c2, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

}  // namespace

__global__ void __launch_bounds__(kPThreads, 1)
k_gateup_pair(const __grid_constant__ CUtensorMap tmWg, const __grid_constant__ CUtensorMap tmWu,
              const __grid_constant__ CUtensorMap tmSg, const __grid_constant__ CUtensorMap tmSu,
              GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;   // same offset in both CTAs
    uint8_t* base = smem_raw + (sbase - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + kPBarOff);  // [S] own weight half landed
    uint64_t* bfull = full + kPStages;                               // [S] own x landed (both)
    uint64_t* pfull = bfull + kPStages;                              // [S] peer's x landed (rank 0)
    uint64_t* empty = pfull + kPStages;                              // [S] stage free (both)
    uint64_t* tfull = empty + kPStages;                              // [2] accumulator ready (both)
    uint64_t* tempty = tfull + 2;                                    // [2] accumulator free (rank 0)
    uint64_t* dbar = tempty + 2;                                     // MMA drain (rank 0)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dbar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(bfull + s, 128);   // the loader threads' copies
            mbar_init(pfull + s, 2);     // the forwarders of both ranks
            mbar_init(empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull + i, 1);
            mbar_init(tempty + i, 256);  // 128 epilogue threads of each CTA
        }
        mbar_init(dbar, 1);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kPTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmWg); prefetch_tmap(&tmWu); prefetch_tmap(&tmSg); prefetch_tmap(&tmSu);
    }
    pdl_wait();   // see common.cuh
    pdl_trigger();
    const int nunits = __ldg(a.n_units);
    const int nc = active_workers(nunits, (int)cluster_count());   // balanced rounds
    const int c0 = (int)cluster_id() < nc ? (int)cluster_id() : nunits;
    const int rbase = 128 * (int)rank;   // this CTA's rows of each unit

    auto give_up = [&]() {
        if (!*abort_flag) { *abort_flag = 1; status_add(a.status, MOE_STATUS_WAIT_TIMEOUT, 1); }
    };
    const uint64_t kWaitNs = a.wait_ns ? a.wait_ns : kPairWaitNs;   // pipeline waits

    if (warp == 0) {
        // ------------------------------------------------- weight-half producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_first();   // routed weights: evict first
            const CUtensorMap* mR = leader ? &tmWg : &tmWu;
            const CUtensorMap* mS = leader ? &tmSg : &tmSu;
            int stage = 0, nfills = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = c0; ok && u < nunits; u += nc) {
                const int4 un = __ldg(a.units + u);
                if (!unit_valid(un, a, kLargeNGU, false, 128)) continue;
                const int g = un.x, m = un.y;
                for (int kb = 0; kb < (a.H >> 6); ++kb) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    const uint32_t sW = sbase + stage * kPStageBytes;
                    mbar_expect_tx(full + stage, (uint32_t)kPTile);  // this CTA's half
                    for (int hb = 0; hb < 2; ++hb) {
                        const int row = m * 128 + 64 * hb;
                        if (g == a.E) tma_load_2d(sW + hb * 64 * 128, mS, kb * 64, row, full + stage);
                        else tma_load_3d_h(sW + hb * 64 * 128, mR, kb * 64, row, g, full + stage, pol);
                    }
                    ++nfills;
                    if (++stage == kPStages) { stage = 0; phase ^= 1u; }
                }
            }
            // drain: the last fill of every stage has landed (consumed or not),
            // so no copy into this CTA's shared memory is in flight at exit
            for (int s = 0; s < kPStages; ++s) {
                if (nfills < kPStages && s >= nfills) break;
                const uint32_t par = s < stage ? phase : (phase ^ 1u);
                if (!mbar_wait_bounded(full + s, par, never, kPairDrainNs)) give_up();
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16_f32(256, 256);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = c0; ok && u < nunits; u += nc) {
                if (!unit_valid(__ldg(a.units + u), a, kLargeNGU, false, 128)) {
                    status_add(a.status, MOE_STATUS_BAD_UNIT, 1);
                    continue;
                }
                if (!mbar_wait_cluster_bounded(tempty + acc, acc_phase ^ 1u, abort_flag, kWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kPAccCols);
                for (int kb = 0; kb < (a.H >> 6); ++kb) {
                    // both ranks' x tiles and weight halves (the forwarders)
                    if (!mbar_wait_cluster_bounded(pfull + stage, phase, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sW = sbase + stage * kPStageBytes;
                    const uint32_t sX = sW + kPTile;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16_pair(d, smem_desc_sw128(sX + kk * 32), smem_desc_sw128(sW + kk * 32),
                                         idesc, (kb | kk) != 0);
                    tc_commit_pair(empty + stage);
                    if (++stage == kPStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair(tfull + acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // drain: arrives (on this CTA's barrier) once every MMA issued
            // above has completed
            tc_commit_pair_local(dbar);
            if (!mbar_wait_bounded(dbar, 0, never, kPairDrainNs)) give_up();
        }
    } else if (warp >= 6 && warp < 10) {
        // ----------------------------------------------------------- x loaders
        // Row i of the CTA's part of a unit is copied by 8 threads, 16 bytes
        // each, into the 128-byte swizzled row of the x tile: chunk c of row i
        // lands at chunk c ^ (i & 7).
        const int lt = threadIdx.x - 192;            // 0..127
        const int lw = lt >> 5, r4 = (lt & 31) >> 3, ch = lt & 7;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = c0; ok && u < nunits; u += nc) {
            const int4 un = __ldg(a.units + u);
            if (!unit_valid(un, a, kLargeNGU, false, 128)) continue;
            const int g = un.x, start = un.z + rbase;
            const int nr = min(128, max(0, un.w - rbase));
            const __nv_bfloat16* src[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = j * 16 + lw * 4 + r4;
                const int row = i >= nr ? -1
                              : g != a.E ? __ldg(a.pair_row + start + i)
                              : (a.shared_rows ? __ldg(a.shared_rows + start + i) : start + i);
                src[j] = row >= 0 ? a.x + (size_t)row * a.H + ch * 8 : nullptr;
            }
            for (int kb = 0; kb < (a.H >> 6); ++kb) {
                if (!mbar_wait_bounded(empty + stage, phase ^ 1u, abort_flag, kWaitNs)) {
                    give_up();
                    ok = false;
                    break;
                }
                const uint32_t sX = sbase + stage * kPStageBytes + kPTile;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = j * 16 + lw * 4 + r4;
                    if (src[j]) cp_async16(sX + i * 128 + ((ch ^ (i & 7)) << 4), src[j] + kb * 64);
                }
                cp_async_arrive(bfull + stage);
                if (++stage == kPStages) { stage = 0; phase ^= 1u; }
            }
        }
        cp_async_wait_all();  // nothing of this thread lands after the loop
    } else if (warp == 10) {
        if (lane == 0) {
            // ------------------------------------------- x-stage forwarder
            // Once the CTA's x tile and weight half of a stage have landed, fence
            // the x tile (written by cp.async) for the async proxy and arrive on
            // rank 0's `pfull`; the MMA thread waits for that barrier alone.
            const uint32_t pfull0 = mapa_shared(smem_u32(pfull), 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = c0; ok && u < nunits; u += nc) {
                if (!unit_valid(__ldg(a.units + u), a, kLargeNGU, false, 128)) continue;
                for (int kb = 0; kb < (a.H >> 6); ++kb) {
                    if (!mbar_wait_bounded(bfull + stage, phase, abort_flag, kWaitNs) ||
                        !mbar_wait_bounded(full + stage, phase, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    fence_proxy_async_smem();   // the x tile was written by cp.async
                    mbar_arrive_cluster(pfull0 + stage * 8);
                    if (++stage == kPStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = c0; u < nunits; u += nc) {
            const int4 un = __ldg(a.units + u);
            if (!unit_valid(un, a, kLargeNGU, false, 128)) continue;
            const int g = un.x, m = un.y, start = un.z + rbase;
            const int nr = min(128, max(0, un.w - rbase));
            const bool ok = mbar_wait_bounded(tfull + acc, acc_phase, abort_flag, kWaitNs);
            if (__any_sync(0xffffffffu, !ok)) { give_up(); break; }
            __syncwarp();
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kPAccCols);
            // lane = row t of this CTA's part: g of intermediate index m*128 + c
            // in column c, u in column 128 + c
            const bool sh = g == a.E;
            const int ld = sh ? a.Is : a.I;
            const int t = q * 32 + lane;
            __nv_bfloat16* orow = (sh ? a.hs + (size_t)(start + t) * (2 * ld)
                                      : a.h + (size_t)(start + t) * ld) + m * 128;
            const int cmax = min(128, ld - m * 128);  // intermediate indices of the tile
            for (int c = 0; c < 128; c += 16) {
                float gv[16], uv[16];
                __syncwarp();  // tcgen05.ld is warp-collective
                tmem_ld16x2(tb + (uint32_t)c, tb + (uint32_t)(128 + c), gv, uv);
                if (t < nr && c < cmax) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float h0 = silu_fast(gv[2 * j]) * uv[2 * j];
                        const float h1 = silu_fast(gv[2 * j + 1]) * uv[2 * j + 1];
                        const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
                        hi[j] = *reinterpret_cast<const uint32_t*>(&b);
                        const __nv_bfloat162 l =
                            __floats2bfloat162_rn(h0 - __low2float(b), h1 - __high2float(b));
                        lo[j] = *reinterpret_cast<const uint32_t*>(&l);
                    }
                    uint4* o = reinterpret_cast<uint4*>(orow + c);
                    o[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    o[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                    if (sh) {  // lo part: columns Is .. 2 Is - 1 of the shared row
                        uint4* ol = reinterpret_cast<uint4*>(orow + ld + c);
                        ol[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        ol[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_cluster(tempty0 + acc * 8);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA leaves while its peer may still signal or read it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kPTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Down GEMM for many pairs per expert on a CTA pair.
//
// A unit is (group g, 256 hidden outputs m, up to 256 pairs of the group).  Two
// CTAs on neighbouring SMs run one tcgen05.mma.cta_group::2 of M = 256, N = 256
// per 16 of K:
//
//   A (M = 256): h rows start + 128 r .. + 127 of the unit's pairs in rank r
//                (TMA; rows past the unit's count feed TMEM lanes that are
//                never read);
//   B (N = 256): W_down rows m * 256 + 128 r .. + 127 in rank r (TMA);
//   D:           each CTA's TMEM holds its 128 pairs x the unit's 256 hidden
//                outputs.
//
// A single-SM M = 128, N = 256 tile loads 16 KB of weights and 32 KB of h per
// 64-wide K step; here each SM loads 16 + 16 KB for the same work.  For the
// shared expert, K runs over [hi | lo] (2 Is columns of hs) while the weights
// wrap around their Is columns.  An epilogue thread owns one pair (a TMEM
// lane): it scales the pair's outputs by its renormalised weight (1 for the
// shared expert) and converts them to fp16; the warp trades its 32 pairs' rows
// through shared memory (128-byte swizzle) so that eight lanes write each
// 128-byte line of the staging rows; a quarter whose largest finite magnitude is
// 2^15 or more is stored as v * 2^-s with the smallest s that brings it below
// 2^15 (s to ysx, the call's `scaled` flag set; k_combine multiplies it back
// exactly); infinities and NaNs pass through the scaling unchanged.
//
// Roles (224 threads per CTA):
//   warp 0 lane 0   TMA producer of the CTA's weight and h halves, completing
//                   on the CTA's own `full`; the first stages' W_down tiles are
//                   issued before the wait for the gate/up GEMM (their h is
//                   held back)
//   warp 1          TMEM allocation (both ranks); lane 0 of rank 0 issues the
//                   MMAs and the commits (stage `empty`, accumulator `tfull`,
//                   multicast to both ranks)
//   warps 2..5      epilogue; the accumulator is released on rank 0's `tempty`
//   warp 6 lane 0   forwarder: waits for the CTA's `full` and arrives on rank
//                   0's `pfull` (one arrival per rank and stage), which the MMA
//                   thread waits for alone
// Waits, abort and drain as in k_gateup_pair.
constexpr int kDStages = 6;
constexpr int kDThreads = 224;
constexpr int kDStageBytes = 2 * kPTile;   // the weight half, then the h half
constexpr int kDXOff = kDStages * kDStageBytes;   // per epilogue warp: 32 rows x 128 B
constexpr int kDBarOff = kDXOff + 4 * 32 * 128;
constexpr int kDSmem = kDBarOff + 512 + 1024;
static_assert(kDSmem <= 227 * 1024, "shared memory budget");
static_assert(8 * (3 * kDStages + 5) + 12 <= 512, "barrier region");
static_assert(kLargeNDown == 256, "N = 256: 128 pairs per rank");

__global__ void __launch_bounds__(kDThreads, 1)
k_down_pair(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
            const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmHs,
            GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;   // same offset in both CTAs
    uint8_t* base = smem_raw + (sbase - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + kDBarOff);  // [S] own halves landed
    uint64_t* pfull = full + kDStages;                               // [S] both ranks' (rank 0)
    uint64_t* empty = pfull + kDStages;                              // [S] stage free (both)
    uint64_t* tfull = empty + kDStages;                              // [2] accumulator ready (both)
    uint64_t* tempty = tfull + 2;                                    // [2] accumulator free (rank 0)
    uint64_t* dbar = tempty + 2;                                     // MMA drain (rank 0)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dbar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(pfull + s, 2);     // the forwarders of both ranks
            mbar_init(empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull + i, 1);
            mbar_init(tempty + i, 256);  // 128 epilogue threads of each CTA
        }
        mbar_init(dbar, 1);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, kPTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmW); prefetch_tmap(&tmS); prefetch_tmap(&tmH); prefetch_tmap(&tmHs);
    }
    // Every role but the producer waits for the gate/up GEMM first.  Before its
    // own wait the producer reads only the unit list (written by the scatter,
    // which the gate/up GEMM waited for before letting this kernel start) and
    // the weights.  No role triggers the combine's launch: it launches when
    // this kernel ends (common.cuh).
    if (warp != 0) pdl_wait();
    const int nunits = __ldg(a.n_units);
    const int nc = (int)cluster_count();   // plain stride: neighbouring units share h
    const int c0 = (int)cluster_id();
    const int half = 128 * (int)rank;      // this CTA's rows of A and of B

    auto give_up = [&]() {
        if (!*abort_flag) { *abort_flag = 1; status_add(a.status, MOE_STATUS_WAIT_TIMEOUT, 1); }
    };
    auto valid = [&](int4 un) { return unit_valid(un, a, kLargeNDown, true, 128, 256); };
    const uint64_t kWaitNs = a.wait_ns ? a.wait_ns : kPairWaitNs;   // pipeline waits

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            struct HeldB { uint32_t sB; const CUtensorMap* map; int kc, row; uint64_t* bar; };
            HeldB held[kDStages];
            int nheld = 0;
            bool waited = false;
            auto release_held = [&]() {
                pdl_wait();
                for (int i = 0; i < nheld; ++i)
                    tma_load_2d(held[i].sB, held[i].map, held[i].kc, held[i].row, held[i].bar);
                nheld = 0;
                waited = true;
            };
            int stage = 0, nfills = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = c0; ok && u < nunits; u += nc) {
                const int4 un = __ldg(a.units + u);
                if (!valid(un)) continue;
                const int g = un.x, m = un.y, start = un.z;
                const bool sh = g == a.E;
                const int Kw = sh ? a.Is : a.I;      // the weights' K extent
                const int K = sh ? 2 * a.Is : a.I;   // h's: [hi | lo] for the shared expert
                for (int kb = 0; kb < (K >> 6); ++kb) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    const uint32_t sW = sbase + stage * kDStageBytes, sH = sW + kPTile;
                    mbar_expect_tx(full + stage, (uint32_t)kDStageBytes);
                    const int kcw = (kb * 64) % Kw, roww = m * 256 + half;
                    if (sh) tma_load_2d(sW, &tmS, kcw, roww, full + stage);
                    else tma_load_3d(sW, &tmW, kcw, roww, g, full + stage);
                    const HeldB hb{sH, sh ? &tmHs : &tmH, kb * 64, start + half, full + stage};
                    if (waited) tma_load_2d(hb.sB, hb.map, hb.kc, hb.row, hb.bar);
                    else held[nheld++] = hb;
                    if (!waited && nheld == kDStages) release_held();
                    ++nfills;
                    if (++stage == kDStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!waited) release_held();   // every posted byte count gets its copies
            // drain: the last fill of every stage has landed (consumed or not)
            for (int s = 0; s < kDStages; ++s) {
                if (nfills < kDStages && s >= nfills) break;
                const uint32_t par = s < stage ? phase : (phase ^ 1u);
                if (!mbar_wait_bounded(full + s, par, never, kPairDrainNs)) give_up();
            }
        } else {
            pdl_wait();
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16_f32(256, 256);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = c0; ok && u < nunits; u += nc) {
                const int4 un = __ldg(a.units + u);
                if (!valid(un)) {
                    status_add(a.status, MOE_STATUS_BAD_UNIT, 1);
                    continue;
                }
                const int K = un.x == a.E ? 2 * a.Is : a.I;
                if (!mbar_wait_cluster_bounded(tempty + acc, acc_phase ^ 1u, abort_flag, kWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kPAccCols);
                for (int kb = 0; kb < (K >> 6); ++kb) {
                    // both ranks' halves of the stage (the forwarders)
                    if (!mbar_wait_cluster_bounded(pfull + stage, phase, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sW = sbase + stage * kDStageBytes, sH = sW + kPTile;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // A = pairs (h), B = hidden outputs (W)
                        tc_mma_bf16_pair(d, smem_desc_sw128(sH + kk * 32), smem_desc_sw128(sW + kk * 32),
                                         idesc, (kb | kk) != 0);
                    tc_commit_pair(empty + stage);
                    if (++stage == kDStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair(tfull + acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // drain: arrives (on this CTA's barrier) once every MMA issued
            // above has completed
            tc_commit_pair_local(dbar);
            if (!mbar_wait_bounded(dbar, 0, never, kPairDrainNs)) give_up();
        }
    } else if (warp == 6) {
        if (lane == 0) {
            // ---------------------------------------------------- forwarder
            const uint32_t pfull0 = mapa_shared(smem_u32(pfull), 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int u = c0; ok && u < nunits; u += nc) {
                const int4 un = __ldg(a.units + u);
                if (!valid(un)) continue;
                const int K = un.x == a.E ? 2 * a.Is : a.I;
                for (int kb = 0; kb < (K >> 6); ++kb) {
                    if (!mbar_wait_bounded(full + stage, phase, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster(pfull0 + stage * 8);
                    if (++stage == kDStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = c0; u < nunits; u += nc) {
            const int4 un = __ldg(a.units + u);
            if (!valid(un)) continue;
            const int g = un.x, m = un.y, start = un.z, n = un.w;
            const int pi = half + q * 32 + lane;   // this thread's pair of the unit
            const bool live = pi < n;
            const float wv = !live ? 0.0f : g == a.E ? 1.0f : __ldg(a.pair_w + start + pi);
            const bool ok = mbar_wait_bounded(tfull + acc, acc_phase, abort_flag, kWaitNs);
            if (__any_sync(0xffffffffu, !ok)) { give_up(); break; }
            __syncwarp();
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kPAccCols);
            const size_t row0 = (size_t)(g == a.E ? a.shared_row0 : 0) + start + half + q * 32;
            uint8_t* xq = a.ysx + (size_t)(m * 8) * a.ld_x + row0 + lane;   // quarter j at + j * ld_x
            uint8_t* xw = base + kDXOff + (warp - 2) * 32 * 128;   // this warp's rows
            bool any_big = false;
#pragma unroll 1
            for (int jp = 0; jp < 4; ++jp) {   // 64-column pieces of the unit's outputs
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {   // its two 32-column quarters
                    const int j = 2 * jp + hq;
                    float v[32];
                    __syncwarp();  // tcgen05.ld is warp-collective
                    tmem_ld16x2(tb + (uint32_t)(32 * j), tb + (uint32_t)(32 * j + 16), v, v + 16);
                    float mx = 0.0f;   // fmaxf skips NaN
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        v[t] *= wv;
                        mx = fmaxf(mx, fabsf(v[t]));
                    }
                    uint32_t sc = 0;
                    if (live && mx >= 32768.0f) {   // the quarter's largest finite magnitude sets s
                        uint32_t mb = 0;
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            const uint32_t ab = __float_as_uint(v[t]) & 0x7FFFFFFFu;
                            mb = max(mb, ab < 0x7F800000u ? ab : 0u);
                        }
                        const int sh = (int)(mb >> 23) - 141;   // biased exponent - (127 + 14)
                        sc = sh > 0 ? (uint32_t)sh : 0u;
                        const float f = __uint_as_float((127u - sc) << 23);   // 2^-s, exact
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] *= f;
                        any_big = true;
                    }
                    // row `lane`, 16-byte chunk c4 of the 128-byte piece at c4 ^ (lane & 7)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t w4[4];
#pragma unroll
                        for (int i2 = 0; i2 < 4; ++i2) {
                            const __half2 hv = __floats2half2_rn(v[8 * c + 2 * i2], v[8 * c + 2 * i2 + 1]);
                            w4[i2] = *reinterpret_cast<const uint32_t*>(&hv);
                        }
                        const int c4 = 4 * hq + c;
                        *reinterpret_cast<uint4*>(xw + lane * 128 + ((c4 ^ (lane & 7)) << 4)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    if (live) xq[(size_t)j * a.ld_x] = (uint8_t)sc;
                }
                __syncwarp();
                // lanes 8 i .. 8 i + 7 write row 4 s + i's 128 bytes
#pragma unroll
                for (int s4 = 0; s4 < 8; ++s4) {
                    const int r = 4 * s4 + (lane >> 3), c8 = lane & 7;
                    const uint4 val = *reinterpret_cast<const uint4*>(xw + r * 128 + ((c8 ^ (r & 7)) << 4));
                    if (half + q * 32 + r < n)
                        *reinterpret_cast<uint4*>(a.ys + (row0 + r) * a.H + m * 256 + jp * 64 + c8 * 8) = val;
                }
            }
            if (__any_sync(0xffffffffu, any_big) && lane == 0) *a.scaled = 1;
            tc_fence_before();
            mbar_arrive_cluster(tempty0 + acc * 8);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no CTA leaves while its peer may still signal or read it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kPTmemCols);
    }
}

// ---------------------------------------------------------------------------

static int g_pair_clusters = 0;   // clusters resident at once (0: not yet known)

cudaError_t gateup_pair_set_attributes(int num_sms) {
    cudaError_t e = cudaFuncSetAttribute(k_gateup_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_gateup_pair, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    g_pair_clusters = n < num_sms / 2 ? n : num_sms / 2;
    return cudaSuccess;
}

cudaError_t launch_gateup_pair(const GemmMaps& mp, const GemmArgs& a, cudaStream_t st) {
    if (g_pair_clusters <= 0) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * g_pair_clusters);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_gateup_pair, mp.a0, mp.a1, mp.a2, mp.a3, a);
}

static int g_down_clusters = 0;   // clusters resident at once (0: not yet known)

cudaError_t down_pair_set_attributes(int num_sms) {
    cudaError_t e = cudaFuncSetAttribute(k_down_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = kDSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_down_pair, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    g_down_clusters = n < num_sms / 2 ? n : num_sms / 2;
    return cudaSuccess;
}

// mp.a0 / a2: W_down and the shared W_down (128-row boxes); mp.b0 / b1: h and
// hs (128-row boxes).
cudaError_t launch_down_pair(const GemmMaps& mp, const GemmArgs& a, cudaStream_t st) {
    if (g_down_clusters <= 0) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * g_down_clusters);
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = kDSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_down_pair, mp.a0, mp.a2, mp.b0, mp.b1, a);
}

}  // namespace moe
