// Shared device helpers of libmoeblock: status counters, workspace layout and
// thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor) and the
// 5th-generation tensor core (tcgen05 + TMEM) on sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_block.h"

namespace moe {

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the caller's workspace base).  Every
// region starts on a 1024-byte boundary (TMA needs 16 B; 1 KB keeps rows of
// the bf16 staging buffers on swizzle-atom boundaries).

struct Layout {
    size_t status;       // uint32[MOE_STATUS_WORDS]
    size_t route_cnt;    // uint32[max_rows]          router row / row-group tickets
    size_t logits;       // fp32 [max_rows, E]        router logits (before bias)
    size_t wnorm;        // fp32 [E]                  |w_e|_2
    size_t prank;        // int32 [max_pairs]         pair rank within (block, expert)
    size_t hist;         // int32 [max_blocks, E]     pairs per (block, expert) / bases
    size_t count;        // int32 [E]                 surviving pairs per expert
    size_t expert_off;   // int32 [E + 1]
    size_t misc;         // int32[16]: [0] ticket, [1] units gate/up, [2] units down, [3] pairs,
                         // [4] set when a staged output quarter needed an exponent
    size_t units_gu;     // int4 [max_units_gu]
    size_t units_dn;     // int4 [max_units_dn]
    size_t pair_row;     // int32 [max_pairs]
    size_t pair_w;       // fp32 [max_pairs]
    size_t h;            // bf16 [max_pairs, I]       routed SwiGLU activations
    size_t hs;           // bf16 [max_rows, 2Is]      shared-expert activations, hi | lo
    size_t inv;          // int32 [max_pairs]         staging row of each (row, slot)
    size_t shared_rows;  // int32 [max_rows]          live rows in order (the shared expert's rows)
    size_t shared_inv;   // int32 [max_rows]          index of a row in shared_rows, or -1 (dead)
    size_t live_base;    // int32 [max_blocks]        live rows of a block, then rows before it
    size_t ys;           // fp16 [max_pairs + max_rows, H] staged per-pair and shared outputs
    size_t ysx;          // uint8 [H / 32, max_pairs + max_rows] power-of-two exponent of each
                         // 32-column quarter of a staged row (ys holds value * 2^-exponent)
    size_t total;
    int64_t max_pairs, max_units_gu, max_units_dn;
};

// Rows of x per unit of grouped-GEMM work.  A call with few rows uses kSmallN
// for both GEMMs (the MMA N extent); otherwise the gate/up GEMM takes kLargeNGU
// rows per unit (a CTA pair, 128 rows of x each as the MMA's M) and the down
// GEMM kLargeNDown (its N extent).
constexpr int kSmallN = 32;
constexpr int kLargeNGU = 256;
constexpr int kLargeNDown = 256;
// Calls of up to this many rows run the down GEMM in the streaming shape
// (kSmallN rows per unit) even when the gate/up GEMM runs on CTA pairs.
constexpr int kStreamDownRows = 512;

// Large-batch router: calls of at least kTcRouteMinRows rows screen with the
// tensor cores.  Few rows give few 128-row tiles, so the screen splits H over
// several CTAs per tile; its partial logits ([parts][R, E]) take at most
// kTcSplitRows rows' worth of the logits region.
constexpr int kTcRouteMinRows = 256;
constexpr int kTcSplitRows = 16384;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Rows of E fp32 logits the workspace holds for plans of up to max_rows rows.
inline int64_t logit_rows(int64_t max_rows) {
    if (max_rows < kTcRouteMinRows) return max_rows;
    const int64_t r8 = 8 * max_rows;
    return r8 < kTcSplitRows ? r8 : (max_rows > kTcSplitRows ? max_rows : kTcSplitRows);
}

inline Layout make_layout(const moe_dims& d) {
    Layout L{};
    const int64_t R = d.max_rows, E = d.E, H = d.H;
    const int64_t P = R * d.k;
    // Unit counts with the smaller chunk size bound both kernel shapes.
    const int64_t chunks = (P + kSmallN - 1) / kSmallN + E;
    const int64_t schunks = (R + kSmallN - 1) / kSmallN;
    L.max_pairs = P;
    L.max_units_gu = chunks * (d.I / 64) + schunks * (d.Is / 64);
    L.max_units_dn = (chunks + schunks) * (H / 128);
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 1024); return at; };
    L.status = take(sizeof(uint32_t) * 64);
    L.route_cnt = take(sizeof(uint32_t) * (size_t)R);
    L.logits = take(sizeof(float) * (size_t)(logit_rows(R) * E));
    L.wnorm = take(sizeof(float) * (size_t)E);
    L.prank = take(sizeof(int32_t) * (size_t)P);
    L.hist = take(sizeof(int32_t) * (size_t)d.max_blocks * (size_t)E);
    L.count = take(sizeof(int32_t) * (size_t)E);
    L.expert_off = take(sizeof(int32_t) * (size_t)(E + 1));
    L.misc = take(sizeof(int32_t) * 16);
    L.units_gu = take(sizeof(int4) * (size_t)L.max_units_gu);
    L.units_dn = take(sizeof(int4) * (size_t)L.max_units_dn);
    L.pair_row = take(sizeof(int32_t) * (size_t)P);
    L.pair_w = take(sizeof(float) * (size_t)P);
    L.h = take(2 * (size_t)(P * d.I));
    L.hs = take(2 * (size_t)(R * 2 * d.Is));
    L.inv = take(sizeof(int32_t) * (size_t)P);
    L.shared_rows = take(sizeof(int32_t) * (size_t)R);
    L.shared_inv = take(sizeof(int32_t) * (size_t)R);
    L.live_base = take(sizeof(int32_t) * (size_t)d.max_blocks);
    L.ys = take(2 * (size_t)(P + R) * (size_t)H);
    L.ysx = take((size_t)(H / 32) * (size_t)(P + R));
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ void status_add(uint32_t* status, int word, uint32_t v) {
    if (v) atomicAdd(status + word, v);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization, so it may be scheduled while the
// kernel before it on the stream is still running.  The rule that keeps this
// safe: a thread calls pdl_wait() -- which returns once the preceding kernel
// has completed and its writes are visible -- before it reads or writes any
// global memory that another kernel writes or reads; the only thing done
// before it is reading the weights (read-only for every kernel).  pdl_trigger()
// lets the next kernel be scheduled; it is called right after the wait, so at
// most two kernels of a stream overlap.  The down GEMM on CTA pairs
// (k_down_pair, bf16 calls over kStreamDownRows rows) does not call it: the
// combine then launches when the down GEMM ends, since combine CTAs made
// resident early, waiting, slowed the down GEMM's last units (8192 rows: step
// 556 -> 545 us without the early trigger, with the four-CTA combine).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Kernel launch through cudaLaunchKernelEx (one call site style for all kernels).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-suspending test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Limits below this are the short ones a test of the failure path sets: such
// waits poll without suspending (try_wait may suspend the thread until the
// phase completes, so a short limit would rarely be seen to run out).
constexpr uint64_t kShortWaitNs = 1000000ull;

// Wait for the phase with the given parity to complete, for at most
// `limit_ns`, giving up early when another role of the CTA raised `abort`.
// Returns false when it gave up (the caller then records the timeout and
// leaves its loop); no wait in this library is unbounded.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, uint64_t limit_ns) {
    if (limit_ns < kShortWaitNs) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_test_wait(bar, parity)) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
        return true;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

// ---- cp.async (16-byte global -> shared copies, L2 only) ----------------------

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Make this thread's generic-proxy writes to shared memory visible to the
// async proxy (TMA, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA ----------------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Gather four rows (r0..r3, one-row box of the map) at column c0 into 4
// consecutive box rows of shared memory; rows out of range read as zero.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int c0, int r0,
                                            int r1, int r2, int r3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
        "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 / TMEM -------------------------------------------------------------

// Allocate `ncols` TMEM columns (power of two >= 32); the whole warp calls it.
// The allocated base address is written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major bf16 operand stored as rows of
// 128 bytes (64 elements) in the 128-byte swizzle pattern TMA writes; groups of
// 8 rows (1 KB) follow each other, so the stride-dimension offset is 1024 B.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
    d |= (uint64_t)1 << 16;                          // leading-dim offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;               // stride-dim offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                          // descriptor version (tcgen05)
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major, shape M x N.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
    uint32_t d = 0;
    d |= 1u << 4;                          // D format: f32
    d |= 1u << 7;                          // A format: bf16
    d |= 1u << 10;                         // B format: bf16
    d |= (uint32_t)(N >> 3) << 17;         // N / 8
    d |= (uint32_t)(M >> 4) << 24;         // M / 16
    return d;
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// As tc_mma_bf16 with A read from tensor memory: M = 128 rows in lanes 0..127
// from column a_tmem on, each 32-bit column holding two consecutive K
// elements of its row (the lower K index in the low half), K-major.
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 16 columns of 32-bit TMEM data from registers: thread i of the
// warp writes lane (base lane + i), columns col .. col+15.  Completion is
// awaited with tmem_st_wait.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 16 columns of 32-bit TMEM data: thread i of the warp receives
// lane (base lane + i), columns col .. col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Sixteen single columns cols[j] (the same in every lane) of a 32-lane TMEM
// slice, one wait.
__device__ __forceinline__ void tmem_ld_cols16(uint32_t taddr, const int* cols, float* v) {
    uint32_t r[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                     : "=r"(r[j])
                     : "r"(taddr + (uint32_t)cols[j]));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 32-lane x 16-column loads (e.g. the gate and the up accumulator of the
// same rows), one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
    uint32_t r[16], q[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(ta));
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]),
          "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]),
          "=r"(q[13]), "=r"(q[14]), "=r"(q[15])
        : "r"(tb));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(q[i]);
    }
}

// ---- small math ---------------------------------------------------------------

// Units of a persistent GEMM in balanced rounds: with U units and G resident
// CTAs (or CTA pairs) the launch needs ceil(U / G) rounds; spreading the units
// over the fewest workers that still finish in that many rounds gives every
// active worker the same count (to within one) instead of leaving most of them
// idle during a short last round.  Worker i takes units i, i + n, i + 2n, ...
// with n = active_workers(U, G); workers i >= n take none.
__device__ __forceinline__ int active_workers(int units, int workers) {
    if (units <= 0 || workers <= 0) return 0;
    const int rounds = (units + workers - 1) / workers;
    return (units + rounds - 1) / rounds;
}

// silu(g) = g / (1 + e^-g) with the fast exponential and division intrinsics:
// relative error near 2^-21, far below the bf16 rounding (2^-9) that h gets
// next.  Below g = -87 the quotient is 0 (the exact value is under 1e-36);
// NaN stays NaN.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ int find_block(const int32_t* off, int nb, int r) {
    // largest b in [0, nb) with off[b] <= r (off need not be valid: result is clamped)
    int lo = 0, hi = nb - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(off + mid) <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace moe
