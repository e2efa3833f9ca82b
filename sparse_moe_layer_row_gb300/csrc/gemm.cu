// Grouped SwiGLU expert GEMMs on the 5th-generation tensor core (sm_103a).
//
// Expert e computes W_down[e] (silu(W_gate[e] x) * (W_up[e] x)) for every row
// x routed to it (model card "Clover-35B-A3B-Preview -- CMF", intro: top-8 of
// 256 experts plus a shared expert; the shared expert is one more group).
//
// Orientation ("weights as M"): a unit of work is (group g, weight tile m,
// a chunk of at most NMAX rows of x).  The MMA is D[128 x N] = A[128 x K] B^T
// with A = 128 weight rows (K-major, straight from the [E, rows, K] weight
// tensor by a 3-D TMA box whose outer coordinate is the expert id) and
// B = N rows of activations (K-major).  So each touched expert's weights
// stream through shared memory once per launch, whatever the number of rows
// routed to it, and N only has to be a multiple of 16.
//
//  gate/up:  A rows 0..63 = gate rows, 64..127 = up rows of the same 64
//            intermediate indices (two 64-row TMA boxes per stage).  TMEM lane
//            quadrants 0-1 hold g, 2-3 hold u; the epilogue warps trade half
//            of each 16-column chunk through shared memory and each computes
//            h = silu(g) * u for its half.  Routed pairs store h in bf16; the
//            shared expert, whose output enters every row with weight 1,
//            stores two bf16 parts hi = bf16(h), lo = bf16(h - hi) (about 16
//            significant bits).  The rounding of h is the largest error of
//            the path: a routed pair's share of it is scaled by the pair's
//            weight (the weights of a row sum to 1), the shared expert's is
//            not, and one bf16 part there too would leave almost no margin in
//            the output tolerance.
//  down:     A = 128 rows of W_down[e] (hidden outputs), B = rows of h.  For
//            the shared expert, D = W (h_hi + h_lo): both parts of h are loaded
//            in one stage and two MMAs are issued per K step (W read once).
//            The epilogue scales by the pair's renormalised weight
//            and stages the pair's output row in fp16 (the shared expert with
//            weight 1, in its own rows), with a power-of-two exponent per 32
//            columns for values beyond fp16's range; k_combine sums the rows.
// This kernel is the streaming shape: units of up to 32 rows, the weights
// streamed once per call.  With many rows per expert both GEMMs run on CTA
// pairs (gemm_pair.cu); calls of up to 512 rows keep this down GEMM.
//
// Pipeline (two CTAs per SM, persistent over the unit list):
//   warp 0 lane 0  TMA producer: STAGES-deep ring of (A tile, B tile) stages
//   warp 1 lane 0  MMA issuer: 4 x tcgen05.mma (K = 16 each) per 64-wide stage,
//                  tcgen05.commit frees the stage; accumulators double-buffered
//                  in TMEM so the epilogue of one unit overlaps the next unit
//   warps 2..5     epilogue: tcgen05.ld 32 lanes x 16 columns, math, stores
// Every wait is bounded (see mbar_wait_bounded): a wait that gives up raises
// a CTA-wide abort flag and a device status counter; all roles then leave
// their loops.  Before the CTA exits, whether it aborted or not, the producer
// waits for the `full` phase of the last fill of every stage (a TMA copy
// completes whether or not the MMA consumes it, so no copy is left in flight)
// and the MMA thread commits once more to a drain barrier and waits for it
// (every MMA it issued has completed); only then is the TMEM released.  These
// drain waits have their own limit, apart from the pipeline waits'.
#include "kernels.cuh"

namespace moe {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any legal wait
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s when draining after an abort

template <int MODE, int NMAX, int STAGES, int QB = 0>
struct GemmCfg {
    // the streaming shape only (many rows per expert run on CTA pairs,
    // gemm_pair.cu); gate/up: 64 gate + 64 up rows in one 128-row A tile, g and
    // u traded in the epilogue
    static_assert(NMAX == kSmallN, "the streaming shape; many rows run in gemm_pair.cu");
    static constexpr int kGURows = 64;  // intermediate rows per gate/up unit
    // rows per B box: the gate/up GEMM's whole 32-row tile (or all of x when a
    // call has at most 32 rows); 16 for the down GEMM's h rows.  Each TMA
    // instruction costs the producer on the order of 200 cycles to issue under
    // load, so a stage takes as few as it can.
    static constexpr int kBoxRows = MODE == kGateUp ? 32 : 16;
    static constexpr int kABytes = 128 * 128;
    // down: the shared expert's lo part of h rides in the same stage as its hi
    // part (a second MMA per K step, the weight tile read once)
    static constexpr bool kDualLo = MODE == kDown;
    static constexpr int kBBytes = (kDualLo ? 2 : 1) * NMAX * 128;
    // quantised weights (QB = 8 or 4 bits, streaming shape only): a stage holds
    // the B tile, the 128 weight rows' raw codes for its 64 K (swizzled by the
    // copy: 64-byte mode for 8 bits, 32-byte for 4) and their scales (two
    // blocks of 32 per row); converter warps dequantise the codes into one of
    // kNA bf16 A slots in tensor memory, from which the MMA reads A
    static constexpr bool kQuant = QB != 0;
    static_assert(QB == 0 || ((QB == 8 || QB == 4) && NMAX == kSmallN), "quantised: streaming shape");
    static constexpr int kRawBytes = QB == 8 ? 128 * 64 : (QB == 4 ? 128 * 32 : 0);
    static constexpr int kScaleBytes = kQuant ? 2 * 128 * 2 : 0;
    static constexpr int kNA = kQuant ? 4 : 0;
    static constexpr int kThreads = kQuant ? 320 : 192;
    static constexpr int kMinBlocks = 2;
    static constexpr int kStageBytes =
        kQuant ? (kBBytes + kRawBytes + kScaleBytes + 1023) / 1024 * 1024 : kABytes + kBBytes;
    static constexpr int kXchgOff = STAGES * kStageBytes;
    // down: pairs of the output tile staged at a time (all of them)
    static constexpr int kStageRows = NMAX;
    // gate/up: g <-> u exchange; down: fp16 output rows of kStageRows pairs
    static constexpr int kXchgBytes = MODE == kGateUp ? 2 * 64 * 9 * 4 : kStageRows * 128 * 2;
    static constexpr int kRowsOff = kXchgOff + kXchgBytes;             // gate/up: rows of x of a unit
    static constexpr int kRowsBytes = MODE == kGateUp && NMAX == kSmallN ? NMAX * 4 : 0;
    static constexpr int kBarOff = kRowsOff + kRowsBytes;
    static constexpr int kSmem = kBarOff + 512 + 1024;
    static constexpr int kAccCols = NMAX;   // TMEM columns per accumulator
    // quantised: the A slots after the two accumulators, 32 columns (64 K of
    // bf16) each
    static constexpr int kACol = 2 * kAccCols;
    static constexpr int kTmemNeed = kACol + kNA * 32;
    static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : 256;
    static_assert(kTmemNeed <= kTmemCols, "TMEM columns");
    // two CTAs per SM: their shared memory (each with 1 KB reserved) and TMEM
    static_assert(kSmem + 1024 <= 233472 / kMinBlocks && kTmemCols * kMinBlocks <= 512, "two CTAs per SM");
    static_assert(8 * (2 * STAGES + 2 * kNA + 7) + 16 <= 512, "barrier region");
    static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
    static_assert(NMAX % 16 == 0 && NMAX <= 256 && NMAX % (NMAX >= 64 ? 64 : 16) == 0, "MMA N extent");
};

// h of (pair or shared row) p, intermediate index il: routed rows [p][ld] bf16;
// shared rows [p][2 ld] = hi | lo.
__device__ __forceinline__ void store_h(__nv_bfloat16* out, bool shared, int ld, int p, int il, float hv) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
    if (shared) {
        __nv_bfloat16* o = out + (size_t)p * (2 * ld);
        o[il] = hi;
        o[ld + il] = __float2bfloat16_rn(hv - __bfloat162float(hi));
    } else {
        out[(size_t)p * ld + il] = hi;
    }
}

// Dequantise weight row r of one stage (thread r of the 128 converter
// threads): its 64 K codes (row r at raw + r * 64 bytes for 8 bits, r * 32 for
// 4, 16-byte chunks in the copy's swizzle: chunk c of row r at c ^ ((r >> 1) & 3)
// for 8 bits, c ^ ((r >> 2) & 1) for 4, so the 8 rows a quarter-warp reads
// together fall in distinct banks) and its two scales (bf16, block-major:
// block j of row r at sc[128 j + r]) become 64 bf16 weights, stored as 32
// columns of tensor memory from taddr on (column j: K elements 2j and 2j + 1,
// the even one in the low half), the A operand layout of the MMA.  The
// arithmetic is bf16x2: a pair of codes becomes two exact bf16 integers (|q| <=
// 128 has at most 8 significant bits) by byte permutes and one subtraction,
// and one bf16x2 product rounds each exact q * d once, to nearest even.
template <int QB>
__device__ __forceinline__ void dequant_row(const uint8_t* raw, const __nv_bfloat16* sc, int r,
                                            uint32_t taddr) {
    if (QB == 8) {
        const uint8_t* row = raw + r * 64;
        const int sw = (r >> 1) & 3;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {   // K elements 32 blk .. 32 blk + 31: chunks 2 blk, 2 blk + 1
            const __nv_bfloat162 d2 = __bfloat162bfloat162(sc[blk * 128 + r]);
            uint32_t o[16];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * blk + cc;
                const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
                const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
                // a code byte b (two's complement) as bf16: 128 + (b & 0x7F) (its low
                // seven bits in the mantissa of 128, exact) minus 128, or minus 256
                // when b's top bit is set (0x4300 or 0x4380): q exactly
#pragma unroll
                for (int w4 = 0; w4 < 4; ++w4) {   // codes 4 w4 .. 4 w4 + 3 of the chunk (bytes, in order)
                    const uint32_t lo7 = wd[w4] & 0x7F7F7F7Fu, top = wd[w4] & 0x80808080u;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {   // codes 4 w4 + 2 h2, 4 w4 + 2 h2 + 1
                        const uint32_t sel = h2 ? 0x5342u : 0x5140u;
                        const uint32_t m2 = __byte_perm(lo7, 0x43434343u, sel);
                        const uint32_t c2 = __byte_perm(top, 0x43434343u, sel);
                        const __nv_bfloat162 q2 = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&m2),
                                                          *reinterpret_cast<const __nv_bfloat162*>(&c2));
                        const __nv_bfloat162 v = __hmul2(q2, d2);
                        o[8 * cc + 2 * w4 + h2] = *reinterpret_cast<const uint32_t*>(&v);
                    }
                }
            }
            tmem_st16(taddr + 16 * blk, o);
        }
    } else {
        const uint8_t* row = raw + r * 32;
        const int sw = (r >> 2) & 1;
        // q + 8 (0..15) as the low mantissa bits of bf16 128 (0x4300): the
        // value 128 + q + 8, exact; minus 136 gives q exactly
        const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
        for (int c = 0; c < 2; ++c) {   // 32 codes (two per byte, even element low) = block c
            const __nv_bfloat162 d2 = __bfloat162bfloat162(sc[c * 128 + r]);
            const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
            const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
            uint32_t o[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {   // elements 8j .. 8j + 7 of the block
                const uint32_t xb = wd[j] ^ 0x88888888u;     // q + 8 per nibble
                const uint32_t lo = xb & 0x0F0F0F0Fu;          // byte i: element 2i
                const uint32_t hi = (xb >> 4) & 0x0F0F0F0Fu;   // byte i: element 2i + 1
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t t = __byte_perm(lo, hi, (uint32_t)(i | ((4 + i) << 4)));
                    const uint32_t m2 = __byte_perm(t, 0x43434343u, 0x5140u);   // {0x43 m0, 0x43 m1}
                    const __nv_bfloat162 q2 = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&m2), k136);
                    const __nv_bfloat162 v = __hmul2(q2, d2);
                    o[4 * j + i] = *reinterpret_cast<const uint32_t*>(&v);
                }
            }
            tmem_st16(taddr + 16 * c, o);
        }
    }
}

template <int MODE, int NMAX, int STAGES, int QB>
__global__ void __launch_bounds__(GemmCfg<MODE, NMAX, STAGES, QB>::kThreads,
                                  GemmCfg<MODE, NMAX, STAGES, QB>::kMinBlocks)
k_gemm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
       const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmA3,
       const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
       const __grid_constant__ CUtensorMap tmBg, const __grid_constant__ CUtensorMap tmS0,
       const __grid_constant__ CUtensorMap tmS1, const __grid_constant__ CUtensorMap tmS2,
       const __grid_constant__ CUtensorMap tmS3, GemmArgs a) {
    using C = GemmCfg<MODE, NMAX, STAGES, QB>;
    // gate/up units gather their rows of x (pair_row; shared_rows on a
    // live-row pass) with TMA gather4 (about 7 bytes per clock per SM: enough
    // for 32-row tiles, far too few for larger ones)
    constexpr bool kGather = MODE == kGateUp && NMAX == kSmallN;
    // A call of at most NMAX rows: every gate/up unit's B is all of x (one
    // 32-row box per stage, no gathers), the MMA runs every row, and the
    // epilogue reads the accumulator column of each pair's row of x.
    const bool allrows = kGather && a.R <= NMAX;
    extern __shared__ uint8_t smem_raw[];

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kBarOff);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* xbar = tempty + 2;  // [2] epilogue exchange (128 arrivals each)
    uint64_t* dbar = xbar + 2;    // MMA drain: every MMA issued has completed
    uint64_t* conv = dbar + 1;    // [kNA] A slot dequantised (quantised weights)
    uint64_t* aempty = conv + C::kNA;   // [kNA] A slot free
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aempty + C::kNA);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* never = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull + i, 1);
            mbar_init(tempty + i, 128);
            mbar_init(xbar + i, 128);
        }
        mbar_init(dbar, 1);
        for (int i = 0; i < C::kNA; ++i) {
            mbar_init(conv + i, 128);   // the converter threads
            mbar_init(aempty + i, 1);
        }
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA0); prefetch_tmap(&tmA1); prefetch_tmap(&tmA2);
        prefetch_tmap(&tmA3); prefetch_tmap(&tmB1);
        if (C::kQuant) {
            prefetch_tmap(&tmS0); prefetch_tmap(&tmS1); prefetch_tmap(&tmS2); prefetch_tmap(&tmS3);
        }
        if (kGather) prefetch_tmap(&tmBg);
        if (MODE == kDown) prefetch_tmap(&tmB0);  // h
    }
    // Programmatic dependent launch (common.cuh).  Every role waits here for
    // the preceding kernel, except the down GEMM's producer: the down GEMM
    // follows the gate/up GEMM, and its first stages' W_down tiles do not
    // depend on it, so the producer issues those before it waits (its unit
    // list was written by the scatter, which the gate/up GEMM waited for
    // before letting this kernel start).
    constexpr bool kEarlyA = MODE == kDown;
    if (!(kEarlyA && warp == 0)) {
        pdl_wait();
        pdl_trigger();
    }
    const int nunits = __ldg(a.n_units);
    // balanced rounds (common.cuh)
    const int nact = active_workers(nunits, gridDim.x);
    const int ufirst = (int)blockIdx.x < nact ? (int)blockIdx.x : nunits;

    auto give_up = [&]() {
        if (!*abort_flag) { *abort_flag = 1; status_add(a.status, MOE_STATUS_WAIT_TIMEOUT, 1); }
    };
    const uint64_t kWaitNs = a.wait_ns ? a.wait_ns : kWaitLimitNs;   // pipeline waits

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        // (the whole warp runs the loop; lane 0 issues the copies)
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int nfills = 0;   // stages filled (TMA issued) so far
        int* s_rows = reinterpret_cast<int*>(base + C::kRowsOff);
        // B copies of the first stages, held back until the wait (down GEMM)
        struct HeldB { uint32_t sB; int g, start, nbox, K, kc; uint64_t* bar; };
        HeldB held[kEarlyA ? STAGES : 1];
        int nheld = 0;
        bool waited = !kEarlyA;
        auto issue_b = [&](uint32_t sB, int g, int start, int nbox, int K, int kc, uint64_t* bar) {
            constexpr int kBoxBytes = C::kBoxRows * 128;
            const CUtensorMap* mB = g == a.E ? &tmB1 : &tmB0;
            for (int t = 0; t < nbox; ++t)
                tma_load_2d(sB + t * kBoxBytes, mB, kc, start + t * C::kBoxRows, bar);
            if (C::kDualLo && g == a.E)  // lo part of h: columns K .. 2K-1 of the same rows
                for (int t = 0; t < nbox; ++t)
                    tma_load_2d(sB + NMAX * 128 + t * kBoxBytes, mB, K + kc, start + t * C::kBoxRows, bar);
        };
        auto release_held = [&]() {
            pdl_wait();
            pdl_trigger();
            if (lane == 0)
                for (int i = 0; i < nheld; ++i)
                    issue_b(held[i].sB, held[i].g, held[i].start, held[i].nbox, held[i].K, held[i].kc,
                            held[i].bar);
            nheld = 0;
            waited = true;
        };
        for (int u = ufirst; ok && u < nunits; u += nact) {
            const int4 un = __ldg(a.units + u);
            if (!unit_valid(un, a, NMAX, MODE == kDown, C::kGURows)) continue;
            const int g = un.x, m = un.y, start = un.z, n = un.w;
            // B rows actually loaded: gathered units load ceil(n/4) rows x 4; the
            // others whole boxes of kBoxRows.  Rows of the tile past n only feed
            // output columns that are never read, so they need not be loaded.
            // gathered: routed rows (pair_row), and the shared expert's rows when
            // only some rows are live (shared_rows)
            const bool gathered = kGather && !allrows && (g != a.E || a.shared_rows != nullptr);
            const int nb4 = (n + 3) >> 2;
            const int nbox = (n + C::kBoxRows - 1) / C::kBoxRows;
            // K steps: gate/up H; down I (routed) or, for the shared expert, Is
            // (streaming shape: hi and lo in one stage) or 2 Is (h = [hi | lo],
            // A wrapping around its Is columns)
            const int Ka = MODE == kGateUp ? a.H : (g == a.E ? a.Is : a.I);
            const int K = MODE == kDown && g == a.E && !C::kDualLo ? 2 * a.Is : Ka;
            const uint32_t bbytes = gathered  ? (uint32_t)nb4 * 512u
                                    : allrows ? (uint32_t)(C::kBoxRows * 128)
                                              : (uint32_t)(nbox * C::kBoxRows * 128);
            const int parts = C::kDualLo && g == a.E ? 2 : 1;
            const uint32_t abytes = C::kQuant ? (uint32_t)(C::kRawBytes + C::kScaleBytes)
                                              : (uint32_t)C::kABytes;
            const uint32_t bytes = abytes + parts * bbytes;
            if (gathered) {
                // the unit's rows of x, padded to a multiple of 4 with R (read as zeros);
                // copies of the previous unit took their coordinates when issued
                __syncwarp();
                const int32_t* rl = g == a.E ? a.shared_rows : a.pair_row;
                for (int i = lane; i < nb4 * 4; i += 32)
                    s_rows[i] = i < n ? __ldg(rl + start + i) : a.R;
                __syncwarp();
            }
            for (int kb = 0; kb < (K >> 6); ++kb) {
                const bool w_ok = mbar_wait_bounded(empty + stage, phase ^ 1u, abort_flag, kWaitNs);
                if (__any_sync(0xffffffffu, !w_ok)) {
                    if (lane == 0) give_up();
                    ok = false;
                    break;
                }
                const uint32_t sA = sbase + stage * C::kStageBytes;
                // quantised: [B | raw codes | scales]; bf16: [A | B]
                const uint32_t sB = C::kQuant ? sA : sA + C::kABytes;
                const int kc = kb * 64;
                if (lane == 0) {
                    mbar_expect_tx(full + stage, bytes);
                    if (C::kQuant) {
                        // raw codes: K bytes kc (8 bits) or kc / 2 (4 bits); scales:
                        // blocks kc / 32 and kc / 32 + 1 of the rows (block-major)
                        const uint32_t sR = sA + C::kBBytes, sS = sR + C::kRawBytes;
                        const int kq = QB == 8 ? kc : kc / 2;
                        if (MODE == kGateUp) {
                            // the interleaved gate/up tensor: rows 128 m .. 128 m + 127
                            // are gate rows 64 m .. 64 m + 63, then the same up rows
                            const int rows = m * 128;
                            if (g == a.E) {
                                tma_load_2d(sR, &tmA2, kq, rows, full + stage);
                                tma_load_2d(sS, &tmS2, rows, kc / 32, full + stage);
                            } else {
                                tma_load_3d(sR, &tmA0, kq, rows, g, full + stage);
                                tma_load_3d(sS, &tmS0, rows, kc / 32, g, full + stage);
                            }
                        } else {
                            const int Kc = g == a.E ? a.Is : a.I;
                            const int kca = kc % Kc, kqa = QB == 8 ? kca : kca / 2;
                            if (g == a.E) {
                                tma_load_2d(sR, &tmA2, kqa, m * 128, full + stage);
                                tma_load_2d(sS, &tmS2, m * 128, kca / 32, full + stage);
                            } else {
                                tma_load_3d(sR, &tmA0, kqa, m * 128, g, full + stage);
                                tma_load_3d(sS, &tmS0, m * 128, kca / 32, g, full + stage);
                            }
                        }
                    } else if (MODE == kGateUp) {
                        // 64-row boxes: gate rows, then up rows (rows past I read as zeros)
                        constexpr int kHalf = C::kGURows / 64;  // boxes per weight
                        const int rows = m * C::kGURows;
#pragma unroll
                        for (int hb = 0; hb < kHalf; ++hb) {
                            const uint32_t dg = sA + hb * 64 * 128, du = dg + kHalf * 64 * 128;
                            if (g == a.E) {
                                tma_load_2d(dg, &tmA2, kc, rows + 64 * hb, full + stage);
                                tma_load_2d(du, &tmA3, kc, rows + 64 * hb, full + stage);
                            } else {
                                tma_load_3d(dg, &tmA0, kc, rows + 64 * hb, g, full + stage);
                                tma_load_3d(du, &tmA1, kc, rows + 64 * hb, g, full + stage);
                            }
                        }
                    } else {
                        const int kca = kc % Ka;
                        if (g == a.E) tma_load_2d(sA, &tmA2, kca, m * 128, full + stage);
                        else tma_load_3d(sA, &tmA0, kca, m * 128, g, full + stage);
                    }
                    if (allrows) tma_load_2d(sB, &tmB1, kc, 0, full + stage);   // all of x
                    else if (!gathered) {
                        if (waited) issue_b(sB, g, start, nbox, K, kc, full + stage);
                        else held[nheld] = HeldB{sB, g, start, nbox, K, kc, full + stage};
                    }
                }
                if (!waited && ++nheld == STAGES) release_held();
                if (gathered) {
                    // the gathers are spread over the lanes (issued after the
                    // expected byte count is posted by lane 0)
                    __syncwarp();
                    for (int t = lane; t < nb4; t += 32) {
                        const int4 rr = *reinterpret_cast<const int4*>(s_rows + 4 * t);
                        tma_gather4(sB + t * 512, &tmBg, kc, rr.x, rr.y, rr.z, rr.w, full + stage);
                    }
                }
                ++nfills;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!waited) release_held();
        // Drain: the last fill of every stage completes its `full` phase when
        // its copies land, consumed or not; wait for each (bounded), so no
        // copy into this CTA's shared memory is in flight when it exits.
        // Stage s < stage was last filled in this wrap (parity `phase`), the
        // others in the wrap before (if filled at all).
        if (lane == 0) {
            for (int s = 0; s < STAGES; ++s) {
                if (nfills < STAGES && s >= nfills) break;
                const uint32_t par = s < stage ? phase : (phase ^ 1u);
                if (!mbar_wait_bounded(full + s, par, never, kDrainLimitNs)) give_up();
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
            int stage = 0, acc = 0, aslot = 0;
            uint32_t phase = 0, acc_phase = 0, aphase = 0;
            bool ok = true;
            for (int u = ufirst; ok && u < nunits; u += nact) {
                const int4 un = __ldg(a.units + u);
                if (!unit_valid(un, a, NMAX, MODE == kDown, C::kGURows)) {
                    status_add(a.status, MOE_STATUS_BAD_UNIT, 1);
                    continue;
                }
                const int g = un.x, n = un.w;
                const int n16 = allrows ? ((a.R + 15) & ~15) : (n + 15) & ~15;   // MMA N
                const int K = MODE == kGateUp ? a.H
                                              : (g == a.E ? (C::kDualLo ? a.Is : 2 * a.Is) : a.I);
                const uint32_t idesc = idesc_bf16_f32(128, n16);
                if (!mbar_wait_bounded(tempty + acc, acc_phase ^ 1u, abort_flag, kWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * C::kAccCols);
                for (int kb = 0; kb < (K >> 6); ++kb) {
                    // quantised: the converter's A slot (it waited for the stage's
                    // copies, the B tile included); bf16: the stage itself
                    if (!mbar_wait_bounded(C::kQuant ? conv + aslot : full + stage,
                                           C::kQuant ? aphase : phase, abort_flag, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sSt = sbase + stage * C::kStageBytes;
                    const uint32_t sB = C::kQuant ? sSt : sSt + C::kABytes;
                    // quantised: A in tensor memory, 8 columns per 16 K
                    const uint32_t ta = tmem + (uint32_t)(C::kACol + aslot * 32);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = smem_desc_sw128(sB + kk * 32);
                        const uint64_t bdl = smem_desc_sw128(sB + NMAX * 128 + kk * 32);
                        if (C::kQuant) {
                            tc_mma_bf16_ta(d, ta + kk * 8, bd, idesc, (kb | kk) != 0);
                            if (C::kDualLo && g == a.E)  // shared expert: lo part of h
                                tc_mma_bf16_ta(d, ta + kk * 8, bdl, idesc, 1u);
                        } else {
                            const uint64_t ad = smem_desc_sw128(sSt + kk * 32);
                            tc_mma_bf16(d, ad, bd, idesc, (kb | kk) != 0);
                            if (C::kDualLo && g == a.E)  // shared expert: lo part of h
                                tc_mma_bf16(d, ad, bdl, idesc, 1u);
                        }
                    }
                    tc_commit(empty + stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (C::kQuant) {
                        tc_commit(aempty + aslot);
                        if (++aslot == C::kNA) { aslot = 0; aphase ^= 1u; }
                    }
                }
                if (!ok) break;
                tc_commit(tfull + acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // drain: arrives once every MMA issued above has completed
            tc_commit(dbar);
            if (!mbar_wait_bounded(dbar, 0, never, kDrainLimitNs)) give_up();
        }
    } else if (C::kQuant && warp >= 6) {
        // ---------------------------------------------------------- converter
        // Stage by stage, in the MMA's order: wait for the stage's copies and a
        // free A slot; thread r turns weight row r's 64 K codes into bf16
        // weights bf16(q * d) in lane r of the slot's tensor-memory columns
        // and, once its stores are complete, hands the slot to the MMA.  A
        // warp may only reach the 32 lanes of its quadrant (warp & 3), so that
        // sets its rows; its waits are voted, since the tensor-memory stores
        // are warp-wide instructions.
        const int r = 32 * (warp & 3) + lane;
        const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)C::kACol;
        int stage = 0, aslot = 0;
        uint32_t phase = 0, aphase = 0;
        bool ok = true;
        for (int u = ufirst; ok && u < nunits; u += nact) {
            const int4 un = __ldg(a.units + u);
            if (!unit_valid(un, a, NMAX, MODE == kDown, C::kGURows)) continue;
            const int g = un.x;
            const int K = MODE == kGateUp ? a.H : (g == a.E ? a.Is : a.I);
            for (int kb = 0; kb < (K >> 6); ++kb) {
                const bool w_ok = mbar_wait_bounded(full + stage, phase, abort_flag, kWaitNs) &&
                                  mbar_wait_bounded(aempty + aslot, aphase ^ 1u, abort_flag, kWaitNs);
                if (__any_sync(0xffffffffu, !w_ok)) {
                    if (!w_ok) give_up();
                    ok = false;
                    break;
                }
                tc_fence_after();   // the MMA that last read the slot has completed
                const uint8_t* raw = base + stage * C::kStageBytes + C::kBBytes;
                const __nv_bfloat16* sc = reinterpret_cast<const __nv_bfloat16*>(raw + C::kRawBytes);
                dequant_row<QB>(raw, sc, r, tq + (uint32_t)(aslot * 32));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(conv + aslot);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                if (++aslot == C::kNA) { aslot = 0; aphase ^= 1u; }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        int acc = 0;
        uint32_t acc_phase = 0, xphase = 0;
        bool alive = true;
        for (int u = ufirst; alive && u < nunits; u += nact) {
            const int4 un = __ldg(a.units + u);
            if (!unit_valid(un, a, NMAX, MODE == kDown, C::kGURows)) continue;
            const int g = un.x, m = un.y, start = un.z, n = un.w;
            const int n16 = (n + 15) & ~15;
            // down: the unit's pair weights, lane l of wreg[j] holding pair
            // 32 j + l (0 past the unit's pairs), loaded while the MMA runs
            float wreg[MODE == kDown ? NMAX / 32 : 1];
            if (MODE == kDown) {
#pragma unroll
                for (int j = 0; j < NMAX / 32; ++j) {
                    const int t = 32 * j + lane;
                    wreg[j] = t < n ? (g == a.E ? 1.0f : __ldg(a.pair_w + start + t)) : 0.0f;
                }
            }
            const bool ok = mbar_wait_bounded(tfull + acc, acc_phase, abort_flag, kWaitNs);
            if (__any_sync(0xffffffffu, !ok)) { give_up(); break; }
            __syncwarp();
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
            bool released = false;  // accumulator handed back to the MMA warp
            if (MODE == kGateUp) {
                // all rows of x in the accumulator: lane l holds the column (row
                // of x) of pair start + l
                int pcol = 0;
                if (allrows && lane < n) {
                    const int32_t* rl = g == a.E ? a.shared_rows : a.pair_row;
                    pcol = rl ? __ldg(rl + start + lane) : start + lane;
                }
                for (int c = 0; alive && c < n16; c += 16) {
                    float v[16];
                    __syncwarp();  // tcgen05.ld is warp-collective
                    if (allrows) {
                        int cols[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) cols[j] = __shfl_sync(0xffffffffu, pcol, (c + j) & 31);
                        tmem_ld_cols16(tb, cols, v);
                    } else {
                        tmem_ld16(tb + (uint32_t)c, v);
                    }
                    // quadrants 0-1: gate rows, 2-3: up rows of intermediate index r
                    const bool is_gate = q < 2;
                    const int r = (q & 1) * 32 + lane;
                    float* xg = reinterpret_cast<float*>(base + C::kXchgOff);  // [64][9]: g, cols 8..15
                    float* xu = xg + 64 * 9;                                    // [64][9]: u, cols 0..7
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        if (is_gate) xg[r * 9 + t] = v[8 + t];
                        else xu[r * 9 + t] = v[t];
                    }
                    // the four epilogue warps meet through an mbarrier (bounded wait)
                    mbar_arrive(xbar);
                    if (__any_sync(0xffffffffu,
                                   !mbar_wait_bounded(xbar, xphase, abort_flag, kWaitNs))) {
                        give_up();
                        alive = false;
                        break;
                    }
                    __nv_bfloat16* out = g == a.E ? a.hs : a.h;
                    const int ld = g == a.E ? a.Is : a.I;
                    const int il = m * 64 + r;
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int col = c + (is_gate ? t : 8 + t);
                        const float gv = is_gate ? v[t] : xg[r * 9 + t];
                        const float uv = is_gate ? xu[r * 9 + t] : v[8 + t];
                        if (col < n) {
                            store_h(out, g == a.E, ld, start + col, il, silu_fast(gv) * uv);
                        }
                    }
                    mbar_arrive(xbar + 1);  // the buffer is reused by the next chunk
                    if (__any_sync(0xffffffffu,
                                   !mbar_wait_bounded(xbar + 1, xphase, abort_flag, kWaitNs))) {
                        give_up();
                        alive = false;
                        break;
                    }
                    xphase ^= 1u;
                }
            } else {
                // Weighted fp16 outputs of the unit's pairs, staged in shared
                // memory ([pair][128 hidden]) kStageRows pairs at a time, so each
                // pair's 128 columns leave as one 256-byte segment; the
                // accumulator is released before the last part's copy-out.
                // fp16 holds |v| < 65504: each warp owns a 32-column
                // quarter (its TMEM lane quadrant) of every pair, and a quarter
                // whose largest finite magnitude is 2^15 or more is stored as
                // v * 2^-s with the smallest s that brings that magnitude below
                // 2^15; s goes to ysx and the call's `scaled` flag is set;
                // k_combine multiplies it back exactly.  Other quarters are
                // stored as they are (s = 0); infinities and NaNs pass through
                // the scaling unchanged.  The common case costs one max per
                // value: the exact per-pair exponents are only worked out for
                // a group of 32 pairs in which some lane saw 2^15 or more.
                __half* xs = reinterpret_cast<__half*>(base + C::kXchgOff);
                const int hl = q * 32 + lane;
                const size_t row0 = (size_t)(g == a.E ? a.shared_row0 : 0) + start;
                uint8_t* xq = a.ysx + (size_t)(m * 4 + q) * a.ld_x + row0;  // this quarter's exponents
                const int et = (warp - 2) * 32 + lane;  // 0..127 over the epilogue warps
                bool any_big = false;
                constexpr int kParts = NMAX / C::kStageRows, kGroups = C::kStageRows / 32;
#pragma unroll
                for (int hp = 0; hp < kParts; ++hp) {
                    const int p0 = hp * C::kStageRows;   // first pair of this part
                    if (p0 >= n16) break;
#pragma unroll
                    for (int jj = 0; jj < kGroups; ++jj) {
                        const int j = hp * kGroups + jj;
                        const int c = 32 * j;
                        if (c >= n16) break;
                        float v[32];
                        __syncwarp();  // tcgen05.ld is warp-collective
                        // columns c .. c + 31 (those past n16 are inside the
                        // accumulator and never copied out)
                        tmem_ld16x2(tb + (uint32_t)c, tb + (uint32_t)(c + 16), v, v + 16);
                        float mx = 0.0f;   // fmaxf skips NaN: the tail's 0 * garbage
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            v[t] *= __shfl_sync(0xffffffffu, wreg[j], t);
                            mx = fmaxf(mx, fabsf(v[t]));
                        }
                        uint32_t my_s = 0;  // lane t: the exponent of pair c + t
                        if (__any_sync(0xffffffffu, mx >= 32768.0f)) {
                            any_big = true;
#pragma unroll
                            for (int t = 0; t < 32; ++t) {
                                const uint32_t ab = __float_as_uint(v[t]) & 0x7FFFFFFFu;
                                const uint32_t mb = __reduce_max_sync(0xffffffffu, ab < 0x7F800000u ? ab : 0u);
                                const int sh = (int)(mb >> 23) - 141;   // biased exponent - (127 + 14)
                                const uint32_t st = sh > 0 ? (uint32_t)sh : 0u;
                                v[t] *= __uint_as_float((127u - st) << 23);   // 2^-s, exact
                                if (lane == t) my_s = st;
                            }
                        }
#pragma unroll
                        for (int t = 0; t < 32; ++t) xs[(c - p0 + t) * 128 + hl] = __float2half_rn(v[t]);
                        if (c + lane < n) xq[c + lane] = (uint8_t)my_s;
                    }
                    if (hp == kParts - 1 || p0 + C::kStageRows >= n16) {
                        // the last TMEM read of the unit: hand the accumulator back
                        if (any_big && lane == 0) *a.scaled = 1;
                        tc_fence_before();
                        mbar_arrive(tempty + acc);
                        released = true;
                    }
                    mbar_arrive(xbar);
                    if (__any_sync(0xffffffffu, !mbar_wait_bounded(xbar, xphase, abort_flag, kWaitNs))) {
                        give_up();
                        alive = false;
                        break;
                    }
                    const int np = min(C::kStageRows, n - p0);   // pairs of this part
                    for (int idx = et; idx < np * 16; idx += 128) {  // np rows x 16 segments of 16 B
                        const int t = idx >> 4, seg = idx & 15;
                        const uint4 val = *reinterpret_cast<const uint4*>(xs + t * 128 + seg * 8);
                        *reinterpret_cast<uint4*>(a.ys + (row0 + p0 + t) * a.H + m * 128 + seg * 8) = val;
                    }
                    mbar_arrive(xbar + 1);  // the rows are rewritten by the next part
                    if (__any_sync(0xffffffffu,
                                   !mbar_wait_bounded(xbar + 1, xphase, abort_flag, kWaitNs))) {
                        give_up();
                        alive = false;
                        break;
                    }
                    xphase ^= 1u;
                }
            }
            if (!alive) break;
            if (!released) {
                tc_fence_before();
                mbar_arrive(tempty + acc);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------------------

template <int MODE, int NMAX, int STAGES, int QB = 0>
static cudaError_t launch_one(const GemmMaps& mp, const GemmArgs& a, int grid, cudaStream_t st) {
    using C = GemmCfg<MODE, NMAX, STAGES, QB>;
    return launch_kernel(k_gemm<MODE, NMAX, STAGES, QB>, dim3(grid), dim3(C::kThreads), C::kSmem, st,
                         mp.a0, mp.a1, mp.a2, mp.a3, mp.b0, mp.b1, mp.bg, mp.s0, mp.s1, mp.s2, mp.s3,
                         a);
}

template <int MODE, int NMAX, int STAGES, int QB = 0>
static cudaError_t set_attr() {
    using C = GemmCfg<MODE, NMAX, STAGES, QB>;
    return cudaFuncSetAttribute(k_gemm<MODE, NMAX, STAGES, QB>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
}

// (rows per unit, pipeline depth) of each kernel shape: small = few rows per
// expert (weight streaming: two CTAs per SM, each with its own ring, keep more
// TMA streams in flight); many rows per expert run on CTA pairs
// (k_gateup_pair, k_down_pair).  Quantised weights stream with the small shape
// at every row count.
constexpr int kSmallStagesGU = 5, kSmallStagesDN = 4;
constexpr int kSmallCtasPerSm = 2;
// quantised stages hold no A tile (it is built in tensor memory), so more fit
constexpr int kQuantStagesGU = 7, kQuantStagesDN = 5;

cudaError_t gemm_set_attributes() {
    cudaError_t e;
    if ((e = set_attr<kGateUp, kSmallN, kSmallStagesGU>()) != cudaSuccess) return e;
    if ((e = set_attr<kDown, kSmallN, kSmallStagesDN>()) != cudaSuccess) return e;
    if ((e = set_attr<kGateUp, kSmallN, kQuantStagesGU, 8>()) != cudaSuccess) return e;
    if ((e = set_attr<kDown, kSmallN, kQuantStagesDN, 8>()) != cudaSuccess) return e;
    if ((e = set_attr<kGateUp, kSmallN, kQuantStagesGU, 4>()) != cudaSuccess) return e;
    return set_attr<kDown, kSmallN, kQuantStagesDN, 4>();
}

cudaError_t launch_gemm(int mode, bool small, int qbits, const GemmMaps& mp, const GemmArgs& a,
                        int grid, cudaStream_t st) {
    if (qbits) {
        grid *= kSmallCtasPerSm;
        if (qbits == 8)
            return mode == kGateUp ? launch_one<kGateUp, kSmallN, kQuantStagesGU, 8>(mp, a, grid, st)
                                   : launch_one<kDown, kSmallN, kQuantStagesDN, 8>(mp, a, grid, st);
        return mode == kGateUp ? launch_one<kGateUp, kSmallN, kQuantStagesGU, 4>(mp, a, grid, st)
                               : launch_one<kDown, kSmallN, kQuantStagesDN, 4>(mp, a, grid, st);
    }
    if (small) {
        grid *= kSmallCtasPerSm;
        return mode == kGateUp ? launch_one<kGateUp, kSmallN, kSmallStagesGU>(mp, a, grid, st)
                               : launch_one<kDown, kSmallN, kSmallStagesDN>(mp, a, grid, st);
    }
    return mode == kGateUp ? launch_gateup_pair(mp, a, st) : launch_down_pair(mp, a, st);
}

}  // namespace moe
