// Block coreset: restrict each block's experts to the smallest set carrying a
// fraction tau of the block's routing mass, then renormalise each row.
//
// Model card "Clover-35B-A3B-Preview -- CMF", Usage: "the block's experts
// restricted to the set that carries 90% of its routing"; InfiniLM PR #604,
// Summary (preview passes use block coreset routing) and Notes (full-route
// replay: the coreset disabled, here tau >= 1).
//
// The arithmetic is exact so that membership matches bit for bit:
//   * q = floor(w * 2^32) per (row, slot) (w in [0, 1], the scaling is exact);
//     w is the slot's routing weight, or, under the probability-mass reading
//     (InfiniLM PR #604, Summary: "block coreset routing"; the pages do not fix
//     the mass), its probability under the softmax over all experts, given
//     apart from the weights; the renormalisation always divides the weights;
//     Q_e = sum of q over the block (64-bit integers, any order);
//   * theta = ceil(tau * T), T = sum_e Q_e, with tau = M * 2^-s taken from its
//     fp32 encoding and the product formed in 128 bits;
//   * experts ranked by (Q desc, id asc); the coreset is the shortest prefix
//     of that order whose mass reaches theta: an expert is in it iff the mass
//     of the experts ranked above it is still below theta.  The ranks come
//     from one 64-bit key per expert.  Up to 256 experts: a thread per expert
//     counts, over the compacted keys of the block's touched experts, the
//     keys above its own and their mass.  More experts: with many blocks
//     (CTAs sharing SMs, so throughput counts) a bitonic sort of the keys in
//     shared memory; with few, a group of lanes counts the keys above each
//     expert's own.  All give the same ranks;
//   * an expert budget B > 0 (InfiniLM PR #604, Summary, names it without
//     defining it) keeps at most the first B experts of that order; rows are
//     copied unchanged only when tau >= 1 and nothing is dropped.
// One CTA per block.
#include "coreset_dev.cuh"

namespace moe {

__global__ void __launch_bounds__(kCoreThreads) k_coreset(CoresetArgs a) {
    pdl_wait();  // see common.cuh: nothing global is touched before
    pdl_trigger();
    __shared__ CoresetSmem sm;
    coreset_block(a, blockIdx.x, sm, gridDim.x >= kSortBlocks);
}

cudaError_t launch_coreset(const CoresetArgs& a, cudaStream_t st) {
    if (a.nb <= 0) return cudaSuccess;
    const int threads = a.E <= 256 ? kCoreThreadsSmallE : (a.nb >= kSortBlocks ? kCoreThreadsSort : kCoreThreads);
    return launch_kernel(k_coreset, dim3(a.nb), dim3(threads), 0, st, a);
}

}  // namespace moe
