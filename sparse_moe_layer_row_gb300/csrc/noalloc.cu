// moe_block_route_noalloc: the router for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand this library a workspace. Examples: an
// engine that reserves all of its device memory up front and forbids any
// later cudaMalloc; a plugin that may only touch the buffers it is given; code
// that must not grow its memory footprint while serving. For them this entry
// point runs the fixed-order (SIMT) router, whose outputs are bit-identical to
// moe_block_route's, with its scratch (the router logits and the row-group
// tickets) in a fixed array compiled into the library instead of in a caller
// workspace.  It never takes the tensor-core screen that moe_block_route uses
// from 256 rows on, so there it is slower for the same ids and weights.
//
// Properties a user must know:
//   * The array holds kNoAllocScratchBytes (1 MiB) on every GPU that loads the
//     library, for as long as the library stays loaded.
//   * Calls needing more scratch than that are rejected with
//     MOE_ERR_UNSUPPORTED and nothing is launched.  A call needs 4 * R * E
//     bytes of logits, 4 * R bytes of tickets rounded up to 256, and 256
//     bytes of status; at E = 256 that allows up to 1019 rows.
//   * All calls share the one array, which keeps what the last call left in
//     it. The tickets that must start at zero are cleared on the stream at the
//     start of every call. Calls that overlap on the GPU (different streams,
//     or different host threads) race on the array and must not be issued.
//   * The first call on a device, with that device current, resolves the
//     array's device address (cudaGetSymbolAddress). Make that first call
//     before any stream capture.  Calls outside a capture resolve the address
//     again (it can move when the device's context is reset and the module
//     reloaded); a call during a capture uses the address of the last call.
//   * Non-finite logits are counted into a status word inside the array, which
//     is not reported to the caller.
#include <mutex>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;
constexpr size_t kStatusBytes = 256;      // status words of these calls (not reported)

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];        // device address of g_route_scratch, per device

// The array's address on the current device.  Outside a stream capture it is
// looked up every time (cheap; the address can change after a context reset);
// during a capture, where the lookup is not allowed, the last one is used.
moe_status scratch_address(int device, cudaStream_t st, unsigned char** out) {
    if (device < 0 || device >= kMaxDevices)
        return set_error(MOE_ERR_UNSUPPORTED, "device ordinal too large for the static scratch");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess)
        return set_error(MOE_ERR_CUDA, "cudaStreamIsCapturing failed");
    std::lock_guard<std::mutex> lock(g_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess || !p)
            return set_error(MOE_ERR_CUDA, "cudaGetSymbolAddress of the router scratch failed");
        g_scratch_addr[device] = p;
    } else if (!g_scratch_addr[device]) {
        return set_error(MOE_ERR_INVALID_ARG,
                         "first call on this device is inside a stream capture; call once before");
    }
    *out = static_cast<unsigned char*>(g_scratch_addr[device]);
    return MOE_OK;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_block_route_noalloc(const moe_plan* plan, const void* x, int32_t R,
                                              const int32_t* block_offsets, int32_t nb,
                                              const float* logit_bias, int32_t* topk_idx,
                                              float* topk_w, moe_stream_t stream) {
    PlanView pv;
    if (!plan_view(plan, &pv)) return set_error(MOE_ERR_INVALID_ARG, "plan is NULL");
    if (R < 0 || R > pv.d.max_rows) return set_error(MOE_ERR_INVALID_ARG, "R outside [0, max_rows]");
    if (nb < 1 || nb > pv.d.max_blocks)
        return set_error(MOE_ERR_INVALID_ARG, "nb outside [1, max_blocks]");
    if (!block_offsets || !aligned_to(block_offsets, 4))
        return set_error(MOE_ERR_INVALID_ARG, "block_offsets NULL or misaligned");
    if (!x || !aligned_to(x, 16)) return set_error(MOE_ERR_INVALID_ARG, "x NULL or not 16-byte aligned");
    if (!topk_idx || !topk_w || !aligned_to(topk_idx, 4) || !aligned_to(topk_w, 4))
        return set_error(MOE_ERR_INVALID_ARG, "topk_idx/topk_w NULL or misaligned");
    if (logit_bias && !aligned_to(logit_bias, 4))
        return set_error(MOE_ERR_INVALID_ARG, "logit_bias misaligned");
    const size_t cnt_bytes = align_up(sizeof(uint32_t) * (size_t)R, 256);
    const size_t logit_bytes = sizeof(float) * (size_t)R * (size_t)pv.d.E;
    if (kStatusBytes + cnt_bytes + logit_bytes > kNoAllocScratchBytes)
        return set_error(MOE_ERR_UNSUPPORTED,
                         "R * E too large for the 1 MiB static router scratch (use moe_block_route)");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != pv.device)
        return set_error(MOE_ERR_INVALID_ARG, "current device is not the plan's device");
    if (R == 0) return set_error(MOE_OK, "");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned char* base = nullptr;
    moe_status s = scratch_address(dev, st, &base);
    if (s != MOE_OK) return s;
    uint32_t* status = reinterpret_cast<uint32_t*>(base);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(base + kStatusBytes);
    float* logits = reinterpret_cast<float*>(base + kStatusBytes + cnt_bytes);
    cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes + cnt_bytes, st);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "clearing the router scratch failed");
    RouteArgs a{static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(pv.w_router),
                logit_bias, block_offsets, R, pv.d.H, pv.d.E, pv.d.k, nb, logits, cnt, topk_idx,
                topk_w, status};
    e = launch_route(a, pv.num_sms, st);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, cudaGetErrorString(e));
    return set_error(MOE_OK, "");
}
