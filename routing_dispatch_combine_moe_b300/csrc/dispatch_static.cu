// moe_dispatch_static: the dispatch of moe_dispatch for callers that cannot give
// the library any device memory of their own for scratch. Examples: a serving loop
// that forbids device allocations after start-up (cudaMalloc can synchronise the
// device and stall a latency-critical step), or a plugin whose host framework owns
// every device buffer and exposes only the tensors it passes in.
//
// The dispatch needs scratch beyond its inputs and outputs: a per-block histogram
// of E x blocks ints and E drop offsets. Here they live in one file-scope device
// array (g_dispatch_scratch below), which every GPU that loads this library holds
// until the process exits. This entry point allocates nothing: it calls no
// cudaMalloc, cudaFree or allocating library routine.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is looked up with
// cudaGetSymbolAddress on the first call made in each device context (once per
// device, with that device current, and again if cudaDeviceReset re-creates the
// context); that first call should therefore come before any stream capture.
#include <mutex>
#include <string>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kStaticScratchInts = MOE_STATIC_SCRATCH_BYTES / sizeof(int32_t);

// [0]: status word, [1]: the scan's ticket, [64, 64 + N*blocks): histogram, then N drop
// offsets, N+1 routed offsets and (gate drop policy) the T*K per-expert assignment list.
__device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchInts];

// Device address of g_dispatch_scratch in the current context, looked up once per
// context: once per device, and again after a cudaDeviceReset re-creates the device's
// context (the module, and with it the array, is then loaded anew).
PerContext<int32_t*> g_scratch_addr;

cudaError_t scratch_address(int32_t** out) {
    const cudaError_t e = g_scratch_addr.get(out, [](int32_t** p) {
        void* q = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&q, g_dispatch_scratch);
        *p = static_cast<int32_t*>(q);
        return err;
    });
    if (e == cudaSuccess && !*out) return cudaErrorInvalidSymbol;
    return e;
}

}  // namespace

extern thread_local std::string g_last_cuda_error;

}  // namespace moe

using namespace moe;

extern "C" int moe_dispatch_static(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                   const float* topk_gate, const moe_dispatch_map* map, void* xperm,
                                   moe_stream_t stream) {
    const int rc = moe_validate_config(cfg);
    if (rc != MOE_OK) return rc;
    if (!x || !topk_idx || !map || (!xperm && moe_rows_capacity(cfg) > 0)) return MOE_ERR_ARG;
    const bool by_gate = cfg->drop_policy == MOE_DROP_LOW_GATE && cfg->capacity >= 0;
    if (by_gate && !topk_gate) return MOE_ERR_ARG;
    if (!map->counts_routed || !map->counts_kept || !map->offsets || !map->rank_offsets || !map->pos ||
        !map->row_src || !map->drop_list || !map->n_dropped)
        return MOE_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(xperm) & 15u)) return MOE_ERR_ALIGN;
    const int N = cfg->E + cfg->n_shared, K = cfg->k + cfg->n_shared;
    const int64_t A = int64_t(cfg->T) * K;
    const size_t hist_ints = size_t(N) * size_t(dispatch_blocks(A));
    const size_t list_ints = by_gate ? 2 * size_t(A) : 0;  // assignment ids, then their gates' order keys
    if (64 + hist_ints + 2 * size_t(N) + 1 + list_ints > kStaticScratchInts) return MOE_ERR_WORKSPACE;

    int32_t* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, 2 * sizeof(int32_t), stream);
    if (e != cudaSuccess) {
        g_last_cuda_error = std::string("moe_dispatch_static: ") + cudaGetErrorName(e) + " (" +
                            cudaGetErrorString(e) + ")";
        return MOE_ERR_CUDA;
    }
    DispatchArgs a{};
    a.T = cfg->T; a.d = cfg->d; a.E = N; a.k = K; a.D = cfg->D;
    a.E_capped = cfg->E;
    a.drop_policy = cfg->drop_policy;
    a.layout = cfg->layout;
    a.topk_gate = topk_gate;
    a.capacity = cfg->capacity;
    a.act_bytes = cfg->act_dtype == MOE_F32 ? 4 : 2;
    a.x = x;
    a.topk_idx = topk_idx;
    a.counts_routed = map->counts_routed;
    a.counts_kept = map->counts_kept;
    a.offsets = map->offsets;
    a.rank_offsets = map->rank_offsets;
    a.pos = map->pos;
    a.row_src = map->row_src;
    a.drop_list = map->drop_list;
    a.n_dropped = map->n_dropped;
    a.xperm = xperm;
    a.status = scratch;
    a.scan_ticket = scratch + 1;
    a.hist = scratch + 64;
    a.drop_offsets = scratch + 64 + hist_ints;
    a.routed_offsets = a.drop_offsets + N;
    a.elist = by_gate ? a.routed_offsets + N + 1 : nullptr;
    e = launch_dispatch(a, stream);
    if (e != cudaSuccess) {
        g_last_cuda_error = std::string("moe_dispatch_static: ") + cudaGetErrorName(e) + " (" +
                            cudaGetErrorString(e) + ")";
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
