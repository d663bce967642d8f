// sparse_attn_decode_noalloc: the decode step for callers that cannot allocate
// device memory.
//
// Some callers have no way to call cudaMalloc or to hand over a workspace:
// code running inside another framework's allocator-less hooks, plugins whose
// host process owns every allocation, or code paths that must not allocate
// once serving has started. For them this entry point runs exactly the same
// kernels as sparse_attn_decode, but its scratch memory (scores, kept
// positions, split partials, tickets) lives in one file-scope __device__ array
// of fixed size that the library carries with it. The caller still passes the
// inputs and the outputs.
//
// Costs and rules:
//   - every GPU that loads the library holds SA_DECODE_NOALLOC_SCRATCH_BYTES
//     of device memory for this array until the process exits;
//   - requests whose sa_decode_workspace_size exceeds that limit are rejected
//     with SA_ERR_WORKSPACE before anything is enqueued;
//   - all calls share the one array, and it keeps the previous call's
//     contents: the decode step clears what has to start at zero (its tickets)
//     itself, but two calls whose work overlaps on the GPU (different streams,
//     or different host threads) race on the array and give wrong results;
//   - the device address of the array is looked up once per device, with that
//     device current, on the first call made on that device: make that first
//     call before any stream capture begins.
#include <cuda_runtime.h>
#include <mutex>

#include "../../include/sparse_attn.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[SA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_lock;
void* g_scratch_ptr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device (host code may
// not use the symbol itself: on the host it names a stand-in, not device memory).
int scratch_on_current_device(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        (void)cudaGetLastError();
        return SA_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> guard(g_lock);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return SA_ERR_LAUNCH;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SA_OK;
}

}  // namespace

extern "C" SA_API int sparse_attn_decode_noalloc(const sa_decode_args* args, cudaStream_t stream)
{
    const size_t need = sa_decode_workspace_size(args);
    if (need == 0) return sparse_attn_decode(args, nullptr, 0, stream);   // reports the argument error
    if (need > (size_t)SA_DECODE_NOALLOC_SCRATCH_BYTES) return SA_ERR_WORKSPACE;
    void* ws = nullptr;
    const int st = scratch_on_current_device(&ws);
    if (st != SA_OK) return st;
    return sparse_attn_decode(args, ws, (size_t)SA_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
