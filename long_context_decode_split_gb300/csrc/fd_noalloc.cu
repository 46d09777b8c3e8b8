// fd_noalloc.cu -- fd_decode_dense_noalloc: the dense split-KV decode for
// callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plug-in running inside a
// host engine that has already reserved all device memory for itself and
// hands out no allocator, or a latency-critical decode loop that must not
// call cudaMalloc/cudaFree because those calls can synchronise the device.
// This entry point takes its scratch (the per-chunk partial results) from a
// fixed array in this library's device memory instead of a caller buffer.
//
// The array is a file-scope __device__ object of FD_NOALLOC_SCRATCH_BYTES
// bytes (fd.h).
// Every GPU that loads the library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the address is
// looked up with cudaGetSymbolAddress once per device, on the first call made
// with that device current, and then passed to the kernels.
#include <atomic>

#include <cuda_runtime.h>

#include "fd.h"

namespace {

constexpr size_t kNoAllocScratchBytes = FD_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (nullptr on
// failure).  Looked up once per device and cached; host threads making their
// first calls at the same time may each look it up, and store the same value.
void* scratch_address() {
    static std::atomic<void*> cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < kMaxDevices) {
        void* hit = cache[dev].load(std::memory_order_relaxed);
        if (hit) return hit;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(p, std::memory_order_relaxed);
    return p;
}

}  // namespace

extern "C" {

int fd_decode_dense_noalloc(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                            int B, int Hq, int Hkv, int L_max, int d, float scale, int num_splits,
                            void* out, int out_dtype, float* lse, void* stream) {
    // The same plan fd_decode_dense would make; its workspace must fit the array.
    const size_t need = fd_decode_workspace_size(B, Hq, Hkv, L_max, d, num_splits, seq_lens != nullptr);
    if (need > kNoAllocScratchBytes) return FD_ERR_WORKSPACE_TOO_SMALL;
    void* ws = nullptr;
    if (need > 0) {
        ws = scratch_address();
        if (!ws) return FD_ERR_CUDA;
    }
    return fd_decode_dense(q, k, v, seq_lens, B, Hq, Hkv, L_max, d, scale, num_splits, out, out_dtype, lse,
                           ws, ws ? kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"
