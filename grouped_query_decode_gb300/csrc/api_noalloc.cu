// gqa_decode_noalloc: the decode step for callers that must not allocate
// device memory at call time.
//
// Some callers cannot let a library call cudaMalloc once they are running: a
// serving engine that reserved all device memory for its own pool at start-up
// (a cudaMalloc then fails or steals from the KV cache), a plugin inside
// another framework that is handed tensors but no allocator, or a decode loop
// that must not take cudaMalloc's implicit device synchronisation on its hot
// path. For them this entry point takes its split-KV scratch from a fixed
// array in device memory that the library reserves when it is loaded, instead
// of from cudaMalloc. The caller still passes inputs and outputs.
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "gqa_decode.h"

namespace {

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
std::map<int, void*> g_scratch_ptr;  // device id -> device address of the array

// The array's name is only a host-side stand-in in host code; the device
// address is looked up once per device, with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GQA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    auto it = g_scratch_ptr.find(dev);
    if (it == g_scratch_ptr.end()) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return GQA_ERR_CUDA;
        it = g_scratch_ptr.emplace(dev, p).first;
    }
    *out = it->second;
    return GQA_OK;
}

}  // namespace

extern "C" int gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* seq_lens, float scale, void* out, float* lse,
                                  int B, int sq, int H, int G, int D, int Tmax,
                                  cudaStream_t stream) {
    const size_t need = gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax);
    if (need == 0)  // bad arguments or no device: let the checks report which
        return gqa_decode_ex(q, k_cache, v_cache, seq_lens, scale, out, lse, B, sq, H, G, D,
                             Tmax, nullptr, 0, stream);
    if (need > (size_t)GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != GQA_OK) return st;
    return gqa_decode_ex(q, k_cache, v_cache, seq_lens, scale, out, lse, B, sq, H, G, D, Tmax,
                         scratch, (size_t)GQA_NOALLOC_SCRATCH_BYTES, stream);
}
