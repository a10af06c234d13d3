// lora_linear_static_scratch: the layer for callers that cannot allocate.
//
// lora_plan / lora_linear keep their per-step state (the plan arrays and the
// shrink result U) in a workspace the caller allocates. Some callers have no
// way to do that: a host program that hands out device memory only from its
// own fixed arena and forbids third-party cudaMalloc; a C caller with no
// device allocator at hand; a latency-critical decode loop that cannot afford
// cudaMalloc / cudaFree, which may synchronize the whole device. For them this
// entry point keeps that state in a fixed array of this library instead.
//
// The array lives in device memory for as long as the library is loaded, on
// every GPU that loads it (kScratchBytes bytes each). Its name is only a
// host-side stand-in for the device address, so the address is looked up once
// per device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device; make that first call before any stream capture.
// All calls share the array and it keeps the last call's contents; every call
// rewrites all of it that it reads, so nothing needs clearing, but calls whose
// work overlaps on the GPU (other streams, other host threads) race on it.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>
#include "lora_gb300.h"

namespace {

// Plan + U for up to 256 token rows, 64 slots and rank 64 (a decode-sized
// batch; such batches need no plan-ordered copy of x).
constexpr int kStaticMaxT = 256;
constexpr int kStaticMaxS = 64;
constexpr int kStaticMaxR = 64;
constexpr size_t kScratchBytes = 72 * 1024;

static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

// Device address of g_static_scratch, per device (null until looked up).
void* scratch_address() {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" lora_status lora_linear_static_scratch(const void* x, const void* W, int T, int d_in, int d_out,
                                                  const lora_pool* pool, const int32_t* ids, void* y,
                                                  void* stream) {
    if (!pool || T < 0) return LORA_EINVAL;
    if (T > kStaticMaxT || pool->S > kStaticMaxS || pool->R_max > kStaticMaxR) return LORA_ESCRATCH;
    const size_t need = lora_plan_workspace_bytes(T, pool->S, pool->R_max, d_in);
    if (need == 0) return LORA_EINVAL;
    if (need > kScratchBytes) return LORA_ESCRATCH;
    if (T == 0) return LORA_OK;
    void* ws = scratch_address();
    if (!ws) return LORA_ECUDA;
    lora_plan_t plan;
    lora_status st = lora_plan_init(&plan, ws, kScratchBytes, T, pool->S, pool->R_max, d_in);
    if (st != LORA_OK) return st;
    st = lora_plan(ids, T, &plan, stream);
    if (st != LORA_OK) return st;
    return lora_linear(x, W, T, d_in, d_out, pool, &plan, y, stream);
}
