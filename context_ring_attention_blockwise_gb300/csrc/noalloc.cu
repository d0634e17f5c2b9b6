// noalloc.cu -- cpattn_forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code that runs inside a memory allocator's own
// hooks (calling the allocator again would recurse), a plug-in loaded into a host process that
// owns every device memory pool, a real-time loop that may not wait on an allocation. For them
// this file holds the forward's scratch in a statically sized device array that the CUDA runtime
// places when the library is loaded, so the call itself allocates nothing: not on the device, and
// not on the host either (the unit-order table reaches the device inside kernel parameters, not
// through a page-locked staging copy).
//
// The array is kNoAllocScratchBytes (64 MiB) plus alignment slack. Every GPU that loads the
// library keeps it until the process exits. All calls share it and it keeps whatever the last
// call left there; the forward's own prologue clears the parts that must start at zero (the
// error header, the tile counters, the scheduler counters) on every call. Calls whose work
// overlaps on the GPU (different streams, or different host threads) race on the array; issue
// them on one stream, one after another. A device-side timeout of such a call is recorded in the
// array's header and read back by cpattn_check_noalloc.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

// Device-side scratch. In host code this name is only a stand-in for the symbol: its device
// address comes from cudaGetSymbolAddress on each device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes + 1024];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The 1024-byte aligned start of the scratch on the current device. Set-up, once per device with
// that device current: ask the runtime where it placed the array on this device. The first call
// of any entry point below on a device does this.
cpattn_status_t scratch_on_current_device(const char* who, void** ws) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        cpattn::set_last_error(std::string(who) + ": no usable current CUDA device");
        return CPATTN_ERR_CUDA;
    }
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_addr[dev]) {
            void* ptr = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr) {
                cpattn::set_last_error(std::string(who) + ": cudaGetSymbolAddress failed: " + cudaGetErrorString(e));
                return CPATTN_ERR_CUDA;
            }
            g_scratch_addr[dev] = ptr;
        }
        base = g_scratch_addr[dev];
    }
    // The forward wants a 1024-byte aligned workspace; the slack after the array covers it.
    const uintptr_t p = reinterpret_cast<uintptr_t>(base);
    *ws = reinterpret_cast<void*>((p + 1023) & ~uintptr_t(1023));
    return CPATTN_OK;
}

}  // namespace

extern "C" cpattn_status_t cpattn_forward_noalloc(cpattn_plan_t plan, int B, const void* q, const void* k,
                                                  const void* v, const int32_t* pos, float scale, void* o,
                                                  float* lse, cpattn_stream_t stream) {
    if (!plan || B <= 0) {
        cpattn::set_last_error("cpattn_forward_noalloc: plan and B > 0 required");
        return CPATTN_ERR_INVALID;
    }
    size_t need = 0;
    cpattn_status_t s = cpattn_workspace_size(plan, B, &need);
    if (s != CPATTN_OK) return s;
    if (need > kNoAllocScratchBytes) {
        char buf[240];
        std::snprintf(buf, sizeof buf,
                      "cpattn_forward_noalloc: this problem needs %zu bytes of scratch but the static scratch "
                      "holds %zu bytes (64 MiB); use cpattn_forward with a caller-owned workspace",
                      need, kNoAllocScratchBytes);
        cpattn::set_last_error(buf);
        return CPATTN_ERR_WORKSPACE;
    }
    void* ws = nullptr;
    if ((s = scratch_on_current_device("cpattn_forward_noalloc", &ws))) return s;
    // The unit order reaches the scratch inside kernel parameters (as for every forward): no
    // host copy is made.
    return cpattn::forward_with_workspace(plan, B, q, k, v, pos, scale, o, lse, ws, kNoAllocScratchBytes, stream);
}

extern "C" cpattn_status_t cpattn_check_noalloc(cpattn_plan_t plan) {
    void* ws = nullptr;
    if (cpattn_status_t s = scratch_on_current_device("cpattn_check_noalloc", &ws)) return s;
    return cpattn_check(plan, ws);
}

extern "C" cpattn_status_t cpattn_selftest_wait_timeout_noalloc(uint64_t timeout_ns, cpattn_stream_t stream) {
    void* ws = nullptr;
    if (cpattn_status_t s = scratch_on_current_device("cpattn_selftest_wait_timeout_noalloc", &ws)) return s;
    return cpattn_selftest_wait_timeout(ws, kNoAllocScratchBytes, timeout_ns, stream);
}
