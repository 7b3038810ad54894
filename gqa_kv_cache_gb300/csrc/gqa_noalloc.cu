// Decode step for callers that cannot allocate device memory.
//
// Some callers cannot give this library a workspace: plugin hosts that hand
// an operator no scratch buffer and forbid device allocation while it runs
// (allocating in the middle of a step would synchronise the device or break
// the host's planned memory layout), and plain C callers with no device
// allocator of their own. For them gqa_decode_step_noalloc runs the dense /
// continuous-batch decode step with its scratch in a fixed array that lives in
// the library image itself, so the call allocates nothing.
//
// The array is a file-scope __device__ variable of kScratchBytes (8 MiB): every
// GPU that loads the library holds it until the process exits. In host code
// its name is only a stand-in, not a device address, so the address is looked
// up with cudaGetSymbolAddress once per device, with that device current, on
// the first call made on that device; that first call should therefore come
// before any stream capture. The address is kept for the life of the process,
// so the entry point must not be used on a device after cudaDeviceReset (or
// anything else that destroys its primary context and reloads the module). All calls share the one array and it keeps the
// last call's contents: calls whose kernels overlap on the GPU (two streams,
// or two threads) race on it and must be serialised by the caller. Of the
// scratch only the per-(row, head) arrival counters must start at zero (a
// completed call leaves all of it zero); each call still clears the counters
// (an asynchronous memset on its stream, no allocation) before its kernel, so
// even a call left incomplete cannot affect the next.
#include <cuda_runtime.h>

#include <mutex>

#include "gqa_common.cuh"
#include "gqa_decode.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of g_scratch on the current device (looked up once per device).
gqa_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return GQA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return GQA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
            return GQA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GQA_OK;
}

}  // namespace

extern "C" {

size_t gqa_noalloc_scratch_bytes(void) { return kScratchBytes; }

gqa_status gqa_decode_step_noalloc(const void *q, const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *lengths,
                                   const int32_t *slot_ids, float *out, int B, int Hq, int Hkv,
                                   int D, int R, int Smax, gqa_dtype dt, int32_t *d_status,
                                   void *stream)
{
    const size_t need = gqa_workspace_bytes(B, Hq, Hkv, D, dt, nullptr);
    if (need > kScratchBytes)
        return GQA_ERR_TOO_LARGE;
    void *ws = nullptr;
    const gqa_status st = scratch_address(&ws);
    if (st != GQA_OK)
        return st;
    // need == 0 means the sizes are invalid: the regular entry point reports why.
    // The per-(row, head) arrival counters must start at zero: clear them on
    // this stream before the kernel (a memset, no allocation).
    if (need != 0 && B > 0 && Hkv > 0) {
        const size_t cnt = gqa::workspace_layout(B, Hkv, Hq / Hkv, D, 0).cnt_bytes;
        if (cudaMemsetAsync(ws, 0, cnt, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return GQA_ERR_CUDA;
    }
    return gqa_decode_step(q, k_new, v_new, k_cache, v_cache, lengths, slot_ids, out, B, Hq, Hkv,
                           D, R, Smax, dt, ws, kScratchBytes, d_status, stream);
}

}  // extern "C"
