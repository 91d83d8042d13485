// fr_noalloc.cu -- fr_decode_attn for callers that cannot allocate device memory.
//
// Some hosts cannot hand this library a workspace: their device memory is
// planned once, up front, by an allocator they do not control (a graph
// allocator that sizes every buffer before the first evaluation, or a plugin
// living inside another framework's memory pool), or they run a real-time loop
// that must not allocate after start-up so its latency stays predictable. They
// can still pass inputs and outputs. For them, fr_decode_attn_noalloc uses a
// fixed scratch array compiled into the library in place of the caller's
// workspace.
//
// The array below lives in every GPU that loads the library, from load until
// the process exits (kScratchBytes per device).
#include <mutex>

#include <cuda_runtime.h>

#include "fr_attn.h"
#include "fr_kernels.h"

namespace {

constexpr size_t kScratchBytes = (size_t)9 << 20;   // 9 MiB
constexpr size_t kTicketsBegin = 256;                // arrival tickets: [256, 1024)
constexpr size_t kTicketsEnd = 1024;                 // (the status word at [0, 4) is kept)
constexpr int kMaxDevices = 64;

// Scratch for the split-KV partial states, the arrival tickets and the status
// word. In host code this name is only a stand-in: the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices];

// Set-up, once per device, with that device current: look up the device
// address of the scratch array.
fr_status scratch_address(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FR_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return FR_OK;
}

}  // namespace

extern "C" fr_status fr_decode_attn_noalloc(const uint16_t* q16, const float* q, int64_t q_tok_stride,
                                            const int32_t* pos, const fr_rope_params* rp, float q_scale,
                                            const uint16_t* k, int64_t k_row_stride, const uint16_t* v,
                                            int64_t v_row_stride, const uint16_t* mask,
                                            int64_t mask_row_stride, int n_tok, int n_head, int hd, int n_kv,
                                            float kq_scale, float* out, cudaStream_t stream) {
    if (n_tok < 1 || n_head < 1 || n_kv < 1) return FR_ERR_INVALID_ARG;
    const size_t need = fr::decode_attn_min_workspace_bytes(n_tok, n_head, hd, n_kv);
    if (need == 0) return FR_ERR_UNSUPPORTED;
    if (need > kScratchBytes) return FR_ERR_WORKSPACE;       // beyond the fixed scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FR_ERR_UNSUPPORTED;
    void* ws = nullptr;
    const fr_status st = scratch_address(dev, &ws);
    if (st != FR_OK) return st;
    // The array keeps whatever the previous call left: the arrival tickets must
    // start at zero. The status word is left alone, so that a device-side
    // timeout stays visible until fr_decode_attn_noalloc_check reads it.
    if (cudaMemsetAsync(static_cast<unsigned char*>(ws) + kTicketsBegin, 0, kTicketsEnd - kTicketsBegin, stream) !=
        cudaSuccess)
        return FR_ERR_CUDA;
    return fr_decode_attn(q16, q, q_tok_stride, pos, rp, q_scale, k, k_row_stride, v, v_row_stride, mask,
                          mask_row_stride, n_tok, n_head, hd, n_kv, kq_scale, out, ws, kScratchBytes, stream);
}

extern "C" fr_status fr_decode_attn_noalloc_check(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FR_ERR_UNSUPPORTED;
    void* ws = nullptr;
    const fr_status st = scratch_address(dev, &ws);
    if (st != FR_OK) return st;
    return fr_workspace_check(ws, stream);
}
