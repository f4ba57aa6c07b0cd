// pa_decode_attention_static_ws: decode attention for callers that cannot
// allocate device memory.  The split-K partials and merge counters live in a
// workspace owned by this library (a file-scope device array) instead of one
// the caller allocates.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pa.h"

namespace {

constexpr size_t kStaticWsBytes = PA_STATIC_WORKSPACE_BYTES;

// The workspace itself.  Every GPU that loads this library holds one copy of
// it until the process exits.  In host code the name is only a host-side
// stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
void* g_ws_addr[kMaxDevices] = {};
std::mutex g_ws_mu;

// Device address of g_static_ws on the current device; looked up once per
// device, with that device current.
pa_status static_ws_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    if (!g_ws_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p) return PA_ERR_CUDA;
        g_ws_addr[dev] = p;
    }
    *out = g_ws_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_attention_static_ws(
    void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, const int32_t* seq_lens, int batch,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
    int num_blocks, float scale, int num_splits, int kv_dtype, void* stream) {
    if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
        num_splits < 0)
        return PA_ERR_INVALID;
    if (batch == 0) return PA_OK;
    const size_t need = pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                                                  max_blocks_per_seq, num_splits);
    if (need == 0 || need > kStaticWsBytes) return PA_ERR_INVALID;  // too large for the static workspace
    void* ws = nullptr;
    const pa_status st = static_ws_address(&ws);
    if (st != PA_OK) return st;
    // The merge counters are the workspace's last part and must start at zero;
    // the array keeps whatever the previous call left.
    const size_t zero_bytes = (((size_t)batch * num_kv_heads * sizeof(int)) + 255) & ~(size_t)255;
    if (cudaMemsetAsync(static_cast<char*>(ws) + (need - zero_bytes), 0, zero_bytes,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    return pa_decode_attention(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, batch,
                               num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                               num_blocks, scale, num_splits, ws, kStaticWsBytes, kv_dtype, stream);
}
