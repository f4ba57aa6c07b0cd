// pa_decode_attention_static_ws: decode attention for callers that cannot
// allocate device memory.  The split-K partials and merge counters live in a
// workspace owned by this library (a file-scope device array) instead of one
// the caller allocates.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kStaticWsBytes = PA_STATIC_WORKSPACE_BYTES;

// The workspace itself.  Every GPU that loads this library holds one copy of
// it until the process exits.  In host code the name is only a host-side
// stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// The device address is looked up once per CUDA context, with the device
// current, and cached under the context's unique id: after a
// cudaDeviceReset the runtime makes a new primary context (with a new id and
// a new copy of the array), so the stale address is never reused.
constexpr int kMaxDevices = 64;
struct WsAddr {
    unsigned long long ctx_id;
    void* addr;
};
WsAddr g_ws[kMaxDevices] = {};
std::mutex g_ws_mu;

struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
    static CtxFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    return f;
}

// Device address of g_static_ws in the current device's current context.
pa_status static_ws_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    const CtxFns& f = ctx_fns();
    if (!f.get_current || !f.get_id) return PA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
    if (!ctx) {
        // no context is bound to this thread yet: the symbol lookup makes the
        // runtime bind the device's primary context
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return PA_ERR_CUDA;
        if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return PA_ERR_CUDA;
    }
    unsigned long long id = 0;
    if (f.get_id(ctx, &id) != CUDA_SUCCESS) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    if (!g_ws[dev].addr || g_ws[dev].ctx_id != id) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p) return PA_ERR_CUDA;
        g_ws[dev].addr = p;
        g_ws[dev].ctx_id = id;
    }
    *out = g_ws[dev].addr;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_attention_static_ws(
    void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, const int32_t* seq_lens, int batch,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
    int num_blocks, float scale, int num_splits, int kv_dtype, void* stream) {
    pa::CallRange range("pa_decode_attention_static_ws");
    // every argument check first: a refused call queues no work on the array
    const pa_status chk = pa::decode_check(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, batch,
                                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                           num_blocks, scale, num_splits, kv_dtype, nullptr, nullptr);
    if (chk != PA_OK || batch == 0) return chk;
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
