// pa_decode_attention_static: paged decode attention for callers that cannot
// allocate device memory.
//
// Some callers of this library have no way to obtain scratch memory: a plugin
// inside a host framework that owns every device allocation, or a serving
// loop that must not allocate once it is running.  They cannot hand
// pa_decode_attention the workspace it needs for split-sequence partials.
// This entry point instead uses one statically sized buffer
// per GPU, held in this library's device image for as long as the process
// runs, and otherwise runs the same decode path.
#include <mutex>

#include "pa_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = (size_t)PA_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// Device scratch shared by every call on a device.  In host code this name is
// only a stand-in for the symbol, never a device address: the address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mu;
void* g_workspace_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device, looked up once per device.
pa_status static_workspace(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_workspace_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_workspace_ptr[dev] = p;
    }
    *out = g_workspace_ptr[dev];
    return PA_OK;
}


}  // namespace

extern "C" pa_status pa_decode_attention_static(void* out, const void* q, const void* k_pool, const void* v_pool,
                                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                int32_t block_size, int32_t num_blocks, float scale,
                                                int32_t partition_tokens, pa_dtype dtype, int32_t* dev_status_out,
                                                void* stream) {
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(dev_status_out) & 3u) return PA_ERR_INVALID_ARG;
    void* ws = nullptr;
    pa_status s = static_workspace(&ws);
    if (s != PA_OK) return s;
    // The buffer keeps the previous call's contents.  The decode checks every
    // argument first, refuses a launch whose grid needs more scratch than the
    // buffer holds (PA_ERR_WORKSPACE_TOO_SMALL, nothing enqueued), and only then
    // zeroes the status word and the merge counters at the buffer's head; the
    // partial slots are written before they are read.
    s = pa::decode_common(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                          num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_tokens, ws,
                          kStaticWorkspaceBytes, dtype, 1.f, 1.f, stream, /*clear_status=*/true);
    if (s != PA_OK) return s;
    if (dev_status_out && cudaMemcpyAsync(dev_status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}
