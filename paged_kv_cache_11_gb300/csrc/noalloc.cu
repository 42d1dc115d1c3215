// noalloc.cu -- paged_attention_decode_static: paged decode attention for
// callers that cannot allocate device memory.
//
// paged_attention_decode needs a caller-provided workspace for its split-K
// partials whenever a context spans more than one partition.  Some callers
// have no way to provide one:
//   - a process whose device memory has all been handed to another
//     allocator up front (for example a serving engine that reserves nearly
//     all of HBM for its KV-cache pool at start-up), so a cudaMalloc for a
//     per-call workspace fails or competes with that pool;
//   - a latency-critical decode loop that must not call cudaMalloc, because
//     the allocation can implicitly synchronise the device and stall every
//     stream in the process.
// This entry point takes no workspace.  The partials live in a file-scope
// device array of kStaticWorkspaceBytes (16 MiB) that every GPU which loads
// the library holds until the process exits.
//
// Set-up: the first call on a device looks up the array's device address
// with cudaGetSymbolAddress while that device is current and caches it; that
// first call should therefore come before any stream capture.  The array is
// shared by every call on the device and keeps the last call's contents; the
// decode kernels write every partial they later read, so nothing has to start
// at zero.  Calls whose kernels overlap on the GPU (for example on two
// streams) race on the array and must be serialised by the caller.
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {

constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_pkv_static_workspace[kStaticWorkspaceBytes];

constexpr int kStaticMaxDevices = 64;
static std::mutex g_static_ws_mutex;
static void* g_static_ws_ptr[kStaticMaxDevices] = {};

// Device address of this device's copy of the array.  In host code the
// array's name is only a host-side stand-in, never a device address.
static void* static_workspace() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_static_ws_mutex);
    if (!g_static_ws_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_pkv_static_workspace) != cudaSuccess) {
            (void)cudaGetLastError();  // the caller reports PKV_ERR_CUDA; leave no sticky error behind
            return nullptr;
        }
        g_static_ws_ptr[dev] = ptr;
    }
    return g_static_ws_ptr[dev];
}

}  // namespace pkv

extern "C" pkv_status paged_attention_decode_static(const void* q, const void* k_cache, const void* v_cache,
                                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                    const int32_t* context_lens, int32_t num_seqs,
                                                    int32_t num_q_heads, int32_t max_context_len, float scale,
                                                    void* out, int32_t out_dtype, const pkv_cache_desc* cache,
                                                    int32_t partition_size, void* stream) {
    if (!cache) return PKV_ERR_INVALID_ARG;
    const size_t need =
        paged_attention_workspace_bytes(num_seqs, num_q_heads, cache->head_dim, max_context_len, partition_size);
    if (need > pkv::kStaticWorkspaceBytes) return PKV_ERR_WORKSPACE;  // beyond the fixed 16 MiB array
    void* ws = nullptr;
    if (need > 0) {
        ws = pkv::static_workspace();
        if (!ws) return PKV_ERR_CUDA;
    }
    return paged_attention_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                  num_q_heads, max_context_len, scale, out, out_dtype, cache, partition_size, ws,
                                  ws ? pkv::kStaticWorkspaceBytes : 0, stream);
}
