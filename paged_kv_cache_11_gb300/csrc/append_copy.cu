// append_copy.cu -- the data-movement kernels of the paged cache:
//   - the block write (tonho.wtf "vllm", "o que isso custou": the method
//     needs its own kernel for block write; "como funciona": slots are
//     filled left to right);
//   - whole-block moves: the batched copy-on-write copy ("como funciona": a
//     write into the last shared block copies that block and only it; "o que
//     isso custou": batched block copy) and swapping blocks out to CPU RAM
//     and back ("como funciona": evicted sequences are swapped to CPU RAM or
//     recomputed);
//   - token-row moves into fresh target blocks (gist.science "Zipage",
//     Compressed PagedAttention: the kept tokens of a request are rewritten
//     into new target blocks so that shared prefix blocks stay intact).
//
// All are pure data movement.  Rows and blocks are moved as 16-byte vectors
// so that every warp issues fully coalesced 512-byte transactions; each
// thread keeps several vectors in flight.  A pool may live in page-locked
// host memory the GPU addresses directly (over NVLink-C2C on GB300).
#include "pkv_internal.cuh"

namespace pkv {

// One thread per 16-byte vector of a (token, KV head) row, for K and V.
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
    pdl_launch_dependents();
    pdl_wait();  // the previous kernel may still read the slots written here
    const int64_t per_token = (int64_t)p.num_kv_heads * p.row_vecs;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.num_tokens * per_token) return;
    const int64_t t = i / per_token;
    const int64_t rem = i - t * per_token;
    const int h = (int)(rem / p.row_vecs);
    const int c = (int)(rem - (int64_t)h * p.row_vecs);
    const int64_t slot = __ldg(p.slot_mapping + t);
    if (slot < 0) return;  // padding token
    if (slot >= p.num_slots) {
        if (rem == 0) record_error(p.err, PKV_DEVERR_SLOT);
        return;
    }
    const int64_t blk = slot / p.block_size, off = slot - blk * p.block_size;
    const int64_t dst = ((blk * p.num_kv_heads + h) * p.block_size + off) * p.row_vecs + c;
    const uint4 kv = __ldg(p.k + i);
    const uint4 vv = __ldg(p.v + i);
    p.k_cache[dst] = kv;
    p.v_cache[dst] = vv;
}

// grid: x = pair, y = 4096-vector chunk of the block, z = 2 * layer + (0: K, 1: V)
constexpr int kCopyThreads = 256;
constexpr int kCopyVecsPerThread = 4;
constexpr int kCopyChunk = kCopyThreads * kCopyVecsPerThread * 4;  // vectors per CTA (64 KiB)

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int pair = blockIdx.x;
    const int layer = blockIdx.z >> 1;
    const int64_t src = __ldg(p.pairs + 2 * pair), dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.src_blocks || dst < 0 || dst >= p.dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_error(p.err, p.err_code);
        return;
    }
    const uint4* from = ((blockIdx.z & 1) ? p.src_v[layer] : p.src_k[layer]) + src * p.block_vecs;
    uint4* to = ((blockIdx.z & 1) ? p.dst_v[layer] : p.dst_k[layer]) + dst * p.block_vecs;
    const int64_t begin = (int64_t)blockIdx.y * kCopyChunk;
    const int64_t end = min(p.block_vecs, begin + kCopyChunk);
    for (int64_t i0 = begin + threadIdx.x; i0 < end; i0 += (int64_t)kCopyThreads * kCopyVecsPerThread) {
        uint4 r[kCopyVecsPerThread];
#pragma unroll
        for (int u = 0; u < kCopyVecsPerThread; ++u) {
            const int64_t i = i0 + (int64_t)u * kCopyThreads;
            if (i < end) r[u] = from[i];
        }
#pragma unroll
        for (int u = 0; u < kCopyVecsPerThread; ++u) {
            const int64_t i = i0 + (int64_t)u * kCopyThreads;
            if (i < end) to[i] = r[u];
        }
    }
}

// One thread per 16-byte vector of a (token, KV head) row, for K and V.
__global__ void __launch_bounds__(256) compact_kernel(const CompactParams p) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t per_token = (int64_t)p.num_kv_heads * p.row_vecs;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.num_tokens * per_token) return;
    const int64_t t = i / per_token;
    const int64_t rem = i - t * per_token;
    const int h = (int)(rem / p.row_vecs);
    const int c = (int)(rem - (int64_t)h * p.row_vecs);
    const int64_t from = __ldg(p.src_slots + t), to = __ldg(p.dst_slots + t);
    if (from < 0 || to < 0) return;  // padding
    if (from >= p.num_slots || to >= p.num_slots) {
        if (rem == 0) record_error(p.err, PKV_DEVERR_SLOT);
        return;
    }
    const int64_t fb = from / p.block_size, fo = from - fb * p.block_size;
    const int64_t tb = to / p.block_size, to_ = to - tb * p.block_size;
    const int64_t src = ((fb * p.num_kv_heads + h) * p.block_size + fo) * p.row_vecs + c;
    const int64_t dst = ((tb * p.num_kv_heads + h) * p.block_size + to_) * p.row_vecs + c;
    const uint4 kv = p.k_cache[src];
    const uint4 vv = p.v_cache[src];
    p.k_cache[dst] = kv;
    p.v_cache[dst] = vv;
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream, int* launches) {
    const int64_t total = p.num_tokens * p.num_kv_heads * p.row_vecs;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    const cudaError_t e = launch_pdl(append_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, p);
    if (e == cudaSuccess) ++*launches;
    return e;
}

cudaError_t launch_compact(const CompactParams& p, cudaStream_t stream, int* launches) {
    const int64_t total = p.num_tokens * p.num_kv_heads * p.row_vecs;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    const cudaError_t e = launch_pdl(compact_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, p);
    if (e == cudaSuccess) ++*launches;
    return e;
}

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream, int* launches) {
    if (p.num_pairs == 0 || p.num_layers == 0) return cudaSuccess;
    const int64_t chunks = (p.block_vecs + kCopyChunk - 1) / kCopyChunk;
    const dim3 grid((unsigned)p.num_pairs, (unsigned)chunks, (unsigned)(2 * p.num_layers));
    const cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), 0, stream, p);
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace pkv
