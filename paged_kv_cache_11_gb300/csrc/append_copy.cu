// append_copy.cu -- the block write and the batched copy-on-write block copy
// (tonho.wtf "vllm", "o que isso custou": the method needs its own kernels
// for block write and batched block copy; "como funciona": slots are filled
// left to right, and a write into the last shared block copies that block
// and only it).
//
// Both are pure data movement.  Rows and blocks are moved as 16-byte vectors
// so that every warp issues fully coalesced 512-byte transactions; each
// thread keeps several vectors in flight.
#include "pkv_internal.cuh"

namespace pkv {

// One thread per 16-byte vector of a (token, KV head) row, for K and V.
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
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
    const int pair = blockIdx.x;
    const int layer = blockIdx.z >> 1;
    const int64_t src = __ldg(p.pairs + 2 * pair), dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_error(p.err, PKV_DEVERR_COPY_ID);
        return;
    }
    uint4* base = (blockIdx.z & 1) ? p.v[layer] : p.k[layer];
    const uint4* from = base + src * p.block_vecs;
    uint4* to = base + dst * p.block_vecs;
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

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream, int* launches) {
    const int64_t total = p.num_tokens * p.num_kv_heads * p.row_vecs;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    append_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) ++*launches;
    return e;
}

cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream, int* launches) {
    if (p.num_pairs == 0 || p.num_layers == 0) return cudaSuccess;
    const int64_t chunks = (p.block_vecs + kCopyChunk - 1) / kCopyChunk;
    const dim3 grid((unsigned)p.num_pairs, (unsigned)chunks, (unsigned)(2 * p.num_layers));
    copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) ++*launches;
    return e;
}

}  // namespace pkv
