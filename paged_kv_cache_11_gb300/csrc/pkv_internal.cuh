// pkv_internal.cuh -- internal declarations shared by the library's
// translation units: launch parameter blocks, launcher entry points, the
// per-device error word and thin inline-PTX wrappers (mbarrier, TMA,
// ldmatrix, mma.sync) for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

constexpr int kHeadDim = 128;          // supported head_dim
constexpr int kAutoPartition = 512;    // smallest automatic split-K partition (tokens)
constexpr int kDecodeCtasPerSm = 5;    // resident decode CTAs per SM the kernel is tuned for
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bound on any in-CTA wait (2 s)
// Split-K calls with at most this many partitions per sequence merge inside
// the decode kernel (the last partition to finish merges); longer ones use
// the separate merge kernel.
#ifndef PKV_FUSE_MERGE_MAX_PARTS
#define PKV_FUSE_MERGE_MAX_PARTS 16
#endif
constexpr int kFuseMergeMaxParts = PKV_FUSE_MERGE_MAX_PARTS;

// The per-device error word lives in the API translation unit; kernels get
// its device address as a parameter.  First error wins (atomicCAS from 0).
__device__ __forceinline__ void record_error(int* err, int code) { atomicCAS(err, 0, code); }

// ---------------------------------------------------------------------------
// Launch parameters
// ---------------------------------------------------------------------------
struct DecodeParams {
    const void* q;               // [B][Hq][D]
    const int32_t* block_tables; // [B][max_blocks_per_seq]
    const int32_t* context_lens; // [B]
    void* out;                   // [B][Hq][D] of out_dtype
    float* part_o;               // [B][Hq][max_parts][D]   (split only)
    float* part_lse;             // [B][Hq][max_parts], log2 domain (split only)
    int* err;                    // device error word
    // fused merge: one 64-bit arrival counter per (sequence, head group),
    // holding (epoch << 16) | arrivals; a counter whose epoch is not this
    // call's counts as zero, so the counters never need clearing.
    unsigned long long* merge_ctr;  // [B][Hkv * head_tiles]
    unsigned long long epoch;       // this call's epoch, 1 .. 2^48 - 1
    int fuse_merge;                 // 1: the last partition of a row merges
    // fused block write (paged_attention_append_decode): sequence s's new
    // token, k_new/v_new [B][Hkv][D], goes to slot_mapping[s], which must be
    // the slot of its last context position
    const uint4* k_new;
    const uint4* v_new;
    const int64_t* slot_mapping;
    uint4* k_cache;
    uint4* v_cache;
    int fused_append;
    int64_t num_blocks;
    int num_seqs, num_q_heads, num_kv_heads;
    int max_blocks_per_seq;
    int len_limit;               // min(max_context_len, max_blocks_per_seq * block_size)
    int partition_size;          // tokens, multiple of block_size
    int max_parts;               // partial slots per (sequence, query head): ceil(max_context_len /
                                 // partition_size) (+ prefix_parts in grouped decode), >= 1
    int group;                   // G = Hq / Hkv
    int head_tiles;              // ceil(G / decode_head_tile(G))
    int out_dtype;               // pkv_dtype
    int split;                   // 1: sequences with > 1 partition write partials
    int block_size;
    float scale_log2;            // scale * log2(e)
    // grouped decode (paged_attention_decode_grouped): sequence s's first
    // prefix_lens[s] tokens are attended by the prefix kernel through the
    // block table of its group's first member, in prefix partitions of
    // prefix_partition tokens (partial indices 0 .. npre-1); the decode
    // kernel attends tokens prefix_lens[s] .. L-1 (partial indices npre ..).
    const int32_t* prefix_lens;     // [B]; nullptr: plain decode
    const int32_t* group_starts;    // [num_groups + 1]: members of group g are group_starts[g] .. [g+1]-1
    int* seq_group;                 // [B]: group the prefix kernel took s into (a hint: see group_verified)
    int max_prefix_len;
    int prefix_partition;           // tokens, multiple of block_size
    int prefix_parts;               // ceil(max_prefix_len / prefix_partition)
    int num_groups;
    int members_per_tile;           // group members per prefix CTA (whole members, <= 64 query rows)
    int row_tiles;                  // prefix CTAs per (group, KV head, prefix partition)
    int parts_in_x;                 // plain decode with > 65535 partitions: partition index in grid x
    // grouped decode: the prefix kernel ran first and let this kernel start
    // only once the kernels before the call had completed, so the decode
    // kernel reads its inputs at once and waits for the prefix kernel only
    // before it reads what that kernel writes (group hints, partials)
    int early_inputs;
};

// Prefix partitions of grouped decode (tokens): chosen per call between the
// smallest (which sizes the workspace) and the largest.
constexpr int kPrefixPartition = 256;
constexpr int kPrefixPartitionMax = 1024;
// Resident prefix CTAs per SM (about 214 KiB of shared memory and 512 TMEM columns each).
constexpr int kPrefixCtasPerSm = 1;
// Query rows of one prefix CTA (each fed twice to the prefix kernel's M = 128 products).
constexpr int kPrefixRows = 64;

// Query heads of one GQA group handled by one decode CTA (8 or 16).
__host__ __device__ inline int decode_head_tile(int group) { return group <= 8 ? 8 : 16; }

// Host-side launchers (decode.cu); return a cudaError_t from the launch.
cudaError_t launch_decode(const DecodeParams& p, int dtype, int block_size, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, cudaStream_t stream, int* launches);
// Grouped decode: the shared-prefix kernel (group_prefix.cu), then the
// decode kernel over each sequence's own tokens.
cudaError_t launch_group_prefix(const DecodeParams& p, int dtype, int block_size, const CUtensorMap& tmk,
                                const CUtensorMap& tmv, cudaStream_t stream, int* launches);

struct AppendParams {
    int* err;
    const uint4* k;
    const uint4* v;
    const int64_t* slot_mapping;
    uint4* k_cache;
    uint4* v_cache;
    int64_t num_tokens;
    int64_t num_slots;   // num_blocks * block_size
    int num_kv_heads, block_size, row_vecs;  // row_vecs = head_dim * elt / 16
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream, int* launches);

// Whole-block moves between two pools (the same pool for copy-on-write
// copies; a GPU pool and a host pool for swapping), up to kCopyMaxLayers
// layers per launch.
constexpr int kCopyMaxLayers = 32;
struct CopyParams {
    int* err;
    int err_code;                 // PKV_DEVERR_* recorded for an id outside a pool
    const uint4* src_k[kCopyMaxLayers];
    const uint4* src_v[kCopyMaxLayers];
    uint4* dst_k[kCopyMaxLayers];
    uint4* dst_v[kCopyMaxLayers];
    const int64_t* pairs;         // [num_pairs][2] = (src, dst)
    int64_t src_blocks, dst_blocks;
    int64_t block_vecs;           // 16-byte vectors per block of one cache
    int num_layers, num_pairs;
};
cudaError_t launch_copy_blocks(const CopyParams& p, cudaStream_t stream, int* launches);

// Token-row moves inside one pool: rows of every KV head from slot src[i]
// to slot dst[i] (compaction into fresh target blocks).
struct CompactParams {
    int* err;
    const int64_t* src_slots;
    const int64_t* dst_slots;
    uint4* k_cache;
    uint4* v_cache;
    int64_t num_tokens;
    int64_t num_slots;
    int num_kv_heads, block_size, row_vecs;
};
cudaError_t launch_compact(const CompactParams& p, cudaStream_t stream, int* launches);

// Launch a kernel with programmatic stream serialisation: it may start while
// the previous kernel on the stream is still running, and must call
// pdl_wait() before touching any memory that kernel could write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------------------
// Inline PTX
// ---------------------------------------------------------------------------
// Wait until the grid this one depends on has completed and its memory is
// visible (returns at once when there is none).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Order this thread's generic-proxy global writes before later async-proxy
// (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// GPU-scope acquire-release fence.  After a CTA barrier, one thread's fence
// releases the writes every thread of the CTA made before the barrier (and,
// after an atomic that observed other CTAs' releases, acquires theirs for the
// threads behind the next barrier).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Allow the next kernel on the stream to start launching its CTAs.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase of parity `parity` to complete; gives up after
// limit_ns and returns false.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// The bounded wait of every copy pipeline: kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled TMA load (coordinates innermost first) into this CTA's shared
// memory, completion counted on the mbarrier `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// 4-D tiled TMA load, as tma_load_3d.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            int w, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A * B, m16n8k16, fp32 accumulate; A row-major 16x16, B col-major 16x8.
template <bool kBF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (kBF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Pack two floats (lo in the low half) into a 16-bit pair, round to nearest
// even; also return the value each element rounded to.
template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi, float& lo_r, float& hi_r) {
    if constexpr (kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        lo_r = __low2float(v);
        hi_r = __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        lo_r = __low2float(v);
        hi_r = __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    float a, b;
    return pack2<kBF16>(lo, hi, a, b);
}

}  // namespace pkv

namespace pkv {
// Transpose an 8x8 matrix of 16-bit elements held in the standard warp
// fragment layout (thread l: row l/4, columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
}  // namespace pkv
