// api.cu -- the C ABI declared in include/pagedkv.h: argument checks on the
// host, TMA descriptor encoding, the per-device error word, and dispatch to
// the kernels in decode.cu and append_copy.cu.
#include <climits>
#include <cstring>
#include <atomic>
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {

// First device-side error since the last pkv_check_device_error, per device.
static __device__ int g_pkv_error = 0;

static std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
static std::mutex g_err_mutex;
static int* g_err_ptr[kMaxDevices] = {};

// Device address of this device's error word (looked up once per device).
static int* error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (!g_err_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_pkv_error) != cudaSuccess) {
            (void)cudaGetLastError();  // reported as PKV_ERR_CUDA; leave no sticky error behind
            return nullptr;
        }
        g_err_ptr[dev] = static_cast<int*>(ptr);
    }
    return g_err_ptr[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// The pool viewed as a 2-D tensor [num_blocks * Hkv * bs rows][128 columns];
// box = one 64-column half of a (block, KV head) tile, 128-byte swizzle.
// Tensor maps of a K or V pool, 128-byte swizzle (a 64-element, 128-byte
// row per line).  Rank 2: the pool as [rows][128] (rows = blocks x KV heads
// x block size), box [BS][64]: one copy brings one dims half of a (block,
// KV head) tile.  Rank 3: the same memory as [2 halves][rows][64], the two
// halves of a row 128 bytes apart, box [2][BS][64]: one copy brings the
// whole tile as its two halves back to back, the layout the rank-2 copies
// of both halves give.  Rank 4: the same memory as [rows / 8 groups][2
// halves][8 rows][64], box [BS / 8][2][8][64]: one copy brings the whole
// tile as 8-row groups of 2 KiB, each holding both halves of its 8 rows, so
// that tiles copied back to back keep every half's 8-row groups 2 KiB apart
// across tile boundaries (the layout the prefix kernel's 128-token tensor
// core operands need).  Every coordinate stays inside the pool.  No L2
// promotion: every copy is a whole contiguous tile half or tile, and
// promotion to 256-byte lines measured slightly slower on decode.
static pkv_status encode_cache_map(CUtensorMap* m, const void* base, const pkv_cache_desc& c, int rank) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    const cuuint64_t rows = (cuuint64_t)c.num_blocks * c.num_kv_heads * c.block_size;
    const CUtensorMapDataType dt =
        c.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r;
    if (rank == 2) {
        const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, rows};
        const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)c.block_size};
        r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (rank == 3) {
        const cuuint64_t dims[3] = {64, rows, 2};
        const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, 128};
        const cuuint32_t box[3] = {64, (cuuint32_t)c.block_size, 2};
        r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint32_t estr4[4] = {1, 1, 1, 1};
        const cuuint64_t dims[4] = {64, 8, 2, rows / 8};  // block_size is a multiple of 8
        const cuuint64_t strides[3] = {(cuuint64_t)kHeadDim * 2, 128, (cuuint64_t)kHeadDim * 2 * 8};
        const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)c.block_size / 8};
        r = fn(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr4, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_INVALID_ARG;
}

// Workspace of a split-K call: first the arrival counters of the in-kernel
// merge (one per sequence and query head, an upper bound on the head groups),
// then the partial outputs [B][Hq][parts][D] and log-sum-exps [B][Hq][parts],
// each region 256-byte aligned.
// Grouped decode adds one group index per sequence after the counters.
struct WorkspaceLayout {
    int64_t ctr_off, group_off, o_off, lse_off, total;
};

static int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

static WorkspaceLayout workspace_layout(int64_t num_seqs, int64_t num_q_heads, int64_t head_dim, int64_t rows,
                                        bool grouped = false) {
    WorkspaceLayout w;
    w.ctr_off = 0;
    w.group_off = round256(num_seqs * num_q_heads * 8);
    w.o_off = w.group_off + (grouped ? round256(num_seqs * 4) : 0);
    w.lse_off = w.o_off + round256(rows * head_dim * 4);
    w.total = w.lse_off + round256(rows * 4);
    return w;
}

// Prefix partitions of grouped decode for the longest shared prefix.
static int64_t prefix_parts_of(int64_t max_prefix_len, int64_t partition = kPrefixPartition) {
    return (max_prefix_len + partition - 1) / partition;
}

// Epoch of a decode call: a process-wide counter, 48 bits, never 0.
static std::atomic<unsigned long long> g_epoch{0};
static unsigned long long next_epoch() {
    for (;;) {
        const unsigned long long e = (g_epoch.fetch_add(1) + 1) & ((1ull << 48) - 1);
        if (e != 0) return e;
    }
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Shape checks common to every call on a cache.
static pkv_status check_cache(const pkv_cache_desc* c) {
    if (!c) return PKV_ERR_INVALID_ARG;
    if (c->num_blocks < 1 || c->num_kv_heads < 1 || c->block_size < 1 || c->head_dim < 1) return PKV_ERR_INVALID_ARG;
    if (c->dtype != PKV_BF16 && c->dtype != PKV_FP16) return PKV_ERR_UNSUPPORTED;
    if ((c->head_dim * 2) % 16 != 0) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// Streaming multiprocessors of the current device (cached per device).
static int sm_count() {
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

// Tokens per split-K partition.  An explicit size is used as given.  The
// automatic choice takes the largest of 512, 1024, 2048, 4096 tokens for which the
// work units (sequence x KV head x head tile x partition, counted at
// max_context_len) still fill the GPU's resident decode CTAs at least twice;
// longer partitions amortise each CTA's start-up, shorter ones balance the
// load.  The workspace is always sized for 512 (the smallest choice).
static int resolve_partition(int32_t partition_size, int64_t rows, int32_t max_context_len) {
    if (partition_size != 0) return partition_size;
    const int64_t slots = (int64_t)(sm_count() > 0 ? sm_count() : 148) * kDecodeCtasPerSm;
    int best = kAutoPartition;
    for (int P = 1024; P <= 4096; P *= 2) {
        const int64_t units = rows * (((int64_t)max_context_len + P - 1) / P);
        if (units >= 2 * slots) best = P;
    }
    return best;
}


// Tokens per prefix partition of grouped decode: the largest of 256, 512,
// 1024 for which the prefix CTAs (group x KV head x row tile x partition,
// counted at max_prefix_len) still fill three quarters of the device's
// resident prefix CTAs (kPrefixCtasPerSm per SM).  Fewer, longer partitions
// leave fewer partials to merge; below that count the launch leaves SMs idle.
static int resolve_prefix_partition(int64_t tiles, int32_t max_prefix_len) {
    const int64_t slots = (int64_t)(sm_count() > 0 ? sm_count() : 148) * kPrefixCtasPerSm;
    int best = kPrefixPartition;
    for (int P = 2 * kPrefixPartition; P <= kPrefixPartitionMax; P *= 2)
        if (4 * tiles * prefix_parts_of(max_prefix_len, P) >= 3 * slots) best = P;
    return best;
}

// How a decode call divides its work (see paged_attention_plan).
struct Plan {
    int kind;        // PKV_PLAN_*
    int partition;   // split-K partition (tokens)
    int max_parts;   // split-K partitions of the longest sequence
};

static Plan make_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t head_tiles, int32_t max_context_len,
                      int32_t partition_size) {
    Plan pl;
    const int64_t groups = (int64_t)num_seqs * num_kv_heads * head_tiles;  // (sequence, head group) rows
    pl.partition = resolve_partition(partition_size, groups, max_context_len);
    pl.max_parts = max_context_len == 0 ? 1 : (max_context_len + pl.partition - 1) / pl.partition;
    if (pl.max_parts <= 1)
        pl.kind = PKV_PLAN_SINGLE;
    else
        pl.kind = pl.max_parts <= kFuseMergeMaxParts ? PKV_PLAN_SPLIT : PKV_PLAN_SPLIT_REDUCE;
    return pl;
}

}  // namespace pkv

using namespace pkv;

// pkv_wait_selftest: one thread waits on phase 0 of a fresh mbarrier that
// expects one arrival nobody makes; the bounded wait runs out after limit_ns
// and the error is recorded the way the copy pipelines record theirs.
__global__ void wait_selftest_kernel(int* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    pdl_wait();
    if (threadIdx.x == 0) {
        const uint32_t b = smem_addr(&bar);
        mbar_init(b, 1);
        fence_barrier_init();
        if (!mbar_wait_for(b, 0, limit_ns)) record_error(err, PKV_DEVERR_TIMEOUT);
    }
}

extern "C" {

const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA call failed";
        case PKV_ERR_DEVICE_METADATA: return "device-side metadata error";
    }
    return "unknown status";
}

int pkv_version(void) { return 100; }

uint64_t pkv_launch_count(void) { return g_launches.load(); }

pkv_status paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
                           void* k_cache, void* v_cache, const pkv_cache_desc* cache, void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    const int row_vecs = cache->head_dim * 2 / 16;
    const int64_t total = num_tokens * cache->num_kv_heads * row_vecs;
    if (total / num_tokens != (int64_t)cache->num_kv_heads * row_vecs || (total + 255) / 256 > INT_MAX)
        return PKV_ERR_INVALID_ARG;
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    AppendParams p;
    p.err = err;
    p.k = static_cast<const uint4*>(k);
    p.v = static_cast<const uint4*>(v);
    p.slot_mapping = slot_mapping;
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.num_tokens = num_tokens;
    p.num_slots = cache->num_blocks * cache->block_size;
    p.num_kv_heads = cache->num_kv_heads;
    p.block_size = cache->block_size;
    p.row_vecs = row_vecs;
    int launches = 0;
    const cudaError_t e = launch_append(p, static_cast<cudaStream_t>(stream), &launches);
    g_launches += launches;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                       int32_t max_context_len, int32_t partition_size) {
    if (num_seqs < 0 || num_q_heads < 1 || head_dim < 1 || max_context_len < 0 || partition_size < 0) return 0;
    const int64_t P = partition_size == 0 ? kAutoPartition : partition_size;  // auto never goes below 512
    const int64_t parts = max_context_len == 0 ? 1 : (max_context_len + P - 1) / P;
    if (parts <= 1) return 0;
    const int64_t rows = (int64_t)num_seqs * num_q_heads * parts;
    const WorkspaceLayout w = workspace_layout(num_seqs, num_q_heads, head_dim, rows);
    return (size_t)w.total;
}

size_t paged_attention_grouped_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                               int32_t max_context_len, int32_t max_prefix_len,
                                               int32_t partition_size) {
    if (num_seqs < 0 || num_q_heads < 1 || head_dim < 1 || max_context_len < 0 || max_prefix_len < 0 ||
        max_prefix_len > max_context_len || partition_size < 0)
        return 0;
    const int64_t P = partition_size == 0 ? kAutoPartition : partition_size;  // auto never goes below 512
    const int64_t parts = prefix_parts_of(max_prefix_len) + (max_context_len == 0 ? 1 : (max_context_len + P - 1) / P);
    const int64_t rows = (int64_t)num_seqs * num_q_heads * parts;
    return (size_t)workspace_layout(num_seqs, num_q_heads, head_dim, rows, true).total;
}

int32_t paged_attention_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t block_size,
                             int32_t max_context_len, int32_t partition_size) {
    if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 ||
        max_context_len < 0 || partition_size < 0 || block_size < 1)
        return -1;
    const int group = num_q_heads / num_kv_heads;
    const int head_tiles = (group + decode_head_tile(group) - 1) / decode_head_tile(group);
    return make_plan(num_seqs, num_kv_heads, head_tiles, max_context_len, partition_size).kind;
}

int32_t paged_attention_partition_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t max_context_len, int32_t partition_size) {
    if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0 ||
        max_context_len < 0 || partition_size < 0)
        return 0;
    const int group = num_q_heads / num_kv_heads;
    const int head_tiles = (group + decode_head_tile(group) - 1) / decode_head_tile(group);
    return resolve_partition(partition_size, (int64_t)num_seqs * num_kv_heads * head_tiles, max_context_len);
}

}  // extern "C"

// Shared-prefix groups of paged_attention_decode_grouped.
struct GroupArgs {
    const int32_t* group_starts;
    int32_t num_groups, max_group_size;
    const int32_t* prefix_lens;
    int32_t max_prefix_len;
};

// paged_attention_decode, optionally with the block write of one new token
// per sequence fused in (k_new != nullptr), or with shared-prefix groups
// (grp != nullptr).
static pkv_status decode_impl(const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                              const void* k_cache, const void* v_cache, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                              int32_t num_q_heads, int32_t max_context_len, float scale, void* out,
                              int32_t out_dtype, const pkv_cache_desc* cache, int32_t partition_size,
                              void* workspace, size_t workspace_bytes, void* stream, const GroupArgs* grp = nullptr) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (cache->head_dim != kHeadDim) return PKV_ERR_UNSUPPORTED;
    if (cache->block_size != 16 && cache->block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_seqs > 65535 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (out_dtype != PKV_FP32 && out_dtype != PKV_BF16 && out_dtype != PKV_FP16) return PKV_ERR_INVALID_ARG;
    if (max_blocks_per_seq < 1 || max_context_len < 0 ||
        (int64_t)max_blocks_per_seq * cache->block_size > INT_MAX ||
        max_context_len > (int64_t)max_blocks_per_seq * cache->block_size)
        return PKV_ERR_INVALID_ARG;
    if (partition_size < 0 || (partition_size > 0 && partition_size % cache->block_size != 0))
        return PKV_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PKV_ERR_INVALID_ARG;
    // tile rows must be addressable by a 32-bit TMA coordinate
    if (cache->num_blocks * cache->num_kv_heads * cache->block_size > INT_MAX) return PKV_ERR_UNSUPPORTED;
    const int group = num_q_heads / cache->num_kv_heads;
    const int head_tiles = (group + decode_head_tile(group) - 1) / decode_head_tile(group);
    if ((int64_t)cache->num_kv_heads * head_tiles > 65535) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID_ARG;
    const bool fused_append = k_new != nullptr;
    if (fused_append && (!v_new || !slot_mapping || !aligned(k_new, 16) || !aligned(v_new, 16) ||
                         !aligned(slot_mapping, 8)))
        return PKV_ERR_INVALID_ARG;

    int members_per_tile = 0, row_tiles = 0, prefix_parts = 0, prefix_partition = kPrefixPartition;
    if (grp) {
        if (group > kPrefixRows) return PKV_ERR_UNSUPPORTED;
        if (grp->num_groups < 0 || grp->num_groups > 65535 || grp->max_prefix_len < 0 ||
            grp->max_prefix_len > max_context_len || (grp->num_groups > 0 && grp->max_group_size < 1))
            return PKV_ERR_INVALID_ARG;
        if (!grp->prefix_lens || !aligned(grp->prefix_lens, 4) ||
            (grp->num_groups > 0 && (!grp->group_starts || !aligned(grp->group_starts, 4))))
            return PKV_ERR_INVALID_ARG;
        members_per_tile = kPrefixRows / group;
        row_tiles = grp->num_groups > 0 ? (grp->max_group_size + members_per_tile - 1) / members_per_tile : 0;
        if ((int64_t)cache->num_kv_heads * row_tiles > 65535) return PKV_ERR_UNSUPPORTED;
        prefix_partition = resolve_prefix_partition(
            (int64_t)grp->num_groups * cache->num_kv_heads * row_tiles, grp->max_prefix_len);
        prefix_parts = (int)prefix_parts_of(grp->max_prefix_len, prefix_partition);
    }
    const size_t need = grp ? paged_attention_grouped_workspace_bytes(num_seqs, num_q_heads, kHeadDim,
                                                                      max_context_len, grp->max_prefix_len,
                                                                      partition_size)
                            : paged_attention_workspace_bytes(num_seqs, num_q_heads, kHeadDim, max_context_len,
                                                              partition_size);
    const bool have_ws = need > 0 && workspace && workspace_bytes >= need && aligned(workspace, 256);
    const Plan pl = make_plan(num_seqs, cache->num_kv_heads, head_tiles, max_context_len, partition_size);
    const int P = pl.partition, max_parts = pl.max_parts + prefix_parts;
    const bool split = grp || pl.kind != PKV_PLAN_SINGLE;
    if (split && !have_ws) return PKV_ERR_WORKSPACE;

    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    // whole tiles: halves back to back (rank 3) for the decode kernel, 8-row
    // groups (rank 4) for the prefix kernel
    CUtensorMap tmk, tmv, tmk4, tmv4;
    st = encode_cache_map(&tmk, k_cache, *cache, 3);
    if (st != PKV_OK) return st;
    st = encode_cache_map(&tmv, v_cache, *cache, 3);
    if (st != PKV_OK) return st;
    if (grp) {
        st = encode_cache_map(&tmk4, k_cache, *cache, 4);
        if (st != PKV_OK) return st;
        st = encode_cache_map(&tmv4, v_cache, *cache, 4);
        if (st != PKV_OK) return st;
    }

    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    if (split) {
        const int64_t rows = (int64_t)num_seqs * num_q_heads * max_parts;
        const WorkspaceLayout w = workspace_layout(num_seqs, num_q_heads, kHeadDim, rows, grp != nullptr);
        char* base = static_cast<char*>(workspace);
        p.merge_ctr = reinterpret_cast<unsigned long long*>(base + w.ctr_off);
        p.part_o = reinterpret_cast<float*>(base + w.o_off);
        p.part_lse = reinterpret_cast<float*>(base + w.lse_off);
        p.fuse_merge = max_parts <= kFuseMergeMaxParts ? 1 : 0;
        p.epoch = next_epoch();
        if (grp) {
            p.seq_group = reinterpret_cast<int*>(base + w.group_off);
            p.prefix_lens = grp->prefix_lens;
            p.group_starts = grp->group_starts;
            p.max_prefix_len = grp->max_prefix_len;
            p.prefix_partition = prefix_partition;
            p.prefix_parts = prefix_parts;
            p.num_groups = grp->num_groups;
            p.members_per_tile = members_per_tile;
            p.row_tiles = row_tiles;
        }
    }
    p.err = err;
    p.num_blocks = cache->num_blocks;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = cache->num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.len_limit = max_context_len;  // already <= max_blocks_per_seq * block_size
    p.partition_size = P;
    p.max_parts = max_parts;
    p.group = group;
    p.head_tiles = head_tiles;
    p.out_dtype = out_dtype;
    p.split = split ? 1 : 0;
    p.block_size = cache->block_size;
    p.parts_in_x = max_parts > 65535 ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    if (fused_append) {
        p.fused_append = 1;
        p.k_new = static_cast<const uint4*>(k_new);
        p.v_new = static_cast<const uint4*>(v_new);
        p.slot_mapping = slot_mapping;
        p.k_cache = static_cast<uint4*>(const_cast<void*>(k_cache));
        p.v_cache = static_cast<uint4*>(const_cast<void*>(v_cache));
    }
    int launches = 0;
    cudaError_t e = cudaSuccess;
    if (grp && prefix_parts > 0 && grp->num_groups > 0) {
        e = launch_group_prefix(p, cache->dtype, cache->block_size, tmk4, tmv4, static_cast<cudaStream_t>(stream),
                                &launches);
        p.early_inputs = 1;  // the prefix kernel releases the decode kernel after its own wait
    }
    if (e == cudaSuccess)
        e = launch_decode(p, cache->dtype, cache->block_size, tmk, tmv, static_cast<cudaStream_t>(stream), &launches);
    g_launches += launches;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Shared by copy_blocks and swap_blocks: whole blocks from a source pool to
// a destination pool (which are the same pool for copy_blocks).
static pkv_status move_blocks(void* const* src_k, void* const* src_v, int64_t src_blocks, void* const* dst_k,
                              void* const* dst_v, int64_t dst_blocks, int32_t num_layers,
                              const int64_t* src_dst_pairs, int32_t num_pairs, const pkv_cache_desc* cache,
                              int err_code, void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_layers < 0 || num_pairs < 0 || src_blocks < 1 || dst_blocks < 1) return PKV_ERR_INVALID_ARG;
    if (num_layers == 0 || num_pairs == 0) return PKV_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !src_dst_pairs || !aligned(src_dst_pairs, 8))
        return PKV_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l)
        if (!src_k[l] || !src_v[l] || !dst_k[l] || !dst_v[l] || !aligned(src_k[l], 16) || !aligned(src_v[l], 16) ||
            !aligned(dst_k[l], 16) || !aligned(dst_v[l], 16))
            return PKV_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)cache->num_kv_heads * cache->block_size * cache->head_dim * 2;
    if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    const int64_t block_vecs = block_bytes / 16;
    if ((block_vecs + 4095) / 4096 > 65535) return PKV_ERR_UNSUPPORTED;
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    int launches = 0;
    cudaError_t e = cudaSuccess;
    for (int l0 = 0; l0 < num_layers && e == cudaSuccess; l0 += kCopyMaxLayers) {
        CopyParams p;
        std::memset(&p, 0, sizeof(p));
        p.err = err;
        p.err_code = err_code;
        p.num_layers = num_layers - l0 < kCopyMaxLayers ? num_layers - l0 : kCopyMaxLayers;
        for (int l = 0; l < p.num_layers; ++l) {
            p.src_k[l] = static_cast<const uint4*>(src_k[l0 + l]);
            p.src_v[l] = static_cast<const uint4*>(src_v[l0 + l]);
            p.dst_k[l] = static_cast<uint4*>(dst_k[l0 + l]);
            p.dst_v[l] = static_cast<uint4*>(dst_v[l0 + l]);
        }
        p.pairs = src_dst_pairs;
        p.src_blocks = src_blocks;
        p.dst_blocks = dst_blocks;
        p.block_vecs = block_vecs;
        p.num_pairs = num_pairs;
        e = launch_copy_blocks(p, static_cast<cudaStream_t>(stream), &launches);
    }
    g_launches += launches;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" {

pkv_status paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len, float scale, void* out, int32_t out_dtype,
                                  const pkv_cache_desc* cache, int32_t partition_size, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    return decode_impl(q, nullptr, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_q_heads, max_context_len, scale, out, out_dtype, cache,
                       partition_size, workspace, workspace_bytes, stream);
}

pkv_status paged_attention_append_decode(const void* q, const void* k_new, const void* v_new,
                                         const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_context_len, float scale, void* out, int32_t out_dtype,
                                         const pkv_cache_desc* cache, int32_t partition_size, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    if (num_seqs > 0 && !k_new) return PKV_ERR_INVALID_ARG;
    return decode_impl(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_q_heads, max_context_len, scale, out, out_dtype, cache,
                       partition_size, workspace, workspace_bytes, stream);
}

pkv_status paged_attention_decode_grouped(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_context_len, const int32_t* group_starts,
                                          int32_t num_groups, int32_t max_group_size, const int32_t* prefix_lens,
                                          int32_t max_prefix_len, float scale, void* out, int32_t out_dtype,
                                          const pkv_cache_desc* cache, int32_t partition_size, void* workspace,
                                          size_t workspace_bytes, void* stream) {
    const GroupArgs grp{group_starts, num_groups, max_group_size, prefix_lens, max_prefix_len};
    return decode_impl(q, nullptr, nullptr, nullptr, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_q_heads, max_context_len, scale, out, out_dtype, cache,
                       partition_size, workspace, workspace_bytes, stream, &grp);
}

pkv_status paged_attention_append_decode_grouped(const void* q, const void* k_new, const void* v_new,
                                                 const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                 const int32_t* context_lens, int32_t num_seqs,
                                                 int32_t num_q_heads, int32_t max_context_len,
                                                 const int32_t* group_starts, int32_t num_groups,
                                                 int32_t max_group_size, const int32_t* prefix_lens,
                                                 int32_t max_prefix_len, float scale, void* out, int32_t out_dtype,
                                                 const pkv_cache_desc* cache, int32_t partition_size,
                                                 void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs > 0 && !k_new) return PKV_ERR_INVALID_ARG;
    const GroupArgs grp{group_starts, num_groups, max_group_size, prefix_lens, max_prefix_len};
    return decode_impl(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_q_heads, max_context_len, scale, out, out_dtype, cache,
                       partition_size, workspace, workspace_bytes, stream, &grp);
}

pkv_status copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                       const int64_t* src_dst_pairs, int32_t num_pairs, const pkv_cache_desc* cache,
                       void* stream) {
    if (!cache) return PKV_ERR_INVALID_ARG;
    return move_blocks(k_caches, v_caches, cache->num_blocks, k_caches, v_caches, cache->num_blocks, num_layers,
                       src_dst_pairs, num_pairs, cache, PKV_DEVERR_COPY_ID, stream);
}

pkv_status swap_blocks(void* const* src_k_caches, void* const* src_v_caches, int64_t src_num_blocks,
                       void* const* dst_k_caches, void* const* dst_v_caches, int64_t dst_num_blocks,
                       int32_t num_layers, const int64_t* src_dst_pairs, int32_t num_pairs,
                       const pkv_cache_desc* cache, void* stream) {
    return move_blocks(src_k_caches, src_v_caches, src_num_blocks, dst_k_caches, dst_v_caches, dst_num_blocks,
                       num_layers, src_dst_pairs, num_pairs, cache, PKV_DEVERR_COPY_ID, stream);
}

pkv_status compact_tokens(const int64_t* src_slots, const int64_t* dst_slots, int64_t num_tokens, void* k_cache,
                          void* v_cache, const pkv_cache_desc* cache, void* stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!src_slots || !dst_slots || !k_cache || !v_cache || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(src_slots, 8) || !aligned(dst_slots, 8))
        return PKV_ERR_INVALID_ARG;
    const int row_vecs = cache->head_dim * 2 / 16;
    const int64_t total = num_tokens * cache->num_kv_heads * row_vecs;
    if (total / num_tokens != (int64_t)cache->num_kv_heads * row_vecs || (total + 255) / 256 > INT_MAX)
        return PKV_ERR_INVALID_ARG;
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    CompactParams p;
    p.err = err;
    p.src_slots = src_slots;
    p.dst_slots = dst_slots;
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.num_tokens = num_tokens;
    p.num_slots = cache->num_blocks * cache->block_size;
    p.num_kv_heads = cache->num_kv_heads;
    p.block_size = cache->block_size;
    p.row_vecs = row_vecs;
    int launches = 0;
    const cudaError_t e = launch_compact(p, static_cast<cudaStream_t>(stream), &launches);
    g_launches += launches;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_wait_selftest(int32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 2000000) return PKV_ERR_INVALID_ARG;
    int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    const cudaError_t e = launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, static_cast<cudaStream_t>(stream), err,
                                     (uint64_t)limit_us * 1000ull);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    ++g_launches;
    return PKV_OK;
}

pkv_status pkv_check_device_error(void* stream, int32_t* first_error_code) {
    if (first_error_code) *first_error_code = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pkv_error, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    if (v == 0) return PKV_OK;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_pkv_error, &zero, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    if (first_error_code) *first_error_code = v;
    return PKV_ERR_DEVICE_METADATA;
}

}  // extern "C"
