// group_prefix.cu -- the shared-prefix half of grouped decode, on the
// 5th-generation tensor cores (tcgen05, operands and accumulators in tensor
// memory).
//
// Sequences forked from one prompt (parallel samples, beams, a common
// system prompt) hold the prompt's K/V in the same physical blocks: the
// block table of every member maps the prompt's logical blocks to the same
// ids, with a reference count per block (tonho.wtf "vllm", "como funciona";
// techtrendfeed "KV Cache Administration", "How PagedAttention Works", step
// 4; aitalk.it "PagedAttention e RadixAttention" on reusing a common
// prefix).  Plain paged decode reads those blocks once per member.  Here
// one CTA takes a partition of the shared blocks for one KV head and
// attends it for the query heads of up to 64 / G members at once, so a
// shared block leaves HBM once per (group, KV head).  Each member's own
// tokens are attended by the decode kernel (decode.cu), and the two halves
// are combined by the same log-sum-exp merge as split-K partitions: the
// softmax over a union of token sets is the weighted merge of the softmaxes
// over its parts.
//
// With up to 64 query rows per shared tile this is a dense contraction, so
// both products run as tcgen05.mma.kind::f16 with fp32 accumulators in
// tensor memory (TMEM), M = 128 rows, 128 tokens per chunk:
//   S = Q K^T   A = Q from TMEM [128 rows x 128 dims], B = K from shared
//               memory [128 tokens x 128 dims], K-major, 128-byte swizzle,
//               N = 128                              -> TMEM columns [0, 128) or [128, 256)
//   O += P V    A = P from TMEM [128 rows x 128 tokens], B = V from shared
//               memory read dims-major (MN-major), 16 tokens per product
//                                                    -> TMEM columns [256, 384)
// The tile's 64 query rows are held twice as Q (TMEM lanes r and r + 64), so
// lanes r and r + 64 hold the same row of S.  Eight softmax warps work on
// the 128 lanes, two per lane (warps w and w + 4 may both access lanes
// 32 (w % 4) .. +31): the four threads of a row take 32 tokens of each chunk
// apiece and exchange their maxima.  P keeps ~16 significant bits as a
// 16-bit high part plus a 16-bit residual: lane r of P holds the high part of
// query row r and lane r + 64 its residual, so one product accumulates both,
// in lanes r and r + 64 of O, which the epilogue adds.  Each thread packs the
// high and residual parts of its own tokens; it swaps the half that belongs
// in the other lane with its partner there through shared memory and writes
// P over the S columns it was computed from.  With Q and P in TMEM the
// products read only K and V from shared memory, whose bandwidth (128 bytes
// per cycle) otherwise sets the pace of a product with N <= 128.
//
// Shared-memory layout of a chunk: each (block, KV head) tile of K or V
// lands in one TMA copy as 8-token groups of 2 KiB (the two 64-dim halves of
// the 8 rows back to back, 128-byte swizzle), tile after tile, so that the
// 8-token groups of the whole chunk sit 2 KiB apart across block boundaries
// and one descriptor spans 128 tokens.
//
// The partition streams through in chunks of 128 tokens, pipelined across
// three roles that hand off on mbarriers:
//   TMA warp: the chunk's tiles of K and V into a 3-stage ring (one copy per
//     tile and tensor, issued from separate lanes);
//   MMA warp (one thread): S(c+1) = Q K(c+1)^T into the other S buffer while
//     the softmax works on chunk c, then O += P(c) V(c) once P(c) is in
//     TMEM; each product's completion is signalled by tcgen05.commit;
//   softmax warps 0-7 (TMEM lanes 0-127, two warps per lane quarter): S(c)
//     from TMEM, the online softmax in the log2 domain with the running max
//     raised lazily (as in the decode warp core; O and l are rescaled when it
//     is), P(c) into TMEM, and at the end the normalised output and
//     log-sum-exp, written a row at a time through shared memory.
// Every wait is bounded; a wait that runs out records PKV_DEVERR_TIMEOUT.
// The softmax warps then stop together at their next barrier and the other
// roles at their next wait; the copies and products already issued are
// waited for (bounded) before the CTA frees its tensor memory or exits.
#include "decode_common.cuh"

namespace pkv {

constexpr int kSoftWarps = 8;             // two per TMEM lane quarter: warps w and w + 4 share lanes 32 (w % 4) ..
constexpr int kTmaWarp = kSoftWarps;      // K/V loads
constexpr int kMmaWarp = kSoftWarps + 1;  // tensor-core products (lane 0)
constexpr int kPrefixThreads = (kSoftWarps + 2) * 32;
constexpr int kChunk = 128;               // tokens per pipeline step
constexpr int kUmmaM = 128;               // M of both products
constexpr int kRing = 3;                  // K/V chunks in flight
constexpr uint32_t kTmemCols = 512;       // S: [0, 128), [128, 256); O: [256, 384); Q: [384, 448)
constexpr uint32_t kOCol = 256;
constexpr uint32_t kQCol = 384;

// ---- tcgen05 wrappers (PTX ISA: tcgen05 instructions, shared memory and
// instruction descriptors)

// Shared-memory matrix descriptor for a 128-byte-swizzled operand: start
// address, leading- and stride-dimension byte offsets (all in 16-byte
// units), the fixed 0b001 at bits 46-48, swizzle mode 2 (128 B) at 61-63.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulate, A and B both bf16 or
// both fp16, operand majorness, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__device__ __forceinline__ uint32_t umma_idesc(bool bf16, int M, int N, bool a_mn_major, bool b_mn_major) {
    const uint32_t t = bf16 ? 1u : 0u;
    return (1u << 4) | (t << 7) | (t << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) = A B^T (+ D when accumulate), A in TMEM (row i in lane i, two
// 16-bit elements of K per 32-bit column), B in shared memory; one thread.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp w reads
// lanes 32w .. 32w+31); every lane of the warp executes it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The reverse: 32 columns of this thread's lane from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
    tmem_st32(taddr, r);
}

// Barrier over the softmax warps only (named barrier 1).
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory"); }

// Barrier over the softmax warps and the MMA warp, not the TMA warp (named
// barrier 2).
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 2, %0;" ::"n"((kSoftWarps + 1) * 32) : "memory");
}

struct PrefixSmem {
    static constexpr int kStage = kChunk * kHeadDim * 2;  // a chunk of K or V: 128 tokens x 128 dims, 32 KiB
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + kRing * kStage;
    // the pair exchange of P: [4 chunks of 16 bytes][256 softmax threads]
    static constexpr int kXOff = kVOff + kRing * kStage;
    static constexpr int kXBytes = 4 * kSoftWarps * 32 * 16;
    static constexpr int kBarOff = kXOff + kXBytes;
    // kvfull[kRing], kvempty[kRing], sfull[2], pfull[2], pvdone
    static constexpr int kNumBars = 2 * kRing + 5;
    static constexpr int kSlotOff = kBarOff + kNumBars * 8;
    // per member of the tile: sequence, prefix tokens (0 when it takes no
    // part), partitions in all, whether the prefix side merges; per (member,
    // head tile): merge verdict
    static constexpr int kMemOff = kSlotOff + 16;
    static constexpr int kMemBytes = kPrefixRows * 4 * 4 + kPrefixRows * 4 * 4;
    // [2][256] chunk maxima, [256] row sums (one per softmax thread)
    static constexpr int kXchOff = kMemOff + kMemBytes;
    static constexpr int kFlagOff = kXchOff + 3 * kSoftWarps * 32 * 4;
    static constexpr int kTotal = kFlagOff + 32;
    static constexpr int kDynamic = kTotal + 1024;  // slack to align the base to 1024 B
    // epilogue: the residual lanes' O rows, [64][kRedStride] floats over the K/V ring
    static constexpr int kRedOff = kKOff;
    static_assert(kPrefixRows * kRedStride * 4 + kPrefixRows * 12 <= 2 * kRing * kStage, "O rows fit the ring");
    static_assert(kDynamic <= 227 * 1024, "shared memory of one CTA");
};

template <bool kBF16, int BS>
__global__ void __launch_bounds__(kPrefixThreads, 1)
    group_prefix_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const DecodeParams p) {
    using S = PrefixSmem;
    constexpr int D = kHeadDim;
    constexpr int kBlocksPerChunk = kChunk / BS;
    static_assert(kChunk % BS == 0 && BS % 8 == 0 && kBlocksPerChunk <= 16, "whole blocks per chunk, one copy per lane");
    static_assert(2 * kPrefixRows == kUmmaM && kSoftWarps * 32 == 2 * kUmmaM,
                  "each row twice, two softmax threads per TMEM lane");
    static_assert(kPrefixPartitionMax / 16 <= 64, "a partition's block ids fit two registers per lane");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_sa = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_sa + 1023u) & ~1023u) - raw_sa);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int part = blockIdx.x;
    const int kvh = blockIdx.y / p.row_tiles, rt = blockIdx.y - kvh * p.row_tiles;
    const int g = blockIdx.z;
    const int G = p.group;

    if (tid == 32 * kTmaWarp) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    // Launched with programmatic stream serialisation.  Wait for the kernels
    // before the call, then let the decode kernel start: it reads the call's
    // inputs at once and waits for this kernel only before reading what this
    // kernel writes.
    pdl_wait();
    pdl_launch_dependents();

    int* mem_s = reinterpret_cast<int*>(smem + S::kMemOff);   // [64]
    int* mem_lim = mem_s + kPrefixRows;                       // [64]
    int* mem_np = mem_lim + kPrefixRows;                      // [64] partitions in all
    int* mem_arrive = mem_np + kPrefixRows;                   // [64] 1: the prefix side merges
    int* verdict = mem_arrive + kPrefixRows;                  // [64 * 4]
    // [0]: bad block id (bit 0) / a wait ran out (bit 1); [1]: tile token
    // end; [2], [4]: a softmax warp's wait ran out, read by every softmax
    // thread after the barrier that follows the wait ([2]: S, [4]: the
    // previous product); [3]: some member's partials are merged on this side
    int* flags = reinterpret_cast<int*>(smem + S::kFlagOff);
    float* xch = reinterpret_cast<float*>(smem + S::kXchOff);
    const uint32_t bar0 = smem_addr(smem + S::kBarOff);
    const uint32_t kvfull0 = bar0, kvempty0 = bar0 + 8 * kRing, sfull0 = bar0 + 16 * kRing, pfull0 = sfull0 + 16,
                   pvdone = pfull0 + 16;
    const uint32_t slot = smem_addr(smem + S::kSlotOff);

    const int gs0 = p.group_starts[g], gs1 = p.group_starts[g + 1];
    const bool bad_group = gs0 < 0 || gs1 < gs0 || gs1 > p.num_seqs;
    const int m0 = rt * p.members_per_tile;
    const int nmem = bad_group ? 0 : max(0, min(p.members_per_tile, gs1 - gs0 - m0));
    const int tok0 = part * p.prefix_partition;

    if (tid == 0) {
        // a range out of order or out of bounds is skipped; members past the
        // row tiles' capacity are not attended (the decode kernel zeroes them)
        if (part == 0 && kvh == 0 && rt == 0 &&
            (bad_group || gs1 - gs0 > p.row_tiles * p.members_per_tile))
            record_error(p.err, PKV_DEVERR_GROUP);
        for (int i = 0; i < 8; ++i) flags[i] = 0;
        for (int i = 0; i < kRing; ++i) {
            mbar_init(kvfull0 + 8 * i, 1);
            mbar_init(kvempty0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(sfull0 + 8 * i, 1);
            mbar_init(pfull0 + 8 * i, kSoftWarps);
        }
        mbar_init(pvdone, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // The TMA warp loads the block ids of the partition from the group's
    // first member's table (block j in ids[j / 32] of lane j % 32) while the
    // member metadata below is read; ids past the tile's token end (known
    // after that) are not used.
    int ids[2] = {0, 0};
    if (warp == kTmaWarp && nmem > 0) {
        const int32_t* table = p.block_tables + (int64_t)gs0 * p.max_blocks_per_seq + tok0 / BS;
        const int jmax = min(p.prefix_partition / BS, p.max_blocks_per_seq - tok0 / BS);  // within the table row
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int j = 32 * k + lane;
            if (j < jmax) ids[k] = __ldg(table + j);
        }
    }
    // Member metadata.  The first CTA of each row tile also records each
    // member's group (the decode kernel's hint, see group_verified).
    for (int i = tid; i < nmem; i += blockDim.x) {
        const int s = gs0 + m0 + i;
        const SeqSpan sp = seq_span(p, s, BS);
        if (part == 0 && kvh == 0) p.seq_group[s] = g;
        mem_s[i] = s;
        mem_lim[i] = sp.err ? 0 : sp.plen;  // bad metadata: the decode kernel zeroes the output
        mem_np[i] = sp.npre + sp.nsuf;
        // with no own partition, the prefix partitions merge among themselves
        // (with one, the decode kernel folds them in; with more, it merges)
        mem_arrive[i] = sp.nsuf == 0 ? 1 : 0;
        if (!sp.err && sp.plen > tok0) atomicMax(flags + 1, min(sp.plen, tok0 + p.prefix_partition));
        if (sp.nsuf == 0 && sp.npre > 1 && sp.plen > tok0) flags[3] = 1;  // some row merges here
    }
    __syncthreads();
    const int tok1 = flags[1];
    if (tok1 <= tok0) return;  // no member's prefix reaches this partition
    const int ntok = tok1 - tok0;  // whole blocks (prefix lengths are)
    const int nchunks = (ntok + kChunk - 1) / kChunk;
    const int rows = nmem * G;  // <= 64

    // ---- TMEM (MMA warp) and Q (softmax warps: this lane's row, zeros past
    // the tile's rows, into TMEM columns [kQCol, kQCol + 64)).  The TMA warp
    // needs neither and starts its copies at once.
    if (warp == kMmaWarp) tmem_alloc(slot, kTmemCols);
    // Softmax thread roles: warp w works on TMEM lanes 32 (w % 4) .. +31 (lane
    // L = 32 (w % 4) + lane); sub = w / 4 splits each lane's work in two.
    const int lane_q = 32 * (warp & 3) + lane;  // TMEM lane
    const int sub = (warp >> 2) & 1;
    uint32_t qa[32];
    if (warp < kSoftWarps) {
        // dims 64 sub .. 64 sub + 63 of row lane_q % 64
        const int r = lane_q & (kPrefixRows - 1);
        const uint4* src = nullptr;
        if (r < rows) {
            const int mi = r / G;
            src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                 ((int64_t)mem_s[mi] * p.num_q_heads + kvh * G + r - mi * G) * D) +
                  8 * sub;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 a = src ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
            qa[4 * k] = a.x, qa[4 * k + 1] = a.y, qa[4 * k + 2] = a.z, qa[4 * k + 3] = a.w;
        }
    }
    uint32_t tmem = 0;
    if (warp != kTmaWarp) {
        tc_fence_before();
        compute_sync();  // the TMEM address is in shared memory
        tc_fence_after();
        tmem = *reinterpret_cast<volatile uint32_t*>(smem + S::kSlotOff);
        if (warp < kSoftWarps) {
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
            tmem_st32(lane_addr + kQCol + 32 * sub, qa);  // two dims per column
        }
        tc_fence_before();
        compute_sync();  // Q is in TMEM
        tc_fence_after();
    }

    float m_run = -INFINITY;  // softmax threads: running max of the row (raised lazily)

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ K/V loads
        const uint64_t policy = l2_policy_evict_first();
        const int nblk = ntok / BS;  // <= kPrefixPartitionMax / 16 = 64
        bool bad = false;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int j = 32 * k + lane;
            if (j >= nblk) {
                ids[k] = 0;
            } else if (ids[k] < 0 || (int64_t)ids[k] >= p.num_blocks) {
                bad = true;
                ids[k] = 0;  // keep the shape; the outputs are zeroed later
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) {
            atomicOr(flags, 1);
            record_error(p.err, PKV_DEVERR_BLOCK_ID);
        }
        int issued = 0;
        for (int c = 0; c < nchunks; ++c) {
            const int st = c % kRing;
            const int b0 = c * kBlocksPerChunk, nb = min(kBlocksPerChunk, nblk - b0);
            bool ok = true;
            if (lane == 0 && c >= kRing) ok = mbar_wait(kvempty0 + 8 * st, ((c / kRing) - 1) & 1);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                if (lane == 0) {
                    atomicOr(flags, 2);
                    record_error(p.err, PKV_DEVERR_TIMEOUT);
                }
                break;
            }
            const uint32_t fb = kvfull0 + 8 * st;
            if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)nb * BS * D * 2 * 2);
            __syncwarp();
            // lane b: block b's K tile; lane 16 + b: its V tile.  A tile lands
            // as BS / 8 groups of 8 tokens x both dims halves (2 KiB each),
            // tile after tile, so the chunk's 8-token groups are 2 KiB apart.
            const int b = lane & 15;
            const int j = (b0 + b) & 63;  // in range whenever b < nb
            const int lo = __shfl_sync(0xffffffffu, ids[0], j & 31), hi = __shfl_sync(0xffffffffu, ids[1], j & 31);
            const int pid = j < 32 ? lo : hi;
            if (b < nb) {
                const int grp = (pid * p.num_kv_heads + kvh) * (BS / 8);  // first 8-row group of the tile
                const uint32_t dst = smem_addr(smem + (lane < 16 ? S::kKOff : S::kVOff) + st * S::kStage) +
                                     b * BS * D * 2;
                tma_load_4d(dst, lane < 16 ? &tmk : &tmv, fb, 0, 0, 0, grp, policy);
            }
            ++issued;
        }
        // every copy issued has landed before the ring is reused or freed
        // (already true when the products consumed them; bounded otherwise)
        if (lane == 0)
            for (int st = 0; st < kRing && st < issued; ++st)
                mbar_wait(kvfull0 + 8 * st, ((st + kRing * ((issued - 1 - st) / kRing)) / kRing) & 1);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ products
        if (lane == 0) {
            const uint32_t id_o = umma_idesc(kBF16, kUmmaM, D, false, true);
            uint32_t last_bar = 0, last_par = 0;  // the latest commit and its phase parity
            bool ok = true;
            for (int c = -1; c < nchunks && ok; ++c) {
                // S(c+1) = Q K(c+1)^T into S buffer (c+1) & 1, ahead of the
                // softmax.  That buffer last held P(c-1), which PV(c-1),
                // issued before this product, has read (the tensor core runs
                // one thread's products in issue order).
                const int cs = c + 1;
                if (cs < nchunks) {
                    const int st = cs % kRing, sb = cs & 1;
                    ok = mbar_wait(kvfull0 + 8 * st, (cs / kRing) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kb = smem_addr(smem + S::kKOff + st * S::kStage);
                    const int nt = min(kChunk, ntok - cs * kChunk);  // a multiple of 16
                    const uint32_t id_s = umma_idesc(kBF16, kUmmaM, nt, false, false);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        // dims 16 ks .. 16 ks + 15: half ks / 4 of each 8-token group
                        const uint32_t b = kb + (ks >> 2) * 1024 + (ks & 3) * 32;
                        umma_f16_ts(tmem + sb * kChunk, tmem + kQCol + 8 * ks, umma_desc_sw128(b, 16, 2048), id_s,
                                    ks > 0);
                    }
                    umma_commit(sfull0 + 8 * sb);
                    last_bar = sfull0 + 8 * sb;
                    last_par = (cs >> 1) & 1;
                }
                if (c < 0) continue;
                // O += P(c) V(c): lanes 0-63 the high part, lanes 64-127 the residual
                const int sb = c & 1;
                ok = mbar_wait(pfull0 + 8 * sb, (c >> 1) & 1);
                if (!ok) break;
                tc_fence_after();
                const int st = c % kRing;
                const uint32_t vb = smem_addr(smem + S::kVOff + st * S::kStage);
                const int nk = min(kChunk, ntok - c * kChunk) / 16;
                // 16 tokens = two 8-token groups (4 KiB); the dims halves of a
                // group are 1 KiB apart, the groups 2 KiB
                for (int ks = 0; ks < nk; ++ks)
                    umma_f16_ts(tmem + kOCol, tmem + sb * kChunk + 8 * ks, umma_desc_sw128(vb + ks * 4096, 1024, 2048),
                                id_o, c > 0 || ks > 0);
                umma_commit(kvempty0 + 8 * st);
                umma_commit(pvdone);
                last_bar = pvdone;
                last_par = c & 1;
            }
            if (!ok) {
                atomicOr(flags, 2);
                record_error(p.err, PKV_DEVERR_TIMEOUT);
            }
            // every product issued has completed before TMEM is read or freed
            if (last_bar) mbar_wait(last_bar, last_par);
        }
    } else {
        // ------------------------------------------------------------ softmax
        // Row r = L % 64 is held by lanes r and r + 64 (half = L / 64); the
        // four threads (half, sub) of the row take chunk tokens
        // 64 half + 32 sub .. +31 each.
        const int r = lane_q & (kPrefixRows - 1);
        const int half = lane_q >> 6;
        const int tq = 64 * half + 32 * sub;  // first chunk token of this thread
        const int lim = r < rows ? min(ntok, mem_lim[r / G] - tok0) : 0;  // tokens row r attends (<= 0: none)
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const float sl2 = p.scale_log2;
        uint4* xbuf = reinterpret_cast<uint4*>(smem + S::kXOff);  // [4][256]
        const int partner = tid ^ 64;                             // lane L ^ 64, same sub
        float l = 0.f;  // this thread's share of the row sum
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const int sb = c & 1;
            float v[32];
            ok = __all_sync(0xffffffffu, mbar_wait(sfull0 + 8 * sb, (c >> 1) & 1));
            if (ok) {
                tc_fence_after();
                tmem_ld32(lane_addr + sb * kChunk + tq, v);
            } else if (lane == 0) {
                flags[2] = 1;
            }
            const int t0 = c * kChunk + tq;  // partition token of v[0]
            float mx = -INFINITY;
            if (ok && t0 + 32 <= lim) {  // every token valid (the common case)
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] *= sl2;
                    mx = fmaxf(mx, v[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] = ok && t0 + j < lim ? v[j] * sl2 : -INFINITY;
                    mx = fmaxf(mx, v[j]);
                }
            }
            float* xm = xch + sb * (kSoftWarps * 32);
            xm[tid] = mx;
            softmax_sync();
            if (flags[2]) {  // every softmax thread sees the same verdict here
                ok = false;
                break;
            }
            // the row's four threads: tid, tid ^ 64 (other half), tid ^ 128
            // (other sub), tid ^ 192
            mx = fmaxf(fmaxf(mx, xm[tid ^ 64]), fmaxf(xm[tid ^ 128], xm[tid ^ 192]));
            // raise m only when a score exceeds it by more than kLazyMargin;
            // the row's threads take the same decision
            const bool raise = mx > m_run + kLazyMargin;
            float alpha = 1.f;
            if (raise) {
                alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - mx);
                m_run = mx;
            }
            const float ms = m_run == -INFINITY ? 0.f : m_run;
            l *= alpha;
            // this thread's 32 tokens as 16 columns of high parts and 16 of
            // residuals; it keeps the ones of its own lane (lane r: high,
            // lane r + 64: residual) and hands the others to its partner on
            // the other lane
            uint32_t keep[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t send[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = 4 * q + i;
                    const float p0 = exp2f(v[2 * e] - ms), p1 = exp2f(v[2 * e + 1] - ms);
                    l += p0 + p1;
                    float r0, r1;
                    const uint32_t hw = pack2<kBF16>(p0, p1, r0, r1);
                    const uint32_t lw = pack2<kBF16>(p0 - r0, p1 - r1);
                    keep[e] = half ? lw : hw;
                    send[i] = half ? hw : lw;
                }
                xbuf[q * (kSoftWarps * 32) + tid] = make_uint4(send[0], send[1], send[2], send[3]);
            }
            // O is rescaled once the previous chunk's product is in it
            const bool rescale = c > 0 && __any_sync(0xffffffffu, alpha != 1.f);
            if (rescale && !__all_sync(0xffffffffu, mbar_wait(pvdone, (c - 1) & 1)) && lane == 0) flags[4] = 1;
            softmax_sync();
            if (flags[4]) {  // as flags[2]: written only before this barrier
                ok = false;
                break;
            }
            uint32_t recv[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 x = xbuf[q * (kSoftWarps * 32) + partner];
                recv[4 * q] = x.x, recv[4 * q + 1] = x.y, recv[4 * q + 2] = x.z, recv[4 * q + 3] = x.w;
            }
            tc_fence_after();
            if (rescale) {
                // columns 64 sub .. +63 of this lane's row of O (the high or
                // the residual product)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float o[32];
                    const uint32_t oa = lane_addr + kOCol + 64 * sub + 32 * q;
                    tmem_ld32(oa, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= alpha;
                    tmem_st32(oa, o);
                }
            }
            // P over this lane's S columns (two tokens per column): this
            // thread's tokens and, at the same columns of the other half, the
            // partner's
            tmem_st16(lane_addr + sb * kChunk + tq / 2, keep);
            tmem_st16(lane_addr + sb * kChunk + (tq ^ 64) / 2, recv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull0 + 8 * sb);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(pvdone, (nchunks - 1) & 1));
        tc_fence_after();
        if (!ok && lane == 0) {
            atomicOr(flags, 2);
            record_error(p.err, PKV_DEVERR_TIMEOUT);
        }
        xch[2 * (kSoftWarps * 32) + tid] = l;  // the row sum's four shares, combined below
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const int fl = flags[0];
    // Each row's normalised output (high + residual product) and
    // log-sum-exp.  The residual lanes (r + 64) put their O columns in shared
    // memory (the ring is idle now); the high lanes (r) add their own, scale
    // the row in place and write its log-sum-exp; then every thread copies
    // rows out, a row's 512 bytes by 32 consecutive threads.  TMEM loads are
    // warp-collective, so every lane runs them.
    float* red = reinterpret_cast<float*>(smem + S::kRedOff);  // [64 rows][kRedStride]
    // per row: where it goes (a partial's row, or null) and whether it is the
    // output itself (a member whose context is all prefix, in one partition)
    float** rowdst = reinterpret_cast<float**>(red + kPrefixRows * kRedStride);  // [64]
    int* rowout = reinterpret_cast<int*>(rowdst + kPrefixRows);                  // [64]
    if (warp < kSoftWarps) {
        const int er = lane_q & (kPrefixRows - 1), ehalf = lane_q >> 6;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        float o[64];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float v[32];
            if (!(fl & 2)) {
                tmem_ld32(lane_addr + kOCol + 64 * sub + 32 * q, v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) o[32 * q + j] = v[j];
        }
        float* row = red + er * kRedStride + 64 * sub;
        if (ehalf) {
#pragma unroll
            for (int j = 0; j < 64; j += 4)
                *reinterpret_cast<float4*>(row + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
        }
        softmax_sync();
        if (!ehalf) {
            const float* ls = xch + 2 * (kSoftWarps * 32);
            const float lsum = (ls[tid] + ls[tid ^ 64]) + (ls[tid ^ 128] + ls[tid ^ 192]);
            const float inv = fl != 0 || !(lsum > 0.f) ? 0.f : 1.f / lsum;  // bad metadata: zeros
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                const float4 b4 = *reinterpret_cast<const float4*>(row + j);
                *reinterpret_cast<float4*>(row + j) = make_float4((o[j] + b4.x) * inv, (o[j + 1] + b4.y) * inv,
                                                                  (o[j + 2] + b4.z) * inv, (o[j + 3] + b4.w) * inv);
            }
            if (sub == 0) {
                const int mi = er / G;
                const bool has = er < rows && tok0 < mem_lim[mi];  // the row's member has prefix tokens here
                const bool partial = has && mem_np[mi] > 1;
                const int64_t idx = ((int64_t)mem_s[mi] * p.num_q_heads + kvh * G + er - mi * G) * p.max_parts + part;
                if (partial) p.part_lse[idx] = fl != 0 ? INFINITY : m_run + log2f(lsum);
                rowdst[er] = partial ? p.part_o + idx * D : nullptr;
                rowout[er] = has && !partial;
            }
        }
    }
    __syncthreads();
    // Rows out, a row's 512 bytes by 32 consecutive threads; every shared
    // load of a thread is issued before its stores.
    constexpr int kOutIters = (kPrefixRows * (D / 4) + kPrefixThreads - 1) / kPrefixThreads;
#pragma unroll
    for (int k = 0; k < kOutIters; ++k) {
        const int i = tid + k * kPrefixThreads, er = i / (D / 4), c4 = i % (D / 4);
        if (er < rows) {
            float* dst = rowdst[er];
            if (dst) *reinterpret_cast<float4*>(dst + 4 * c4) = *reinterpret_cast<const float4*>(red + er * kRedStride + 4 * c4);
        }
    }
    // members whose whole context is prefix, in one partition: the output itself
    for (int i = tid; i < rows * (D / 4); i += blockDim.x) {
        const int er = i / (D / 4), c4 = i % (D / 4);
        if (!rowout[er]) continue;
        const int mi = er / G, s = mem_s[mi], h = kvh * G + er - mi * G;
        const float4 v = *reinterpret_cast<const float4*>(red + er * kRedStride + 4 * c4);
        store_out(p, s, h, 4 * c4, v.x);
        store_out(p, s, h, 4 * c4 + 1, v.y);
        store_out(p, s, h, 4 * c4 + 2, v.z);
        store_out(p, s, h, 4 * c4 + 3, v.w);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);

    if (p.fuse_merge && flags[3]) {
        // One arrival per (member, head tile of the decode kernel) that takes
        // a partial from this partition; the last arrival merges the row.
        // (Members with partitions of their own are merged by the decode
        // kernel, which folds these partials in or counts them.)
        // The partials every thread wrote before the barrier are released by
        // the arriving thread's fence; an arrival that is last acquires the
        // other partitions' before the barrier that starts the merges.
        const int units = nmem * p.head_tiles;
        __syncthreads();
        for (int u = tid; u < units; u += blockDim.x) {
            const int mi = u / p.head_tiles, ht = u - mi * p.head_tiles;
            bool last = false;
            if (tok0 < mem_lim[mi] && mem_np[mi] > 1 && mem_arrive[mi]) {
                const int64_t c = (int64_t)mem_s[mi] * p.num_kv_heads * p.head_tiles + kvh * p.head_tiles + ht;
                fence_acq_rel_gpu();
                last = arrive_last(p.merge_ctr + c, p.epoch, mem_np[mi]);
                if (last) fence_acq_rel_gpu();
            }
            verdict[u] = last ? 1 : 0;
        }
        __syncthreads();
        const int HT = decode_head_tile(G);
        for (int u = 0; u < units; ++u) {
            if (!verdict[u]) continue;
            const int mi = u / p.head_tiles, ht = u - mi * p.head_tiles;
            merge_row_partials(p, mem_s[mi], kvh * G + ht * HT, min(HT, G - ht * HT), mem_np[mi],
                               reinterpret_cast<float*>(smem));  // the ring's start: free now
            __syncthreads();  // the scratch is reused by the next merge
        }
    }
}

template <bool kBF16, int BS>
static cudaError_t launch_prefix_t(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                   cudaStream_t stream, int* launches) {
    using S = PrefixSmem;
    auto kern = group_prefix_kernel<kBF16, BS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kDynamic);
    if (e != cudaSuccess) return e;
    const dim3 grid(p.prefix_parts, p.num_kv_heads * p.row_tiles, p.num_groups);
    e = launch_pdl(kern, grid, dim3(kPrefixThreads), S::kDynamic, stream, tmk, tmv, p);
    if (e == cudaSuccess) ++*launches;
    return e;
}

cudaError_t launch_group_prefix(const DecodeParams& p, int dtype, int block_size, const CUtensorMap& tmk,
                                const CUtensorMap& tmv, cudaStream_t stream, int* launches) {
    const bool bf16 = dtype == PKV_BF16;
    if (block_size == 16)
        return bf16 ? launch_prefix_t<true, 16>(p, tmk, tmv, stream, launches)
                    : launch_prefix_t<false, 16>(p, tmk, tmv, stream, launches);
    return bf16 ? launch_prefix_t<true, 32>(p, tmk, tmv, stream, launches)
                : launch_prefix_t<false, 32>(p, tmk, tmv, stream, launches);
}

}  // namespace pkv
