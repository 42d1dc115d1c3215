// decode.cu -- paged decode attention for sm_103a.
//
// What it computes (tonho.wtf "vllm", "como funciona"; techtrendfeed "KV
// Cache Administration", "How PagedAttention Works", step 2): for one new
// query token per sequence, the keys of one block at a time give that
// block's slice of the scores, and the output is accumulated against the
// same block's values; the block table says where each block lives, so
// blocks need not be adjacent.  The block-by-block accumulation is the
// online-softmax rescaling (running max m, running sum l, output rescaled by
// exp(m_old - m_new)), which the pages imply but do not spell out.
//
// Work decomposition.  One CTA per (partition of the context, KV head, GQA
// head tile of <= 16 query heads, sequence).  A partition is a run of
// `partition_size` tokens (chosen per call from 512 to 4096 unless the
// caller fixes it); when a sequence has more than one partition, each CTA
// writes its normalised partial output and log-sum-exp and the last
// partition to finish (or reduce_kernel, for many partitions) merges them
// (split-K).  All query heads of a GQA group share one pass over
// each K/V tile, so a tile is read from HBM once per KV head (once per 16
// query heads when the group is larger than 16).  Partitions are numbered
// from the end of each sequence and that number is the slowest grid
// dimension.  The hardware starts CTAs in linear index order, so every
// sequence's last partition (usually shorter than the others) starts first,
// then the full partitions before it, and the first partitions of the
// sequences with the most partitions end the launch.  This order measured
// faster than starting from the first partitions, and faster than running
// all full partitions before the last ones.
//
// CTA layout: NCW consumer warps + 1 producer warp.
//   producer: reads the partition's block ids (32 at a time, coalesced),
//     checks them against the pool, and for block j issues two TMA loads
//     (K and V; each brings the tile's two 64-column halves, 128-byte
//     swizzle) into ring stage j % NST, completing on that stage's "full"
//     mbarrier.  One copy per tile rather than per half: the SM's TMA unit
//     takes a roughly fixed time per copy of this size.
//   consumer warp w: takes blocks j = w, w + NCW, ...; per 16-token sub-block
//     S = Q K^T with mma.sync m16n8k16 (Q rows = the head tile, padded to 16
//     with zeros; two interleaved score accumulators), masks tokens past the
//     context, updates its own running max/sum (the max is raised only when a
//     score exceeds it by more than 2^8, which skips the reduction and the
//     rescale on most blocks), then O += P V with P split into a 16-bit high
//     part and a 16-bit residual so that P keeps ~16 significant bits.  It
//     releases the stage on its "empty" mbarrier.
//   epilogue: the NCW per-warp (m, l, O) states are merged through shared
//     memory in warp order (fixed, so the result depends only on logical
//     token positions and never on physical block ids).
//
// Shared-memory tile layout: a (block, KV head) tile of K is BS rows x 128
// columns; it lands as two [BS][64] halves, 128 bytes per row, with the TMA
// 128-byte swizzle (16-byte chunk c of row r stored at chunk c ^ (r & 7)),
// which makes the ldmatrix row gathers below bank-conflict free.
#include "decode_common.cuh"

namespace pkv {

template <int BS, int NCW, int NST, int HT>
struct DecodeSmem {
    static constexpr int kTileBytes = BS * kHeadDim * 2;  // one (block, KV head) tile of K or V
    static constexpr int kHalfBytes = kTileBytes / 2;     // its 64-column half
    static constexpr int kStageBytes = 2 * kTileBytes;    // K + V
    static constexpr int kStagesBytes = NST * kStageBytes;
    // per-warp rows, per-warp (m, l), per-row merge weights and lse
    static constexpr int kRedBytes = NCW * HT * kRedStride * 4 + NCW * HT * 2 * 4 + HT * (NCW + 1) * 4;
    // the merge buffer reuses the ring once every stage has been consumed
    static constexpr int kRingBytes = ((kStagesBytes > kRedBytes ? kStagesBytes : kRedBytes) + 1023) / 1024 * 1024;
    static constexpr int kBarOffset = kRingBytes;
    static constexpr int kFlagOffset = kBarOffset + 2 * NST * 8;
    static constexpr int kTotal = kFlagOffset + 16;  // flags[0]: errors, [1]: last-arrival verdict, [2]: no group
    static constexpr int kDynamic = kTotal + 1024;        // slack to align the base to 1024 B
};

// NH: 8-head n-tiles per CTA (1: up to 8 query heads of a group, 2: up to 16).
// kPrefix: grouped decode -- attend only tokens prefix_lens[s] .. L-1 (the
// shared prefix is the prefix kernel's), partial indices after the prefix's.
template <bool kBF16, int BS, int NH, int NCW, int NST, bool kPrefix>
__global__ void __launch_bounds__((NCW + 1) * 32, NH == 1 ? PKV_MINB : PKV_MINB - 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
    using S = DecodeSmem<BS, NCW, NST, 8 * NH>;
    constexpr int D = kHeadDim;
    constexpr int HT = 8 * NH;     // query heads per CTA
    static_assert(BS % 16 == 0, "block size must be a multiple of 16");
    static_assert(NST % NCW == 0, "each ring stage must belong to one consumer warp");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_sa = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_sa + 1023u) & ~1023u) - raw_sa);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Grid: grouped decode (prefix, head group, sequence); plain decode (head
    // group, sequence, partition counted from the end of the sequence): the
    // hardware starts CTAs in linear index order, so the last partitions of
    // all sequences start first.
    // (More than 65535 partitions do not fit the slowest dimension; such a
    // call uses the grouped layout with the partition in x.)
    const bool part_x = kPrefix || p.parts_in_x;
    const int ygrp = part_x ? blockIdx.y : blockIdx.x;  // KV head x head tile
    const int kvh = ygrp / p.head_tiles;
    const int ht = ygrp - kvh * p.head_tiles;
    const int s = part_x ? blockIdx.z : blockIdx.y;
    const int h0 = kvh * p.group + ht * HT;  // first query head of this CTA
    const int rows = min(HT, p.group - ht * HT);

    // Launched with programmatic stream serialisation: the previous kernel on
    // the stream (e.g. the block write) may still be running.  Let the next
    // kernel start launching, then wait for the previous one to finish before
    // reading anything it may have written.  In a grouped call whose prefix
    // kernel ran first (early_inputs), that kernel released this one only
    // after the kernels before the call had completed: the inputs are read at
    // once, and the wait comes before the first read of the prefix kernel's
    // results.
    pdl_launch_dependents();
    if (tid == 32 * NCW) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    const bool early = kPrefix && p.early_inputs;
    if (!early) pdl_wait();
    // A single-pass call (every sequence one partition) starts every CTA's
    // blocks at the sequence's first: the producer loads the first 32 block
    // ids together with the context length, not after it.
    const bool first_ids = !kPrefix && !p.split && warp == NCW;
    int id0 = 0;
    if (first_ids && lane < p.max_blocks_per_seq)
        id0 = __ldg(p.block_tables + (int64_t)s * p.max_blocks_per_seq + lane);

    int L, tok0, nparts, pidx, narrive, part;
    bool shared = false;  // grouped decode: s has a shared prefix; its group is checked before the epilogue
    int fold = 0;         // grouped decode: prefix partials this CTA folds into its own result
    if constexpr (kPrefix) {
        part = blockIdx.x;
        const SeqSpan sp = seq_span(p, s, BS);
        if (sp.err || part >= sp.nsuf) {
            // Partition 0 owns the output of a sequence with nothing to
            // attend (L == 0), with bad metadata, or whose shared prefix no
            // group attended: zeros.  (L == prefix > 0 and attended: the
            // prefix kernel wrote it.)
            if (part == 0) {
                if (early) pdl_wait();
                int err = sp.err;
                if (!err && sp.plen > 0 && !group_verified(p, s)) err = PKV_DEVERR_GROUP;
                if (err || sp.L == 0) {
                    if (err && tid == 0) record_error(p.err, err);
                    for (int i = tid; i < rows * D; i += blockDim.x) store_out(p, s, h0 + i / D, i % D, 0.f);
                }
            }
            return;
        }
        L = sp.L;
        tok0 = sp.plen + part * p.partition_size;  // whole blocks: the prefix length is a multiple of BS
        nparts = sp.npre + sp.nsuf;
        pidx = sp.npre + part;
        narrive = sp.nsuf;  // the prefix partials are complete: only this side's partitions arrive
        shared = sp.plen > 0;
        fold = folds_prefix(sp) ? sp.npre : 0;
    } else {
        const int from_end = part_x ? blockIdx.x : blockIdx.z;
        L = p.context_lens[s];
        const bool bad_len = L < 0 || L > p.len_limit;
        nparts = (bad_len || L == 0) ? 1 : (L + p.partition_size - 1) / p.partition_size;
        if (from_end >= nparts) return;  // the sequence has no such partition
        part = nparts - 1 - from_end;
        if (bad_len || L == 0) {
            // The single partition of a sequence with nothing to attend
            // (L == 0) or with an invalid length owns its output: zeros.
            if (bad_len && tid == 0) record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
            for (int i = tid; i < rows * D; i += blockDim.x) store_out(p, s, h0 + i / D, i % D, 0.f);
            return;
        }
        tok0 = part * p.partition_size;
        pidx = part;
        narrive = nparts;
    }
    const int tok1 = min(L, tok0 + p.partition_size);
    const int nblk = (tok1 - tok0 + BS - 1) / BS;
    const int blk0 = tok0 / BS;
    const bool write_partial = p.split && nparts > 1 && !fold;

    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOffset);
    int* flags = reinterpret_cast<int*>(smem + S::kFlagOffset);  // bit 0: bad block id, bit 1: timeout
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + NST);

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        flags[0] = 0;
        flags[2] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    WarpAcc<NH> acc;  // consumer state (registers); see decode_common.cuh
    acc_reset(acc);
    int issued = 0;  // producer lane 0: TMA stages issued

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        const uint64_t policy = l2_policy_evict_first();
        const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks_per_seq + blk0;
        if (p.fused_append && tok1 == L) {
            // Block write fused into the decode: this partition holds the last
            // position, so this CTA writes that token's row for its KV head
            // before any TMA load can read it.
            const int64_t slot = p.slot_mapping[s];
            if (slot >= 0) {
                const int pos = L - 1;
                const int pb = p.block_tables[(int64_t)s * p.max_blocks_per_seq + pos / BS];
                if (pb >= 0 && (int64_t)pb < p.num_blocks) {  // a bad id is reported by the loads below
                    if (slot == (int64_t)pb * BS + pos % BS) {
                        const int64_t row = ((int64_t)pb * p.num_kv_heads + kvh) * BS + pos % BS;
                        const int64_t src = ((int64_t)s * p.num_kv_heads + kvh) * (kHeadDim / 8);
                        if (lane < 16)
                            p.k_cache[row * (kHeadDim / 8) + lane] = p.k_new[src + lane];
                        else
                            p.v_cache[row * (kHeadDim / 8) + lane - 16] = p.v_new[src + lane - 16];
                        fence_proxy_async_global();
                    } else if (lane == 0) {
                        record_error(p.err, PKV_DEVERR_SLOT);
                    }
                }
                __syncwarp();
            }
        }
        bool ok = true;
        for (int c = 0; c < nblk; c += 32) {
            const int j = c + lane;
            int id = 0;
            bool bad = false;
            if (j < nblk) {
                id = first_ids && c == 0 ? id0 : __ldg(table + j);
                bad = id < 0 || (int64_t)id >= p.num_blocks;
                if (bad) id = 0;  // keep the pipeline's shape; the output is zeroed later
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) {
                atomicOr(flags, 1);
                record_error(p.err, PKV_DEVERR_BLOCK_ID);
            }
            const int n = min(32, nblk - c);
            for (int i = 0; i < n; ++i) {
                const int pid = __shfl_sync(0xffffffffu, id, i);
                if (lane == 0 && ok) {
                    const int jj = c + i, st = jj % NST, round = jj / NST;
                    if (round > 0) ok = mbar_wait(empty0 + 8 * st, (round - 1) & 1);
                    if (ok) {
                        const uint32_t fb = full0 + 8 * st;
                        mbar_arrive_expect_tx(fb, S::kStageBytes);
                        const uint32_t dst = smem_addr(stages + st * S::kStageBytes);
                        const int y = (pid * p.num_kv_heads + kvh) * BS;  // row of the tile in [rows][128]
                        tma_load_3d(dst, &tmk, fb, 0, y, 0, policy);  // both dims halves of the tile
                        tma_load_3d(dst + S::kTileBytes, &tmv, fb, 0, y, 0, policy);
                        ++issued;
                    } else {
                        atomicOr(flags, 2);
                        record_error(p.err, PKV_DEVERR_TIMEOUT);
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        QFrag<NH> qf;
        load_q_frag(qf, p, s, h0, rows, lane);
        const float sl2 = p.scale_log2;
        for (int jj = warp; jj < nblk; jj += NCW) {
            const int st = jj % NST, round = jj / NST;
            // every lane waits (each needs the acquire of the TMA writes); the
            // verdict is made warp-uniform so that a timeout never splits the warp
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, round & 1))) {
                if (lane == 0) {
                    atomicOr(flags, 2);
                    record_error(p.err, PKV_DEVERR_TIMEOUT);
                }
                break;
            }
            const int valid = min(BS, tok1 - (tok0 + jj * BS));  // >= 1
            const uint32_t kb = smem_addr(stages + st * S::kStageBytes);
            attend_block<kBF16, BS, NH, false, true>(acc, qf, kb, kb + S::kTileBytes, valid, sl2, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }
        acc_finish(acc);
    }
    if (early) pdl_wait();  // the prefix kernel's group hints and partials are read below
    __syncthreads();

    const int fl = flags[0];
    if ((fl & 2) && warp == NCW && lane == 0) {
        // A wait ran out: let every TMA load already issued land before the
        // stage memory is reused or the CTA exits (bounded as well).
        for (int st = 0; st < NST && st < issued; ++st) {
            const int last_round = (issued - 1 - st) / NST;
            mbar_wait(full0 + 8 * st, last_round & 1);
        }
    }
    if constexpr (kPrefix) {
        if (shared && tid == 0 && !group_verified(p, s)) flags[2] = 1;
    }
    __syncthreads();
    if constexpr (kPrefix) {
        if (flags[2]) {
            // no group attended this sequence's shared prefix: partition 0
            // zeroes the output, nothing else is written
            if (part == 0) {
                if (tid == 0) record_error(p.err, PKV_DEVERR_GROUP);
                for (int i = tid; i < rows * D; i += blockDim.x) store_out(p, s, h0 + i / D, i % D, 0.f);
            }
            return;
        }
    }

    // ---- merge the per-warp states (stage memory is free now).  Warp w's
    // state (O_w, m_w, l_w) counts 2^(m_w - M) of the row, M = max_w m_w: the
    // row's output is sum_w f_w O_w / sum_w f_w l_w with f_w = 2^(m_w - M).
    // The per-row weights f_w / sum are found once, then every output
    // element is a weighted sum of the warps' rows, a float4 at a time.
    float* red = reinterpret_cast<float*>(smem);      // [NCW][HT][kRedStride]
    float* ml = red + NCW * HT * kRedStride;           // [NCW][HT][2]
    float* wts = ml + NCW * HT * 2;                    // [HT][NCW + 1]: weights, then the row's lse
    if (warp < NCW) acc_to_smem(acc, red, ml, warp, rows, lane);
    __syncthreads();
    if (tid < rows) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml[(w * HT + tid) * 2]);
        float f[NCW], lsum = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float mw = ml[(w * HT + tid) * 2];
            f[w] = mw == -INFINITY ? 0.f : exp2f(mw - M);
            lsum += f[w] * ml[(w * HT + tid) * 2 + 1];
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;  // 0: no warp saw a token (a wait ran out)
#pragma unroll
        for (int w = 0; w < NCW; ++w) wts[tid * (NCW + 1) + w] = f[w] * inv;
        wts[tid * (NCW + 1) + NCW] = M + log2f(lsum);
    }
    __syncthreads();
    // this partition's normalised output, float4 c4 of row hr
    auto own_out = [&](int hr, int c4) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float ww = wts[hr * (NCW + 1) + w];
            const float4 r = *reinterpret_cast<const float4*>(red + (w * HT + hr) * kRedStride + 4 * c4);
            o.x += ww * r.x;
            o.y += ww * r.y;
            o.z += ww * r.z;
            o.w += ww * r.w;
        }
        return o;
    };

    const bool bad = fl != 0;
    if constexpr (kPrefix) {
        if (fold) {
            // out = (2^lse_own o_own + sum_j 2^lse_j o_j) / (2^lse_own + sum_j 2^lse_j)
            // over this partition and the prefix partials j < fold; every
            // load of a row chunk is issued before any is used.
            constexpr int MP = kFuseMergeMaxParts;
            for (int i = tid; i < rows * (D / 4); i += blockDim.x) {
                const int hr = i / (D / 4), c4 = i - hr * (D / 4);
                const int64_t row = (int64_t)s * p.num_q_heads + h0 + hr;
                const float* plse = p.part_lse + row * p.max_parts;
                const float4* po = reinterpret_cast<const float4*>(p.part_o + row * p.max_parts * D) + c4;
                float lj[MP];
                float4 vj[MP];
#pragma unroll
                for (int j = 0; j < MP; ++j)
                    if (j < fold) {
                        lj[j] = __ldcg(plse + j);
                        vj[j] = __ldcg(po + j * (D / 4));
                    }
                const float lse = wts[hr * (NCW + 1) + NCW];
                const float4 o = own_out(hr, c4);
                float M = lse;
#pragma unroll
                for (int j = 0; j < MP; ++j)
                    if (j < fold) M = fmaxf(M, lj[j]);
                const bool zero = bad || M == INFINITY;  // +inf: a prefix partition saw bad metadata
                const float w0 = zero ? 0.f : exp2f(lse - M);
                float sum = w0;
                float4 acc = make_float4(w0 * o.x, w0 * o.y, w0 * o.z, w0 * o.w);
#pragma unroll
                for (int j = 0; j < MP; ++j)
                    if (j < fold) {
                        const float wj = zero ? 0.f : exp2f(lj[j] - M);
                        sum += wj;
                        acc.x += wj * vj[j].x;
                        acc.y += wj * vj[j].y;
                        acc.z += wj * vj[j].z;
                        acc.w += wj * vj[j].w;
                    }
                const float inv = zero ? 0.f : 1.f / sum;
                store_out4(p, s, h0 + hr, 4 * c4, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
            }
            return;
        }
    }
    for (int i = tid; i < rows * (D / 4); i += blockDim.x) {
        const int hr = i / (D / 4), c4 = i - hr * (D / 4);
        const int h = h0 + hr;
        const float4 o = bad ? make_float4(0.f, 0.f, 0.f, 0.f) : own_out(hr, c4);
        if (write_partial) {
            const int64_t idx = ((int64_t)s * p.num_q_heads + h) * p.max_parts + pidx;
            *reinterpret_cast<float4*>(p.part_o + idx * D + 4 * c4) = o;
            // +inf marks a partition whose metadata was bad: the merge zeroes the output.
            if (c4 == 0) p.part_lse[idx] = bad ? INFINITY : wts[hr * (NCW + 1) + NCW];
        } else {
            store_out4(p, s, h, 4 * c4, o);
        }
    }

    if (write_partial && p.fuse_merge) {
        // Every partition of this (sequence, head group) arrives on its
        // counter once its partials are globally visible; the last to arrive
        // merges them.  Nothing ever waits for another CTA.  Thread 0
        // releases the partials every thread wrote before the barrier with
        // one fence, and the last arrival acquires the other partitions'
        // before the barrier that starts the merge.  (A fence in every
        // thread measured ~3 us per CTA under load.)
        __syncthreads();
        if (tid == 0) {
            fence_acq_rel_gpu();
            const bool last =
                arrive_last(p.merge_ctr + (int64_t)s * p.num_kv_heads * p.head_tiles + ygrp, p.epoch, narrive);
            if (last) fence_acq_rel_gpu();
            flags[1] = last ? 1 : 0;
        }
        __syncthreads();
        if (flags[1]) merge_row_partials(p, s, h0, rows, nparts, reinterpret_cast<float*>(smem));
    }
}

// Split-K merge for sequences with many partitions (the decode kernel merges
// the others itself): out = sum_p 2^(lse_p - LSE) o_p, LSE = log2 sum_p
// 2^lse_p.  One CTA per (query head, sequence).  Warp w takes partitions
// w, w + kReduceWarps, ..., kReduceUnroll of them per round with every load
// of the round issued together; lane l holds columns 4l .. 4l+3 as a float4.
// Each warp keeps its own running maximum, sum and weighted output (the
// online form of the merge), and the warps are combined in warp order
// through shared memory, so the result depends only on the partition count.
// The sequence's length is read beside the first round of partials, which
// lie inside the row's workspace slots whatever the length turns out to be.
constexpr int kReduceWarps = 8;
constexpr int kReduceUnroll = 8;

__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(const DecodeParams p) {
    pdl_wait();  // the decode kernel's partials must be complete
    const int h = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kStep = kReduceWarps * kReduceUnroll;
    const int64_t base = ((int64_t)s * p.num_q_heads + h) * p.max_parts;
    const float* lse = p.part_lse + base;
    const float4* po = reinterpret_cast<const float4*>(p.part_o + base * kHeadDim) + lane;
    // first round, before the length is known: partitions < max_parts only
    float lj[kReduceUnroll];
    float4 vj[kReduceUnroll];
#pragma unroll
    for (int u = 0; u < kReduceUnroll; ++u) {
        const int j = warp + u * kReduceWarps;
        if (j < p.max_parts) {
            lj[u] = __ldcg(lse + j);
            vj[u] = __ldcg(po + (int64_t)j * (kHeadDim / 4));
        }
    }
    const SeqSpan sp = seq_span(p, s, p.block_size);
    if (sp.err) return;                   // the decode kernel already zeroed it
    if (sp.plen > 0 && !group_verified(p, s)) return;
    const int np = sp.npre + sp.nsuf;
    if (np <= 1 || folds_prefix(sp)) return;  // written directly by the kernel that attended it
    float m = -INFINITY, l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool bad = false;  // a partition marked +inf (bad metadata) zeroes the row
    for (int j0 = warp;;) {
#pragma unroll
        for (int u = 0; u < kReduceUnroll; ++u) {
            const int j = j0 + u * kReduceWarps;
            if (j < np) {
                if (lj[u] == INFINITY) {
                    bad = true;
                } else if (lj[u] > -INFINITY) {
                    const float mn = fmaxf(m, lj[u]);
                    const float a = exp2f(m - mn), b = exp2f(lj[u] - mn);  // m = -inf: a = 0
                    l = l * a + b;
                    acc.x = acc.x * a + b * vj[u].x;
                    acc.y = acc.y * a + b * vj[u].y;
                    acc.z = acc.z * a + b * vj[u].z;
                    acc.w = acc.w * a + b * vj[u].w;
                    m = mn;
                }
            }
        }
        j0 += kStep;
        if (j0 >= np) break;
#pragma unroll
        for (int u = 0; u < kReduceUnroll; ++u) {
            const int j = j0 + u * kReduceWarps;
            if (j < np) {
                lj[u] = __ldcg(lse + j);
                vj[u] = __ldcg(po + (int64_t)j * (kHeadDim / 4));
            }
        }
    }
    __shared__ float4 red_acc[kReduceWarps][kHeadDim / 4];
    __shared__ float red_m[kReduceWarps], red_l[kReduceWarps];
    __shared__ int red_bad;
    if (threadIdx.x == 0) red_bad = 0;
    __syncthreads();
    red_acc[warp][lane] = acc;
    if (lane == 0) {
        red_m[warp] = m;
        red_l[warp] = l;
        if (bad) red_bad = 1;
    }
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
        const int d = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) M = fmaxf(M, red_m[w]);
        float sum = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) {
            const float f = exp2f(red_m[w] - M);  // a warp with no partition: m = -inf, f = 0
            sum += f * red_l[w];
            o += f * reinterpret_cast<const float*>(&red_acc[w][0])[d];
        }
        store_out(p, s, h, d, red_bad || !(sum > 0.f) ? 0.f : o / sum);
    }
}

template <bool kBF16, int BS, int NH>
static cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                   cudaStream_t stream, int* launches) {
    constexpr int NCW = PKV_NCW;
    constexpr int NST = BS == 16 ? PKV_NST16 : PKV_NST32;
    using S = DecodeSmem<BS, NCW, NST, 8 * NH>;
    auto kern = p.prefix_lens ? decode_kernel<kBF16, BS, NH, NCW, NST, true>
                              : decode_kernel<kBF16, BS, NH, NCW, NST, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kDynamic);
    if (e != cudaSuccess) return e;
    // grouped decode: partitions of the sequences' own tokens only
    const dim3 grid = p.prefix_lens || p.parts_in_x
                          ? dim3(p.max_parts - p.prefix_parts, p.num_kv_heads * p.head_tiles, p.num_seqs)
                          : dim3(p.num_kv_heads * p.head_tiles, p.num_seqs, p.max_parts);
    e = launch_pdl(kern, grid, dim3((NCW + 1) * 32), S::kDynamic, stream, tmk, tmv, p);
    if (e != cudaSuccess) return e;
    ++*launches;
    if (p.split && !p.fuse_merge) {
        e = launch_pdl(reduce_kernel, dim3(p.num_q_heads, p.num_seqs), dim3(kReduceWarps * 32), 0, stream, p);
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int block_size, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, cudaStream_t stream, int* launches) {
    const bool bf16 = dtype == PKV_BF16;
    const bool wide = decode_head_tile(p.group) == 16;
#define PKV_DISPATCH(BS_)                                                                              \
    return bf16 ? (wide ? launch_decode_t<true, BS_, 2>(p, tmk, tmv, stream, launches)                 \
                        : launch_decode_t<true, BS_, 1>(p, tmk, tmv, stream, launches))                \
                : (wide ? launch_decode_t<false, BS_, 2>(p, tmk, tmv, stream, launches)                \
                        : launch_decode_t<false, BS_, 1>(p, tmk, tmv, stream, launches));
    if (block_size == 16) {
        PKV_DISPATCH(16)
    }
    PKV_DISPATCH(32)
#undef PKV_DISPATCH
}

}  // namespace pkv
