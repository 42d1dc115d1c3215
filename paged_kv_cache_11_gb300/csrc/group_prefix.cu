// group_prefix.cu -- the shared-prefix half of grouped decode.
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
// CTA layout: 4 consumer warps + 1 producer warp.  The producer streams the
// partition's (block, KV head) tiles into a ring with TMA exactly as the
// decode kernel does; every consumer warp reads every stage.  Consumer warp
// w owns query rows 16w .. 16w+15 of the CTA's row tile (row r = member
// r / G, head r % G of that member's KV head) and runs the decode warp core
// (decode_common.cuh) over them: S^T = K Q^T with the 16 rows as the N
// dimension, online softmax, O^T += V^T P^T.  A member whose shared prefix
// ends before a block masks its columns for that block.
#include "decode_common.cuh"

namespace pkv {

constexpr int kPrefixWarps = kPrefixRows / 16;  // consumer warps

#ifndef PKV_PNST16
#define PKV_PNST16 8
#endif
#ifndef PKV_PNST32
#define PKV_PNST32 4
#endif

template <int BS, int NST>
struct PrefixSmem {
    static constexpr int kTileBytes = BS * kHeadDim * 2;
    static constexpr int kHalfBytes = kTileBytes / 2;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStagesBytes = NST * kStageBytes;
    // epilogue: the rows' outputs [64][kRedStride] and (m, l) [64][2]
    static constexpr int kRedBytes = kPrefixRows * kRedStride * 4 + kPrefixRows * 2 * 4;
    static constexpr int kRingBytes = ((kStagesBytes > kRedBytes ? kStagesBytes : kRedBytes) + 1023) / 1024 * 1024;
    static constexpr int kBarOffset = kRingBytes;
    // per member of the tile: sequence, prefix tokens (0 when it takes no
    // part), partitions in all, whether the prefix side merges; per (member,
    // head tile): merge verdict
    static constexpr int kMemOffset = kBarOffset + 2 * NST * 8;
    static constexpr int kMemBytes = kPrefixRows * 4 * 4 + kPrefixRows * 4 * 4;
    static constexpr int kFlagOffset = kMemOffset + kMemBytes;
    static constexpr int kTotal = kFlagOffset + 16;
    static constexpr int kDynamic = kTotal + 1024;
};

template <bool kBF16, int BS, int NST>
__global__ void __launch_bounds__((kPrefixWarps + 1) * 32, 2)
    group_prefix_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const DecodeParams p) {
    using S = PrefixSmem<BS, NST>;
    constexpr int D = kHeadDim;
    constexpr int NH = 2;  // 16 rows per consumer warp
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_sa = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_sa + 1023u) & ~1023u) - raw_sa);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int part = blockIdx.x;
    const int kvh = blockIdx.y / p.row_tiles, rt = blockIdx.y - kvh * p.row_tiles;
    const int g = blockIdx.z;
    const int G = p.group;

    pdl_launch_dependents();
    if (tid == 32 * kPrefixWarps) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    pdl_wait();

    int* mem_s = reinterpret_cast<int*>(smem + S::kMemOffset);  // [64]
    int* mem_lim = mem_s + kPrefixRows;                         // [64]
    int* mem_np = mem_lim + kPrefixRows;                        // [64] partitions in all
    int* mem_arrive = mem_np + kPrefixRows;                     // [64] 1: the prefix side merges
    int* verdict = mem_arrive + kPrefixRows;                    // [64 * 4]
    int* flags = reinterpret_cast<int*>(smem + S::kFlagOffset); // [0]: bad block / timeout, [1]: tile token end
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOffset);
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + NST);

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
        flags[0] = 0;
        flags[1] = 0;
        for (int i = 0; i < NST; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kPrefixWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
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
    }
    __syncthreads();
    const int tok1 = flags[1];
    if (tok1 <= tok0) return;  // no member's prefix reaches this partition
    const int nblk = (tok1 - tok0) / BS;  // prefix lengths are whole blocks
    const int blk0 = tok0 / BS;

    WarpAcc<NH> acc;
    acc_reset(acc);
    int issued = 0;

    if (warp == kPrefixWarps) {
        // ------------------------------------------------------------ producer
        const uint64_t policy = l2_policy_evict_first();
        const int32_t* table = p.block_tables + (int64_t)gs0 * p.max_blocks_per_seq + blk0;
        bool ok = true;
        for (int c = 0; c < nblk; c += 32) {
            const int j = c + lane;
            int id = 0;
            bool bad = false;
            if (j < nblk) {
                id = __ldg(table + j);
                bad = id < 0 || (int64_t)id >= p.num_blocks;
                if (bad) id = 0;
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
                        const uint32_t dst = smem_addr(smem + st * S::kStageBytes);
                        const int y = (pid * p.num_kv_heads + kvh) * BS;
                        tma_load_2d(dst, &tmk, fb, 0, y, policy);
                        tma_load_2d(dst + S::kHalfBytes, &tmk, fb, 64, y, policy);
                        tma_load_2d(dst + S::kTileBytes, &tmv, fb, 0, y, policy);
                        tma_load_2d(dst + S::kTileBytes + S::kHalfBytes, &tmv, fb, 64, y, policy);
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
        // rows of this warp: 16 warp + 8 n + (lane / 4) for the Q operand,
        // columns 16 warp + 8 n + 2 (lane % 4) + c for the scores it holds
        const int gq = lane >> 2, t = lane & 3;
        QFrag<NH> qf;
#pragma unroll
        for (int n = 0; n < NH; ++n) {
            const int r = 16 * warp + 8 * n + gq, mi = r / G;
            const uint32_t* qr =
                mi < nmem ? reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) +
                                                              ((int64_t)mem_s[mi] * p.num_q_heads + kvh * G + r - mi * G) *
                                                                  kHeadDim)
                          : nullptr;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                qf.b[n][ks][0] = qr ? __ldg(qr + 8 * ks + t) : 0u;
                qf.b[n][ks][1] = qr ? __ldg(qr + 8 * ks + 4 + t) : 0u;
            }
        }
        int lim[NH][2];  // prefix tokens of each held column's member (0: none)
#pragma unroll
        for (int n = 0; n < NH; ++n)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int mi = (16 * warp + 8 * n + 2 * t + c) / G;
                lim[n][c] = mi < nmem ? mem_lim[mi] : 0;
            }
        const float sl2 = p.scale_log2;
        for (int jj = 0; jj < nblk; ++jj) {
            const int st = jj % NST, round = jj / NST;
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, round & 1))) {
                if (lane == 0) {
                    atomicOr(flags, 2);
                    record_error(p.err, PKV_DEVERR_TIMEOUT);
                }
                break;
            }
            const int tb = tok0 + jj * BS;
            uint32_t cols = 0;
#pragma unroll
            for (int n = 0; n < NH; ++n)
#pragma unroll
                for (int c = 0; c < 2; ++c) cols |= (tb < lim[n][c] ? 1u : 0u) << (2 * n + c);
            const uint32_t kb = smem_addr(smem + st * S::kStageBytes);
            attend_block<kBF16, BS, NH, true, true>(acc, qf, kb, kb + S::kTileBytes, BS, sl2, lane, cols);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }
        acc_finish(acc);
    }
    __syncthreads();

    const int fl = flags[0];
    if ((fl & 2) && warp == kPrefixWarps && lane == 0) {
        for (int st = 0; st < NST && st < issued; ++st) {
            const int last_round = (issued - 1 - st) / NST;
            mbar_wait(full0 + 8 * st, last_round & 1);
        }
    }
    __syncthreads();

    // ---- each warp's 16 rows are complete: stage them, then write them out
    float* red = reinterpret_cast<float*>(smem);  // [64][kRedStride]
    float* ml = red + kPrefixRows * kRedStride;    // [64][2]
    if (warp < kPrefixWarps) acc_to_smem(acc, red + 16 * warp * kRedStride, ml + 16 * warp * 2, 0, 16, lane);
    __syncthreads();

    const bool bad = fl != 0;
    const int rows = nmem * G;
    for (int i = tid; i < rows * (D / 4); i += blockDim.x) {
        const int r = i / (D / 4), c4 = i - r * (D / 4);
        const int mi = r / G;
        if (tok0 >= mem_lim[mi]) continue;  // this member's prefix ends before the partition
        const int s = mem_s[mi], h = kvh * G + r - mi * G;
        const float l = ml[r * 2 + 1];
        const float inv = 1.f / l;
        const float* src = red + r * kRedStride + 4 * c4;
        float4 o = make_float4(src[0] * inv, src[1] * inv, src[2] * inv, src[3] * inv);
        if (bad) o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mem_np[mi] > 1) {
            const int64_t idx = ((int64_t)s * p.num_q_heads + h) * p.max_parts + part;
            reinterpret_cast<float4*>(p.part_o + idx * D)[c4] = o;
            if (c4 == 0) p.part_lse[idx] = bad ? INFINITY : ml[r * 2] + log2f(l);
        } else {
            store_out(p, s, h, 4 * c4, o.x);
            store_out(p, s, h, 4 * c4 + 1, o.y);
            store_out(p, s, h, 4 * c4 + 2, o.z);
            store_out(p, s, h, 4 * c4 + 3, o.w);
        }
    }

    if (p.fuse_merge) {
        // One arrival per (member, head tile of the decode kernel) that takes
        // a partial from this partition; the last arrival merges the row.
        const int units = nmem * p.head_tiles;
        __threadfence();
        __syncthreads();
        for (int u = tid; u < units; u += blockDim.x) {
            const int mi = u / p.head_tiles, ht = u - mi * p.head_tiles;
            bool last = false;
            if (tok0 < mem_lim[mi] && mem_np[mi] > 1 && mem_arrive[mi]) {
                const int64_t c = (int64_t)mem_s[mi] * p.num_kv_heads * p.head_tiles + kvh * p.head_tiles + ht;
                last = arrive_last(p.merge_ctr + c, p.epoch, mem_np[mi]);
            }
            verdict[u] = last ? 1 : 0;
        }
        __syncthreads();
        const int HT = decode_head_tile(G);
        for (int u = 0; u < units; ++u) {
            if (!verdict[u]) continue;
            const int mi = u / p.head_tiles, ht = u - mi * p.head_tiles;
            __threadfence();
            merge_row_partials(p, mem_s[mi], kvh * G + ht * HT, min(HT, G - ht * HT), mem_np[mi],
                               reinterpret_cast<float*>(smem));
            __syncthreads();  // the scratch is reused by the next merge
        }
    }
}

template <bool kBF16, int BS>
static cudaError_t launch_prefix_t(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                   cudaStream_t stream, int* launches) {
    constexpr int NST = BS == 16 ? PKV_PNST16 : PKV_PNST32;
    using S = PrefixSmem<BS, NST>;
    auto kern = group_prefix_kernel<kBF16, BS, NST>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kDynamic);
    if (e != cudaSuccess) return e;
    const dim3 grid(p.prefix_parts, p.num_kv_heads * p.row_tiles, p.num_groups);
    e = launch_pdl(kern, grid, dim3((kPrefixWarps + 1) * 32), S::kDynamic, stream, tmk, tmv, p);
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
