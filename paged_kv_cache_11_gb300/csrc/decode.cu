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
// `partition_size` tokens (512 by default); when a sequence has more than one
// partition, each CTA writes its normalised partial output and log-sum-exp
// and reduce_kernel merges them (split-K).  All query heads of a GQA group
// share one pass over each K/V tile, so a tile is read from HBM once per KV
// head (once per 16 query heads when the group is larger than 16).
//
// CTA layout: NCW consumer warps + 1 producer warp.
//   producer: reads the partition's block ids (32 at a time, coalesced),
//     checks them against the pool, and for block j issues four 2-D TMA
//     loads (K and V, two 64-column halves each, 128-byte swizzle) into ring
//     stage j % NST, completing on that stage's "full" mbarrier.
//   consumer warp w: takes blocks j = w, w + NCW, ...; per 16-token sub-block
//     S = Q K^T with mma.sync m16n8k16 (Q rows = the head tile, padded to 16
//     with zeros), masks tokens past the context, updates its own running
//     max/sum, then O += P V with P split into a 16-bit high part and a
//     16-bit residual so that P keeps ~16 significant bits.  It releases the
//     stage on its "empty" mbarrier.
//   epilogue: the NCW per-warp (m, l, O) states are merged through shared
//     memory in warp order (fixed, so the result depends only on logical
//     token positions and never on physical block ids).
//
// Shared-memory tile layout: a (block, KV head) tile of K is BS rows x 128
// columns; it lands as two [BS][64] halves, 128 bytes per row, with the TMA
// 128-byte swizzle (16-byte chunk c of row r stored at chunk c ^ (r & 7)),
// which makes the ldmatrix row gathers below bank-conflict free.
#include "pkv_internal.cuh"

namespace pkv {

template <int BS, int NCW, int NST>
struct DecodeSmem {
    static constexpr int kTileBytes = BS * kHeadDim * 2;  // one (block, KV head) tile of K or V
    static constexpr int kHalfBytes = kTileBytes / 2;     // its 64-column half
    static constexpr int kStageBytes = 2 * kTileBytes;    // K + V
    static constexpr int kStagesBytes = NST * kStageBytes;
    static constexpr int kRedStride = kHeadDim + 4;       // floats per merged row
    static constexpr int kRedBytes = NCW * kHeadTile * kRedStride * 4 + NCW * kHeadTile * 2 * 4;
    static constexpr int kBarOffset = kStagesBytes;
    static constexpr int kFlagOffset = kBarOffset + 2 * NST * 8;
    static constexpr int kTotal = kFlagOffset + 16;
    static constexpr int kDynamic = kTotal + 1024;        // slack to align the base to 1024 B
    static_assert(kRedBytes <= kStagesBytes, "merge buffer must fit in the stage ring");
};

__device__ __forceinline__ void store_out(const DecodeParams& p, int s, int h, int d, float v) {
    const int64_t i = ((int64_t)s * p.num_q_heads + h) * kHeadDim + d;
    if (p.out_dtype == PKV_FP32)
        static_cast<float*>(p.out)[i] = v;
    else if (p.out_dtype == PKV_BF16)
        static_cast<__nv_bfloat16*>(p.out)[i] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(p.out)[i] = __float2half_rn(v);
}

template <bool kBF16, int BS, int NCW, int NST>
__global__ void __launch_bounds__((NCW + 1) * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
    using S = DecodeSmem<BS, NCW, NST>;
    constexpr int D = kHeadDim;
    constexpr int kSub = BS / 16;  // 16-token sub-blocks per block
    static_assert(BS % 16 == 0, "block size must be a multiple of 16");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_sa = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_sa + 1023u) & ~1023u) - raw_sa);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int part = blockIdx.x;
    const int kvh = blockIdx.y / p.head_tiles;
    const int ht = blockIdx.y - kvh * p.head_tiles;
    const int s = blockIdx.z;
    const int h0 = kvh * p.group + ht * kHeadTile;  // first query head of this CTA
    const int rows = min(kHeadTile, p.group - ht * kHeadTile);

    const int L = __ldg(p.context_lens + s);
    const bool bad_len = L < 0 || L > p.len_limit;
    if (bad_len || part * p.partition_size >= L) {
        // Partition 0 owns the output of a sequence with nothing to attend
        // (L == 0) or with an invalid length: zeros.
        if (part == 0) {
            if (bad_len && tid == 0) record_error(p.err, PKV_DEVERR_CONTEXT_LEN);
            for (int i = tid; i < rows * D; i += blockDim.x) store_out(p, s, h0 + i / D, i % D, 0.f);
        }
        return;
    }
    const int tok0 = part * p.partition_size;
    const int tok1 = min(L, tok0 + p.partition_size);
    const int nblk = (tok1 - tok0 + BS - 1) / BS;
    const int blk0 = tok0 / BS;
    const int nparts = (L + p.partition_size - 1) / p.partition_size;
    const bool write_partial = p.split && nparts > 1;

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
        fence_barrier_init();
    }
    __syncthreads();

    // consumer state (registers)
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int issued = 0;  // producer lane 0: TMA stages issued

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        const uint64_t policy = l2_policy_evict_first();
        const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks_per_seq + blk0;
        bool ok = true;
        for (int c = 0; c < nblk; c += 32) {
            const int j = c + lane;
            int id = 0;
            bool bad = false;
            if (j < nblk) {
                id = __ldg(table + j);
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
        const int r0 = lane >> 2, r1 = r0 + 8, cq = 2 * (lane & 3);
        // Q as the A operand of S = Q K^T: 8 k-steps of 16 dims.
        uint32_t qa[8][4];
        {
            const uint32_t* q0 = r0 < rows ? reinterpret_cast<const uint32_t*>(
                                                 static_cast<const uint16_t*>(p.q) +
                                                 ((int64_t)s * p.num_q_heads + h0 + r0) * D)
                                           : nullptr;
            const uint32_t* q1 = r1 < rows ? reinterpret_cast<const uint32_t*>(
                                                 static_cast<const uint16_t*>(p.q) +
                                                 ((int64_t)s * p.num_q_heads + h0 + r1) * D)
                                           : nullptr;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int c0 = (16 * ks + cq) >> 1, c1 = (16 * ks + 8 + cq) >> 1;
                qa[ks][0] = q0 ? __ldg(q0 + c0) : 0u;
                qa[ks][1] = q1 ? __ldg(q1 + c0) : 0u;
                qa[ks][2] = q0 ? __ldg(q0 + c1) : 0u;
                qa[ks][3] = q1 ? __ldg(q1 + c1) : 0u;
            }
        }
        const float sl2 = p.scale_log2;
        const int mi = lane >> 3, rr = lane & 7;

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
            const uint32_t vb = kb + S::kTileBytes;

#pragma unroll
            for (int sub = 0; sub < kSub; ++sub) {
                if (sub * 16 >= valid) break;  // warp-uniform: nothing valid left in this block
                // ---- S = Q K^T for tokens sub*16 .. sub*16+15
                float sc[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
                {
                    // matrices: (tokens 0-7 | 8-15) x (dims lo | hi of the k-step)
                    const int tok = sub * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int chunk = 2 * ks + (mi & 1);
                        const int line = (chunk >> 3) * BS + tok;
                        const uint32_t addr = kb + line * 128 + (((chunk & 7) ^ rr) << 4);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        mma_16816<kBF16>(sc[0], qa[ks], b0, b1);
                        mma_16816<kBF16>(sc[1], qa[ks], b2, b3);
                    }
                }
                // ---- scale (log2 domain), mask past the context, online softmax
                const int tb = sub * 16 + cq;  // token of sc[nt][0] is tb + 8 nt; sc[nt][1] is one more
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int t = tb + 8 * nt;
                    sc[nt][0] = t < valid ? sc[nt][0] * sl2 : -INFINITY;
                    sc[nt][1] = t + 1 < valid ? sc[nt][1] * sl2 : -INFINITY;
                    sc[nt][2] = t < valid ? sc[nt][2] * sl2 : -INFINITY;
                    sc[nt][3] = t + 1 < valid ? sc[nt][3] * sl2 : -INFINITY;
                    mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
                    mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
                const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
                const float ms0 = mn0 == -INFINITY ? 0.f : mn0;
                const float ms1 = mn1 == -INFINITY ? 0.f : mn1;
                m0 = mn0;
                m1 = mn1;
                float pr[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    pr[nt][0] = exp2f(sc[nt][0] - ms0);
                    pr[nt][1] = exp2f(sc[nt][1] - ms0);
                    pr[nt][2] = exp2f(sc[nt][2] - ms1);
                    pr[nt][3] = exp2f(sc[nt][3] - ms1);
                }
                l0 = l0 * al0 + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
                l1 = l1 * al1 + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
#pragma unroll
                for (int n2 = 0; n2 < 16; ++n2) {
                    o[n2][0] *= al0;
                    o[n2][1] *= al0;
                    o[n2][2] *= al1;
                    o[n2][3] *= al1;
                }
                // ---- P as the A operand: high part + residual
                uint32_t ph[4], pl[4];
                {
                    float ra, rb;
                    ph[0] = pack2<kBF16>(pr[0][0], pr[0][1], ra, rb);
                    pl[0] = pack2<kBF16>(pr[0][0] - ra, pr[0][1] - rb);
                    ph[1] = pack2<kBF16>(pr[0][2], pr[0][3], ra, rb);
                    pl[1] = pack2<kBF16>(pr[0][2] - ra, pr[0][3] - rb);
                    ph[2] = pack2<kBF16>(pr[1][0], pr[1][1], ra, rb);
                    pl[2] = pack2<kBF16>(pr[1][0] - ra, pr[1][1] - rb);
                    ph[3] = pack2<kBF16>(pr[1][2], pr[1][3], ra, rb);
                    pl[3] = pack2<kBF16>(pr[1][2] - ra, pr[1][3] - rb);
                }
                // ---- O += P V over the 16 tokens
                {
                    // matrices: (tokens 0-7 | 8-15) x (8-column n-tiles 2qd | 2qd+1), transposed
                    const int tok = sub * 16 + (mi & 1) * 8 + rr;
                    const bool tail = sub * 16 + 16 > valid;
                    // V rows past the context may hold anything (even NaN): zero them
                    // in the B fragments rather than rely on p == 0.
                    const uint32_t keep0 = (tb < valid ? 0x0000ffffu : 0u) | (tb + 1 < valid ? 0xffff0000u : 0u);
                    const uint32_t keep1 =
                        (tb + 8 < valid ? 0x0000ffffu : 0u) | (tb + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
                    for (int qd = 0; qd < 8; ++qd) {
                        const int chunk = 2 * qd + (mi >> 1);
                        const int line = (chunk >> 3) * BS + tok;
                        const uint32_t addr = vb + line * 128 + (((chunk & 7) ^ rr) << 4);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_trans(addr, b0, b1, b2, b3);
                        if (tail) {
                            b0 &= keep0;
                            b1 &= keep1;
                            b2 &= keep0;
                            b3 &= keep1;
                        }
                        mma_16816<kBF16>(o[2 * qd], ph, b0, b1);
                        mma_16816<kBF16>(o[2 * qd], pl, b0, b1);
                        mma_16816<kBF16>(o[2 * qd + 1], ph, b2, b3);
                        mma_16816<kBF16>(o[2 * qd + 1], pl, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
        }
        // full row sums: the four lanes of a quad hold disjoint token columns
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
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
    __syncthreads();

    // ---- merge the per-warp states (stage memory is free now)
    float* red = reinterpret_cast<float*>(smem);                // [NCW][16][kRedStride]
    float* ml = red + NCW * kHeadTile * S::kRedStride;          // [NCW][16][2]
    if (warp < NCW) {
        const int r0 = lane >> 2, r1 = r0 + 8, cq = 2 * (lane & 3);
        if (r0 < rows) {
            float* dst = red + (warp * kHeadTile + r0) * S::kRedStride + cq;
#pragma unroll
            for (int n2 = 0; n2 < 16; ++n2) *reinterpret_cast<float2*>(dst + 8 * n2) = make_float2(o[n2][0], o[n2][1]);
            if ((lane & 3) == 0) {
                ml[(warp * kHeadTile + r0) * 2] = m0;
                ml[(warp * kHeadTile + r0) * 2 + 1] = l0;
            }
        }
        if (r1 < rows) {
            float* dst = red + (warp * kHeadTile + r1) * S::kRedStride + cq;
#pragma unroll
            for (int n2 = 0; n2 < 16; ++n2) *reinterpret_cast<float2*>(dst + 8 * n2) = make_float2(o[n2][2], o[n2][3]);
            if ((lane & 3) == 0) {
                ml[(warp * kHeadTile + r1) * 2] = m1;
                ml[(warp * kHeadTile + r1) * 2 + 1] = l1;
            }
        }
    }
    __syncthreads();

    const bool bad = fl != 0;
    for (int i = tid; i < rows * D; i += blockDim.x) {
        const int g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml[(w * kHeadTile + g) * 2]);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float mw = ml[(w * kHeadTile + g) * 2];
            if (mw != -INFINITY) {
                const float f = exp2f(mw - M);
                lsum += f * ml[(w * kHeadTile + g) * 2 + 1];
                acc += f * red[(w * kHeadTile + g) * S::kRedStride + d];
            }
        }
        const int h = h0 + g;
        if (write_partial) {
            const int64_t idx = ((int64_t)s * p.num_q_heads + h) * p.max_parts + part;
            p.part_o[idx * D + d] = bad ? 0.f : acc / lsum;
            // +inf marks a partition whose metadata was bad: the merge zeroes the output.
            if (d == 0) p.part_lse[idx] = bad ? INFINITY : M + log2f(lsum);
        } else {
            store_out(p, s, h, d, bad ? 0.f : acc / lsum);
        }
    }
}

// Split-K merge: out = sum_p 2^(lse_p - LSE) o_p with LSE = log2 sum_p 2^lse_p,
// for sequences with at least two partitions.  One CTA per (query head,
// sequence); thread d owns output column d.
__global__ void __launch_bounds__(kHeadDim) reduce_kernel(const DecodeParams p) {
    const int h = blockIdx.x, s = blockIdx.y, d = threadIdx.x;
    const int L = __ldg(p.context_lens + s);
    if (L < 0 || L > p.len_limit) return;  // the decode kernel already zeroed it
    const int np = (L + p.partition_size - 1) / p.partition_size;
    if (np <= 1) return;                   // written directly by the decode kernel
    const int64_t base = ((int64_t)s * p.num_q_heads + h) * p.max_parts;
    const float* lse = p.part_lse + base;
    const float* po = p.part_o + base * kHeadDim + d;
    float M = -INFINITY;
    bool bad = false;
    for (int i = 0; i < np; ++i) {
        const float v = lse[i];
        bad |= v == INFINITY;
        M = fmaxf(M, v);
    }
    float acc = 0.f, sum = 0.f;
    if (!bad) {
#pragma unroll 8
        for (int i = 0; i < np; ++i) {
            const float w = exp2f(lse[i] - M);
            sum += w;
            acc += w * po[(int64_t)i * kHeadDim];
        }
    }
    store_out(p, s, h, d, bad ? 0.f : acc / sum);
}

template <bool kBF16, int BS, int NCW, int NST>
static cudaError_t launch_decode_t(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                   cudaStream_t stream, int* launches) {
    using S = DecodeSmem<BS, NCW, NST>;
    auto kern = decode_kernel<kBF16, BS, NCW, NST>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kDynamic);
    if (e != cudaSuccess) return e;
    const dim3 grid(p.max_parts, p.num_kv_heads * p.head_tiles, p.num_seqs);
    kern<<<grid, (NCW + 1) * 32, S::kDynamic, stream>>>(tmk, tmv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ++*launches;
    if (p.split) {
        reduce_kernel<<<dim3(p.num_q_heads, p.num_seqs), kHeadDim, 0, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int block_size, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, cudaStream_t stream, int* launches) {
    const bool bf16 = dtype == PKV_BF16;
    if (block_size == 16)
        return bf16 ? launch_decode_t<true, 16, 4, 8>(p, tmk, tmv, stream, launches)
                    : launch_decode_t<false, 16, 4, 8>(p, tmk, tmv, stream, launches);
    return bf16 ? launch_decode_t<true, 32, 4, 4>(p, tmk, tmv, stream, launches)
                : launch_decode_t<false, 32, 4, 4>(p, tmk, tmv, stream, launches);
}

}  // namespace pkv
