// decode_common.cuh -- the per-warp attention core of the decode kernel
// (decode.cu), kept apart from the grid and pipeline code around it.
//
// A consumer warp owns the running state of up to NH x 8 query heads of one
// GQA group: O^T accumulators, running max m and running sum l per head.
// attend_block() folds one (block, KV head) tile of K and V, staged in shared
// memory by TMA with the 128-byte swizzle, into that state:
//   S^T = K Q^T   (mma.sync m16n8k16; tokens are M, query heads are N)
//   online softmax per head (log2 domain, scale folded into sl2)
//   O^T += V^T P^T (P^T moved to operand layout with movmatrix.trans,
//                   P split into a 16-bit high part and a 16-bit residual)
// This is the block-by-block accumulation of tonho.wtf "vllm", "como
// funciona": the current token's query against one block's keys, the output
// accumulated against the same block's values.
#pragma once

#include "pkv_internal.cuh"

// Tunables (compile-time): consumer warps per CTA, ring stages for 16- and
// 32-token blocks, and the minimum resident CTAs per SM the register
// allocation must allow.
#ifndef PKV_NCW
#define PKV_NCW 2
#endif
#ifndef PKV_NST16
#define PKV_NST16 4
#endif
#ifndef PKV_NST32
#define PKV_NST32 2
#endif
#ifndef PKV_MINB
#define PKV_MINB kDecodeCtasPerSm
#endif

namespace pkv {

constexpr int kRedStride = kHeadDim + 4;  // floats per row of the warp-merge buffer

__device__ __forceinline__ void store_out(const DecodeParams& p, int s, int h, int d, float v) {
    const int64_t i = ((int64_t)s * p.num_q_heads + h) * kHeadDim + d;
    if (p.out_dtype == PKV_FP32)
        static_cast<float*>(p.out)[i] = v;
    else if (p.out_dtype == PKV_BF16)
        static_cast<__nv_bfloat16*>(p.out)[i] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(p.out)[i] = __float2half_rn(v);
}

// Four consecutive output elements d .. d + 3 (d a multiple of 4) of query
// head h of sequence s; the output is 16-byte aligned.
__device__ __forceinline__ void store_out4(const DecodeParams& p, int s, int h, int d, float4 v) {
    const int64_t i = ((int64_t)s * p.num_q_heads + h) * kHeadDim + d;
    if (p.out_dtype == PKV_FP32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.out) + i) = v;
    } else if (p.out_dtype == PKV_BF16) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + i) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    } else {
        const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        *reinterpret_cast<uint2*>(static_cast<__half*>(p.out) + i) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    }
}

// Count one arrival of this call (epoch) on a (epoch << 16 | count) counter
// and report whether it was the nparts-th.  A counter left by another call
// (different epoch) counts as zero, so stale or garbage contents never
// matter; the last arrival also resets the count, so a replay of the same
// launch (same epoch, e.g. from a captured graph) starts from zero too.
// Lock-free: a failed CAS means another CTA's arrival got in first, so the
// loop ends after at most nparts tries.
__device__ __forceinline__ bool arrive_last(unsigned long long* ctr, unsigned long long epoch, int nparts) {
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr);
    for (;;) {
        const unsigned long long cnt = (old >> 16) == epoch ? (old & 0xFFFFull) + 1 : 1;
        const bool last = cnt == (unsigned long long)nparts;
        const unsigned long long prev = atomicCAS(ctr, old, (epoch << 16) | (last ? 0ull : cnt));
        if (prev == old) return last;
        old = prev;
    }
}

// Merge the nparts partial (o_p, lse_p) of query heads h0 .. h0+rows-1 of
// sequence s into out: out = sum_p 2^(lse_p - LSE) o_p, LSE = log2 sum_p
// 2^lse_p.  A partition marked +inf (bad metadata) zeroes the row.  Runs in
// the CTA that arrived last, so it sits on the critical path of the row: all
// loads of a phase are issued together (L2 latency once per phase, not once
// per partition).  Partials written by other CTAs are read through L2
// (ld.global.cg).  `w` is shared scratch of rows x (kFuseMergeMaxParts + 1)
// floats.
static __device__ __noinline__ void merge_row_partials(const DecodeParams& p, int s, int h0, int rows, int nparts,
                                                float* w) {
    constexpr int MP = kFuseMergeMaxParts;
    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)s * p.num_q_heads + h0;
    for (int i = tid; i < rows * nparts; i += blockDim.x) {
        const int r = i / nparts, j = i - r * nparts;
        w[r * MP + j] = __ldcg(p.part_lse + (row0 + r) * p.max_parts + j);
    }
    __syncthreads();
    for (int r = tid; r < rows; r += blockDim.x) {
        float M = -INFINITY;
        for (int j = 0; j < nparts; ++j) M = fmaxf(M, w[r * MP + j]);
        const bool bad = M == INFINITY;  // a bad row merges to exact zeros
        float sum = 0.f;
        for (int j = 0; j < nparts; ++j) {
            const float e = bad ? 0.f : exp2f(w[r * MP + j] - M);
            w[r * MP + j] = e;
            sum += e;
        }
        w[rows * MP + r] = bad ? 0.f : 1.f / sum;
    }
    __syncthreads();
    // one float4 of one row per item; every partition's load issued up front
    for (int i = tid; i < rows * (kHeadDim / 4); i += blockDim.x) {
        const int r = i / (kHeadDim / 4), c = i - r * (kHeadDim / 4);
        const float4* po = reinterpret_cast<const float4*>(p.part_o + (row0 + r) * p.max_parts * kHeadDim) + c;
        float4 v[MP];
#pragma unroll
        for (int j = 0; j < MP; ++j)
            if (j < nparts) v[j] = __ldcg(po + j * (kHeadDim / 4));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < MP; ++j)
            if (j < nparts) {
                const float wj = w[r * MP + j];
                acc.x += wj * v[j].x;
                acc.y += wj * v[j].y;
                acc.z += wj * v[j].z;
                acc.w += wj * v[j].w;
            }
        const float inv = w[rows * MP + r];
        store_out4(p, s, h0 + r, 4 * c, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
}

// What sequence s of a decode call attends.  L tokens in all; in grouped
// decode the first plen of them are attended by the prefix kernel in npre
// prefix partitions and the rest by the decode kernel in nsuf partitions
// (plain decode: plen = npre = 0).  err != 0 is the PKV_DEVERR_* code of bad
// metadata: the sequence then attends nothing and its output is zero.
struct SeqSpan {
    int L, plen, npre, nsuf, err;
};

__device__ __forceinline__ SeqSpan seq_span(const DecodeParams& p, int s, int block_size) {
    SeqSpan r;
    r.L = p.context_lens[s];
    r.plen = p.prefix_lens ? p.prefix_lens[s] : 0;
    r.err = 0;
    if (r.L < 0 || r.L > p.len_limit)
        r.err = PKV_DEVERR_CONTEXT_LEN;
    else if (r.plen < 0 || r.plen > r.L || r.plen > p.max_prefix_len || r.plen % block_size != 0)
        r.err = PKV_DEVERR_PREFIX_LEN;
    if (r.err) {
        r.L = r.plen = r.npre = r.nsuf = 0;
        return r;
    }
    r.npre = r.plen > 0 ? (r.plen + p.prefix_partition - 1) / p.prefix_partition : 0;
    r.nsuf = (r.L - r.plen + p.partition_size - 1) / p.partition_size;
    return r;
}

// Grouped decode: how a sequence's partials come together.  The prefix
// kernel has completed before the decode kernel starts, so a sequence with
// one partition of its own (and not too many prefix partitions) is finished
// by that partition's CTA, which folds the prefix partials into its own
// state.  Otherwise the last arrival among the CTAs of the side that runs
// last merges every partial -- the sequence's own partitions when it has
// several, else its prefix partitions -- or the merge kernel does, when the
// call has more partitions than an in-kernel merge takes.
__device__ __forceinline__ bool folds_prefix(const SeqSpan& sp) {
    return sp.nsuf == 1 && sp.npre >= 1 && sp.npre + 1 <= kFuseMergeMaxParts;
}

// Grouped decode: was sequence s's shared prefix attended by this call's
// prefix kernel?  The kernel stores, for every member it takes, the index of
// its group in seq_group[s]; the value read here may also be a stale one from
// an earlier call (or garbage), so it is only a hint, checked against this
// call's group_starts: every group whose range is valid is taken in full up
// to the row-tile capacity, so a hint that names a valid group containing s
// within that capacity proves s was attended, whoever wrote it.  Readable
// once the prefix kernel has completed.
__device__ __forceinline__ bool group_verified(const DecodeParams& p, int s) {
    const int m = __ldcg(p.seq_group + s);
    if (m < 0 || m >= p.num_groups) return false;
    const int a = p.group_starts[m], b = p.group_starts[m + 1];
    return a >= 0 && a <= s && s < b && b <= p.num_seqs && s - a < p.row_tiles * p.members_per_tile;
}

// Q^T as the B operand of S^T = K Q^T: for k-step ks, b[n][ks][0] holds
// q[head 8n + g][16 ks + 2t .. +1] and b[n][ks][1] q[head 8n + g][16 ks + 8 + 2t .. +1]
// (g = lane / 4, t = lane % 4); heads past `rows` are zero.
template <int NH>
struct QFrag {
    uint32_t b[NH][8][2];
};

// One warp's running state: O^T accumulators (m-tile of 16 dims x n-tile x
// fragment) and per-head running max / sum for heads 8n + 2t, 8n + 2t + 1.
template <int NH>
struct WarpAcc {
    float o[8][NH][4];
    float m[NH][2];
    float l[NH][2];
};

template <int NH>
__device__ __forceinline__ void load_q_frag(QFrag<NH>& q, const DecodeParams& p, int s, int h0, int rows,
                                            int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int n = 0; n < NH; ++n) {
        const int hr = 8 * n + g;
        const uint32_t* qr =
            hr < rows ? reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) +
                                                          ((int64_t)s * p.num_q_heads + h0 + hr) * kHeadDim)
                      : nullptr;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            q.b[n][ks][0] = qr ? __ldg(qr + 8 * ks + t) : 0u;
            q.b[n][ks][1] = qr ? __ldg(qr + 8 * ks + 4 + t) : 0u;
        }
    }
}

template <int NH>
__device__ __forceinline__ void acc_reset(WarpAcc<NH>& a) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int n = 0; n < NH; ++n) a.o[mt][n][0] = a.o[mt][n][1] = a.o[mt][n][2] = a.o[mt][n][3] = 0.f;
#pragma unroll
    for (int n = 0; n < NH; ++n) a.m[n][0] = a.m[n][1] = -INFINITY, a.l[n][0] = a.l[n][1] = 0.f;
}

// Fold one staged tile (K at shared address kb, V at vb; `valid` tokens of
// the block, >= 1) into the warp state.  With kColMask, bit 2n + c of
// `cols` says whether this thread's query column 8n + 2t + c attends the
// block at all (a cleared bit masks every token of the block for that
// column; used when the rows of one tile attend different token ranges).
// kIlp is for compute-heavier callers (the prefix kernel).  It orders the
// MMAs for more independent work in flight: two score accumulators per
// n-tile, and the residual half of P V one m-tile behind the high half.  It
// also keeps the running max m lazily.  m is raised, and O and l are
// rescaled, only when some score of the warp exceeds its column's m by more
// than kLazyMargin (log2 units; a warp vote).  Otherwise p = 2^(s - m) <=
// 2^kLazyMargin is accumulated against the unchanged m.  O and l always
// share one m, so the result is the same softmax; the common case skips the
// max reduction and the rescale.
constexpr float kLazyMargin = 8.f;
template <bool kBF16, int BS, int NH, bool kColMask = false, bool kIlp = false>
__device__ __forceinline__ void attend_block(WarpAcc<NH>& a, const QFrag<NH>& q, uint32_t kb, uint32_t vb,
                                             int valid, float sl2, int lane, uint32_t cols = 0xffffffffu) {
    constexpr int kSub = BS / 16;  // 16-token sub-blocks per block
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
    for (int sub = 0; sub < kSub; ++sub) {
        if (sub * 16 >= valid) break;  // warp-uniform: nothing valid left in this block
        // ---- S^T = K Q^T for tokens sub*16 .. sub*16+15 (M) x heads (N)
        float sc[NH][4];
#pragma unroll
        for (int n = 0; n < NH; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        {
            // A = K rows: matrices (tokens 0-7 | 8-15) x (dims lo | hi of the k-step)
            const int tok = sub * 16 + (mi & 1) * 8 + rr;
            float sc2[kIlp ? NH : 1][4];
            if constexpr (kIlp) {
#pragma unroll
                for (int n = 0; n < NH; ++n) sc2[n][0] = sc2[n][1] = sc2[n][2] = sc2[n][3] = 0.f;
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int chunk = 2 * ks + (mi >> 1);
                const int line = (chunk >> 3) * BS + tok;
                const uint32_t addr = kb + line * 128 + (((chunk & 7) ^ rr) << 4);
                uint32_t af[4];
                ldsm_x4(addr, af[0], af[1], af[2], af[3]);
#pragma unroll
                for (int n = 0; n < NH; ++n) {
                    if (kIlp && (ks & 1))
                        mma_16816<kBF16>(sc2[kIlp ? n : 0], af, q.b[n][ks][0], q.b[n][ks][1]);
                    else
                        mma_16816<kBF16>(sc[n], af, q.b[n][ks][0], q.b[n][ks][1]);
                }
            }
            if constexpr (kIlp) {
#pragma unroll
                for (int n = 0; n < NH; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[n][e] += sc2[n][e];
            }
        }
        // ---- scale (log2 domain), mask past the context, online softmax per head
        const int ta = sub * 16 + g, tb = ta + 8;  // tokens of sc[.][0..1] and sc[.][2..3]
        const bool va = ta < valid, vb_ = tb < valid;
        uint32_t ph[NH][2], pl[NH][2];
#pragma unroll
        for (int n = 0; n < NH; ++n) {
            const bool c0 = !kColMask || ((cols >> (2 * n)) & 1u), c1 = !kColMask || ((cols >> (2 * n + 1)) & 1u);
            sc[n][0] = va && c0 ? sc[n][0] * sl2 : -INFINITY;
            sc[n][1] = va && c1 ? sc[n][1] * sl2 : -INFINITY;
            sc[n][2] = vb_ && c0 ? sc[n][2] * sl2 : -INFINITY;
            sc[n][3] = vb_ && c1 ? sc[n][3] * sl2 : -INFINITY;
        }
        bool rescale = true;
        if constexpr (kIlp) {
            bool need = false;
#pragma unroll
            for (int n = 0; n < NH; ++n)
                need |= fmaxf(sc[n][0], sc[n][2]) > a.m[n][0] + kLazyMargin ||
                        fmaxf(sc[n][1], sc[n][3]) > a.m[n][1] + kLazyMargin;
            rescale = __any_sync(0xffffffffu, need);
        }
#pragma unroll
        for (int n = 0; n < NH; ++n) {
            float ms0, ms1;
            if (rescale) {
                float mx0 = fmaxf(sc[n][0], sc[n][2]), mx1 = fmaxf(sc[n][1], sc[n][3]);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                }
                const float mn0 = fmaxf(a.m[n][0], mx0), mn1 = fmaxf(a.m[n][1], mx1);
                const float al0 = mn0 == -INFINITY ? 1.f : exp2f(a.m[n][0] - mn0);
                const float al1 = mn1 == -INFINITY ? 1.f : exp2f(a.m[n][1] - mn1);
                ms0 = mn0 == -INFINITY ? 0.f : mn0;
                ms1 = mn1 == -INFINITY ? 0.f : mn1;
                a.m[n][0] = mn0;
                a.m[n][1] = mn1;
                a.l[n][0] *= al0;
                a.l[n][1] *= al1;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    a.o[mt][n][0] *= al0;
                    a.o[mt][n][1] *= al1;
                    a.o[mt][n][2] *= al0;
                    a.o[mt][n][3] *= al1;
                }
            } else {
                ms0 = a.m[n][0] == -INFINITY ? 0.f : a.m[n][0];  // a column with nothing yet: p = 0
                ms1 = a.m[n][1] == -INFINITY ? 0.f : a.m[n][1];
            }
            const float p0 = exp2f(sc[n][0] - ms0), p1 = exp2f(sc[n][1] - ms1);
            const float p2 = exp2f(sc[n][2] - ms0), p3 = exp2f(sc[n][3] - ms1);
            a.l[n][0] += p0 + p2;
            a.l[n][1] += p1 + p3;
            // P^T rows (tokens) x columns (heads) in the accumulator layout;
            // movmatrix.trans turns each 8x8 half into the B operand layout of
            // O^T = V^T P^T.  High part + residual.
            float r0, r1, r2, r3;
            const uint32_t h01 = pack2<kBF16>(p0, p1, r0, r1);
            const uint32_t h23 = pack2<kBF16>(p2, p3, r2, r3);
            const uint32_t l01 = pack2<kBF16>(p0 - r0, p1 - r1);
            const uint32_t l23 = pack2<kBF16>(p2 - r2, p3 - r3);
            ph[n][0] = movmatrix_trans(h01);
            ph[n][1] = movmatrix_trans(h23);
            pl[n][0] = movmatrix_trans(l01);
            pl[n][1] = movmatrix_trans(l23);
        }
        // ---- O^T += V^T P^T over the 16 tokens
        {
            // A = V^T: matrices (tokens 0-7 | 8-15) x (dims 16mt+0..7 | +8..15), transposed
            const int tok = sub * 16 + (mi >> 1) * 8 + rr;
            const bool tail = sub * 16 + 16 > valid;
            // V rows past the context may hold anything (even NaN): zero them
            // in the A fragments rather than rely on p == 0.
            const int tt = sub * 16 + 2 * t;
            const uint32_t keep0 = (tt < valid ? 0x0000ffffu : 0u) | (tt + 1 < valid ? 0xffff0000u : 0u);
            const uint32_t keep1 = (tt + 8 < valid ? 0x0000ffffu : 0u) | (tt + 9 < valid ? 0xffff0000u : 0u);
            uint32_t prev[4];  // kIlp: the previous m-tile's V fragment, for its residual MMAs
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const int chunk = 2 * mt + (mi & 1);
                const int line = (chunk >> 3) * BS + tok;
                const uint32_t addr = vb + line * 128 + (((chunk & 7) ^ rr) << 4);
                uint32_t af[4];
                ldsm_x4_trans(addr, af[0], af[1], af[2], af[3]);
                if (tail) {
                    af[0] &= keep0;
                    af[1] &= keep0;
                    af[2] &= keep1;
                    af[3] &= keep1;
                }
                if constexpr (kIlp) {
#pragma unroll
                    for (int n = 0; n < NH; ++n) mma_16816<kBF16>(a.o[mt][n], af, ph[n][0], ph[n][1]);
                    if (mt > 0) {
#pragma unroll
                        for (int n = 0; n < NH; ++n) mma_16816<kBF16>(a.o[mt - 1][n], prev, pl[n][0], pl[n][1]);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) prev[e] = af[e];
                } else {
#pragma unroll
                    for (int n = 0; n < NH; ++n) {
                        mma_16816<kBF16>(a.o[mt][n], af, ph[n][0], ph[n][1]);
                        mma_16816<kBF16>(a.o[mt][n], af, pl[n][0], pl[n][1]);
                    }
                }
            }
            if constexpr (kIlp) {
#pragma unroll
                for (int n = 0; n < NH; ++n) mma_16816<kBF16>(a.o[7][n], prev, pl[n][0], pl[n][1]);
            }
        }
    }
}

// Full per-head sums: the eight lanes g = 0..7 hold disjoint tokens.
template <int NH>
__device__ __forceinline__ void acc_finish(WarpAcc<NH>& a) {
#pragma unroll
    for (int n = 0; n < NH; ++n)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            a.l[n][0] += __shfl_xor_sync(0xffffffffu, a.l[n][0], o);
            a.l[n][1] += __shfl_xor_sync(0xffffffffu, a.l[n][1], o);
        }
}

// Write a warp's state for rows < `rows` into the merge buffer:
// red[warp][head][kRedStride], ml[warp][head][2] = (m, l).
template <int NH>
__device__ __forceinline__ void acc_to_smem(const WarpAcc<NH>& a, float* red, float* ml, int warp, int rows,
                                            int lane) {
    constexpr int HT = 8 * NH;
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int n = 0; n < NH; ++n) {
        const int ha = 8 * n + 2 * t, hb = ha + 1;
        float* ra = red + (warp * HT + ha) * kRedStride;
        float* rb = red + (warp * HT + hb) * kRedStride;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d0 = 16 * mt + g;
            if (ha < rows) {
                ra[d0] = a.o[mt][n][0];
                ra[d0 + 8] = a.o[mt][n][2];
            }
            if (hb < rows) {
                rb[d0] = a.o[mt][n][1];
                rb[d0 + 8] = a.o[mt][n][3];
            }
        }
        if (g == 0) {
            if (ha < rows) {
                ml[(warp * HT + ha) * 2] = a.m[n][0];
                ml[(warp * HT + ha) * 2 + 1] = a.l[n][0];
            }
            if (hb < rows) {
                ml[(warp * HT + hb) * 2] = a.m[n][1];
                ml[(warp * HT + hb) * 2 + 1] = a.l[n][1];
            }
        }
    }
}

}  // namespace pkv
