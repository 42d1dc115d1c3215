/*
 * pkv_oracle.c -- the oracle for the paged KV cache decode path.
 *
 * TEST INFRASTRUCTURE.  This is a plain, slow, fp64 CPU statement of what the
 * path computes, written to be checked by eye against the pages it follows.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header or table with the CUDA library, and it
 * includes nothing from it.
 *
 * Sources (web pages on paged KV caches; page title, then section):
 *   [vLLM]   tonho.wtf encyclopedia entry "vllm", sections "como funciona"
 *            (fixed-size KV blocks, block table mapping logical to physical
 *            blocks, slots filled left to right, attention rewritten block
 *            by block over non-adjacent blocks; sharing with refcounts and a
 *            copy of the last shared block on write) and "o que isso custou"
 *            (the three kernels: block write, fused paged read + attention,
 *            batched block copy).
 *   [KVCM]   techtrendfeed "KV Cache Administration: PagedAttention &
 *            RadixAttention", "How PagedAttention Works", steps 1-4, and
 *            "Why this modified LLM serving" (paging changes neither the
 *            attention algorithm nor the model's outputs).
 *   [aitalk] aitalk.it "PagedAttention e RadixAttention", section
 *            "PagedAttention: la memoria come un sistema operativo" (the
 *            same four steps; outputs unchanged).
 *   [Zipage] gist.science summary of "Zipage: Maintain High Request
 *            Concurrency for LLM Reasoning through Compressed
 *            PagedAttention", technical summary, section 2 (a request holds
 *            at most N_max blocks; kept tokens are rewritten into new target
 *            blocks, the first N_max - 1 of them, leaving shared blocks
 *            intact).
 *
 * Readings where the pages leave a point open:
 *   - cache layout: k_cache and v_cache are [num_blocks][num_kv_heads]
 *     [block_size][head_dim], row-major; token position t of a sequence lives
 *     in logical block t / block_size at offset t % block_size;
 *   - a flat slot is physical_block * block_size + offset; a negative slot is
 *     a padding token and is skipped;
 *   - context_lens[s] counts every token attended, including the one
 *     appended this step;
 *   - query head h reads KV head h / (num_q_heads / num_kv_heads);
 *   - a context of length 0 gives an output of zeros;
 *   - the attention itself is the plain definition
 *       out = sum_t softmax_t(scale * q . K_t) V_t
 *     over the context gathered in logical order; the maximum score is
 *     subtracted before exp, which changes nothing mathematically;
 *   - split-K (sequence partitions merged through their log-sum-exp) is the
 *     same quantity regrouped; oracle_decode with partition_size > 0 states
 *     it so that the regrouping can be checked against the plain form.
 *
 * Element types: 0 = bfloat16, 1 = IEEE binary16; both held as raw 16-bit
 * patterns and decoded exactly into double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_FP16 1

/* Exact decode of one 16-bit storage element into double. */
double oracle_elem_to_f64(uint16_t bits, int dtype) {
    int sign = (bits >> 15) & 1;
    double mag;
    if (dtype == ORC_BF16) {
        /* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits */
        int e = (bits >> 7) & 0xFF;
        int f = bits & 0x7F;
        if (e == 0xFF)
            mag = f ? NAN : INFINITY;
        else if (e == 0)
            mag = ldexp((double)f, -126 - 7);
        else
            mag = ldexp((double)(128 + f), e - 127 - 7);
    } else {
        /* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits */
        int e = (bits >> 10) & 0x1F;
        int f = bits & 0x3FF;
        if (e == 0x1F)
            mag = f ? NAN : INFINITY;
        else if (e == 0)
            mag = ldexp((double)f, -14 - 10);
        else
            mag = ldexp((double)(1024 + f), e - 15 - 10);
    }
    if (isnan(mag)) return mag;
    return sign ? -mag : mag;
}

void oracle_to_f64(const uint16_t* in, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_elem_to_f64(in[i], dtype);
}

/*
 * Block write [vLLM "o que isso custou"; "como funciona"]: the new token's
 * K and V rows go to the slot its sequence's block table gives.
 * k, v: [num_tokens][num_kv_heads][head_dim]; slot_mapping: [num_tokens].
 * Returns the number of tokens whose slot lies outside the pool (skipped).
 */
int64_t oracle_append(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping, int64_t num_tokens,
                      uint16_t* k_cache, uint16_t* v_cache, int64_t num_blocks, int num_kv_heads, int block_size,
                      int head_dim) {
    int64_t bad = 0;
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue; /* padding token */
        if (slot >= num_blocks * block_size) {
            ++bad;
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_dim;
            int64_t src = t * row + (int64_t)h * head_dim;
            memcpy(k_cache + dst, k + src, sizeof(uint16_t) * (size_t)head_dim);
            memcpy(v_cache + dst, v + src, sizeof(uint16_t) * (size_t)head_dim);
        }
    }
    return bad;
}

/*
 * Copy-on-write block copy [vLLM "como funciona": a write into the last
 * shared block copies that block and only it; "o que isso custou": batched
 * block copy].  pairs: [num_pairs][2] = (src, dst) physical block ids; each
 * copies every KV head and slot of the block, K and V.  Returns the number
 * of pairs with an id outside the pool (skipped).
 */
int64_t oracle_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int64_t* pairs, int64_t num_pairs,
                           int64_t num_blocks, int num_kv_heads, int block_size, int head_dim) {
    int64_t bad = 0;
    int64_t blk = (int64_t)num_kv_heads * block_size * head_dim;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++bad;
            continue;
        }
        memcpy(k_cache + dst * blk, k_cache + src * blk, sizeof(uint16_t) * (size_t)blk);
        memcpy(v_cache + dst * blk, v_cache + src * blk, sizeof(uint16_t) * (size_t)blk);
    }
    return bad;
}

/*
 * Swap of whole blocks between two pools [vLLM "como funciona": the blocks
 * of an evicted sequence go to CPU RAM and are brought back]: block src of
 * the source pool becomes block dst of the destination pool, every KV head
 * and slot, K and V.  Returns the number of pairs with an id outside its
 * pool (skipped).
 */
int64_t oracle_swap_blocks(const uint16_t* src_k, const uint16_t* src_v, int64_t src_num_blocks, uint16_t* dst_k,
                           uint16_t* dst_v, int64_t dst_num_blocks, const int64_t* pairs, int64_t num_pairs,
                           int num_kv_heads, int block_size, int head_dim) {
    int64_t bad = 0;
    int64_t blk = (int64_t)num_kv_heads * block_size * head_dim;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
            ++bad;
            continue;
        }
        memcpy(dst_k + dst * blk, src_k + src * blk, sizeof(uint16_t) * (size_t)blk);
        memcpy(dst_v + dst * blk, src_v + src * blk, sizeof(uint16_t) * (size_t)blk);
    }
    return bad;
}

/*
 * Token-level compaction [Zipage, Compressed PagedAttention: the kept tokens
 * of a request are rewritten into new target blocks]: the K and V rows of
 * every KV head move from slot src_slots[i] to slot dst_slots[i].  Negative
 * slots are skipped; slots outside the pool are counted and skipped.
 */
int64_t oracle_compact(uint16_t* k_cache, uint16_t* v_cache, const int64_t* src_slots, const int64_t* dst_slots,
                       int64_t num_tokens, int64_t num_blocks, int num_kv_heads, int block_size, int head_dim) {
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t a = src_slots[t], b = dst_slots[t];
        if (a < 0 || b < 0) continue;
        if (a >= num_blocks * block_size || b >= num_blocks * block_size) {
            ++bad;
            continue;
        }
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t from = (((a / block_size) * num_kv_heads + h) * block_size + a % block_size) * head_dim;
            int64_t to = (((b / block_size) * num_kv_heads + h) * block_size + b % block_size) * head_dim;
            memcpy(k_cache + to, k_cache + from, sizeof(uint16_t) * (size_t)head_dim);
            memcpy(v_cache + to, v_cache + from, sizeof(uint16_t) * (size_t)head_dim);
        }
    }
    return bad;
}

typedef struct {
    int dtype;
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int num_seqs, num_q_heads, num_kv_heads, block_size, head_dim;
    int64_t num_blocks;
    double scale;
    int partition_size; /* 0: plain form; > 0: partitioned form */
    double* out;
    const int32_t* select; /* optional [nsel][2] (seq, q head) pairs */
    int64_t nsel;
    int32_t* status; /* per sequence: 0 ok, 1 bad metadata */
    /* work distribution */
    int64_t next;
    pthread_mutex_t lock;
} dec_job;

static int head_selected(const dec_job* j, int s, int h) {
    if (!j->select) return 1;
    for (int64_t i = 0; i < j->nsel; ++i)
        if (j->select[2 * i] == s && j->select[2 * i + 1] == h) return 1;
    return 0;
}

/*
 * Plain softmax attention of one query row over a contiguous context
 * K, V: [len][head_dim] in double.  Writes out[head_dim]; also returns the
 * row's log-sum-exp of the scaled scores through *lse (used by the
 * partitioned form).
 */
static void attend_rows(const double* qrow, const double* K, const double* V, int64_t len, int head_dim,
                        double scale, double* z, double* out, double* lse) {
    double zmax = -INFINITY;
    for (int64_t t = 0; t < len; ++t) {
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d) acc += qrow[d] * K[t * head_dim + d];
        z[t] = scale * acc;
        if (z[t] > zmax) zmax = z[t];
    }
    double denom = 0.0;
    for (int64_t t = 0; t < len; ++t) {
        z[t] = exp(z[t] - zmax);
        denom += z[t];
    }
    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < len; ++t)
        for (int d = 0; d < head_dim; ++d) out[d] += z[t] * V[t * head_dim + d];
    for (int d = 0; d < head_dim; ++d) out[d] /= denom;
    *lse = zmax + log(denom);
}

/*
 * One (sequence, KV head) group: gather the sequence's K and V rows of this
 * KV head in logical order through the block table [vLLM "como funciona";
 * KVCM step 2], then attend every selected query head of the group.
 */
static void decode_group(dec_job* j, int s, int kvh, double* K, double* V, double* z) {
    const int D = j->head_dim, bs = j->block_size;
    const int G = j->num_q_heads / j->num_kv_heads;
    int64_t L = j->context_lens[s];
    int ok = L >= 0 && L <= (int64_t)j->max_blocks_per_seq * bs;
    for (int64_t t = 0; ok && t < L; ++t) {
        int64_t pb = j->block_tables[(int64_t)s * j->max_blocks_per_seq + t / bs];
        if (pb < 0 || pb >= j->num_blocks) {
            ok = 0;
            break;
        }
        const uint16_t* kr = j->k_cache + ((pb * j->num_kv_heads + kvh) * bs + t % bs) * D;
        const uint16_t* vr = j->v_cache + ((pb * j->num_kv_heads + kvh) * bs + t % bs) * D;
        for (int d = 0; d < D; ++d) {
            K[t * D + d] = oracle_elem_to_f64(kr[d], j->dtype);
            V[t * D + d] = oracle_elem_to_f64(vr[d], j->dtype);
        }
    }
    double qrow[1024], part[1024];
    for (int g = 0; g < G; ++g) {
        int h = kvh * G + g;
        if (!head_selected(j, s, h)) continue;
        double* o = j->out + ((int64_t)s * j->num_q_heads + h) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (!ok) {
            pthread_mutex_lock(&j->lock);
            j->status[s] = 1;
            pthread_mutex_unlock(&j->lock);
            continue;
        }
        if (L == 0) continue;
        for (int d = 0; d < D; ++d)
            qrow[d] = oracle_elem_to_f64(j->q[((int64_t)s * j->num_q_heads + h) * D + d], j->dtype);
        double lse;
        if (j->partition_size <= 0) {
            attend_rows(qrow, K, V, L, D, j->scale, z, o, &lse);
        } else {
            /*
             * Partitioned form: attend each run of partition_size tokens on
             * its own, keep (o_p, lse_p), then merge with weights
             * exp(lse_p - LSE), LSE = log sum_p exp(lse_p).
             */
            int64_t P = j->partition_size;
            int64_t np = (L + P - 1) / P;
            double* lses = (double*)malloc(sizeof(double) * (size_t)np);
            double* outs = (double*)malloc(sizeof(double) * (size_t)(np * D));
            double lmax = -INFINITY;
            for (int64_t p = 0; p < np; ++p) {
                int64_t b = p * P, e = b + P < L ? b + P : L;
                attend_rows(qrow, K + b * D, V + b * D, e - b, D, j->scale, z, outs + p * D, &lses[p]);
                if (lses[p] > lmax) lmax = lses[p];
            }
            double sum = 0.0;
            for (int64_t p = 0; p < np; ++p) sum += exp(lses[p] - lmax);
            double LSE = lmax + log(sum);
            for (int64_t p = 0; p < np; ++p) {
                double w = exp(lses[p] - LSE);
                for (int d = 0; d < D; ++d) part[d] = w * outs[p * D + d];
                for (int d = 0; d < D; ++d) o[d] += part[d];
            }
            free(lses);
            free(outs);
        }
    }
}

static void* dec_worker(void* arg) {
    dec_job* j = (dec_job*)arg;
    int64_t maxL = (int64_t)j->max_blocks_per_seq * j->block_size;
    double* K = (double*)malloc(sizeof(double) * (size_t)(maxL * j->head_dim + 1));
    double* V = (double*)malloc(sizeof(double) * (size_t)(maxL * j->head_dim + 1));
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxL + 1));
    int64_t total = (int64_t)j->num_seqs * j->num_kv_heads;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int64_t w = j->next++;
        pthread_mutex_unlock(&j->lock);
        if (w >= total) break;
        int s = (int)(w / j->num_kv_heads), kvh = (int)(w % j->num_kv_heads);
        /* skip groups with no selected head */
        int G = j->num_q_heads / j->num_kv_heads, any = 0;
        for (int g = 0; g < G && !any; ++g) any = head_selected(j, s, kvh * G + g);
        if (any) decode_group(j, s, kvh, K, V, z);
    }
    free(K);
    free(V);
    free(z);
    return 0;
}

/*
 * Decode attention [vLLM "como funciona"; KVCM "Why this modified LLM
 * serving"]: for every sequence s and query head h (or only the (s, h) pairs
 * listed in `select`), out[s][h][:] = softmax(scale * q[s][h] . K_s) V_s in
 * double, K_s and V_s gathered through block_tables.
 *
 * q: [num_seqs][num_q_heads][head_dim]; caches as in the file header;
 * block_tables: [num_seqs][max_blocks_per_seq]; out: [num_seqs]
 * [num_q_heads][head_dim] double.  status[s] is set to 1 (and that
 * sequence's selected outputs are zero) when its context length or one of
 * its block ids lies outside the pool.  partition_size > 0 selects the
 * partitioned (split-K) form.  Returns -1 on a bad argument, else the number
 * of sequences with bad metadata.
 */
int64_t oracle_decode(int dtype, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                      int num_seqs, int num_q_heads, int num_kv_heads, int block_size, int head_dim,
                      int64_t num_blocks, double scale, int partition_size, double* out,
                      const int32_t* select, int64_t nsel, int32_t* status, int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads || head_dim <= 0 || head_dim > 1024 ||
        block_size <= 0 || (dtype != ORC_BF16 && dtype != ORC_FP16))
        return -1;
    dec_job j;
    j.dtype = dtype;
    j.q = q;
    j.k_cache = k_cache;
    j.v_cache = v_cache;
    j.block_tables = block_tables;
    j.max_blocks_per_seq = max_blocks_per_seq;
    j.context_lens = context_lens;
    j.num_seqs = num_seqs;
    j.num_q_heads = num_q_heads;
    j.num_kv_heads = num_kv_heads;
    j.block_size = block_size;
    j.head_dim = head_dim;
    j.num_blocks = num_blocks;
    j.scale = scale;
    j.partition_size = partition_size;
    j.out = out;
    j.select = select;
    j.nsel = nsel;
    j.status = status;
    j.next = 0;
    pthread_mutex_init(&j.lock, 0);
    for (int s = 0; s < num_seqs; ++s) status[s] = 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    pthread_t th[512];
    int started[512] = {0};
    for (int t = 1; t < nthreads; ++t) started[t] = pthread_create(&th[t], 0, dec_worker, &j) == 0;
    dec_worker(&j);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) pthread_join(th[t], 0);
    pthread_mutex_destroy(&j.lock);
    int64_t bad = 0;
    for (int s = 0; s < num_seqs; ++s) bad += status[s] != 0;
    return bad;
}
