// Paged decode attention: plain fp64 CPU oracle.
//
// TEST INFRASTRUCTURE ONLY. This file is the reference the GPU library is
// checked against. Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg load it. It shares no code, header, table or helper with
// the CUDA library, and it is written for readability, not speed: scalar
// loops, no blocking, no fusion, no reordering beyond what the method states.
//
// What it computes (sources, by page title and section):
//  * "39 · PagedAttention" §1-§2: one new query per (sequence, head) is
//    compared with the key of every earlier token in logical order, a softmax
//    turns the scores into weights that sum to one, and the output is the
//    weighted sum of the value vectors. The paged version walks the logical
//    blocks in order, follows the block table to each physical block, scores
//    every key of the block, applies one softmax over all scores, and then
//    walks the blocks again to sum the weighted values. That is exactly
//    ordinary attention plus one indirection per block.
//  * "FlashAttention vs PagedAttention", "What does FlashAttention optimize?":
//    the score is q.k scaled by 1/sqrt(d); the caller passes that scale.
//  * "PagedAttention: The Cache Was Storing Nothing" §2.2: fixed-size blocks
//    of 16 or 32 tokens, one block table per request mapping logical block
//    i to a physical block id anywhere in the pool.
//  * "PagedAttention: The Cache Was Storing Nothing" §3.1: grouped-query
//    attention gives each group of query heads one key/value head. Query head
//    h reads kv head floor(h / g) with g = Hq / Hkv (consecutive groups).
//  * "39 · PagedAttention" §3: two partials (m1, l1), (m2, l2) combine as
//    m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m); the weighted value sums
//    are rescaled by the same factors.
//
// Storage convention (a reading: the pages do not fix a layout): each pool is
// [num_blocks][Hkv][block_size][D] row-major; token t of sequence b, kv head
// j lives at pool[table[b][t / bs]][j][t % bs][:]. Slots past the sequence
// length and table entries past ceil(L / bs) are never read.
//
// Element storage: dtype 0 = IEEE float32, dtype 1 = bfloat16 bit patterns
// (the upper 16 bits of a float32). Every stored value is widened exactly to
// double before any arithmetic.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// Widen one stored element to double (exact for both storage types).
double load_elem(const void* base, int64_t index, int dtype) {
    if (dtype == 0) {
        return static_cast<double>(static_cast<const float*>(base)[index]);
    }
    const uint16_t bits = static_cast<const uint16_t*>(base)[index];
    const uint32_t wide = static_cast<uint32_t>(bits) << 16;
    float f;
    std::memcpy(&f, &wide, sizeof(f));
    return static_cast<double>(f);
}

struct Problem {
    const void* q;
    const void* kpool;
    const void* vpool;
    const int32_t* table;
    int max_blocks;
    const int32_t* seq_lens;
    int B, Hq, Hkv, D, bs, num_blocks;
    double scale;
    int dtype;
};

// Offset of element 0 of token t (kv head j) of sequence b inside a pool, or
// -1 when the table entry does not name a block of the pool.
int64_t token_offset(const Problem& p, int b, int j, int64_t t) {
    const int64_t logical_block = t / p.bs;
    const int64_t slot = t % p.bs;
    const int32_t phys = p.table[static_cast<int64_t>(b) * p.max_blocks + logical_block];
    if (phys < 0 || phys >= p.num_blocks) return -1;
    return ((static_cast<int64_t>(phys) * p.Hkv + j) * p.bs + slot) * p.D;
}

// Pass 1 of the paged walk: the scores s_t = scale * sum_d q[d] k_t[d] for
// t in [t0, t1), visiting the logical blocks in order through the table.
// Returns false on a table entry outside the pool.
bool scores(const Problem& p, int b, int h, int64_t t0, int64_t t1, std::vector<double>& s) {
    const int g = p.Hq / p.Hkv;
    const int j = h / g;
    const int64_t qoff = (static_cast<int64_t>(b) * p.Hq + h) * p.D;
    s.assign(static_cast<size_t>(t1 - t0), 0.0);
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t koff = token_offset(p, b, j, t);
        if (koff < 0) return false;
        double dot = 0.0;
        for (int d = 0; d < p.D; ++d) {
            dot += load_elem(p.q, qoff + d, p.dtype) * load_elem(p.kpool, koff + d, p.dtype);
        }
        s[static_cast<size_t>(t - t0)] = p.scale * dot;
    }
    return true;
}

bool check_len(const Problem& p, int b) {
    const int32_t L = p.seq_lens[b];
    return L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_blocks) * p.bs;
}

// The three passes for one (sequence, query head): scores, one softmax over
// all of them, weighted value sum. Writes D doubles to out and, when w is not
// null, the L normalised weights to w.
bool attend_one(const Problem& p, int b, int h, double* out, double* w) {
    if (!check_len(p, b)) return false;
    const int64_t L = p.seq_lens[b];
    std::vector<double> s;
    if (!scores(p, b, h, 0, L, s)) return false;

    // Pass 2: softmax over all L scores (max subtracted for range only).
    double m = -std::numeric_limits<double>::infinity();
    for (double v : s) m = v > m ? v : m;
    double z = 0.0;
    for (double& v : s) {
        v = std::exp(v - m);
        z += v;
    }
    for (double& v : s) v /= z;
    if (w) {
        for (int64_t t = 0; t < L; ++t) w[t] = s[static_cast<size_t>(t)];
    }

    // Pass 3: walk the blocks again and add up the weighted values.
    const int j = h / (p.Hq / p.Hkv);
    for (int d = 0; d < p.D; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t voff = token_offset(p, b, j, t);
        if (voff < 0) return false;
        const double wt = s[static_cast<size_t>(t)];
        for (int d = 0; d < p.D; ++d) out[d] += wt * load_elem(p.vpool, voff + d, p.dtype);
    }
    return true;
}

bool valid_shape(int B, int Hq, int Hkv, int D, int bs, int num_blocks, int max_blocks, int dtype) {
    return B >= 0 && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 && D >= 1 && bs >= 1 &&
           num_blocks >= 1 && max_blocks >= 1 && (dtype == 0 || dtype == 1);
}

}  // namespace

extern "C" {

// Number of fixed-size blocks a sequence of L tokens occupies: ceil(L / bs)
// ("PagedAttention: The Cache Was Storing Nothing" §2.1: 200 tokens in
// 16-token blocks take 13 blocks).
int64_t oracle_num_blocks(int64_t L, int64_t bs) {
    if (L <= 0 || bs <= 0) return 0;
    return (L + bs - 1) / bs;
}

// Cached elements per token: 2 (keys and values) x heads x head_dim x layers
// ("PagedAttention: The Cache Was Storing Nothing" §3).
int64_t oracle_kv_elems_per_token(int64_t kv_heads, int64_t head_dim, int64_t layers) {
    return 2 * kv_heads * head_dim * layers;
}

// Bytes of algorithmic HBM traffic of one decode call: every K and V element
// of every attended token once, one table entry per attended block, the
// queries, the sequence lengths and the output. Pads inside a partly filled
// last block are not counted.
int64_t oracle_decode_bytes(const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs,
                            int kv_elem_bytes, int out_elem_bytes) {
    int64_t total = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t L = seq_lens[b];
        total += oracle_kv_elems_per_token(Hkv, D, 1) * L * kv_elem_bytes;
        total += 4 * oracle_num_blocks(L, bs);
    }
    total += static_cast<int64_t>(B) * Hq * D * kv_elem_bytes;  // queries
    total += 4 * static_cast<int64_t>(B);                       // sequence lengths
    total += static_cast<int64_t>(B) * Hq * D * out_elem_bytes; // output
    return total;
}

// Decode attention for all (b, h), or for the npairs listed (b, h) pairs
// when pairs is not null (pairs[2i] = b, pairs[2i+1] = h; output row i).
// out holds B*Hq*D (or npairs*D) doubles. Returns 0 on success, -1 on a bad
// shape, -2 on a sequence length outside [1, max_blocks*bs], -3 on a table
// entry outside the pool.
int oracle_decode(const void* q, const void* kpool, const void* vpool, const int32_t* table,
                  int max_blocks, const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs,
                  int num_blocks, float scale, int dtype, double* out, const int32_t* pairs,
                  int npairs, int nthreads) {
    if (!valid_shape(B, Hq, Hkv, D, bs, num_blocks, max_blocks, dtype)) return -1;
    const Problem p{q, kpool, vpool, table, max_blocks, seq_lens, B, Hq, Hkv, D, bs, num_blocks,
                    static_cast<double>(scale), dtype};
    const int64_t n = pairs ? npairs : static_cast<int64_t>(B) * Hq;
    for (int64_t i = 0; i < n; ++i) {
        const int b = pairs ? pairs[2 * i] : static_cast<int>(i / Hq);
        const int h = pairs ? pairs[2 * i + 1] : static_cast<int>(i % Hq);
        if (b < 0 || b >= B || h < 0 || h >= Hq) return -1;
        if (!check_len(p, b)) return -2;
    }
    if (nthreads < 1) nthreads = 1;
    std::vector<int> status(static_cast<size_t>(nthreads), 0);
    auto work = [&](int tid) {
        for (int64_t i = tid; i < n; i += nthreads) {
            const int b = pairs ? pairs[2 * i] : static_cast<int>(i / Hq);
            const int h = pairs ? pairs[2 * i + 1] : static_cast<int>(i % Hq);
            if (!attend_one(p, b, h, out + i * D, nullptr)) {
                status[static_cast<size_t>(tid)] = -3;
                return;
            }
        }
    };
    if (nthreads == 1) {
        work(0);
    } else {
        std::vector<std::thread> pool;
        for (int tid = 0; tid < nthreads; ++tid) pool.emplace_back(work, tid);
        for (auto& th : pool) th.join();
    }
    for (int st : status) {
        if (st != 0) return st;
    }
    return 0;
}

// The normalised softmax weights w_t (t < L) of one (b, h): pass 2 exposed.
int oracle_weights(const void* q, const void* kpool, const int32_t* table, int max_blocks,
                   const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs, int num_blocks,
                   float scale, int dtype, int b, int h, double* w) {
    if (!valid_shape(B, Hq, Hkv, D, bs, num_blocks, max_blocks, dtype)) return -1;
    if (b < 0 || b >= B || h < 0 || h >= Hq) return -1;
    const Problem p{q, kpool, kpool, table, max_blocks, seq_lens, B, Hq, Hkv, D, bs, num_blocks,
                    static_cast<double>(scale), dtype};
    if (!check_len(p, b)) return -2;
    std::vector<double> o(static_cast<size_t>(D));
    return attend_one(p, b, h, o.data(), w) ? 0 : -3;
}

// One partial over the token range [t0, t1) of (b, h): m = max score,
// l = sum e^(s-m), acc[d] = sum e^(s-m) v[d]. An empty range gives
// m = -inf, l = 0, acc = 0.
int oracle_partial(const void* q, const void* kpool, const void* vpool, const int32_t* table,
                   int max_blocks, const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs,
                   int num_blocks, float scale, int dtype, int b, int h, int64_t t0, int64_t t1,
                   double* m_out, double* l_out, double* acc) {
    if (!valid_shape(B, Hq, Hkv, D, bs, num_blocks, max_blocks, dtype)) return -1;
    if (b < 0 || b >= B || h < 0 || h >= Hq) return -1;
    const Problem p{q, kpool, vpool, table, max_blocks, seq_lens, B, Hq, Hkv, D, bs, num_blocks,
                    static_cast<double>(scale), dtype};
    if (!check_len(p, b)) return -2;
    if (t0 < 0 || t1 > seq_lens[b] || t0 > t1) return -1;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    *m_out = -std::numeric_limits<double>::infinity();
    *l_out = 0.0;
    if (t0 == t1) return 0;
    std::vector<double> s;
    if (!scores(p, b, h, t0, t1, s)) return -3;
    double m = -std::numeric_limits<double>::infinity();
    for (double v : s) m = v > m ? v : m;
    double l = 0.0;
    const int j = h / (Hq / Hkv);
    for (int64_t t = t0; t < t1; ++t) {
        const double e = std::exp(s[static_cast<size_t>(t - t0)] - m);
        l += e;
        const int64_t voff = token_offset(p, b, j, t);
        if (voff < 0) return -3;
        for (int d = 0; d < D; ++d) acc[d] += e * load_elem(vpool, voff + d, dtype);
    }
    *m_out = m;
    *l_out = l;
    return 0;
}

// Combine n partials in order with the two-partial rule, then normalise:
// out[d] = acc[d] / l. m, l have n entries, acc is n x D.
int oracle_merge(int n, const double* m, const double* l, const double* acc, int D, double* out) {
    if (n < 1 || D < 1) return -1;
    double mm = m[0];
    double ll = l[0];
    std::vector<double> aa(acc, acc + D);
    for (int i = 1; i < n; ++i) {
        const double mn = m[i] > mm ? m[i] : mm;
        if (mn == -std::numeric_limits<double>::infinity()) continue;  // both empty
        const double f_old = std::exp(mm - mn);
        const double f_new = std::exp(m[i] - mn);
        ll = ll * f_old + l[i] * f_new;
        for (int d = 0; d < D; ++d) aa[static_cast<size_t>(d)] = aa[static_cast<size_t>(d)] * f_old + acc[static_cast<int64_t>(i) * D + d] * f_new;
        mm = mn;
    }
    if (!(ll > 0.0)) return -2;
    for (int d = 0; d < D; ++d) out[d] = aa[static_cast<size_t>(d)] / ll;
    return 0;
}

// KV append: write each sequence's new key/value rows into slot
// cache_len % bs of physical block table[b][cache_len / bs], as raw bytes
// (a bit-exact copy). k_new/v_new are [B][Hkv][D]. Returns -3 on a table
// entry outside the pool, -2 on a cache length outside [0, max_blocks*bs).
int oracle_append(const void* k_new, const void* v_new, void* kpool, void* vpool,
                  const int32_t* table, int max_blocks, const int32_t* cache_lens, int B, int Hkv,
                  int D, int bs, int num_blocks, int elem_bytes) {
    if (B < 0 || Hkv < 1 || D < 1 || bs < 1 || num_blocks < 1 || max_blocks < 1) return -1;
    if (elem_bytes != 2 && elem_bytes != 4) return -1;
    for (int b = 0; b < B; ++b) {
        const int64_t pos = cache_lens[b];
        if (pos < 0 || pos >= static_cast<int64_t>(max_blocks) * bs) return -2;
        const int32_t phys = table[static_cast<int64_t>(b) * max_blocks + pos / bs];
        if (phys < 0 || phys >= num_blocks) return -3;
        for (int j = 0; j < Hkv; ++j) {
            const int64_t dst = ((static_cast<int64_t>(phys) * Hkv + j) * bs + pos % bs) * D;
            const int64_t src = (static_cast<int64_t>(b) * Hkv + j) * D;
            std::memcpy(static_cast<char*>(kpool) + dst * elem_bytes,
                        static_cast<const char*>(k_new) + src * elem_bytes,
                        static_cast<size_t>(D) * elem_bytes);
            std::memcpy(static_cast<char*>(vpool) + dst * elem_bytes,
                        static_cast<const char*>(v_new) + src * elem_bytes,
                        static_cast<size_t>(D) * elem_bytes);
        }
    }
    return 0;
}

// Block copies for copy-on-write ("PagedAttention: The Cache Was Storing
// Nothing" §2.3: a shared block is copied only when a sequence diverges and
// writes into it). Copies whole blocks (every kv head, every slot) of both
// pools, pair i copying block src[i] to block dst[i], in order. block_bytes is
// the size of one block of one pool. Returns -3 on an id outside the pool.
int oracle_copy_blocks(void* kpool, void* vpool, const int32_t* src, const int32_t* dst, int n,
                       int num_blocks, int64_t block_bytes) {
    if (n < 0 || num_blocks < 1 || block_bytes < 1) return -1;
    for (int i = 0; i < n; ++i) {
        if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) return -3;
        char* k = static_cast<char*>(kpool);
        char* v = static_cast<char*>(vpool);
        std::memmove(k + dst[i] * block_bytes, k + src[i] * block_bytes, static_cast<size_t>(block_bytes));
        std::memmove(v + dst[i] * block_bytes, v + src[i] * block_bytes, static_cast<size_t>(block_bytes));
    }
    return 0;
}

// PagedEviction page scores (Pith review of arXiv 2509.04377, "Core claim" and
// "What carries the argument"): a token's importance is S = ||V||_2 / ||K||_2
// of its cached value and key, a page's importance is the mean of S over its
// tokens, and when the most recent page has just filled (L % bs == 0) the page
// with the lowest mean is the one to evict. Readings: K and V of a token are
// its vectors over all kv heads together (one block table serves every head,
// so a page is evicted for all heads at once); ||K|| = 0 gives S = +inf; every
// full page is a candidate; ties go to the lowest logical page.
// scores[b * max_blocks + p] receives the mean over the valid tokens of
// logical page p < ceil(L_b / bs) (other entries untouched); victims[b] the
// page to evict, or -1 when L_b % bs != 0. Returns -2 / -3 on a bad length /
// table entry.
int oracle_page_scores(const void* kpool, const void* vpool, const int32_t* table, int max_blocks,
                       const int32_t* seq_lens, int B, int Hkv, int D, int bs, int num_blocks,
                       int dtype, double* scores, int32_t* victims) {
    if (B < 0 || Hkv < 1 || D < 1 || bs < 1 || num_blocks < 1 || max_blocks < 1) return -1;
    if (dtype != 0 && dtype != 1) return -1;
    for (int b = 0; b < B; ++b) {
        const int64_t L = seq_lens[b];
        if (L < 1 || L > static_cast<int64_t>(max_blocks) * bs) return -2;
        const int64_t nb = (L + bs - 1) / bs;
        for (int64_t p = 0; p < nb; ++p) {
            const int32_t phys = table[static_cast<int64_t>(b) * max_blocks + p];
            if (phys < 0 || phys >= num_blocks) return -3;
            const int64_t n = std::min<int64_t>(bs, L - p * bs);
            double sum = 0.0;
            for (int64_t slot = 0; slot < n; ++slot) {
                double kk = 0.0, vv = 0.0;
                for (int j = 0; j < Hkv; ++j) {
                    const int64_t off = ((static_cast<int64_t>(phys) * Hkv + j) * bs + slot) * D;
                    for (int d = 0; d < D; ++d) {
                        const double k = load_elem(kpool, off + d, dtype);
                        const double v = load_elem(vpool, off + d, dtype);
                        kk += k * k;
                        vv += v * v;
                    }
                }
                sum += kk > 0.0 ? std::sqrt(vv) / std::sqrt(kk)
                                : std::numeric_limits<double>::infinity();
            }
            scores[static_cast<int64_t>(b) * max_blocks + p] = sum / static_cast<double>(n);
        }
        int32_t victim = -1;
        if (L % bs == 0) {
            for (int64_t p = 0; p < nb; ++p) {
                const double sp = scores[static_cast<int64_t>(b) * max_blocks + p];
                if (victim < 0 || sp < scores[static_cast<int64_t>(b) * max_blocks + victim])
                    victim = static_cast<int32_t>(p);
            }
        }
        victims[b] = victim;
    }
    return 0;
}

// Paged multi-query attention (chunked prefill, speculative verification):
// the n_b = q_start[b+1] - q_start[b] newest tokens of sequence b are queries;
// query i sits at position pos = L_b - n_b + i and attends, causally, to the
// tokens t <= pos through the block table ("FlashAttention vs PagedAttention",
// "How prefill and decode change the diagnosis": prefill processes many prompt
// positions at once; decode is the case n_b = 1). q and out are
// [q_start[B]][Hq][D]; each row is the three-pass attention of decode over
// L = pos + 1 tokens. Returns -2 on n_b < 1 or n_b > L_b.
int oracle_prefill(const void* q, const void* kpool, const void* vpool, const int32_t* table,
                   int max_blocks, const int32_t* seq_lens, const int32_t* q_start, int B, int Hq,
                   int Hkv, int D, int bs, int num_blocks, float scale, int dtype, double* out,
                   int nthreads) {
    if (!valid_shape(B, Hq, Hkv, D, bs, num_blocks, max_blocks, dtype)) return -1;
    for (int b = 0; b < B; ++b) {
        const int32_t n = q_start[b + 1] - q_start[b];
        if (n < 1 || n > seq_lens[b] || static_cast<int64_t>(seq_lens[b]) > static_cast<int64_t>(max_blocks) * bs)
            return -2;
    }
    const int64_t rows = q_start[B];
    // One "sequence" per query row: the same table row, length pos + 1.
    std::vector<int32_t> row_seq(static_cast<size_t>(rows)), row_len(static_cast<size_t>(rows));
    for (int b = 0; b < B; ++b) {
        const int32_t n = q_start[b + 1] - q_start[b];
        for (int32_t i = 0; i < n; ++i) {
            row_seq[static_cast<size_t>(q_start[b] + i)] = b;
            row_len[static_cast<size_t>(q_start[b] + i)] = seq_lens[b] - n + i + 1;
        }
    }
    if (nthreads < 1) nthreads = 1;
    std::vector<int> status(static_cast<size_t>(nthreads), 0);
    auto work = [&](int tid) {
        for (int64_t i = tid; i < rows * Hq; i += nthreads) {
            const int64_t r = i / Hq;
            const int h = static_cast<int>(i % Hq);
            const int b = row_seq[static_cast<size_t>(r)];
            const int32_t len = row_len[static_cast<size_t>(r)];
            // The query row r becomes "sequence 0" of a one-sequence problem over
            // sequence b's table with length len; q offsets index row r directly.
            const Problem p{static_cast<const char*>(q) + (r * Hq) * D * (dtype == 0 ? 4 : 2),
                            kpool, vpool, table + static_cast<int64_t>(b) * max_blocks, max_blocks,
                            &len, 1, Hq, Hkv, D, bs, num_blocks, static_cast<double>(scale), dtype};
            if (!attend_one(p, 0, h, out + i * D, nullptr)) {
                status[static_cast<size_t>(tid)] = -3;
                return;
            }
        }
    };
    if (nthreads == 1) {
        work(0);
    } else {
        std::vector<std::thread> pool;
        for (int tid = 0; tid < nthreads; ++tid) pool.emplace_back(work, tid);
        for (auto& th : pool) th.join();
    }
    for (int st : status)
        if (st != 0) return st;
    return 0;
}

}  // extern "C"
