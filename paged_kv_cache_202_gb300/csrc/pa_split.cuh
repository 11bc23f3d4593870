// Split paged decode attention for bf16 KV pools.
//
// Work decomposition. Every (sequence b, kv unit u) pair is a "segment": the
// ordered list of the nb_b = ceil(L_b / BS) logical blocks ("pages") the
// query heads of unit u attend over ("39 · PagedAttention" §2: walk the
// logical blocks in order through the block table). A kv unit is one kv head
// and one slice of at most 16 of the query heads that share it
// ("PagedAttention: The Cache Was Storing Nothing" §3.1). All segments are
// concatenated into one stream of P pages and cut into contiguous ranges: one
// equal static range per resident warp of a persistent grid for most of the
// stream, then small pieces claimed dynamically by whichever warp is free, so
// the work is balanced whatever the length mix and whatever the speed of each
// SM. A range produces a finished output row for every segment it covers
// completely, and a partial (m, l, acc) for at most two segments cut by its
// boundaries. The merge kernel combines those with the two-partial rule of
// "39 · PagedAttention" §3.
// Splitting along the sequence is what keeps the chip busy when a decode has
// only one query row ("PagedAttention: The Cache Was Storing Nothing", "Where
// this goes next").
//
// Data movement. Each warp runs its own pipeline of `stages` shared-memory
// stages. One page of one kv head is a contiguous [BS][D] bf16 block in the
// pool; lane 0 reads its physical id from the block table (one indirection
// per page) and moves the K and V pages into a stage with tiled bulk tensor
// copies in 64-column boxes with the 128-byte swizzle, completing on the
// stage's mbarrier. The first page of a segment also brings the segment's
// query rows. Consumers read the stage with ldmatrix / 128-bit loads that the
// swizzle keeps free of bank conflicts.
//
// Arithmetic. Scores are kept in the log2 domain (s * scale * log2 e) so the
// exponentials are single ex2 instructions. Slots past a sequence's length
// are excluded by predicate, never multiplied by zero: their scores become
// -inf and, on the tensor-core path, their V elements are replaced by zero
// before the product so that NaN or garbage there cannot leak into a sum.
//   * FMA path (one query head per kv head): lane = (d-half, token); each
//     lane dots half a key with half the query, a shuffle joins the halves.
//   * MMA path (a GQA group of g >= 2 query heads): S^T[16 tok x 8 heads] =
//     K[16 x D] Q^T via bf16 m16n8k16 tiles with fp32 accumulation; the
//     probabilities are split into a bf16 pair hi + lo (about 16 significant
//     bits together), transposed in registers (movmatrix) and fed to
//     O^T[D x 8 heads] += V^T[D x 16 tok] (P_hi^T + P_lo^T).
#pragma once

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace split {

struct Cursor {
    int b, u, p, nb;  // sequence, kv unit, logical page, pages of sequence b
};

__device__ __forceinline__ int seq_pages(const int* pre, int b) { return pre[b + 1] - pre[b]; }

__device__ __forceinline__ void advance(Cursor& c, const int* pre, int U, int B) {
    if (++c.p == c.nb) {
        c.p = 0;
        if (++c.u == U) {
            c.u = 0;
            do {
                ++c.b;
            } while (c.b < B && seq_pages(pre, c.b) == 0);
            c.nb = (c.b < B) ? seq_pages(pre, c.b) : 0;
        }
    }
}

// Block-wide: validate the lengths and build the page prefix sums pre[0..B]
// and the attended lengths len[0..B) in shared memory. Invalid lengths count
// as zero pages (their rows are written as zeros by the merge kernel). With
// several queries per sequence (q_start != null), a sequence is also invalid
// unless it has 1 .. nq queries, at least as many tokens, and its query rows
// lie within the num_q rows of q and out.
template <int BS>
__device__ void scan_lengths(const int32_t* __restrict__ seq_lens, int B, int limit, int* pre,
                             int* len, int* err, const int32_t* q_start = nullptr, int nq = 0,
                             int num_q = 0) {
    __shared__ int warp_tot[32];
    const int T = blockDim.x, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
    const int chunk = (B + T - 1) / T;
    const int lo = min(tid * chunk, B), hi = min(lo + chunk, B);
    int sum = 0;
    bool bad = false;
    for (int b = lo; b < hi; ++b) {
        const int L = seq_lens[b];
        bool ok = L >= 1 && L <= limit;
        if (q_start) {
            const int nqb = q_start[b + 1] - q_start[b];
            ok = ok && nqb >= 1 && nqb <= nq && nqb <= L && q_start[b] >= 0 && q_start[b + 1] <= num_q;
        }
        bad |= !ok;
        len[b] = ok ? L : 0;
        sum += ok ? (L + BS - 1) / BS : 0;
    }
    if (bad && blockIdx.x == 0 && err) atomicOr(err, kErrSeqLen);
    int x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += y;
        }
        if (lane < nwarps) warp_tot[lane] = t;
    }
    __syncthreads();
    int run = x - sum + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int b = lo; b < hi; ++b) {
        pre[b] = run;
        run += (len[b] + BS - 1) / BS;
    }
    if (tid == T - 1) pre[B] = run;
    __syncthreads();
}

__device__ __forceinline__ uint32_t swz(uint32_t region, int chunk, int tok, int BS) {
    // 16-byte chunk `chunk` of row `tok` in a [BS][D] page stored as D/64 boxes
    // of [BS][64] with the 128-byte swizzle.
    return region + (chunk >> 3) * (BS * 128) + tok * 128 + ((((chunk & 7) ^ (tok & 7))) << 4);
}

// ------------------------------------------------------------------ FMA path
template <int D, int BS>
struct FmaState {
    static constexpr bool kQS = false;   // query rows staged contiguously, read once per segment
    static constexpr int HALF = D / 2;   // query elements per lane
    static constexpr int DPL = D / 32;   // output elements per lane
    static constexpr int TPL = BS / 16;  // tokens per lane
    float qf[HALF];
    float acc[DPL];
    float m, l;

    __device__ __forceinline__ void start(uint32_t qst, int /*nh*/, int lane) {
        const int hh = lane >> 4;
#pragma unroll
        for (int c = 0; c < HALF / 8; ++c) {
            const uint4 w = lds_u128(qst + hh * D + c * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qf[c * 8 + 2 * e] = bf16_lo(ws[e]);
                qf[c * 8 + 2 * e + 1] = bf16_hi(ws[e]);
            }
        }
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
        m = -INFINITY;
        l = 0.f;
    }

    __device__ __forceinline__ void page(uint32_t kst, uint32_t vst, int nv, float scale_log2,
                                         int lane) {
        const int hh = lane >> 4, tl = lane & 15;
        float sc[TPL];
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
            const int tok = tl + 16 * j;
            float dot = 0.f;
#pragma unroll
            for (int c = 0; c < HALF / 8; ++c) {
                const uint4 w = lds_u128(swz(kst, hh * (HALF / 8) + c, tok, BS));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dot = fmaf(qf[c * 8 + 2 * e], bf16_lo(ws[e]), dot);
                    dot = fmaf(qf[c * 8 + 2 * e + 1], bf16_hi(ws[e]), dot);
                }
            }
            dot += __shfl_xor_sync(0xffffffffu, dot, 16);
            sc[j] = tok < nv ? dot * scale_log2 : -INFINITY;
        }
        float mx = sc[0];
#pragma unroll
        for (int j = 1; j < TPL; ++j) mx = fmaxf(mx, sc[j]);
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m - m_use);
        float p[TPL];
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
            p[j] = fast_exp2(sc[j] - m_use);
            psum += p[j];
        }
        l = l * alpha + (hh == 0 ? psum : 0.f);
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] *= alpha;
        m = m_new;
        // Weighted values: lane owns DPL consecutive dims, token by token.
        const int d0 = lane * DPL;
        const int chunk = d0 >> 3;
        const uint32_t within = (d0 & 7) * 2;
#pragma unroll
        for (int j = 0; j < TPL; ++j) {
          const int nt_j = min(16, nv - 16 * j);
          for (int tt = 0; tt < nt_j; ++tt) {
            const int t = 16 * j + tt;
            const float pt = __shfl_sync(0xffffffffu, p[j], tt);
            const uint32_t addr = swz(vst, chunk, t, BS) + within;
            if constexpr (DPL == 4) {
                const uint2 w = lds_u64(addr);
                acc[0] = fmaf(pt, bf16_lo(w.x), acc[0]);
                acc[1] = fmaf(pt, bf16_hi(w.x), acc[1]);
                acc[2] = fmaf(pt, bf16_lo(w.y), acc[2]);
                acc[3] = fmaf(pt, bf16_hi(w.y), acc[3]);
            } else {
                const uint32_t w = lds_u32(addr);
                acc[0] = fmaf(pt, bf16_lo(w), acc[0]);
                acc[1] = fmaf(pt, bf16_hi(w), acc[1]);
            }
          }
        }
    }

    __device__ __forceinline__ void finish(const SplitArgs& a, int b, int hq0, int nh, bool full,
                                           bool poison, int slot, int lane) {
        (void)nh;
        float lt = l;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
        const int d0 = lane * DPL;
        if (full) {
            const float inv = poison ? 0.f : 1.f / lt;
            const size_t row = (static_cast<size_t>(b) * a.Hq + hq0) * D;
            if (a.out_bf16) {
                uint16_t* o = static_cast<uint16_t*>(a.out) + row + d0;
                if constexpr (DPL == 4) {
                    uint2 w;
                    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
                    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
                    *reinterpret_cast<uint2*>(o) = w;
                } else {
                    *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
                }
            } else {
                float* o = static_cast<float*>(a.out) + row + d0;
#pragma unroll
                for (int i = 0; i < DPL; ++i) o[i] = acc[i] * inv;
            }
        } else {
            float* o = a.ws_acc + static_cast<size_t>(slot) * a.GS * D + d0;
#pragma unroll
            for (int i = 0; i < DPL; ++i) o[i] = poison ? 0.f : acc[i];
            if (lane == 0) {
                a.ws_ml[static_cast<size_t>(slot) * a.GS * 2 + 0] = poison ? __int_as_float(0x7fc00000) : m;
                a.ws_ml[static_cast<size_t>(slot) * a.GS * 2 + 1] = poison ? 0.f : lt;
            }
        }
    }
};

// ------------------------------------------------------------------ MMA path
// QS: the query fragments are read from the stage's query rows (row pitch
// mq_q_pitch(D)) at every chunk instead of being held in registers for the
// whole segment. Tiles of two n-tiles (9-16 columns: several queries per
// sequence, or 9-16 query heads per kv head) do this, which saves 32
// registers a thread; their stage keeps the segment's query rows because
// they run one stage per warp.
template <int D, int BS, int NT, bool QS = false>
struct MmaState {
    static constexpr bool kQS = QS;
    static constexpr int KS = D / 16;     // k-steps of the score product, m-tiles of the value product
    static constexpr int TILES = BS / 16; // 16-token tiles per page
    static constexpr int QP = QS ? mq_q_pitch(D) : D * 2;  // query row pitch in the stage
    uint32_t qb[QS ? 1 : KS][NT][2];      // Q^T fragments (B operand), held unless QS
    float o[KS][NT][4];                   // O^T accumulators
    float m[NT][2], l[NT][2];

    // Fragment (kk, nt) of Q^T from the stage: rows past nh read as zero.
    __device__ __forceinline__ void q_frag(uint32_t qst, int nh, int lane, int kk, int nt,
                                           uint32_t& b0, uint32_t& b1) const {
        const int row = nt * 8 + (lane >> 2);
        const uint32_t addr = qst + row * QP + (16 * kk + 2 * (lane & 3)) * 2;
        b0 = row < nh ? lds_u32(addr) : 0u;
        b1 = row < nh ? lds_u32(addr + 16) : 0u;
    }

    __device__ __forceinline__ void start(uint32_t qst, int nh, int lane) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if constexpr (!QS) {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) q_frag(qst, nh, lane, kk, nt, qb[kk][nt][0], qb[kk][nt][1]);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                m[nt][j] = -INFINITY;
                l[nt][j] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
        }
    }

    // nv: tokens of this chunk before the end of the sequence. With MQ, column
    // c of the tile is query c / g (of nqb, the newest tokens) and head c % g,
    // and query i sees only the tokens before rem - (nqb - 1 - i), rem being
    // the tokens from the chunk's start to the end of the sequence.
    template <bool MQ = false>
    __device__ __forceinline__ void page(uint32_t kst, uint32_t vst, int nv, float scale_log2,
                                         int lane, int rem = 0, int nqb = 0, int g = 1,
                                         uint32_t qst = 0, int nh = 0) {
        int lim[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if constexpr (MQ) {
                    const int col = nt * 8 + 2 * (lane & 3) + j;
                    lim[nt][j] = min(nv, rem - (nqb - 1 - col / g));
                } else {
                    lim[nt][j] = nv;
                }
            }
        float s[TILES][NT][4];
#pragma unroll
        for (int t = 0; t < TILES; ++t)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s[t][nt][i] = 0.f;
        // Scores S^T = K Q^T.
        if constexpr (QS) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t b[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) q_frag(qst, nh, lane, kk, nt, b[nt][0], b[nt][1]);
#pragma unroll
                for (int t = 0; t < TILES; ++t) {
                    const int tok = t * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(swz(kst, 2 * kk + (lane >> 4), tok, BS), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(s[t][nt], a0, a1, a2, a3, b[nt][0], b[nt][1]);
                }
            }
        } else {
#pragma unroll
            for (int t = 0; t < TILES; ++t) {
                const int tok = t * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(swz(kst, 2 * kk + (lane >> 4), tok, BS), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(s[t][nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
                }
            }
        }
        // Scale to the log2 domain, mask the tail, column maxima over the tokens.
        float mx[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mx[nt][0] = -INFINITY;
            mx[nt][1] = -INFINITY;
        }
#pragma unroll
        for (int t = 0; t < TILES; ++t) {
            const int tok = t * 16 + (lane >> 2);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tk = tok + (i >= 2 ? 8 : 0);
                    const float v = tk < lim[nt][i & 1] ? s[t][nt][i] * scale_log2 : -INFINITY;
                    s[t][nt][i] = v;
                    mx[nt][i & 1] = fmaxf(mx[nt][i & 1], v);
                }
            }
        }
        float alpha[NT][2], m_use[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float x = mx[nt][j];
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
                const float m_new = fmaxf(m[nt][j], x);
                m_use[nt][j] = m_new == -INFINITY ? 0.f : m_new;
                alpha[nt][j] = fast_exp2(m[nt][j] - m_use[nt][j]);
                m[nt][j] = m_new;
            }
        }
        // Probabilities as a bf16 pair hi + lo (hi = bf16(p), lo = bf16(p - hi)),
        // transposed in registers into the B operand of P V. With MQ (twice
        // the columns, so twice the products per page) only hi is used, as in
        // the prefill kernel: 8 significant bits of p, well inside the bf16
        // output's tolerance.
        uint32_t pb[TILES][NT][2][2];  // [tile][n-tile][hi/lo][token half]
        float ps[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            ps[nt][0] = 0.f;
            ps[nt][1] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < TILES; ++t) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) p[i] = fast_exp2(s[t][nt][i] - m_use[nt][i & 1]);
                ps[nt][0] += p[0] + p[2];
                ps[nt][1] += p[1] + p[3];
                const uint32_t top = pack_bf16x2(p[0], p[1]);
                const uint32_t bot = pack_bf16x2(p[2], p[3]);
                pb[t][nt][0][0] = movmatrix_trans(top);
                pb[t][nt][0][1] = movmatrix_trans(bot);
                if constexpr (!MQ) {
                    const uint32_t top_lo = pack_bf16x2(p[0] - bf16_lo(top), p[1] - bf16_hi(top));
                    const uint32_t bot_lo = pack_bf16x2(p[2] - bf16_lo(bot), p[3] - bf16_hi(bot));
                    pb[t][nt][1][0] = movmatrix_trans(top_lo);
                    pb[t][nt][1][1] = movmatrix_trans(bot_lo);
                }
            }
        }
        bool rescale = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                l[nt][j] = l[nt][j] * alpha[nt][j] + ps[nt][j];
                rescale |= alpha[nt][j] != 1.f;
            }
        }
        if (__any_sync(0xffffffffu, rescale)) {  // skipped while no running max moves
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[mt][nt][i] *= alpha[nt][i & 1];
        }
        // Values O^T += V^T P^T.
        const bool tail = nv < BS;
        const int t0 = 2 * (lane & 3);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
            for (int t = 0; t < TILES; ++t) {
                const int tok = t * 16 + (lane >> 4) * 8 + (lane & 7);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(swz(vst, 2 * mt + ((lane >> 3) & 1), tok, BS), a0, a1, a2, a3);
                if (tail) {
                    const int tb = t * 16 + t0;
                    const uint32_t keep01 = (tb < nv ? 0x0000ffffu : 0u) | (tb + 1 < nv ? 0xffff0000u : 0u);
                    const uint32_t keep89 = (tb + 8 < nv ? 0x0000ffffu : 0u) | (tb + 9 < nv ? 0xffff0000u : 0u);
                    a0 &= keep01;
                    a1 &= keep01;
                    a2 &= keep89;
                    a3 &= keep89;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_bf16_16816(o[mt][nt], a0, a1, a2, a3, pb[t][nt][0][0], pb[t][nt][0][1]);
                    if constexpr (!MQ)
                        mma_bf16_16816(o[mt][nt], a0, a1, a2, a3, pb[t][nt][1][0], pb[t][nt][1][1]);
                }
            }
        }
    }

    // With MQ, column `head` is query head / g of the sequence (row qrow0 + it
    // of out) and head hq0 + head % g; otherwise head hq0 + head of row b.
    template <bool MQ = false>
    __device__ __forceinline__ void finish(const SplitArgs& a, int b, int hq0, int nh, bool full,
                                           bool poison, int slot, int lane, int qrow0 = 0) {
        float lt[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float x = l[nt][j];
                x += __shfl_xor_sync(0xffffffffu, x, 4);
                x += __shfl_xor_sync(0xffffffffu, x, 8);
                x += __shfl_xor_sync(0xffffffffu, x, 16);
                lt[nt][j] = x;
            }
        const int dr = lane >> 2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int head = nt * 8 + 2 * (lane & 3) + j;
                if (head >= nh) continue;
                if (full) {
                    const float inv = poison ? 0.f : 1.f / lt[nt][j];
                    size_t row;
                    if constexpr (MQ)
                        row = ((static_cast<size_t>(qrow0) + head / a.g) * a.Hq + hq0 + head % a.g) * D;
                    else
                        row = (static_cast<size_t>(b) * a.Hq + hq0 + head) * D;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const int d = mt * 16 + dr + 8 * r;
                            const float v = o[mt][nt][2 * r + j] * inv;
                            if (a.out_bf16)
                                static_cast<uint16_t*>(a.out)[row + d] = f32_to_bf16_bits(v);
                            else
                                static_cast<float*>(a.out)[row + d] = v;
                        }
                    }
                } else {
                    float* acc = a.ws_acc + (static_cast<size_t>(slot) * a.GS + head) * D;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                        for (int r = 0; r < 2; ++r)
                            acc[mt * 16 + dr + 8 * r] = poison ? 0.f : o[mt][nt][2 * r + j];
                    if (dr == 0) {
                        float* ml = a.ws_ml + (static_cast<size_t>(slot) * a.GS + head) * 2;
                        ml[0] = poison ? __int_as_float(0x7fc00000) : m[nt][j];
                        ml[1] = poison ? 0.f : lt[nt][j];
                    }
                }
            }
        }
    }
};

// ------------------------------------------------------------------ kernel
// One pipeline stage holds a chunk of CT = kChunkTokens consecutive tokens of
// one segment: two 16-token pages stacked (block size 16) or one 32-token
// page. Both give the same shared-memory image, [D/64 boxes][32 rows][128 B]
// with the 128-byte swizzle, so the arithmetic sees one 32-token tile pair.
// Ranges of the page stream. The first (1 - f) of the stream is cut into equal
// static ranges, one per warp; the last fraction f into small dynamic pieces of
// dyn_pages pages that warps claim through an atomic counter once their static
// range is done (guided self-scheduling: warps that run faster take more of the
// tail). A range id r owns partial slots 2r (head) and 2r + 1 (tail): static
// ranges have ids 0 .. NW-1, dynamic piece j has id NW + j.
struct Range {
    int x0, x1, id;
};

__device__ __forceinline__ void sts_v4i(uint32_t addr, int a0, int a1, int a2) {
    asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a0), "r"(a1), "r"(a2), "r"(0)
                 : "memory");
}

__device__ __forceinline__ void sts_u128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ int4 lds_v4i(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Number of ranges that hold part of pages [x0, x1) of the stream: static
// ranges of `per` pages up to A, then dynamic pieces of qd pages. Each writes
// one partial of a segment that occupies those pages.
__device__ __forceinline__ int ranges_over(int x0, int x1, int per, int A, int qd) {
    int n = 0;
    if (x0 < A) n += (min(x1, A) - 1) / per - x0 / per + 1;
    if (x1 > A) n += (x1 - 1 - A) / qd - (max(x0, A) - A) / qd + 1;
    return n;
}

// Fused merge: fold the partials of the segment on pages [x0, x1) for its nh
// query-head columns and write the normalised rows row0 .. row0 + nh - 1 --
// the two-partial rule of "39 · PagedAttention" §3 applied to batches of
// partials against a running maximum (log2 domain), as the merge kernel does.
// Run by the warp that wrote the segment's last partial; the partials of
// other warps are read from L2 (ld.global.cg), past the fence that published
// them.
template <int D>
__device__ __forceinline__ void fold_segment(const SplitArgs& a, int x0, int x1, int per, int A,
                                          int NW, int qd, size_t row0, int nh, int lane) {
    constexpr int DPL = D / 32;
    constexpr int kBatch = 8;
    auto range_of = [&](int x) { return x < A ? x / per : NW + (x - A) / qd; };
    auto holds = [&](int r) { return r >= NW || static_cast<long long>(r) * per < A; };
    const int rf = range_of(x0), rl = range_of(x1 - 1);
    const int d0 = lane * DPL;
    for (int j = 0; j < nh; ++j) {
        float m = -INFINITY, l = 0.f, acc[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
        bool poison = false;
        for (int r0 = rf; r0 <= rl; r0 += kBatch) {
            float mi[kBatch], li[kBatch], v[kBatch][DPL];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int r = r0 + k;
                mi[k] = -INFINITY;
                li[k] = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i) v[k][i] = 0.f;
                if (r <= rl && holds(r)) {
                    const size_t base = static_cast<size_t>(r == rf ? 2 * r + 1 : 2 * r) * a.GS + j;
                    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.ws_ml) + base);
                    mi[k] = ml.x;
                    li[k] = ml.y;
                    const float* src = a.ws_acc + base * D + d0;
                    if constexpr (DPL == 4) {
                        const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
                        v[k][0] = t.x; v[k][1] = t.y; v[k][2] = t.z; v[k][3] = t.w;
                    } else {
                        const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
                        v[k][0] = t.x; v[k][1] = t.y;
                    }
                }
            }
            float mb = m;
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                poison |= mi[k] != mi[k];   // the poison marker of a bad table entry
                mb = fmaxf(mb, mi[k]);      // fmaxf passes over NaN
            }
            if (mb == -INFINITY) continue;
            const float fo = fast_exp2(m - mb);
            l *= fo;
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] *= fo;
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const float f = fast_exp2(mi[k] - mb);
                l = fmaf(li[k], f, l);
#pragma unroll
                for (int i = 0; i < DPL; ++i) acc[i] = fmaf(v[k][i], f, acc[i]);
            }
            m = mb;
        }
        // A poisoned partial (bad table entry) makes the sums NaN: the row is
        // written as zeros, not scaled by zero.
        const bool zero = poison || !(l > 0.f);
        const float inv = zero ? 0.f : 1.f / l;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = zero ? 0.f : acc[i];
        const size_t o = (row0 + j) * D + d0;
        if (a.out_bf16) {
            uint16_t* dst = static_cast<uint16_t*>(a.out) + o;
            if constexpr (DPL == 4) {
                uint2 w;
                w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
                w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
                *reinterpret_cast<uint2*>(dst) = w;
            } else {
                *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            }
        } else {
            float* dst = static_cast<float*>(a.out) + o;
#pragma unroll
            for (int i = 0; i < DPL; ++i) dst[i] = acc[i] * inv;
        }
    }
}

// APPEND: the step's new K/V rows are appended by this kernel (one stage per
// warp). The warp whose chunk holds a segment's last page loads the rows
// before it waits for the stage, writes them into the staged page at
// position seq_len - 1 once the copy has landed, and (first slice of the kv
// head) into the pools. No other warp reads that slot in this call: every
// page belongs to one range, and the other slices of a kv head patch their
// own staged copies.
template <int D, int BS, typename State, bool MQ = false, bool FUSED = false, bool APPEND = false>
__device__ __forceinline__ void split_body(const CUtensorMap* kmap, const CUtensorMap* vmap,
                                           const SplitArgs& a) {
    static_assert(!(MQ && FUSED), "the fused merge serves one query per sequence");
    static_assert(!(APPEND && (MQ || FUSED)), "the fused append serves the plain decode");
    static_assert(!MQ || State::kQS, "the multi-query tile reads its query rows from the stage");
    constexpr int CT = kChunkTokens;
    constexpr int CP = CT / BS;  // pages per chunk
    extern __shared__ uint8_t smem_raw[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    int* pre = reinterpret_cast<int*>(smem_raw + (base - raw));
    int* len = pre + (a.B + 1);
    const int S = a.stages;
    const uint32_t ring0 = base + a.lens_bytes;
    const uint32_t bars0 = ring0 + static_cast<uint32_t>(W * S * a.stage_bytes);
    // Per stage: range x0, x1, id (16-byte records, so 16-byte aligned).
    const uint32_t meta0 = bars0 + ((static_cast<uint32_t>(W * S * 8) + 15u) & ~15u);
    // An mbarrier that nothing completes: the wait-expiry probe's first wait.
    const uint32_t probe_bar = meta0 + static_cast<uint32_t>(W * S * 16);
    // The two-n-tile decode keeps its query rows per warp after the rest
    // (one stage per warp); the other kernels carry them in the stage after
    // K and V.
    constexpr bool kQRegion = State::kQS && !MQ;
    const uint32_t q_region0 = probe_bar + 16;

    if (threadIdx.x == 0) {
        prefetch_tensormap(kmap);
        prefetch_tensormap(vmap);
        if (a.probe_wait) {
            mbar_init(probe_bar, 1);
            fence_barrier_init();
        }
    }
    // Everything below may read what the previous kernel of the stream wrote.
    griddep_wait();
    griddep_launch_dependents();
    const int limit = min(a.max_seq_len, a.max_blocks * BS);
    if constexpr (MQ)
        scan_lengths<BS>(a.seq_lens, a.B, limit, pre, len, a.err, a.q_start, a.nq, a.num_q);
    else
        scan_lengths<BS>(a.seq_lens, a.B, limit, pre, len, a.err);

    const int P = a.U * pre[a.B];
    const int NW = gridDim.x * W;
    // Dynamic tail: a fraction of the stream in pieces of dyn_pages (none for
    // small streams, where the static ranges are already short).
    const int qd = a.dyn_pages;
    const int Dp = (P >= 8 * NW * qd) ? (static_cast<int>(static_cast<long long>(P) * a.dyn_permille / 1000) / qd) * qd : 0;
    const int A = P - Dp;
    const int per = max(1, (A + NW - 1) / NW);
    const int nd = Dp / qd;
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= a.B; i += blockDim.x) a.ws_meta[kMetaHeader + i] = pre[i];
        if (threadIdx.x == 0) {
            a.ws_meta[0] = P;
            a.ws_meta[1] = per;
            a.ws_meta[2] = NW;
            // [3] is the dynamic-piece counter: zero on entry, reset by the merge.
            a.ws_meta[4] = A;
            a.ws_meta[5] = qd;
            a.ws_meta[6] = nd;
        }
    }
    const int gw = blockIdx.x * W + warp;
    if constexpr (FUSED) {
        // No merge kernel follows: rows of invalid sequences get zeros here.
        for (int b = gw; b < a.B; b += NW) {
            if (len[b] != 0) continue;
            const size_t row0 = static_cast<size_t>(b) * a.Hq * D;
            for (int i = lane; i < a.Hq * D; i += 32) {
                if (a.out_bf16) static_cast<uint16_t*>(a.out)[row0 + i] = 0;
                else static_cast<float*>(a.out)[row0 + i] = 0.f;
            }
        }
    }
    // Every warp calls this once, as it leaves (warp-collective). With the
    // fused merge the last warp of the grid to leave resets the dynamic-piece
    // counter for the next call and, if any warp gave up, the segment
    // counters (whose partials may never have arrived).
    auto leave = [&](bool gave_up) {
        if constexpr (FUSED) {
            int done = 0;
            if (lane == 0) {
                if (gave_up) atomicExch(a.ws_meta + 8, 1);
                __threadfence();
                done = atomicAdd(a.ws_meta + 7, 1);
            }
            done = __shfl_sync(0xffffffffu, done, 0);
            if (done == NW - 1) {
                __threadfence();
                const bool clear = *reinterpret_cast<volatile int*>(a.ws_meta + 8) != 0;
                if (clear)
                    for (int i = lane; i < a.B * a.U; i += 32) a.ws_cnt[i] = 0;
                if (lane == 0) {
                    a.ws_meta[3] = 0;
                    a.ws_meta[7] = 0;
                    a.ws_meta[8] = 0;
                }
            }
        }
    };
    const uint32_t my_bars = bars0 + warp * S * 8;
    const uint32_t my_meta = meta0 + warp * S * 16;
    const uint32_t my_ring = ring0 + static_cast<uint32_t>(warp * S * a.stage_bytes);
    const uint32_t my_q = q_region0 + static_cast<uint32_t>(warp * a.q_bytes);
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(my_bars + 8 * s, 1);
        fence_barrier_init();
    }
    __syncwarp();

    auto claim = [&]() -> Range {
        int j = 0;
        if (lane == 0) j = atomicAdd(a.ws_meta + 3, 1);
        j = __shfl_sync(0xffffffffu, j, 0);
        if (j >= nd) return Range{-1, -1, -1};
        return Range{A + j * qd, min(A + (j + 1) * qd, P), NW + j};
    };
    auto locate = [&](int x) {
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.U * pre[mid] <= x) lo = mid; else hi = mid - 1;
        }
        const int nb = seq_pages(pre, lo);
        const int off = x - a.U * pre[lo];
        return Cursor{lo, off / nb, off % nb, nb};
    };

    Range ri{gw * per, min(gw * per + per, A), gw};
    if (ri.x0 >= ri.x1) ri = claim();
    if (ri.id < 0) {
        leave(false);
        return;
    }
    Cursor ci = locate(ri.x0);
    int xi = ri.x0;
    bool issue_done = false;
    const uint32_t page_bytes = 2u * BS * D * 2u;  // K + V of one page
    const uint64_t policy = policy_evict_first();
    int tb_row = -1, tb_base = -1, tbl = -1;  // table batch: entries [tb_base, tb_base+32) of row tb_row
    uint32_t badmask = 0, phase = 0;

    auto table_entry = [&](int b, int p, int nb) {
        const int pbase = p & ~31;
        if (b != tb_row || pbase != tb_base) {
            tb_row = b;
            tb_base = pbase;
            tbl = (pbase + lane < nb)
                      ? __ldg(a.tables + static_cast<size_t>(b) * a.max_blocks + pbase + lane)
                      : -1;
        }
        return __shfl_sync(0xffffffffu, tbl, p - pbase);
    };

    // Issue the chunk at the issue cursor into stage s; warp-collective.
    auto issue = [&](int s) {
        const int n = min(min(CP, ci.nb - ci.p), ri.x1 - xi);
        const bool qstart = xi == ri.x0 || ci.p == 0;
        int phys[CP];
        bool bad = false;
#pragma unroll
        for (int j = 0; j < CP; ++j) {
            phys[j] = j < n ? table_entry(ci.b, ci.p + j, ci.nb) : 0;
            bad |= j < n && (phys[j] < 0 || phys[j] >= a.num_blocks);
        }
        badmask = bad ? (badmask | (1u << s)) : (badmask & ~(1u << s));
        if (lane == 0) {
            const uint32_t bar = my_bars + 8 * s;
            const uint32_t stg = my_ring + static_cast<uint32_t>(s * a.stage_bytes);
            sts_v4i(my_meta + 16 * s, ri.x0, ri.x1, ri.id);  // released by the arrive below
            const int kvh = ci.u / a.nslices, slice = ci.u - kvh * a.nslices;
            int nh, qrow0 = 0;
            if constexpr (MQ) {
                qrow0 = a.q_start[ci.b];
                nh = (a.q_start[ci.b + 1] - qrow0) * a.g;  // validated: 1 .. nq queries
            } else {
                nh = min(a.GS, a.g - slice * a.GS);
            }
            const uint32_t qbytes = qstart ? static_cast<uint32_t>(nh * D * 2) : 0u;
            if (bad) {
                atomicOr(a.err, kErrTable);
                if (qstart) {
                    mbar_arrive_expect_tx(bar, qbytes);
                } else {
                    mbar_arrive(bar);
                }
            } else {
                mbar_arrive_expect_tx(bar, n * page_bytes + qbytes);
                for (int j = 0; j < n; ++j) {
                    const int row = phys[j] * a.Hkv + kvh;
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        const uint32_t off = h * (CT * 128) + j * (BS * 128);
                        tma_load_3d(stg + off, kmap, h * 64, 0, row, bar, policy);
                        tma_load_3d(stg + CT * D * 2 + off, vmap, h * 64, 0, row, bar, policy);
                    }
                }
            }
            if (qstart) {
                if constexpr (State::kQS) {
                    // One row of D values per copy at the padded pitch. With MQ,
                    // column c = i * g + j is head kvh * g + j of query row
                    // qrow0 + i; otherwise head kvh * g + slice * GS + c of row b.
                    for (int c = 0; c < nh; ++c) {
                        size_t row;
                        if constexpr (MQ) {
                            const int i = c / a.g, j = c - i * a.g;
                            row = (static_cast<size_t>(qrow0) + i) * a.Hq + kvh * a.g + j;
                        } else {
                            row = static_cast<size_t>(ci.b) * a.Hq + kvh * a.g + slice * a.GS + c;
                        }
                        bulk_load((kQRegion ? my_q : stg + 2 * CT * D * 2) + c * mq_q_pitch(D),
                                  a.q + row * D, D * 2, bar);
                    }
                } else {
                    const uint16_t* src =
                        a.q + (static_cast<size_t>(ci.b) * a.Hq + kvh * a.g + slice * a.GS) * D;
                    bulk_load(stg + 2 * CT * D * 2, src, qbytes, bar);
                }
            }
        }
        for (int j = 0; j < n; ++j) advance(ci, pre, a.U, a.B);
        xi += n;
        if (xi == ri.x1) {  // next range: a dynamic piece, if any is left
            ri = claim();
            if (ri.id < 0) {
                issue_done = true;
            } else {
                ci = locate(ri.x0);
                xi = ri.x0;
            }
        }
    };

    int n_issued = 0;
    for (int s = 0; s < S && !issue_done; ++s, ++n_issued) issue(s);

    State st;
    Range rc{-1, -1, -1};
    Cursor cc{0, 0, 0, 0};
    int xc = 0;
    int p_first = 0, hq0 = 0, nh = 0, qrow0 = 0, nqb = 0;
    bool poison = false;
    int s = 0, n_done = 0;
    while (n_done < n_issued) {
        const uint32_t bar = my_bars + 8 * s;
        const uint32_t stg = my_ring + static_cast<uint32_t>(s * a.stage_bytes);
        // Fused append: does this stage hold a segment's last page? The range
        // record is this warp's own earlier write, readable before the wait.
        constexpr int RV = D / 8;  // 16-byte vectors of one K or V row
        int ap_row = -1, ap_kvh = 0, ap_slice = 0, ap_phys = 0, ap_slot = 0;
        uint4 ap_w = make_uint4(0, 0, 0, 0);
        if constexpr (APPEND) {
            const int4 p4 = lds_v4i(my_meta + 16 * s);
            const bool fresh = p4.z != rc.id;
            const Cursor pc = fresh ? locate(p4.x) : cc;
            const int pn = min(min(CP, pc.nb - pc.p), fresh ? p4.y - p4.x : rc.x1 - xc);
            if (pc.p + pn == pc.nb && !((badmask >> s) & 1u)) {
                ap_kvh = pc.u / a.nslices;
                ap_slice = pc.u - ap_kvh * a.nslices;
                ap_slot = (len[pc.b] - 1) % BS;
                ap_row = (pc.nb - 1 - pc.p) * BS + ap_slot;
                ap_phys = table_entry(pc.b, pc.nb - 1, pc.nb);
                if (lane < 2 * RV) {
                    const uint16_t* src = (lane < RV ? a.k_new : a.v_new) +
                                          (static_cast<size_t>(pc.b) * a.Hkv + ap_kvh) * D +
                                          (lane % RV) * 8;
                    ap_w = *reinterpret_cast<const uint4*>(src);
                }
            }
        }
        const bool ready = (a.probe_wait && n_done == 0)
                               ? mbar_wait_bounded(probe_bar, 0, kProbeLimitNs)
                               : mbar_wait_bounded(bar, (phase >> s) & 1u, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ready)) {
            // Give up: report, wait (bounded) for this warp's copies in flight, return.
            if (lane == 0) atomicOr(a.err, kErrTimeout);
            for (int j = n_done; j < n_issued; ++j) {
                const int sj = j % S;
                mbar_wait_bounded(my_bars + 8 * sj, (phase >> sj) & 1u, kWaitLimitNs);
            }
            leave(true);
            return;
        }
        phase ^= 1u << s;
        const int4 m4 = lds_v4i(my_meta + 16 * s);
        if (m4.z != rc.id) {  // first chunk of a new range
            rc = Range{m4.x, m4.y, m4.z};
            xc = rc.x0;
            cc = locate(xc);
        }
        const int n = min(min(CP, cc.nb - cc.p), rc.x1 - xc);
        if (xc == rc.x0 || cc.p == 0) {
            const int kvh = cc.u / a.nslices, slice = cc.u - kvh * a.nslices;
            if constexpr (MQ) {
                qrow0 = a.q_start[cc.b];
                nqb = a.q_start[cc.b + 1] - qrow0;
                nh = nqb * a.g;
                hq0 = kvh * a.g;
            } else {
                nh = min(a.GS, a.g - slice * a.GS);
                hq0 = kvh * a.g + slice * a.GS;
            }
            st.start(kQRegion ? my_q : stg + 2 * CT * D * 2, nh, lane);
            p_first = cc.p;
            poison = false;
        }
        if constexpr (APPEND) {
            if (ap_row >= 0) {
                if (lane < 2 * RV) {
                    const uint32_t region = stg + (lane < RV ? 0u : static_cast<uint32_t>(CT * D * 2));
                    sts_u128(swz(region, lane % RV, ap_row, CT), ap_w);
                    if (ap_slice == 0) {
                        uint16_t* pool = lane < RV ? a.kpool_w : a.vpool_w;
                        const size_t off =
                            ((static_cast<size_t>(ap_phys) * a.Hkv + ap_kvh) * BS + ap_slot) * D;
                        *reinterpret_cast<uint4*>(pool + off + (lane % RV) * 8) = ap_w;
                    }
                }
                __syncwarp();
            }
        }
        if ((badmask >> s) & 1u) {
            poison = true;
        } else {
            const int rem = len[cc.b] - cc.p * BS;  // tokens from the chunk start to the end
            const int nv = min(n * BS, rem);
            if constexpr (MQ)
                st.template page<true>(stg, stg + CT * D * 2, nv, a.scale_log2, lane, rem, nqb, a.g,
                                       stg + 2 * CT * D * 2, nh);
            else if constexpr (State::kQS)
                st.page(stg, stg + CT * D * 2, nv, a.scale_log2, lane, 0, 0, 1, my_q, nh);
            else
                st.page(stg, stg + CT * D * 2, nv, a.scale_log2, lane);
        }
        __syncwarp();
        if (!issue_done) {
            fence_proxy_async_smem();
            issue(s);
            ++n_issued;
        }
        const int p_last = cc.p + n - 1;
        if (p_last == cc.nb - 1 || xc + n == rc.x1) {
            const bool full = p_first == 0 && p_last == cc.nb - 1;
            const int slot = rc.id * 2 + (p_first > 0 ? 0 : 1);
            if constexpr (MQ)
                st.template finish<true>(a, cc.b, hq0, nh, full, poison, slot, lane, qrow0);
            else
                st.finish(a, cc.b, hq0, nh, full, poison, slot, lane);
            if constexpr (FUSED) {
                if (!full) {
                    // Publish this partial, count it; the warp that writes the
                    // segment's last partial folds them all.
                    __threadfence();
                    __syncwarp();
                    const int x0 = a.U * pre[cc.b] + cc.u * cc.nb;
                    const int parts = ranges_over(x0, x0 + cc.nb, per, A, qd);
                    int prev = 0;
                    if (lane == 0) prev = atomicAdd(a.ws_cnt + cc.b * a.U + cc.u, 1);
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    if (prev == parts - 1) {
                        __threadfence();
                        fold_segment<D>(a, x0, x0 + cc.nb, per, A, NW, qd,
                                        static_cast<size_t>(cc.b) * a.Hq + hq0, nh, lane);
                        if (lane == 0) a.ws_cnt[cc.b * a.U + cc.u] = 0;
                    }
                }
            }
        }
        for (int j = 0; j < n; ++j) advance(cc, pre, a.U, a.B);
        xc += n;
        ++n_done;
        if (++s == S) s = 0;
    }
    leave(false);
}

}  // namespace split
}  // namespace pa
