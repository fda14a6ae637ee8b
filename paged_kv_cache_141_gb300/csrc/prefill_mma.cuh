// prefill_mma.cuh -- multi-query paged attention for a few query tokens per
// sequence (a speculative verification step) on warp-level tensor-core MMA.
//
// Work unit: a sequence s, a KV head hk and 8 NT of the sequence's R = Q_s G
// query rows, token-major (row r is query token r / G and query head
// hk G + r % G, as in the tcgen05 kernel), cut into NT n-tiles of 8 rows.
// Query token i sits at position L - Q_s + i and sees keys 0..L - Q_s + i
// ("Lecture 3: PagedAttention and vLLM", "the paged implementation of
// attention"; the queries there carry a num_queries axis).
//
// Two kernels, both the tensor-core decode (decode_mma.cuh) with the MMA's
// eight columns holding query rows instead of the query heads of one token.
// The producer warp loads each 32-key stage of K and V once per CTA (tensor
// TMA, 128-byte swizzle), whatever the number of rows. Per warp and 16-key
// row tile: S^T (16 keys x 8 rows) = K Q^T, each column masked at its row's
// causal limit, an online softmax per row (base 2, against a reference max
// that moves only past 2^8), O^T += V^T P^T with P as two bf16 terms (bf16
// caches) or one binary16 term (f16 caches, E4M3 caches widened to binary16:
// at most 2^-11 relative error per weight).
//
//  * paged_prefill_mma_kernel, up to 16 rows (NT = 1 or 2 n-tiles of 8):
//    consumer warp w (of 4) owns n-tile w mod NT; the NT warps of different
//    n-tiles all read every stage, the 4 / NT warps of one n-tile take
//    alternate stages and are merged at the end as in the decode. The query
//    fragments stay in registers.
//  * paged_prefill_mma2_kernel, 17 to 32 rows (head size <= 128): a warp owns
//    two n-tiles, so each K or V fragment it loads feeds two MMAs; warps w and
//    w + 2 take alternate stages. The query rows sit in shared memory and are
//    read with ldmatrix, leaving the registers to two n-tiles' accumulators.
//
// Why these next to the tcgen05 kernels: for the 32 or fewer rows of a
// verification step a 128-row tcgen05 tile is mostly padding, and its one
// CTA per SM leaves the SM idle while a unit starts and drains. Here one CTA
// streams its sequence's K/V once for all its rows at a few times the
// decode's MMA work per byte, with 3 (16-bit) to 4 (E4M3) CTAs per SM
// overlapping one another's starts and ends. (One n-tile per warp at 32 rows,
// four warps per stage, was latency-bound below the tcgen05 kernel; beyond
// 32 rows the tcgen05 kernels are faster.)
//
// Keys past a stage's last needed key are masked by a select on the scores
// (never a multiply) and their V^T fragments are zeroed in registers, so stale
// or poisoned shared memory never reaches an output (0 x NaN). Every wait is
// bounded (PA_DEV_TIMEOUT).
#pragma once

#include "decode_mma.cuh"

namespace pagedkv {

// Rows of one CTA: 8 NT, NT = 1 or 2.
constexpr int kMqMaxTiles = 2;
// A column's reference max moves only when a score exceeds it by more than
// this (base 2): weights stay below 2^8.
constexpr float kMqRescaleLog2 = 8.0f;

// CTAs per SM the registers must allow (shared memory allows 3 for 16-bit
// caches at head size <= 128, more for E4M3: there 4 CTAs of 96 registers,
// with a few spilled words, ran faster than 3 without spills or 5 with more).
template <int D>
constexpr int mq_min_blocks() {
    return D <= 128 ? 4 : 2;
}

// The producer warp of both multi-query MMA kernels: walks sequence s's block
// table ("the paged implementation of attention": logical block -> physical
// block) and loads keys [0, Tend) of KV head kvh, 32 per stage, K and V with
// tensor TMA (one box per block segment and 128-byte column span) into ring
// slot k mod NST, once the slot's consumers have released it; at the end it
// waits for its copies in flight. Every wait is bounded.
template <typename CT, int D, int NST>
__device__ __forceinline__ void mq_load_stages(const TmaDecodeParams& tp, int s, int kvh, int Tend,
                                               uint8_t* ring, uint64_t* full, uint64_t* empty,
                                               int lane) {
    using S = TmaShape<CT, D>;
    const DecodeParams& p = tp.p;
    const int n_st = (Tend + kTmaStageTokens - 1) / kTmaStageTokens;
    const int B = p.block_size;
    const int rows = tp.box_rows;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
    if (lane == 0) {
        tma_prefetch_map(&tp.k_map);
        tma_prefetch_map(&tp.v_map);
    }
    int issued = 0;
    for (int k = 0; k < n_st; ++k) {
        const int slot = k % NST;
        if (k >= NST) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(&empty[slot], ((k / NST) - 1) & 1, p.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
        }
        const int t_lo = k * kTmaStageTokens;
        const int t_hi = min(t_lo + kTmaStageTokens, Tend);
        const int j0 = t_lo / B;
        const int nseg = (t_hi - 1) / B - j0 + 1;
        uint32_t bytes = 0;
        int y = 0, r0 = 0;
        if (lane < nseg) {
            const int j = j0 + lane;
            const int pb = table[j];
            if (pb < 0 || (int64_t)pb >= p.num_blocks) {
                if (p.status) atomicOr(p.status, PA_DEV_BAD_BLOCK_ID);
            } else {
                const int off = (B >= kTmaStageTokens) ? (t_lo - j * B) : 0;
                y = (pb * p.num_kv_heads + kvh) * B + off;
                r0 = (B >= kTmaStageTokens) ? 0 : j * B - t_lo;
                bytes = (uint32_t)(rows * S::kRowBytes);
            }
        }
        uint32_t total = bytes;
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) total += __shfl_xor_sync(0xffffffffu, total, m);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2 * total);
        __syncwarp();
        if (bytes) {
            uint8_t* st = ring + (size_t)slot * S::kStageBytes;
#pragma unroll
            for (int sp = 0; sp < S::kSpans; ++sp) {
                const int x = sp * (128 / S::kElem);
                uint8_t* kd = st + sp * S::kSpanTileBytes + r0 * 128;
                tma_load_2d(kd, &tp.k_map, x, y, &full[slot]);
                tma_load_2d(kd + S::kTileBytes, &tp.v_map, x, y, &full[slot]);
            }
        }
        issued = k + 1;
    }
    if (lane == 0) {
        for (int k = max(0, issued - NST); k < issued; ++k)
            mbar_wait_bounded(&full[k % NST], (k / NST) & 1, p.status);
    }
}

template <typename QT, typename CT, int D, int NT>
__global__ void __launch_bounds__(kTmaThreads, mq_min_blocks<D>())
paged_prefill_mma_kernel(const __grid_constant__ TmaDecodeParams tp) {
    constexpr int CW = kTmaConsumerWarps;                // consumer warps; warp CW loads
    using S = TmaShape<CT, D>;
    using Smem = MmaSmem<CT, D>;
    using MT = typename MathType<CT>::T;
    using Ops = MmaOps<MT>;
    constexpr bool kFp8 = std::is_same<CT, e4m3_t>::value;
    // binary16 MMAs (f16 caches, E4M3 widened): P as one term, at most 2^-11
    // relative error per weight; bf16: P_hi + P_lo
    constexpr bool kOneTerm = std::is_same<MT, __half>::value;
    constexpr int NST = Smem::kNst;
    constexpr int WPT = CW / NT;                         // warps per n-tile
    static_assert(NT == 1 || NT == kMqMaxTiles, "n-tiles per CTA");
    // a slot's successive stages belong to the same warps, so a warp waiting
    // on a slot is never two phases ahead of it
    static_assert(NST % WPT == 0, "slot ownership");
    constexpr int KS = D / 16;                           // k-steps of the score product
    const DecodeParams& p = tp.p;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBarOffset);
    uint64_t* empty = full + NST;

    const int kvh = blockIdx.y;
    const int row0 = blockIdx.x * 8 * NT;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;                             // fragment row / B column
    const int t4 = lane & 3;                             // fragment column pair
    // the sequence: launch position z, or the caller's order (longest first)
    const int s = p.seq_order ? __ldg(p.seq_order + blockIdx.z) : (int)blockIdx.z;
    if (s < 0 || s >= p.num_seqs) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0 && p.status)
            atomicOr(p.status, PA_DEV_BAD_ORDER);
        return;
    }

    const int q0 = __ldg(p.query_start + s);
    const int Q = __ldg(p.query_start + s + 1) - q0;
    const int L = __ldg(p.context_lens + s);
    {
        int cap = p.max_context_len;
        const long long tab = (long long)p.max_blocks * p.block_size;
        if (tab < cap) cap = (int)tab;
        if (Q < 0 || Q > p.max_queries || L < Q || L > cap) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0 && p.status)
                atomicOr(p.status, PA_DEV_BAD_LEN);
            return;
        }
    }
    const int G = p.group;
    const int R = Q * G;
    if (row0 >= R) return;
    // keys seen by the CTA's last row; every other row sees a prefix of them
    const int Tend = L - Q + (min(R, row0 + 8 * NT) - 1) / G + 1;
    const int n_st = (Tend + kTmaStageTokens - 1) / kTmaStageTokens;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NT);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        mq_load_stages<CT, D, NST>(tp, s, kvh, Tend, ring, full, empty, lane);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int nt = warp % NT;                            // this warp's n-tile
    const int rw = row0 + 8 * nt;                        // its first row
    // Q^T fragments (B operand of S = K Q^T): column g = row rw + g, zero past
    // the sequence's rows. For E4M3 the k index of a 16-wide step maps to d as
    // the widened ldmatrix bytes come (decode_mma.cuh): k = 2t+j <-> d = 4t+j,
    // k = 2t+8+j <-> d = 4t+2+j, for K and Q alike.
    uint32_t qb[KS][2];
    {
        const int r = rw + g;
        const bool valid = r < R;
        const int i = valid ? r / G : 0;
        const QT* qp = reinterpret_cast<const QT*>(p.query) +
                       ((size_t)(q0 + i) * p.num_q_heads + (size_t)kvh * G + (valid ? r - i * G : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (!valid) {
                qb[ks][0] = 0u;
                qb[ks][1] = 0u;
            } else if constexpr (kFp8) {
                const QT* q4 = qp + 16 * ks + 4 * t4;
                qb[ks][0] = Ops::pack(to_float(q4[0]), to_float(q4[1]));
                qb[ks][1] = Ops::pack(to_float(q4[2]), to_float(q4[3]));
            } else {
                qb[ks][0] = *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * t4);
                qb[ks][1] = *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * t4 + 8);
            }
        }
    }
    // causal limits of this lane's two columns (rows rw + 2 t4 + j): keys
    // < kend. Padding columns (zero queries, never written) take every key
    // of the CTA, so that their running max is finite like the others'.
    int kend[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int r = rw + 2 * t4 + j;
        kend[j] = r < R ? L - Q + r / G + 1 : Tend;
    }
    // below this key no column of the warp is masked (rows are token-major,
    // so the warp's first row has the smallest limit)
    const int kfree = rw < R ? L - Q + rw / G + 1 : Tend;
    float acc[KS][4];                                    // O^T fragments: rows d, columns rows
#pragma unroll
    for (int i = 0; i < KS; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    // per column: the reference max m (base 2) the weights and O are taken
    // against, and this lane's share of the sum of weights. m moves (and O is
    // rescaled) only when a score exceeds it by more than 2^8, so weights
    // stay below 2^8 and most stages need no cross-lane max.
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const float qk_mul = kFp8 ? p.q_mul * 256.f : p.q_mul;
    const int mi = lane >> 3, r8 = lane & 7;             // ldmatrix: lane -> (matrix, row)

    for (int k = warp / NT; k < n_st; k += WPT) {
        const int slot = k % NST;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (k / NST) & 1, p.status));
        if (!ok) break;
        const uint8_t* Kst = ring + (size_t)slot * S::kStageBytes;
        const uint8_t* Vst = Kst + S::kTileBytes;
        const int key0 = k * kTmaStageTokens;
        const int nvalid = min(kTmaStageTokens, Tend - key0);

        // ---- S = K Q^T for both 16-key row tiles, even and odd k-steps in
        // separate accumulators (four independent MMA chains)
        float sc[2][4];
        {
            float sx[2][2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j < 4; ++j) sx[mt][h][j] = 0.f;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int row = 16 * mt + (mi & 1) * 8 + r8;
                const uint8_t* rbase = Kst + row * 128;
                if constexpr (kFp8) {
#pragma unroll
                    for (int kp = 0; kp < KS / 2; ++kp) {
                        const int c = 2 * kp + (mi >> 1);
                        uint32_t x[4];
                        ldmatrix_x4(x, rbase + (c >> 3) * S::kSpanTileBytes + (((c & 7) ^ (row & 7)) << 4));
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const uint32_t a[4] = {
                                e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2], 0u, 0x4140)),
                                e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2 + 1], 0u, 0x4140)),
                                e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2], 0u, 0x4342)),
                                e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2 + 1], 0u, 0x4342))};
                            Ops::mma(sx[mt][h2], a, qb[2 * kp + h2][0], qb[2 * kp + h2][1]);
                        }
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int c = 2 * ks + (mi >> 1);
                        uint32_t a[4];
                        ldmatrix_x4(a, rbase + (c >> 3) * S::kSpanTileBytes + (((c & 7) ^ (row & 7)) << 4));
                        Ops::mma(sx[mt][ks & 1], a, qb[ks][0], qb[ks][1]);
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int j = 0; j < 4; ++j) sc[mt][j] = (sx[mt][0][j] + sx[mt][1][j]) * qk_mul;
        }

        // ---- online softmax per column (this lane: columns 2 t4 + j; keys g,
        // g + 8 of each 16-key tile); masked scores are -inf (a select, never
        // a multiply), only in a stage that reaches a column's limit
        if (key0 + kTmaStageTokens > kfree) {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int key = key0 + 16 * mt + g + 8 * hr;
                        if (key >= kend[j]) sc[mt][2 * hr + j] = -INFINITY;
                    }
        }
        float lmax[2];
        bool up = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            lmax[j] = fmaxf(fmaxf(sc[0][j], sc[0][2 + j]), fmaxf(sc[1][j], sc[1][2 + j]));
            up |= m_run[j] == -INFINITY || lmax[j] > m_run[j] + kMqRescaleLog2;
        }
        if (__any_sync(0xffffffffu, up)) {
            // a new reference max for each column: the column's max over
            // its eight lanes, if it exceeds the old one by more than 2^8
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = lmax[j];
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                if (m_run[j] == -INFINITY || mx > m_run[j] + kMqRescaleLog2) {
                    const float alpha = m_run[j] == -INFINITY ? 0.f : fast_exp2(m_run[j] - mx);
                    if (mx != -INFINITY) {
                        l_run[j] *= alpha;
#pragma unroll
                        for (int i = 0; i < KS; ++i) {
                            acc[i][j] *= alpha;
                            acc[i][2 + j] *= alpha;
                        }
                        m_run[j] = mx;
                    }
                }
            }
        }
        // weights exp2(s - m) <= 2^8; -inf scores (and a column with no key
        // yet, m = -inf) give 0
        float pv[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mj = m_run[e & 1];
                pv[mt][e] = mj == -INFINITY ? 0.f : fast_exp2(sc[mt][e] - mj);
            }

        // ---- P^T fragments: hi + residual, transposed from the S layout
        uint32_t bh[2][2], bl[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float w0 = pv[mt][2 * hr], w1 = pv[mt][2 * hr + 1];
                const uint32_t hi = Ops::pack(w0, w1);
                if constexpr (kOneTerm) {
                    // binary16 weights as one term: the sums take the
                    // rounded weights the products use
                    const float2 hf = Ops::unpack(hi);
                    l_run[0] += hf.x;
                    l_run[1] += hf.y;
                } else {
                    // hi + lo is the weight to 2^-17: the sums take the weight
                    const float2 hf = Ops::unpack(hi);
                    l_run[0] += w0;
                    l_run[1] += w1;
                    bl[mt][hr] = movmatrix_trans(Ops::pack(w0 - hf.x, w1 - hf.y));
                }
                bh[mt][hr] = movmatrix_trans(hi);
            }
        }

        // V^T fragment masks: a fragment's registers 0-1 hold keys 2 t4, 2 t4 + 1
        // of its 16-key step, registers 2-3 keys 2 t4 + 8, 2 t4 + 9 (low half
        // the even key); keys at or past nvalid are zeroed
        uint32_t vmask[2][2];
#pragma unroll
        for (int kt = 0; kt < 2; ++kt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int key = 16 * kt + 2 * t4 + 8 * h;
                vmask[kt][h] = (key < nvalid ? 0x0000ffffu : 0u) | (key + 1 < nvalid ? 0xffff0000u : 0u);
            }
        const bool ragged = nvalid < kTmaStageTokens;

        // ---- O^T += V^T P^T
        if constexpr (kFp8) {
#pragma unroll
            for (int md = 0; md < KS; ++md) {
                const int row = 8 * mi + r8;                         // key
                uint32_t y[4];
                ldmatrix_x4_trans(y, Vst + (md >> 3) * S::kSpanTileBytes + row * 128 +
                                         (((md & 7) ^ (row & 7)) << 4));
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const uint32_t lo = y[2 * kt], hi = y[2 * kt + 1];
                    uint32_t a[4] = {e4m3x2_to_f16x2_scaled(__byte_perm(lo, 0u, 0x4240)),
                                     e4m3x2_to_f16x2_scaled(__byte_perm(lo, 0u, 0x4341)),
                                     e4m3x2_to_f16x2_scaled(__byte_perm(hi, 0u, 0x4240)),
                                     e4m3x2_to_f16x2_scaled(__byte_perm(hi, 0u, 0x4341))};
                    if (ragged) {
                        a[0] &= vmask[kt][0];
                        a[1] &= vmask[kt][0];
                        a[2] &= vmask[kt][1];
                        a[3] &= vmask[kt][1];
                    }
                    Ops::mma(acc[md], a, bh[kt][0], bh[kt][1]);
                }
            }
        } else {
#pragma unroll
            for (int md = 0; md < KS; ++md) {
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const int row = 16 * kt + (mi >> 1) * 8 + r8;       // key
                    const int c = 2 * md + (mi & 1);                     // 16-byte chunk of d
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, Vst + (c >> 3) * S::kSpanTileBytes + row * 128 +
                                             (((c & 7) ^ (row & 7)) << 4));
                    if (ragged) {
                        a[0] &= vmask[kt][0];
                        a[1] &= vmask[kt][0];
                        a[2] &= vmask[kt][1];
                        a[3] &= vmask[kt][1];
                    }
                    Ops::mma(acc[md], a, bh[kt][0], bh[kt][1]);
                    if constexpr (!kOneTerm) Ops::mma(acc[md], a, bl[kt][0], bl[kt][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ------------------------------------------ merge the warps of each n-tile
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
    }
    named_barrier(1, CW * 32);                           // ring is free: every stage was consumed
    float* cm = reinterpret_cast<float*>(smem);          // [CW][8]
    float* cl = cm + CW * 8;                             // [CW][8]
    float* co = cl + CW * 8;                             // [CW][8][D]
    if (g == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            cm[warp * 8 + 2 * t4 + j] = m_run[j];
            cl[warp * 8 + 2 * t4 + j] = l_run[j];
        }
    }
#pragma unroll
    for (int md = 0; md < KS; ++md) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int d = kFp8 ? 16 * md + 2 * g + hr : 16 * md + g + 8 * hr;
                co[(warp * 8 + 2 * t4 + j) * D + d] = acc[md][2 * hr + j];
            }
    }
    named_barrier(1, CW * 32);

    // row c of n-tile t was computed by warps t, t + NT, ...; the CTA's rows
    // are written row by row, d contiguous
    const int nrows = min(8 * NT, R - row0);
    const float vm = kFp8 ? p.v_mul * 256.f : p.v_mul;
    QT* out = reinterpret_cast<QT*>(p.out);
    for (int idx = threadIdx.x; idx < nrows * D; idx += CW * 32) {
        const int rr = idx / D;
        const int e = idx - rr * D;
        const int t = rr >> 3, c = rr & 7;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WPT; ++w) M = fmaxf(M, cm[(t + NT * w) * 8 + c]);
        float W = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < WPT; ++w) {
            const int src = (t + NT * w) * 8 + c;
            const float mw = cm[src];
            const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
            W = fmaf(f, cl[src], W);
            O = fmaf(f, co[src * D + e], O);
        }
        const int r = row0 + rr;
        const int i = r / G;
        const size_t orow = (size_t)(q0 + i) * p.num_q_heads + (size_t)kvh * G + (r - i * G);
        out[orow * D + e] = from_float<QT>(__fdiv_rn(O, W) * vm);
    }
}

// ---------------------------------------------------------------- 32 rows
// Four 8-row n-tiles per CTA (up to 32 rows: 8 draft tokens at G = 4), for
// 16-bit and E4M3 caches at head size <= 128. A warp takes two n-tiles (16 rows), so
// each K or V fragment it loads feeds two MMAs, and a stage is read by two
// warps instead of four; warps w and w + 2 take the same rows on alternate
// stages and are merged at the end. The query rows sit in shared memory in
// the swizzled layout of the K tiles and are read with ldmatrix as the B
// operand (both n-tiles' fragments of a k-step in one load), which leaves
// the registers to the two n-tiles' accumulators. For E4M3 caches the rows
// are stored as binary16 in the k order of the widened K fragments (as the
// query registers of the kernel above), and K/V fragments are widened in
// registers.
constexpr int kMq2Rows = 32;

template <typename CT, int D>
struct Mq2Smem {
    using Ring = MmaSmem<CT, D>;
    static constexpr int kNst = Ring::kNst;
    static constexpr int kQBytes = kMq2Rows * D * 2;             // the CTA's query rows
    static constexpr int kCombineBytes = kTmaConsumerWarps * 16 * (D + 2) * 4;
    static constexpr int kBody =
        Ring::kRingBytes > kCombineBytes ? Ring::kRingBytes : kCombineBytes;
    static constexpr int kQOffset = (kBody + 1023) / 1024 * 1024;
    static constexpr int kBarOffset = kQOffset + kQBytes;
    static constexpr int kBytes = kBarOffset + 2 * kNst * 8;
    static constexpr int kAlloc = kBytes + 1024;                // room to align the ring to 1 KB
};

template <typename QT, typename CT, int D>
__global__ void __launch_bounds__(kTmaThreads, 3)
paged_prefill_mma2_kernel(const __grid_constant__ TmaDecodeParams tp) {
    using S = TmaShape<CT, D>;
    using Smem = Mq2Smem<CT, D>;
    using MT = typename MathType<CT>::T;
    using Ops = MmaOps<MT>;
    constexpr bool kFp8 = std::is_same<CT, e4m3_t>::value;
    constexpr int CW = kTmaConsumerWarps;                // consumer warps; warp CW loads
    constexpr int NST = Smem::kNst;
    static_assert(NST % 2 == 0, "a slot's stages belong to one warp pair");
    static_assert(D <= 128, "two n-tiles' accumulators in registers");
    constexpr bool kOneTerm = std::is_same<MT, __half>::value;  // binary16 P as one term
    constexpr int KS = D / 16;
    constexpr int kQSpan = kMq2Rows * 128;               // bytes of one 128-byte column span
    const DecodeParams& p = tp.p;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* ring = smem;
    uint8_t* qsm = smem + Smem::kQOffset;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBarOffset);
    uint64_t* empty = full + NST;

    const int kvh = blockIdx.y;
    const int row0 = blockIdx.x * kMq2Rows;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t4 = lane & 3;
    const int s = p.seq_order ? __ldg(p.seq_order + blockIdx.z) : (int)blockIdx.z;
    if (s < 0 || s >= p.num_seqs) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0 && p.status)
            atomicOr(p.status, PA_DEV_BAD_ORDER);
        return;
    }
    const int q0 = __ldg(p.query_start + s);
    const int Q = __ldg(p.query_start + s + 1) - q0;
    const int L = __ldg(p.context_lens + s);
    {
        int cap = p.max_context_len;
        const long long tab = (long long)p.max_blocks * p.block_size;
        if (tab < cap) cap = (int)tab;
        if (Q < 0 || Q > p.max_queries || L < Q || L > cap) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0 && p.status)
                atomicOr(p.status, PA_DEV_BAD_LEN);
            return;
        }
    }
    const int G = p.group;
    const int R = Q * G;
    if (row0 >= R) return;
    const int Tend = L - Q + (min(R, row0 + kMq2Rows) - 1) / G + 1;
    const int n_st = (Tend + kTmaStageTokens - 1) / kTmaStageTokens;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 2);                     // the two warps of a stage phase
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        mq_load_stages<CT, D, NST>(tp, s, kvh, Tend, ring, full, empty, lane);
        return;
    }

    // ---- the CTA's query rows -> shared memory, zero past the sequence's,
    // row r's 16-byte chunk c of span c / 8 at chunk (c mod 8) ^ (r mod 8).
    // E4M3: binary16, chunk c = 2 ks + h holding positions 8 h .. 8 h + 7 of
    // k-step ks, position 2 t + j <-> d = 16 ks + 4 t + 2 h + j.
    constexpr int CPR = D / 8;
    for (int i = threadIdx.x; i < kMq2Rows * CPR; i += CW * 32) {
        const int r = i / CPR, c = i - r * CPR;
        const int rg = row0 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (rg < R) {
            const int ti = rg / G;
            const QT* qrow_g = reinterpret_cast<const QT*>(p.query) +
                               ((size_t)(q0 + ti) * p.num_q_heads + (size_t)kvh * G + (rg - ti * G)) * D;
            if constexpr (kFp8) {
                const QT* q4 = qrow_g + 16 * (c >> 1) + 2 * (c & 1);
                uint32_t w[4];
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    w[t] = Ops::pack(to_float(q4[4 * t]), to_float(q4[4 * t + 1]));
                v = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                v = *reinterpret_cast<const uint4*>(qrow_g + c * 8);
            }
        }
        *reinterpret_cast<uint4*>(qsm + (c >> 3) * kQSpan + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
    }
    named_barrier(2, CW * 32);

    // ---- consumers: warp w takes CTA rows 16 (w mod 2) .. + 15 (n-tiles
    // nt = 0, 1 of 8 rows) on stages k = w / 2 (mod 2)
    const int pi = warp & 1;
    const int ph = warp >> 1;
    const int mi = lane >> 3, r8 = lane & 7;
    int kend[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = row0 + 16 * pi + 8 * nt + 2 * t4 + j;
            kend[nt][j] = r < R ? L - Q + r / G + 1 : Tend;
        }
    const int rfirst = row0 + 16 * pi;
    const int kfree = rfirst < R ? L - Q + rfirst / G + 1 : Tend;
    float acc[2][KS][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][i][e] = 0.f;
    float m_run[2][2], l_run[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            m_run[nt][j] = -INFINITY;
            l_run[nt][j] = 0.f;
        }
    const float qk_mul = kFp8 ? p.q_mul * 256.f : p.q_mul;  // E4M3: the widening's 2^-8
    // B fragments of a k-step: matrix mi = (n-tile mi / 2, 8-element half mi mod 2)
    const int qrow = 16 * pi + 8 * (mi >> 1) + r8;
    const uint8_t* qbase = qsm + qrow * 128;

    for (int k = ph; k < n_st; k += 2) {
        const int slot = k % NST;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (k / NST) & 1, p.status));
        if (!ok) break;
        const uint8_t* Kst = ring + (size_t)slot * S::kStageBytes;
        const uint8_t* Vst = Kst + S::kTileBytes;
        const int key0 = k * kTmaStageTokens;
        const int nvalid = min(kTmaStageTokens, Tend - key0);

        // ---- S = K Q^T: [n-tile][16-key tile], four independent chains
        float sc[2][2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[nt][mt][e] = 0.f;
        if constexpr (kFp8) {
            // one ldmatrix.x4 of E4M3 bytes covers two k-steps of 16 keys,
            // widened in registers (decode_mma.cuh)
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
                uint32_t b[2][4];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int cq = 2 * (2 * kp + h2) + (mi & 1);
                    ldmatrix_x4(b[h2], qbase + (cq >> 3) * kQSpan + (((cq & 7) ^ (qrow & 7)) << 4));
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int row = 16 * mt + (mi & 1) * 8 + r8;
                    const int c = 2 * kp + (mi >> 1);
                    uint32_t x[4];
                    ldmatrix_x4(x, Kst + (c >> 3) * S::kSpanTileBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4));
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const uint32_t a[4] = {
                            e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2], 0u, 0x4140)),
                            e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2 + 1], 0u, 0x4140)),
                            e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2], 0u, 0x4342)),
                            e4m3x2_to_f16x2_scaled(__byte_perm(x[2 * h2 + 1], 0u, 0x4342))};
                        Ops::mma(sc[0][mt], a, b[h2][0], b[h2][1]);
                        Ops::mma(sc[1][mt], a, b[h2][2], b[h2][3]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int cq = 2 * ks + (mi & 1);
                uint32_t b[4];
                ldmatrix_x4(b, qbase + (cq >> 3) * kQSpan + (((cq & 7) ^ (qrow & 7)) << 4));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int row = 16 * mt + (mi & 1) * 8 + r8;
                    const int c = 2 * ks + (mi >> 1);
                    uint32_t a[4];
                    ldmatrix_x4(a, Kst + (c >> 3) * S::kSpanTileBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4));
                    Ops::mma(sc[0][mt], a, b[0], b[1]);
                    Ops::mma(sc[1][mt], a, b[2], b[3]);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[nt][mt][e] *= qk_mul;

        // ---- causal mask (a select), only in a stage that reaches a limit
        if (key0 + kTmaStageTokens > kfree) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int key = key0 + 16 * mt + g + 8 * hr;
                            if (key >= kend[nt][j]) sc[nt][mt][2 * hr + j] = -INFINITY;
                        }
        }
        // ---- reference max per column, moved only past 2^8 (a warp vote)
        float lmax[2][2];
        bool up = false;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                lmax[nt][j] = fmaxf(fmaxf(sc[nt][0][j], sc[nt][0][2 + j]),
                                    fmaxf(sc[nt][1][j], sc[nt][1][2 + j]));
                up |= m_run[nt][j] == -INFINITY || lmax[nt][j] > m_run[nt][j] + kMqRescaleLog2;
            }
        if (__any_sync(0xffffffffu, up)) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float mx = lmax[nt][j];
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    if (m_run[nt][j] == -INFINITY || mx > m_run[nt][j] + kMqRescaleLog2) {
                        const float alpha =
                            m_run[nt][j] == -INFINITY ? 0.f : fast_exp2(m_run[nt][j] - mx);
                        if (mx != -INFINITY) {
                            l_run[nt][j] *= alpha;
#pragma unroll
                            for (int i = 0; i < KS; ++i) {
                                acc[nt][i][j] *= alpha;
                                acc[nt][i][2 + j] *= alpha;
                            }
                            m_run[nt][j] = mx;
                        }
                    }
                }
        }
        // ---- weights and their P^T fragments (hi + residual)
        uint32_t bh[2][2][2], bl[2][2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const float m0 = m_run[nt][0], m1 = m_run[nt][1];
                    const float w0 = m0 == -INFINITY ? 0.f : fast_exp2(sc[nt][mt][2 * hr] - m0);
                    const float w1 = m1 == -INFINITY ? 0.f : fast_exp2(sc[nt][mt][2 * hr + 1] - m1);
                    const uint32_t hi = Ops::pack(w0, w1);
                    const float2 hf = Ops::unpack(hi);
                    bh[nt][mt][hr] = movmatrix_trans(hi);
                    if constexpr (kOneTerm) {
                        // the sums take the rounded weights the products use
                        l_run[nt][0] += hf.x;
                        l_run[nt][1] += hf.y;
                    } else {
                        // hi + lo is the weight to 2^-17: the sums take the weight
                        l_run[nt][0] += w0;
                        l_run[nt][1] += w1;
                        bl[nt][mt][hr] = movmatrix_trans(Ops::pack(w0 - hf.x, w1 - hf.y));
                    }
                }

        // ---- O^T += V^T P^T for both n-tiles; keys at or past nvalid zeroed
        // in the V^T fragments (registers 0-1: keys 2 t4, 2 t4 + 1 of the
        // 16-key step; 2-3: keys 2 t4 + 8, 2 t4 + 9)
        const bool ragged = nvalid < kTmaStageTokens;
        uint32_t vmask[2][2];
#pragma unroll
        for (int kt = 0; kt < 2; ++kt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int key = 16 * kt + 2 * t4 + 8 * h;
                vmask[kt][h] = (key < nvalid ? 0x0000ffffu : 0u) | (key + 1 < nvalid ? 0xffff0000u : 0u);
            }
        if constexpr (kFp8) {
            // one 16-byte chunk = 16 d of all 32 keys (decode_mma.cuh):
            // fragment row g <-> d 2g, row g + 8 <-> d 2g + 1
#pragma unroll
            for (int md = 0; md < KS; ++md) {
                const int row = 8 * mi + r8;
                uint32_t y[4];
                ldmatrix_x4_trans(y, Vst + (md >> 3) * S::kSpanTileBytes + row * 128 +
                                         (((md & 7) ^ (row & 7)) << 4));
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const uint32_t lo = y[2 * kt], hi = y[2 * kt + 1];
                    uint32_t a[4] = {e4m3x2_to_f16x2_scaled(__byte_perm(lo, 0u, 0x4240)),
                                     e4m3x2_to_f16x2_scaled(__byte_perm(lo, 0u, 0x4341)),
                                     e4m3x2_to_f16x2_scaled(__byte_perm(hi, 0u, 0x4240)),
                                     e4m3x2_to_f16x2_scaled(__byte_perm(hi, 0u, 0x4341))};
                    if (ragged) {
                        a[0] &= vmask[kt][0];
                        a[1] &= vmask[kt][0];
                        a[2] &= vmask[kt][1];
                        a[3] &= vmask[kt][1];
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        Ops::mma(acc[nt][md], a, bh[nt][kt][0], bh[nt][kt][1]);
                }
            }
        } else {
#pragma unroll
            for (int md = 0; md < KS; ++md) {
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const int row = 16 * kt + (mi >> 1) * 8 + r8;
                    const int c = 2 * md + (mi & 1);
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, Vst + (c >> 3) * S::kSpanTileBytes + row * 128 +
                                             (((c & 7) ^ (row & 7)) << 4));
                    if (ragged) {
                        a[0] &= vmask[kt][0];
                        a[1] &= vmask[kt][0];
                        a[2] &= vmask[kt][1];
                        a[3] &= vmask[kt][1];
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        Ops::mma(acc[nt][md], a, bh[nt][kt][0], bh[nt][kt][1]);
                        if constexpr (!kOneTerm) Ops::mma(acc[nt][md], a, bl[nt][kt][0], bl[nt][kt][1]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ------------------------------------------ merge the two stage phases
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 4);
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 8);
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 16);
        }
    named_barrier(1, CW * 32);                           // ring is free: every stage was consumed
    float* cm = reinterpret_cast<float*>(smem);          // [CW][16]
    float* cl = cm + CW * 16;                            // [CW][16]
    float* co = cl + CW * 16;                            // [CW][16][D]
    if (g == 0) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                cm[warp * 16 + 8 * nt + 2 * t4 + j] = m_run[nt][j];
                cl[warp * 16 + 8 * nt + 2 * t4 + j] = l_run[nt][j];
            }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int md = 0; md < KS; ++md)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    co[(warp * 16 + 8 * nt + 2 * t4 + j) * D +
                       (kFp8 ? 16 * md + 2 * g + hr : 16 * md + g + 8 * hr)] = acc[nt][md][2 * hr + j];
    named_barrier(1, CW * 32);

    // CTA row rr = 16 pair + c was computed by warps pair and pair + 2
    const int nrows = min(kMq2Rows, R - row0);
    const float vm = kFp8 ? p.v_mul * 256.f : p.v_mul;
    QT* out = reinterpret_cast<QT*>(p.out);
    for (int idx = threadIdx.x; idx < nrows * D; idx += CW * 32) {
        const int rr = idx / D;
        const int e = idx - rr * D;
        const int a0 = (rr >> 4) * 16 + (rr & 15);       // warp pair, phase 0
        const int a1 = a0 + 2 * 16;                      // phase 1
        const float ma = cm[a0], mb = cm[a1];
        const float M = fmaxf(ma, mb);
        const float fa = ma == -INFINITY ? 0.f : fast_exp2(ma - M);
        const float fb = mb == -INFINITY ? 0.f : fast_exp2(mb - M);
        const float W = fmaf(fa, cl[a0], fb * cl[a1]);
        const float O = fmaf(fa, co[a0 * D + e], fb * co[a1 * D + e]);
        const int r = row0 + rr;
        const int i = r / G;
        const size_t orow = (size_t)(q0 + i) * p.num_q_heads + (size_t)kvh * G + (r - i * G);
        out[orow * D + e] = from_float<QT>(__fdiv_rn(O, W) * vm);
    }
}

template <typename QT, typename CT, int D>
cudaError_t launch_prefill_mma2(const TmaDecodeParams& tp, cudaStream_t stream) {
    using Smem = Mq2Smem<CT, D>;
    auto kern = paged_prefill_mma2_kernel<QT, CT, D>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Smem::kAlloc);
    if (e != cudaSuccess) return e;
    const DecodeParams& p = tp.p;
    const long long rows = (long long)p.max_queries * p.group;
    const long long groups = (rows + kMq2Rows - 1) / kMq2Rows;
    if (groups > 0x7fffffffll) return cudaErrorInvalidValue;
    dim3 grid((unsigned)groups, p.num_kv_heads, p.num_seqs);
    kern<<<grid, kTmaThreads, Smem::kAlloc, stream>>>(tp);
    return cudaGetLastError();
}

template <typename QT, typename CT, int D, int NT>
cudaError_t launch_prefill_mma_variant(const TmaDecodeParams& tp, cudaStream_t stream) {
    using Smem = MmaSmem<CT, D>;
    auto kern = paged_prefill_mma_kernel<QT, CT, D, NT>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Smem::kAlloc);
    if (e != cudaSuccess) return e;
    const DecodeParams& p = tp.p;
    const long long rows = (long long)p.max_queries * p.group;
    const long long groups = (rows + 8 * NT - 1) / (8 * NT);
    if (groups > 0x7fffffffll) return cudaErrorInvalidValue;
    dim3 grid((unsigned)groups, p.num_kv_heads, p.num_seqs);
    kern<<<grid, kTmaThreads, Smem::kAlloc, stream>>>(tp);
    return cudaGetLastError();
}

// The fewest n-tiles that hold max_queries * group rows, at most kMqMaxTiles
// (more rows would take several CTAs per sequence and KV head).
template <typename QT, typename CT, int D>
cudaError_t launch_prefill_mma_d(const TmaDecodeParams& tp, cudaStream_t stream) {
    const long long rows = (long long)tp.p.max_queries * tp.p.group;
    if (rows <= 8) return launch_prefill_mma_variant<QT, CT, D, 1>(tp, stream);
    if constexpr (D <= 128) {
        if (rows > 8 * kMqMaxTiles) return launch_prefill_mma2<QT, CT, D>(tp, stream);
    }
    return launch_prefill_mma_variant<QT, CT, D, kMqMaxTiles>(tp, stream);
}

template <typename QT, typename CT>
cudaError_t launch_prefill_mma(const DecodeParams& p, int head_size, cudaStream_t stream) {
    constexpr int eb = TypeInfo<CT>::bytes;
    TmaDecodeParams tp;
    tp.p = p;
    tp.box_rows = p.block_size < kTmaStageTokens ? p.block_size : kTmaStageTokens;
    const unsigned long long rows =
        (unsigned long long)p.num_blocks * p.num_kv_heads * p.block_size;
    cudaError_t e = encode_cache_map(&tp.k_map, p.k_cache, eb, head_size, rows, tp.box_rows);
    if (e == cudaSuccess) e = encode_cache_map(&tp.v_map, p.v_cache, eb, head_size, rows, tp.box_rows);
    if (e != cudaSuccess) return e;
    if constexpr (eb == 2) {
        switch (head_size) {
        case 64: return launch_prefill_mma_d<QT, CT, 64>(tp, stream);
        case 128: return launch_prefill_mma_d<QT, CT, 128>(tp, stream);
        case 256: return launch_prefill_mma_d<QT, CT, 256>(tp, stream);
        }
    } else {
        switch (head_size) {
        case 128: return launch_prefill_mma_d<QT, CT, 128>(tp, stream);
        case 256: return launch_prefill_mma_d<QT, CT, 256>(tp, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace pagedkv
