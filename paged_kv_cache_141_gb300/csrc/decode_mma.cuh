// decode_mma.cuh -- the paged decode for 16-bit caches with the GQA group's
// two contractions on the tensor cores (warp-level mma m16n8k16).
//
// Work unit, producer and shared-memory layout are those of the tensor-TMA
// kernel (decode_tma.cuh): a producer warp walks the block table ("Lecture 3:
// PagedAttention and vLLM", "the paged implementation of attention") and
// loads each 32-token stage of K and V with cp.async.bulk.tensor into the
// 128-byte swizzled layout. Here each stage belongs to one consumer warp
// (stage k -> warp k mod 4), which computes, per 16-token row tile:
//   S (16 tokens x 8 heads) = K_tile (16 x d) . Q^T (d x 8), K fragments read
//     with ldmatrix from the swizzled tile, Q^T fragments kept in registers;
//   an online softmax over the tokens for each head (base 2, float32);
//   O^T (d x 8 heads) += V^T (d x 16 tokens) . P^T (16 tokens x 8 heads),
//     V^T fragments read with ldmatrix.trans, P^T fragments made from the S
//     accumulators with movmatrix. P is split into a 16-bit high part and a
//     16-bit residual, two MMAs, so the weights keep ~16 significant bits
//     (E4M3 caches: binary16 weights as one term, 11 bits, far below the
//     codes' own error).
// E4M3 caches are widened to binary16 in registers by integer operations
// (e4m3x2_to_f16x2_scaled) and multiplied on binary16 MMAs. (Warp-level MMAs
// with E4M3 operands were measured to cost as many instructions as this
// widening on this GPU, with the query and weights cut to two E4M3 terms.)
// Heads beyond the group (up to the MMA's 8 columns) carry zero queries and
// are never written out. Rows of V past the context are zeroed before the
// P.V product, since 0 x NaN would otherwise poison every output component.
// At the end the four warps' (max, sum, output) are merged as in the other
// kernels; the output is O / sum (the partition's normalised output).
#pragma once

#include "decode_tma.cuh"

namespace pagedkv {

template <typename CT> struct MmaOps;

template <> struct MmaOps<__nv_bfloat16> {
    __device__ __forceinline__ static void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // (lo, hi) floats -> packed pair, round to nearest even; and the residuals
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
};

template <> struct MmaOps<__half> {
    __device__ __forceinline__ static void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    }
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(smem_row)));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(smem_row)));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Consumer warps of the tensor-core decode: 4, as in the tensor-TMA kernel
// (6 or 8 for E4M3 caches, one ring slot each, measured no faster: 8 with
// three CTAs per SM took 152 us against 89 us on the shared-prefix pool).
template <typename CT, int D>
constexpr int mma_consumer_warps() {
    return kTmaConsumerWarps;
}

// Shared memory of the tensor-core decode: the stage ring (reused for the
// final merge of the consumer warps) and the stage barriers.
// Stage k belongs to warp k mod W (W consumer warps) and sits in slot k mod
// NST; NST is a multiple of W so that every slot has one owner and its
// mbarrier phases advance one stage at a time (a parity wait cannot alias an
// older phase).
template <typename CT, int D>
struct MmaSmem {
    using S = TmaShape<CT, D>;
    static constexpr int kConsumers = mma_consumer_warps<CT, D>();
    // E4M3 stages are half the bytes: one stage per consumer warp keeps the
    // ring at 32 KB, so that the register file, not shared memory, limits the
    // CTAs per SM (5) for these latency-bound tiles
    static constexpr int kNstCap = std::is_same<CT, e4m3_t>::value ? kConsumers : 1 << 30;
    static constexpr int kNstT = S::kNst < kNstCap ? S::kNst : kNstCap;
    static constexpr int kNst0 = kNstT / kConsumers * kConsumers;
    static constexpr int kNst = kNst0 < kConsumers ? kConsumers : kNst0;
    static constexpr int kRingBytes = kNst * S::kStageBytes;
    static constexpr int kCombineBytes = kConsumers * 8 * (D + 2) * 4;
    static constexpr int kBody = kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes;
    static constexpr int kBarOffset = (kBody + 127) / 128 * 128;
    // full[kNst], empty[kNst], and two rendezvous barriers of shared-prefix units
    static constexpr int kBytes = kBarOffset + (2 * kNst + 2) * 8;
    static constexpr int kAlloc = kBytes + 1024;                // room to align the ring to 1 KB
};

// E4M3 caches run the MMAs in binary16 (every E4M3 value is exact in it):
// K and V fragments are widened in registers, the query is rounded to f16.
// The widened values are the codes' values times 2^-8 (see
// e4m3x2_to_f16x2_scaled); the score and output scales carry the 2^8.
template <typename CT> struct MathType { using T = CT; };
template <> struct MathType<e4m3_t> { using T = __half; };

// Two E4M3 codes, in bytes 0 and 2 of t (bytes 1 and 3 zero), to the binary16
// pair of their values times 2^-8, exactly, in integer operations: the
// exponent field (bias 7) and 3 mantissa bits moved up 7 places are a binary16
// exponent (bias 15) and mantissa of the value times 2^-8 (a subnormal code
// gives the binary16 subnormal of that value), and the sign, moved to bit 14,
// is carried into bit 15 by adding it to itself. The saturating write never
// stores the NaN codes 0x7f / 0xff.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t t) {
    const uint32_t x = t << 7;
    return x + (x & 0x40004000u);
}

// CTAs per SM the registers must allow: 4 at head size <= 128 (shared memory
// allows 3 for 16-bit caches), 5 for E4M3 caches whose 32 KB ring allows more;
// 2 at head size 256.
template <typename CT, int D>
constexpr int mma_min_blocks() {
    return D <= 128 ? (std::is_same<CT, e4m3_t>::value ? 5 : 4) : 2;
}

template <typename CT, int D>
constexpr int mma_threads() {
    return (mma_consumer_warps<CT, D>() + 1) * 32;
}

// One consumer warp's share of the decode: the query's B fragments, the
// O^T accumulators and the online-softmax state of the heads this lane holds
// (2 t4 and 2 t4 + 1), and the work on one 32-token stage of K and V.
// kOneTermP: the weights as one 16-bit term (E4M3 values, widened in
// registers or staged as binary16 tiles); otherwise high part + residual.
template <typename QT, typename CT, int D, int GS,
          bool kOneTermP = std::is_same<CT, e4m3_t>::value>
struct MmaWarp {
    using S = TmaShape<CT, D>;
    using MT = typename MathType<CT>::T;
    using Ops = MmaOps<MT>;
    static constexpr bool kFp8 = std::is_same<CT, e4m3_t>::value;
    static constexpr int KS = D / 16;          // k-steps of the score product
    // Q^T fragments (B operand of S = K Q^T): column g = head g, rows = d.
    // For E4M3 the k index of a 16-wide step maps to d as the widened ldmatrix
    // bytes come: k = 2t+j <-> d = 4t+j and k = 2t+8+j <-> d = 4t+2+j (a
    // permutation of the reduction, applied to K and Q alike).
    uint32_t qb[KS][2];
    float qk_mul;                               // scale * log2(e) (E4M3: k_scale and 2^8 too)
    float acc[KS][4];                           // O^T fragments: rows d, columns heads
    float m_run[2];                             // heads 2*t4 and 2*t4+1
    float l_run[2];                             // this lane's share of the sums

    // qp: the query row of the unit's first head; q_mul: scale * log2(e)
    // (E4M3: * k_scale).
    __device__ __forceinline__ void load_query(const QT* __restrict__ qp, float q_mul, int lane) {
        const int g = lane >> 2;
        const int t4 = lane & 3;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (g >= GS) {
                qb[ks][0] = 0u;
                qb[ks][1] = 0u;
            } else if constexpr (kFp8) {
                const QT* q4 = qp + g * D + 16 * ks + 4 * t4;
                qb[ks][0] = Ops::pack(to_float(q4[0]), to_float(q4[1]));
                qb[ks][1] = Ops::pack(to_float(q4[2]), to_float(q4[3]));
            } else {
                qb[ks][0] = *reinterpret_cast<const uint32_t*>(qp + g * D + 16 * ks + 2 * t4);
                qb[ks][1] = *reinterpret_cast<const uint32_t*>(qp + g * D + 16 * ks + 2 * t4 + 8);
            }
        }
        // the widened E4M3 codes are their values times 2^-8
        qk_mul = kFp8 ? q_mul * 256.f : q_mul;
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
    }

    // 16-bit math on tiles of another source (widened E4M3): the query rows
    // of type Q2 rounded to this warp's 16-bit type, natural d order.
    template <typename Q2>
    __device__ __forceinline__ void load_query_as(const Q2* __restrict__ qp, float q_mul, int lane) {
        static_assert(!kFp8, "16-bit math only");
        const int g = lane >> 2;
        const int t4 = lane & 3;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (g >= GS) {
                qb[ks][0] = 0u;
                qb[ks][1] = 0u;
            } else {
                const Q2* q2 = qp + g * D + 16 * ks + 2 * t4;
                qb[ks][0] = Ops::pack(to_float(q2[0]), to_float(q2[1]));
                qb[ks][1] = Ops::pack(to_float(q2[8]), to_float(q2[9]));
            }
        }
        qk_mul = q_mul;
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
    }

    // One stage: K and V tiles of 32 tokens in the 128-byte swizzled layout,
    // the first nvalid of them in the context (V rows past it already zero).
    __device__ __forceinline__ void consume(const uint8_t* Kst, const uint8_t* Vst, int nvalid,
                                            int lane) {
        const int g = lane >> 2;
        const int mi = lane >> 3, r8 = lane & 7;   // ldmatrix row addresses: lane -> (matrix, row)
        // ---- S = K Q^T for both 16-token row tiles
        float sc[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
            for (int j = 0; j < 4; ++j) sc[mt][j] = 0.f;
            const int row = 16 * mt + (mi & 1) * 8 + r8;
            const uint8_t* rbase = Kst + row * 128;
            if constexpr (kFp8) {
                // one ldmatrix.x4 covers two 16-byte chunks (32 d) of 16 tokens
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
                        Ops::mma(sc[mt], a, qb[2 * kp + h2][0], qb[2 * kp + h2][1]);
                    }
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int c = 2 * ks + (mi >> 1);
                    uint32_t a[4];
                    ldmatrix_x4(a, rbase + (c >> 3) * S::kSpanTileBytes + (((c & 7) ^ (row & 7)) << 4));
                    Ops::mma(sc[mt], a, qb[ks][0], qb[ks][1]);
                }
            }
        }

        // ---- online softmax per head (this lane: heads 2*t4, 2*t4+1; tokens g, g+8 of each tile)
        float pv[2][4];
        float alpha[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int tok = 16 * mt + g + 8 * hr;
                    float v = sc[mt][2 * hr + j] * qk_mul;
                    v = tok < nvalid ? v : -INFINITY;          // select, never multiply
                    sc[mt][2 * hr + j] = v;
                    mx = fmaxf(mx, v);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[j], mx);
            alpha[j] = (m_new == -INFINITY) ? 1.f
                     : ((m_run[j] == -INFINITY) ? 0.f : fast_exp2(m_run[j] - m_new));
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const float v = sc[mt][2 * hr + j];
                    const float w = (v == -INFINITY) ? 0.f : fast_exp2(v - m_new);
                    pv[mt][2 * hr + j] = w;
                }
            m_run[j] = m_new;
            l_run[j] = l_run[j] * alpha[j];
        }
#pragma unroll
        for (int i = 0; i < KS; ++i) {
            acc[i][0] *= alpha[0];
            acc[i][1] *= alpha[1];
            acc[i][2] *= alpha[0];
            acc[i][3] *= alpha[1];
        }

        // ---- P^T fragments: hi + residual, transposed from the S layout
        uint32_t bh[2][2], bl[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float w0 = pv[mt][2 * hr], w1 = pv[mt][2 * hr + 1];
                const uint32_t hi = Ops::pack(w0, w1);
                const float2 hf = Ops::unpack(hi);
                // the sums use exactly the weights the products use
                if constexpr (kOneTermP) {
                    // binary16 weights as one term: relative error at most
                    // 2^-11, far inside the E4M3 codes' own 2^-4
                    l_run[0] += hf.x;
                    l_run[1] += hf.y;
                } else {
                    const uint32_t lo = Ops::pack(w0 - hf.x, w1 - hf.y);
                    const float2 lf = Ops::unpack(lo);
                    l_run[0] += hf.x + lf.x;
                    l_run[1] += hf.y + lf.y;
                    bl[mt][hr] = movmatrix_trans(lo);
                }
                bh[mt][hr] = movmatrix_trans(hi);
            }
        }

        // ---- O^T += V^T P^T
        if constexpr (kFp8) {
            // one 16-byte chunk = 16 d of all 32 tokens: ldmatrix.trans on byte
            // pairs gives lane (tokens 2t, 2t+1) x (d 2g, 2g+1); a byte permute
            // regroups them by d. Fragment row g <-> d 2g, row g+8 <-> d 2g+1.
#pragma unroll
            for (int md = 0; md < KS; ++md) {
                const int row = 8 * mi + r8;                        // token
                uint32_t y[4];
                ldmatrix_x4_trans(y, Vst + (md >> 3) * S::kSpanTileBytes + row * 128 +
                                         (((md & 7) ^ (row & 7)) << 4));
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const uint32_t lo = y[2 * kt], hi = y[2 * kt + 1];
                    const uint32_t a[4] = {e4m3x2_to_f16x2_scaled(__byte_perm(lo, 0u, 0x4240)),
                                           e4m3x2_to_f16x2_scaled(__byte_perm(lo, 0u, 0x4341)),
                                           e4m3x2_to_f16x2_scaled(__byte_perm(hi, 0u, 0x4240)),
                                           e4m3x2_to_f16x2_scaled(__byte_perm(hi, 0u, 0x4341))};
                    Ops::mma(acc[md], a, bh[kt][0], bh[kt][1]);
                }
            }
        } else {
#pragma unroll
            for (int md = 0; md < KS; ++md) {
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const int row = 16 * kt + (mi >> 1) * 8 + r8;      // token
                    const int c = 2 * md + (mi & 1);                    // 16-byte chunk of d
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, Vst + (c >> 3) * S::kSpanTileBytes + row * 128 +
                                             (((c & 7) ^ (row & 7)) << 4));
                    Ops::mma(acc[md], a, bh[kt][0], bh[kt][1]);
                    if constexpr (!kOneTermP) Ops::mma(acc[md], a, bl[kt][0], bl[kt][1]);
                }
            }
        }
    }
};

// The threads [tid, nthreads) share the widening of one E4M3 stage (K and V
// tiles of 32 rows, 128-byte swizzled) into binary16 tiles of the same
// swizzled layout (rows of 2 D bytes), values times 2^-8 as
// e4m3x2_to_f16x2_scaled gives them: 16 codes in, two 16-byte chunks out.
template <int D>
__device__ __forceinline__ void widen_stage_f16(const uint8_t* codes_k, const uint8_t* codes_v,
                                                uint8_t* f16_k, uint8_t* f16_v, int tid,
                                                int nthreads) {
    using S8 = TmaShape<e4m3_t, D>;
    using SF = TmaShape<__half, D>;
    constexpr int C = S8::kChunks;               // 16-code chunks per row
    constexpr int kItems = 2 * kTmaStageTokens * C;
    for (int i = tid; i < kItems; i += nthreads) {
        const int t = i / (kTmaStageTokens * C);
        const int r = (i / C) % kTmaStageTokens;
        const int c = i % C;
        const uint8_t* src = (t ? codes_v : codes_k) + (c >> 3) * S8::kSpanTileBytes + r * 128 +
                             (((c & 7) ^ (r & 7)) << 4);
        const uint4 w = *reinterpret_cast<const uint4*>(src);
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
        uint32_t out[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            out[2 * q] = e4m3x2_to_f16x2_scaled(__byte_perm(in[q], 0u, 0x4140));
            out[2 * q + 1] = e4m3x2_to_f16x2_scaled(__byte_perm(in[q], 0u, 0x4342));
        }
        uint8_t* dst = t ? f16_v : f16_k;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int cc = 2 * c + h;
            *reinterpret_cast<uint4*>(dst + (cc >> 3) * SF::kSpanTileBytes + r * 128 +
                                      (((cc & 7) ^ (r & 7)) << 4)) =
                make_uint4(out[4 * h], out[4 * h + 1], out[4 * h + 2], out[4 * h + 3]);
        }
    }
}

// Shared-prefix partitions ("TGI PagedAttention deep-dive" (lpnh.cn) sec. 5:
// requests that share a prompt prefix share its KV blocks). A unit is up to
// NCW sequences whose block tables agree over their first `parts` partitions;
// CTA (partition, KV head group, unit) reads each stage of that partition
// once, from the first valid member's table, and every consumer warp consumes
// every stage for its own member's query, so the shared blocks are read once
// per unit instead of once per sequence. These CTAs run in the partition
// kernel's own launch, ahead of the per-sequence ones (grid z = units, then
// sequences), so that the two kinds of latency-bound work overlap. Each warp
// writes its member's partials (maximum, sum, normalised output) for the
// partition itself; the partition kernel skips those partitions (skip_parts)
// and the merge is unchanged.
// A member is computed here only if its context holds the shared partitions
// and at least one more token, its skip_parts entry equals the unit's parts
// and its table agrees with the first member's over the partition; otherwise
// PA_DEV_BAD_PREFIX is set (the partition kernel computes a sequence whose
// length fails the first rule itself).
template <typename QT, typename CT, int D, int GS>
__device__ __forceinline__ void shared_unit_cta(const TmaDecodeParams& tp, uint8_t* smem, int u) {
    using S = TmaShape<CT, D>;
    using Smem = MmaSmem<CT, D>;
    constexpr bool kFp8 = std::is_same<CT, e4m3_t>::value;
    constexpr int NST = Smem::kNst;
    constexpr int NCW = Smem::kConsumers;
    constexpr int KS = D / 16;
    static_assert(GS <= 8, "one MMA covers eight heads");
    static_assert(NCW == PA_SHARED_UNIT_MEMBERS, "one consumer warp per unit member");
    const DecodeParams& p = tp.p;

    // E4M3: the codes use two ring slots; the other two hold one binary16 K/V
    // tile pair that the four warps widen each stage into once, so that the
    // unit's members do not each widen it (16-bit math from there)
    using SF = TmaShape<__half, D>;
    constexpr int NSTU = kFp8 ? 2 : NST;
    static_assert(!kFp8 || 2 * SF::kTileBytes <= (NST - NSTU) * S::kStageBytes, "staging fits");
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBarOffset);
    uint64_t* empty = full + NST;
    uint64_t* conv = empty + NST;                // the stage's binary16 tiles are complete
    uint64_t* done = conv + 1;                   // every warp has finished reading them
    uint8_t* stg_k = ring + NSTU * S::kStageBytes;
    uint8_t* stg_v = stg_k + SF::kTileBytes;

    const int part = blockIdx.x;
    const int kvh = blockIdx.y / p.sub_groups;
    const int sub = blockIdx.y - kvh * p.sub_groups;
    const int hq0 = kvh * p.group + sub * GS;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int parts = p.unit_parts[u];
    if (part >= parts) return;
    const int P = p.partition_size;
    int cap = p.max_context_len;
    {
        const long long tab = (long long)p.max_blocks * p.block_size;
        if (tab < cap) cap = (int)tab;
    }
    // a member: in range, its context holds the shared partitions and one more
    // token, and its own skip count names this unit's partitions
    auto member_ok = [&](int m) {
        if (m < 0 || m >= p.num_seqs) return false;
        const int L = p.context_lens[m];
        return L > (long long)parts * P && L <= cap && p.skip_parts[m] == parts;
    };
    // the first valid member's table names the blocks the unit reads
    int leader = -1;
    for (int w = 0; w < NCW && leader < 0; ++w) {
        const int cand = p.unit_seqs[(size_t)u * NCW + w];
        if (member_ok(cand)) leader = cand;
    }
    if (leader < 0) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, PA_DEV_BAD_PREFIX);
        return;
    }
    const int T0 = part * P;
    const int n_st = P / kTmaStageTokens;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTU; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);           // every consumer reads every stage
        }
        mbar_init(conv, NCW);
        mbar_init(done, NCW);
        fence_barrier_init();
    }
    __syncthreads();

    const int32_t* lead_table = p.block_tables + (size_t)leader * p.max_blocks;
    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        const int B = p.block_size;
        const int rows = tp.box_rows;
        if (lane == 0) {
            tma_prefetch_map(&tp.k_map);
            tma_prefetch_map(&tp.v_map);
        }
        int issued = 0;
        for (int k = 0; k < n_st; ++k) {
            const int slot = k % NSTU;
            if (k >= NSTU) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&empty[slot], ((k / NSTU) - 1) & 1, p.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            const int t_lo = T0 + k * kTmaStageTokens;
            const int t_hi = t_lo + kTmaStageTokens;
            const int j0 = t_lo / B;
            const int nseg = (t_hi - 1) / B - j0 + 1;
            uint32_t bytes = 0;
            int y = 0, row0 = 0;
            if (lane < nseg) {
                const int j = j0 + lane;
                const int pb = lead_table[j];
                if (pb < 0 || (int64_t)pb >= p.num_blocks) {
                    if (p.status) atomicOr(p.status, PA_DEV_BAD_BLOCK_ID);
                } else {
                    const int off = (B >= kTmaStageTokens) ? (t_lo - j * B) : 0;
                    y = (pb * p.num_kv_heads + kvh) * B + off;
                    row0 = (B >= kTmaStageTokens) ? 0 : j * B - t_lo;
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
                    uint8_t* kd = st + sp * S::kSpanTileBytes + row0 * 128;
                    tma_load_2d(kd, &tp.k_map, x, y, &full[slot]);
                    tma_load_2d(kd + S::kTileBytes, &tp.v_map, x, y, &full[slot]);
                }
            }
            issued = k + 1;
        }
        if (lane == 0) {
            for (int k = max(0, issued - NSTU); k < issued; ++k)
                mbar_wait_bounded(&full[k % NSTU], (k / NSTU) & 1, p.status);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int m = p.unit_seqs[(size_t)u * NCW + warp];
    bool active = member_ok(m);
    if (active && m != leader) {
        // the member's table must name the leader's blocks over the partition
        const int B = p.block_size;
        const int32_t* t = p.block_tables + (size_t)m * p.max_blocks;
        bool same = true;
        for (int j = T0 / B + lane; j < (T0 + P + B - 1) / B; j += 32) same &= t[j] == lead_table[j];
        active = __all_sync(0xffffffffu, same);
    }
    if (!active && m >= 0 && lane == 0 && p.status) atomicOr(p.status, PA_DEV_BAD_PREFIX);
    using Warp = std::conditional_t<kFp8, MmaWarp<__half, __half, D, GS, true>,
                                    MmaWarp<QT, CT, D, GS>>;
    Warp cw;
    if (active) {
        const QT* qp = reinterpret_cast<const QT*>(p.query) + ((size_t)m * p.num_q_heads + hq0) * D;
        if constexpr (kFp8) cw.load_query_as(qp, p.q_mul * 256.f, lane);   // widened values are 2^-8 x
        else cw.load_query(qp, p.q_mul, lane);
    }
    bool ok = true;
    for (int k = 0; k < n_st; ++k) {
        const int slot = k % NSTU;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (k / NSTU) & 1, p.status));
        if (!ok) break;
        uint8_t* Kst = ring + (size_t)slot * S::kStageBytes;
        if constexpr (kFp8) {
            if (k > 0) {                         // the previous stage's tiles have been read
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(done, (k - 1) & 1, p.status));
                if (!ok) break;
            }
            widen_stage_f16<D>(Kst, Kst + S::kTileBytes, stg_k, stg_v, threadIdx.x, NCW * 32);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(conv);
                mbar_arrive(&empty[slot]);       // the codes' slot may be refilled
            }
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(conv, k & 1, p.status));
            if (!ok) break;
            if (active) cw.consume(stg_k, stg_v, kTmaStageTokens, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(done);
        } else {
            if (active) cw.consume(Kst, Kst + S::kTileBytes, kTmaStageTokens, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    if (!active || !ok) return;

    // ---------------------------------------------- this member's partials
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        cw.l_run[j] += __shfl_xor_sync(0xffffffffu, cw.l_run[j], 4);
        cw.l_run[j] += __shfl_xor_sync(0xffffffffu, cw.l_run[j], 8);
        cw.l_run[j] += __shfl_xor_sync(0xffffffffu, cw.l_run[j], 16);
    }
    const int g = lane >> 2;
    const int t4 = lane & 3;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int h = 2 * t4 + j;
        if (h >= GS) continue;
        const size_t row = ((size_t)m * p.num_q_heads + hq0 + h) * p.max_parts + part;
        const float inv = (kFp8 ? p.v_mul * 256.f : p.v_mul) / cw.l_run[j];
#pragma unroll
        for (int md = 0; md < KS; ++md)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int d = 16 * md + g + 8 * hr;          // 16-bit math: natural order
                p.tmp_out[row * D + d] = cw.acc[md][2 * hr + j] * inv;
            }
        if (g == 0) {
            p.max_logits[row] = cw.m_run[j] * kLn2;
            p.exp_sums[row] = cw.l_run[j];
        }
    }
}

// kShared: a split launch with shared-prefix units (grid z: units, then
// sequences); a separate instantiation, so that the plain kernels carry
// neither the unit path nor the skip test.
template <typename QT, typename CT, int D, int GS, bool kSplit, bool kShared = false>
__global__ void __launch_bounds__(mma_threads<CT, D>(), mma_min_blocks<CT, D>())
paged_decode_mma_kernel(const __grid_constant__ TmaDecodeParams tp) {
    using S = TmaShape<CT, D>;
    using Smem = MmaSmem<CT, D>;
    constexpr bool kFp8 = std::is_same<CT, e4m3_t>::value;
    constexpr int NST = Smem::kNst;
    constexpr int NCW = Smem::kConsumers;
    static_assert(NST % NCW == 0, "one owner per slot");
    constexpr int KS = D / 16;                 // k-steps of the score product
    static_assert(GS <= 8, "one MMA covers eight heads");
    const DecodeParams& p = tp.p;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBarOffset);
    uint64_t* empty = full + NST;

    int zs = blockIdx.z;
    if constexpr (kShared) {
        static_assert(kSplit, "units are partitions");
        if (zs < p.num_units) {                 // a shared-prefix unit (grid z: units first)
            shared_unit_cta<QT, CT, D, GS>(tp, smem, zs);
            return;
        }
        zs -= p.num_units;
    }
    const int s = zs;
    const int kvh = blockIdx.y / p.sub_groups;
    const int sub = blockIdx.y - kvh * p.sub_groups;
    const int hq0 = kvh * p.group + sub * GS;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;                   // fragment row / B column
    const int t4 = lane & 3;                   // fragment column pair

    int L = p.context_lens[s];
    {
        int cap = p.max_context_len;
        const long long tab = (long long)p.max_blocks * p.block_size;
        if (tab < cap) cap = (int)tab;
        if (L < 0 || L > cap) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && sub == 0 && p.status)
                atomicOr(p.status, PA_DEV_BAD_LEN);
            L = L < 0 ? 0 : cap;
        }
    }
    int T0, Tend;
    if constexpr (kSplit) {
        if (kShared && p.skip_parts) {
            // partitions this launch's unit CTAs compute for this sequence
            // (their rule: the context extends past them and is within the bound)
            const int sk = p.skip_parts[s];
            const int Lr = p.context_lens[s];
            if (sk > 0 && (int)blockIdx.x < sk && Lr > (long long)sk * p.partition_size &&
                Lr <= p.max_context_len && Lr <= (long long)p.max_blocks * p.block_size)
                return;
        }
        T0 = blockIdx.x * p.partition_size;
        if (T0 >= L) return;
        Tend = min(T0 + p.partition_size, L);
    } else {
        T0 = 0;
        Tend = L;
        if (L == 0) {
            QT* out = reinterpret_cast<QT*>(p.out);
            for (int i = threadIdx.x; i < GS * D; i += blockDim.x)
                out[((size_t)s * p.num_q_heads + hq0) * D + i] = from_float<QT>(0.f);
            return;
        }
    }
    const int n_st = (Tend - T0 + kTmaStageTokens - 1) / kTmaStageTokens;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        const int B = p.block_size;
        const int rows = tp.box_rows;
        const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
        if (lane == 0) {
            tma_prefetch_map(&tp.k_map);
            tma_prefetch_map(&tp.v_map);
        }
        // the fused write of position L - 1 (in stage kw of this range): its
        // stores go out once the ring's first stages are issued, overlapping
        // the wait for a free slot, and the fence right before stage kw's copy
        const bool writes = p.new_key && L - 1 >= T0 && L - 1 < Tend;
        const int kw = writes ? (L - 1 - T0) / kTmaStageTokens : -1;
        const int kstore = kw < NST ? kw : NST;
        int issued = 0;
        for (int k = 0; k < n_st; ++k) {
            const int slot = k % NST;
            if (k == kstore) fused_store_token<QT, CT, D>(p, s, kvh, L, lane);
            if (k >= NST) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&empty[slot], ((k / NST) - 1) & 1, p.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            const int t_lo = T0 + k * kTmaStageTokens;
            const int t_hi = min(t_lo + kTmaStageTokens, Tend);
            if (k == kw) fused_write_fence();
            const int j0 = t_lo / B;
            const int nseg = (t_hi - 1) / B - j0 + 1;
            uint32_t bytes = 0;
            int y = 0, row0 = 0;
            if (lane < nseg) {
                const int j = j0 + lane;
                const int pb = table[j];
                if (pb < 0 || (int64_t)pb >= p.num_blocks) {
                    if (p.status) atomicOr(p.status, PA_DEV_BAD_BLOCK_ID);
                } else {
                    const int off = (B >= kTmaStageTokens) ? (t_lo - j * B) : 0;
                    y = (pb * p.num_kv_heads + kvh) * B + off;
                    row0 = (B >= kTmaStageTokens) ? 0 : j * B - t_lo;
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
                    uint8_t* kd = st + sp * S::kSpanTileBytes + row0 * 128;
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
        return;
    }

    // ---------------------------------------------------------------- consumers
    MmaWarp<QT, CT, D, GS> cw;
    cw.load_query(reinterpret_cast<const QT*>(p.query) + ((size_t)s * p.num_q_heads + hq0) * D,
                  p.q_mul, lane);

    for (int k = warp; k < n_st; k += NCW) {
        const int slot = k % NST;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (k / NST) & 1, p.status));
        if (!ok) break;
        uint8_t* Kst = ring + (size_t)slot * S::kStageBytes;
        uint8_t* Vst = Kst + S::kTileBytes;
        const int nvalid = min(kTmaStageTokens, Tend - (T0 + k * kTmaStageTokens));
        if (nvalid < kTmaStageTokens) {
            // rows past the context: zero V so that 0-weights stay 0 in the MMA
            const int n16 = (kTmaStageTokens - nvalid) * S::kRowBytes / 16;
            for (int i = lane; i < n16; i += 32) {
                const int row = nvalid + i / (S::kRowBytes / 16);
                const int c = i % (S::kRowBytes / 16);
                *reinterpret_cast<uint4*>(Vst + (c >> 3) * S::kSpanTileBytes + row * 128 + ((c & 7) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        cw.consume(Kst, Vst, nvalid, lane);
        if (nvalid < kTmaStageTokens) {
            // the generic-proxy zeroing must be ordered before the next bulk copy into this slot
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ------------------------------------------------- merge the four warps
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        cw.l_run[j] += __shfl_xor_sync(0xffffffffu, cw.l_run[j], 4);
        cw.l_run[j] += __shfl_xor_sync(0xffffffffu, cw.l_run[j], 8);
        cw.l_run[j] += __shfl_xor_sync(0xffffffffu, cw.l_run[j], 16);
    }
    named_barrier(1, NCW * 32);    // ring is free: every stage was consumed
    float* cm = reinterpret_cast<float*>(smem);                 // [NCW][8]
    float* cl = cm + NCW * 8;                                   // [NCW][8]
    float* co = cl + NCW * 8;                                   // [NCW][8][D]
    if (g == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            cm[warp * 8 + 2 * t4 + j] = cw.m_run[j];
            cl[warp * 8 + 2 * t4 + j] = cw.l_run[j];
        }
    }
#pragma unroll
    for (int md = 0; md < KS; ++md) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = 2 * t4 + j;
                const int d = kFp8 ? 16 * md + 2 * g + hr : 16 * md + g + 8 * hr;
                if (h < GS) co[(warp * 8 + h) * D + d] = cw.acc[md][2 * hr + j];
            }
    }
    named_barrier(1, NCW * 32);

    for (int i = threadIdx.x; i < GS * D; i += NCW * 32) {
        const int h = i / D;
        const int e = i - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, cm[w * 8 + h]);
        float W = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float mw = cm[w * 8 + h];
            const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
            W = fmaf(f, cl[w * 8 + h], W);
            O = fmaf(f, co[(w * 8 + h) * D + e], O);
        }
        const float val = __fdiv_rn(O, W) * (kFp8 ? p.v_mul * 256.f : p.v_mul);
        const int hq = hq0 + h;
        if constexpr (kSplit) {
            const size_t row = ((size_t)s * p.num_q_heads + hq) * p.max_parts + blockIdx.x;
            p.tmp_out[row * D + e] = val;
            if (e == 0) {
                p.max_logits[row] = M * kLn2;
                p.exp_sums[row] = W;
            }
        } else {
            QT* out = reinterpret_cast<QT*>(p.out);
            out[((size_t)s * p.num_q_heads + hq) * D + e] = from_float<QT>(val);
        }
    }
}

template <typename QT, typename CT, int D, int GS, bool kSplit, bool kShared = false>
cudaError_t launch_mma_variant(const TmaDecodeParams& tp, cudaStream_t stream) {
    using Smem = MmaSmem<CT, D>;
    auto kern = paged_decode_mma_kernel<QT, CT, D, GS, kSplit, kShared>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Smem::kAlloc);
    if (e != cudaSuccess) return e;
    const DecodeParams& p = tp.p;
    dim3 grid(kSplit ? p.max_parts : 1, p.num_kv_heads * p.sub_groups,
              p.num_seqs + (kShared ? p.num_units : 0));
    kern<<<grid, mma_threads<CT, D>(), Smem::kAlloc, stream>>>(tp);
    return cudaGetLastError();
}

template <typename QT, typename CT, int D>
cudaError_t launch_mma_d(const TmaDecodeParams& tp, int gs, bool split, cudaStream_t stream) {
#define PA_MMA_CASE(G)                                                        \
    case G:                                                                   \
        if (split && tp.p.num_units > 0)                                      \
            return launch_mma_variant<QT, CT, D, G, true, true>(tp, stream);  \
        return split ? launch_mma_variant<QT, CT, D, G, true>(tp, stream)     \
                     : launch_mma_variant<QT, CT, D, G, false>(tp, stream);
    switch (gs) {
        PA_MMA_CASE(1)
        PA_MMA_CASE(2)
        PA_MMA_CASE(4)
        PA_MMA_CASE(8)
    }
#undef PA_MMA_CASE
    return cudaErrorInvalidValue;
}

// Query type QT (16-bit); cache CT of the same type, or E4M3 codes; rows of
// 128, 256 or 512 bytes; heads_per_unit 1, 2, 4 or 8.
template <typename QT, typename CT>
cudaError_t launch_mma(const DecodeParams& p, int head_size, int gs, bool split,
                       cudaStream_t stream) {
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
        case 64: return launch_mma_d<QT, CT, 64>(tp, gs, split, stream);
        case 128: return launch_mma_d<QT, CT, 128>(tp, gs, split, stream);
        case 256: return launch_mma_d<QT, CT, 256>(tp, gs, split, stream);
        }
    } else {
        switch (head_size) {
        case 128: return launch_mma_d<QT, CT, 128>(tp, gs, split, stream);
        case 256: return launch_mma_d<QT, CT, 256>(tp, gs, split, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace pagedkv
