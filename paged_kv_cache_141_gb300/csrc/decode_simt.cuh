// decode_simt.cuh -- the generic paged decode kernel (CUDA cores).
//
// One CTA computes one work unit: a sequence, a group of GS query heads that
// share one KV head, and a token range (the whole context for the single-pass
// decode, or one partition for the split decode, cf. "TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 4.1, PagedAttention V1/V2).
//
// Data movement. Warp 4 is a producer: it walks the sequence's block table
// ("Lecture 3: PagedAttention and vLLM", "the paged implementation of
// attention": logical block -> physical block) and, for each 32-token stage,
// issues one bulk copy (the TMA engine, cp.async.bulk) per block segment for K
// and for V into a ring of NST shared-memory stages, completing on the stage's
// mbarrier. Each lane copies one block segment, so a stage that spans 32 blocks
// of one token (block_size 1) is issued in one warp instruction.
//
// Math. Warps 0-3 are consumers; warp w takes tokens 8w..8w+7 of every stage
// and keeps its own online softmax (running max m, running sum l, running
// output o) per query head. Lane l owns head_size/32 consecutive components of
// every row. A pass scores TOK tokens x GS heads: each lane forms partial dot
// products over its components, and a transposing butterfly (each step sends
// half of the remaining values to the partner lane and adds the half it
// receives) leaves one finished score per lane, with 31 shuffles for 32
// scores. Softmax weights go through a per-warp shared buffer to the P.V loop,
// in which each lane accumulates its components for all GS heads. At the end
// the four warps' (m, l, o) are merged with the max / sum-exp rule.
//
// Scores are kept in base 2: q is pre-multiplied by scale * log2(e), so
// exp(s - m) = 2^(s2 - m2); the workspace stores natural-log maxima.
#pragma once

#include "device_common.cuh"
#include "kv_store.cuh"
#include "launch.h"

namespace pagedkv {

constexpr int kConsumerWarps = 4;
constexpr int kStageTokens = 32;
constexpr int kTokensPerWarp = kStageTokens / kConsumerWarps;   // 8
constexpr int kSimtThreads = (kConsumerWarps + 1) * 32;         // 160

template <typename CT, int D>
struct SimtShape {
    static constexpr int kRowBytes = D * TypeInfo<CT>::bytes;
    static constexpr int kStageBytes = 2 * kStageTokens * kRowBytes;      // K then V
    static constexpr int kRingTarget = 64 * 1024;
    static constexpr int kNst0 = kRingTarget / kStageBytes;
    static constexpr int kNst = kNst0 < 2 ? 2 : (kNst0 > 8 ? 8 : kNst0);
    static constexpr int kRingBytes = kNst * kStageBytes;
};

template <int GS>
struct SimtScratch {
    // per consumer warp: softmax weights of one pass, and the rescale factors
    float p[kConsumerWarps][kTokensPerWarp][GS];
    float alpha[kConsumerWarps][GS];
};

template <typename CT, int D, int GS>
struct SimtSmem {
    using Shape = SimtShape<CT, D>;
    static constexpr int kCombineBytes = kConsumerWarps * GS * (D + 2) * 4;
    static constexpr int kBody = Shape::kRingBytes > kCombineBytes ? Shape::kRingBytes : kCombineBytes;
    static constexpr int kBarOffset = (kBody + 127) / 128 * 128;
    static constexpr int kScratchOffset = kBarOffset + 2 * Shape::kNst * 8;
    static constexpr int kBytes = kScratchOffset + (int)sizeof(SimtScratch<GS>);
};

// Transposing butterfly: N partial values per lane (N a power of two, <= 32).
// Returns the full sum of value index idx = lane >> (5 - log2 N); lanes that
// share idx hold the same sum.
template <int N, int M>
__device__ __forceinline__ void transpose_reduce(float* v, int lane) {
    if constexpr (M >= 1) {
        if constexpr (N > 1) {
            constexpr int H = N / 2;
            const bool up = (lane & M) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = up ? v[i] : v[i + H];
                const float keep = up ? v[i + H] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            transpose_reduce<H, M / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
            transpose_reduce<1, M / 2>(v, lane);
        }
    }
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <typename QT, typename CT, int D, int GS, bool kSplit>
__global__ void __launch_bounds__(kSimtThreads)
paged_decode_simt_kernel(const DecodeParams p) {
    using Shape = SimtShape<CT, D>;
    using Smem = SimtSmem<CT, D, GS>;
    constexpr int NST = Shape::kNst;
    constexpr int EPL = D / 32;                                   // components per lane
    constexpr int TOK = (32 / GS) < kTokensPerWarp ? (32 / GS) : kTokensPerWarp;
    constexpr int NV = TOK * GS;                                  // values per pass
    constexpr int SHIFT = 5 - ilog2(NV);                          // lane -> value index
    constexpr int GSB = ilog2(GS);
    constexpr int TOKEN_MASK_LO = 1 << (SHIFT + GSB);             // lowest lane bit of the token
    constexpr int PASSES = kTokensPerWarp / TOK;

    extern __shared__ __align__(128) uint8_t smem[];
    CT* ring = reinterpret_cast<CT*>(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBarOffset);
    uint64_t* empty = full + NST;
    SimtScratch<GS>& scr = *reinterpret_cast<SimtScratch<GS>*>(smem + Smem::kScratchOffset);

    int s = blockIdx.z;
    size_t qrow = (size_t)s;                                      // row of query / out
    const int kvh = blockIdx.y / p.sub_groups;
    const int sub = blockIdx.y - kvh * p.sub_groups;
    const int hq0 = kvh * p.group + sub * GS;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // context length, clamped to what the table and the grid can cover
    int L;
    int cap = p.max_context_len;
    {
        const long long tab = (long long)p.max_blocks * p.block_size;
        if (tab < cap) cap = (int)tab;
    }
    if constexpr (!kSplit) {
        if (p.query_start) {
            // multi-query: blockIdx.x is a query token; its sequence is the
            // last s with query_start[s] <= token
            const int t = blockIdx.x;
            qrow = (size_t)t;
            int lo = 0, hi = p.num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.query_start[mid] <= t) lo = mid;
                else hi = mid - 1;
            }
            s = lo;
            const int qs0 = p.query_start[s], qs1 = p.query_start[s + 1];
            const int Ls = p.context_lens[s];
            if (t < qs0 || t >= qs1 || Ls > cap || qs1 - qs0 > Ls) {
                if (threadIdx.x == 0 && sub == 0 && p.status) atomicOr(p.status, PA_DEV_BAD_LEN);
                return;
            }
            L = Ls - (qs1 - qs0) + (t - qs0) + 1;
        }
    }
    if (kSplit || !p.query_start) {
        L = p.context_lens[s];
        if (L < 0 || L > cap) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && sub == 0 && p.status)
                atomicOr(p.status, PA_DEV_BAD_LEN);
            L = L < 0 ? 0 : cap;
        }
    }
    int T0, Tend;
    if constexpr (kSplit) {
        T0 = blockIdx.x * p.partition_size;
        if (T0 >= L) return;                                      // no such partition
        Tend = min(T0 + p.partition_size, L);
    } else {
        T0 = 0;
        Tend = L;
        if (L == 0) {                                             // empty context: zeros
            QT* out = reinterpret_cast<QT*>(p.out);
            for (int i = threadIdx.x; i < GS * D; i += blockDim.x)
                out[(qrow * p.num_q_heads + hq0) * D + i] = from_float<QT>(0.f);
            return;
        }
    }
    const int n_st = (Tend - T0 + kStageTokens - 1) / kStageTokens;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const int B = p.block_size;
        const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
        const CT* kbase = reinterpret_cast<const CT*>(p.k_cache);
        const CT* vbase = reinterpret_cast<const CT*>(p.v_cache);
        int issued = 0;
        for (int k = 0; k < n_st; ++k) {
            const int slot = k % NST;
            if (k >= NST) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&empty[slot], ((k / NST) - 1) & 1, p.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            const int t_lo = T0 + k * kStageTokens;
            const int t_hi = min(t_lo + kStageTokens, Tend);
            if (p.new_key && L - 1 >= t_lo && L - 1 < t_hi)
                fused_write_token<QT, CT, D>(p, s, kvh, L, lane);
            const int j0 = t_lo / B;
            const int nseg = (t_hi - 1) / B - j0 + 1;             // <= 32
            uint32_t bytes = 0;
            int seg_lo = 0, pb = 0, j = 0;
            if (lane < nseg) {
                j = j0 + lane;
                seg_lo = max(t_lo, j * B);
                const int seg_hi = min(t_lo + kStageTokens, (j + 1) * B);
                pb = table[j];
                if (pb < 0 || (int64_t)pb >= p.num_blocks) {
                    if (p.status) atomicOr(p.status, PA_DEV_BAD_BLOCK_ID);
                } else {
                    bytes = (uint32_t)(seg_hi - seg_lo) * Shape::kRowBytes;
                }
            }
            uint32_t total = bytes;
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) total += __shfl_xor_sync(0xffffffffu, total, m);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2 * total);
            __syncwarp();
            if (bytes) {
                uint8_t* stage = reinterpret_cast<uint8_t*>(ring) + (size_t)slot * Shape::kStageBytes;
                const size_t src = (((size_t)pb * p.num_kv_heads + kvh) * B + (seg_lo - j * B)) * D;
                const int row = seg_lo - t_lo;
                bulk_copy_g2s(stage + row * Shape::kRowBytes, kbase + src, bytes, &full[slot]);
                bulk_copy_g2s(stage + (kStageTokens + row) * Shape::kRowBytes, vbase + src, bytes,
                              &full[slot]);
            }
            issued = k + 1;
        }
        // drain: this CTA does not exit while a copy it issued is in flight
        if (lane == 0) {
            for (int k = max(0, issued - NST); k < issued; ++k)
                mbar_wait_bounded(&full[k % NST], (k / NST) & 1, p.status);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    float q[GS][EPL];
    {
        const QT* qp = reinterpret_cast<const QT*>(p.query) + (qrow * p.num_q_heads + hq0) * D;
#pragma unroll
        for (int h = 0; h < GS; ++h) {
            float x[EPL];
            RowLoader<QT, EPL>::load(qp + h * D + lane * EPL, x);
#pragma unroll
            for (int e = 0; e < EPL; ++e) q[h][e] = x[e] * p.q_mul;
        }
    }
    float o[GS][EPL];
#pragma unroll
    for (int h = 0; h < GS; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;

    const int idx = lane >> SHIFT;             // this lane's value index in a pass
    const int my_t = idx >> GSB;               // token within the pass
    const int my_h = idx & (GS - 1);           // head within the group
    const bool canonical = (lane & ((1 << SHIFT) - 1)) == 0;
    float m_run = -INFINITY;                   // running max (base 2) of head my_h
    float l_run = 0.f;                         // this lane's share of the running sum

    for (int k = 0; k < n_st; ++k) {
        const int slot = k % NST;
        // every lane acquires the stage itself: the bulk copies wrote it
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (k / NST) & 1, p.status));
        if (!ok) break;

        const CT* Ks = ring + (size_t)slot * (Shape::kStageBytes / TypeInfo<CT>::bytes);
        const CT* Vs = Ks + kStageTokens * D;
        const int nvalid = min(kStageTokens, Tend - (T0 + k * kStageTokens));
        const int wbase = warp * kTokensPerWarp;

#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass) {
            const int tb = wbase + pass * TOK;
            const int nv = min(TOK, nvalid - tb);
            if (nv <= 0) break;                                   // warp-uniform

            float acc[NV];
#pragma unroll
            for (int t = 0; t < TOK; ++t) {
                float kx[EPL];
                RowLoader<CT, EPL>::load(Ks + (tb + t) * D + lane * EPL, kx);
#pragma unroll
                for (int h = 0; h < GS; ++h) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) a = fmaf(q[h][e], kx[e], a);
                    acc[t * GS + h] = a;
                }
            }
            transpose_reduce<NV, 16>(acc, lane);
            const float sc = (my_t < nv) ? acc[0] : -INFINITY;   // select, never multiply
            float mx = sc;
#pragma unroll
            for (int m = TOKEN_MASK_LO; m <= 16; m <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
            const float pw = (sc == -INFINITY) ? 0.f : fast_exp2(sc - m_new);
            l_run = l_run * alpha + (canonical ? pw : 0.f);
            m_run = m_new;
            scr.p[warp][my_t][my_h] = pw;
            if (my_t == 0) scr.alpha[warp][my_h] = alpha;
            __syncwarp();
#pragma unroll
            for (int h = 0; h < GS; ++h) {
                const float a = scr.alpha[warp][h];
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[h][e] *= a;
            }
            for (int t = 0; t < nv; ++t) {
                float vx[EPL];
                RowLoader<CT, EPL>::load(Vs + (tb + t) * D + lane * EPL, vx);
#pragma unroll
                for (int h = 0; h < GS; ++h) {
                    const float pw_t = scr.p[warp][t][h];
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(pw_t, vx[e], o[h][e]);
                }
            }
            __syncwarp();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ------------------------------------------------- merge the four warps
    float l_sum = l_run;
#pragma unroll
    for (int m = TOKEN_MASK_LO; m <= 16; m <<= 1) l_sum += __shfl_xor_sync(0xffffffffu, l_sum, m);
    // every stage's copies have landed, so the ring is free for the merge
    named_barrier(1, kConsumerWarps * 32);
    float* cm = reinterpret_cast<float*>(smem);                  // [4][GS]
    float* cl = cm + kConsumerWarps * GS;                        // [4][GS]
    float* co = cl + kConsumerWarps * GS;                        // [4][GS][D]
    if (canonical && my_t == 0) {
        cm[warp * GS + my_h] = m_run;
        cl[warp * GS + my_h] = l_sum;
    }
#pragma unroll
    for (int h = 0; h < GS; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) co[(warp * GS + h) * D + lane * EPL + e] = o[h][e];
    named_barrier(1, kConsumerWarps * 32);

    for (int i = threadIdx.x; i < GS * D; i += kConsumerWarps * 32) {
        const int h = i / D;
        const int e = i - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w * GS + h]);
        // o of each warp is unnormalised (sum of 2^(s - m_w) v), so it is
        // rescaled by 2^(m_w - M) alone; the sums l_w get the same factor.
        float W = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = cm[w * GS + h];
            const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
            W = fmaf(f, cl[w * GS + h], W);
            O = fmaf(f, co[(w * GS + h) * D + e], O);
        }
        const float val = __fdiv_rn(O, W) * p.v_mul;
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
            out[(qrow * p.num_q_heads + hq) * D + e] = from_float<QT>(val);
        }
    }
}

template <typename QT, typename CT, int D, int GS, bool kSplit>
cudaError_t launch_simt_variant(const DecodeParams& p, cudaStream_t stream) {
    using Smem = SimtSmem<CT, D, GS>;
    auto kern = paged_decode_simt_kernel<QT, CT, D, GS, kSplit>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Smem::kBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.query_start ? p.num_queries : (kSplit ? p.max_parts : 1),
              p.num_kv_heads * p.sub_groups, p.query_start ? 1 : p.num_seqs);
    kern<<<grid, kSimtThreads, Smem::kBytes, stream>>>(p);
    return cudaGetLastError();
}

template <typename QT, typename CT, int D>
cudaError_t launch_simt_d(const DecodeParams& p, int gs, bool split, cudaStream_t stream) {
    switch (gs) {
    case 1: return split ? launch_simt_variant<QT, CT, D, 1, true>(p, stream)
                         : launch_simt_variant<QT, CT, D, 1, false>(p, stream);
    case 2: return split ? launch_simt_variant<QT, CT, D, 2, true>(p, stream)
                         : launch_simt_variant<QT, CT, D, 2, false>(p, stream);
    case 4: return split ? launch_simt_variant<QT, CT, D, 4, true>(p, stream)
                         : launch_simt_variant<QT, CT, D, 4, false>(p, stream);
    case 8:
        if constexpr (D <= 128)
            return split ? launch_simt_variant<QT, CT, D, 8, true>(p, stream)
                         : launch_simt_variant<QT, CT, D, 8, false>(p, stream);
        break;
    }
    return cudaErrorInvalidValue;
}

template <typename QT, typename CT>
cudaError_t launch_simt(const DecodeParams& p, int head_size, int gs, bool split,
                        cudaStream_t stream) {
    switch (head_size) {
    case 64: return launch_simt_d<QT, CT, 64>(p, gs, split, stream);
    case 128: return launch_simt_d<QT, CT, 128>(p, gs, split, stream);
    case 256: return launch_simt_d<QT, CT, 256>(p, gs, split, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pagedkv
