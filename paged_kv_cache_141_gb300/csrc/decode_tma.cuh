// decode_tma.cuh -- the paged decode kernel for the common shapes (rows of
// 128, 256 or 512 bytes, block sizes that are multiples of 8).
//
// One CTA computes one work unit: a sequence, a group of GS query heads that
// share one KV head, and a token range (the whole context for the single-pass
// decode, or one partition of the split decode; "TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 4.1, PagedAttention V1/V2).
//
// Data movement. Warp 4 walks the block table ("Lecture 3: PagedAttention and
// vLLM", "the paged implementation of attention": logical block -> physical
// block) and loads each 32-token stage of K and V with tensor TMA copies
// (cp.async.bulk.tensor, one box per block segment and 128-byte column span)
// into shared memory in the 128-byte swizzled layout: row r's 16-byte chunk c
// sits at chunk c ^ (r mod 8). Stage k belongs to consumer warp k mod 4, and
// each ring slot is only ever used by one warp.
//
// Math. In a stage, lane t owns token t: it reads its own K row chunk by chunk
// (the swizzle makes the 32 lanes' reads of one chunk conflict-free) against
// the query group, which sits in shared memory as float32 and is read as a
// broadcast; products accumulate in packed FP32x2 FMAs. No cross-lane
// reduction is needed for the scores. Each warp keeps its own online softmax
// (base 2) per head; weights go through a per-warp buffer to the P.V loop, in
// which lane l owns head_size/32 components and a packed accumulator holds the
// even- and odd-token partial sums of each component. At the end the four
// warps' (max, sum, output) are merged.
#pragma once

#include <cuda.h>

#include "device_common.cuh"
#include "kv_store.cuh"
#include "launch.h"

namespace pagedkv {

// Shared-memory ring per CTA (bytes); with 64 KB, three CTAs fit on an SM.
#ifndef PA_TMA_RING_BYTES
#define PA_TMA_RING_BYTES (64 * 1024)
#endif

constexpr int kTmaConsumerWarps = 4;
constexpr int kTmaThreads = (kTmaConsumerWarps + 1) * 32;
constexpr int kTmaStageTokens = 32;

template <typename CT, int D>
struct TmaShape {
    static constexpr int kElem = TypeInfo<CT>::bytes;
    static constexpr int kRowBytes = D * kElem;                 // 128, 256 or 512
    static constexpr int kSpans = kRowBytes / 128;              // 128-byte swizzle spans
    static constexpr int kSpanTileBytes = kTmaStageTokens * 128;
    static constexpr int kTileBytes = kTmaStageTokens * kRowBytes;  // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kNst0 = PA_TMA_RING_BYTES / kStageBytes;
    static constexpr int kNst = kNst0 < 2 ? 2 : (kNst0 > 8 ? 8 : kNst0);
    static constexpr int kRingBytes = kNst * kStageBytes;
    static constexpr int kChunks = kRowBytes / 16;              // 16-byte chunks per row
    static constexpr int kChunksPerWarp = kChunks / kTmaConsumerWarps;
    static constexpr int kEpc = 16 / kElem;                     // elements per chunk
    static constexpr int kEpl = D / 32;                         // P.V components per lane
    static_assert(kRowBytes == 128 || kRowBytes == 256 || kRowBytes == 512, "row bytes");
    static_assert(kChunksPerWarp >= 1, "chunks");
};

constexpr int kTmaTokensPerWarp = kTmaStageTokens / kTmaConsumerWarps;   // 8

template <typename CT, int D, int GS>
struct TmaSmem {
    using S = TmaShape<CT, D>;
    static constexpr int kQBytes = D * GS * 4;                                      // q, float32
    static constexpr int kPartBytes = 2 * kTmaConsumerWarps * kTmaStageTokens * GS * 4;  // partial scores
    static constexpr int kPBytes = kTmaConsumerWarps * GS * kTmaTokensPerWarp * 4;      // weights
    static constexpr int kABytes = kTmaConsumerWarps * GS * 4;                          // rescales
    static constexpr int kCombineBytes = kTmaConsumerWarps * GS * (D + 2) * 4;
    static constexpr int kBody = S::kRingBytes > kCombineBytes ? S::kRingBytes : kCombineBytes;
    static constexpr int kQOffset = (kBody + 127) / 128 * 128;
    static constexpr int kPartOffset = kQOffset + kQBytes;
    static constexpr int kPOffset = kPartOffset + kPartBytes;
    static constexpr int kAOffset = kPOffset + kPBytes;
    static constexpr int kBarOffset = (kAOffset + kABytes + 7) / 8 * 8;
    static constexpr int kBytes = kBarOffset + 2 * S::kNst * 8;
    static constexpr int kAlloc = kBytes + 1024;                // room to align the ring to 1 KB
};

// Parameters of the TMA decode: the generic ones plus the two tensor maps.
struct TmaDecodeParams {
    DecodeParams p;
    CUtensorMap k_map;   // K pool viewed as [num_blocks*Hkv*B rows][D], box [128 B][rows]
    CUtensorMap v_map;
    int box_rows;        // min(block_size, 32)
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 16 bytes of stored elements widened to float2 pairs (consecutive elements).
template <typename CT> struct Widen16;
template <> struct Widen16<float> {
    static constexpr int kPairs = 2;
    __device__ __forceinline__ static void run(const uint4& w, float2 (&f)[2]) {
        f[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
        f[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
};
template <> struct Widen16<__nv_bfloat16> {
    static constexpr int kPairs = 4;
    __device__ __forceinline__ static void run(const uint4& w, float2 (&f)[4]) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)   // bfloat16 -> float32 is a 16-bit shift
            f[i] = make_float2(__uint_as_float(ws[i] << 16), __uint_as_float(ws[i] & 0xffff0000u));
    }
};
template <> struct Widen16<__half> {
    static constexpr int kPairs = 4;
    __device__ __forceinline__ static void run(const uint4& w, float2 (&f)[4]) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __half22float2(*reinterpret_cast<const __half2*>(&ws[i]));
    }
};
template <> struct Widen16<e4m3_t> {
    static constexpr int kPairs = 8;
    __device__ __forceinline__ static void run(const uint4& w, float2 (&f)[8]) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = e4m3x2_to_float2(static_cast<uint16_t>(ws[i] & 0xffffu));
            f[2 * i + 1] = e4m3x2_to_float2(static_cast<uint16_t>(ws[i] >> 16));
        }
    }
};

// The EPL components one lane owns in the P.V loop, widened to float.
template <typename CT, int EPL>
__device__ __forceinline__ void load_slice(const uint8_t* p, float (&x)[EPL]) {
    if constexpr (std::is_same<CT, e4m3_t>::value) {
        RowLoader<e4m3_t, EPL>::load(reinterpret_cast<const e4m3_t*>(p), x);
    } else if constexpr (std::is_same<CT, __nv_bfloat16>::value) {
        if constexpr (EPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(p);
            x[0] = __uint_as_float(w.x << 16); x[1] = __uint_as_float(w.x & 0xffff0000u);
            x[2] = __uint_as_float(w.y << 16); x[3] = __uint_as_float(w.y & 0xffff0000u);
        } else {
            RowLoader<__nv_bfloat16, EPL>::load(reinterpret_cast<const __nv_bfloat16*>(p), x);
        }
    } else {
        RowLoader<CT, EPL>::load(reinterpret_cast<const CT*>(p), x);
    }
}

template <typename QT, typename CT, int D, int GS, bool kSplit>
__global__ void __launch_bounds__(kTmaThreads)
paged_decode_tma_kernel(const __grid_constant__ TmaDecodeParams tp) {
    using S = TmaShape<CT, D>;
    using Smem = TmaSmem<CT, D, GS>;
    constexpr int NST = S::kNst;
    constexpr int EPL = S::kEpl;
    const DecodeParams& p = tp.p;

    extern __shared__ uint8_t smem_raw[];
    // the swizzle follows shared-memory address bits 4-9: align the ring to 1 KB
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* ring = smem;
    float* qs = reinterpret_cast<float*>(smem + Smem::kQOffset);       // [chunk][GS][epc]
    float* part = reinterpret_cast<float*>(smem + Smem::kPartOffset);  // [2][warp][GS][32]
    float* ps = reinterpret_cast<float*>(smem + Smem::kPOffset);       // [warp][GS][8]
    float* as = reinterpret_cast<float*>(smem + Smem::kAOffset);       // [warp][GS]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::kBarOffset);
    uint64_t* empty = full + NST;

    const int s = blockIdx.z;
    const int kvh = blockIdx.y / p.sub_groups;
    const int sub = blockIdx.y - kvh * p.sub_groups;
    const int hq0 = kvh * p.group + sub * GS;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

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
            mbar_init(&empty[i], kTmaConsumerWarps);
        }
        fence_barrier_init();
    }
    if (warp < kTmaConsumerWarps) {
        // query group -> shared memory as float32 [chunk][head][epc], pre-scaled
        const QT* qp = reinterpret_cast<const QT*>(p.query) + ((size_t)s * p.num_q_heads + hq0) * D;
        for (int i = threadIdx.x; i < GS * D; i += kTmaConsumerWarps * 32) {
            const int h = i / D, e = i - h * D;
            const int c = e / S::kEpc, j = e - c * S::kEpc;
            qs[(c * GS + h) * S::kEpc + j] = to_float(qp[i]) * p.q_mul;
        }
    }
    __syncthreads();

    if (warp == kTmaConsumerWarps) {
        // ------------------------------------------------------------ producer
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
            const int t_lo = T0 + k * kTmaStageTokens;
            const int t_hi = min(t_lo + kTmaStageTokens, Tend);
            if (p.new_key && L - 1 >= t_lo && L - 1 < t_hi)
                fused_write_token<QT, CT, D>(p, s, kvh, L, lane);
            const int j0 = t_lo / B;
            const int nseg = (t_hi - 1) / B - j0 + 1;           // 1 when B >= 32
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
    // Softmax / P.V lane layout: warp w owns tokens 8w..8w+7 of every stage;
    // lane l holds VPL (token, head) values, value index l*VPL + i (mod NV).
    constexpr int NV = kTmaTokensPerWarp * GS;
    constexpr int VPL = NV >= 32 ? NV / 32 : 1;
    constexpr int TOKMASK_LO = GS / VPL;          // lowest lane bit that changes the token
    float m_run[VPL], l_run[VPL];
    float2 o2[GS][EPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < GS; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e) o2[h][e] = make_float2(0.f, 0.f);
    int my_t[VPL], my_h[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int idx = (lane * VPL + i) % NV;
        my_t[i] = idx / GS;
        my_h[i] = idx % GS;
    }
    const bool canonical = lane * VPL < NV;       // lanes past NV repeat earlier values
    float* pw_buf = ps + warp * GS * kTmaTokensPerWarp;          // [GS][8]
    float* a_buf = as + warp * GS;                               // [GS]
    // this lane's P.V components: byte offset within a row, split into span / chunk
    const int vb = lane * EPL * S::kElem;
    const int v_span = vb >> 7, v_chunk = (vb & 127) >> 4, v_in = vb & 15;
    const int c0 = warp * S::kChunksPerWarp;                     // this warp's score chunks

    for (int k = 0; k < n_st; ++k) {
        const int slot = k % NST;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (k / NST) & 1, p.status));
        const uint8_t* Kst = ring + (size_t)slot * S::kStageBytes;
        const uint8_t* Vst = Kst + S::kTileBytes;
        const int nvalid = min(kTmaStageTokens, Tend - (T0 + k * kTmaStageTokens));

        // partial scores over this warp's quarter of the row: lane owns token `lane`
        // (after a timed-out wait the values are garbage; the vote below ends the loop)
        float2 acc[GS];
#pragma unroll
        for (int h = 0; h < GS; ++h) acc[h] = make_float2(0.f, 0.f);
        const uint8_t* krow = Kst + lane * 128;
        const int sw = lane & 7;
#pragma unroll
        for (int cc = 0; cc < S::kChunksPerWarp; ++cc) {
            const int c = c0 + cc;
            const uint4 kw = *reinterpret_cast<const uint4*>(
                krow + (c >> 3) * S::kSpanTileBytes + (((c & 7) ^ sw) << 4));
            float2 kf[Widen16<CT>::kPairs];
            Widen16<CT>::run(kw, kf);
#pragma unroll
            for (int h = 0; h < GS; ++h) {
                const float4* qv = reinterpret_cast<const float4*>(qs + (c * GS + h) * S::kEpc);
#pragma unroll
                for (int j = 0; j < Widen16<CT>::kPairs / 2; ++j) {
                    const float4 q4 = qv[j];
                    acc[h] = __ffma2_rn(kf[2 * j], make_float2(q4.x, q4.y), acc[h]);
                    acc[h] = __ffma2_rn(kf[2 * j + 1], make_float2(q4.z, q4.w), acc[h]);
                }
            }
        }
        float* pbuf = part + (k & 1) * (kTmaConsumerWarps * GS * kTmaStageTokens);
#pragma unroll
        for (int h = 0; h < GS; ++h)
            pbuf[(warp * GS + h) * kTmaStageTokens + lane] = acc[h].x + acc[h].y;
        // all four warps' partials are in place; a timed-out wait anywhere ends
        // the loop for every consumer warp at once
        if (!named_barrier_and(1, kTmaConsumerWarps * 32, ok)) break;

        // full scores of this warp's tokens, online softmax per head
        float pw[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int tok = warp * kTmaTokensPerWarp + my_t[i];
            float sc = 0.f;
#pragma unroll
            for (int w = 0; w < kTmaConsumerWarps; ++w)
                sc += pbuf[(w * GS + my_h[i]) * kTmaStageTokens + tok];
            const bool valid = tok < nvalid;
            sc = valid ? sc : -INFINITY;                              // select, never multiply
            float mx = sc;
#pragma unroll
            for (int m = TOKMASK_LO; m <= 16; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            const float m_new = fmaxf(m_run[i], mx);
            const float alpha = (m_new == -INFINITY) ? 1.f
                              : ((m_run[i] == -INFINITY) ? 0.f : fast_exp2(m_run[i] - m_new));
            pw[i] = valid ? fast_exp2(sc - m_new) : 0.f;
            l_run[i] = l_run[i] * alpha + (canonical ? pw[i] : 0.f);
            m_run[i] = m_new;
            pw_buf[my_h[i] * kTmaTokensPerWarp + my_t[i]] = pw[i];
            if (my_t[i] == 0) a_buf[my_h[i]] = alpha;
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < GS; ++h) {
            const float a = a_buf[h];
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o2[h][e] = __fmul2_rn(o2[h][e], a2);
        }

        // P.V over this warp's tokens: lane owns EPL components; even/odd tokens
        // accumulate in the two halves of a packed pair
        const int tw0 = warp * kTmaTokensPerWarp;
        const int nv = min(kTmaTokensPerWarp, nvalid - tw0);          // may be <= 0
        const uint8_t* vbase = Vst + v_span * S::kSpanTileBytes + v_in;
        int t = 0;
        for (; t + 1 < nv; t += 2) {
            const int ra = tw0 + t, rb = ra + 1;
            float va[EPL], vb2[EPL];
            load_slice<CT, EPL>(vbase + ra * 128 + ((v_chunk ^ (ra & 7)) << 4), va);
            load_slice<CT, EPL>(vbase + rb * 128 + ((v_chunk ^ (rb & 7)) << 4), vb2);
#pragma unroll
            for (int h = 0; h < GS; ++h) {
                const float2 pp = *reinterpret_cast<const float2*>(pw_buf + h * kTmaTokensPerWarp + t);
#pragma unroll
                for (int e = 0; e < EPL; ++e)
                    o2[h][e] = __ffma2_rn(make_float2(va[e], vb2[e]), pp, o2[h][e]);
            }
        }
        if (t < nv) {
            const int ra = tw0 + t;
            float va[EPL];
            load_slice<CT, EPL>(vbase + ra * 128 + ((v_chunk ^ (ra & 7)) << 4), va);
#pragma unroll
            for (int h = 0; h < GS; ++h) {
                const float pt = pw_buf[h * kTmaTokensPerWarp + t];
#pragma unroll
                for (int e = 0; e < EPL; ++e) o2[h][e].x = fmaf(va[e], pt, o2[h][e].x);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ------------------------------------------------- merge the four warps
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
#pragma unroll
        for (int m = TOKMASK_LO; m <= 16; m <<= 1) l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], m);
    }
    named_barrier(1, kTmaConsumerWarps * 32);    // ring is free: every stage was consumed
    float* cm = reinterpret_cast<float*>(smem);                 // [4][GS]
    float* cl = cm + kTmaConsumerWarps * GS;                    // [4][GS]
    float* co = cl + kTmaConsumerWarps * GS;                    // [4][GS][D]
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        if (canonical && my_t[i] == 0) {
            cm[warp * GS + my_h[i]] = m_run[i];
            cl[warp * GS + my_h[i]] = l_run[i];
        }
    }
#pragma unroll
    for (int h = 0; h < GS; ++h)
#pragma unroll
        for (int e = 0; e < EPL; ++e)
            co[(warp * GS + h) * D + lane * EPL + e] = o2[h][e].x + o2[h][e].y;
    named_barrier(1, kTmaConsumerWarps * 32);

    for (int i = threadIdx.x; i < GS * D; i += kTmaConsumerWarps * 32) {
        const int h = i / D;
        const int e = i - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kTmaConsumerWarps; ++w) M = fmaxf(M, cm[w * GS + h]);
        float W = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kTmaConsumerWarps; ++w) {
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
            out[((size_t)s * p.num_q_heads + hq) * D + e] = from_float<QT>(val);
        }
    }
}

// ---------------------------------------------------------------- host side

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
inline cudaError_t encode_cache_map(CUtensorMap* map, const void* base, int elem_bytes,
                                    int head_size, unsigned long long rows, int box_rows) {
    using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static std::atomic<EncodeFn> fn{nullptr};
    EncodeFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        f = reinterpret_cast<EncodeFn>(ptr);
        fn.store(f, std::memory_order_release);
    }
    const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT32;
    const cuuint64_t dims[2] = {(cuuint64_t)head_size, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)head_size * elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = f(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename QT, typename CT, int D, int GS, bool kSplit>
cudaError_t launch_tma_variant(const TmaDecodeParams& tp, cudaStream_t stream) {
    using Smem = TmaSmem<CT, D, GS>;
    auto kern = paged_decode_tma_kernel<QT, CT, D, GS, kSplit>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Smem::kAlloc);
    if (e != cudaSuccess) return e;
    const DecodeParams& p = tp.p;
    dim3 grid(kSplit ? p.max_parts : 1, p.num_kv_heads * p.sub_groups, p.num_seqs);
    kern<<<grid, kTmaThreads, Smem::kAlloc, stream>>>(tp);
    return cudaGetLastError();
}

template <typename QT, typename CT, int D>
cudaError_t launch_tma_d(const TmaDecodeParams& tp, int gs, bool split, cudaStream_t stream) {
#define PA_TMA_CASE(G)                                                                 \
    case G:                                                                            \
        return split ? launch_tma_variant<QT, CT, D, G, true>(tp, stream)              \
                     : launch_tma_variant<QT, CT, D, G, false>(tp, stream);
    // heads per unit are capped so that the P.V accumulators (GS x D/32
    // float2) stay within 32 register pairs
    switch (gs) {
        PA_TMA_CASE(1)
        PA_TMA_CASE(2)
        PA_TMA_CASE(4)
    }
    if constexpr (D <= 128) {
        if (gs == 8) return split ? launch_tma_variant<QT, CT, D, 8, true>(tp, stream)
                                  : launch_tma_variant<QT, CT, D, 8, false>(tp, stream);
    }
    if constexpr (D <= 64) {
        if (gs == 16) return split ? launch_tma_variant<QT, CT, D, 16, true>(tp, stream)
                                   : launch_tma_variant<QT, CT, D, 16, false>(tp, stream);
    }
#undef PA_TMA_CASE
    return cudaErrorInvalidValue;
}

// Build the tensor maps and launch; head_size must give 128/256/512-byte rows.
template <typename QT, typename CT>
cudaError_t launch_tma(const DecodeParams& p, int head_size, int gs, bool split,
                       cudaStream_t stream) {
    TmaDecodeParams tp;
    tp.p = p;
    tp.box_rows = p.block_size < kTmaStageTokens ? p.block_size : kTmaStageTokens;
    const unsigned long long rows =
        (unsigned long long)p.num_blocks * p.num_kv_heads * p.block_size;
    cudaError_t e = encode_cache_map(&tp.k_map, p.k_cache, TypeInfo<CT>::bytes, head_size, rows,
                                     tp.box_rows);
    if (e == cudaSuccess)
        e = encode_cache_map(&tp.v_map, p.v_cache, TypeInfo<CT>::bytes, head_size, rows,
                             tp.box_rows);
    if (e != cudaSuccess) return e;
    const int row_bytes = head_size * TypeInfo<CT>::bytes;
    if (row_bytes == 128) {
        if constexpr (TypeInfo<CT>::bytes == 1) return launch_tma_d<QT, CT, 128>(tp, gs, split, stream);
        if constexpr (TypeInfo<CT>::bytes == 2) return launch_tma_d<QT, CT, 64>(tp, gs, split, stream);
    } else if (row_bytes == 256) {
        if constexpr (TypeInfo<CT>::bytes == 1) return launch_tma_d<QT, CT, 256>(tp, gs, split, stream);
        if constexpr (TypeInfo<CT>::bytes == 2) return launch_tma_d<QT, CT, 128>(tp, gs, split, stream);
        if constexpr (TypeInfo<CT>::bytes == 4) return launch_tma_d<QT, CT, 64>(tp, gs, split, stream);
    } else if (row_bytes == 512) {
        if constexpr (TypeInfo<CT>::bytes == 2) return launch_tma_d<QT, CT, 256>(tp, gs, split, stream);
        if constexpr (TypeInfo<CT>::bytes == 4) return launch_tma_d<QT, CT, 128>(tp, gs, split, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pagedkv
