// prefill_tc.cuh -- multi-query paged attention on the 5th-generation tensor
// cores (tcgen05): the queries of a prefill chunk or of a speculative
// verification step attend causally to the paged cache ("Lecture 3:
// PagedAttention and vLLM", "the paged implementation of attention": logical
// block -> physical block; the queries there already carry a num_queries axis).
//
// Work unit. One CTA takes one (sequence s, KV head, query tile). The tile's
// 128 rows are (query token, head in the group) pairs, token-major: row r is
// token r / G and query head hk*G + r % G, so the G query heads that share the
// KV head read each key once. Query token i of s sits at position
// L - Q + i and sees keys 0..position.
//
// Data movement. Warp 4 (one lane) walks the block table and loads each
// 128-key (64 for head size 256) tile of K and V with tensor TMA copies into
// 128-byte-swizzled shared memory, one box per block segment and 64-element
// column span, on rings of KS (K) and VS (V) stages.
//
// Tensor cores. Warp 5 (one lane) issues tcgen05.mma: S = Q.K^T for tile j
// into one of two TMEM score buffers (A = Q and B = K both K-major), then
// O += P.V for tile j-1 (A = P K-major, B = V with the head dimension
// contiguous, i.e. MN-major). Commits on mbarriers hand S to the softmax, free
// K and V stages, and report each P.V done.
//
// Softmax. Warps 0-3: thread t owns TMEM lane t, i.e. row t. It loads its row
// of S, applies the causal mask, keeps the running max m and sum l in base 2,
// writes the weights P into shared memory (swizzled, K-major) and rescales its
// row of O in TMEM when the max has grown by more than 2^8 since the last
// rescale (weights up to 2^8 cannot overflow). At the end it divides by l and
// stores its output row.
//
// Precision. A weight rounded to bf16 carries a relative error up to 2^-8,
// which on a row with few keys moves the output by up to ~2^-8 |v - out|,
// beyond a 2e-3 bound. So P goes to the tensor cores as two 16-bit terms,
// P_hi = round(p) and P_lo = round(p - P_hi) (relative error ~2^-16), and O
// accumulates P_hi.V + P_lo.V: three MMAs per key tile instead of two.
//
// Every wait is bounded; a wait that runs out raises PA_DEV_TIMEOUT and a
// shared abort flag that ends every role's loop, and the CTA drains its copies
// and MMAs before it frees TMEM.
#pragma once

#include <cuda.h>

#include "decode_tma.cuh"   // tma_load_2d, encode_cache_map
#include "device_common.cuh"
#include "launch.h"

namespace pagedkv {

constexpr int kTcRows = 128;                  // MMA M: rows of a query tile
constexpr int kTcThreads = 6 * 32;            // 4 softmax warps, producer, MMA
constexpr int kTcProducerWarp = 4;
constexpr int kTcMmaWarp = 5;
constexpr float kTcRescaleLog2 = 8.0f;        // lazy rescale threshold (base 2)

template <int D>
struct TcShape {
    static constexpr int N = D == 256 ? 64 : 128;            // keys per tile
    static constexpr int KS = 2;                             // K stages
    static constexpr int VS = 2;                             // V stages
    static constexpr int kSpans = D / 64;                    // 128-byte column spans per row
    static constexpr int kQBytes = kTcRows * D * 2;
    static constexpr int kKvBytes = N * D * 2;               // one stage of K (or V)
    static constexpr int kPBytes = kTcRows * N * 2;          // one of P_hi, P_lo
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;
    static constexpr int kVOff = kKOff + KS * kKvBytes;
    static constexpr int kPOff = kVOff + VS * kKvBytes;
    static constexpr int kBarOff = kPOff + 2 * kPBytes;
    // barriers: k_full[KS] k_empty[KS] v_full[VS] v_empty[VS] s_full[2] s_free[2] p_full pv_done drain
    static constexpr int kNumBars = 2 * KS + 2 * VS + 7;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
    static constexpr int kBytes = kMiscOff + 16;
    // one CTA per SM: the CTA allocates all 512 TMEM columns
    static constexpr int kAlloc0 = kBytes + 1024;
    static constexpr int kAlloc = kAlloc0 < 120 * 1024 ? 120 * 1024 : kAlloc0;
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0;                          // score buffers at 0 and N
    static constexpr int kOCol = 2 * N;
    static_assert(2 * N + D <= kTmemCols, "TMEM columns");
    static_assert(kAlloc <= 227 * 1024, "shared memory");
};

struct TcPrefillParams {
    PrefillParams p;
    CUtensorMap k_map;            // pool as [num_blocks*Hkv*B rows][D], box [64 elements][box_rows]
    CUtensorMap v_map;
    int box_rows;                 // min(block_size, keys per tile)
};

// ---------------------------------------------------------------- tcgen05 wrappers

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (all >> 4), descriptor version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: F32 accumulator, A/B both bf16 or both
// f16, A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
template <typename T>
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, int b_mn) {
    constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
          "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
          "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Two floats to a packed pair of 16-bit values (low half = first), RNE.
template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <typename T> __device__ __forceinline__ float2 unpack2(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<__half2*>(&w));
}

// Bounded mbarrier wait that also gives up once another role has aborted.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                        volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            if (status) atomicOr(status, PA_DEV_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// Byte offset of 16-byte chunk c (0..D/8-1) of row r in a [rows x D] operand
// stored as D/64 column spans of rows x 128 bytes, 128-byte swizzled.
template <int ROWS>
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
    return (uint32_t)((c >> 3) * (ROWS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- the kernel

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ TcPrefillParams tp) {
    using Sh = TcShape<D>;
    constexpr int N = Sh::N;
    constexpr int KS = Sh::KS;
    constexpr int VS = Sh::VS;
    const PrefillParams& p = tp.p;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::kBarOff);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + KS;
    uint64_t* v_full = k_empty + KS;
    uint64_t* v_empty = v_full + VS;
    uint64_t* s_full = v_empty + VS;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* pv_done = p_full + 1;
    uint64_t* drain = pv_done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Sh::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Sh::kMiscOff + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- the work unit
    const int tile = blockIdx.x % p.q_tiles;
    const int rest = blockIdx.x / p.q_tiles;
    const int hk = rest % p.num_kv_heads;
    const int s = rest / p.num_kv_heads;
    const int q0 = p.query_start[s];
    const int Q = p.query_start[s + 1] - q0;
    const int L = p.context_lens[s];
    {
        int cap = p.max_context_len;
        const long long tab = (long long)p.max_blocks * p.block_size;
        if (tab < cap) cap = (int)tab;
        if (Q < 0 || Q > p.max_queries || L < Q || L > cap) {
            if (tid == 0 && tile == 0 && hk == 0 && p.status) atomicOr(p.status, PA_DEV_BAD_LEN);
            return;
        }
    }
    const int Tq = p.tokens_per_tile;
    const int tok0 = tile * Tq;
    if (tok0 >= Q) return;                                   // no such tile
    const int ntok = min(Tq, Q - tok0);
    const int first_pos = L - Q + tok0;
    const int kend = first_pos + ntok;                       // keys [0, kend)
    const int ntiles = (kend + N - 1) / N;

    // ---- setup: barriers, TMEM, the query tile
    if (tid == kTcProducerWarp * 32) {
        for (int i = 0; i < KS; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
        for (int i = 0; i < VS; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_free[i], 128); }
        mbar_init(p_full, 128);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_map(&tp.k_map);
        tma_prefetch_map(&tp.v_map);
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(Sh::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    const int G = p.group;
    if (warp < 4) {
        // rows (token, head) of the tile; padding rows are zero
        const T* qbase = reinterpret_cast<const T*>(p.query);
        constexpr int CPR = D / 8;                           // 16-byte chunks per row
        for (int idx = tid; idx < kTcRows * CPR; idx += 128) {
            const int r = idx / CPR, c = idx - r * CPR;
            const int i = r / G, g = r - i * G;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (i < ntok) {
                const size_t row = (size_t)(q0 + tok0 + i) * p.num_q_heads + (size_t)hk * G + g;
                v = *reinterpret_cast<const uint4*>(qbase + row * D + c * 8);
            }
            *reinterpret_cast<uint4*>(sm + Sh::kQOff + sw128_chunk<kTcRows>(r, c)) = v;
        }
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTcProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
            const int rows = tp.box_rows;
            const int B = p.block_size;
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int ks = j % KS, vs = j % VS;
                if (j >= KS && !tc_wait(&k_empty[ks], (uint32_t)((j / KS - 1) & 1), p.status, abort_flag)) break;
                if (j >= VS && !tc_wait(&v_empty[vs], (uint32_t)((j / VS - 1) & 1), p.status, abort_flag)) break;
                const int key0 = j * N;
                const int nvalid = min(N, kend - key0);
                // count the boxes first: the barrier must expect exactly what lands
                uint32_t boxes = 0;
                for (int r0 = 0; r0 < nvalid; r0 += rows) {
                    const int key = key0 + r0;
                    const int32_t blk = table[key / B];
                    if (blk >= 0 && blk < p.num_blocks) ++boxes;
                }
                const uint32_t bytes = boxes * (uint32_t)rows * 128u * Sh::kSpans;
                mbar_arrive_expect_tx(&k_full[ks], bytes);
                mbar_arrive_expect_tx(&v_full[vs], bytes);
                uint8_t* kd = sm + Sh::kKOff + ks * Sh::kKvBytes;
                uint8_t* vd = sm + Sh::kVOff + vs * Sh::kKvBytes;
                for (int r0 = 0; r0 < nvalid; r0 += rows) {
                    const int key = key0 + r0;
                    const int32_t blk = table[key / B];
                    if (blk < 0 || blk >= p.num_blocks) {
                        if (p.status) atomicOr(p.status, PA_DEV_BAD_BLOCK_ID);
                        continue;
                    }
                    const int y = (int)(((int64_t)blk * p.num_kv_heads + hk) * B + key % B);
#pragma unroll
                    for (int h = 0; h < Sh::kSpans; ++h) {
                        tma_load_2d(kd + h * (N * 128) + r0 * 128, &tp.k_map, h * 64, y, &k_full[ks]);
                        tma_load_2d(vd + h * (N * 128) + r0 * 128, &tp.v_map, h * 64, y, &v_full[vs]);
                    }
                }
                issued = j + 1;
            }
            // copies still in flight (only after an abort) land before the CTA ends
            for (int j = issued - 1; j >= 0 && j >= issued - KS; --j)
                mbar_wait_bounded(&k_full[j % KS], (uint32_t)((j / KS) & 1), p.status);
            for (int j = issued - 1; j >= 0 && j >= issued - VS; --j)
                mbar_wait_bounded(&v_full[j % VS], (uint32_t)((j / VS) & 1), p.status);
        }
    } else if (warp == kTcMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc_idesc<T>(kTcRows, N, 0);
            constexpr uint32_t idO = tc_idesc<T>(kTcRows, D, 1);
            const uint32_t qa = smem_u32(sm + Sh::kQOff);
            const uint32_t pa = smem_u32(sm + Sh::kPOff);
            auto pv = [&](int j) -> bool {
                const int vs = j % VS;
                if (!tc_wait(p_full, (uint32_t)(j & 1), p.status, abort_flag)) return false;
                if (!tc_wait(&v_full[vs], (uint32_t)((j / VS) & 1), p.status, abort_flag)) return false;
                tc_fence_after();
                const uint32_t va = smem_u32(sm + Sh::kVOff + vs * Sh::kKvBytes);
#pragma unroll
                for (int kk = 0; kk < N / 16; ++kk) {
                    const uint64_t a = tc_desc(pa + (kk >> 2) * (kTcRows * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = tc_desc(va + kk * 2048, N * 128, 1024);
                    tc_mma(tmem + Sh::kOCol, a, b, idO, j > 0 || kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < N / 16; ++kk) {
                    const uint64_t a = tc_desc(pa + Sh::kPBytes + (kk >> 2) * (kTcRows * 128) + (kk & 3) * 32,
                                               16, 1024);
                    const uint64_t b = tc_desc(va + kk * 2048, N * 128, 1024);
                    tc_mma(tmem + Sh::kOCol, a, b, idO, true);
                }
                tc_commit(&v_empty[vs]);
                tc_commit(pv_done);
                return true;
            };
            bool ok = true;
            for (int j = 0; j < ntiles && ok; ++j) {
                const int ks = j % KS, b = j & 1;
                ok = tc_wait(&k_full[ks], (uint32_t)((j / KS) & 1), p.status, abort_flag);
                if (ok && j >= 2)
                    ok = tc_wait(&s_free[b], (uint32_t)((j / 2 - 1) & 1), p.status, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm + Sh::kKOff + ks * Sh::kKvBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    const uint64_t a = tc_desc(qa + (kk >> 2) * (kTcRows * 128) + off, 16, 1024);
                    const uint64_t bd = tc_desc(ka + (kk >> 2) * (N * 128) + off, 16, 1024);
                    tc_mma(tmem + Sh::kSCol + b * N, a, bd, idS, kk > 0);
                }
                tc_commit(&k_empty[ks]);
                tc_commit(&s_full[b]);
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok) pv(ntiles - 1);
            // everything issued has finished before TMEM is freed
            tc_commit(drain);
            mbar_wait_bounded(drain, 0, p.status);
        }
    } else {
        // ------------------------------------------------------------ softmax (rows)
        const int r = tid;                                   // TMEM lane = row
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const int i = r / G;
        const bool row_valid = i < ntok && r < Tq * G;
        const int pos = first_pos + (row_valid ? i : ntok - 1);
        const float qm = p.q_mul;
        float m = -INFINITY;                                 // running max (base 2, scaled)
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int b = j & 1;
            ok = tc_wait(&s_full[b], (uint32_t)((j >> 1) & 1), p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            float x[N];
#pragma unroll
            for (int c = 0; c < N; c += 32) {
                uint32_t rr[32];
                tc_ld32(lane_base + Sh::kSCol + b * N + c, rr);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) x[c + e] = __uint_as_float(rr[e]);
            }
            tc_fence_before();
            mbar_arrive(&s_free[b]);
            const int key0 = j * N;
            if (key0 + N - 1 > pos) {                        // the causal edge crosses this tile
#pragma unroll
                for (int c = 0; c < N; ++c)
                    if (key0 + c > pos) x[c] = -INFINITY;
            }
            float mx = x[0];
#pragma unroll
            for (int c = 1; c < N; ++c) mx = fmaxf(mx, x[c]);
            const float m_cand = fmaxf(m, mx * qm);
            const bool rescale = m_cand > m + kTcRescaleLog2;
            const float m_use = rescale ? m_cand : m;
            const float alpha = fast_exp2(m - m_use);        // 0 on the first tile, 1 if kept
            float sum = 0.f;
            uint32_t phi[N / 2], plo[N / 2];
#pragma unroll
            for (int c = 0; c < N; c += 2) {
                const float e0 = fast_exp2(fmaf(x[c], qm, -m_use));
                const float e1 = fast_exp2(fmaf(x[c + 1], qm, -m_use));
                sum += e0 + e1;
                phi[c / 2] = pack2<T>(e0, e1);
                const float2 h = unpack2<T>(phi[c / 2]);
                plo[c / 2] = pack2<T>(e0 - h.x, e1 - h.y);
            }
            l = fmaf(l, alpha, sum);
            m = m_use;
            // the previous P.V must be done: P's buffer is reused and O is read
            if (j > 0) {
                ok = tc_wait(pv_done, (uint32_t)((j - 1) & 1), p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tc_ld32(lane_base + Sh::kOCol + c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc_st32(lane_base + Sh::kOCol + c, o);
                    }
                    tc_wait_st();
                }
            }
            // P row, 16-byte chunks into the swizzled K-major tiles
#pragma unroll
            for (int c = 0; c < N / 8; ++c) {
                const uint32_t off = Sh::kPOff + sw128_chunk<kTcRows>(r, c);
                *reinterpret_cast<uint4*>(sm + off) =
                    make_uint4(phi[4 * c], phi[4 * c + 1], phi[4 * c + 2], phi[4 * c + 3]);
                *reinterpret_cast<uint4*>(sm + off + Sh::kPBytes) =
                    make_uint4(plo[4 * c], plo[4 * c + 1], plo[4 * c + 2], plo[4 * c + 3]);
            }
            if (key0 + N > kend) {
                // last tile: V rows at or past kend hold stale data or cache
                // poison; zero them so that 0-weights stay 0 in the MMA
                const int vs = j % VS;
                ok = tc_wait(&v_full[vs], (uint32_t)((j / VS) & 1), p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const int first = kend - key0;
                constexpr int CPR = D / 8;
                uint8_t* vd = sm + Sh::kVOff + vs * Sh::kKvBytes;
                for (int idx = tid; idx < (N - first) * CPR; idx += 128) {
                    const int rr = first + idx / CPR, c = idx % CPR;
                    *reinterpret_cast<uint4*>(vd + sw128_chunk<N>(rr, c)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // ---- epilogue: O / l to the output row
        if (ok) {
            ok = tc_wait(pv_done, (uint32_t)((ntiles - 1) & 1), p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            T* orow = reinterpret_cast<T*>(p.out) +
                      ((size_t)(q0 + tok0 + (row_valid ? i : 0)) * p.num_q_heads + (size_t)hk * G +
                       (r - i * G)) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tc_ld32(lane_base + Sh::kOCol + c, o);
                tc_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pack2<T>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        v.y = pack2<T>(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        v.z = pack2<T>(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        v.w = pack2<T>(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c + e) = v;
                    }
                }
            }
        }
    }

    // ---- teardown: all TMEM traffic has completed
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tmem), "r"(Sh::kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------- host side

template <typename T, int D>
cudaError_t launch_prefill_tc_d(const TcPrefillParams& tp, cudaStream_t stream) {
    using Sh = TcShape<D>;
    auto kern = paged_prefill_tc_kernel<T, D>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Sh::kAlloc);
    if (e != cudaSuccess) return e;
    const PrefillParams& p = tp.p;
    const long long units = (long long)p.num_seqs * p.num_kv_heads * p.q_tiles;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    kern<<<(unsigned)units, kTcThreads, Sh::kAlloc, stream>>>(tp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_tc(const PrefillParams& p, int head_size, cudaStream_t stream) {
    TcPrefillParams tp;
    tp.p = p;
    const int n = head_size == 256 ? TcShape<256>::N : TcShape<128>::N;
    tp.box_rows = p.block_size < n ? p.block_size : n;
    const unsigned long long rows =
        (unsigned long long)p.num_blocks * p.num_kv_heads * p.block_size;
    cudaError_t e = encode_cache_map(&tp.k_map, p.k_cache, 2, head_size, rows, tp.box_rows);
    if (e == cudaSuccess) e = encode_cache_map(&tp.v_map, p.v_cache, 2, head_size, rows, tp.box_rows);
    if (e != cudaSuccess) return e;
    switch (head_size) {
    case 64: return launch_prefill_tc_d<T, 64>(tp, stream);
    case 128: return launch_prefill_tc_d<T, 128>(tp, stream);
    case 256: return launch_prefill_tc_d<T, 256>(tp, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pagedkv
