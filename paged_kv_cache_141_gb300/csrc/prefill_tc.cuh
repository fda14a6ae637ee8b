// prefill_tc.cuh -- multi-query paged attention on the 5th-generation tensor
// cores (tcgen05): the queries of a prefill chunk or of a speculative
// verification step attend causally to the paged cache ("Lecture 3:
// PagedAttention and vLLM", "the paged implementation of attention": logical
// block -> physical block; the queries there already carry a num_queries axis).
//
// Work unit. One CTA takes one (sequence s, KV head, query tile) (the
// two-tile kernel further down takes two query tiles). The tile's
// 128 rows are (query token, head in the group) pairs, token-major: row r is
// token r / G and query head hk*G + r % G, so the G query heads that share the
// KV head read each key once. Query token i of s sits at position
// L - Q + i and sees keys 0..position.
//
// Data movement. Warp 8 walks the block table and loads each 128-key (64 for
// head size 256) tile of K with tensor TMA copies into 128-byte-swizzled
// shared memory, one box per block segment and 64-element column span, lane i
// taking box i; warp 10 does the same for V. K and V have rings of their own
// (three stages each at head size 128), so a K tile is fetched as soon as the
// S = Q.K^T of the tile three stages back has consumed its slot, whatever P.V
// is doing. The block-table entries of a unit's first four key tiles are read
// at kernel entry, alongside the sequence's lengths.
//
// Tensor cores. Warp 9 (one lane) issues tcgen05.mma in the order S_0, S_1,
// PV_0, S_2, PV_1, ...: S_j = Q.K_j^T into TMEM score buffer j mod 2 (A = Q
// and B = K, both K-major in shared memory), then O += P_j.V_j with P_j read
// from TMEM and V_j (head dimension contiguous, i.e. MN-major) from shared
// memory. The tensor pipe runs one CTA's MMAs in issue order, so S_{j+2}
// overwriting P_j's buffer after PV_j needs no extra wait. Commits on
// mbarriers hand S to the softmax, free K and V slots and report each P.V.
//
// Softmax. Warps 0-7: a TMEM lane (row) is readable by warps w and w + 4, so
// thread t takes row t mod 128 and half t / 128 of the tile's key columns;
// two warps per SM sub-partition hide each other's latencies. Both halves
// take the max of the whole masked row of S (each loads the whole row, or,
// with the E4M3 products, its own columns, and the halves trade their
// maxima through two spare TMEM columns per score buffer), so they keep the
// same running max m (base 2) and make the same rescale decisions;
// each exponentiates its own columns, keeps their running sum, and stores
// their weights P over the same TMEM buffer. O is rescaled in TMEM (each half its
// half of the columns) only when the max has grown by more than 2^8 since the
// last rescale (weights up to 2^8 cannot overflow; the rescale waits for the
// previous P.V). At the end the two halves' sums are added through shared
// memory and each half divides and stores its half of the output row.
//
// Precision. A weight rounded to bf16 carries a relative error up to 2^-8,
// which on a row with few keys moves the output by up to ~2^-8 |v - out|,
// beyond a 2e-3 bound. So P goes to the tensor cores as two 16-bit terms,
// P_hi = round(p) and P_lo = round(p - P_hi) (relative error ~2^-16), packed
// side by side in the score buffer, and O accumulates P_hi.V + P_lo.V: three
// MMAs per key tile instead of two. Binary16 operands (f16 caches, and E4M3
// caches widened to binary16) keep 11 significant bits, a relative error of
// at most 2^-11 per weight: P goes as one term and the P_lo product is skipped.
// The E4M3 products (both kernels; E4M3 cache, bf16 query, head size 128)
// take the query and the weights as two E4M3 terms each (8 significant bits:
// exact for a bf16 query in E4M3's normal range, ~2^-8 for a weight), within
// the E4M3 cache's 3e-2 bound; an f16 query keeps the widened path. The K and
// V tiles then go to the tensor cores as they are stored, by TMA, in rings of
// six (one-tile) or five (two-tile) 16 KB stages.
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
constexpr int kTcSoftmaxThreads = 256;       // 8 softmax warps: two per row quarter
constexpr int kTcThreads = 11 * 32;           // softmax, K loads, MMA, V loads
constexpr int kTcKWarp = 8;
constexpr int kTcMmaWarp = 9;
constexpr int kTcVWarp = 10;
// E4M3 caches: 16 warps, the tiles widened by two warps per operand (K: warps
// 8 and 11, V: warps 10 and 13, one per SM sub-partition), registers moved
// from the producer warpgroups (2 and 3) to the softmax ones (0 and 1)
constexpr int kTcThreadsFp8 = 16 * 32;
constexpr int kTcK2Warp = 11;
constexpr int kTcV2Warp = 13;
constexpr int kTcSoftmaxRegs = 168;                 // 2 x 128 x 168 + 2 x 128 x 88 = 512 x 128
constexpr int kTcProducerRegs = 88;
static_assert(2 * 128 * kTcSoftmaxRegs + 2 * 128 * kTcProducerRegs <= kTcThreadsFp8 * 128,
              "register split within the launch's allocation");
constexpr float kTcRescaleLog2 = 8.0f;        // lazy rescale threshold (base 2)
constexpr int kTcSmemLimit = 227 * 1024;

// kFp8: E4M3 caches. Their tiles land row-major (D bytes per key) in two
// staging slots per K and V, and two producer warps per operand widen them to
// binary16 in the 16-bit rings the MMAs read.
template <int D, bool kFp8 = false>
struct TcShape {
    static constexpr int N = D == 256 ? 64 : 128;            // keys per tile
    static constexpr int kSpans = D / 64;                    // 128-byte column spans per row
    static constexpr int kQBytes = kTcRows * D * 2;
    static constexpr int kKvBytes = N * D * 2;               // one stage of K (or V)
    static constexpr int kStage8Bytes = kFp8 ? N * D : 0;    // one E4M3 staging slot
    static constexpr int kFixed = kQBytes + 1024 + 256 + 1024 + 4 * kStage8Bytes;
    static constexpr int kStages0 = (kTcSmemLimit - kFixed) / (2 * kKvBytes);
    static constexpr int NS = kStages0 > 4 ? 4 : kStages0;   // K stages = V stages
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;
    static constexpr int kVOff = kKOff + NS * kKvBytes;
    static constexpr int kK8Off = kVOff + NS * kKvBytes;     // E4M3 staging: K[2], V[2]
    static constexpr int kV8Off = kK8Off + 2 * kStage8Bytes;
    static constexpr int kBarOff = kV8Off + 2 * kStage8Bytes;
    // barriers: k_full[NS] k_empty[NS] v_full[NS] v_empty[NS] s_full[2] p_full pv_done drain
    // q_ready, then (E4M3) k_staged[2][2] v_staged[2][2] (per half and staging slot)
    static constexpr int kNumBars = 4 * NS + 6 + (kFp8 ? 8 : 0);
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
    static constexpr int kLsumOff = kMiscOff + 16;           // row sums of the two halves
    static constexpr int kBytes = kLsumOff + kTcSoftmaxThreads * 4;
    static constexpr int kAlloc = kBytes + 1024;
    // TMEM: two score buffers of N columns (S as f32, then P_hi | P_lo as
    // packed 16-bit pairs, N/2 columns each) and O (D columns). The CTA takes
    // all 512 columns, so one CTA runs per SM; the shared memory it asks for
    // keeps a second one off the SM.
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0;
    static constexpr int kOCol = 2 * N;
    static_assert(NS >= 2, "stages");
    static_assert(2 * N + D <= kTmemCols, "TMEM columns");
    static_assert(kAlloc <= kTcSmemLimit, "shared memory");
    static_assert(2 * kAlloc > 228 * 1024, "one CTA per SM");
    static_assert(!kFp8 || D <= 128, "E4M3 staging fits at head size <= 128");
};

// The MMAs' operand type: the query's for 16-bit caches; binary16 for E4M3
// caches (every E4M3 value is exact in it; the query is rounded to it).
template <typename QT, typename CT> struct TcMath { using T = QT; };
// whether weights in this MMA type need the P_lo correction term
template <typename T> constexpr bool kTcPLo = std::is_same<T, __nv_bfloat16>::value;
template <typename QT> struct TcMath<QT, e4m3_t> { using T = __half; };

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

// Same, with A read from TMEM (a_tmem: lane = row, 16-bit pairs per column).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// Instruction descriptor of kind::f8f6f4 with A and B both E4M3 (format 0),
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), F32 accumulator,
// shape M x N.
__host__ __device__ constexpr uint32_t tc_idesc_e4m3(int M, int N, int b_mn = 0) {
    return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
// D (+)= A.B^T on E4M3 operands from shared memory: K = 32 codes per step.
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}
// The same with A from TMEM (a_tmem: lane = row, four E4M3 codes per column).
__device__ __forceinline__ void tc_mma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                               uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
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

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// NC consecutive columns (16 or a multiple of 32) from r[0..NC).
__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7])
        : "memory");
}
// One 32-bit TMEM column of this thread's lane: store, and load with its
// wait (the register is tied to the wait, so no use moves above it).
__device__ __forceinline__ void tc_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t tc_ld1_wait(uint32_t taddr) {
    uint32_t v;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr) : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(v)::"memory");
    return v;
}
template <int NC>
__device__ __forceinline__ void tc_st_n(uint32_t taddr, const uint32_t* r) {
    static_assert(NC == 8 || NC == 16 || NC % 32 == 0, "columns");
    if constexpr (NC == 8) {
        tc_st8(taddr, r);
    } else if constexpr (NC == 16) {
        tc_st16(taddr, r);
    } else {
#pragma unroll
        for (int c = 0; c < NC; c += 32)
            tc_st32(taddr + c, *reinterpret_cast<const uint32_t(*)[32]>(r + c));
    }
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

// Two E4M3 codes, in bytes 0 and 2 of t (bytes 1 and 3 zero), to the binary16
// pair of their values times 2^-8, exactly, in integer operations: E4M3's
// exponent field (bias 7) and 3 mantissa bits moved up 7 places become a
// binary16 exponent (bias 15) and mantissa of the same value times 2^-8, an
// E4M3 subnormal becomes the binary16 subnormal of that value, and the sign
// (moved to bit 14) is carried into bit 15 by adding it to itself. The 2^8 is
// folded into the score and output scales. (Codes 0x7f/0xff, NaN, are never
// stored by the saturating write.)
__device__ __forceinline__ uint32_t e4m3x2_spread_to_f16x2_scaled(uint32_t t) {
    const uint32_t x = t << 7;
    return x + (x & 0x40004000u);
}

// max(a, b, c) in one instruction (three-input max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
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

// One role's loads, by a whole warp: K (or V) tiles of the unit into the
// ring `ring` of NS slots, each slot freed by a commit on `empty`, filled on
// `full`. Lane i owns box i of a tile (keys i*box_rows ..): it reads that
// box's block-table entry and issues the box's copies. The entries of the
// next kAhead tiles are in flight while the current ones are issued, so the
// table's latency is not paid per tile.
constexpr int kTcAhead = 4;                   // key tiles whose table entries load together

// The sequence of launch position i: i, or the caller's order (longest
// context first); -1 (and PA_DEV_BAD_ORDER, raised by `report`) for an entry
// outside [0, S).
__device__ __forceinline__ int tc_sequence(const PrefillParams& p, int i, bool report) {
    const int s = p.seq_order ? __ldg(p.seq_order + i) : i;
    if (s < 0 || s >= p.num_seqs) {
        if (report && p.status) atomicOr(p.status, PA_DEV_BAD_ORDER);
        return -1;
    }
    return s;
}

// The block-table entries of a unit's first kTcAhead key tiles for this
// lane's box, read before the sequence's lengths are known: every unit's keys
// start at 0, so they depend on the sequence alone (entries past the context
// are dropped once kend is known, and none past max_blocks is read). The
// table read then overlaps the length reads and the CTA's setup instead of
// following them.
template <typename Sh>
__device__ __forceinline__ void tc_ring_first(const TcPrefillParams& tp, int s, int lane,
                                              int64_t (&first)[kTcAhead]) {
    constexpr int N = Sh::N;
    const PrefillParams& p = tp.p;
    const int r0 = lane * tp.box_rows;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
#pragma unroll
    for (int k = 0; k < kTcAhead; ++k) {
        const int e = (k * N + r0) / p.block_size;
        first[k] = (r0 < N && e < p.max_blocks) ? (int64_t)__ldg(table + e) : -1;
    }
}

template <typename Sh, int NS>
__device__ __forceinline__ void tc_load_ring(const TcPrefillParams& tp, const CUtensorMap* map,
                                             uint8_t* ring, uint64_t* full, uint64_t* empty,
                                             int s, int hk, int ntiles, int kend, int lane,
                                             const int64_t (&first)[kTcAhead],
                                             volatile int* abort_flag) {
    constexpr int N = Sh::N;
    static_assert(NS >= 2, "ring stages");
    constexpr int64_t kNone = -1;
    const PrefillParams& p = tp.p;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
    const int rows = tp.box_rows;                            // >= 8, so <= 16 boxes per tile
    const int B = p.block_size;
    const int r0 = lane * rows;
    auto fetch = [&](int j) -> int64_t {
        const int key = j * N + r0;
        if (r0 < N && key < kend) return (int64_t)table[key / B];
        return kNone;
    };
    // Entries for groups of kAhead tiles: the next group's loads are issued
    // when a group starts and read when it ends, so no register copy waits on
    // a load still in flight. The first group's were read at kernel entry.
    constexpr int kAhead = kTcAhead;
    int64_t cur[kAhead], nxt[kAhead];
#pragma unroll
    for (int k = 0; k < kAhead; ++k)
        cur[k] = (k < ntiles && r0 < N && k * N + r0 < kend) ? first[k] : kNone;
    int issued = 0;
    bool live = true;
    for (int j0 = 0; j0 < ntiles && live; j0 += kAhead) {
#pragma unroll
        for (int k = 0; k < kAhead; ++k) nxt[k] = j0 + kAhead + k < ntiles ? fetch(j0 + kAhead + k) : kNone;
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            const int j = j0 + k;
            if (j >= ntiles || !live) break;
            const int64_t blk = cur[k];
            const int st = j % NS;
            if (j >= NS) {
                bool ok = true;
                if (lane == 0) ok = tc_wait(&empty[st], (uint32_t)((j / NS - 1) & 1), p.status, abort_flag);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    live = false;
                    break;
                }
            }
            const bool has = blk != kNone;
            const bool valid = has && blk >= 0 && blk < p.num_blocks;
            if (has && !valid && p.status) atomicOr(p.status, PA_DEV_BAD_BLOCK_ID);
            // the barrier must expect exactly the bytes that land
            const uint32_t boxes = __popc(__ballot_sync(0xffffffffu, valid));
            if (lane == 0) mbar_arrive_expect_tx(&full[st], boxes * (uint32_t)rows * 128u * Sh::kSpans);
            __syncwarp();
            if (valid) {
                const int key = j * N + r0;
                const int y = (int)((blk * p.num_kv_heads + hk) * B + key % B);
                uint8_t* dst = ring + st * Sh::kKvBytes + r0 * 128;
#pragma unroll
                for (int h = 0; h < Sh::kSpans; ++h)
                    tma_load_2d(dst + h * (N * 128), map, h * 64, y, &full[st]);
            }
            issued = j + 1;
        }
#pragma unroll
        for (int k = 0; k < kAhead; ++k) cur[k] = nxt[k];
    }
    // copies still in flight (only after an abort) land before the CTA ends
    if (lane == 0)
        for (int j = issued - 1; j >= 0 && j >= issued - NS; --j)
            mbar_wait_bounded(&full[j % NS], (uint32_t)((j / NS) & 1), p.status);
}

// E4M3 K (or V) tiles, loaded and widened in halves by two warps (both
// tcgen05 kernels): warp `half` owns rows [half * N/2, (half + 1) * N/2) of
// every tile -- it reads their block-table entries (a tile ahead), copies
// them into its half of one of two staging slots (plain boxes of at most
// N/2 rows, so no box spans both halves; a barrier per half and slot),
// widens them to binary16 into the ring slot the MMAs read once that slot is
// free (`empty`), orders its writes for the tensor cores (fence.proxy.async,
// which also orders its reads of the staging rows before the next copy into
// them), arrives on `full` (count 2), and refills its half of the staging
// slot with the tile two ahead. The two warps never wait for each other.
// Measured on GB300: a warp whose proxy fence follows tensor copies it issued
// itself passes it in ~200 cycles, one that issued none waited ~2,800, so
// both warps issue.
template <int N, int D, int NS>
__device__ __forceinline__ void tc_load_widen_halves(const TcPrefillParams& tp,
                                                     const CUtensorMap* map, uint8_t* staging,
                                                     uint8_t* ring, uint64_t* staged,
                                                     uint64_t* full, uint64_t* empty, int s,
                                                     int hk, int ntiles, int kend, int half,
                                                     int lane, volatile int* abort_flag) {
    constexpr int kKvBytes = N * D * 2;                      // one binary16 ring slot
    constexpr int kStage8Bytes = N * D;                      // one E4M3 staging slot
    constexpr int kSlots = 2;                                // staging slots
    constexpr int kRow8 = D;                                 // bytes of an E4M3 row
    constexpr int kHalfChunks = N * kRow8 / 16 / 2;          // 16-code chunks per warp and tile
    constexpr int64_t kNone = -1;
    const PrefillParams& p = tp.p;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks;
    const int rows = tp.box_rows;                            // divides N/2
    const int B = p.block_size;
    const int r0 = half * (N / 2) + lane * rows;             // this lane's box
    const bool owner = lane * rows < N / 2;
    uint64_t* my_staged = staged + kSlots * half;            // [slot] of this half
    auto fetch = [&](int j) -> int64_t {
        const int key = j * N + r0;
        if (owner && j < ntiles && key < kend) return (int64_t)table[key / B];
        return kNone;
    };
    auto issue = [&](int j, int64_t blk) {
        const bool has = blk != kNone;
        const bool valid = has && blk >= 0 && blk < p.num_blocks;
        if (has && !valid && p.status) atomicOr(p.status, PA_DEV_BAD_BLOCK_ID);
        const uint32_t boxes = __popc(__ballot_sync(0xffffffffu, valid));
        if (lane == 0) mbar_arrive_expect_tx(&my_staged[j % kSlots], boxes * (uint32_t)rows * kRow8);
        __syncwarp();
        if (valid) {
            const int key = j * N + r0;
            const int y = (int)((blk * p.num_kv_heads + hk) * B + key % B);
            tma_load_2d(staging + (j % kSlots) * kStage8Bytes + r0 * kRow8, map, 0, y,
                        &my_staged[j % kSlots]);
        }
    };
    int issued = 0;
    for (; issued < kSlots && issued < ntiles; ++issued) issue(issued, fetch(issued));
    int64_t next = fetch(kSlots);
    bool live = true;
    for (int j = 0; j < ntiles && live; ++j) {
        const int64_t after = fetch(j + kSlots + 1);         // in flight while tile j is widened
        bool ok = true;
        if (lane == 0) {
            ok = tc_wait(&my_staged[j % kSlots], (uint32_t)((j / kSlots) & 1), p.status, abort_flag);
            if (ok && j >= NS)
                ok = tc_wait(&empty[j % NS], (uint32_t)((j / NS - 1) & 1), p.status, abort_flag);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
            live = false;
            break;
        }
        const uint8_t* src = staging + (j % kSlots) * kStage8Bytes;
        uint8_t* dst = ring + (j % NS) * kKvBytes;
#pragma unroll 4
        for (int k = 0; k < kHalfChunks / 32; ++k) {
            const int q = half * kHalfChunks + lane + 32 * k;
            const int r = q / (kRow8 / 16), c = q - r * (kRow8 / 16);
            const uint4 w = *reinterpret_cast<const uint4*>(src + r * kRow8 + c * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                h[2 * e] = e4m3x2_spread_to_f16x2_scaled(__byte_perm(ws[e], 0u, 0x4140));
                h[2 * e + 1] = e4m3x2_spread_to_f16x2_scaled(__byte_perm(ws[e], 0u, 0x4342));
            }
            *reinterpret_cast<uint4*>(dst + sw128_chunk<N>(r, 2 * c)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(dst + sw128_chunk<N>(r, 2 * c + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[j % NS]);
        if (j + kSlots < ntiles) {
            issue(j + kSlots, next);                         // this half of staging slot j % kSlots
            issued = j + kSlots + 1;
        }
        next = after;
    }
    // copies still in flight (only after an abort) land before the CTA ends
    if (lane == 0)
        for (int j = issued - 1; j >= 0 && j >= issued - kSlots; --j)
            mbar_wait_bounded(&my_staged[j % kSlots], (uint32_t)((j / kSlots) & 1), p.status);
}

// Weights of the E4M3 products are y = P 2^6 <= 448: the softmax rescales O
// whenever the row's maximum has grown by more than log2(448 / 64) = 2.8,
// and y below E4M3's normal range (P < 2^-12) keeps an absolute error under
// 2^-16 in P.
constexpr int kTcWeightLog2E4M3 = 6;
constexpr float kTcRescaleLog2E4M3 = 2.8f;
// The E4M3 K ring as tc_load_ring sees it: one 128-byte span per key.
struct TcRingE4M3 {
    static constexpr int N = 128;
    static constexpr int kSpans = 1;
    static constexpr int kKvBytes = N * 128;
};
// Whether a tcgen05 kernel takes the E4M3 products: E4M3 cache, head size 128,
// bf16 query (its 8 significant bits are exactly the two E4M3 terms; an f16
// query's 11 are not, and a test with rows up to 32 times N(0,1) measured
// errors of 7e-2 that way, so f16 queries keep the widened K).
template <typename QT, typename CT, int D>
constexpr bool kTcE4M3Products =
    std::is_same<CT, e4m3_t>::value && D == 128 && std::is_same<QT, __nv_bfloat16>::value;

// The one-tile kernel with the E4M3 products: the query's two E4M3 terms in
// the 32 KB its bf16 rows land in, K and V rings of six 16 KB stages filled
// straight from the cache (128-byte swizzled boxes), barriers, row sums.
struct TcShapeE4M3Products {
    static constexpr int D = 128;
    static constexpr int N = 128;                            // keys per tile
    static constexpr int kQTermBytes = kTcRows * D;          // one E4M3 term of the query tile
    static constexpr int kQBytes = 2 * kQTermBytes;          // hi, then lo
    static constexpr int kKvBytes = N * D;                   // one E4M3 K (or V) stage
    static constexpr int NS = 6;                             // K stages = V stages
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;
    static constexpr int kVOff = kKOff + NS * kKvBytes;
    static constexpr int kBarOff = kVOff + NS * kKvBytes;
    // k_full[NS] k_empty[NS] v_full[NS] v_empty[NS] s_full[2] p_full pv_done drain
    // q_ready q_land
    static constexpr int kNumBars = 4 * NS + 7;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
    static constexpr int kLsumOff = kMiscOff + 16;           // row sums of the two halves
    static constexpr int kBytes = kLsumOff + kTcSoftmaxThreads * 4;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr int kTmemCols = 512;
    static constexpr int kSCol = 0;
    static constexpr int kOCol = 2 * N;
    static constexpr int kXCol = kOCol + D;                  // row-max exchange: [tile parity][half]
    static_assert(kXCol + 4 <= kTmemCols, "TMEM columns");
    static_assert(kQBytes == kTcRows * D * 2, "the bf16 query rows land in the E4M3 region");
    static_assert(2 * N + D <= kTmemCols, "TMEM columns");
    static_assert(kAlloc <= kTcSmemLimit, "shared memory");
    static_assert(2 * kAlloc > 228 * 1024, "one CTA per SM");
};

template <typename QT, typename CT, int D>
__global__ void __launch_bounds__(std::is_same<CT, e4m3_t>::value ? kTcThreadsFp8 : kTcThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ TcPrefillParams tp) {
    using MT = typename TcMath<QT, CT>::T;                  // MMA operand type
    constexpr bool kFp8 = std::is_same<CT, e4m3_t>::value;
    constexpr bool kF8S = kTcE4M3Products<QT, CT, D>;        // both products on kind::f8f6f4
    using Sh = std::conditional_t<kF8S, TcShapeE4M3Products, TcShape<D, kFp8>>;
    constexpr int N = Sh::N;
    constexpr int NS = Sh::NS;
    const PrefillParams& p = tp.p;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::kBarOff);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + NS;
    uint64_t* v_full = k_empty + NS;
    uint64_t* v_empty = v_full + NS;
    uint64_t* s_full = v_empty + NS;
    uint64_t* p_full = s_full + 2;
    uint64_t* pv_done = p_full + 1;
    uint64_t* drain = pv_done + 1;
    uint64_t* q_ready = drain + 1;
    uint64_t* q_land = q_ready + 1;                          // E4M3 products: the query rows landed
    uint64_t* k_staged = q_ready + 1;                        // widened E4M3: [half][slot]
    uint64_t* v_staged = k_staged + 4;                       // widened E4M3: [half][slot]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Sh::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Sh::kMiscOff + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- the work unit
    const int tile = blockIdx.x % p.q_tiles;
    const int rest = blockIdx.x / p.q_tiles;
    const int hk = rest % p.num_kv_heads;
    const int s = tc_sequence(p, rest / p.num_kv_heads, tid == 0 && tile == 0 && hk == 0);
    if (s < 0) return;
    int64_t first[kTcAhead] = {-1, -1, -1, -1};              // producers: first table entries
    if constexpr (!kFp8) {
        if (warp == kTcKWarp || warp == kTcVWarp) tc_ring_first<Sh>(tp, s, lane, first);
    } else if constexpr (kF8S) {
        if (warp == kTcKWarp || warp == kTcVWarp) tc_ring_first<TcRingE4M3>(tp, s, lane, first);
    }
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

    // ---- setup: barriers and TMEM; the K/V producers start at once, while
    // the softmax warps load the query tile (the MMA issuer waits for it)
    if (tid == kTcKWarp * 32) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&k_full[i], kFp8 && !kF8S ? 2 : 1);    // widened E4M3: two warps
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], kFp8 && !kF8S ? 2 : 1);
            mbar_init(&v_empty[i], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(p_full, kTcSoftmaxThreads);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        mbar_init(q_ready, kTcSoftmaxThreads);
        if constexpr (kF8S) mbar_init(q_land, 1);
        if constexpr (kFp8 && !kF8S) {
            for (int i = 0; i < 4; ++i) {
                mbar_init(&k_staged[i], 1);
                mbar_init(&v_staged[i], 1);
            }
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_map(&tp.k_map);
        tma_prefetch_map(&tp.v_map);
    }
    if constexpr (kF8S) {
        // E4M3 products: the query rows arrive by bulk copies, one per token
        // (its G heads' rows are contiguous), token-major into the query
        // region, converted in place below
        if (warp == kTcKWarp) {
            const uint32_t tok_bytes = (uint32_t)(p.group * D * sizeof(QT));
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(q_land, (uint32_t)ntok * tok_bytes);
            __syncwarp();
            const QT* qbase = reinterpret_cast<const QT*>(p.query);
            for (int i = lane; i < ntok; i += 32) {
                const QT* src = qbase + ((size_t)(q0 + tok0 + i) * p.num_q_heads +
                                         (size_t)hk * p.group) * D;
                bulk_copy_g2s(sm + Sh::kQOff + i * tok_bytes, src, tok_bytes, q_land);
            }
        }
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(Sh::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int G = p.group;
    float q_row_mul = 1.f;                                   // E4M3 products: the row's inverse scale
    if constexpr (kF8S) {
        if (tid < kTcSoftmaxThreads) {
            // the softmax warpgroups' registers, taken before the conversion
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTcSoftmaxRegs));
            // Each row times a power of two that puts its largest |element|
            // in [128, 256), as hi = the value rounded to E4M3's four
            // significant bits (integer operations, ties to even; exact in
            // E4M3 there) and lo = E4M3(value - hi), stored K-major with one
            // 128-byte swizzled span per row, hi then lo, over the landed
            // 16-bit rows once every thread has read its row. Both threads of
            // a row read all of it (the scale needs its maximum) and convert
            // their half of its chunks; each visits its half's chunks from
            // chunk r mod 8 on, so rows 256 bytes apart spread over the banks.
            const int r = tid & (kTcRows - 1);
            const int hf = tid / kTcRows;
            const bool live_row = r / G < ntok;
            const bool okq = tc_wait(q_land, 0u, p.status, abort_flag);
            const uint8_t* qs8 = sm + Sh::kQOff + r * (D * 2);
            uint4 qv[D / 8];                                 // [0, 8): this half's chunks
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const int cc = ((c >> 3) ^ hf) * 8 + ((c + r) & 7);
                qv[c] = live_row && okq ? *reinterpret_cast<const uint4*>(qs8 + cc * 16)
                                        : make_uint4(0u, 0u, 0u, 0u);
            }
            named_barrier(3, kTcSoftmaxThreads);             // every row read before any is overwritten
            uint32_t m2 = 0u;                                // 16-bit magnitudes order as integers
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                m2 = __vmaxu2(m2, qv[c].x & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, qv[c].y & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, qv[c].z & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, qv[c].w & 0x7FFF7FFFu);
            }
            const float mx = unpack2<QT>(max(m2 & 0xFFFFu, m2 >> 16)).x;
            int ex = 0;
            (void)frexpf(mx, &ex);                           // mx = m 2^ex, m in [0.5, 1)
            const float qsc = mx > 0.f ? ldexpf(1.f, 8 - max(ex, -100)) : 1.f;
            q_row_mul = 1.f / qsc;
            auto round4 = [](float y) -> float {
                uint32_t b = __float_as_uint(y);
                b += 0x7FFFFu + ((b >> 20) & 1u);
                return __uint_as_float(b & 0xFFF00000u);
            };
            uint8_t* qd = sm + Sh::kQOff;
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                const uint32_t in[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
                uint32_t hw[2], lw[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint32_t h4 = 0u, l4 = 0u;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float2 f2 = unpack2<QT>(in[2 * e + u]);
                        const float y0 = f2.x * qsc, y1 = f2.y * qsc;
                        const float h0 = round4(y0), h1 = round4(y1);
                        const __nv_fp8x2_storage_t hc =
                            __nv_cvt_float2_to_fp8x2(make_float2(h0, h1), __NV_SATFINITE, __NV_E4M3);
                        const __nv_fp8x2_storage_t lc = __nv_cvt_float2_to_fp8x2(
                            make_float2(y0 - h0, y1 - h1), __NV_SATFINITE, __NV_E4M3);
                        h4 |= (uint32_t)hc << (16 * u);
                        l4 |= (uint32_t)lc << (16 * u);
                    }
                    hw[e] = h4;
                    lw[e] = l4;
                }
                const int cc = hf * 8 + ((c + r) & 7);           // the chunk qv[c] holds
                const uint32_t off = (uint32_t)(r * 128 + ((((cc * 8) >> 4) ^ (r & 7)) << 4) + ((cc * 8) & 15));
                *reinterpret_cast<uint2*>(qd + off) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2*>(qd + Sh::kQTermBytes + off) = make_uint2(lw[0], lw[1]);
            }
            fence_async_smem();
            mbar_arrive(q_ready);
        }
    } else if (tid < kTcSoftmaxThreads) {
        // rows (token, head) of the tile; padding rows are zero. All of a
        // thread's loads are in flight before the first store.
        const QT* qbase = reinterpret_cast<const QT*>(p.query);
        constexpr int CPR = D / 8;                           // 16-byte chunks per row
        constexpr int PER = kTcRows * CPR / kTcSoftmaxThreads;  // chunks per thread
        uint4 v[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int idx = tid + k * kTcSoftmaxThreads;
            const int r = idx / CPR, c = idx - r * CPR;
            const int i = r / G, g = r - i * G;
            v[k] = make_uint4(0u, 0u, 0u, 0u);
            if (i < ntok) {
                const size_t row = (size_t)(q0 + tok0 + i) * p.num_q_heads + (size_t)hk * G + g;
                v[k] = __ldg(reinterpret_cast<const uint4*>(qbase + row * D + c * 8));
            }
        }
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int idx = tid + k * kTcSoftmaxThreads;
            const int r = idx / CPR, c = idx - r * CPR;
            uint4 w = v[k];
            if constexpr (!std::is_same<QT, MT>::value) {
                // E4M3 caches: the query in the MMAs' binary16
                const uint32_t in[4] = {w.x, w.y, w.z, w.w};
                uint32_t o4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack2<QT>(in[e]);
                    o4[e] = pack2<MT>(f.x, f.y);
                }
                w = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
            *reinterpret_cast<uint4*>(sm + Sh::kQOff + sw128_chunk<kTcRows>(r, c)) = w;
        }
        fence_async_smem();
        mbar_arrive(q_ready);
    }


    if (warp >= kTcSoftmaxThreads / 32) {
    // producer warpgroup(s); E4M3: they give up registers to the softmax
    // warpgroups (every warp of a warpgroup runs the same instruction, before
    // the warps part ways)
    if constexpr (kFp8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTcProducerRegs));
    if (warp == kTcKWarp || (kFp8 && !kF8S && warp == kTcK2Warp)) {
        // ------------------------------------------------------------ K loads
        if constexpr (kF8S) {
            tc_load_ring<TcRingE4M3, NS>(tp, &tp.k_map, sm + Sh::kKOff, k_full, k_empty, s, hk,
                                         ntiles, kend, lane, first, abort_flag);
            // the query copies this warp issued land before the CTA ends
            if (lane == 0) mbar_wait_bounded(q_land, 0u, p.status);
        } else if constexpr (kFp8)
            tc_load_widen_halves<N, D, NS>(tp, &tp.k_map, sm + Sh::kK8Off, sm + Sh::kKOff,
                                           k_staged, k_full, k_empty, s, hk, ntiles, kend,
                                           warp == kTcKWarp ? 0 : 1, lane, abort_flag);
        else
            tc_load_ring<Sh, NS>(tp, &tp.k_map, sm + Sh::kKOff, k_full, k_empty, s, hk, ntiles,
                                 kend, lane, first, abort_flag);
    } else if (warp == kTcVWarp || (kFp8 && !kF8S && warp == kTcV2Warp)) {
        // ------------------------------------------------------------ V loads
        if constexpr (kF8S)
            tc_load_ring<TcRingE4M3, NS>(tp, &tp.v_map, sm + Sh::kVOff, v_full, v_empty, s, hk,
                                         ntiles, kend, lane, first, abort_flag);
        else if constexpr (kFp8)
            tc_load_widen_halves<N, D, NS>(tp, &tp.v_map, sm + Sh::kV8Off, sm + Sh::kVOff,
                                           v_staged, v_full, v_empty, s, hk, ntiles, kend,
                                           warp == kTcVWarp ? 0 : 1, lane, abort_flag);
        else
            tc_load_ring<Sh, NS>(tp, &tp.v_map, sm + Sh::kVOff, v_full, v_empty, s, hk, ntiles,
                                 kend, lane, first, abort_flag);
    } else if (warp == kTcMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc_idesc<MT>(kTcRows, N, 0);
            constexpr uint32_t idO = tc_idesc<MT>(kTcRows, D, 1);
            const uint32_t qa = smem_u32(sm + Sh::kQOff);
            auto qk = [&](int j) -> bool {
                const int st = j % NS;
                if (!tc_wait(&k_full[st], (uint32_t)((j / NS) & 1), p.status, abort_flag)) return false;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm + Sh::kKOff + st * Sh::kKvBytes);
                const uint32_t sc = tmem + Sh::kSCol + (j & 1) * N;
                if constexpr (kF8S) {
                    // the query's two terms against the E4M3 K tile, 32 codes a step
                    constexpr uint32_t idS8 = tc_idesc_e4m3(kTcRows, N);
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int kk = 0; kk < D / 32; ++kk) {
                            const uint64_t a = tc_desc(qa + u * Sh::kQTermBytes + kk * 32, 16, 1024);
                            const uint64_t b = tc_desc(ka + kk * 32, 16, 1024);
                            tc_mma_e4m3(sc, a, b, idS8, u > 0 || kk > 0);
                        }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (uint32_t)(kk & 3) * 32u;
                        const uint64_t a = tc_desc(qa + (kk >> 2) * (kTcRows * 128) + off, 16, 1024);
                        const uint64_t b = tc_desc(ka + (kk >> 2) * (N * 128) + off, 16, 1024);
                        tc_mma(sc, a, b, idS, kk > 0);
                    }
                }
                tc_commit(&k_empty[st]);
                tc_commit(&s_full[j & 1]);
                return true;
            };
            auto pv = [&](int j) -> bool {
                const int st = j % NS;
                if (!tc_wait(p_full, (uint32_t)(j & 1), p.status, abort_flag)) return false;
                if (!tc_wait(&v_full[st], (uint32_t)((j / NS) & 1), p.status, abort_flag)) return false;
                tc_fence_after();
                const uint32_t va = smem_u32(sm + Sh::kVOff + st * Sh::kKvBytes);
                const uint32_t pt = tmem + Sh::kSCol + (j & 1) * N;   // P_hi | P_lo
                if constexpr (kF8S) {
                    // the weights' two E4M3 terms (32 columns each) against
                    // the E4M3 V tile as an MN-major operand, 32 keys a step
                    constexpr uint32_t idO8 = tc_idesc_e4m3(kTcRows, D, 1);
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int kk = 0; kk < N / 32; ++kk) {
                            const uint64_t b = tc_desc(va + kk * 32 * 128, N * 128, 1024);
                            tc_mma_e4m3_ts(tmem + Sh::kOCol, pt + u * (N / 4) + kk * 8, b, idO8,
                                           j > 0 || u > 0 || kk > 0);
                        }
                } else {
#pragma unroll
                    for (int kk = 0; kk < N / 16; ++kk) {
                        const uint64_t b = tc_desc(va + kk * 2048, N * 128, 1024);
                        tc_mma_ts(tmem + Sh::kOCol, pt + kk * 8, b, idO, j > 0 || kk > 0);
                    }
                }
                if constexpr (kTcPLo<MT>) {
#pragma unroll
                    for (int kk = 0; kk < N / 16; ++kk) {
                        const uint64_t b = tc_desc(va + kk * 2048, N * 128, 1024);
                        tc_mma_ts(tmem + Sh::kOCol, pt + N / 2 + kk * 8, b, idO, true);
                    }
                }
                tc_commit(&v_empty[st]);
                tc_commit(pv_done);
                return true;
            };
            bool ok = tc_wait(q_ready, 0u, p.status, abort_flag);
            tc_fence_after();
            if (ok) ok = qk(0);
            for (int j = 0; j < ntiles && ok; ++j) {
                if (j + 1 < ntiles) ok = qk(j + 1);
                if (ok) ok = pv(j);
            }
            // everything issued has finished before the epilogue reads O and
            // before TMEM is freed
            tc_commit(drain);
            mbar_wait_bounded(drain, 0, p.status);
        }
    }
    } else {
        // ------------------------------------------------------------ softmax (rows)
        if constexpr (kFp8 && !kF8S) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTcSoftmaxRegs));
        // Thread t: row r = t mod 128 (its warp's TMEM lane quarter), half
        // hf = t / 128 of the key columns. Both halves take the same row max
        // (each reads the whole row; with the E4M3 products each reads its
        // own columns and the halves trade their maxima through TMEM), so
        // they make the same rescale decision; each exponentiates, sums and
        // stores only its own columns.
        constexpr int NH = N / 2;
        const int r = tid & (kTcRows - 1);
        const int hf = tid / kTcRows;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int i = r / G;
        const bool row_valid = i < ntok && r < Tq * G;
        const int pos = first_pos + (row_valid ? i : ntok - 1);
        const float qm = p.q_mul * q_row_mul;                // E4M3 products: the row's scale out
        const float2 qm2 = make_float2(qm, qm);
        float m = -INFINITY;                                 // running max (base 2, scaled)
        float l = 0.f;                                       // this half's running sum
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int b = j & 1;
            const uint32_t sbuf = lane_base + Sh::kSCol + b * N;
            if (ok) {
                ok = tc_wait(&s_full[b], (uint32_t)((j >> 1) & 1), p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (!ok) {
                // after an abort the thread still meets the halves' barrier
                // once per key tile (and does nothing else), so every softmax
                // thread passes it ntiles times and no half waits there for
                // one that has stopped
                named_barrier(2, kTcSoftmaxThreads);
                continue;
            }
            tc_fence_after();
            const int key0 = j * N;
            constexpr int R = 8;
            float m_row;                                     // the row's max of S over this tile
            float x[kF8S ? NH : N];
            if constexpr (kF8S) {
                // this half's columns only; the halves trade their maxima
                // through TMEM columns kXCol + 2 (j mod 2) + half (a column
                // is rewritten two tiles on, after the partner's read of it
                // has passed the barrier of the tile between)
                uint32_t xr[NH];
#pragma unroll
                for (int c = 0; c < NH; c += 32)
                    tc_ld32(sbuf + hf * NH + c, *reinterpret_cast<uint32_t(*)[32]>(xr + c));
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < NH; ++c) x[c] = __uint_as_float(xr[c]);
                if (key0 + N - 1 > pos) {                    // the causal edge crosses this tile
#pragma unroll
                    for (int c = 0; c < NH; ++c)
                        if (key0 + hf * NH + c > pos) x[c] = -INFINITY;
                }
                float mr[R];
#pragma unroll
                for (int k = 0; k < R; ++k) mr[k] = x[k];
#pragma unroll
                for (int c = R; c + 1 < NH; c += 2) mr[(c / 2) % R] = fmax3(mr[(c / 2) % R], x[c], x[c + 1]);
#pragma unroll
                for (int w = R / 2; w >= 1; w /= 2)
#pragma unroll
                    for (int k = 0; k < w; ++k) mr[k] = fmaxf(mr[k], mr[k + w]);
                const uint32_t xcol = lane_base + Sh::kXCol + 2 * (j & 1);
                tc_st1(xcol + hf, __float_as_uint(mr[0]));
                tc_wait_st();
                // the other half of this row must also have read its S before
                // either half writes its weights over the buffer
                tc_fence_before();
                named_barrier(2, kTcSoftmaxThreads);
                tc_fence_after();
                m_row = fmaxf(mr[0], __uint_as_float(tc_ld1_wait(xcol + (hf ^ 1))));
            } else {
            // the whole row in flight at once, one wait
            uint32_t xr[N];
#pragma unroll
            for (int c = 0; c < N; c += 32)
                tc_ld32(sbuf + c, *reinterpret_cast<uint32_t(*)[32]>(xr + c));
            tc_wait_ld();
            // the other half of this row must have read S before either half
            // writes its weights over it
            tc_fence_before();
            named_barrier(2, kTcSoftmaxThreads);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < N; ++c) x[c] = __uint_as_float(xr[c]);
            if (key0 + N - 1 > pos) {                        // the causal edge crosses this tile
#pragma unroll
                for (int c = 0; c < N; ++c)
                    if (key0 + c > pos) x[c] = -INFINITY;
            }
            // the max as 8 independent chains
            float mr[R];
#pragma unroll
            for (int k = 0; k < R; ++k) mr[k] = x[k];
#pragma unroll
            for (int c = R; c + 1 < N; c += 2) mr[(c / 2) % R] = fmax3(mr[(c / 2) % R], x[c], x[c + 1]);
#pragma unroll
            for (int w = R / 2; w >= 1; w /= 2)
#pragma unroll
                for (int k = 0; k < w; ++k) mr[k] = fmaxf(mr[k], mr[k + w]);
            m_row = mr[0];
            }
            const float m_cand = fmaxf(m, m_row * qm);
            const bool rescale = m_cand > m + (kF8S ? kTcRescaleLog2E4M3 : kTcRescaleLog2);
            const float m_use = rescale ? m_cand : m;
            const float alpha = fast_exp2(m - m_use);        // 0 on the first tile, 1 if kept
            const float2 nm2 = make_float2(-m_use, -m_use);
            // this half's weights: 2^(x qm - m), as hi + lo 16-bit pairs
            uint32_t phi[NH / 2], plo[NH / 2];
            float2 sr[R / 2];
#pragma unroll
            for (int k = 0; k < R / 2; ++k) sr[k] = make_float2(0.f, 0.f);
            auto weights = [&](auto off) {
                constexpr int c0 = decltype(off)::value;
#pragma unroll
                for (int c = 0; c < NH; c += 2) {
                    const float2 t = __ffma2_rn(make_float2(x[c0 + c], x[c0 + c + 1]), qm2, nm2);
                    const float2 e = make_float2(fast_exp2(t.x), fast_exp2(t.y));
                    sr[(c / 2) % (R / 2)] = __fadd2_rn(sr[(c / 2) % (R / 2)], e);
                    phi[c / 2] = pack2<MT>(e.x, e.y);
                    if constexpr (kTcPLo<MT>) {
                        const float2 lo = __ffma2_rn(unpack2<MT>(phi[c / 2]), make_float2(-1.f, -1.f), e);
                        plo[c / 2] = pack2<MT>(lo.x, lo.y);
                    }
                }
            };
            // E4M3 products: y = P 2^6 (the 2^6 in the exponent) as hi =
            // E4M3(y) and lo = E4M3(y - hi), the remainder taken in binary16;
            // four codes per 32-bit column, hi in columns [0, N/4) and lo in
            // [N/4, N/2) of the buffer, this half's keys a half of each; its
            // two quarters of 32 keys stored one after the other
            auto weights8 = [&](const float (&xh)[NH]) {
                const float2 nm8 = make_float2(kTcWeightLog2E4M3 - m_use, kTcWeightLog2E4M3 - m_use);
#pragma unroll
                for (int h = 0; h < NH / 32; ++h) {
                    uint32_t hq8[8], lq8[8];
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const int cc = h * 32 + c;
                        uint32_t hq = 0u, lq = 0u;
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const float2 t2 = __ffma2_rn(make_float2(xh[cc + 2 * u], xh[cc + 2 * u + 1]), qm2, nm8);
                            const float2 y = make_float2(fast_exp2(t2.x), fast_exp2(t2.y));
                            sr[(c / 2 + u) % (R / 2)] = __fadd2_rn(sr[(c / 2 + u) % (R / 2)], y);
                            const __nv_fp8x2_storage_t hc = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
                            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hc, __NV_E4M3);
                            const __half2 rem = __hsub2(__float22half2_rn(y), *reinterpret_cast<const __half2*>(&hr));
                            const __nv_fp8x2_storage_t lc = __nv_cvt_halfraw2_to_fp8x2(
                                *reinterpret_cast<const __half2_raw*>(&rem), __NV_SATFINITE, __NV_E4M3);
                            hq |= (uint32_t)hc << (16 * u);
                            lq |= (uint32_t)lc << (16 * u);
                        }
                        hq8[c / 4] = hq;
                        lq8[c / 4] = lq;
                    }
                    tc_st_n<8>(sbuf + hf * (NH / 4) + h * 8, hq8);
                    tc_st_n<8>(sbuf + N / 4 + hf * (NH / 4) + h * 8, lq8);
                }
            };
            if constexpr (kF8S) {
                weights8(x);
            } else {
                if (hf == 0) weights(std::integral_constant<int, 0>{});
                else weights(std::integral_constant<int, NH>{});
            }
#pragma unroll
            for (int w = R / 4; w >= 1; w /= 2)
#pragma unroll
                for (int k = 0; k < w; ++k) sr[k] = __fadd2_rn(sr[k], sr[k + w]);
            l = fmaf(l, alpha, sr[0].x + sr[0].y);
            m = m_use;
            // P over S in the same buffer: P_hi pairs in columns [0, N/2), P_lo
            // in [N/2, N); this half's keys are a quarter of the buffer each
            if constexpr (!kF8S) {
                tc_st_n<NH / 2>(sbuf + hf * (NH / 2), phi);
                if constexpr (kTcPLo<MT>) tc_st_n<NH / 2>(sbuf + N / 2 + hf * (NH / 2), plo);
            }
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                // O holds tiles < j once the previous P.V is done; each half
                // rescales its half of the columns
                ok = tc_wait(pv_done, (uint32_t)((j - 1) & 1), p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) continue;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 2; c += 32) {
                    const uint32_t oa = lane_base + Sh::kOCol + hf * (D / 2) + c;
                    uint32_t o[32];
                    tc_ld32(oa, o);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc_st32(oa, o);
                }
            }
            tc_wait_st();
            if (key0 + N > kend) {
                // last tile: V rows at or past kend hold stale data or cache
                // poison; zero them so that 0-weights stay 0 in the MMA
                const int st = j % NS;
                ok = tc_wait(&v_full[st], (uint32_t)((j / NS) & 1), p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) continue;
                const int first = kend - key0;
                constexpr int CPR = kF8S ? 8 : D / 8;            // 16-byte chunks of a V row
                uint8_t* vd = sm + Sh::kVOff + st * Sh::kKvBytes;
                for (int idx = tid; idx < (N - first) * CPR; idx += kTcSoftmaxThreads) {
                    const int rr = first + idx / CPR, c = idx % CPR;
                    *reinterpret_cast<uint4*>(vd + sw128_chunk<N>(rr, c)) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_async_smem();
            }
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // ---- epilogue: O / l to the output row, once every MMA has finished
        // (the MMA issuer's final commit; pv_done could alias two phases here)
        float* lsum = reinterpret_cast<float*>(sm + Sh::kLsumOff);
        lsum[tid] = l;
        named_barrier(1, kTcSoftmaxThreads);
        // E4M3: V's scale comes in here (the widened tiles also lack 2^8, the
        // E4M3 products' weights carry 2^6 as the row sums do)
        const float inv = p.v_mul / (lsum[r] + lsum[r + kTcRows]);
        if (ok) {
            ok = tc_wait(drain, 0u, p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            QT* orow = reinterpret_cast<QT*>(p.out) +
                      ((size_t)(q0 + tok0 + (row_valid ? i : 0)) * p.num_q_heads + (size_t)hk * G +
                       (r - i * G)) * D + hf * (D / 2);
#pragma unroll 1
            for (int c = 0; c < D / 2; c += 32) {
                uint32_t o[32];
                tc_ld32(lane_base + Sh::kOCol + hf * (D / 2) + c, o);
                tc_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pack2<QT>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        v.y = pack2<QT>(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        v.z = pack2<QT>(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        v.w = pack2<QT>(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
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

// ---------------------------------------------------------------- two query tiles per CTA

// Shapes of the two-tile kernel (head size 64 or 128): two 128-row query
// tiles share every K/V tile, so each loaded tile feeds twice the rows.
// kFp8: E4M3 caches, whose tiles land row-major in two staging slots per
// operand and are widened to binary16 into the rings (for every 256 rows,
// not 128 as in the one-tile kernel). At head size 128 that leaves one K
// stage: a K tile is widened while tile 0's softmax runs, after both tiles'
// S products of the previous key tile, which finish early in each key tile.
template <int D, bool kPLo, bool kFp8 = false>
struct TcShape2 {
    static constexpr int N = 128;                            // keys per tile
    static constexpr int kSpans = D / 64;
    static constexpr int kQBytes = kTcRows * D * 2;          // one query tile
    static constexpr int kKvBytes = N * D * 2;
    static constexpr int kStage8Bytes = kFp8 ? N * D : 0;    // one E4M3 staging slot
    // Q0, Q1, slack, barriers, staging (K[2], V[2])
    static constexpr int kFixed = 2 * kQBytes + 1024 + 256 + 4 * kStage8Bytes;
    static constexpr int kStages0 = (kTcSmemLimit - kFixed) / (2 * kKvBytes);
    // K and V rings of their own depths: a K slot is free once both tiles'
    // S products have read it, a V slot only after both P.V products, so V
    // takes the stage that is left over (head size 128: 2 K, 3 V stages).
    // With the P_lo term (bf16) the softmax's registers are at their limit
    // and the deeper V ring measured slower: K and V get equal depths.
    static constexpr int NSK = kStages0 > 4 ? 4 : kStages0;
    static constexpr int kStagesV0 = (kTcSmemLimit - kFixed - NSK * kKvBytes) / kKvBytes;
    static constexpr int kStagesV1 = kPLo ? NSK : kStagesV0;
    static constexpr int NSV = kStagesV1 > 4 ? 4 : kStagesV1;
    static constexpr int kKBytes = kKvBytes;                 // one K stage
    static constexpr int kVBytes = kKvBytes;                 // one V stage
    static constexpr int kQOff = 0;                          // Q0, then Q1
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + NSK * kKvBytes;
    static constexpr int kK8Off = kVOff + NSV * kKvBytes;    // E4M3 staging: K[2], V[2]
    static constexpr int kV8Off = kK8Off + 2 * kStage8Bytes;
    static constexpr int kBarOff = kV8Off + 2 * kStage8Bytes;
    // k_full[NSK] k_empty[NSK] v_full[NSV] v_empty[NSV] s_full[2] p_full[2] drain q_ready,
    // then (E4M3) k_staged[2][2] v_staged[2][2] (per half and staging slot)
    static constexpr int kNumBars = 2 * NSK + 2 * NSV + 6 + (kFp8 ? 8 : 0);
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kBytes = kMiscOff + 16;
    static constexpr int kAlloc = kBytes + 1024;
    // TMEM: per query tile t, S_t (N columns; S as f32, then P_hi | P_lo)
    // and O_t (D columns)
    static constexpr int kTmemCols = 512;
    static constexpr int kTileCols = N + D;
    static_assert(D == 64 || D == 128, "head size");
    static_assert(NSK >= (kFp8 ? 1 : 2) && NSV >= 2, "stages");
    static_assert(2 * kTileCols <= kTmemCols, "TMEM columns");
    static_assert(kAlloc <= kTcSmemLimit, "shared memory");
    static_assert(2 * kAlloc > 228 * 1024, "one CTA per SM");
};

// The two-tile kernel on E4M3 caches at head size 128 with a bf16 query:
// both products on kind::f8f6f4, straight from the E4M3 tiles (TMA, 128-byte
// swizzle, no widening). S = Q.K^T with the query as two E4M3 terms hi + lo
// of its row scaled by a power of two (exact for a bf16 value in E4M3's
// normal range); O += P.V with the weights as two E4M3 terms of P 2^6 in TMEM
// and V an MN-major operand. Shared memory: Q 4 x 16 KB (tile, term), K and V
// rings of five 16 KB stages, barriers.
struct TcShape2E4M3Scores {
    static constexpr int D = 128;
    static constexpr int N = 128;                            // keys per tile
    static constexpr int kSpans = 1;                         // 128-byte rows
    static constexpr int kQTermBytes = kTcRows * D;          // one E4M3 term of one query tile
    static constexpr int kQBytes = 2 * kQTermBytes;          // one query tile: hi, then lo
    static constexpr int kKBytes = N * D;                    // one E4M3 K stage
    static constexpr int kVBytes = N * D;                    // one E4M3 V stage
    static constexpr int kKvBytes = kVBytes;
    static constexpr int NSK = 5;
    static constexpr int NSV = 5;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + NSK * kKBytes;
    static constexpr int kBarOff = kVOff + NSV * kVBytes;
    // k_full[NSK] k_empty[NSK] v_full[NSV] v_empty[NSV] s_full[2] p_full[2] drain q_ready
    // q_land
    static constexpr int kNumBars = 2 * NSK + 2 * NSV + 7;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kBytes = kMiscOff + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static constexpr int kTmemCols = 512;
    static constexpr int kTileCols = N + D;
    static_assert(kQBytes == kTcRows * D * 2, "a tile's bf16 query rows land in its E4M3 region");
    static_assert(2 * kTileCols <= kTmemCols, "TMEM columns");
    static_assert(kAlloc <= kTcSmemLimit, "shared memory");
    static_assert(2 * kAlloc > 228 * 1024, "one CTA per SM");
};
// Two query tiles per CTA: warps 0-3 run the softmax of tile 0, warps 4-7 of
// tile 1, each thread a whole row of 128 keys. The MMA issuer interleaves the
// tiles -- S0_0, S1_0, PV0_0, S0_1, PV1_0, S1_1, PV0_1, ... -- so one tile's
// softmax runs while the tensor cores work for the other. S_t_{j+1} is issued
// after PV_t_j, so a softmax that sees S_t_j also sees O_t final for the
// earlier key tiles and can rescale it at once. A K slot is freed after the
// second tile's S, a V slot after its P.V. Without a second tile (the last
// group of a sequence with an odd tile count) warps 4-7 idle and the tile-1
// MMAs are skipped. E4M3 caches: warps 8/11 and 10/13 load and widen the K
// and V tiles by halves (tc_load_widen_halves), and the registers move from the producer
// warpgroups to the softmax ones as in the one-tile kernel.
template <typename QT, typename CT, int D>
__global__ void __launch_bounds__(std::is_same<CT, e4m3_t>::value ? kTcThreadsFp8 : kTcThreads, 1)
paged_prefill_tc2_kernel(const __grid_constant__ TcPrefillParams tp) {
    using T = typename TcMath<QT, CT>::T;                    // MMA operand type
    constexpr bool kFp8 = std::is_same<CT, e4m3_t>::value;
    constexpr bool kF8S = kTcE4M3Products<QT, CT, D>;          // E4M3 scores (kind::f8f6f4)
    using Sh = std::conditional_t<kF8S, TcShape2E4M3Scores, TcShape2<D, kTcPLo<T>, kFp8>>;
    constexpr int N = Sh::N;
    constexpr int NSK = Sh::NSK;                             // K ring stages
    constexpr int NSV = Sh::NSV;                             // V ring stages
    const PrefillParams& p = tp.p;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::kBarOff);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + NSK;
    uint64_t* v_full = k_empty + NSK;
    uint64_t* v_empty = v_full + NSV;
    uint64_t* s_full = v_empty + NSV;                        // [2], per query tile
    uint64_t* p_full = s_full + 2;                           // [2]
    uint64_t* drain = p_full + 2;
    uint64_t* q_ready = drain + 1;
    uint64_t* q_land = q_ready + 1;                          // E4M3 scores: the query rows landed
    uint64_t* k_staged = q_ready + 1;                        // widened E4M3 K: [half][slot]
    uint64_t* v_staged = kF8S ? q_ready + 1 : k_staged + 4;  // E4M3 V: [half][slot]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Sh::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Sh::kMiscOff + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- the work unit: query tiles 2g and 2g+1 of (sequence s, KV head hk)
    const int groups = (p.q_tiles + 1) / 2;
    const int g = blockIdx.x % groups;
    const int rest = blockIdx.x / groups;
    const int hk = rest % p.num_kv_heads;
    const int s = tc_sequence(p, rest / p.num_kv_heads, tid == 0 && g == 0 && hk == 0);
    if (s < 0) return;
    int64_t first[kTcAhead] = {-1, -1, -1, -1};              // producers: first table entries
    if constexpr (!kFp8) {
        if (warp == kTcKWarp || warp == kTcVWarp) tc_ring_first<Sh>(tp, s, lane, first);
    } else if constexpr (kF8S) {
        if (warp == kTcKWarp || warp == kTcVWarp) tc_ring_first<TcRingE4M3>(tp, s, lane, first);
    }
    const int q0 = p.query_start[s];
    const int Q = p.query_start[s + 1] - q0;
    const int L = p.context_lens[s];
    {
        int cap = p.max_context_len;
        const long long tab = (long long)p.max_blocks * p.block_size;
        if (tab < cap) cap = (int)tab;
        if (Q < 0 || Q > p.max_queries || L < Q || L > cap) {
            if (tid == 0 && g == 0 && hk == 0 && p.status) atomicOr(p.status, PA_DEV_BAD_LEN);
            return;
        }
    }
    const int Tq = p.tokens_per_tile;
    const int tok0 = 2 * g * Tq;
    if (tok0 >= Q) return;                                   // no such group
    const int ntok0 = min(Tq, Q - tok0);
    const int ntok1 = max(0, min(Tq, Q - tok0 - Tq));
    const bool two = ntok1 > 0;
    const int kend = L - Q + tok0 + ntok0 + ntok1;           // keys [0, kend)
    const int ntiles = (kend + N - 1) / N;
    float q_row_mul = 1.f;                                   // E4M3 scores: the row's inverse scale
    if (tid == kTcKWarp * 32) {
        for (int i = 0; i < NSK; ++i) {
            mbar_init(&k_full[i], kFp8 && !kF8S ? 2 : 1);    // widened E4M3: two warps
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(&v_full[i], kFp8 && !kF8S ? 2 : 1);    // widened E4M3: two warps
            mbar_init(&v_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], kTcRows);
        }
        mbar_init(drain, 1);
        mbar_init(q_ready, kTcSoftmaxThreads);
        if constexpr (kF8S) mbar_init(q_land, 1);
        if constexpr (kFp8 && !kF8S) {
            for (int i = 0; i < 4; ++i) {
                mbar_init(&k_staged[i], 1);
                mbar_init(&v_staged[i], 1);
            }
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_map(&tp.k_map);
        tma_prefetch_map(&tp.v_map);
    }
    if constexpr (kF8S) {
        // E4M3 scores: the query rows arrive by bulk copies, one per token
        // (its G heads' rows are contiguous), each tile's rows (token-major)
        // into that tile's query region, converted in place below
        if (warp == kTcKWarp) {
            const uint32_t tok_bytes = (uint32_t)(p.group * D * sizeof(QT));
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(q_land, (uint32_t)(ntok0 + ntok1) * tok_bytes);
            __syncwarp();
            const QT* qbase = reinterpret_cast<const QT*>(p.query);
            for (int k = lane; k < ntok0 + ntok1; k += 32) {
                const int t = k < ntok0 ? 0 : 1, i = k - t * ntok0;
                const QT* src = qbase + ((size_t)(q0 + tok0 + t * Tq + i) * p.num_q_heads +
                                         (size_t)hk * p.group) * D;
                bulk_copy_g2s(sm + Sh::kQOff + t * Sh::kQBytes + i * tok_bytes, src, tok_bytes, q_land);
            }
        }
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(Sh::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int G = p.group;
    const int qt = tid / kTcRows;                            // softmax threads: query tile
    if (tid < kTcSoftmaxThreads) {
        // tile qt's rows (token, head); padding rows are zero
        const int r = tid & (kTcRows - 1);
        (void)r;
        const QT* qbase = reinterpret_cast<const QT*>(p.query);
        const int tt0 = tok0 + qt * Tq;
        const int nt = qt == 0 ? ntok0 : ntok1;
        constexpr int CPR = D / 8;
        constexpr int PER = kF8S ? 1 : CPR;                  // 128 rows x CPR chunks / 128 threads
        uint4 v[PER];
        if constexpr (!kF8S) {
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int idx = (tid & (kTcRows - 1)) + k * kTcRows;
            const int rr = idx / CPR, c = idx - rr * CPR;
            const int i = rr / G, gg = rr - i * G;
            v[k] = make_uint4(0u, 0u, 0u, 0u);
            if (i < nt) {
                const size_t row = (size_t)(q0 + tt0 + i) * p.num_q_heads + (size_t)hk * G + gg;
                v[k] = __ldg(reinterpret_cast<const uint4*>(qbase + row * D + c * 8));
            }
        }
        }
        uint8_t* qd = sm + Sh::kQOff + qt * Sh::kQBytes;
        if constexpr (kF8S) {
            // E4M3 scores: the thread's row times a power of two that puts its
            // largest |element| in [128, 256), as hi = the value rounded to
            // E4M3's four significant bits (integer operations, ties to even;
            // exact in E4M3 there) and lo = E4M3(value - hi), stored K-major
            // with one 128-byte swizzled span per row, hi then lo, over the
            // landed 16-bit rows once every thread has read its own (each
            // thread starts at chunk r mod 16 of its row: rows 256 bytes apart
            // would otherwise all hit the same banks)
            const int r = tid & (kTcRows - 1);
            const bool live_row = r / G < nt;
            bool okq = tc_wait(q_land, 0u, p.status, abort_flag);
            uint4 qv[D / 8];
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const int cc = (c + r) & (D / 8 - 1);
                qv[c] = live_row && okq ? *reinterpret_cast<const uint4*>(qd + r * (D * 2) + cc * 16)
                                        : make_uint4(0u, 0u, 0u, 0u);
            }
            named_barrier(3, kTcSoftmaxThreads);             // every row read before any is overwritten
            uint32_t m2 = 0u;                                // 16-bit magnitudes order as integers
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                m2 = __vmaxu2(m2, qv[c].x & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, qv[c].y & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, qv[c].z & 0x7FFF7FFFu);
                m2 = __vmaxu2(m2, qv[c].w & 0x7FFF7FFFu);
            }
            const float mx = unpack2<QT>(max(m2 & 0xFFFFu, m2 >> 16)).x;
            int ex = 0;
            (void)frexpf(mx, &ex);                           // mx = m 2^ex, m in [0.5, 1)
            const float qs = mx > 0.f ? ldexpf(1.f, 8 - max(ex, -100)) : 1.f;
            q_row_mul = 1.f / qs;
            auto round4 = [](float y) -> float {
                uint32_t b = __float_as_uint(y);
                b += 0x7FFFFu + ((b >> 20) & 1u);
                return __uint_as_float(b & 0xFFF00000u);
            };
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint32_t in[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
                uint32_t hw[2], lw[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint32_t h4 = 0u, l4 = 0u;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float2 f2 = unpack2<QT>(in[2 * e + u]);
                        const float y0 = f2.x * qs, y1 = f2.y * qs;
                        const float h0 = round4(y0), h1 = round4(y1);
                        const __nv_fp8x2_storage_t hc =
                            __nv_cvt_float2_to_fp8x2(make_float2(h0, h1), __NV_SATFINITE, __NV_E4M3);
                        const __nv_fp8x2_storage_t lc = __nv_cvt_float2_to_fp8x2(
                            make_float2(y0 - h0, y1 - h1), __NV_SATFINITE, __NV_E4M3);
                        h4 |= (uint32_t)hc << (16 * u);
                        l4 |= (uint32_t)lc << (16 * u);
                    }
                    hw[e] = h4;
                    lw[e] = l4;
                }
                const int cc = (c + r) & (D / 8 - 1);            // the chunk qv[c] holds
                const uint32_t off = (uint32_t)(r * 128 + ((((cc * 8) >> 4) ^ (r & 7)) << 4) + ((cc * 8) & 15));
                *reinterpret_cast<uint2*>(qd + off) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2*>(qd + Sh::kQTermBytes + off) = make_uint2(lw[0], lw[1]);
            }
        } else {
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int idx = (tid & (kTcRows - 1)) + k * kTcRows;
            const int rr = idx / CPR, c = idx - rr * CPR;
            uint4 w = v[k];
            if constexpr (!std::is_same<QT, T>::value) {
                // E4M3 caches: the query in the MMAs' binary16
                const uint32_t in[4] = {w.x, w.y, w.z, w.w};
                uint32_t o4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack2<QT>(in[e]);
                    o4[e] = pack2<T>(f.x, f.y);
                }
                w = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
            *reinterpret_cast<uint4*>(qd + sw128_chunk<kTcRows>(rr, c)) = w;
        }
        }
        fence_async_smem();
        mbar_arrive(q_ready);
    }

    if (warp >= kTcSoftmaxThreads / 32) {
    // producer warpgroup(s); E4M3: they give up registers to the softmax
    // warpgroups (every warp of a warpgroup runs the same instruction)
    if constexpr (kFp8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTcProducerRegs));
    if (warp == kTcKWarp || (kFp8 && !kF8S && warp == kTcK2Warp)) {
        if constexpr (kF8S) {
            tc_load_ring<TcRingE4M3, NSK>(tp, &tp.k_map, sm + Sh::kKOff, k_full, k_empty, s, hk,
                                          ntiles, kend, lane, first, abort_flag);
            // the query copies this warp issued land before the CTA ends
            if (lane == 0) mbar_wait_bounded(q_land, 0u, p.status);
        }
        else if constexpr (kFp8)
            tc_load_widen_halves<N, D, NSK>(tp, &tp.k_map, sm + Sh::kK8Off, sm + Sh::kKOff,
                                            k_staged, k_full, k_empty, s, hk, ntiles, kend,
                                            warp == kTcKWarp ? 0 : 1, lane, abort_flag);
        else
            tc_load_ring<Sh, NSK>(tp, &tp.k_map, sm + Sh::kKOff, k_full, k_empty, s, hk, ntiles,
                                  kend, lane, first, abort_flag);
    } else if (warp == kTcVWarp || (kFp8 && !kF8S && warp == kTcV2Warp)) {
        if constexpr (kF8S)
            tc_load_ring<TcRingE4M3, NSV>(tp, &tp.v_map, sm + Sh::kVOff, v_full, v_empty, s, hk,
                                          ntiles, kend, lane, first, abort_flag);
        else if constexpr (kFp8)
            tc_load_widen_halves<N, D, NSV>(tp, &tp.v_map, sm + Sh::kV8Off, sm + Sh::kVOff,
                                            v_staged, v_full, v_empty, s, hk, ntiles, kend,
                                            warp == kTcVWarp ? 0 : 1, lane, abort_flag);
        else
            tc_load_ring<Sh, NSV>(tp, &tp.v_map, sm + Sh::kVOff, v_full, v_empty, s, hk, ntiles,
                                  kend, lane, first, abort_flag);
    } else if (warp == kTcMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc_idesc<T>(kTcRows, N, 0);
            constexpr uint32_t idO = tc_idesc<T>(kTcRows, D, 1);
            const int last_t = two ? 1 : 0;
            auto qk = [&](int t, int j) -> bool {
                const int st = j % NSK;
                if (t == 0) {
                    if (!tc_wait(&k_full[st], (uint32_t)((j / NSK) & 1), p.status, abort_flag))
                        return false;
                    tc_fence_after();
                }
                const uint32_t qa = smem_u32(sm + Sh::kQOff + t * Sh::kQBytes);
                const uint32_t ka = smem_u32(sm + Sh::kKOff + st * Sh::kKBytes);
                const uint32_t sc = tmem + t * Sh::kTileCols;
                if constexpr (kF8S) {
                    // the query's two terms against the E4M3 K tile, 32 codes a step
                    constexpr uint32_t idS8 = tc_idesc_e4m3(kTcRows, N);
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int kk = 0; kk < D / 32; ++kk) {
                            const uint64_t a = tc_desc(qa + u * Sh::kQTermBytes + kk * 32, 16, 1024);
                            const uint64_t b = tc_desc(ka + kk * 32, 16, 1024);
                            tc_mma_e4m3(sc, a, b, idS8, u > 0 || kk > 0);
                        }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (uint32_t)(kk & 3) * 32u;
                        const uint64_t a = tc_desc(qa + (kk >> 2) * (kTcRows * 128) + off, 16, 1024);
                        const uint64_t b = tc_desc(ka + (kk >> 2) * (N * 128) + off, 16, 1024);
                        tc_mma(sc, a, b, idS, kk > 0);
                    }
                }
                if (t == last_t) tc_commit(&k_empty[st]);
                tc_commit(&s_full[t]);
                return true;
            };
            auto pv = [&](int t, int j) -> bool {
                const int st = j % NSV;
                if (!tc_wait(&p_full[t], (uint32_t)(j & 1), p.status, abort_flag)) return false;
                if (t == 0 &&
                    !tc_wait(&v_full[st], (uint32_t)((j / NSV) & 1), p.status, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t va = smem_u32(sm + Sh::kVOff + st * Sh::kVBytes);
                const uint32_t pt = tmem + t * Sh::kTileCols;          // P_hi | P_lo
                const uint32_t oc = pt + N;
                if constexpr (kF8S) {
                    // the weights' two E4M3 terms (32 columns each) against
                    // the E4M3 V tile as an MN-major operand, 32 keys a step
                    constexpr uint32_t idO8 = tc_idesc_e4m3(kTcRows, D, 1);
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int kk = 0; kk < N / 32; ++kk) {
                            const uint64_t b = tc_desc(va + kk * 32 * 128, N * 128, 1024);
                            tc_mma_e4m3_ts(oc, pt + u * (N / 4) + kk * 8, b, idO8,
                                           j > 0 || u > 0 || kk > 0);
                        }
                } else {
#pragma unroll
                for (int kk = 0; kk < N / 16; ++kk) {
                    const uint64_t b = tc_desc(va + kk * 2048, N * 128, 1024);
                    tc_mma_ts(oc, pt + kk * 8, b, idO, j > 0 || kk > 0);
                }
                }
                if constexpr (kTcPLo<T>) {
#pragma unroll
                    for (int kk = 0; kk < N / 16; ++kk) {
                        const uint64_t b = tc_desc(va + kk * 2048, N * 128, 1024);
                        tc_mma_ts(oc, pt + N / 2 + kk * 8, b, idO, true);
                    }
                }
                if (t == last_t) tc_commit(&v_empty[st]);
                return true;
            };
            bool ok = tc_wait(q_ready, 0u, p.status, abort_flag);
            tc_fence_after();
            if (ok) ok = qk(0, 0);
            if (ok && two) ok = qk(1, 0);
            for (int j = 0; j < ntiles && ok; ++j) {
                ok = pv(0, j);
                if (ok && j + 1 < ntiles) ok = qk(0, j + 1);
                if (ok && two) {
                    ok = pv(1, j);
                    if (ok && j + 1 < ntiles) ok = qk(1, j + 1);
                }
            }
            // everything issued has finished before the epilogue reads O and
            // before TMEM is freed
            tc_commit(drain);
            mbar_wait_bounded(drain, 0, p.status);
        }
    }
    } else if (qt == 0 || two) {
        // ------------------------------------------------------------ softmax (tile qt)
        if constexpr (kFp8) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTcSoftmaxRegs));
        const int r = tid & (kTcRows - 1);
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t sbuf = lane_base + qt * Sh::kTileCols;
        const uint32_t obuf = sbuf + N;
        const int i = r / G;
        const int nt = qt == 0 ? ntok0 : ntok1;
        const bool row_valid = i < nt && r < Tq * G;
        const int pos = L - Q + tok0 + qt * Tq + (row_valid ? i : nt - 1);
        const float qm = p.q_mul * q_row_mul;                // E4M3 scores: the row's scale out
        const float2 qm2 = make_float2(qm, qm);
        float m = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            ok = tc_wait(&s_full[qt], (uint32_t)(j & 1), p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t xr[N];
#pragma unroll
            for (int c = 0; c < N; c += 32)
                tc_ld32(sbuf + c, *reinterpret_cast<uint32_t(*)[32]>(xr + c));
            tc_wait_ld();
            float x[N];
#pragma unroll
            for (int c = 0; c < N; ++c) x[c] = __uint_as_float(xr[c]);
            const int key0 = j * N;
            if (key0 + N - 1 > pos) {
#pragma unroll
                for (int c = 0; c < N; ++c)
                    if (key0 + c > pos) x[c] = -INFINITY;
            }
            constexpr int R = 8;
            float mr[R];
#pragma unroll
            for (int k = 0; k < R; ++k) mr[k] = x[k];
#pragma unroll
            for (int c = R; c + 1 < N; c += 2) mr[(c / 2) % R] = fmax3(mr[(c / 2) % R], x[c], x[c + 1]);
#pragma unroll
            for (int w = R / 2; w >= 1; w /= 2)
#pragma unroll
                for (int k = 0; k < w; ++k) mr[k] = fmaxf(mr[k], mr[k + w]);
            const float m_cand = fmaxf(m, mr[0] * qm);
            const bool rescale = m_cand > m + (kF8S ? kTcRescaleLog2E4M3 : kTcRescaleLog2);
            const float m_use = rescale ? m_cand : m;
            const float alpha = fast_exp2(m - m_use);
            const float2 nm2 = make_float2(-m_use, -m_use);
            float2 sr[R / 2];
#pragma unroll
            for (int k = 0; k < R / 2; ++k) sr[k] = make_float2(0.f, 0.f);
            // weights in four quarters of 32 keys: each quarter's P_hi and
            // P_lo go to TMEM before the next is formed, so few packed words
            // are live next to the scores not yet used
            if constexpr (kF8S) {
                // E4M3 weights: y = P 2^6 (the 2^6 in the exponent) as hi =
                // E4M3(y) and lo = E4M3(y - hi), the remainder taken in
                // binary16; four codes per 32-bit column, hi in columns
                // [0, N/4), lo in [N/4, N/2); each quarter of 32 keys stored
                // before the next is formed
                const float2 nm8 = make_float2(kTcWeightLog2E4M3 - m_use, kTcWeightLog2E4M3 - m_use);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t phi[N / 16], plo[N / 16];
#pragma unroll
                    for (int c = 0; c < N / 4; c += 4) {
                        const int cc = h * (N / 4) + c;
                        uint32_t hq = 0u, lq = 0u;
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const float2 t2 = __ffma2_rn(make_float2(x[cc + 2 * u], x[cc + 2 * u + 1]), qm2, nm8);
                            const float2 y = make_float2(fast_exp2(t2.x), fast_exp2(t2.y));
                            sr[(c / 2 + u) % (R / 2)] = __fadd2_rn(sr[(c / 2 + u) % (R / 2)], y);
                            const __nv_fp8x2_storage_t hc = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
                            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hc, __NV_E4M3);
                            const __half2 rem = __hsub2(__float22half2_rn(y), *reinterpret_cast<const __half2*>(&hr));
                            const __nv_fp8x2_storage_t lc = __nv_cvt_halfraw2_to_fp8x2(
                                *reinterpret_cast<const __half2_raw*>(&rem), __NV_SATFINITE, __NV_E4M3);
                            hq |= (uint32_t)hc << (16 * u);
                            lq |= (uint32_t)lc << (16 * u);
                        }
                        phi[c / 4] = hq;
                        plo[c / 4] = lq;
                    }
                    tc_st_n<N / 16>(sbuf + h * (N / 16), phi);
                    tc_st_n<N / 16>(sbuf + N / 4 + h * (N / 16), plo);
                }
            } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t phi[N / 8], plo[N / 8];
#pragma unroll
                for (int c = 0; c < N / 4; c += 2) {
                    const int cc = h * (N / 4) + c;
                    const float2 t2 = __ffma2_rn(make_float2(x[cc], x[cc + 1]), qm2, nm2);
                    const float2 e = make_float2(fast_exp2(t2.x), fast_exp2(t2.y));
                    sr[(c / 2) % (R / 2)] = __fadd2_rn(sr[(c / 2) % (R / 2)], e);
                    phi[c / 2] = pack2<T>(e.x, e.y);
                    if constexpr (kTcPLo<T>) {
                        const float2 lo = __ffma2_rn(unpack2<T>(phi[c / 2]), make_float2(-1.f, -1.f), e);
                        plo[c / 2] = pack2<T>(lo.x, lo.y);
                    }
                }
                tc_st_n<N / 8>(sbuf + h * (N / 8), phi);
                if constexpr (kTcPLo<T>) tc_st_n<N / 8>(sbuf + N / 2 + h * (N / 8), plo);
            }
            }
#pragma unroll
            for (int w = R / 4; w >= 1; w /= 2)
#pragma unroll
                for (int k = 0; k < w; ++k) sr[k] = __fadd2_rn(sr[k], sr[k + w]);
            l = fmaf(l, alpha, sr[0].x + sr[0].y);
            m = m_use;
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                // O_t already holds key tiles < j (S_t_j came after PV_t_{j-1})
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tc_ld32(obuf + c, o);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc_st32(obuf + c, o);
                }
            }
            tc_wait_st();
            if (qt == 0 && key0 + N > kend) {
                // last tile: V rows at or past kend hold stale data or cache
                // poison; zero them before either tile's P.V reads the slot
                const int st = j % NSV;
                ok = tc_wait(&v_full[st], (uint32_t)((j / NSV) & 1), p.status, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const int first = kend - key0;
                constexpr int CPR = kF8S ? 8 : D / 8;            // 16-byte chunks of a V row
                uint8_t* vd = sm + Sh::kVOff + st * Sh::kVBytes;
                for (int idx = r; idx < (N - first) * CPR; idx += kTcRows) {
                    const int rr = first + idx / CPR, c = idx % CPR;
                    *reinterpret_cast<uint4*>(vd + sw128_chunk<N>(rr, c)) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&p_full[qt]);
        }
        if (ok) {
            ok = tc_wait(drain, 0u, p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            // E4M3: the values were widened without their scale; it comes in here
            const float inv = kFp8 ? p.v_mul / l : 1.f / l;
            QT* orow = reinterpret_cast<QT*>(p.out) +
                       ((size_t)(q0 + tok0 + qt * Tq + (row_valid ? i : 0)) * p.num_q_heads +
                        (size_t)hk * G + (r - i * G)) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tc_ld32(obuf + c, o);
                tc_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pack2<QT>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        v.y = pack2<QT>(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        v.z = pack2<QT>(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        v.w = pack2<QT>(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c + e) = v;
                    }
                }
            }
        }
    }

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

// Host: a [rows][head_size] byte tensor (E4M3 cache) with unswizzled boxes
// [head_size bytes][box_rows].
inline cudaError_t encode_plain_map(CUtensorMap* map, const void* base, int head_size,
                                    unsigned long long rows, int box_rows) {
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
    const cuuint64_t dims[2] = {(cuuint64_t)head_size, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)head_size};
    const cuuint32_t box[2] = {(cuuint32_t)head_size, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = f(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}



template <typename T, int D>
cudaError_t launch_prefill_tc_d(const TcPrefillParams& tp, cudaStream_t stream) {
    const PrefillParams& p = tp.p;
    // two query tiles per CTA when sequences have at least two (head size
    // <= 128); otherwise one tile with double-buffered scores
    if constexpr (D <= 128) {
        if (p.q_tiles >= 2) {
            using Sh = TcShape2<D, kTcPLo<T>>;
            auto kern = paged_prefill_tc2_kernel<T, T, D>;
            cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Sh::kAlloc);
            if (e != cudaSuccess) return e;
            const long long units = (long long)p.num_seqs * p.num_kv_heads * ((p.q_tiles + 1) / 2);
            if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
            kern<<<(unsigned)units, kTcThreads, Sh::kAlloc, stream>>>(tp);
            return cudaGetLastError();
        }
    }
    using Sh = TcShape<D>;
    auto kern = paged_prefill_tc_kernel<T, T, D>;
    cudaError_t e = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Sh::kAlloc);
    if (e != cudaSuccess) return e;
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

// E4M3 caches (head size 64 or 128): two query tiles per CTA when sequences
// have at least two, else the one-tile kernel. Both maps view the cache as
// [num_blocks*Hkv*B rows][D bytes] with boxes of min(B, 64) rows within one
// block segment: plain (unswizzled) where the tiles are widened to binary16,
// 128-byte swizzled for the E4M3 products (head size 128, bf16 query), the
// layout the kind::f8f6f4 MMAs read.
template <typename QT>
cudaError_t launch_prefill_tc_e4m3(const PrefillParams& p, int head_size, cudaStream_t stream) {
    TcPrefillParams tp;
    tp.p = p;
    const bool e4m3_scores = kTcE4M3Products<QT, e4m3_t, 128> && head_size == 128;
    // the widened tiles hold K and V times 2^-8 (e4m3x2_spread_to_f16x2_scaled);
    // the E4M3 products read K and V as they are stored (their weights carry
    // a power of two that the row sums carry too)
    if (!e4m3_scores) {
        tp.p.q_mul *= 256.f;
        tp.p.v_mul *= 256.f;
    }
    constexpr int n = TcShape<128, true>::N;
    static_assert(TcShape<64, true>::N == n, "one box height for both head sizes");
    // the tiles load by halves: boxes of at most n/2 rows
    tp.box_rows = p.block_size < n / 2 ? p.block_size : n / 2;
    const unsigned long long rows =
        (unsigned long long)p.num_blocks * p.num_kv_heads * p.block_size;
    cudaError_t e = e4m3_scores ? encode_cache_map(&tp.k_map, p.k_cache, 1, head_size, rows, tp.box_rows)
                                : encode_plain_map(&tp.k_map, p.k_cache, head_size, rows, tp.box_rows);
    if (e == cudaSuccess)
        e = e4m3_scores ? encode_cache_map(&tp.v_map, p.v_cache, 1, head_size, rows, tp.box_rows)
                        : encode_plain_map(&tp.v_map, p.v_cache, head_size, rows, tp.box_rows);
    if (e != cudaSuccess) return e;
    static_assert(TcShape2E4M3Scores::N == n && TcShape2<64, false, true>::N == n &&
                      TcShapeE4M3Products::N == n,
                  "the kernels' box height");
    auto go = [&](auto dtag) -> cudaError_t {
        constexpr int D = decltype(dtag)::value;
        if (p.q_tiles >= 2) {
            using Sh2 = std::conditional_t<kTcE4M3Products<QT, e4m3_t, D>, TcShape2E4M3Scores,
                                           TcShape2<D, false, true>>;
            auto kern2 = paged_prefill_tc2_kernel<QT, e4m3_t, D>;
            cudaError_t e2 = ensure_smem_attribute(reinterpret_cast<const void*>(kern2), Sh2::kAlloc);
            if (e2 != cudaSuccess) return e2;
            const long long units = (long long)p.num_seqs * p.num_kv_heads * ((p.q_tiles + 1) / 2);
            if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
            kern2<<<(unsigned)units, kTcThreadsFp8, Sh2::kAlloc, stream>>>(tp);
            return cudaGetLastError();
        }
        using Sh = std::conditional_t<kTcE4M3Products<QT, e4m3_t, D>, TcShapeE4M3Products,
                                      TcShape<D, true>>;
        auto kern = paged_prefill_tc_kernel<QT, e4m3_t, D>;
        cudaError_t e2 = ensure_smem_attribute(reinterpret_cast<const void*>(kern), Sh::kAlloc);
        if (e2 != cudaSuccess) return e2;
        const long long units = (long long)p.num_seqs * p.num_kv_heads * p.q_tiles;
        if (units <= 0) return cudaSuccess;
        if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
        kern<<<(unsigned)units, kTcThreadsFp8, Sh::kAlloc, stream>>>(tp);
        return cudaGetLastError();
    };
    switch (head_size) {
    case 64: return go(std::integral_constant<int, 64>{});
    case 128: return go(std::integral_constant<int, 128>{});
    }
    return cudaErrorInvalidValue;
}

}  // namespace pagedkv
