// Chunked causal prefill on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA), bf16 operands with fp32 accumulation.
//
// Method (BASED reading notes, "Simple linear attention language models
// balance the recall-throughput tradeoff", sec. 2.5, blockwise form):
//   num_b = (M_b o Phi_Qb Phi_Kb^T) V_b + Phi_Qb S_<b,   den_b likewise with 1
//   S_<b+1 = S_<b + Phi_Kb^T V_b
// over 128-token chunks, starting from the caller's initial state
// ("Understanding and Improving Length Generalization in Recurrent Models"
// reading notes, sec. 2.5 Eq. (4)).
//
// GB300 design (one CTA per (b, h), 512 threads, 1 CTA per SM):
//  * Intra-chunk term without feature vectors: T = Q K^T on the tensor core
//    (K = 16), then P = 1 + T/4 + T^2/32 (the Taylor kernel, BASED sec. 2.3)
//    with the causal mask in registers, then P V and P 1 on the tensor core.
//  * Inter-chunk terms on the tensor core with a symmetric-compact feature
//    map inside the kernel: 136 quadratic features (a <= b) + 1 + 16 + 7 pad
//    = 160 instead of 273 (BASED sec. 2.3 table: 1 + d' + d'(d'+1)/2 = 153).
//    Query features carry xbar_a xbar_b, key features xbar_a xbar_b (a < b)
//    and xbar_a^2 / 2, so Phi'_Q . Phi'_K = 1 + q.k/4 + (q.k)^2/32 exactly.
//    The state is held as S' (160 x 64 fp32 in TMEM); it is converted from /
//    to the 273-row layout of the C ABI at the start / end (the antisymmetric
//    part of a caller's s0 cannot influence any output and is passed through).
//  * The normaliser rides on the same MMAs with N = 16 operands: z' via a
//    ones matrix (z' += Phi'_K^T 1), and den via Phi'_Q z' and P 1.
//  * Roles: warp 0 TMA producer (q, k, v chunks, zero-filled past N), warp 1
//    MMA issuer, warpgroup 1 feature generation (one token per thread),
//    warpgroup 2 P epilogue and output epilogue y = num / den, warpgroup 3
//    state conversion S' (TMEM, fp32) -> bf16 shared-memory operand for the
//    next chunk's read-out, and the final state store.
//  * Every wait is bounded: after ~1 s the kernel records a timeout in the
//    device status word and every role unwinds.
#include <utility>

#include "la_internal.h"
#include "tc_common.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;          // tokens per chunk
constexpr int kThreads = 512;
constexpr int kNQuad = 136;      // a <= b pairs
constexpr int kFConst = 136;
constexpr int kFLin = 137;
constexpr int kNReal = 153;

// TMEM columns (512 allocated)
constexpr uint32_t kTmS0 = 0, kTmS1 = 64, kTmZ0 = 128, kTmZ1 = 144;
__host__ __device__ constexpr uint32_t tm_den(int nb) { return nb ? 176u : 160u; }
__host__ __device__ constexpr uint32_t tm_num(int nb) { return nb ? 256u : 192u; }
constexpr uint32_t kTmT = 384;

// Shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kSmPhiQ = 0;        // [blk0 16K][blk1 16K][blk2 8K]: rows = tokens
constexpr uint32_t kSmPhiK = 40960;    // same layout
constexpr uint32_t kSmP = 81920;       // [2][128 rows][128 B] K-major SW128
constexpr uint32_t kSmSb = 114688;     // [160][64] bf16 MN-major SW128
constexpr uint32_t kSmZb = 135168;     // [160][16] bf16 MN-major SW32
constexpr uint32_t kSmOnes = 140288;   // [128][16] bf16 ones
constexpr uint32_t kSmQ = 144384;      // 3 x [128][16] bf16 SW32
constexpr uint32_t kSmK = 156672;      // 3 x [128][16] bf16 SW32
constexpr uint32_t kSmV = 168960;      // 3 x [128][64] bf16 SW128
constexpr uint32_t kSmBar = 218112;
constexpr uint32_t kSmTotal = kSmBar + 512;
constexpr uint32_t kSmAlloc = kSmTotal + 1024;
constexpr int kStages = 3;

// barrier indices
enum {
    B_QK_FULL = 0, B_QK_EMPTY = 3, B_V_FULL = 6, B_V_EMPTY = 9,
    B_T_FULL = 12, B_T_EMPTY, B_P_FULL, B_P_EMPTY, B_PHQ_FULL, B_PHQ_EMPTY,
    B_PHK_FULL, B_PHK_EMPTY, B_NUM_FULL, B_NUM_EMPTY = B_NUM_FULL + 2,
    B_S_FULL = B_NUM_EMPTY + 2, B_SB_FULL, B_FINAL, B_COUNT
};
constexpr uint32_t kSmTmemSlot = kSmBar + 8 * B_COUNT;
constexpr uint32_t kSmAbort = kSmTmemSlot + 4;
static_assert(kSmAbort + 4 <= kSmTotal, "barrier area");

constexpr uint32_t kIdQK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdPV = idesc_bf16(128, 64, false, true);
constexpr uint32_t kIdPV16 = idesc_bf16(128, 16, false, true);
constexpr uint32_t kIdUp = idesc_bf16(128, 64, true, true);
constexpr uint32_t kIdUp16 = idesc_bf16(128, 16, true, true);

constexpr float kSqrt2 = 1.41421356237309504880f;
constexpr float kRSqrt2 = 0.70710678118654752440f;

// (a, b) of compact quadratic feature f: row-major over a <= b.
__host__ __device__ constexpr int pair_a(int f) {
    int a = 0, base = 0;
    while (f >= base + (16 - a)) { base += 16 - a; ++a; }
    return a;
}
__host__ __device__ constexpr int pair_b(int f) {
    int a = pair_a(f);
    return f - (16 * a - a * (a - 1) / 2) + a;
}
static_assert(pair_a(135) == 15 && pair_b(135) == 15 && pair_a(16) == 1 && pair_b(16) == 1, "");

// Compact feature F of xbar (x / 2).  Key features halve the squares.
template <bool kKey, int F>
__device__ __forceinline__ float feat(const float (&x)[16]) {
    if constexpr (F < kNQuad) {
        constexpr int a = pair_a(F), b = pair_b(F);
        if constexpr (kKey && a == b) return 0.5f * (x[a] * x[b]);
        else return x[a] * x[b];
    } else if constexpr (F == kFConst) {
        return 1.0f;
    } else if constexpr (F < kNReal) {
        return x[F - kFLin];
    } else {
        return 0.0f;
    }
}

// Shared-memory byte offset of 16-byte chunk J (features 8J..8J+7) of row t
// in a feature buffer: two 128-B-swizzled 64-feature blocks + one 64-B-swizzled
// 32-feature block.
__device__ __forceinline__ uint32_t feat_chunk_off(int J, int t) {
    if (J < 8) return (uint32_t)(t * 128 + ((J ^ (t & 7)) << 4));
    if (J < 16) return 16384u + (uint32_t)(t * 128 + (((J - 8) ^ (t & 7)) << 4));
    return 32768u + (uint32_t)(t * 64 + (((J - 16) ^ ((t >> 1) & 3)) << 4));
}

template <bool kKey, int J>
__device__ __forceinline__ void emit_chunk(const float (&x)[16], uint32_t base, int t, bool zero) {
    uint32_t w[4];
    w[0] = pack_bf16(feat<kKey, 8 * J + 0>(x), feat<kKey, 8 * J + 1>(x));
    w[1] = pack_bf16(feat<kKey, 8 * J + 2>(x), feat<kKey, 8 * J + 3>(x));
    w[2] = pack_bf16(feat<kKey, 8 * J + 4>(x), feat<kKey, 8 * J + 5>(x));
    w[3] = pack_bf16(feat<kKey, 8 * J + 6>(x), feat<kKey, 8 * J + 7>(x));
    if (zero) w[0] = w[1] = w[2] = w[3] = 0u;
    st_shared_v4(base + feat_chunk_off(J, t), w[0], w[1], w[2], w[3]);
}

template <bool kKey, int... J>
__device__ __forceinline__ void emit_features(const float (&x)[16], uint32_t base, int t,
                                              bool zero, std::integer_sequence<int, J...>) {
    (emit_chunk<kKey, J>(x, base, t, zero), ...);
}

// Read token row t (16 bf16) of a [128][16] SW32 tile as xbar = x / 2.
__device__ __forceinline__ void load_row16(uint32_t tile, int t, float (&x)[16]) {
    const uint32_t sw = (uint32_t)((t >> 2) & 1);
    const uint4 lo = ld_shared_v4(tile + t * 32 + ((0u ^ sw) << 4));
    const uint4 hi = ld_shared_v4(tile + t * 32 + ((1u ^ sw) << 4));
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = 0.5f * bf16lo(w[i]);
        x[2 * i + 1] = 0.5f * bf16hi(w[i]);
    }
}

// ABI row(s) of compact feature f: r1, r2 (r2 < 0 if none); kind 0 = square,
// 1 = off-diagonal pair, 2 = constant / linear, 3 = padding.
struct Rows { int r1, r2, kind; };
__device__ __forceinline__ Rows abi_rows(int f) {
    if (f < kNQuad) {
        int a = 0, base = 0;
        while (f >= base + (16 - a)) { base += 16 - a; ++a; }
        const int b = f - base + a;
        if (a == b) return {17 + 17 * a, -1, 0};
        return {17 + 16 * a + b, 17 + 16 * b + a, 1};
    }
    if (f == kFConst) return {0, -1, 2};
    if (f < kNReal) return {1 + (f - kFLin), -1, 2};
    return {-1, -1, 3};
}

// Compact S' row f (64 values) and z'[f] from the ABI initial state.
__device__ __forceinline__ void load_initial(const float *s0, const float *z0, int64_t bh, int f,
                                             float (&srow)[64], float &zf) {
    const Rows r = abi_rows(f);
#pragma unroll
    for (int j = 0; j < 64; ++j) srow[j] = 0.f;
    zf = 0.f;
    if (!s0 || r.kind == 3) return;
    const float4 *p1 = reinterpret_cast<const float4 *>(s0 + (bh * kD + r.r1) * kDV);
    const float z1 = z0[bh * kD + r.r1];
    if (r.kind == 2) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 a = p1[j];
            srow[4 * j] = a.x; srow[4 * j + 1] = a.y; srow[4 * j + 2] = a.z; srow[4 * j + 3] = a.w;
        }
        zf = z1;
    } else if (r.kind == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 a = p1[j];
            srow[4 * j] = a.x * kRSqrt2; srow[4 * j + 1] = a.y * kRSqrt2;
            srow[4 * j + 2] = a.z * kRSqrt2; srow[4 * j + 3] = a.w * kRSqrt2;
        }
        zf = z1 * kRSqrt2;
    } else {
        const float4 *p2 = reinterpret_cast<const float4 *>(s0 + (bh * kD + r.r2) * kDV);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 a = p1[j], b = p2[j];
            srow[4 * j] = (a.x + b.x) * kRSqrt2; srow[4 * j + 1] = (a.y + b.y) * kRSqrt2;
            srow[4 * j + 2] = (a.z + b.z) * kRSqrt2; srow[4 * j + 3] = (a.w + b.w) * kRSqrt2;
        }
        zf = (z1 + z0[bh * kD + r.r2]) * kRSqrt2;
    }
}

// Write compact row f of the final state back to the ABI layout.
__device__ __forceinline__ void store_final(const float *s0, const float *z0, float *s_out,
                                            float *z_out, int64_t bh, int f,
                                            const float (&srow)[64], float zf) {
    const Rows r = abi_rows(f);
    if (r.kind == 3) return;
    if (r.kind == 1) {
        // S'/sqrt2 is the symmetric part; the antisymmetric part of s0 passes through.
        float4 *o1 = s_out ? reinterpret_cast<float4 *>(s_out + (bh * kD + r.r1) * kDV) : nullptr;
        float4 *o2 = s_out ? reinterpret_cast<float4 *>(s_out + (bh * kD + r.r2) * kDV) : nullptr;
        const float4 *a1 = s0 ? reinterpret_cast<const float4 *>(s0 + (bh * kD + r.r1) * kDV) : nullptr;
        const float4 *a2 = s0 ? reinterpret_cast<const float4 *>(s0 + (bh * kD + r.r2) * kDV) : nullptr;
        if (o1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float4 sym = make_float4(srow[4 * j] * kRSqrt2, srow[4 * j + 1] * kRSqrt2,
                                         srow[4 * j + 2] * kRSqrt2, srow[4 * j + 3] * kRSqrt2);
                float4 anti = make_float4(0.f, 0.f, 0.f, 0.f);
                if (a1) {
                    const float4 x = a1[j], y = a2[j];
                    anti = make_float4(0.5f * (x.x - y.x), 0.5f * (x.y - y.y), 0.5f * (x.z - y.z),
                                       0.5f * (x.w - y.w));
                }
                o1[j] = make_float4(sym.x + anti.x, sym.y + anti.y, sym.z + anti.z, sym.w + anti.w);
                o2[j] = make_float4(sym.x - anti.x, sym.y - anti.y, sym.z - anti.z, sym.w - anti.w);
            }
        }
        if (z_out) {
            const float sym = zf * kRSqrt2;
            const float anti = z0 ? 0.5f * (z0[bh * kD + r.r1] - z0[bh * kD + r.r2]) : 0.f;
            z_out[bh * kD + r.r1] = sym + anti;
            z_out[bh * kD + r.r2] = sym - anti;
        }
        return;
    }
    const float sc = r.kind == 0 ? kSqrt2 : 1.0f;
    if (s_out) {
        float4 *o = reinterpret_cast<float4 *>(s_out + (bh * kD + r.r1) * kDV);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            o[j] = make_float4(srow[4 * j] * sc, srow[4 * j + 1] * sc, srow[4 * j + 2] * sc,
                               srow[4 * j + 3] * sc);
    }
    if (z_out) z_out[bh * kD + r.r1] = zf * sc;
}

// bf16 copy of S' row f (64 values) into the MN-major SW128 operand, and z'[f]
// into column 0 of the [160][16] SW32 operand.
__device__ __forceinline__ void write_state_operand(uint32_t sb, uint32_t zb, int f,
                                                    const float (&srow)[64], float zf) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        st_shared_v4(sb + f * 128 + ((j ^ (f & 7)) << 4),
                     pack_bf16(srow[8 * j + 0], srow[8 * j + 1]),
                     pack_bf16(srow[8 * j + 2], srow[8 * j + 3]),
                     pack_bf16(srow[8 * j + 4], srow[8 * j + 5]),
                     pack_bf16(srow[8 * j + 6], srow[8 * j + 7]));
    }
    st_shared_v4(zb + f * 32 + (((f >> 2) & 1) << 4), pack_bf16(zf, 0.f), 0u, 0u, 0u);
}

__device__ __forceinline__ void tmem_load_row64(uint32_t taddr, float (&srow)[64]) {
    uint32_t r0[32], r1[32];
    tmem_ld32(taddr, r0);
    tmem_ld32(taddr + 32, r1);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        srow[j] = __uint_as_float(r0[j]);
        srow[32 + j] = __uint_as_float(r1[j]);
    }
}

__device__ __forceinline__ void tmem_store_row64(uint32_t taddr, const float (&srow)[64]) {
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(srow[j]);
    tmem_st32(taddr, r);
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(srow[32 + j]);
    tmem_st32(taddr + 32, r);
}

__device__ __forceinline__ void tmem_store_z16(uint32_t taddr, float zf) {
    uint32_t r[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(zf);
    tmem_st16(taddr, r);
}

// Drain wait used when unwinding: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return;
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const float *__restrict__ s0,
                  const float *__restrict__ z0, __nv_bfloat16 *__restrict__ y,
                  float *__restrict__ s_out, float *__restrict__ z_out, int N, float eps,
                  unsigned *status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) { return sb + kSmBar + 8u * (uint32_t)i; };
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kSmAbort);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t bh = blockIdx.x;
    const int n = (N + kC - 1) / kC;

    // ---- set-up: barriers, TMEM, constant operands
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_QK_FULL + s), 1);
            mbar_init(bar(B_QK_EMPTY + s), 1 + 4);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        mbar_init(bar(B_T_FULL), 1);
        mbar_init(bar(B_T_EMPTY), 4);
        mbar_init(bar(B_P_FULL), 4);
        mbar_init(bar(B_P_EMPTY), 1);
        mbar_init(bar(B_PHQ_FULL), 4);
        mbar_init(bar(B_PHQ_EMPTY), 1);
        mbar_init(bar(B_PHK_FULL), 4);
        mbar_init(bar(B_PHK_EMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_NUM_FULL + i), 1);
            mbar_init(bar(B_NUM_EMPTY + i), 4);
        }
        mbar_init(bar(B_S_FULL), 1);
        mbar_init(bar(B_SB_FULL), 4);
        mbar_init(bar(B_FINAL), 1);
        *abort = 0;
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(sb + kSmTmemSlot, 512);
        tmem_relinquish();
    }
    // ones operand, and zero the z' operand (only its column 0 is rewritten later)
    for (int i = tid; i < 4096 / 16; i += kThreads)
        st_shared_v4(sb + kSmOnes + 16 * i, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    for (int i = tid; i < 5120 / 16; i += kThreads) st_shared_v4(sb + kSmZb + 16 * i, 0u, 0u, 0u, 0u);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kSmTmemSlot);

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            int issued_qk = 0, issued_v = 0;
            for (int c = 0; c < n; ++c) {
                const int st = c % kStages;
                const uint32_t ph = ((uint32_t)(c / kStages) & 1u) ^ 1u;
                if (!mbar_wait(bar(B_QK_EMPTY + st), ph, abort, status)) break;
                mbar_expect_tx(bar(B_QK_FULL + st), 2 * kC * 16 * 2);
                tma_load_3d(sb + kSmQ + st * 4096, &tq, bar(B_QK_FULL + st), 0, c * kC, (int)bh);
                tma_load_3d(sb + kSmK + st * 4096, &tk, bar(B_QK_FULL + st), 0, c * kC, (int)bh);
                issued_qk = c + 1;
                if (!mbar_wait(bar(B_V_EMPTY + st), ph, abort, status)) break;
                mbar_expect_tx(bar(B_V_FULL + st), kC * 64 * 2);
                tma_load_3d(sb + kSmV + st * 16384, &tv, bar(B_V_FULL + st), 0, c * kC, (int)bh);
                issued_v = c + 1;
            }
            if (*abort) {
                // every issued load must land before the CTA may exit; the last
                // kStages chunks are the latest use of each stage
                for (int c = (issued_qk > kStages ? issued_qk - kStages : 0); c < issued_qk; ++c)
                    drain_wait(bar(B_QK_FULL + c % kStages), (uint32_t)(c / kStages) & 1u);
                for (int c = (issued_v > kStages ? issued_v - kStages : 0); c < issued_v; ++c)
                    drain_wait(bar(B_V_FULL + c % kStages), (uint32_t)(c / kStages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            auto qdesc = [&](int st) { return smem_desc(sb + kSmQ + st * 4096, 16, 256, kSw32); };
            auto kdesc = [&](int st) { return smem_desc(sb + kSmK + st * 4096, 16, 256, kSw32); };
            auto vdesc = [&](int st, int s) {
                return smem_desc(sb + kSmV + st * 16384 + s * 2048, 16384, 1024, kSw128);
            };
            auto onesdesc = [&](int s) { return smem_desc(sb + kSmOnes + s * 512, 4096, 256, kSw32); };
            auto pdesc = [&](int s) {
                return smem_desc(sb + kSmP + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024, kSw128);
            };
            auto phiqdesc = [&](int s) {
                return s < 8 ? smem_desc(sb + kSmPhiQ + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024, kSw128)
                             : smem_desc(sb + kSmPhiQ + 32768 + (s - 8) * 32, 16, 512, kSw64);
            };
            auto sbdesc = [&](int s) { return smem_desc(sb + kSmSb + s * 2048, 16384, 1024, kSw128); };
            auto zbdesc = [&](int s) { return smem_desc(sb + kSmZb + s * 512, 4096, 256, kSw32); };
            auto phik0desc = [&](int s) { return smem_desc(sb + kSmPhiK + s * 2048, 16384, 1024, kSw128); };
            auto phik1desc = [&](int s) { return smem_desc(sb + kSmPhiK + 32768 + s * 1024, 8192, 512, kSw64); };

            bool ok = mbar_wait(bar(B_QK_FULL + 0), 0, abort, status);
            if (ok) {
                tc_fence_after();
                mma_bf16(tmem + kTmT, qdesc(0), kdesc(0), kIdQK, 0);
                mma_commit(bar(B_T_FULL));
                mma_commit(bar(B_QK_EMPTY + 0));
            }
            for (int c = 0; ok && c < n; ++c) {
                const int vs = c % kStages, nb = c & 1;
                const uint32_t pc = (uint32_t)c & 1u;
                ok = mbar_wait(bar(B_P_FULL), pc, abort, status) &&
                     mbar_wait(bar(B_V_FULL + vs), (uint32_t)(c / kStages) & 1u, abort, status) &&
                     mbar_wait(bar(B_NUM_EMPTY + nb), ((uint32_t)(c >> 1) & 1u) ^ 1u, abort, status);
                if (!ok) break;
                tc_fence_after();
                // intra-chunk: num = P V, den = P 1
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    mma_bf16(tmem + tm_num(nb), pdesc(s), vdesc(vs, s), kIdPV, s > 0);
                    mma_bf16(tmem + tm_den(nb), pdesc(s), onesdesc(s), kIdPV16, s > 0);
                }
                mma_commit(bar(B_P_EMPTY));
                // next chunk's Q K^T as soon as its tiles are in
                if (c + 1 < n) {
                    const int st = (c + 1) % kStages;
                    ok = mbar_wait(bar(B_QK_FULL + st), (uint32_t)((c + 1) / kStages) & 1u, abort, status) &&
                         mbar_wait(bar(B_T_EMPTY), pc, abort, status);
                    if (!ok) break;
                    tc_fence_after();
                    mma_bf16(tmem + kTmT, qdesc(st), kdesc(st), kIdQK, 0);
                    mma_commit(bar(B_T_FULL));
                    mma_commit(bar(B_QK_EMPTY + st));
                }
                // inter-chunk read-out: num += Phi'_Q S', den += Phi'_Q z'
                ok = mbar_wait(bar(B_SB_FULL), pc, abort, status) &&
                     mbar_wait(bar(B_PHQ_FULL), pc, abort, status);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 10; ++s) {
                    mma_bf16(tmem + tm_num(nb), phiqdesc(s), sbdesc(s), kIdPV, 1);
                    mma_bf16(tmem + tm_den(nb), phiqdesc(s), zbdesc(s), kIdPV16, 1);
                }
                mma_commit(bar(B_NUM_FULL + nb));
                mma_commit(bar(B_PHQ_EMPTY));
                // state update: S' += Phi'_K^T V, z' += Phi'_K^T 1
                ok = mbar_wait(bar(B_PHK_FULL), pc, abort, status);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    mma_bf16(tmem + kTmS0, phik0desc(s), vdesc(vs, s), kIdUp, 1);
                    mma_bf16(tmem + kTmZ0, phik0desc(s), onesdesc(s), kIdUp16, 1);
                }
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    mma_bf16(tmem + kTmS1, phik1desc(s), vdesc(vs, s), kIdUp, 1);
                    mma_bf16(tmem + kTmZ1, phik1desc(s), onesdesc(s), kIdUp16, 1);
                }
                mma_commit(bar(B_S_FULL));
                mma_commit(bar(B_PHK_EMPTY));
                mma_commit(bar(B_V_EMPTY + vs));
            }
            // every issued MMA must finish before TMEM is released
            mma_commit(bar(B_FINAL));
            drain_wait(bar(B_FINAL), 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ================= feature generation (one token per thread) =================
        const int t = tid - 128;
        for (int c = 0; c < n; ++c) {
            const int st = c % kStages;
            const uint32_t pc = (uint32_t)c & 1u;
            if (!mbar_wait(bar(B_QK_FULL + st), (uint32_t)(c / kStages) & 1u, abort, status)) break;
            float xq[16], xk[16];
            load_row16(sb + kSmQ + st * 4096, t, xq);
            load_row16(sb + kSmK + st * 4096, t, xk);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QK_EMPTY + st));
            if (!mbar_wait(bar(B_PHQ_EMPTY), pc ^ 1u, abort, status)) break;
            emit_features<false>(xq, sb + kSmPhiQ, t, false, std::make_integer_sequence<int, 20>{});
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PHQ_FULL));
            const bool pad = c * kC + t >= N;  // past the end: no contribution to S', z'
            if (!mbar_wait(bar(B_PHK_EMPTY), pc ^ 1u, abort, status)) break;
            emit_features<true>(xk, sb + kSmPhiK, t, pad, std::make_integer_sequence<int, 20>{});
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PHK_FULL));
        }
    } else if (warp >= 8 && warp < 12) {
        // ================= P epilogue and output epilogue =================
        const int w = warp - 8;
        const int i = tid - 256;  // query row within the chunk (= TMEM lane)
        const uint32_t lanebase = (uint32_t)(32 * w) << 16;
        auto do_p = [&](int c) -> bool {
            const uint32_t pc = (uint32_t)c & 1u;
            if (!mbar_wait(bar(B_T_FULL), pc, abort, status)) return false;
            if (!mbar_wait(bar(B_P_EMPTY), pc ^ 1u, abort, status)) return false;
            tc_fence_after();
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t pw[16];
                if (p <= w) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lanebase + kTmT + 32 * p, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float t0 = __uint_as_float(r[2 * j]), t1 = __uint_as_float(r[2 * j + 1]);
                        float p0 = fmaf(t0, fmaf(t0, 0.03125f, 0.25f), 1.0f);
                        float p1 = fmaf(t1, fmaf(t1, 0.03125f, 0.25f), 1.0f);
                        if (p == w) {
                            if (32 * p + 2 * j > i) p0 = 0.f;
                            if (32 * p + 2 * j + 1 > i) p1 = 0.f;
                        }
                        pw[j] = pack_bf16(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) pw[j] = 0u;
                }
                const uint32_t blk = sb + kSmP + (uint32_t)(p >> 1) * 16384 + i * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int J = (p & 1) * 4 + q;
                    st_shared_v4(blk + ((J ^ (i & 7)) << 4), pw[4 * q], pw[4 * q + 1], pw[4 * q + 2],
                                 pw[4 * q + 3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_T_EMPTY));
                mbar_arrive(bar(B_P_FULL));
            }
            return true;
        };
        auto do_y = [&](int c) -> bool {
            const int nb = c & 1;
            if (!mbar_wait(bar(B_NUM_FULL + nb), (uint32_t)(c >> 1) & 1u, abort, status)) return false;
            tc_fence_after();
            uint32_t r0[32], r1[32], dr;
            tmem_ld32(tmem + lanebase + tm_num(nb), r0);
            tmem_ld32(tmem + lanebase + tm_num(nb) + 32, r1);
            tmem_ld1(tmem + lanebase + tm_den(nb), dr);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_NUM_EMPTY + nb));
            const int row = c * kC + i;
            if (row < N) {
                const float inv = 1.0f / (__uint_as_float(dr) + eps);
                uint4 *dst = reinterpret_cast<uint4 *>(y + ((int64_t)bh * N + row) * kDV);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    dst[j] = make_uint4(
                        pack_bf16(__uint_as_float(r0[8 * j + 0]) * inv, __uint_as_float(r0[8 * j + 1]) * inv),
                        pack_bf16(__uint_as_float(r0[8 * j + 2]) * inv, __uint_as_float(r0[8 * j + 3]) * inv),
                        pack_bf16(__uint_as_float(r0[8 * j + 4]) * inv, __uint_as_float(r0[8 * j + 5]) * inv),
                        pack_bf16(__uint_as_float(r0[8 * j + 6]) * inv, __uint_as_float(r0[8 * j + 7]) * inv));
                    dst[4 + j] = make_uint4(
                        pack_bf16(__uint_as_float(r1[8 * j + 0]) * inv, __uint_as_float(r1[8 * j + 1]) * inv),
                        pack_bf16(__uint_as_float(r1[8 * j + 2]) * inv, __uint_as_float(r1[8 * j + 3]) * inv),
                        pack_bf16(__uint_as_float(r1[8 * j + 4]) * inv, __uint_as_float(r1[8 * j + 5]) * inv),
                        pack_bf16(__uint_as_float(r1[8 * j + 6]) * inv, __uint_as_float(r1[8 * j + 7]) * inv));
                }
            }
            return true;
        };
        if (do_p(0)) {
            for (int c = 0; c < n; ++c) {
                if (c + 1 < n && !do_p(c + 1)) break;
                if (!do_y(c)) break;
            }
        }
    } else if (warp >= 12) {
        // ================= state conversion =================
        const int w = warp - 12;
        const int f = 32 * w + lane;          // compact feature of TMEM tile 0 (lane f)
        const int f1 = 128 + lane;            // compact feature of tile 1 (warp 12 only)
        const uint32_t lanebase = (uint32_t)(32 * w) << 16;
        {
            float srow[64], zf;
            load_initial(s0, z0, bh, f, srow, zf);
            tmem_store_row64(tmem + lanebase + kTmS0, srow);
            tmem_store_z16(tmem + lanebase + kTmZ0, zf);
            write_state_operand(sb + kSmSb, sb + kSmZb, f, srow, zf);
            if (w == 0) {
                load_initial(s0, z0, bh, f1, srow, zf);
                tmem_store_row64(tmem + kTmS1, srow);
                tmem_store_z16(tmem + kTmZ1, zf);
                write_state_operand(sb + kSmSb, sb + kSmZb, f1, srow, zf);
            }
            tmem_wait_st();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_SB_FULL));
        }
        for (int c = 0; c < n; ++c) {
            if (!mbar_wait(bar(B_S_FULL), (uint32_t)c & 1u, abort, status)) break;
            tc_fence_after();
            float srow[64];
            uint32_t zr;
            const bool last = (c == n - 1);
            tmem_ld1(tmem + lanebase + kTmZ0, zr);
            tmem_load_row64(tmem + lanebase + kTmS0, srow);
            if (!last) {
                write_state_operand(sb + kSmSb, sb + kSmZb, f, srow, __uint_as_float(zr));
            } else {
                store_final(s0, z0, s_out, z_out, bh, f, srow, __uint_as_float(zr));
            }
            if (w == 0) {
                tmem_ld1(tmem + kTmZ1, zr);
                tmem_load_row64(tmem + kTmS1, srow);
                if (!last) write_state_operand(sb + kSmSb, sb + kSmZb, f1, srow, __uint_as_float(zr));
                else store_final(s0, z0, s_out, z_out, bh, f1, srow, __uint_as_float(zr));
            }
            if (!last) {
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_SB_FULL));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    }
    return fn;
}

}  // namespace

// [BH][N][width] bf16 rows as a 3-D tensor map with a {width, 128, 1} box;
// rows past N read as zero.
bool make_row_tmap(CUtensorMap *map, const void *base, int64_t BH, int64_t N, int width,
                   bool swizzle128) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)N * width * 2};
    const cuuint32_t box[3] = {(cuuint32_t)width, 128u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    if (a.N > (int64_t)0x7FFFFFFF - kC) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv;
    if (!make_row_tmap(&tq, a.q, BH, a.N, 16, false) || !make_row_tmap(&tk, a.k, BH, a.N, 16, false) ||
        !make_row_tmap(&tv, a.v, BH, a.N, 64, true))
        return cudaErrorInvalidValue;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e != cudaSuccess) return e;
        configured_for = dev;
    }
    prefill_tc_kernel<<<(unsigned)BH, kThreads, kSmAlloc, st>>>(
        tq, tk, tv, a.s0, a.z0, (__nv_bfloat16 *)a.y, a.s_out, a.z_out, (int)a.N, a.eps, a.status);
    return cudaGetLastError();
}

}  // namespace la
