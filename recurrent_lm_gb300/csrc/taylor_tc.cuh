// Device helpers shared by the tensor-core kernels: the internal compact
// Taylor feature map, its packed generation, and the conversion between the
// internal state rows and the 273-row state layout of the C ABI.
//
// Feature map (BASED reading notes, "Simple linear attention language models
// balance the recall-throughput tradeoff", sec. 2.3): phi(x) = [1, xbar,
// vec(xbar xbar^T)/sqrt(2)], xbar = x / 2, so phi(q).phi(k) = 1 + q.k/4 +
// (q.k)^2/32.  Inside the kernels the symmetric-compact form is used
// (1 + 16 + 136 features, the table on the same page), padded to 160.
#pragma once

#include <stdint.h>
#include <utility>

#include "la_internal.h"
#include "tc_common.cuh"

namespace la {
namespace taylor {

using namespace tc;

constexpr int kNFeat = 160;      // compact features (153 real + 7 zero)

constexpr float kSqrt2 = 1.41421356237309504880f;
constexpr float kRSqrt2 = 0.70710678118654752440f;

// Compact feature order (160 features = 80 packed bf16 pairs), chosen so that
// every pair of quadratic features is one bf16x2 product of packed inputs:
//   pairs  0..7   squares (2j, 2j) and (2j+1, 2j+1)
//   pairs  8..63  for offset d = 1..15, j < (16 - d) / 2: (2j, 2j+d), (2j+1, 2j+1+d)
//   pairs 64..67  the leftovers (4i, 15), (4i+2, 15) of the odd offsets
//   pairs 68..75  linear xbar_{2j}, xbar_{2j+1};  pair 76: (1, 0);  77..79: 0
// Query features are xbar_a xbar_b; key features the same except the squares,
// which are halved, so Phi'_Q . Phi'_K = 1 + qbar.kbar + (qbar.kbar)^2 / 2.
struct PairSpec { int kind, j, d; };  // kind 0 square, 1 off-diagonal, 2 leftover, 3 linear, 4 const, 5 zero
__host__ __device__ constexpr PairSpec pair_spec(int r) {
    if (r < 8) return {0, r, 0};
    int k = 8;
    for (int d = 1; d <= 15; ++d) {
        const int m = (16 - d) / 2;
        if (r < k + m) return {1, r - k, d};
        k += m;
    }
    if (r < 68) return {2, r - 64, 0};
    if (r < 76) return {3, r - 68, 0};
    if (r == 76) return {4, 0, 0};
    return {5, 0, 0};
}
static_assert(pair_spec(63).kind == 1 && pair_spec(63).d == 14 && pair_spec(64).kind == 2, "layout");

// (a, b) of the two quadratic features of pair r (b = -1: linear / constant / zero).
__host__ __device__ constexpr void pair_ab(int r, int e, int &a, int &b) {
    const PairSpec p = pair_spec(r);
    if (p.kind == 0) { a = b = 2 * p.j + e; return; }
    if (p.kind == 1) { a = 2 * p.j + e; b = a + p.d; return; }
    if (p.kind == 2) { a = 4 * p.j + 2 * e; b = 15; return; }
    a = b = -1;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t x, uint32_t y) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
}

// Packed features of one token: X[j] = (xbar_2j, xbar_2j+1) as bf16x2, Y[j] =
// (xbar_2j+1, xbar_2j+2), H[j] = X[j] / 2 (keys only).  XL[j] is the left
// factor of every product: X[j] itself, or X[j] times a per-token scale when
// the whole feature vector is scaled (then cst = (scale, 0) is the constant
// feature), so scaling costs 8 multiplies instead of 80.
template <bool kKey, int R>
__device__ __forceinline__ uint32_t feat_pair(const uint32_t (&XL)[8], const uint32_t (&X)[8],
                                              const uint32_t (&Y)[7], const uint32_t (&H)[8],
                                              uint32_t b15, uint32_t cst) {
    constexpr PairSpec p = pair_spec(R);
    if constexpr (p.kind == 0) {
        if constexpr (kKey) return hmul2(XL[p.j], H[p.j]);
        else return hmul2(XL[p.j], X[p.j]);
    } else if constexpr (p.kind == 1) {
        if constexpr (p.d % 2 == 0) return hmul2(XL[p.j], X[p.j + p.d / 2]);
        else return hmul2(XL[p.j], Y[p.j + (p.d - 1) / 2]);
    } else if constexpr (p.kind == 2) {
        return hmul2(__byte_perm(XL[2 * p.j], XL[2 * p.j + 1], 0x5410), b15);
    } else if constexpr (p.kind == 3) {
        return XL[p.j];
    } else if constexpr (p.kind == 4) {
        return cst;  // (1.0, 0), or (scale, 0)
    } else {
        return 0u;
    }
}

// Shared-memory byte offset of 16-byte chunk J (features 8J..8J+7) of token
// row t: two 128-B-swizzled 64-feature blocks, then features 128..159 in a
// 64-B-swizzled block (queries, K-major A) or in a 128-B-swizzled block
// (keys, MN-major B: one 64-feature atom of which 32 are used).
template <bool kKey>
__device__ __forceinline__ uint32_t feat_chunk_off(int J, int t) {
    if (J < 8) return (uint32_t)(t * 128 + ((J ^ (t & 7)) << 4));
    if (J < 16) return 16384u + (uint32_t)(t * 128 + (((J - 8) ^ (t & 7)) << 4));
    if (kKey) return 32768u + (uint32_t)(t * 128 + (((J - 16) ^ (t & 7)) << 4));
    return 32768u + (uint32_t)(t * 64 + (((J - 16) ^ ((t >> 1) & 3)) << 4));
}

template <bool kKey, int J>
__device__ __forceinline__ void emit_chunk(const uint32_t (&XL)[8], const uint32_t (&X)[8],
                                           const uint32_t (&Y)[7], const uint32_t (&H)[8], uint32_t b15,
                                           uint32_t cst, uint32_t base, int t, bool zero) {
    uint32_t w0 = feat_pair<kKey, 4 * J + 0>(XL, X, Y, H, b15, cst);
    uint32_t w1 = feat_pair<kKey, 4 * J + 1>(XL, X, Y, H, b15, cst);
    uint32_t w2 = feat_pair<kKey, 4 * J + 2>(XL, X, Y, H, b15, cst);
    uint32_t w3 = feat_pair<kKey, 4 * J + 3>(XL, X, Y, H, b15, cst);
    if (zero) w0 = w1 = w2 = w3 = 0u;
    st_shared_v4(base + feat_chunk_off<kKey>(J, t), w0, w1, w2, w3);
}

// xbar as packed bf16 pairs from the raw token row.  kDk = 16: xbar = x / 2
// (exact).  kDk = 8: the row holds x in dims 0..7 and zeros in 8..15, and
// xbar = x / 8^(1/4) = x 2^-3/4 (one rounding to bf16); the d' = 8 map is then
// the d' = 16 map of the padded row, restricted to the dims 0..7 (its other
// features are zero): 16^(1/4) (2^(1/4) x) / 16^(1/4) = x 2^-3/4 per input,
// so the feature values coincide.
template <int kDk>
__device__ __forceinline__ void xbar_pairs(const uint32_t (&raw)[8], uint32_t (&X)[8]) {
    if constexpr (kDk == 16) {
#pragma unroll
        for (int j = 0; j < 8; ++j) X[j] = hmul2(raw[j], 0x3F003F00u);
    } else {
        static_assert(kDk == 8, "d' = 16 or 8");
        constexpr float kS = 0.59460355750136053f;  // 2^-3/4
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(raw[j] << 16), hi = __uint_as_float(raw[j] & 0xFFFF0000u);
            X[j] = pack_bf16(lo * kS, hi * kS);
        }
#pragma unroll
        for (int j = 4; j < 8; ++j) X[j] = 0u;
    }
}

// Feature vector of one token into its row of the feature tile; with kScaled
// every feature is multiplied by scale2 (a bf16x2 pair of the same scale).
template <bool kKey, bool kScaled = false, int kDk = 16, int... J>
__device__ __forceinline__ void emit_features(const uint4 &lo, const uint4 &hi, uint32_t base, int t,
                                              bool zero, std::integer_sequence<int, J...>,
                                              uint32_t scale2 = 0x3F803F80u) {
    // xbar, its odd-shifted pairs, and halves for the key squares
    const uint32_t raw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t X[8], Y[7], H[8];
    xbar_pairs<kDk>(raw, X);
#pragma unroll
    for (int j = 0; j < 7; ++j) Y[j] = __byte_perm(X[j], X[j + 1], 0x5432);
#pragma unroll
    for (int j = 0; j < 8; ++j) H[j] = kKey ? hmul2(X[j], 0x3F003F00u) : 0u;
    const uint32_t b15 = __byte_perm(X[7], X[7], 0x3232);
    if constexpr (kScaled) {
        uint32_t XL[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) XL[j] = hmul2(X[j], scale2);
        const uint32_t cst = scale2 & 0xFFFFu;
        (emit_chunk<kKey, J>(XL, X, Y, H, b15, cst, base, t, zero), ...);
    } else {
        (emit_chunk<kKey, J>(X, X, Y, H, b15, 0x00003F80u, base, t, zero), ...);
    }
}

// Feature vector of one token into its TMEM lane (columns taddr + r for the
// 80 packed pairs r, the layout of an A operand in TMEM: two consecutive K
// elements per 32-bit column), with 5 warp-collective stores of 16 columns.
template <bool kKey, int G, int... J>
__device__ __forceinline__ void store_feature_group(const uint32_t (&XL)[8], const uint32_t (&X)[8],
                                                    const uint32_t (&Y)[7], const uint32_t (&H)[8],
                                                    uint32_t b15, uint32_t cst, uint32_t taddr,
                                                    std::integer_sequence<int, J...>) {
    uint32_t w[16];
    ((w[J] = feat_pair<kKey, 16 * G + J>(XL, X, Y, H, b15, cst)), ...);
    tmem_store16_sync(taddr + 16 * G, w);
}
template <bool kKey, bool kScaled = false, int kDk = 16, int... G>
__device__ __forceinline__ void emit_features_tmem(const uint4 &lo, const uint4 &hi, uint32_t taddr,
                                                   std::integer_sequence<int, G...>,
                                                   uint32_t scale2 = 0x3F803F80u) {
    const uint32_t raw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t X[8], Y[7], H[8];
    xbar_pairs<kDk>(raw, X);
#pragma unroll
    for (int j = 0; j < 7; ++j) Y[j] = __byte_perm(X[j], X[j + 1], 0x5432);
#pragma unroll
    for (int j = 0; j < 8; ++j) H[j] = kKey ? hmul2(X[j], 0x3F003F00u) : 0u;
    const uint32_t b15 = __byte_perm(X[7], X[7], 0x3232);
    if constexpr (kScaled) {
        uint32_t XL[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) XL[j] = hmul2(X[j], scale2);
        (store_feature_group<kKey, G>(XL, X, Y, H, b15, scale2 & 0xFFFFu, taddr,
                                      std::make_integer_sequence<int, 16>{}), ...);
    } else {
        (store_feature_group<kKey, G>(X, X, Y, H, b15, 0x00003F80u, taddr,
                                      std::make_integer_sequence<int, 16>{}), ...);
    }
}

// Raw token row t (16 bf16 as two 16-byte halves) of a [128][16] SW32 tile.
__device__ __forceinline__ void load_row16_raw(uint32_t tile, int t, uint4 &lo, uint4 &hi) {
    const uint32_t sw = (uint32_t)((t >> 2) & 1);
    lo = ld_shared_v4(tile + t * 32 + ((0u ^ sw) << 4));
    hi = ld_shared_v4(tile + t * 32 + ((1u ^ sw) << 4));
}

// ABI row(s) of compact feature f: r1, r2 (r2 < 0 if none); kind 0 = square,
// 1 = off-diagonal pair, 2 = constant / linear, 3 = padding.
struct Rows { int r1, r2, kind; };
__host__ __device__ constexpr Rows abi_rows(int f) {
    const int r = f >> 1, e = f & 1;
    const PairSpec p = pair_spec(r);
    if (p.kind <= 2) {
        int a = 0, b = 0;
        pair_ab(r, e, a, b);
        if (a == b) return {17 + 17 * a, -1, 0};
        return {17 + 16 * a + b, 17 + 16 * b + a, 1};
    }
    if (p.kind == 3) return {1 + 2 * p.j + e, -1, 2};
    if (p.kind == 4 && e == 0) return {0, -1, 2};
    return {-1, -1, 3};
}
static_assert(abi_rows(0).r1 == 17 && abi_rows(152).r1 == 0 && abi_rows(153).kind == 3, "feature order");

// The same for the state layout of d' = kDk (1 + kDk + kDk^2 rows; kDk = 8:
// row 0 constant, 1 + a linear, 9 + 8 a + b quadratic).  At kDk = 8 the
// features that involve dims 8..15 are zero and have no row (padding).
template <int kDk>
__host__ __device__ constexpr Rows abi_rows_t(int f) {
    if (kDk == 16) return abi_rows(f);
    const int r = f >> 1, e = f & 1;
    const PairSpec p = pair_spec(r);
    if (p.kind <= 2) {
        int a = 0, b = 0;
        pair_ab(r, e, a, b);
        if (a >= kDk || b >= kDk) return {-1, -1, 3};
        if (a == b) return {1 + kDk + (kDk + 1) * a, -1, 0};
        return {1 + kDk + kDk * a + b, 1 + kDk + kDk * b + a, 1};
    }
    if (p.kind == 3) {
        const int a = 2 * p.j + e;
        return a < kDk ? Rows{1 + a, -1, 2} : Rows{-1, -1, 3};
    }
    if (p.kind == 4 && e == 0) return {0, -1, 2};
    return {-1, -1, 3};
}
static_assert(abi_rows_t<8>(0).r1 == 9 && abi_rows_t<8>(152).r1 == 0 && abi_rows_t<8>(142).kind == 2 &&
                  abi_rows_t<8>(142).r1 == 7 && abi_rows_t<8>(7).kind == 0 && abi_rows_t<8>(7).r1 == 72 &&
                  abi_rows_t<8>(14).kind == 3 && abi_rows_t<8>(150).kind == 3,
              "d' = 8 rows");

// The conversions between the 273-row ABI state and the compact rows are
// written per feature with the feature index F as a template argument, so the
// kind and the ABI rows of every feature are compile-time constants (no row
// table, no branches, no dummy loads).

// Reads of the ABI column `col` (rows `stride` elements apart) that compact
// feature F needs: its row, and for an off-diagonal pair the mirrored row.
template <int F, int kDk = 16>
__device__ __forceinline__ void abi_reads(const float *col, int64_t stride, float &a, float &b) {
    constexpr Rows e = abi_rows_t<kDk>(F);
    a = b = 0.f;
    if constexpr (e.kind != 3) a = __ldcg(col + e.r1 * stride);
    if constexpr (e.kind == 1) b = __ldcg(col + e.r2 * stride);
}

// Compact entry of feature F: squares carry 1/sqrt2, pairs the symmetric sum
// over (a,b) and (b,a) times 1/sqrt2.
template <int F, int kDk = 16>
__device__ __forceinline__ uint32_t compact_entry(float a, float b) {
    constexpr Rows e = abi_rows_t<kDk>(F);
    if constexpr (e.kind == 3) return 0u;
    else if constexpr (e.kind == 2) return __float_as_uint(a);
    else if constexpr (e.kind == 0) return __float_as_uint(a * kRSqrt2);
    else return __float_as_uint((a + b) * kRSqrt2);
}

// Compact entries of the initial state for the 32 features of group G from
// the ABI column `col` (NULL: zero state).  Every read is issued before any is
// used, so they are in flight together.
template <int G, int kDk = 16, int... J>
__device__ __forceinline__ void compact_initial_group(const float *col, int64_t stride, uint32_t (&r)[32],
                                                      std::integer_sequence<int, J...>) {
    if (!col) {
        ((r[J] = 0u), ...);
        return;
    }
    float a[32], b[32];
    (abi_reads<32 * G + J, kDk>(col, stride, a[J], b[J]), ...);
    ((r[J] = compact_entry<32 * G + J, kDk>(a[J], b[J])), ...);
}

// ABI value(s) of compact feature F with entry x: the rows' values, the
// antisymmetric part anti (of a pair) added to (a,b) and subtracted from (b,a).
// kStage: written into a shared-memory image at stage_d + 4 * 64 * row (value
// column d: rows 256 bytes apart), else to out[row * stride] in global memory.
template <bool kStage, int F, int kDk = 16>
__device__ __forceinline__ void abi_write(float x, float anti, uint32_t stage_d, float *out, int64_t stride) {
    constexpr Rows e = abi_rows_t<kDk>(F);
    if constexpr (e.kind == 3) return;
    float v1, v2 = 0.f;
    if constexpr (e.kind == 2) v1 = x;
    else if constexpr (e.kind == 0) v1 = x * kSqrt2;
    else {
        v1 = x * kRSqrt2 + anti;
        v2 = x * kRSqrt2 - anti;
    }
    if constexpr (kStage) {
        st_shared_f32(stage_d + 256u * (uint32_t)e.r1, v1);
        if constexpr (e.kind == 1) st_shared_f32(stage_d + 256u * (uint32_t)e.r2, v2);
    } else {
        out[e.r1 * stride] = v1;
        if constexpr (e.kind == 1) out[e.r2 * stride] = v2;
    }
}

// One group G of the final ABI state from its compact entries r: the
// antisymmetric part of the initial state's column col0 (NULL: none), scaled
// by anti_scale, is read for the pairs (all reads issued together) and added.
template <bool kStage, int G, int kDk = 16, int... J>
__device__ __forceinline__ void final_group(const uint32_t (&r)[32], const float *col0, int64_t stride,
                                            float anti_scale, uint32_t stage_d, float *out,
                                            std::integer_sequence<int, J...>) {
    float a[32], b[32];
    if (col0) {
        (abi_reads<32 * G + J, kDk>(col0, stride, a[J], b[J]), ...);
    } else {
        ((a[J] = 0.f), ...);
        ((b[J] = 0.f), ...);
    }
    const float h = 0.5f * anti_scale;
    (abi_write<kStage, 32 * G + J, kDk>(__uint_as_float(r[J]), h * (a[J] - b[J]), stage_d, out, stride), ...);
}

// Drain wait used when unwinding: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return;
}

// Final ABI state of feature group G from TMEM rows, for one warp's lanes:
// value rows (column d of each ABI row) and the z' row (lane 64, by lane 0 of
// the warp that owns lanes 64..95).  The value rows go to the shared-memory
// image at `stage` (kStage, a [273][64] fp32 array) or to s_outh; z' goes to
// z_outh.  A NULL destination is skipped.
template <bool kStage, int G, int kDk = 16>
__device__ __forceinline__ void final_group_rows(uint32_t taddr, int d, bool zrow, int lane, const float *s0h,
                                                 uint32_t stage, float *s_outh, const float *z0h, float *z_outh,
                                                 float anti_scale) {
    const auto js = std::make_integer_sequence<int, 32>{};
    uint32_t r[32];
    tmem_load32_sync(taddr + 32 * G, r);
    if (zrow) {
        if (lane == 0 && z_outh) final_group<false, G, kDk>(r, z0h, 1, anti_scale, 0u, z_outh, js);
    } else if (kStage || s_outh) {
        final_group<kStage, G, kDk>(r, s0h ? s0h + d : nullptr, kDV, anti_scale, stage + 4u * (uint32_t)d,
                               s_outh ? s_outh + d : nullptr, js);
    }
    __syncwarp();
}

// Feature groups G0 + I... of the final ABI state (see final_group_rows).  Runs
// once per CTA, so it is kept out of line.
template <bool kStage, int G0, int kDk = 16, int... I>
static __device__ __noinline__ void final_groups(uint32_t taddr, int d, bool zrow, int lane, const float *s0h,
                                                 uint32_t stage, float *s_outh, const float *z0h, float *z_outh,
                                                 float anti_scale, std::integer_sequence<int, I...>) {
    (final_group_rows<kStage, G0 + I, kDk>(taddr, d, zrow, lane, s0h, stage, s_outh, z0h, z_outh, anti_scale),
     ...);
}

// ---- compact state layout in memory (153 rows: 0 constant, 1 + a linear,
// 17 + c(a, b) quadratic for a <= b, c(a, b) = 16 a - a (a - 1) / 2 + (b - a)),
// with the symmetric map of the BASED notes, sec. 2.3: squares carry 1/sqrt2
// on both sides, cross terms none.  The internal entry of a square is then
// the memory entry / sqrt2 (the internal key side carries xbar_a^2 / 2), every
// other internal entry equals its memory entry.  kDCompact (153) is la::kDCompact.

// Row of compact feature f in the 153-row layout, -1 for padding.
__host__ __device__ constexpr int compact_row(int f) {
    const Rows e = abi_rows(f);
    if (e.kind == 3) return -1;
    if (e.kind == 2) return e.r1;  // constant and linear rows coincide with the 273-row layout
    const int x = (e.r1 - 17) / 16, y = (e.r1 - 17) % 16;
    const int a = x < y ? x : y, b = x < y ? y : x;
    return 17 + 16 * a - a * (a - 1) / 2 + (b - a);
}
static_assert(compact_row(0) == 17 && compact_row(152) == 0 && compact_row(153) == -1, "compact rows");

template <int F>
__device__ __forceinline__ float compact_io_read(const float *col, int64_t stride) {
    constexpr int r = compact_row(F);
    if constexpr (r < 0) return 0.f;
    else return __ldcg(col + r * stride);
}

template <int F>
__device__ __forceinline__ uint32_t compact_io_entry(float x) {
    constexpr Rows e = abi_rows(F);
    if constexpr (e.kind == 3) return 0u;
    else if constexpr (e.kind == 0) return __float_as_uint(x * kRSqrt2);
    else return __float_as_uint(x);
}

// Internal entries of the initial state for the 32 features of group G from
// the compact-layout column `col` (NULL: zero state); every read is issued
// before any is used.
template <int G, int... J>
__device__ __forceinline__ void compact_io_initial_group(const float *col, int64_t stride, uint32_t (&r)[32],
                                                         std::integer_sequence<int, J...>) {
    if (!col) {
        ((r[J] = 0u), ...);
        return;
    }
    float a[32];
    ((a[J] = compact_io_read<32 * G + J>(col, stride)), ...);
    ((r[J] = compact_io_entry<32 * G + J>(a[J])), ...);
}

// Memory entry of compact feature F from its internal entry x: written into
// the shared-memory image at stage_d + 256 * row (kStage) or to out[row * stride].
template <bool kStage, int F>
__device__ __forceinline__ void compact_io_write(float x, uint32_t stage_d, float *out, int64_t stride) {
    constexpr Rows e = abi_rows(F);
    constexpr int r = compact_row(F);
    if constexpr (r < 0) return;
    else {
        const float v = e.kind == 0 ? x * kSqrt2 : x;
        if constexpr (kStage) st_shared_f32(stage_d + 256u * (uint32_t)r, v);
        else out[r * stride] = v;
    }
}

// Final compact-layout state of feature group G from TMEM rows (the
// counterpart of final_group_rows; there is no antisymmetric part to add).
template <bool kStage, int G, int... J>
__device__ __forceinline__ void final_group_rows_compact(uint32_t taddr, int d, bool zrow, int lane,
                                                         uint32_t stage, float *s_outh, float *z_outh,
                                                         std::integer_sequence<int, J...>) {
    uint32_t r[32];
    tmem_load32_sync(taddr + 32 * G, r);
    if (zrow) {
        if (lane == 0 && z_outh) (compact_io_write<false, 32 * G + J>(__uint_as_float(r[J]), 0u, z_outh, 1), ...);
    } else if (kStage || s_outh) {
        (compact_io_write<kStage, 32 * G + J>(__uint_as_float(r[J]), stage + 4u * (uint32_t)d,
                                              s_outh ? s_outh + d : nullptr, kDV), ...);
    }
    __syncwarp();
}

template <bool kStage, int G0, int... I>
static __device__ __noinline__ void final_groups_compact(uint32_t taddr, int d, bool zrow, int lane,
                                                         uint32_t stage, float *s_outh, float *z_outh,
                                                         std::integer_sequence<int, I...>) {
    (final_group_rows_compact<kStage, G0 + I>(taddr, d, zrow, lane, stage, s_outh, z_outh,
                                              std::make_integer_sequence<int, 32>{}), ...);
}

}  // namespace taylor
}  // namespace la
