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

// Feature vector of one token into its row of the feature tile; with kScaled
// every feature is multiplied by scale2 (a bf16x2 pair of the same scale).
template <bool kKey, bool kScaled = false, int... J>
__device__ __forceinline__ void emit_features(const uint4 &lo, const uint4 &hi, uint32_t base, int t,
                                              bool zero, std::integer_sequence<int, J...>,
                                              uint32_t scale2 = 0x3F803F80u) {
    // xbar = x / 2 (exact), its odd-shifted pairs, and halves for the key squares
    const uint32_t raw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t X[8], Y[7], H[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) X[j] = hmul2(raw[j], 0x3F003F00u);
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

// Raw token row t (16 bf16 as two 16-byte halves) of a [128][16] SW32 tile.
__device__ __forceinline__ void load_row16_raw(uint32_t tile, int t, uint4 &lo, uint4 &hi) {
    const uint32_t sw = (uint32_t)((t >> 2) & 1);
    lo = ld_shared_v4(tile + t * 32 + ((0u ^ sw) << 4));
    hi = ld_shared_v4(tile + t * 32 + ((1u ^ sw) << 4));
}

// ABI row(s) of compact feature f: r1, r2 (r2 < 0 if none); kind 0 = square,
// 1 = off-diagonal pair, 2 = constant / linear, 3 = padding.
struct Rows { int r1, r2, kind; };
__device__ __forceinline__ Rows abi_rows(int f) {
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

// Compact entries of the initial state for the 32 features of one row group
// (rows table entries e[0..31]): squares carry 1/sqrt2, pairs the symmetric
// sum over (a,b) and (b,a) times 1/sqrt2.  The loads are unconditional
// (padding reads row 0, unpaired features read their row twice) and all issued
// before any is used, so each half's 32 reads are in flight together instead of
// paying one DRAM latency each.
__device__ __forceinline__ void compact_initial_group(const float *col, int stride, const int4 *e,
                                                      uint32_t (&r)[32]) {
    if (!col) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = 0u;
        return;
    }
#pragma unroll
    for (int h = 0; h < 32; h += 16) {  // two halves of 16 features: fewer live registers
        float a[16], b[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int4 t = e[h + j];
            const int r1 = t.z == 3 ? 0 : t.x;
            const int r2 = t.z == 1 ? t.y : r1;
            a[j] = __ldg(col + (int64_t)r1 * stride);
            b[j] = __ldg(col + (int64_t)r2 * stride);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int k = e[h + j].z;
            const float x = k == 3 ? 0.f : k == 2 ? a[j] : k == 0 ? a[j] * kRSqrt2 : (a[j] + b[j]) * kRSqrt2;
            r[h + j] = __float_as_uint(x);
        }
    }
}

// Drain wait used when unwinding: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return;
}

// Final ABI state from TMEM rows, for one warp's lanes and feature groups
// [g0, g0 + ng): value rows d < 64 (column d of each ABI row), and the z' row
// (lane 64, by lane 0 of the warp that owns lanes 64..95).  Each group's reads
// of the initial state are issued together before its stores.  Runs once per
// CTA, so it is kept out of line.
static __device__ __noinline__ void store_final_groups(uint32_t taddr, int g0, int ng, int d, bool zrow, int lane,
                                                       const int4 *rows_tab, const float *s0h, float *s_outh,
                                                       const float *z0h, float *z_outh, float anti_scale) {
    const float *col0 = zrow ? z0h : (s0h ? s0h + d : nullptr);
    float *out = zrow ? z_outh : (s_outh ? s_outh + d : nullptr);
    const int64_t stride = zrow ? 1 : kDV;
    for (int g = g0; g < g0 + ng; ++g) {
        uint32_t r[32];
        tmem_load32_sync(taddr + 32 * g, r);
        if (out && (!zrow || lane == 0)) {
            // antisymmetric part of the initial state for the pairs: unconditional
            // loads (other features read row 0 and discard it) so all are in flight at once
            float anti[32];
            if (col0) {
                float a[32], b[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int4 e = rows_tab[32 * g + j];
                    const int r1 = e.z == 1 ? e.x : 0, r2 = e.z == 1 ? e.y : 0;
                    a[j] = __ldg(col0 + r1 * stride);
                    b[j] = __ldg(col0 + r2 * stride);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    anti[j] = rows_tab[32 * g + j].z == 1 ? (0.5f * anti_scale) * (a[j] - b[j]) : 0.f;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) anti[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int4 e = rows_tab[32 * g + j];
                const float x = __uint_as_float(r[j]);
                if (e.z == 2) {
                    out[e.x * stride] = x;
                } else if (e.z == 0) {
                    out[e.x * stride] = x * kSqrt2;
                } else if (e.z == 1) {
                    const float sym = x * kRSqrt2;
                    out[e.x * stride] = sym + anti[j];
                    out[e.y * stride] = sym - anti[j];
                }
            }
        }
        __syncwarp();
    }
}

}  // namespace taylor
}  // namespace la
