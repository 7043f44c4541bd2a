// Chunked prefill for d' = 24 and 32 (bf16 activations) with its dense
// contractions on the tensor cores, through cuBLASLt batched GEMMs.
//
// Method: BASED reading notes ("Simple linear attention language models
// balance the recall-throughput tradeoff"), sec. 2.5, blockwise form over
// 128-token chunks c:
//   num_c = (M o P_c) [V_c | 1] + Phi_Qc S_<c,   S_<c+1 = S_<c + Phi_Kc^T [V_c | 1]
// with the second-order Taylor map of sec. 2.3 for a general d' (the page's
// feature-dimension ablations), started from the caller's state
// ("Understanding and Improving Length Generalization in Recurrent Models"
// reading notes, sec. 2.5 Eq. (4)).
//
// The feature map is the symmetric compact one, phi_c(x) = [1, xbar_a,
// xbar_a^2 / sqrt(2), xbar_a xbar_b (a < b)], xbar = x / d'^(1/4): 325 (d' = 24)
// or 561 (d' = 32) features instead of 601 or 1057, with phi_c(q).phi_c(k) =
// 1 + q.k / sqrt(d') + (q.k)^2 / (2 d') exactly.  The state is held in that
// form (pairs folded: s_c[ab] = (s[ab] + s[ba]) / sqrt(2)); the antisymmetric
// part of the caller's s0, which no output can see, passes through to s_out.
//
// Steps (one stream, every buffer in the caller's workspace):
//   1. feat_kernel: Phi_Q, Phi_K (bf16, padded to a multiple of 8 features)
//      and [v | 1 | 0] (80 columns) for every token, zero past N;
//   2. GEMM: dS_c = Phi_Kc^T [V_c | 1], fp32, all chunks of all heads at once;
//   3. scan_kernel: S_<c (bf16 copies, the read-out operand) by a running sum
//      over the chunks from the folded s0, and the final state unfolded into
//      the ABI rows;
//   4. GEMM: num_c = Phi_Qc S_<c (fp32);
//   5. intra_p_kernel: P_c = 1 + T/sqrt(d') + T^2/(2 d') for key <= query,
//      T = Q_c K_c^T in fp32 (bf16 out);
//   6. GEMM: num_c += P_c [V_c | 1];
//   7. y_kernel: y = num[:, :64] / (num[:, 64] + eps).
// The GEMMs (bf16 operands, fp32 accumulation) are plain library GEMMs; the
// feature map, the scan with the state conversion, the masked kernel matrix
// and the normalisation are this file's kernels.
#include <cublasLt.h>

#include <mutex>

#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kCG = 128;   // tokens per chunk
constexpr int kNV = 80;    // [v | 1 | 0]: 64 values, the ones column (z), 15 zero columns
constexpr size_t kLtWorkspace = size_t(32) << 20;

template <int DK>
struct GDims {
    static constexpr int kDc = 1 + DK + DK * (DK + 1) / 2;  // compact features
    static constexpr int kDp = (kDc + 7) / 8 * 8;           // padded: rows of 16-byte multiples
    static constexpr int kD = 1 + DK + DK * DK;             // ABI rows
};

// Compact feature f as a product xe[ia] * xe[ib] * scale over xe = [1, xbar]:
// the constant (0, 0, 1), linear a (1 + a, 0, 1), square (1 + a, 1 + a,
// 1/sqrt(2)), pair a < b (1 + a, 1 + b, 1), in the order constant, linear
// a = 0..d'-1, then a = 0..d'-1, b = a..d'-1; padding features have scale 0.
// code = ia | ib << 8 | kind << 16 (kind 0: scale 0, 1: scale 1, 2: 1/sqrt(2)).
template <int DK>
struct FeatTable {
    uint32_t code[GDims<DK>::kDp];
    constexpr FeatTable() : code() {
        int f = 0;
        code[f++] = 0u | (0u << 8) | (1u << 16);
        for (int a = 0; a < DK; ++a) code[f++] = (uint32_t)(1 + a) | (0u << 8) | (1u << 16);
        for (int a = 0; a < DK; ++a)
            for (int b = a; b < DK; ++b)
                code[f++] = (uint32_t)(1 + a) | ((uint32_t)(1 + b) << 8) | ((a == b ? 2u : 1u) << 16);
        while (f < GDims<DK>::kDp) code[f++] = 0u;
    }
};
__device__ const FeatTable<24> kFeat24{};
__device__ const FeatTable<32> kFeat32{};

template <int DK>
__device__ __forceinline__ uint32_t feat_code(int f) {
    if constexpr (DK == 24) return __ldg(&kFeat24.code[f]);
    else return __ldg(&kFeat32.code[f]);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 h) { return __bfloat162float(h); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// 1. A CTA per 32 tokens (of Np = chunks * 128 per head): the query and key
// features (each thread 8 consecutive features of one token, one 16-byte
// store per side: a warp's stores cover consecutive 16-byte pieces of a
// token's rows) and [v | 1 | 0], all zero for t >= N.
constexpr int kFT = 32;  // tokens per CTA
template <int DK>
__global__ void __launch_bounds__(256) feat_kernel(const __nv_bfloat16 *__restrict__ q,
                                                   const __nv_bfloat16 *__restrict__ k,
                                                   const __nv_bfloat16 *__restrict__ v, uint4 *__restrict__ phq,
                                                   uint4 *__restrict__ phk, uint4 *__restrict__ ve,
                                                   int64_t N, int64_t Np, float xscale) {
    constexpr int Dp = GDims<DK>::kDp, G = Dp / 8, XE = DK + 1;
    __shared__ float xq[kFT][XE], xk[kFT][XE];
    __shared__ __align__(16) uint32_t code[Dp];
    const int tid = threadIdx.x;
    // the CTA's 32 tokens lie in one head (Np is a multiple of 128)
    const int64_t tok0 = (int64_t)blockIdx.x * kFT;  // first token (bh * Np + t)
    const int64_t bh = tok0 / Np, t0 = tok0 % Np;
    for (int f = tid; f < Dp; f += blockDim.x) code[f] = feat_code<DK>(f);
    for (int e = tid; e < kFT * XE; e += blockDim.x) {
        const int r = e / XE, c = e % XE;
        const int64_t t = t0 + r;
        float xqv = 0.f, xkv = 0.f;
        if (c == 0) {
            xqv = xkv = 1.f;
        } else if (t < N) {
            xqv = xscale * bf2f(q[(bh * N + t) * DK + c - 1]);
            xkv = xscale * bf2f(k[(bh * N + t) * DK + c - 1]);
        }
        xq[r][c] = xqv;
        xk[r][c] = xkv;
    }
    __syncthreads();
    for (int it = tid; it < kFT * G; it += blockDim.x) {
        const int r = it / G, g = it % G;
        const int64_t tok = tok0 + r;
        const bool in = t0 + r < N;
        const uint4 c0 = *reinterpret_cast<const uint4 *>(&code[8 * g]);
        const uint4 c1 = *reinterpret_cast<const uint4 *>(&code[8 * g + 4]);
        const uint32_t cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t wq[4], wk[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float oq[2], ok[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t c = cs[2 * h + e];
                const int ia = c & 0xFF, ib = (c >> 8) & 0xFF, kind = c >> 16;
                const float sc = kind == 0 ? 0.f : (kind == 1 ? 1.f : kInvSqrt2);
                oq[e] = xq[r][ia] * xq[r][ib] * sc;
                ok[e] = xk[r][ia] * xk[r][ib] * sc;
            }
            wq[h] = in ? pack2(oq[0], oq[1]) : 0u;
            wk[h] = in ? pack2(ok[0], ok[1]) : 0u;
        }
        phq[tok * G + g] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        phk[tok * G + g] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
    }
    for (int it = tid; it < kFT * (kNV / 8); it += blockDim.x) {
        const int r = it / (kNV / 8), g = it % (kNV / 8);
        const int64_t tok = tok0 + r, t = t0 + r;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (t < N) {
            if (g < kDV / 8) w = reinterpret_cast<const uint4 *>(v + (bh * N + t) * kDV)[g];
            else if (g == kDV / 8) w.x = pack2(1.f, 0.f);  // the ones column (z)
        }
        ve[tok * (kNV / 8) + g] = w;
    }
}

// 3. One thread per (bh, compact feature f, column col of [v | 1 | 0]): the
// state before each chunk (bf16, the read-out operand), from s0 folded into
// the compact form, then the final state unfolded into the ABI rows (value
// columns into s_out, the ones column into z_out).
template <int DK>
__global__ void __launch_bounds__(256) scan_kernel(const float *__restrict__ dS, __nv_bfloat16 *__restrict__ Sb,
                                                   const float *__restrict__ s0, const float *__restrict__ z0,
                                                   float *__restrict__ s_out, float *__restrict__ z_out,
                                                   int64_t BH, int nch) {
    constexpr int Dc = GDims<DK>::kDc, Dp = GDims<DK>::kDp, D = GDims<DK>::kD;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= BH * Dp * kNV) return;
    const int col = (int)(idx % kNV);
    const int f = (int)((idx / kNV) % Dp);
    const int64_t bh = idx / ((int64_t)kNV * Dp);
    const bool live = f < Dc && col <= kDV;  // value columns and the z column
    // ABI rows of feature f: r1 (and r2 for a pair a < b: rows ab and ba)
    int r1 = 0, r2 = -1;
    if (f < Dc) {
        const uint32_t c = feat_code<DK>(f);
        const int ia = c & 0xFF, ib = (c >> 8) & 0xFF;  // indices into [1, xbar]
        if (ia == 0) r1 = 0;                            // the constant
        else if (ib == 0) r1 = ia;                      // linear: row 1 + a
        else {
            const int a = ia - 1, b = ib - 1;
            r1 = 1 + DK + a * DK + b;
            if (a != b) r2 = 1 + DK + b * DK + a;
        }
    }
    auto in_abi = [&](int r) -> float {
        if (col < kDV) return s0 ? s0[(bh * D + r) * kDV + col] : 0.f;
        return z0 ? z0[bh * D + r] : 0.f;
    };
    float S = 0.f, anti = 0.f;
    if (live) {
        if (r2 < 0) {
            S = in_abi(r1);
        } else {
            const float x1 = in_abi(r1), x2 = in_abi(r2);
            S = (x1 + x2) * kInvSqrt2;
            anti = 0.5f * (x1 - x2);
        }
    }
    const int64_t blk = (int64_t)Dp * kNV;
    const float *d = dS + bh * nch * blk + (int64_t)f * kNV + col;
    __nv_bfloat16 *o = Sb + bh * nch * blk + (int64_t)f * kNV + col;
    for (int c = 0; c < nch; ++c) {
        o[c * blk] = __float2bfloat16_rn(S);
        S += d[c * blk];  // zero outside the live entries (zero features / columns)
    }
    if (!live) return;
    auto out_abi = [&](int r, float x) {
        if (col < kDV) {
            if (s_out) s_out[(bh * D + r) * kDV + col] = x;
        } else if (z_out) {
            z_out[bh * D + r] = x;
        }
    };
    if (r2 < 0) {
        out_abi(r1, S);
    } else {
        out_abi(r1, S * kInvSqrt2 + anti);
        out_abi(r2, S * kInvSqrt2 - anti);
    }
}

// 5. One CTA per (bh, chunk): P[i][j] = 1 + T/sqrt(d') + T^2/(2 d') for
// j <= i, else 0, T = q_i . k_j in fp32 from the bf16 inputs (rows past N read
// as zero: their P entries meet zero rows of [v | 1]).  Thread t: an 8 x 8
// tile of (i, j), queries 8 (t / 16), keys 8 (t % 16), from d'-major copies
// of Q and K in shared memory (two 16-byte reads feed 64 FMAs).
template <int DK>
__global__ void __launch_bounds__(256) intra_p_kernel(const __nv_bfloat16 *__restrict__ q,
                                                      const __nv_bfloat16 *__restrict__ k,
                                                      uint4 *__restrict__ P, int64_t N, int nch) {
    __shared__ __align__(16) float qs[DK][kCG];
    __shared__ __align__(16) float ks[DK][kCG];
    const int64_t bc = blockIdx.x;
    const int64_t bh = bc / nch;
    const int c = (int)(bc % nch);
    const int tid = threadIdx.x;
    // thread: 8 dims of one token (16 bytes); a warp's smem writes go to 32
    // consecutive tokens of a row, conflict-free
    for (int e = tid; e < kCG * (DK / 8); e += blockDim.x) {
        const int t = e % kCG, d8 = e / kCG;
        const int64_t tok = (int64_t)c * kCG + t;
        uint4 wq = make_uint4(0u, 0u, 0u, 0u), wk = wq;
        if (tok < N) {
            wq = reinterpret_cast<const uint4 *>(q + (bh * N + tok) * DK)[d8];
            wk = reinterpret_cast<const uint4 *>(k + (bh * N + tok) * DK)[d8];
        }
        const uint32_t aq[4] = {wq.x, wq.y, wq.z, wq.w}, ak[4] = {wk.x, wk.y, wk.z, wk.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            qs[8 * d8 + 2 * h][t] = __uint_as_float(aq[h] << 16);
            qs[8 * d8 + 2 * h + 1][t] = __uint_as_float(aq[h] & 0xFFFF0000u);
            ks[8 * d8 + 2 * h][t] = __uint_as_float(ak[h] << 16);
            ks[8 * d8 + 2 * h + 1][t] = __uint_as_float(ak[h] & 0xFFFF0000u);
        }
    }
    __syncthreads();
    const int i0 = 8 * (tid >> 4), j0 = 8 * (tid & 15);
    float T[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) T[a][b] = 0.f;
#pragma unroll 4
    for (int dd = 0; dd < DK; ++dd) {
        const float4 qa = *reinterpret_cast<const float4 *>(&qs[dd][i0]);
        const float4 qb = *reinterpret_cast<const float4 *>(&qs[dd][i0 + 4]);
        const float4 ka = *reinterpret_cast<const float4 *>(&ks[dd][j0]);
        const float4 kb = *reinterpret_cast<const float4 *>(&ks[dd][j0 + 4]);
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const float kv[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int b = 0; b < 8; ++b) T[a][b] = fmaf(qv[a], kv[b], T[a][b]);
    }
    const float c1 = rsqrtf((float)DK), c2 = 0.5f / (float)DK;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int i = i0 + a;
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int j = j0 + 2 * h;
            const float p0 = j <= i ? fmaf(T[a][2 * h], fmaf(T[a][2 * h], c2, c1), 1.f) : 0.f;
            const float p1 = j + 1 <= i ? fmaf(T[a][2 * h + 1], fmaf(T[a][2 * h + 1], c2, c1), 1.f) : 0.f;
            w[h] = pack2(p0, p1);
        }
        P[(bc * kCG + i) * (kCG / 8) + j0 / 8] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 7. y = num[:, :64] / (num[:, 64] + eps) for t < N, 8 values per thread.
__global__ void __launch_bounds__(256) y_kernel(const float *__restrict__ num, __nv_bfloat16 *__restrict__ y,
                                                int64_t BH, int64_t N, int64_t Np, float eps) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= BH * N * (kDV / 8)) return;
    const int g = (int)(idx % (kDV / 8));
    const int64_t tok = idx / (kDV / 8);
    const int64_t bh = tok / N, t = tok % N;
    const float *r = num + (bh * Np + t) * kNV;
    const float inv = 1.0f / (r[kDV] + eps);
    const float4 a = *reinterpret_cast<const float4 *>(r + 8 * g);
    const float4 b = *reinterpret_cast<const float4 *>(r + 8 * g + 4);
    reinterpret_cast<uint4 *>(y + tok * kDV)[g] =
        make_uint4(pack2(a.x * inv, a.y * inv), pack2(a.z * inv, a.w * inv), pack2(b.x * inv, b.y * inv),
                   pack2(b.z * inv, b.w * inv));
}

// ---------------------------------------------------------------- host side
struct GLayout {
    size_t phq, phk, ve, ds, sb, num, p, lt, total;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

GLayout g_layout(int64_t BH, int64_t N, int dk) {
    const int Dp = dk == 24 ? GDims<24>::kDp : GDims<32>::kDp;
    const int64_t nch = (N + kCG - 1) / kCG, Np = nch * kCG;
    GLayout L{};
    size_t off = 0;
    L.phq = off; off = al256(off + 2 * (size_t)BH * Np * Dp);
    L.phk = off; off = al256(off + 2 * (size_t)BH * Np * Dp);
    L.ve = off;  off = al256(off + 2 * (size_t)BH * Np * kNV);
    L.ds = off;  off = al256(off + 4 * (size_t)BH * nch * Dp * kNV);
    L.sb = off;  off = al256(off + 2 * (size_t)BH * nch * Dp * kNV);
    L.num = off; off = al256(off + 4 * (size_t)BH * Np * kNV);
    L.p = off;   off = al256(off + 2 * (size_t)BH * nch * kCG * kCG);
    L.lt = off;  off += kLtWorkspace;
    L.total = off;
    return L;
}

constexpr int kMaxDevLt = 64;
std::mutex g_lt_mu;
cublasLtHandle_t g_lt[kMaxDevLt] = {};

cublasLtHandle_t lt_handle() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevLt) return nullptr;
    std::lock_guard<std::mutex> lock(g_lt_mu);
    if (!g_lt[dev] && cublasLtCreate(&g_lt[dev]) != CUBLAS_STATUS_SUCCESS) g_lt[dev] = nullptr;
    return g_lt[dev];
}

// D (m x n, column-major, ld m, fp32) = A (m x k, column-major, ld m, bf16) *
// op(B) (+ beta D), B bf16 column-major: k x n (ld k) or, transposed, n x k
// (ld n); `batch` problems at the given element strides.
cudaError_t gemm(cublasLtHandle_t h, int m, int n, int k, const void *A, int64_t sA, const void *B, bool transb,
                 int64_t sB, float *D, int64_t sD, int batch, float beta, void *ws, cudaStream_t st) {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    bool ok = cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS;
    const cublasOperation_t tn = CUBLAS_OP_N, tb = transb ? CUBLAS_OP_T : CUBLAS_OP_N;
    ok = ok && cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &tn, sizeof(tn)) == CUBLAS_STATUS_SUCCESS;
    ok = ok && cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) == CUBLAS_STATUS_SUCCESS;
    ok = ok && cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, m, k, m) == CUBLAS_STATUS_SUCCESS;
    ok = ok && cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, transb ? n : k, transb ? k : n, transb ? n : k) ==
                   CUBLAS_STATUS_SUCCESS;
    ok = ok && cublasLtMatrixLayoutCreate(&ld, CUDA_R_32F, m, n, m) == CUBLAS_STATUS_SUCCESS;
    const cublasLtMatrixLayout_t lays[3] = {la, lb, ld};
    const int64_t strides[3] = {sA, sB, sD};
    for (int i = 0; ok && i < 3; ++i) {
        ok = cublasLtMatrixLayoutSetAttribute(lays[i], CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &batch, sizeof(batch)) ==
                 CUBLAS_STATUS_SUCCESS &&
             cublasLtMatrixLayoutSetAttribute(lays[i], CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &strides[i],
                                              sizeof(strides[i])) == CUBLAS_STATUS_SUCCESS;
    }
    ok = ok && cublasLtMatmulPreferenceCreate(&pref) == CUBLAS_STATUS_SUCCESS;
    const size_t wsb = kLtWorkspace;
    ok = ok && cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb,
                                                    sizeof(wsb)) == CUBLAS_STATUS_SUCCESS;
    cublasLtMatmulHeuristicResult_t res{};
    int found = 0;
    ok = ok && cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, ld, ld, pref, 1, &res, &found) ==
                   CUBLAS_STATUS_SUCCESS && found > 0;
    const float alpha = 1.f;
    ok = ok && cublasLtMatmul(h, op, &alpha, A, la, B, lb, &beta, D, ld, D, ld, &res.algo, ws, wsb, st) ==
                   CUBLAS_STATUS_SUCCESS;
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (ld) cublasLtMatrixLayoutDestroy(ld);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return ok ? cudaSuccess : cudaErrorUnknown;
}

template <int DK>
cudaError_t run_general_tc(const PrefillArgs &a, char *ws, cudaStream_t st) {
    constexpr int Dp = GDims<DK>::kDp;
    const int64_t BH = a.B * a.H, N = a.N;
    const int nch = (int)((N + kCG - 1) / kCG);
    const int64_t Np = (int64_t)nch * kCG;
    const GLayout L = g_layout(BH, N, DK);
    cublasLtHandle_t h = lt_handle();
    if (!h) return cudaErrorUnknown;
    auto *phq = reinterpret_cast<__nv_bfloat16 *>(ws + L.phq);
    auto *phk = reinterpret_cast<__nv_bfloat16 *>(ws + L.phk);
    auto *ve = reinterpret_cast<__nv_bfloat16 *>(ws + L.ve);
    auto *dS = reinterpret_cast<float *>(ws + L.ds);
    auto *Sb = reinterpret_cast<__nv_bfloat16 *>(ws + L.sb);
    auto *num = reinterpret_cast<float *>(ws + L.num);
    auto *P = reinterpret_cast<__nv_bfloat16 *>(ws + L.p);
    void *ltws = ws + L.lt;
    const auto *q = static_cast<const __nv_bfloat16 *>(a.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(a.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(a.v);
    const float xscale = 1.0f / sqrtf(sqrtf((float)DK));
    const int batch = (int)(BH * nch);

    feat_kernel<DK><<<(unsigned)(BH * Np / kFT), 256, 0, st>>>(
        q, k, v, reinterpret_cast<uint4 *>(phq), reinterpret_cast<uint4 *>(phk), reinterpret_cast<uint4 *>(ve), N,
        Np, xscale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. dS_c (Dp x 80, row-major) = Phi_Kc^T [V_c | 1]: column-major 80 x Dp = [V_c | 1]^T Phi_Kc
    if ((e = gemm(h, kNV, Dp, kCG, ve, (int64_t)kCG * kNV, phk, true, (int64_t)kCG * Dp, dS, (int64_t)Dp * kNV,
                  batch, 0.f, ltws, st)) != cudaSuccess)
        return e;
    const int64_t nscan = BH * Dp * kNV;
    scan_kernel<DK><<<(unsigned)((nscan + 255) / 256), 256, 0, st>>>(dS, Sb, a.s0, a.z0, a.s_out, a.z_out, BH, nch);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. num_c (128 x 80, row-major) = Phi_Qc S_<c: column-major 80 x 128 = S_<c^T Phi_Qc^T
    if ((e = gemm(h, kNV, kCG, Dp, Sb, (int64_t)Dp * kNV, phq, false, (int64_t)kCG * Dp, num, (int64_t)kCG * kNV,
                  batch, 0.f, ltws, st)) != cudaSuccess)
        return e;
    intra_p_kernel<DK><<<(unsigned)batch, 256, 0, st>>>(q, k, reinterpret_cast<uint4 *>(P), N, nch);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 6. num_c += P_c [V_c | 1]: column-major 80 x 128 += [V_c | 1]^T P_c^T
    if ((e = gemm(h, kNV, kCG, kCG, ve, (int64_t)kCG * kNV, P, false, (int64_t)kCG * kCG, num, (int64_t)kCG * kNV,
                  batch, 1.f, ltws, st)) != cudaSuccess)
        return e;
    const int64_t ny = BH * N * (kDV / 8);
    y_kernel<<<(unsigned)((ny + 255) / 256), 256, 0, st>>>(num, static_cast<__nv_bfloat16 *>(a.y), BH, N, Np, a.eps);
    return cudaGetLastError();
}

}  // namespace

size_t general_tc_workspace(int64_t BH, int64_t N, int dk) {
    if ((dk != 24 && dk != 32) || N <= 0 || BH <= 0) return 0;
    // every grid and the GEMMs' batch count fit 32 bits while B*H*Np <= 2^31
    const int64_t Np = (N + kCG - 1) / kCG * kCG;
    if (BH > (int64_t(1) << 31) / Np) return 0;
    return g_layout(BH, N, dk).total;
}

cudaError_t launch_prefill_general_tc(const PrefillArgs &a, int dk, void *workspace, cudaStream_t st) {
    char *ws = static_cast<char *>(workspace);
    return dk == 24 ? run_general_tc<24>(a, ws, st) : run_general_tc<32>(a, ws, st);
}

}  // namespace la
