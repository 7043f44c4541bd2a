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

// Compact feature f: 0xFFFF the constant, a | 0xFF00 the linear feature a,
// a | b << 8 the product of a <= b (in the order a = 0..d'-1, b = a..d'-1).
template <int DK>
struct FeatTable {
    uint16_t code[GDims<DK>::kDc];
    constexpr FeatTable() : code() {
        int f = 0;
        code[f++] = 0xFFFF;
        for (int a = 0; a < DK; ++a) code[f++] = (uint16_t)(a | 0xFF00);
        for (int a = 0; a < DK; ++a)
            for (int b = a; b < DK; ++b) code[f++] = (uint16_t)(a | (b << 8));
    }
};
__device__ const FeatTable<24> kFeat24{};
__device__ const FeatTable<32> kFeat32{};

template <int DK>
__device__ __forceinline__ uint16_t feat_code(int f) {
    if constexpr (DK == 24) return __ldg(&kFeat24.code[f]);
    else return __ldg(&kFeat32.code[f]);
}

template <int DK>
__device__ __forceinline__ float feat_value(const float *x, int f) {
    if (f >= GDims<DK>::kDc) return 0.f;
    const uint16_t c = feat_code<DK>(f);
    if (c == 0xFFFF) return 1.f;
    const int a = c & 0xFF, b = c >> 8;
    if (b == 0xFF) return x[a];
    return a == b ? x[a] * x[a] * kInvSqrt2 : x[a] * x[b];
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 h) { return __bfloat162float(h); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// 1. One warp per token (bh, t), t < Np = chunks * 128: the query and key
// features and [v | 1 | 0], all zero for t >= N.
template <int DK>
__global__ void __launch_bounds__(256) feat_kernel(const __nv_bfloat16 *__restrict__ q,
                                                   const __nv_bfloat16 *__restrict__ k,
                                                   const __nv_bfloat16 *__restrict__ v, uint32_t *__restrict__ phq,
                                                   uint32_t *__restrict__ phk, uint32_t *__restrict__ ve,
                                                   int64_t BH, int64_t N, int64_t Np, float xscale) {
    constexpr int Dp = GDims<DK>::kDp;
    __shared__ float xs[8][2][DK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)blockIdx.x * 8 + warp;
    if (tok >= BH * Np) return;
    const int64_t bh = tok / Np, t = tok % Np;
    const bool in = t < N;
    if (lane < DK) {
        xs[warp][0][lane] = in ? xscale * bf2f(q[(bh * N + t) * DK + lane]) : 0.f;
        xs[warp][1][lane] = in ? xscale * bf2f(k[(bh * N + t) * DK + lane]) : 0.f;
    }
    __syncwarp();
    uint32_t *oq = phq + tok * (Dp / 2), *ok = phk + tok * (Dp / 2);
    for (int j = lane; j < Dp / 2; j += 32) {
        const int f = 2 * j;
        oq[j] = in ? pack2(feat_value<DK>(xs[warp][0], f), feat_value<DK>(xs[warp][0], f + 1)) : 0u;
        ok[j] = in ? pack2(feat_value<DK>(xs[warp][1], f), feat_value<DK>(xs[warp][1], f + 1)) : 0u;
    }
    uint32_t *ov = ve + tok * (kNV / 2);
    for (int j = lane; j < kNV / 2; j += 32) {
        uint32_t w = 0u;
        if (in && 2 * j < kDV) w = *reinterpret_cast<const uint32_t *>(v + (bh * N + t) * kDV + 2 * j);
        else if (in && 2 * j == kDV) w = pack2(1.f, 0.f);  // the ones column (z) and a zero
        ov[j] = w;
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
        const uint16_t c = feat_code<DK>(f);
        const int a = c & 0xFF, b = c >> 8;
        if (c == 0xFFFF) r1 = 0;
        else if (b == 0xFF) r1 = 1 + a;
        else {
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
// as zero: their P entries meet zero rows of [v | 1]).  Thread t: query row
// t / 2, keys 64 (t % 2) .. + 63, written as 8 x 16 bytes.
template <int DK>
__global__ void __launch_bounds__(256) intra_p_kernel(const __nv_bfloat16 *__restrict__ q,
                                                      const __nv_bfloat16 *__restrict__ k,
                                                      uint4 *__restrict__ P, int64_t N, int nch) {
    __shared__ float ks[kCG][DK + 1];
    __shared__ float qs[kCG][DK + 1];
    const int64_t bc = blockIdx.x;
    const int64_t bh = bc / nch;
    const int c = (int)(bc % nch);
    const int tid = threadIdx.x;
    for (int e = tid; e < kCG * DK; e += blockDim.x) {
        const int t = e / DK, dd = e % DK;
        const int64_t tok = (int64_t)c * kCG + t;
        const bool in = tok < N;
        qs[t][dd] = in ? bf2f(q[(bh * N + tok) * DK + dd]) : 0.f;
        ks[t][dd] = in ? bf2f(k[(bh * N + tok) * DK + dd]) : 0.f;
    }
    __syncthreads();
    const int i = tid >> 1, j0 = (tid & 1) * 64;
    float qr[DK];
#pragma unroll
    for (int dd = 0; dd < DK; ++dd) qr[dd] = qs[i][dd];
    const float c1 = rsqrtf((float)DK), c2 = 0.5f / (float)DK;
    uint4 *row = P + (bc * kCG + i) * (kCG / 8) + j0 / 8;
#pragma unroll 1
    for (int g = 0; g < 8; ++g) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float p2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = j0 + 8 * g + 2 * h + e;
                float T = 0.f;
#pragma unroll
                for (int dd = 0; dd < DK; ++dd) T = fmaf(qr[dd], ks[j][dd], T);
                p2[e] = j <= i ? fmaf(T, fmaf(T, c2, c1), 1.f) : 0.f;
            }
            w[h] = pack2(p2[0], p2[1]);
        }
        row[g] = make_uint4(w[0], w[1], w[2], w[3]);
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

    feat_kernel<DK><<<(unsigned)((BH * Np + 7) / 8), 256, 0, st>>>(
        q, k, v, reinterpret_cast<uint32_t *>(phq), reinterpret_cast<uint32_t *>(phk),
        reinterpret_cast<uint32_t *>(ve), BH, N, Np, xscale);
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
    if ((dk != 24 && dk != 32) || N <= 0) return 0;
    return g_layout(BH, N, dk).total;
}

cudaError_t launch_prefill_general_tc(const PrefillArgs &a, int dk, void *workspace, cudaStream_t st) {
    char *ws = static_cast<char *>(workspace);
    return dk == 24 ? run_general_tc<24>(a, ws, st) : run_general_tc<32>(a, ws, st);
}

}  // namespace la
