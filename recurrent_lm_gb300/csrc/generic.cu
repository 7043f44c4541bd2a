// CUDA-core prefill and decode step for feature dimensions d' other than 16
// (d' in {8, 24, 32}; D = 1 + d' + d'^2 = 73, 601, 1057), any activation dtype.
//
// Method: BASED reading notes ("Simple linear attention language models
// balance the recall-throughput tradeoff"), sec. 2.2 Eqs. (1)-(3), with the
// second-order Taylor map of sec. 2.3 for a general d' (the page's ablations
// vary the feature dimension): phi(x) = [1, xbar, vec(xbar xbar^T)/sqrt(2)],
// xbar = x / d'^(1/4), so phi(q).phi(k) = 1 + q.k/sqrt(d') + (q.k)^2/(2 d').
//
// Layout: one CTA per (b, h, slice of 8 value columns), 256 threads.  The
// CTA keeps its D x 8 slice of the fp32 state in registers (thread t: column
// t % 8, rows t / 8 + 32 j), so even D = 1057 needs 34 registers a thread;
// every slice keeps its own copy of z (D floats, shared memory) for the
// normaliser.  Per token the features are built in shared memory, the state
// rows are updated and read, and the numerator and normaliser are reduced.
// This is the general-d' path, not a tuned one: d' = 16 has the tensor-core
// kernels.
#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreadsG = 256;
constexpr int kCols = 8;                       // value columns per CTA
constexpr int kSlices = kDV / kCols;           // 8 CTAs per head
constexpr int kRowGroups = kThreadsG / kCols;  // 32

template <int DK>
struct Dims {
    static constexpr int D = 1 + DK + DK * DK;
    static constexpr int kRowsPer = (D + kRowGroups - 1) / kRowGroups;
};

template <int DK>
__device__ __forceinline__ float phi_general(const float *xbar, int f) {
    if (f == 0) return 1.0f;
    if (f <= DK) return xbar[f - 1];
    const int a = (f - 1 - DK) / DK, b = (f - 1 - DK) % DK;
    return xbar[a] * xbar[b] * kInvSqrt2;
}

// y for tokens [0, N) of one (b, h) and 8 value columns, from (s0, z0) to
// (s_out, z_out).  write_z: this launch writes z_out (slice 0 of each head).
template <typename T, int DK>
__global__ void __launch_bounds__(kThreadsG, 1)
prefill_general_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       const float *s0, const float *z0, T *__restrict__ y, float *s_out, float *z_out,
                       int64_t N, float eps, float xscale, bool write_z) {
    constexpr int D = Dims<DK>::D, kRowsPer = Dims<DK>::kRowsPer;
    __shared__ float xq[DK], xk[DK], vs[kCols];
    __shared__ float phq[D], phk[D], zsh[D];
    __shared__ float red[kRowGroups][kCols];
    __shared__ float den_part[kThreadsG / 32];

    const int64_t bh = blockIdx.x;
    const int slice = blockIdx.y;
    const int tid = threadIdx.x;
    const int c = tid % kCols, g = tid / kCols;
    const int col = slice * kCols + c;

    float s[kRowsPer];
#pragma unroll
    for (int j = 0; j < kRowsPer; ++j) {
        const int r = g + j * kRowGroups;
        s[j] = (s0 && r < D) ? s0[(bh * D + r) * kDV + col] : 0.f;
    }
    for (int f = tid; f < D; f += kThreadsG) zsh[f] = z0 ? z0[bh * D + f] : 0.f;

    for (int64_t i = 0; i < N; ++i) {
        const int64_t t = bh * N + i;
        if (tid < DK) xq[tid] = xscale * Act<T>::load(q, t * DK + tid);
        else if (tid >= 32 && tid < 32 + DK) xk[tid - 32] = xscale * Act<T>::load(k, t * DK + tid - 32);
        else if (tid >= 64 && tid < 64 + kCols) vs[tid - 64] = Act<T>::load(v, t * kDV + slice * kCols + tid - 64);
        __syncthreads();
        float dpart = 0.f;
        for (int f = tid; f < D; f += kThreadsG) {
            const float pk = phi_general<DK>(xk, f), pq = phi_general<DK>(xq, f);
            phk[f] = pk;
            phq[f] = pq;
            const float zn = zsh[f] + pk;
            zsh[f] = zn;
            dpart = fmaf(pq, zn, dpart);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, o);
        if ((tid & 31) == 0) den_part[tid >> 5] = dpart;
        __syncthreads();
        const float vc = vs[c];
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j) {
            const int r = g + j * kRowGroups;
            if (r < D) {
                s[j] = fmaf(phk[r], vc, s[j]);
                acc = fmaf(phq[r], s[j], acc);
            }
        }
        red[g][c] = acc;
        __syncthreads();
        if (tid < kCols) {
            float den = eps;
#pragma unroll
            for (int w = 0; w < kThreadsG / 32; ++w) den += den_part[w];
            float num = 0.f;
#pragma unroll
            for (int gg = 0; gg < kRowGroups; ++gg) num += red[gg][tid];
            Act<T>::store(y, t * kDV + slice * kCols + tid, num / den);
        }
        // the next token's first barrier orders these reads before the
        // shared buffers are overwritten
    }
    if (s_out) {
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j) {
            const int r = g + j * kRowGroups;
            if (r < D) s_out[(bh * D + r) * kDV + col] = s[j];
        }
    }
    __syncthreads();
    if (write_z && slice == 0 && z_out)
        for (int f = tid; f < D; f += kThreadsG) z_out[bh * D + f] = zsh[f];
}

// z_out = z_in + phi(k) for one decode token per (b, h): a separate launch so
// that an in-place update cannot race with the slices still reading z_in.
template <typename T, int DK>
__global__ void decode_z_kernel(const T *__restrict__ k, const float *z_in, float *z_out, float xscale) {
    constexpr int D = Dims<DK>::D;
    __shared__ float xk[DK];
    const int64_t bh = blockIdx.x;
    if (threadIdx.x < DK) xk[threadIdx.x] = xscale * Act<T>::load(k, bh * DK + threadIdx.x);
    __syncthreads();
    for (int f = threadIdx.x; f < D; f += blockDim.x) z_out[bh * D + f] = z_in[bh * D + f] + phi_general<DK>(xk, f);
}

template <typename T, int DK>
cudaError_t launch_prefill_dk(const void *q, const void *k, const void *v, const float *s0, const float *z0,
                              void *y, float *s_out, float *z_out, int64_t BH, int64_t N, float eps,
                              bool write_z, cudaStream_t st) {
    const float xscale = (float)(1.0 / sqrt(sqrt((double)DK)));
    dim3 grid((unsigned)BH, kSlices);
    prefill_general_kernel<T, DK><<<grid, kThreadsG, 0, st>>>(
        (const T *)q, (const T *)k, (const T *)v, s0, z0, (T *)y, s_out, z_out, N, eps, xscale, write_z);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_t(int dk, const void *q, const void *k, const void *v, const float *s0,
                             const float *z0, void *y, float *s_out, float *z_out, int64_t BH, int64_t N,
                             float eps, bool write_z, cudaStream_t st) {
    switch (dk) {
        case 8: return launch_prefill_dk<T, 8>(q, k, v, s0, z0, y, s_out, z_out, BH, N, eps, write_z, st);
        case 24: return launch_prefill_dk<T, 24>(q, k, v, s0, z0, y, s_out, z_out, BH, N, eps, write_z, st);
        case 32: return launch_prefill_dk<T, 32>(q, k, v, s0, z0, y, s_out, z_out, BH, N, eps, write_z, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_decode_z(int dk, const void *k, const float *z_in, float *z_out, int64_t BH, cudaStream_t st) {
    const float xscale = (float)(1.0 / sqrt(sqrt((double)dk)));
    switch (dk) {
        case 8: decode_z_kernel<T, 8><<<(unsigned)BH, 128, 0, st>>>((const T *)k, z_in, z_out, xscale); break;
        case 24: decode_z_kernel<T, 24><<<(unsigned)BH, 256, 0, st>>>((const T *)k, z_in, z_out, xscale); break;
        case 32: decode_z_kernel<T, 32><<<(unsigned)BH, 256, 0, st>>>((const T *)k, z_in, z_out, xscale); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_general(const PrefillArgs &a, int dk, la_dtype dt, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    if (dt == LA_DTYPE_BF16)
        return launch_prefill_t<__nv_bfloat16>(dk, a.q, a.k, a.v, a.s0, a.z0, a.y, a.s_out, a.z_out, BH, a.N,
                                               a.eps, true, st);
    return launch_prefill_t<float>(dk, a.q, a.k, a.v, a.s0, a.z0, a.y, a.s_out, a.z_out, BH, a.N, a.eps, true,
                                   st);
}

cudaError_t launch_decode_general(const DecodeArgs &a, int dk, la_dtype dt, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    cudaError_t e;
    // y and the state update (all slices read z_in), then z_out = z_in + phi(k)
    if (dt == LA_DTYPE_BF16) {
        e = launch_prefill_t<__nv_bfloat16>(dk, a.q, a.k, a.v, a.s_in, a.z_in, a.y, a.s_out, nullptr, BH, 1,
                                            a.eps, false, st);
        if (e == cudaSuccess) e = launch_decode_z<__nv_bfloat16>(dk, a.k, a.z_in, a.z_out, BH, st);
    } else {
        e = launch_prefill_t<float>(dk, a.q, a.k, a.v, a.s_in, a.z_in, a.y, a.s_out, nullptr, BH, 1, a.eps,
                                    false, st);
        if (e == cudaSuccess) e = launch_decode_z<float>(dk, a.k, a.z_in, a.z_out, BH, st);
    }
    return e;
}

}  // namespace la
