// CUDA-core (fp32 FFMA) kernels: the token-by-token prefill used for fp32
// activations (its initial state is s0 plus, for the prefix call, the
// per-segment prefix partial states added in segment order, so the sum is
// deterministic), the per-segment prefix-state partial sums for fp32
// activations, and the state copy used when N == 0.
//
// Prefill: BASED reading notes ("Simple linear attention language models
// balance the recall-throughput tradeoff"), sec. 2.2 Eqs. (1)-(3); initial
// state: "Understanding and Improving Length Generalization in Recurrent
// Models" reading notes, sec. 2.5 Eq. (4).  Prefix state: "Just read twice"
// reading notes, sec. 2.6 Eqs. (3)-(4).
//
// One CTA owns one (b, h) and keeps the whole 273 x 64 fp32 state in
// registers: thread t holds column c = t % 64 of the rows r = t / 64 + 4 j.
// Per token the feature vectors phi(q), phi(k) are built in shared memory,
// every thread updates its rows and accumulates its share of phi(q)^T s,
// and the four row-group partials plus the normaliser are reduced in shared
// memory.  This path exists for fp32 accuracy (the tensor-core path rounds
// operands to bf16); it is not the fast path.
#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kRowGroups = kThreads / kDV;                          // 4
constexpr int kRowsPerThread = (kD + kRowGroups - 1) / kRowGroups;  // 69

template <typename T>
__device__ __forceinline__ void load_token(const T *q, const T *k, const T *v,
                                           int64_t qi, int64_t vi, float *xq,
                                           float *xk, float *vs, int tid) {
    if (tid < kDFeat) xq[tid] = 0.5f * Act<T>::load(q, qi + tid);
    else if (tid < 2 * kDFeat) xk[tid - kDFeat] = 0.5f * Act<T>::load(k, qi + tid - kDFeat);
    else if (tid >= 64 && tid < 64 + kDV) vs[tid - 64] = Act<T>::load(v, vi + tid - 64);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
prefill_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                    const T *__restrict__ v, const float *__restrict__ s0,
                    const float *__restrict__ z0, T *__restrict__ y,
                    float *__restrict__ s_out, float *__restrict__ z_out,
                    int64_t N, float eps, const int32_t *__restrict__ left_pad, int64_t H,
                    unsigned *status, const float *__restrict__ gamma,
                    const float *__restrict__ part_s, const float *__restrict__ part_z, int64_t nseg) {
    __shared__ float xq[kDFeat], xk[kDFeat], vs[kDV];
    __shared__ float phq[kD], phk[kD];
    __shared__ float zsh[kD];
    __shared__ float red[kRowGroups][kDV];
    __shared__ float den_part[kThreads / 32];

    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int c = tid % kDV, g = tid / kDV;

    float s[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int r = g + j * kRowGroups;
        s[j] = (s0 && r < kD) ? s0[(bh * kD + r) * kDV + c] : 0.f;
    }
    for (int f = tid; f < kD; f += kThreads) zsh[f] = z0 ? z0[bh * kD + f] : 0.f;
    // prefix call: + the partial states of the prefix segments, in order
    for (int64_t sg = 0; part_s && sg < nseg; ++sg) {
        const float *ps = part_s + (bh * nseg + sg) * (int64_t)kD * kDV;
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) {
            const int r = g + j * kRowGroups;
            if (r < kD) s[j] += ps[r * kDV + c];
        }
        const float *pz = part_z + (bh * nseg + sg) * (int64_t)kD;
        for (int f = tid; f < kD; f += kThreads) zsh[f] += pz[f];
    }

    // leading padding positions of this batch row: y = 0, no state change
    const int64_t lpad = row_left_pad(left_pad, bh / H, N, status, tid == 0);
    // per-head decay (s = gamma s + phi(k) v^T), clamped to [0, 1] and reported
    const bool decay = gamma != nullptr;
    float gam = 1.f;
    if (decay) {
        gam = gamma[bh % H];
        if (!(gam >= 0.f && gam <= 1.f)) {
            if (tid == 0) atomicOr(status, kStatusBadDecay);
            gam = (gam > 1.f) ? 1.f : 0.f;
        }
    }
    for (int64_t i = 0; i < lpad; ++i)
        if (tid < kDV) Act<T>::store(y, (bh * N + i) * kDV + tid, 0.f);
    for (int64_t i = lpad; i < N; ++i) {
        const int64_t t = bh * N + i;
        load_token(q, k, v, t * kDFeat, t * kDV, xq, xk, vs, tid);
        __syncthreads();
        float dpart = 0.f;
        for (int f = tid; f < kD; f += kThreads) {
            const float pk = phi_feature(xk, f), pq = phi_feature(xq, f);
            phk[f] = pk;
            phq[f] = pq;
            const float zn = (decay ? gam * zsh[f] : zsh[f]) + pk;
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
        for (int j = 0; j < kRowsPerThread; ++j) {
            const int r = g + j * kRowGroups;
            if (r < kD) {
                s[j] = fmaf(phk[r], vc, decay ? gam * s[j] : s[j]);
                acc = fmaf(phq[r], s[j], acc);
            }
        }
        red[g][c] = acc;
        __syncthreads();
        if (tid < kDV) {
            float den = eps;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) den += den_part[w];
            float num = 0.f;
#pragma unroll
            for (int gg = 0; gg < kRowGroups; ++gg) num += red[gg][tid];
            Act<T>::store(y, t * kDV + tid, num / den);
        }
        // the next iteration's first barrier orders these reads before the
        // shared buffers are overwritten
    }
    if (s_out) {
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) {
            const int r = g + j * kRowGroups;
            if (r < kD) s_out[(bh * kD + r) * kDV + c] = s[j];
        }
    }
    __syncthreads();
    if (z_out)
        for (int f = tid; f < kD; f += kThreads) z_out[bh * kD + f] = zsh[f];
}

// Partial prefix state of one token segment: sum phi(k_e_j) v_e_j^T and
// sum phi(k_e_j) over j in [seg * seg_len, min(M, (seg + 1) * seg_len)).
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
prefix_partial_simt_kernel(const T *__restrict__ ke, const T *__restrict__ ve,
                           int64_t M, int64_t seg_len, int64_t nseg,
                           float *__restrict__ part_s, float *__restrict__ part_z,
                           const int32_t *__restrict__ left_pad, int64_t H, int64_t N) {
    __shared__ float xk[kDFeat], vs[kDV];
    __shared__ float phk[kD];
    __shared__ float zsh[kD];
    const int64_t bh = blockIdx.x, seg = blockIdx.y;
    const int tid = threadIdx.x;
    const int c = tid % kDV, g = tid / kDV;
    const int64_t j1 = (seg * seg_len + seg_len < M) ? seg * seg_len + seg_len : M;
    // prefix positions below min(left pad, M) are padding (range reported by the prefill)
    const int64_t pe = min(M, row_left_pad(left_pad, bh / H, N, nullptr, false));
    const int64_t j0 = max(seg * seg_len, pe);

    float s[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) s[j] = 0.f;
    for (int f = tid; f < kD; f += kThreads) zsh[f] = 0.f;

    for (int64_t jj = j0; jj < j1; ++jj) {
        const int64_t t = bh * M + jj;
        if (tid < kDFeat) xk[tid] = 0.5f * Act<T>::load(ke, t * kDFeat + tid);
        else if (tid >= 64 && tid < 64 + kDV) vs[tid - 64] = Act<T>::load(ve, t * kDV + tid - 64);
        __syncthreads();
        for (int f = tid; f < kD; f += kThreads) {
            const float pk = phi_feature(xk, f);
            phk[f] = pk;
            zsh[f] += pk;
        }
        __syncthreads();
        const float vc = vs[c];
#pragma unroll
        for (int j = 0; j < kRowsPerThread; ++j) {
            const int r = g + j * kRowGroups;
            if (r < kD) s[j] = fmaf(phk[r], vc, s[j]);
        }
        __syncthreads();
    }
    float *ps = part_s + (bh * nseg + seg) * (int64_t)kD * kDV;
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int r = g + j * kRowGroups;
        if (r < kD) ps[r * kDV + c] = s[j];
    }
    float *pz = part_z + (bh * nseg + seg) * (int64_t)kD;
    for (int f = tid; f < kD; f += kThreads) pz[f] = zsh[f];
}

__global__ void state_copy_kernel(const float *__restrict__ s0,
                                  const float *__restrict__ z0, float *s_out,
                                  float *z_out, int64_t BH, int64_t D) {
    const int64_t ns = BH * D * kDV, nz = BH * D;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < ns + nz;
         e += (int64_t)gridDim.x * blockDim.x) {
        if (e < ns) {
            if (s_out) s_out[e] = s0 ? s0[e] : 0.f;
        } else if (z_out) {
            z_out[e - ns] = z0 ? z0[e - ns] : 0.f;
        }
    }
}

int grid_for(int64_t n, int threads) {
    int64_t b = (n + threads - 1) / threads;
    const int64_t cap = 152 * 16;
    return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, la_dtype dt, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    if (dt == LA_DTYPE_BF16)
        prefill_simt_kernel<__nv_bfloat16><<<(unsigned)BH, kThreads, 0, st>>>(
            (const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k,
            (const __nv_bfloat16 *)a.v, a.s0, a.z0, (__nv_bfloat16 *)a.y, a.s_out,
            a.z_out, a.N, a.eps, a.left_pad, a.H, a.status, a.gamma, a.part_s, a.part_z, a.nseg);
    else
        prefill_simt_kernel<float><<<(unsigned)BH, kThreads, 0, st>>>(
            (const float *)a.q, (const float *)a.k, (const float *)a.v, a.s0, a.z0,
            (float *)a.y, a.s_out, a.z_out, a.N, a.eps, a.left_pad, a.H, a.status, a.gamma, a.part_s,
            a.part_z, a.nseg);
    return cudaGetLastError();
}

cudaError_t launch_prefix_partials_simt(const PrefixArgs &a, la_dtype dt, cudaStream_t st) {
    if (a.nseg > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)(a.B * a.H), (unsigned)a.nseg);
    if (dt == LA_DTYPE_BF16)
        prefix_partial_simt_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            (const __nv_bfloat16 *)a.k_e, (const __nv_bfloat16 *)a.v_e, a.M,
            a.seg_len, a.nseg, a.part_s, a.part_z, a.left_pad, a.H, a.N);
    else
        prefix_partial_simt_kernel<float><<<grid, kThreads, 0, st>>>(
            (const float *)a.k_e, (const float *)a.v_e, a.M, a.seg_len, a.nseg,
            a.part_s, a.part_z, a.left_pad, a.H, a.N);
    return cudaGetLastError();
}

cudaError_t launch_state_copy(int64_t D, const float *s0, const float *z0, float *s_out,
                              float *z_out, int64_t BH, cudaStream_t st) {
    const int64_t total = BH * (D * kDV + D);
    state_copy_kernel<<<grid_for(total, 256), 256, 0, st>>>(s0, z0, s_out, z_out, BH, D);
    return cudaGetLastError();
}

}  // namespace la
