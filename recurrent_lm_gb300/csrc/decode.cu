// Recurrent decode step: one token per (b, h), bandwidth bound.
//
// BASED reading notes ("Simple linear attention language models balance the
// recall-throughput tradeoff"), sec. 2.2 Eq. (2) for a single token, and
// sec. 2.5: the decode kernel fuses the outer-product write with the query
// read-out but still reads and writes the whole persistent state.
//
// Per head the state is s [273][64] fp32 (69,888 B) + z [273] fp32; one CTA
// streams it once: every thread owns one float4 column group (16 per row) of
// a strided set of rows, issues all of its row loads before using any (so a
// CTA keeps ~70 KB in flight), applies s += phi(k)_r v, writes the row back
// and accumulates phi(q)_r * s_r for the numerator.  Partial numerators are
// summed across the 16 row groups in shared memory; the normaliser phi(q).z
// uses a warp-shuffle reduction.
//
// Steps are launched with programmatic dependent launch, so a step's CTAs are
// scheduled while the previous kernel in the stream drains; each waits for it
// (griddepcontrol.wait) before reading anything, since that kernel may have
// produced q, k, v or the state.
#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kColGroups = kDV / 4;              // 16 float4 per state row
constexpr int kRowGroups = kThreads / kColGroups;  // 16
constexpr int kRowsPerThread = (kD + kRowGroups - 1) / kRowGroups;  // 18

// kDecay: s = gamma_h s + phi(k) v^T, z = gamma_h z + phi(k) (a fixed per-head
// decay, the general recurrence of the length-generalization notes, sec. 2.1
// Eq. (1), with A_t = gamma I); a separate instantiation.
template <typename T, bool kDecay>
__global__ void __launch_bounds__(kThreads, 2)
decode_step_kernel(const T *__restrict__ q, const T *__restrict__ k,
                   const T *__restrict__ v, const float *s_in, const float *z_in,
                   float *s_out, float *z_out, T *__restrict__ y, float eps,
                   const float *__restrict__ gamma, int64_t H, unsigned *status) {
    __shared__ float xq[kDFeat], xk[kDFeat];
    __shared__ float phq[kD + 15], phk[kD + 15];
    __shared__ float4 red[kRowGroups][kColGroups];
    __shared__ float den_part[kThreads / 32];

    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_wait();  // the previous kernel's outputs (q, k, v, the state) are complete from here on
    float g = 1.f;
    if constexpr (kDecay) {
        g = gamma[bh % H];
        if (!(g >= 0.f && g <= 1.f)) {  // clamped; reported by one thread
            if (tid == 0) atomicOr(status, kStatusBadDecay);
            g = (g > 1.f) ? 1.f : 0.f;
        }
    }
    if (tid < kDFeat) xq[tid] = 0.5f * Act<T>::load(q, bh * kDFeat + tid);
    else if (tid < 2 * kDFeat) xk[tid - kDFeat] = 0.5f * Act<T>::load(k, bh * kDFeat + tid - kDFeat);

    const int cg = tid % kColGroups;   // float4 column group
    const int rg = tid / kColGroups;   // row group: rows rg, rg + 16, ...
    const float4 *src = reinterpret_cast<const float4 *>(s_in + bh * (int64_t)kD * kDV);
    float4 *dst = reinterpret_cast<float4 *>(s_out + bh * (int64_t)kD * kDV);

    // Issue every state load of this thread up front.
    float4 sr[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int r = rg + j * kRowGroups;
        if (r < kD) sr[j] = src[r * kColGroups + cg];
    }
    const float zin0 = z_in[bh * kD + tid];
    const float zin1 = (tid + kThreads < kD) ? z_in[bh * kD + tid + kThreads] : 0.f;
    float4 vv;
    vv.x = Act<T>::load(v, bh * kDV + cg * 4 + 0);
    vv.y = Act<T>::load(v, bh * kDV + cg * 4 + 1);
    vv.z = Act<T>::load(v, bh * kDV + cg * 4 + 2);
    vv.w = Act<T>::load(v, bh * kDV + cg * 4 + 3);
    __syncthreads();

    for (int f = tid; f < kD; f += kThreads) {
        phq[f] = phi_feature(xq, f);
        phk[f] = phi_feature(xk, f);
    }
    __syncthreads();

    // z update and the normaliser phi(q).z_new.
    float dpart = 0.f;
    {
        const float zn = (kDecay ? g * zin0 : zin0) + phk[tid];
        z_out[bh * kD + tid] = zn;
        dpart = phq[tid] * zn;
        if (tid + kThreads < kD) {
            const int f = tid + kThreads;
            const float zn1 = (kDecay ? g * zin1 : zin1) + phk[f];
            z_out[bh * kD + f] = zn1;
            dpart += phq[f] * zn1;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, o);
    if ((tid & 31) == 0) den_part[tid >> 5] = dpart;

    // s update (write back) and the numerator partials.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int r = rg + j * kRowGroups;
        if (r < kD) {
            const float pk = phk[r], pq = phq[r];
            float4 s = sr[j];
            if constexpr (kDecay) {
                s.x *= g;
                s.y *= g;
                s.z *= g;
                s.w *= g;
            }
            s.x = fmaf(pk, vv.x, s.x);
            s.y = fmaf(pk, vv.y, s.y);
            s.z = fmaf(pk, vv.z, s.z);
            s.w = fmaf(pk, vv.w, s.w);
            dst[r * kColGroups + cg] = s;
            acc.x = fmaf(pq, s.x, acc.x);
            acc.y = fmaf(pq, s.y, acc.y);
            acc.z = fmaf(pq, s.z, acc.z);
            acc.w = fmaf(pq, s.w, acc.w);
        }
    }
    red[rg][cg] = acc;
    pdl_trigger();  // this CTA's state is written; the next step may be scheduled
    __syncthreads();

    if (tid < kDV) {
        float den = eps;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) den += den_part[w];
        const int c4 = tid >> 2, lane4 = tid & 3;
        float num = 0.f;
#pragma unroll
        for (int g = 0; g < kRowGroups; ++g) {
            const float4 p = red[g][c4];
            num += lane4 == 0 ? p.x : lane4 == 1 ? p.y : lane4 == 2 ? p.z : p.w;
        }
        Act<T>::store(y, bh * kDV + tid, num / den);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, la_dtype dt, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    if (BH == 0) return cudaSuccess;
    dim3 grid((unsigned)BH), block(kThreads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dt == LA_DTYPE_BF16) {
        auto kern = a.gamma ? decode_step_kernel<__nv_bfloat16, true> : decode_step_kernel<__nv_bfloat16, false>;
        return cudaLaunchKernelEx(&cfg, kern, (const __nv_bfloat16 *)a.q, (const __nv_bfloat16 *)a.k,
                                  (const __nv_bfloat16 *)a.v, a.s_in, a.z_in, a.s_out, a.z_out,
                                  (__nv_bfloat16 *)a.y, a.eps, a.gamma, a.H, a.status);
    }
    auto kern = a.gamma ? decode_step_kernel<float, true> : decode_step_kernel<float, false>;
    return cudaLaunchKernelEx(&cfg, kern, (const float *)a.q, (const float *)a.k, (const float *)a.v, a.s_in,
                              a.z_in, a.s_out, a.z_out, (float *)a.y, a.eps, a.gamma, a.H, a.status);
}

}  // namespace la
