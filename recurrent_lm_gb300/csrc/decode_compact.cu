// Compact-state decode step and the conversions between the 273-row and the
// 153-row compact state layouts.
//
// BASED reading notes ("Simple linear attention language models balance the
// recall-throughput tradeoff"), sec. 2.3: the Taylor map's quadratic block
// vec(xbar xbar^T) / sqrt2 holds every cross product twice, so the same
// kernel 1 + q.k/4 + (q.k)^2/32 comes from 153 features
//   phi_c(x) = [1, xbar_a, xbar_a^2 / sqrt2 (a = b), xbar_a xbar_b (a < b)],
// rows 0, 1 + a, 17 + c(a, b) with c(a, b) = 16 a - a (a - 1) / 2 + (b - a).
// Sec. 2.5: decoding reads and writes the whole state each step, so the
// 153-row state moves 1.78x fewer bytes than the 273-row one.
//
// The decode kernel has the structure of the 273-row one (one CTA per (b, h)
// streams its state once with every load issued up front, float4 columns,
// shared-memory row-group reduction of the numerator, warp shuffles for the
// normaliser); per head it moves 39,168 B of s and 612 B of z each way.  Steps
// are launched with programmatic dependent launch (see decode.cu).
#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kColGroups = kDV / 4;                                     // 16 float4 per row
constexpr int kRowGroups = kThreads / kColGroups;                       // 16
constexpr int kRowsPerThread = (kDCompact + kRowGroups - 1) / kRowGroups;  // 10
static_assert(kDCompact <= kThreads, "one z entry per thread");

// (a, b), a <= b, of quadratic compact index c = row - 17 in 0..135.
__device__ __forceinline__ void quad_ab(int c, int &a, int &b) {
    a = 0;
    while (c >= 16 - a) {
        c -= 16 - a;
        ++a;
    }
    b = a + c;
}

// phi_c feature of compact row f, xbar already scaled (x / 2).
__device__ __forceinline__ float phi_c_feature(const float *xbar, int f) {
    if (f == 0) return 1.0f;
    if (f <= kDFeat) return xbar[f - 1];
    int a, b;
    quad_ab(f - 1 - kDFeat, a, b);
    const float p = xbar[a] * xbar[b];
    return a == b ? p * kInvSqrt2 : p;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 4)
decode_compact_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                      const float *s_in, const float *z_in, float *s_out, float *z_out,
                      T *__restrict__ y, float eps) {
    __shared__ float xq[kDFeat], xk[kDFeat];
    __shared__ float phq[kThreads], phk[kThreads];
    __shared__ float4 red[kRowGroups][kColGroups];
    __shared__ float den_part[kThreads / 32];

    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    pdl_wait();  // the previous kernel's outputs (q, k, v, the state) are complete from here on
    if (tid < kDFeat) xq[tid] = 0.5f * Act<T>::load(q, bh * kDFeat + tid);
    else if (tid < 2 * kDFeat) xk[tid - kDFeat] = 0.5f * Act<T>::load(k, bh * kDFeat + tid - kDFeat);

    const int cg = tid % kColGroups;
    const int rg = tid / kColGroups;  // rows rg, rg + 16, ...
    const float4 *src = reinterpret_cast<const float4 *>(s_in + bh * (int64_t)kDCompact * kDV);
    float4 *dst = reinterpret_cast<float4 *>(s_out + bh * (int64_t)kDCompact * kDV);

    float4 sr[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int r = rg + j * kRowGroups;
        if (r < kDCompact) sr[j] = src[r * kColGroups + cg];
    }
    const float zin = tid < kDCompact ? z_in[bh * kDCompact + tid] : 0.f;
    float4 vv;
    vv.x = Act<T>::load(v, bh * kDV + cg * 4 + 0);
    vv.y = Act<T>::load(v, bh * kDV + cg * 4 + 1);
    vv.z = Act<T>::load(v, bh * kDV + cg * 4 + 2);
    vv.w = Act<T>::load(v, bh * kDV + cg * 4 + 3);
    __syncthreads();

    // one feature per thread (rows >= 153 are zero and never read)
    phq[tid] = tid < kDCompact ? phi_c_feature(xq, tid) : 0.f;
    phk[tid] = tid < kDCompact ? phi_c_feature(xk, tid) : 0.f;
    __syncthreads();

    float dpart = 0.f;
    if (tid < kDCompact) {
        const float zn = zin + phk[tid];
        z_out[bh * kDCompact + tid] = zn;
        dpart = phq[tid] * zn;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, o);
    if ((tid & 31) == 0) den_part[tid >> 5] = dpart;

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kRowsPerThread; ++j) {
        const int r = rg + j * kRowGroups;
        if (r < kDCompact) {
            const float pk = phk[r], pq = phq[r];
            float4 s = sr[j];
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

// 273-row -> compact: one thread per float4 of s_c (and per z_c entry).
__global__ void state_to_compact_kernel(const float *__restrict__ s, const float *__restrict__ z,
                                        float *__restrict__ s_c, float *__restrict__ z_c, int64_t BH) {
    const int64_t ns = BH * kDCompact * kColGroups;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < ns + BH * kDCompact;
         e += (int64_t)gridDim.x * blockDim.x) {
        const bool is_s = e < ns;
        const int64_t u = is_s ? e : e - ns;
        const int64_t bh = is_s ? u / (kDCompact * kColGroups) : u / kDCompact;
        const int rc = is_s ? (int)(u / kColGroups % kDCompact) : (int)(u % kDCompact);
        // 273-row rows r1 (and r2 for a cross term) of compact row rc
        int r1 = rc, r2 = -1;
        if (rc > kDFeat) {
            int a, b;
            quad_ab(rc - 1 - kDFeat, a, b);
            r1 = 1 + kDFeat + kDFeat * a + b;
            if (a != b) r2 = 1 + kDFeat + kDFeat * b + a;
        }
        if (is_s) {
            const int cg = (int)(u % kColGroups);
            const float4 *sh = reinterpret_cast<const float4 *>(s + bh * (int64_t)kD * kDV);
            float4 x = sh[r1 * kColGroups + cg];
            if (r2 >= 0) {
                const float4 w = sh[r2 * kColGroups + cg];
                x.x = (x.x + w.x) * kInvSqrt2;
                x.y = (x.y + w.y) * kInvSqrt2;
                x.z = (x.z + w.z) * kInvSqrt2;
                x.w = (x.w + w.w) * kInvSqrt2;
            }
            reinterpret_cast<float4 *>(s_c)[u] = x;
        } else {
            float x = z[bh * kD + r1];
            if (r2 >= 0) x = (x + z[bh * kD + r2]) * kInvSqrt2;
            z_c[u] = x;
        }
    }
}

// compact -> 273-row: one thread per float4 of s (and per z entry); cross
// terms are split evenly between (a, b) and (b, a).
__global__ void state_from_compact_kernel(const float *__restrict__ s_c, const float *__restrict__ z_c,
                                          float *__restrict__ s, float *__restrict__ z, int64_t BH) {
    const int64_t ns = BH * kD * kColGroups;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < ns + BH * kD;
         e += (int64_t)gridDim.x * blockDim.x) {
        const bool is_s = e < ns;
        const int64_t u = is_s ? e : e - ns;
        const int64_t bh = is_s ? u / (kD * kColGroups) : u / kD;
        const int r = is_s ? (int)(u / kColGroups % kD) : (int)(u % kD);
        int rc = r;
        float scale = 1.f;
        if (r > kDFeat) {
            const int x = (r - 1 - kDFeat) / kDFeat, y = (r - 1 - kDFeat) % kDFeat;
            const int a = x < y ? x : y, b = x < y ? y : x;
            rc = 1 + kDFeat + kDFeat * a - a * (a - 1) / 2 + (b - a);
            if (a != b) scale = kInvSqrt2;
        }
        if (is_s) {
            const int cg = (int)(u % kColGroups);
            float4 w = reinterpret_cast<const float4 *>(s_c + bh * (int64_t)kDCompact * kDV)[rc * kColGroups + cg];
            w.x *= scale;
            w.y *= scale;
            w.z *= scale;
            w.w *= scale;
            reinterpret_cast<float4 *>(s)[u] = w;
        } else {
            z[u] = z_c[bh * kDCompact + rc] * scale;
        }
    }
}

unsigned conv_grid(int64_t work) {
    const int64_t blocks = (work + 255) / 256;
    return (unsigned)(blocks < 152 * 16 ? (blocks > 0 ? blocks : 1) : 152 * 16);
}

}  // namespace

cudaError_t launch_decode_compact(const DecodeArgs &a, la_dtype dt, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    if (BH == 0) return cudaSuccess;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)BH);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dt == LA_DTYPE_BF16)
        return cudaLaunchKernelEx(&cfg, decode_compact_kernel<__nv_bfloat16>, (const __nv_bfloat16 *)a.q,
                                  (const __nv_bfloat16 *)a.k, (const __nv_bfloat16 *)a.v, a.s_in, a.z_in, a.s_out,
                                  a.z_out, (__nv_bfloat16 *)a.y, a.eps);
    return cudaLaunchKernelEx(&cfg, decode_compact_kernel<float>, (const float *)a.q, (const float *)a.k,
                              (const float *)a.v, a.s_in, a.z_in, a.s_out, a.z_out, (float *)a.y, a.eps);
}

cudaError_t launch_state_to_compact(const float *s, const float *z, float *s_c, float *z_c, int64_t BH,
                                    cudaStream_t st) {
    state_to_compact_kernel<<<conv_grid(BH * kDCompact * (kColGroups + 1)), 256, 0, st>>>(s, z, s_c, z_c, BH);
    return cudaGetLastError();
}

cudaError_t launch_state_from_compact(const float *s_c, const float *z_c, float *s, float *z, int64_t BH,
                                      cudaStream_t st) {
    state_from_compact_kernel<<<conv_grid(BH * kD * (kColGroups + 1)), 256, 0, st>>>(s_c, z_c, s, z, BH);
    return cudaGetLastError();
}

}  // namespace la
