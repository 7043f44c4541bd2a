// Prefix-state partial sums on the tensor cores (bf16 operands, fp32
// accumulate): for each (b, h) and each segment of up to 2048 prefix tokens,
//   s_E,seg = sum_j phi(k_e_j) v_e_j^T,   z_E,seg = sum_j phi(k_e_j)
// ("Just read twice" reading notes, sec. 2.6: the non-causal encoder state of
// prefix linear attention; sec. 2.8: the encoder state is accumulated first
// and then seeds the causal scan).  Each partial is written as the kernel
// holds it, in the internal compact rows ([160][64] values and [160] z', fp32,
// row = compact feature); the causal prefill's set-up adds the segments to
// its initial state in segment order (deterministic), so there is no
// separate reduction pass.
//
// Same update as the causal prefill kernel: [S'^T ; z'] += [V | 1]^T Phi'_K
// per 128-token chunk (8 MMAs of M = 128, N = 160, K = 16), with the compact
// feature map generated one token per thread.  Splitting the prefix over
// segments spreads the reduction over all SMs instead of lengthening each
// (b, h) scan.  256 threads, about 111 KB of shared memory and 256 TMEM
// columns per CTA, so two CTAs share an SM.
#include "la_internal.h"
#include "taylor_tc.cuh"
#include "tc_common.cuh"

namespace la {
namespace {

using namespace tc;
using namespace taylor;

constexpr int kC = 128;
constexpr int kThreads = 256;
constexpr int kStages = 3;

// Shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kSmPhiK = 0;        // MN-major B: 3 x 16K SW128
constexpr uint32_t kSmV = 49152;       // 3 x [128][64] bf16 SW128
constexpr uint32_t kSmOnes = 98304;    // [16][64] bf16 ones: rows 64..127 of [V | 1]^T for every K step
constexpr uint32_t kSmK = 100352;      // 3 x [128][16] bf16 SW32
constexpr uint32_t kSmBar = 112640;
constexpr uint32_t kSmTotal = kSmBar + 256;
constexpr uint32_t kSmAlloc = kSmTotal + 1024;

// Phi'_K is produced and consumed in two halves of 64 tokens (K steps 0..3 and
// 4..7), each with its own full / empty barrier, so that the features of one
// half of chunk c + 1 are generated while the update reads the other half of
// chunk c.
enum { B_KV_FULL = 0, B_KV_EMPTY = kStages, B_PHK_FULL = 2 * kStages, B_PHK_EMPTY = 2 * kStages + 2,
       B_S_FULL = 2 * kStages + 4, B_COUNT };
constexpr uint32_t kSmTmemSlot = kSmBar + 8 * B_COUNT;
constexpr uint32_t kSmAbort = kSmTmemSlot + 4;
static_assert(kSmAbort + 4 <= kSmTotal, "barrier area");
static_assert(kSmV + kStages * 16384 <= kSmOnes && kSmOnes + 2048 <= kSmK && kSmK + kStages * 4096 <= kSmBar,
              "shared memory map");
static_assert(2 * (kSmAlloc + 1024) <= 233472, "two CTAs per SM");

constexpr uint32_t kIdUp = idesc_bf16(128, kNFeat, true, true);  // [V | 1]^T x Phi'_K

// Optional per-role timeline of CTA (0, 0) (compile with -DLA_TRACE): SM clock
// offsets from kernel entry for events of each role and chunk.
#ifdef LA_TRACE
constexpr int kPTraceChunks = 256;
__device__ uint32_t g_ptrace[3][kPTraceChunks][4];
#define LA_PTR(role, c, ev)                                                              \
    do {                                                                                 \
        if (blockIdx.x == 0 && blockIdx.y == 0 && (c) < kPTraceChunks)                   \
            g_ptrace[role][c][ev] = (uint32_t)(clock64() - t_start);                     \
    } while (0)
#else
#define LA_PTR(role, c, ev) do { } while (0)
#endif

// kPad: the launch carries left-padding counts (a separate instantiation, so
// the unpadded one carries none of the skip code).
template <bool kPad>
__global__ void __launch_bounds__(kThreads, 2)
prefix_partial_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                         int M, int seg_len, int nseg, float *__restrict__ part_s,
                         float *__restrict__ part_z, unsigned *status,
                         const int32_t *__restrict__ left_pad, int64_t H, int64_t N) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) { return sb + kSmBar + 8u * (uint32_t)i; };
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kSmAbort);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t bh = blockIdx.x;
    const int seg = blockIdx.y;
#ifdef LA_TRACE
    const long long t_start = clock64();
#endif
    const int js = seg * seg_len;  // the segment: prefix positions [js, j1)
    const int j1 = min(M, js + seg_len);
    // prefix positions below min(left pad, M) are padding (range reported by the prefill)
    const int pe = (int)min((int64_t)M, row_left_pad(left_pad, bh / H, N, status, false));
    // the segment's whole chunks below pe add nothing and are skipped (a segment
    // that is all padding runs no chunk and writes a zero partial state)
    const int skip = kPad ? max(0, min((pe - js) / kC, (j1 - js + kC - 1) / kC)) : 0;
    const int j0 = js + skip * kC;               // first chunk processed
    const int n = (j1 - js + kC - 1) / kC - skip;  // chunks processed

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KV_FULL + s), 1);
            mbar_init(bar(B_KV_EMPTY + s), 1 + 4);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(B_PHK_FULL + h), 2);  // the two generation warps of the half
            mbar_init(bar(B_PHK_EMPTY + h), 1);
        }
        mbar_init(bar(B_S_FULL), 1);
        *abort = 0;
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(sb + kSmTmemSlot, 256);
        tmem_relinquish();
    }
    for (int i = tid; i < 2048 / 16; i += kThreads)
        st_shared_v4(sb + kSmOnes + 16 * i, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kSmTmemSlot);

    if (warp == 0) {
        // ================= TMA producer: k_e, v_e chunks of the segment =================
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            int issued = 0;
            for (int c = 0; c < n; ++c) {
                const int st = c % kStages;
                LA_PTR(0, c, 0);
                if (!mbar_wait(bar(B_KV_EMPTY + st), ((uint32_t)(c / kStages) & 1u) ^ 1u, abort, status))
                    break;
                LA_PTR(0, c, 1);
                mbar_expect_tx(bar(B_KV_FULL + st), kC * 16 * 2 + kC * 64 * 2);
                tma_load_3d(sb + kSmK + st * 4096, &tk, bar(B_KV_FULL + st), 0, j0 + c * kC, (int)bh);
                tma_load_3d(sb + kSmV + st * 16384, &tv, bar(B_KV_FULL + st), 0, j0 + c * kC, (int)bh);
                issued = c + 1;
            }
            if (*abort)
                for (int c = (issued > kStages ? issued - kStages : 0); c < issued; ++c)
                    drain_wait(bar(B_KV_FULL + c % kStages), (uint32_t)(c / kStages) & 1u);
        }
    } else if (warp == 1) {
        // ================= MMA issuer: [S'^T ; z'] += [V | 1]^T Phi'_K =================
        if (lane == 0) {
            const uint64_t dPhiK = smem_desc(sb + kSmPhiK, 16384, 1024, kSw128);
            bool ok = true;
            for (int c = 0; c < n && ok; ++c) {
                const int st = c % kStages;
                ok = mbar_wait(bar(B_KV_FULL + st), (uint32_t)(c / kStages) & 1u, abort, status);
                for (int h = 0; h < 2 && ok; ++h) {
                    if (!(ok = mbar_wait(bar(B_PHK_FULL + h), (uint32_t)c & 1u, abort, status))) break;
                    if (h == 0) LA_PTR(1, c, 0);
                    tc_fence_after();
                    // A = [V | 1]^T, MN-major: K step s reads value rows 0..63 from its
                    // 16 tokens of the V stage and rows 64..127 from the one 2 KB ones
                    // block (the leading byte offset is the distance between the two)
#pragma unroll
                    for (int s = 4 * h; s < 4 * h + 4; ++s) {
                        const uint32_t va = kSmV + (uint32_t)st * 16384u + (uint32_t)s * 2048u;
                        mma_bf16(tmem, smem_desc(sb + va, kSmOnes - va, 1024, kSw128), dPhiK + s * (2048 >> 4),
                                 kIdUp, (c > 0 || s > 0));
                    }
                    mma_commit(bar(B_PHK_EMPTY + h));
                }
                if (ok) mma_commit(bar(B_KV_EMPTY + st));
                LA_PTR(1, c, 1);
            }
            mma_commit(bar(B_S_FULL));  // also covers an early exit: every issued MMA completes first
        }
    } else if (warp >= 4) {
        // ================= feature generation (one token per thread) =================
        const int t = tid - 128;
        const int h = t >> 6;  // the half of the Phi'_K tile this warp writes
        for (int c = 0; c < n; ++c) {
            const int st = c % kStages;
            if (!mbar_wait(bar(B_KV_FULL + st), (uint32_t)(c / kStages) & 1u, abort, status)) break;
            if (tid == 128) LA_PTR(2, c, 0);
            uint4 klo, khi;
            load_row16_raw(sb + kSmK + st * 4096, t, klo, khi);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_KV_EMPTY + st));
            if (!mbar_wait(bar(B_PHK_EMPTY + h), ((uint32_t)c & 1u) ^ 1u, abort, status)) break;
            if (tid == 128) LA_PTR(2, c, 1);
            // outside this segment, or left padding: no contribution
            const bool pad = j0 + c * kC + t >= j1 || j0 + c * kC + t < pe;
            emit_features<true>(klo, khi, sb + kSmPhiK, t, pad, std::make_integer_sequence<int, 20>{});
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PHK_FULL + h));
            if (tid == 128) LA_PTR(2, c, 2);
        }
        // ---- partial state of this segment in the internal compact rows (value
        // d: lanes 0..63 of warps 4, 5, entry (F, d) at [F * 64 + d]; z': lane
        // 64, warp 6, entry F at [F]).  An empty segment writes zeros.
        if (warp < 7) {
            const int w = warp - 4;
            const bool zrow = (w == 2);
            const bool ok = n == 0 || mbar_wait(bar(B_S_FULL), 0, abort, status);
            __syncwarp();
            tc_fence_after();
            if (ok) {
                const int64_t slot = bh * nseg + seg;
                float *dst = zrow ? part_z + slot * kNFeat : part_s + slot * kNFeat * kDV + 32 * w + lane;
                const int64_t stride = zrow ? 1 : kDV;
#pragma unroll 1
                for (int G = 0; G < kNFeat / 32; ++G) {
                    uint32_t r[32];
                    if (n > 0) {
                        tmem_load32_sync(tmem + ((uint32_t)(32 * w) << 16) + 32 * G, r);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    if (!zrow || lane == 0) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) __stcg(dst + (32 * G + j) * stride, __uint_as_float(r[j]));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

#ifdef LA_TRACE
extern "C" LA_API int la_debug_prefix_trace(void *host, size_t bytes) {
    if (bytes > sizeof(g_ptrace)) bytes = sizeof(g_ptrace);
    return (int)cudaMemcpyFromSymbol(host, g_ptrace, bytes);
}
#endif

cudaError_t launch_prefix_partials_tc(const PrefixArgs &a, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    if (a.M > (int64_t)0x7FFFFFFF - kC || a.nseg > 65535) return cudaErrorInvalidValue;
    CUtensorMap tk, tv;
    if (!make_row_tmap(&tk, a.k_e, BH, a.M, 16, false) || !make_row_tmap(&tv, a.v_e, BH, a.M, 64, true))
        return cudaErrorInvalidValue;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        cudaError_t e = cudaFuncSetAttribute(prefix_partial_tc_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefix_partial_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmAlloc);
        if (e != cudaSuccess) return e;
        configured_for = dev;
    }
    dim3 grid((unsigned)BH, (unsigned)a.nseg);
    auto kern = a.left_pad ? prefix_partial_tc_kernel<true> : prefix_partial_tc_kernel<false>;
    kern<<<grid, kThreads, kSmAlloc, st>>>(tk, tv, (int)a.M, (int)a.seg_len, (int)a.nseg, a.part_s, a.part_z,
                                           a.status, a.left_pad, a.H, a.N);
    return cudaGetLastError();
}

}  // namespace la
