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
//    with the causal mask in registers, written back in place into TMEM as
//    bf16, then [num | den] = P [V | 1] with P as the TMEM A operand.
//  * Inter-chunk terms with a symmetric-compact feature map inside the
//    kernel: 136 quadratic features (a <= b) + 1 + 16 + 7 pad = 160 instead
//    of 273 (BASED sec. 2.3 table: 1 + d' + d'(d'+1)/2 = 153).  Query features
//    carry xbar_a xbar_b, key features xbar_a xbar_b (a < b) and xbar_a^2 / 2,
//    so Phi'_Q . Phi'_K = 1 + q.k/4 + (q.k)^2/32 exactly.
//  * The state is kept transposed, S'^T (values x features, fp32 in TMEM),
//    and updated as [S'^T ; z'] += [V | 1]^T Phi'_K: one M = 128, N = 160 MMA
//    per 16 tokens (the 64 value rows plus ones rows that yield z').  Its
//    bf16 copy is then directly the K-major B operand of the read-out
//    [num | den] += Phi'_Q [S' | z'].  The 273-row C-ABI state is converted
//    at the start and the end (the antisymmetric part of a caller's s0 cannot
//    influence any output and is passed through unchanged).
//  * These MMAs have small N and are bound by shared-memory operand
//    bandwidth, so the layout minimises operand bytes per chunk.
//  * Roles: warp 0 TMA producer (q, k, v chunks, zero-filled past N; warp 3
//    issues the first chunks' loads during set-up), warp 1 MMA issuer,
//    warps 2, 3 the P epilogue of keys 64..127 for rows 64..127, warpgroup 1
//    feature generation (one token per thread) and the state conversion
//    (TMEM fp32 -> bf16 operand) of feature groups 3, 4, warpgroup 2 the P
//    epilogue of keys 0..63 and the conversion of groups 0..2, warpgroup 3
//    the output epilogue y = num / den (TMA stores).  The final state is
//    assembled in shared memory and written with one bulk copy.  With decay
//    the y warps also form P of keys 0..63, warpgroup 2 converts (and
//    rescales) all five groups, and the feature warps only emit features.
//  * Every wait is bounded: after ~1 s the kernel records a timeout in the
//    device status word and every role unwinds.
#include <type_traits>
#include <utility>

#include "la_internal.h"
#include "taylor_tc.cuh"
#include "tc_common.cuh"

namespace la {
namespace {

using namespace tc;
using namespace taylor;

constexpr int kC = 128;          // tokens per chunk
constexpr int kThreads = 512;
constexpr int kNB = 80;          // B columns of the value side: 64 values + 16 normaliser

// TMEM columns (all 512): S'^T|z' (160), Phi'_Q (80: 160 bf16 features, two
// per 32-bit column, the A operand of the read-out), num|den (80), T = Q K^T
// (128 fp32) and P (64: 128 x 128 bf16, two keys per 32-bit column, the A
// operand of P V).  Keeping Phi'_Q in TMEM rather than shared memory takes
// 80 KB per chunk (its stores and the read-out's operand reads) off the
// shared-memory data path, which the tensor core's other operand reads, the
// TMA, the feature stores and every barrier operation share.  With P in its
// own buffer, Q K^T of the next chunk may overwrite T as soon as the P warps
// have read it.
constexpr uint32_t kTmS = 0;
constexpr uint32_t kTmPhiQ = 160;
constexpr uint32_t kTmNum = 240;
constexpr uint32_t kTmT = 320;
constexpr uint32_t kTmP = 448;

// Shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kSmPhiQ = 0;        // 40 KB, free during the chunk loop (Phi'_Q lives in TMEM)
constexpr uint32_t kSmPhiK = 40960;    // MN-major B: 3 x 16K SW128 (blk2: 32 of 64 features used)
constexpr uint32_t kSmSb = 90112;      // K-major B [80 rows][160]: 2 x 10K SW128 + 5K SW64
constexpr uint32_t kSmV = 116736;      // 3 x [128][64] bf16 SW128
constexpr uint32_t kSmOnes = 165888;   // [128][64] bf16 ones (the extra rows/columns of [V | 1])
constexpr uint32_t kSmQ = 182272;      // 3 x [128][16] bf16 SW32
constexpr uint32_t kSmK = 194560;      // 3 x [128][16] bf16 SW32
constexpr uint32_t kSmY = 206848;      // 4 x [32 rows][64] bf16 SW128: y staging for TMA stores
constexpr uint32_t kSmBar = kSmY + 16384;
// decay: [129] float2 (gamma^d, gamma^(d-1)), then at kPowInvOff [32] float2
// (gamma^-2j, gamma^-2j)
constexpr uint32_t kSmPow = kSmBar + 512;
constexpr uint32_t kPowInvOff = 1040;
constexpr uint32_t kSmTotal = kSmPow + kPowInvOff + 256;
constexpr uint32_t kSmAlloc = kSmTotal + 1024;
constexpr int kStages = 3;

// barrier indices
enum {
    B_QK_FULL = 0, B_QK_EMPTY = 3, B_V_FULL = 6, B_V_EMPTY = 9,
    B_T_FULL = 12,   // Q K^T of the chunk is in T
    // PV_READY(c): P(c) (P warps) and num drained after chunk c - 1 (y warps);
    // RO_READY(c): Phi'_Q(c) (gen warps) and the state operand after chunk c - 1
    // (conversion warps).  Merged so the MMA issuer waits once for each: its
    // waits are expensive after MMA issue.  With decay RO_READY(c) also covers
    // Phi'_K(c) (PHK_FULL is unused there): one wait fewer per chunk, which pays
    // in the decayed kernel, whose issuer is not its bottleneck, and not in
    // the plain one, where the update's operand lands after the read-out's.
    B_PV_READY = 14, B_RO_READY, B_PHK_FULL,
    B_NUM_FULL, B_S_FULL, B_FINAL,
    B_STAGED,   // the final state's value rows are in the shared-memory image
    B_COUNT
};
constexpr uint32_t kSmTmemSlot = kSmBar + 8 * B_COUNT;
constexpr uint32_t kSmAbort = kSmTmemSlot + 4;
static_assert(kSmAbort + 4 <= kSmTotal, "barrier area");
static_assert(kSmSb + 25600 <= kSmV && kSmV + 3 * 16384 == kSmOnes && kSmOnes + 16384 == kSmQ &&
              kSmQ + 3 * 4096 == kSmK && kSmK + 3 * 4096 == kSmY && kSmAlloc <= 232448, "smem map");

constexpr uint32_t kIdQK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdPV = idesc_bf16(128, kNB, false, true);   // P (TMEM) x [V | 1]
constexpr uint32_t kIdRO = idesc_bf16(128, kNB, false, false);  // Phi'_Q x [S' | z'] (K-major)
constexpr uint32_t kIdUp = idesc_bf16(128, kNFeat, true, true); // [V | 1]^T x Phi'_K

// Byte offset of 16-byte chunk j (features 8j..8j+7) of row d in the K-major
// [80][160] state operand.
__device__ __forceinline__ uint32_t sb_chunk_off(int d, int j) {
    if (j < 8) return (uint32_t)(d * 128 + ((j ^ (d & 7)) << 4));
    if (j < 16) return 10240u + (uint32_t)(d * 128 + (((j - 8) ^ (d & 7)) << 4));
    return 20480u + (uint32_t)(d * 64 + (((j - 16) ^ ((d >> 1) & 3)) << 4));
}

// Write 32 consecutive features (group g) of state row d as bf16.
__device__ __forceinline__ void write_sb_group(uint32_t sbase, int d, int g, const uint32_t (&r)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st_shared_v4(sbase + sb_chunk_off(d, 4 * g + q),
                     pack_bf16(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1])),
                     pack_bf16(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3])),
                     pack_bf16(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5])),
                     pack_bf16(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7])));
}

// bf16 operand rows of the state after a chunk, for one warp's TMEM lanes and
// feature groups [kG0, kG0 + kNG) (32 features each): value rows d < 64 and
// the z' row 64 (lane 0 of the warp owning lanes 64..95).
// With kDecay the fp32 state in TMEM is then multiplied by `decay` (gamma to
// the next chunk's length) for the next update, while the operand keeps the
// undecayed state that the next read-out needs.
template <int kG0, int kNG, bool kDecay = false>
__device__ __forceinline__ void convert_groups(uint32_t taddr, uint32_t sbase, int d, bool zrow, int lane,
                                               float decay = 1.f) {
    uint32_t r[32 * kNG];
    if constexpr (kNG == 2) {
        uint32_t (&r64)[64] = reinterpret_cast<uint32_t (&)[64]>(r);
        tmem_load64_sync(taddr + 32 * kG0, r64);
    } else {
        uint32_t (&r32)[32] = reinterpret_cast<uint32_t (&)[32]>(r);
        tmem_load32_sync(taddr + 32 * kG0, r32);
    }
    if (!zrow || lane == 0) {
#pragma unroll
        for (int g = 0; g < kNG; ++g)
            write_sb_group(sbase, zrow ? 64 : d, kG0 + g, *reinterpret_cast<const uint32_t (*)[32]>(r + 32 * g));
    }
    if constexpr (kDecay) {
        // rescaled in place and written back with one store and one wait
        __syncwarp();  // tcgen05.st is warp-collective
#pragma unroll
        for (int j = 0; j < 16 * kNG; ++j) {  // packed fp32x2 multiplies
            const uint64_t p = fmul2((uint64_t)r[2 * j] | ((uint64_t)r[2 * j + 1] << 32), f2pack(decay, decay));
            r[2 * j] = (uint32_t)p;
            r[2 * j + 1] = (uint32_t)(p >> 32);
        }
        if constexpr (kNG == 2)
            tmem_store64_sync(taddr + 32 * kG0, reinterpret_cast<const uint32_t (&)[64]>(r));
        else
            tmem_store32_sync(taddr + 32 * kG0, reinterpret_cast<const uint32_t (&)[32]>(r));
    }
}

// P = 1 + T/4 + T^2/32 for the keys 64 pp .. 64 pp + 63 of query row i (TMEM
// lane quarter w, 2 pp <= w), with the causal mask (key > i), left padding
// (key < kmin) and, with decay, the factor gamma^(i - key) from the tables at
// `pow` (powers gamma^d, and gamma^-2j at kPowInvOff).  Reads T at `tsrc` +
// 64 pp; once the previous chunk's P V has read the P buffer (phase `wpar` of
// the barrier `wbar`; wbar = 0: no wait) writes the 32 packed bf16 columns to
// `tdst`.  Returns false if that wait gave up.  Kept out of line: the warps
// that form P share one copy of this code (the kernel's roles together run
// more code than the instruction cache holds).
template <bool kPad, bool kDecay, int kDk = 16>
static __device__ __noinline__ bool p_block(uint32_t tsrc, uint32_t tdst, int pp, int i, int w, int kmin,
                                            uint32_t pow, uint32_t wbar, uint32_t wpar, volatile int *abort,
                                            unsigned *status) {
    uint32_t pw[32];
    {
        // K(q, k) = 1 + q.k / sqrt(d') + (q.k)^2 / (2 d')
        constexpr float kLin = kDk == 16 ? 0.25f : 0.35355339059327376f, kQuad = 1.0f / (2 * kDk);
        const uint64_t c32 = f2pack(kQuad, kQuad), c4 = f2pack(kLin, kLin), c1 = f2pack(1.0f, 1.0f);
        const bool diag = 64 * pp + 63 >= 32 * w;  // this block reaches the diagonal
        if constexpr (kDecay) {
            // times the decay factors gamma^(i-key) (key > i is masked below)
            uint32_t r[64];
            tmem_load64_sync(tsrc + 64 * pp, r);
            if (__uint_as_float((uint32_t)ld_shared_u64(pow + 8u)) >= 0.25f) {
                // separable within the block: gamma^(i-key) = gamma^(i-64pp) gamma^(-2j)
                // for the key pair 64pp + 2j, +1.  The row's factor scales the
                // polynomial's coefficients; the key's factor (warp-uniform, a
                // broadcast read, below 2^124 for gamma >= 1/4) multiplies P.
                const uint64_t a2 = ld_shared_u64(pow + 8u * (uint32_t)(i - 64 * pp));  // i >= 64 pp
                const uint64_t e1 = a2, e4 = fmul2(c4, a2), e32 = fmul2(c32, a2);
#pragma unroll
                for (int j2 = 0; j2 < 16; ++j2) {
                    const uint4 u = ld_shared_v4(pow + kPowInvOff + 16u * (uint32_t)j2);  // (gamma^-2j) x 2, j = 2 j2, +1
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 2 * j2 + h, key = 64 * pp + 2 * j;
                        const uint64_t uj = h ? ((uint64_t)u.z | ((uint64_t)u.w << 32))
                                              : ((uint64_t)u.x | ((uint64_t)u.y << 32));
                        const uint64_t t2 = (uint64_t)r[2 * j] | ((uint64_t)r[2 * j + 1] << 32);
                        const uint64_t p2 = fmul2(ffma2(t2, ffma2(t2, e32, e4), e1), uj);
                        float p0 = __uint_as_float((uint32_t)p2), p1 = __uint_as_float((uint32_t)(p2 >> 32));
                        if (diag) {
                            if (key > i) p0 = 0.f;
                            if (key + 1 > i) p1 = 0.f;
                        }
                        pw[j] = pack_bf16(p0, p1);
                    }
                }
            } else {
                // small rates: (gamma^(i-key), gamma^(i-key-1)) from the power table
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int key = 64 * pp + 2 * j;
                    const uint64_t t2 = (uint64_t)r[2 * j] | ((uint64_t)r[2 * j + 1] << 32);
                    const uint64_t f2 = ld_shared_u64(pow + 8u * (uint32_t)max(i - key, 0));
                    const uint64_t p2 = fmul2(ffma2(t2, ffma2(t2, c32, c4), c1), f2);
                    float p0 = __uint_as_float((uint32_t)p2), p1 = __uint_as_float((uint32_t)(p2 >> 32));
                    if (diag) {
                        if (key > i) p0 = 0.f;
                        if (key + 1 > i) p1 = 0.f;
                    }
                    pw[j] = pack_bf16(p0, p1);
                }
            }
        } else {
            uint32_t r[64];
            tmem_load64_sync(tsrc + 64 * pp, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint64_t t2 = (uint64_t)r[2 * j] | ((uint64_t)r[2 * j + 1] << 32);
                const uint64_t p2 = ffma2(t2, ffma2(t2, c32, c4), c1);
                float p0 = __uint_as_float((uint32_t)p2), p1 = __uint_as_float((uint32_t)(p2 >> 32));
                if (diag) {
                    const int key = 64 * pp + 2 * j;
                    if (key > i) p0 = 0.f;
                    if (key + 1 > i) p1 = 0.f;
                }
                pw[j] = pack_bf16(p0, p1);
            }
        }
        if (kPad && kmin > 64 * pp) {  // chunk holds left padding: drop padded keys
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int key = 64 * pp + 2 * j;
                if (key + 1 < kmin) pw[j] = 0u;
                else if (key < kmin) pw[j] &= 0xFFFF0000u;  // low half = the even key
            }
        }
    }
    if (wbar && !__all_sync(0xffffffffu, mbar_wait(wbar, wpar, abort, status))) return false;
    tmem_store32_sync(tdst, pw);
    return true;
}

// r[j] += sum over the nseg segments, in order, of part[seg * seg_stride +
// (32 G + j) * stride]: the prefix partial states (internal compact rows) of
// feature group G, for one value column (or z').  The 32 reads of a segment
// are issued together.
template <int G>
__device__ __forceinline__ void add_partials(const float *part, int64_t stride, int64_t seg_stride, int nseg,
                                             uint32_t (&r)[32]) {
#pragma unroll 1
    for (int sg = 0; sg < nseg; ++sg) {
        const float *p = part + sg * seg_stride + (32 * G) * stride;
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) a[j] = __ldcg(p + j * stride);
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + a[j]);
    }
}

// A head split in two pieces hands its state over through a transfer slot
// (kXferFloats floats): the first piece writes its final state there as it
// would to s_out (same layout: values, then z) and then publishes a flag word
// equal to the launch's call id; the second piece waits for it (bounded) and
// reads the slot as its initial state.
static_assert(kXferFloats >= kD * kDV + kD && kXferFloats % 4 == 0, "transfer slot");

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Bounded wait for *flag == v (about one second); on expiry the timeout is
// recorded and the CTA's abort flag set.
__device__ __forceinline__ bool wait_flag(const unsigned long long *flag, unsigned long long v,
                                          volatile int *abort, unsigned *status) {
    const long long t0 = clock64();
    while (ld_acquire_u64(flag) != v) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitCycles) {
            atomicOr(status, kStatusTimeout);
            *abort = 1;
            return false;
        }
        __nanosleep(256);
    }
    return true;
}

// Image of one head's final [273][64] fp32 state in shared memory, written
// out with a single bulk copy once the last update has completed (the
// feature-operand buffers it overlays are free by then).
constexpr uint32_t kSmStage = kSmPhiQ;
constexpr uint32_t kStageBytes = (uint32_t)kD * kDV * 4;
constexpr uint32_t kStageBytesCompact = (uint32_t)kDCompact * kDV * 4;  // the 153-row layout
static_assert(kSmStage + kStageBytes <= kSmSb, "final state image overlays Phi'_Q and Phi'_K only");

// Optional per-role timeline of CTA 0 (compile with -DLA_TRACE): SM clock
// offsets from kernel entry for events of each role and chunk.
#ifdef LA_TRACE
constexpr int kTraceChunks = 512;
__device__ uint32_t g_trace[5][kTraceChunks][8];
#define LA_TR(role, c, ev)                                                         \
    do {                                                                           \
        if (blockIdx.x == 0 && (c) < kTraceChunks)                                 \
            g_trace[role][c][ev] = (uint32_t)(clock64() - t_start);                \
    } while (0)
#else
#define LA_TR(role, c, ev) do { } while (0)
#endif
enum { TR_TMA = 0, TR_MMA, TR_GEN, TR_EPI, TR_CONV };

// kPad: the launch carries per-row left-padding counts; kDecay: a per-head
// decay gamma (s_i = gamma s_(i-1) + phi(k_i) v_i^T).  Separate instantiations,
// so the plain kernel carries none of their code.  With decay, token t of a
// chunk of length L reads gamma^(t+1) Phi'_Q . S (scaled query features),
// writes gamma^(L-1-t) Phi'_K (scaled key features), the intra-chunk kernel
// entries carry gamma^(i-j), and the state is multiplied by gamma^L in TMEM
// before each update.
template <bool kPad, bool kDecay, bool kCompact = false, bool kPrefix = false, int kDk = 16>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap ty,
                  const float *__restrict__ s0,
                  const float *__restrict__ z0, const int32_t *__restrict__ left_pad,
                  const float *__restrict__ gamma, int64_t H,
                  float *__restrict__ s_out, float *__restrict__ z_out, int N, float eps,
                  unsigned *status, const float *__restrict__ part_s, const float *__restrict__ part_z,
                  int nseg, int bh_total, int split_r, int split_n1, float *__restrict__ xfer,
                  unsigned long long *__restrict__ xflag, unsigned long long call_id) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) { return sb + kSmBar + 8u * (uint32_t)i; };
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kSmAbort);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef LA_TRACE
    const long long t_start = clock64();
#endif
    // Work of this CTA: a whole head, or a piece of one of the last split_r
    // heads, which are split at chunk split_n1.  Block order: split_r whole
    // heads, the split_r first pieces, the other whole heads, the split_r
    // second pieces (launch_prefill_tc explains the schedule).
    const int n_all = (N + kC - 1) / kC;
    int64_t bh_ = blockIdx.x;
    int c0_ = 0, n_ = n_all, piece_ = 0;  // piece 0: whole head, 1: first piece, 2: second piece
    if (split_r > 0) {
        const int b = blockIdx.x;
        if (b < split_r) {
        } else if (b < 2 * split_r) {
            bh_ = bh_total - split_r + (b - split_r);
            n_ = split_n1;
            piece_ = 1;
        } else if (b < bh_total) {
            bh_ = b - split_r;
        } else {
            bh_ = bh_total - split_r + (b - bh_total);
            c0_ = split_n1;
            n_ = n_all - split_n1;
            piece_ = 2;
        }
    }
    const int64_t bh = bh_;
    const int piece = piece_;
    // leading padding positions of this batch row: no contribution to any sum, y = 0
    const int lpad = kPad ? (int)row_left_pad(left_pad, bh / H, N, status, tid == 0) : 0;
    // chunks that lie entirely in the left padding add nothing to the state:
    // a CTA whose chunks start there skips them (keeping at least one chunk)
    // and only writes their y, as zeros (the y warps, before their loop)
    const int skip = kPad ? max(0, min(lpad / kC - c0_, n_ - 1)) : 0;
    const int c0 = c0_ + skip;  // first chunk of this CTA's work
    const int n = n_ - skip;    // chunks of this CTA's work
    float *xs = piece ? xfer + (bh - (bh_total - split_r)) * (int64_t)kXferFloats : nullptr;
    unsigned long long *xf = piece ? xflag + (bh - (bh_total - split_r)) : nullptr;
    // per-head columns of the state in memory (the 273-row layout, or with
    // kCompact the 153-row one): entry (row r, value d) at [r * 64 + d]
    constexpr int64_t kRowsIO = kCompact ? kDCompact : (kDk == 8 ? 73 : kD);
    // a second piece starts from the transfer slot (which holds s0 and, for
    // the prefix call, the prefix sum already); a first piece ends there
    const float *s0h = piece == 2 ? xs : (s0 ? s0 + bh * kRowsIO * kDV : nullptr);
    const float *z0h = piece == 2 ? xs + kRowsIO * kDV : (z0 ? z0 + bh * kRowsIO : nullptr);
    float *s_outh = piece == 1 ? xs : (s_out ? s_out + bh * kRowsIO * kDV : nullptr);
    float *z_outh = piece == 1 ? xs + kRowsIO * kDV : (z_out ? z_out + bh * kRowsIO : nullptr);

    // ---- set-up: barriers, TMEM, constant operands, feature -> row table
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_QK_FULL + s), 1);
            mbar_init(bar(B_QK_EMPTY + s), 4 + 1);  // gen warps read q, k; Q K^T of the chunk completed
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        mbar_init(bar(B_T_FULL), 1);
        // P warps 8..11, 2, 3; y warps (with decay the y warps write P of keys
        // 0..63 instead of warps 8..11)
        mbar_init(bar(B_PV_READY), (kDecay ? 2 : 6) + 4);
        // P warps; gen warps twice (Phi'_Q, conversion), with decay three times (+ Phi'_K)
        mbar_init(bar(B_RO_READY), 4 + (kDecay ? 12 : 8));
        mbar_init(bar(B_PHK_FULL), 4);
        mbar_init(bar(B_NUM_FULL), 1);
        mbar_init(bar(B_S_FULL), 1);
        mbar_init(bar(B_FINAL), 1);
        mbar_init(bar(B_STAGED), 4 + 4);  // P and gen warps
        *abort = 0;
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(sb + kSmTmemSlot, 512);
        tmem_relinquish();
    }
    for (int i = tid; i < 16384 / 16; i += kThreads)
        st_shared_v4(sb + kSmOnes + 16 * i, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    // rows 65..79 of the state operand stay zero (only the z' row 64 is used)
    for (int i = tid; i < 15 * 20; i += kThreads) {
        const int d = 65 + i / 20, j = i % 20;
        st_shared_v4(sb + kSmSb + sb_chunk_off(d, j), 0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kSmTmemSlot);

    // decay: the head's gamma (clamped to [0, 1]; out of range is reported) and
    // its powers (gamma^d, gamma^(d-1)) for d = 0..128
    auto pow_gamma = [&](int d) {
        return kDecay ? __uint_as_float((uint32_t)ld_shared_u64(sb + kSmPow + 8u * (uint32_t)d)) : 1.f;
    };
    if constexpr (kDecay) {
        float g = gamma[bh % H];
        if (!(g >= 0.f && g <= 1.f)) {
            if (tid == 0) atomicOr(status, kStatusBadDecay);
            g = (g > 1.f) ? 1.f : 0.f;
        }
        if (tid <= 128)
            reinterpret_cast<float2 *>(smem + kSmPow)[tid] =
                make_float2(powf(g, (float)tid), tid > 0 ? powf(g, (float)(tid - 1)) : 0.f);
        else if (tid >= 160 && tid < 192) {  // read only for gamma >= 1/4 (finite there)
            const float u = powf(g, -2.f * (float)(tid - 160));
            reinterpret_cast<float2 *>(smem + kSmPow + kPowInvOff)[tid - 160] = make_float2(u, u);
        }
        __syncthreads();
    }
    // length of chunk c (the last may be short)
    auto chunk_len = [&](int c) { return min(kC, N - (c0 + c) * kC); };
    // the antisymmetric part of the initial state bypasses the compact state: it
    // decays by gamma to the number of tokens this CTA covers (N for a whole
    // head; a split head's pieces hand it over through the transfer slot)
    const float anti_decay =
        kDecay ? powf(pow_gamma(1), (float)(min(N, (c0 + n) * kC) - c0 * kC)) : 1.f;

    // the first kStages chunks' loads (their stages start empty) go out now, so
    // that they land while the initial state is read; warp 3 has no state rows
    // (not in the decayed variant, whose registers are already tight)
    const int n_early = kDecay ? 0 : (n < kStages ? n : kStages);
    if (!kDecay && warp == 3 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        for (int c = 0; c < n_early; ++c) {
            mbar_expect_tx(bar(B_QK_FULL + c), 2 * kC * 16 * 2);
            tma_load_3d(sb + kSmQ + c * 4096, &tq, bar(B_QK_FULL + c), 0, (c0 + c) * kC, (int)bh);
            tma_load_3d(sb + kSmK + c * 4096, &tk, bar(B_QK_FULL + c), 0, (c0 + c) * kC, (int)bh);
            mbar_expect_tx(bar(B_V_FULL + c), kC * 64 * 2);
            tma_load_3d(sb + kSmV + c * 16384, &tv, bar(B_V_FULL + c), 0, (c0 + c) * kC, (int)bh);
        }
    }

    // initial state, before any role starts: S'^T rows (values d = 0..63, TMEM lane
    // quarters 0, 1) and z' (lane 64, quarter 2) in TMEM, and their bf16 operand
    // rows.  The 5 feature groups of each quarter are spread over the quarter's 4
    // warps (warp % 4 selects the quarter) so that their loads are in flight together.
    if ((warp & 3) < 3) {
        const int w = warp & 3;
        const int d = 32 * w + lane;
        const bool zrow = (w == 2);
        const uint32_t lanebase = (uint32_t)(32 * w) << 16;
        const float *col0 = zrow ? z0h : (s0h ? s0h + d : nullptr);
        const int64_t stride = zrow ? 1 : kDV;
        // a second piece waits until its first piece has handed its state over
        if (piece == 2) __all_sync(0xffffffffu, wait_flag(xf, call_id, abort, status));
        auto load_group = [&](auto gc) {
            constexpr int G = decltype(gc)::value;
            uint32_t r[32];
            if constexpr (kCompact)
                compact_io_initial_group<G>(col0, stride, r, std::make_integer_sequence<int, 32>{});
            else
                compact_initial_group<G, kDk>(col0, stride, r, std::make_integer_sequence<int, 32>{});
            if constexpr (kPrefix) {
                // + the prefix segments' partial states (internal compact rows), in
                // order; a second piece's slot holds them already
                const float *p = zrow ? part_z + bh * nseg * kNFeat : part_s + bh * nseg * kNFeat * kDV + d;
                add_partials<G>(p, stride, zrow ? kNFeat : kNFeat * kDV, piece == 2 ? 0 : nseg, r);
            }
            __syncwarp();
            if (!zrow || lane == 0) write_sb_group(sb + kSmSb, zrow ? 64 : d, G, r);
            if constexpr (kDecay) {  // the first update starts from gamma^L0 s0
                const float d0 = pow_gamma(chunk_len(0));
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * d0);
            }
            tmem_store32_sync(tmem + lanebase + kTmS + 32 * G, r);
        };
        switch (warp >> 2) {  // warps 0..2 take groups 0 and 4
            case 0:
                load_group(std::integral_constant<int, 0>{});
                load_group(std::integral_constant<int, 4>{});
                break;
            case 1: load_group(std::integral_constant<int, 1>{}); break;
            case 2: load_group(std::integral_constant<int, 2>{}); break;
            default: load_group(std::integral_constant<int, 3>{}); break;
        }
        fence_async_smem();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            if (kDecay) {
                prefetch_tmap(&tq);
                prefetch_tmap(&tk);
                prefetch_tmap(&tv);
            }
            int issued_qk = n_early, issued_v = n_early;
            for (int c = n_early; c < n; ++c) {
                const int st = c % kStages;
                const uint32_t ph = ((uint32_t)(c / kStages) & 1u) ^ 1u;
                if (!mbar_wait(bar(B_QK_EMPTY + st), ph, abort, status)) break;
                LA_TR(TR_TMA, c, 0);
                mbar_expect_tx(bar(B_QK_FULL + st), 2 * kC * 16 * 2);
                tma_load_3d(sb + kSmQ + st * 4096, &tq, bar(B_QK_FULL + st), 0, (c0 + c) * kC, (int)bh);
                tma_load_3d(sb + kSmK + st * 4096, &tk, bar(B_QK_FULL + st), 0, (c0 + c) * kC, (int)bh);
                issued_qk = c + 1;
                if (!mbar_wait(bar(B_V_EMPTY + st), ph, abort, status)) break;
                LA_TR(TR_TMA, c, 1);
                mbar_expect_tx(bar(B_V_FULL + st), kC * 64 * 2);
                tma_load_3d(sb + kSmV + st * 16384, &tv, bar(B_V_FULL + st), 0, (c0 + c) * kC, (int)bh);
                issued_v = c + 1;
                if (!kCompact && c == n - 1 && s0h && piece != 1) {
                    // the final state store reads s0 again (its antisymmetric part)
                    prefetch_l2_bulk(s0h, (uint32_t)kRowsIO * kDV * 4);
                    for (int o = 0; o < kRowsIO; o += 32) prefetch_l2(z0h + o);
                }
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
        // ================= MMA issuer (the whole warp; one elected lane issues) =================
        {
            // every wait's result is made warp-uniform so the warp stays converged
            auto wwait = [&](uint32_t b_, uint32_t par) {
                return __all_sync(0xffffffffu, mbar_wait(b_, par, abort, status));
            };
            // descriptor bases; per-step offsets are added in 16-byte units
            const uint64_t dQ = smem_desc(sb + kSmQ, 16, 256, kSw32);
            const uint64_t dK = smem_desc(sb + kSmK, 16, 256, kSw32);
            const uint64_t dSb = smem_desc(sb + kSmSb, 16, 1024, kSw128);
            const uint64_t dSb2 = smem_desc(sb + kSmSb + 20480, 16, 512, kSw64);
            const uint64_t dPhiK = smem_desc(sb + kSmPhiK, 16384, 1024, kSw128);
            // [V | 1]: V stage st plus the ones atom at a fixed distance past it;
            // the B operand of P V and (as MN-major A) of the state update
            const uint64_t dV0 = smem_desc(sb + kSmV, kSmOnes - kSmV, 1024, kSw128);
            auto dVst = [&](int st) {
                return dV0 + (uint64_t)(st * (16384 >> 4)) - ((uint64_t)(st * (16384 >> 4)) << 16);
            };
            auto issue_qk = [&](int c) {  // T = Q_c K_c^T
                const int st = c % kStages;
                mma_bf16_warp(tmem + kTmT, dQ + st * (4096 >> 4), dK + st * (4096 >> 4), kIdQK, 0);
                mma_commit_warp(bar(B_T_FULL));  // also frees the q, k stage (P epilogue forwards it)
            };
            bool ok = wwait(bar(B_QK_FULL + 0), 0);
            if (ok) {
                tc_fence_after();
                issue_qk(0);
            }
            for (int c = 0; ok && c < n; ++c) {
                const int vs = c % kStages;
                const uint64_t dV = dVst(vs);
                const uint32_t pc = (uint32_t)c & 1u;
                // P(c) is in the P buffer (so the P warps have read T, which may take
                // Q K^T(c + 1)); V(c) is in; num was drained for chunk c - 1; q, k of
                // c + 1 (PV_READY(c) also covers V(c) and q, k of chunk c + 1: a y warp
                // observes those loads before it arrives, sparing this thread the waits)
                ok = wwait(bar(B_PV_READY), pc);
                if (!ok) break;
                if (lane == 0) LA_TR(TR_MMA, c, 0);
                tc_fence_after();
                if (c + 1 < n) issue_qk(c + 1);
                if (lane == 0) LA_TR(TR_MMA, c, 1);
                // intra-chunk: [num | den] = P [V | 1], P from TMEM (keys 16 s.. in
                // packed columns 8 s..)
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16_ts_warp(tmem + kTmNum, tmem + kTmP + 8 * s, dV + s * (2048 >> 4), kIdPV, s > 0);
                // inter-chunk read-out operands: the state after chunk c - 1, Phi'_Q(c)
                ok = wwait(bar(B_RO_READY), pc);
                if (!ok) break;
                if (lane == 0) LA_TR(TR_MMA, c, 2);
                tc_fence_after();
                // inter-chunk read-out: [num | den] += Phi'_Q [S' | z'], Phi'_Q from TMEM
                // (features 16 s.. in columns 8 s..), the state K-major in shared memory
#pragma unroll
                for (int s = 0; s < 10; ++s) {
                    const uint64_t db = s < 8 ? dSb + ((uint32_t)((s >> 2) * 10240 + (s & 3) * 32) >> 4)
                                              : dSb2 + ((uint32_t)((s - 8) * 32) >> 4);
                    mma_bf16_ts_warp(tmem + kTmNum, tmem + kTmPhiQ + 8 * s, db, kIdRO, 1);
                }
                mma_commit_warp(bar(B_NUM_FULL));  // also: Phi'_Q and the P buffer free
                // state update operand Phi'_K(c) (with decay part of RO_READY(c))
                if (!kDecay && !(ok = wwait(bar(B_PHK_FULL), pc))) break;
                if (lane == 0) LA_TR(TR_MMA, c, 3);
                tc_fence_after();
                // state update: [S'^T ; z'] += [V | 1]^T Phi'_K, 16 tokens per MMA
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16_warp(tmem + kTmS, dV + s * (2048 >> 4), dPhiK + s * (2048 >> 4), kIdUp, 1);
                mma_commit_warp(bar(B_S_FULL));  // also: Phi'_K and V(c) buffers free (gen forwards the latter)
                if (lane == 0) LA_TR(TR_MMA, c, 4);
            }
            // every issued MMA must finish before TMEM is released
            __syncwarp();
            mma_commit_warp(bar(B_FINAL));
            drain_wait(bar(B_FINAL), 0);
        }
    } else if (warp == 2 || warp == 3) {
        // ================= P epilogue, keys 64..127 of the rows of lane quarter 2 or 3 =================
        // (rows 64..127 see up to 128 keys; the P warps 10, 11 take keys 0..63)
        const int w = warp;
        const int i = 32 * w + lane;
        const uint32_t lanebase = (uint32_t)(32 * w) << 16;
        const int kmin = kPad ? lpad : 0;
        for (int c = 0; c < n; ++c) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_T_FULL), (uint32_t)c & 1u, abort, status))) break;
            tc_fence_after();
            // P V of chunk c - 1 completed with the read-out (NUM_FULL(c - 1))
            if (!p_block<kPad, kDecay, kDk>(tmem + lanebase + kTmT, tmem + lanebase + kTmP + 32, 1, i, w,
                                       kmin - (c0 + c) * kC,
                                       sb + kSmPow, c > 0 ? bar(B_NUM_FULL) : 0u, (uint32_t)(c - 1) & 1u, abort,
                                       status))
                break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PV_READY));
        }
    } else if (warp >= 4 && warp < 8) {
        // ================= feature generation (one token per thread) =================
        // and the conversion of state feature groups 3, 4 after each update
        const int t = tid - 128;
        const int wq = warp - 4;                        // TMEM lane quarter of this warp
        const uint32_t lanebase = (uint32_t)(32 * wq) << 16;
        const bool zrow = (wq == 2);                    // lane 64 holds z'
        if (lane == 0) mbar_arrive(bar(B_RO_READY));  // phase 0: initial operand written in set-up
        bool gen_done = false;
        for (int c = 0; c < n; ++c) {
            const int st = c % kStages;
            const uint32_t pc = (uint32_t)c & 1u;
            if (!mbar_wait(bar(B_QK_FULL + st), (uint32_t)(c / kStages) & 1u, abort, status)) break;
            if (tid == 128) LA_TR(TR_GEN, c, 0);
            uint4 qlo, qhi, klo, khi;
            load_row16_raw(sb + kSmQ + st * 4096, t, qlo, qhi);
            load_row16_raw(sb + kSmK + st * 4096, t, klo, khi);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_QK_EMPTY + st));
            // the read-out of chunk c - 1 (NUM_FULL) released Phi'_Q; it goes into this
            // thread's TMEM lane (token t), the read-out's A operand
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_NUM_FULL), pc ^ 1u, abort, status))) break;
            tc_fence_after();
            if constexpr (kDecay) {  // token t reads gamma^(t+1) of the state before the chunk
                const float lq = pow_gamma(t + 1);
                emit_features_tmem<false, true, kDk>(qlo, qhi, tmem + lanebase + kTmPhiQ,
                                                std::make_integer_sequence<int, 5>{}, pack_bf16(lq, lq));
            } else {
                emit_features_tmem<false, false, kDk>(qlo, qhi, tmem + lanebase + kTmPhiQ,
                                                      std::make_integer_sequence<int, 5>{});
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_RO_READY));
            if (tid == 128) LA_TR(TR_GEN, c, 1);
            // past the end or left padding: no contribution to S', z'
            bool pad = (c0 + c) * kC + t >= N;
            if constexpr (kPad) pad = pad || (c0 + c) * kC + t < lpad;
            // the update of chunk c - 1 (S_FULL) released the Phi'_K buffer and V(c - 1)
            if (!mbar_wait(bar(B_S_FULL), pc ^ 1u, abort, status)) break;
            if (c > 0 && tid == 128) LA_TR(TR_CONV, c - 1, 2);
            if (c > 0 && tid == 128) mbar_arrive(bar(B_V_EMPTY + (c - 1) % kStages));
            if (c > 0) {
                // state after chunk c - 1, feature groups 3, 4 (with decay only 4: the
                // rescale would hold up the key features below) -> operand of the
                // read-out of c
                __syncwarp();
                tc_fence_after();
                if constexpr (!kDecay)
                    if (wq < 3)
                        convert_groups<3, 2, false>(tmem + lanebase + kTmS, sb + kSmSb, 32 * wq + lane, zrow, lane);
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_RO_READY));
            }
            if (tid == 128) LA_TR(TR_GEN, c, 2);
            if constexpr (kDecay) {  // token t enters the state after the chunk with gamma^(L-1-t)
                const float lk = pow_gamma(max(chunk_len(c) - 1 - t, 0));
                emit_features<true, true, kDk>(klo, khi, sb + kSmPhiK, t, pad, std::make_integer_sequence<int, 20>{},
                                          pack_bf16(lk, lk));
            } else {
                emit_features<true, false, kDk>(klo, khi, sb + kSmPhiK, t, pad, std::make_integer_sequence<int, 20>{});
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kDecay ? B_RO_READY : B_PHK_FULL));
            if (tid == 128) LA_TR(TR_GEN, c, 3);
            if (c == n - 1) gen_done = true;
        }
        // final state, feature groups 3, 4, once the last update completed (the
        // loop observed every earlier update phase in order)
        if (gen_done && mbar_wait(bar(B_S_FULL), (uint32_t)(n - 1) & 1u, abort, status)) {
            __syncwarp();
            tc_fence_after();
            if (tid == 128) LA_TR(TR_CONV, n - 1, 4);
            if (wq < 3) {
                if constexpr (kCompact)
                    final_groups_compact<true, 3>(tmem + lanebase + kTmS, 32 * wq + lane, zrow, lane,
                                                  sb + kSmStage, s_outh, z_outh, std::make_integer_sequence<int, 2>{});
                else
                    final_groups<true, 3, kDk>(tmem + lanebase + kTmS, 32 * wq + lane, zrow, lane, s0h, sb + kSmStage,
                                          s_outh, z0h, z_outh, anti_decay, std::make_integer_sequence<int, 2>{});
            }
            fence_async_smem();
            if (piece == 1) __threadfence();  // the z' row, before the hand-over flag
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_STAGED));
            // every value row is in the image: one bulk copy to s_out (a first
            // piece: to its transfer slot, then the hand-over flag)
            if (tid == 128 && s_outh && mbar_wait(bar(B_STAGED), 0u, abort, status)) {
                bulk_store(s_outh, sb + kSmStage, kCompact ? kStageBytesCompact : (uint32_t)kRowsIO * kDV * 4);
                bulk_commit();
                bulk_wait0();
                if (piece == 1) {
                    __threadfence();
                    st_release_u64(xf, call_id);
                }
            }
            if (tid == 128) LA_TR(TR_CONV, n - 1, 5);
        }
    } else if (warp >= 8 && warp < 12) {
        // ================= P epilogue: P = 1 + T/4 + T^2/32, causal, in place =================
        const int w = warp - 8;
        const int i = tid - 256;  // query row within the chunk (= TMEM lane)
        const uint32_t lanebase = (uint32_t)(32 * w) << 16;
        const bool zrow = (w == 2);  // warp 10: lane 64 holds z'
        // rows 0..63 see no key of 64..127: their P columns 32..63 stay zero
        // (with decay the y warps write them, before their first arrival)
        if (!kDecay && w < 2) {
            uint32_t zero[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) zero[j] = 0u;
            tmem_store32_sync(tmem + lanebase + kTmP + 32, zero);
        }
        auto do_p = [&](int c) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_T_FULL), (uint32_t)c & 1u, abort, status))) return false;
            if (tid == 256) mbar_arrive(bar(B_QK_EMPTY + c % kStages));  // Q K^T(c) has read its q, k stage
            if (tid == 256 + 96) LA_TR(TR_EPI, c, 0);
            tc_fence_after();
            const int kmin = kPad ? lpad - (c0 + c) * kC : 0;  // keys below kmin are left padding
            // keys 0..63 -> P columns 0..31; keys 64..127 of lane quarters 2, 3 are
            // warps 2, 3's share (P columns 32..63).  The store waits until P V of
            // chunk c - 1 has completed (NUM_FULL(c - 1)).
            if (!p_block<kPad, kDecay, kDk>(tmem + lanebase + kTmT, tmem + lanebase + kTmP, 0, i, w, kmin, sb + kSmPow,
                                       c > 0 ? bar(B_NUM_FULL) : 0u, (uint32_t)(c - 1) & 1u, abort, status))
                return false;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PV_READY));
            if (tid == 256 + 96) LA_TR(TR_EPI, c, 1);
            return true;
        };
        // After P(c + 1) (done well before the update of chunk c completes), the
        // state after chunk c, feature groups 0..2: the operand of the read-out of
        // chunk c + 1, or the final state (groups 3, 4: gen warps).
        // (With decay the y warps take the P blocks: these warps only convert.)
        if (lane == 0) mbar_arrive(bar(B_RO_READY));  // phase 0: initial operand written in set-up
        bool ok = kDecay ? true : do_p(0);
        for (int c = 0; ok && c < n; ++c) {
            if (!kDecay && c + 1 < n && !(ok = do_p(c + 1))) break;
            if (!(ok = mbar_wait(bar(B_S_FULL), (uint32_t)c & 1u, abort, status))) break;
            if (tid == 256) LA_TR(TR_CONV, c, 0);
            __syncwarp();
            tc_fence_after();
            const bool last = (c == n - 1);
            if (w < 3) {
                if (!last) {
                    const float dn = pow_gamma(chunk_len(c + 1));
                    convert_groups<0, 2, kDecay>(tmem + lanebase + kTmS, sb + kSmSb, i, zrow, lane, dn);
                    __syncwarp();
                    if constexpr (kDecay) {  // with decay these warps convert every group
                        convert_groups<2, 1, true>(tmem + lanebase + kTmS, sb + kSmSb, i, zrow, lane, dn);
                        __syncwarp();
                        convert_groups<3, 1, true>(tmem + lanebase + kTmS, sb + kSmSb, i, zrow, lane, dn);
                        __syncwarp();
                        convert_groups<4, 1, true>(tmem + lanebase + kTmS, sb + kSmSb, i, zrow, lane, dn);
                    } else
                        convert_groups<2, 1, false>(tmem + lanebase + kTmS, sb + kSmSb, i, zrow, lane, dn);
                } else if constexpr (kCompact) {
                    final_groups_compact<true, 0>(tmem + lanebase + kTmS, i, zrow, lane, sb + kSmStage, s_outh,
                                                  z_outh, std::make_integer_sequence<int, 3>{});
                } else {
                    final_groups<true, 0, kDk>(tmem + lanebase + kTmS, i, zrow, lane, s0h, sb + kSmStage, s_outh, z0h,
                                          z_outh, anti_decay, std::make_integer_sequence<int, 3>{});
                }
                __syncwarp();
            }
            if (last) {
                fence_async_smem();
                if (piece == 1) __threadfence();  // the z' row, before the hand-over flag
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_STAGED));
            } else {
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_RO_READY));
            }
            if (tid == 256) LA_TR(TR_CONV, c, 1);
        }
    } else if (warp >= 12) {
        // ========== output epilogue y = num / den ==========
        const int w = warp - 12;
        const int i = 32 * w + lane;          // query row (num lane)
        const uint32_t lanebase = (uint32_t)(32 * w) << 16;
        if constexpr (kPad) {
            if (skip > 0) {  // y of the skipped (fully padded) chunks: zero tiles of this warp's 32 rows
                const uint32_t stage = sb + kSmY + (uint32_t)w * 4096;
                for (int j = lane; j < 4096 / 16; j += 32) st_shared_v4(stage + 16u * (uint32_t)j, 0u, 0u, 0u, 0u);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    for (int c = c0 - skip; c < c0; ++c)
                        if (c * kC + 32 * w < N) tma_store_3d(&ty, stage, 0, c * kC + 32 * w, (int)bh);
                    bulk_commit();  // the loop's first bulk_wait_read0 covers these reads of the tile
                }
                __syncwarp();
            }
        }
        // PV_READY(c) from the y warps: num drained after chunk c - 1, and (one
        // lane) the loads P V(c) and Q K^T(c + 1) read.  The lane observes those
        // loads before it waits for the numerator (they have landed long before),
        // so that the numerator drain alone sits on the path to the next P V.
        auto observe = [&](int c) -> bool {
            return tid != 384 || c >= n ||
                   (mbar_wait(bar(B_V_FULL + c % kStages), (uint32_t)(c / kStages) & 1u, abort, status) &&
                    (c + 1 >= n || mbar_wait(bar(B_QK_FULL + (c + 1) % kStages), (uint32_t)((c + 1) / kStages) & 1u,
                                             abort, status)));
        };
        // With decay these warps also form P of keys 0..63 for their rows (the
        // P warps' role without decay): P(c + 1) once Q K^T(c + 1) is in T, stored
        // once P V(c) has completed (NUM_FULL(c)), before num(c) is drained, so
        // that one arrival covers both.
        auto p_next = [&](int c) -> bool {  // P(c)
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_T_FULL), (uint32_t)c & 1u, abort, status))) return false;
            if (tid == 384) mbar_arrive(bar(B_QK_EMPTY + c % kStages));  // Q K^T(c) has read its q, k stage
            tc_fence_after();
            return p_block<kPad, kDecay, kDk>(tmem + lanebase + kTmT, tmem + lanebase + kTmP, 0, i, w,
                                              kPad ? lpad - (c0 + c) * kC : 0, sb + kSmPow,
                                              c > 0 ? bar(B_NUM_FULL) : 0u, (uint32_t)(c - 1) & 1u, abort, status);
        };
        bool ok = __all_sync(0xffffffffu, observe(0));
        if constexpr (kDecay) {
            if (w < 2) {  // rows 0..63 see no key of 64..127: their P columns 32..63 stay zero
                uint32_t zero[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) zero[j] = 0u;
                tmem_store32_sync(tmem + lanebase + kTmP + 32, zero);
            }
            ok = ok && p_next(0);
            tc_fence_before();
            __syncwarp();
        }
        if (ok && lane == 0) mbar_arrive(bar(B_PV_READY));  // phase 0: num starts drained (with decay: P(0))
        for (int c = 0; ok && c < n; ++c) {
            // ---- y(c)
            const bool seen = observe(c + 1);
            if constexpr (kDecay)
                if (c + 1 < n && !p_next(c + 1)) break;
            if (!mbar_wait(bar(B_NUM_FULL), (uint32_t)c & 1u, abort, status)) break;
            if (tid == 384) LA_TR(TR_EPI, c, 2);
            __syncwarp();
            tc_fence_after();
            {
                uint32_t r[64], dr;
                tmem_load64_1_sync(tmem + lanebase + kTmNum, 64, r, dr);
                tc_fence_before();
                __syncwarp();
                ok = __all_sync(0xffffffffu, seen);  // warp-uniform result
                if (ok && lane == 0) mbar_arrive(bar(B_PV_READY));  // num of chunk c drained
                // y rows of this warp -> its 4 KB staging tile -> one bulk tensor store
                // (rows past N are clipped by the store)
                float inv = 1.0f / (__uint_as_float(dr) + eps);
                if constexpr (kPad)
                    if ((c0 + c) * kC + i < lpad) inv = 0.f;  // padded query rows (left padding) output 0
                const uint64_t inv2 = f2pack(inv, inv);
                const uint32_t stage = sb + kSmY + (uint32_t)w * 4096;
                if (lane == 0) bulk_wait_read0();  // previous chunk's store has read the tile
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t o[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        o[h] = pack_bf16x2(fmul2((uint64_t)r[8 * j + 2 * h] | ((uint64_t)r[8 * j + 2 * h + 1] << 32),
                                                 inv2));
                    st_shared_v4(stage + lane * 128 + ((j ^ (lane & 7)) << 4), o[0], o[1], o[2], o[3]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0 && (c0 + c) * kC + 32 * w < N) {
                    tma_store_3d(&ty, stage, 0, (c0 + c) * kC + 32 * w, (int)bh);
                    bulk_commit();
                }
            }
            if (tid == 384) LA_TR(TR_EPI, c, 3);
        }
        if (tid == 384) LA_TR(TR_CONV, n - 1, 6);
        if (lane == 0) bulk_wait0();  // y stores complete before the CTA exits
        if (tid == 384) LA_TR(TR_CONV, n - 1, 7);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();  // lane 0 ran the producer loop alone; dealloc is warp-collective
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

#ifdef LA_TRACE
}  // namespace
extern "C" LA_API int la_debug_prefill_trace(void *host, size_t bytes) {
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    return (int)cudaMemcpyFromSymbol(host, g_trace, bytes);
}
namespace {
#endif

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
                   bool swizzle128, int box_rows, int box_width) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)N * width * 2};
    const cuuint32_t box[3] = {(cuuint32_t)(box_width ? box_width : width), (cuuint32_t)box_rows, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t st) {
    const int64_t BH = a.B * a.H;
    if (a.N > (int64_t)0x7FFFFFFF - kC) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv, ty;
    // d' = 8: the q, k rows are 8 wide; the box reads 16 columns, the upper 8
    // out of bounds and so zero (the padded rows of the d' = 16 map)
    if (a.dk != 16 && a.dk != 8) return cudaErrorInvalidValue;
    if (!make_row_tmap(&tq, a.q, BH, a.N, a.dk, false, 128, 16) ||
        !make_row_tmap(&tk, a.k, BH, a.N, a.dk, false, 128, 16) ||
        !make_row_tmap(&tv, a.v, BH, a.N, 64, true) || !make_row_tmap(&ty, a.y, BH, a.N, 64, true, 32))
        return cudaErrorInvalidValue;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<false, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<false, false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<false, false, false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<true, false, false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<false, false, false, false, 8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e != cudaSuccess) return e;
        configured_for = dev;
    }
    if (a.left_pad && a.gamma) return cudaErrorInvalidValue;  // no padded decayed variant
    if (a.compact && (a.left_pad || a.gamma)) return cudaErrorInvalidValue;  // plain prefill only
    const bool prefix = a.part_s != nullptr;
    if (prefix && (a.gamma || a.compact || a.nseg < 1 || a.nseg > 65535)) return cudaErrorInvalidValue;
    const int nseg = (int)a.nseg;
    // split heads (see the schedule above): grid = BH + split_r
    const int r = a.split_r;
    if (r < 0 || (r > 0 && (!a.xfer || !a.xflag || 2 * (int64_t)r > BH || a.split_n1 < 1 ||
                            a.split_n1 >= (a.N + kC - 1) / kC)))
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)(BH + r);
#define LA_PREFILL_ARGS                                                                                    \
    tq, tk, tv, ty, a.s0, a.z0, a.left_pad, a.gamma, a.H, a.s_out, a.z_out, (int)a.N, a.eps, a.status, a.part_s, \
        a.part_z, nseg, (int)BH, r, a.split_n1, a.xfer, a.xflag, a.call_id
    // d' = 8: the plain prefill only (padding, decay, the prefix and the compact
    // state exist for d' = 16)
    if (a.dk == 8 && (prefix || a.compact || a.left_pad || a.gamma)) return cudaErrorInvalidValue;
    if (a.dk == 8)
        prefill_tc_kernel<false, false, false, false, 8><<<grid, kThreads, kSmAlloc, st>>>(LA_PREFILL_ARGS);
    else if (prefix && a.left_pad)
        prefill_tc_kernel<true, false, false, true><<<grid, kThreads, kSmAlloc, st>>>(LA_PREFILL_ARGS);
    else if (prefix)
        prefill_tc_kernel<false, false, false, true><<<grid, kThreads, kSmAlloc, st>>>(LA_PREFILL_ARGS);
    else if (a.compact)
        prefill_tc_kernel<false, false, true><<<grid, kThreads, kSmAlloc, st>>>(LA_PREFILL_ARGS);
    else if (a.left_pad)
        prefill_tc_kernel<true, false><<<grid, kThreads, kSmAlloc, st>>>(LA_PREFILL_ARGS);
    else if (a.gamma)
        prefill_tc_kernel<false, true><<<grid, kThreads, kSmAlloc, st>>>(LA_PREFILL_ARGS);
    else
        prefill_tc_kernel<false, false><<<grid, kThreads, kSmAlloc, st>>>(LA_PREFILL_ARGS);
#undef LA_PREFILL_ARGS
    return cudaGetLastError();
}

}  // namespace la
