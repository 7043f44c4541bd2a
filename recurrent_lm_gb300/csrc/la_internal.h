// Internal interface between the C-ABI layer (la_api.cu) and the kernel
// translation units.  Launchers assume their arguments were validated by the
// ABI layer and return the cudaError_t of the launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "linattn.h"

namespace la {

constexpr int kDFeat = 16;     // d'
constexpr int kDV = 64;        // d_v
constexpr int kD = 273;        // 1 + d' + d'^2
constexpr int kStateFloats = kD * kDV + kD;  // one head's s and z

// Bits of the device status word (one per failure class).
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBadPad = 2u;   // a left-padding count outside [0, N] (clamped)
constexpr unsigned kStatusBadDecay = 4u; // a decay rate outside [0, 1] (clamped)

// Leading padding positions of batch row b: left_pad[b] clamped to [0, N]
// (NULL: none).  An out-of-range count sets kStatusBadPad (by one thread).
__device__ __forceinline__ int64_t row_left_pad(const int32_t *left_pad, int64_t b, int64_t N,
                                                unsigned *status, bool report) {
    if (!left_pad) return 0;
    const int64_t p = left_pad[b];
    if (p < 0 || p > N) {
        if (report) atomicOr(status, kStatusBadPad);
        return p < 0 ? 0 : N;
    }
    return p;
}

struct PrefillArgs {
    const void *q, *k, *v;
    const float *s0, *z0;
    void *y;
    float *s_out, *z_out;
    int64_t B, H, N;
    float eps;
    unsigned *status;   // device status word
    const int32_t *left_pad;  // [B] leading padding positions per batch row, or NULL
    const float *gamma;       // [H] per-head decay in [0, 1], or NULL (no decay)
    bool compact = false;     // s0/z0 and s_out/z_out in the 153-row compact layout
    int dk = 16;              // d' (the tensor-core path: 16, or 8 on the padded map)
    // Prefix partial states added, segment by segment in order, to the initial
    // state (NULL: none): the bf16 tensor-core path reads its internal compact
    // rows, part_s [BH][nseg][160][64] and part_z [BH][nseg][160]; the fp32
    // path the 273-row ones, part_s [BH][nseg][273][64] and part_z [BH][nseg][273].
    const float *part_s = nullptr, *part_z = nullptr;
    int64_t nseg = 0;
    // Split heads (bf16 tensor-core path): the last split_r heads run as two
    // pieces, chunks [0, split_n1) and [split_n1, n); the first hands its state
    // to the second through xfer ([split_r][kXferFloats] fp32) and the flag
    // words xflag ([split_r], set to call_id).  split_r = 0: no split.
    int split_r = 0, split_n1 = 0;
    float *xfer = nullptr;
    unsigned long long *xflag = nullptr;
    unsigned long long call_id = 0;
};

struct DecodeArgs {
    const void *q, *k, *v;
    const float *s_in, *z_in;
    float *s_out, *z_out;
    void *y;
    int64_t B, H;
    float eps;
    const float *gamma;       // [H] per-head decay in [0, 1], or NULL (no decay)
    unsigned *status;
};

// Per-segment partial prefix states (fp32), in the layouts PrefillArgs
// describes; the prefill adds them to its initial state.
struct PrefixArgs {
    const void *k_e, *v_e;
    int64_t B, H, M;
    int64_t seg_len, nseg;
    float *part_s, *part_z;
    unsigned *status;
    const int32_t *left_pad;  // [B]: prefix positions j < min(left_pad[b], M) are padding
    int64_t N;                // causal length (the range of left_pad)
};

// Smallest workspace la_prefix_prefill accepts (the prefix partial states
// only; la_prefix_workspace_size adds the split heads' hand-over region).
size_t prefix_workspace_min(int64_t B, int64_t H, int64_t M);

// One transfer slot of a split head: a state in the layout of s0 / s_out
// ([273][64] values, then [273] z, fp32; or the 153-row compact layout),
// padded to a multiple of 16 bytes.
constexpr int kXferFloats = (kD * kDV + kD + 3) / 4 * 4;

// Split of the M prefix tokens into segments, one CTA each: enough segments
// for about 256 CTAs over all (b, h) (at most 16 per head, at least one
// 128-token chunk each), segment length a multiple of 128.
struct PrefixSplit {
    int64_t seg_len, nseg;
};
inline PrefixSplit prefix_split(int64_t BH, int64_t M) {
    if (M <= 0 || BH <= 0) return {0, 0};
    int64_t n = (256 + BH - 1) / BH;
    if (n > 16) n = 16;
    const int64_t chunks = (M + 127) / 128;
    if (n > chunks) n = chunks;
    const int64_t seg_len = (M + n - 1) / n;
    const int64_t seg = (seg_len + 127) / 128 * 128;
    return {seg, (M + seg - 1) / seg};
}

// Feature dimensions d' with a kernel: 16 (tensor-core and CUDA-core paths)
// and 8, 24, 32 (the general CUDA-core path).  D = 1 + d' + d'^2.
inline bool supported_dk(int dk) { return dk == 8 || dk == 16 || dk == 24 || dk == 32; }
inline int64_t feat_dim(int dk) { return 1 + (int64_t)dk + (int64_t)dk * dk; }
cudaError_t launch_prefill_general(const PrefillArgs &a, int dk, la_dtype dt, cudaStream_t st);
// d' = 24, 32 with bf16 activations on the tensor cores (cuBLASLt batched GEMMs
// and this library's kernels), in a workspace of general_tc_workspace bytes
// (0 for other d' or N = 0).
size_t general_tc_workspace(int64_t BH, int64_t N, int dk);
cudaError_t launch_prefill_general_tc(const PrefillArgs &a, int dk, void *workspace, cudaStream_t st);
cudaError_t launch_decode_general(const DecodeArgs &a, int dk, la_dtype dt, cudaStream_t st);

cudaError_t launch_decode(const DecodeArgs &a, la_dtype dt, cudaStream_t st);
cudaError_t launch_prefill_simt(const PrefillArgs &a, la_dtype dt, cudaStream_t st);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t st);
cudaError_t launch_prefix_partials_simt(const PrefixArgs &a, la_dtype dt, cudaStream_t st);
cudaError_t launch_prefix_partials_tc(const PrefixArgs &a, cudaStream_t st);
cudaError_t launch_state_copy(int64_t D, const float *s0, const float *z0, float *s_out,
                              float *z_out, int64_t BH, cudaStream_t st);
cudaError_t launch_timeout_probe(unsigned *status, cudaStream_t st);

// Compact state layout (d' = 16): 153 rows, see linattn.h.
constexpr int kDCompact = 153;
cudaError_t launch_decode_compact(const DecodeArgs &a, la_dtype dt, cudaStream_t st);
cudaError_t launch_state_to_compact(const float *s, const float *z, float *s_c, float *z_c, int64_t BH,
                                    cudaStream_t st);
cudaError_t launch_state_from_compact(const float *s_c, const float *z_c, float *s, float *z, int64_t BH,
                                      cudaStream_t st);

}  // namespace la
