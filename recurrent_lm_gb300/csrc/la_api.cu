// C-ABI layer of liblinattn.so: argument validation on the host, workspace
// carving, and dispatch to the kernel launchers.  Nothing is launched unless
// every argument check passes.  See include/linattn.h for the contract.
#include <atomic>
#include <mutex>

#include "la_internal.h"

namespace {

using la::kD;
using la::kDV;
using la::kDFeat;

__device__ unsigned g_la_status = 0;

constexpr int kMaxDevices = 64;
unsigned *g_status_ptr[kMaxDevices] = {};
int g_cc[kMaxDevices] = {};  // major*10+minor, 0 = not queried yet
int g_sms[kMaxDevices] = {};  // multiprocessor count
std::mutex g_mu;
std::atomic<unsigned long long> g_call_id{1};  // flag value of split heads' state hand-over

// Per-device set-up: compute capability and the status word's address.
la_status device_setup(int *dev_out, unsigned **status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cc[dev] == 0) {
        int major = 0, minor = 0;
        int sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return LA_ERR_CUDA;
        g_sms[dev] = sms;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_la_status) != cudaSuccess) return LA_ERR_CUDA;
        g_status_ptr[dev] = static_cast<unsigned *>(p);
        g_cc[dev] = major * 10 + minor;
    }
    if (g_cc[dev] != 103) return LA_ERR_UNSUPPORTED;  // kernels are built for sm_103a only
    *dev_out = dev;
    *status = g_status_ptr[dev];
    return LA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    const void *p;
    size_t bytes;
};

bool overlaps(Range a, Range b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Checks that no output range overlaps any input range or another output.
bool any_overlap(const Range *in, int nin, const Range *out, int nout) {
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlaps(out[i], in[j])) return true;
        for (int j = i + 1; j < nout; ++j)
            if (overlaps(out[i], out[j])) return true;
    }
    return false;
}

// Shape limits: every grid dimension used is (B*H) or segments; element
// counts are 64-bit everywhere in the kernels.
constexpr int64_t kMaxBH = (int64_t(1) << 31) - 1;
constexpr int64_t kMaxTokens = int64_t(1) << 40;

la_status check_common(int64_t B, int64_t H, int64_t N, int d_feat, int d_v, la_dtype dtype) {
    if (!la::supported_dk(d_feat) || d_v != kDV) return LA_ERR_UNSUPPORTED;
    if (dtype != LA_DTYPE_F32 && dtype != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || N < 0) return LA_ERR_INVALID_ARG;
    if (B > kMaxBH / H) return LA_ERR_INVALID_ARG;
    if (N > kMaxTokens / (B * H)) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

size_t esize(la_dtype dt) { return dt == LA_DTYPE_BF16 ? 2 : 4; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Split heads of the bf16 prefill.  One CTA per head and per SM, so B*H heads
// run in W = ceil(B*H / SMs) waves, the last with r heads and SMs - r idle
// SMs.  The r heads of the last wave are split at chunk n1 into a first piece
// (chunks [0, n1)) and a second piece (the rest), and the block order is
//   r whole heads, r first pieces, the other whole heads, r second pieces.
// So r SMs run whole heads and then a second piece, and the other SMs run
// k = ceil(r / (SMs - r)) first pieces before their whole heads; the first
// pieces are done long before the second pieces start (blocks are dispatched
// in order).  n1 balances the two kinds of SM, counting f chunk times of fixed
// cost per CTA (set-up and final state): n - n1 + f = k (n1 + f).  f = 16 was
// measured best (f = 6 / 10 / 14 / 18 / 24 at B=16, H=16, N=32768: 0.607 /
// 0.599 / 0.591 / 0.588 / 0.592 ms; the prefix call is best at 14).
struct SplitPlan {
    int r = 0, n1 = 0;
};
SplitPlan split_plan(int64_t BH, int64_t N, int sms) {
    SplitPlan p;
    const int64_t n = (N + 127) / 128;
    if (sms < 2 || n < 32) return p;
    const int64_t W = (BH + sms - 1) / sms;
    if (W < 2) return p;
    const int64_t r = BH - (W - 1) * sms;
    if (r <= 0 || r >= sms) return p;
    const int64_t k = (r + (sms - r) - 1) / (sms - r);
    const int64_t f = 16;
    const int64_t n2 = (k * n + (k - 1) * f) / (k + 1);
    const int64_t n1 = n - n2;
    if (n1 < 4 || n2 < 4) return p;
    p.r = (int)r;
    p.n1 = (int)n1;
    return p;
}

// Transfer slots and flag words of the split heads, for up to B*H heads.
size_t xfer_bytes(int64_t BH) { return align256(sizeof(float) * BH * la::kXferFloats); }
size_t xflag_bytes(int64_t BH) { return align256(sizeof(unsigned long long) * BH); }

// Fills the split fields of `a` for a bf16 prefill when a workspace region
// (xfer: xfer_bytes(B*H), then xflag_bytes(B*H)) is available.
void plan_split(la::PrefillArgs &a, int dev, char *xfer_region) {
    if (!xfer_region) return;
    const SplitPlan p = split_plan(a.B * a.H, a.N, g_sms[dev]);
    if (p.r == 0) return;
    a.split_r = p.r;
    a.split_n1 = p.n1;
    a.xfer = reinterpret_cast<float *>(xfer_region);
    a.xflag = reinterpret_cast<unsigned long long *>(xfer_region + xfer_bytes(a.B * a.H));
    a.call_id = g_call_id.fetch_add(1);
}

// Workspace of the prefix call: the per-segment partial states, sized for
// the 273-row layout of the fp32 path (the bf16 path uses the first 160 rows'
// worth of each part).
struct PrefixLayout {
    size_t part_s, part_z, base_total, xfer, total;  // base_total: without the split heads' region
};

PrefixLayout prefix_layout(int64_t BH, int64_t M) {
    PrefixLayout L{};
    if (M <= 0) return L;
    const int64_t nseg = la::prefix_split(BH, M).nseg;
    size_t off = 0;
    L.part_s = off; off = align256(off + sizeof(float) * BH * nseg * kD * kDV);
    L.part_z = off; off = align256(off + sizeof(float) * BH * nseg * kD);
    L.base_total = off;
    L.xfer = off;   off += xfer_bytes(BH) + xflag_bytes(BH);  // split heads of the prefill (optional)
    L.total = off;
    return L;
}

cudaError_t run_prefill(const la::PrefillArgs &a, la_dtype dtype, cudaStream_t st, int dk = kDFeat) {
    const int64_t BH = a.B * a.H;
    if (a.N == 0) {
        if (!a.s_out && !a.z_out) return cudaSuccess;
        return la::launch_state_copy(a.compact ? la::kDCompact : la::feat_dim(dk), a.s0, a.z0, a.s_out,
                                     a.z_out, BH, st);
    }
    if (dtype == LA_DTYPE_BF16 && (dk == kDFeat || dk == 8)) {  // tensor cores (d' = 8: padded map)
        la::PrefillArgs b = a;
        b.dk = dk;
        return la::launch_prefill_tc(b, st);
    }
    if (dk != kDFeat) return la::launch_prefill_general(a, dk, dtype, st);
    return la::launch_prefill_simt(a, dtype, st);
}

la_status to_status(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

}  // namespace

extern "C" {

int la_version(void) { return 100; }

const char *la_status_string(la_status s) {
    switch (s) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument (shape, NULL pointer, M > N or overlapping buffers)";
        case LA_ERR_UNSUPPORTED:
            return "unsupported (d_feat 8/16/24/32 (padding, decay and prefix: 16 only), d_v 64, dtype f32/bf16, "
                   "device sm_103)";
        case LA_ERR_MISALIGNED: return "a buffer is not 16-byte aligned";
        case LA_ERR_CUDA: return "CUDA runtime error or kernel launch failure";
        case LA_ERR_TIMEOUT: return "a bounded device-side wait gave up";
        case LA_ERR_SCRATCH_TOO_SMALL:
            return "problem needs more scratch than the no-allocation buffer holds (use la_prefix_prefill)";
    }
    return "unknown status";
}

}  // extern "C"

namespace {

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

la_status prefill_impl(const void *q, const void *k, const void *v, const float *s0,
                       const float *z0, const int32_t *left_pad, void *y, float *s_out,
                       float *z_out, int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                       la_dtype dtype, float eps, la_stream_t stream, const float *gamma = nullptr,
                       bool compact = false, void *workspace = nullptr, size_t workspace_bytes = 0) {
    la_status st = check_common(B, H, N, d_feat, d_v, dtype);
    if (st != LA_OK) return st;
    // padding and decay exist for d' = 16 only
    if ((left_pad || gamma) && d_feat != kDFeat) return LA_ERR_UNSUPPORTED;
    // compact states: the bf16 tensor-core path of the plain prefill only
    if (compact && (d_feat != kDFeat || dtype != LA_DTYPE_BF16 || left_pad || gamma)) return LA_ERR_UNSUPPORTED;
    const int64_t D = compact ? la::kDCompact : la::feat_dim(d_feat);
    if ((s0 == nullptr) != (z0 == nullptr)) return LA_ERR_INVALID_ARG;
    if (N > 0 && (!q || !k || !v || !y)) return LA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, s0, z0, y, s_out, z_out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    const int64_t BH = B * H;
    const size_t es = esize(dtype);
    const Range in[] = {{q, es * BH * N * d_feat}, {k, es * BH * N * d_feat},
                        {v, es * BH * N * kDV}, {s0, sizeof(float) * BH * D * kDV},
                        {z0, sizeof(float) * BH * D}};
    const Range out[] = {{y, es * BH * N * kDV}, {s_out, sizeof(float) * BH * D * kDV},
                         {z_out, sizeof(float) * BH * D}};
    if (any_overlap(in, 5, out, 3)) return LA_ERR_INVALID_ARG;
    if (workspace) {
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return LA_ERR_MISALIGNED;
        const Range ws{workspace, workspace_bytes};
        for (const Range &r : in)
            if (overlaps(ws, r)) return LA_ERR_INVALID_ARG;
        for (const Range &r : out)
            if (overlaps(ws, r)) return LA_ERR_INVALID_ARG;
    }
    if ((left_pad && !aligned4(left_pad)) || (gamma && !aligned4(gamma))) return LA_ERR_MISALIGNED;
    for (const Range &o : out)
        if (overlaps({left_pad, sizeof(int32_t) * B}, o) || overlaps({gamma, sizeof(float) * H}, o))
            return LA_ERR_INVALID_ARG;
    int dev;
    unsigned *status;
    if ((st = device_setup(&dev, &status)) != LA_OK) return st;
    la::PrefillArgs a{q, k, v, s0, z0, y, s_out, z_out, B, H, N, eps, status, left_pad, gamma};
    a.compact = compact;
    // d' = 24, 32 (bf16) on the tensor cores, given room for its buffers
    if (workspace && dtype == LA_DTYPE_BF16 && (d_feat == 24 || d_feat == 32)) {
        const size_t need = la::general_tc_workspace(BH, N, d_feat);  // 0: not this path
        if (need > 0 && workspace_bytes >= need)
            return to_status(
                la::launch_prefill_general_tc(a, d_feat, workspace, reinterpret_cast<cudaStream_t>(stream)));
    }
    // split heads on the bf16 tensor-core path, given room for the hand-over
    if (workspace && dtype == LA_DTYPE_BF16 && (d_feat == kDFeat || d_feat == 8) &&
        workspace_bytes >= xfer_bytes(BH) + xflag_bytes(BH))
        plan_split(a, dev, static_cast<char *>(workspace));
    return to_status(run_prefill(a, dtype, reinterpret_cast<cudaStream_t>(stream), d_feat));
}

la_status prefix_impl(const void *q, const void *k, const void *v, const void *k_e,
                      const void *v_e, int64_t M, const float *s0, const float *z0,
                      const int32_t *left_pad, void *y, float *s_out, float *z_out,
                      void *workspace, size_t workspace_bytes, int64_t B, int64_t H,
                      int64_t N, int d_feat, int d_v, la_dtype dtype, float eps,
                      la_stream_t stream) {
    la_status st = check_common(B, H, N, d_feat, d_v, dtype);
    if (st != LA_OK) return st;
    if (d_feat != kDFeat) return LA_ERR_UNSUPPORTED;  // the prefix path exists for d' = 16
    if (M < 0 || M > N) return LA_ERR_INVALID_ARG;
    if (M == 0)
        return prefill_impl(q, k, v, s0, z0, left_pad, y, s_out, z_out, B, H, N, d_feat, d_v,
                            dtype, eps, stream);
    if ((s0 == nullptr) != (z0 == nullptr)) return LA_ERR_INVALID_ARG;
    if (!q || !k || !v || !y || !k_e || !v_e || !workspace) return LA_ERR_INVALID_ARG;
    const int64_t BH = B * H;
    const PrefixLayout L = prefix_layout(BH, M);
    if (workspace_bytes < L.base_total) return LA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, k_e, v_e, s0, z0, y, s_out, z_out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return LA_ERR_MISALIGNED;
    const size_t es = esize(dtype);
    const Range in[] = {{q, es * BH * N * kDFeat}, {k, es * BH * N * kDFeat},
                        {v, es * BH * N * kDV}, {k_e, es * BH * M * kDFeat},
                        {v_e, es * BH * M * kDV}, {s0, sizeof(float) * BH * kD * kDV},
                        {z0, sizeof(float) * BH * kD}};
    const Range out[] = {{y, es * BH * N * kDV}, {s_out, sizeof(float) * BH * kD * kDV},
                         {z_out, sizeof(float) * BH * kD}, {workspace, workspace_bytes}};
    if (any_overlap(in, 7, out, 4)) return LA_ERR_INVALID_ARG;
    if (left_pad) {
        if (!aligned4(left_pad)) return LA_ERR_MISALIGNED;
        const Range lp{left_pad, sizeof(int32_t) * B};
        for (const Range &o : out)
            if (overlaps(lp, o)) return LA_ERR_INVALID_ARG;
    }
    int dev;
    unsigned *status;
    if ((st = device_setup(&dev, &status)) != LA_OK) return st;

    char *ws = static_cast<char *>(workspace);
    const la::PrefixSplit split = la::prefix_split(BH, M);
    la::PrefixArgs pa{};
    pa.k_e = k_e; pa.v_e = v_e; pa.B = B; pa.H = H; pa.M = M;
    pa.seg_len = split.seg_len; pa.nseg = split.nseg;
    pa.part_s = reinterpret_cast<float *>(ws + L.part_s);
    pa.part_z = reinterpret_cast<float *>(ws + L.part_z);
    pa.status = status;
    pa.left_pad = left_pad;
    pa.N = N;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // the partial states, then the prefill, whose set-up adds them (in segment
    // order) to s0, z0
    cudaError_t e = dtype == LA_DTYPE_BF16 ? la::launch_prefix_partials_tc(pa, cs)
                                           : la::launch_prefix_partials_simt(pa, dtype, cs);
    if (e != cudaSuccess) return LA_ERR_CUDA;
    la::PrefillArgs a{q, k, v, s0, z0, y, s_out, z_out, B, H, N, eps, status, left_pad};
    a.part_s = pa.part_s;
    a.part_z = pa.part_z;
    a.nseg = pa.nseg;
    if (dtype == LA_DTYPE_BF16 && workspace_bytes >= L.total) plan_split(a, dev, ws + L.xfer);
    return to_status(run_prefill(a, dtype, cs));
}

}  // namespace

extern "C" {

la_status la_prefill(const void *q, const void *k, const void *v, const float *s0,
                     const float *z0, void *y, float *s_out, float *z_out, int64_t B,
                     int64_t H, int64_t N, int d_feat, int d_v, la_dtype dtype, float eps,
                     la_stream_t stream) {
    return prefill_impl(q, k, v, s0, z0, nullptr, y, s_out, z_out, B, H, N, d_feat, d_v, dtype,
                        eps, stream);
}

size_t la_prefill_workspace_size(int64_t B, int64_t H, int64_t N, int d_feat, la_dtype dtype) {
    if (B < 1 || H < 1 || N < 0 || B > kMaxBH / H) return 0;
    if (dtype != LA_DTYPE_BF16) return 0;
    if (d_feat == 24 || d_feat == 32) return la::general_tc_workspace(B * H, N, d_feat);
    if (d_feat != kDFeat && d_feat != 8) return 0;
    return xfer_bytes(B * H) + xflag_bytes(B * H);
}

la_status la_prefill_split_info(int64_t B, int64_t H, int64_t N, int *split_heads, int *split_chunk) {
    if (!split_heads || !split_chunk) return LA_ERR_INVALID_ARG;
    *split_heads = *split_chunk = 0;
    if (B < 1 || H < 1 || N < 0 || B > kMaxBH / H) return LA_ERR_INVALID_ARG;
    int dev;
    unsigned *status;
    const la_status st = device_setup(&dev, &status);
    if (st != LA_OK) return st;
    const SplitPlan p = split_plan(B * H, N, g_sms[dev]);
    *split_heads = p.r;
    *split_chunk = p.n1;
    return LA_OK;
}

la_status la_prefill_ws(const void *q, const void *k, const void *v, const float *s0, const float *z0, void *y,
                        float *s_out, float *z_out, void *workspace, size_t workspace_bytes, int64_t B, int64_t H,
                        int64_t N, int d_feat, int d_v, la_dtype dtype, float eps, la_stream_t stream) {
    return prefill_impl(q, k, v, s0, z0, nullptr, y, s_out, z_out, B, H, N, d_feat, d_v, dtype, eps, stream,
                        nullptr, false, workspace, workspace ? workspace_bytes : 0);
}

la_status la_prefill_decay_ws(const void *q, const void *k, const void *v, const float *s0, const float *z0,
                              const float *gamma, void *y, float *s_out, float *z_out, void *workspace,
                              size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                              la_dtype dtype, float eps, la_stream_t stream) {
    if (!gamma) return LA_ERR_INVALID_ARG;
    return prefill_impl(q, k, v, s0, z0, nullptr, y, s_out, z_out, B, H, N, d_feat, d_v, dtype, eps, stream,
                        gamma, false, workspace, workspace ? workspace_bytes : 0);
}

la_status la_prefill_padded(const void *q, const void *k, const void *v, const float *s0,
                            const float *z0, const int32_t *left_pad, void *y, float *s_out,
                            float *z_out, int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                            la_dtype dtype, float eps, la_stream_t stream) {
    if (!left_pad) return LA_ERR_INVALID_ARG;
    return prefill_impl(q, k, v, s0, z0, left_pad, y, s_out, z_out, B, H, N, d_feat, d_v, dtype,
                        eps, stream);
}

size_t la_prefix_workspace_size(int64_t B, int64_t H, int64_t M) {
    if (B < 1 || H < 1 || M <= 0 || B > kMaxBH / H) return 0;
    return prefix_layout(B * H, M).total;
}

}  // extern "C"

namespace la {
size_t prefix_workspace_min(int64_t B, int64_t H, int64_t M) {
    if (B < 1 || H < 1 || M <= 0 || B > kMaxBH / H) return 0;
    return prefix_layout(B * H, M).base_total;
}
}  // namespace la

extern "C" {

la_status la_prefix_prefill(const void *q, const void *k, const void *v, const void *k_e,
                            const void *v_e, int64_t M, const float *s0, const float *z0,
                            void *y, float *s_out, float *z_out, void *workspace,
                            size_t workspace_bytes, int64_t B, int64_t H, int64_t N,
                            int d_feat, int d_v, la_dtype dtype, float eps,
                            la_stream_t stream) {
    return prefix_impl(q, k, v, k_e, v_e, M, s0, z0, nullptr, y, s_out, z_out, workspace,
                       workspace_bytes, B, H, N, d_feat, d_v, dtype, eps, stream);
}

la_status la_prefix_prefill_padded(const void *q, const void *k, const void *v, const void *k_e,
                                   const void *v_e, int64_t M, const float *s0, const float *z0,
                                   const int32_t *left_pad, void *y, float *s_out, float *z_out,
                                   void *workspace, size_t workspace_bytes, int64_t B, int64_t H,
                                   int64_t N, int d_feat, int d_v, la_dtype dtype, float eps,
                                   la_stream_t stream) {
    if (!left_pad) return LA_ERR_INVALID_ARG;
    return prefix_impl(q, k, v, k_e, v_e, M, s0, z0, left_pad, y, s_out, z_out, workspace,
                       workspace_bytes, B, H, N, d_feat, d_v, dtype, eps, stream);
}

}  // extern "C"

namespace {

la_status decode_impl(const void *q, const void *k, const void *v, const float *gamma,
                      const float *s_in, const float *z_in, float *s_out, float *z_out, void *y,
                      int64_t B, int64_t H, int d_feat, int d_v, la_dtype dtype, float eps,
                      la_stream_t stream, bool compact = false) {
    la_status st = check_common(B, H, 1, d_feat, d_v, dtype);
    if (st != LA_OK) return st;
    if (gamma && d_feat != kDFeat) return LA_ERR_UNSUPPORTED;  // decay exists for d' = 16 only
    if (compact && (d_feat != kDFeat || gamma)) return LA_ERR_UNSUPPORTED;
    const int64_t D = compact ? la::kDCompact : la::feat_dim(d_feat);
    if (!q || !k || !v || !s_in || !z_in || !s_out || !z_out || !y) return LA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, s_in, z_in, s_out, z_out, y};
    for (const void *p : ptrs)
        if (!aligned16(p)) return LA_ERR_MISALIGNED;
    const int64_t BH = B * H;
    const size_t es = esize(dtype);
    const size_t sb = sizeof(float) * BH * D * kDV, zb = sizeof(float) * BH * D;
    // exact aliasing s_out == s_in / z_out == z_in is the in-place update
    const Range in[] = {{q, es * BH * d_feat}, {k, es * BH * d_feat}, {v, es * BH * kDV},
                        {s_out == s_in ? nullptr : s_in, sb},
                        {z_out == z_in ? nullptr : z_in, zb}};
    const Range out[] = {{y, es * BH * kDV}, {s_out, sb}, {z_out, zb}};
    if (any_overlap(in, 5, out, 3)) return LA_ERR_INVALID_ARG;
    // an in-place state must not overlap the other state buffer or y either
    if (s_out == s_in && (overlaps({s_in, sb}, {z_in, zb}) || overlaps({s_in, sb}, {y, es * BH * kDV})))
        return LA_ERR_INVALID_ARG;
    if (gamma) {
        if (!aligned4(gamma)) return LA_ERR_MISALIGNED;
        for (const Range &o : out)
            if (overlaps({gamma, sizeof(float) * H}, o)) return LA_ERR_INVALID_ARG;
    }
    int dev;
    unsigned *status;
    if ((st = device_setup(&dev, &status)) != LA_OK) return st;
    la::DecodeArgs a{q, k, v, s_in, z_in, s_out, z_out, y, B, H, eps, gamma, status};
    if (compact) return to_status(la::launch_decode_compact(a, dtype, reinterpret_cast<cudaStream_t>(stream)));
    if (d_feat != kDFeat)
        return to_status(la::launch_decode_general(a, d_feat, dtype, reinterpret_cast<cudaStream_t>(stream)));
    return to_status(la::launch_decode(a, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

la_status la_decode_step(const void *q, const void *k, const void *v, const float *s_in,
                         const float *z_in, float *s_out, float *z_out, void *y, int64_t B,
                         int64_t H, int d_feat, int d_v, la_dtype dtype, float eps,
                         la_stream_t stream) {
    return decode_impl(q, k, v, nullptr, s_in, z_in, s_out, z_out, y, B, H, d_feat, d_v, dtype, eps,
                       stream);
}

la_status la_decode_step_decay(const void *q, const void *k, const void *v, const float *gamma,
                               const float *s_in, const float *z_in, float *s_out, float *z_out,
                               void *y, int64_t B, int64_t H, int d_feat, int d_v, la_dtype dtype,
                               float eps, la_stream_t stream) {
    if (!gamma) return LA_ERR_INVALID_ARG;
    return decode_impl(q, k, v, gamma, s_in, z_in, s_out, z_out, y, B, H, d_feat, d_v, dtype, eps,
                       stream);
}

la_status la_decode_step_compact(const void *q, const void *k, const void *v, const float *s_in_c,
                                 const float *z_in_c, float *s_out_c, float *z_out_c, void *y, int64_t B,
                                 int64_t H, int d_feat, int d_v, la_dtype dtype, float eps,
                                 la_stream_t stream) {
    return decode_impl(q, k, v, nullptr, s_in_c, z_in_c, s_out_c, z_out_c, y, B, H, d_feat, d_v, dtype, eps,
                       stream, true);
}

la_status la_prefill_compact(const void *q, const void *k, const void *v, const float *s0_c,
                             const float *z0_c, void *y, float *s_out_c, float *z_out_c, int64_t B,
                             int64_t H, int64_t N, int d_feat, int d_v, la_dtype dtype, float eps,
                             la_stream_t stream) {
    return prefill_impl(q, k, v, s0_c, z0_c, nullptr, y, s_out_c, z_out_c, B, H, N, d_feat, d_v, dtype, eps,
                        stream, nullptr, true);
}

}  // extern "C"

namespace {

// Shared checks of the two state conversions: from (rows_in) to (rows_out).
la_status convert_check(const float *s_in, const float *z_in, const float *s_out, const float *z_out,
                        int64_t B, int64_t H, int d_feat, int d_v, int64_t rows_in, int64_t rows_out,
                        unsigned **status) {
    if (d_feat != kDFeat || d_v != kDV) return LA_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || B > kMaxBH / H) return LA_ERR_INVALID_ARG;
    if (!s_in || !z_in || !s_out || !z_out) return LA_ERR_INVALID_ARG;
    const void *ptrs[] = {s_in, z_in, s_out, z_out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return LA_ERR_MISALIGNED;
    const int64_t BH = B * H;
    const Range in[] = {{s_in, sizeof(float) * BH * rows_in * kDV}, {z_in, sizeof(float) * BH * rows_in}};
    const Range out[] = {{s_out, sizeof(float) * BH * rows_out * kDV}, {z_out, sizeof(float) * BH * rows_out}};
    if (any_overlap(in, 2, out, 2)) return LA_ERR_INVALID_ARG;
    int dev;
    return device_setup(&dev, status);
}

}  // namespace

extern "C" {

la_status la_state_to_compact(const float *s, const float *z, float *s_c, float *z_c, int64_t B, int64_t H,
                              int d_feat, int d_v, la_stream_t stream) {
    unsigned *status;
    la_status st = convert_check(s, z, s_c, z_c, B, H, d_feat, d_v, kD, la::kDCompact, &status);
    if (st != LA_OK) return st;
    return to_status(la::launch_state_to_compact(s, z, s_c, z_c, B * H, reinterpret_cast<cudaStream_t>(stream)));
}

la_status la_state_from_compact(const float *s_c, const float *z_c, float *s, float *z, int64_t B, int64_t H,
                                int d_feat, int d_v, la_stream_t stream) {
    unsigned *status;
    la_status st = convert_check(s_c, z_c, s, z, B, H, d_feat, d_v, la::kDCompact, kD, &status);
    if (st != LA_OK) return st;
    return to_status(
        la::launch_state_from_compact(s_c, z_c, s, z, B * H, reinterpret_cast<cudaStream_t>(stream)));
}

la_status la_prefill_decay(const void *q, const void *k, const void *v, const float *s0,
                           const float *z0, const float *gamma, void *y, float *s_out,
                           float *z_out, int64_t B, int64_t H, int64_t N, int d_feat, int d_v,
                           la_dtype dtype, float eps, la_stream_t stream) {
    if (!gamma) return LA_ERR_INVALID_ARG;
    return prefill_impl(q, k, v, s0, z0, nullptr, y, s_out, z_out, B, H, N, d_feat, d_v, dtype, eps,
                        stream, gamma);
}

}  // extern "C"

namespace {

// la_prefill_host: the (b, h) rows are processed in up to kHostSlices slices;
// kHostBuffers slices are in flight at once, each on its own stream with its
// own device buffers (copy in, compute, copy out), so the two copy directions
// and the kernels overlap.
constexpr int64_t kHostSlices = 8;
constexpr int64_t kHostBuffers = 3;

struct HostSliceLayout {
    size_t q, k, v, y, s0, z0, s, z, total;
};

HostSliceLayout host_slice_layout(int64_t R, int64_t N, int dk, size_t es) {
    const int64_t D = la::feat_dim(dk);
    HostSliceLayout L{};
    size_t off = 0;
    L.q = off; off = align256(off + es * R * N * dk);
    L.k = off; off = align256(off + es * R * N * dk);
    L.v = off; off = align256(off + es * R * N * kDV);
    L.y = off; off = align256(off + es * R * N * kDV);
    L.s0 = off; off = align256(off + sizeof(float) * R * D * kDV);
    L.z0 = off; off = align256(off + sizeof(float) * R * D);
    L.s = off; off = align256(off + sizeof(float) * R * D * kDV);
    L.z = off; off = align256(off + sizeof(float) * R * D);
    L.total = off;
    return L;
}

int64_t host_slice_rows(int64_t BH) { return (BH + kHostSlices - 1) / kHostSlices; }

size_t host_workspace_bytes(int64_t BH, int64_t N, int dk, size_t es) {
    const int64_t R = host_slice_rows(BH);
    const int64_t nslice = (BH + R - 1) / R;
    const int64_t nb = nslice < kHostBuffers ? nslice : kHostBuffers;
    return (size_t)nb * host_slice_layout(R, N, dk, es).total;
}

}  // namespace

extern "C" {

size_t la_prefill_host_workspace_size(int64_t B, int64_t H, int64_t N, int d_feat, la_dtype dtype) {
    if (check_common(B, H, N, d_feat, kDV, dtype) != LA_OK) return 0;
    return host_workspace_bytes(B * H, N, d_feat, esize(dtype));
}

la_status la_prefill_host(const void *q, const void *k, const void *v, const float *s0,
                          const float *z0, void *y, float *s_out, float *z_out, void *workspace,
                          size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int d_feat,
                          int d_v, la_dtype dtype, float eps, la_stream_t stream) {
    la_status st = check_common(B, H, N, d_feat, d_v, dtype);
    if (st != LA_OK) return st;
    if ((s0 == nullptr) != (z0 == nullptr)) return LA_ERR_INVALID_ARG;
    if (N > 0 && (!q || !k || !v || !y)) return LA_ERR_INVALID_ARG;
    const int64_t BH = B * H;
    const size_t es = esize(dtype);
    const int64_t D = la::feat_dim(d_feat);
    if (!workspace || workspace_bytes < host_workspace_bytes(BH, N, d_feat, es)) return LA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return LA_ERR_MISALIGNED;
    const Range in[] = {{q, es * BH * N * d_feat}, {k, es * BH * N * d_feat}, {v, es * BH * N * kDV},
                        {s0, sizeof(float) * BH * D * kDV}, {z0, sizeof(float) * BH * D}};
    // the workspace is written by the call too: no input or output may overlap it
    const Range out[] = {{y, es * BH * N * kDV}, {s_out, sizeof(float) * BH * D * kDV},
                         {z_out, sizeof(float) * BH * D},
                         {workspace, host_workspace_bytes(BH, N, d_feat, es)}};
    if (any_overlap(in, 5, out, 4)) return LA_ERR_INVALID_ARG;
    int dev;
    unsigned *status;
    if ((st = device_setup(&dev, &status)) != LA_OK) return st;

    const int64_t R = host_slice_rows(BH);
    const int64_t nslice = (BH + R - 1) / R;
    const int nb = (int)(nslice < kHostBuffers ? nslice : kHostBuffers);
    const HostSliceLayout L = host_slice_layout(R, N, d_feat, es);
    cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t ss[kHostBuffers] = {};
    cudaEvent_t fork = nullptr, join[kHostBuffers] = {};
    bool ok = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) == cudaSuccess;
    for (int j = 0; ok && j < nb; ++j)
        ok = cudaStreamCreateWithFlags(&ss[j], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&join[j], cudaEventDisableTiming) == cudaSuccess;
    // the internal streams start after the caller's earlier work
    ok = ok && cudaEventRecord(fork, caller) == cudaSuccess;
    for (int j = 0; ok && j < nb; ++j) ok = cudaStreamWaitEvent(ss[j], fork, 0) == cudaSuccess;
    la_status result = ok ? LA_OK : LA_ERR_CUDA;
    auto copy = [&](void *dst, const void *src, size_t bytes, cudaStream_t cs) {
        if (result == LA_OK && bytes > 0 && cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, cs) != cudaSuccess)
            result = LA_ERR_CUDA;
    };
    for (int64_t i = 0; ok && result == LA_OK && i < nslice; ++i) {
        const int j = (int)(i % nb);
        cudaStream_t cs = ss[j];
        char *base = static_cast<char *>(workspace) + (size_t)j * L.total;
        const int64_t r0 = i * R, nr = (BH - r0) < R ? (BH - r0) : R;
        const size_t qk = es * N * d_feat, vy = es * N * kDV, sr = sizeof(float) * D * kDV,
                     zr = sizeof(float) * D;
        copy(base + L.q, static_cast<const char *>(q) + r0 * qk, nr * qk, cs);
        copy(base + L.k, static_cast<const char *>(k) + r0 * qk, nr * qk, cs);
        copy(base + L.v, static_cast<const char *>(v) + r0 * vy, nr * vy, cs);
        if (s0) {
            copy(base + L.s0, reinterpret_cast<const char *>(s0) + r0 * sr, nr * sr, cs);
            copy(base + L.z0, reinterpret_cast<const char *>(z0) + r0 * zr, nr * zr, cs);
        }
        if (result != LA_OK) break;
        // the slice's rows as nr independent sequences of one batch row each
        result = prefill_impl(base + L.q, base + L.k, base + L.v,
                              s0 ? reinterpret_cast<float *>(base + L.s0) : nullptr,
                              s0 ? reinterpret_cast<float *>(base + L.z0) : nullptr, nullptr, base + L.y,
                              s_out ? reinterpret_cast<float *>(base + L.s) : nullptr,
                              z_out ? reinterpret_cast<float *>(base + L.z) : nullptr, nr, 1, N, d_feat,
                              d_v, dtype, eps, reinterpret_cast<la_stream_t>(cs));
        copy(static_cast<char *>(y) + r0 * vy, base + L.y, nr * vy, cs);
        if (s_out) copy(reinterpret_cast<char *>(s_out) + r0 * sr, base + L.s, nr * sr, cs);
        if (z_out) copy(reinterpret_cast<char *>(z_out) + r0 * zr, base + L.z, nr * zr, cs);
    }
    // the caller's stream continues after every slice (also after a failure,
    // so that no enqueued copy outlives the call's ordering)
    for (int j = 0; j < nb; ++j) {
        if (ss[j] && join[j] && cudaEventRecord(join[j], ss[j]) == cudaSuccess)
            cudaStreamWaitEvent(caller, join[j], 0);
        else if (ss[j])
            cudaStreamSynchronize(ss[j]);
    }
    // released once their work completes
    for (int j = 0; j < nb; ++j) {
        if (join[j]) cudaEventDestroy(join[j]);
        if (ss[j]) cudaStreamDestroy(ss[j]);
    }
    if (fork) cudaEventDestroy(fork);
    return result;
}

la_status la_debug_timeout_probe(la_stream_t stream) {
    int dev;
    unsigned *status;
    la_status st = device_setup(&dev, &status);
    if (st != LA_OK) return st;
    return to_status(la::launch_timeout_probe(status, reinterpret_cast<cudaStream_t>(stream)));
}

la_status la_check_device_status(la_stream_t stream) {
    int dev;
    unsigned *status;
    la_status st = device_setup(&dev, &status);
    if (st != LA_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LA_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LA_ERR_CUDA;
    if (word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return LA_ERR_CUDA;
        return (word & la::kStatusTimeout) ? LA_ERR_TIMEOUT : LA_ERR_INVALID_ARG;
    }
    return LA_OK;
}

}  // extern "C"
