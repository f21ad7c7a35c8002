// gdn_replay.cu -- libgdnreplay: ReplaySSM verify / accept / flush of Gated
// DeltaNet state for sm_103a.  The C ABI and the layouts are documented in
// include/gdnreplay.h; this file holds the kernels and host validation.
//
// Method: "The inference stack behind OCRia" (LlamaIndex engineering blog),
// section "Making speculative verification cheaper" -- a checkpoint of the state
// and a buffer of committed inputs per sequence; verify replays both, flush
// rewrites the checkpoint, accept moves the buffer length.  Recurrence: the
// gated delta rule of "Gated Delta Networks" (ICLR 2025),
//     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t (scale q_t).
//
// Per-token replay kernels (this file).  Every row i of S evolves on its own:
// S_t[i,:] depends only on S_{t-1}[i,:], k_t, v_t[i], a_t and b_t.  A CTA owns
// 64 rows of one (sequence, head); TPR = d_k/16 threads own one state row,
// thread `part` holding the 16-byte column chunks {TPR*m + part} (16 floats),
// so the TPR threads of a row read TPR*16 contiguous bytes per load and a warp
// touches whole 32-byte sectors.  Keys, queries, values and gates of all
// replayed tokens are staged once into shared memory as fp32; the row dot
// products are reduced across the row's threads with log2(TPR) shuffles.
//
// Decay factoring.  The kernels keep S = c * St with a per-(b,h) scalar c, so
// one token costs a dot product and one FMA per element instead of a scale,
// a multiply and an add:  c' = a c,  w = b (v - c' (St k)),  St += (w / c') k.
// When c' falls below 2^-64 the factor is folded back into St (rare; it
// happens only after a run of near-reset gates).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "replay_common.h"

namespace {

using gdn::ReplayArgs;
using gdn::launch_pdl;
using gdn::pdl_release;
using gdn::pdl_wait;

constexpr int kRows = 64;               // state rows per CTA
constexpr float kRenorm = 5.421011e-20f;  // 2^-64

template <typename TIn> struct InVec;   // one 16-byte vector of input elements
template <> struct InVec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void to_f32(const uint4 &r, float *f) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 x = __bfloat1622float2(p[i]);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
};
template <> struct InVec<float> {
    static constexpr int N = 4;
    __device__ static void to_f32(const uint4 &r, float *f) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
};


// Copy `n` token rows of width D (elements of TIn) into fp32 shared memory,
// rows [dst0, dst0 + n).  Token r comes from src + r * src_stride.  When
// `copy_to` is set the raw vectors are also written to copy_to + r * dst_stride.
template <typename TIn, int D>
__device__ __forceinline__ void stage_rows(float *sm, int dst0, int n,
                                           const TIn *src, long src_stride,
                                           TIn *copy_to, long copy_stride)
{
    constexpr int VE = InVec<TIn>::N;
    constexpr int VPR = D / VE;                 // vectors per row
    for (int e = threadIdx.x; e < n * VPR; e += blockDim.x) {
        const int r = e / VPR, c = e % VPR;
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src + r * src_stride) + c);
        if (copy_to) reinterpret_cast<uint4 *>(copy_to + r * copy_stride)[c] = raw;
        float f[VE];
        InVec<TIn>::to_f32(raw, f);
        float4 *d = reinterpret_cast<float4 *>(sm + (size_t)(dst0 + r) * D + c * VE);
#pragma unroll
        for (int i = 0; i < VE / 4; ++i) d[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
    }
}

template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Shared-memory footprint of one CTA (floats): keys and values of up to `cap`
// tokens, T queries, and a, b per token.
__host__ __device__ inline size_t replay_smem_floats(int dk, int dv, int cap, int T) {
    return (size_t)cap * dk + (size_t)T * dk + (size_t)cap * dv + 2 * (size_t)cap;
}

// MODE 0 (verify): checkpoint + buffer + draft, outputs, stage draft into buffer.
// MODE 1 (flush):  replay the buffer onto the checkpoint and store it.
// MODE 2 (verify with fold): as verify, and a unit whose buffer reached the
//   threshold also stores the state after its buffered tokens and stages the
//   draft at buffer slot 0 (one CTA owns all rows of the unit in this mode).
enum { kVerify = 0, kFlush = 1, kVerifyFold = 2 };

template <int DK, int DV, typename TIn, int MODE>
__device__ __forceinline__ void replay_pertoken(const ReplayArgs &a)
{
    constexpr bool VERIFY = MODE != kFlush;
    constexpr int ROWS = MODE == kVerifyFold ? DV : kRows;
    constexpr int TPR = DK / 16;                         // threads per state row
    extern __shared__ __align__(16) float smem[];
    const int h = blockIdx.x, b = blockIdx.y;
    pdl_wait();
    pdl_release();
    const int slot = a.state_idx ? a.state_idx[b] : b;
    if (slot < 0 || slot >= a.n_slot) {
        if (threadIdx.x == 0 && h == 0 && blockIdx.z == 0) atomicOr(a.status, GDN_STATUS_BAD_SLOT);
        return;
    }
    const int len = a.buf_len[slot];
    int n_tok;
    const bool fold = MODE == kVerifyFold && len >= a.threshold && len <= a.cap;
    if (VERIFY) {
        if (len < 0 || (!fold && len + a.T > a.cap)) {
            if (threadIdx.x == 0 && h == 0 && blockIdx.z == 0)
                atomicOr(a.status, len < 0 || len > a.cap ? GDN_STATUS_BAD_LEN : GDN_STATUS_NO_ROOM);
            return;
        }
        n_tok = len + a.T;
    } else {
        if (len < 0 || len > a.cap) return;              // reported by the length kernel
        if (!(len >= a.threshold || (a.force && len > 0))) return;
        n_tok = len;
    }
    const int cap = a.cap, T = a.T, H = a.H;
    const int cmax = MODE == kVerifyFold ? cap + T : cap;   // most tokens one unit replays
    float *sk = smem;                                    // [cmax][DK]
    float *sq = sk + (size_t)cmax * DK;                  // [T][DK]
    float *sv = sq + (size_t)T * DK;                     // [cmax][DV]
    float *sa = sv + (size_t)cmax * DV;                  // [cmax] alpha
    float *sb = sa + cmax;                               // [cmax] beta

    const size_t unit = (size_t)slot * H + h;
    const TIn *bk = reinterpret_cast<const TIn *>(a.buf_k) + unit * cap * DK;
    const TIn *bv = reinterpret_cast<const TIn *>(a.buf_v) + unit * cap * DV;
    const float *bg = a.buf_g + unit * cap, *bb = a.buf_beta + unit * cap;

    // ---- stage committed tokens (and the draft block) into shared memory
    stage_rows<TIn, DK>(sk, 0, len, bk, DK, nullptr, 0);
    stage_rows<TIn, DV>(sv, 0, len, bv, DV, nullptr, 0);
    for (int t = threadIdx.x; t < len; t += blockDim.x) { sa[t] = expf(bg[t]); sb[t] = bb[t]; }
    if (VERIFY) {
        const bool writer = blockIdx.z == 0 && !fold;    // one CTA per (b, h) stages the draft
        const long tk = (long)H * DK, tv = (long)H * DV;
        const TIn *dk_ = reinterpret_cast<const TIn *>(a.k) + ((size_t)b * T * H + h) * DK;
        const TIn *dq_ = reinterpret_cast<const TIn *>(a.q) + ((size_t)b * T * H + h) * DK;
        const TIn *dv_ = reinterpret_cast<const TIn *>(a.v) + ((size_t)b * T * H + h) * DV;
        TIn *wk = writer ? reinterpret_cast<TIn *>(a.buf_k) + (unit * cap + len) * DK : nullptr;
        TIn *wv = writer ? reinterpret_cast<TIn *>(a.buf_v) + (unit * cap + len) * DV : nullptr;
        stage_rows<TIn, DK>(sk, len, T, dk_, tk, wk, DK);
        stage_rows<TIn, DV>(sv, len, T, dv_, tv, wv, DV);
        stage_rows<TIn, DK>(sq, 0, T, dq_, tk, nullptr, 0);
        for (int t = threadIdx.x; t < T; t += blockDim.x) {
            const size_t gi = ((size_t)b * T + t) * H + h;
            const float gg = a.g[gi], be = a.beta[gi];
            sa[len + t] = expf(gg);
            sb[len + t] = be;
            if (writer) {
                a.buf_g[unit * cap + len + t] = gg;
                a.buf_beta[unit * cap + len + t] = be;
            }
        }
    }
    __syncthreads();

    // ---- state row chunk into registers
    constexpr int NC = 4;                                // float4 chunks per thread
    const int row = blockIdx.z * ROWS + threadIdx.x / TPR, part = threadIdx.x % TPR;
    const float *src = (MODE == kVerify ? a.state_in : a.state_out) + (unit * DV + row) * DK;
    float4 s[NC];
#pragma unroll
    for (int m = 0; m < NC; ++m)                         // flush rewrites what it reads: coherent loads
        s[m] = MODE == kVerify ? __ldg(reinterpret_cast<const float4 *>(src) + TPR * m + part)
                               : reinterpret_cast<const float4 *>(src)[TPR * m + part];

    float c = 1.0f;
    for (int t = 0; t < n_tok; ++t) {
        const float4 *kt = reinterpret_cast<const float4 *>(sk + (size_t)t * DK);
        float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);   // four independent FMA chains
#pragma unroll
        for (int m = 0; m < NC; ++m) {
            const float4 kv = kt[TPR * m + part];
            acc4.x = fmaf(s[m].x, kv.x, acc4.x); acc4.y = fmaf(s[m].y, kv.y, acc4.y);
            acc4.z = fmaf(s[m].z, kv.z, acc4.z); acc4.w = fmaf(s[m].w, kv.w, acc4.w);
        }
        const float acc = row_sum<TPR>((acc4.x + acc4.y) + (acc4.z + acc4.w));   // (St k_t)_row
        c *= sa[t];                                      // c' = a_t c
        const float w = sb[t] * (sv[(size_t)t * DV + row] - c * acc);
        const float coef = __fdividef(w, c);
#pragma unroll
        for (int m = 0; m < NC; ++m) {                   // keys re-read from shared memory
            const float4 kv = kt[TPR * m + part];
            s[m].x = fmaf(coef, kv.x, s[m].x); s[m].y = fmaf(coef, kv.y, s[m].y);
            s[m].z = fmaf(coef, kv.z, s[m].z); s[m].w = fmaf(coef, kv.w, s[m].w);
        }
        if (c < kRenorm) {                               // uniform across the CTA
#pragma unroll
            for (int m = 0; m < NC; ++m) { s[m].x *= c; s[m].y *= c; s[m].z *= c; s[m].w *= c; }
            c = 1.0f;
        }
        if (MODE == kVerifyFold && fold && t == len - 1) {   // the flushed checkpoint
            float4 *dst = reinterpret_cast<float4 *>(a.state_out + (unit * DV + row) * DK);
#pragma unroll
            for (int m = 0; m < NC; ++m)
                dst[TPR * m + part] = make_float4(s[m].x * c, s[m].y * c, s[m].z * c, s[m].w * c);
        }
        if (VERIFY && t >= len) {
            const float4 *qt = reinterpret_cast<const float4 *>(sq + (size_t)(t - len) * DK);
            float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < NC; ++m) {
                const float4 qv = qt[TPR * m + part];
                o4.x = fmaf(s[m].x, qv.x, o4.x); o4.y = fmaf(s[m].y, qv.y, o4.y);
                o4.z = fmaf(s[m].z, qv.z, o4.z); o4.w = fmaf(s[m].w, qv.w, o4.w);
            }
            const float o = row_sum<TPR>((o4.x + o4.y) + (o4.z + o4.w));
            if (part == 0) a.out[(((size_t)b * T + (t - len)) * H + h) * DV + row] = o * c * a.scale;
        }
    }
    if (!VERIFY) {
        float4 *dst = reinterpret_cast<float4 *>(a.state_out + (unit * DV + row) * DK);
#pragma unroll
        for (int m = 0; m < NC; ++m)
            dst[TPR * m + part] = make_float4(s[m].x * c, s[m].y * c, s[m].z * c, s[m].w * c);
    }
    if (MODE == kVerifyFold && fold) {
        // the draft becomes buffer tokens 0 .. T-1; every buffer read was staged before
        // the barrier above, and this CTA is the only reader of the unit's buffer
        const int T = a.T, H = a.H, cap = a.cap;
        constexpr int VE = InVec<TIn>::N;
        TIn *wk = reinterpret_cast<TIn *>(a.buf_k) + unit * cap * DK;
        TIn *wv = reinterpret_cast<TIn *>(a.buf_v) + unit * cap * DV;
        const TIn *dk_ = reinterpret_cast<const TIn *>(a.k) + ((size_t)b * T * H + h) * DK;
        const TIn *dv_ = reinterpret_cast<const TIn *>(a.v) + ((size_t)b * T * H + h) * DV;
        for (int e = threadIdx.x; e < T * (DK / VE); e += blockDim.x) {
            const int r = e / (DK / VE), cc = e % (DK / VE);
            reinterpret_cast<uint4 *>(wk + (size_t)r * DK)[cc] =
                __ldg(reinterpret_cast<const uint4 *>(dk_ + (size_t)r * H * DK) + cc);
        }
        for (int e = threadIdx.x; e < T * (DV / VE); e += blockDim.x) {
            const int r = e / (DV / VE), cc = e % (DV / VE);
            reinterpret_cast<uint4 *>(wv + (size_t)r * DV)[cc] =
                __ldg(reinterpret_cast<const uint4 *>(dv_ + (size_t)r * H * DV) + cc);
        }
        for (int t = threadIdx.x; t < T; t += blockDim.x) {
            const size_t gi = ((size_t)b * T + t) * H + h;
            a.buf_g[unit * cap + t] = a.g[gi];
            a.buf_beta[unit * cap + t] = a.beta[gi];
        }
    }
}

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kRows * (DK / 16), 2) verify_pertoken_kernel(ReplayArgs a) {
    replay_pertoken<DK, DV, TIn, kVerify>(a);
}

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kRows * (DK / 16), 2) flush_pertoken_kernel(ReplayArgs a) {
    replay_pertoken<DK, DV, TIn, kFlush>(a);
}

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(DV * (DK / 16), 1) verify_fold_pertoken_kernel(ReplayArgs a) {
    replay_pertoken<DK, DV, TIn, kVerifyFold>(a);
}

// After the flush kernel: one thread per sequence resets the length of every
// flushed slot (all CTAs of the flush have read it by then) and reports
// corrupt lengths.  When a fold gave up on a bounded wait (GDN_STATUS_TIMEOUT in
// *status) no length is reset, so no buffered token is dropped unfolded.
__global__ void flush_lengths_kernel(int32_t *buf_len, const int32_t *state_idx, int B, int n_slot,
                                     int cap, int threshold, int force, int32_t *status)
{
    pdl_wait();
    pdl_release();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    if (*status & GDN_STATUS_TIMEOUT) return;
    const int slot = state_idx ? state_idx[b] : b;
    if (slot < 0 || slot >= n_slot) { atomicOr(status, GDN_STATUS_BAD_SLOT); return; }
    const int len = buf_len[slot];
    if (len < 0 || len > cap) { atomicOr(status, GDN_STATUS_BAD_LEN); return; }
    if (len >= threshold || (force && len > 0)) buf_len[slot] = 0;
}

__global__ void accept_kernel(int32_t *buf_len, const int32_t *state_idx, const int32_t *accepted,
                              int B, int n_slot, int T, int cap, int32_t *status)
{
    pdl_wait();
    pdl_release();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int slot = state_idx ? state_idx[b] : b;
    if (slot < 0 || slot >= n_slot) { atomicOr(status, GDN_STATUS_BAD_SLOT); return; }
    const int p = accepted[b];
    if (p < 0 || p > T) { atomicOr(status, GDN_STATUS_BAD_ACCEPT); return; }
    const int len = buf_len[slot];
    if (len < 0 || len + p > cap) { atomicOr(status, GDN_STATUS_BAD_LEN); return; }
    buf_len[slot] = len + p;
}

// After a verify with fold: sequences whose buffer reached the threshold restart
// at length 0 (their draft sits in slots 0 .. T-1), then the accepted prefix is kept.
// After a timed-out verify_fold (GDN_STATUS_TIMEOUT) every length is left as it is.
__global__ void accept_fold_kernel(int32_t *buf_len, const int32_t *state_idx, const int32_t *accepted,
                                   int B, int n_slot, int T, int cap, int threshold, int32_t *status)
{
    pdl_wait();
    pdl_release();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    if (*status & GDN_STATUS_TIMEOUT) return;
    const int slot = state_idx ? state_idx[b] : b;
    if (slot < 0 || slot >= n_slot) { atomicOr(status, GDN_STATUS_BAD_SLOT); return; }
    const int p = accepted[b];
    if (p < 0 || p > T) { atomicOr(status, GDN_STATUS_BAD_ACCEPT); return; }
    int len = buf_len[slot];
    if (len < 0 || len > cap) { atomicOr(status, GDN_STATUS_BAD_LEN); return; }
    if (len >= threshold) len = 0;
    if (len + p > cap) { atomicOr(status, GDN_STATUS_BAD_LEN); return; }
    buf_len[slot] = len + p;
}

// ------------------------------------------------------------------ host side
bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

int check_dims(const gdn_replay_dims *d) {
    if (!d) return GDN_ERR_NULL;
    if (d->in_dtype != GDN_DTYPE_BF16 && d->in_dtype != GDN_DTYPE_F32) return GDN_ERR_DTYPE;
    if (d->B < 0 || d->H < 1 || d->n_slot < d->B) return GDN_ERR_DIMS;
    if ((d->dk != 64 && d->dk != 128) || (d->dv != 64 && d->dv != 128)) return GDN_ERR_DIMS;
    if (d->T < 1 || d->T > 64 || d->cap < d->T || d->cap > 256) return GDN_ERR_DIMS;
    if (d->threshold < 1 || d->threshold > d->cap) return GDN_ERR_DIMS;
    if (d->flags & ~GDN_FLAG_TEST_EXPIRE) return GDN_ERR_DIMS;
    if ((long long)d->B * d->H > 0x7fffffffLL) return GDN_ERR_DIMS;
    if (replay_smem_floats(d->dk, d->dv, d->cap, d->T) * sizeof(float) > 227 * 1024) return GDN_ERR_DIMS;
    return GDN_OK;
}

template <int DK, int DV, typename TIn, int MODE>
int launch_replay(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s) {
    auto kern = MODE == kVerify ? verify_pertoken_kernel<DK, DV, TIn>
              : MODE == kFlush  ? flush_pertoken_kernel<DK, DV, TIn>
                                : verify_fold_pertoken_kernel<DK, DV, TIn>;
    const size_t smem = replay_smem_floats(DK, DV, MODE == kVerifyFold ? d->cap + d->T : d->cap, d->T) *
                        sizeof(float);
    if (smem > 227 * 1024) return GDN_ERR_DIMS;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int rows = MODE == kVerifyFold ? DV : kRows;
    return launch_pdl(kern, dim3(d->H, d->B, DV / rows), dim3(rows * (DK / 16)), smem, s, a) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

template <int MODE>
int dispatch_replay(const gdn_replay_dims *d, const ReplayArgs &a, cudaStream_t s) {
    const bool bf = d->in_dtype == GDN_DTYPE_BF16;
#define GDN_CASE(DK_, DV_)                                                                   \
    if (d->dk == DK_ && d->dv == DV_)                                                        \
        return bf ? launch_replay<DK_, DV_, __nv_bfloat16, MODE>(d, a, s)                    \
                  : launch_replay<DK_, DV_, float, MODE>(d, a, s);
    GDN_CASE(128, 128) GDN_CASE(128, 64) GDN_CASE(64, 128) GDN_CASE(64, 64)
#undef GDN_CASE
    return GDN_ERR_DIMS;
}

}  // namespace

extern "C" {

int gdn_replay_verify(const gdn_replay_dims *d, const float *state, const int32_t *state_idx,
                      void *buf_k, void *buf_v, float *buf_g, float *buf_beta,
                      const int32_t *buf_len, const void *q, const void *k, const void *v,
                      const float *g, const float *beta, float *out, int32_t *status,
                      cudaStream_t stream)
{
    const int rc = check_dims(d);
    if (rc) return rc;
    if (d->B == 0) return GDN_OK;
    if (!state || !buf_k || !buf_v || !buf_g || !buf_beta || !buf_len || !q || !k || !v || !g ||
        !beta || !out || !status)
        return GDN_ERR_NULL;
    if (!aligned(state, 16) || !aligned(buf_k, 16) || !aligned(buf_v, 16) || !aligned(q, 16) ||
        !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 4))
        return GDN_ERR_DIMS;
    ReplayArgs a{};
    a.state_in = state; a.state_idx = state_idx;
    a.buf_k = buf_k; a.buf_v = buf_v; a.buf_g = buf_g; a.buf_beta = buf_beta; a.buf_len = buf_len;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out; a.status = status;
    a.B = d->B; a.H = d->H; a.T = d->T; a.cap = d->cap; a.threshold = d->threshold;
    a.n_slot = d->n_slot; a.scale = d->scale; a.flags = d->flags;
    const int tc = gdn::tc_verify(d, a, stream);
    if (tc <= 0) return tc;
    return dispatch_replay<kVerify>(d, a, stream);
}

int gdn_replay_accept(const gdn_replay_dims *d, int32_t *buf_len, const int32_t *state_idx,
                      const int32_t *accepted, int32_t *status, cudaStream_t stream)
{
    const int rc = check_dims(d);
    if (rc) return rc;
    if (d->B == 0) return GDN_OK;
    if (!buf_len || !accepted || !status) return GDN_ERR_NULL;
    return launch_pdl(accept_kernel, dim3((d->B + 127) / 128), dim3(128), 0, stream, buf_len, state_idx,
                      accepted, d->B, d->n_slot, d->T, d->cap, status) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

int gdn_replay_flush(const gdn_replay_dims *d, float *state, const int32_t *state_idx,
                     const void *buf_k, const void *buf_v, const float *buf_g,
                     const float *buf_beta, int32_t *buf_len, int32_t force, int32_t *status,
                     cudaStream_t stream)
{
    const int rc = check_dims(d);
    if (rc) return rc;
    if (d->B == 0) return GDN_OK;
    if (!state || !buf_k || !buf_v || !buf_g || !buf_beta || !buf_len || !status) return GDN_ERR_NULL;
    if (!aligned(state, 16) || !aligned(buf_k, 16) || !aligned(buf_v, 16)) return GDN_ERR_DIMS;
    ReplayArgs a{};
    a.state_out = state; a.state_idx = state_idx;
    a.buf_k = const_cast<void *>(buf_k); a.buf_v = const_cast<void *>(buf_v);
    a.buf_g = const_cast<float *>(buf_g); a.buf_beta = const_cast<float *>(buf_beta);
    a.buf_len = buf_len; a.status = status;
    a.B = d->B; a.H = d->H; a.T = d->T; a.cap = d->cap; a.threshold = d->threshold;
    a.force = force ? 1 : 0; a.n_slot = d->n_slot; a.scale = d->scale; a.flags = d->flags;
    int r = gdn::tc_flush(d, a, stream);
    if (r > 0) r = dispatch_replay<kFlush>(d, a, stream);
    if (r) return r;
    return launch_pdl(flush_lengths_kernel, dim3((d->B + 127) / 128), dim3(128), 0, stream, buf_len,
                      state_idx, d->B, d->n_slot, d->cap, d->threshold, a.force, status) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

int gdn_replay_verify_fold(const gdn_replay_dims *d, float *state, const int32_t *state_idx,
                           void *buf_k, void *buf_v, float *buf_g, float *buf_beta,
                           const int32_t *buf_len, const void *q, const void *k, const void *v,
                           const float *g, const float *beta, float *out, int32_t *status,
                           cudaStream_t stream)
{
    const int rc = check_dims(d);
    if (rc) return rc;
    if (d->B == 0) return GDN_OK;
    if (!state || !buf_k || !buf_v || !buf_g || !buf_beta || !buf_len || !q || !k || !v || !g ||
        !beta || !out || !status)
        return GDN_ERR_NULL;
    if (!aligned(state, 16) || !aligned(buf_k, 16) || !aligned(buf_v, 16) || !aligned(q, 16) ||
        !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 4))
        return GDN_ERR_DIMS;
    if (d->threshold + d->T - 1 > d->cap) return GDN_ERR_DIMS;   // room for the draft when not folding
    ReplayArgs a{};
    a.state_in = state; a.state_out = state; a.state_idx = state_idx;
    a.buf_k = buf_k; a.buf_v = buf_v; a.buf_g = buf_g; a.buf_beta = buf_beta; a.buf_len = buf_len;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out; a.status = status;
    a.B = d->B; a.H = d->H; a.T = d->T; a.cap = d->cap; a.threshold = d->threshold;
    a.n_slot = d->n_slot; a.scale = d->scale; a.flags = d->flags;
    const int tc = gdn::tc_verify_fold(d, a, stream);
    if (tc <= 0) return tc;
    return dispatch_replay<kVerifyFold>(d, a, stream);
}

int gdn_replay_accept_fold(const gdn_replay_dims *d, int32_t *buf_len, const int32_t *state_idx,
                           const int32_t *accepted, int32_t *status, cudaStream_t stream)
{
    const int rc = check_dims(d);
    if (rc) return rc;
    if (d->B == 0) return GDN_OK;
    if (!buf_len || !accepted || !status) return GDN_ERR_NULL;
    return launch_pdl(accept_fold_kernel, dim3((d->B + 127) / 128), dim3(128), 0, stream, buf_len, state_idx,
                      accepted, d->B, d->n_slot, d->T, d->cap, d->threshold, status) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

int gdn_replay_kernel_family(const gdn_replay_dims *d) {
    const int rc = check_dims(d);
    if (rc) return rc;
    return gdn::tc_shape(d) ? GDN_FAMILY_TCGEN05 : GDN_FAMILY_PERTOKEN;
}

const char *gdn_replay_strerror(int code) {
    switch (code) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "a required pointer is NULL";
        case GDN_ERR_DIMS: return "unsupported or inconsistent dims (or misaligned pointer)";
        case GDN_ERR_DTYPE: return "unsupported input dtype";
        case GDN_ERR_LAUNCH: return "CUDA launch failed";
        default: return "unknown gdn_replay error";
    }
}

int gdn_replay_version(void) { return 200; }

}  // extern "C"
