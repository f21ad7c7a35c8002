// gdn_nonreplay.cu -- the non-replay baseline for sm_103a (C ABI and layouts:
// include/gdnnonreplay.h): the state is always current, the verify stores the
// state after every draft token and the accept restores by copying one of those
// snapshots ("The inference stack behind OCRia", section "Making speculative
// verification cheaper": restoring a recurrent state moves a lot of data).
//
// A streaming kernel pair.  At d = 128 the verify reads 64 KB of state per
// (sequence, head) and writes T x 64 KB of snapshots; its arithmetic (a rank-one
// update and two dot products per token and row) is a few flops per stored
// byte, so it runs on the CUDA cores with the state rows in registers and the
// snapshot stores as the only large stream.  No tensor cores: the update is
// rank one and every intermediate state has to be materialised anyway.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdnnonreplay.h"
#include "replay_common.h"

namespace {

using gdn::launch_pdl;
using gdn::pdl_release;
using gdn::pdl_wait;

constexpr int kRowsPerCta = 32;     // state rows of one CTA
constexpr int kLanesPerRow = 8;     // threads sharing one state row
constexpr int kNrThreads = kRowsPerCta * kLanesPerRow;
constexpr int kCopyThreads = 256;

struct NrArgs {
    const float *state;
    float *state_w;
    const int32_t *state_idx;
    const void *q, *k, *v;
    const float *g, *beta;
    float *out;
    float *snap;
    const int32_t *accepted;
    int32_t *status;
    int B, H, T, dv, n_slot;
    float scale;
};

template <typename TIn> __device__ __forceinline__ float to_f(TIn x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// One CTA per (32 state rows, head, sequence).  Thread (r, l) owns DK/8 columns of
// row r, as DK/32 groups of four: columns 32 i + 4 l .. 32 i + 4 l + 3, so that store
// i of the row's 8 lanes covers 128 contiguous bytes (whole sectors; with 16 consecutive
// columns per lane every 16-byte store landed in a different half-sector and the
// snapshot stream ran at 2.98 TB/s against 7.4 TB/s for a plain fill).  The row
// reductions are shuffles over the row's 8 lanes.  Shared memory: k_t and scale q_t of
// every draft token (fp32), the values of the CTA's rows, alpha_t = exp(g_t) and beta_t.
// Snapshots leave with streaming stores: the accept reads back one snapshot in T.
template <int DK, typename TIn>
__global__ void __launch_bounds__(kNrThreads) nonreplay_verify_kernel(const NrArgs a)
{
    constexpr int NC = DK / kLanesPerRow;
    extern __shared__ float smem[];
    const int T = a.T, H = a.H, dv = a.dv;
    const int row0 = blockIdx.x * kRowsPerCta, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, r = tid / kLanesPerRow, c0 = (tid % kLanesPerRow) * 4;   // + 32 i
    float *sK = smem, *sQ = sK + T * DK, *sV = sQ + T * DK, *sA = sV + T * kRowsPerCta, *sB = sA + T;
    pdl_wait();
    pdl_release();
    const int slot = a.state_idx ? a.state_idx[b] : b;
    if (slot < 0 || slot >= a.n_slot) {
        if (tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(a.status, GDN_STATUS_BAD_SLOT);
        return;
    }
    const size_t unit = static_cast<size_t>(slot) * H + h;
    float S[NC];
    {
        const float4 *src = reinterpret_cast<const float4 *>(a.state + (unit * dv + row0 + r) * DK + c0);
#pragma unroll
        for (int i = 0; i < NC / 4; ++i) {
            const float4 x = src[8 * i];
            S[4 * i] = x.x; S[4 * i + 1] = x.y; S[4 * i + 2] = x.z; S[4 * i + 3] = x.w;
        }
    }
    const TIn *qi = static_cast<const TIn *>(a.q), *ki = static_cast<const TIn *>(a.k);
    const TIn *vi = static_cast<const TIn *>(a.v);
    for (int e = tid; e < T * DK; e += kNrThreads) {
        const int t = e / DK, j = e - t * DK;
        const size_t off = ((static_cast<size_t>(b) * T + t) * H + h) * DK + j;
        sK[e] = to_f(ki[off]);
        sQ[e] = a.scale * to_f(qi[off]);
    }
    for (int e = tid; e < T * kRowsPerCta; e += kNrThreads) {
        const int t = e / kRowsPerCta, i = e - t * kRowsPerCta;
        sV[e] = to_f(vi[((static_cast<size_t>(b) * T + t) * H + h) * dv + row0 + i]);
    }
    for (int t = tid; t < T; t += kNrThreads) {
        const size_t gi = (static_cast<size_t>(b) * T + t) * H + h;
        sA[t] = expf(a.g[gi]);
        sB[t] = a.beta[gi];
    }
    __syncthreads();
    const size_t snap_t = static_cast<size_t>(dv) * DK;          // floats per snapshot
    float *snap = a.snap + ((static_cast<size_t>(b) * H + h) * T * dv + row0 + r) * DK + c0;
    float *out = a.out + (static_cast<size_t>(b) * T * H + h) * dv + row0 + r;
    for (int t = 0; t < T; ++t) {
        float kv[NC], qv[NC];
#pragma unroll
        for (int i = 0; i < NC / 4; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(sK + t * DK + c0 + 32 * i);
            const float4 y = *reinterpret_cast<const float4 *>(sQ + t * DK + c0 + 32 * i);
            kv[4 * i] = x.x; kv[4 * i + 1] = x.y; kv[4 * i + 2] = x.z; kv[4 * i + 3] = x.w;
            qv[4 * i] = y.x; qv[4 * i + 1] = y.y; qv[4 * i + 2] = y.z; qv[4 * i + 3] = y.w;
        }
        float sk = 0.f;                                           // (S_{t-1} k_t)_r
#pragma unroll
        for (int c = 0; c < NC; ++c) sk = fmaf(S[c], kv[c], sk);
#pragma unroll
        for (int m = 1; m < kLanesPerRow; m <<= 1) sk += __shfl_xor_sync(0xffffffffu, sk, m);
        const float alpha = sA[t];
        const float w = sB[t] * (sV[t * kRowsPerCta + r] - alpha * sk);
        float o = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            S[c] = fmaf(w, kv[c], alpha * S[c]);
            o = fmaf(S[c], qv[c], o);
        }
#pragma unroll
        for (int m = 1; m < kLanesPerRow; m <<= 1) o += __shfl_xor_sync(0xffffffffu, o, m);
        if ((tid % kLanesPerRow) == 0) out[static_cast<size_t>(t) * H * dv] = o;
        float4 *dst = reinterpret_cast<float4 *>(snap + t * snap_t);
#pragma unroll
        for (int i = 0; i < NC / 4; ++i) __stcs(dst + 8 * i, make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]));
    }
}

// One CTA per (head, sequence): copy snapshot p - 1 over the state.
__global__ void __launch_bounds__(kCopyThreads) nonreplay_accept_kernel(const NrArgs a, int dk)
{
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    pdl_wait();
    pdl_release();
    const int slot = a.state_idx ? a.state_idx[b] : b;
    if (slot < 0 || slot >= a.n_slot) {
        if (h == 0 && tid == 0) atomicOr(a.status, GDN_STATUS_BAD_SLOT);
        return;
    }
    const int p = a.accepted[b];
    if (p < 0 || p > a.T) {
        if (h == 0 && tid == 0) atomicOr(a.status, GDN_STATUS_BAD_ACCEPT);
        return;
    }
    if (p == 0) return;                                           // everything rejected
    const size_t n = static_cast<size_t>(a.dv) * dk;
    const float4 *src = reinterpret_cast<const float4 *>(a.snap + ((static_cast<size_t>(b) * a.H + h) * a.T + p - 1) * n);
    float4 *dst = reinterpret_cast<float4 *>(a.state_w + (static_cast<size_t>(slot) * a.H + h) * n);
    for (size_t i = tid; i < n / 4; i += kCopyThreads) dst[i] = __ldcs(src + i);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_nr(const gdn_replay_dims *d, const int32_t *state_idx) {
    if (!d) return GDN_ERR_NULL;
    if (d->in_dtype != GDN_DTYPE_BF16 && d->in_dtype != GDN_DTYPE_F32) return GDN_ERR_DTYPE;
    if (d->B < 0 || d->B > 65535 || d->H < 1 || d->H > 65535 || d->n_slot < 0) return GDN_ERR_DIMS;
    if (!state_idx && d->n_slot < d->B) return GDN_ERR_DIMS;
    if ((d->dk != 64 && d->dk != 128) || (d->dv != 64 && d->dv != 128)) return GDN_ERR_DIMS;
    if (d->T < 1 || d->T > 64 || d->flags != 0) return GDN_ERR_DIMS;
    return GDN_OK;
}

template <int DK, typename TIn>
int launch_nr_verify(const gdn_replay_dims *d, const NrArgs &a, cudaStream_t s) {
    const size_t smem = (2 * static_cast<size_t>(d->T) * DK + d->T * kRowsPerCta + 2 * d->T) * sizeof(float);
    auto kern = nonreplay_verify_kernel<DK, TIn>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    return launch_pdl(kern, dim3(d->dv / kRowsPerCta, d->H, d->B), dim3(kNrThreads), smem, s, a) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

}  // namespace

extern "C" int gdn_nonreplay_verify(const gdn_replay_dims *dims, const float *state, const int32_t *state_idx,
                                    const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, float *out, float *snap, int32_t *status,
                                    cudaStream_t stream) {
    const int rc = check_nr(dims, state_idx);
    if (rc) return rc;
    if (dims->B == 0) return GDN_OK;
    if (!state || !q || !k || !v || !g || !beta || !out || !snap || !status) return GDN_ERR_NULL;
    if (!aligned16(state) || !aligned16(snap)) return GDN_ERR_DIMS;
    NrArgs a = {state, nullptr, state_idx, q, k, v, g, beta, out, snap, nullptr, status,
                dims->B, dims->H, dims->T, dims->dv, dims->n_slot, dims->scale};
    const bool bf = dims->in_dtype == GDN_DTYPE_BF16;
    if (dims->dk == 128)
        return bf ? launch_nr_verify<128, __nv_bfloat16>(dims, a, stream) : launch_nr_verify<128, float>(dims, a, stream);
    return bf ? launch_nr_verify<64, __nv_bfloat16>(dims, a, stream) : launch_nr_verify<64, float>(dims, a, stream);
}

extern "C" int gdn_nonreplay_accept(const gdn_replay_dims *dims, float *state, const int32_t *state_idx,
                                    const float *snap, const int32_t *accepted, int32_t *status,
                                    cudaStream_t stream) {
    const int rc = check_nr(dims, state_idx);
    if (rc) return rc;
    if (dims->B == 0) return GDN_OK;
    if (!state || !snap || !accepted || !status) return GDN_ERR_NULL;
    if (!aligned16(state) || !aligned16(snap)) return GDN_ERR_DIMS;
    NrArgs a = {nullptr, state, state_idx, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                const_cast<float *>(snap), accepted, status,
                dims->B, dims->H, dims->T, dims->dv, dims->n_slot, dims->scale};
    return launch_pdl(nonreplay_accept_kernel, dim3(dims->H, dims->B), dim3(kCopyThreads), 0, stream, a,
                      dims->dk) == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// The baseline step for callers that cannot allocate device memory: the snapshots
// live in this fixed area (GDN_NONREPLAY_STATIC_SNAP_BYTES) instead of a caller
// buffer.  Host code must not hand the array's name to a kernel -- on the host it is
// only a stand-in for the symbol -- so its device address is looked up, on every call:
// a context created after a device reset loads the library again, possibly elsewhere.
static __device__ __align__(256) float g_static_snap[GDN_NONREPLAY_STATIC_SNAP_BYTES / sizeof(float)];

namespace {

// Device address of g_static_snap in the current context (the first lookup in a
// context loads the library's device code there).
int static_snap_address(float **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_snap) != cudaSuccess || !p) return GDN_ERR_LAUNCH;
    *out = static_cast<float *>(p);
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_nonreplay_step_static(const gdn_replay_dims *dims, float *state, const int32_t *state_idx,
                                         const void *q, const void *k, const void *v, const float *g,
                                         const float *beta, const int32_t *accepted, float *out,
                                         int32_t *status, cudaStream_t stream) {
    int rc = check_nr(dims, state_idx);
    if (rc) return rc;
    if (dims->B == 0) return GDN_OK;
    if (!state || !q || !k || !v || !g || !beta || !accepted || !out || !status) return GDN_ERR_NULL;
    const size_t need = static_cast<size_t>(dims->B) * dims->H * dims->T * dims->dv * dims->dk * sizeof(float);
    if (need > GDN_NONREPLAY_STATIC_SNAP_BYTES) return GDN_ERR_DIMS;
    float *snap = nullptr;
    if ((rc = static_snap_address(&snap)) != GDN_OK) return rc;
    if ((rc = gdn_nonreplay_verify(dims, state, state_idx, q, k, v, g, beta, out, snap, status, stream)) != GDN_OK)
        return rc;
    return gdn_nonreplay_accept(dims, state, state_idx, snap, accepted, status, stream);
}
