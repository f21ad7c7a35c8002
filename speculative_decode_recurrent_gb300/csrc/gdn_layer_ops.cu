// gdn_layer_ops.cu -- the GDN layer steps either side of the recurrence, for
// sm_103a: the causal convolution with pointer rollback, and the gated RMSNorm
// fused with FP8 (E4M3) quantisation.  C ABI and layouts: include/gdnlayer.h.
//
// Both are streaming kernels (a few flops per byte): the design goal is whole
// 16-byte vectors per thread, every load of a thread issued before its first use,
// and no intermediate written to HBM.  "The inference stack behind OCRia"
// (LlamaIndex engineering blog), section "Avoiding unnecessary memory transfers":
// fusing consecutive steps keeps their intermediates on chip.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "gdnlayer.h"
#include "replay_common.h"

namespace {

using gdn::launch_pdl;
using gdn::pdl_release;
using gdn::pdl_wait;

constexpr int kConvThreads = 128;
constexpr int kTaps = 4;            // widest kernel; narrower ones get leading zero taps
constexpr int kChunk = 8;           // draft tokens whose loads are in flight together

struct ConvArgs {
    void *ring;
    const int32_t *ring_pos;
    const int32_t *state_idx;
    const void *x;
    const float *weight, *bias;
    void *y;
    int32_t *status;
    int B, D, W, T, cap, n_slot, act;
};

// 16 bytes of inputs <-> floats
__device__ __forceinline__ void unpack(const uint4 &r, float (&f)[8]) {
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __bfloat1622float2(p[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}
__device__ __forceinline__ void unpack(const uint4 &r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}

template <typename T> struct Vec { static constexpr int N = 16 / sizeof(T); };

template <typename TOut, int V>
__device__ __forceinline__ void store_out(TOut *dst, const float (&v)[V]);
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16, 8>(__nv_bfloat16 *dst, const float (&v)[8]) {
    uint4 r;
    uint32_t *w = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&p);
    }
    *reinterpret_cast<uint4 *>(dst) = r;
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16, 4>(__nv_bfloat16 *dst, const float (&v)[4]) {
    uint2 r;
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]), p1 = __floats2bfloat162_rn(v[2], v[3]);
    r.x = *reinterpret_cast<const uint32_t *>(&p0);
    r.y = *reinterpret_cast<const uint32_t *>(&p1);
    *reinterpret_cast<uint2 *>(dst) = r;
}
template <>
__device__ __forceinline__ void store_out<float, 8>(float *dst, const float (&v)[8]) {
    reinterpret_cast<float4 *>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store_out<float, 4>(float *dst, const float (&v)[4]) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

// One thread owns V consecutive channels (one 16-byte input vector) of one
// sequence for every position: it reads the W-1 window vectors, then the draft
// vectors in chunks whose loads are all in flight before the first is used, emits
// the T outputs and stages the raw draft vectors in the ring.  No two threads touch
// the same bytes, so reading the window before staging needs no barrier.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(kConvThreads) conv_verify_kernel(const ConvArgs a)
{
    constexpr int V = Vec<TIn>::N;
    const int b = blockIdx.y;
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * V;
    pdl_wait();
    pdl_release();
    if (c0 >= a.D) return;
    const int slot = a.state_idx ? a.state_idx[b] : b;
    if (slot < 0 || slot >= a.n_slot) {
        if (c0 == 0) atomicOr(a.status, GDN_STATUS_BAD_SLOT);
        return;
    }
    const int pos = a.ring_pos[slot];
    if (pos < 0 || pos >= a.cap) {
        if (c0 == 0) atomicOr(a.status, GDN_STATUS_BAD_LEN);
        return;
    }
    const int D = a.D, W = a.W, T = a.T, cap = a.cap;
    TIn *ring = reinterpret_cast<TIn *>(a.ring) + static_cast<size_t>(slot) * cap * D + c0;
    const TIn *x = reinterpret_cast<const TIn *>(a.x) + static_cast<size_t>(b) * T * D + c0;
    TOut *y = reinterpret_cast<TOut *>(a.y) + static_cast<size_t>(b) * T * D + c0;

    // window: h[j] is input x_{j-3}; only the last W-1 exist for this kernel width
    uint4 hraw[kTaps - 1];
#pragma unroll
    for (int j = 0; j < kTaps - 1; ++j) {
        hraw[j] = make_uint4(0u, 0u, 0u, 0u);
        if (j >= kTaps - W) {
            const int r = (pos - (kTaps - 1) + j + cap) % cap;
            hraw[j] = *reinterpret_cast<const uint4 *>(ring + static_cast<size_t>(r) * D);
        }
    }
    // taps padded on the left: wt[i][j] multiplies x_{t-3+j}
    float wt[V][kTaps], bias[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        bias[i] = a.bias ? __ldg(a.bias + c0 + i) : 0.f;
#pragma unroll
        for (int j = 0; j < kTaps; ++j) {
            const int jj = j - (kTaps - W);
            wt[i][j] = jj >= 0 ? __ldg(a.weight + static_cast<size_t>(c0 + i) * W + jj) : 0.f;
        }
    }
    float h[kTaps - 1][V];
#pragma unroll
    for (int j = 0; j < kTaps - 1; ++j) unpack(hraw[j], h[j]);

    for (int t0 = 0; t0 < T; t0 += kChunk) {
        uint4 xr[kChunk];
#pragma unroll
        for (int u = 0; u < kChunk; ++u)
            xr[u] = t0 + u < T ? __ldg(reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t0 + u) * D))
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
            const int t = t0 + u;
            if (t >= T) break;
            float xv[V], o[V];
            unpack(xr[u], xv);
#pragma unroll
            for (int i = 0; i < V; ++i) {
                float acc = bias[i];
                acc = fmaf(wt[i][0], h[0][i], acc);
                acc = fmaf(wt[i][1], h[1][i], acc);
                acc = fmaf(wt[i][2], h[2][i], acc);
                acc = fmaf(wt[i][3], xv[i], acc);
                o[i] = a.act == GDN_CONV_ACT_SILU ? acc / (1.f + expf(-acc)) : acc;
            }
            store_out<TOut, V>(y + static_cast<size_t>(t) * D, o);
            const int r = (pos + t) % cap;
            *reinterpret_cast<uint4 *>(ring + static_cast<size_t>(r) * D) = xr[u];
#pragma unroll
            for (int i = 0; i < V; ++i) {
                h[0][i] = h[1][i];
                h[1][i] = h[2][i];
                h[2][i] = xv[i];
            }
        }
    }
}

__global__ void conv_accept_kernel(int32_t *ring_pos, const int32_t *state_idx, const int32_t *accepted,
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
    const int pos = ring_pos[slot];
    if (pos < 0 || pos >= cap) { atomicOr(status, GDN_STATUS_BAD_LEN); return; }
    ring_pos[slot] = (pos + p) % cap;
}

// ------------------------------------------------- gated RMSNorm + E4M3 codes
constexpr int kNormWarps = 8;

template <int E>
__device__ __forceinline__ void load_f32(const float *p, float (&v)[E]) {
    if constexpr (E == 8) {
        const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if constexpr (E == 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
        const float2 a = *reinterpret_cast<const float2 *>(p);
        v[0] = a.x; v[1] = a.y;
    }
}
template <int E>
__device__ __forceinline__ void load_gate(const __nv_bfloat16 *p, float (&v)[E]) {
#pragma unroll
    for (int i = 0; i < E; i += 2) {
        const float2 f = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(p)[i / 2]);
        v[i] = f.x;
        v[i + 1] = f.y;
    }
}
template <int E>
__device__ __forceinline__ void load_gate(const float *p, float (&v)[E]) { load_f32<E>(p, v); }

// One warp per row of D values; lane l owns elements E l .. E l + E - 1, so every
// load and the E-byte store of codes are contiguous across the warp.
template <int D, typename TZ>
__global__ void __launch_bounds__(kNormWarps * 32) gated_rmsnorm_fp8_kernel(
    int rows, const float *__restrict__ o, const TZ *__restrict__ z, const float *__restrict__ w,
    float eps, float inv_scale, uint8_t *__restrict__ q)
{
    constexpr int E = D / 32;
    pdl_wait();
    pdl_release();
    const int row = blockIdx.x * kNormWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= rows) return;
    const size_t base = static_cast<size_t>(row) * D + lane * E;
    float ov[E], zv[E], wv[E];
    load_f32<E>(o + base, ov);
    load_gate<E>(z + base, zv);
    load_f32<E>(w + lane * E, wv);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) ss = fmaf(ov[i], ov[i], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = 1.f / sqrtf(ss / D + eps);
    uint8_t codes[E];
#pragma unroll
    for (int i = 0; i < E; i += 2) {
        float v[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float g = zv[i + k] / (1.f + expf(-zv[i + k]));
            v[k] = ov[i + k] * r * wv[i + k] * g * inv_scale;
        }
        const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(make_float2(v[0], v[1]), __NV_SATFINITE, __NV_E4M3);
        codes[i] = static_cast<uint8_t>(p & 0xffu);
        codes[i + 1] = static_cast<uint8_t>(p >> 8);
    }
    if constexpr (E == 8) {
        uint2 out;
        out.x = codes[0] | (codes[1] << 8) | (codes[2] << 16) | (static_cast<uint32_t>(codes[3]) << 24);
        out.y = codes[4] | (codes[5] << 8) | (codes[6] << 16) | (static_cast<uint32_t>(codes[7]) << 24);
        *reinterpret_cast<uint2 *>(q + base) = out;
    } else if constexpr (E == 4) {
        *reinterpret_cast<uint32_t *>(q + base) =
            codes[0] | (codes[1] << 8) | (codes[2] << 16) | (static_cast<uint32_t>(codes[3]) << 24);
    } else {
        *reinterpret_cast<uint16_t *>(q + base) = static_cast<uint16_t>(codes[0] | (codes[1] << 8));
    }
}

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

int check_conv(const gdn_conv_dims *d) {
    if (!d) return GDN_ERR_NULL;
    if ((d->in_dtype != GDN_DTYPE_BF16 && d->in_dtype != GDN_DTYPE_F32) ||
        (d->out_dtype != GDN_DTYPE_BF16 && d->out_dtype != GDN_DTYPE_F32))
        return GDN_ERR_DTYPE;
    if (d->B < 0 || d->n_slot < d->B || d->D < 8 || d->D % 8 != 0) return GDN_ERR_DIMS;
    if (d->W < 1 || d->W > kTaps || d->T < 1 || d->T > 64) return GDN_ERR_DIMS;
    if (d->cap < d->W - 1 + d->T || d->cap > 4096) return GDN_ERR_DIMS;
    if (d->act != GDN_CONV_ACT_NONE && d->act != GDN_CONV_ACT_SILU) return GDN_ERR_DIMS;
    if (static_cast<long long>(d->n_slot) * d->cap * d->D > 0x7fffffffLL) return GDN_ERR_DIMS;
    return GDN_OK;
}

template <typename TIn, typename TOut>
int launch_conv(const gdn_conv_dims *d, const ConvArgs &a, cudaStream_t s) {
    constexpr int V = Vec<TIn>::N;
    const int vecs = d->D / V;
    const dim3 grid((vecs + kConvThreads - 1) / kConvThreads, d->B);
    return launch_pdl(conv_verify_kernel<TIn, TOut>, grid, dim3(kConvThreads), 0, s, a) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

template <int D>
int launch_norm(int rows, const float *o, const void *z, int32_t z_dtype, const float *w, float eps,
                float inv_scale, uint8_t *q, cudaStream_t s) {
    const dim3 grid((rows + kNormWarps - 1) / kNormWarps);
    const cudaError_t e =
        z_dtype == GDN_DTYPE_BF16
            ? launch_pdl(gated_rmsnorm_fp8_kernel<D, __nv_bfloat16>, grid, dim3(kNormWarps * 32), 0, s, rows, o,
                         static_cast<const __nv_bfloat16 *>(z), w, eps, inv_scale, q)
            : launch_pdl(gated_rmsnorm_fp8_kernel<D, float>, grid, dim3(kNormWarps * 32), 0, s, rows, o,
                         static_cast<const float *>(z), w, eps, inv_scale, q);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int gdn_conv_verify(const gdn_conv_dims *d, void *ring, const int32_t *ring_pos, const int32_t *state_idx,
                    const void *x, const float *weight, const float *bias, void *y, int32_t *status,
                    cudaStream_t stream)
{
    const int rc = check_conv(d);
    if (rc) return rc;
    if (d->B == 0) return GDN_OK;
    if (!ring || !ring_pos || !x || !weight || !y || !status) return GDN_ERR_NULL;
    if (!aligned(ring, 16) || !aligned(x, 16) || !aligned(y, 16) || !aligned(weight, 4) ||
        (bias && !aligned(bias, 4)))
        return GDN_ERR_DIMS;
    ConvArgs a{ring, ring_pos, state_idx, x, weight, bias, y, status,
               d->B, d->D, d->W, d->T, d->cap, d->n_slot, d->act};
    const bool in_bf = d->in_dtype == GDN_DTYPE_BF16, out_bf = d->out_dtype == GDN_DTYPE_BF16;
    if (in_bf) return out_bf ? launch_conv<__nv_bfloat16, __nv_bfloat16>(d, a, stream)
                             : launch_conv<__nv_bfloat16, float>(d, a, stream);
    return out_bf ? launch_conv<float, __nv_bfloat16>(d, a, stream) : launch_conv<float, float>(d, a, stream);
}

int gdn_conv_accept(const gdn_conv_dims *d, int32_t *ring_pos, const int32_t *state_idx,
                    const int32_t *accepted, int32_t *status, cudaStream_t stream)
{
    const int rc = check_conv(d);
    if (rc) return rc;
    if (d->B == 0) return GDN_OK;
    if (!ring_pos || !accepted || !status) return GDN_ERR_NULL;
    return launch_pdl(conv_accept_kernel, dim3((d->B + 127) / 128), dim3(128), 0, stream, ring_pos, state_idx,
                      accepted, d->B, d->n_slot, d->T, d->cap, status) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

int gdn_gated_rmsnorm_fp8(int32_t rows, int32_t d, const float *o, const void *z, int32_t z_dtype,
                          const float *weight, float eps, float inv_scale, uint8_t *q, cudaStream_t stream)
{
    if (rows < 0 || (d != 64 && d != 128 && d != 256)) return GDN_ERR_DIMS;
    if (z_dtype != GDN_DTYPE_BF16 && z_dtype != GDN_DTYPE_F32) return GDN_ERR_DTYPE;
    if (!(eps >= 0.f) || !(inv_scale > 0.f)) return GDN_ERR_DIMS;
    if (rows == 0) return GDN_OK;
    if (!o || !z || !weight || !q) return GDN_ERR_NULL;
    if (!aligned(o, 16) || !aligned(z, 16) || !aligned(weight, 16) || !aligned(q, 8)) return GDN_ERR_DIMS;
    switch (d) {
        case 64: return launch_norm<64>(rows, o, z, z_dtype, weight, eps, inv_scale, q, stream);
        case 128: return launch_norm<128>(rows, o, z, z_dtype, weight, eps, inv_scale, q, stream);
        default: return launch_norm<256>(rows, o, z, z_dtype, weight, eps, inv_scale, q, stream);
    }
}

}  // extern "C"
