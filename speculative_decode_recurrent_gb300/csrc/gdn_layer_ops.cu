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
constexpr int kTaps = 4;            // widest kernel
constexpr int kChunk = 4;           // draft positions per thread (8: 4 % slower, 2: 15 % slower)

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

// Four consecutive channels of an input row: 8 bytes of bf16 or 16 bytes of fp32.
template <typename TIn> struct In4;
template <> struct In4<__nv_bfloat16> {
    using Raw = uint2;
    __device__ static void unpack(const uint2 &r, float (&f)[4]) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
};
template <> struct In4<float> {
    using Raw = uint4;
    __device__ static void unpack(const uint4 &r, float (&f)[4]) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
};

template <typename TOut>
__device__ __forceinline__ void store_out4(TOut *dst, const float (&v)[4]);
template <>
__device__ __forceinline__ void store_out4<__nv_bfloat16>(__nv_bfloat16 *dst, const float (&v)[4]) {
    uint2 r;
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]), p1 = __floats2bfloat162_rn(v[2], v[3]);
    r.x = *reinterpret_cast<const uint32_t *>(&p0);
    r.y = *reinterpret_cast<const uint32_t *>(&p1);
    *reinterpret_cast<uint2 *>(dst) = r;
}
template <>
__device__ __forceinline__ void store_out4<float>(float *dst, const float (&v)[4]) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

// One thread owns 4 consecutive channels of one sequence for a chunk of kChunk draft
// positions (a warp covers 128 channels: whole 128-byte lines for bf16 rows): it reads
// the W-1 inputs before its chunk (from the ring for the first chunk, from the draft
// otherwise) and the chunk's draft inputs, all requested before the first is used,
// emits the outputs and stages its raw draft inputs in the ring.  Staged positions
// pos .. pos+T-1 never meet the window pos-W+1 .. pos-1 (cap >= W - 1 + T), and no two
// threads write the same bytes, so no barrier is needed.  64 registers at W = 4 with
// bf16 rows: eight CTAs per SM, so the decode shape's 1536 CTAs run in about 1.3 waves
// (chunks of 8 positions fit in one wave but keep fewer loads in flight: 4 % slower).
template <typename TIn, typename TOut, int W>
__global__ void __launch_bounds__(kConvThreads) conv_verify_kernel(const ConvArgs a)
{
    using Raw = typename In4<TIn>::Raw;
    const int b = blockIdx.y, t0 = blockIdx.z * kChunk;
    const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 4;
    pdl_wait();
    pdl_release();
    if (c0 >= a.D) return;
    const int D = a.D, T = a.T, cap = a.cap;
    const TIn *x = reinterpret_cast<const TIn *>(a.x) + static_cast<size_t>(b) * T * D + c0;
    TOut *y = reinterpret_cast<TOut *>(a.y) + static_cast<size_t>(b) * T * D + c0;

    // inputs x_{t0-W+1} .. x_{t0-1}, then the chunk.  The draft rows (the chunk, and the
    // window past the first chunk) do not depend on the ring position: they are in
    // flight while the slot and the position are read.
    Raw hraw[W > 1 ? W - 1 : 1], xr[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
        if (t0 + u < T) xr[u] = __ldg(reinterpret_cast<const Raw *>(x + static_cast<size_t>(t0 + u) * D));
    }
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
        const int u = t0 - (W - 1) + j;
        if (u >= 0) hraw[j] = __ldg(reinterpret_cast<const Raw *>(x + static_cast<size_t>(u) * D));
    }
    // the 4 channels' taps: 4 W consecutive floats
    float wt[4 * W], bias[4];
#pragma unroll
    for (int q = 0; q < W; ++q) {
        const float4 w4 = __ldg(reinterpret_cast<const float4 *>(a.weight + static_cast<size_t>(c0) * W) + q);
        wt[4 * q] = w4.x; wt[4 * q + 1] = w4.y; wt[4 * q + 2] = w4.z; wt[4 * q + 3] = w4.w;
    }
    if (a.bias) {
        const float4 b4 = __ldg(reinterpret_cast<const float4 *>(a.bias + c0));
        bias[0] = b4.x; bias[1] = b4.y; bias[2] = b4.z; bias[3] = b4.w;
    } else {
        bias[0] = bias[1] = bias[2] = bias[3] = 0.f;
    }
    const int slot = a.state_idx ? a.state_idx[b] : b;
    if (slot < 0 || slot >= a.n_slot) {
        if (c0 == 0 && t0 == 0) atomicOr(a.status, GDN_STATUS_BAD_SLOT);
        return;
    }
    const int pos = a.ring_pos[slot];
    if (pos < 0 || pos >= a.cap) {
        if (c0 == 0 && t0 == 0) atomicOr(a.status, GDN_STATUS_BAD_LEN);
        return;
    }
    TIn *ring = reinterpret_cast<TIn *>(a.ring) + static_cast<size_t>(slot) * cap * D + c0;
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {                    // the committed window (first chunk)
        const int u = t0 - (W - 1) + j;
        if (u < 0) hraw[j] = __ldg(reinterpret_cast<const Raw *>(ring + static_cast<size_t>(u + pos + cap) % cap * D));
    }
    float h[W][4];                                       // h[W-1] is the current input
#pragma unroll
    for (int j = 0; j < W - 1; ++j) In4<TIn>::unpack(hraw[j], h[j]);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
        const int t = t0 + u;
        if (t >= T) break;
        In4<TIn>::unpack(xr[u], h[W - 1]);
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float acc = bias[i];
#pragma unroll
            for (int j = 0; j < W; ++j) acc = fmaf(wt[i * W + j], h[j][i], acc);
            o[i] = a.act == GDN_CONV_ACT_SILU ? __fdividef(acc, 1.f + __expf(-acc)) : acc;   // 0 below -87
        }
        store_out4<TOut>(y + static_cast<size_t>(t) * D, o);
        *reinterpret_cast<Raw *>(ring + static_cast<size_t>((pos + t) % cap) * D) = xr[u];
#pragma unroll
        for (int j = 0; j + 1 < W; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) h[j][i] = h[j + 1][i];
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
            const float g = __fdividef(zv[i + k], 1.f + __expf(-zv[i + k]));   // silu; 0 below -87
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

template <typename TIn, typename TOut, int W>
int launch_conv_w(const gdn_conv_dims *d, const ConvArgs &a, cudaStream_t s) {
    const int vecs = d->D / 4;
    const dim3 grid((vecs + kConvThreads - 1) / kConvThreads, d->B, (d->T + kChunk - 1) / kChunk);
    return launch_pdl(conv_verify_kernel<TIn, TOut, W>, grid, dim3(kConvThreads), 0, s, a) == cudaSuccess
               ? GDN_OK : GDN_ERR_LAUNCH;
}

template <typename TIn, typename TOut>
int launch_conv(const gdn_conv_dims *d, const ConvArgs &a, cudaStream_t s) {
    switch (d->W) {
        case 1: return launch_conv_w<TIn, TOut, 1>(d, a, s);
        case 2: return launch_conv_w<TIn, TOut, 2>(d, a, s);
        case 3: return launch_conv_w<TIn, TOut, 3>(d, a, s);
        default: return launch_conv_w<TIn, TOut, 4>(d, a, s);
    }
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
    if (!aligned(ring, 16) || !aligned(x, 16) || !aligned(y, 16) || !aligned(weight, 16) ||
        (bias && !aligned(bias, 16)))
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
